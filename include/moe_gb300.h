/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) MoE-LoRA expert layer.
 *
 * The layer is the MoE expert block that the Unsloth "Faster MoE" docs and the
 * Unsloth x NVIDIA training article optimise for LoRA fine-tuning:
 *
 *   routing   flatten the [T,k] top-k expert ids, stable-sort them by expert id,
 *             count them with one bincount, turn the counts into offsets and
 *             permute the token rows once (article, section "Optimisation 3:
 *             MoE routing done in one grouped pass", steps 1-5);
 *   experts   per expert a SwiGLU MLP, gate_up then down, with "split LoRA":
 *             X W^T + s (X A^T) B^T, never forming B A (docs, sections "What is
 *             torch._grouped_mm" and "Faster LoRA MoE training"; the
 *             split-LoRA equations of "Implementation details");
 *   combine   Y[t] = sum_j w[t,j] * expert_{ids[t,j]}(X[t]) (the plain top-k
 *             mixture; the pages do not print this step);
 *   backward  dX, the routing-weight gradient and dA, dB of both adapters for
 *             frozen base weights (docs: the router and base weights are frozen,
 *             "loss, gradients and outputs are unchanged").
 *
 * Conventions for every call
 *   - Every pointer is caller-owned DEVICE memory unless stated otherwise.  The
 *     library never allocates or frees device memory and never synchronises,
 *     except moe_status(), which synchronises the given stream.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Calls are stream-ordered; results are valid once the stream
 *     reaches them.
 *   - Tensors are dense row-major.  bf16 values are passed as 16-bit patterns
 *     (moe_bf16).  Every bf16 matrix row must start on a 16-byte boundary: the
 *     base pointers 16-byte aligned and d, f, r multiples of 8.
 *   - Argument errors are detected on the host before anything is launched and
 *     returned synchronously (MOE_ERR_INVALID_ARG / MOE_ERR_WORKSPACE /
 *     MOE_ERR_UNSUPPORTED); moe_last_error() then describes the problem.
 *     Launch failures return MOE_ERR_CUDA.  Errors found by kernels (an expert
 *     id outside [0,E), a pipeline wait that timed out) are recorded in a
 *     per-device status word read by moe_status().
 *   - Determinism: no floating-point atomics; equal inputs give bit-identical
 *     outputs.
 *
 * Notation
 *   T tokens, d hidden size, f expert intermediate size, E routed experts,
 *   k experts per token, r LoRA rank, s = lora_scale = alpha / r.
 *   shared_expert = 1 adds one always-active expert with weight 1 (group E).
 *   G = E + shared_expert expert groups, K = k + shared_expert slots per token,
 *   N = T * K routed rows (flat index i = t*K + j; slot j = k is the shared one).
 *
 * Permuted row layout used between calls
 *   Permuted buffers have N rows in sorted order: row p holds sorted position
 *   p, so expert g's rows are the contiguous slice [offsets[g], offsets[g+1])
 *   (article step 5, "slice the token list by offsets").  The grouped GEMMs
 *   cut each slice into 128-row tiles (MOE_TILE_M) that start at offsets[g];
 *   tile_off numbers those tiles.  A tile's last rows may run into the next
 *   expert's slice: they are computed but never stored.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;                 /* bf16 bit pattern */
typedef struct CUstream_st* moe_stream_t;  /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer */
  MOE_ERR_UNSUPPORTED = -2, /* valid but outside what this library supports */
  MOE_ERR_WORKSPACE = -3,   /* workspace too small */
  MOE_ERR_CUDA = -4,        /* a CUDA runtime / driver call failed */
  MOE_ERR_BAD_IDS = -5,     /* (device) an expert id outside [0,E) was seen */
  MOE_ERR_TIMEOUT = -6      /* (device) a pipeline wait gave up */
} moe_status_t;

#define MOE_TILE_M 128      /* rows per grouped-GEMM tile */
#define MOE_MAX_EXPERTS 1024

typedef struct moe_dims {
  int32_t T, d, f, E, k, r;
  float lora_scale;        /* s = alpha / r */
  int32_t shared_expert;   /* 0 or 1 */
} moe_dims;

/* ------------------------------------------------------------------------ */
/* Router (upstream of the layer; the docs keep the router frozen).          */
/* ------------------------------------------------------------------------ */

/* Softmax over the E logits of each token, top-k by descending logit (equal
 * logits: lower expert id first), weights renormalised to sum to one -- the
 * router rule of the layer workloads.  The renormalised weights equal a
 * softmax over the k selected logits, which is what is computed (fp32).
 *   logits  [T,E] fp32 (read)        ids [T,k] int32 (written)
 *   weights [T,k] fp32 (written)     1 <= k <= min(E, 32), E <= MOE_MAX_EXPERTS */
MOE_API int moe_router_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                    int32_t* ids, float* weights, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Routing: article section "Optimisation 3", steps 1-5.                     */
/* ------------------------------------------------------------------------ */

/* The router and the routing pass in one call, from the logits: the top-k
 * ids and renormalised weights of moe_router_topk (written to ids [T,k] and
 * weights [T,k]), then the routing tables of moe_route from those ids, all
 * enqueued on `stream` with no host round trip in between.  Same arguments,
 * checks and results as the two calls in sequence; every check runs before
 * anything is launched. */
MOE_API int moe_route_logits(const float* logits, int32_t T, int32_t E, int32_t k,
                             int32_t shared_expert, int32_t* ids, float* weights,
                             int32_t* counts, int32_t* offsets, int32_t* tile_off,
                             int32_t* sorted_src, int32_t* dest_pos, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Bytes of scratch moe_route needs for T tokens, K slots, G groups. */
MOE_API size_t moe_route_workspace_size(int32_t T, int32_t K, int32_t G);

/* Kernels moe_route (and moe_route_noalloc) launch for T tokens, K slots and
 * G groups: 3 (per-chunk histogram, scan over chunks, scatter), or 2 when
 * there are at most 64 chunks and the scatter kernel scans the histogram
 * itself.  MOE_ERR_INVALID_ARG for a non-positive size. */
MOE_API int32_t moe_route_kernel_count(int32_t T, int32_t K, int32_t G);

/* Flatten ids [T,k] row-major (the shared slot j = k carries id E when
 * shared_expert = 1), stable-sort by expert id, bincount, offsets:
 *   counts    [G]    counts[g] = #{i : id(i) = g}
 *   offsets   [G+1]  exclusive prefix sum of counts
 *   tile_off  [G+1]  exclusive prefix sum of ceil(counts / MOE_TILE_M)
 *   sorted_src[N]    flat index i at each sorted position (stable: equal ids
 *                    keep ascending i)
 *   dest_pos  [N]    inverse permutation: sorted_src[dest_pos[i]] = i
 * No data-dependent value reaches the host.  An id outside [0,E) sets
 * MOE_ERR_BAD_IDS in the status word; that assignment is left out of counts
 * and its dest_pos is -1 (sorted positions past the valid total are -1).
 * ws: device scratch of at least moe_route_workspace_size() bytes, 16-byte
 * aligned; its contents need no initialisation. */
MOE_API int moe_route(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t shared_expert,
              int32_t* counts, int32_t* offsets, int32_t* tile_off,
              int32_t* sorted_src, int32_t* dest_pos,
              void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_route without a workspace argument.  The pages have no counterpart to
 * this call; it exists for callers that cannot allocate device memory: hosts
 * that own all device memory through their own pool and hand a library only
 * raw pointers and a stream (plugin interfaces whose enqueue step must not
 * allocate, serving runtimes that forbid allocation after start-up).
 * Same arguments and results as moe_route, minus ws / ws_bytes.  The routing
 * histogram lives in a 2 MiB array inside this library, which every GPU that
 * loads the library holds until the process exits; this call itself never
 * allocates or frees memory.  Limit: the histogram moe_route would need,
 * moe_route_workspace_size(T, k + shared_expert, E + shared_expert), must not
 * exceed 2 MiB (e.g. up to 256 experts with 8,388,608 routed rows); larger
 * problems return MOE_ERR_WORKSPACE -- use moe_route with a workspace for them.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array: calls whose work overlaps on the
 * GPU (other streams, other threads) race on it and must be serialised by the
 * caller.  The array is never cleared; no result depends on its old contents.
 * It accepts exactly the shapes moe_route accepts (plus the 2 MiB limit), and
 * the timing probe traces it under the kernel name "route", like moe_route. */
MOE_API int moe_route_noalloc(const int32_t* ids, int32_t T, int32_t k, int32_t E,
                              int32_t shared_expert, int32_t* counts, int32_t* offsets,
                              int32_t* tile_off, int32_t* sorted_src, int32_t* dest_pos,
                              moe_stream_t stream);

/* Row permute (article step 5, "slice the token list by offsets"): every
 * token's row goes to the sorted positions of its slots,
 *   dst[dest_pos[t*K + j], :] = src[t, :]   for j < K, dest_pos >= 0,
 * i.e. dst[p] = src[sorted_src[p] / K] for every valid sorted position p.
 *   src [T,d] bf16 (each row read once);  dst [N,d] bf16 (N = T*K).  Used for
 *   X (forward) and for the upstream gradient dY (backward).  K <= 33. */
MOE_API int moe_permute(const moe_bf16* src, int32_t T, int32_t d, int32_t K,
                        const int32_t* dest_pos, moe_bf16* dst, moe_stream_t stream);

/* Combine (unpermute + reduce): for every token t, with p(t,j) = dest_pos[t*K+j]
 * the permuted row of slot j:
 *   out[t,:] = bf16( sum_{j<K} c_j * rows[p(t,j),:] ),  fp32 sum in j order,
 *   c_j = weights[t,j] for j < k and 1 for the shared slot, or c_j = 1 when
 *   weights is NULL (rows already scaled, or a gradient sum);
 *   slot_out[t,j] = row_scalars[p(t,j)] for j < k when both are non-NULL.
 *   rows [N,d] bf16; out [T,d] bf16; weights [T,k] fp32 or NULL;
 *   row_scalars [N] fp32 or NULL; slot_out [T,k] fp32 or NULL.
 * Slots with dest_pos = -1 (out-of-range ids) contribute nothing. */
MOE_API int moe_unpermute_combine(const moe_bf16* rows, const int32_t* dest_pos, int32_t T,
                                  int32_t d, int32_t k, int32_t shared_expert,
                                  const float* weights, const float* row_scalars,
                                  float* slot_out, moe_bf16* out, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Grouped split-LoRA SwiGLU expert MLP (docs: "Faster LoRA MoE training",    */
/* "Implementation details").                                                */
/* ------------------------------------------------------------------------ */
/* Weights, all bf16, row-major, G groups (shared expert last):
 *   W_gu [G,2f,d]  rows [0,f) gate, rows [f,2f) up   A_gu [G,r,d]  B_gu [G,2f,r]
 *   W_dn [G,d,f]                                      A_dn [G,r,f]  B_dn [G,d,r]
 * Per permuted row p of group g with routing weight w_p (w of its slot; 1 for
 * the shared slot):
 *   xa   = Xp A_gu^T             h = Xp W_gu^T + s xa B_gu^T      [.,2f]
 *   act  = silu(h[:, :f]) * h[:, f:]                               [.,f]
 *   xa_dn = act A_dn^T           o = act W_dn^T + s xa_dn B_dn^T  [.,d]
 *   Yp   = w_p * o
 * B A is never formed.  Accumulation is fp32 on tensor cores. */

/* Precision of saved intermediates.  Every value that later feeds a sum over
 * the rows of an expert (the LoRA weight gradients and the routing-weight
 * gradient) keeps ~16 significant bits: h is stored in fp32 (interleaved in
 * 16-feature chunks so that each chunk is one 128-byte line), and the other
 * such intermediates as "pair" buffers [2, P, cols] of bf16 with
 * value = pair[0] + pair[1] (pair[0] = bf16(v), pair[1] = bf16(v - pair[0])).
 * The tensor cores consume a pair as two bf16 operands (extra K steps).
 * Here P = N = T * K (permuted rows). */

/* Forward.  Row input: either Xp = moe_permute(X) [P,d], or X itself [T,d]
 * with Xp = NULL, in which case the GEMMs gather each permuted row's token row
 * straight from X while loading it (16-byte cp.async copies picked by
 * sorted_src; no permuted copy is made).  The permuted input is the faster
 * of the two on GB300 (its tiles load with TMA); the gathered one needs no
 * [P,d] buffer.
 * Other inputs: the routing outputs (counts is
 * not read; offsets and tile_off define the tiles, sorted_src locates each
 * row's routing weight), topk weights [T,k] fp32, the six weight tensors.  Outputs:
 *   Yp    [P,d]    bf16  w-scaled expert outputs (feed moe_unpermute_combine
 *                        with weights = NULL)
 *   h     [P,hs]   fp32  saved gate and up pre-activations, hs = 32*ceil(f/16):
 *                        features in chunks of 16, row layout
 *                        [gate c*16..c*16+15 | up c*16..c*16+15] for chunk c
 *   act   [2,P,f]  bf16 pair  saved w_p * silu(gate) * up (scaled by the row's
 *                              routing weight w_p; 1 for shared-expert rows)
 *   xa_gu [2,P,r]  bf16 pair  saved s * Xp A_gu^T
 *   xa_dn [2,P,r]  bf16 pair  saved s * act A_dn^T (so also scaled by w_p)
 * The down projection consumes the high halves: Yp = act W_dn^T + xa_dn B_dn^T
 * is w_p * o without a separate scaling step (Yp is a bf16 output). */
MOE_API int moe_lora_grouped_mlp_fwd(const moe_dims* dims, const moe_bf16* Xp,
                             const moe_bf16* X, const int32_t* counts, const int32_t* offsets,
                             const int32_t* tile_off, const int32_t* sorted_src,
                             const float* topk_w,
                             const moe_bf16* W_gu, const moe_bf16* A_gu, const moe_bf16* B_gu,
                             const moe_bf16* W_dn, const moe_bf16* A_dn, const moe_bf16* B_dn,
                             moe_bf16* Yp, float* h, moe_bf16* act,
                             moe_bf16* xa_gu, moe_bf16* xa_dn, moe_stream_t stream);

/* Bytes of scratch moe_lora_grouped_mlp_bwd needs. */
MOE_API size_t moe_mlp_bwd_workspace_size(const moe_dims* dims);

/* Backward for frozen W (and frozen router).  Row inputs as in the forward:
 * dYp = moe_permute of the upstream gradient dY (unscaled) or dY itself [T,d]
 * with dYp = NULL (gathered), and Xp or X likewise; h, act, xa_gu, xa_dn as
 * saved by the forward.  With dO = w_p dYp:
 *   dw_rows[p] = <dYp_p, o_p> = <act_p, g_p>  [P] fp32, the gradient of the
 *                routing weight of row p (moe_unpermute_combine gathers it
 *                to [T,k] through row_scalars / slot_out)
 *   g = dYp W_dn + s u A_dn with u = dYp B_dn;  dact = w_p g
 *   dh = [dact*up*silu'(gate) | dact*silu(gate)];  v = dh B_gu
 *   dXp = dh W_gu + s v A_gu              [P,d] bf16 (combine -> dX)
 *   dB_dn[g] = s sum_p dO^T (act_p A_dn^T) = sum_p dYp^T xa_dn   [G,d,r] fp32
 *   dA_dn[g] = s sum_p (dO B_dn)^T act_p = sum_p (s u)^T act       [G,r,f] fp32
 *              (act_p unscaled; the saved act and xa_dn already carry w_p)
 *   dB_gu[g] = s sum_p dh^T xa             [G,2f,r] fp32
 *   dA_gu[g] = s sum_p v^T Xp              [G,r,d] fp32
 * Full fine-tuning (optional; the Faster MoE docs' introduction: the kernels
 * serve full fine-tuning as well as LoRA): with dW_gu and/or dW_dn non-NULL
 * the call also writes the gradients of the expert weights themselves,
 *   dW_dn[g] = sum_p dO^T act_p = sum_p dYp^T act   [G,d,f]  fp32
 *   dW_gu[g] = sum_p dh^T Xp                        [G,2f,d] fp32
 * (act and dh as hi/lo pairs, so the sums keep ~16-bit terms).  They need the
 * permuted rows (Xp and dYp non-NULL), else MOE_ERR_UNSUPPORTED.
 * Gradients are overwritten (not accumulated); groups with no rows get zeros.
 * With a shared expert (which sees every token), the LoRA gradients of each
 * group with more than max(1024, 1.25 x the mean group) rows are summed in
 * parts of that many rows, and the parts' fp32 sums added in part order, so
 * results stay bit-for-bit reproducible.
 * ws: >= moe_mlp_bwd_workspace_size bytes of device scratch, 16-byte aligned
 * (the dh, u and v intermediates, dw partials, and the parts' partial sums
 * with their arrival counters, which the call zeroes on its own stream).
 * The weight-gradient GEMMs run on a second stream that the library
 * creates once per device (no device memory); it forks from `stream` after
 * their inputs exist and joins back before the call returns, so all results
 * are ordered on `stream` as if everything ran there.  Calls from several host
 * threads serialise their enqueueing on that stream. */
MOE_API int moe_lora_grouped_mlp_bwd(const moe_dims* dims, const moe_bf16* dYp,
                             const moe_bf16* dY, const moe_bf16* Xp, const moe_bf16* X,
                             const int32_t* counts, const int32_t* offsets,
                             const int32_t* tile_off, const int32_t* sorted_src,
                             const float* topk_w,
                             const moe_bf16* W_gu, const moe_bf16* A_gu, const moe_bf16* B_gu,
                             const moe_bf16* W_dn, const moe_bf16* A_dn, const moe_bf16* B_dn,
                             const float* h, const moe_bf16* act,
                             const moe_bf16* xa_gu, const moe_bf16* xa_dn,
                             moe_bf16* dXp, float* dw_rows,
                             float* dA_gu, float* dB_gu, float* dA_dn, float* dB_dn,
                             float* dW_gu, float* dW_dn,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Expert parallelism                                                        */
/* ------------------------------------------------------------------------ */
/* With the experts split into contiguous ranges over P ranks (the Unsloth x
 * NVIDIA article's closing section points multi-GPU training at data and
 * expert sharding), a rank's permuted rows for the experts of rank q are the
 * contiguous slice [offsets[e_q], offsets[e_{q+1}]) of its sorted order, so
 * one all-to-all per direction moves them (the collective itself is the
 * caller's: NCCL through torch.distributed in the Python layer).  Received
 * rows arrive rank-major, expert-minor; moe_route on their local expert ids
 * (moe_ep_segment_ids) regroups them by expert, moe_permute with K = 1 moves
 * them, and moe_unpermute_combine with K = 1 moves results back.  These two
 * calls are the only kernels expert parallelism adds. */

/* Blocks (rank, local expert) a received-row count matrix may have. */
#define MOE_EP_MAX_BLOCKS 16384

/* Routing weight of every sorted position, so it can travel with its row:
 *   row_w[dest_pos[t*K + j]] = topk_w[t, j]  (j < k),  1 for the shared slot
 * (K = k + shared_expert).  topk_w [T,k] fp32, dest_pos [T*K] from moe_route
 * (entries < 0, bad ids, are skipped), row_w [T*K] fp32. */
MOE_API int moe_ep_row_weights(const float* topk_w, const int32_t* dest_pos, int32_t T,
                               int32_t k, int32_t shared_expert, float* row_w,
                               moe_stream_t stream);

/* Local expert id of every received row.  counts [P, E_loc] int32 (device):
 * counts[r, e] rows from rank r for local expert e, received rank-major then
 * expert-minor; ids [n_rows] int32 gets e for each of them.  n_rows must equal
 * the sum of counts: otherwise nothing is written and MOE_ERR_BAD_IDS is
 * recorded in the status word.  P * E_loc <= MOE_EP_MAX_BLOCKS.  n_rows = 0 is
 * a no-op. */
MOE_API int moe_ep_segment_ids(const int32_t* counts, int32_t P, int32_t E_loc, int64_t n_rows,
                               int32_t* ids, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */

/* Synchronises `stream`, then returns and clears the current device's status
 * word: MOE_OK, MOE_ERR_BAD_IDS or MOE_ERR_TIMEOUT (first error recorded), or
 * MOE_ERR_CUDA if the synchronisation itself failed. */
MOE_API int moe_status(moe_stream_t stream);

/* Message for the last error returned on this thread ("" if none). */
MOE_API const char* moe_last_error(void);

/* Self-test of the failure path that every pipeline wait of the GEMM kernels
 * takes: enqueues one GPU thread that waits on an mbarrier no one arrives on,
 * bounded by timeout_us microseconds (1 .. 2,000,000), through the same wait
 * routine; when the limit passes it records MOE_ERR_TIMEOUT in the device
 * status word and returns, leaving the context usable.  moe_status(stream)
 * then returns MOE_ERR_TIMEOUT.  Returns MOE_OK once enqueued, or
 * MOE_ERR_INVALID_ARG for a timeout out of range. */
MOE_API int moe_selftest_wait_timeout(uint32_t timeout_us, moe_stream_t stream);

/* Read-stream probe (measurement): reads `bytes` of device memory at `src`
 * into shared memory with the asynchronous copies the grouped GEMMs load
 * their operands with, one CTA per SM, computes nothing and discards them.
 * Timing it (caller-owned events on `stream`) gives the rate at which this
 * GPU streams reads alone -- the ceiling for read-dominated kernels, which a
 * copy peak (reads and writes mixed) does not show.  Patterns:
 *   MOE_PROBE_LINEAR  32 KB bulk copies, neighbouring CTAs on neighbouring
 *                     chunks; bytes a multiple of 16
 *   MOE_PROBE_TILES   src as a [bytes/4096, 2048] bf16 matrix read the way a
 *                     GEMM reads an operand: 128B-swizzled TMA boxes of 128
 *                     rows x 64 columns, each CTA over the whole K extent of
 *                     its own 128-row blocks; bytes a multiple of 512 KiB
 * src: device pointer, 16-byte aligned.  Returns MOE_OK once enqueued,
 * MOE_ERR_INVALID_ARG for a bad pointer, pattern or size.  Its waits are
 * bounded like the GEMMs' (MOE_ERR_TIMEOUT in the status word). */
enum { MOE_PROBE_LINEAR = 0, MOE_PROBE_TILES = 1 };
MOE_API int moe_probe_read_stream(const void* src, size_t bytes, int32_t pattern,
                                  moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Tracing: timing probe                                                     */
/* ------------------------------------------------------------------------ */

/* Kernel names the probe knows, i = 0, 1, ...; NULL past the last one:
 * route, permute, combine, router_topk, the grouped GEMMs xa_gu, gate_up,
 * xa_dn, down, u, dgrad_dn, v, dgrad_gu, the weight-gradient GEMMs dB_dn,
 * dA_dn, dB_gu, dA_gu, dw_reduce, and the full weight-gradient GEMMs dW_dn
 * and dW_gu.  ("route" covers all of its kernels: moe_route_kernel_count.) */
MOE_API const char* moe_kernel_name(int32_t i);

/* Arms the probe of one kernel: its next n launches record start_events[i]
 * before and stop_events[i] after the launch on the launch stream (cudaEvent_t
 * handles, caller-owned, created with timing enabled); later launches are not
 * recorded.  n = 0 disarms.  The arrays are copied.  Costs nothing when no
 * kernel is armed. */
MOE_API int moe_probe_arm(const char* kernel, void* const* start_events,
                          void* const* stop_events, int32_t n);

/* Launches of `kernel` recorded since it was armed (-1: unknown name). */
MOE_API int32_t moe_probe_count(const char* kernel);

/* Library ABI version (bumped on any signature change). */
MOE_API int moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
