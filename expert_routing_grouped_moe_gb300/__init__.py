"""GB300-native (sm_103a) MoE-LoRA expert layer.

Grouped routing (flatten, stable sort by expert, one bincount, offsets, one
row permute), split-LoRA SwiGLU experts as tcgen05 grouped GEMMs, weighted
combine, and the backward pass for frozen base weights -- all in the CUDA
library under ``csrc/``, exposed through the C ABI of ``include/moe_gb300.h``.

Importing this package does not load the library; the first call does, and
fails loudly if ``build.build()`` has not produced it.
"""
from . import _lib as lib  # noqa: F401
from . import synth  # noqa: F401
from .layer import MoELoRALayer, LAUNCHES_FWD, LAUNCHES_BWD  # noqa: F401
