"""Both tile modes of the large row-tile GEMMs against the oracle.

gate_up, down, dgrad_dn and dgrad_gu run either on single CTAs (128-row
tiles) or on CTA pairs (256-row tiles, tcgen05 cta_group::2); the library
picks per kernel and shape, and MOE_PAIR_TILES in the environment (read once
per process) forces a choice.  The seeded random-shape parity module runs
here in child processes with every GEMM on pairs and with none on pairs, so
each mode meets the same ragged shapes whatever the default picks."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("mode", ["1", "0", "gate_up,dgrad_dn"])
def test_random_shapes_in_tile_mode(mode):
    """The random shapes, and the edge cases (one token, all rows on one
    expert, 300 and 600 experts, exact tiles, duplicates) of the layer tests."""
    env = dict(os.environ, MOE_PAIR_TILES=mode)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p",
                        "no:cacheprovider", os.path.join(HERE, "test_gpu_random_shapes.py"),
                        os.path.join(HERE, "test_gpu_layer.py"), "-k",
                        "random_shape or edge_cases"],
                       env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
