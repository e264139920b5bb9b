"""mx_gemm_chain through the persistent one-kernel path (MX_CHAIN_PERSISTENT=1).

The same checks as tests/test_gpu_chain.py: bit-exact with composing the
separately verified entry points (the kernel splits each projection's K-range
as mx_gemm's plan does, keeps its per-CTA chunk order and adds the split
partials in rank order), and the independent oracle's bounds. Also checks that
calls of different shapes in a row agree with the composition: the kernel's
per-tile counters must start every call at zero.
"""
import os

import pytest

from gpu_helpers import handle
from test_gpu_chain import _composition, _vs_oracle

pytestmark = pytest.mark.gpu

DECODE = [(2048, 5120), (8192, 1536), (5120, 8192)]
SMALL = [(384, 640), (256, 256), (512, 256)]


@pytest.fixture(scope="module")
def ph():
    """A handle created with MX_CHAIN_PERSISTENT=1 (read once, at mx_create)."""
    import mxfp8_block_scaled_06_gb300 as mx

    handle()  # builds and loads the library
    old = os.environ.get("MX_CHAIN_PERSISTENT")
    os.environ["MX_CHAIN_PERSISTENT"] = "1"
    try:
        h = mx.mx_create(0)
    finally:
        if old is None:
            del os.environ["MX_CHAIN_PERSISTENT"]
        else:
            os.environ["MX_CHAIN_PERSISTENT"] = old
    yield h
    h.close()


@pytest.mark.parametrize("m", [1, 5, 16])
def test_persistent_equals_composition_small(ph, m):
    _composition(m, SMALL, 256, seed=7, chain_handle=ph)


@pytest.mark.parametrize("m", [1, 8, 16])
def test_persistent_equals_composition_decode_shapes(ph, m):
    _composition(m, DECODE, 1536, seed=2, chain_handle=ph)


@pytest.mark.parametrize("m", [1, 4, 16])
def test_persistent_vs_oracle_decode_shapes(ph, m):
    _vs_oracle(m, DECODE, 1536, seed=2, chain_handle=ph)


def test_persistent_alternating_shapes(ph):
    for m, shapes, g1 in [(3, SMALL, 256), (2, DECODE, 1536), (9, SMALL, 256), (1, DECODE, 1536)]:
        _composition(m, shapes, g1, seed=5, chain_handle=ph)
