"""mx_gemm_chain through the persistent one-kernel path (MX_CHAIN_PERSISTENT=1).

The same checks as tests/test_gpu_chain.py: bit-exact with composing the
separately verified entry points (the kernel splits each projection's K-range
as mx_gemm's plan does, keeps its per-CTA chunk order and adds the split
partials in rank order), and the independent oracle's bounds. Also checks that
calls of different shapes in a row agree with the composition: the kernel's
per-tile counters must start every call at zero.
"""
import pytest

from test_gpu_chain import _composition, _vs_oracle

pytestmark = pytest.mark.gpu

DECODE = [(2048, 5120), (8192, 1536), (5120, 8192)]
SMALL = [(384, 640), (256, 256), (512, 256)]


@pytest.fixture(autouse=True)
def persistent(monkeypatch):
    monkeypatch.setenv("MX_CHAIN_PERSISTENT", "1")


@pytest.mark.parametrize("m", [1, 5, 16])
def test_persistent_equals_composition_small(m):
    _composition(m, SMALL, 256, seed=7)


@pytest.mark.parametrize("m", [1, 8, 16])
def test_persistent_equals_composition_decode_shapes(m):
    _composition(m, DECODE, 1536, seed=2)


@pytest.mark.parametrize("m", [1, 4, 16])
def test_persistent_vs_oracle_decode_shapes(m):
    _vs_oracle(m, DECODE, 1536, seed=2)


def test_persistent_alternating_shapes():
    for m, shapes, g1 in [(3, SMALL, 256), (2, DECODE, 1536), (9, SMALL, 256), (1, DECODE, 1536)]:
        _composition(m, shapes, g1, seed=5)
