"""The row sweep toward the compute-bound crossover at its full sizes: M in
{64, 96, 128, 192, 256} activation rows against the (N, K) = (8192, 5120) and
(5120, 8192) weights, launched the way the benchmark launches them
(programmatic dependent launch on, and replayed from a CUDA graph), every output
element within 1e-2 |ref| + 1e-3 rms(ref) of the fp64 oracle. The weights are
quantized once per shape on the GPU and checked byte for byte against the
oracle's codes first, so both sides contract the same operands."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_gemm_close, handle, operands, quantize_on_gpu, u8

pytestmark = pytest.mark.gpu

SHAPES = [(8192, 5120), (5120, 8192)]
ROWS = [64, 96, 128, 192, 256]
_WEIGHTS = {}


def _weights(n, k):
    if (n, k) not in _WEIGHTS:
        bits, _, (rw, rsw) = operands(70 + n // 1024, synth.TAG_W, n, k)
        wq, wsc = quantize_on_gpu(bits)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(u8(wq), rw)
        _WEIGHTS[(n, k)] = (wq, wsc, rw, rsw)
    return _WEIGHTS[(n, k)]


@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("m", ROWS)
def test_row_sweep_full_size(m, n, k):
    import mxfp8_block_scaled_06_gb300 as mx

    wq, wsc, rw, rsw = _weights(n, k)
    a_bits, _, (ra, rsa) = operands(71 + m, synth.TAG_A, m, k)
    aq, asc = quantize_on_gpu(a_bits)
    out = mx.mx_gemm(handle(), aq, asc, wq, wsc, pdl=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u8(aq), ra)
    assert mx.mx_device_status(handle()) == mx.MX_OK
    assert_gemm_close(out, oracle.mx_gemm(ra, rsa, rw, rsw), f"row sweep M={m} N={n} K={k}")


def test_row_sweep_graph_replay_equals_eager():
    """Graph-replayed PDL launches (the benchmark's form) give the eager bits."""
    import mxfp8_block_scaled_06_gb300 as mx

    n, k = SHAPES[1]
    wq, wsc, _, _ = _weights(n, k)
    acts = [quantize_on_gpu(synth.block_scaled_bf16(72 + m, synth.TAG_A, m, k, -6, 6)) for m in (64, 256)]
    eager = [mx.mx_gemm(handle(), a, s, wq, wsc) for a, s in acts]
    outs = [torch.empty_like(e) for e in eager]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        mx.mx_gemm(handle(), *acts[0], wq, wsc, out=outs[0], pdl=True, stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for (a, s), o in zip(acts, outs):
                mx.mx_gemm(handle(), a, s, wq, wsc, out=o, pdl=True, stream=stream)
        for o in outs:
            o.fill_(0)
        g.replay()
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    for e, o in zip(eager, outs):
        assert torch.equal(e.view(torch.int16), o.view(torch.int16))
