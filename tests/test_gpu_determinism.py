"""Run-to-run determinism of the GPU path: the split-K partials are summed over
the cluster in rank order and every kernel's work split is fixed by its plan,
so repeated calls, CUDA-graph replays and PDL on or off give bit-identical
outputs. A race between the pipeline stages or in the cluster reduction would
show up here as differing bits."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_to_device, handle, quantize_on_gpu

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("m,n,k", [(1, 2048, 5120), (16, 8192, 1536), (8, 5120, 8192), (64, 2048, 5120)])
def test_gemm_repeats_bit_identically(m, n, k):
    import mxfp8_block_scaled_06_gb300 as mx

    aq, asc = quantize_on_gpu(synth.block_scaled_bf16(31, synth.TAG_A, m, k, -6, 6))
    wq, wsc = quantize_on_gpu(synth.block_scaled_bf16(31, synth.TAG_W, n, k, -6, 6))
    first = mx.mx_gemm(handle(), aq, asc, wq, wsc)
    outs = [mx.mx_gemm(handle(), aq, asc, wq, wsc, pdl=(i % 2 == 0)) for i in range(6)]
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    ref = _bits(first)
    for o in outs:
        np.testing.assert_array_equal(_bits(o), ref)


def test_graph_replays_match_eager_calls():
    """Thirty chained launches captured in a CUDA graph (PDL on, as the bench
    runs them), replayed three times: every output equals the eager one."""
    import mxfp8_block_scaled_06_gb300 as mx

    m, n, k = 4, 2048, 5120
    aq, asc = quantize_on_gpu(synth.block_scaled_bf16(32, synth.TAG_A, m, k, -6, 6))
    ws = [quantize_on_gpu(synth.block_scaled_bf16(40 + j, synth.TAG_W, n, k, -6, 6)) for j in range(3)]
    eager = [_bits(mx.mx_gemm(handle(), aq, asc, *ws[j])) for j in range(3)]
    outs = [torch.empty((m, n), dtype=torch.bfloat16, device="cuda") for _ in range(30)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mx.mx_gemm(handle(), aq, asc, *ws[0], out=outs[0], pdl=True, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(30):
                mx.mx_gemm(handle(), aq, asc, *ws[i % 3], out=outs[i], pdl=True, stream=s)
        for _ in range(3):
            for o in outs:
                o.fill_(0)
            g.replay()
            torch.cuda.synchronize()
            for i, o in enumerate(outs):
                np.testing.assert_array_equal(_bits(o), eager[i % 3])
    assert mx.mx_device_status(handle()) == mx.MX_OK


def test_chain_and_wo_a_repeat_bit_identically():
    import mxfp8_block_scaled_06_gb300 as mx

    m = 8
    shapes = [(2048, 5120), (8192, 1536), (5120, 8192)]
    ws = [quantize_on_gpu(synth.block_scaled_bf16(50 + i, synth.TAG_W, n, k, -6, 6))
          for i, (n, k) in enumerate(shapes)]
    a1 = quantize_on_gpu(synth.block_scaled_bf16(51, synth.TAG_A, m, 5120, -4, 4))
    outs = [mx.mx_gemm_chain(handle(), a1[0], a1[1], ws)["out"] for _ in range(3)]
    G, H, R, D = 4, 8, 1024, 512
    ww = quantize_on_gpu(synth.block_scaled_bf16(52, synth.TAG_WOA, G * R, H * D, -6, 6))
    cs = torch.from_numpy(synth.rope_cos_sin_cache(65536)).cuda()
    x = bf16_to_device(synth.normal_bf16(53, synth.TAG_X, (5, G * H, D)))
    pos = torch.from_numpy(synth.positions(53, synth.TAG_POS, 5)).cuda()
    qs = [mx.wo_a_grouped(handle(), x, pos, cs, *ww, G, H, R)["q"] for _ in range(3)]
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    for o in outs[1:]:
        np.testing.assert_array_equal(_bits(o), _bits(outs[0]))
    for q in qs[1:]:
        assert torch.equal(q, qs[0])
