"""Zero-copy host I/O: mx_quantize_rows reading its bf16 rows straight from
pinned host memory and mx_gemm writing its bf16 output straight into pinned
host memory give, bit for bit, what the same calls give on device buffers; rows
of the host output beyond M keep their bytes."""
import pytest
import torch

import synth
from gpu_helpers import bf16_to_device, handle, quantize_on_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,k", [(1, 5120), (5, 640), (130, 256)])
def test_quantize_reads_pinned_host_rows(m, k):
    import mxfp8_block_scaled_06_gb300 as mx

    bits = synth.block_scaled_bf16(40 + m, synth.TAG_A, m, k, -6, 6)
    x_dev = bf16_to_device(bits)
    x_host = x_dev.cpu().pin_memory()
    q_ref, s_ref = mx.mx_quantize_rows(handle(), x_dev)
    q, s = mx.mx_quantize_rows(handle(), x_host)
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    assert q.is_cuda and s.is_cuda
    assert torch.equal(q, q_ref) and torch.equal(s, s_ref)


@pytest.mark.parametrize("m,n,k", [(1, 2048, 5120), (8, 2048, 5120), (17, 384, 640)])
def test_gemm_writes_pinned_host_output(m, n, k):
    import mxfp8_block_scaled_06_gb300 as mx

    aq, asc = quantize_on_gpu(synth.block_scaled_bf16(41, synth.TAG_A, m, k, -4, 4))
    wq, wsc = quantize_on_gpu(synth.block_scaled_bf16(41, synth.TAG_W, n, k, -6, 6))
    ref = mx.mx_gemm(handle(), aq, asc, wq, wsc, pdl=True)
    host = torch.full((m + 3, n), 7.0, dtype=torch.bfloat16).pin_memory()  # 3 guard rows
    mx.mx_gemm(handle(), aq, asc, wq, wsc, out=host[:m], pdl=True)
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    assert torch.equal(host[:m].view(torch.int16), ref.cpu().view(torch.int16))
    assert bool((host[m:] == 7.0).all()), "rows beyond M were written"


def test_step_through_host_memory_matches_device_step():
    """The bench's end-to-end step: activations read from one pinned buffer,
    outputs written to another, four row counts in a row with PDL."""
    import mxfp8_block_scaled_06_gb300 as mx

    k, n, rows = 5120, 2048, (1, 2, 4, 8)
    wq, wsc = quantize_on_gpu(synth.block_scaled_bf16(42, synth.TAG_W, n, k, -6, 6))
    bits = synth.block_scaled_bf16(42, synth.TAG_A, sum(rows), k, -4, 4)
    x_dev = bf16_to_device(bits)
    x_host = x_dev.cpu().pin_memory()
    out_host = torch.empty((sum(rows), n), dtype=torch.bfloat16).pin_memory()
    o = 0
    for m in rows:
        q, s = mx.mx_quantize_rows(handle(), x_host[o:o + m])
        mx.mx_gemm(handle(), q, s, wq, wsc, out=out_host[o:o + m], pdl=True)
        o += m
    ref = []
    o = 0
    for m in rows:
        q, s = mx.mx_quantize_rows(handle(), x_dev[o:o + m])
        ref.append(mx.mx_gemm(handle(), q, s, wq, wsc, pdl=True))
        o += m
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    assert torch.equal(out_host.view(torch.int16), torch.cat(ref).cpu().view(torch.int16))
