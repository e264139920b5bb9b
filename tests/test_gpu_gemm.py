"""mx_gemm on the GPU against the fp64 oracle: every output element within
1e-2 |ref| + 1e-3 rms(ref), across tiles, K-splits, ragged activation rows and
the decode-projection shapes, plus the zero-input and untouched-rows cases."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_gemm_close, bf16_to_device, handle, operands, quantize_on_gpu, u8

pytestmark = pytest.mark.gpu


def _run(m, n, k, seed=0, pdl=False, a_range=(-6, 6)):
    import mxfp8_block_scaled_06_gb300 as mx

    a_bits, _, (ra, rsa) = operands(seed, synth.TAG_A, m, k, *a_range)
    w_bits, _, (rw, rsw) = operands(seed, synth.TAG_W, n, k)
    aq, asc = quantize_on_gpu(a_bits)
    wq, wsc = quantize_on_gpu(w_bits)
    out = mx.mx_gemm(handle(), aq, asc, wq, wsc, pdl=pdl)
    torch.cuda.synchronize()
    # the operands the GPU used are the oracle's, byte for byte
    np.testing.assert_array_equal(u8(aq), ra)
    np.testing.assert_array_equal(u8(wq), rw)
    ref = oracle.mx_gemm(ra, rsa, rw, rsw)
    assert_gemm_close(out, ref, f"mx_gemm M={m} N={n} K={k}")
    assert mx.mx_device_status(handle()) == mx.MX_OK


def test_gemm_tiny_config():
    _run(4, 256, 512)


@pytest.mark.parametrize("m", [1, 2, 4, 8])
def test_gemm_single_decode_projection(m):
    _run(m, 2048, 5120, seed=1)


@pytest.mark.parametrize("m", [1, 3, 15, 16, 17, 31, 33, 48, 63, 64, 100, 128])
def test_gemm_ragged_rows(m):
    _run(m, 384, 640, seed=m)


@pytest.mark.parametrize("n,k", [(128, 128), (128, 256), (256, 1024), (1024, 128), (640, 4096)])
def test_gemm_tile_and_split_shapes(n, k):
    _run(5, n, k, seed=n + k)


@pytest.mark.parametrize("m", [129, 192, 256])
def test_gemm_two_activation_row_tiles(m):
    _run(m, 256, 1024, seed=m)


def test_gemm_pdl_flag():
    _run(8, 2048, 5120, seed=5, pdl=True)


def test_gemm_zero_input_gives_zero():
    # all-zero codes with all-zero scale bytes (the warm-up input of the page)
    import mxfp8_block_scaled_06_gb300 as mx

    m, n, k = 8, 512, 1024
    w_bits, _, _ = operands(2, synth.TAG_W, n, k)
    wq, wsc = quantize_on_gpu(w_bits)
    a = torch.zeros((m, k), dtype=torch.uint8, device="cuda")
    asc = torch.zeros(mx.mx_scale_bytes(m, k), dtype=torch.uint8, device="cuda")
    out = mx.mx_gemm(handle(), a, asc, wq, wsc)
    torch.cuda.synchronize()
    assert (out.float() == 0).all()


def test_gemm_leaves_rows_beyond_m_untouched():
    import mxfp8_block_scaled_06_gb300 as mx

    m, n, k = 3, 256, 512
    a_bits, _, (ra, rsa) = operands(4, synth.TAG_A, m, k)
    w_bits, _, (rw, rsw) = operands(4, synth.TAG_W, n, k)
    aq, asc = quantize_on_gpu(a_bits)
    wq, wsc = quantize_on_gpu(w_bits)
    canary = torch.full((m + 2, n), 7.0, dtype=torch.bfloat16, device="cuda")
    mx.mx_gemm(handle(), aq, asc, wq, wsc, out=canary[:m])
    torch.cuda.synchronize()
    assert (canary[m:].float() == 7.0).all()
    assert_gemm_close(canary[:m], oracle.mx_gemm(ra, rsa, rw, rsw))


def test_gemm_invalid_arguments_launch_nothing():
    import mxfp8_block_scaled_06_gb300 as mx

    lib = mx.load_library()
    h = handle()
    m, n, k = 4, 256, 512
    a = torch.zeros((m, k), dtype=torch.uint8, device="cuda")
    asc = torch.zeros(mx.mx_scale_bytes(m, k), dtype=torch.uint8, device="cuda")
    w = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
    wsc = torch.zeros(mx.mx_scale_bytes(n, k), dtype=torch.uint8, device="cuda")
    out = torch.full((m, n), 3.0, dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()
    cases = [
        ((h.ptr, 0, n, k, p(a), p(asc), p(w), p(wsc), p(out), 0, None), mx.MX_ERR_INVALID_ARG),
        ((h.ptr, 257, n, k, p(a), p(asc), p(w), p(wsc), p(out), 0, None), mx.MX_ERR_UNSUPPORTED),
        ((h.ptr, m, 200, k, p(a), p(asc), p(w), p(wsc), p(out), 0, None), mx.MX_ERR_UNSUPPORTED),
        ((h.ptr, m, n, 96, p(a), p(asc), p(w), p(wsc), p(out), 0, None), mx.MX_ERR_UNSUPPORTED),
        ((h.ptr, m, n, 100, p(a), p(asc), p(w), p(wsc), p(out), 0, None), mx.MX_ERR_INVALID_ARG),
        ((h.ptr, m, n, k, p(a) + 1, p(asc), p(w), p(wsc), p(out), 0, None), mx.MX_ERR_INVALID_ARG),
        ((h.ptr, m, n, k, p(a), p(asc), p(w), p(wsc) + 16, p(out), 0, None), mx.MX_ERR_INVALID_ARG),
        ((h.ptr, m, n, k, p(a), p(asc), p(w), p(wsc), None, 0, None), mx.MX_ERR_INVALID_ARG),
        ((h.ptr, m, n, k, None, p(asc), p(w), p(wsc), p(out), 0, None), mx.MX_ERR_INVALID_ARG),
        ((h.ptr, m, n, k, p(a), p(asc), p(w), p(wsc), p(out), 8, None), mx.MX_ERR_INVALID_ARG),
    ]
    for args, want in cases:
        assert lib.mx_gemm(*args) == want, args
    torch.cuda.synchronize()
    assert (out.float() == 3.0).all()
