"""mx_gemm_bf16 (activation quantization inside the GEMM) on the GPU.

It must equal, bit for bit, mx_quantize_rows followed by mx_gemm: the codes and
scales it builds in shared memory are the quantizer's, and the contraction and
the K-split reduction are the same kernel's. Against the fp64 oracle (quantize
then dequantized matmul) every element stays within 1e-2 |ref| + 1e-3 rms(ref).
Covers single and multiple row batches of the in-kernel staging (32 rows),
two activation row tiles, ragged rows, strided rows, special blocks, and the
argument checks."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_gemm_close, bf16_to_device, handle, operands, quantize_on_gpu

pytestmark = pytest.mark.gpu


def _composed(x, wq, wsc, m):
    import mxfp8_block_scaled_06_gb300 as mx

    aq, asc = mx.mx_quantize_rows(handle(), x[:m] if x.shape[0] > m else x)
    return mx.mx_gemm(handle(), aq, asc, wq, wsc)


def _run(m, n, k, seed=0, ldx=None, pdl=False):
    import mxfp8_block_scaled_06_gb300 as mx

    a_bits, _, (ra, rsa) = operands(seed, synth.TAG_A, m, k)
    w_bits, _, (rw, rsw) = operands(seed, synth.TAG_W, n, k)
    wq, wsc = quantize_on_gpu(w_bits)
    if ldx is None:
        x = bf16_to_device(a_bits)
    else:
        big = np.zeros((m, ldx), dtype=np.uint16)
        big[:, :k] = a_bits
        x = bf16_to_device(big)[:, :k]  # row stride ldx
    out = mx.mx_gemm_bf16(handle(), x, wq, wsc, pdl=pdl)
    ref_dev = _composed(bf16_to_device(a_bits), wq, wsc, m)
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    np.testing.assert_array_equal(out.view(torch.int16).cpu().numpy(), ref_dev.view(torch.int16).cpu().numpy())
    ref = oracle.mx_gemm(ra, rsa, rw, rsw)
    assert_gemm_close(out, ref, f"mx_gemm_bf16 M={m} N={n} K={k}")


def test_bf16_tiny_config():
    _run(4, 256, 512)


@pytest.mark.parametrize("m", [1, 2, 4, 8, 16])
def test_bf16_decode_projection(m):
    _run(m, 2048, 5120, seed=11, pdl=True)


@pytest.mark.parametrize("m", [1, 7, 15, 17, 31, 32, 33, 47, 64])
def test_bf16_ragged_rows_and_row_batches(m):
    _run(m, 384, 640, seed=20 + m)


@pytest.mark.parametrize("m", [130, 256])
def test_bf16_two_activation_row_tiles(m):
    _run(m, 256, 512, seed=3)


@pytest.mark.parametrize("n,k", [(128, 128), (1024, 128), (640, 4096), (8192, 1536)])
def test_bf16_tile_and_split_shapes(n, k):
    _run(6, n, k, seed=n + k)


@pytest.mark.parametrize("m,n,k", [(3, 2048, 1408), (3, 2048, 2432)])
def test_bf16_ragged_k_splits(m, n, k):
    # 11 / 19 chunks over 8 K-splits: CTAs with one or two (two or three)
    # chunks, so one launch splits its 32-blocks over 8 and 4 (4 and 2) threads
    _run(m, n, k, seed=k)


def test_bf16_strided_rows():
    _run(5, 512, 1024, seed=4, ldx=1024 + 40)


def test_bf16_special_blocks():
    """Zero, subnormal, saturating and non-finite 32-blocks quantize as the
    quantizer does (checked through the bit-exact output)."""
    import mxfp8_block_scaled_06_gb300 as mx

    m, n, k = 3, 256, 256
    a = synth.block_scaled_bf16(7, synth.TAG_A, m, k, -6, 6).copy()
    a[0, 0:32] = 0                      # zero block
    a[0, 32:64] = 0x0001                # bf16 subnormals
    a[1, 64:96] = 0x43E0                # 448: at the E4M3 maximum
    a[1, 96:128] = 0x4400               # 512 -> saturates after scaling
    a[2, 128] = 0x7FC0                  # NaN: the block's scale becomes 0xFF
    w_bits = synth.block_scaled_bf16(7, synth.TAG_W, n, k, -6, 6)
    wq, wsc = quantize_on_gpu(w_bits)
    x = bf16_to_device(a)
    out = mx.mx_gemm_bf16(handle(), x, wq, wsc)
    ref = _composed(x, wq, wsc, m)
    torch.cuda.synchronize()
    got, want = out.view(torch.int16).cpu().numpy(), ref.view(torch.int16).cpu().numpy()
    # rows 0 and 1 are finite: identical bits; row 2 holds a NaN block: NaN in the same places
    np.testing.assert_array_equal(got[:2], want[:2])
    g2, w2 = out[2].float().cpu().numpy(), ref[2].float().cpu().numpy()
    np.testing.assert_array_equal(np.isnan(g2), np.isnan(w2))
    np.testing.assert_array_equal(g2[~np.isnan(g2)], w2[~np.isnan(w2)])


def test_bf16_rejects_bad_arguments():
    import mxfp8_block_scaled_06_gb300 as mx

    lib = mx.load_library()
    w_bits = synth.block_scaled_bf16(1, synth.TAG_W, 256, 512, -6, 6)
    wq, wsc = quantize_on_gpu(w_bits)
    x = torch.zeros((4, 512), dtype=torch.bfloat16, device="cuda")
    out = torch.full((4, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    h = handle().ptr

    def call(m=4, n=256, k=512, xp=x.data_ptr(), ldx=512):
        return lib.mx_gemm_bf16(h, m, n, k, xp, ldx, wq.data_ptr(), wsc.data_ptr(), out.data_ptr(), 0, None)

    assert call(ldx=500) == mx.MX_ERR_INVALID_ARG      # ldx < K
    assert call(ldx=516) == mx.MX_ERR_INVALID_ARG      # rows not 16-byte aligned
    assert call(xp=x.data_ptr() + 2) == mx.MX_ERR_INVALID_ARG
    assert call(m=0) == mx.MX_ERR_INVALID_ARG
    assert call(m=257) == mx.MX_ERR_UNSUPPORTED
    assert call(n=200) == mx.MX_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (out.float() == 7.0).all()  # nothing launched
