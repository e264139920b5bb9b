"""mx_quantize_rows on the GPU is bit-exact with the oracle: codes, swizzled
scales (including zero padding) and the plain scale layout."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import bf16_to_device, handle, u8

pytestmark = pytest.mark.gpu


def _check(bits, swizzled=True, ldx=None):
    import mxfp8_block_scaled_06_gb300 as mx

    m, k = bits.shape
    vals = synth.bf16_bits_to_f64(bits)
    rc, rs = oracle.mx_quantize(vals)
    if ldx is None:
        x = bf16_to_device(bits)
    else:
        full = np.zeros((m, ldx), np.uint16)
        full[:, :k] = bits
        x = bf16_to_device(full)[:, :k]
    q, s = mx.mx_quantize_rows(handle(), x, swizzled=swizzled)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u8(q), rc)
    if swizzled:
        np.testing.assert_array_equal(u8(s), oracle.swizzle_scales(rs))
    else:
        np.testing.assert_array_equal(u8(s), rs)


@pytest.mark.parametrize("m,k", [(4, 512), (1, 5120), (2, 5120), (8, 5120), (3, 96), (130, 160),
                                 (16, 1536), (64, 8192), (256, 4096), (33, 32)])
@pytest.mark.parametrize("swizzled", [True, False])
def test_quantize_block_scaled_normal(m, k, swizzled):
    _check(synth.block_scaled_bf16(11, m * 7 + k, m, k, -6, 6), swizzled)


def test_quantize_weight_full_size():
    # the single decode projection's weight [2048, 5120]
    _check(synth.block_scaled_bf16(1, synth.TAG_W, 2048, 5120, -6, 6))


def test_quantize_max_rows():
    # the largest row count the entry point takes, and one more
    import mxfp8_block_scaled_06_gb300 as mx

    _check(synth.block_scaled_bf16(5, 12, 65536, 64, -6, 6))
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((2, 64), dtype=torch.uint8, device="cuda")
    s = torch.zeros(mx.mx_scale_bytes(2, 64), dtype=torch.uint8, device="cuda")
    rc = mx.load_library().mx_quantize_rows(handle().ptr, 65537, 64, x.data_ptr(), 64, q.data_ptr(),
                                            s.data_ptr(), 1, None)
    assert rc == mx.MX_ERR_INVALID_ARG


def test_quantize_strided_rows():
    _check(synth.block_scaled_bf16(3, 9, 5, 512, -4, 4), ldx=512 + 64)


def test_quantize_every_bf16_pattern():
    # all 65536 bf16 bit patterns, in blocks of 32 consecutive patterns: covers
    # zeros, subnormals, the top binade, saturation, NaN and Inf blocks
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(64, 1024)
    _check(bits)


def test_quantize_special_blocks():
    rows = []
    z = np.zeros(32)
    rows.append(z)                                    # zero block
    rows.append(-z)                                   # negative zeros
    rows.append(np.arange(32) * 2.0**-133)            # bf16 subnormals
    r = np.zeros(32); r[0] = 448 * 2.0**3; r[1] = 511 * 2.0**3; r[2] = -500 * 2.0**3
    rows.append(r)                                    # saturation in the top binade
    r = np.zeros(32); r[0] = 256.0; r[1] = 1.0625; r[2] = 1.1875; r[3] = 2.0**-10; r[4] = 1.5 * 2.0**-9
    rows.append(r)                                    # ties
    r = np.full(32, 2.0**100); rows.append(r)          # huge exponent
    r = np.full(32, -2.0**-120); rows.append(r)        # exponent clamp
    r = np.ones(32); r[7] = np.inf; rows.append(r)     # non-finite
    r = np.ones(32); r[9] = np.nan; rows.append(r)
    x = np.stack(rows)
    bits = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    _check(bits)
    _check(bits, swizzled=False)
