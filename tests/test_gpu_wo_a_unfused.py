"""wo_a_grouped_unfused (RoPE + quantize, then one grouped GEMM) on the GPU.

* the RoPE'd, per-32 quantized activation it writes (xq and its swizzled
  scales, padding included) is bit-exact with the oracle's, and with the fused
  kernel's debug copy where both run;
* z (bf16) is within the GEMM tolerance of the oracle's fp64 contraction;
* q / q_scales equal mx_quantize_rows of the GPU's own bf16 z, bit for bit, and
  agree with the oracle's on every 32-block whose bf16 z agrees;
* token counts beyond the fused kernel's limit (129..256, two activation row
  tiles) and token strides wider than the heads read are covered.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_gemm_close, bf16_to_device, handle, operands, quantize_on_gpu, u8

pytestmark = pytest.mark.gpu

G, H, R, D = 4, 8, 1024, 512
_CACHE = {}


def _setup(seed=3):
    if seed not in _CACHE:
        w_bits, _, (rw, rws) = operands(seed, synth.TAG_WOA, G * R, H * D)
        wq, wsc = quantize_on_gpu(w_bits)
        cs = synth.rope_cos_sin_cache(65536)
        _CACHE[seed] = ((wq, wsc), (rw, rws), cs, torch.from_numpy(cs).cuda())
    return _CACHE[seed]


def _run(t, seed=5, extra_heads=0):
    import mxfp8_block_scaled_06_gb300 as mx

    (wq, wsc), (rw, rws), cs, cs_dev = _setup()
    heads = G * H + extra_heads
    x_bits = synth.normal_bf16(seed + t, synth.TAG_X, (t, heads, D))
    pos = synth.positions(seed + t, synth.TAG_POS, t)
    x = bf16_to_device(x_bits)[:, :G * H, :]
    pos_dev = torch.from_numpy(pos).cuda()
    res = mx.wo_a_grouped_unfused(handle(), x, pos_dev, cs_dev, wq, wsc, G, H, R, z=True)
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    xv = synth.bf16_bits_to_f64(x_bits[:, :G * H, :])
    ora = oracle.wo_a_grouped(xv, pos, cs, rw, rws, G, H, 448, 64, R)
    return res, ora, (x, pos_dev, cs_dev, wq, wsc)


def _check(res, ora, t):
    import mxfp8_block_scaled_06_gb300 as mx

    np.testing.assert_array_equal(u8(res["xq"]), ora["xq"])
    np.testing.assert_array_equal(u8(res["xq_scales"]), oracle.swizzle_scales(ora["xs"]))
    assert_gemm_close(res["z"], ora["z"], "unfused WO-A z")
    q2, s2 = mx.mx_quantize_rows(handle(), res["z"])
    torch.cuda.synchronize()
    assert torch.equal(res["q"], q2) and torch.equal(res["q_scales"], s2)
    zb_gpu = res["z"].view(torch.int16).cpu().numpy().view(np.uint16)
    zb_ora = oracle.bf16_bits(ora["zb"])
    same_block = (zb_gpu.reshape(t, -1, 32) == zb_ora.reshape(t, -1, 32)).all(axis=-1)
    gq = u8(res["q"]).reshape(t, -1, 32)
    assert (gq[same_block] == ora["q"].reshape(t, -1, 32)[same_block]).all()
    assert same_block.mean() >= 0.95


@pytest.mark.parametrize("t", [1, 8, 32])
def test_unfused_decode_tokens(t):
    res, ora, _ = _run(t)
    _check(res, ora, t)


@pytest.mark.parametrize("t", [129, 200, 256])
def test_unfused_beyond_the_fused_limit(t):
    res, ora, _ = _run(t)
    _check(res, ora, t)


def test_unfused_strided_heads():
    res, ora, _ = _run(6, extra_heads=8)
    _check(res, ora, 6)


def test_unfused_matches_fused_activation():
    import mxfp8_block_scaled_06_gb300 as mx

    t = 17
    res, _, (x, pos_dev, cs_dev, wq, wsc) = _run(t)
    fused = mx.wo_a_grouped(handle(), x, pos_dev, cs_dev, wq, wsc, G, H, R, debug=True)
    torch.cuda.synchronize()
    assert torch.equal(res["xq"], fused["xq"])
    plain = oracle.unswizzle_scales(u8(res["xq_scales"]), t, G * H * D // 32)
    np.testing.assert_array_equal(plain, u8(fused["xs"]))


def test_unfused_rejects_unsupported():
    import mxfp8_block_scaled_06_gb300 as mx

    (wq, wsc), _, _, cs_dev = _setup()
    x = torch.zeros((257, G * H, D), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(257, dtype=torch.int64, device="cuda")
    with pytest.raises(mx.MxError) as e:
        mx.wo_a_grouped_unfused(handle(), x, pos, cs_dev, wq, wsc, G, H, R)
    assert e.value.code == mx.MX_ERR_UNSUPPORTED
    x4 = torch.zeros((4, G * H, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MxError) as e:
        mx.wo_a_grouped_unfused(handle(), x4, pos[:4], torch.zeros((1024, 128), device="cuda"), wq, wsc,
                                G, H, R, d_nope=384, d_rope=128)
    assert e.value.code == mx.MX_ERR_UNSUPPORTED
