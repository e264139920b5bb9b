"""wo_a_grouped on the GPU against the oracle.

* the RoPE'd, per-32 quantized activation the contraction reads (debug copy)
  is bit-exact with the oracle's (float32 rotation without FMA, MX rule);
* z (bf16, before requantization) is within the GEMM tolerance of the
  oracle's fp64 contraction;
* q / q_scales equal mx_quantize_rows of the GPU's own bf16 z, bit for bit,
  and agree with the oracle's on every 32-block whose bf16 z agrees;
* the wo_b GEMM on q (K = 4096, N = 5120) stays within the GEMM tolerance plus
  the exact effect of the few codes that differ;
* called without the debug copy of the activation above 8 tokens, the call
  takes the two launches on the handle's scratch: the same checks, plus bit
  equality with wo_a_grouped_unfused, also for calls of shrinking sizes in a row.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import (assert_gemm_close, bf16_to_device, handle, operands, quantize_on_gpu,
                         u8)

pytestmark = pytest.mark.gpu

G, H, R, D = 4, 8, 1024, 512
_CACHE = {}


def _setup(seed=3):
    if seed not in _CACHE:
        w_bits, _, (rw, rws) = operands(seed, synth.TAG_WOA, G * R, H * D)
        wq, wsc = quantize_on_gpu(w_bits)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(u8(wq), rw)
        cs = synth.rope_cos_sin_cache(65536)
        _CACHE[seed] = ((wq, wsc), (rw, rws), cs, torch.from_numpy(cs).cuda())
    return _CACHE[seed]


def _run(t, seed=3, extra_heads=0, early_trigger=False):
    import mxfp8_block_scaled_06_gb300 as mx

    (wq, wsc), (rw, rws), cs, cs_dev = _setup()
    heads = G * H + extra_heads
    x_bits = synth.normal_bf16(seed + t, synth.TAG_X, (t, heads, D))
    pos = synth.positions(seed + t, synth.TAG_POS, t)
    x = bf16_to_device(x_bits)[:, :G * H, :]
    res = mx.wo_a_grouped(handle(), x, torch.from_numpy(pos).cuda(), cs_dev, wq, wsc, G, H, R,
                          debug=True, early_trigger=early_trigger)
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    xv = synth.bf16_bits_to_f64(x_bits[:, :G * H, :])
    ora = oracle.wo_a_grouped(xv, pos, cs, rw, rws, G, H, 448, 64, R)
    return res, ora


@pytest.mark.parametrize("t", [1, 8, 32])
def test_wo_a_decode_tokens(t):
    _check(*_run(t), t)


@pytest.mark.parametrize("t", [2, 17, 50, 64, 100, 128])
def test_wo_a_ragged_tokens(t):
    _check(*_run(t), t)


def test_wo_a_strided_heads_and_early_trigger():
    # attn_out carries more heads than the projection reads: token stride > G*H*D
    _check(*_run(5, extra_heads=8, early_trigger=True), 5)


def _check(res, ora, t):
    import mxfp8_block_scaled_06_gb300 as mx

    np.testing.assert_array_equal(u8(res["xq"]), ora["xq"])
    np.testing.assert_array_equal(u8(res["xs"]), ora["xs"])
    assert_gemm_close(res["z"], ora["z"], "WO-A z")
    q2, s2 = mx.mx_quantize_rows(handle(), res["z"])
    torch.cuda.synchronize()
    assert torch.equal(res["q"], q2) and torch.equal(res["q_scales"], s2)
    zb_gpu = res["z"].view(torch.int16).cpu().numpy().view(np.uint16)
    zb_ora = oracle.bf16_bits(ora["zb"])
    same_block = (zb_gpu.reshape(t, -1, 32) == zb_ora.reshape(t, -1, 32)).all(axis=-1)
    gq = u8(res["q"]).reshape(t, -1, 32)
    assert (gq[same_block] == ora["q"].reshape(t, -1, 32)[same_block]).all()
    assert same_block.mean() >= 0.95


def test_wo_a_then_wo_b():
    import mxfp8_block_scaled_06_gb300 as mx

    t = 8
    res, ora = _run(t)
    wb_bits, _, (rb, rbs) = operands(4, synth.TAG_WOB, 5120, G * R)
    wbq, wbs = quantize_on_gpu(wb_bits)
    out = mx.mx_gemm(handle(), res["q"], res["q_scales"], wbq, wbs, pdl=True)
    torch.cuda.synchronize()
    ref = oracle.mx_gemm(ora["q"], ora["qs"], rb, rbs)
    gq = u8(res["q"])
    gs_plain = np.zeros_like(ora["qs"])
    buf = u8(res["q_scales"])
    rr, cc = np.meshgrid(np.arange(t), np.arange(G * R // 32), indexing="ij")
    gs_plain[rr, cc] = buf[((rr // 128) * (G * R // 128) + cc // 4) * 512 + (rr % 32) * 16
                           + ((rr % 128) // 32) * 4 + cc % 4]
    dq = lambda c, s: (torch.from_numpy(c).view(torch.float8_e4m3fn).double().reshape(t, -1, 32)
                       * torch.from_numpy(s).view(torch.float8_e8m0fnu).double()[..., None]
                       ).reshape(t, -1).numpy()
    delta = np.abs(dq(gq, gs_plain) - dq(ora["q"], ora["qs"]))
    extra = 1.01 * (delta @ np.abs(oracle.mx_dequantize(rb, rbs)).T)
    got = out.float().cpu().numpy().astype(np.float64)
    assert (np.abs(got - ref) <= oracle.gemm_tolerance(ref) + extra).all()


FUSED_MAX_TOKENS = 8  # wo_a_grouped's documented switch to the two launches


def _without_debug_copy(t, seed=3):
    """wo_a_grouped asked for z only (no debug copy of the activation): above 8
    tokens it runs the two launches on the handle's scratch. Checked against the
    oracle like the fused kernel, and there bit for bit against
    wo_a_grouped_unfused on caller buffers."""
    import mxfp8_block_scaled_06_gb300 as mx

    (wq, wsc), (rw, rws), cs, cs_dev = _setup()
    x_bits = synth.normal_bf16(seed + t, synth.TAG_X, (t, G * H, D))
    pos = synth.positions(seed + t, synth.TAG_POS, t)
    x = bf16_to_device(x_bits)
    pos_dev = torch.from_numpy(pos).cuda()
    res = mx.wo_a_grouped(handle(), x, pos_dev, cs_dev, wq, wsc, G, H, R, z=True, early_trigger=True)
    torch.cuda.synchronize()
    assert mx.mx_device_status(handle()) == mx.MX_OK
    assert res["xq"] is None and res["xs"] is None
    if t > FUSED_MAX_TOKENS:
        ref = mx.wo_a_grouped_unfused(handle(), x, pos_dev, cs_dev, wq, wsc, G, H, R, z=True)
        torch.cuda.synchronize()
        assert torch.equal(res["z"], ref["z"])
        assert torch.equal(res["q"], ref["q"]) and torch.equal(res["q_scales"], ref["q_scales"])
    ora = oracle.wo_a_grouped(synth.bf16_bits_to_f64(x_bits), pos, cs, rw, rws, G, H, 448, 64, R)
    assert_gemm_close(res["z"], ora["z"], "WO-A z (two launches)")
    q2, s2 = mx.mx_quantize_rows(handle(), res["z"])
    torch.cuda.synchronize()
    assert torch.equal(res["q"], q2) and torch.equal(res["q_scales"], s2)
    zb_gpu = res["z"].view(torch.int16).cpu().numpy().view(np.uint16)
    same_block = (zb_gpu.reshape(t, -1, 32) == oracle.bf16_bits(ora["zb"]).reshape(t, -1, 32)).all(-1)
    gq = u8(res["q"]).reshape(t, -1, 32)
    assert (gq[same_block] == ora["q"].reshape(t, -1, 32)[same_block]).all()
    assert same_block.mean() >= 0.95


@pytest.mark.parametrize("t", [8, 9, 17, 32, 100, 128])
def test_wo_a_without_debug_copy(t):
    _without_debug_copy(t)


def test_wo_a_two_launch_scratch_reused_across_calls():
    # the handle's scratch keeps the previous call's activation: a smaller call
    # after a larger one must not read any of it
    for t in (128, 24, 64, 9):
        _without_debug_copy(t, seed=9)


def test_wo_a_rejects_unsupported_shapes():
    import mxfp8_block_scaled_06_gb300 as mx

    (wq, wsc), _, _, cs_dev = _setup()
    x = torch.zeros((4, G * H, D), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(4, dtype=torch.int64, device="cuda")
    cs128 = torch.zeros((1024, 128), dtype=torch.float32, device="cuda")  # a cache matching d_rope
    with pytest.raises(mx.MxError) as e:
        mx.wo_a_grouped(handle(), x, pos, cs128, wq, wsc, G, H, R, d_nope=384, d_rope=128)
    assert e.value.code == mx.MX_ERR_UNSUPPORTED
    x129 = torch.zeros((129, G * H, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MxError) as e:
        mx.wo_a_grouped(handle(), x129, torch.zeros(129, dtype=torch.int64, device="cuda"),
                        cs_dev, wq, wsc, G, H, R)
    assert e.value.code == mx.MX_ERR_UNSUPPORTED
