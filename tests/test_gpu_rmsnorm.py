"""mx_rmsnorm_quantize_rows and mx_gemm_chain_norm on the GPU.

* the normalized row y (bf16) is within one bf16 ulp of the oracle's float64
  normalization rounded to bf16 (the GPU works in float32), and equal for the
  vast majority of elements;
* q / scales equal mx_quantize_rows of the GPU's own y, bit for bit, and the
  oracle's codes on every 32-block whose y agrees;
* closed forms: a constant row with weight 1 and eps 0 normalizes to exactly
  +-1; a zero row with eps > 0 stays zero (scale byte 0);
* the chain with the norm equals composing the entry points on the GPU
  (mx_gemm, mx_rmsnorm_quantize_rows, mx_gemm, mx_quantize_rows, mx_gemm), bit
  for bit, in both of its forms (up to 16 rows the norm and quantization run
  in G2's prologue; above, the norm kernel runs between G1 and G2), and its
  output stays within the GEMM tolerance of the oracle's GEMM on the GPU's own
  last activation.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_gemm_close, bf16_to_device, handle, operands, quantize_on_gpu, u8

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _weight(k, seed):
    return synth.norm_weight_bf16(seed, k)


def _run(m, k, seed, eps=1e-6, ldx=None, swizzled=True):
    import mxfp8_block_scaled_06_gb300 as mx

    x_bits = synth.block_scaled_bf16(seed, synth.TAG_A, m, k, -4, 4)
    w_bits = _weight(k, seed)
    if ldx is None:
        x = bf16_to_device(x_bits)
    else:
        big = np.zeros((m, ldx), dtype=np.uint16)
        big[:, :k] = x_bits
        x = bf16_to_device(big)[:, :k]
    wg = bf16_to_device(w_bits)
    q, s, y = mx.mx_rmsnorm_quantize_rows(handle(), x, wg, eps, swizzled=swizzled, y=True)
    torch.cuda.synchronize()
    xv = synth.bf16_bits_to_f64(x_bits)
    y_ora = oracle.round_bf16(oracle.rms_norm(xv, synth.bf16_bits_to_f64(w_bits), eps))
    return q, s, y, y_ora


@pytest.mark.parametrize("m,k", [(1, 1536), (5, 1536), (130, 256), (3, 96), (8, 4096)])
def test_rmsnorm_quantize_vs_oracle(m, k):
    import mxfp8_block_scaled_06_gb300 as mx

    q, s, y, y_ora = _run(m, k, seed=m + k)
    yg = y.double().cpu().numpy()
    ulp = np.abs(y_ora) * 2.0 ** -7  # one bf16 ulp at most (8 significant bits)
    assert (np.abs(yg - y_ora) <= ulp + 1e-300).all()
    same = _bits(y) == oracle.bf16_bits(y_ora)
    assert same.mean() >= 0.99
    q2, s2 = mx.mx_quantize_rows(handle(), y)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s, s2)
    oc, _ = oracle.mx_quantize(y_ora)
    blocks = same.reshape(m, -1, 32).all(axis=-1)
    assert (u8(q).reshape(m, -1, 32)[blocks] == oc.reshape(m, -1, 32)[blocks]).all()


def test_rmsnorm_strided_rows_and_plain_scales():
    import mxfp8_block_scaled_06_gb300 as mx

    q, s, y, _ = _run(4, 512, seed=3, ldx=512 + 24, swizzled=False)
    q2, s2 = mx.mx_quantize_rows(handle(), y, swizzled=False)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s, s2)


def test_rmsnorm_closed_forms():
    import mxfp8_block_scaled_06_gb300 as mx

    k = 256
    x = torch.full((2, k), -3.25, dtype=torch.bfloat16, device="cuda")
    x[1] = 0
    ones = torch.ones(k, dtype=torch.bfloat16, device="cuda")
    q, s, y = mx.mx_rmsnorm_quantize_rows(handle(), x, ones, 0.0, swizzled=False, y=True)
    torch.cuda.synchronize()
    assert (y[0].float() == -1.0).all()
    oc, os_ = oracle.mx_quantize(np.full((1, k), -1.0))
    np.testing.assert_array_equal(u8(q)[0], oc[0])
    np.testing.assert_array_equal(u8(s)[0], os_[0])
    q, s, y = mx.mx_rmsnorm_quantize_rows(handle(), x[1:], ones, 1e-6, swizzled=False, y=True)
    torch.cuda.synchronize()
    assert (y.float() == 0).all() and (u8(s) == 0).all()


def test_rmsnorm_rejects_bad_arguments():
    import mxfp8_block_scaled_06_gb300 as mx

    lib = mx.load_library()
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((2, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros(mx.mx_scale_bytes(2, 256), dtype=torch.uint8, device="cuda")
    h = handle().ptr
    call = lambda k=256, ldx=256, eps=1e-6, wp=w.data_ptr(): lib.mx_rmsnorm_quantize_rows(
        h, 2, k, x.data_ptr(), ldx, wp, eps, None, q.data_ptr(), s.data_ptr(), 1, None)
    assert call(k=250) == mx.MX_ERR_INVALID_ARG
    assert call(ldx=200) == mx.MX_ERR_INVALID_ARG
    assert call(eps=-1.0) == mx.MX_ERR_INVALID_ARG
    assert call(eps=float("nan")) == mx.MX_ERR_INVALID_ARG
    assert call(wp=0) == mx.MX_ERR_INVALID_ARG


def _plain_test_side(buf: np.ndarray, rows: int, ncols: int) -> np.ndarray:
    """Plain [rows, ncols] scales from a 128x4-tiled buffer (the test's own reshape)."""
    rpad, cpad = (rows + 127) // 128 * 128, (ncols + 3) // 4 * 4
    t = buf.reshape(rpad // 128, cpad // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4)
    return t.reshape(rpad, cpad)[:rows, :ncols]


def _dequant_torch(codes: np.ndarray, plain_scales: np.ndarray) -> np.ndarray:
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    sc = torch.from_numpy(plain_scales).view(torch.float8_e8m0fnu).to(torch.float64)
    m, k = codes.shape
    return (v.reshape(m, k // 32, 32) * sc[..., None]).reshape(m, k).numpy()


def _chain_norm_composition(m, shapes, g1_cols, seed):
    """mx_gemm_chain_norm against the composition of the entry points, bit for bit."""
    import mxfp8_block_scaled_06_gb300 as mx

    wops = [operands(seed + i, synth.TAG_W + i, n, k) for i, (n, k) in enumerate(shapes)]
    ws = [quantize_on_gpu(bits) for bits, _, _ in wops]
    a_bits, _, (ra, rsa) = operands(seed + 1, synth.TAG_A, m, shapes[0][1], -4, 4)
    aq, asc = quantize_on_gpu(a_bits)
    nw_bits = _weight(g1_cols, seed + 2)
    nw = bf16_to_device(nw_bits)
    h = handle()
    res = mx.mx_gemm_chain_norm(h, aq, asc, ws, nw, 1e-6, g1_cols=g1_cols, debug=True)
    o1 = mx.mx_gemm(h, aq, asc, *ws[0])
    a2, a2s, y = mx.mx_rmsnorm_quantize_rows(h, o1[:, :g1_cols], nw, 1e-6, y=True)
    o2 = mx.mx_gemm(h, a2, a2s, *ws[1])
    a3, a3s = mx.mx_quantize_rows(h, o2)
    o3 = mx.mx_gemm(h, a3, a3s, *ws[2])
    torch.cuda.synchronize()
    assert mx.mx_device_status(h) == mx.MX_OK
    # 1. the chain is the composition of the entry points, bit for bit
    for name, got, want in [("out1", res["out1"], o1), ("y", res["y"], y), ("a2", res["a2"], a2),
                            ("a2_scales", res["a2_scales"], a2s), ("out2", res["out2"], o2),
                            ("a3", res["a3"], a3), ("a3_scales", res["a3_scales"], a3s),
                            ("out", res["out"], o3)]:
        assert torch.equal(got.view(torch.uint8), want.view(torch.uint8)), name
    return res, wops, ra, rsa, nw_bits


@pytest.mark.parametrize("m", [1, 16])
def test_chain_norm_small_shapes(m):
    # a shorter normalized row (g1_cols = 256: 8 blocks, fewer than a lane's loads)
    _chain_norm_composition(m, [(384, 640), (256, 256), (512, 256)], 256, seed=70)


# 1, 2, 3 and 5 rows: G2 splits each 32-block of its prologue over 8, 4, 2 and
# 2 threads (its K-range holds 12 blocks a row), from 16 rows one thread a block
@pytest.mark.parametrize("m", [1, 2, 3, 5, 16, 17, 40, 130])
def test_chain_norm_equals_composition_and_oracle(m):
    shapes = [(2048, 5120), (8192, 1536), (5120, 8192)]
    res, wops, ra, rsa, nw_bits = _chain_norm_composition(m, shapes, 1536, seed=60)
    # 2. against the oracle chain on the oracle's own operands
    ora = oracle.chain_norm(ra, rsa, [ops[2] for ops in wops], synth.bf16_bits_to_f64(nw_bits), 1e-6)
    assert_gemm_close(res["out1"], ora["out1"], "chain-norm G1")
    gc2 = u8(res["a2"])
    assert (gc2 != ora["a2"]).mean() <= 5e-3  # only where a bf16 rounding went the other way
    gc3 = u8(res["a3"])
    gs3 = _plain_test_side(u8(res["a3_scales"]), m, 8192 // 32)
    delta = np.abs(_dequant_torch(gc3, gs3) - _dequant_torch(ora["a3"], ora["a3s"]))
    w3 = _dequant_torch(*wops[2][2])
    extra = 1.01 * (delta @ np.abs(w3).T)
    got = res["out"].float().cpu().numpy().astype(np.float64)
    ref = ora["out3"]
    assert (np.abs(got - ref) <= oracle.gemm_tolerance(ref) + extra).all()
