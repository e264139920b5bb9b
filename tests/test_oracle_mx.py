"""Pins of the oracle's MX block quantization, scale layout, GEMM, chain and
WO-A against brute force, exact rational arithmetic, closed forms and
invariants (none of them re-calls the function under test)."""
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth


# ---------------------------------------------------------------- brute force
def _table():
    codes = np.arange(0x7F)
    return codes, [Fraction(float(v)) for v in oracle.e4m3_decode(codes)]


def _brute_code(x: Fraction) -> int:
    codes, vals = _table()
    a = abs(x)
    if a >= 448:
        c = 0x7E
    else:
        best = min(abs(a - v) for v in vals)
        tied = [int(c) for c, v in zip(codes, vals) if abs(a - v) == best]
        even = [c for c in tied if c % 2 == 0]
        c = even[0] if even else tied[0]
    return c | (0x80 if x < 0 or (x == 0 and math.copysign(1.0, float(x)) < 0) else 0)


def _brute_block(xs):
    """Scale exponent = the smallest e with every |x| < 2**(e + 9) (i.e. the
    largest binade of E4M3, 2**8, holds amax), searched over [-127, 127]."""
    amax = max(abs(Fraction(float(v))) for v in xs)
    if amax == 0:
        e = -127
    else:
        e = -127
        while not amax < Fraction(2) ** (e + 9):
            e += 1
        e = min(e, 127)
    codes = []
    for v in xs:
        fv = Fraction(float(v)) / Fraction(2) ** e
        c = _brute_code(fv)
        if fv == 0 and math.copysign(1.0, float(v)) < 0:
            c = 0x80
        codes.append(c)
    return codes, e + 127


# --------------------------------------------------------------- quantization
def test_quantize_matches_brute_force_tiny():
    bits = synth.block_scaled_bf16(7, 1, 3, 96, -6, 6)
    x = synth.bf16_bits_to_f64(bits)
    x[1, 40] = -0.0
    x[2, 64:96] = 0.0
    codes, sb = oracle.mx_quantize(x)
    for r in range(3):
        for b in range(3):
            c, s = _brute_block(x[r, 32 * b:32 * b + 32])
            assert sb[r, b] == s
            assert list(codes[r, 32 * b:32 * b + 32]) == c


def test_quantize_exact_for_representable_blocks():
    rng = np.random.default_rng(1)
    for e in [-127, -40, -3, 0, 5, 100, 119]:
        c = rng.integers(0, 0x7F, size=(16, 32))
        c[:, 0] = rng.integers(0x78, 0x7F, size=16)  # amax code in [256, 448]
        c = np.where(rng.random((16, 32)) < 0.5, c | 0x80, c).astype(np.uint8)
        x = oracle.e4m3_decode(c) * 2.0**e
        codes, sb = oracle.mx_quantize(x)
        assert (sb == e + 127).all()
        np.testing.assert_array_equal(oracle.mx_dequantize(codes, sb), x)


def test_quantize_powers_of_two():
    for j in range(-100, 120, 7):
        x = np.full((1, 32), 2.0**j)
        codes, sb = oracle.mx_quantize(x)
        assert sb[0, 0] == j - 8 + 127
        assert (codes == 0x78).all()  # 2**8 = S.1111.000


def test_quantize_zero_and_subnormal_blocks():
    codes, sb = oracle.mx_quantize(np.zeros((2, 64)))
    assert (sb == 0).all() and (codes == 0).all()
    x = np.full((1, 32), -0.0)
    codes, sb = oracle.mx_quantize(x)
    assert sb[0, 0] == 0 and (codes == 0x80).all()
    # bf16 subnormals: amax 2**-130 -> exponent clamps at -127, values scale by 2**127
    x = np.arange(32, dtype=np.float64)[None, :] * 2.0**-135
    codes, sb = oracle.mx_quantize(x)
    assert sb[0, 0] == 0
    np.testing.assert_array_equal(codes[0], oracle.e4m3_encode(x[0] * 2.0**127))


def test_quantize_saturates_top_binade():
    # amax / 2**e in [448, 512) maps to 448
    for v in [448.0, 449.0, 464.0, 480.0, 511.0]:
        x = np.zeros((1, 32))
        x[0, 3] = v * 2.0**5
        x[0, 4] = -v * 2.0**5
        codes, sb = oracle.mx_quantize(x)
        assert sb[0, 0] == 5 + 127
        assert codes[0, 3] == 0x7E and codes[0, 4] == 0xFE


def test_quantize_ties_to_even():
    x = np.zeros((1, 32))
    x[0, 0] = 256.0               # sets e = 0
    x[0, 1] = 1.0625              # between 1 (even) and 1.125
    x[0, 2] = 1.1875              # between 1.125 and 1.25 (even)
    x[0, 3] = 0.0009765625        # half the smallest subnormal -> 0
    x[0, 4] = 0.0029296875        # 1.5 * 2**-9 -> 2 * 2**-9
    codes, sb = oracle.mx_quantize(x)
    assert list(codes[0, :5]) == [0x78, 0x38, 0x3A, 0x00, 0x02]


def test_quantize_nonfinite_block():
    x = np.ones((1, 64))
    x[0, 5] = np.nan
    codes, sb = oracle.mx_quantize(x)
    assert sb[0, 0] == 0xFF and (codes[0, :32] == 0x7F).all()
    assert sb[0, 1] == 127 - 8 and (codes[0, 32:] == 0x78).all()


# --------------------------------------------------------------- scale layout
@pytest.mark.parametrize("rows,k", [(1, 128), (4, 512), (130, 160), (300, 5120), (128, 96)])
def test_swizzle_bijection_and_size(rows, k):
    c = k // 32
    rpad, cpad = oracle.ceil_to(rows, 128), oracle.ceil_to(c, 4)
    assert oracle.mx_scale_bytes(rows, k) == rpad * cpad
    rr, cc = np.meshgrid(np.arange(rpad), np.arange(cpad), indexing="ij")
    off = oracle.swizzled_offset(rr, cc, c).ravel()
    assert sorted(off.tolist()) == list(range(rpad * cpad))


@pytest.mark.parametrize("rows,k", [(4, 512), (130, 160), (256, 5120)])
def test_swizzle_matches_tile_reshape(rows, k):
    """An independent construction: pad to [R, C], cut 128x4 tiles with
    reshape, and inside a tile order (row % 32, row // 32, col)."""
    c = k // 32
    s = np.random.default_rng(2).integers(1, 255, size=(rows, c)).astype(np.uint8)
    rpad, cpad = oracle.ceil_to(rows, 128), oracle.ceil_to(c, 4)
    p = np.zeros((rpad, cpad), np.uint8)
    p[:rows, :c] = s
    t = p.reshape(rpad // 128, 4, 32, cpad // 4, 4)      # (rt, r//32, r%32, ct, c%4)
    want = t.transpose(0, 3, 2, 1, 4).reshape(-1)          # (rt, ct, r%32, r//32, c%4)
    np.testing.assert_array_equal(oracle.swizzle_scales(s), want)
    np.testing.assert_array_equal(oracle.unswizzle_scales(want, rows, c), s)


def test_swizzle_golden_offsets():
    # documented examples: within the first tile, row 32 sits 4 bytes after row 0,
    # row 1 sits 16 bytes after row 0; the second 4-column tile starts at 512
    assert oracle.swizzled_offset(0, 0, 8) == 0
    assert oracle.swizzled_offset(0, 1, 8) == 1
    assert oracle.swizzled_offset(1, 0, 8) == 16
    assert oracle.swizzled_offset(32, 0, 8) == 4
    assert oracle.swizzled_offset(127, 3, 8) == 31 * 16 + 3 * 4 + 3
    assert oracle.swizzled_offset(0, 4, 8) == 512
    assert oracle.swizzled_offset(128, 0, 8) == 1024


# ----------------------------------------------------------------------- GEMM
def _c0_operands(m=4, n=256, k=512, seed=0):
    a = synth.bf16_bits_to_f64(synth.block_scaled_bf16(seed, synth.TAG_A, m, k, -6, 6))
    w = synth.bf16_bits_to_f64(synth.block_scaled_bf16(seed, synth.TAG_W, n, k, -6, 6))
    return oracle.mx_quantize(a), oracle.mx_quantize(w)


def _exact_gemm_int(ac, asb, wc, wsb):
    """Exact sum with integers: each E4M3 value is an integer multiple of 2**-9,
    so a 32-block's code products sum exactly in int64; blocks combine as
    rationals with their power-of-two scales."""
    ia = np.rint(oracle.e4m3_decode(ac) * 512).astype(np.int64)
    iw = np.rint(oracle.e4m3_decode(wc) * 512).astype(np.int64)
    m, k = ia.shape
    n = iw.shape[0]
    nb = k // 32
    blk = np.einsum("mbj,nbj->mnb", ia.reshape(m, nb, 32), iw.reshape(n, nb, 32))
    out = [[Fraction(0)] * n for _ in range(m)]
    for i in range(m):
        for j in range(n):
            tot = Fraction(0)
            for b in range(nb):
                e = int(asb[i, b]) + int(wsb[j, b]) - 254 - 18
                tot += Fraction(int(blk[i, j, b])) * (Fraction(2) ** e)
            out[i][j] = tot
    return out


def test_gemm_exact_on_tiny_config():
    (ac, asb), (wc, wsb) = _c0_operands()
    got = oracle.mx_gemm(ac, asb, wc, wsb)
    exact = _exact_gemm_int(ac, asb, wc, wsb)
    mag = np.abs(oracle.mx_dequantize(ac, asb)) @ np.abs(oracle.mx_dequantize(wc, wsb)).T
    for i in range(got.shape[0]):
        for j in range(got.shape[1]):
            assert abs(Fraction(float(got[i, j])) - exact[i][j]) <= Fraction(float(mag[i, j])) * Fraction(2) ** -45


def test_gemm_rational_brute_force():
    (ac, asb), (wc, wsb) = _c0_operands(3, 5, 64, seed=3)
    exact = oracle.mx_gemm_exact(ac, asb, wc, wsb)
    assert exact == _exact_gemm_int(ac, asb, wc, wsb)


def test_gemm_one_hot_orientation():
    # A has one non-zero at (m0, k0); W one at (n0, k0): only out[m0, n0] is set.
    m, n, k = 3, 5, 64
    ac = np.zeros((m, k), np.uint8)
    wc = np.zeros((n, k), np.uint8)
    asb = np.full((m, 2), 127, np.uint8)
    wsb = np.full((n, 2), 127, np.uint8)
    ac[2, 40] = 0x40   # 2.0
    wc[4, 40] = 0xB8   # -1.0
    asb[2, 1] = 130    # x 8
    wsb[4, 1] = 125    # x 1/4
    out = oracle.mx_gemm(ac, asb, wc, wsb)
    want = np.zeros((m, n))
    want[2, 4] = 2.0 * 8 * -1.0 / 4
    np.testing.assert_array_equal(out, want)


def test_gemm_zero_input_gives_zero():
    ac = np.zeros((8, 256), np.uint8)
    asb = np.zeros((8, 8), np.uint8)
    (_, _), (wc, wsb) = _c0_operands(1, 64, 256)
    assert (oracle.mx_gemm(ac, asb, wc, wsb) == 0).all()


def test_tolerance_rule():
    ref = np.array([3.0, -4.0, 0.0])
    np.testing.assert_allclose(oracle.gemm_tolerance(ref), 1e-2 * np.abs(ref) + 1e-3 * math.sqrt(25 / 3))


# ---------------------------------------------------------------------- chain
def _nearest_bf16(v: Fraction) -> float:
    """The bf16 number nearest the rational v, ties to the even significand,
    found by searching the bf16 neighbours of v's float32 neighbours."""
    f = float(v)
    cands = {f, float(np.nextafter(np.float32(f), np.float32(np.inf))),
             float(np.nextafter(np.float32(f), np.float32(-np.inf)))}
    bf = set()
    for c in cands:
        b = np.array([c], np.float32).view(np.uint32)[0] & np.uint32(0xFFFF0000)
        for d in (0, 1, -1):
            bb = np.uint32(int(b) + d * 0x10000)
            bf.add(float(np.array([bb], np.uint32).view(np.float32)[0]))
    return min(bf, key=lambda y: (abs(Fraction(y) - v), (np.array([y], np.float32).view(np.uint32)[0] >> 16) & 1))


def _exact_stage(ac, asb, wc, wsb) -> np.ndarray:
    """One projection evaluated exactly with rationals, rounded once to bf16."""
    ex = oracle.mx_gemm_exact(ac, asb, wc, wsb)
    return np.array([[_nearest_bf16(v) for v in row] for row in ex])


def _brute_requant(b, cols):
    """(codes [rows][32-blocks], scale bytes) of b's first cols columns by brute force."""
    blocks = [_brute_block(b[r, 32 * c:32 * c + 32]) for r in range(b.shape[0]) for c in range(cols // 32)]
    return [c for c, _ in blocks], [s for _, s in blocks]


def _blocks(codes):
    return [[int(x) for x in blk] for blk in np.asarray(codes).reshape(-1, 32)]


def test_chain_tiny_brute_force():
    m, k1, n1, g1, n2, n3 = 2, 64, 96, 64, 64, 32
    a = synth.bf16_bits_to_f64(synth.block_scaled_bf16(5, 1, m, k1, -4, 4))
    ws = [synth.bf16_bits_to_f64(synth.block_scaled_bf16(5, 10 + i, n, kk, -6, 6))
          for i, (n, kk) in enumerate([(n1, k1), (n2, g1), (n3, n2)])]
    aq = oracle.mx_quantize(a)
    wq = [oracle.mx_quantize(w) for w in ws]
    got = oracle.chain(aq[0], aq[1], wq, g1_cols=g1)

    b1 = _exact_stage(aq[0], aq[1], *wq[0])
    np.testing.assert_array_equal(got["b1"], b1)
    a2 = [_brute_block(b1[r, 32 * c:32 * c + 32]) for r in range(m) for c in range(g1 // 32)]
    assert [int(x) for x in got["a2s"].ravel()] == [s for _, s in a2]
    assert [[int(x) for x in blk] for blk in got["a2"].reshape(-1, 32)] == [c for c, _ in a2]
    b2 = _exact_stage(got["a2"], got["a2s"], *wq[1])
    np.testing.assert_array_equal(got["b2"], b2)
    a3 = [_brute_block(b2[r, 32 * c:32 * c + 32]) for r in range(m) for c in range(n2 // 32)]
    assert [int(x) for x in got["a3s"].ravel()] == [s for _, s in a3]
    assert [[int(x) for x in blk] for blk in got["a3"].reshape(-1, 32)] == [c for c, _ in a3]
    b3 = _exact_stage(got["a3"], got["a3s"], *wq[2])
    np.testing.assert_array_equal(got["b3"], b3)


# ----------------------------------------------------------------------- RoPE
def test_rope_cache_closed_forms():
    cs = synth.rope_cos_sin_cache(max_pos=1000)
    np.testing.assert_array_equal(cs[0], np.r_[np.ones(32), np.zeros(32)].astype(np.float32))
    for p, i in [(1, 0), (999, 5), (17, 31)]:
        th = p * 10000.0 ** (-2 * i / 64)
        assert cs[p, i] == np.float32(math.cos(th))
        assert cs[p, 32 + i] == np.float32(math.sin(th))


def test_rope_identity_at_position_zero():
    x = synth.bf16_bits_to_f64(synth.normal_bf16(1, 2, (3, 4, 512))).astype(np.float32)
    act = oracle.wo_a_activation(x, np.zeros(3, np.int64), synth.rope_cos_sin_cache(8))
    np.testing.assert_array_equal(act, x)


def test_rope_direction_quarter_turn():
    # cos = 0, sin = 1 is theta = pi/2: rotating by -theta maps (a, b) to (b, -a)
    x = np.array([[1.5, -2.25, 3.0, 0.5]], np.float32)
    out = oracle.rope_rotate_inverse(x, np.zeros((1, 2), np.float32), np.ones((1, 2), np.float32))
    np.testing.assert_array_equal(out, [[-2.25, -1.5, 0.5, -3.0]])


def test_rope_matches_float64_rotation_and_inverts():
    cs = synth.rope_cos_sin_cache(65536)
    pos = synth.positions(3, 1, 64)
    x = synth.bf16_bits_to_f64(synth.normal_bf16(3, 2, (64, 2, 512))).astype(np.float32)
    act = oracle.wo_a_activation(x, pos, cs)
    c = cs[pos][:, None, :32].astype(np.float64)
    s = cs[pos][:, None, 32:].astype(np.float64)
    a = x[..., 448::2].astype(np.float64)
    b = x[..., 449::2].astype(np.float64)
    np.testing.assert_allclose(act[..., 448::2], a * c + b * s, rtol=0, atol=4e-7 * (abs(a) + abs(b)).max())
    np.testing.assert_allclose(act[..., 449::2], b * c - a * s, rtol=0, atol=4e-7 * (abs(a) + abs(b)).max())
    # norms preserved, nope dims untouched
    n0 = np.hypot(a, b)
    n1 = np.hypot(act[..., 448::2].astype(np.float64), act[..., 449::2].astype(np.float64))
    np.testing.assert_allclose(n1, n0, rtol=1e-6, atol=1e-30)
    np.testing.assert_array_equal(act[..., :448], x[..., :448])
    # rotating forward by +theta (a c - b s, a s + b c) returns the input
    r = act[..., 448:].astype(np.float64)
    back_a = r[..., 0::2] * c - r[..., 1::2] * s
    back_b = r[..., 0::2] * s + r[..., 1::2] * c
    np.testing.assert_allclose(back_a, a, atol=1e-6 * (abs(a) + abs(b)).max())
    np.testing.assert_allclose(back_b, b, atol=1e-6 * (abs(a) + abs(b)).max())


# ----------------------------------------------------------------------- WO-A
def test_wo_a_tiny_brute_force():
    t, g, h, r = 1, 2, 2, 16  # two heads per group: the group takes contiguous heads
    x = synth.bf16_bits_to_f64(synth.normal_bf16(9, 1, (t, g * h, 512)))
    pos = np.array([12345], np.int64)
    cs = synth.rope_cos_sin_cache(65536)
    w = synth.bf16_bits_to_f64(synth.block_scaled_bf16(9, 2, g * r, h * 512, -6, 6))
    wc, ws = oracle.mx_quantize(w)
    got = oracle.wo_a_grouped(x, pos, cs, wc, ws, n_groups=g, heads_per_group=h, o_lora_rank=r)
    # rope by scalar float32 arithmetic, element by element
    act = x.astype(np.float32).copy()
    c_row, s_row = cs[pos[0], :32], cs[pos[0], 32:]
    for hh in range(g * h):
        for i in range(32):
            a = np.float32(x[0, hh, 448 + 2 * i])
            b = np.float32(x[0, hh, 449 + 2 * i])
            act[0, hh, 448 + 2 * i] = np.float32(np.float32(a * c_row[i]) + np.float32(b * s_row[i]))
            act[0, hh, 449 + 2 * i] = np.float32(np.float32(b * c_row[i]) - np.float32(a * s_row[i]))
    np.testing.assert_array_equal(got["act"], act)
    for gg in range(g):
        xg = act[0, gg * h:(gg + 1) * h].reshape(-1).astype(np.float64)
        for blk in range(xg.size // 32):
            codes, s = _brute_block(xg[32 * blk:32 * blk + 32])
            col = gg * h * 512 + 32 * blk
            assert list(got["xq"][0, col:col + 32]) == codes
            assert got["xs"][0, col // 32] == s
        ex = oracle.mx_gemm_exact(got["xq"][:, gg * 512 * h:(gg + 1) * 512 * h],
                                  got["xs"][:, gg * 16 * h:(gg + 1) * 16 * h],
                                  wc[gg * r:(gg + 1) * r], ws[gg * r:(gg + 1) * r])
        for j in range(r):
            assert abs(Fraction(float(got["z"][0, gg * r + j])) - ex[0][j]) <= abs(ex[0][j]) * Fraction(2) ** -40 + Fraction(2) ** -200
            assert got["zb"][0, gg * r + j] == _nearest_bf16(ex[0][j])
    codes, scales = _brute_requant(got["zb"], g * r)
    assert _blocks(got["q"]) == codes
    assert [int(x) for x in got["qs"].ravel()] == scales


# ------------------------------------------------------------ RMS norm split
def test_rms_norm_closed_forms():
    # [3, 4]: mean square 12.5, so y = (3, 4) / (5 / sqrt 2) = (3 sqrt2 / 5, 4 sqrt2 / 5)
    y = oracle.rms_norm(np.array([[3.0, 4.0]]), np.ones(2), 0.0)
    np.testing.assert_allclose(y[0], [3 * np.sqrt(2) / 5, 4 * np.sqrt(2) / 5], rtol=0, atol=1e-15)
    # a constant row normalizes to the weight itself (eps = 0), with the row's sign
    w = np.array([0.5, -2.0, 3.0, 1.0])
    np.testing.assert_array_equal(oracle.rms_norm(np.full((1, 4), -7.25), w, 0.0)[0], -w)
    # a zero row stays zero with eps > 0
    assert (oracle.rms_norm(np.zeros((1, 8)), np.ones(8), 1e-6) == 0).all()


def test_rms_norm_invariants():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 96))
    y = oracle.rms_norm(x, np.ones(96), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)  # unit RMS
    for k in (-20, -3, 5, 40):  # scale invariance: powers of two scale exactly
        np.testing.assert_array_equal(oracle.rms_norm(np.ldexp(x, k), np.ones(96), 0.0), y)
    # eps lowers the result toward zero, by sqrt(ms / (ms + eps))
    ms = np.mean(x * x, axis=-1, keepdims=True)
    np.testing.assert_allclose(oracle.rms_norm(x, np.ones(96), 0.25), y * np.sqrt(ms / (ms + 0.25)),
                               rtol=1e-13)


def test_split_qkv_and_norm_parts():
    rng = np.random.default_rng(6)
    out1 = oracle.round_bf16(rng.standard_normal((3, 2048)) * 4)
    w = oracle.round_bf16(rng.uniform(0.5, 1.5, 1536))
    sp = oracle.split_qkv_and_norm(out1, w, 1e-6)
    np.testing.assert_array_equal(sp["kv"], out1[:, 1536:])
    assert sp["y"].shape == (3, 1536) and (oracle.round_bf16(sp["y"]) == sp["y"]).all()
    q2, s2 = oracle.mx_quantize(sp["y"])
    np.testing.assert_array_equal(sp["q"], q2)
    np.testing.assert_array_equal(sp["qs"], s2)
    # the norm runs over the first 1536 columns only: scaling or zeroing the kv
    # columns changes nothing in y, q or qs
    for kv in (out1[:, 1536:] * 64, np.zeros((3, 512))):
        sp2 = oracle.split_qkv_and_norm(np.concatenate([out1[:, :1536], kv], axis=1), w, 1e-6)
        for key in ("y", "q", "qs"):
            np.testing.assert_array_equal(sp2[key], sp[key])
    # with a unit weight and eps 0, each normalized row has unit mean square
    # (up to the bf16 rounding of y, relative 2**-8 per element)
    y1 = oracle.split_qkv_and_norm(out1, np.ones(1536), 0.0)["y"]
    assert np.all(np.abs(np.mean(y1 * y1, axis=-1) - 1.0) <= 2.0 ** -7)


def _decimal_rms_norm_bf16(row, weight, eps) -> np.ndarray:
    """RMS norm of one row evaluated in 60-digit decimal arithmetic, each
    element rounded once to the nearest bf16."""
    getcontext().prec = 60
    xs = [Decimal(Fraction(float(v)).numerator) / Decimal(Fraction(float(v)).denominator) for v in row]
    ms = sum(x * x for x in xs) / len(xs)
    inv = 1 / (ms + Decimal(eps)).sqrt()
    out = []
    for x, w in zip(xs, weight):
        v = Fraction(x * inv * (Decimal(Fraction(float(w)).numerator) / Decimal(Fraction(float(w)).denominator)))
        out.append(_nearest_bf16(v))
    return np.array(out)


def test_chain_norm_tiny_brute_force():
    m, k1, n1, g1, n2, n3 = 2, 64, 96, 64, 64, 32
    a = synth.bf16_bits_to_f64(synth.block_scaled_bf16(8, 1, m, k1, -4, 4))
    ws = [synth.bf16_bits_to_f64(synth.block_scaled_bf16(8, 10 + i, n, kk, -6, 6))
          for i, (n, kk) in enumerate([(n1, k1), (n2, g1), (n3, n2)])]
    nw = synth.bf16_bits_to_f64(synth.norm_weight_bf16(8, g1))
    aq = oracle.mx_quantize(a)
    wq = [oracle.mx_quantize(w) for w in ws]
    got = oracle.chain_norm(aq[0], aq[1], wq, nw, 1e-6, g1_cols=g1)
    b1 = _exact_stage(aq[0], aq[1], *wq[0])
    np.testing.assert_array_equal(got["b1"], b1)
    np.testing.assert_array_equal(got["kv"], b1[:, g1:])
    y = np.stack([_decimal_rms_norm_bf16(b1[r, :g1], nw, 1e-6) for r in range(m)])
    np.testing.assert_array_equal(got["y"], y)
    codes, scales = _brute_requant(y, g1)
    assert _blocks(got["a2"]) == codes and [int(x) for x in got["a2s"].ravel()] == scales
    b2 = _exact_stage(got["a2"], got["a2s"], *wq[1])
    np.testing.assert_array_equal(got["b2"], b2)
    codes, scales = _brute_requant(b2, n2)
    assert _blocks(got["a3"]) == codes and [int(x) for x in got["a3s"].ravel()] == scales
    np.testing.assert_array_equal(got["b3"], _exact_stage(got["a3"], got["a3s"], *wq[2]))


def test_chain_norm_removes_the_input_scale():
    """Scaling the layer input by 2**k scales G1's output by 2**k exactly; with
    eps = 0 the norm divides it out again, so everything after it is unchanged."""
    m, k1, n1, g1, n2, n3 = 3, 128, 256, 128, 128, 128
    a = synth.bf16_bits_to_f64(synth.block_scaled_bf16(9, 1, m, k1, -2, 2))
    wq = [oracle.mx_quantize(synth.bf16_bits_to_f64(synth.block_scaled_bf16(9, 10 + i, n, kk, -2, 2)))
          for i, (n, kk) in enumerate([(n1, k1), (n2, g1), (n3, n2)])]
    nw = synth.bf16_bits_to_f64(synth.norm_weight_bf16(9, g1))
    ac, asb = oracle.mx_quantize(a)
    base = oracle.chain_norm(ac, asb, wq, nw, 0.0, g1_cols=g1)
    for k in (-5, 3, 9):
        got = oracle.chain_norm(ac, (asb.astype(np.int64) + k).astype(np.uint8), wq, nw, 0.0, g1_cols=g1)
        np.testing.assert_array_equal(got["b1"], np.ldexp(base["b1"], k))
        for key in ("y", "a2", "a2s", "b2", "a3", "a3s", "b3"):
            np.testing.assert_array_equal(got[key], base[key])
