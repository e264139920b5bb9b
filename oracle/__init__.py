"""CPU oracle for the low-batch MXFP8 block-scaled projections.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
(and its ``--impl reference`` arm) call it. It shares no code with the CUDA
library; the only thing both sides share is the seeded input generator in
``synth`` (random numbers, none of the arithmetic below).

Everything is plain numpy, evaluated exactly or in float64, in the order the
method states; a library matmul is the only borrowed step. Sources:

* "vllm ... specialized_decode.attention.mxfp8" (MXFP8 attention projections):
  module docstring (E4M3 data, UE8M0 scales, F8_128x4 activation scales),
  ``launch_low_latency`` (out = a x W with W column-major [K, N], bf16 out, no
  scale or bias), ``compile_low_latency`` (Float8E4M3FN / Float8E8M0FNU operands,
  sf_vec_size 32, float32 accumulator), ``_zeros`` (zero data with zero scale
  bytes is a valid input).
* "vllm ... ops.o_proj" (DSV4.1 output projection): ``_can_fuse_wo_a`` (448 nope
  + 64 rope dims, per-32 FP8 weight recipe (1, 1, 32), groups of <= 8 heads,
  o_lora_rank % 128 == 0), ``dsv41_o_proj`` (RoPE from the cos/sin cache, grouped
  contraction, the result handed on as an MXFP8 activation (q, scales)).
* The MX block rule (scale exponent = floor(log2 amax) - 8, saturating
  round-to-nearest-even into E4M3) as the OCP Microscaling format fixes it for
  E4M3 elements (largest power of two of E4M3 is 2**8).

Readings where the pages are silent (each also listed in the design notes):
  - an all-zero block gets scale byte 0 and +-0 codes (``_zeros`` uses zero
    scale bytes); the exponent is clamped to [-127, 127];
  - a block holding NaN or Inf gets scale byte 0xFF and NaN codes (0x7F);
  - the F8_128x4 layout is NVIDIA's documented 128x4 block-scale-factor layout
    (see ``swizzled_offset``);
  - the projection chain rounds each product to bf16 (RNE) before requantizing;
  - WO-A rotates the rope pairs in float32 without fused multiply-add, keeps the
    rotated values in float32 (no bf16 round) and quantizes per 32 elements.
  - the split between G1 and G2 (``_split_qkv_and_norm``, shown only as a call):
    qr = G1's first 1536 bf16 columns, RMS-normalized over them with a given
    weight and epsilon, rounded to bf16, MX-quantized; kv = the other columns.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(exhaustive codec tables, torch's independent float8 cast, brute force, exact
rational evaluation, closed forms, an independent reshape construction of the
scale layout). The WO-A operation order is a reading, pinned only by its
closed-form special cases (identity rotation at position 0, exact inverse).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN = 0x7F
SCALE_NAN = 0xFF
SF_VEC = 32  # elements per scale (sf_vec_size)


# ----------------------------------------------------------------------------
# E4M3 (fn) codec: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinity,
# S.1111.111 is NaN, largest finite 448, subnormals k * 2**-9.
# ----------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 byte, float64 (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0**-9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e4m3_encode(v) -> np.ndarray:
    """Round float64 values to E4M3 codes: nearest, ties to the even code,
    finite magnitudes above 448 (and +-Inf) saturate to +-448, NaN -> 0x7F,
    the sign of zero (and of values that round to zero) is kept."""
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # quantum of a's binade; binades below 2**-6 share the subnormal quantum 2**-9
    _, ex = np.frexp(a)
    binade = np.maximum(np.where(a > 0, ex - 1, -6), -6)
    quantum = np.exp2(binade - 3.0)
    val = np.rint(a / quantum) * quantum  # a / quantum is exact; rint is half-even
    val = np.minimum(val, E4M3_MAX)
    # bits of the rounded magnitude
    _, ex2 = np.frexp(val)
    ev = np.where(val > 0, ex2 - 1, 0)
    is_norm = val >= 2.0**-6
    mant_norm = np.where(is_norm, val / np.exp2(ev) * 8.0 - 8.0, 0.0)
    code_norm = ((ev + 7) << 3) + mant_norm.astype(np.int64)
    code_sub = (val / 2.0**-9).astype(np.int64)
    code = np.where(is_norm, code_norm, code_sub)
    code = np.where(neg, code | 0x80, code)
    code = np.where(nan, E4M3_NAN, code)
    return code.astype(np.uint8)


def ue8m0_decode(s) -> np.ndarray:
    """Value of UE8M0 scale bytes: 2**(s - 127); 0xFF is NaN."""
    s = np.asarray(s).astype(np.int64)
    return np.where(s == SCALE_NAN, np.nan, np.exp2(s - 127.0))


# ----------------------------------------------------------------------------
# MX block quantization (one UE8M0 scale per 32 consecutive K elements)
# ----------------------------------------------------------------------------
def mx_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """Quantize rows of x (float64 holding exact bf16 / fp32 values), shape
    [R, K] with K % 32 == 0, to (E4M3 codes uint8 [R, K], scale bytes uint8
    [R, K/32] in plain row-major order).

    Per block of 32: amax = max |x|; e = floor(log2 amax) - 8 clamped to
    [-127, 127] (e = -127 for an all-zero block); codes = E4M3(x * 2**-e) with
    saturating nearest-even rounding; scale byte = e + 127.
    """
    x = np.asarray(x, dtype=np.float64)
    r, k = x.shape
    assert k % SF_VEC == 0, "K must be a multiple of 32"
    blk = x.reshape(r, k // SF_VEC, SF_VEC)
    finite = np.isfinite(blk).all(axis=-1)
    amax = np.max(np.abs(np.where(np.isfinite(blk), blk, 0.0)), axis=-1)
    _, ex = np.frexp(amax)
    e = np.where(amax > 0, (ex - 1) - 8, -127)  # frexp: amax = f * 2**ex, f in [0.5, 1)
    e = np.clip(e, -127, 127)
    scaled = np.ldexp(np.where(np.isfinite(blk), blk, 0.0), -e[..., None])
    codes = e4m3_encode(scaled)
    codes = np.where(finite[..., None], codes, E4M3_NAN).astype(np.uint8)
    sbytes = np.where(finite, e + 127, SCALE_NAN).astype(np.uint8)
    return codes.reshape(r, k), sbytes


def mx_dequantize(codes, sbytes) -> np.ndarray:
    """float64 values of an MXFP8 tensor given codes [R, K] and plain scale bytes [R, K/32]."""
    codes = np.asarray(codes)
    r, k = codes.shape
    vals = e4m3_decode(codes).reshape(r, k // SF_VEC, SF_VEC)
    return (vals * ue8m0_decode(sbytes)[..., None]).reshape(r, k)


# ----------------------------------------------------------------------------
# F8_128x4 swizzled scale layout (NVIDIA's 128x4 block-scale-factor layout):
# the [rows, K/32] scale matrix is padded to a multiple of 128 rows and 4
# columns and cut into 128x4 tiles of 512 contiguous bytes, tiles ordered
# row-major; inside a tile, (r, c) sits at 16 * (r % 32) + 4 * (r // 32) + c.
# ----------------------------------------------------------------------------
def ceil_to(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def mx_scale_bytes(rows: int, k: int) -> int:
    """Size of the swizzled scale buffer of a [rows, k] operand."""
    return ceil_to(rows, 128) * ceil_to(k // SF_VEC, 4)


def swizzled_offset(r, c, n_cols: int):
    """Byte offset of scale (row r, block column c) for n_cols = K/32 block columns."""
    cpad = ceil_to(n_cols, 4)
    tile = (np.asarray(r) // 128) * (cpad // 4) + np.asarray(c) // 4
    inner = (np.asarray(r) % 32) * 16 + ((np.asarray(r) % 128) // 32) * 4 + np.asarray(c) % 4
    return tile * 512 + inner


def swizzle_scales(sbytes) -> np.ndarray:
    """Plain [R, C] scale bytes -> swizzled flat buffer, padding bytes zero."""
    sbytes = np.asarray(sbytes, dtype=np.uint8)
    r, c = sbytes.shape
    out = np.zeros(ceil_to(r, 128) * ceil_to(c, 4), dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(r), np.arange(c), indexing="ij")
    out[swizzled_offset(rr, cc, c)] = sbytes
    return out


def unswizzle_scales(buf, rows: int, n_cols: int) -> np.ndarray:
    """Swizzled flat buffer -> plain [rows, n_cols] scale bytes."""
    rr, cc = np.meshgrid(np.arange(rows), np.arange(n_cols), indexing="ij")
    return np.asarray(buf, dtype=np.uint8)[swizzled_offset(rr, cc, n_cols)]


# ----------------------------------------------------------------------------
# bfloat16 rounding (nearest-even, one rounding from float64)
# ----------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round float64 to the nearest bfloat16 value (ties to even), as float64."""
    x = np.asarray(x, dtype=np.float64)
    _, ex = np.frexp(x)
    # bf16 has 8 significant bits; its subnormal quantum is 2**-133
    quantum = np.exp2(np.maximum(np.where(x != 0, ex, -125) - 8, -133).astype(np.float64))
    return np.rint(x / quantum) * quantum


def bf16_bits(x) -> np.ndarray:
    """Bit patterns (uint16) of float64 values that are exact bfloat16 numbers."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
    return (f >> np.uint32(16)).astype(np.uint16)


# ----------------------------------------------------------------------------
# The block-scaled GEMM
# ----------------------------------------------------------------------------
def mx_gemm(a_codes, a_sbytes, w_codes, w_sbytes) -> np.ndarray:
    """out[m, n] = sum_k dA[m, k] * dW[n, k] in float64, where dX is the E4M3
    value times 2**(s - 127) of its 32-block. A is [M, K], W is [N, K] (the
    column-major [K, N] weight of ``launch_low_latency``). Scales are plain
    [rows, K/32]."""
    return mx_dequantize(a_codes, a_sbytes) @ mx_dequantize(w_codes, w_sbytes).T


def mx_gemm_exact(a_codes, a_sbytes, w_codes, w_sbytes) -> list[list[Fraction]]:
    """The same contraction evaluated exactly with rationals (tiny shapes only)."""
    da = mx_dequantize(a_codes, a_sbytes)
    dw = mx_dequantize(w_codes, w_sbytes)
    m, k = da.shape
    n = dw.shape[0]
    fa = [[Fraction(float(da[i, j])) for j in range(k)] for i in range(m)]
    fw = [[Fraction(float(dw[i, j])) for j in range(k)] for i in range(n)]
    return [[sum(fa[i][j] * fw[c][j] for j in range(k)) for c in range(n)] for i in range(m)]


# ----------------------------------------------------------------------------
# Three-projection chain (fused_wqa_wkv -> wq_b -> wo_b of the decode step)
# ----------------------------------------------------------------------------
def chain(a1_codes, a1_sbytes, weights, g1_cols: int = 1536) -> dict:
    """G1 on the MXFP8 layer input; its bf16 output's first g1_cols columns are
    requantized and fed to G2; G2's whole bf16 output is requantized and fed to
    G3. weights = [(codes, plain scale bytes)] * 3. Returns every stage."""
    (w1, s1), (w2, s2), (w3, s3) = weights
    out1 = mx_gemm(a1_codes, a1_sbytes, w1, s1)
    b1 = round_bf16(out1)
    a2, a2s = mx_quantize(b1[:, :g1_cols])
    out2 = mx_gemm(a2, a2s, w2, s2)
    b2 = round_bf16(out2)
    a3, a3s = mx_quantize(b2)
    out3 = mx_gemm(a3, a3s, w3, s3)
    return dict(out1=out1, b1=b1, a2=a2, a2s=a2s, out2=out2, b2=b2, a3=a3, a3s=a3s,
                out3=out3, b3=round_bf16(out3))


def rms_norm(x, weight, eps: float) -> np.ndarray:
    """Each row over its last axis: x / sqrt(mean(x^2) + eps) * weight, float64."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(weight, dtype=np.float64)


def split_qkv_and_norm(out1_bf16, norm_weight, eps: float, q_cols: int = 1536) -> dict:
    """The split between the first two projections (`_split_qkv_and_norm` in
    `AttentionStep.run`; reading: the pages show only its call). qr = the first
    q_cols columns of G1's bf16 output, RMS-normalized over those columns with
    the given weight and epsilon, rounded to bf16 and MX-quantized for G2; kv =
    the remaining columns, unchanged."""
    out1_bf16 = np.asarray(out1_bf16, dtype=np.float64)
    y = round_bf16(rms_norm(out1_bf16[:, :q_cols], norm_weight, eps))
    q, qs = mx_quantize(y)
    return dict(y=y, q=q, qs=qs, kv=out1_bf16[:, q_cols:])


def chain_norm(a1_codes, a1_sbytes, weights, norm_weight, eps: float, g1_cols: int = 1536) -> dict:
    """`chain` with the split-and-norm between G1 and G2 instead of the plain
    requantization of G1's first g1_cols columns."""
    (w1, s1), (w2, s2), (w3, s3) = weights
    out1 = mx_gemm(a1_codes, a1_sbytes, w1, s1)
    b1 = round_bf16(out1)
    sp = split_qkv_and_norm(b1, norm_weight, eps, g1_cols)
    out2 = mx_gemm(sp["q"], sp["qs"], w2, s2)
    b2 = round_bf16(out2)
    a3, a3s = mx_quantize(b2)
    out3 = mx_gemm(a3, a3s, w3, s3)
    return dict(out1=out1, b1=b1, y=sp["y"], a2=sp["q"], a2s=sp["qs"], kv=sp["kv"], out2=out2,
                b2=b2, a3=a3, a3s=a3s, out3=out3, b3=round_bf16(out3))


# ----------------------------------------------------------------------------
# Grouped WO-A with RoPE, feeding wo_b as MXFP8
# ----------------------------------------------------------------------------
def rope_rotate_inverse(xr, cos, sin) -> np.ndarray:
    """Rotate adjacent pairs (x[2i], x[2i+1]) of float32 xr [..., 2h] by -theta_i:
    a' = a cos + b sin, b' = b cos - a sin, each product and sum rounded to
    float32 (no fused multiply-add). cos, sin: float32 [..., h]."""
    xr = np.asarray(xr, dtype=np.float32)
    a, b = xr[..., 0::2], xr[..., 1::2]
    c = np.asarray(cos, dtype=np.float32)
    s = np.asarray(sin, dtype=np.float32)
    a2 = (a * c) + (b * s)
    b2 = (b * c) - (a * s)
    out = np.empty_like(xr)
    out[..., 0::2] = a2
    out[..., 1::2] = b2
    return out


def wo_a_activation(x, positions, cos_sin, d_nope: int = 448, d_rope: int = 64) -> np.ndarray:
    """float32 [T, heads, d_nope + d_rope]: nope dims as given, rope dims rotated
    by -pos * f_i with cos/sin read from the float32 cache row of each token."""
    x = np.asarray(x, dtype=np.float32)
    half = d_rope // 2
    rows = np.asarray(cos_sin, dtype=np.float32)[np.asarray(positions, dtype=np.int64)]
    cos = rows[:, None, :half]
    sin = rows[:, None, half:2 * half]
    act = x.copy()
    act[..., d_nope:d_nope + d_rope] = rope_rotate_inverse(x[..., d_nope:d_nope + d_rope], cos, sin)
    return act


def wo_a_grouped(x, positions, cos_sin, w_codes, w_sbytes, n_groups: int = 4,
                 heads_per_group: int = 8, d_nope: int = 448, d_rope: int = 64,
                 o_lora_rank: int = 1024) -> dict:
    """x: [T, n_groups * heads_per_group, d] exact bf16 values (float64 or float32);
    w_codes [n_groups * o_lora_rank, heads_per_group * d], w_sbytes plain scales.
    z[t, g R + r] = sum_k dXg[t, k] dWg[r, k] with Xg the group's heads, RoPE'd and
    MX-quantized; z is rounded to bf16 and MX-quantized for wo_b."""
    d = d_nope + d_rope
    t = x.shape[0]
    act = wo_a_activation(x, positions, cos_sin, d_nope, d_rope)
    kg = heads_per_group * d
    xq = np.zeros((t, n_groups * kg), dtype=np.uint8)
    xs = np.zeros((t, n_groups * kg // SF_VEC), dtype=np.uint8)
    z = np.zeros((t, n_groups * o_lora_rank))
    for g in range(n_groups):
        xg = act[:, g * heads_per_group:(g + 1) * heads_per_group, :].reshape(t, kg)
        cq, cs = mx_quantize(xg.astype(np.float64))
        xq[:, g * kg:(g + 1) * kg] = cq
        xs[:, g * kg // SF_VEC:(g + 1) * kg // SF_VEC] = cs
        rows = slice(g * o_lora_rank, (g + 1) * o_lora_rank)
        z[:, rows] = mx_gemm(cq, cs, w_codes[rows], w_sbytes[rows])
    zb = round_bf16(z)
    q, qs = mx_quantize(zb)
    return dict(act=act, xq=xq, xs=xs, z=z, zb=zb, q=q, qs=qs)


# ----------------------------------------------------------------------------
# Acceptance rule for GEMM outputs
# ----------------------------------------------------------------------------
def gemm_tolerance(ref) -> np.ndarray:
    """Per-element bound 1e-2 |ref| + 1e-3 rms(ref)."""
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    return 1e-2 * np.abs(ref) + 1e-3 * rms
