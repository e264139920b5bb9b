"""Pins of the oracle's E4M3 codec, UE8M0 scales and bf16 rounding against
things other than itself: torch's independent float8/bfloat16 casts, the OCP
format table (tests/golden/e4m3_points.txt), and a brute-force nearest-code search."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _positive_table():
    codes = np.arange(0x7F, dtype=np.uint8)  # 0x00..0x7E: every finite non-negative code
    return codes, oracle.e4m3_decode(codes)


def _brute_encode(v):
    """Nearest finite code by exhaustive search, ties to the even code,
    magnitudes above the largest value clamp to it; sign copied."""
    codes, vals = _positive_table()
    a = np.abs(v)
    d = np.abs(a[:, None] - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates prefer the even code
    even = cand & (codes[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    out = codes[pick].astype(np.uint8)
    out = np.where(a >= 448.0, np.uint8(0x7E), out)
    return np.where(np.signbit(v), out | 0x80, out).astype(np.uint8)


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert nan.sum() == 2  # 0x7F and 0xFF
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert np.signbit(got[0x80])  # -0 keeps its sign


def test_decode_closed_forms():
    assert oracle.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert oracle.e4m3_decode(np.array([0x01]))[0] == 2.0**-9
    assert oracle.e4m3_decode(np.array([0x08]))[0] == 2.0**-6
    assert oracle.e4m3_decode(np.array([0x38]))[0] == 1.0


def test_encode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    assert codes.size == 254
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_encode_golden_points():
    rows = []
    for line in open(os.path.join(GOLDEN, "e4m3_points.txt")):
        line = line.split("#")[0].strip()
        if line:
            v, c = line.split()
            rows.append((float(v), int(c, 16)))
    vals = np.array([r[0] for r in rows])
    want = np.array([r[1] for r in rows], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(vals), want)
    assert oracle.e4m3_encode(np.array([np.nan]))[0] == 0x7F
    assert oracle.e4m3_encode(np.array([np.inf]))[0] == 0x7E
    assert oracle.e4m3_encode(np.array([-np.inf]))[0] == 0xFE


def _all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        v = bits.view(np.float32).astype(np.float64)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("shift", [0, 8, -8])
def test_encode_matches_brute_force_on_every_bf16(shift):
    v = _all_bf16_values() * 2.0**shift
    v = v[np.abs(v) < 2.0**12]  # bigger magnitudes all saturate; keep the table small
    np.testing.assert_array_equal(oracle.e4m3_encode(v), _brute_encode(v))


def test_encode_matches_brute_force_on_midpoints():
    _, vals = _positive_table()
    mids = (vals[1:] + vals[:-1]) / 2
    eps = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9)])
    v = np.concatenate([eps, -eps])
    np.testing.assert_array_equal(oracle.e4m3_encode(v), _brute_encode(v))


def test_encode_matches_torch_in_range():
    v = _all_bf16_values()
    v = v[np.abs(v) < 464.0]  # torch's cast does not saturate: NaN beyond 464
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


def test_ue8m0_decode():
    s = np.arange(256)
    got = oracle.ue8m0_decode(s)
    assert np.isnan(got[255])
    np.testing.assert_array_equal(got[:255], [2.0 ** (i - 127) for i in range(255)])
    ref = torch.from_numpy(s.astype(np.uint8)).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    np.testing.assert_array_equal(got[:255], ref[:255])


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000)),
        (np.arange(1, 20000) * 2.0**-140),  # bf16 subnormal neighbourhood
    ]).astype(np.float32)
    # ties: values exactly half way between two bf16 numbers
    base = (rng.integers(0, 2**15, 10000).astype(np.uint32) << 16) | np.uint32(0x8000)
    x = np.concatenate([x, base.view(np.float32)])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


def test_round_bf16_float64_single_rounding():
    # 1 + 2**-8 + 2**-40 lies just above the bf16 midpoint 1 + 2**-8: rounds up,
    # while a float32 first step would land on the midpoint and round to even (1.0).
    x = 1.0 + 2.0**-8 + 2.0**-40
    assert oracle.round_bf16(np.array([x]))[0] == 1.0 + 2.0**-7
    assert oracle.round_bf16(np.array([1.0 + 2.0**-8]))[0] == 1.0
    assert oracle.round_bf16(np.array([1.0 + 3 * 2.0**-8]))[0] == 1.0 + 4 * 2.0**-8
