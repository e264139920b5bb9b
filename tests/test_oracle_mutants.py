"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a single oracle function -- a wrong constant, a
dropped term, a wrong sign or index, a transposed or misplaced operand -- by
editing that function's source text and installing the edited copy in the oracle
module (on the CPU, for this test only). The pins of ``test_oracle_mx`` and
``test_oracle_codec`` then run against the mutated oracle, and at least one of
them has to fail. A mutant that every pin accepts would mark a hole in the pins.
"""
import inspect
import textwrap

import pytest

import oracle
import test_oracle_codec
import test_oracle_mx

# (function, [(old text, new text), ...], what the mistake is)
MUTANTS = [
    ("mx_quantize", [("(ex - 1) - 8", "(ex - 1) - 7")], "scale exponent floor(log2 amax) - 7"),
    ("mx_quantize", [("np.clip(e, -127, 127)", "np.clip(e, -126, 127)")], "exponent clamp one binade short"),
    ("mx_quantize", [("e + 127, SCALE_NAN", "e + 128, SCALE_NAN")], "scale byte bias 128"),
    ("mx_quantize", [("codes = np.where(finite[..., None], codes, E4M3_NAN)", "codes = np.where(True, codes, 0)")],
     "non-finite blocks not marked NaN"),
    ("e4m3_encode", [("np.rint(a / quantum)", "np.floor(a / quantum + 0.5)")], "ties rounded away from zero"),
    ("e4m3_encode", [("np.minimum(val, E4M3_MAX)", "val")], "no saturation at 448"),
    ("e4m3_encode", [("ex - 1, -6), -6)", "ex - 1, -7), -7)")], "subnormal quantum 2**-10"),
    ("e4m3_encode", [("code = np.where(neg, code | 0x80, code)", "code = code")], "sign dropped"),
    ("e4m3_decode", [("m * 2.0**-9", "m * 2.0**-10")], "subnormal values halved"),
    ("e4m3_decode", [("np.exp2(e - 7.0)", "np.exp2(e - 8.0)")], "exponent bias 8"),
    ("ue8m0_decode", [("s - 127.0", "s - 128.0")], "scale bias 128"),
    ("mx_dequantize", [("ue8m0_decode(sbytes)[..., None]", "ue8m0_decode(sbytes)[:, ::-1][..., None]")],
     "scale of the wrong K block"),
    ("swizzled_offset", [("(np.asarray(r) % 32) * 16 + ((np.asarray(r) % 128) // 32) * 4",
                          "(np.asarray(r) % 128) * 4")], "128x4 tile without the 32-row interleave"),
    ("swizzled_offset", [("(np.asarray(r) % 32) * 16 + ((np.asarray(r) % 128) // 32) * 4",
                          "(np.asarray(r) % 32) * 4 + ((np.asarray(r) % 128) // 32) * 128")],
     "32-row interleave transposed"),
    ("swizzled_offset", [("(np.asarray(r) // 128) * (cpad // 4) + np.asarray(c) // 4",
                          "(np.asarray(c) // 4) * (cpad // 4) + np.asarray(r) // 128")], "tiles in column order"),
    ("mx_scale_bytes", [("ceil_to(k // SF_VEC, 4)", "k // SF_VEC")], "scale columns not padded to 4"),
    ("round_bf16", [("np.rint(x / quantum)", "np.trunc(x / quantum)")], "bf16 by truncation"),
    ("round_bf16", [("- 8, -133)", "- 7, -133)")], "bf16 with 7 significant bits"),
    ("mx_gemm", [("mx_dequantize(a_codes, a_sbytes) @ mx_dequantize(w_codes, w_sbytes).T",
                  "mx_dequantize(a_codes, a_sbytes)[:, :-32] @ mx_dequantize(w_codes, w_sbytes)[:, :-32].T")],
     "last K block dropped"),
    ("mx_gemm", [("mx_dequantize(w_codes, w_sbytes).T", "e4m3_decode(w_codes).T")], "weight scales ignored"),
    ("chain", [("mx_quantize(b1[:, :g1_cols])", "mx_quantize(b1[:, -g1_cols:])")], "G2 fed G1's last columns"),
    ("chain", [("mx_quantize(b1[:, :g1_cols])", "mx_quantize(out1[:, :g1_cols])")], "G1 output not rounded to bf16"),
    ("chain", [("a3, a3s = mx_quantize(b2)", "a3, a3s = mx_quantize(out2)")], "G2 output not rounded to bf16"),
    ("rope_rotate_inverse", [("a2 = (a * c) + (b * s)", "a2 = (a * c) - (b * s)"),
                             ("b2 = (b * c) - (a * s)", "b2 = (b * c) + (a * s)")], "forward rotation"),
    ("rope_rotate_inverse", [("a, b = xr[..., 0::2], xr[..., 1::2]",
                              "a, b = xr[..., :xr.shape[-1] // 2], xr[..., xr.shape[-1] // 2:]")],
     "rotate-half pairs instead of adjacent pairs"),
    ("wo_a_activation", [("act[..., d_nope:d_nope + d_rope] = rope_rotate_inverse(x[..., d_nope:d_nope + d_rope]",
                          "act[..., :d_rope] = rope_rotate_inverse(x[..., :d_rope]")], "rotation on the nope dims"),
    ("wo_a_activation", [("sin = rows[:, None, half:2 * half]", "sin = -rows[:, None, half:2 * half]")],
     "sine sign flipped"),
    ("wo_a_grouped", [("mx_gemm(cq, cs, w_codes[rows], w_sbytes[rows])",
                       "mx_gemm(cq, cs, w_codes[:o_lora_rank], w_sbytes[:o_lora_rank])")],
     "every group contracted with group 0's weights"),
    ("wo_a_grouped", [("zb = round_bf16(z)", "zb = z")], "z not rounded to bf16 before requantization"),
    ("rms_norm", [("np.mean(x * x", "np.sum(x * x")], "sum of squares instead of the mean"),
    ("rms_norm", [("np.sqrt(ms + eps)", "(np.sqrt(ms) + eps)")], "epsilon outside the square root"),
    ("split_qkv_and_norm", [("rms_norm(out1_bf16[:, :q_cols], norm_weight, eps)",
                             "rms_norm(out1_bf16, np.r_[norm_weight, np.ones(out1_bf16.shape[1] - q_cols)], "
                             "eps)[:, :q_cols]")], "norm taken over the whole G1 row"),
    ("split_qkv_and_norm", [("y = round_bf16(rms_norm(", "y = (rms_norm(")], "normalized row not rounded to bf16"),
    ("chain_norm", [("sp = split_qkv_and_norm(b1,", "sp = split_qkv_and_norm(out1,")],
     "norm applied to G1's unrounded output"),
    ("chain_norm", [("out2 = mx_gemm(sp[\"q\"], sp[\"qs\"], w2, s2)",
                     "out2 = mx_gemm(*mx_quantize(b1[:, :g1_cols]), w2, s2)")], "norm skipped"),
    ("gemm_tolerance", [("1e-3 * rms", "1e-3 * np.abs(ref)")], "tolerance without the rms floor"),
    ("mx_quantize", [("amax = np.max(np.abs(np.where(np.isfinite(blk), blk, 0.0)), axis=-1)",
                      "amax = np.max(np.where(np.isfinite(blk), blk, 0.0), axis=-1)")], "amax without the magnitude"),
    ("wo_a_grouped", [("act[:, g * heads_per_group:(g + 1) * heads_per_group, :]", "act[:, g::n_groups, :]")],
     "groups take every n_groups-th head"),
    ("wo_a_activation", [("[np.asarray(positions, dtype=np.int64)]", "[np.asarray(positions, dtype=np.int64) + 1]")],
     "cache row of the next position"),
    ("wo_a_activation", [("cos = rows[:, None, :half]", "cos = rows[:, None, half:2 * half]"),
                         ("sin = rows[:, None, half:2 * half]", "sin = rows[:, None, :half]")],
     "cos and sin halves of the cache swapped"),
    ("unswizzle_scales", [("[swizzled_offset(rr, cc, n_cols)]", "[swizzled_offset(rr, cc, n_cols) ^ 4]")],
     "unswizzle reads the neighbouring 32-row group"),
]


def _pins():
    """Every pin of the two oracle test modules, parametrized cases expanded."""
    out = []
    for mod in (test_oracle_codec, test_oracle_mx):
        for name, fn in vars(mod).items():
            if not (name.startswith("test_") and callable(fn)):
                continue
            cases = [{}]
            for mark in getattr(fn, "pytestmark", []):
                if mark.name != "parametrize":
                    continue
                names = [s.strip() for s in mark.args[0].split(",")]
                vals = [v if len(names) > 1 else (v,) for v in mark.args[1]]
                cases = [dict(c, **dict(zip(names, v))) for c in cases for v in vals]
            out += [(f"{mod.__name__}.{name}{sorted(c.items()) if c else ''}", fn, c) for c in cases]
    return out


PINS = _pins()


def _install(monkeypatch, fname, edits):
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fname)))
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor not unique in {fname}: {old!r}"
        src = src.replace(old, new)
    ns = dict(vars(oracle))
    exec(compile(src, f"<mutant of oracle.{fname}>", "exec"), ns)
    monkeypatch.setattr(oracle, fname, ns[fname])


@pytest.mark.parametrize("fname,edits,what", MUTANTS, ids=[m[2] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(monkeypatch, fname, edits, what):
    _install(monkeypatch, fname, edits)
    for label, fn, kwargs in PINS:
        try:
            fn(**kwargs)
        except Exception:  # an assertion, or the mistake breaking a shape
            return
    pytest.fail(f"no pin fails with the planted mistake '{what}' in oracle.{fname}")


def test_pins_pass_on_the_oracle_as_written():
    assert len(PINS) >= 40
    for label, fn, kwargs in PINS:
        fn(**kwargs)
