"""The C-ABI library builds, loads and exports every entry point include/mx.h
declares; host-side logic that needs no GPU (scale-buffer size, status names,
argument checks that fail before touching a device)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import mxfp8_block_scaled_06_gb300 as mx

    return mx.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "mx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for f in ["mx_create", "mx_destroy", "mx_scale_bytes", "mx_quantize_rows", "mx_gemm",
              "mx_gemm_chain", "wo_a_grouped", "mx_device_status", "mx_status_string"]:
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    path = lib._name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [f for f in _declared_functions() if f not in exported]
    assert not missing, missing
    for f in _declared_functions():
        assert hasattr(lib, f)


def test_binding_names_match_header():
    import mxfp8_block_scaled_06_gb300 as mx

    assert sorted(mx.EXPORTS) == _declared_functions()
    for f in ["mx_create", "mx_scale_bytes", "mx_quantize_rows", "mx_gemm", "mx_gemm_chain",
              "wo_a_grouped", "mx_device_status"]:
        assert callable(getattr(mx, f))


@pytest.mark.parametrize("rows,k", [(1, 5120), (4, 512), (8, 1536), (64, 8192), (128, 4096),
                                    (129, 4096), (256, 5120), (3, 96), (0, 128)])
def test_scale_bytes_matches_oracle(lib, rows, k):
    assert lib.mx_scale_bytes(rows, k) == oracle.mx_scale_bytes(rows, k)


def test_scale_bytes_rejects_bad_k(lib):
    assert lib.mx_scale_bytes(4, 100) == 0
    assert lib.mx_scale_bytes(-1, 128) == 0


def test_warmup_bytes_follows_the_documented_layout(lib):
    """Host-only: the zero activation (largest rows*k codes, largest scale
    bytes), then one bf16 output per distinct (n, k) and row count, each
    rounded to 256 bytes. A repeated shape adds nothing."""
    import mxfp8_block_scaled_06_gb300 as mx

    shapes = [(2048, 5120), (8192, 1536), (2048, 5120)]
    ws = (mx.MxWeight * 3)(*[mx.MxWeight(None, None, n, k) for n, k in shapes])
    rows = (ctypes.c_int * 2)(1, 16)
    r256 = lambda v: (v + 255) // 256 * 256
    want = (r256(16 * 5120) + r256(oracle.mx_scale_bytes(16, 5120))
            + sum(r256(r * n * 2) for n in (2048, 8192) for r in (1, 16)))
    assert lib.mx_warmup_bytes(ws, 3, rows, 2) == want
    assert lib.mx_warmup_bytes(ws, 0, rows, 2) == 0
    assert lib.mx_warmup_bytes(ws, 3, rows, 0) == 0
    bad = (ctypes.c_int * 1)(0)
    assert lib.mx_warmup_bytes(ws, 3, bad, 1) == 0


def test_status_strings(lib):
    import mxfp8_block_scaled_06_gb300 as mx

    names = [mx.status_string(c) for c in range(6)]
    assert names == ["MX_OK", "MX_ERR_INVALID_ARG", "MX_ERR_UNSUPPORTED", "MX_ERR_DEVICE",
                     "MX_ERR_CUDA", "MX_ERR_TIMEOUT"]
    assert mx.status_string(99) == "MX_ERR_UNKNOWN"


def test_null_handle_is_rejected_before_any_device_call(lib):
    import mxfp8_block_scaled_06_gb300 as mx

    assert lib.mx_gemm(None, 1, 128, 128, None, None, None, None, None, 0, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_quantize_rows(None, 1, 32, None, 32, None, None, 1, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_gemm_chain(None, 1, None, None, None, 1536, None, None, None, None, None, None,
                             None, None) == mx.MX_ERR_INVALID_ARG
    assert lib.wo_a_grouped(None, 1, None, 0, None, None, 1, None, None, 4, 8, 448, 64, 1024, None,
                            None, None, None, None, 0, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_wait_selftest(None, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_destroy(None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_create(None, 0) == mx.MX_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_a_device_fails_cleanly(lib):
    import mxfp8_block_scaled_06_gb300 as mx

    p = ctypes.c_void_p()
    rc = lib.mx_create(ctypes.byref(p), 0)
    assert rc in (mx.MX_ERR_CUDA, mx.MX_ERR_DEVICE)
    assert p.value is None
    with pytest.raises(mx.MxError):
        mx.mx_create(0)
