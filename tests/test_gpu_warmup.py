"""mx_warmup: the registered weight shapes' GEMMs run once on a zero MXFP8
activation (the mxfp8 page's `compile_pinned` / `run_zeros` / `_zeros` over
`shape_representatives`).

* every run's output is exactly zero (zero codes and zero scale bytes times
  finite weights), one output per distinct (n, k) and row count;
* the plans the warm-up keeps serve later calls: a real GEMM on the warmed
  handle equals, bit for bit, the same GEMM on a fresh handle;
* a rejected row count or a short scratch buffer fails before any launch and
  leaves the scratch untouched.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_to_device, handle, quantize_on_gpu

pytestmark = pytest.mark.gpu

SHAPES = [(2048, 5120), (8192, 1536), (5120, 8192), (2048, 5120)]  # the last repeats the first
ROWS = [1, 4, 16, 64]


def _weights(seed):
    return [quantize_on_gpu(synth.block_scaled_bf16(seed + i, synth.TAG_W + i, n, k, -6, 6))
            for i, (n, k) in enumerate(SHAPES)]


def test_warmup_outputs_are_zero():
    import mxfp8_block_scaled_06_gb300 as mx

    h = handle()
    outs = mx.mx_warmup(h, _weights(30), ROWS)
    torch.cuda.synchronize()
    assert mx.mx_device_status(h) == mx.MX_OK
    distinct = sorted(set(SHAPES))
    assert len(outs) == len(distinct) * len(ROWS)
    for i, (n, _) in enumerate(distinct):
        for j, r in enumerate(ROWS):
            o = outs[i * len(ROWS) + j]
            assert o.shape == (r, n)
            assert not torch.any(o.view(torch.int16) != 0), f"({n}, {r}) not all +0"


def test_warmed_plans_serve_later_calls():
    import mxfp8_block_scaled_06_gb300 as mx

    ws = _weights(31)
    warmed = mx.mx_create(0)
    fresh = mx.mx_create(0)
    try:
        mx.mx_warmup(warmed, ws, ROWS)
        for (wq, wsc), m in [(ws[0], 4), (ws[1], 16), (ws[2], 1)]:
            a = bf16_to_device(synth.block_scaled_bf16(32, synth.TAG_A + m, m, wq.shape[1], -4, 4))
            aq, asc = mx.mx_quantize_rows(warmed, a)
            o_w = mx.mx_gemm(warmed, aq, asc, wq, wsc, pdl=True)
            o_f = mx.mx_gemm(fresh, aq, asc, wq, wsc, pdl=True)
            torch.cuda.synchronize()
            assert torch.equal(o_w.view(torch.int16), o_f.view(torch.int16))
        assert mx.mx_device_status(warmed) == mx.MX_OK
    finally:
        warmed.close()
        fresh.close()


@pytest.mark.parametrize("case", ["rows_too_many", "scratch_short"])
def test_rejected_warmup_launches_nothing(case):
    import mxfp8_block_scaled_06_gb300 as mx

    lib, h = mx.load_library(), handle()
    ws = _weights(33)[:2]
    w_arr = (mx.MxWeight * 2)(*[mx.MxWeight(w.data_ptr(), s.data_ptr(), w.shape[0], w.shape[1])
                                for w, s in ws])
    rows = [1, 300] if case == "rows_too_many" else [1, 8]
    r_arr = (ctypes.c_int * 2)(*rows)
    need = lib.mx_warmup_bytes(w_arr, 2, r_arr, 2)
    assert need > 0
    have = need if case == "rows_too_many" else need - 256
    buf = torch.full((need + 512,), 0xA5, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    rc = lib.mx_warmup(h.ptr, w_arr, 2, r_arr, 2, buf.data_ptr() + off, have,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == (mx.MX_ERR_UNSUPPORTED if case == "rows_too_many" else mx.MX_ERR_INVALID_ARG)
    torch.cuda.synchronize()
    assert (buf.cpu().numpy() == 0xA5).all(), "a rejected warm-up wrote its scratch"
    assert mx.mx_device_status(h) == mx.MX_OK
