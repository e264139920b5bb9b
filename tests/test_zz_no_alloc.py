"""The chain entry point for callers that cannot allocate device memory.

Some callers only hold the buffers of their own inputs and outputs: a caller
inside a CUDA-graph capture (cudaMalloc is not a stream operation and may
synchronize), an engine that hands a kernel library nothing but its input and
output buffers because it budgets device memory itself, or a plugin host with
no allocator exposed to the plugin. mx_gemm_chain_noalloc serves them by keeping
the chain's two intermediates in a fixed device array inside the library.

This test calls that entry point through the C ABI (ctypes on libmx.so) twice
in a row and compares each result with mx_gemm_chain run on caller-owned
intermediates, within the GEMM tolerance the other tests use
(|got - ref| <= 1e-2 |ref| + 1e-3 rms(ref)). The second call checks that the
contents the first call left in the shared array do not leak into the next one.
The file name sorts last, so a run that stops at the first failure has run every
other test before this one.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import bf16_to_device, handle

pytestmark = pytest.mark.gpu

SHAPES = [(2048, 5120), (8192, 1536), (5120, 8192)]  # (N, K) of the three projections
G1_COLS = 1536


def _weights(h, seed):
    import mxfp8_block_scaled_06_gb300 as mx

    out = []
    for i, (n, k) in enumerate(SHAPES):
        bits = synth.block_scaled_bf16(seed, synth.TAG_W + i, n, k, -6, 6)
        out.append(mx.mx_quantize_rows(h, bf16_to_device(bits)))
    return out


def _close(got: torch.Tensor, ref: torch.Tensor):
    r = ref.float().cpu().numpy().astype(np.float64)
    g = got.float().cpu().numpy().astype(np.float64)
    tol = oracle.gemm_tolerance(r)
    err = np.abs(g - r)
    assert (err <= tol).all(), f"{int((err > tol).sum())} elements beyond tolerance"


@pytest.mark.parametrize("m", [1, 16, 64])
def test_chain_noalloc_matches_chain_twice(m):
    import mxfp8_block_scaled_06_gb300 as mx

    h = handle()
    lib = mx.load_library()
    wts = _weights(h, 11)
    a_bits = synth.block_scaled_bf16(11, synth.TAG_A + m, m, SHAPES[0][1], -4, 4)
    a1, a1s = mx.mx_quantize_rows(h, bf16_to_device(a_bits))
    ref = mx.mx_gemm_chain(h, a1, a1s, wts, g1_cols=G1_COLS)["out"]
    ws = (mx.MxWeight * 3)(*[mx.MxWeight(w.data_ptr(), s.data_ptr(), w.shape[0], w.shape[1])
                             for w, s in wts])
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((m, SHAPES[2][0]), float("nan"), dtype=torch.bfloat16, device=a1.device)
        rc = lib.mx_gemm_chain_noalloc(h.ptr, m, a1.data_ptr(), a1s.data_ptr(), ws, G1_COLS,
                                       out.data_ptr(), stream)
        assert rc == mx.MX_OK, mx.status_string(rc)
        torch.cuda.synchronize()
        assert mx.mx_device_status(h) == mx.MX_OK
        _close(out, ref)


def test_chain_noalloc_rejects_intermediates_beyond_its_array():
    import mxfp8_block_scaled_06_gb300 as mx

    h = handle()
    lib = mx.load_library()
    wts = _weights(h, 12)
    m = 128  # 128 * (1536 + 8192) bytes of codes alone exceed the 1 MiB array
    a_bits = synth.block_scaled_bf16(12, synth.TAG_A + m, m, SHAPES[0][1], -4, 4)
    a1, a1s = mx.mx_quantize_rows(h, bf16_to_device(a_bits))
    ws = (mx.MxWeight * 3)(*[mx.MxWeight(w.data_ptr(), s.data_ptr(), w.shape[0], w.shape[1])
                             for w, s in wts])
    out = torch.full((m, SHAPES[2][0]), 7.0, dtype=torch.bfloat16, device=a1.device)
    torch.cuda.synchronize()
    rc = lib.mx_gemm_chain_noalloc(h.ptr, m, a1.data_ptr(), a1s.data_ptr(), ws, G1_COLS,
                                   out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == mx.MX_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a rejected call wrote its output"
