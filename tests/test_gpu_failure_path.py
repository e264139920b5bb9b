"""The failure path of the kernels' bounded waits, taken on purpose on the GPU.

Every pipeline wait in the library (TMA landings, MMA completion, cluster
partners) is an mbarrier wait with a one-second limit; on expiry the kernel sets
a bit in the handle's status word and returns instead of spinning forever.
``mx_wait_selftest`` runs that same wait against a barrier nothing completes --
no fault, no bad address, just a flag that is never set -- so this test checks
that the wait ends, that the host reads MX_ERR_TIMEOUT, that reading clears it,
and that the context still computes correctly afterwards."""
import time

import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_gemm_close, handle, operands, quantize_on_gpu

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_survives():
    import mxfp8_block_scaled_06_gb300 as mx

    h = handle()
    assert mx.mx_device_status(h) == mx.MX_OK  # read-and-clear anything earlier
    t0 = time.perf_counter()
    mx.mx_wait_selftest(h)
    status = mx.mx_device_status(h)  # synchronizes: the kernel has returned
    waited = time.perf_counter() - t0
    assert status == mx.MX_ERR_TIMEOUT
    assert 0.9 <= waited < 30.0
    assert mx.mx_device_status(h) == mx.MX_OK  # the read cleared it

    # the same context still runs the GEMM correctly, and reports no error
    a_bits, _, (ra, rsa) = operands(90, synth.TAG_A, 4, 512)
    w_bits, _, (rw, rsw) = operands(90, synth.TAG_W, 256, 512)
    aq, asc = quantize_on_gpu(a_bits)
    wq, wsc = quantize_on_gpu(w_bits)
    out = mx.mx_gemm(h, aq, asc, wq, wsc)
    torch.cuda.synchronize()
    assert_gemm_close(out, oracle.mx_gemm(ra, rsa, rw, rsw), "GEMM after an expired wait")
    assert mx.mx_device_status(h) == mx.MX_OK
