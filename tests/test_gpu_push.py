"""The push reduction (every K-split stores the partials of the units another
rank owns straight into that rank's shared memory) against the forms that read
the peers' partials: each output is the same rank-order sum of the same fp32
partials, so the two agree bit for bit, for every split count a cluster can
hold and for row counts that leave ranks without units, split a unit's rows
(M = 3, 5, 13) or give a rank several units. The output is also checked against
the oracle. Plans are read when a handle is created, so each variant gets one."""
import os

import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_gemm_close, handle, operands, quantize_on_gpu

pytestmark = pytest.mark.gpu

ROWS = (1, 2, 3, 4, 5, 8, 13, 16)


def _handle_with(env: dict):
    import mxfp8_block_scaled_06_gb300 as mx

    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        return mx.mx_create(0)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.fixture(scope="module")
def no_push():
    h = _handle_with({"MX_PUSH_ROWS": "0"})
    yield h
    h.close()


def _run(h, aq, asc, wq, wsc):
    import mxfp8_block_scaled_06_gb300 as mx

    out = mx.mx_gemm(h, aq, asc, wq, wsc, pdl=True)
    torch.cuda.synchronize()
    assert mx.mx_device_status(h) == mx.MX_OK
    return out


@pytest.mark.parametrize("n,k", [(2048, 5120), (8192, 1536), (5120, 8192), (384, 640)])
def test_push_equals_peer_reads(no_push, n, k):
    wq, wsc = quantize_on_gpu(synth.block_scaled_bf16(60, synth.TAG_W, n, k, -6, 6))
    for m in ROWS:
        aq, asc = quantize_on_gpu(synth.block_scaled_bf16(60 + m, synth.TAG_A, m, k, -4, 4))
        got = _run(handle(), aq, asc, wq, wsc)
        ref = _run(no_push, aq, asc, wq, wsc)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (n, k, m)


@pytest.mark.parametrize("splits", range(1, 9))
def test_push_every_split_count(splits):
    """N = 256, K = 1024 (8 chunks): 1 to 8 ranks per cluster, push and not."""
    n, k = 256, 1024
    spec = f"{n}x{k}:{splits}"
    hp = _handle_with({"MX_PLAN_AT": spec})
    hn = _handle_with({"MX_PLAN_AT": spec, "MX_PUSH_ROWS": "0"})
    try:
        wbits, _, (rw, rsw) = operands(61, synth.TAG_W, n, k)
        wq, wsc = quantize_on_gpu(wbits)
        for m in ROWS:
            abits, _, (ra, rsa) = operands(61 + m, synth.TAG_A, m, k, -4, 4)
            aq, asc = quantize_on_gpu(abits)
            got = _run(hp, aq, asc, wq, wsc)
            ref = _run(hn, aq, asc, wq, wsc)
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (splits, m)
            assert_gemm_close(got, oracle.mx_gemm(ra, rsa, rw, rsw), f"splits={splits} m={m}")
    finally:
        hp.close()
        hn.close()
