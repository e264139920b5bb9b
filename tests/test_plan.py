"""Plan queries (host only, no GPU): the reduction form each launch takes, the
push exchange's receive area in the shared-memory budget, and the chain's
co-residency rule, checked as an invariant recomputed here from the plans the
library returns."""
import itertools
import math

import pytest

import mxfp8_block_scaled_06_gb300 as mx

SM_COUNT, SMEM_PER_SM, RESERVED, MAX_SMEM = 152, 233472, 1024, 232448
CHAIN = [(2048, 5120), (8192, 1536), (5120, 8192)]


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()


def _area(m, s, compact):
    """The receive area from the documented geometry: units of g rows (4, or m
    when m < 3) by one 32-column block, U = 4 ceil(m / g), a slot of
    ceil(U / s) units x 32 lanes x g floats per rank (per peer when compact)."""
    g = m if m < 3 else 4
    units = 4 * math.ceil(m / g)
    slot = math.ceil(units / s) * 128 * g
    return (s - 1 if compact else s) * slot


def test_decode_projection_takes_push_up_to_16_rows():
    for m in range(1, 257):
        p = mx.mx_plan_gemm(m, 2048, 5120)
        if m <= 16:
            assert p["reduction"] == mx.MX_REDUCE_PUSH and p["splits"] == 8, (m, p)
        else:
            rows = p["splits"] <= 4 and m >= 8 * p["splits"]
            assert p["reduction"] == (mx.MX_REDUCE_ROWS if rows else mx.MX_REDUCE_ITEMS), (m, p)
        assert p["mtile"] == (m + 15) // 16 * 16


@pytest.mark.parametrize("n,k", [(2048, 5120), (8192, 1536), (5120, 8192), (5120, 4096), (384, 640),
                                 (256, 2048)])
@pytest.mark.parametrize("fused,norm", [(False, False), (True, False), (True, True)])
def test_receive_area_is_in_the_budget(n, k, fused, norm):
    """Same ring and splits with and without push; the difference in shared
    memory is the receive area (plus under 128 bytes of alignment); a push
    plan never exceeds the per-CTA maximum. With the norm (the chain's G2) the
    prologue's row sums and norm weight share the budget."""
    for m in range(1, 17):
        none = mx.mx_plan_gemm(m, n, k, fused=fused, norm=norm, push=mx.MX_PUSH_NONE)
        for push, red, compact in ((mx.MX_PUSH_FULL, mx.MX_REDUCE_PUSH, False),
                                   (mx.MX_PUSH_COMPACT, mx.MX_REDUCE_PUSH_COMPACT, True)):
            p = mx.mx_plan_gemm(m, n, k, fused=fused, norm=norm, push=push)
            assert (p["splits"], p["stages"], p["tmem_cols"]) == (none["splits"], none["stages"], none["tmem_cols"])
            if p["reduction"] != red:  # push left out: it did not fit
                assert none["smem"] + _area(m, p["splits"], compact) > MAX_SMEM or none["smem"] > MAX_SMEM
                assert p == none
                continue
            extra = p["smem"] - none["smem"]
            assert 0 <= extra - _area(m, p["splits"], compact) < 128, (m, p, none)
            assert p["smem"] <= MAX_SMEM


def _fits(prev, prev_n, nxt):
    k = math.ceil(prev_n // 128 * prev["splits"] / SM_COUNT)
    return (k * (prev["smem"] + RESERVED) + nxt["smem"] + RESERVED <= SMEM_PER_SM
            and k * prev["tmem_cols"] + nxt["tmem_cols"] <= 512)


@pytest.mark.parametrize("m", list(range(1, 17)) + [24, 32, 64])
def test_chain_keeps_every_neighbour_pair_resident(m):
    """For each pair of neighbours (G3 before the next step's G1) that fits an
    SM without receive areas, the chosen push forms fit too."""
    modes = mx.mx_plan_chain_push(m, CHAIN)
    assert all(x in (mx.MX_PUSH_NONE, mx.MX_PUSH_COMPACT, mx.MX_PUSH_FULL) for x in modes)
    # the plain chain's projections as planned (G2 and G3 without the norm)
    plans = [mx.mx_plan_gemm(m, n, k, push=modes[i]) for i, (n, k) in enumerate(CHAIN)]
    bare = [mx.mx_plan_gemm(m, n, k, push=mx.MX_PUSH_NONE) for n, k in CHAIN]
    for i in range(3):
        p = (i + 2) % 3
        if _fits(bare[p], CHAIN[p][0], bare[i]):
            assert _fits(plans[p], CHAIN[p][0], plans[i]), (m, modes, p, i)
    for i in range(3):
        if m > 16:
            assert modes[i] == mx.MX_PUSH_NONE


def test_chain_forms_at_the_decode_row_counts():
    """The forms the design notes report for the decode chain on a GB300."""
    assert mx.mx_plan_chain_push(1, CHAIN) == [mx.MX_PUSH_FULL] * 3
    assert mx.mx_plan_chain_push(4, CHAIN) == [mx.MX_PUSH_FULL, mx.MX_PUSH_FULL, mx.MX_PUSH_COMPACT]
    assert mx.mx_plan_chain_push(16, CHAIN) == [mx.MX_PUSH_FULL, mx.MX_PUSH_NONE, mx.MX_PUSH_NONE]
    assert mx.mx_plan_chain_push(64, CHAIN) == [mx.MX_PUSH_NONE] * 3


def test_chain_with_room_to_spare_keeps_every_push():
    for m, norm in itertools.product((1, 4, 8, 16), (False, True)):
        assert mx.mx_plan_chain_push(m, CHAIN, norm=norm, smem_per_sm=10 * SMEM_PER_SM) == [mx.MX_PUSH_FULL] * 3


def test_plan_queries_reject_bad_arguments():
    for args in ((0, 2048, 5120), (257, 2048, 5120), (1, 2000, 5120), (1, 2048, 5000)):
        with pytest.raises(mx.MxError):
            mx.mx_plan_gemm(*args)
    with pytest.raises(mx.MxError):
        mx.mx_plan_gemm(1, 2048, 5120, norm=True)  # the norm only with in-kernel quantization
    with pytest.raises(mx.MxError):
        mx.mx_plan_gemm(1, 2048, 5120, sm_count=0)
    with pytest.raises(mx.MxError):
        mx.mx_plan_chain_push(1, [(2048, 5120), (8192, 1536), (5120, 4096)])  # G3's k != G2's n
    with pytest.raises(mx.MxError):
        mx.mx_plan_chain_push(1, [(1024, 5120), (8192, 1536), (5120, 8192)])  # G2's k > G1's n
