"""The split-K planner and unit order, on the host (the library's plan query, no GPU).

A split call with P segments per sequence runs pass 1 (segment 0 and the maps M_p, N_p of
the middle segments), a fix-up, then pass 2 (segments 1..P-1 from their fixed-up
states): the split-K partition of "flashinfer.cudnn.cudnn_chunk_gated_delta_rule"
(Parameters, batch_invariant) read as the "T precompute -> MN precompute -> state fixup
-> CP prefill" sequence of "flashinfer.gdn_prefill" (Cake GDN CP).  Whatever order a plan
picks, each pass must walk every unit it owns exactly once; the per-CTA walk lengths
give the plan's time in whole-sequence walks.
"""
import random
from collections import Counter
from fractions import Fraction

import pytest

import gated_delta_rule_24_gb300 as gdn


def seg_len(plan, seg):
    return Fraction(plan["num"][seg + 1] - plan["num"][seg], plan["den"])


def check_plan(N, H, T, sms):
    """Coverage of both passes, and the time of each pass (the longest per-CTA sum of
    segment fractions) for equal-length sequences."""
    plan = gdn.testing_split_plan(N, H, T, sms)
    P, U = plan["P"], N * H
    if P == 1:
        return plan, None
    assert plan["num"][0] == 0 and plan["num"][P] == plan["den"]
    assert all(a < b for a, b in zip(plan["num"], plan["num"][1:]))
    times = []
    for ps, kinds in ((0, 2 * P - 3), (1, P - 1)):
        grid = plan["grid"][ps]
        assert 0 < grid <= sms
        units = plan["units"][ps]
        real = [x for x in units if x != (-1, -1)]
        assert Counter(real) == Counter((nh, k) for nh in range(U) for k in range(kinds)), (ps, plan["P"])
        load = Counter()
        for u, (nh, k) in enumerate(units):
            if nh < 0:
                continue
            seg = (k if k <= P - 2 else k - (P - 2)) if ps == 0 else k + 1
            load[u % grid] += seg_len(plan, seg)
        times.append(max(load.values()))
    return plan, times


def test_workload4_takes_the_four_segment_plan():
    """2 x 65536 tokens, 32 heads, 152 SMs: segments of 3, 1, 1, 2 sevenths; pass 1 takes
    3/7 (64 CTAs walk segment 0, 88 CTAs walk the 256 one-seventh maps, three at most),
    pass 2 takes 2/7 (segments 1 and 2 on one CTA, segment 3 on another)."""
    plan, times = check_plan(2, 32, 2 * 65536, 152)
    assert plan["P"] == 4 and plan["num"] == [0, 3, 4, 5, 7] and plan["den"] == 7
    assert plan["grid"] == [152, 128]
    assert times == [Fraction(3, 7), Fraction(2, 7)]


def test_skewed_three_segment_plan():
    """64 units of 32 chunks: too short for the four-segment plan (segments of 8 chunks
    or more), so P = 3 with 1/2, 1/4, 1/4: pass 1 takes 1/2, pass 2 1/4."""
    plan, times = check_plan(4, 16, 4 * 2048, 152)
    assert plan["P"] == 3 and plan["num"] == [0, 2, 3, 4] and plan["den"] == 4
    assert times == [Fraction(1, 2), Fraction(1, 4)]


def test_uniform_and_unsplit_plans():
    plan, times = check_plan(1, 2, 16384, 152)  # two units: eight uniform segments
    assert plan["P"] == 8 and plan["den"] == 8 and times == [Fraction(1, 8), Fraction(1, 8)]
    plan, _ = check_plan(16, 32, 16 * 4096, 152)  # 512 units fill every SM
    assert plan["P"] == 1


def test_forced_uniform_plans(force_split):
    for P in range(2, 9):
        force_split(P)
        plan, times = check_plan(3, 4, 3 * 1000, 152)
        assert plan["P"] == P and plan["num"] == list(range(P + 1))
        U = 3 * 4  # units of 1/P, round-robin over min(units, SMs) CTAs
        assert times == [Fraction(-(-U * (2 * P - 3) // 152), P), Fraction(-(-U * (P - 1) // 152), P)]


@pytest.mark.parametrize("seed", range(4))
def test_random_shapes_cover_every_unit(seed):
    """Any shape the planner meets: both passes walk every unit once, and whatever plan it
    takes is modelled at least a fifth faster than the unsplit walk."""
    rng = random.Random(seed)
    for _ in range(40):
        N = rng.randint(1, 8)
        H = rng.choice([1, 2, 4, 8, 16, 32, 64])
        T = N * rng.choice([64, 1000, 4096, 16384, 65536])
        sms = rng.choice([16, 100, 148, 152])
        plan, times = check_plan(N, H, T, sms)
        if plan["P"] > 1:
            waves = -(-N * H // sms)
            assert sum(times) <= Fraction(4, 5) * waves, (N, H, T, sms, plan["P"], times)


def test_plan_query_rejects_bad_sizes():
    with pytest.raises(gdn.GdnError):
        gdn.testing_split_plan(0, 4, 100, 152)
    with pytest.raises(gdn.GdnError):
        gdn.testing_split_plan(2, 4, 100, 0)
