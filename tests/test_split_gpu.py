"""GPU parity of the split-K path (batch_invariant=False): pass 1 over segment 0 and
the affine maps of the middle segments, the fp32 state fix-up, pass 2 over the rest.

The library picks the number of segments P itself (P = 1 whenever splitting would
not pay); the testing aid gdn_testing_force_splits forces P so that every segment layout is exercised on
small problems, including segments with no chunk at all.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import compare, rel_l2, run_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_rule_24_gb300 import build
    build.build()
    import oracle
    oracle.build()
    gdn.gdn_init(0)
    yield
    assert gdn.device_status() == 0


def _run(p, **kw):
    out, st = gdn.run_problem(p, device=DEV, **kw)
    torch.cuda.synchronize()
    return out, st


LENGTHS = [1, 63, 64, 65, 700, 0, 1500, 129]


@pytest.mark.parametrize("P", [2, 3, 4, 5, 8])
def test_forced_split_matches_oracle(force_split, P):
    force_split(str(P))
    p = W.make_problem(LENGTHS, 2, 4, gates="mamba", init="fp32", init_std=0.05, seed=80 + P,
                       batch_invariant=False)
    out, st = _run(p)
    compare(p, out, st)


def test_forced_split_bf16_pools_and_indices(force_split):
    """bf16 state pools addressed through int32 state_indices, int64 cu_seqlens."""
    force_split("4")
    lengths = [int(x) for x in np.random.default_rng(7).integers(200, 900, size=24)]
    p = W.make_problem(lengths, 8, 16, gates="uniform", init="bf16", init_std=0.05,
                       state_dtype=torch.bfloat16, pool_slots=64, cu_dtype=torch.int64,
                       seed=90, batch_invariant=False)
    out, st = _run(p)
    compare(p, out, st)


def test_split_is_deterministic(force_split):
    force_split("3")
    p = W.make_problem([900, 333], 2, 2, gates="mamba", init="fp32", seed=95, batch_invariant=False)
    o1, s1 = _run(p)
    o2, s2 = _run(p)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_split_without_state_buffers(force_split):
    """No initial state and no output state: the workspace still carries S_p."""
    force_split("5")
    p = W.make_problem([1000], 1, 2, init=None, seed=97, batch_invariant=False)
    out, _ = _run(p)
    compare(p, out, None)


def test_auto_split_single_long_sequence(force_split):
    """One 16384-token sequence, 2 heads: the unsplit grid would use 2 SMs, so the
    library splits it on its own."""
    force_split(0)
    p = W.make_problem([16384], 1, 2, gates="mamba", init="fp32", init_std=0.05, seed=99,
                       batch_invariant=False)
    out, st = _run(p)
    compare(p, out, st)


def test_split_bad_inputs_set_error_bits(force_split):
    force_split("3")
    p = W.make_problem([400, 400, 400], 1, 2, seed=101, batch_invariant=False)
    p.cu_seqlens = torch.tensor([0, 400, 300, 1200], dtype=torch.int32)
    _run(p)
    assert gdn.device_status() & gdn.binding.DEVERR_CU_SEQLENS
    p = W.make_problem([300], 1, 1, seed=102, batch_invariant=False)
    out, st = _run(p)
    compare(p, out, st)
    assert gdn.device_status() == 0


@pytest.mark.parametrize("forced", [None, "4"])
def test_workload4_split(force_split, forced):
    """2 x 65536 tokens with batch_invariant=False: sampled units match the oracle."""
    if forced is None:
        force_split(0)
    else:
        force_split(forced)
    p = W.make_workload(4, batch_invariant=False)
    out, st = _run(p)
    compare(p, out, st, units=[(0, 0), (0, 7), (0, 16), (0, 31), (1, 1), (1, 14), (1, 21), (1, 30)])
    assert torch.isfinite(out.float()).all()


def test_planner_skewed_split_matches_oracle(force_split):
    """64 (sequence, head) units of 32 chunks on 152 SMs: the planner splits every
    sequence into segments of 1/2, 1/4 and 1/4 of its chunks (pass 1 pairs the map walks
    on the CTAs that take two units); every unit matches the oracle, and the result is
    deterministic."""
    force_split(0)
    p = W.make_problem([2048] * 4, 8, 16, gates="mamba", init="fp32", init_std=0.05, seed=91,
                       batch_invariant=False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = gdn.testing_split_plan(p.N, p.H, p.T, sms)
    if sms == 152:
        assert plan["P"] == 3 and plan["num"] == [0, 2, 3, 4]
    out, st = _run(p)
    compare(p, out, st)
    out2, st2 = _run(p)
    assert torch.equal(out, out2) and torch.equal(st, st2)


def test_planner_four_segment_split_matches_oracle(force_split):
    """64 (sequence, head) units of 64 chunks on 152 SMs: the planner splits every sequence
    into segments of 3, 1, 1 and 2 sevenths (pass 1: segment 0 on 64 CTAs, the 256 maps
    three to a CTA on the other 88, with idle indices between; pass 2: segments 1 and 2
    on one CTA, segment 3 on another); every unit matches the oracle, and the result is
    deterministic."""
    force_split(0)
    p = W.make_problem([4096] * 4, 8, 16, gates="mamba", init="fp32", init_std=0.05, seed=92,
                       batch_invariant=False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = gdn.testing_split_plan(p.N, p.H, p.T, sms)
    if sms == 152:
        assert plan["P"] == 4 and plan["num"] == [0, 3, 4, 5, 7] and plan["grid"] == [152, 128]
    out, st = _run(p)
    compare(p, out, st)
    out2, st2 = _run(p)
    assert torch.equal(out, out2) and torch.equal(st, st2)


def _tail_state(p, n, begin):
    """Oracle final state of sequence n over its tokens from row ``begin`` on, from a zero
    state: what the state would be if everything before ``begin`` were forgotten."""
    b, e = int(p.cu_seqlens[n]), int(p.cu_seqlens[n + 1])
    rows = slice(begin, e)
    sub = dataclasses.replace(p, q=p.q[rows], k=p.k[rows], v=p.v[rows], g=p.g[rows], beta=p.beta[rows],
                              initial_state=None, state_indices=None,
                              cu_seqlens=torch.tensor([0, e - begin], dtype=p.cu_seqlens.dtype))
    return run_oracle(sub)[1][0]


@pytest.mark.parametrize("P", [2, 3, 4, 8])
def test_forced_split_with_slow_decay(P, force_split):
    """Gates close to one (log g ~ U(-0.004, 0)): a segment's map M_p stays far from zero,
    so the fix-up's S_p M_p term carries real weight (with faster decays it underflows
    and any M_p would pass).  The input is checked for that first: the final state of the
    long sequence differs from the one its last segment alone would leave."""
    force_split(P)
    p = W.make_problem([3000, 1, 777, 2048], 2, 4, gates="slow", init="fp32", init_std=0.05, seed=210 + P,
                       batch_invariant=False)
    o_ref, s_ref = run_oracle(p)
    chunks = (3000 + 63) // 64
    last_begin = (chunks * (P - 1) // P) * 64  # first row of the last segment of sequence 0
    forgot = _tail_state(p, 0, last_begin)
    assert rel_l2(forgot, s_ref[0]) > 0.05
    out, st = _run(p)
    compare(p, out, st, o_ref=o_ref, s_ref=s_ref)


def test_planner_splits_with_slow_decay(force_split):
    """The planner's own plans (the skewed three-segment one and the four-segment one) on
    slowly decaying gates, where the segment maps matter."""
    force_split(0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for lens, hqk, hv in (([2048] * 4, 8, 16), ([4096] * 4, 8, 16)):
        p = W.make_problem(lens, hqk, hv, gates="slow", init="fp32", init_std=0.05, seed=230 + len(lens),
                           batch_invariant=False)
        plan = gdn.testing_split_plan(p.N, p.H, p.T, sms)
        assert plan["P"] > 1
        o_ref, s_ref = run_oracle(p)
        num, den = plan["num"], plan["den"]
        chunks = lens[0] // 64
        forgot = _tail_state(p, 0, (chunks * num[-2] // den) * 64)
        assert rel_l2(forgot, s_ref[0]) > 0.05
        out, st = _run(p)
        compare(p, out, st, o_ref=o_ref, s_ref=s_ref)
