"""GPU parity of the split-K path (batch_invariant=False): pass 1 over segment 0 and
the affine maps of the middle segments, the fp32 state fix-up, pass 2 over the rest.

The library picks the number of segments P itself (P = 1 whenever splitting would
not pay); the testing aid gdn_testing_force_splits forces P so that every segment layout is exercised on
small problems, including segments with no chunk at all.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import compare

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
    out, st = _run(p)
    compare(p, out, st)
    out2, st2 = _run(p)
    assert torch.equal(out, out2) and torch.equal(st, st2)
