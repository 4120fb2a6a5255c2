"""GPU parity of the mid-sequence f32 state checkpoints of gdn_chunk_prefill_checkpointed:
checkpoint m of a sequence is the state after its first (m + 1) * every * 64 tokens,
which the oracle gives as the final state of that prefix."""
import dataclasses

import numpy as np
import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import compare, rel_l2, run_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SENTINEL = 7.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_rule_24_gb300 import build
    build.build()
    import oracle
    oracle.build()
    gdn.gdn_init(0)
    yield
    assert gdn.device_status() == 0


def _prefix(p, lengths):
    """Problem ``p`` cut to the first ``lengths[n]`` tokens of each sequence."""
    cu = p.cu_seqlens.tolist()
    rows = torch.cat([torch.arange(cu[n], cu[n] + L) for n, L in enumerate(lengths)])
    cu_p = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return dataclasses.replace(p, q=p.q[rows], k=p.k[rows], v=p.v[rows],
                               g=None if p.g is None else p.g[rows],
                               beta=None if p.beta is None else p.beta[rows],
                               cu_seqlens=torch.tensor(cu_p))


def _run(p, M, every):
    dev = torch.device(DEV)
    out = torch.empty(p.T, p.H, 128, dtype=torch.bfloat16, device=dev)
    st = torch.zeros(p.state_slots, p.H, 128, 128, dtype=p.state_dtype, device=dev)
    ck = torch.full((p.N * M, p.H, 128, 128), SENTINEL, device=dev)
    gdn.gdn_chunk_prefill_checkpointed(
        p.q.to(dev), p.k.to(dev), p.v.to(dev), p.g.to(dev), p.beta.to(dev), p.scale,
        None if p.initial_state is None else p.initial_state.to(dev),
        None if p.state_indices is None else p.state_indices.to(dev), st, p.cu_seqlens.to(dev),
        p.use_qk_l2norm, p.batch_invariant, out, ck, M, every)
    torch.cuda.synchronize()
    return out, st, ck.cpu()


def _check_checkpoints(p, ck, M, every):
    lens = np.diff(p.cu_seqlens.numpy())
    span = 64 * every
    for m in range(M):
        have = [n for n in range(p.N) if lens[n] >= (m + 1) * span]
        for n in set(range(p.N)) - set(have):  # never written
            assert torch.all(ck[n * M + m] == SENTINEL), (n, m)
        if not have:
            continue
        cut = [int(min(lens[n], (m + 1) * span)) for n in range(p.N)]
        _, s_ref = run_oracle(_prefix(p, cut))
        # every (sequence, head) block on its own, so one bad block cannot hide
        worst = max((rel_l2(ck[n * M + m, h].numpy(), s_ref[n, h]), n, h) for n in have for h in range(p.H))
        assert worst[0] <= 1e-3, (m, worst)


@pytest.mark.parametrize("every", [1, 3])
def test_checkpoints_match_prefix_states(every):
    p = W.make_problem([700, 64, 130, 0, 1300, 63], 2, 4, gates="mamba", init="fp32", init_std=0.05,
                       seed=300 + every)
    M = 8
    out, st, ck = _run(p, M, every)
    compare(p, out, st)
    _check_checkpoints(p, ck, M, every)


def test_checkpoints_under_split_k(force_split):
    """Segments of a split sequence write the checkpoints that fall inside them."""
    force_split("3")
    p = W.make_problem([1500, 900, 256], 1, 2, gates="uniform", init="bf16", init_std=0.05,
                       state_dtype=torch.bfloat16, pool_slots=5, seed=310, batch_invariant=False)
    M, every = 12, 2
    out, st, ck = _run(p, M, every)
    compare(p, out, st)
    _check_checkpoints(p, ck, M, every)


def test_checkpoints_under_planner_split_slow_gates(force_split):
    """The planner's own split of 64 units of 64 chunks (on 152 SMs: segments of 3, 1, 1
    and 2 sevenths) on slowly decaying gates, so the states that segments 1-3 start from
    come through the fix-up with weight: every checkpoint matches the oracle's state of
    that prefix, the ones inside the later segments included."""
    force_split(0)
    p = W.make_problem([4096] * 4, 8, 16, gates="slow", init="fp32", init_std=0.05, seed=320,
                       batch_invariant=False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = gdn.testing_split_plan(p.N, p.H, p.T, sms)
    assert plan["P"] > 1
    M, every = 8, 8  # after 512, 1024, ..., 4096 tokens
    out, st, ck = _run(p, M, every)
    compare(p, out, st)
    _check_checkpoints(p, ck, M, every)
