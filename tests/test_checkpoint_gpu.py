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
        got = np.stack([ck[n * M + m].numpy() for n in have])
        want = np.stack([s_ref[n] for n in have])
        assert rel_l2(got, want) <= 1e-3, (m, rel_l2(got, want))


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
