"""GPU parity of the decode step (one token per batch row, state updated in place)
against the fp64 CPU oracle, through the C ABI.

A decode batch of B rows is the recurrence over B sequences of one token each, so the
oracle is the same token recurrence the prefill tests use.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import compare, run_oracle, rel_l2, OUT_REL_L2, STATE_REL_L2

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


def _decode(p, pool):
    """One decode step of problem ``p`` (T == N rows) on ``pool`` (device, in place)."""
    dev = torch.device(DEV)
    out = torch.empty(p.T, p.H, 128, dtype=torch.bfloat16, device=dev)
    gdn.gdn_decode_step(p.q.to(dev), p.k.to(dev), p.v.to(dev),
                        None if p.g is None else p.g.to(dev),
                        None if p.beta is None else p.beta.to(dev), p.scale, pool,
                        None if p.state_indices is None else p.state_indices.to(dev),
                        p.use_qk_l2norm, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("state", ["fp32", "bf16"])
@pytest.mark.parametrize("heads", [(1, 1), (2, 4), (4, 2), (3, 6), (6, 3)])
def test_decode_matches_oracle(state, heads):
    dt = {"fp32": torch.float32, "bf16": torch.bfloat16}[state]
    p = W.make_problem([1] * 37, heads[0], heads[1], gates="mamba", init=state, init_std=0.1,
                       state_dtype=dt, pool_slots=50, idx_dtype=torch.int64, seed=200 + heads[1])
    pool = p.initial_state.to(DEV).clone()
    out = _decode(p, pool)
    compare(p, out, pool)
    # slots no row addresses are untouched
    untouched = sorted(set(range(p.state_slots)) - set(p.state_indices.tolist()))
    assert torch.equal(pool[untouched].cpu(), p.initial_state[untouched])


def test_decode_defaults_no_gates_no_indices():
    p = W.make_problem([1] * 9, 2, 2, init="fp32", init_std=0.1, with_g=False, with_beta=False,
                       use_qk_l2norm=False, seed=210)
    p.k = (p.k.float() / 12.0).to(torch.bfloat16)
    pool = p.initial_state.to(DEV).clone()
    p.scale = 0.0
    out = _decode(p, pool)
    p.scale = 1.0 / np.sqrt(128.0)
    compare(p, out, pool)


def test_prefill_then_decode_handoff():
    """Prefill a batch into a bf16 state pool, then three decode steps through the same
    pool: outputs and final states match the oracle run over the whole sequences."""
    prompt = [300, 129, 64, 1]
    steps = 3
    full = W.make_problem([L + steps for L in prompt], 2, 4, gates="mamba", init="bf16",
                          init_std=0.05, state_dtype=torch.bfloat16, pool_slots=8, seed=220)
    cu = full.cu_seqlens.tolist()
    o_ref, s_ref = run_oracle(full)
    pool = full.initial_state.to(DEV).clone()
    # prefill over the prompts, final states written in place of the initial ones
    rows = torch.cat([torch.arange(cu[n], cu[n] + L) for n, L in enumerate(prompt)])
    cu_p = [0]
    for L in prompt:
        cu_p.append(cu_p[-1] + L)
    pre = dataclasses.replace(full, q=full.q[rows], k=full.k[rows], v=full.v[rows], g=full.g[rows],
                              beta=full.beta[rows], cu_seqlens=torch.tensor(cu_p, dtype=torch.int32))
    staging = torch.empty_like(pool)
    staging.copy_(pool)
    out_pre, _ = gdn.run_problem(pre, device=DEV, output_state=staging)
    torch.cuda.synchronize()
    pool.copy_(staging)
    o_pre = np.concatenate([o_ref[cu[n]:cu[n] + L] for n, L in enumerate(prompt)])
    assert rel_l2(out_pre.float().cpu().numpy(), o_pre) <= OUT_REL_L2
    for j in range(steps):
        rows = torch.tensor([cu[n] + L + j for n, L in enumerate(prompt)])
        step = dataclasses.replace(full, q=full.q[rows], k=full.k[rows], v=full.v[rows], g=full.g[rows],
                                   beta=full.beta[rows],
                                   cu_seqlens=torch.arange(len(prompt) + 1, dtype=torch.int32))
        out = _decode(step, pool)
        want = o_ref[rows.numpy()]
        assert rel_l2(out.float().cpu().numpy(), want) <= OUT_REL_L2, j
    idx = full.state_indices.tolist()
    got = np.stack([pool[idx[n]].float().cpu().numpy() for n in range(len(prompt))])
    assert rel_l2(got, s_ref) <= STATE_REL_L2[torch.bfloat16]


def test_decode_bad_index_sets_error_bit():
    p = W.make_problem([1] * 4, 1, 2, init="fp32", pool_slots=6, seed=230)
    p.state_indices = torch.tensor([0, 9, 2, 3], dtype=torch.int32)
    pool = p.initial_state.to(DEV).clone()
    _decode(p, pool)
    assert gdn.device_status() & gdn.binding.DEVERR_STATE_INDEX
    assert torch.equal(pool[1].cpu(), p.initial_state[1])  # row 1's would-be slot: none touched
    p = W.make_problem([1] * 4, 1, 2, init="fp32", pool_slots=6, seed=231)
    pool = p.initial_state.to(DEV).clone()
    compare(p, _decode(p, pool), pool)
    assert gdn.device_status() == 0


def test_decode_workload_full_size_sampled():
    """The decode batch that follows workload 5: 1024 rows, 8 q/k heads, 16 v heads, a
    4096-slot bf16 pool through int32 state_indices (sampled (row, head) units)."""
    p = W.make_decode_workload(device=DEV)
    pool = p.initial_state.clone()
    out = _decode(p, pool)
    rng = np.random.default_rng(240)
    units = [(int(rng.integers(p.N)), int(rng.integers(p.H))) for _ in range(64)]
    idx = p.state_indices.cpu().tolist()
    small = dataclasses.replace(p, q=p.q.cpu(), k=p.k.cpu(), v=p.v.cpu(), g=p.g.cpu(), beta=p.beta.cpu(),
                                initial_state=p.initial_state.cpu(), state_indices=p.state_indices.cpu(),
                                cu_seqlens=p.cu_seqlens.cpu())
    o_ref, s_ref = run_oracle(small, units)
    got_o = np.stack([out[n, h].float().cpu().numpy() for n, h in units])
    want_o = np.stack([o_ref[n, h] for n, h in units])
    assert rel_l2(got_o, want_o) <= OUT_REL_L2
    got_s = np.stack([pool[idx[n], h].float().cpu().numpy() for n, h in units])
    want_s = np.stack([s_ref[n, h] for n, h in units])
    assert rel_l2(got_s, want_s) <= STATE_REL_L2[torch.bfloat16]
