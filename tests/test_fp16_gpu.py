"""fp16 inputs and states (q/k/v/output fp16, every tensor-core operand fp16, fp16 or f32
state pools, fp16 gates) against the fp64 oracle, for the prefill, split-K and the
decode step."""
import numpy as np
import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
F16 = torch.float16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_rule_24_gb300 import build
    build.build()
    import oracle
    oracle.build()
    gdn.gdn_init(0)
    yield
    assert gdn.device_status() == 0


def _run(p):
    out, st = gdn.run_problem(p, device=DEV)
    torch.cuda.synchronize()
    return out, st


@pytest.mark.parametrize("state", ["fp16", "fp32"])
@pytest.mark.parametrize("heads", [(1, 1), (2, 4)])
def test_prefill_fp16(state, heads):
    dt = {"fp16": F16, "fp32": torch.float32}[state]
    p = W.make_problem([1, 63, 64, 65, 300, 0, 777], heads[0], heads[1], gates="mamba", init=state,
                       init_std=0.05, state_dtype=dt, qkv_dtype=F16, seed=400 + heads[1])
    out, st = _run(p)
    assert out.dtype == F16
    compare(p, out, st)


def test_prefill_fp16_gates_and_pool():
    p = W.make_problem([200, 129, 1000], 2, 4, gates="uniform", init="fp16", init_std=0.05,
                       state_dtype=F16, pool_slots=7, cu_dtype=torch.int64, qkv_dtype=F16, seed=410)
    p.g = p.g.to(F16)
    p.beta = p.beta.to(F16)
    out, st = _run(p)
    compare(p, out, st)


@pytest.mark.parametrize("gates", ["mamba", "slow"])
def test_prefill_fp16_split_k(force_split, gates):
    """Forced P = 3; the slow gates keep the segment maps from underflowing."""
    force_split("3")
    p = W.make_problem([900, 64, 1500], 1, 2, gates=gates, init="fp32", init_std=0.05,
                       qkv_dtype=F16, seed=420, batch_invariant=False)
    out, st = _run(p)
    compare(p, out, st)


def test_prefill_fp16_planner_split(force_split):
    """The planner's own split of 64 units of 64 chunks, fp16 operands and fp16 states,
    slow gates."""
    force_split(0)
    p = W.make_problem([4096] * 4, 8, 16, gates="slow", init="fp16", init_std=0.05, state_dtype=F16,
                       qkv_dtype=F16, seed=425, batch_invariant=False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert gdn.testing_split_plan(p.N, p.H, p.T, sms)["P"] > 1
    out, st = _run(p)
    compare(p, out, st)


@pytest.mark.parametrize("state", ["fp16", "fp32"])
def test_decode_fp16(state):
    dt = {"fp16": F16, "fp32": torch.float32}[state]
    p = W.make_problem([1] * 33, 2, 4, gates="mamba", init=state, init_std=0.1, state_dtype=dt,
                       pool_slots=40, qkv_dtype=F16, seed=430)
    pool = p.initial_state.to(DEV).clone()
    out = torch.empty(p.T, p.H, 128, dtype=F16, device=DEV)
    gdn.gdn_decode_step(p.q.to(DEV), p.k.to(DEV), p.v.to(DEV), p.g.to(DEV), p.beta.to(DEV), p.scale, pool,
                        p.state_indices.to(DEV), p.use_qk_l2norm, out)
    torch.cuda.synchronize()
    compare(p, out, pool)
