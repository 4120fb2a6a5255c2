"""GPU parity of the CUDA prefill against the fp64 CPU oracle, through the C ABI.

Every comparison runs the library kernel (via the ctypes binding of
gdn_chunk_prefill) and the oracle on the same seeded inputs.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import compare, run_oracle

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


def test_workload1_single_sequence():
    p = W.make_workload(1)
    out, st = _run(p)
    compare(p, out, st)


def test_workload1_zero_initial_state_equals_null():
    """An explicit zero fp32 initial state gives bit-identical results to none."""
    p = W.make_workload(1)
    out0, st0 = _run(p)
    p.initial_state = torch.zeros(1, 1, 128, 128)
    out1, st1 = _run(p)
    assert torch.equal(out0, out1) and torch.equal(st0, st1)


def test_workload2_varlen():
    p = W.make_workload(2)
    out, st = _run(p)
    compare(p, out, st)


@pytest.mark.parametrize("lengths", [[1, 63, 64, 65, 127, 128, 129], [0, 5, 0, 200, 0], [300]])
@pytest.mark.parametrize("heads", [(1, 1), (2, 4), (4, 2), (3, 6), (6, 3)])
def test_edge_lengths_and_head_maps(lengths, heads):
    p = W.make_problem(lengths, heads[0], heads[1], gates="uniform", init="fp32", seed=sum(lengths))
    out, st = _run(p)
    compare(p, out, st)


def test_defaults_null_gates_and_state_no_l2norm():
    """g, beta and the initial state absent; scale 0 means 1/sqrt(128); no L2 norm."""
    p = W.make_problem([70, 33], 2, 2, init=None, with_g=False, with_beta=False,
                       use_qk_l2norm=False, seed=21)
    # without the L2 norm and with g = beta = 1 the state grows with |k|^2 ~ 128 per
    # token; scale the keys so the recurrence stays well conditioned
    p.k = (p.k.float() / 12.0).to(torch.bfloat16)
    p.scale = 0.0
    out, st = _run(p)
    p.scale = 1.0 / np.sqrt(128.0)
    compare(p, out, st)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_long_memory_slow_gates(state_dtype):
    """Gates close to one (log g ~ U(-0.001, 0), beta ~ U(0, 0.1)): the state carries
    information across the whole 4096-token sequence, so the inter-chunk path (state
    update, its 16-bit operand copy, the decay of the carried state) is weighted over 64
    chunks, not only over the last one or two as with faster decays."""
    p = W.make_problem([4096, 1000, 65], 2, 4, gates="slow", init="fp32", init_std=0.05,
                       state_dtype=state_dtype, seed=41)
    out, st = _run(p)
    compare(p, out, st)


def test_gate_and_state_dtypes():
    """bf16 g and beta, bf16 initial state into an fp32 output state, int64 cu_seqlens."""
    p = W.make_problem([100, 64, 17], 2, 4, gates="mamba", init="bf16", init_std=0.05,
                       state_dtype=torch.float32, cu_dtype=torch.int64, seed=31)
    p.g = p.g.to(torch.bfloat16)
    p.beta = p.beta.to(torch.bfloat16)
    out, st = _run(p)
    compare(p, out, st)
    p.g = p.g.to(torch.float16)
    p.state_dtype = torch.bfloat16
    out, st = _run(p)
    compare(p, out, st)


def test_state_pool_with_indices():
    """Workload-5 style pools: int32 state_indices into bf16 pools, int64 cu_seqlens."""
    p = W.make_workload(5, seqs=48)
    out, st = _run(p)
    compare(p, out, st)
    # slots not addressed by state_indices are left untouched
    untouched = sorted(set(range(p.state_slots)) - set(p.state_indices.tolist()))[:64]
    assert not st[untouched].float().abs().sum().item()


def test_strided_qkv_from_fused_buffer():
    """q, k, v as column slices of one fused [T, (2*Hqk + Hv) * 128] buffer."""
    p = W.make_problem([90, 40], 2, 4, seed=41)
    T = p.T
    fused = torch.empty(T, (2 * 2 + 4) * 128, dtype=torch.bfloat16)
    fused[:, :256] = p.q.reshape(T, -1)
    fused[:, 256:512] = p.k.reshape(T, -1)
    fused[:, 512:] = p.v.reshape(T, -1)
    fd = fused.to(DEV)
    q = fd[:, :256].view(T, 2, 128)
    k = fd[:, 256:512].view(T, 2, 128)
    v = fd[:, 512:].view(T, 4, 128)
    assert not q.is_contiguous()
    out = torch.empty(T, 4, 128, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(p.N, 4, 128, 128, device=DEV)
    gdn.gdn_chunk_prefill(q, k, v, p.g.to(DEV), p.beta.to(DEV), p.scale,
                          p.initial_state.to(DEV), None, st, p.cu_seqlens.to(DEV), True, True, out)
    torch.cuda.synchronize()
    compare(p, out, st)


def _sub(p, rows, cu, init, **kw):
    """A problem made of rows ``rows`` of ``p`` with new cu_seqlens and initial states."""
    pick = {name: (None if getattr(p, name) is None else getattr(p, name)[rows])
            for name in ("q", "k", "v", "g", "beta")}
    return dataclasses.replace(p, **pick, cu_seqlens=torch.tensor(cu, dtype=torch.int32),
                               initial_state=init, state_indices=None,
                               state_slots=len(cu) - 1, **kw)


def test_batch_invariance_bitwise():
    """With batch_invariant every bit of a sequence's output and state is independent
    of what else is in the batch and where the sequence sits in the packing."""
    p = W.make_problem([150, 77, 300, 1], 2, 4, gates="mamba", init="fp32", init_std=0.05, seed=51)
    out, st = _run(p)
    cu = p.cu_seqlens.tolist()
    pad = 37
    for n in range(p.N):
        a, b = cu[n], cu[n + 1]
        rows = torch.cat([torch.arange(pad), torch.arange(a, b)])
        other = (n + 1) % p.N
        init = torch.cat([p.initial_state[other:other + 1], p.initial_state[n:n + 1]])
        q = _sub(p, rows, [0, pad, pad + b - a], init)
        o2, s2 = _run(q)
        assert torch.equal(o2[pad:], out[a:b]), n
        assert torch.equal(s2[1], st[n]), n


def test_workload3_full_size_sampled_units():
    p = W.make_workload(3)
    out, st = _run(p)
    rng = np.random.default_rng(3)
    units = [(int(rng.integers(p.N)), int(rng.integers(p.H))) for _ in range(6)]
    compare(p, out, st, units=units)
    assert torch.isfinite(out.float()).all()


# eight (sequence, head) units of workload 4, both sequences, heads spread over 0..31
# (both heads of a q/k pair among them)
WORKLOAD4_UNITS = [(0, 0), (0, 5), (0, 17), (0, 30), (1, 2), (1, 3), (1, 21), (1, 31)]


def test_workload4_full_size_batch_invariant():
    """2 x 65536 tokens with batch_invariant: sampled units match the oracle, and each
    sequence run alone reproduces the batch result bit for bit."""
    p = W.make_workload(4, batch_invariant=True)
    out, st = _run(p)
    compare(p, out, st, units=WORKLOAD4_UNITS)
    for n in range(2):
        a, b = n * 65536, (n + 1) * 65536
        q = _sub(p, slice(a, b), [0, 65536], p.initial_state[n:n + 1])
        o2, s2 = _run(q)
        assert torch.equal(o2, out[a:b]) and torch.equal(s2[0], st[n]), n


def test_workload5_full_size_sampled_units():
    p = W.make_workload(5, device=DEV)
    out, st = _run(p)
    rng = np.random.default_rng(5)
    units = [(int(rng.integers(p.N)), int(rng.integers(p.H))) for _ in range(24)]
    compare(p.to("cpu"), out, st, units=units)


def test_device_detected_bad_inputs_do_not_fault():
    """Decreasing cu_seqlens and out-of-range state indices set device error bits,
    skip the affected sequences and leave the context usable."""
    p = W.make_problem([40, 40, 40], 1, 2, seed=61)
    p.cu_seqlens = torch.tensor([0, 40, 30, 120], dtype=torch.int32)
    out, st = _run(p)
    assert gdn.device_status() & gdn.binding.DEVERR_CU_SEQLENS
    p = W.make_workload(5, seqs=8)
    p.state_indices = p.state_indices.clone()
    p.state_indices[3] = 5000
    out, st = _run(p)
    assert gdn.device_status() & gdn.binding.DEVERR_STATE_INDEX
    # the context still works
    p = W.make_workload(1)
    out, st = _run(p)
    compare(p, out, st)
    assert gdn.device_status() == 0


def test_many_units_per_cta_with_pools_and_gaps():
    """Several units per CTA through 16-bit pools (the incoming and final states move by
    TMA, staged through the output stage and a held K-copy slot), with empty, one-token,
    partial and exact-chunk sequences in between and one unit whose state index is out of
    range: that unit is skipped with its error bit, every other unit matches the oracle,
    and slots nobody addresses stay untouched."""
    pattern = [0, 1, 63, 64, 65, 130, 200, 0, 7, 128]
    lens = [pattern[(3 * n) % len(pattern)] for n in range(400)]
    p = W.make_problem(lens, 2, 4, gates="slow", init="bf16", init_std=0.05, state_dtype=torch.bfloat16,
                       pool_slots=1024, seed=62)
    out, st = _run(p)
    assert gdn.device_status() == 0
    compare(p, out, st)
    bad = 137
    p.state_indices = p.state_indices.clone()
    p.state_indices[bad] = 5000
    out, st = _run(p)
    assert gdn.device_status() & gdn.binding.DEVERR_STATE_INDEX
    units = [(n, h) for n in range(p.N) for h in range(p.H) if n != bad]
    q = dataclasses.replace(p, state_indices=p.state_indices.clone())
    q.state_indices[bad] = 0  # any valid slot for the oracle; that unit is not compared
    o_ref, s_ref = run_oracle(q, units)
    rows = torch.ones(p.T, dtype=torch.bool)
    rows[int(p.cu_seqlens[bad]):int(p.cu_seqlens[bad + 1])] = False
    o = out.float().cpu()[rows].numpy()
    ref = o_ref[rows.numpy()]
    assert np.linalg.norm(o - ref) / np.linalg.norm(ref) <= 5e-3
    compare(q, out, st, units=units, o_ref=o_ref, s_ref=s_ref)


def test_all_empty_batch():
    p = W.make_problem([0, 0, 0], 1, 2, init="fp32", seed=71)
    out, st = _run(p)
    assert torch.equal(st.cpu(), p.initial_state)


def test_workload5_batch_order_permuted_bitwise():
    """With batch_invariant, permuting the order of the sequences in the packed batch
    (their rows, states and state slots moved together) changes no bit of any
    sequence's output or final state."""
    p = W.make_workload(5, seqs=160, batch_invariant=True)
    out, st = _run(p)
    cu = p.cu_seqlens.tolist()
    perm = np.random.default_rng(55).permutation(p.N)
    rows = torch.cat([torch.arange(cu[n], cu[n + 1]) for n in perm])
    lens = [cu[n + 1] - cu[n] for n in perm]
    cu2 = np.concatenate([[0], np.cumsum(lens)]).tolist()
    pick = {name: getattr(p, name)[rows] for name in ("q", "k", "v", "g", "beta")}
    q = dataclasses.replace(p, **pick, cu_seqlens=torch.tensor(cu2, dtype=p.cu_seqlens.dtype),
                            state_indices=p.state_indices[torch.as_tensor(perm)])
    o2, s2 = _run(q)
    for j, n in enumerate(perm):
        assert torch.equal(o2[cu2[j]:cu2[j + 1]], out[cu[n]:cu[n + 1]]), n
    slots = p.state_indices.tolist()
    assert torch.equal(s2[slots], st[slots])
