"""Pins of the CPU oracle to facts other than itself.

The pages print no worked example, so each function is pinned by exact
arithmetic, closed forms, invariants of the recurrence, or a hand-worked case;
a dropped term, a wrong sign or index, or a transposed state fails at least
one of these.  The recurrence being pinned is the Gated Delta Rule stated for
flashinfer's chunked GDN prefill (flashinfer.gdn_prefill), with the argument
semantics of flashinfer.cudnn.cudnn_chunk_gated_delta_rule (Parameters).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_24_gb300 import workloads as W

pytestmark = pytest.mark.usefixtures("oracle_lib")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(lengths, H_qk, H_v, D, seed, *, gates=True, beta=True, init=True, dyadic=False):
    gen = torch.Generator().manual_seed(seed)
    T, N, H = sum(lengths), len(lengths), max(H_qk, H_v)
    if dyadic:   # small dyadic rationals: exact in fp64, so only rounding differs
        q = torch.randint(-8, 9, (T, H_qk, D), generator=gen).double() / 8
        k = torch.randint(-8, 9, (T, H_qk, D), generator=gen).double() / 8
        v = torch.randint(-8, 9, (T, H_v, D), generator=gen).double() / 8
        g = torch.randint(1, 9, (T, H), generator=gen).double() / 8
        b = torch.randint(0, 9, (T, H), generator=gen).double() / 16
        s0 = torch.randint(-8, 9, (N, H, D, D), generator=gen).double() / 8
    else:
        q = torch.randn(T, H_qk, D, generator=gen, dtype=torch.float64)
        k = torch.randn(T, H_qk, D, generator=gen, dtype=torch.float64)
        v = torch.randn(T, H_v, D, generator=gen, dtype=torch.float64)
        g = torch.exp(-torch.rand(T, H, generator=gen, dtype=torch.float64) * 0.5)
        b = torch.rand(T, H, generator=gen, dtype=torch.float64)
        s0 = torch.randn(N, H, D, D, generator=gen, dtype=torch.float64) * 0.3
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int64)
    return dict(q=q, k=k, v=v, g=g if gates else None, beta=b if beta else None,
                initial_state=s0 if init else None, cu_seqlens=cu)


def _frac_bruteforce(P, scale, H_qk, H_v):
    """Exact rational recurrence with the literal matrix product
    S <- g S (I - b k k^T) + b v k^T."""
    q, k, v = P["q"].numpy(), P["k"].numpy(), P["v"].numpy()
    g, b, s0 = P["g"].numpy(), P["beta"].numpy(), P["initial_state"].numpy()
    cu = P["cu_seqlens"].tolist()
    T, _, D = q.shape
    H = max(H_qk, H_v)
    F = lambda x: Fraction(float(x))  # noqa: E731  (exact: inputs are dyadic)
    out = [[None] * H for _ in range(T)]
    fin = {}
    for n in range(len(cu) - 1):
        for h in range(H):
            hq, hv = h // (H // H_qk), h // (H // H_v)
            S = [[F(s0[n, h, i, j]) for j in range(D)] for i in range(D)]
            for t in range(cu[n], cu[n + 1]):
                kt = [F(x) for x in k[t, hq]]
                qt = [F(x) for x in q[t, hq]]
                vt = [F(x) for x in v[t, hv]]
                a, bb = F(g[t, h]), F(b[t, h])
                M = [[(1 if i == j else 0) - bb * kt[i] * kt[j] for j in range(D)] for i in range(D)]
                S = [[a * sum(S[i][m] * M[m][j] for m in range(D)) + bb * vt[i] * kt[j]
                      for j in range(D)] for i in range(D)]
                out[t][h] = [scale * sum(S[i][j] * qt[j] for j in range(D)) for i in range(D)]
            fin[(n, h)] = S
    return out, fin


@pytest.mark.parametrize("impl", ["recurrence", "chunked"])
def test_exact_rational_bruteforce(impl):
    """fp64 oracle vs exact rational arithmetic at head_dim 4 (pins every term)."""
    lengths, H_qk, H_v, D = [5, 3, 0, 1], 1, 2, 4
    P = _problem(lengths, H_qk, H_v, D, seed=7, dyadic=True)
    scale = Fraction(1, 2)
    ref_o, ref_s = _frac_bruteforce(P, scale, H_qk, H_v)
    fn = oracle.recurrence if impl == "recurrence" else \
        (lambda **kw: oracle.chunked(chunk=2, **kw))
    o, s = fn(**P, scale=0.5, use_qk_l2norm=False)
    for t in range(sum(lengths)):
        for h in range(2):
            exact = np.array([float(x) for x in ref_o[t][h]])
            np.testing.assert_allclose(o[t, h], exact, rtol=1e-13, atol=1e-13)
    for (n, h), S in ref_s.items():
        exact = np.array([[float(x) for x in row] for row in S])
        np.testing.assert_allclose(s[n, h], exact, rtol=1e-13, atol=1e-13)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    return vals


@pytest.mark.parametrize("impl", ["recurrence", "chunked"])
def test_hand_worked_d2(impl):
    """Two steps worked by hand at head_dim 2 (tests/golden/hand_d2_t2.txt)."""
    G = _read_golden("hand_d2_t2.txt")
    q = torch.tensor(np.stack([G["q1"], G["q2"]]))[:, None, :]
    k = torch.tensor(np.stack([G["k1"], G["k2"]]))[:, None, :]
    v = torch.tensor(np.stack([G["v1"], G["v2"]]))[:, None, :]
    g = torch.tensor([G["g1"][0], G["g2"][0]])[:, None]
    b = torch.tensor([G["b1"][0], G["b2"][0]])[:, None]
    s0 = torch.tensor(G["S0"].reshape(1, 1, 2, 2))
    fn = oracle.recurrence if impl == "recurrence" else oracle.chunked
    o, s = fn(q=q, k=k, v=v, g=g, beta=b, scale=1.0, initial_state=s0,
              cu_seqlens=[0, 2], use_qk_l2norm=False)
    np.testing.assert_allclose(o[0, 0], G["o1"], atol=1e-15)
    np.testing.assert_allclose(o[1, 0], G["o2"], atol=1e-15)
    np.testing.assert_allclose(s[0, 0].reshape(-1), G["S2"], atol=1e-15)


@pytest.mark.parametrize("impl", ["recurrence", "chunked"])
def test_beta_zero_closed_form(impl):
    """beta = 0: S_t = (prod_{s<=t} g_s) S_0 and o_t = scale (prod g) S_0 q_t."""
    P = _problem([70, 9], 1, 1, 16, seed=3)
    P["beta"] = torch.zeros_like(P["g"])
    fn = oracle.recurrence if impl == "recurrence" else oracle.chunked
    o, s = fn(**P, scale=0.25, use_qk_l2norm=False)
    cu = P["cu_seqlens"].tolist()
    for n in range(2):
        lg = torch.cumsum(torch.log(P["g"][cu[n]:cu[n + 1], 0]), 0)
        decay = torch.exp(lg).numpy()
        S0 = P["initial_state"][n, 0].numpy()
        want = 0.25 * decay[:, None] * (P["q"][cu[n]:cu[n + 1], 0].numpy() @ S0.T)
        np.testing.assert_allclose(o[cu[n]:cu[n + 1], 0], want, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(s[n, 0], decay[-1] * S0, rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("impl", ["recurrence", "chunked"])
def test_g_one_beta_zero_keeps_state(impl):
    """g = 1 and beta = 0 leave the state unchanged."""
    P = _problem([67], 1, 1, 8, seed=4)
    P["g"] = torch.ones_like(P["g"])
    P["beta"] = torch.zeros_like(P["g"])
    fn = oracle.recurrence if impl == "recurrence" else oracle.chunked
    o, s = fn(**P, scale=1.0, use_qk_l2norm=False)
    S0 = P["initial_state"][0, 0].numpy()
    np.testing.assert_array_equal(s[0, 0], S0)
    np.testing.assert_allclose(o[:, 0], P["q"][:, 0].numpy() @ S0.T, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("impl", ["recurrence", "chunked"])
def test_delta_rule_stores_value(impl):
    """beta = 1 with unit keys: S_t k_t = v_t for any g and any prior state
    ((I - k k^T) k = 0).  Reading with q_t = k_t gives o_t = scale v_t; this pins
    the V-major orientation and that o_t uses the post-update state."""
    P = _problem([130], 1, 1, 32, seed=5)
    k = P["k"] / P["k"].norm(dim=-1, keepdim=True)
    P["k"], P["q"] = k, k.clone()
    P["beta"] = torch.ones_like(P["g"])
    fn = oracle.recurrence if impl == "recurrence" else oracle.chunked
    o, _ = fn(**P, scale=0.5, use_qk_l2norm=False)
    np.testing.assert_allclose(o[:, 0], 0.5 * P["v"][:, 0].numpy(), rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("impl", ["recurrence", "chunked"])
def test_orthonormal_memory(impl):
    """g = 1, beta = 1, orthonormal keys from a zero state: S = sum_i v_i k_i^T,
    so every stored key recalls its value (the textbook delta-rule memory)."""
    D = 16
    gen = torch.Generator().manual_seed(6)
    Qm, _ = torch.linalg.qr(torch.randn(D, D, generator=gen, dtype=torch.float64))
    keys = Qm.T.contiguous()                      # rows orthonormal
    v = torch.randn(D, 1, D, generator=gen, dtype=torch.float64)
    fn = oracle.recurrence if impl == "recurrence" else oracle.chunked
    o, s = fn(q=keys[:, None, :], k=keys[:, None, :], v=v, g=None, beta=None, scale=1.0,
              initial_state=None, cu_seqlens=[0, D], use_qk_l2norm=False)
    np.testing.assert_allclose(s[0, 0], v[:, 0].numpy().T @ keys.numpy(), atol=1e-12)
    np.testing.assert_allclose(s[0, 0] @ keys.numpy().T, v[:, 0].numpy().T, atol=1e-12)


@pytest.mark.parametrize("impl", ["recurrence", "chunked"])
def test_split_invariance(impl):
    """Running [0, t) then [t, T) with final_state -> initial_state equals [0, T)."""
    P = _problem([200], 2, 4, 16, seed=8)
    fn = oracle.recurrence if impl == "recurrence" else oracle.chunked
    o, s = fn(**P, scale=0.3, use_qk_l2norm=True)
    t = 77
    A = {k: (v[:t] if k in ("q", "k", "v", "g", "beta") else v) for k, v in P.items()}
    A["cu_seqlens"] = [0, t]
    oa, sa = fn(**A, scale=0.3, use_qk_l2norm=True)
    B = {k: (v[t:] if k in ("q", "k", "v", "g", "beta") else v) for k, v in P.items()}
    B["cu_seqlens"] = [0, 200 - t]
    B["initial_state"] = torch.tensor(sa)
    ob, sb = fn(**B, scale=0.3, use_qk_l2norm=True)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(sb, s, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("length", [1, 63, 64, 65, 129, 200])
def test_chunked_matches_recurrence(length):
    """The numpy chunked form and the C recurrence agree to fp64 round-off."""
    P = _problem([length, 3], 2, 4, 128, seed=length)
    o1, s1 = oracle.recurrence(**P, scale=None, use_qk_l2norm=True)
    o2, s2 = oracle.chunked(**P, scale=None, use_qk_l2norm=True)
    assert np.abs(o1 - o2).max() <= 1e-12 * np.abs(o1).max()
    assert np.abs(s1 - s2).max() <= 1e-12 * np.abs(s1).max()


def test_chunked_matches_recurrence_workload2():
    P = W.make_workload(2)
    args = dict(q=P.q, k=P.k, v=P.v, g=P.g, beta=P.beta, scale=P.scale,
                initial_state=P.initial_state, state_indices=P.state_indices,
                cu_seqlens=P.cu_seqlens, use_qk_l2norm=P.use_qk_l2norm,
                units=[(n, h) for n in range(P.N) for h in (0, 5)])
    o1, s1 = oracle.recurrence(**args)
    o2, s2 = oracle.chunked(**args)
    m = ~np.isnan(o1)
    assert np.abs(o1[m] - o2[m]).max() <= 1e-12 * np.abs(o1[m]).max()
    for n in range(P.N):
        for h in (0, 5):
            assert np.abs(s1[n, h] - s2[n, h]).max() <= 1e-12 * np.abs(s1[n, h]).max()


def test_l2norm_is_scale_invariant():
    """With the fused L2 norm, rescaling q and k by positive factors changes the
    result only through the 1e-6 epsilon."""
    P = _problem([90], 1, 1, 32, seed=9)
    o, s = oracle.recurrence(**P, scale=0.2, use_qk_l2norm=True)
    P2 = dict(P, q=P["q"] * 7.0, k=P["k"] * 0.25)
    o2, s2 = oracle.recurrence(**P2, scale=0.2, use_qk_l2norm=True)
    np.testing.assert_allclose(o2, o, rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(s2, s, rtol=2e-5, atol=1e-6)
    # and it really normalises: unit-norm inputs are (nearly) left alone
    P3 = dict(P, q=P["q"] / P["q"].norm(dim=-1, keepdim=True),
              k=P["k"] / P["k"].norm(dim=-1, keepdim=True))
    o3, s3 = oracle.recurrence(**P3, scale=0.2, use_qk_l2norm=False)
    np.testing.assert_allclose(o, o3, rtol=1e-5, atol=1e-6)


def test_scale_default_and_linearity():
    """scale None or 0.0 means 1/sqrt(head_dim); the output is linear in scale
    and the state does not depend on it."""
    P = _problem([40], 1, 1, 64, seed=10)
    o_none, s_none = oracle.recurrence(**P, scale=None)
    o_zero, _ = oracle.recurrence(**P, scale=0.0)
    o_exp, s_exp = oracle.recurrence(**P, scale=1 / math.sqrt(64))
    np.testing.assert_array_equal(o_none, o_exp)
    np.testing.assert_array_equal(o_zero, o_exp)
    o_two, s_two = oracle.recurrence(**P, scale=2 / math.sqrt(64))
    np.testing.assert_allclose(o_two, 2 * o_exp, rtol=1e-14)
    np.testing.assert_array_equal(s_two, s_exp)


def test_head_grouping():
    """Sab head h reads q/k head h // (H/H_qk) and v head h // (H/H_v): each
    unit equals the single-head problem built from those slices."""
    P = _problem([33, 20], 2, 4, 16, seed=11)
    o, s = oracle.recurrence(**P, scale=0.5, use_qk_l2norm=True)
    for h in range(4):
        hq = h // 2
        Q = dict(q=P["q"][:, hq:hq + 1], k=P["k"][:, hq:hq + 1], v=P["v"][:, h:h + 1],
                 g=P["g"][:, h:h + 1], beta=P["beta"][:, h:h + 1],
                 initial_state=P["initial_state"][:, h:h + 1], cu_seqlens=P["cu_seqlens"])
        o1, s1 = oracle.recurrence(**Q, scale=0.5, use_qk_l2norm=True)
        np.testing.assert_array_equal(o[:, h], o1[:, 0])
        np.testing.assert_array_equal(s[:, h], s1[:, 0])


def test_state_indices_gather():
    """With state_indices, sequence n starts from pool slot state_indices[n]."""
    P = _problem([10, 0, 25], 1, 2, 16, seed=12)
    pool = torch.randn(7, 2, 16, 16, generator=torch.Generator().manual_seed(1),
                       dtype=torch.float64)
    idx = torch.tensor([5, 0, 3], dtype=torch.int32)
    o, s = oracle.recurrence(**dict(P, initial_state=pool), state_indices=idx, scale=0.5)
    o2, s2 = oracle.recurrence(**dict(P, initial_state=pool[idx.long()]), scale=0.5)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(s, s2)


def test_empty_sequences_pass_state_through():
    P = _problem([0, 4, 0], 1, 1, 8, seed=13)
    o, s = oracle.recurrence(**P, scale=1.0)
    np.testing.assert_array_equal(s[0, 0], P["initial_state"][0, 0].numpy())
    np.testing.assert_array_equal(s[2, 0], P["initial_state"][2, 0].numpy())
    P["initial_state"] = None
    o, s = oracle.recurrence(**P, scale=1.0)
    assert not s[0].any() and not s[2].any()
    o, s = oracle.recurrence(**dict(P, cu_seqlens=[0, 0, 0]), scale=1.0)
    assert not s.any()


def test_workload_generators_are_seeded():
    a, b = W.make_workload(2), W.make_workload(2)
    for x, y in [(a.q, b.q), (a.v, b.v), (a.g, b.g), (a.initial_state, b.initial_state)]:
        assert torch.equal(x, y)
    assert a.lengths()[:0] == [] and sorted(a.lengths())[:1] == [1]
    assert {1, 63, 64, 65} <= set(a.lengths()) and len(a.lengths()) == 8
    # workload-5 structure on a small pool (the full 4096-slot pool is slow to draw on a CPU)
    p5 = W.make_problem(W.short_lengths(1005)[:32], 8, 16, init="bf16", init_std=0.05,
                        state_dtype=torch.bfloat16, pool_slots=64, cu_dtype=torch.int64,
                        idx_dtype=torch.int32, seed=1005)
    assert p5.cu_seqlens.dtype == torch.int64 and p5.state_indices.dtype == torch.int32
    assert len(set(p5.state_indices.tolist())) == 32
    assert all(16 <= n <= 256 for n in p5.lengths())
