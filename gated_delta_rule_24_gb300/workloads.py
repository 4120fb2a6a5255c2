"""Seeded synthetic inputs for chunked Gated Delta Rule prefill.

This module only draws random tensors with the shapes, dtypes and value
distributions of the prefill workloads; it holds none of the method's
arithmetic.  Both the CUDA path (through the binding) and the CPU oracle are
fed from it, so each side sees bit-identical inputs.

Layouts follow the flashinfer ``cudnn_chunk_gated_delta_rule`` documentation
(Parameters: q/k/v, g, beta, initial_state, cu_seqlens):

* q, k: ``[T, H_qk, 128]`` bf16, v: ``[T, H_v, 128]`` bf16, packed varlen;
* g (linear-space forget gate, alpha = exp(log g)) and beta (post-sigmoid
  update gate): ``[T, H]`` fp32, with ``H = max(H_qk, H_v)`` sab heads;
* states: ``[slots, H, 128, 128]`` V-major (row = value index);
* cu_seqlens: ``[N + 1]`` int32 or int64.

All randomness comes from one ``torch.Generator`` seeded per workload, drawn
on the CPU (bit-identical on every host) unless ``device`` asks otherwise.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

HEAD_DIM = 128


@dataclasses.dataclass
class Problem:
    """One prefill call's inputs plus the description of its outputs."""

    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: Optional[torch.Tensor]
    beta: Optional[torch.Tensor]
    scale: float
    initial_state: Optional[torch.Tensor]
    state_indices: Optional[torch.Tensor]
    cu_seqlens: torch.Tensor
    use_qk_l2norm: bool
    batch_invariant: bool
    output_final_state: bool
    state_dtype: torch.dtype          # dtype of the state the call writes
    state_slots: int                  # first dim of the output-state buffer
    seed: int

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def H_qk(self) -> int:
        return int(self.q.shape[1])

    @property
    def H_v(self) -> int:
        return int(self.v.shape[1])

    @property
    def H(self) -> int:
        return max(self.H_qk, self.H_v)

    @property
    def N(self) -> int:
        return int(self.cu_seqlens.shape[0]) - 1

    def lengths(self) -> list[int]:
        cu = self.cu_seqlens.tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]

    def to(self, device) -> "Problem":
        def mv(x):
            return None if x is None else x.to(device)
        return dataclasses.replace(
            self, q=mv(self.q), k=mv(self.k), v=mv(self.v), g=mv(self.g),
            beta=mv(self.beta), initial_state=mv(self.initial_state),
            state_indices=mv(self.state_indices), cu_seqlens=mv(self.cu_seqlens))


def _cu(lengths: Sequence[int], dtype) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=dtype)


def _gates(kind: str, T: int, H: int, gen: torch.Generator, device):
    """Forget gate g (linear space) and update gate beta, fp32 ``[T, H]``."""
    if kind == "weak":            # g = exp(u), u ~ U(-0.1, 0); beta ~ U(0, 1)
        u = torch.rand(T, H, generator=gen, device=device) * -0.1
        g = torch.exp(u)
        beta = torch.rand(T, H, generator=gen, device=device)
    elif kind == "uniform":       # log g ~ U(-0.5, 0); beta = sigmoid(N(0, 1))
        lg = torch.rand(T, H, generator=gen, device=device) * -0.5
        g = torch.exp(lg)
        beta = torch.sigmoid(torch.randn(T, H, generator=gen, device=device))
    elif kind == "slow":          # log g ~ U(-0.001, 0), beta ~ U(0, 0.1): memory over thousands of tokens
        lg = torch.rand(T, H, generator=gen, device=device) * -0.001
        g = torch.exp(lg)
        beta = torch.rand(T, H, generator=gen, device=device) * 0.1
    elif kind == "mamba":         # g = exp(-exp(A_h) softplus(x)), A_h ~ U(-2, 1)
        A = torch.rand(H, generator=gen, device=device) * 3.0 - 2.0
        x = torch.randn(T, H, generator=gen, device=device)
        g = torch.exp(-torch.exp(A)[None, :] * torch.nn.functional.softplus(x))
        beta = torch.sigmoid(torch.randn(T, H, generator=gen, device=device))
    else:
        raise ValueError(f"unknown gate distribution {kind!r}")
    return g.float().contiguous(), beta.float().contiguous()


def make_problem(lengths: Sequence[int], H_qk: int, H_v: int, *, gates: str = "uniform",
                 use_qk_l2norm: bool = True, init: Optional[str] = "fp32",
                 init_std: float = 0.1, state_dtype: torch.dtype = torch.float32,
                 pool_slots: Optional[int] = None, cu_dtype=torch.int32,
                 idx_dtype=torch.int32, batch_invariant: bool = True,
                 output_final_state: bool = True, seed: int = 0,
                 device="cpu", name: str = "custom", with_g: bool = True,
                 with_beta: bool = True, scale: Optional[float] = None,
                 qkv_dtype: torch.dtype = torch.bfloat16) -> Problem:
    """A seeded varlen problem.

    ``init`` is ``None`` (no initial state), ``"fp32"`` or ``"bf16"``; with
    ``pool_slots`` the initial states form a pool of that many slots addressed
    through a unique random ``state_indices`` permutation.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    T = int(sum(lengths))
    N = len(lengths)
    H = max(H_qk, H_v)
    q = torch.randn(T, H_qk, HEAD_DIM, generator=gen, device=device).to(qkv_dtype)
    k = torch.randn(T, H_qk, HEAD_DIM, generator=gen, device=device).to(qkv_dtype)
    v = torch.randn(T, H_v, HEAD_DIM, generator=gen, device=device).to(qkv_dtype)
    g, beta = _gates(gates, T, H, gen, device)
    slots = N if pool_slots is None else int(pool_slots)
    init_state = None
    if init is not None:
        dt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[init]
        init_state = (torch.randn(slots, H, HEAD_DIM, HEAD_DIM, generator=gen, device=device)
                      * init_std).to(dt)
    state_indices = None
    if pool_slots is not None:
        state_indices = torch.randperm(slots, generator=gen, device=device)[:N].to(idx_dtype)
    return Problem(
        name=name, q=q, k=k, v=v, g=g if with_g else None, beta=beta if with_beta else None,
        scale=(1.0 / math.sqrt(HEAD_DIM)) if scale is None else float(scale),
        initial_state=init_state, state_indices=state_indices,
        cu_seqlens=_cu(lengths, cu_dtype).to(device), use_qk_l2norm=use_qk_l2norm,
        batch_invariant=batch_invariant, output_final_state=output_final_state,
        state_dtype=state_dtype, state_slots=slots, seed=seed)


def varlen_lengths(seed: int) -> list[int]:
    """Eight lengths: 1, 63, 64, 65 forced in plus four drawn from U[1, 2048], shuffled."""
    gen = torch.Generator()
    gen.manual_seed(seed)
    drawn = torch.randint(1, 2049, (4,), generator=gen).tolist()
    lens = [1, 63, 64, 65] + drawn
    perm = torch.randperm(8, generator=gen).tolist()
    return [lens[i] for i in perm]


def short_lengths(seed: int, n: int = 1024, lo: int = 16, hi: int = 256) -> list[int]:
    gen = torch.Generator()
    gen.manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


# The five prefill workloads.  Seeds are 1000 + workload number.
WORKLOADS = {
    1: "single sequence T=256, 1 q/k head, 1 v head, fp32 state, zero initial state",
    2: "8 varlen sequences (1, 63, 64, 65 + 4 x U[1,2048]), 4 q/k heads, 8 v heads, fp32 state",
    3: "16 x 4096 tokens, 16 q/k heads, 32 v heads, bf16 state (hybrid-LLM GDN layer prefill)",
    4: "2 x 65536 tokens, 16 q/k heads, 32 v heads, fp32 state",
    5: "1024 sequences of U[16,256] tokens, 8 q/k heads, 16 v heads, bf16 state pools of 4096 slots",
}


def make_workload(i: int, *, device="cpu", batch_invariant: Optional[bool] = None,
                  seqs: Optional[int] = None) -> Problem:
    """Workload ``i`` (1..5) with its seed.  ``seqs`` truncates the number of
    sequences (same distributions, fewer of them) for bounded CPU samples.

    ``batch_invariant`` is False, the API default of cudnn_chunk_gated_delta_rule, for
    every workload whose statement does not set it; workload 4 names both settings and
    is built with False (pass ``batch_invariant=True`` for its second run)."""
    seed = 1000 + i
    if i == 1:
        p = make_problem([256], 1, 1, gates="weak", init=None, state_dtype=torch.float32,
                         seed=seed, device=device, name="w1_single_256")
    elif i == 2:
        p = make_problem(varlen_lengths(seed), 4, 8, gates="uniform", init="fp32",
                         init_std=0.1, state_dtype=torch.float32, seed=seed,
                         device=device, name="w2_varlen8")
    elif i == 3:
        n = 16 if seqs is None else seqs
        p = make_problem([4096] * n, 16, 32, gates="mamba", init="bf16", init_std=0.05,
                         state_dtype=torch.bfloat16, seed=seed, device=device,
                         name="w3_16x4096_h16x32_bf16state")
    elif i == 4:
        n = 2 if seqs is None else seqs
        p = make_problem([65536] * n, 16, 32, gates="mamba", init="fp32", init_std=0.05,
                         state_dtype=torch.float32, seed=seed, device=device,
                         batch_invariant=False, name="w4_2x65536_h16x32_fp32state")
    elif i == 5:
        lens = short_lengths(seed)
        if seqs is not None:
            lens = lens[:seqs]
        p = make_problem(lens, 8, 16, gates="uniform", init="bf16", init_std=0.05,
                         state_dtype=torch.bfloat16, pool_slots=4096, cu_dtype=torch.int64,
                         idx_dtype=torch.int32, seed=seed, device=device,
                         name="w5_1024short_h8x16_pool4096")
    else:
        raise ValueError(f"workload {i} does not exist (1..5)")
    p.batch_invariant = False if batch_invariant is None else batch_invariant
    return p


def make_decode_workload(*, device="cpu", rows: int = 1024) -> Problem:
    """The decode batch that follows workload 5: ``rows`` sequences taking one token
    each, 8 q/k heads and 16 v heads, gates as in workload 2, the states a 4096-slot
    bf16 pool addressed through a unique int32 ``state_indices`` permutation."""
    return make_problem([1] * rows, 8, 16, gates="uniform", init="bf16", init_std=0.05,
                        state_dtype=torch.bfloat16, pool_slots=4096, idx_dtype=torch.int32,
                        seed=1006, device=device, name=f"decode_{rows}_h8x16_bf16pool4096")
