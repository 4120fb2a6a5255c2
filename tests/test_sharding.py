"""Sequence sharding across ranks: host logic, checked with world-size-2 gloo ranks
on CPU (each rank runs its shard through the CPU oracle; rank 0 reassembles and
compares with the unsharded batch)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from gated_delta_rule_24_gb300 import workloads as W
from gated_delta_rule_24_gb300.sharding import shard_problem, split_sequences


def test_split_covers_every_sequence_once():
    for lengths in ([5, 0, 7, 100, 1, 1, 64], [3], [0, 0], [10] * 9):
        cu = np.concatenate([[0], np.cumsum(lengths)]).tolist()
        for world in (1, 2, 3, 8):
            sh = split_sequences(cu, world)
            assert len(sh) == world
            seqs = [i for s in sh for i in range(s.seq_begin, s.seq_end)]
            assert seqs == list(range(len(lengths)))
            for s in sh:
                assert s.row_end - s.row_begin == sum(lengths[s.seq_begin:s.seq_end])
                assert s.cu_local[-1] == s.row_end - s.row_begin
                assert s.slots == list(range(s.seq_begin, s.seq_end))


def test_split_balances_tokens():
    lengths = W.short_lengths(5, n=1024)
    cu = np.concatenate([[0], np.cumsum(lengths)]).tolist()
    sh = split_sequences(cu, 4)
    tok = [s.row_end - s.row_begin for s in sh]
    assert max(tok) - min(tok) <= 2 * max(lengths)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    p = W.make_problem([70, 3, 130, 0, 64, 20], 1, 2, init="fp32", pool_slots=9, seed=91)
    s, sub = shard_problem(p, world, rank)
    rows = slice(s.row_begin, s.row_end)
    # the shard as a call of its own, in the library's argument contract: its rows, its
    # cu_seqlens from 0, the global slots of its sequences into the unchanged pools
    assert sub.cu_seqlens.tolist() == s.cu_local and sub.cu_seqlens[0] == 0
    assert sub.cu_seqlens.dtype == p.cu_seqlens.dtype
    assert sub.state_indices.tolist() == p.state_indices[s.seq_begin:s.seq_end].tolist()
    assert sub.state_indices.dtype == p.state_indices.dtype
    assert sub.initial_state is p.initial_state and sub.state_slots == p.state_slots
    assert torch.equal(sub.q, p.q[rows]) and torch.equal(sub.beta, p.beta[rows]) and sub.T == s.row_end - s.row_begin
    o, st = oracle.recurrence(sub.q, sub.k, sub.v, sub.g, sub.beta, sub.scale, sub.initial_state,
                              sub.state_indices, sub.cu_seqlens, sub.use_qk_l2norm)
    # gather (padded) outputs and states to every rank
    T, H = p.T, p.H
    full_o = torch.zeros(T, H, 128, dtype=torch.float64)
    full_o[rows] = torch.from_numpy(o)
    full_s = torch.zeros(p.N, H, 128, 128, dtype=torch.float64)
    full_s[s.seq_begin:s.seq_end] = torch.from_numpy(st)
    dist.all_reduce(full_o)
    dist.all_reduce(full_s)
    if rank == 0:
        o_ref, s_ref = oracle.recurrence(p.q, p.k, p.v, p.g, p.beta, p.scale, p.initial_state,
                                         p.state_indices, p.cu_seqlens, p.use_qk_l2norm)
        ok = np.array_equal(full_o.numpy(), o_ref) and np.array_equal(full_s.numpy(), s_ref)
        with open(result_path, "w") as f:
            f.write("ok" if ok else "mismatch")
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gloo_sharded_batch_equals_whole(tmp_path, oracle_lib):
    path = str(tmp_path / "result.txt")
    mp.spawn(_worker, args=(2, _free_port(), path), nprocs=2, join=True)
    assert open(path).read() == "ok"
