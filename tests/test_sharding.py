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
from gated_delta_rule_24_gb300.sharding import split_sequences


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
    shards = split_sequences(p.cu_seqlens.tolist(), world, p.state_indices.tolist())
    s = shards[rank]
    rows = slice(s.row_begin, s.row_end)
    o, st = oracle.recurrence(p.q[rows], p.k[rows], p.v[rows], p.g[rows], p.beta[rows], p.scale,
                              p.initial_state, torch.tensor(s.slots, dtype=torch.int64),
                              s.cu_local, p.use_qk_l2norm)
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
