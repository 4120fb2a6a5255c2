"""Shared comparison helpers for the GPU parity tests.

Tolerances (the fixed bar for this operation): bf16 output relative-L2 <= 5e-3
and max-abs <= 3e-2; fp32 final state relative-L2 <= 1e-3.  A bf16 final
state carries its own rounding (~1e-3 relative-L2 from storage alone), so it is
held to relative-L2 <= 5e-3; an fp16 one (~1.5e-4 from storage) to 2e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

OUT_REL_L2 = 5e-3
OUT_MAX_ABS = 3e-2
STATE_REL_L2 = {torch.float32: 1e-3, torch.bfloat16: 5e-3, torch.float16: 2e-3}


def rel_l2(a, b) -> float:
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / d) if d > 0 else float(np.linalg.norm(a - b))


def run_oracle(p, units=None):
    return oracle.recurrence(p.q, p.k, p.v, p.g, p.beta, p.scale, p.initial_state,
                             p.state_indices, p.cu_seqlens, p.use_qk_l2norm, units=units)


def compare(p, out, out_state, units=None, o_ref=None, s_ref=None):
    """Check GPU results of problem ``p`` against the oracle on ``units``
    (all units if None).  Outputs are held to the bars over all compared rows; the
    final state of every (sequence, head) unit is held to its bar on its own, so
    one bad unit cannot hide among good ones.  Returns a dict of the measured errors
    (state_rel_l2 is the worst unit, state_rel_l2_all the pooled value)."""
    if o_ref is None:
        o_ref, s_ref = run_oracle(p, units)
    o = out.float().cpu().numpy()
    mask = ~np.isnan(o_ref)
    res = {}
    if mask.any():
        res["out_rel_l2"] = rel_l2(o[mask], o_ref[mask])
        res["out_max_abs"] = float(np.abs(o[mask] - o_ref[mask]).max())
        assert res["out_rel_l2"] <= OUT_REL_L2, res
        assert res["out_max_abs"] <= OUT_MAX_ABS, res
    if out_state is not None:
        st = out_state.float().cpu()
        idx = p.state_indices.tolist() if p.state_indices is not None else list(range(p.N))
        if units is None:
            units = [(n, h) for n in range(p.N) for h in range(p.H)]
        got = np.stack([st[idx[n], h].numpy() for n, h in units])
        want = np.stack([s_ref[n, h] for n, h in units])
        per_unit = [rel_l2(gu, wu) for gu, wu in zip(got, want)]
        worst = int(np.argmax(per_unit))
        res["state_rel_l2"] = per_unit[worst]
        res["state_worst_unit"] = tuple(units[worst])
        res["state_rel_l2_all"] = rel_l2(got, want)
        res["state_max_abs"] = float(np.abs(got - want).max())
        assert res["state_rel_l2"] <= STATE_REL_L2[out_state.dtype], res
    return res
