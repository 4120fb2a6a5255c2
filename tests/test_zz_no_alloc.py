"""The allocation-free entry point (gdn_chunk_prefill_noalloc) against the
regular one.  Collected last (file name), so it also runs after every other GPU
test has used the regular entry point and its allocations on the same device.
"""
import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import OUT_MAX_ABS, OUT_REL_L2, STATE_REL_L2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gated_delta_rule_24_gb300 import build
    build.build()
    gdn.gdn_init(0)
    yield


def _rel_l2(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


def _args(p):
    dev = torch.device(DEV)
    q, k, v = (x.to(dev) for x in (p.q, p.k, p.v))
    g = None if p.g is None else p.g.to(dev)
    beta = None if p.beta is None else p.beta.to(dev)
    s0 = None if p.initial_state is None else p.initial_state.to(dev)
    idx = None if p.state_indices is None else p.state_indices.to(dev)
    return q, k, v, g, beta, s0, idx, p.cu_seqlens.to(dev)


def _call(fn, p, a, **kw):
    q, k, v, g, beta, s0, idx, cu = a
    out = torch.empty(p.T, p.H, 128, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(p.state_slots, p.H, 128, 128, dtype=p.state_dtype, device=DEV)
    fn(q, k, v, g, beta, p.scale, s0, idx, st, cu, p.use_qk_l2norm, p.batch_invariant, out, **kw)
    return out, st


def _close(out, st, out_ref, st_ref):
    d = (out.float() - out_ref.float()).abs().max().item()
    assert _rel_l2(out.float(), out_ref.float()) <= OUT_REL_L2 and d <= OUT_MAX_ABS
    assert _rel_l2(st.float(), st_ref.float()) <= STATE_REL_L2[st.dtype]


@pytest.mark.parametrize("case", ["split", "invariant"])
def test_two_calls_match_the_regular_entry(force_split, case):
    if case == "split":  # split-K: the static scratch carries the segment maps
        force_split("4")
        p = W.make_problem([700, 65, 1300, 0, 257], 2, 4, gates="mamba", init="fp32",
                           init_std=0.05, seed=120, batch_invariant=False)
    else:  # bf16 pools through int32 state_indices, int64 cu_seqlens
        lengths = [16 + (37 * n) % 241 for n in range(40)]
        p = W.make_problem(lengths, 8, 16, gates="uniform", init="bf16", init_std=0.05,
                           state_dtype=torch.bfloat16, pool_slots=96, cu_dtype=torch.int64, seed=119)
    a = _args(p)
    out_ref, st_ref = _call(gdn.gdn_chunk_prefill, p, a)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        out, st = _call(gdn.gdn_chunk_prefill_noalloc, p, a, device_error=err)
        torch.cuda.synchronize()
        _close(out, st, out_ref, st_ref)
    assert int(err.item()) == 0
    assert gdn.device_status() == 0


def test_device_errors_reach_the_callers_word():
    p = W.make_problem([40, 40, 40], 1, 2, seed=121)
    p.cu_seqlens = torch.tensor([0, 40, 30, 120], dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    _call(gdn.gdn_chunk_prefill_noalloc, p, _args(p), device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & gdn.binding.DEVERR_CU_SEQLENS
    # without a caller word the bits are dropped; the call still runs
    _call(gdn.gdn_chunk_prefill_noalloc, p, _args(p))
    torch.cuda.synchronize()


def test_split_beyond_the_static_scratch_is_rejected(force_split):
    """64 sequences x 8 heads at P = 8 need 608 MiB of maps: refused on the host."""
    force_split("8")
    p = W.make_problem([16] * 64, 4, 8, seed=122, batch_invariant=False)
    with pytest.raises(gdn.GdnError) as ei:
        _call(gdn.gdn_chunk_prefill_noalloc, p, _args(p))
    assert ei.value.status == 2 and "static scratch" in str(ei.value)


def test_entries_work_again_after_shutdown(force_split):
    """gdn_shutdown drops every per-device resource and cached setting; the next calls
    set them up again: the regular entry (split-K, so its workspace is grown anew) and the
    allocation-free one give bit-identical results to their calls from before."""
    force_split("3")
    p = W.make_problem([700, 65, 1300], 2, 4, gates="slow", init="fp32", init_std=0.05, seed=123,
                       batch_invariant=False)
    a = _args(p)
    out0, st0 = _call(gdn.gdn_chunk_prefill, p, a)
    out1, st1 = _call(gdn.gdn_chunk_prefill_noalloc, p, a)
    torch.cuda.synchronize()
    gdn.binding.load_library().gdn_shutdown()
    gdn.gdn_init(0)
    out2, st2 = _call(gdn.gdn_chunk_prefill, p, a)
    out3, st3 = _call(gdn.gdn_chunk_prefill_noalloc, p, a)
    torch.cuda.synchronize()
    assert torch.equal(out0, out2) and torch.equal(st0, st2)
    assert torch.equal(out1, out3) and torch.equal(st1, st3)
    assert gdn.device_status() == 0
