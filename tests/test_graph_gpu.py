"""CUDA-graph capture and replay of the entry points: a captured prefill (one pass, and
split-K after gdn_reserve_workspace) and a captured decode step, replayed on new input
values written into the captured buffers, match the fp64 oracle for those values."""
import dataclasses

import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import workloads as W
from tests.parity import compare

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


def _device_problem(p):
    to = lambda x: None if x is None else x.to(DEV)  # noqa: E731
    return dataclasses.replace(p, q=to(p.q), k=to(p.k), v=to(p.v), g=to(p.g), beta=to(p.beta),
                               initial_state=to(p.initial_state), state_indices=to(p.state_indices),
                               cu_seqlens=to(p.cu_seqlens))


def _load(dst, src):
    """Write problem ``src``'s input values into the captured buffers of ``dst``."""
    for name in ("q", "k", "v", "g", "beta", "initial_state"):
        getattr(dst, name).copy_(getattr(src, name))


def _capture_prefill(p_dev, out, st):
    gdn.run_problem(p_dev, device=DEV, output=out, output_state=st)  # warm-up: one-time set-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.run_problem(p_dev, device=DEV, output=out, output_state=st)
    return graph


@pytest.mark.parametrize("split", [1, 3])
def test_prefill_graph_replay(split, force_split):
    force_split(str(split))
    lens, hqk, hv = [700, 64, 0, 1300, 63], 2, 4
    mk = lambda seed: W.make_problem(lens, hqk, hv, gates="mamba", init="fp32", init_std=0.05,  # noqa: E731
                                     seed=seed, batch_invariant=(split == 1))
    p0 = mk(500 + split)
    if split > 1:
        gdn.gdn_reserve_workspace(gdn.gdn_split_workspace_bytes(p0.N, p0.H, 8))
    p_dev = _device_problem(p0)
    out = torch.empty(p0.T, p0.H, 128, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(p0.state_slots, p0.H, 128, 128, dtype=p0.state_dtype, device=DEV)
    graph = _capture_prefill(p_dev, out, st)
    for seed in (510 + split, 520 + split):
        p1 = mk(seed)
        _load(p_dev, _device_problem(p1))
        out.fill_(0)
        st.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        compare(p1, out, st)


def test_split_capture_without_reserve_is_refused(force_split):
    """Growing the split-K workspace inside a capture is refused before anything is
    enqueued; after a reserve the same capture succeeds."""
    force_split("3")
    gdn.binding.load_library().gdn_shutdown()  # drop the workspace earlier calls grew
    gdn.gdn_init(0)
    p = W.make_problem([700, 1300], 1, 2, gates="mamba", init=None, seed=530, batch_invariant=False)
    p_dev = _device_problem(p)
    out = torch.empty(p.T, p.H, 128, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(p.state_slots, p.H, 128, 128, device=DEV)
    graph = torch.cuda.CUDAGraph()
    with pytest.raises(gdn.GdnError, match="gdn_reserve_workspace"):
        with torch.cuda.graph(graph):
            gdn.run_problem(p_dev, device=DEV, output=out, output_state=st)
    torch.cuda.synchronize()
    gdn.gdn_reserve_workspace(gdn.gdn_split_workspace_bytes(p.N, p.H, 3))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.run_problem(p_dev, device=DEV, output=out, output_state=st)
    graph.replay()
    torch.cuda.synchronize()
    compare(p, out, st)


def test_decode_graph_replay():
    hqk, hv, B = 2, 4, 37
    mk = lambda seed: W.make_problem([1] * B, hqk, hv, gates="mamba", init="bf16", init_std=0.1,  # noqa: E731
                                     state_dtype=torch.bfloat16, pool_slots=50, seed=seed)
    p0 = mk(540)
    d = _device_problem(p0)
    pool = d.initial_state.clone()
    out = torch.empty(B, p0.H, 128, dtype=torch.bfloat16, device=DEV)

    def step():
        gdn.gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, d.scale, pool, d.state_indices,
                            d.use_qk_l2norm, out)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (541, 542):
        p1 = mk(seed)
        p1.state_indices = p0.state_indices  # the captured index buffer keeps its values
        d1 = _device_problem(p1)
        for name in ("q", "k", "v", "g", "beta"):
            getattr(d, name).copy_(getattr(d1, name))
        pool.copy_(d1.initial_state)
        graph.replay()
        torch.cuda.synchronize()
        compare(p1, out, pool)
