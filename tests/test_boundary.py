"""Host-side tests of the C ABI: the library loads, exports every symbol
include/gdn.h declares, and rejects bad arguments with the documented status
before touching any GPU (these run on a machine without one)."""
import os
import re

import pytest
import torch

import gated_delta_rule_24_gb300 as gdn
from gated_delta_rule_24_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load_library()


def test_exports_every_declared_symbol(lib):
    header = open(os.path.join(ROOT, "include", "gdn.h")).read()
    declared = set(re.findall(r"^\s*(?:gdn_status_t|const char\*|void|size_t)\s+(gdn_\w+)\s*\(",
                              header, flags=re.M))
    assert declared, "no declarations found"
    assert declared == set(binding.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_last_error_initially_empty(lib):
    assert lib.gdn_last_error() in (b"", None) or isinstance(lib.gdn_last_error(), bytes)


def _args(T=10, Hqk=2, Hv=4, N=2):
    q = torch.zeros(T, Hqk, 128, dtype=torch.bfloat16)
    k = torch.zeros(T, Hqk, 128, dtype=torch.bfloat16)
    v = torch.zeros(T, Hv, 128, dtype=torch.bfloat16)
    H = max(Hqk, Hv)
    return dict(q=q, k=k, v=v, g=torch.ones(T, H), beta=torch.ones(T, H), scale=0.0,
                initial_state=torch.zeros(N, H, 128, 128), state_indices=None,
                output_state=torch.zeros(N, H, 128, 128),
                cu_seqlens=torch.tensor([0, 4, T], dtype=torch.int32), use_qk_l2norm=True,
                batch_invariant=True, output=torch.empty(T, H, 128, dtype=torch.bfloat16))


def _status(**kw):
    a = _args()
    a.update(kw)
    try:
        gdn.gdn_chunk_prefill(**a, stream=0)
    except binding.GdnError as e:
        return e.status, str(e)
    return 0, ""


INVALID, UNSUPPORTED, ALIAS, CUDA = 1, 2, 3, 4
BF = torch.bfloat16

CASES = {
    "q_fp32": (dict(q=torch.zeros(10, 2, 128)), UNSUPPORTED),
    "head_dim_64": (dict(q=torch.zeros(10, 2, 64, dtype=BF), k=torch.zeros(10, 2, 64, dtype=BF)),
                    UNSUPPORTED),
    "hq_ne_hk": (dict(k=torch.zeros(10, 1, 128, dtype=BF)), UNSUPPORTED),
    "heads_not_multiple": (dict(v=torch.zeros(10, 3, 128, dtype=BF)), UNSUPPORTED),
    "v_token_count": (dict(v=torch.zeros(9, 4, 128, dtype=BF)), INVALID),
    "g_shape": (dict(g=torch.ones(10, 3)), INVALID),
    "beta_i32": (dict(beta=torch.ones(10, 4, dtype=torch.int32)), UNSUPPORTED),
    "qkv_mixed_dtypes": (dict(q=torch.zeros(10, 2, 128, dtype=torch.float16)), UNSUPPORTED),
    "output_not_q_dtype": (dict(output=torch.empty(10, 4, 128, dtype=torch.float16)), UNSUPPORTED),
    "state_shape": (dict(initial_state=torch.zeros(2, 4, 64, 128)), INVALID),
    "state_i32": (dict(initial_state=torch.zeros(2, 4, 128, 128, dtype=torch.int32)), UNSUPPORTED),
    "state_k_major": (dict(initial_state=torch.zeros(2, 4, 128, 128).transpose(2, 3)), INVALID),
    "too_few_slots": (dict(initial_state=torch.zeros(1, 4, 128, 128)), INVALID),
    "cu_float": (dict(cu_seqlens=torch.tensor([0.0, 4.0, 10.0])), UNSUPPORTED),
    "cu_empty": (dict(cu_seqlens=torch.zeros(0, dtype=torch.int32)), INVALID),
    "indices_length": (dict(state_indices=torch.tensor([0, 1, 2], dtype=torch.int32)), INVALID),
    "output_fp32": (dict(output=torch.empty(10, 4, 128)), UNSUPPORTED),
    "output_heads": (dict(output=torch.empty(10, 2, 128, dtype=BF)), INVALID),
    "scale_inf": (dict(scale=float("inf")), INVALID),
    "scale_nan": (dict(scale=float("nan")), INVALID),
    "misaligned_q": (dict(q=torch.zeros(10 * 260 + 4, dtype=BF).as_strided((10, 2, 128), (260, 128, 1), 4),
                          k=torch.zeros(10, 2, 128, dtype=BF)), INVALID),
    "same_state_buffer": (dict(initial_state=torch.zeros(2, 4, 128, 128)), None),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_validation_status(lib, name):
    case, expect = CASES[name]
    if name == "same_state_buffer":
        s = case["initial_state"]
        st, msg = _status(initial_state=s, output_state=s)
        assert st == ALIAS, msg
        pool = torch.zeros(4, 4, 128, 128)
        st, msg = _status(initial_state=pool[:2], output_state=pool[1:3])  # partial overlap
        assert st == ALIAS, msg
        return
    st, msg = _status(**case)
    assert st == expect, msg
    assert msg


def test_output_aliasing_an_input_rejected(lib):
    v = torch.zeros(10, 4, 128, dtype=BF)
    st, msg = _status(v=v, output=v)
    assert st == ALIAS, msg


def test_unknown_dtype_refused_by_binding(lib):
    with pytest.raises(TypeError):
        _status(g=torch.ones(10, 4, dtype=torch.float64))


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    st, msg = _status()
    assert st == CUDA, msg
    # strided views of a fused buffer pass validation and also stop at the device
    fused = torch.zeros(10, 2 * 256, dtype=BF)
    q = fused[:, :256].view(10, 2, 128)
    k = fused[:, 256:].view(10, 2, 128)
    st, msg = _status(q=q, k=k)
    assert st == CUDA, msg


def test_python_api_signature():
    import inspect
    names = list(inspect.signature(gdn.chunk_gated_delta_rule).parameters)
    assert names[:13] == ["q", "k", "v", "g", "beta", "scale", "initial_state", "output_final_state",
                          "cu_seqlens", "use_qk_l2norm_in_kernel", "output", "output_state",
                          "batch_invariant"]


def _decode_args(B=3, Hqk=2, Hv=4, slots=5):
    H = max(Hqk, Hv)
    return dict(q=torch.zeros(B, Hqk, 128, dtype=BF), k=torch.zeros(B, Hqk, 128, dtype=BF),
                v=torch.zeros(B, Hv, 128, dtype=BF), g=torch.ones(B, H), beta=torch.ones(B, H),
                scale=0.0, state=torch.zeros(slots, H, 128, 128),
                state_indices=torch.tensor([4, 0, 2], dtype=torch.int32), use_qk_l2norm=True,
                output=torch.empty(B, H, 128, dtype=BF))


def _decode_status(**kw):
    a = _decode_args()
    a.update(kw)
    try:
        gdn.gdn_decode_step(**a, stream=0)
    except binding.GdnError as e:
        return e.status, str(e)
    return 0, ""


DECODE_CASES = {
    "no_state": (dict(state=None), INVALID),
    "state_i32": (dict(state=torch.zeros(5, 4, 128, 128, dtype=torch.int32)), UNSUPPORTED),
    "qkv_mixed_dtypes": (dict(v=torch.zeros(3, 4, 128, dtype=torch.float16)), UNSUPPORTED),
    "state_heads": (dict(state=torch.zeros(5, 2, 128, 128)), INVALID),
    "indices_length": (dict(state_indices=torch.tensor([0, 1], dtype=torch.int32)), INVALID),
    "too_few_slots": (dict(state=torch.zeros(2, 4, 128, 128), state_indices=None), INVALID),
    "g_rows": (dict(g=torch.ones(2, 4)), INVALID),
    "v_rows": (dict(v=torch.zeros(2, 4, 128, dtype=BF)), INVALID),
    "output_fp32": (dict(output=torch.empty(3, 4, 128)), UNSUPPORTED),
    "scale_inf": (dict(scale=float("inf")), INVALID),
}


@pytest.mark.parametrize("name", sorted(DECODE_CASES))
def test_decode_validation_status(lib, name):
    case, expect = DECODE_CASES[name]
    st, msg = _decode_status(**case)
    assert st == expect, msg
    assert msg


def test_decode_state_aliasing_rejected(lib):
    out = torch.empty(3, 4, 128, dtype=BF)
    st, msg = _decode_status(v=out, output=out)
    assert st == ALIAS, msg
    pool = torch.zeros(5 * 4 * 128 * 128)
    st, msg = _decode_status(state=pool.view(5, 4, 128, 128), g=pool[:12].view(3, 4))
    assert st == ALIAS, msg


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_decode_valid_call_without_gpu_reports_cuda_error(lib):
    st, msg = _decode_status()
    assert st == CUDA, msg


def _ck_status(ck, M=2, every=1, **kw):
    a = _args()
    a.update(kw)
    try:
        gdn.gdn_chunk_prefill_checkpointed(**a, checkpoints=ck, checkpoints_per_seq=M, checkpoint_every=every,
                                           stream=0)
    except binding.GdnError as e:
        return e.status, str(e)
    return 0, ""


def test_checkpoint_validation(lib):
    ok = torch.zeros(2 * 2, 4, 128, 128)
    assert _ck_status(ok, every=0)[0] == INVALID
    assert _ck_status(ok, M=3)[0] == INVALID  # N * M rows
    assert _ck_status(ok, M=0)[0] == INVALID
    assert _ck_status(torch.zeros(4, 4, 128, 128, dtype=torch.bfloat16))[0] == UNSUPPORTED
    assert _ck_status(torch.zeros(4, 2, 128, 128))[0] == INVALID  # heads
    assert _ck_status(torch.zeros(4, 4, 128, 128).transpose(2, 3))[0] == INVALID
    st, msg = _ck_status(None)
    assert st == INVALID and "checkpoints" in msg
    pool = torch.zeros(8, 4, 128, 128)
    st, msg = _ck_status(pool[:4], output_state=pool[2:4])
    assert st == ALIAS, msg


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_checkpointed_valid_call_without_gpu_reports_cuda_error(lib):
    assert _ck_status(torch.zeros(4, 4, 128, 128))[0] == CUDA


def test_split_workspace_bytes():
    """N * H * (3P - 5) blocks of 64 KiB for P segments; nothing without a split."""
    assert gdn.gdn_split_workspace_bytes(5, 4, 1) == 0
    assert gdn.gdn_split_workspace_bytes(0, 4, 8) == 0
    assert gdn.gdn_split_workspace_bytes(5, 4, 2) == 5 * 4 * 1 * 65536
    assert gdn.gdn_split_workspace_bytes(5, 4, 3) == 5 * 4 * 4 * 65536
    assert gdn.gdn_split_workspace_bytes(64, 16, 8) == 64 * 16 * 19 * 65536
