"""Thin ctypes binding of the C ABI in ``include/gdn.h``.

Only argument marshalling happens here: torch tensors are described to the
library (pointer, dtype, shape, strides) and every step of the computation runs
in the library's CUDA kernels.  There is no fallback: if the compiled library
is missing, or the GPU is not an sm_103 part, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB as _LIB_PATH

GDN_OK = 0
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARGUMENT", 2: "GDN_ERR_UNSUPPORTED",
                3: "GDN_ERR_ALIAS", 4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE_INPUT"}
DEVERR_CU_SEQLENS, DEVERR_STATE_INDEX, DEVERR_TIMEOUT = 0x1, 0x2, 0x4
_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.int32: 3, torch.int64: 4}
# symbols include/gdn.h declares; the tests check the library exports all of them
EXPORTED = ["gdn_init", "gdn_chunk_prefill", "gdn_chunk_prefill_checkpointed", "gdn_chunk_prefill_noalloc",
            "gdn_decode_step", "gdn_reserve_workspace", "gdn_split_workspace_bytes",
            "gdn_get_device_status", "gdn_last_error", "gdn_shutdown", "gdn_testing_force_splits",
            "gdn_testing_wait_limit", "gdn_testing_split_plan"]


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class GdnTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -m gated_delta_rule_24_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER(GdnTensor)
        lib.gdn_init.argtypes = [ctypes.c_int]
        lib.gdn_init.restype = ctypes.c_int
        lib.gdn_chunk_prefill.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, P, P, ctypes.c_int,
                                          ctypes.c_int, P, ctypes.c_void_p]
        lib.gdn_chunk_prefill.restype = ctypes.c_int
        lib.gdn_chunk_prefill_noalloc.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, P, P, ctypes.c_int,
                                                  ctypes.c_int, P, ctypes.c_void_p, ctypes.c_void_p]
        lib.gdn_chunk_prefill_noalloc.restype = ctypes.c_int
        lib.gdn_chunk_prefill_checkpointed.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, P, P, ctypes.c_int,
                                                       ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int,
                                                       ctypes.c_void_p]
        lib.gdn_chunk_prefill_checkpointed.restype = ctypes.c_int
        lib.gdn_reserve_workspace.argtypes = [ctypes.c_size_t, ctypes.c_void_p]
        lib.gdn_reserve_workspace.restype = ctypes.c_int
        lib.gdn_split_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
        lib.gdn_split_workspace_bytes.restype = ctypes.c_size_t
        lib.gdn_decode_step.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, ctypes.c_int, P, ctypes.c_void_p]
        lib.gdn_decode_step.restype = ctypes.c_int
        lib.gdn_get_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
        lib.gdn_get_device_status.restype = ctypes.c_int
        lib.gdn_last_error.argtypes = []
        lib.gdn_last_error.restype = ctypes.c_char_p
        lib.gdn_shutdown.argtypes = []
        lib.gdn_shutdown.restype = None
        lib.gdn_testing_force_splits.argtypes = [ctypes.c_int]
        lib.gdn_testing_force_splits.restype = ctypes.c_int
        lib.gdn_testing_wait_limit.argtypes = [ctypes.c_uint64, ctypes.c_int]
        lib.gdn_testing_wait_limit.restype = ctypes.c_int
        lib.gdn_testing_split_plan.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.gdn_testing_split_plan.restype = ctypes.c_int
        _lib = lib
    return _lib


def describe(t: Optional[torch.Tensor]):
    """A GdnTensor describing ``t`` (None -> a null pointer)."""
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError("at most 4 dims")
    d = GdnTensor()
    d.data = t.data_ptr() if t.numel() > 0 else (t.data_ptr() or None)
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _check(status: int):
    if status != GDN_OK:
        msg = load_library().gdn_last_error().decode(errors="replace")
        raise GdnError(status, msg)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def gdn_init(device: int = 0) -> None:
    _check(load_library().gdn_init(int(device)))


def gdn_chunk_prefill(q, k, v, g, beta, scale: float, initial_state, state_indices, output_state,
                      cu_seqlens, use_qk_l2norm: bool, batch_invariant: bool, output,
                      stream=None) -> None:
    """Same names and order as the C entry point; raises GdnError on a non-OK status."""
    lib = load_library()
    descs = [describe(x) for x in (q, k, v, g, beta)]
    s_in, idx, s_out, cu, out = (describe(x) for x in (initial_state, state_indices, output_state,
                                                      cu_seqlens, output))
    st = lib.gdn_chunk_prefill(_ref(descs[0]), _ref(descs[1]), _ref(descs[2]), _ref(descs[3]),
                               _ref(descs[4]), ctypes.c_float(float(scale)), _ref(s_in), _ref(idx),
                               _ref(s_out), _ref(cu), int(bool(use_qk_l2norm)),
                               int(bool(batch_invariant)), _ref(out),
                               ctypes.c_void_p(_stream_handle(stream)))
    _check(st)


def gdn_chunk_prefill_noalloc(q, k, v, g, beta, scale: float, initial_state, state_indices,
                              output_state, cu_seqlens, use_qk_l2norm: bool, batch_invariant: bool,
                              output, device_error=None, stream=None) -> None:
    """The allocation-free entry point: same names and order as the C function
    (``device_error`` is an optional int32 device tensor of one element)."""
    lib = load_library()
    descs = [describe(x) for x in (q, k, v, g, beta)]
    s_in, idx, s_out, cu, out = (describe(x) for x in (initial_state, state_indices, output_state,
                                                      cu_seqlens, output))
    err_ptr = None
    if device_error is not None:
        if device_error.dtype != torch.int32 or device_error.numel() < 1 or not device_error.is_cuda:
            raise ValueError("device_error must be an int32 CUDA tensor")
        err_ptr = device_error.data_ptr()
    st = lib.gdn_chunk_prefill_noalloc(_ref(descs[0]), _ref(descs[1]), _ref(descs[2]), _ref(descs[3]),
                                       _ref(descs[4]), ctypes.c_float(float(scale)), _ref(s_in),
                                       _ref(idx), _ref(s_out), _ref(cu), int(bool(use_qk_l2norm)),
                                       int(bool(batch_invariant)), _ref(out), ctypes.c_void_p(err_ptr),
                                       ctypes.c_void_p(_stream_handle(stream)))
    _check(st)


def gdn_chunk_prefill_checkpointed(q, k, v, g, beta, scale: float, initial_state, state_indices,
                                   output_state, cu_seqlens, use_qk_l2norm: bool, batch_invariant: bool,
                                   output, checkpoints, checkpoints_per_seq: int, checkpoint_every: int,
                                   stream=None) -> None:
    """Prefill that also writes f32 state checkpoints every ``checkpoint_every`` chunks;
    same names and order as the C entry point."""
    lib = load_library()
    d = [describe(x) for x in (q, k, v, g, beta, initial_state, state_indices, output_state, cu_seqlens,
                               output, checkpoints)]
    st = lib.gdn_chunk_prefill_checkpointed(
        _ref(d[0]), _ref(d[1]), _ref(d[2]), _ref(d[3]), _ref(d[4]), ctypes.c_float(float(scale)),
        _ref(d[5]), _ref(d[6]), _ref(d[7]), _ref(d[8]), int(bool(use_qk_l2norm)), int(bool(batch_invariant)),
        _ref(d[9]), _ref(d[10]), int(checkpoints_per_seq), int(checkpoint_every),
        ctypes.c_void_p(_stream_handle(stream)))
    _check(st)


def gdn_decode_step(q, k, v, g, beta, scale: float, state, state_indices, use_qk_l2norm: bool, output,
                    stream=None) -> None:
    """One decode token per batch row, updating ``state`` in place; same names and order
    as the C entry point."""
    lib = load_library()
    d = [describe(x) for x in (q, k, v, g, beta, state, state_indices, output)]
    st = lib.gdn_decode_step(_ref(d[0]), _ref(d[1]), _ref(d[2]), _ref(d[3]), _ref(d[4]),
                             ctypes.c_float(float(scale)), _ref(d[5]), _ref(d[6]),
                             int(bool(use_qk_l2norm)), _ref(d[7]), ctypes.c_void_p(_stream_handle(stream)))
    _check(st)


def gdn_reserve_workspace(nbytes: int, stream=None) -> None:
    """Grow the split-K workspace now (e.g. before capturing a CUDA graph)."""
    _check(load_library().gdn_reserve_workspace(ctypes.c_size_t(int(nbytes)),
                                                ctypes.c_void_p(_stream_handle(stream))))


def gdn_split_workspace_bytes(num_seqs: int, num_sab_heads: int, splits: int) -> int:
    """Workspace bytes of a split-K call with ``splits`` segments per sequence."""
    return int(load_library().gdn_split_workspace_bytes(int(num_seqs), int(num_sab_heads), int(splits)))


def testing_force_splits(splits: int) -> None:
    """Testing aid: force ``splits`` segments per sequence for this thread's later
    calls with batch_invariant=False (0 restores the planner)."""
    _check(load_library().gdn_testing_force_splits(int(splits)))


def testing_wait_limit(limit_ns: int, withhold_local_ready: bool = False) -> None:
    """Testing aid: bound the prefill kernel's hand-off waits by ``limit_ns`` (0: the
    default) and optionally withhold one hand-off so that a wait runs out."""
    _check(load_library().gdn_testing_wait_limit(int(limit_ns), int(bool(withhold_local_ready))))


def testing_split_plan(num_seqs: int, num_sab_heads: int, total_tokens: int, num_sms: int) -> dict:
    """Testing aid (host only): the split-K plan a batch_invariant=False call would take.
    Returns P, the segment bounds (numerators over ``den``) and, per pass, the grid and
    for every unit index its (sequence * heads + head, kind) pair, (-1, -1) when idle."""
    lib = load_library()
    plan = (ctypes.c_int32 * 16)()
    cap = 3 * int(num_sms) + 16 * int(num_seqs) * int(num_sab_heads) + 64
    units = (ctypes.c_int32 * (2 * cap * 2))()
    _check(lib.gdn_testing_split_plan(int(num_seqs), int(num_sab_heads), int(total_tokens), int(num_sms),
                                      ctypes.cast(plan, ctypes.c_void_p), ctypes.cast(units, ctypes.c_void_p), cap))
    P, den = plan[0], plan[1]
    res = {"P": P, "den": den, "num": list(plan[2:3 + P]), "grid": [plan[11], plan[12]],
           "units": [[], []]}
    for ps in range(2 if P > 1 else 0):
        n = plan[13 + ps]
        base = ps * cap * 2
        res["units"][ps] = [(units[base + 2 * u], units[base + 2 * u + 1]) for u in range(n)]
    return res


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error bits."""
    lib = load_library()
    word = ctypes.c_int32(0)
    st = lib.gdn_get_device_status(ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(word))
    if st not in (GDN_OK, 5):
        _check(st)
    return int(word.value)


def chunk_gated_delta_rule(q, k, v, g=None, beta=None, scale: Optional[float] = None,
                           initial_state=None, output_final_state: bool = False,
                           cu_seqlens=None, use_qk_l2norm_in_kernel: bool = False, output=None,
                           output_state=None, batch_invariant: bool = False,
                           state_indices=None, stream=None):
    """Chunked Gated Delta Rule prefill with the argument meanings of
    ``flashinfer.cudnn.cudnn_chunk_gated_delta_rule`` (plus ``state_indices``).

    Returns ``output``, or ``(output, final_state)`` when ``output_final_state``.
    With ``output_final_state`` unset no state is written at all (``output_state``
    is then ignored).  A state buffer the call allocates has the initial state's
    dtype, or fp32 without an initial state, and one slot per sequence (or the
    initial pool's slot count when ``state_indices`` addresses a pool).
    """
    if cu_seqlens is None:
        raise ValueError("cu_seqlens is required")
    T = q.shape[0]
    H = max(q.shape[1], v.shape[1])
    N = cu_seqlens.shape[0] - 1
    if output is None:
        output = torch.empty(T, H, q.shape[2], dtype=q.dtype, device=q.device)
    final_state = None
    if output_final_state:
        if output_state is None:
            slots = initial_state.shape[0] if (state_indices is not None and initial_state is not None) else N
            dt = initial_state.dtype if initial_state is not None else torch.float32
            output_state = torch.empty(slots, H, v.shape[2], q.shape[2], dtype=dt, device=q.device)
        final_state = output_state
    gdn_chunk_prefill(q, k, v, g, beta, 0.0 if scale is None else float(scale), initial_state,
                      state_indices, final_state, cu_seqlens, use_qk_l2norm_in_kernel,
                      batch_invariant, output, stream)
    return (output, final_state) if output_final_state else output


def run_problem(p, device="cuda", output_state=None, output=None, stream=None):
    """Run a :class:`workloads.Problem` (tensors already on ``device`` or moved
    there).  Returns (output, output_state or None)."""
    dev = torch.device(device)
    q, k, v = (x.to(dev) for x in (p.q, p.k, p.v))
    g = None if p.g is None else p.g.to(dev)
    beta = None if p.beta is None else p.beta.to(dev)
    s0 = None if p.initial_state is None else p.initial_state.to(dev)
    idx = None if p.state_indices is None else p.state_indices.to(dev)
    cu = p.cu_seqlens.to(dev)
    if output is None:
        output = torch.empty(p.T, p.H, 128, dtype=p.q.dtype, device=dev)
    if p.output_final_state and output_state is None:
        output_state = torch.zeros(p.state_slots, p.H, 128, 128, dtype=p.state_dtype, device=dev)
    gdn_chunk_prefill(q, k, v, g, beta, p.scale, s0, idx,
                      output_state if p.output_final_state else None, cu, p.use_qk_l2norm,
                      p.batch_invariant, output, stream)
    return output, (output_state if p.output_final_state else None)
