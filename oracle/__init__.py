"""CPU oracle for chunked Gated Delta Rule prefill.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The library never imports
this package, and this package imports nothing from the library.

Two independent implementations of the same definition:

* :func:`recurrence` -- the fp64 token-by-token recurrence (plain C in
  ``gdn_recurrence.c``, threaded over (sequence, head) units).  This is the
  definition the CUDA path is judged against.
* :func:`chunked` (``chunked.py``) -- the chunked WY/UT form in numpy fp64,
  cross-checked against the recurrence by the tests.

Semantics follow "flashinfer.cudnn.cudnn_chunk_gated_delta_rule", Parameters:
q/k ``[T, H_qk, D]``, v ``[T, H_v, D]``, g/beta ``[T, H]`` (all ones when
absent), scale (``1/sqrt(D)`` when absent or 0), initial_state
``[slots, H, Dv, Dk]`` V-major (zero when absent), cu_seqlens ``[N+1]``.
Readings where the pages are silent:

* H = max(H_qk, H_v) sab heads; sab head h reads q/k head ``h // (H // H_qk)``
  and v head ``h // (H // H_v)`` (consecutive grouping);
* L2 normalisation is ``x / sqrt(sum(x^2) + 1e-6)``, applied to q and k
  before the recurrence; the scale multiplies ``S_t q_t``;
* with ``state_indices`` both the initial and the final state of sequence n
  live in slot ``state_indices[n]`` of their pools; without it, slot n;
* an empty sequence writes no output rows and its final state is its initial
  state.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Iterable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_recurrence.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
L2NORM_EPS = 1e-6
_lib = None


def build(force: bool = False) -> str:
    """Compile the C recurrence with gcc into ``oracle/_build``."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.gdn_oracle_recurrence.argtypes = [
            ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P, P,
            ctypes.c_double, ctypes.c_int, ctypes.c_double, P, P, P, ctypes.c_int]
        lib.gdn_oracle_recurrence.restype = ctypes.c_int
        _lib = lib
    return _lib


def _np64(x) -> Optional[np.ndarray]:
    """Exact conversion of a torch tensor (any float dtype) or array to float64."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _ints(x) -> Optional[list]:
    if x is None:
        return None
    if hasattr(x, "detach"):
        return [int(a) for a in x.detach().to("cpu").tolist()]
    return [int(a) for a in x]


def resolve_scale(scale, dk: int) -> float:
    """``scale`` None or 0.0 means 1/sqrt(head_dim)."""
    return 1.0 / math.sqrt(dk) if (scale is None or scale == 0.0) else float(scale)


class Units:
    """The (sequence, sab head) units one oracle call computes, with their
    inputs gathered into compact fp64 arrays."""

    def __init__(self, q, k, v, g, beta, initial_state, state_indices, cu_seqlens,
                 units: Optional[Iterable[tuple]] = None):
        cu = _ints(cu_seqlens)
        self.N = len(cu) - 1
        self.T, self.H_qk, self.dk = (int(s) for s in q.shape)
        self.H_v, self.dv = int(v.shape[1]), int(v.shape[2])
        self.H = max(self.H_qk, self.H_v)
        if self.H % self.H_qk or self.H % self.H_v:
            raise ValueError("H must be a multiple of both H_qk and H_v")
        if units is None:
            units = [(n, h) for n in range(self.N) for h in range(self.H)]
        self.units = [(int(n), int(h)) for n, h in units]
        idx = _ints(state_indices)
        gq, gv = self.H // self.H_qk, self.H // self.H_v
        lens, offs, rows_q, rows_v, rows_gh = [], [], [], [], []
        off = 0
        for n, h in self.units:
            bos, eos = cu[n], cu[n + 1]
            lens.append(eos - bos)
            offs.append(off)
            off += eos - bos
            t = np.arange(bos, eos)
            rows_q.append((t, h // gq))
            rows_v.append((t, h // gv))
            rows_gh.append((t, h))
        self.len = np.asarray(lens, dtype=np.int64)
        self.off = np.asarray(offs, dtype=np.int64)

        # slice in the source dtype first, then widen: exact and memory-light
        qs = [q[_ti(t), hh] for t, hh in rows_q]
        ks = [k[_ti(t), hh] for t, hh in rows_q]
        vs = [v[_ti(t), hh] for t, hh in rows_v]
        self.q = _cat(qs, self.dk)
        self.k = _cat(ks, self.dk)
        self.v = _cat(vs, self.dv)
        self.g = None if g is None else _cat1([g[_ti(t), hh] for t, hh in rows_gh])
        self.beta = None if beta is None else _cat1([beta[_ti(t), hh] for t, hh in rows_gh])
        self.slot = [(idx[n] if idx is not None else n) for n, _ in self.units]
        if initial_state is None:
            self.s0 = None
        else:
            self.s0 = np.ascontiguousarray(np.stack(
                [_np64(initial_state[s, h]) for s, (_, h) in zip(self.slot, self.units)])
                if self.units else np.zeros((0, self.dv, self.dk)))


def _ti(t):
    """Index a torch tensor or an array by a contiguous row range."""
    return slice(int(t[0]), int(t[-1]) + 1) if len(t) else slice(0, 0)


def _cat(parts, d):
    arrs = [_np64(p).reshape(-1, d) for p in parts]
    return np.ascontiguousarray(np.concatenate(arrs, axis=0)) if arrs else np.zeros((0, d))


def _cat1(parts):
    arrs = [_np64(p).reshape(-1) for p in parts]
    return np.ascontiguousarray(np.concatenate(arrs)) if arrs else np.zeros(0)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def recurrence_units(U: Units, scale, use_qk_l2norm: bool, nthreads: Optional[int] = None):
    """Run the C recurrence on gathered units.  Returns (out [R, Dv] compact
    rows in unit order, final states [n_units, Dv, Dk]), both float64."""
    lib = _load()
    R = int(U.len.sum()) if len(U.len) else 0
    out = np.zeros((R, U.dv))
    sf = np.zeros((len(U.units), U.dv, U.dk))
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib.gdn_oracle_recurrence(
        len(U.units), _ptr(U.len), _ptr(U.off), U.dk, U.dv, _ptr(U.q), _ptr(U.k),
        _ptr(U.v), _ptr(U.g), _ptr(U.beta), resolve_scale(scale, U.dk),
        int(bool(use_qk_l2norm)), L2NORM_EPS, _ptr(U.s0), _ptr(out), _ptr(sf), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle recurrence rejected its arguments")
    return out, sf


def scatter(U: Units, out_rows: np.ndarray, states: np.ndarray, cu_seqlens):
    """Place compact unit results at their packed positions: output
    ``[T, H, Dv]`` (NaN where no unit was computed) and final states keyed by
    sequence, ``{(n, h): [Dv, Dk]}``."""
    cu = _ints(cu_seqlens)
    o = np.full((U.T, U.H, U.dv), np.nan)
    fs = {}
    for i, (n, h) in enumerate(U.units):
        a, L = int(U.off[i]), int(U.len[i])
        o[cu[n]:cu[n] + L, h] = out_rows[a:a + L]
        fs[(n, h)] = states[i]
    return o, fs


def recurrence(q, k, v, g=None, beta=None, scale=None, initial_state=None,
               state_indices=None, cu_seqlens=None, use_qk_l2norm=False,
               units: Optional[Sequence[tuple]] = None, nthreads: Optional[int] = None):
    """fp64 oracle over whole problems.  Returns (output ``[T, H, Dv]`` float64,
    final state ``[N, H, Dv, Dk]`` float64 indexed by sequence).  With
    ``units`` only those (n, h) pairs are computed; the other entries are NaN."""
    if cu_seqlens is None:
        cu_seqlens = [0, int(q.shape[0])]
    U = Units(q, k, v, g, beta, initial_state, state_indices, cu_seqlens, units)
    rows, sf = recurrence_units(U, scale, use_qk_l2norm, nthreads)
    o, fs = scatter(U, rows, sf, cu_seqlens)
    final = np.full((U.N, U.H, U.dv, U.dk), np.nan)
    for (n, h), s in fs.items():
        final[n, h] = s
    return o, final


from .chunked import chunked  # noqa: E402  (numpy chunked form)

__all__ = ["build", "recurrence", "chunked", "Units", "recurrence_units", "scatter",
           "resolve_scale", "L2NORM_EPS"]
