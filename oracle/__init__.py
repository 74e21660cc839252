"""fp64 CPU oracle for the predictive sparse-KV decode step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path (``sparse_kv_prefetch_gb300``) never does.
It shares no code with the CUDA path; both are fed by ``synth``.

This module is argument marshalling around ``oracle.c``.  That file holds every
step of the arithmetic and cites the passage of the DualDecoder paper (and its
summary page) that each step follows.  No function here is "parity unpinned":
``tests/test_oracle_pins.py`` pins each one against closed forms, invariants and
brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1


def build(src: str = _SRC, out: str = _LIB, extra_flags: tuple = ()) -> str:
    """Compile oracle.c with gcc (no fast-math: IEEE fp64 throughout)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", *extra_flags, "-o", out, src,
           "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "n_q_heads", "n_kv_heads", "head_dim", "ctx_len", "top_k", "window", "dtype")]


@dataclass(frozen=True)
class Shape:
    """One layer: B, H_q, H_kv, d, n, k, W and the stored dtype (F32 or BF16)."""
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx_len: int
    top_k: int
    window: int
    dtype: int

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def c(self) -> _Shape:
        return _Shape(self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim,
                      self.ctx_len, self.top_k, self.window, self.dtype)


def _ptr(x) -> int:
    """Address of a host buffer: numpy array, CPU torch tensor or a raw int."""
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"]
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        assert not x.is_cuda and x.is_contiguous()
        return x.data_ptr()
    raise TypeError(type(x))


_P = ctypes.c_void_p
_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int32)


class Oracle:
    """ctypes handle on one compiled oracle library (tests may load a variant)."""

    def __init__(self, lib_path: str = _LIB):
        if lib_path == _LIB and (not os.path.exists(_LIB)
                                 or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
            build()
        self.lib = L = ctypes.CDLL(lib_path)
        S = ctypes.POINTER(_Shape)
        L.orc_score_unit.argtypes = [S, _P, _P, ctypes.c_int, ctypes.c_int, _D, _D]
        L.orc_selection_score.argtypes = [S, _D, _D, _D]
        L.orc_select_unit.argtypes = [S, _D, _I, _D, _D]
        L.orc_attend_unit.argtypes = [S, _P, _P, _P, ctypes.c_int, ctypes.c_int, _I,
                                      ctypes.c_int64, ctypes.c_int, _D]
        L.orc_dense_unit.argtypes = [S, _P, _P, _P, ctypes.c_int, ctypes.c_int, _D]
        L.orc_layer.argtypes = [S, _P, _P, _P, _P, _I, _D, _D, _D, _D, ctypes.c_int64,
                                ctypes.c_int64, ctypes.c_int]
        L.orc_landmarks_unit.argtypes = [S, ctypes.c_int, _P, ctypes.c_int, ctypes.c_int, _D]
        L.orc_landmark_select_unit.argtypes = [S, ctypes.c_int, _P, _D, ctypes.c_int, ctypes.c_int,
                                               _I, _D, _D, _D]
        for f in ("orc_score_unit", "orc_selection_score", "orc_select_unit",
                  "orc_attend_unit", "orc_dense_unit", "orc_layer", "orc_landmarks_unit",
                  "orc_landmark_select_unit"):
            getattr(L, f).restype = None

    # -- steps 1-2 ---------------------------------------------------------
    def score_unit(self, s: Shape, q_spec, K, b: int, hk: int):
        """Logits [G][n] and LSE [G] of unit (b, hk)."""
        logits = np.empty((s.group, s.ctx_len), np.float64)
        lse = np.empty(s.group, np.float64)
        self.lib.orc_score_unit(ctypes.byref(s.c()), _ptr(q_spec), _ptr(K), b, hk,
                                logits.ctypes.data_as(_D), lse.ctypes.data_as(_D))
        return logits, lse

    # -- step 3 -------------------------------------------------------------
    def selection_score(self, s: Shape, logits: np.ndarray, lse: np.ndarray) -> np.ndarray:
        logits = np.ascontiguousarray(logits, np.float64)
        lse = np.ascontiguousarray(lse, np.float64)
        a = np.empty(s.ctx_len, np.float64)
        self.lib.orc_selection_score(ctypes.byref(s.c()), logits.ctypes.data_as(_D),
                                     lse.ctypes.data_as(_D), a.ctypes.data_as(_D))
        return a

    # -- step 4 -------------------------------------------------------------
    def select_unit(self, s: Shape, a: np.ndarray):
        """(idx ascending [k], a[idx] [k], relative gap between k-th and (k+1)-th)."""
        a = np.ascontiguousarray(a, np.float64)
        idx = np.empty(s.top_k, np.int32)
        sel = np.empty(s.top_k, np.float64)
        gap = ctypes.c_double()
        self.lib.orc_select_unit(ctypes.byref(s.c()), a.ctypes.data_as(_D),
                                 idx.ctypes.data_as(_I), sel.ctypes.data_as(_D),
                                 ctypes.byref(gap))
        return idx, sel, gap.value

    # -- step 5 / 6 ---------------------------------------------------------
    def attend_unit(self, s: Shape, q, K, V, b: int, hk: int, idx, include_window=True):
        """Attention output [G][d] of unit (b, hk) over idx (+ window)."""
        idx = np.ascontiguousarray(idx, np.int32)
        out = np.empty((s.group, s.head_dim), np.float64)
        self.lib.orc_attend_unit(ctypes.byref(s.c()), _ptr(q), _ptr(K), _ptr(V), b, hk,
                                 idx.ctypes.data_as(_I), idx.size, int(include_window),
                                 out.ctypes.data_as(_D))
        return out

    def dense_unit(self, s: Shape, q, K, V, b: int, hk: int):
        out = np.empty((s.group, s.head_dim), np.float64)
        self.lib.orc_dense_unit(ctypes.byref(s.c()), _ptr(q), _ptr(K), _ptr(V), b, hk,
                                out.ctypes.data_as(_D))
        return out

    # -- landmark (chunk) selection ----------------------------------------
    def landmarks_unit(self, s: Shape, chunk: int, K, b: int, hk: int) -> np.ndarray:
        """Landmarks [M][d] of unit (b, hk): the mean key of each chunk of
        [0, n - W)."""
        M = (s.ctx_len - s.window) // chunk
        L = np.empty((M, s.head_dim), np.float64)
        self.lib.orc_landmarks_unit(ctypes.byref(s.c()), chunk, _ptr(K), b, hk,
                                    L.ctypes.data_as(_D))
        return L

    def landmark_select_unit(self, s: Shape, chunk: int, q_spec, L: np.ndarray, b: int, hk: int):
        """(rows [k] ascending, chunk scores [k/c], chunk LSE [G], gap) of unit (b, hk)."""
        L = np.ascontiguousarray(L, np.float64)
        rows = np.empty(s.top_k, np.int32)
        sel = np.empty(s.top_k // chunk, np.float64)
        lse = np.empty(s.group, np.float64)
        gap = ctypes.c_double()
        self.lib.orc_landmark_select_unit(ctypes.byref(s.c()), chunk, _ptr(q_spec),
                                          L.ctypes.data_as(_D), b, hk, rows.ctypes.data_as(_I),
                                          sel.ctypes.data_as(_D), lse.ctypes.data_as(_D),
                                          ctypes.byref(gap))
        return rows, sel, lse, gap.value

    # -- whole layer -------------------------------------------------------
    def layer(self, s: Shape, q_spec, q, K, V, nthreads: int = 1, units=None):
        """Steps 1-5 on units [lo, hi) of a layer (all units by default)."""
        U = s.batch * s.n_kv_heads
        lo, hi = units if units is not None else (0, U)
        idx = np.zeros((U, s.top_k), np.int32)
        sel = np.zeros((U, s.top_k), np.float64)
        lse = np.zeros((s.batch, s.n_q_heads), np.float64)
        gap = np.zeros(U, np.float64)
        out = np.zeros((s.batch, s.n_q_heads, s.head_dim), np.float64)
        self.lib.orc_layer(ctypes.byref(s.c()), _ptr(q_spec), _ptr(q), _ptr(K), _ptr(V),
                           idx.ctypes.data_as(_I), sel.ctypes.data_as(_D),
                           lse.ctypes.data_as(_D), gap.ctypes.data_as(_D),
                           out.ctypes.data_as(_D), lo, hi, nthreads)
        return {"idx": idx, "sel": sel, "lse": lse, "gap": gap, "out": out}


_default = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
