"""Seeded synthetic workloads for the predictive sparse-KV decode step.

The one module that feeds both the fp64 oracle and the CUDA path.  It holds no
arithmetic of the method (no scoring, selection, gather or attention): only
the workload shapes and a counter-based generator (SplitMix64 + Box-Muller,
written in ``synth.c``) that fills caller-provided host buffers.

Workloads are shaped like the DualDecoder paper's long-context decode steps
(LLaMA-2-7B/13B, 32K-128K context; paper summary page, worked example and
experimental results) and stand in for the long-context suites the paper
evaluates on; no suite data is used.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

F32, BF16 = 0, 1
PLANT_NONE, PLANT_RANDOM, PLANT_SPREAD = 0, 1, 2


def build() -> str:
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", _LIB, _SRC, "-lm",
                    "-lpthread"], check=True)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("ctx_len", ctypes.c_int32), ("window", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("n_planted", ctypes.c_int32),
                ("plant_mode", ctypes.c_int32), ("key_scale", ctypes.c_int32),
                ("q_noise", ctypes.c_float), ("plant_noise", ctypes.c_float),
                ("plant_gain", ctypes.c_float)]


@dataclass(frozen=True)
class Workload:
    """One decode-step workload: L layers cycling through D distinct layer slots."""
    name: str
    cfg_id: int
    n_layers: int
    n_slots: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx_len: int
    top_k: int
    window: int
    dtype: int
    n_planted: int
    plant_mode: int
    key_scale: bool = False
    q_noise: float = 0.1
    plant_noise: float = 0.1
    plant_gain: float = 3.0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def elt(self) -> int:
        return 2 if self.dtype == BF16 else 4

    @property
    def units(self) -> int:
        return self.batch * self.n_kv_heads

    def seed(self, slot: int) -> int:
        return 1234 + 1000 * self.cfg_id + slot

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)

    # bytes of one layer, as counted by the roofline model
    def k_bytes(self) -> int:
        return self.batch * self.n_kv_heads * self.ctx_len * self.head_dim * self.elt

    def gather_bytes(self) -> int:
        return 2 * self.batch * self.n_kv_heads * self.top_k * self.head_dim * self.elt

    def attn_bytes(self) -> int:
        rows = self.top_k + self.window
        return 2 * self.batch * self.n_kv_heads * rows * self.head_dim * self.elt

    def c(self) -> _Cfg:
        return _Cfg(self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim, self.ctx_len,
                    self.window, self.dtype, self.n_planted, self.plant_mode,
                    int(self.key_scale), self.q_noise, self.plant_noise, self.plant_gain)


# The five workloads.  Shapes follow LLaMA-2-7B (32 heads x 128) and
# LLaMA-2-13B (40 heads x 128); c5 is a grouped-query variant (32 query / 8 KV heads).
C1 = Workload("c1-tiny-f32", 1, n_layers=1, n_slots=1, batch=1, n_q_heads=4, n_kv_heads=4,
              head_dim=64, ctx_len=2048, top_k=64, window=16, dtype=F32, n_planted=16,
              plant_mode=PLANT_RANDOM)
C2 = Workload("c2-7b-32k", 2, n_layers=32, n_slots=8, batch=8, n_q_heads=32, n_kv_heads=32,
              head_dim=128, ctx_len=32768, top_k=128, window=64, dtype=BF16, n_planted=32,
              plant_mode=PLANT_RANDOM)
C3 = Workload("c3-7b-128k", 3, n_layers=32, n_slots=8, batch=4, n_q_heads=32, n_kv_heads=32,
              head_dim=128, ctx_len=131072, top_k=1024, window=64, dtype=BF16, n_planted=32,
              plant_mode=PLANT_SPREAD)
C4 = Workload("c4-13b-64k", 4, n_layers=40, n_slots=8, batch=16, n_q_heads=40, n_kv_heads=40,
              head_dim=128, ctx_len=65536, top_k=512, window=64, dtype=BF16, n_planted=0,
              plant_mode=PLANT_NONE, key_scale=True)
C5 = Workload("c5-gqa-128k", 5, n_layers=32, n_slots=4, batch=32, n_q_heads=32, n_kv_heads=8,
              head_dim=128, ctx_len=131072, top_k=2048, window=0, dtype=BF16, n_planted=64,
              plant_mode=PLANT_RANDOM)
WORKLOADS = {w.name: w for w in (C1, C2, C3, C4, C5)}


class _Gen:
    def __init__(self):
        if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            build()
        L = self.lib = ctypes.CDLL(_LIB)
        C = ctypes.POINTER(_Cfg)
        P = ctypes.c_void_p
        L.syn_queries.argtypes = [C, ctypes.c_uint64, P, P, P]
        L.syn_kv.argtypes = [C, ctypes.c_uint64, P, P, P, P, ctypes.c_int]
        L.syn_fill_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                      ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                                      ctypes.c_int, P, ctypes.c_int]
        L.syn_stream.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.syn_stream.restype = ctypes.c_uint64
        L.syn_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.syn_u64.restype = ctypes.c_uint64
        L.syn_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.syn_normal.restype = ctypes.c_double
        for f in ("syn_queries", "syn_kv", "syn_fill_normal"):
            getattr(L, f).restype = None


_gen = None


def gen() -> _Gen:
    global _gen
    if _gen is None:
        _gen = _Gen()
    return _gen


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"]
        return x.ctypes.data
    assert not x.is_cuda and x.is_contiguous()
    return x.data_ptr()


def nthreads_default() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def fill_slot(w: Workload, slot: int, q_spec, q, K, V, planted=None, nthreads=None):
    """Fill one layer slot's host buffers.

    q_spec, q: [B][H_q][d]; K, V: [B][H_kv][n][d] (stored dtype; V may be None);
    planted: optional int32 [B][H_kv][P].  Any buffer is a numpy array, a CPU torch
    tensor (pinned or not) or a raw address.
    """
    g = gen()
    seed = w.seed(slot)
    qf = np.empty(w.batch * w.n_q_heads * w.head_dim, np.float32)
    g.lib.syn_queries(ctypes.byref(w.c()), seed, _addr(q_spec), _addr(q), qf.ctypes.data)
    g.lib.syn_kv(ctypes.byref(w.c()), seed, qf.ctypes.data, _addr(K), _addr(V), _addr(planted),
                 nthreads or nthreads_default())


def np_dtype(w: Workload):
    return np.uint16 if w.dtype == BF16 else np.float32


def slot_numpy(w: Workload, slot: int, with_v: bool = True):
    """Convenience for small workloads: one slot as numpy arrays (bf16 as uint16 bits)."""
    dt = np_dtype(w)
    q_spec = np.empty((w.batch, w.n_q_heads, w.head_dim), dt)
    q = np.empty_like(q_spec)
    K = np.empty((w.batch, w.n_kv_heads, w.ctx_len, w.head_dim), dt)
    V = np.empty_like(K) if with_v else None
    P = max(w.n_planted, 1)
    planted = np.zeros((w.batch, w.n_kv_heads, P), np.int32)
    fill_slot(w, slot, q_spec, q, K, V, planted)
    return {"q_spec": q_spec, "q": q, "K": K, "V": V,
            "planted": planted[..., :w.n_planted]}


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    """Widen stored bf16 bit patterns (uint16) to float32 (exact)."""
    return (x.astype(np.uint32) << 16).view(np.float32)
