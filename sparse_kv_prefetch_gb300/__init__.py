"""GB300-native predictive sparse-KV decode step (DualDecoder's hot path).

Thin ctypes binding of ``libdd.so`` (declared in ``include/dd.h``): argument
marshalling only, with the C names.  Every step runs in the library's CUDA
kernels; there is no CPU fallback, and every call raises if the library has not
been built (``python -m sparse_kv_prefetch_gb300.build``).

Buffers are torch tensors (device tensors for device arguments, page-locked CPU
tensors for the host KV store) or raw integer addresses.  Streams are
``torch.cuda.Stream`` objects, raw ``cudaStream_t`` integers, or None for the
current torch stream.

A decode step over L layers::

    import torch, sparse_kv_prefetch_gb300 as dd
    shape = dd.Shape(B, H_q, H_kv, d, n, k, W, dd.DD_BF16)
    ctx = dd.Ctx(shape)                     # scratch slots, workspace, events
    layers = [dd.LayerIO(q_spec[l], q[l],   # device [B][H_q][d]
                         K_dev[l],          # device [B][H_kv][n][d]
                         K_host[l], V_host[l],  # pinned host [B][H_kv][n][d]
                         V_win[l],          # device [B][H_kv][W][d]
                         out[l])            # device fp32 [B][H_q][d]
              for l in range(L)]
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    ctx.decode_step(layers, compute=compute, copy=copy)   # asynchronous

or, for fixed buffers, ``ctx.capture_step(layers, compute, copy=copy)`` once and
``ctx.replay_step(compute)`` per step.  Landmark (chunk) selection:
``build_landmarks`` per layer, ``ctx.set_landmark_chunk(c)``, the landmarks in
``LayerIO(..., landmarks=L)`` and ``decode_step(..., landmarks=True)``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import NamedTuple, Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdd.so")

DD_OK, DD_ERR_INVALID_ARG, DD_ERR_UNSUPPORTED, DD_ERR_OOM, DD_ERR_CUDA, DD_ERR_TIMEOUT = range(6)
DD_F32, DD_BF16 = 0, 1
DD_STEP_TIMING = 1
DD_STEP_LATE_GATHER = 2
DD_STEP_GATHER_LSU = 4
DD_STEP_PIPELINE = 8
DD_STEP_CORRECT_MISSES = 16
DD_STEP_LANDMARKS = 32
DD_STEP_TIMING_LIGHT = 64
DD_STEP_FUSED_TOPK = 128
DD_STEP_GATHER_BESIDE_ATTN = 256
DD_STEP_DEBUG_DELAY_COPY = 512
DD_STEP_DEBUG_DELAY_COMPUTE = 1024


class DDError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib().dd_status_string(status).decode()} (status {status})")


class dd_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "n_q_heads", "n_kv_heads", "head_dim", "ctx_len", "top_k", "window", "dtype")]


class dd_layer_io(ctypes.Structure):
    _fields_ = [("q_spec", ctypes.c_void_p), ("q", ctypes.c_void_p), ("k_dev", ctypes.c_void_p),
                ("k_host", ctypes.c_void_p), ("v_host", ctypes.c_void_p),
                ("v_win", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("landmarks", ctypes.c_void_p), ("k_win", ctypes.c_void_p),
                ("kv_host", ctypes.c_void_p)]


class dd_phase_times(ctypes.Structure):
    _fields_ = [("step_ms", ctypes.c_float), ("score_ms", ctypes.c_float),
                ("topk_ms", ctypes.c_float), ("gather_ms", ctypes.c_float),
                ("attn_ms", ctypes.c_float), ("n_layers", ctypes.c_int32),
                ("launches", ctypes.c_int32)]


@dataclass(frozen=True)
class Shape:
    """One layer: B, H_q, H_kv, d, n, k, W, dtype (DD_F32 or DD_BF16)."""
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx_len: int
    top_k: int
    window: int
    dtype: int

    def c(self) -> dd_shape:
        return dd_shape(self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim,
                        self.ctx_len, self.top_k, self.window, self.dtype)


_L = None


def _lib():
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m sparse_kv_prefetch_gb300.build` (there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, S = ctypes.c_void_p, ctypes.POINTER(dd_shape)
        sig = {
            "dd_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "dd_version": ([], ctypes.c_int),
            "dd_check_device": ([], ctypes.c_int),
            "dd_host_alloc": ([ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
            "dd_host_free": ([ctypes.c_void_p], ctypes.c_int),
            "dd_host_page_bytes": ([], ctypes.c_size_t),
            "dd_host_store_kind": ([ctypes.c_void_p], ctypes.c_int),
            "dd_host_alloc_pinned": ([ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)],
                                     ctypes.c_int),
            "dd_host_store_locked": ([ctypes.c_void_p], ctypes.c_int),
            "dd_workspace_size": ([S, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
            "dd_score_tensor_cores": ([S], ctypes.c_int),
            "dd_set_gather_geometry": ([ctypes.c_int, ctypes.c_int, ctypes.c_int], ctypes.c_int),
            "dd_set_gather_lsu_geometry": ([ctypes.c_int, ctypes.c_int], ctypes.c_int),
            "dd_score_topk": ([S, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "dd_gather_h2d": ([S, P, P, P, P, P, ctypes.c_int, P], ctypes.c_int),
            "dd_gather_h2d_kv": ([S, P, P, P, P, ctypes.c_int, P], ctypes.c_int),
            "dd_sparse_decode_attn": ([S, P, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
            "dd_sparse_decode_attn_noalloc": ([S, P, P, P, P, P, P, P], ctypes.c_int),
            "dd_ctx_create": ([S, ctypes.POINTER(P)], ctypes.c_int),
            "dd_ctx_destroy": ([P], None),
            "dd_ctx_device_bytes": ([P], ctypes.c_size_t),
            "dd_decode_step": ([P, ctypes.POINTER(dd_layer_io), ctypes.c_int, P, P, ctypes.c_int],
                               ctypes.c_int),
            "dd_ctx_timings": ([P, ctypes.POINTER(dd_phase_times)], ctypes.c_int),
            "dd_ctx_score_times": ([P, ctypes.POINTER(ctypes.c_float), ctypes.c_int],
                                   ctypes.c_int),
            "dd_correct_misses": ([S, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P],
                                  ctypes.c_int),
            "dd_correct_misses_kv": ([S, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P],
                                     ctypes.c_int),
            "dd_ctx_correction_stats": ([P, P, P, ctypes.c_int], ctypes.c_int),
            "dd_landmarks_size": ([S, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
                                  ctypes.c_int),
            "dd_landmarks_workspace_size": ([S, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
                                            ctypes.c_int),
            "dd_build_landmarks": ([S, ctypes.c_int, P, P, P], ctypes.c_int),
            "dd_score_topk_landmarks": ([S, ctypes.c_int, P, P, P, P, P, P, ctypes.c_size_t, P],
                                        ctypes.c_int),
            "dd_ctx_set_landmark_chunk": ([P, ctypes.c_int], ctypes.c_int),
            "dd_ctx_set_timing_depth": ([P, ctypes.c_int], ctypes.c_int),
            "dd_ctx_capture_step": ([P, ctypes.POINTER(dd_layer_io), ctypes.c_int, P, P,
                                     ctypes.c_int], ctypes.c_int),
            "dd_ctx_replay_step": ([P, P], ctypes.c_int),
            "dd_debug_expire_wait": ([ctypes.c_uint64, P], ctypes.c_int),
            "dd_ctx_step_timings": ([P, ctypes.c_int, ctypes.POINTER(dd_phase_times)],
                                    ctypes.c_int),
            "dd_ctx_step_score_times": ([P, ctypes.c_int, ctypes.POINTER(ctypes.c_float),
                                         ctypes.c_int], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _L = L
    return _L


def lib():
    """The loaded libdd.so (ctypes.CDLL)."""
    return _lib()


def _check(status: int, what: str):
    if status != DD_OK:
        raise DDError(status, what)


def _dev(x) -> Optional[int]:
    """Address of a device buffer (CUDA tensor or raw int; None -> NULL)."""
    if x is None or isinstance(x, int):
        return x
    if not x.is_cuda:
        raise TypeError("expected a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def _store_bytes(shape: "Shape") -> int:
    """Bytes of one layer's host K (or V) store [B][H_kv][n][d] for this shape."""
    elt = 2 if shape.dtype == DD_BF16 else 4
    return shape.batch * shape.n_kv_heads * shape.ctx_len * shape.head_dim * elt


def _host(x, need: Optional[int] = None) -> Optional[int]:
    """Address of a page-locked host buffer (pinned CPU tensor, a tensor from
    host_empty, or raw int).  With `need`, a tensor must hold at least that
    many bytes: the GPU reads the store by the shape alone, so a smaller one
    would be read past its end."""
    if x is None or isinstance(x, int):
        return x
    if x.is_cuda or not x.is_contiguous():
        raise TypeError("expected a contiguous CPU tensor")
    if need is not None and x.numel() * x.element_size() < need:
        raise ValueError(f"host store of {x.numel() * x.element_size()} bytes; the shape "
                         f"reads {need}")
    if not x.is_pinned() and not _lib().dd_host_store_kind(x.data_ptr()):
        raise ValueError("the host KV store must be page-locked (pin_memory=True or host_empty)")
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def version() -> int:
    return _lib().dd_version()


def host_empty(shape, dtype, kind: str = "huge"):
    """An uninitialised CPU tensor in a page-locked host KV store from the
    library: kind "huge" (dd_host_alloc: locked transparent huge pages) or
    "pinned" (dd_host_alloc_pinned: driver-allocated, exact size).  Freed with
    dd_host_free when the tensor and all its views are gone."""
    import weakref

    import torch
    numel = 1
    for s_ in shape:
        numel *= int(s_)
    nbytes = max(1, numel * torch.empty((), dtype=dtype).element_size())
    p = ctypes.c_void_p()
    if kind == "huge":
        _check(_lib().dd_host_alloc(nbytes, ctypes.byref(p)), "dd_host_alloc")
    elif kind == "pinned":
        _check(_lib().dd_host_alloc_pinned(nbytes, ctypes.byref(p)), "dd_host_alloc_pinned")
    else:
        raise ValueError(f"unknown host store kind {kind!r}")
    buf = (ctypes.c_char * nbytes).from_address(p.value)
    weakref.finalize(buf, _lib().dd_host_free, ctypes.c_void_p(p.value))
    t = torch.frombuffer(buf, dtype=torch.uint8, count=nbytes)
    return t.view(dtype)[:numel].view(*shape) if numel else t.view(dtype)[:0].view(*shape)


def host_page_bytes() -> int:
    return _lib().dd_host_page_bytes()


def host_store_locked(t) -> bool:
    """True if the tensor lies in a dd_host_alloc store whose pages are locked."""
    return bool(_lib().dd_host_store_locked(t.data_ptr()))


def debug_expire_wait(limit_ns: int, stream=None):
    """Test hook: a device wait that nothing completes gives up after limit_ns;
    the next check_device raises DD_ERR_TIMEOUT (see dd.h)."""
    _check(_lib().dd_debug_expire_wait(limit_ns, _stream(stream)), "dd_debug_expire_wait")


def check_device():
    """Raise DDError(DD_ERR_TIMEOUT) if a bounded device-side wait gave up."""
    _check(_lib().dd_check_device(), "dd_check_device")


def set_gather_geometry(grid_pct: int = 100, tile_bytes: int = 4096, stages: int = 3):
    """Geometry of the bulk-copy gather for later launches (see dd.h)."""
    _check(_lib().dd_set_gather_geometry(grid_pct, tile_bytes, stages), "dd_set_gather_geometry")


def set_gather_lsu_geometry(grid_pct: int = 100, threads: int = 256):
    """Geometry of the load/store gather for later launches (see dd.h)."""
    _check(_lib().dd_set_gather_lsu_geometry(grid_pct, threads), "dd_set_gather_lsu_geometry")


def workspace_size(shape: Shape) -> int:
    n = ctypes.c_size_t()
    _check(_lib().dd_workspace_size(ctypes.byref(shape.c()), ctypes.byref(n)), "dd_workspace_size")
    return n.value


def score_tensor_cores(shape: Shape) -> bool:
    """Whether this shape's logits are computed on the tensor cores (see dd.h)."""
    r = _lib().dd_score_tensor_cores(ctypes.byref(shape.c()))
    if r < 0:
        _check(-r, "dd_score_tensor_cores")
    return r == 1


def score_topk(shape: Shape, q_spec, k_dev, idx_out, sel_score_out, lse_out, workspace,
               stream=None, ws_bytes: Optional[int] = None):
    """Steps 1-2 (scoring + per-KV-head top-k) of one layer; see dd.h."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().dd_score_topk(ctypes.byref(shape.c()), _dev(q_spec), _dev(k_dev),
                                _dev(idx_out), _dev(sel_score_out), _dev(lse_out),
                                _dev(workspace), ws_bytes, _stream(stream)), "dd_score_topk")


def gather_h2d(shape: Shape, k_host, v_host, idx, k_buf, v_buf, mode: int = 0, stream=None):
    """Step 3: gather the selected K/V rows from pinned host memory; see dd.h."""
    nb = _store_bytes(shape)
    _check(_lib().dd_gather_h2d(ctypes.byref(shape.c()), _host(k_host, nb), _host(v_host, nb),
                                _dev(idx), _dev(k_buf), _dev(v_buf), mode, _stream(stream)),
           "dd_gather_h2d")


def gather_h2d_kv(shape: Shape, kv_host, idx, k_buf, v_buf, mode: int = 0, stream=None):
    """Step 3 from one interleaved host store [B][H_kv][n][2][d]; see dd.h."""
    _check(_lib().dd_gather_h2d_kv(ctypes.byref(shape.c()), _host(kv_host, 2 * _store_bytes(shape)),
                                   _dev(idx),
                                   _dev(k_buf), _dev(v_buf), mode, _stream(stream)),
           "dd_gather_h2d_kv")


def sparse_decode_attn(shape: Shape, q, k_buf, v_buf, k_dev, v_win, out, workspace, stream=None,
                       ws_bytes: Optional[int] = None):
    """Step 4: split-k attention over the gathered rows plus the window; see dd.h."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().dd_sparse_decode_attn(ctypes.byref(shape.c()), _dev(q), _dev(k_buf),
                                        _dev(v_buf), _dev(k_dev), _dev(v_win), _dev(out),
                                        _dev(workspace), ws_bytes, _stream(stream)),
           "dd_sparse_decode_attn")


def correct_misses(shape: Shape, q, k_dev, idx_spec, k_buf_spec, v_buf_spec, k_host, v_host,
                   idx_true_out, k_buf_out, v_buf_out, miss_out, mass_out, workspace,
                   stream=None, ws_bytes: Optional[int] = None):
    """Miss correction for one layer: the real query's top-k and its rows,
    copied from the prefetched buffers or fetched from the host store; see dd.h."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().dd_correct_misses(
        ctypes.byref(shape.c()), _dev(q), _dev(k_dev), _dev(idx_spec), _dev(k_buf_spec),
        _dev(v_buf_spec), _host(k_host, _store_bytes(shape)), _host(v_host, _store_bytes(shape)),
        _dev(idx_true_out), _dev(k_buf_out),
        _dev(v_buf_out), _dev(miss_out), _dev(mass_out), _dev(workspace), ws_bytes,
        _stream(stream)), "dd_correct_misses")


def correct_misses_kv(shape: Shape, q, k_dev, idx_spec, k_buf_spec, v_buf_spec, kv_host,
                      idx_true_out, k_buf_out, v_buf_out, miss_out, mass_out, workspace,
                      stream=None, ws_bytes: Optional[int] = None):
    """correct_misses with the host rows read from one interleaved store
    [B][H_kv][n][2][d]; see dd.h."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().dd_correct_misses_kv(
        ctypes.byref(shape.c()), _dev(q), _dev(k_dev), _dev(idx_spec), _dev(k_buf_spec),
        _dev(v_buf_spec), _host(kv_host, 2 * _store_bytes(shape)), _dev(idx_true_out),
        _dev(k_buf_out),
        _dev(v_buf_out), _dev(miss_out), _dev(mass_out), _dev(workspace), ws_bytes,
        _stream(stream)), "dd_correct_misses_kv")


def landmarks_size(shape: Shape, chunk: int) -> int:
    """Bytes of one layer's chunk landmarks (fp32 [B][H_kv][(n-W)/chunk][d])."""
    n = ctypes.c_size_t()
    _check(_lib().dd_landmarks_size(ctypes.byref(shape.c()), chunk, ctypes.byref(n)),
           "dd_landmarks_size")
    return n.value


def landmarks_workspace_size(shape: Shape, chunk: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib().dd_landmarks_workspace_size(ctypes.byref(shape.c()), chunk, ctypes.byref(n)),
           "dd_landmarks_workspace_size")
    return n.value


def build_landmarks(shape: Shape, chunk: int, k_dev, landmarks_out, stream=None):
    """Chunk-mean landmarks of one layer's keys; see dd.h."""
    _check(_lib().dd_build_landmarks(ctypes.byref(shape.c()), chunk, _dev(k_dev),
                                     _dev(landmarks_out), _stream(stream)), "dd_build_landmarks")


def score_topk_landmarks(shape: Shape, chunk: int, q_spec, landmarks, idx_out, chunk_score_out,
                         lse_out, workspace, stream=None, ws_bytes: Optional[int] = None):
    """Landmark selection: top k/chunk chunks per KV head, expanded to k rows; see dd.h."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib().dd_score_topk_landmarks(ctypes.byref(shape.c()), chunk, _dev(q_spec),
                                          _dev(landmarks), _dev(idx_out), _dev(chunk_score_out),
                                          _dev(lse_out), _dev(workspace), ws_bytes,
                                          _stream(stream)), "dd_score_topk_landmarks")


NOALLOC_SCRATCH_BYTES = 32 << 20


def sparse_decode_attn_noalloc(shape: Shape, q, k_buf, v_buf, k_dev, v_win, out, stream=None):
    """Step 4 without a workspace: the partials use the library's static device
    array (NOALLOC_SCRATCH_BYTES, shared by every call; calls must not overlap
    on the GPU).  For callers that cannot allocate device memory; see dd.h."""
    _check(_lib().dd_sparse_decode_attn_noalloc(ctypes.byref(shape.c()), _dev(q), _dev(k_buf),
                                                _dev(v_buf), _dev(k_dev), _dev(v_win),
                                                _dev(out), _stream(stream)),
           "dd_sparse_decode_attn_noalloc")


class LayerIO(NamedTuple):
    q_spec: object
    q: object
    k_dev: object
    k_host: object
    v_host: object
    v_win: object
    out: object
    landmarks: object = None
    k_win: object = None
    kv_host: object = None


class Ctx:
    """Layer-scoped state (double-buffered scratch, workspace, events) for one shape."""

    def __init__(self, shape: Shape):
        self.shape = shape
        h = ctypes.c_void_p()
        _check(_lib().dd_ctx_create(ctypes.byref(shape.c()), ctypes.byref(h)), "dd_ctx_create")
        self._h = h
        self._keep = None

    @property
    def device_bytes(self) -> int:
        return _lib().dd_ctx_device_bytes(self._h)

    def close(self):
        if self._h:
            _lib().dd_ctx_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def pack(layers: Sequence[LayerIO], shape: Optional[Shape] = None):
        """Marshal the per-layer buffers once (reuse across steps).  With the
        shape, host stores smaller than it reads are refused."""
        arr = (dd_layer_io * len(layers))()
        nb = None if shape is None else _store_bytes(shape)
        for i, io in enumerate(layers):
            arr[i] = dd_layer_io(_dev(io.q_spec), _dev(io.q), _dev(io.k_dev),
                                 _host(io.k_host, nb), _host(io.v_host, nb), _dev(io.v_win),
                                 _dev(io.out), _dev(io.landmarks), _dev(io.k_win),
                                 _host(io.kv_host, None if nb is None else 2 * nb))
        return arr

    def set_landmark_chunk(self, chunk: int):
        """Chunk size of landmark selection (decode_step(landmarks=True))."""
        _check(_lib().dd_ctx_set_landmark_chunk(self._h, chunk), "dd_ctx_set_landmark_chunk")

    def decode_step(self, layers, compute=None, copy=None, timing=False,
                    late_gather: bool = False, gather_mode: int = 0, pipeline: bool = False,
                    correct_misses: bool = False, landmarks: bool = False,
                    fused_topk: bool = False, debug_delay: str = "", guarded: bool = False):
        """Enqueue one decode step over the layers (LayerIO list or a packed array)."""
        arr = layers if isinstance(layers, ctypes.Array) else self.pack(layers, self.shape)
        cs = _stream(compute)
        xs = None if copy is None else _stream(copy)
        # timing: False, True (every phase) or "light" (step and scoring only)
        flags = self._flags(late_gather, gather_mode, pipeline, correct_misses, landmarks,
                            fused_topk, timing, debug_delay, guarded)
        _check(_lib().dd_decode_step(self._h, arr, len(arr), cs, xs, flags), "dd_decode_step")
        self._keep = arr

    @staticmethod
    def _flags(late_gather=False, gather_mode=0, pipeline=False, correct_misses=False,
               landmarks=False, fused_topk=False, timing=False, debug_delay="",
               guarded=False):
        return ((DD_STEP_DEBUG_DELAY_COPY if "copy" in debug_delay else 0)
                | (DD_STEP_GATHER_BESIDE_ATTN if guarded else 0)
                | (DD_STEP_DEBUG_DELAY_COMPUTE if "compute" in debug_delay else 0)
                | (DD_STEP_TIMING_LIGHT if timing == "light" else DD_STEP_TIMING if timing else 0)
                | (DD_STEP_LATE_GATHER if late_gather else 0)
                | (DD_STEP_GATHER_LSU if gather_mode == 1 else 0)
                | (DD_STEP_PIPELINE if pipeline else 0)
                | (DD_STEP_CORRECT_MISSES if correct_misses else 0)
                | (DD_STEP_LANDMARKS if landmarks else 0)
                | (DD_STEP_FUSED_TOPK if fused_topk else 0))

    def capture_step(self, layers, compute, copy=None, **schedule):
        """Capture one decode step into a CUDA graph held by the context (the
        step runs once directly first); replay it with replay_step.  `compute`
        must be a created stream (capture is not possible on the default one)."""
        arr = layers if isinstance(layers, ctypes.Array) else self.pack(layers, self.shape)
        _check(_lib().dd_ctx_capture_step(self._h, arr, len(arr), _stream(compute),
                                          None if copy is None else _stream(copy),
                                          self._flags(**schedule)), "dd_ctx_capture_step")
        self._keep_graph = arr

    def replay_step(self, stream=None):
        """Launch the captured step (one graph launch)."""
        _check(_lib().dd_ctx_replay_step(self._h, _stream(stream)), "dd_ctx_replay_step")

    def set_timing_depth(self, depth: int):
        """Keep the events of the last `depth` timed steps (read with back=...)."""
        _check(_lib().dd_ctx_set_timing_depth(self._h, depth), "dd_ctx_set_timing_depth")

    def timings(self, back: int = 0) -> dict:
        """Phase times of the timed step `back` steps before the last one."""
        t = dd_phase_times()
        _check(_lib().dd_ctx_step_timings(self._h, back, ctypes.byref(t)), "dd_ctx_step_timings")
        return {f: getattr(t, f) for f, _ in dd_phase_times._fields_}

    def correction_stats(self, n_layers: int):
        """(misses [n_layers][units] int32, mass [n_layers][units][2] float32) of the
        last step run with correct_misses=True."""
        import numpy as np
        U = self.shape.batch * self.shape.n_kv_heads
        misses = np.zeros((n_layers, U), np.int32)
        mass = np.zeros((n_layers, U, 2), np.float32)
        _check(_lib().dd_ctx_correction_stats(self._h, misses.ctypes.data, mass.ctypes.data,
                                              n_layers), "dd_ctx_correction_stats")
        return misses, mass

    def score_times(self, n: int, back: int = 0):
        buf = (ctypes.c_float * n)()
        _check(_lib().dd_ctx_step_score_times(self._h, back, buf, n), "dd_ctx_step_score_times")
        return list(buf)
