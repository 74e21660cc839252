"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/dd.h declares, and rejects bad arguments synchronously
with the documented status codes, before touching the device."""
import ctypes
import os
import re

import pytest

import sparse_kv_prefetch_gb300 as dd
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(dd_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_function_is_exported():
    lib = ctypes.CDLL(dd.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings_and_version():
    lib = dd.lib()
    for s in range(6):
        assert lib.dd_status_string(s)
    assert lib.dd_status_string(99) == b"unknown status"
    assert dd.version() >= 10000


def _shape(**kw):
    base = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, ctx_len=4096, top_k=64,
                window=16, dtype=dd.DD_BF16)
    base.update(kw)
    return dd.Shape(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(window=4096), dd.DD_ERR_INVALID_ARG),          # W >= n
    (dict(top_k=4096 - 15), dd.DD_ERR_INVALID_ARG),      # k > n - W
    (dict(top_k=0), dd.DD_ERR_INVALID_ARG),
    (dict(n_kv_heads=3), dd.DD_ERR_INVALID_ARG),         # H_q % H_kv != 0
    (dict(batch=0), dd.DD_ERR_INVALID_ARG),
    (dict(window=-1), dd.DD_ERR_INVALID_ARG),
    (dict(head_dim=96), dd.DD_ERR_UNSUPPORTED),
    (dict(head_dim=256, dtype=dd.DD_F32), dd.DD_ERR_UNSUPPORTED),
    (dict(n_q_heads=6, n_kv_heads=2), dd.DD_ERR_UNSUPPORTED),  # group of 3
    (dict(dtype=7), dd.DD_ERR_UNSUPPORTED),
])
def test_bad_shapes_rejected(kw, status):
    n = ctypes.c_size_t()
    st = dd.lib().dd_workspace_size(ctypes.byref(_shape(**kw).c()), ctypes.byref(n))
    assert st == status


def test_scoring_form_query():
    """bf16 keys with a GQA group are scored on the tensor cores; one head per
    KV head and fp32 keys in the per-lane form; bad shapes give the negated
    status of dd_workspace_size."""
    for g in (2, 4, 8):
        assert dd.score_tensor_cores(_shape(n_q_heads=2 * g)) is True
    assert dd.score_tensor_cores(_shape(n_q_heads=2)) is False
    assert dd.score_tensor_cores(_shape(head_dim=64, dtype=dd.DD_F32)) is False
    assert dd.lib().dd_score_tensor_cores(ctypes.byref(_shape(head_dim=96).c())) == \
        -dd.DD_ERR_UNSUPPORTED
    with pytest.raises(dd.DDError) as e:
        dd.score_tensor_cores(_shape(window=4096))
    assert e.value.status == dd.DD_ERR_INVALID_ARG


def test_workspace_size_layout():
    """Logits [B][H_q][round_up(n, 4)] fp32 dominate; the rest is small."""
    for w in (synth.C1, synth.C2, synth.C3, synth.C4, synth.C5):
        shp = dd.Shape(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ctx_len, w.top_k,
                       w.window, w.dtype)
        ws = dd.workspace_size(shp)
        logits = w.batch * w.n_q_heads * ((w.ctx_len + 3) // 4 * 4) * 4
        assert logits <= ws <= logits * 1.1 + (1 << 20)
        assert ws % 256 == 0


def test_gather_geometry_ranges():
    """dd_set_gather_geometry takes grid 1..800 % of the SMs, tiles of a
    multiple of 512 bytes up to 16 KiB, 1..8 stages, and at most 227 KiB of
    shared memory per CTA; anything else is refused and changes nothing."""
    lib = dd.lib()
    for bad in ((0, 4096, 3), (801, 4096, 3), (100, 4000, 3), (100, 256, 3),
                (100, 32768, 1), (100, 4096, 0), (100, 4096, 9), (100, 16384, 8)):
        assert lib.dd_set_gather_geometry(*bad) == dd.DD_ERR_INVALID_ARG, bad
    for good in ((1, 512, 1), (800, 16384, 6), (100, 4096, 3)):
        assert lib.dd_set_gather_geometry(*good) == dd.DD_OK, good
    for bad in ((0, 256), (100, 48), (100, 288), (100, 0), (801, 32)):
        assert lib.dd_set_gather_lsu_geometry(*bad) == dd.DD_ERR_INVALID_ARG, bad
    for good in ((100, 32), (50, 128), (100, 256)):
        assert lib.dd_set_gather_lsu_geometry(*good) == dd.DD_OK, good


def test_null_and_misaligned_pointers_rejected():
    lib = dd.lib()
    shp = _shape().c()
    st = lib.dd_score_topk(ctypes.byref(shp), None, 16, 16, 16, None, 16, 1 << 30, None)
    assert st == dd.DD_ERR_INVALID_ARG
    st = lib.dd_score_topk(ctypes.byref(shp), 17, 16, 16, 16, None, 16, 1 << 30, None)
    assert st == dd.DD_ERR_INVALID_ARG
    st = lib.dd_sparse_decode_attn(ctypes.byref(shp), 16, 16, 16, 16, None, 16, 16, 1 << 30,
                                   None)  # W > 0 needs the window V
    assert st == dd.DD_ERR_INVALID_ARG
    st = lib.dd_gather_h2d(ctypes.byref(shp), 16, 16, 16, 16, 16, 2, None)
    assert st == dd.DD_ERR_UNSUPPORTED  # modes 0 (bulk copy) and 1 (load/store) only
    st = lib.dd_score_topk(ctypes.byref(shp), 16, 16, 16, 16, None, 16, 1024, None)
    assert st == dd.DD_ERR_INVALID_ARG  # workspace too small
    assert lib.dd_decode_step(None, None, 0, None, None, 0) == dd.DD_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,chunk,status", [
    (dict(), 1, dd.DD_ERR_UNSUPPORTED),                 # a chunk of one row is not a chunk
    (dict(), 0, dd.DD_ERR_UNSUPPORTED),
    (dict(), 32, dd.DD_ERR_UNSUPPORTED),                # 32 divides k = 64, not n - W = 4080
    (dict(), 17, dd.DD_ERR_UNSUPPORTED),                # 17 divides n - W = 4080, not k = 64
    (dict(head_dim=256), 16, dd.DD_ERR_UNSUPPORTED),    # landmarks: d in {64, 128}
    (dict(window=4096), 16, dd.DD_ERR_INVALID_ARG),     # the shape itself is invalid
])
def test_bad_landmark_chunks_rejected(kw, chunk, status):
    n = ctypes.c_size_t()
    st = dd.lib().dd_landmarks_size(ctypes.byref(_shape(**kw).c()), chunk, ctypes.byref(n))
    assert st == status


def test_landmark_sizes():
    shp = _shape()  # n - W = 4080 = 255 * 16, k = 64 = 4 * 16
    M = 4080 // 16
    assert dd.landmarks_size(shp, 16) == 2 * 2 * M * 128 * 4
    ws = dd.landmarks_workspace_size(shp, 16)
    assert ws % 256 == 0
    assert ws >= 2 * 8 * M * 4 + 2 * 8 * 128 * 4 + 2 * 2 * 4 * 4  # logits, fp32 q, chunk ids
    assert ws < dd.workspace_size(shp)  # M = (n - W) / c logits instead of n
    lib = dd.lib()
    c = shp.c()
    assert lib.dd_build_landmarks(ctypes.byref(c), 16, None, 16, None) == dd.DD_ERR_INVALID_ARG
    assert lib.dd_build_landmarks(ctypes.byref(c), 16, 16, 8, None) == dd.DD_ERR_INVALID_ARG
    st = lib.dd_score_topk_landmarks(ctypes.byref(c), 16, 16, 16, 16, 16, None, 16, 1024, None)
    assert st == dd.DD_ERR_INVALID_ARG  # workspace too small
    st = lib.dd_score_topk_landmarks(ctypes.byref(c), 16, 16, 16, None, 16, None, 16, ws, None)
    assert st == dd.DD_ERR_INVALID_ARG  # no index output
    assert lib.dd_ctx_set_landmark_chunk(None, 16) == dd.DD_ERR_INVALID_ARG


def test_timing_calls_reject_null_context():
    lib = dd.lib()
    t = dd.dd_phase_times()
    assert lib.dd_ctx_set_timing_depth(None, 4) == dd.DD_ERR_INVALID_ARG
    assert lib.dd_ctx_step_timings(None, 0, ctypes.byref(t)) == dd.DD_ERR_INVALID_ARG
    assert lib.dd_ctx_timings(None, ctypes.byref(t)) == dd.DD_ERR_INVALID_ARG
    assert lib.dd_ctx_capture_step(None, None, 1, None, None, 0) == dd.DD_ERR_INVALID_ARG
    assert lib.dd_ctx_replay_step(None, None) == dd.DD_ERR_INVALID_ARG
    assert lib.dd_debug_expire_wait(0, None) == dd.DD_ERR_INVALID_ARG
    assert lib.dd_debug_expire_wait(200_000_000, None) == dd.DD_ERR_INVALID_ARG


def test_pageable_host_store_rejected_by_binding():
    import torch
    shp = _shape()
    full = torch.empty((2, 2, 4096, 128), dtype=torch.bfloat16)  # the shape's size, pageable
    with pytest.raises(ValueError, match="page-locked"):
        dd.gather_h2d(shp, full, full, 16, 16, 16)
    kv = torch.empty((2, 2, 4096, 2, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="page-locked"):
        dd.gather_h2d_kv(shp, kv, 16, 16, 16)


def test_host_store_smaller_than_the_shape_rejected_by_binding():
    """The GPU reads a host store by the shape alone, so the binding refuses
    one with fewer bytes than the shape reads, before anything is launched."""
    import torch
    shp = _shape()
    small = torch.empty((2, 2, 4095, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="the shape reads"):
        dd.gather_h2d(shp, small, small, 16, 16, 16)
    one_tensor = torch.empty((2, 2, 4096, 128), dtype=torch.bfloat16)  # K only, not K and V
    with pytest.raises(ValueError, match="the shape reads"):
        dd.gather_h2d_kv(shp, one_tensor, 16, 16, 16)
    with pytest.raises(ValueError, match="the shape reads"):
        dd.correct_misses(shp, 16, 16, 16, 16, 16, small, small, 16, 16, 16, 16, 16, 16,
                          ws_bytes=1)
    with pytest.raises(ValueError, match="the shape reads"):
        dd.correct_misses_kv(shp, 16, 16, 16, 16, 16, one_tensor, 16, 16, 16, 16, 16, 16,
                             ws_bytes=1)
    io = dd.LayerIO(16, 16, 16, None, None, None, 16, kv_host=one_tensor)
    with pytest.raises(ValueError, match="the shape reads"):
        dd.Ctx.pack([io], shp)
    dd.Ctx.pack([io._replace(kv_host=None, k_host=16, v_host=16)], shp)  # raw addresses pass


def test_product_path_never_touches_the_oracle():
    """The package and its sources import neither the oracle nor the generator."""
    pkg = os.path.join(ROOT, "sparse_kv_prefetch_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\b(import|from)\s+(oracle|synth)\b", text), f
                assert "liboracle" not in text and "libsynth" not in text, f
