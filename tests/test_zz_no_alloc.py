"""The allocation-free attention call against the regular one.

dd_sparse_decode_attn_noalloc serves callers that cannot allocate device
memory.  Examples: an engine whose KV-cache pool already owns all free HBM, or
a plugin whose host framework owns every device allocation.  Its split-k
partials live in a static device array inside libdd.so instead of a
caller-provided workspace.

This file is named so that pytest collects it last.  A run that stops at the
first failure has then already run every other test.
"""
import ctypes

import pytest
import torch

import sparse_kv_prefetch_gb300 as dd
import synth
from gpu_util import TOL_OUT, Outputs, Slot, dd_shape, run_layer

CASES = [
    synth.C2.scaled(batch=2, n_q_heads=4, n_kv_heads=4, ctx_len=5000),
    synth.C5.scaled(batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=12000),
    synth.C1,
]


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_on_consecutive_calls():
    """Three calls in a row (two shapes, then the first again) each match the
    workspace entry point within the attention tolerance."""
    prepared = []
    for w in CASES:
        s, o = Slot(w), Outputs(w)
        run_layer(w, s, o)  # regular entry points: indices, gathered rows, reference output
        prepared.append((w, s, o))
    torch.cuda.synchronize()
    for w, s, o in prepared + [prepared[0]]:
        got = torch.full_like(o.out, float("nan"))
        status = dd.lib().dd_sparse_decode_attn_noalloc(
            ctypes.byref(dd_shape(w).c()), s.q.data_ptr(), o.k_buf.data_ptr(),
            o.v_buf.data_ptr(), s.K.data_ptr(),
            s.v_win.data_ptr() if s.v_win is not None else None, got.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert status == dd.DD_OK, dd.lib().dd_status_string(status)
        torch.cuda.synchronize()
        err = (got - o.out).abs().max().item()
        assert err <= TOL_OUT[w.dtype], f"{w.name}: max-abs difference {err:.3g}"


def test_noalloc_rejects_shapes_beyond_its_static_scratch():
    """A shape whose partials exceed the static array is refused up front."""
    big = dd.Shape(64, 64, 64, 128, 16384, 8192, 0, dd.DD_BF16)
    S = (8192 + 63) // 64
    assert 64 * 64 * S * 128 * 4 > dd.NOALLOC_SCRATCH_BYTES
    status = dd.lib().dd_sparse_decode_attn_noalloc(ctypes.byref(big.c()), 16, 16, 16, 16, None,
                                                    16, None)
    assert status == dd.DD_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_rejects_the_pointers_the_workspace_call_rejects():
    """Both attention entry points share one pointer check: a page-locked host
    buffer passed as the query (or as the output) is refused by each with
    DD_ERR_INVALID_ARG before anything is launched."""
    w = CASES[0]
    s, o = Slot(w), Outputs(w)
    run_layer(w, s, o)
    torch.cuda.synchronize()
    q_host = s.q.cpu().pin_memory()
    out_host = torch.empty(o.out.shape, dtype=o.out.dtype).pin_memory()
    shape = ctypes.byref(dd_shape(w).c())
    stream = torch.cuda.current_stream().cuda_stream
    v_win = s.v_win.data_ptr() if s.v_win is not None else None
    for q_ptr, out_ptr in ((q_host.data_ptr(), o.out.data_ptr()),
                           (s.q.data_ptr(), out_host.data_ptr())):
        st_noalloc = dd.lib().dd_sparse_decode_attn_noalloc(
            shape, q_ptr, o.k_buf.data_ptr(), o.v_buf.data_ptr(), s.K.data_ptr(), v_win, out_ptr,
            stream)
        st_ws = dd.lib().dd_sparse_decode_attn(
            shape, q_ptr, o.k_buf.data_ptr(), o.v_buf.data_ptr(), s.K.data_ptr(), v_win, out_ptr,
            o.ws.data_ptr(), o.ws.numel(), stream)
        assert st_noalloc == dd.DD_ERR_INVALID_ARG
        assert st_ws == dd.DD_ERR_INVALID_ARG
