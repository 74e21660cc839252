"""Helpers for the GPU parity tests: one layer slot on host and device, and the
parity checks against the fp64 oracle (tolerances from the method's statement:
indices exact outside a 1e-3 relative tie band, attention within 2e-3 (bf16)
or 1e-5 (fp32) max-abs, LSE within 1e-3 / 1e-4)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_kv_prefetch_gb300 as dd
import synth

BAND = 1e-3
TOL_OUT = {synth.F32: 1e-5, synth.BF16: 2e-3}
TOL_LSE = {synth.F32: 1e-4, synth.BF16: 1e-3}


def torch_dtype(w):
    return torch.bfloat16 if w.dtype == synth.BF16 else torch.float32


def dd_shape(w) -> dd.Shape:
    return dd.Shape(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ctx_len, w.top_k,
                    w.window, w.dtype)


def orc_shape(w) -> oracle.Shape:
    return oracle.Shape(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ctx_len, w.top_k,
                        w.window, w.dtype)


class Slot:
    """One layer slot: pinned host store (q_spec, q, K, V) and device copies."""

    def __init__(self, w, slot: int = 0, device: str = "cuda", fill=True, huge_pages=False,
                 store: str = "torch"):
        dt = torch_dtype(w)
        B, Hq, Hkv, d, n, W = (w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ctx_len,
                               w.window)
        self.w = w
        self.q_spec_h = torch.empty((B, Hq, d), dtype=dt, pin_memory=True)
        self.q_h = torch.empty((B, Hq, d), dtype=dt, pin_memory=True)
        if huge_pages or store in ("huge", "pinned"):  # the library's host store allocators
            kind = "huge" if huge_pages else store
            self.K_h = dd.host_empty((B, Hkv, n, d), dt, kind=kind)
            self.V_h = dd.host_empty((B, Hkv, n, d), dt, kind=kind)
        else:  # plain page-locked memory from torch
            self.K_h = torch.empty((B, Hkv, n, d), dtype=dt, pin_memory=True)
            self.V_h = torch.empty((B, Hkv, n, d), dtype=dt, pin_memory=True)
        self.planted = np.zeros((B, Hkv, max(w.n_planted, 1)), np.int32)
        if fill:
            synth.fill_slot(w, slot, self.q_spec_h, self.q_h, self.K_h, self.V_h, self.planted)
        self.to_device(device)

    def to_device(self, device="cuda"):
        w = self.w
        self.q_spec = self.q_spec_h.to(device)
        self.q = self.q_h.to(device)
        self.K = self.K_h.to(device)
        self.v_win = (self.V_h[:, :, w.ctx_len - w.window:, :].contiguous().to(device)
                      if w.window > 0 else None)


class Outputs:
    """Device outputs of one layer."""

    def __init__(self, w, device="cuda"):
        U = w.units
        self.idx = torch.empty((U, w.top_k), dtype=torch.int32, device=device)
        self.sel = torch.empty((U, w.top_k), dtype=torch.float32, device=device)
        self.lse = torch.empty((w.batch, w.n_q_heads), dtype=torch.float32, device=device)
        dt = torch_dtype(w)
        self.k_buf = torch.empty((U, w.top_k, w.head_dim), dtype=dt, device=device)
        self.v_buf = torch.empty_like(self.k_buf)
        self.out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32,
                               device=device)
        self.ws = torch.empty(dd.workspace_size(dd_shape(w)), dtype=torch.uint8, device=device)


def run_layer(w, s: Slot, o: Outputs, stream=None):
    """The three per-layer calls in order on one stream."""
    shp = dd_shape(w)
    dd.score_topk(shp, s.q_spec, s.K, o.idx, o.sel, o.lse, o.ws, stream=stream)
    dd.gather_h2d(shp, s.K_h, s.V_h, o.idx, o.k_buf, o.v_buf, stream=stream)
    dd.sparse_decode_attn(shp, s.q, o.k_buf, o.v_buf, s.K, s.v_win, o.out, o.ws, stream=stream)


def check_unit_topk(w, s: Slot, u: int, gpu_idx: np.ndarray, gpu_sel: np.ndarray,
                    gpu_lse, orc=None, query=None):
    """Selection of unit u against the oracle: exact set when the oracle's
    k-th / (k+1)-th relative gap exceeds BAND, otherwise a valid top-k within
    the band; selected scores (if given) and LSE (if given) within tolerance.
    The query defaults to the speculated one.  Returns the gap."""
    orc = orc or oracle.get()
    os_ = orc_shape(w)
    b, hk = divmod(u, w.n_kv_heads)
    logits, lse = orc.score_unit(os_, s.q_spec_h if query is None else query, s.K_h, b, hk)
    a = orc.selection_score(os_, logits, lse)
    want, want_sel, gap = orc.select_unit(os_, a)
    G, k, span = w.group, w.top_k, w.ctx_len - w.window
    if gpu_lse is not None:
        np.testing.assert_allclose(gpu_lse[b, hk * G:(hk + 1) * G], lse, rtol=0,
                                   atol=TOL_LSE[w.dtype], err_msg=f"LSE unit {u}")
    got = gpu_idx.astype(np.int64)
    assert np.all(np.diff(got) > 0), f"unit {u}: indices not strictly ascending"
    assert got[0] >= 0 and got[-1] < span, f"unit {u}: index outside [0, n-W)"
    if gap > BAND:
        assert np.array_equal(got, want), f"unit {u}: set differs (gap {gap:.3g})"
    else:
        kth = want_sel.min()
        must = np.nonzero(a[:span] > kth * (1 + BAND))[0]
        assert np.all(np.isin(must, got)), f"unit {u}: misses an entry above the band"
        assert np.all(a[got] >= kth * (1 - BAND)), f"unit {u}: takes an entry below the band"
    if gpu_sel is not None:
        np.testing.assert_allclose(gpu_sel, a[got], rtol=2e-3, atol=1e-12,
                                   err_msg=f"selection scores unit {u}")
    return gap


def oracle_selection_score(w, s: Slot, u: int, query, orc=None):
    """The oracle's selection score a[j] of unit u for a given query."""
    orc = orc or oracle.get()
    os_ = orc_shape(w)
    b, hk = divmod(u, w.n_kv_heads)
    logits, lse = orc.score_unit(os_, query, s.K_h, b, hk)
    return orc.selection_score(os_, logits, lse)


def check_unit_attention(w, s: Slot, u: int, gpu_idx: np.ndarray, gpu_out: np.ndarray, orc=None):
    """Attention of unit u recomputed by the oracle on the GPU's index set."""
    orc = orc or oracle.get()
    b, hk = divmod(u, w.n_kv_heads)
    G = w.group
    want = orc.attend_unit(orc_shape(w), s.q_h, s.K_h, s.V_h, b, hk, gpu_idx, True)
    got = gpu_out[b, hk * G:(hk + 1) * G].astype(np.float64)
    err = np.max(np.abs(got - want))
    assert err <= TOL_OUT[w.dtype], f"unit {u}: attention max-abs error {err:.3g}"
    return err


def check_gather(w, s: Slot, gpu_idx: np.ndarray, k_buf: torch.Tensor, v_buf: torch.Tensor,
                 units):
    """Gathered rows equal the host rows bit for bit."""
    Kh = s.K_h.view(w.units, w.ctx_len, w.head_dim)
    Vh = s.V_h.view(w.units, w.ctx_len, w.head_dim)
    kb = k_buf.cpu().view(w.units, w.top_k, w.head_dim)
    vb = v_buf.cpu().view(w.units, w.top_k, w.head_dim)
    for u in units:
        ix = torch.from_numpy(gpu_idx[u].astype(np.int64))
        assert torch.equal(kb[u].view(torch.int16 if kb.dtype == torch.bfloat16 else torch.int32),
                           Kh[u][ix].view(torch.int16 if kb.dtype == torch.bfloat16 else torch.int32))
        assert torch.equal(vb[u].view(torch.int16 if vb.dtype == torch.bfloat16 else torch.int32),
                           Vh[u][ix].view(torch.int16 if vb.dtype == torch.bfloat16 else torch.int32))


def sample_units(U: int, n: int = 6, seed: int = 0):
    rng = np.random.default_rng(seed)
    base = {0, U - 1, U // 2}
    extra = rng.choice(U, size=min(U, n), replace=False).tolist()
    return sorted(base | set(extra))
