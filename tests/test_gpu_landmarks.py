"""Landmark (chunk) selection through the C ABI, against the fp64 oracle.

DualDecoder paper, Sec. 1: the retrieval index comes from the current token
and static GPU-resident KV landmarks; Sec. 2.2: adjacent KV entries are
grouped into chunks with compressed landmarks and whole chunks are selected.
Checked here: the landmarks (chunk-mean keys), the chunk selection under the
same tie-band rule as the key-level top-k, its expansion to rows, the
attention over those rows, and the layer loop with DD_STEP_LANDMARKS
bit-identical to the standalone calls in every schedule.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import sparse_kv_prefetch_gb300 as dd
import synth
from gpu_util import (BAND, TOL_LSE, Outputs, Slot, check_gather, check_unit_attention,
                      dd_shape, orc_shape, sample_units)

pytestmark = pytest.mark.gpu

C1, C2, C5 = synth.C1, synth.C2, synth.C5

# (workload, chunk): every case has c | (n - W) and c | k
SMALL = {
    "c1_c16": (C1, 16),
    "c1_c8": (C1, 8),
    "c2_mini_c16": (C2.scaled(batch=2, n_q_heads=4, n_kv_heads=4, ctx_len=5184), 16),
    "c5_mini_c32": (C5.scaled(batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=12288), 32),
    "gqa2_d64_c4": (C2.scaled(batch=2, n_q_heads=4, n_kv_heads=2, head_dim=64, ctx_len=4116,
                              top_k=100, window=16, n_planted=20), 4),
    "f32_gqa2_d128_c8": (C1.scaled(batch=1, n_q_heads=4, n_kv_heads=2, head_dim=128,
                                   ctx_len=3000, top_k=96, window=8, n_planted=10), 8),
    "c2_mini_c2": (C2.scaled(batch=1, n_q_heads=2, n_kv_heads=2, ctx_len=2112), 2),
}
FULL = {"c2_c16": (C2, 16), "c5_c32": (C5, 32)}


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _unit_chunk_scores(w, s, chunk, u, Lu, orc):
    """The oracle's chunk selection scores of unit u over all M chunks: its
    scoring applied to the unit's landmarks (rounded to fp32, as stored) as a
    one-unit key cache with no window."""
    b, hk = divmod(u, w.n_kv_heads)
    G, M = w.group, Lu.shape[0]
    one = oracle.Shape(1, G, 1, w.head_dim, M, w.top_k // chunk, 0, synth.F32)
    q = s.q_spec_h[b, hk * G:(hk + 1) * G].float().contiguous()
    K = np.ascontiguousarray(Lu, dtype=np.float32)
    logits, lse = orc.score_unit(one, q, K, 0, 0)
    return orc.selection_score(one, logits, lse)


class Landmarks:
    """GPU landmarks and landmark selection of one slot."""

    def __init__(self, w, s: Slot, chunk: int):
        shp = dd_shape(w)
        M = (w.ctx_len - w.window) // chunk
        kc = w.top_k // chunk
        assert dd.landmarks_size(shp, chunk) == w.units * M * w.head_dim * 4
        self.L = torch.empty((w.batch, w.n_kv_heads, M, w.head_dim), dtype=torch.float32,
                             device="cuda")
        dd.build_landmarks(shp, chunk, s.K, self.L)
        self.idx = torch.empty((w.units, w.top_k), dtype=torch.int32, device="cuda")
        self.csel = torch.empty((w.units, kc), dtype=torch.float32, device="cuda")
        self.lse = torch.empty((w.batch, w.n_q_heads), dtype=torch.float32, device="cuda")
        self.ws = torch.empty(dd.landmarks_workspace_size(shp, chunk), dtype=torch.uint8,
                              device="cuda")
        dd.score_topk_landmarks(shp, chunk, s.q_spec, self.L, self.idx, self.csel, self.lse,
                                self.ws)
        torch.cuda.synchronize()


def _oracle_landmarks(w, s, chunk, u, orc):
    b, hk = divmod(u, w.n_kv_heads)
    return orc.landmarks_unit(orc_shape(w), chunk, s.K_h, b, hk)


def check_unit_landmark_selection(w, s, chunk, u, Lu, rows, csel, lse, orc):
    """Chunk selection of unit u (oracle landmarks Lu [M][d]) against the
    oracle: the exact chunk set when the oracle's k/c-th vs next chunk gap
    exceeds the band, else a valid selection within the band; rows = the
    chunks' positions; chunk scores and LSE within tolerance.  Returns the gap."""
    b, hk = divmod(u, w.n_kv_heads)
    G, kc = w.group, w.top_k // chunk
    want_rows, want_sel, want_lse, gap = orc.landmark_select_unit(orc_shape(w), chunk,
                                                                  s.q_spec_h, Lu, b, hk)
    a = _unit_chunk_scores(w, s, chunk, u, Lu, orc)
    np.testing.assert_allclose(lse[b, hk * G:(hk + 1) * G], want_lse, rtol=0,
                               atol=TOL_LSE[synth.F32], err_msg=f"chunk LSE unit {u}")
    got = rows.astype(np.int64)
    assert np.all(np.diff(got) > 0) and got[0] >= 0 and got[-1] < w.ctx_len - w.window
    chunks = got.reshape(kc, chunk)
    assert np.all(chunks % chunk == np.arange(chunk)), f"unit {u}: rows are not whole chunks"
    assert np.all(chunks - chunks[:, :1] == np.arange(chunk)), f"unit {u}: chunk split"
    cid = chunks[:, 0] // chunk
    if gap > BAND:
        assert np.array_equal(got, want_rows), f"unit {u}: chunk set differs (gap {gap:.3g})"
        np.testing.assert_allclose(csel, want_sel, rtol=2e-3, atol=1e-12)
    else:
        kth = np.sort(a)[::-1][kc - 1]
        must = np.nonzero(a > kth * (1 + BAND))[0]
        assert np.all(np.isin(must, cid)), f"unit {u}: misses a chunk above the band"
        assert np.all(a[cid] >= kth * (1 - BAND)), f"unit {u}: takes a chunk below the band"
    np.testing.assert_allclose(csel, a[cid], rtol=2e-3, atol=1e-12,
                               err_msg=f"chunk scores unit {u}")
    return gap


@pytest.mark.parametrize("name", list(SMALL))
def test_landmark_selection_small(name):
    w, chunk = SMALL[name]
    orc = oracle.get()
    s = Slot(w)
    lmk = Landmarks(w, s, chunk)
    Lg = lmk.L.cpu().numpy().reshape(w.units, -1, w.head_dim)
    rows, csel, lse = lmk.idx.cpu().numpy(), lmk.csel.cpu().numpy(), lmk.lse.cpu().numpy()
    gaps = []
    for u in range(w.units):
        Lu = _oracle_landmarks(w, s, chunk, u, orc)
        # fp32 sums of c values: a relative error of a few ulps times c
        np.testing.assert_allclose(Lg[u], Lu, rtol=1e-5, atol=1e-6 * chunk)
        gaps.append(check_unit_landmark_selection(w, s, chunk, u, Lu, rows[u], csel[u], lse,
                                                  orc))
    assert max(gaps) > BAND  # the exact-set branch is exercised
    # the rows feed the unchanged gather and attention
    o = Outputs(w)
    shp = dd_shape(w)
    dd.gather_h2d(shp, s.K_h, s.V_h, lmk.idx, o.k_buf, o.v_buf)
    dd.sparse_decode_attn(shp, s.q, o.k_buf, o.v_buf, s.K, s.v_win, o.out, o.ws)
    torch.cuda.synchronize()
    check_gather(w, s, rows, o.k_buf, o.v_buf, range(w.units))
    out = o.out.cpu().numpy()
    for u in range(w.units):
        check_unit_attention(w, s, u, rows[u], out, orc)


def test_chunk_of_identical_keys_has_that_key_as_landmark():
    """Every chunk made of one repeated key: each landmark is that key exactly
    (bf16 keys: the fp32 sum of 8 copies and its division by 8 are exact)."""
    w = C2.scaled(batch=1, n_q_heads=2, n_kv_heads=2, ctx_len=576, top_k=32, window=64)
    chunk = 8
    s = Slot(w)
    K = s.K_h.view(w.units, w.ctx_len, w.head_dim)
    M = (w.ctx_len - w.window) // chunk
    for u in range(w.units):
        K[u, :M * chunk] = K[u, 0:M * chunk:chunk].repeat_interleave(chunk, dim=0)
    s.to_device()
    lmk = Landmarks(w, s, chunk)
    want = K[:, 0:M * chunk:chunk].reshape(w.batch, w.n_kv_heads, M, w.head_dim)
    assert torch.equal(lmk.L.cpu(), want.float())


def _layers(w, slots, outs, lms, L, k_wins=None):
    """Layer inputs; with k_wins (one window-key buffer per slot, or None for
    W = 0) the key cache itself is left out."""
    return [dd.LayerIO(slots[l % len(slots)].q_spec, slots[l % len(slots)].q,
                       slots[l % len(slots)].K if k_wins is None else None,
                       slots[l % len(slots)].K_h, slots[l % len(slots)].V_h,
                       slots[l % len(slots)].v_win, outs[l], lms[l % len(lms)].L,
                       None if k_wins is None else k_wins[l % len(slots)])
            for l in range(L)]


@pytest.mark.parametrize("name", ["c1_c16", "c2_mini_c16", "c5_mini_c32"])
def test_landmark_decode_step_equals_calls_in_every_schedule(name):
    w, chunk = SMALL[name]
    D, L = 2, 5
    slots = [Slot(w, d) for d in range(D)]
    lms = [Landmarks(w, slots[d], chunk) for d in range(D)]
    ref = []
    shp = dd_shape(w)
    for d in range(D):
        o = Outputs(w)
        dd.gather_h2d(shp, slots[d].K_h, slots[d].V_h, lms[d].idx, o.k_buf, o.v_buf)
        dd.sparse_decode_attn(shp, slots[d].q, o.k_buf, o.v_buf, slots[d].K, slots[d].v_win,
                              o.out, o.ws)
        ref.append(o.out)
    ctx = dd.Ctx(shp)
    with pytest.raises(dd.DDError):  # no chunk set yet
        ctx.decode_step(_layers(w, slots, [ref[0]] * L, lms, L), landmarks=True)
    ctx.set_landmark_chunk(chunk)
    compute = torch.cuda.Stream()
    copy = torch.cuda.Stream(priority=-1)
    compute.wait_stream(torch.cuda.current_stream())
    runs = {}
    for sched, kw in {"overlap": dict(copy=copy, timing=True), "serial": dict(copy=None),
                      "late": dict(copy=copy, late_gather=True),
                      "pipeline": dict(copy=copy, pipeline=True),
                      "lsu": dict(copy=copy, gather_mode=1),
                      "fused": dict(copy=copy, fused_topk=True)}.items():
        outs = [torch.full((w.batch, w.n_q_heads, w.head_dim), float("nan"), device="cuda")
                for _ in range(L)]
        ctx.decode_step(_layers(w, slots, outs, lms, L), compute=compute, landmarks=True, **kw)
        if sched == "overlap":
            t = ctx.timings()
        runs[sched] = outs
    # Without the key cache on the device: landmarks plus the window's keys.
    k_wins = [s.K[:, :, w.ctx_len - w.window:, :].contiguous() if w.window else None
              for s in slots]
    for sched, kw in {"overlap_no_k": dict(copy=copy), "serial_no_k": dict(copy=None)}.items():
        outs = [torch.full((w.batch, w.n_q_heads, w.head_dim), float("nan"), device="cuda")
                for _ in range(L)]
        ctx.decode_step(_layers(w, slots, outs, lms, L, k_wins), compute=compute, landmarks=True,
                        **kw)
        runs[sched] = outs
    with pytest.raises(dd.DDError):  # no key cache and no landmark selection
        ctx.decode_step(_layers(w, slots, outs, lms, L, k_wins), compute=compute)
    # captured as a CUDA graph and replayed
    outs = [torch.full((w.batch, w.n_q_heads, w.head_dim), float("nan"), device="cuda")
            for _ in range(L)]
    ctx.capture_step(dd.Ctx.pack(_layers(w, slots, outs, lms, L, k_wins)), compute, copy=copy,
                     landmarks=True)
    for o in outs:
        o.fill_(float("nan"))
    compute.synchronize()
    ctx.replay_step(compute)
    ctx.replay_step(compute)
    compute.synchronize()
    runs["graph_no_k"] = outs
    torch.cuda.synchronize()
    for sched, outs in runs.items():
        for l in range(L):
            assert torch.equal(outs[l], ref[l % D]), f"{sched}, layer {l}: != standalone calls"
    # score (reads a bf16 query itself), top-k (writes the chunks' rows), gather (pinned
    # store: no host-page touch), attention (splits merged in the same kernel)
    per_layer = 1 + 1 + 1 + 1
    assert t["n_layers"] == L and t["launches"] == L * per_layer
    with pytest.raises(dd.DDError):  # not combinable with miss correction
        ctx.decode_step(_layers(w, slots, runs["serial"], lms, L), compute=compute,
                        landmarks=True, correct_misses=True)
    dd.check_device()
    ctx.close()


@pytest.mark.parametrize("name", list(FULL))
def test_landmark_full_size_sampled_units(name):
    """Full per-layer size, through the layer loop; sampled units against the
    oracle; every unit's rows are whole chunks in ascending order."""
    w, chunk = FULL[name]
    orc = oracle.get()
    s = Slot(w)
    lmk = Landmarks(w, s, chunk)
    ctx = dd.Ctx(dd_shape(w))
    ctx.set_landmark_chunk(chunk)
    outs = [torch.empty((w.batch, w.n_q_heads, w.head_dim), device="cuda") for _ in range(2)]
    compute = torch.cuda.Stream()
    copy = torch.cuda.Stream(priority=-1)
    compute.wait_stream(torch.cuda.current_stream())
    ctx.decode_step(_layers(w, [s], outs, [lmk], 2), compute=compute, copy=copy, landmarks=True)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    rows, csel, lse = lmk.idx.cpu().numpy(), lmk.csel.cpu().numpy(), lmk.lse.cpu().numpy()
    out = outs[0].cpu().numpy()
    units = sample_units(w.units, n=4, seed=w.cfg_id)
    for u in units:
        b, hk = divmod(u, w.n_kv_heads)
        Lu = _oracle_landmarks(w, s, chunk, u, orc)
        np.testing.assert_allclose(lmk.L[b, hk].cpu().numpy(), Lu, rtol=1e-5, atol=1e-6 * chunk)
        check_unit_landmark_selection(w, s, chunk, u, Lu, rows[u], csel[u], lse, orc)
        check_unit_attention(w, s, u, rows[u], out, orc)
    r = rows.reshape(w.units, -1, chunk).astype(np.int64)
    assert np.all(np.diff(rows, axis=1) > 0)
    assert np.all(r % chunk == np.arange(chunk))
    assert rows.min() >= 0 and rows.max() < w.ctx_len - w.window
    ctx.close()
    del s, lmk, outs
    _free()


def test_chunk_change_reuses_workspace_and_fused_selection_still_agrees():
    """Setting a smaller chunk after a larger one reuses the context's landmark
    workspace in a new layout; the fused selection (which keeps per-unit
    counters in that workspace) and the two-kernel one still agree."""
    w = C2.scaled(batch=1, n_q_heads=4, n_kv_heads=2, ctx_len=4160, top_k=64, window=64)
    s = Slot(w)
    L = 2
    ctx = dd.Ctx(dd_shape(w))
    ctx.set_landmark_chunk(8)  # M = 512: the larger workspace
    lm8 = Landmarks(w, s, 8)
    outs = [torch.empty((w.batch, w.n_q_heads, w.head_dim), device="cuda") for _ in range(L)]
    ctx.decode_step(_layers(w, [s], outs, [lm8], L), landmarks=True, fused_topk=True)
    ctx.set_landmark_chunk(16)  # M = 256: reuses it
    lm16 = Landmarks(w, s, 16)
    runs = []
    for fused in (True, False, True):
        o = [torch.full_like(outs[0], float("nan")) for _ in range(L)]
        ctx.decode_step(_layers(w, [s], o, [lm16], L), landmarks=True, fused_topk=fused)
        runs.append(o)
    torch.cuda.synchronize()
    for r in runs[1:]:
        for l in range(L):
            assert torch.equal(r[l], runs[0][l])
    dd.check_device()
    ctx.close()


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_every_chunk_selected_gives_every_row(dtype):
    """k = n - W: every chunk is selected, the rows are 0 .. n - W - 1 in
    order, and the attention equals the oracle's over all n positions."""
    base = C1 if dtype == synth.F32 else C2
    w = base.scaled(batch=1, n_q_heads=4, n_kv_heads=2, head_dim=64, ctx_len=528, top_k=512,
                    window=16)
    chunk = 16
    orc = oracle.get()
    s = Slot(w)
    lmk = Landmarks(w, s, chunk)
    rows = lmk.idx.cpu().numpy()
    for u in range(w.units):
        assert rows[u].tolist() == list(range(w.ctx_len - w.window))
    o = Outputs(w)
    shp = dd_shape(w)
    dd.gather_h2d(shp, s.K_h, s.V_h, lmk.idx, o.k_buf, o.v_buf)
    dd.sparse_decode_attn(shp, s.q, o.k_buf, o.v_buf, s.K, s.v_win, o.out, o.ws)
    torch.cuda.synchronize()
    out = o.out.cpu().numpy()
    for u in range(w.units):
        check_unit_attention(w, s, u, rows[u], out, orc)
