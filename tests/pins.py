"""Pins for the fp64 oracle: checks against what the mathematics and the paper fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
failure.  ``test_oracle_pins.py`` runs them on the oracle itself, and
``test_oracle_mutants.py`` runs them on copies of ``oracle.c`` with one planted
mistake each (a dropped term, a wrong sign or index, a swapped operand), which
must fail at least one pin.

None of these re-types the oracle's formulas.  They use closed forms (basis-vector
keys, equal logits, two-row softmax), invariants (probabilities sum to one; the
group score sums to G; k = n - W reproduces dense attention), brute force (every
k-subset of a tiny input) and planted-key recovery.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

from oracle import BF16, F32, Shape

import synth


def _rng(seed):
    return np.random.default_rng(seed)


def _f32(shape, seed, scale=1.0):
    return (_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bit patterns (nearest even)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


# --------------------------------------------------------------------------
# scoring / softmax
# --------------------------------------------------------------------------

def pin_softmax_sums_to_one(orc):
    """sum_j alpha_h[j] = 1 (1e-12) per query head; the group score sums to G."""
    for (B, Hq, Hkv, d, n) in [(2, 2, 2, 8, 257), (2, 4, 2, 16, 130), (1, 8, 2, 64, 77)]:
        s = Shape(B, Hq, Hkv, d, n, 3, 0, F32)
        q = _f32((B, Hq, d), 1)
        K = _f32((B, Hkv, n, d), 2, scale=2.0)
        for b in range(B):
            for hk in range(Hkv):
                lg, lse = orc.score_unit(s, q, K, b, hk)
                for g in range(s.group):
                    assert abs(np.exp(lg[g] - lse[g]).sum() - 1.0) < 1e-12
                a = orc.selection_score(s, lg, lse)
                assert abs(a.sum() - s.group) < 1e-12 * n


def pin_logits_basis_keys(orc):
    """Keys that are scaled basis vectors give hand-computable logits.

    KV head hk holds K[j] = (hk + 1) e_(j mod d), so for the query head h of
    group hk the logit is s_h[j] = (hk + 1) q[h][j mod d] / sqrt(d).  Run with
    B = 2 and GQA (H_q = 4, H_kv = 2), in fp32 and in bf16 with exactly
    representable values, this pins the 1/sqrt(d) scale, the dot-product
    operand order, the query-head -> KV-head map and bf16 widening.
    """
    B, Hq, Hkv, d, n = 2, 4, 2, 4, 11
    qv = np.array([[[1.0, -2.0, 0.5, 3.0], [0.25, 1.5, -1.0, 2.0],
                    [-3.0, 0.75, 4.0, -0.5], [2.5, -1.25, 1.0, 0.125]],
                   [[-1.0, 2.0, -0.5, 0.0], [1.0, 1.0, 1.0, 1.0],
                    [0.5, -0.25, 8.0, -6.0], [-2.0, 3.5, -4.5, 1.75]]], np.float32)
    K = np.zeros((B, Hkv, n, d), np.float32)
    for b in range(B):
        for hk in range(Hkv):
            for j in range(n):
                K[b, hk, j, j % d] = (hk + 1) * (1 + b)
    for dtype in (F32, BF16):
        s = Shape(B, Hq, Hkv, d, n, 2, 0, dtype)
        qs = qv if dtype == F32 else _bf16_bits(qv)
        Ks = K if dtype == F32 else _bf16_bits(K)
        for b in range(B):
            for hk in range(Hkv):
                lg, lse = orc.score_unit(s, qs, Ks, b, hk)
                for g in range(s.group):
                    h = hk * s.group + g
                    want = np.array([(hk + 1) * (1 + b) * float(qv[b, h, j % d]) / 2.0
                                     for j in range(n)])
                    assert np.array_equal(lg[g], want), (dtype, b, hk, g)
                    # log-sum-exp of these hand values, with the largest factored out
                    m = want.max()
                    assert abs(lse[g] - (m + math.log(sum(math.exp(x - m) for x in want)))) < 1e-12


def pin_group_score_two_heads(orc):
    """GQA group of two heads that disagree, in closed form.

    d = 2, q_0 = (c, 0), q_1 = (0, c), keys (1, 0), (0, 1), (0.8, 0.8); with
    t = c / sqrt 2 and Z = e^t + 1 + e^(0.8 t), each head's probabilities are
    a permutation of (e^t, 1, e^(0.8 t)) / Z, so the group score is
    a = ((e^t + 1)/Z, (e^t + 1)/Z, 2 e^(0.8 t)/Z).  For c = sqrt 2 the shared
    key wins (2 e^0.8 > e + 1) although each head alone prefers its own key.
    """
    c = math.sqrt(2.0)
    s = Shape(1, 2, 1, 2, 3, 1, 0, F32)
    q = np.array([[[c, 0.0], [0.0, c]]], np.float32)
    K = np.array([[[[1.0, 0.0], [0.0, 1.0], [0.8, 0.8]]]], np.float32)
    lg, lse = orc.score_unit(s, q, K, 0, 0)
    a = orc.selection_score(s, lg, lse)
    t = float(np.float32(c)) / math.sqrt(2.0)
    e8 = math.exp(float(np.float32(0.8)) * t)
    Z = math.exp(t) + 1.0 + e8
    want = [(math.exp(t) + 1.0) / Z, (math.exp(t) + 1.0) / Z, 2.0 * e8 / Z]
    assert np.max(np.abs(a - want)) < 1e-12
    idx, _, _ = orc.select_unit(s, a)
    assert idx.tolist() == [2]


def pin_lse_equal_logits(orc):
    """q = 0 gives n equal logits: LSE = log n and every alpha = 1/n."""
    for n in (1, 2, 1000, 4097):
        s = Shape(1, 2, 1, 8, n, 1, 0, F32)
        q = np.zeros((1, 2, 8), np.float32)
        K = _f32((1, 1, n, 8), 3)
        lg, lse = orc.score_unit(s, q, K, 0, 0)
        assert np.all(lg == 0.0)
        assert abs(lse[0] - math.log(n)) < 1e-12 and abs(lse[1] - math.log(n)) < 1e-12


def pin_logits_d1(orc):
    """d = 1: q = 2, keys (0, 1, -1, 3) give logits (0, 2, -2, 6) exactly."""
    s = Shape(1, 1, 1, 1, 4, 1, 0, F32)
    q = np.array([[[2.0]]], np.float32)
    K = np.array([[[[0.0], [1.0], [-1.0], [3.0]]]], np.float32)
    lg, lse = orc.score_unit(s, q, K, 0, 0)
    assert np.array_equal(lg[0], [0.0, 2.0, -2.0, 6.0])
    want = 6.0 + math.log(math.exp(-6.0) + math.exp(-4.0) + math.exp(-8.0) + 1.0)
    assert abs(lse[0] - want) < 1e-13


# --------------------------------------------------------------------------
# selection
# --------------------------------------------------------------------------

def _brute_topk(a, span, k):
    """The unique k-subset S of [0, span) such that every member beats every
    non-member in the order (a desc, index asc) -- found by trying all subsets."""
    found = []
    for S in itertools.combinations(range(span), k):
        inside = set(S)
        ok = all((a[i] > a[j]) or (a[i] == a[j] and i < j)
                 for i in inside for j in range(span) if j not in inside)
        if ok:
            found.append(S)
    assert len(found) == 1
    return list(found[0])


def pin_topk_bruteforce(orc):
    """Exhaustive check on tiny inputs, with forced ties and a window."""
    rng = _rng(7)
    for trial in range(60):
        n = int(rng.integers(2, 11))
        W = int(rng.integers(0, min(3, n - 1) + 1))
        span = n - W
        levels = int(rng.integers(1, 5))  # few levels => many exact ties
        a = rng.integers(0, levels, size=n).astype(np.float64) + 0.5
        if trial % 3 == 0:
            a = rng.random(n)
        if W > 0:
            a[span:] = 100.0  # window positions are never candidates
        for k in range(1, span + 1):
            s = Shape(1, 1, 1, 1, n, k, W, F32)
            idx, sel, gap = orc.select_unit(s, a)
            want = _brute_topk(a, span, k)
            assert idx.tolist() == want, (a.tolist(), W, k, idx.tolist(), want)
            assert np.array_equal(sel, a[want])
            # relative gap between the k-th and (k+1)-th value of the order
            order = sorted(range(span), key=lambda j: (-a[j], j))
            if k < span:
                kth, nxt = a[order[k - 1]], a[order[k]]
                assert gap == (kth - nxt) / kth
            else:
                assert gap == math.inf


def pin_topk_window_boundary(orc):
    """The largest value just inside [0, n-W) is taken; one at n-W is not."""
    n, W = 20, 5
    a = np.linspace(0.1, 0.2, n)
    a[n - W] = 9.0
    a[n - W - 1] = 8.0
    s = Shape(1, 1, 1, 1, n, 1, W, F32)
    idx, _, _ = orc.select_unit(s, a)
    assert idx.tolist() == [n - W - 1]


def pin_planted_recovery(orc):
    """Planted high-affinity keys (3 sqrt(d) q_spec/|q_spec| + noise) are all
    selected: tiny fp32 MHA, a bf16 MHA case and a bf16 GQA case."""
    cases = [synth.C1,
             synth.C2.scaled(batch=2, n_q_heads=4, n_kv_heads=4, ctx_len=1500, top_k=40,
                             window=8, n_planted=12),
             synth.C5.scaled(batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=3000, top_k=64,
                             window=0, n_planted=16)]
    for w in cases:
        d = synth.slot_numpy(w, 0)
        s = Shape(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ctx_len, w.top_k,
                  w.window, w.dtype)
        r = orc.layer(s, d["q_spec"], d["q"], d["K"], d["V"], nthreads=4)
        for u in range(w.units):
            b, hk = divmod(u, w.n_kv_heads)
            planted = set(d["planted"][b, hk].tolist())
            assert planted <= set(r["idx"][u].tolist()), (w.name, u)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def _attn_case(B, Hq, Hkv, d, n, W, dtype, seed):
    q = _f32((B, Hq, d), seed)
    K = _f32((B, Hkv, n, d), seed + 1)
    V = _f32((B, Hkv, n, d), seed + 2)
    if dtype == BF16:
        q, K, V = _bf16_bits(q), _bf16_bits(K), _bf16_bits(V)
    return q, K, V


def pin_sparse_full_equals_dense(orc):
    """k = n - W with the window reproduces dense softmax attention (1e-12)."""
    for (B, Hq, Hkv, d, n, W, dt) in [(2, 2, 2, 8, 50, 7, F32), (2, 4, 2, 16, 33, 0, BF16),
                                      (1, 8, 2, 64, 70, 16, BF16)]:
        s = Shape(B, Hq, Hkv, d, n, n - W, W, dt)
        q, K, V = _attn_case(B, Hq, Hkv, d, n, W, dt, 11)
        for b in range(B):
            for hk in range(Hkv):
                sparse = orc.attend_unit(s, q, K, V, b, hk, np.arange(n - W), True)
                dense = orc.dense_unit(s, q, K, V, b, hk)
                assert np.max(np.abs(sparse - dense)) < 1e-12


def pin_attention_single_row(orc):
    """W = 0, k = 1: the softmax over one row is 1, so o = V[j] exactly."""
    B, Hq, Hkv, d, n = 2, 4, 2, 8, 40
    s = Shape(B, Hq, Hkv, d, n, 1, 0, F32)
    q, K, V = _attn_case(B, Hq, Hkv, d, n, 0, F32, 21)
    for b in range(B):
        for hk in range(Hkv):
            j = 3 + 5 * b + 11 * hk
            o = orc.attend_unit(s, q, K, V, b, hk, np.array([j]), True)
            for g in range(s.group):
                assert np.array_equal(o[g], V[b, hk, j].astype(np.float64))


def pin_attention_equal_keys(orc):
    """All keys equal: every row gets weight 1/|S|, so o = mean of V over S."""
    B, Hq, Hkv, d, n, W = 2, 2, 2, 8, 30, 4
    s = Shape(B, Hq, Hkv, d, n, 5, W, F32)
    q = _f32((B, Hq, d), 31)
    K = np.broadcast_to(_f32((1, 1, 1, d), 32), (B, Hkv, n, d)).copy()
    V = _f32((B, Hkv, n, d), 33)
    idx = np.array([0, 4, 9, 17, 20], np.int32)
    for b in range(B):
        for hk in range(Hkv):
            o = orc.attend_unit(s, q, K, V, b, hk, idx, True)
            rows = list(idx) + list(range(n - W, n))
            want = V[b, hk, rows].astype(np.float64).mean(axis=0)
            assert np.max(np.abs(o[0] - want)) < 1e-12


def pin_attention_two_rows(orc):
    """d = 2, q = (c, 0), keys e1, e2, values e1, e2: o = (sigma, 1 - sigma)
    with sigma = 1 / (1 + exp(-c / sqrt 2)), the two-way softmax."""
    for c in (0.0, 1.0, -3.0, 7.5):
        s = Shape(1, 1, 1, 2, 2, 2, 0, F32)
        q = np.array([[[c, 0.0]]], np.float32)
        K = np.array([[[[1.0, 0.0], [0.0, 1.0]]]], np.float32)
        V = K.copy()
        o = orc.attend_unit(s, q, K, V, 0, 0, np.array([0, 1]), True)
        sig = 1.0 / (1.0 + math.exp(-c / math.sqrt(2.0)))
        assert abs(o[0, 0] - sig) < 1e-14 and abs(o[0, 1] - (1.0 - sig)) < 1e-14


def pin_attention_window_only(orc):
    """The window alone: with idx empty, the result only depends on rows
    [n-W, n) -- changing any earlier row of K or V leaves it unchanged, while
    changing the first window row changes it."""
    B, Hq, Hkv, d, n, W = 1, 2, 1, 8, 25, 6
    s = Shape(B, Hq, Hkv, d, n, 1, W, F32)
    q, K, V = _attn_case(B, Hq, Hkv, d, n, W, F32, 41)
    base = orc.attend_unit(s, q, K, V, 0, 0, np.zeros(0, np.int32), True)
    K2, V2 = K.copy(), V.copy()
    K2[0, 0, : n - W] += 5.0
    V2[0, 0, : n - W] -= 3.0
    assert np.array_equal(orc.attend_unit(s, q, K2, V2, 0, 0, np.zeros(0, np.int32), True), base)
    V3 = V.copy()
    V3[0, 0, n - W] += 1.0
    assert not np.array_equal(orc.attend_unit(s, q, K, V3, 0, 0, np.zeros(0, np.int32), True), base)


# --------------------------------------------------------------------------
# landmark (chunk) selection
# --------------------------------------------------------------------------

def pin_landmarks_chunk1_is_plain_topk(orc):
    """With one position per chunk the landmark is the key itself, so chunk
    selection must reproduce the (separately pinned) plain top-k: the same rows,
    for MHA and for a GQA group.  Without a window the chunk softmax covers the
    same positions as the plain one, so the scores and LSE agree too (with a
    window the chunks exclude it and the normalisation differs)."""
    for (B, Hq, Hkv, d, n, k, W, dt) in [(2, 2, 2, 8, 90, 9, 5, F32), (1, 8, 2, 16, 70, 6, 0, BF16)]:
        s = Shape(B, Hq, Hkv, d, n, k, W, dt)
        q, K, _ = _attn_case(B, Hq, Hkv, d, n, W, dt, 51)
        for b in range(B):
            for hk in range(Hkv):
                L = orc.landmarks_unit(s, 1, K, b, hk)
                Kf = K if dt == F32 else synth.bf16_bits_to_f32(K)
                assert np.array_equal(L, Kf[b, hk, : n - W].astype(np.float64))
                rows, sel, lse, gap = orc.landmark_select_unit(s, 1, q, L, b, hk)
                lg, lse0 = orc.score_unit(s, q, K, b, hk)
                a = orc.selection_score(s, lg, lse0)
                idx, sel0, gap0 = orc.select_unit(s, a)
                assert rows.tolist() == idx.tolist()
                if W == 0:
                    np.testing.assert_allclose(sel, sel0, rtol=1e-12)
                    np.testing.assert_allclose(lse, lse0, rtol=1e-12)


def pin_landmark_is_chunk_mean(orc):
    """Keys j * e_t (an arithmetic run) have the closed-form chunk mean
    (m c + (c - 1)/2) e_t; positions of the window form no chunk."""
    B, Hq, Hkv, d, n, W, c = 2, 2, 2, 4, 48, 8, 8
    s = Shape(B, Hq, Hkv, d, n, 8, W, F32)
    K = np.zeros((B, Hkv, n, d), np.float32)
    for b in range(B):
        for hk in range(Hkv):
            K[b, hk, :, (b + 2 * hk) % d] = np.arange(n) * (1 + hk + b)
    for b in range(B):
        for hk in range(Hkv):
            L = orc.landmarks_unit(s, c, K, b, hk)
            assert L.shape == ((n - W) // c, d)
            for m in range(L.shape[0]):
                want = np.zeros(d)
                want[(b + 2 * hk) % d] = (m * c + (c - 1) / 2) * (1 + hk + b)
                assert np.array_equal(L[m], want)


def pin_landmark_selection_by_hand(orc):
    """Chunks of equal keys v_m e_1 and q = (x, 0) give chunk logits x v_m / sqrt 2:
    the chunks with the largest v_m win, ties to the lower chunk, and each
    selected chunk contributes all of its positions."""
    d, c, W = 2, 4, 3
    v = [1.0, 5.0, 2.0, 5.0, 0.5, 4.0, 5.0]  # 7 chunks, a three-way tie at 5
    n = len(v) * c + W
    for kc, want_chunks in [(1, [1]), (2, [1, 3]), (3, [1, 3, 6]), (4, [1, 3, 5, 6])]:
        s = Shape(1, 1, 1, d, n, kc * c, W, F32)
        K = np.zeros((1, 1, n, d), np.float32)
        for m, vm in enumerate(v):
            K[0, 0, m * c:(m + 1) * c, 0] = vm
        K[0, 0, n - W:, 0] = 100.0  # the window never competes
        q = np.array([[[0.7, 0.0]]], np.float32)
        L = orc.landmarks_unit(s, c, K, 0, 0)
        rows, sel, lse, gap = orc.landmark_select_unit(s, c, q, L, 0, 0)
        assert rows.tolist() == [m * c + r for m in want_chunks for r in range(c)], (kc, rows)
        lg = np.array([float(np.float32(0.7)) * vm / math.sqrt(2.0) for vm in v])
        al = np.exp(lg - lg.max()) / np.exp(lg - lg.max()).sum()
        np.testing.assert_allclose(sel, al[want_chunks], rtol=1e-12)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
