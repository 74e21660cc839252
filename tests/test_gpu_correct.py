"""Miss correction and predictability (the real query's top-k against the
prefetched, speculated one), through the C ABI, against the fp64 oracle.

The paper's claim (DualDecoder, Sec. 1): even an imperfect prediction of the
next token predicts most of the KV entries the next step needs, and the
remaining misses are corrected on the critical path.
"""
import numpy as np
import pytest
import torch

import sparse_kv_prefetch_gb300 as dd
import synth
from gpu_util import (Outputs, Slot, check_gather, check_unit_attention, check_unit_topk,
                      dd_shape, oracle_selection_score, run_layer, sample_units)

pytestmark = pytest.mark.gpu

CASES = {
    "c2_mini": synth.C2.scaled(batch=2, n_q_heads=4, n_kv_heads=4, ctx_len=5000),
    "c5_mini": synth.C5.scaled(batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=12000),
    "c1": synth.C1,
}


def _corrected(w, s, o):
    """Run the speculated path, then the correction with the real query."""
    run_layer(w, s, o)
    U = w.units
    idx_true = torch.empty_like(o.idx)
    kb, vb = torch.empty_like(o.k_buf), torch.empty_like(o.v_buf)
    miss = torch.empty(U, dtype=torch.int32, device="cuda")
    mass = torch.empty((U, 2), dtype=torch.float32, device="cuda")
    dd.correct_misses(dd_shape(w), s.q, s.K, o.idx, o.k_buf, o.v_buf, s.K_h, s.V_h, idx_true, kb,
                      vb, miss, mass, o.ws)
    torch.cuda.synchronize()
    return idx_true, kb, vb, miss, mass


@pytest.mark.parametrize("name", list(CASES))
def test_correction_against_oracle(name):
    w = CASES[name]
    s, o = Slot(w), Outputs(w)
    idx_true, kb, vb, miss, mass = _corrected(w, s, o)
    spec = o.idx.cpu().numpy()
    true = idx_true.cpu().numpy()
    miss, mass = miss.cpu().numpy(), mass.cpu().numpy()
    # the real query's top-k, as the oracle defines it
    for u in range(w.units):
        check_unit_topk(w, s, u, true[u], None, None, query=s.q_h)
        hits = np.isin(true[u], spec[u])
        assert miss[u] == w.top_k - hits.sum()
        a = oracle_selection_score(w, s, u, s.q_h)
        np.testing.assert_allclose(mass[u], [a[true[u][hits]].sum(), a[true[u]].sum()],
                                   rtol=2e-3, atol=1e-9)
    # the corrected rows are the host rows of the real top-k, bit for bit
    check_gather(w, s, true, kb, vb, range(w.units))
    # attention over them matches the oracle's attention over the real top-k
    out = torch.empty_like(o.out)
    dd.sparse_decode_attn(dd_shape(w), s.q, kb, vb, s.K, s.v_win, out, o.ws)
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    for u in range(w.units):
        check_unit_attention(w, s, u, true[u], out)
    dd.check_device()


def test_exact_prediction_has_no_misses():
    """With q = q_spec the real and the predicted top-k coincide."""
    w = CASES["c2_mini"].scaled(q_noise=0.0)
    s, o = Slot(w), Outputs(w)
    assert torch.equal(s.q_h, s.q_spec_h)
    idx_true, kb, vb, miss, mass = _corrected(w, s, o)
    assert torch.equal(idx_true, o.idx)
    assert int(miss.sum()) == 0
    assert torch.equal(kb, o.k_buf) and torch.equal(vb, o.v_buf)
    m = mass.cpu().numpy()
    assert np.array_equal(m[:, 0], m[:, 1])


def test_recall_falls_with_prediction_noise():
    """Recall |TopK(q_spec) & TopK(q)| / k is high for a close prediction and
    falls as the real query drifts away from the speculated one."""
    base = CASES["c2_mini"]
    recall = {}
    for sigma in (0.05, 0.3, 3.0):
        w = base.scaled(q_noise=sigma)
        s, o = Slot(w), Outputs(w)
        _, _, _, miss, mass = _corrected(w, s, o)
        recall[sigma] = 1.0 - miss.float().mean().item() / w.top_k
    assert recall[0.05] >= recall[0.3] >= recall[3.0]
    assert recall[0.05] > 0.8 and recall[3.0] < recall[0.05]


@pytest.mark.parametrize("name", ["c2_mini", "c5_mini"])
def test_decode_step_with_correction(name):
    """DD_STEP_CORRECT_MISSES: every layer attends over the real query's top-k;
    outputs and miss counts equal the per-layer calls, in every schedule."""
    w = CASES[name]
    D, L = 2, 4
    slots = [Slot(w, d) for d in range(D)]
    ref_out, ref_miss = [], []
    for d in range(D):
        o = Outputs(w)
        _, kb, vb, miss, _ = _corrected(w, slots[d], o)
        out = torch.empty_like(o.out)
        dd.sparse_decode_attn(dd_shape(w), slots[d].q, kb, vb, slots[d].K, slots[d].v_win, out, o.ws)
        ref_out.append(out)
        ref_miss.append(miss.cpu().numpy())
    ctx = dd.Ctx(dd_shape(w))
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    compute.wait_stream(torch.cuda.current_stream())
    for copy_stream, fused in ((copy, False), (None, False), (copy, True)):
        outs = [torch.full_like(ref_out[0], float("nan")) for _ in range(L)]
        layers = [dd.LayerIO(slots[l % D].q_spec, slots[l % D].q, slots[l % D].K,
                             slots[l % D].K_h, slots[l % D].V_h, slots[l % D].v_win, outs[l])
                  for l in range(L)]
        ctx.decode_step(layers, compute=compute, copy=copy_stream, correct_misses=True,
                        fused_topk=fused)
        misses, mass = ctx.correction_stats(L)
        torch.cuda.synchronize()
        for l in range(L):
            assert torch.equal(outs[l], ref_out[l % D]), f"layer {l}"
            assert np.array_equal(misses[l], ref_miss[l % D]), f"layer {l}"
    dd.check_device()
    ctx.close()


def test_full_size_correction_sampled_units():
    """The 7B-32K layer at full size: the real query's top-k on sampled units
    against the oracle, miss counts against the two index sets, corrected rows
    bit-exact on those units."""
    w = synth.C2
    s, o = Slot(w), Outputs(w)
    idx_true, kb, vb, miss, mass = _corrected(w, s, o)
    spec, true = o.idx.cpu().numpy(), idx_true.cpu().numpy()
    miss = miss.cpu().numpy()
    units = sample_units(w.units, n=4, seed=11)
    for u in units:
        check_unit_topk(w, s, u, true[u], None, None, query=s.q_h)
        assert miss[u] == w.top_k - np.isin(true[u], spec[u]).sum()
    check_gather(w, s, true, kb, vb, units)
    assert np.all(np.diff(true, axis=1) > 0)
    del s, o, kb, vb
    torch.cuda.empty_cache()
