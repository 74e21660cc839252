"""The interleaved host store ([B][H_kv][n][2][d], each position's K row then its
V row) gives exactly the bytes and outputs of separate K and V stores: the
gather in both modes and several geometries, the layer loop in the overlapped
and serial schedules, and miss correction, which reads rows from the store."""
import pytest
import torch

import sparse_kv_prefetch_gb300 as dd
import synth
from gpu_util import Outputs, Slot, dd_shape, run_layer

pytestmark = pytest.mark.gpu

CASES = {
    "c2_mini": synth.C2.scaled(batch=2, n_q_heads=4, n_kv_heads=4, ctx_len=5000),
    "c5_mini": synth.C5.scaled(batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=12000),
    "c1": synth.C1,
}


def interleaved(s: Slot):
    """The slot's K and V host stores as one page-locked [B][H_kv][n][2][d] store."""
    kv = torch.empty(s.K_h.shape[:3] + (2,) + s.K_h.shape[3:], dtype=s.K_h.dtype,
                     pin_memory=True)
    kv[:, :, :, 0, :] = s.K_h
    kv[:, :, :, 1, :] = s.V_h
    return kv


def _bytes(t):
    return t.view(torch.uint8)


@pytest.mark.parametrize("name", list(CASES))
def test_gather_from_interleaved_store_is_identical(name):
    w = CASES[name]
    s, o = Slot(w), Outputs(w)
    run_layer(w, s, o)
    kv = interleaved(s)
    kb, vb = torch.empty_like(o.k_buf), torch.empty_like(o.v_buf)
    try:
        for mode, geom in ((0, (100, 4096, 3)), (0, (200, 8192, 4)), (0, (13, 16384, 6)),
                           (1, (100, 256)), (1, (30, 64))):
            if mode == 0:
                dd.set_gather_geometry(*geom)
            else:
                dd.set_gather_lsu_geometry(*geom)
            kb.zero_()
            vb.zero_()
            dd.gather_h2d_kv(dd_shape(w), kv, o.idx, kb, vb, mode=mode)
            torch.cuda.synchronize()
            assert torch.equal(_bytes(kb), _bytes(o.k_buf)), (mode, geom)
            assert torch.equal(_bytes(vb), _bytes(o.v_buf)), (mode, geom)
    finally:
        dd.set_gather_geometry()
        dd.set_gather_lsu_geometry()
    # runs of consecutive positions (as landmark chunks select) are still copied row by row
    U, k = w.units, w.top_k
    runs = (torch.arange(k, dtype=torch.int32) + 7).repeat(U, 1).contiguous().cuda()
    ka, va = torch.empty_like(kb), torch.empty_like(vb)
    dd.gather_h2d(dd_shape(w), s.K_h, s.V_h, runs, ka, va)
    dd.gather_h2d_kv(dd_shape(w), kv, runs, kb, vb)
    torch.cuda.synchronize()
    assert torch.equal(_bytes(ka), _bytes(kb)) and torch.equal(_bytes(va), _bytes(vb))
    dd.check_device()


@pytest.mark.parametrize("name", ["c2_mini", "c5_mini"])
def test_layer_loop_over_interleaved_store(name):
    w = CASES[name]
    D, L = 2, 4
    slots = [Slot(w, d_) for d_ in range(D)]
    kvs = [interleaved(s) for s in slots]
    shape = dd_shape(w)
    ctx = dd.Ctx(shape)
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream(priority=-1)
    compute.wait_stream(torch.cuda.current_stream())

    def layers(outs, inter):
        return [dd.LayerIO(slots[l % D].q_spec, slots[l % D].q, slots[l % D].K,
                           None if inter else slots[l % D].K_h,
                           None if inter else slots[l % D].V_h,
                           slots[l % D].v_win, outs[l],
                           kv_host=kvs[l % D] if inter else None) for l in range(L)]

    def new_outs():
        return [torch.full((w.batch, w.n_q_heads, w.head_dim), float("nan"), device="cuda")
                for _ in range(L)]

    for kw in (dict(copy=copy), dict(copy=None), dict(copy=copy, correct_misses=True)):
        ref, got = new_outs(), new_outs()
        ctx.decode_step(layers(ref, False), compute=compute, **kw)
        ctx.decode_step(layers(got, True), compute=compute, **kw)
        torch.cuda.synchronize()
        for l in range(L):
            assert torch.equal(ref[l], got[l]), (kw, l)
    # a layer naming both kinds of store, or neither, is refused
    bad = layers(new_outs(), True)
    bad[1] = bad[1]._replace(k_host=slots[1].K_h, v_host=slots[1].V_h)
    with pytest.raises(dd.DDError) as e:
        ctx.decode_step(bad, compute=compute, copy=copy)
    assert e.value.status == dd.DD_ERR_INVALID_ARG
    bad[1] = bad[1]._replace(k_host=None, v_host=None, kv_host=None)
    with pytest.raises(dd.DDError) as e:
        ctx.decode_step(bad, compute=compute, copy=copy)
    assert e.value.status == dd.DD_ERR_INVALID_ARG
    ctx.close()
    dd.check_device()


def test_miss_correction_from_interleaved_store():
    """dd_correct_misses_kv fetches the same rows, counts the same misses and
    the same selection mass as dd_correct_misses over separate stores."""
    w = CASES["c5_mini"]
    s, o = Slot(w), Outputs(w)
    run_layer(w, s, o)
    kv = interleaved(s)
    U, k = w.units, w.top_k
    shape = dd_shape(w)
    outs = []
    for inter in (False, True):
        idx = torch.empty((U, k), dtype=torch.int32, device="cuda")
        kb, vb = torch.empty_like(o.k_buf), torch.empty_like(o.v_buf)
        miss = torch.empty(U, dtype=torch.int32, device="cuda")
        mass = torch.empty((U, 2), dtype=torch.float32, device="cuda")
        if inter:
            dd.correct_misses_kv(shape, s.q, s.K, o.idx, o.k_buf, o.v_buf, kv, idx, kb, vb,
                                 miss, mass, o.ws)
        else:
            dd.correct_misses(shape, s.q, s.K, o.idx, o.k_buf, o.v_buf, s.K_h, s.V_h, idx, kb,
                              vb, miss, mass, o.ws)
        torch.cuda.synchronize()
        outs.append((idx, kb, vb, miss, mass))
    for a, b in zip(*outs):
        assert torch.equal(_bytes(a), _bytes(b))
    assert int(outs[0][3].sum()) > 0  # the real query does miss some rows here
