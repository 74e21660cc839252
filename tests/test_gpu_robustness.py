"""Robustness of the C ABI on the GPU: event ordering under delayed streams,
no writes outside the output buffers (guard canaries), and the bounded
device-side wait giving up with DD_ERR_TIMEOUT while the context stays usable.
No test here faults, traps or hangs the GPU: the delays are bounded sleeps and
the expiring wait is a wait on a barrier nothing arrives at, with a 5 ms limit.
"""
import pytest
import torch

import sparse_kv_prefetch_gb300 as dd
import synth
from gpu_util import Outputs, Slot, dd_shape, run_layer

pytestmark = pytest.mark.gpu

W2 = synth.C2.scaled(batch=2, n_q_heads=4, n_kv_heads=4, ctx_len=5000)
W5 = synth.C5.scaled(batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=12000)


def _layers(w, slots, outs, L):
    return [dd.LayerIO(slots[l % len(slots)].q_spec, slots[l % len(slots)].q,
                       slots[l % len(slots)].K, slots[l % len(slots)].K_h,
                       slots[l % len(slots)].V_h, slots[l % len(slots)].v_win, outs[l])
            for l in range(L)]


@pytest.mark.parametrize("w", [W2, W5], ids=["mha", "gqa"])
def test_delayed_streams_keep_every_schedule_exact(w):
    """A 50 us sleep before every gather (copy stream late) or before every
    attention (compute stream late, so the scratch slots are released late)
    must not change any output: the events, not the timing, order the step."""
    D, L = 2, 5
    slots = [Slot(w, d) for d in range(D)]
    ctx = dd.Ctx(dd_shape(w))
    compute = torch.cuda.Stream()
    copy = torch.cuda.Stream(priority=-1)
    compute.wait_stream(torch.cuda.current_stream())
    ref = [torch.empty((w.batch, w.n_q_heads, w.head_dim), device="cuda") for _ in range(L)]
    ctx.decode_step(_layers(w, slots, ref, L), compute=compute, copy=None)
    for delay in ("copy", "compute", "copy+compute"):
        for sched in (dict(), dict(late_gather=True), dict(pipeline=True), dict(guarded=True)):
            outs = [torch.full_like(ref[0], float("nan")) for _ in range(L)]
            ctx.decode_step(_layers(w, slots, outs, L), compute=compute, copy=copy,
                            debug_delay=delay, **sched)
            compute.synchronize()
            for l in range(L):
                assert torch.equal(outs[l], ref[l]), f"delay {delay}, {sched}, layer {l}"
    dd.check_device()
    ctx.close()


def test_outputs_have_no_writes_outside_their_buffers():
    """Every output of the per-layer calls sits between two guard regions
    filled with a pattern; after the calls the guards are unchanged."""
    w = synth.C2.scaled(batch=2, n_q_heads=4, n_kv_heads=2, ctx_len=3001, top_k=77, window=9)
    s = Slot(w)
    o = Outputs(w)
    G = 4096  # guard elements on each side

    def guarded(t):
        flat = t.reshape(-1)
        buf = torch.empty(flat.numel() + 2 * G, dtype=t.dtype, device="cuda")
        buf.view(torch.uint8).fill_(0xA5)
        inner = buf[G:G + flat.numel()].view(t.shape)
        return buf, inner

    bufs = {}
    for name in ("idx", "sel", "lse", "k_buf", "v_buf", "out"):
        buf, inner = guarded(getattr(o, name))
        bufs[name] = buf
        setattr(o, name, inner)
    run_layer(w, s, o)
    torch.cuda.synchronize()
    for name, buf in bufs.items():
        raw = buf.view(torch.uint8)
        nbytes = G * buf.element_size()
        assert bool((raw[:nbytes] == 0xA5).all()), f"{name}: write before the buffer"
        assert bool((raw[-nbytes:] == 0xA5).all()), f"{name}: write after the buffer"


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """A wait that nothing completes gives up after 5 ms: check_device reports
    DD_ERR_TIMEOUT once, then the device and a context work as before."""
    dd.check_device()
    dd.debug_expire_wait(5_000_000)
    with pytest.raises(dd.DDError) as e:
        dd.check_device()
    assert e.value.status == dd.DD_ERR_TIMEOUT
    dd.check_device()  # the status word was cleared
    w = W2
    s = Slot(w)
    o1, o2 = Outputs(w), Outputs(w)
    run_layer(w, s, o1)
    ctx = dd.Ctx(dd_shape(w))
    out = torch.empty_like(o1.out)
    ctx.decode_step(_layers(w, [s], [out], 1))
    torch.cuda.synchronize()
    assert torch.equal(out, o1.out)
    with pytest.raises(dd.DDError):
        dd.debug_expire_wait(0)  # limits outside (0, 100 ms] are refused
    dd.check_device()
    ctx.close()
