"""The shared input generator and the workload byte accounting."""
import json
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_outputs():
    ref = json.load(open(os.path.join(GOLDEN, "splitmix64.json")))
    g = synth.gen()
    got = [g.lib.syn_u64(ref["state"], i) for i in range(len(ref["outputs_hex"]))]
    assert got == [int(x, 16) for x in ref["outputs_hex"]]


def test_normals_moments_and_counter_property():
    n = 1 << 20
    x = np.empty(n, np.float32)
    synth.gen().lib.syn_fill_normal(99, 3, 0, n, 0.0, 1.0, synth.F32, x.ctypes.data, 4)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    # counter-based: a sub-range regenerated on its own is identical
    y = np.empty(1000, np.float32)
    synth.gen().lib.syn_fill_normal(99, 3, 12345, 1000, 0.0, 1.0, synth.F32, y.ctypes.data, 1)
    assert np.array_equal(y, x[12345:13345])


def test_slot_is_deterministic_and_bf16_rounded():
    w = synth.C2.scaled(batch=1, n_q_heads=2, n_kv_heads=2, ctx_len=300, top_k=16, window=4,
                        n_planted=4)
    a = synth.slot_numpy(w, 0)
    b = synth.slot_numpy(w, 0)
    c = synth.slot_numpy(w, 1)
    for k in ("q_spec", "q", "K", "V", "planted"):
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["K"], c["K"])
    f32 = synth.bf16_bits_to_f32(a["K"])
    # values are bf16: the low 16 bits of their fp32 patterns are zero
    assert np.all((f32.view(np.uint32) & 0xFFFF) == 0)
    # planted positions are distinct and outside the window
    for u in range(2):
        p = a["planted"][0, u]
        assert len(set(p.tolist())) == 4 and p.max() < 300 - 4


def test_spread_planting_positions():
    w = synth.C3.scaled(batch=1, n_q_heads=1, n_kv_heads=1, ctx_len=1000, top_k=16, window=64,
                        n_planted=8)
    p = synth.slot_numpy(w, 0)["planted"][0, 0]
    span = 1000 - 64
    assert p.tolist() == [((2 * i + 1) * span) // 16 for i in range(8)]


def test_worked_example_bytes():
    """The LLaMA-2-7B 32K workload gathers exactly the worked example's ~2 MB per
    layer per request (128 x 2 x 4096 x 2 bytes)."""
    ref = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    want = ref["top_k"] * ref["k_and_v"] * ref["hidden"] * ref["bytes_per_element"]
    assert want == ref["bytes_per_layer_per_request"]
    w = synth.C2
    assert w.n_q_heads * w.head_dim == ref["hidden"] and w.top_k == ref["top_k"]
    assert w.gather_bytes() // w.batch == want


def test_layer_scoped_buffer_independent_of_context():
    """O(n d) -> O(k d): the gathered rows of a layer do not grow with n."""
    a = synth.C2.gather_bytes()
    b = synth.C2.scaled(ctx_len=4 * synth.C2.ctx_len).gather_bytes()
    assert a == b and synth.C2.scaled(ctx_len=4 * synth.C2.ctx_len).k_bytes() == 4 * synth.C2.k_bytes()
