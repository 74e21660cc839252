"""Every logit of the scoring step against the fp64 oracle, to the fp32
rounding bound of a d-term dot product.

The scoring kernel has two consumers: bf16 keys scored by two, four or eight
query heads per KV head go through the tensor cores (16-row tiles, each stage
filled as two halves), single heads and fp32 keys through the per-lane form
(a build option sends bf16 single heads to the tensor cores too; these cases
then cover that).  The shapes below take both, with context lengths whose
last stage ends in the first half, in the second half, and on a stage
boundary, over several chunks per unit.

The logits are read from the workspace, whose first region holds them as fp32
[B][H_q][round_up(n, 4)] (dd_workspace_size).
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_kv_prefetch_gb300 as dd
import synth
from gpu_util import Outputs, Slot, dd_shape, orc_shape

pytestmark = pytest.mark.gpu

C1, C2 = synth.C1, synth.C2
CASES = {
    # tensor-core form (bf16)
    "g4_d128_tail_in_second_half": C2.scaled(batch=2, n_q_heads=8, n_kv_heads=2, ctx_len=3001,
                                             top_k=64, window=0),
    "g4_d128_tail_in_first_half": C2.scaled(batch=1, n_q_heads=8, n_kv_heads=2, ctx_len=2961,
                                            top_k=64, window=0),
    "g4_d128_whole_stages": C2.scaled(batch=1, n_q_heads=4, n_kv_heads=1, ctx_len=4096,
                                      top_k=64, window=0),
    "g2_d64_tail_in_second_half": C2.scaled(batch=2, n_q_heads=4, n_kv_heads=2, head_dim=64,
                                            ctx_len=3050, top_k=64, window=0),
    "g2_d64_tail_in_first_half": C2.scaled(batch=1, n_q_heads=2, n_kv_heads=1, head_dim=64,
                                           ctx_len=3001, top_k=64, window=0),
    "g8_d128": C2.scaled(batch=1, n_q_heads=16, n_kv_heads=2, ctx_len=2500, top_k=64, window=0),
    "g8_d256_tail_in_second_half": C2.scaled(batch=1, n_q_heads=16, n_kv_heads=2, head_dim=256,
                                             ctx_len=3001, top_k=64, window=0),
    "g8_d256_tail_in_first_half": C2.scaled(batch=1, n_q_heads=8, n_kv_heads=1, head_dim=256,
                                            ctx_len=2990, top_k=64, window=0),
    # per-lane form (bf16, one head per KV head)
    "mha_d128_tail_in_second_half": C2.scaled(batch=2, n_q_heads=2, n_kv_heads=2,
                                              ctx_len=3001, top_k=64, window=0),
    "mha_d128_tail_in_first_half": C2.scaled(batch=1, n_q_heads=2, n_kv_heads=2, ctx_len=2961,
                                             top_k=64, window=0),
    "mha_d64": C2.scaled(batch=1, n_q_heads=3, n_kv_heads=3, head_dim=64, ctx_len=3050,
                         top_k=64, window=0),
    "mha_d256": C2.scaled(batch=1, n_q_heads=2, n_kv_heads=2, head_dim=256, ctx_len=3001,
                          top_k=64, window=0),
    # per-lane form (fp32 keys)
    "f32_g4_d128": C1.scaled(batch=1, n_q_heads=8, n_kv_heads=2, head_dim=128, ctx_len=2600,
                             top_k=64, window=0),
    "f32_mha_d64": C1.scaled(batch=2, n_q_heads=2, n_kv_heads=2, ctx_len=3001, top_k=64,
                             window=0),
}


def _as_f64(x, w):
    a = np.asarray(x.cpu() if torch.is_tensor(x) else x)
    if w.dtype == synth.BF16:
        a = a.view(np.uint16) if a.dtype != np.uint16 else a
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


@pytest.mark.parametrize("name", list(CASES))
def test_logits_match_oracle_within_fp32_bound(name):
    w = CASES[name]
    s, o = Slot(w), Outputs(w)
    dd.score_topk(dd_shape(w), s.q_spec, s.K, o.idx, o.sel, o.lse, o.ws)
    torch.cuda.synchronize()
    B, Hq, Hkv, d, n, G = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ctx_len, w.group
    ldn = (n + 3) // 4 * 4
    got = o.ws[:B * Hq * ldn * 4].view(torch.float32).view(B, Hq, ldn)[:, :, :n].cpu().numpy()
    assert np.isfinite(got).all()
    orc = oracle.get()
    os_ = orc_shape(w)
    q = _as_f64(s.q_spec_h.view(torch.int16) if w.dtype == synth.BF16 else s.q_spec_h, w)
    K = _as_f64(s.K_h.view(torch.int16) if w.dtype == synth.BF16 else s.K_h, w)
    scale = 1.0 / np.sqrt(d)
    for b in range(B):
        for hk in range(Hkv):
            want, _ = orc.score_unit(os_, s.q_spec_h, s.K_h, b, hk)
            # |sum_i q_i k_i| rounding bound: d additions of exact products
            # (bf16 x bf16 and fp32 x fp32 products round at most once), each
            # off by at most one fp32 ulp of the running magnitude.
            mag = np.abs(q[b, hk * G:(hk + 1) * G]) @ np.abs(K[b, hk]).T * scale
            tol = (d + 2) * 2.0 ** -23 * mag + 1e-30
            err = np.abs(got[b, hk * G:(hk + 1) * G] - want)
            worst = np.unravel_index(np.argmax(err / tol), err.shape)
            assert np.all(err <= tol), (
                f"unit ({b}, {hk}): head {worst[0]} position {worst[1]}: "
                f"{got[b, hk * G + worst[0], worst[1]]} vs {want[worst]}")
    dd.check_device()
