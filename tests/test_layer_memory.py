"""The layer-scoped buffer is O(k d), not O(n d).

The summary page's core formulas state that prefetching only the critical
entries shrinks the runtime sparse-KV buffer from O(n d) to O(k d), and the
paper (Sec. 1, layer-scoped KV memory manager) keeps only the current
layers' entries on the GPU.  Here that is pinned on the library itself: the
double-buffered scratch a decode-step context owns does not change with the
context length n, and the only device memory that grows with n is the
scoring workspace (fp32 logits, 4 bytes per query head and position, plus
per-chunk softmax partials), which no gathered row ever occupies.
"""
import pytest

import sparse_kv_prefetch_gb300 as dd

# The GQA-128K layer shape (bf16) at four context lengths.
B, HQ, HKV, D, K, W = 32, 32, 8, 128, 2048, 0
NS = (16384, 32768, 65536, 131072)


def shape(n, k=K, dtype=dd.DD_BF16):
    return dd.Shape(B, HQ, HKV, D, n, k, W, dtype)


def test_workspace_grows_only_by_logits_and_chunk_partials():
    """Workspace growth between context lengths is the fp32 logits of the new
    positions (4 B per query head and position) plus at most 8 B per query
    head and 256 positions of per-chunk partials (a scoring chunk holds at
    least 256 positions), up to 256-byte alignment of each region."""
    ws = {n: dd.workspace_size(shape(n)) for n in NS}
    for n1, n2 in zip(NS, NS[1:]):
        logits = B * HQ * (n2 - n1) * 4
        extra = (ws[n2] - ws[n1]) - logits
        assert 0 <= extra <= B * HQ * 8 * ((n2 - n1) // 256 + 1) + 2 * 256, (n1, n2, extra)
    # k does not enter the logits: the same n with a larger k grows only by
    # terms proportional to k, the split-k attention partials (d fp32 values
    # and a (max, sum) pair per query head and 64 attended rows) and the real
    # query's selection scores (4 B per selected row).
    grow = dd.workspace_size(shape(NS[-1], 2 * K)) - ws[NS[-1]]
    per_row = B * HQ * (D * 4 + 8) / 64 + B * HKV * 4
    assert 0 < grow <= per_row * K + B * HQ * (D * 4 + 8) + 3 * 256, grow


@pytest.mark.gpu
def test_context_scratch_is_independent_of_context_length():
    """A context's device bytes minus its workspace are the two layer slots of
    gathered K and V rows (2 x 2 x B x H_kv x k x d x 2 B), their index and
    score lists (2 x 2 x B x H_kv x k x 4 B) and the query heads' LSE (B x H_q
    x 4 B): the same at every n, and doubling with k."""
    U = B * HKV
    want = 2 * (2 * U * K * D * 2) + 2 * (2 * U * K * 4) + B * HQ * 4
    got = {}
    for n in NS:
        ctx = dd.Ctx(shape(n))
        got[n] = ctx.device_bytes - dd.workspace_size(shape(n))
        ctx.close()
    assert all(v == want for v in got.values()), got
    ctx = dd.Ctx(shape(NS[0], 2 * K))
    doubled = ctx.device_bytes - dd.workspace_size(shape(NS[0], 2 * K))
    ctx.close()
    assert doubled == 2 * want - B * HQ * 4
