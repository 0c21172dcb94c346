"""GPU parity of dsv4_indexer_topk: index sets equal the oracle's, except slots
whose oracle score lies within 1e-3 relative of the k-th score."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_gb300 import binding as B
from deepseek_v4_compressed_gb300 import synth

from _util import check_topk, dev, make_decode_inputs, oracle_indexer

pytestmark = pytest.mark.gpu


def run_indexer(d, max_ctx=None, seqs=None):
    plan = B.Plan(B.C4A, d.n_heads, d.batch, d.topk, int(max_ctx or d.ctx.max()), idx_heads=d.idx_heads)
    ws = plan.workspace()
    out_idx = torch.full((d.batch, d.topk), -7, dtype=torch.int32, device="cuda")
    out_len = torch.full((d.batch,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.indexer_topk(plan, d.t["qi"], d.t["w"], d.t["idx"], d.t["idx_bt"], d.t["ctx"], out_idx, out_len, ws,
                   status=status)
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == B.OK, bits
    return out_idx.cpu().numpy(), out_len.cpu().numpy()


def check_all(d, idx, ln, seqs=None):
    tolerated = 0
    for b in (range(d.batch) if seqs is None else seqs):
        tolerated += check_topk(idx[b], int(ln[b]), oracle_indexer(d, b), d.topk)
    return tolerated


def test_tiny_c4a():
    d = make_decode_inputs(4, 1, 512, 8, 4, 32, seed=0, with_comp=False)
    idx, ln = run_indexer(d)
    assert ln[0] == 32
    check_all(d, idx, ln)


def test_ragged_contexts_and_short_sequences():
    # n_c = 0, 1, 25, 64 (= k), 512, 1250: covers n_c <= k, a ragged last tile and empty
    ctx = np.array([3, 4, 100, 256, 2049, 5000], np.int32)
    d = make_decode_inputs(4, len(ctx), ctx, 8, 64, 64, seed=21, with_comp=False)
    idx, ln = run_indexer(d)
    assert list(ln) == [0, 1, 25, 64, 64, 64]
    check_all(d, idx, ln)


def test_c4a_32k_batch32_full_size():
    d = make_decode_inputs(4, 32, 32768, 64, 64, 512, seed=1, with_comp=False)
    idx, ln = run_indexer(d)
    assert np.all(ln == 512)
    tol = check_all(d, idx, ln)
    print("near-tie slots tolerated:", tol)


def _with_zero_weights(d, seqs):
    """All-equal logits (zero head weights) for the given sequences: every
    selection of k of them is a valid top-k."""
    for b in seqs:
        d.w[b] = 0.0
        d.t["w"][b] = 0.0
    return d


def test_cluster_topk_ragged_batch32():
    # a plan for 32 sequences of up to 32768 tokens takes the top-k inside the
    # logits launch (clusters of 4 CTAs): n_c <= k, empty CTAs of a cluster,
    # ragged last tiles, and all-equal rows (zero weights)
    ctx = np.array([3, 4, 100, 2048, 2052, 5000, 32768, 8195, 20000, 4097, 131, 600] * 3, np.int32)[:32]
    d = _with_zero_weights(make_decode_inputs(4, 32, ctx, 8, 64, 512, seed=31, with_comp=False), [7, 9, 30])
    plan = B.Plan(B.C4A, d.n_heads, d.batch, d.topk, 32768, idx_heads=d.idx_heads)
    assert plan.info()["launches_indexer"] == 1
    idx, ln = run_indexer(d, max_ctx=32768)
    assert list(ln) == [min(512, int(c) // 4) for c in ctx]
    check_all(d, idx, ln)


def test_cluster_topk_eight_ctas():
    # 19 sequences of up to 8192 tokens: clusters of 8 CTAs of 2 tiles each
    ctx = np.array([8192, 8000, 7777, 4096, 4100, 257, 1, 0, 6000, 8192, 5555, 3000, 2049, 1024, 999, 8190,
                    7000, 6500, 12], np.int32)
    d = _with_zero_weights(make_decode_inputs(4, 19, ctx, 8, 32, 256, seed=32, with_comp=False), [4])
    plan = B.Plan(B.C4A, d.n_heads, d.batch, d.topk, 8192, idx_heads=d.idx_heads)
    info = plan.info()
    if info["idx_ctas_per_seq"] > 8:
        pytest.skip("this GPU splits a sequence over more than 8 CTAs")
    assert info["launches_indexer"] == 1
    idx, ln = run_indexer(d, max_ctx=8192)
    assert list(ln) == [min(256, int(c) // 4) for c in ctx]
    check_all(d, idx, ln)


def test_plan_max_ctx_larger_than_batch_contexts():
    ctx = np.array([1000, 4001, 16], np.int32)
    d = make_decode_inputs(4, 3, ctx, 8, 16, 128, seed=22, with_comp=False)
    idx, ln = run_indexer(d, max_ctx=70000)
    check_all(d, idx, ln)


def test_long_c4a_1m_full_size():
    d = make_decode_inputs(4, 4, 1048576, 8, 64, 2048, seed=4, with_comp=False)
    idx, ln = run_indexer(d)
    assert np.all(ln == 2048)
    check_all(d, idx, ln)


def test_deterministic_across_runs():
    d = make_decode_inputs(4, 8, 20000, 8, 64, 256, seed=23, with_comp=False)
    first = run_indexer(d)
    for _ in range(5):
        again = run_indexer(d)
        assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])


def test_long_rows_cluster_topk_ragged():
    # plans whose top-k is a separate launch over long rows split across a
    # cluster of CTAs: 4 sequences with up to 32768 slots (128K context), ragged
    # lengths (n_c <= k, CTAs with no slots) and an all-equal row
    ctx = np.array([131072, 70000, 1500, 9000], np.int32)
    d = _with_zero_weights(make_decode_inputs(4, 4, ctx, 8, 16, 512, seed=34, with_comp=False), [3])
    plan = B.Plan(B.C4A, d.n_heads, d.batch, d.topk, 131072, idx_heads=d.idx_heads)
    assert plan.info()["launches_indexer"] == 2
    idx, ln = run_indexer(d, max_ctx=131072)
    assert list(ln) == [min(512, int(c) // 4) for c in ctx]
    check_all(d, idx, ln)


def test_long_rows_candidate_lists_and_their_overflow():
    """A 2M-context plan (clusters of 16 CTAs with 32768 keys each, candidate
    lists of half a warp's run).  Sequence 0 has plain scores.  In sequence 1
    the first 2048 slots score about 8 times higher: warp 0 of the first CTA
    finds more candidates than its list holds, so that CTA scans all of its
    keys while the others walk their lists; the set rule holds for both."""
    d = make_decode_inputs(4, 2, 2097152, 8, 64, 2048, seed=37, with_comp=False)
    g = synth.rng(38)
    n_c = int(d.n_c[1])
    rows = synth.normal(g, (n_c, 128), 1.0 / np.sqrt(128))
    rows[:2048] *= 8.0
    data, sc = oracle.quant_idx_rows(rows)
    oracle.page_write(oracle.IDX_KIND, d.idx, d.idx_bt[1], data, sc, nope_dim=64)
    d.t["idx"] = dev(d.idx)
    plan = B.Plan(B.C4A, d.n_heads, d.batch, d.topk, 2097152, idx_heads=d.idx_heads)
    assert plan.info()["launches_indexer"] == 2
    idx, ln = run_indexer(d)
    assert np.all(ln == 2048)
    check_all(d, idx, ln)
    assert np.count_nonzero(idx[1] < 2048) > 1024


def test_topk_beyond_the_cluster_range():
    # a plan for rows longer than 16 x 32768 slots (context 2.4M) keeps the
    # single-CTA top-k with its keys in global memory; actual rows are short
    ctx = np.array([100000, 3000, 65541], np.int32)
    d = make_decode_inputs(4, 3, ctx, 8, 16, 512, seed=35, with_comp=False)
    idx, ln = run_indexer(d, max_ctx=2400000)
    assert list(ln) == [min(512, int(c) // 4) for c in ctx]
    check_all(d, idx, ln)


def test_indexer_heads_not_a_multiple_of_16():
    # 20 indexer heads: the MMA's N is padded to 32 with zero weights past the heads
    ctx = np.array([9000, 512, 40000], np.int32)
    d = make_decode_inputs(4, 3, ctx, 8, 20, 256, seed=36, with_comp=False)
    idx, ln = run_indexer(d)
    assert list(ln) == [min(256, int(c) // 4) for c in ctx]
    check_all(d, idx, ln)
