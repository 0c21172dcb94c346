"""GPU parity of the FP4 (MXFP4) indexer cache: the compressor's and the row
inserter's FP4 entries bit for bit against the oracle, and dsv4_indexer_topk
over FP4 pages under the same top-k set rule as FP8 (exact, except slots whose
oracle score lies within 1e-3 relative of the k-th score)."""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_gb300 import binding as B
from deepseek_v4_compressed_gb300 import synth

from _util import bf16_bits, bits_tensor, check_topk, dev, make_decode_inputs, oracle_indexer

pytestmark = pytest.mark.gpu

EPS = 1e-6


def fp4_entries_from_pages(cache, bt_row, n):
    pages = cache.reshape(-1, 64 * 68)
    data = np.stack([pages[bt_row[j // 64], (j % 64) * 64:(j % 64 + 1) * 64] for j in range(n)])
    sc = np.stack([pages[bt_row[j // 64], 64 * 64 + (j % 64) * 4:64 * 64 + (j % 64 + 1) * 4] for j in range(n)])
    return data, sc


@pytest.mark.parametrize("chunked", [False, True])
def test_fp4_compressor_stream_bytes_exact(chunked):
    g = synth.rng(71)
    L = 512
    ks = bf16_bits(synth.normal(g, (L, 4 * 128)))
    ape = synth.normal(g, (4, 256), 0.1)
    w = synth.uniform(g, 128, 0.5, 1.5)
    cs = oracle.rope_table(L, 64)
    want_d, want_s = oracle.compress_stream(oracle.IDX_FP4_KIND, 4, ks, ape, w, EPS, cs, nope_dim=64)
    bt = synth.page_tables(g, 1, 2, extra_pages=1)
    cache = torch.zeros(3 * B.IDX_FP4_PAGE_BYTES, dtype=torch.uint8, device="cuda")
    state = torch.zeros((1, 8, 512), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t_ks, seq0 = bits_tensor(ks), dev(np.zeros(L, np.int32))
    step = 37 if chunked else 1
    for p0 in range(0, L, step):
        n = min(step, L - p0)
        B.compress_insert(B.CACHE_IDX_FP4, 4, t_ks[p0:p0 + n], dev(np.arange(p0, p0 + n, dtype=np.int32)),
                          seq0[:n], dev(ape), dev(w), EPS, dev(cs), state, cache, dev(bt), 1,
                          one_token_per_seq=(n == 1), status=status)
    torch.cuda.synchronize()
    assert B.read_device_status(status)[0] == B.OK
    got_d, got_s = fp4_entries_from_pages(cache.cpu().numpy(), bt[0], L // 4)
    assert np.array_equal(got_d, want_d) and np.array_equal(got_s, want_s)


def test_fp4_pair_kernel_and_row_insert_bytes_exact():
    """Both compressor streams in one launch with the indexer stream in FP4,
    over 4 sequences for 64 decode steps; then quantise-and-insert of given
    rows, including zero, tiny and saturating ones."""
    g = synth.rng(72)
    S, L = 4, 64
    ks_m = bf16_bits(synth.normal(g, (S, L, 4 * 576)))
    ks_i = bf16_bits(synth.normal(g, (S, L, 4 * 128)))
    ape_m, ape_i = synth.normal(g, (4, 1152), 0.1), synth.normal(g, (4, 256), 0.1)
    w_m, w_i = np.ones(576, np.float32), synth.uniform(g, 128, 0.5, 1.5)
    cs = oracle.rope_table(L, 64)
    bt = synth.page_tables(g, S, 1, extra_pages=0)
    comp = torch.zeros(S * B.MLA_PAGE_BYTES, dtype=torch.uint8, device="cuda")
    idxc = torch.zeros(S * B.IDX_FP4_PAGE_BYTES, dtype=torch.uint8, device="cuda")
    st_m = torch.zeros((S, 8, 2304), dtype=torch.float32, device="cuda")
    st_i = torch.zeros((S, 8, 512), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    seqs = dev(np.arange(S, dtype=np.int32))
    t_m, t_i = bits_tensor(ks_m), bits_tensor(ks_i)
    for p in range(L):
        pos = dev(np.full(S, p, np.int32))
        B.compress_insert_pair(
            dict(kind=B.CACHE_MLA, ratio=4, kv_score=t_m[:, p].contiguous(), positions=pos, seqs=seqs,
                 ape=dev(ape_m), rms_weight=dev(w_m), rms_eps=EPS, cos_sin=dev(cs), state=st_m, cache=comp,
                 block_table=dev(bt), num_seqs=S, status=status),
            dict(kind=B.CACHE_IDX_FP4, ratio=4, kv_score=t_i[:, p].contiguous(), positions=pos, seqs=seqs,
                 ape=dev(ape_i), rms_weight=dev(w_i), rms_eps=EPS, cos_sin=dev(cs), state=st_i, cache=idxc,
                 block_table=dev(bt), num_seqs=S, status=status))
    torch.cuda.synchronize()
    assert B.read_device_status(status)[0] == B.OK
    host = idxc.cpu().numpy()
    for b in range(S):
        want = oracle.compress_stream(oracle.IDX_FP4_KIND, 4, ks_i[b], ape_i, w_i, EPS, cs, nope_dim=64)
        got = fp4_entries_from_pages(host, bt[b], L // 4)
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]), b
    # rows straight into the cache
    rows = synth.normal(g, (100, 128), 1.0).astype(np.float32)
    rows[0] = 0.0
    rows[1] *= 1e-30
    rows[2, :32] = 6.0e30
    rows[3, 5] = -0.0
    cache = torch.zeros(3 * B.IDX_FP4_PAGE_BYTES, dtype=torch.uint8, device="cuda")
    bt2 = np.array([[2, 0]], np.int32)
    B.cache_insert_rows(B.CACHE_IDX_FP4, dev(rows), dev(np.zeros(100, np.int32)), dev(np.arange(100, dtype=np.int32)),
                        cache, dev(bt2), status=status)
    want_c = np.zeros(3 * oracle.page_bytes(oracle.IDX_FP4_KIND), np.uint8)
    oracle.page_write(oracle.IDX_FP4_KIND, want_c, bt2[0], *oracle.quant_idx_fp4_rows(rows), nope_dim=64)
    torch.cuda.synchronize()
    assert B.read_device_status(status)[0] == B.OK
    assert np.array_equal(cache.cpu().numpy(), want_c)


def run_indexer_fp4(d, max_ctx=None):
    plan = B.Plan(B.C4A, d.n_heads, d.batch, d.topk, int(max_ctx or d.ctx.max()), idx_heads=d.idx_heads,
                  idx_format=B.IDX_FP4)
    ws = plan.workspace()
    out_idx = torch.full((d.batch, d.topk), -7, dtype=torch.int32, device="cuda")
    out_len = torch.full((d.batch,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.indexer_topk(plan, d.t["qi"], d.t["w"], d.t["idx"], d.t["idx_bt"], d.t["ctx"], out_idx, out_len, ws,
                   status=status)
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == B.OK, bits
    return plan, out_idx.cpu().numpy(), out_len.cpu().numpy()


def check_rows(d, idx, ln):
    import concurrent.futures
    with concurrent.futures.ThreadPoolExecutor(max_workers=16) as ex:
        return sum(ex.map(lambda b: check_topk(idx[b], int(ln[b]), oracle_indexer(d, b), d.topk), range(d.batch)))


def test_fp4_indexer_tiny_and_ragged():
    d = make_decode_inputs(4, 1, 512, 8, 4, 32, seed=73, with_comp=False, idx_fp4=True)
    _, idx, ln = run_indexer_fp4(d)
    assert ln[0] == 32
    check_rows(d, idx, ln)
    ctx = np.array([3, 4, 100, 256, 2049, 5000, 9000], np.int32)
    d = make_decode_inputs(4, len(ctx), ctx, 8, 20, 64, seed=74, with_comp=False, idx_fp4=True)
    _, idx, ln = run_indexer_fp4(d)
    assert list(ln) == [min(64, int(c) // 4) for c in ctx]
    check_rows(d, idx, ln)


def test_fp4_indexer_c4a_32k_batch32_full_size():
    d = make_decode_inputs(4, 32, 32768, 64, 64, 512, seed=75, with_comp=False, idx_fp4=True)
    plan, idx, ln = run_indexer_fp4(d)
    assert plan.info()["launches_indexer"] == 1          # top-k inside the logits launch
    assert np.all(ln == 512)
    print("near-tie slots tolerated:", check_rows(d, idx, ln))


def test_fp4_indexer_1m_batch4_full_size():
    d = make_decode_inputs(4, 4, 1048576, 8, 64, 2048, seed=76, with_comp=False, idx_fp4=True)
    plan, idx, ln = run_indexer_fp4(d)
    assert plan.info()["launches_indexer"] == 2          # logits, then the long-row top-k
    assert np.all(ln == 2048)
    print("near-tie slots tolerated:", check_rows(d, idx, ln))


def test_fp4_indexer_wide_exponent_spread_slots():
    """Slots whose four 32-dim blocks lie more than 8 binades apart take the
    kernel's exact per-slot path; their scores (and every other slot's) still
    give the oracle's top-k."""
    g = synth.rng(77)
    B_, n_c, HI, K = 3, 1500, 16, 96
    ctx = np.full(B_, 4 * n_c, np.int32)
    pages = (n_c + 63) // 64
    bt = synth.page_tables(g, B_, pages, extra_pages=1)
    cache = np.zeros((B_ * pages + 1) * oracle.page_bytes(oracle.IDX_FP4_KIND), np.uint8)
    for b in range(B_):
        rows = synth.normal(g, (n_c, 128), 1.0)
        spread = g.random(n_c) < 0.2                     # a fifth of the slots
        shift = g.integers(9, 30, size=n_c)
        rows[spread, :32] *= 2.0 ** shift[spread, None]  # block 0 far above the others
        rows[spread, 96:] *= 2.0 ** -shift[spread, None]
        oracle.page_write(oracle.IDX_FP4_KIND, cache, bt[b], *oracle.quant_idx_fp4_rows(rows), nope_dim=64)
    qi = oracle.f32_to_e4m3(synth.normal(g, (B_, HI, 128)))
    wq = synth.uniform(g, (B_, HI))
    plan = B.Plan(B.C4A, 8, B_, K, int(ctx.max()), idx_heads=HI, idx_format=B.IDX_FP4)
    ws = plan.workspace()
    out_idx = torch.full((B_, K), -7, dtype=torch.int32, device="cuda")
    out_len = torch.full((B_,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.indexer_topk(plan, dev(qi), dev(wq), dev(cache), dev(bt), dev(ctx), out_idx, out_len, ws, status=status)
    torch.cuda.synchronize()
    assert B.read_device_status(status)[0] == B.OK
    idx, ln = out_idx.cpu().numpy(), out_len.cpu().numpy()
    for b in range(B_):
        check_topk(idx[b], int(ln[b]), oracle.indexer_logits_fp4(qi[b], wq[b], cache, bt[b], n_c), K)
