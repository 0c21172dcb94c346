"""End-to-end decode on the GPU (compressor stream -> indexer/top-k -> sparse MLA)
against the oracle, IndexCache reuse, and the device-status paths."""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_gb300 import binding as B
from deepseek_v4_compressed_gb300 import synth

from _util import SCALE, bf16_bits, bits_tensor, check_attention, check_topk, dev

pytestmark = pytest.mark.gpu

EPS = 1e-6


def test_tiny_c4a_end_to_end():
    """512 tokens through both compressors token by token, then one decode query
    (8 heads, 4 indexer heads, top-32 of 128 slots, window 128)."""
    g = synth.rng(0)
    L, H, HI, K = 512, 8, 4, 32
    ks_main = bf16_bits(synth.normal(g, (L, 4 * 576)))
    ks_idx = bf16_bits(synth.normal(g, (L, 4 * 128)))
    ape_main = synth.normal(g, (4, 2 * 576), 0.1)
    ape_idx = synth.normal(g, (4, 2 * 128), 0.1)
    w_main = np.ones(576, np.float32)
    w_idx = np.ones(128, np.float32)
    cs = oracle.rope_table(L, 64)
    swa_rows = bf16_bits(synth.normal(g, (L, 576), SCALE))
    q = bf16_bits(synth.normal(g, (1, H, 576), SCALE))
    qi = oracle.f32_to_e4m3(synth.normal(g, (1, HI, 128)))
    wq = synth.uniform(g, (1, HI))

    # oracle
    main_d, main_s = oracle.compress_stream(0, 4, ks_main, ape_main, w_main, EPS, cs, nope_dim=512)
    idx_d, idx_s = oracle.compress_stream(1, 4, ks_idx, ape_idx, w_idx, EPS, cs, nope_dim=64)
    bt = np.array([[1, 0]], np.int32)
    comp = np.zeros(2 * oracle.page_bytes(0), np.uint8)
    oracle.page_write(0, comp, bt[0], main_d, main_s)
    idxc = np.zeros(2 * oracle.page_bytes(1), np.uint8)
    oracle.page_write(1, idxc, bt[0], idx_d, idx_s, nope_dim=64)
    swa_bt = np.array([[5, 3, 7, 1, 0, 2, 4, 6]], np.int32)
    swa = np.zeros((8 * 64, 576), np.uint16)
    for t in range(L):
        swa[swa_bt[0, t // 64] * 64 + t % 64] = swa_rows[t]
    logits = oracle.indexer_logits(qi[0], wq[0], idxc, bt[0], 128)
    o_idx, o_len = oracle.topk(logits, K)
    ref, ref_lse, _ = oracle.sparse_mla(q[0], comp, bt[0], o_idx, o_len, swa, swa_bt[0], L - 1, SCALE)

    # GPU: the same token stream through the library
    t_bt = dev(bt)
    cache_main = torch.zeros(2 * B.MLA_PAGE_BYTES, dtype=torch.uint8, device="cuda")
    cache_idx = torch.zeros(2 * B.IDX_PAGE_BYTES, dtype=torch.uint8, device="cuda")
    st_main = torch.zeros((1, 8, 4 * 576), dtype=torch.float32, device="cuda")
    st_idx = torch.zeros((1, 8, 4 * 128), dtype=torch.float32, device="cuda")
    km, ki = bits_tensor(ks_main), bits_tensor(ks_idx)
    seq0 = dev(np.zeros(1, np.int32))
    t_cs = dev(cs)
    for p in range(L):
        pos = dev(np.array([p], np.int32))
        B.compress_insert(B.CACHE_MLA, 4, km[p:p + 1], pos, seq0, dev(ape_main), dev(w_main), EPS, t_cs,
                          st_main, cache_main, t_bt, 1)
        B.compress_insert(B.CACHE_IDX, 4, ki[p:p + 1], pos, seq0, dev(ape_idx), dev(w_idx), EPS, t_cs,
                          st_idx, cache_idx, t_bt, 1)
    plan = B.Plan(B.C4A, H, 1, K, L, idx_heads=HI)
    ws = plan.workspace()
    ctx = dev(np.array([L], np.int32))
    out_idx = torch.zeros((1, K), dtype=torch.int32, device="cuda")
    out_len = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.indexer_topk(plan, dev(qi), dev(wq), cache_idx, t_bt, ctx, out_idx, out_len, ws)
    out = torch.zeros((1, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, H), dtype=torch.float32, device="cuda")
    B.sparse_mla_decode(plan, bits_tensor(q), bits_tensor(swa), dev(swa_bt), ctx, out, ws,
                        comp_cache=cache_main, comp_block_table=t_bt, topk_idx=out_idx, topk_len=out_len,
                        lse=lse)
    torch.cuda.synchronize()
    assert np.array_equal(cache_main.cpu().numpy(), comp)
    assert np.array_equal(cache_idx.cpu().numpy(), idxc)
    g_idx, g_len = out_idx.cpu().numpy()[0], int(out_len.cpu()[0])
    tol = check_topk(g_idx, g_len, logits, K)
    if tol:
        # near-ties: the GPU's set is a valid top-k; attend over it in the oracle
        ref, ref_lse, _ = oracle.sparse_mla(q[0], comp, bt[0], g_idx[:g_len].copy(), g_len, swa, swa_bt[0],
                                            L - 1, SCALE)
    check_attention(out.float().cpu().numpy()[0], ref)
    np.testing.assert_allclose(lse.cpu().numpy()[0], ref_lse, rtol=1e-3, atol=1e-3)


def test_indexcache_reuse_layer_reads_its_own_kv():
    """Two c4a layers, the second a reuse layer under freq 2: it takes the first
    layer's indices but attends over its own compressed cache."""
    skip = B.index_schedule([4, 4], True, 2)
    assert skip == [0, 1]
    from _util import make_decode_inputs
    d1 = make_decode_inputs(4, 3, 4096, 16, 16, 64, seed=41)
    d2 = make_decode_inputs(4, 3, 4096, 16, 16, 64, seed=42)
    plan = B.Plan(B.C4A, 16, 3, 64, 4096, idx_heads=16)
    ws = plan.workspace()
    shared_idx = torch.zeros((3, 64), dtype=torch.int32, device="cuda")
    shared_len = torch.zeros(3, dtype=torch.int32, device="cuda")
    outs = []
    for layer, d in enumerate([d1, d2]):
        if not skip[layer]:
            B.indexer_topk(plan, d.t["qi"], d.t["w"], d.t["idx"], d.t["idx_bt"], d.t["ctx"], shared_idx,
                           shared_len, ws)
        out = torch.zeros((3, 16, 512), dtype=torch.bfloat16, device="cuda")
        B.sparse_mla_decode(plan, d.t["q"], d.t["swa"], d.t["swa_bt"], d.t["ctx"], out, ws,
                            comp_cache=d.t["comp"], comp_block_table=d.t["comp_bt"], topk_idx=shared_idx,
                            topk_len=shared_len)
        outs.append(out.float().cpu().numpy())
    torch.cuda.synchronize()
    idx = shared_idx.cpu().numpy()
    ln = shared_len.cpu().numpy()
    for b in range(3):
        logits = oracle.indexer_logits(d1.qi[b], d1.w[b], d1.idx, d1.idx_bt[b], int(d1.n_c[b]))
        assert check_topk(idx[b], int(ln[b]), logits, 64) == 0
        o_idx, o_len = oracle.topk(logits, 64)
        # the reuse layer: layer-1 indices over layer-2's own caches and query
        ref2, _, _ = oracle.sparse_mla(d2.q[b], d2.comp, d2.comp_bt[b], o_idx, o_len, d2.swa, d2.swa_bt[b],
                                       int(d2.p[b]), SCALE)
        check_attention(outs[1][b], ref2, "reuse seq %d" % b)


def test_bounded_wait_times_out_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.selftest_bounded_wait(status, 1000)
    st, bits = B.read_device_status(status)
    assert st == B.ERR_TIMEOUT and bits & B.DEV_TIMEOUT
    # the context is still usable and the word was cleared
    x = torch.ones(1024, device="cuda") * 2
    assert float(x.sum()) == 2048.0
    assert B.read_device_status(status)[0] == B.OK


def test_bad_block_table_is_flagged_not_faulted():
    from _util import make_decode_inputs
    d = make_decode_inputs(4, 2, 2048, 8, 8, 32, seed=43)
    bad_bt = d.t["idx_bt"].clone()
    bad_bt[1, 3] = 10 ** 6                     # points past the cache
    plan = B.Plan(B.C4A, 8, 2, 32, 2048, idx_heads=8)
    ws = plan.workspace()
    out_idx = torch.zeros((2, 32), dtype=torch.int32, device="cuda")
    out_len = torch.zeros(2, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.indexer_topk(plan, d.t["qi"], d.t["w"], d.t["idx"], bad_bt, d.t["ctx"], out_idx, out_len, ws,
                   status=status)
    st, bits = B.read_device_status(status)
    assert st == B.ERR_DEVICE_CHECK and bits & B.DEV_BAD_PAGE
    bad_idx = torch.full((2, 32), 5, dtype=torch.int32, device="cuda")
    bad_idx[0, 0] = 10 ** 6                    # a slot past the block table
    out = torch.zeros((2, 8, 512), dtype=torch.bfloat16, device="cuda")
    B.sparse_mla_decode(plan, d.t["q"], d.t["swa"], d.t["swa_bt"], d.t["ctx"], out, ws,
                        comp_cache=d.t["comp"], comp_block_table=d.t["comp_bt"], topk_idx=bad_idx,
                        topk_len=torch.full((2,), 32, dtype=torch.int32, device="cuda"), status=status)
    st, bits = B.read_device_status(status)
    assert st == B.ERR_DEVICE_CHECK and bits & B.DEV_BAD_INDEX


@pytest.mark.parametrize("case", ["b4_streamed_prefill", "c4a_32k_b32", "b4_streamed_prefill_v4",
                                  "c4a_32k_b32_v4", "b4_streamed_prefill_fp4", "c4a_32k_b32_fp4"])
def test_bench_call_chain_under_dependent_launch(case):
    """The benchmark's decode loop (compress pair -> indexer + top-k -> sparse
    MLA under programmatic dependent launch, captured in a CUDA graph; in the
    V4-native geometry followed by the inverse RoPE + FP8 output quant; with
    the MXFP4 indexer cache) over
    steps that include ratio-4 boundaries: the slot a step's compressor emits
    is selected by that step's indexer and dominates its attention, and every
    cache byte, top-k set and output matches the oracle."""
    from _chain import run_chain
    v4, fp4 = case.endswith("_v4"), case.endswith("_fp4")
    if case.startswith("b4_streamed_prefill"):
        tol, nb = run_chain(4, [1021, 2046, 517, 3072], 6, 64, 64, 64, seed=51, prefill="stream", v4=v4,
                            idx_fp4=fp4)
    else:
        tol, nb = run_chain(32, 32763, 5, 64, 64, 512, seed=52, prefill="direct", v4=v4, idx_fp4=fp4)
    assert nb > 0
    print("boundary steps checked:", nb, "near-tie slots tolerated:", tol)


def test_mixed_stack_plans_b16_64k():
    """The 60-layer stack's per-type plans at its full size (batch 16, context
    65536, 64 heads, top-k 512): a swaonly layer, a c4a layer that runs the
    indexer (16384 slots per sequence: on 152 SMs the logits take 9 CTAs per
    sequence and the top-k a separate cluster launch), a c4a reuse layer under
    IndexCache frequency 2 (the previous c4a layer's indices over its own
    caches and query) and a c128a layer whose metadata selects all 512
    visible slots.  All calls in order on one stream; every output against
    the oracle."""
    import concurrent.futures
    from _util import make_decode_inputs
    ratios = [1, 4, 4, 128]
    skip = B.index_schedule(ratios, True, 2)
    assert skip == [0, 0, 1, 0]
    Bsz, L, H, K = 16, 65536, 64, 512
    d_sw = make_decode_inputs(1, Bsz, L, H, 0, 0, seed=61)
    d_c1 = make_decode_inputs(4, Bsz, L, H, 64, K, seed=62)
    d_c2 = make_decode_inputs(4, Bsz, L, H, 64, K, seed=63)
    d_128 = make_decode_inputs(128, Bsz, L, H, 0, K, seed=64)
    assert np.all(d_128.meta_len == 512) and np.array_equal(d_128.meta_idx[0], np.arange(512))
    p_sw = B.Plan(B.SWAONLY, H, Bsz, 0, L)
    p_c4 = B.Plan(B.C4A, H, Bsz, K, L, idx_heads=64)
    p_128 = B.Plan(B.C128A, H, Bsz, K, L)
    info = p_c4.info()
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert info["idx_ctas_per_seq"] == 9 and info["launches_indexer"] == 2
    ws = torch.zeros(max(p_sw.workspace_bytes, p_c4.workspace_bytes, p_128.workspace_bytes),
                     dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    shared_idx = torch.full((Bsz, K), -9, dtype=torch.int32, device="cuda")
    shared_len = torch.full((Bsz,), -9, dtype=torch.int32, device="cuda")

    def out_buf():
        return (torch.zeros((Bsz, H, 512), dtype=torch.bfloat16, device="cuda"),
                torch.zeros((Bsz, H), dtype=torch.float32, device="cuda"))

    outs = []
    o, l = out_buf()
    B.sparse_mla_decode(p_sw, d_sw.t["q"], d_sw.t["swa"], d_sw.t["swa_bt"], d_sw.t["ctx"], o, ws, lse=l, status=status)
    outs.append((o, l))
    for layer, d in ((1, d_c1), (2, d_c2)):
        if not skip[layer]:
            B.indexer_topk(p_c4, d.t["qi"], d.t["w"], d.t["idx"], d.t["idx_bt"], d.t["ctx"], shared_idx, shared_len,
                           ws, status)
        o, l = out_buf()
        B.sparse_mla_decode(p_c4, d.t["q"], d.t["swa"], d.t["swa_bt"], d.t["ctx"], o, ws, comp_cache=d.t["comp"],
                            comp_block_table=d.t["comp_bt"], topk_idx=shared_idx, topk_len=shared_len, lse=l,
                            status=status)
        outs.append((o, l))
    o, l = out_buf()
    B.sparse_mla_decode(p_128, d_128.t["q"], d_128.t["swa"], d_128.t["swa_bt"], d_128.t["ctx"], o, ws,
                        comp_cache=d_128.t["comp"], comp_block_table=d_128.t["comp_bt"], topk_idx=d_128.t["meta_idx"],
                        topk_len=d_128.t["meta_len"], lse=l, status=status)
    outs.append((o, l))
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == B.OK, bits
    gidx, glen = shared_idx.cpu().numpy(), shared_len.cpu().numpy()
    res = [(x.float().cpu().numpy(), y.cpu().numpy()) for x, y in outs]

    def check(b):
        logits = oracle.indexer_logits(d_c1.qi[b], d_c1.w[b], d_c1.idx, d_c1.idx_bt[b], int(d_c1.n_c[b]))
        tol = check_topk(gidx[b], int(glen[b]), logits, K)
        sel = gidx[b][:glen[b]].copy()
        refs = [oracle.sparse_mla(d_sw.q[b], None, None, None, 0, d_sw.swa, d_sw.swa_bt[b], int(d_sw.p[b]), SCALE)]
        for d in (d_c1, d_c2):
            refs.append(oracle.sparse_mla(d.q[b], d.comp, d.comp_bt[b], sel, int(glen[b]), d.swa, d.swa_bt[b],
                                          int(d.p[b]), SCALE))
        refs.append(oracle.sparse_mla(d_128.q[b], d_128.comp, d_128.comp_bt[b], d_128.meta_idx[b],
                                      int(d_128.meta_len[b]), d_128.swa, d_128.swa_bt[b], int(d_128.p[b]), SCALE))
        for li, ((got, got_lse), (ref, ref_lse, _)) in enumerate(zip(res, refs)):
            check_attention(got[b], ref, "layer %d seq %d" % (li, b))
            np.testing.assert_allclose(got_lse[b], ref_lse, rtol=1e-3, atol=1e-3)
        return tol

    with concurrent.futures.ThreadPoolExecutor(max_workers=16) as ex:
        tol = sum(ex.map(check, range(Bsz)))
    print("near-tie slots tolerated:", tol)
