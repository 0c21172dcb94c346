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
    tol = check_topk(out_idx.cpu().numpy()[0], int(out_len.cpu()[0]), logits, K)
    if tol == 0:
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
