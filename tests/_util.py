"""Test helpers: seeded decode inputs (generator + oracle quantiser), GPU upload,
and the parity checks (bit-exact bytes, top-k set rule, attention tolerances).

Inputs come from deepseek_v4_compressed_gb300.synth; cache bytes from the
oracle's quantiser; expected values from the oracle.  Nothing here takes an
input or an expected value from the CUDA path.
"""
import math

import numpy as np
import torch

import oracle
from deepseek_v4_compressed_gb300 import synth

SCALE = 1.0 / math.sqrt(576)

# Attention tolerances: the stated bf16 bounds plus a relative-L2 bound (outputs
# of near-uniform attention are ~2e-3 in size, so the absolute bounds alone
# would pass an all-zero output).
ATT_MAX_ABS = 2e-2
ATT_MEAN_ABS = 2e-3
ATT_REL_L2 = 1e-2
TOPK_REL = 1e-3

# Top-k parity record of the session: rows compared, slots that differ from
# the oracle's set (all within TOPK_REL of the k-th score, else the check
# fails) and oracle slots inside that band; conftest prints the totals.
TOPK_STATS = {"rows": 0, "differ": 0, "in_band": 0}


def bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def bits_tensor(bits, device="cuda"):
    """uint16 bf16 bit patterns -> torch bfloat16 tensor on device."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def tensor_bits(t):
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DecodeInputs:
    """One layer's decode-step inputs for a batch (host numpy + device tensors)."""


def make_decode_inputs(layer_type, batch, ctx, n_heads, idx_heads, topk, seed, comp_pool=8192,
                       peaky=False, with_comp=True, idx_fp4=False, device="cuda"):
    """ctx: int or per-sequence array of contexts L (query position L - 1).

    c4a: indexer cache with L // 4 oracle-quantised rows per sequence, q_fp8
    and head weights U(0,1); c128a: sorted uniform metadata indices over the
    L // 128 slots; both: a compressed cache (rows drawn from a pool of
    `comp_pool` quantised N(0,1)/sqrt(576) rows), an SWA cache holding the
    window's tokens and bf16 queries N(0,1)/sqrt(576) (or peaky ones)."""
    g = synth.rng(seed)
    ctx = np.broadcast_to(np.asarray(ctx, np.int64), (batch,)).astype(np.int32).copy()
    ratio = {4: 4, 128: 128, 1: 0}[layer_type]
    n_c = (ctx // ratio) if ratio else np.zeros(batch, np.int32)
    d = DecodeInputs()
    d.layer_type, d.batch, d.ctx, d.n_heads, d.idx_heads, d.topk = layer_type, batch, ctx, n_heads, idx_heads, topk
    d.n_c = n_c.astype(np.int32)
    d.p = (ctx - 1).astype(np.int32)

    # SWA cache: window tokens only; other logical pages unmapped (-1)
    swa_lp = int(ctx.max() + 63) // 64
    d.swa_bt = np.full((batch, swa_lp), -1, np.int32)
    n_swa_pages = 0
    for b in range(batch):
        t0 = max(0, int(d.p[b]) - 127)
        for lp in range(t0 // 64, int(d.p[b]) // 64 + 1):
            d.swa_bt[b, lp] = n_swa_pages
            n_swa_pages += 1
    perm = g.permutation(n_swa_pages).astype(np.int32)
    d.swa_bt = np.where(d.swa_bt >= 0, perm[np.maximum(d.swa_bt, 0)], -1).astype(np.int32)
    d.swa = bf16_bits(synth.normal(g, (n_swa_pages * 64, 576), SCALE))

    # compressed cache
    with_comp = with_comp and bool(ratio)
    if with_comp:
        cp = int(max(1, (n_c.max() + 63) // 64))
        d.comp_bt = synth.page_tables(g, batch, cp, extra_pages=1)
        pool_n = int(min(comp_pool, max(1, n_c.sum())))
        pool_data, pool_sc = oracle.quant_mla_rows(synth.normal(g, (pool_n, 576), SCALE))
        d.comp = np.zeros((batch * cp + 1) * oracle.page_bytes(oracle.MLA_KIND), np.uint8)
        d.comp_rows = []
        for b in range(batch):
            pick = g.integers(0, pool_n, size=int(n_c[b]))
            oracle.page_write(oracle.MLA_KIND, d.comp, d.comp_bt[b], pool_data[pick], pool_sc[pick])
            d.comp_rows.append((pool_data[pick], pool_sc[pick]))
    # indexer cache + queries
    if layer_type == 4 and idx_heads > 0:
        ip = int(max(1, (n_c.max() + 63) // 64))
        d.idx_bt = synth.page_tables(g, batch, ip, extra_pages=1)
        kind = oracle.IDX_FP4_KIND if idx_fp4 else oracle.IDX_KIND
        d.idx_fp4 = idx_fp4
        d.idx = np.zeros((batch * ip + 1) * oracle.page_bytes(kind), np.uint8)
        for b in range(batch):
            rows = synth.normal(g, (int(n_c[b]), 128), 1.0 / math.sqrt(128))
            data, sc = oracle.quant_idx_fp4_rows(rows) if idx_fp4 else oracle.quant_idx_rows(rows)
            oracle.page_write(kind, d.idx, d.idx_bt[b], data, sc, nope_dim=64)
        d.qi = oracle.f32_to_e4m3(synth.normal(g, (batch, idx_heads, 128)))
        d.w = synth.uniform(g, (batch, idx_heads))
    if layer_type == 128:
        d.meta_idx = np.full((batch, topk), -1, np.int32)
        d.meta_len = np.zeros(batch, np.int32)
        for b in range(batch):
            s = synth.sorted_sample(g, int(n_c[b]), topk)
            d.meta_idx[b, :len(s)] = s
            d.meta_len[b] = len(s)

    q = synth.normal(g, (batch, n_heads, 576), SCALE)
    if peaky and with_comp:
        # each head leans on 4 of its sequence's compressed rows
        for b in range(batch):
            if n_c[b] == 0:
                continue
            data, sc = d.comp_rows[b]
            for h in range(n_heads):
                pick = g.integers(0, int(n_c[b]), size=4)
                rows = [oracle.e4m3_to_f64(data[s, :512]) * np.repeat(2.0 ** (sc[s].astype(np.int64) - 127), 64)
                        for s in pick]
                q[b, h, :512] = (200.0 * np.sum(rows, axis=0)).astype(np.float32)
    d.q = bf16_bits(q)

    # device copies
    d.t = {}
    d.t["q"] = bits_tensor(d.q, device)
    d.t["swa"] = bits_tensor(d.swa, device)
    d.t["swa_bt"] = dev(d.swa_bt, device)
    d.t["ctx"] = dev(d.ctx, device)
    if with_comp:
        d.t["comp"] = dev(d.comp, device)
        d.t["comp_bt"] = dev(d.comp_bt, device)
    if layer_type == 4 and idx_heads > 0:
        d.t["idx"] = dev(d.idx, device)
        d.t["idx_bt"] = dev(d.idx_bt, device)
        d.t["qi"] = dev(d.qi, device)
        d.t["w"] = dev(d.w, device)
    if layer_type == 128:
        d.t["meta_idx"] = dev(d.meta_idx, device)
        d.t["meta_len"] = dev(d.meta_len, device)
    return d


def oracle_indexer(d, b):
    f = oracle.indexer_logits_fp4 if getattr(d, "idx_fp4", False) else oracle.indexer_logits
    return f(d.qi[b], d.w[b], d.idx, d.idx_bt[b], int(d.n_c[b]))


def check_topk(gpu_idx, gpu_len, logits, k):
    """Top-k set rule: exact, except slots whose oracle score is within 1e-3
    relative of the k-th score.  Returns the number of such tolerated slots."""
    n = logits.size
    TOPK_STATS["rows"] += 1
    o_idx, o_len = oracle.topk(logits, k)
    assert gpu_len == o_len, (gpu_len, o_len)
    g = gpu_idx[:gpu_len]
    assert np.all(gpu_idx[gpu_len:] == -1)
    assert np.all(np.diff(g) > 0), "indices not strictly ascending"
    assert np.all((g >= 0) & (g < n))
    if o_len == n:
        assert np.array_equal(g, np.arange(n))
        return 0
    kth = np.sort(logits)[::-1][k - 1]
    diff = np.setxor1d(g, o_idx[:o_len])
    near = np.abs(logits[diff] - kth) <= TOPK_REL * abs(kth)
    assert np.all(near), "slots %s differ and are not near the k-th score" % diff[~near][:10]
    TOPK_STATS["differ"] += int(diff.size)
    TOPK_STATS["in_band"] += int(np.count_nonzero(np.abs(logits - kth) <= TOPK_REL * abs(kth)))
    return int(diff.size)


def check_attention(out_gpu, out_ref, what=""):
    """out_gpu: float array of the bf16 output; out_ref: oracle double."""
    err = np.abs(out_gpu.astype(np.float64) - out_ref)
    rel = np.linalg.norm(out_gpu.astype(np.float64) - out_ref) / max(np.linalg.norm(out_ref), 1e-30)
    assert err.max() <= ATT_MAX_ABS, "%s max abs %g" % (what, err.max())
    assert err.mean() <= ATT_MEAN_ABS, "%s mean abs %g" % (what, err.mean())
    assert rel <= ATT_REL_L2, "%s rel L2 %g" % (what, rel)
    return float(err.max()), float(err.mean()), float(rel)


SCALE_V4 = 1.0 / math.sqrt(512)
V4_PAGE_BYTES = 64 * 584


def make_v4_decode_inputs(layer_type, batch, ctx, n_heads, topk, seed, comp_pool=8192, peaky=False,
                          device="cuda"):
    """One layer's decode inputs in the V4-native geometry: compressed and SWA
    caches both of 584-byte rows (oracle-quantised N(0,1)/sqrt(512) rows, nope
    448), bf16 queries [batch][n_heads][512], and per sequence either random
    top-k slots (c4a), sorted metadata slots (c128a) or none (swaonly)."""
    g = synth.rng(seed)
    ctx = np.broadcast_to(np.asarray(ctx, np.int64), (batch,)).astype(np.int32).copy()
    ratio = {4: 4, 128: 128, 1: 0}[layer_type]
    d = DecodeInputs()
    d.layer_type, d.batch, d.ctx, d.n_heads, d.topk = layer_type, batch, ctx, n_heads, topk
    d.n_c = ((ctx // ratio) if ratio else np.zeros(batch, np.int64)).astype(np.int32)
    d.p = (ctx - 1).astype(np.int32)
    # SWA: the window's pages only, each page filled with 64 quantised rows
    swa_lp = int(ctx.max() + 63) // 64
    d.swa_bt = np.full((batch, swa_lp), -1, np.int32)
    n_pages = 0
    for b in range(batch):
        for lp in range(max(0, int(d.p[b]) - 127) // 64, int(d.p[b]) // 64 + 1):
            d.swa_bt[b, lp] = n_pages
            n_pages += 1
    perm = g.permutation(n_pages).astype(np.int32)
    d.swa_bt = np.where(d.swa_bt >= 0, perm[np.maximum(d.swa_bt, 0)], -1).astype(np.int32)
    d.swa = np.zeros(n_pages * V4_PAGE_BYTES, np.uint8)
    for pg in range(n_pages):
        data, sc = oracle.quant_mla_rows(synth.normal(g, (64, 512), SCALE_V4), nope_dim=448)
        oracle.page_write(oracle.MLA_KIND, d.swa, np.array([pg], np.int32), data, sc, nope_dim=448)
    d.comp = None
    if ratio:
        cp = int(max(1, (d.n_c.max() + 63) // 64))
        d.comp_bt = synth.page_tables(g, batch, cp, extra_pages=1)
        pool_n = int(min(comp_pool, max(1, d.n_c.sum())))
        pool_z = synth.normal(g, (pool_n, 512), SCALE_V4)
        pool_data, pool_sc = oracle.quant_mla_rows(pool_z, nope_dim=448)
        d.comp = np.zeros((batch * cp + 1) * V4_PAGE_BYTES, np.uint8)
        picks = []
        for b in range(batch):
            pick = g.integers(0, pool_n, size=int(d.n_c[b]))
            oracle.page_write(oracle.MLA_KIND, d.comp, d.comp_bt[b], pool_data[pick], pool_sc[pick], nope_dim=448)
            picks.append(pick)
        d.idx = np.full((batch, topk), -1, np.int32)
        d.idx_len = np.zeros(batch, np.int32)
        for b in range(batch):
            s = synth.sorted_sample(g, int(d.n_c[b]), topk)
            if layer_type == 4:
                s = g.permutation(s)               # c4a: any order
            d.idx[b, :len(s)] = s
            d.idx_len[b] = len(s)
    q = synth.normal(g, (batch, n_heads, 512), SCALE_V4)
    if peaky and ratio:
        for b in range(batch):
            if d.n_c[b] == 0:
                continue
            for h in range(n_heads):
                sel = d.idx[b, g.integers(0, max(1, int(d.idx_len[b])), size=4)]
                q[b, h] = (150.0 * pool_z[picks[b][sel]].sum(axis=0)).astype(np.float32)
    d.q = bf16_bits(q)
    d.t = {"q": bits_tensor(d.q, device), "swa": dev(d.swa, device), "swa_bt": dev(d.swa_bt, device),
           "ctx": dev(d.ctx, device)}
    if ratio:
        d.t.update(comp=dev(d.comp, device), comp_bt=dev(d.comp_bt, device), idx=dev(d.idx, device),
                   idx_len=dev(d.idx_len, device))
    return d


def oracle_v4(d, b):
    if d.comp is None:
        return oracle.sparse_mla_v4(d.q[b], None, None, None, 0, d.swa, d.swa_bt[b], int(d.p[b]), SCALE_V4)
    return oracle.sparse_mla_v4(d.q[b], d.comp, d.comp_bt[b], d.idx[b], int(d.idx_len[b]), d.swa, d.swa_bt[b],
                                int(d.p[b]), SCALE_V4)
