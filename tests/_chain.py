"""A decode loop of one c4a layer exactly as the benchmark runs it: per step
dsv4_compress_insert_pair (both compressor streams, one token per sequence),
dsv4_indexer_topk and dsv4_sparse_mla_decode, back to back on one stream
(programmatic dependent launch between them), captured in a CUDA graph and
replayed.  Steps include ratio-4 boundaries: the slot emitted by the
compressor in a step must be visible to that step's indexer and attention.

With v4=True the layer is in the V4-native geometry: 512-dim main stream
(448 FP8 nope + 64 bf16 rope, 584-byte rows), FP8 SWA rows, K = V attention,
and each step ends with dsv4_inv_rope_fp8_quant of the attention output.

Expected values come from the oracle: cache entries (pool -> RMSNorm -> RoPE
-> quantise), indexer logits, top-k, attention and the output quantisation.  Inputs come from the
seeded generators; at boundary steps the queries are built from the oracle's
entry for the new slot so that the indexer must select it and the attention
must be dominated by it.
"""
import concurrent.futures
import math
import os

import numpy as np
import torch

import oracle
from deepseek_v4_compressed_gb300 import binding as B
from deepseek_v4_compressed_gb300 import synth

from _util import SCALE, SCALE_V4, bf16_bits, bits_tensor, check_attention, check_topk, dev

EPS = 1e-6
D_IDX = 128


def _pool():
    return concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4))


NOPE = {B.CACHE_MLA: 512, B.CACHE_V4: 448, B.CACHE_IDX: 64, B.CACHE_IDX_FP4: 64}


def oracle_entry(kind, ks, ape, w, cs, p):
    """The compressed entry emitted at boundary p (oracle steps, one entry)."""
    nope = NOPE[kind]
    y = oracle.compress_pool(4, ks, ape, p)
    z = oracle.rmsnorm(y, w, EPS)
    z[nope:] = oracle.rope_gptj(z[nope:], cs[(p // 4) * 4])
    if kind == B.CACHE_IDX_FP4:
        d, s = oracle.quant_idx_fp4_rows(z[None])
    elif kind != B.CACHE_IDX:
        d, s = oracle.quant_mla_rows(z[None], nope_dim=nope)
    else:
        d, s = oracle.quant_idx_rows(z[None])
    return d[0], s[0]


def idx_key_values(data, sc, fp4):
    """An indexer entry's 128 key values (FP8 codes x scale, or the MXFP4
    codes x their block exponents)."""
    if fp4:
        codes = np.stack([data & 15, data >> 4], axis=-1).reshape(128)
        return oracle.e2m1_to_f64(codes) * np.repeat(2.0 ** (sc.astype(np.int64) - 127), 32)
    return oracle.e4m3_to_f64(data) * float(sc)


def dequant_nope(data, sc, nope=512):
    return oracle.e4m3_to_f64(data[:nope]) * np.repeat(2.0 ** (sc[:nope // 64].astype(np.int64) - 127), 64)


def dequant_row(data, sc, nope):
    """The whole dequantised key (nope dims, then the bf16 rope dims)."""
    rope = oracle.bf16_to_f32(np.ascontiguousarray(data[nope:]).view(np.uint16)).astype(np.float64)
    return np.concatenate([dequant_nope(data, sc, nope), rope])


def run_chain(batch, L0, n_steps, H, HI, k, seed, prefill, graph=True, v4=False, idx_fp4=False):
    """prefill: 'stream' runs tokens 0..L0-1 through the library's multi-token
    compressor (caches and ring built by the library, checked against the
    oracle's whole-stream entries); 'direct' writes oracle-quantised random
    rows into the slots below L0 // 4 and the ring rows of tokens L0-8..L0-1
    (the compressor state layout of dsv4.h) so that long contexts stay cheap."""
    g = synth.rng(seed)
    kind_m = B.CACHE_V4 if v4 else B.CACHE_MLA
    kind_i = B.CACHE_IDX_FP4 if idx_fp4 else B.CACHE_IDX
    okind_i = oracle.IDX_FP4_KIND if idx_fp4 else oracle.IDX_KIND
    D_MAIN = 512 if v4 else 576
    nope_m = NOPE[kind_m]
    scale = SCALE_V4 if v4 else SCALE
    L0 = np.broadcast_to(np.asarray(L0, np.int64), (batch,)).astype(np.int64).copy()
    T = L0 + n_steps
    Tmax = int(T.max())
    cs = oracle.rope_table(Tmax + 1, 64)
    ape_m = synth.normal(g, (4, 2 * D_MAIN), 0.1)
    ape_i = synth.normal(g, (4, 2 * D_IDX), 0.1)
    w_m = synth.uniform(g, D_MAIN, 0.5, 1.5)
    w_i = synth.uniform(g, D_IDX, 0.5, 1.5)
    lo = np.zeros(batch, np.int64) if prefill == "stream" else np.maximum(L0 - 8, 0)
    ks_m, ks_i = [], []
    for b in range(batch):
        km = np.zeros((int(T[b]), 4 * D_MAIN), np.uint16)
        ki = np.zeros((int(T[b]), 4 * D_IDX), np.uint16)
        km[lo[b]:] = bf16_bits(synth.normal(g, (int(T[b] - lo[b]), 4 * D_MAIN)))
        ki[lo[b]:] = bf16_bits(synth.normal(g, (int(T[b] - lo[b]), 4 * D_IDX)))
        ks_m.append(km)
        ks_i.append(ki)

    # entries of every slot below T // 4, in the oracle
    n_ent = T // 4
    pps = int(max(1, (n_ent.max() + 63) // 64))
    comp_bt = synth.page_tables(g, batch, pps, extra_pages=1)
    idx_bt = synth.page_tables(g, batch, pps, extra_pages=1)
    ent_m, ent_i = [], []

    def entries(b):
        if prefill == "stream":
            dm, sm = oracle.compress_stream(0, 4, ks_m[b], ape_m, w_m, EPS, cs, nope_dim=nope_m)
            di, si = oracle.compress_stream(okind_i, 4, ks_i[b], ape_i, w_i, EPS, cs, nope_dim=64)
            return (dm, sm), (di, si)
        return None

    if prefill == "stream":
        with _pool() as ex:
            res = list(ex.map(entries, range(batch)))
        ent_m = [r[0] for r in res]
        ent_i = [r[1] for r in res]
    else:
        pool_n = 4096
        pm, psm = oracle.quant_mla_rows(synth.normal(g, (pool_n, D_MAIN), 1.0), nope_dim=nope_m)
        for b in range(batch):
            n0 = int(L0[b] // 4)
            pick = g.integers(0, pool_n, size=int(n_ent[b]))
            dm, sm = pm[pick].copy(), psm[pick].copy()
            rows_i = synth.normal(g, (int(n_ent[b]), D_IDX), 1.0)
            di, si = oracle.quant_idx_fp4_rows(rows_i) if idx_fp4 else oracle.quant_idx_rows(rows_i)
            for p in range(int(L0[b]), int(T[b])):
                if (p + 1) % 4 == 0:
                    j = p // 4
                    dm[j], sm[j] = oracle_entry(kind_m, ks_m[b], ape_m, w_m, cs, p)
                    di[j], si[j] = oracle_entry(kind_i, ks_i[b], ape_i, w_i, cs, p)
            assert n0 <= n_ent[b]
            ent_m.append((dm, sm))
            ent_i.append((di, si))
    comp_o = np.zeros((batch * pps + 1) * oracle.page_bytes(0, nope_dim=nope_m), np.uint8)
    idx_o = np.zeros((batch * pps + 1) * oracle.page_bytes(okind_i), np.uint8)
    for b in range(batch):
        oracle.page_write(0, comp_o, comp_bt[b], *ent_m[b], nope_dim=nope_m)
        oracle.page_write(okind_i, idx_o, idx_bt[b], *ent_i[b], nope_dim=64)

    # SWA cache: rows of tokens max(0, L0 - 128) .. T - 1 (the windows of every step)
    swa_lp = (Tmax + 63) // 64
    swa_bt = np.full((batch, swa_lp), -1, np.int32)
    npg = 0
    for b in range(batch):
        for lp in range(max(0, int(L0[b]) - 128) // 64, (int(T[b]) - 1) // 64 + 1):
            swa_bt[b, lp] = npg
            npg += 1
    if v4:
        swa = np.zeros(npg * oracle.page_bytes(0, nope_dim=448), np.uint8)
        for pg in range(npg):
            data, sc = oracle.quant_mla_rows(synth.normal(g, (64, 512), SCALE_V4), nope_dim=448)
            oracle.page_write(0, swa, np.array([pg], np.int32), data, sc, nope_dim=448)
    else:
        swa = bf16_bits(synth.normal(g, (npg * 64, 576), SCALE))

    # per-step queries; at a boundary step the new slot's own codes / latent
    steps = []
    for s in range(n_steps):
        st = dict(p=(L0 + s).astype(np.int32))
        qi = oracle.f32_to_e4m3(synth.normal(g, (batch, HI, 128)))
        wq = synth.uniform(g, (batch, HI))
        q = synth.normal(g, (batch, H, D_MAIN), scale)
        st["boundary"] = [(int(st["p"][b]) + 1) % 4 == 0 for b in range(batch)]
        for b in range(batch):
            if st["boundary"][b]:
                j = int(st["p"][b]) // 4
                qi[b, :, :] = (ent_i[b][0][j] if not idx_fp4 else
                               oracle.f32_to_e4m3(idx_key_values(ent_i[b][0][j], ent_i[b][1][j], True)
                                                  .astype(np.float32) * 8.0))
                q[b, :, :nope_m] = dequant_nope(ent_m[b][0][j], ent_m[b][1][j], nope_m).astype(np.float32)
        st["qi"], st["w"], st["q"] = qi, wq, bf16_bits(q)
        steps.append(st)

    # ---- GPU
    plan = B.Plan(B.C4A, H, batch, k, Tmax, idx_heads=HI, kv_layout=B.KV_V4 if v4 else B.KV_576,
                  idx_format=B.IDX_FP4 if idx_fp4 else B.IDX_FP8)
    ws = plan.workspace()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    comp = torch.zeros(comp_o.size, dtype=torch.uint8, device="cuda")
    idxc = torch.zeros(idx_o.size, dtype=torch.uint8, device="cuda")
    t_comp_bt, t_idx_bt = dev(comp_bt), dev(idx_bt)
    st_m = torch.zeros((batch, 8, 4 * D_MAIN), dtype=torch.float32, device="cuda")
    st_i = torch.zeros((batch, 8, 4 * D_IDX), dtype=torch.float32, device="cuda")
    t_ape_m, t_ape_i, t_w_m, t_w_i, t_cs = dev(ape_m), dev(ape_i), dev(w_m), dev(w_i), dev(cs)
    seqs = dev(np.arange(batch, dtype=np.int32))
    if prefill == "stream":
        for kind, ks, ape, w, st, cache, bt in ((kind_m, ks_m, t_ape_m, t_w_m, st_m, comp, t_comp_bt),
                                                (kind_i, ks_i, t_ape_i, t_w_i, st_i, idxc, t_idx_bt)):
            rows, ps, sq = [], [], []
            for b in range(batch):
                rows.append(ks[b][:L0[b]])
                ps += list(range(int(L0[b])))
                sq += [b] * int(L0[b])
            B.compress_insert(kind, 4, bits_tensor(np.concatenate(rows)), dev(np.array(ps, np.int32)),
                              dev(np.array(sq, np.int32)), ape, w, EPS, t_cs, st, cache, bt, batch,
                              one_token_per_seq=False, status=status)
    else:
        # slots below L0 // 4 hold their entries already; the ring holds tokens L0-8 .. L0-1
        n0 = [int(L0[b] // 4) for b in range(batch)]
        part_c = np.zeros_like(comp_o)
        part_i = np.zeros_like(idx_o)
        for b in range(batch):
            oracle.page_write(0, part_c, comp_bt[b], ent_m[b][0][:n0[b]], ent_m[b][1][:n0[b]], nope_dim=nope_m)
            oracle.page_write(okind_i, part_i, idx_bt[b], ent_i[b][0][:n0[b]], ent_i[b][1][:n0[b]], nope_dim=64)
        comp.copy_(dev(part_c))
        idxc.copy_(dev(part_i))
        ring_m = np.zeros((batch, 8, 4 * D_MAIN), np.float32)
        ring_i = np.zeros((batch, 8, 4 * D_IDX), np.float32)
        for b in range(batch):
            for t in range(int(lo[b]), int(L0[b])):
                for ring, ks, ape, d in ((ring_m, ks_m, ape_m, D_MAIN), (ring_i, ks_i, ape_i, D_IDX)):
                    row = oracle.bf16_to_f32(ks[b][t])
                    ring[b, t % 8, :2 * d] = row[:2 * d]
                    ring[b, t % 8, 2 * d:] = (row[2 * d:] + ape[t % 4]).astype(np.float32)
        st_m.copy_(dev(ring_m))
        st_i.copy_(dev(ring_i))
    t_swa, t_swa_bt = (dev(swa) if v4 else bits_tensor(swa)), dev(swa_bt)
    gin = []
    for s, st in enumerate(steps):
        kvm = bits_tensor(np.stack([ks_m[b][st["p"][b]] for b in range(batch)]))
        kvi = bits_tensor(np.stack([ks_i[b][st["p"][b]] for b in range(batch)]))
        gin.append(dict(kvm=kvm, kvi=kvi, pos=dev(st["p"]), ctx=dev(st["p"] + 1), qi=dev(st["qi"]),
                        w=dev(st["w"]), q=bits_tensor(st["q"]),
                        idx=torch.full((batch, k), -9, dtype=torch.int32, device="cuda"),
                        len=torch.full((batch,), -9, dtype=torch.int32, device="cuda"),
                        out=torch.zeros((batch, H, 512), dtype=torch.bfloat16, device="cuda"),
                        lse=torch.zeros((batch, H), dtype=torch.float32, device="cuda"),
                        codes=torch.zeros((batch, H, 512), dtype=torch.uint8, device="cuda"),
                        scales=torch.zeros((batch, H, 4), dtype=torch.float32, device="cuda")))
    torch.cuda.synchronize()

    def decode_steps():
        for x in gin:
            B.compress_insert_pair(
                dict(kind=kind_m, ratio=4, kv_score=x["kvm"], positions=x["pos"], seqs=seqs, ape=t_ape_m,
                     rms_weight=t_w_m, rms_eps=EPS, cos_sin=t_cs, state=st_m, cache=comp, block_table=t_comp_bt,
                     num_seqs=batch, status=status),
                dict(kind=kind_i, ratio=4, kv_score=x["kvi"], positions=x["pos"], seqs=seqs, ape=t_ape_i,
                     rms_weight=t_w_i, rms_eps=EPS, cos_sin=t_cs, state=st_i, cache=idxc, block_table=t_idx_bt,
                     num_seqs=batch, status=status))
            B.indexer_topk(plan, x["qi"], x["w"], idxc, t_idx_bt, x["ctx"], x["idx"], x["len"], ws, status)
            B.sparse_mla_decode(plan, x["q"], t_swa, t_swa_bt, x["ctx"], x["out"], ws, comp_cache=comp,
                                comp_block_table=t_comp_bt, topk_idx=x["idx"], topk_len=x["len"], lse=x["lse"],
                                status=status)
            if v4:
                B.inv_rope_fp8_quant(x["out"], x["pos"], t_cs, x["codes"], x["scales"], status=status)

    if graph:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            decode_steps()
        gr.replay()
    else:
        decode_steps()
    torch.cuda.synchronize()
    st_code, bits = B.read_device_status(status)
    assert st_code == B.OK, bits

    # ---- checks
    assert np.array_equal(comp.cpu().numpy(), comp_o), "compressed cache bytes differ from the oracle"
    assert np.array_equal(idxc.cpu().numpy(), idx_o), "indexer cache bytes differ from the oracle"
    tolerated = 0
    n_boundary = 0
    for s, (st, x) in enumerate(zip(steps, gin)):
        gidx, glen = x["idx"].cpu().numpy(), x["len"].cpu().numpy()
        gout, glse = x["out"].float().cpu().numpy(), x["lse"].cpu().numpy()
        gcodes, gscales = x["codes"].cpu().numpy(), x["scales"].cpu().numpy()

        def check(b):
            p = int(st["p"][b])
            n_c = (p + 1) // 4
            f = oracle.indexer_logits_fp4 if idx_fp4 else oracle.indexer_logits
            logits = f(st["qi"][b], st["w"][b], idx_o, idx_bt[b], n_c)
            tol = check_topk(gidx[b], int(glen[b]), logits, k)
            if st["boundary"][b]:
                assert p // 4 in set(gidx[b][:glen[b]].tolist()), "step %d seq %d: new slot not selected" % (s, b)
            sel = gidx[b][:glen[b]].copy()
            if v4:
                ref, ref_lse = oracle.sparse_mla_v4(st["q"][b], comp_o, comp_bt[b], sel, int(glen[b]), swa,
                                                    swa_bt[b], p, SCALE_V4)
                # the step's output quantisation, bit for bit on the kernel's own bf16 output
                o_bits = oracle.f32_to_bf16(gout[b].astype(np.float32))
                wc, wsc = oracle.inv_rope_fp8_quant(o_bits, p, cs)
                assert np.array_equal(gcodes[b], wc) and np.array_equal(gscales[b], wsc), \
                    "step %d seq %d: output quant differs" % (s, b)
            else:
                ref, ref_lse, _ = oracle.sparse_mla(st["q"][b], comp_o, comp_bt[b], sel, int(glen[b]), swa,
                                                    swa_bt[b], p, SCALE)
            check_attention(gout[b], ref, "step %d seq %d" % (s, b))
            np.testing.assert_allclose(glse[b], ref_lse, rtol=1e-3, atol=1e-3)
            if st["boundary"][b]:
                # the new slot dominates: the output is close to its latent (V4: its whole row)
                ent = (ent_m[b][0][p // 4], ent_m[b][1][p // 4])
                lat = dequant_row(*ent, nope_m) if v4 else dequant_nope(*ent)
                assert np.linalg.norm(gout[b] - lat[None, :]) / np.linalg.norm(np.broadcast_to(lat, gout[b].shape)) < 0.1
            return tol

        with _pool() as ex:
            tolerated += sum(ex.map(check, range(batch)))
        n_boundary += sum(st["boundary"])
    return tolerated, n_boundary
