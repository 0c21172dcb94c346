"""GPU parity of dsv4_compress_insert / dsv4_cache_insert_rows: cache bytes must
equal the oracle's bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_gb300 import binding as B
from deepseek_v4_compressed_gb300 import synth

from _util import bf16_bits, bits_tensor, dev

pytestmark = pytest.mark.gpu

EPS = 1e-6

# per cache kind: stream dimension, (data, scale) bytes of an entry, page bytes,
# the oracle's kind and nope dims
DIM = {B.CACHE_MLA: 576, B.CACHE_IDX: 128, B.CACHE_V4: 512}
ENTRY = {B.CACHE_MLA: (640, 8), B.CACHE_IDX: (128, 4), B.CACHE_V4: (576, 8)}
ORACLE = {B.CACHE_MLA: (oracle.MLA_KIND, 512), B.CACHE_IDX: (oracle.IDX_KIND, 64), B.CACHE_V4: (oracle.MLA_KIND, 448)}


def make_stream(kind, ratio, n_tok, seed, w_ones=False):
    g = synth.rng(seed)
    d = DIM[kind]
    coff = 2 if ratio == 4 else 1
    ks = bf16_bits(synth.normal(g, (n_tok, 2 * coff * d)))
    ape = synth.normal(g, (ratio, coff * d), 0.1)
    w = np.ones(d, np.float32) if w_ones else synth.uniform(g, d, 0.5, 1.5)
    return ks, ape, w


def entries_from_pages(kind, cache, bt_row, n):
    """Read entries 0..n-1 (slot order) back out of the paged bytes."""
    data_b, sc_b = ENTRY[kind]
    if n == 0:
        return np.zeros((0, data_b), np.uint8), np.zeros((0, sc_b), np.uint8)
    pages = cache.reshape(-1, 64 * (data_b + sc_b))
    data = np.stack([pages[bt_row[j // 64], (j % 64) * data_b:(j % 64 + 1) * data_b] for j in range(n)])
    sc = np.stack([pages[bt_row[j // 64], 64 * data_b + (j % 64) * sc_b: 64 * data_b + (j % 64 + 1) * sc_b]
                   for j in range(n)])
    return data, sc


def run_gpu_streams(kind, ratio, streams, chunks, cos_sin):
    """streams: list of (kv_score bits [T_b, row], ape, w) per sequence -- all sequences
    share ape / w (one layer).  chunks: per-step token counts per sequence (list of
    lists) or None for one token per step.  Returns per-sequence cache entries."""
    nseq = len(streams)
    d = DIM[kind]
    coff = 2 if ratio == 4 else 1
    ape, w = streams[0][1], streams[0][2]
    n_ent = [s[0].shape[0] // ratio for s in streams]
    pps = max(1, (max(n_ent) + 63) // 64)
    g = synth.rng(99)
    bt = synth.page_tables(g, nseq, pps, extra_pages=2)
    page_b = B.PAGE_BYTES[kind]
    cache = torch.zeros((nseq * pps + 2) * page_b, dtype=torch.uint8, device="cuda")
    state = torch.zeros((nseq, coff * ratio, 2 * coff * d), dtype=torch.float32, device="cuda")
    t_ape, t_w, t_cs, t_bt = dev(ape), dev(w), dev(cos_sin), dev(bt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t_ks = [bits_tensor(s[0]) for s in streams]
    pos = [0] * nseq
    step = 0
    while any(pos[b] < streams[b][0].shape[0] for b in range(nseq)):
        rows, ps, sq = [], [], []
        for b in range(nseq):
            n_b = streams[b][0].shape[0]
            if pos[b] >= n_b:
                continue
            take = 1 if chunks is None else chunks[b][step % len(chunks[b])]
            take = min(take, n_b - pos[b])
            rows.append(t_ks[b][pos[b]:pos[b] + take])
            ps += list(range(pos[b], pos[b] + take))
            sq += [b] * take
            pos[b] += take
        kv = torch.cat(rows, 0).contiguous()
        one = len(sq) == len(set(sq))
        B.compress_insert(kind, ratio, kv, dev(np.array(ps, np.int32)), dev(np.array(sq, np.int32)),
                          t_ape, t_w, EPS, t_cs, state, cache, t_bt, nseq, one_token_per_seq=one,
                          status=status)
        step += 1
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == B.OK, bits
    host = cache.cpu().numpy()
    return [entries_from_pages(kind, host, bt[b], n_ent[b]) for b in range(nseq)]


def oracle_entries(kind, ratio, ks, ape, w, cos_sin):
    okind, nope = ORACLE[kind]
    data, sc = oracle.compress_stream(okind, ratio, ks, ape, w, EPS, cos_sin, nope_dim=nope)
    if kind == B.CACHE_IDX:
        sc = sc.view(np.uint8).reshape(-1, 4)
    return data, sc


def assert_bytes_equal(got, want, what):
    gd, gs = got
    wd, ws = want
    assert gd.shape == wd.shape, what
    bad = np.nonzero(np.any(gd != wd, axis=1) | np.any(gs != ws, axis=1))[0]
    assert bad.size == 0, "%s: %d of %d entries differ, first %s" % (what, bad.size, gd.shape[0], bad[:8])


@pytest.mark.parametrize("kind,ratio,n_tok", [(B.CACHE_MLA, 4, 512), (B.CACHE_IDX, 4, 512),
                                              (B.CACHE_MLA, 128, 384), (B.CACHE_V4, 4, 512),
                                              (B.CACHE_V4, 128, 384)])
def test_decode_stream_bit_exact(kind, ratio, n_tok):
    ks, ape, w = make_stream(kind, ratio, n_tok, seed=kind * 10 + ratio, w_ones=(ratio == 4))
    cs = oracle.rope_table(n_tok, 64)
    got = run_gpu_streams(kind, ratio, [(ks, ape, w)], None, cs)[0]
    assert_bytes_equal(got, oracle_entries(kind, ratio, ks, ape, w, cs), "decode stream")


@pytest.mark.parametrize("kind,ratio", [(B.CACHE_MLA, 4), (B.CACHE_IDX, 4), (B.CACHE_MLA, 128),
                                        (B.CACHE_V4, 4), (B.CACHE_V4, 128)])
def test_chunked_stream_bit_exact(kind, ratio):
    n_tok = 700 if ratio == 4 else 600
    ks, ape, w = make_stream(kind, ratio, n_tok, seed=77 + ratio)
    cs = oracle.rope_table(n_tok, 64)
    chunks = [[1, 3, 7, 16, 2, 64, 5, 200, 9]]   # spans ring-size chunks (200 > 128)
    got = run_gpu_streams(kind, ratio, [(ks, ape, w)], chunks, cs)[0]
    assert_bytes_equal(got, oracle_entries(kind, ratio, ks, ape, w, cs), "chunked stream")


@pytest.mark.parametrize("ratio", [4, 128])
def test_batched_sequences_bit_exact(ratio):
    lens = [13, 200, 517, 3] if ratio == 4 else [130, 300, 256]
    ks0, ape, w = make_stream(B.CACHE_MLA, ratio, 1, seed=5)
    streams = []
    for i, L in enumerate(lens):
        ks, _, _ = make_stream(B.CACHE_MLA, ratio, L, seed=500 + i)
        streams.append((ks, ape, w))
    cs = oracle.rope_table(max(lens), 64)
    for chunks in [None, [[1, 2, 3]] * len(lens)]:
        got = run_gpu_streams(B.CACHE_MLA, ratio, streams, chunks, cs)
        for b, (ks, _, _) in enumerate(streams):
            if ks.shape[0] >= ratio:
                assert_bytes_equal(got[b], oracle_entries(B.CACHE_MLA, ratio, ks, ape, w, cs),
                                   "seq %d" % b)


@pytest.mark.parametrize("kind", [B.CACHE_MLA, B.CACHE_IDX, B.CACHE_V4])
def test_insert_rows_bit_exact(kind):
    g = synth.rng(31 + kind)
    d = DIM[kind]
    n = 300
    rows = synth.normal(g, (n, d), 1.0)
    rows *= (10.0 ** g.uniform(-6, 3, size=(n, 1))).astype(np.float32)
    rows[0] = 0.0
    rows[1, :64] = 1e-30
    rows[2, :64] = 448.0
    nseq = 2
    pps = 4
    bt = synth.page_tables(g, nseq, pps)
    seqs = np.array([i % nseq for i in range(n)], np.int32)
    slots = np.array([i // nseq for i in range(n)], np.int32)
    page_b = B.PAGE_BYTES[kind]
    # pre-filled with 0xff: every byte of an entry (the V4 pad byte too) is written
    cache = torch.full((nseq * pps * page_b,), 255, dtype=torch.uint8, device="cuda")
    B.cache_insert_rows(kind, dev(rows), dev(seqs), dev(slots), cache, dev(bt))
    host = cache.cpu().numpy()
    if kind != B.CACHE_IDX:
        wd, ws = oracle.quant_mla_rows(rows, nope_dim=ORACLE[kind][1])
    else:
        wd, wsf = oracle.quant_idx_rows(rows)
        ws = wsf.view(np.uint8).reshape(-1, 4)
    for b in range(nseq):
        sel = seqs == b
        got = entries_from_pages(kind, host, bt[b], int(sel.sum()))
        assert_bytes_equal(got, (wd[sel], ws[sel]), "insert rows seq %d" % b)


@pytest.mark.parametrize("ratio,main_kind", [(4, B.CACHE_MLA), (128, B.CACHE_MLA), (4, B.CACHE_V4),
                                             (128, B.CACHE_V4)])
def test_pair_launch_bit_exact(ratio, main_kind):
    """dsv4_compress_insert_pair (main + indexer streams in one launch, one token
    per sequence per step) writes the same bytes as the oracle for both caches."""
    lens = [300, 129, 517] if ratio == 4 else [300, 256, 384]
    nseq = len(lens)
    cs = oracle.rope_table(max(lens), 64)
    t_cs = dev(cs)
    kinds = {"main": (main_kind, ratio, DIM[main_kind]), "idx": (B.CACHE_IDX, 4, 128)}
    setup = {}
    for name, (kind, r, d) in kinds.items():
        coff = 2 if r == 4 else 1
        _, ape, w = make_stream(kind, r, 1, seed=900 + kind)
        streams = [make_stream(kind, r, L, seed=910 + 7 * kind + i)[0] for i, L in enumerate(lens)]
        n_ent = max(L // r for L in lens)
        pps = max(1, (n_ent + 63) // 64)
        bt = synth.page_tables(synth.rng(40 + kind), nseq, pps, extra_pages=1)
        page_b = B.PAGE_BYTES[kind]
        setup[name] = dict(kind=kind, ratio=r, ape=ape, w=w, streams=streams, bt=bt,
                           t_ks=[bits_tensor(s) for s in streams],
                           cache=torch.zeros((nseq * pps + 1) * page_b, dtype=torch.uint8, device="cuda"),
                           state=torch.zeros((nseq, coff * r, 2 * coff * d), dtype=torch.float32, device="cuda"),
                           t_ape=dev(ape), t_w=dev(w), t_bt=dev(bt))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(max(lens)):
        live = [b for b in range(nseq) if step < lens[b]]
        pos = dev(np.full(len(live), step, np.int32))
        seqs = dev(np.array(live, np.int32))
        args = {}
        for name, st in setup.items():
            kv = torch.cat([st["t_ks"][b][step:step + 1] for b in live], 0).contiguous()
            args[name] = dict(kind=st["kind"], ratio=st["ratio"], kv_score=kv, positions=pos, seqs=seqs,
                              ape=st["t_ape"], rms_weight=st["t_w"], rms_eps=EPS, cos_sin=t_cs,
                              state=st["state"], cache=st["cache"], block_table=st["t_bt"], num_seqs=nseq,
                              status=status)
        B.compress_insert_pair(args["main"], args["idx"])
    torch.cuda.synchronize()
    s, bits = B.read_device_status(status)
    assert s == B.OK, bits
    for name, st in setup.items():
        host = st["cache"].cpu().numpy()
        for b in range(nseq):
            n = lens[b] // st["ratio"]
            got = entries_from_pages(st["kind"], host, st["bt"][b], n)
            want = oracle_entries(st["kind"], st["ratio"], st["streams"][b], st["ape"], st["w"], cs)
            assert_bytes_equal(got, want, "%s seq %d" % (name, b))


@pytest.mark.parametrize("kind,d", [(B.CACHE_IDX, 128), (B.CACHE_MLA, 576)])
def test_rmsnorm_order_sensitive_vector_bytes_equal(kind, d):
    """A stream whose RMSNorm sum of squares rounds differently in ascending
    channel order than in the fixed butterfly-then-groups order (the fp32 mean
    squares differ, asserted here): the kernel's cache bytes still equal the
    oracle's, token by token and in one multi-token call."""
    from _rms_case import ascending_sum, butterfly_sum, mean_square_pair, pooled_vector, token_rows
    y = pooled_vector(d)
    assert ascending_sum(y) != butterfly_sum(y)
    ms_asc, ms_tree = mean_square_pair(d)
    assert ms_asc != ms_tree
    ks = token_rows(d)
    ape = np.zeros((4, 2 * d), np.float32)
    w = np.ones(d, np.float32)
    cs = oracle.rope_table(8, 64)
    want = oracle_entries(kind, 4, ks, ape, w, cs)
    assert want[0].shape[0] == 1
    for chunks in (None, [[4]]):
        got = run_gpu_streams(kind, 4, [(ks, ape, w)], chunks, cs)
        assert_bytes_equal(got[0], want, "order-sensitive d=%d chunks=%s" % (d, chunks))



@pytest.mark.parametrize("kind,d", [(B.CACHE_MLA, 576), (B.CACHE_V4, 512)])
def test_rmsnorm_order_sensitive_vector_bytes_equal_ratio128(kind, d):
    """The same order-sensitive vector through a ratio-128 stream, whose
    boundary spreads a token's 64-channel warps over a cluster of CTAs (the
    warp totals exchanged between them): the cache bytes equal the oracle's,
    token by token and in one multi-token call."""
    from _rms_case import ascending_sum, butterfly_sum, mean_square_pair, pooled_vector, token_rows_c128
    y = pooled_vector(d)
    assert ascending_sum(y) != butterfly_sum(y)
    ms_asc, ms_tree = mean_square_pair(d)
    assert ms_asc != ms_tree
    ks = token_rows_c128(d)
    ape = np.zeros((128, d), np.float32)
    w = np.ones(d, np.float32)
    cs = oracle.rope_table(128, 64)
    want = oracle_entries(kind, 128, ks, ape, w, cs)
    assert want[0].shape[0] == 1
    for chunks in (None, [[128]]):
        got = run_gpu_streams(kind, 128, [(ks, ape, w)], chunks, cs)
        assert_bytes_equal(got[0], want, "order-sensitive ratio 128 d=%d chunks=%s" % (d, chunks))