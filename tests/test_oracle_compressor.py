"""Pins of the oracle's compressor (pool -> RMSNorm -> RoPE -> quantise -> page).

Window membership and RoPE anchors come from the pages' worked examples
(tests/golden/compressor_windows.txt); pooling, normalisation and rotation are
checked against closed forms; the quantised bytes against the (separately
pinned) E4M3 / UE8M0 / bf16 codecs.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def to_bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def parse_tokens(s):
    s = s.strip()
    if s == "-":
        return []
    if ".." in s:
        a, b = s.split("..")
        return list(range(int(a), int(b) + 1))
    return [int(t) for t in s.split()]


def golden_windows():
    rows = []
    with open(os.path.join(GOLDEN, "compressor_windows.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            head, b0, b1 = line.split("|")
            ratio, p, slot, rope_pos = (int(v) for v in head.split())
            rows.append((ratio, p, slot, rope_pos, parse_tokens(b0), parse_tokens(b1)))
    return rows


def signature_stream(ratio, n_tokens, d=4):
    """kv block a of token t = 2^t, block b = 2^(t+8) (ratio 4); block 0 = t (ratio 128);
    all scores and APE zero, so every window row weighs the same."""
    coff = 2 if ratio == 4 else 1
    rows = np.zeros((n_tokens, 2 * coff * d), np.float32)
    for t in range(n_tokens):
        if ratio == 4:
            rows[t, 0:d] = 2.0 ** t
            rows[t, d:2 * d] = 2.0 ** (t + 8)
        else:
            rows[t, 0:d] = float(t)
    ape = np.zeros((ratio, coff * d), np.float32)
    return to_bf16_bits(rows), ape


@pytest.mark.parametrize("row", golden_windows())
def test_window_membership_matches_pages(row):
    ratio, p, slot, rope_pos, block0, block1 = row
    assert slot == p // ratio and (p + 1) % ratio == 0
    assert rope_pos == (p // ratio) * ratio
    n = p + 1
    if ratio == 4:
        assert max(block0 + block1) < 16
        ks, ape = signature_stream(4, n)
        y = oracle.compress_pool(4, ks, ape, p)
        expect_sum = sum(2.0 ** t for t in block0) + sum(2.0 ** (t + 8) for t in block1)
        count = len(block0) + len(block1)
        assert np.all(y == np.float32(expect_sum / count))
    else:
        ks, ape = signature_stream(128, n)
        y = oracle.compress_pool(128, ks, ape, p)
        assert np.all(y == np.float32(sum(block0) / len(block0)))


@pytest.mark.parametrize("ratio", [4, 128])
def test_emission_only_at_boundaries_and_slot_counts(ratio):
    n = 3 * ratio + ratio // 2
    ks, ape = signature_stream(ratio, n)
    for p in range(n):
        y = oracle.compress_pool(ratio, ks, ape, p)
        assert (y is not None) == ((p + 1) % ratio == 0)
    # slot counts n_c = floor(L / ratio), e.g. the talk's N = 128 -> 32 and 1 entries
    for L, expect in [(128, 128 // ratio), (512, 512 // ratio), (n, n // ratio)]:
        g = np.random.default_rng(L)
        coff = 2 if ratio == 4 else 1
        d = 64 + 64
        ks2 = to_bf16_bits(g.normal(size=(L, 2 * coff * d)))
        data, _ = oracle.compress_stream(oracle.IDX_KIND, ratio, ks2,
                                         np.zeros((ratio, coff * d), np.float32),
                                         np.ones(d, np.float32), 1e-6,
                                         oracle.rope_table(L, 64), nope_dim=64)
        assert data.shape[0] == expect
    assert 128 // 4 == 32 and 128 // 128 == 1


def test_equal_scores_give_window_mean():
    g = np.random.default_rng(1)
    d, p = 16, 11
    kv = g.normal(size=(p + 1, 2 * d)).astype(np.float32)
    rows = np.concatenate([kv, np.full((p + 1, 2 * d), 0.75, np.float32)], axis=1)
    ks = to_bf16_bits(rows)
    kvb = oracle.bf16_to_f32(ks[:, : 2 * d]).astype(np.float64)
    y = oracle.compress_pool(4, ks, np.zeros((4, 2 * d), np.float32), p)
    expect = (kvb[p - 7:p - 3, 0:d].sum(0) + kvb[p - 3:p + 1, d:2 * d].sum(0)) / 8
    np.testing.assert_allclose(y, expect, rtol=2e-6, atol=1e-7)


def test_dominant_score_selects_its_row():
    g = np.random.default_rng(2)
    d, p = 8, 7
    kv = g.uniform(0.5, 2.0, size=(p + 1, 2 * d)).astype(np.float32)
    score = g.normal(size=(p + 1, 2 * d)).astype(np.float32) * 0.1
    score[2, 0:d] += 30.0          # token 2 is in the old group: block a decides
    ks = to_bf16_bits(np.concatenate([kv, score], axis=1))
    y = oracle.compress_pool(4, ks, np.zeros((4, 2 * d), np.float32), p)
    np.testing.assert_allclose(y, oracle.bf16_to_f32(ks[2, 0:d]), rtol=1e-6)


def test_ape_is_indexed_by_token_position():
    # ape[t % ratio] boosts the token whose position is 1 mod 4 in each group
    d, p = 8, 7
    g = np.random.default_rng(3)
    kv = g.uniform(0.5, 2.0, size=(p + 1, 2 * d)).astype(np.float32)
    rows = np.concatenate([kv, np.zeros((p + 1, 2 * d), np.float32)], axis=1)
    ks = to_bf16_bits(rows)
    ape = np.zeros((4, 2 * d), np.float32)
    ape[1, 0:d] = 40.0      # residue 1, block a  -> token 1 (old group)
    ape[2, d:2 * d] = 40.0  # residue 2, block b  -> token 6 (new group)
    y = oracle.compress_pool(4, ks, ape, p)
    t1 = oracle.bf16_to_f32(ks[1, 0:d]).astype(np.float64)
    t6 = oracle.bf16_to_f32(ks[6, d:2 * d]).astype(np.float64)
    np.testing.assert_allclose(y, (t1 + t6) / 2, rtol=1e-6)


def test_c128_constant_kv_is_fixed_point():
    g = np.random.default_rng(4)
    d, p = 8, 255
    kv = np.full((p + 1, d), 1.5, np.float32)
    score = g.normal(size=(p + 1, d)).astype(np.float32) * 3
    ks = to_bf16_bits(np.concatenate([kv, score], axis=1))
    y = oracle.compress_pool(128, ks, np.zeros((128, d), np.float32), p)
    np.testing.assert_allclose(y, 1.5, rtol=2e-6)


def test_rmsnorm_closed_form():
    d = 576
    w = np.linspace(0.5, 1.5, d).astype(np.float32)
    z = oracle.rmsnorm(np.full(d, 2.0, np.float32), w, 1e-6)
    np.testing.assert_allclose(z, w * 2.0 / math.sqrt(4.0 + 1e-6), rtol=1e-6)
    g = np.random.default_rng(5)
    y = g.normal(size=d).astype(np.float32) * 3
    z = oracle.rmsnorm(y, np.ones(d, np.float32), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(z.astype(np.float64) ** 2)), 1.0, rtol=1e-6)


def test_rope_table_closed_forms():
    T = oracle.rope_table(300, 64, 10000.0)
    pos = np.arange(300)
    # pair 0 turns at frequency 1: cos(pos), sin(pos)
    np.testing.assert_array_equal(T[:, 0], np.cos(pos.astype(np.float64)).astype(np.float32))
    np.testing.assert_array_equal(T[:, 32], np.sin(pos.astype(np.float64)).astype(np.float32))
    # angle addition: rotation by a then b is rotation by a + b, every pair
    a, b = 37, 211
    ca, sa, cb, sb = T[a, :32], T[a, 32:], T[b, :32], T[b, 32:]
    np.testing.assert_allclose(ca * cb - sa * sb, T[a + b, :32], atol=3e-6)
    np.testing.assert_allclose(sa * cb + ca * sb, T[a + b, 32:], atol=3e-6)
    # last pair: frequency theta^(-62/64)
    f = 10000.0 ** (-62 / 64)
    np.testing.assert_allclose(T[299, 31], math.cos(299 * f), atol=1e-7)


def test_rope_gptj_rotates_interleaved_pairs():
    T = oracle.rope_table(40, 64)
    x = np.zeros(64, np.float32)
    x[0::2] = 1.0                                # every pair (x0, x1) = (1, 0)
    out = oracle.rope_gptj(x, T[36])
    np.testing.assert_array_equal(out[0::2], T[36, :32])
    np.testing.assert_array_equal(out[1::2], T[36, 32:])
    x2 = np.zeros(64, np.float32)
    x2[1::2] = 1.0                               # (0, 1) -> (-sin, cos)
    out2 = oracle.rope_gptj(x2, T[36])
    np.testing.assert_array_equal(out2[0::2], -T[36, 32:])
    np.testing.assert_array_equal(out2[1::2], T[36, :32])


@pytest.mark.parametrize("kind,ratio", [(oracle.MLA_KIND, 4), (oracle.MLA_KIND, 128),
                                        (oracle.IDX_KIND, 4)])
def test_stream_rope_anchor_is_slot_start(kind, ratio):
    """Every emitted entry's rope part equals bf16(rope(norm(pool), (p//r)*r)) and, for
    slots past the first, differs from rotating at p itself."""
    nope = 512 if kind == oracle.MLA_KIND else 64
    d = nope + 64
    coff = 2 if ratio == 4 else 1
    L = 3 * ratio
    g = np.random.default_rng(6 + ratio)
    ks = to_bf16_bits(g.normal(size=(L, 2 * coff * d)))
    ape = g.normal(size=(ratio, coff * d)).astype(np.float32) * 0.1
    w = g.uniform(0.5, 1.5, size=d).astype(np.float32)
    T = oracle.rope_table(L, 64)
    data, scale = oracle.compress_stream(kind, ratio, ks, ape, w, 1e-6, T, nope_dim=nope)
    assert data.shape[0] == 3
    for j in range(3):
        p = ratio * j + ratio - 1
        z = oracle.rmsnorm(oracle.compress_pool(ratio, ks, ape, p), w, 1e-6)
        good = z.copy()
        good[nope:] = oracle.rope_gptj(z[nope:], T[(p // ratio) * ratio])
        bad = z.copy()
        bad[nope:] = oracle.rope_gptj(z[nope:], T[p])
        if kind == oracle.MLA_KIND:
            got = data[j, nope:].view(np.uint16)
            assert np.array_equal(got, oracle.f32_to_bf16(good[nope:]))
            assert not np.array_equal(got, oracle.f32_to_bf16(bad[nope:]))
        else:
            dg, sg = oracle.quant_idx(good)
            db, _ = oracle.quant_idx(bad)
            assert np.array_equal(data[j], dg) and scale[j] == np.float32(sg)
            assert not np.array_equal(data[j], db)


def test_quant_mla_blocks_and_grid_values():
    g = np.random.default_rng(8)
    z = g.normal(size=576).astype(np.float32)
    z[64:128] *= 1e-3
    data, scales = oracle.quant_mla(z)
    for b in range(8):
        e = int(scales[b]) - 127
        blk = z[64 * b:64 * (b + 1)].astype(np.float64)
        assert np.abs(blk).max() <= 448 * 2.0 ** e
        assert np.abs(blk).max() > 448 * 2.0 ** (e - 1)
        deq = oracle.e4m3_to_f64(data[64 * b:64 * (b + 1)]) * 2.0 ** e
        # E4M3 keeps 4 significant bits: relative error <= 2^-4 for normals,
        # absolute <= 2^-10 * 2^e in the subnormal range
        assert np.all(np.abs(deq - blk) <= np.maximum(np.abs(blk) * 2.0 ** -4,
                                                      2.0 ** (e - 10)) + 0.0)
    rope = data[512:].view(np.uint16)
    assert np.array_equal(rope, to_bf16_bits(z[512:]))
    # values already on the scaled E4M3 grid come back exactly
    grid = oracle.e4m3_to_f64(g.integers(0, 0x7E, size=512).astype(np.uint8)) * 2.0 ** -5
    grid[0] = 448 * 2.0 ** -5
    zz = np.concatenate([grid, np.zeros(64)]).astype(np.float32)
    d2, s2 = oracle.quant_mla(zz)
    assert np.all(s2[:8] == 127 - 5)
    np.testing.assert_array_equal(oracle.e4m3_to_f64(d2[:512]) * 2.0 ** -5, grid)


def test_quant_idx_scale_rule():
    g = np.random.default_rng(9)
    z = g.normal(size=128).astype(np.float32)
    data, s = oracle.quant_idx(z)
    assert s == np.float32(np.float32(np.abs(z).max()) / np.float32(448.0))
    deq = oracle.e4m3_to_f64(data) * s
    assert np.all(np.abs(deq - z) <= np.abs(z) * 2.0 ** -4 + 2.0 ** -9 * s)
    d0, s0 = oracle.quant_idx(np.zeros(128, np.float32))
    assert s0 == 1.0 and np.all(d0 == 0)


def test_page_write_follows_block_table():
    g = np.random.default_rng(10)
    n = 150
    data = g.integers(0, 256, size=(n, 640), dtype=np.uint8)
    sc = g.integers(0, 256, size=(n, 8), dtype=np.uint8)
    bt = np.array([4, 0, 2], np.int32)
    cache = np.zeros(5 * oracle.page_bytes(oracle.MLA_KIND), np.uint8)
    oracle.page_write(oracle.MLA_KIND, cache, bt, data, sc)
    pages = cache.reshape(5, -1)
    for j in [0, 63, 64, 100, 149]:
        pg = pages[bt[j // 64]]
        r = j % 64
        assert np.array_equal(pg[r * 640:(r + 1) * 640], data[j])
        assert np.array_equal(pg[64 * 640 + r * 8: 64 * 640 + (r + 1) * 8], sc[j])


def test_rmsnorm_sum_order_is_the_fixed_one():
    """The RMSNorm mean square is summed in one fixed association (channel
    pairs, a 32-way butterfly per 64-channel group, groups in ascending order).
    The crafted stream makes that order matter: summed in ascending channel
    order the mean square rounds to the other fp32 neighbour, and the indexer
    entry's stored fp32 scale (amax / 448) would differ."""
    from _rms_case import ascending_sum, butterfly_sum, mean_square_pair, pooled_vector, token_rows
    d = 128
    y = pooled_vector(d)
    assert ascending_sum(y) != butterfly_sum(y)
    ms_asc, ms_tree = mean_square_pair(d)
    assert ms_asc != ms_tree
    ks = token_rows(d)
    ape = np.zeros((4, 2 * d), np.float32)
    # the compressor pools exactly the constructed vector
    assert np.array_equal(oracle.compress_pool(4, ks, ape, 3), y)

    def scale_for(ms):
        inv = np.float32(1) / np.sqrt(ms + np.float32(1e-6))
        return np.max(np.abs(y * inv)) / np.float32(448)

    cs = oracle.rope_table(4, 64)
    data, sc = oracle.compress_stream(1, 4, ks, ape, np.ones(d, np.float32), 1e-6, cs, nope_dim=64)
    stored = sc.view(np.float32).ravel()[0]
    assert scale_for(ms_tree) != scale_for(ms_asc)
    assert stored == scale_for(ms_tree)
