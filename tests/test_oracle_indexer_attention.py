"""Pins of the oracle's lightning indexer, top-k and sparse MLA.

Indexer: brute force on tiny inputs and the one-head special case that reduces
to a plain matrix-vector product.  Top-k: numpy's stable sort.  Attention:
closed forms (one key, equal scores, two keys) and the sparse path against
dense attention over keys this test gathers itself through the page tables.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_gb300 import synth


def to_bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def fp8_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def make_idx_cache(g, n_c, pages_extra=3):
    n_pages = (n_c + 63) // 64
    bt = synth.page_tables(g, 1, n_pages, extra_pages=pages_extra)[0]
    rows = synth.normal(g, (n_c, 128), 1.0 / math.sqrt(128))
    data, scale = oracle.quant_idx_rows(rows)
    cache = np.zeros((n_pages + pages_extra) * oracle.page_bytes(oracle.IDX_KIND), np.uint8)
    oracle.page_write(oracle.IDX_KIND, cache, bt, data, scale, nope_dim=64)
    return cache, bt, data, scale


def test_indexer_brute_force_tiny():
    g = synth.rng(11)
    n_c, H = 70, 4
    cache, bt, data, scale = make_idx_cache(g, n_c)
    q = oracle.f32_to_e4m3(synth.normal(g, (H, 128)))
    w = synth.uniform(g, H, -0.5, 1.0)
    got = oracle.indexer_logits(q, w, cache, bt, n_c)
    qd, kd = fp8_decode(q), fp8_decode(data)
    for s in range(n_c):
        dots = qd @ kd[s]
        expect = float(scale[s]) * sum(float(w[j]) * max(0.0, dots[j]) for j in range(H))
        assert got[s] == pytest.approx(expect, rel=1e-12, abs=1e-15)


def test_indexer_single_head_is_matvec():
    g = synth.rng(12)
    n_c = 130
    cache, bt, data, scale = make_idx_cache(g, n_c)
    kd = fp8_decode(data) * scale[:, None].astype(np.float64)
    q = oracle.f32_to_e4m3(np.abs(synth.normal(g, (1, 128))))
    # keep only slots with a positive dot so ReLU is the identity
    mv = kd @ fp8_decode(q)[0]
    got = oracle.indexer_logits(q, np.ones(1, np.float32), cache, bt, n_c)
    pos = mv > 0
    np.testing.assert_allclose(got[pos], mv[pos], rtol=1e-12)
    assert np.all(got[~pos] == 0.0)


def test_indexer_page_permutation_invariance():
    g = synth.rng(13)
    n_c = 200
    cache, bt, data, scale = make_idx_cache(g, n_c, pages_extra=0)
    q = oracle.f32_to_e4m3(synth.normal(g, (8, 128)))
    w = synth.uniform(g, 8)
    a = oracle.indexer_logits(q, w, cache, bt, n_c)
    bt2 = np.array([3, 1, 0, 2], np.int32)
    cache2 = np.zeros_like(cache)
    oracle.page_write(oracle.IDX_KIND, cache2, bt2, data, scale, nope_dim=64)
    b = oracle.indexer_logits(q, w, cache2, bt2, n_c)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("n,k", [(1000, 32), (8192, 512), (50, 64), (64, 64), (0, 8)])
def test_topk_against_stable_sort(n, k):
    g = np.random.default_rng(n + k)
    lg = np.round(g.normal(size=n), 2)     # many exact ties
    idx, ln = oracle.topk(lg, k)
    assert ln == min(n, k)
    order = np.lexsort((np.arange(n), -lg))[:ln]  # score desc, then index asc
    assert np.array_equal(idx[:ln], np.sort(order))
    assert np.all(idx[ln:] == -1)
    assert np.all(np.diff(idx[:ln]) > 0)


def test_dense_attention_closed_forms():
    g = np.random.default_rng(14)
    key = g.normal(size=(1, 576))
    q = g.normal(size=(3, 576))
    out, lse = oracle.dense_attention(q, key, 512, 0.1)
    np.testing.assert_allclose(out, np.repeat(key[:, :512], 3, 0), rtol=0, atol=0)
    np.testing.assert_allclose(lse, 0.1 * (q @ key[0]), rtol=1e-13)
    keys = g.normal(size=(37, 576))
    out, lse = oracle.dense_attention(np.zeros((2, 576)), keys, 512, 0.3)
    np.testing.assert_allclose(out[0], keys[:, :512].mean(0), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse, math.log(37), rtol=1e-14)
    # two keys, scores s1 and s2 set through q
    k2 = np.zeros((2, 576))
    k2[0, 0], k2[1, 1] = 1.0, 1.0
    k2[0, 100], k2[1, 100] = 5.0, -3.0
    qq = np.zeros((1, 576))
    qq[0, 0], qq[0, 1] = 2.0, -1.0
    out, lse = oracle.dense_attention(qq, k2, 512, 1.0)
    p0 = math.exp(2.0) / (math.exp(2.0) + math.exp(-1.0))
    assert out[0, 100] == pytest.approx(p0 * 5.0 + (1 - p0) * -3.0, rel=1e-14)
    assert lse[0] == pytest.approx(math.log(math.exp(2.0) + math.exp(-1.0)), rel=1e-14)


def build_mla_inputs(g, n_c, p, n_pages_swa_extra=2):
    """A compressed cache with n_c random entries and an SWA cache covering 0..p."""
    rows = synth.normal(g, (n_c, 576), 1.0 / math.sqrt(576))
    data, sc = oracle.quant_mla_rows(rows)
    cpages = (n_c + 63) // 64
    cbt = synth.page_tables(g, 1, cpages, extra_pages=1)[0]
    comp = np.zeros((cpages + 1) * oracle.page_bytes(oracle.MLA_KIND), np.uint8)
    oracle.page_write(oracle.MLA_KIND, comp, cbt, data, sc)
    spages = p // 64 + 1
    sbt = synth.page_tables(g, 1, spages, extra_pages=n_pages_swa_extra)[0]
    swa = to_bf16_bits(synth.normal(g, ((spages + n_pages_swa_extra) * 64, 576),
                                    1.0 / math.sqrt(576)))
    return comp, cbt, data, sc, swa, sbt


def own_gather(comp_data, comp_sc, idx, swa, sbt, p, window=128):
    """Independent gather: decode selected entries from the entry arrays (not the pages),
    and SWA tokens through the page table."""
    keys = []
    for s in idx:
        nope = fp8_decode(comp_data[s, :512]) * np.repeat(2.0 ** (comp_sc[s].astype(np.int64)
                                                                  - 127), 64)
        rope = torch.from_numpy(comp_data[s, 512:].copy().view(np.int16)).view(torch.bfloat16) \
            .double().numpy()
        keys.append(np.concatenate([nope, rope]))
    for t in range(max(0, p - window + 1), p + 1):
        row = swa[sbt[t // 64] * 64 + t % 64]
        keys.append(torch.from_numpy(row.view(np.int16).copy()).view(torch.bfloat16)
                    .double().numpy())
    return np.array(keys)


@pytest.mark.parametrize("n_c,k,p", [(128, 128, 511), (100, 32, 400), (40, 40, 90),
                                     (0, 0, 60)])
def test_sparse_mla_equals_dense_over_gathered_keys(n_c, k, p):
    g = synth.rng(15 + n_c)
    comp, cbt, data, sc, swa, sbt = build_mla_inputs(g, max(n_c, 1), p)
    idx = synth.sorted_sample(g, n_c, k) if k else np.zeros(0, np.int32)
    q = to_bf16_bits(synth.normal(g, (8, 576), 1.0))
    scale = 1.0 / math.sqrt(576)
    out, lse, n = oracle.sparse_mla(q, comp if k else None, cbt if k else None, idx, k, swa, sbt,
                                    p, scale)
    keys = own_gather(data, sc, idx, swa, sbt, p)
    assert n == len(keys) == k + min(p + 1, 128)
    qd = oracle.bf16_to_f32(q).astype(np.float64)
    s = scale * qd @ keys.T
    m = s.max(1, keepdims=True)
    e = np.exp(s - m)
    ref = (e @ keys[:, :512]) / e.sum(1, keepdims=True)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(lse, m[:, 0] + np.log(e.sum(1)), rtol=1e-12)


def test_sparse_mla_one_key_returns_its_latent():
    g = synth.rng(16)
    comp, cbt, data, sc, swa, sbt = build_mla_inputs(g, 64, 0)
    q = to_bf16_bits(synth.normal(g, (4, 576)))
    # p = 0: exactly one SWA token and no compressed slot
    out, _, n = oracle.sparse_mla(q, None, None, None, 0, swa, sbt, 0, 0.05)
    assert n == 1
    row = swa[sbt[0] * 64]
    v = oracle.bf16_to_f32(row[:512]).astype(np.float64)
    assert np.array_equal(out, np.repeat(v[None], 4, 0))
