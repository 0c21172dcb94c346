"""Pins of the oracle's prefill helpers: dequantise-and-gather of cache rows
into a dense bf16 buffer and the per-token combined index list over it
(_forward_prefill of the vLLM DeepseekV4Attention walkthrough)."""
import math

import numpy as np

import oracle
from deepseek_v4_compressed_gb300 import synth

SCALE = 1.0 / math.sqrt(576)


def test_gather_returns_grid_values_exactly():
    """Rows already on the FP8 grid (per 64-dim block) dequantise to exactly
    the values they were made from; SWA rows come back unchanged."""
    g = synth.rng(81)
    n = 70
    codes = g.integers(0, 126, size=(n, 512)).astype(np.uint8)
    ex = g.integers(-10, 4, size=(n, 8))
    vals = oracle.e4m3_to_f64(codes) * np.repeat(2.0 ** ex, 64, axis=1)
    for r in range(n):
        for b in range(8):   # each block's largest magnitude 448 * 2^e, so the block exponent is e
            vals[r, 64 * b] = 448.0 * 2.0 ** ex[r, b]
    rope = oracle.f32_to_bf16(synth.normal(g, (n, 64)))
    z = np.concatenate([vals, oracle.bf16_to_f32(rope)], axis=1).astype(np.float32)
    data, sc = oracle.quant_mla_rows(z)
    bt = np.array([3, 1, 0, 2], np.int32)
    cache = np.zeros(4 * oracle.page_bytes(0), np.uint8)
    oracle.page_write(0, cache, bt, data, sc)
    got = oracle.dequant_gather(0, cache, bt, 5, 60)
    assert np.array_equal(oracle.bf16_to_f32(got[:, :512]), vals[5:65].astype(np.float32))
    assert np.array_equal(got[:, 512:], rope[5:65])
    swa = oracle.f32_to_bf16(synth.normal(g, (4 * 64, 576)))
    rows = oracle.dequant_gather(1, swa, bt, 100, 50)
    for i in range(50):
        t = 100 + i
        assert np.array_equal(rows[i], swa[bt[t // 64] * 64 + t % 64])


def test_combine_indices_hand_example():
    # buffer: N = 20 compressed slots, then tokens 4..9 of a 10-token sequence
    # (gather_len 6); window 3; the token at position 8 sees tokens 6, 7, 8
    out = oracle.combine_topk_swa_indices(np.array([3, -1, 11], np.int32), 3, 8, 10, 6, 3, 20)
    assert list(out) == [3, 11, 22, 23, 24]
    # the first token: window reaches before the sequence start -> clipped at 0
    out = oracle.combine_topk_swa_indices(np.array([0], np.int32), 1, 1, 4, 4, 3, 1)
    assert list(out) == [0, 1, 2]
    # a window token outside the gathered range is an error
    assert oracle.combine_topk_swa_indices(np.array([0], np.int32), 1, 8, 10, 2, 3, 20) is None


def test_gather_combine_dense_attention_equals_sparse_mla():
    """The pages' prefill flow in the oracle -- gather the compressed slots and
    the SWA tokens into one buffer, combine each query token's top-k with its
    window, attend densely over the listed rows -- equals the decode-form
    sparse attention of each token."""
    g = synth.rng(82)
    L, n_q, H, k = 900, 5, 4, 16
    n_c = L // 4
    bt = synth.page_tables(g, 1, (n_c + 63) // 64, extra_pages=1)[0]
    comp = np.zeros((bt.size + 1) * oracle.page_bytes(0), np.uint8)
    oracle.page_write(0, comp, bt, *oracle.quant_mla_rows(synth.normal(g, (n_c, 576), SCALE)))
    sbt = synth.page_tables(g, 1, (L + 63) // 64, extra_pages=1)[0]
    swa = oracle.f32_to_bf16(synth.normal(g, ((sbt.size + 1) * 64, 576), SCALE))
    gather_len = 128 + n_q - 1
    kv = np.concatenate([oracle.dequant_gather(0, comp, bt, 0, n_c),
                         oracle.dequant_gather(1, swa, sbt, L - gather_len, gather_len)])
    kvd = oracle.bf16_to_f32(kv).astype(np.float64)
    for j in range(n_q):
        pos = L - n_q + j
        q = oracle.f32_to_bf16(synth.normal(g, (H, 576), SCALE))
        sel = synth.sorted_sample(g, (pos + 1) // 4, k)
        ids = oracle.combine_topk_swa_indices(sel, len(sel), pos, L, gather_len, 128, n_c)
        dense, dense_lse = oracle.dense_attention(oracle.bf16_to_f32(q).astype(np.float64), kvd[ids], 512, SCALE)
        ref, ref_lse, _ = oracle.sparse_mla(q, comp, bt, sel, len(sel), swa, sbt, pos, SCALE)
        np.testing.assert_allclose(dense, ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dense_lse, ref_lse, rtol=1e-12)
