"""Pins of the oracle's V4-native geometry ("From MLA to CSA + HCA" 5.5 and
6.4; the V4 internals talk write-up, section 6): the 584-byte cache row read
back by an independent decoder (torch's float8 / bfloat16 views), attention
with K = V over all 512 dims against torch's softmax in double, and the
inverse RoPE + FP8 quantisation against the rotation written as a closed form
and against the identity R(-i) R(j) = R(j - i)."""
import math

import numpy as np
import torch

import oracle
from deepseek_v4_compressed_gb300 import synth

V4_DATA = 576
V4_PAGE = 64 * (V4_DATA + 8)


def t_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)


def t_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64)


def random_v4_pages(g, n_pages):
    """Random bytes in the 584-byte row format: finite E4M3 codes, scale bytes
    near 127, a random pad byte, bf16 RoPE values of unit scale."""
    cache = np.zeros(n_pages * V4_PAGE, np.uint8)
    for pg in range(n_pages):
        base = pg * V4_PAGE
        codes = g.integers(0, 256, size=(64, 448)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x10            # no NaN codes
        rope = synth.normal(g, (64, 64), 0.5).astype(np.float32)
        rope_bits = torch.from_numpy(rope).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint8)
        data = np.concatenate([codes, rope_bits.reshape(64, 128)], axis=1)
        cache[base:base + 64 * V4_DATA] = data.reshape(-1)
        sc = g.integers(118, 136, size=(64, 8)).astype(np.uint8)
        sc[:, 7] = g.integers(0, 256, size=64)          # the pad byte
        cache[base + 64 * V4_DATA:base + V4_PAGE] = sc.reshape(-1)
    return cache


def decode_row(cache, bt, slot):
    """Independent reading of one 584-byte row: [0, 448) E4M3 codes scaled by
    2^(scale byte - 127) per 64 dims, [448, 576) 64 little-endian bf16."""
    base = int(bt[slot // 64]) * V4_PAGE
    r = slot % 64
    data = cache[base + r * V4_DATA:base + (r + 1) * V4_DATA]
    sc = cache[base + 64 * V4_DATA + r * 8:base + 64 * V4_DATA + r * 8 + 7].astype(np.float64)
    nope = t_e4m3(data[:448]) * torch.from_numpy(np.repeat(2.0 ** (sc - 127), 64))
    rope = t_bf16(data[448:].view(np.uint16))
    return torch.cat([nope, rope])


def torch_attention(q_bits, keys, scale):
    q = t_bf16(q_bits)
    k = torch.stack(keys)
    s = scale * (q @ k.T)
    return (torch.softmax(s, -1) @ k).numpy(), torch.logsumexp(s, -1).numpy()


def test_v4_attention_matches_torch():
    g = synth.rng(41)
    comp = random_v4_pages(g, 4)
    swa = random_v4_pages(g, 5)
    comp_bt = np.array([2, 0, 3, 1], np.int32)
    swa_bt = np.array([-1, -1, 4, 1, 3], np.int32)      # tokens 128 .. 319 mapped
    p, window, H = 300, 128, 8
    idx = g.choice(4 * 64, size=100, replace=False).astype(np.int32)
    q = synth.normal(g, (H, 512), 0.05)
    q_bits = torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    scale = 1.0 / math.sqrt(512)
    out, lse = oracle.sparse_mla_v4(q_bits, comp, comp_bt, idx, len(idx), swa, swa_bt, p, scale, window)
    keys = [decode_row(comp, comp_bt, int(s)) for s in idx]
    keys += [decode_row(swa, swa_bt, t) for t in range(p - window + 1, p + 1)]
    ref, ref_lse = torch_attention(q_bits, keys, scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_v4_value_is_the_whole_key():
    """One key (query at position 0, no compressed slots): the output is the
    key row itself, RoPE dims 448..511 included (K = V)."""
    g = synth.rng(42)
    swa = random_v4_pages(g, 1)
    bt = np.array([0], np.int32)
    q_bits = np.full((2, 512), 0x3C00, np.uint16)       # bf16 0.0078125
    out, lse = oracle.sparse_mla_v4(q_bits, None, None, None, 0, swa, bt, 0, 0.25)
    k = decode_row(swa, bt, 0).numpy()
    assert np.array_equal(out[0], k) and np.array_equal(out[1], k)
    np.testing.assert_allclose(lse, 0.25 * 0.0078125 * k.sum(), rtol=1e-13)


def test_v4_window_starts_at_zero_and_pad_is_ignored():
    g = synth.rng(43)
    swa = random_v4_pages(g, 1)
    bt = np.array([0], np.int32)
    q_bits = torch.from_numpy(synth.normal(g, (3, 512), 0.1).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    out, _ = oracle.sparse_mla_v4(q_bits, None, None, None, 0, swa, bt, 5, 0.3)
    ref, _ = torch_attention(q_bits, [decode_row(swa, bt, t) for t in range(6)], 0.3)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
    swa2 = swa.copy()
    swa2[64 * V4_DATA + np.arange(64) * 8 + 7] ^= 0xFF
    out2, _ = oracle.sparse_mla_v4(q_bits, None, None, None, 0, swa2, bt, 5, 0.3)
    assert np.array_equal(out, out2)
    # one more in a scale byte doubles that 64-dim block of that row only
    swa3 = swa.copy()
    swa3[64 * V4_DATA + 0 * 8 + 2] += 1
    k0, k3 = decode_row(swa, bt, 0).numpy(), decode_row(swa3, bt, 0).numpy()
    assert np.array_equal(k3[128:192], 2 * k0[128:192])
    o1, _ = oracle.sparse_mla_v4(q_bits[:1], None, None, None, 0, swa3, bt, 0, 0.3)
    assert np.array_equal(o1[0], k3)


def rotate(x, ang):
    """GPT-J rotation of the interleaved pairs of x by the angles ang (double)."""
    y = x.astype(np.float64).copy()
    c, s = np.cos(ang), np.sin(ang)
    y[0::2] = x[0::2] * c - x[1::2] * s
    y[1::2] = x[0::2] * s + x[1::2] * c
    return y


def angles(pos, rope_dim=64, theta=10000.0):
    return pos * theta ** (-2.0 * np.arange(rope_dim // 2) / rope_dim)


def cos_sin_table(max_pos, rope_dim=64):
    t = np.empty((max_pos, rope_dim), np.float32)
    for pos in range(max_pos):
        a = angles(pos, rope_dim)
        t[pos, :rope_dim // 2] = np.cos(a)
        t[pos, rope_dim // 2:] = np.sin(a)
    return t


def dequant(codes, scales):
    """E4M3 codes [H][512] with fp32 scales [H][4] (128-dim blocks) -> double."""
    return t_e4m3(codes).numpy() * np.repeat(scales.astype(np.float64), 128, axis=1)


def quant_bound(x, scales):
    """Largest E4M3 rounding error of x under the block scales: half a step of
    3 mantissa bits for normals, half the subnormal step 2^-9 below them."""
    s = np.repeat(scales.astype(np.float64), 128, axis=1)
    return np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)


def to_bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_inv_rope_at_position_zero_is_block_quant():
    g = synth.rng(44)
    o_bits = to_bf16_bits(synth.normal(g, (4, 512), 0.3))
    codes, sc = oracle.inv_rope_fp8_quant(o_bits, 0, cos_sin_table(4))
    x = oracle.bf16_to_f32(o_bits)
    for h in range(4):
        for blk in range(4):
            c, s = oracle.quant_idx(x[h, blk * 128:(blk + 1) * 128])
            assert np.array_equal(codes[h, blk * 128:(blk + 1) * 128], c)
            assert sc[h, blk] == np.float32(s)


def test_inv_rope_closed_form():
    g = synth.rng(45)
    H, pos = 6, 3001
    o = synth.normal(g, (H, 512), 0.3)
    o_bits = to_bf16_bits(o)
    x = oracle.bf16_to_f32(o_bits).astype(np.float64)
    codes, sc = oracle.inv_rope_fp8_quant(o_bits, pos, cos_sin_table(pos + 1))
    want = x.copy()
    for h in range(H):
        want[h, 448:] = rotate(x[h, 448:], -angles(pos))
    got = dequant(codes, sc)
    assert np.all(np.abs(got - want) <= quant_bound(want, sc) + 1e-6 * np.abs(want))
    # the unrotated (or wrongly rotated) values miss the bound on most RoPE dims
    wrong = x.copy()
    for h in range(H):
        wrong[h, 448:] = rotate(x[h, 448:], angles(pos))
    for bad in (x, wrong):
        miss = np.abs(got - bad)[:, 448:] > quant_bound(bad, sc)[:, 448:]
        assert miss.mean() > 0.5


def test_inv_rope_undoes_the_key_rotation():
    """R(-i) R(j) k = R(j - i) k: a value rotated at key position j and
    inverse-rotated at query position i carries only the offset j - i."""
    g = synth.rng(46)
    i, j = 777, 700
    table = cos_sin_table(i + 1)
    k = synth.normal(g, (1, 512), 0.3).astype(np.float32)
    o = k.copy()
    o[0, 448:] = oracle.rope_gptj(k[0, 448:], table[j])
    o_bits = to_bf16_bits(o)
    codes, sc = oracle.inv_rope_fp8_quant(o_bits, i, table)
    want = k[0].astype(np.float64).copy()
    want[448:] = rotate(k[0, 448:].astype(np.float64), angles(j - i))
    got = dequant(codes, sc)[0]
    # bf16 input rounding (2^-9 relative) on top of the FP8 bound
    tol = quant_bound(want[None], sc)[0] + 2.0 ** -8 * np.max(np.abs(k[0, 448:])) + 1e-6
    assert np.all(np.abs(got - want) <= tol)


def test_inv_rope_scale_per_128_dim_block():
    g = synth.rng(47)
    o = synth.normal(g, (3, 512), 0.2)
    o[0, 128:256] *= 50.0            # one loud block
    o[1, 256:384] = 0.0              # one silent block
    o_bits = to_bf16_bits(o)
    codes, sc = oracle.inv_rope_fp8_quant(o_bits, 9, cos_sin_table(10))
    dq = t_e4m3(codes).numpy()
    for h in range(3):
        for blk in range(4):
            c = dq[h, blk * 128:(blk + 1) * 128]
            if h == 1 and blk == 2:
                assert sc[h, blk] == 1.0 and np.all(c == 0)
            else:
                assert np.max(np.abs(c)) == 448.0
    assert sc[0, 1] > 20 * sc[0, 0]


def test_v4_rows_written_by_the_quantiser_read_back():
    """quant_mla_rows + page_write at nope 448 produce the 584-byte layout:
    the independent decoder gets the rows back within E4M3 / bf16 rounding,
    each block's scale byte is the smallest 2^e with amax <= 448 * 2^e, and
    the pad byte is zero."""
    g = synth.rng(48)
    z = synth.normal(g, (70, 512), 0.2).astype(np.float32)
    z[3, :64] *= 1000.0
    z[5, 64:128] = 0.0
    data, sc = oracle.quant_mla_rows(z, nope_dim=448)
    assert data.shape == (70, 576) and sc.shape == (70, 8)
    cache = np.zeros(2 * V4_PAGE, np.uint8)
    bt = np.array([1, 0], np.int32)
    oracle.page_write(oracle.MLA_KIND, cache, bt, data, sc, nope_dim=448)
    assert oracle.page_bytes(oracle.MLA_KIND, nope_dim=448) == V4_PAGE
    for s in range(70):
        k = decode_row(cache, bt, s).numpy()
        blk = np.repeat(2.0 ** (sc[s, :7].astype(np.float64) - 127), 64)
        assert np.all(np.abs(k[:448] - z[s, :448]) <= np.maximum(np.abs(z[s, :448]) * 2.0 ** -4,
                                                                 blk * 2.0 ** -10) * (1 + 1e-9))
        rope = torch.from_numpy(z[s, 448:]).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(k[448:], rope)
        base = int(bt[s // 64]) * V4_PAGE + 64 * V4_DATA + (s % 64) * 8
        assert cache[base + 7] == 0
        for b in range(7):
            a = float(np.abs(z[s, 64 * b:64 * b + 64]).max())
            e = int(sc[s, b]) - 127
            if a == 0.0:
                assert e == 0
            else:
                assert a <= 448.0 * 2.0 ** e and a > 448.0 * 2.0 ** (e - 1)


def test_v4_compressor_entry_is_the_normalised_rotated_mean():
    """The compressor at nope 448 (d = 512, ratio 128, equal scores, constant
    kv rows): the entry is RMSNorm(row) with RoPE at the slot's first
    position on dims 448..511, in the 584-byte row."""
    g = synth.rng(49)
    d, ratio = 512, 128
    row = synth.normal(g, (d,), 0.7).astype(np.float32)
    row_bits = to_bf16_bits(row)
    ks = np.zeros((2 * ratio, 2 * d), np.uint16)
    ks[:, :d] = row_bits
    ks[:, d:] = to_bf16_bits(np.full(d, 0.25, np.float32))
    ape = np.zeros((ratio, d), np.float32)
    w = synth.uniform(g, (d,), 0.5, 1.5).astype(np.float32)
    table = cos_sin_table(2 * ratio)
    data, sc = oracle.compress_stream(oracle.MLA_KIND, ratio, ks, ape, w, 1e-6, table, 448)
    assert data.shape == (2, 576)
    y = oracle.bf16_to_f32(row_bits).astype(np.float64)
    z = y / np.sqrt(np.mean(y * y) + 1e-6) * w
    for j in range(2):
        want = z.copy()
        want[448:] = rotate(z[448:], angles(j * ratio))
        cache = np.zeros(V4_PAGE, np.uint8)
        oracle.page_write(oracle.MLA_KIND, cache, np.array([0], np.int32), data[j:j + 1], sc[j:j + 1],
                          nope_dim=448)
        k = decode_row(cache, np.array([0], np.int32), 0).numpy()
        blk = np.repeat(2.0 ** (sc[j, :7].astype(np.float64) - 127), 64)
        assert np.all(np.abs(k[:448] - want[:448]) <= np.maximum(np.abs(want[:448]) * 2.0 ** -4 + 1e-5,
                                                                 blk * 2.0 ** -10))
        np.testing.assert_allclose(k[448:], want[448:], rtol=2.0 ** -8, atol=1e-5)
