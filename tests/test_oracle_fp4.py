"""Pins of the oracle's FP4 (MXFP4) indexer cache: the E2M1 codec against
CUDA's own host-side codec (cuda_fp4.h, built here with g++), the shared
block exponent rule, the quantiser and packing, the page's byte count from
the pages, and the FP4 indexer logits against closed forms."""
import ctypes
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from deepseek_v4_compressed_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
CUDA_INC = "/usr/local/cuda/include"


@pytest.fixture(scope="module")
def cuda_fp4():
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_fp4.h")):
        pytest.skip("g++ or cuda_fp4.h not available")
    d = tempfile.mkdtemp()
    so = os.path.join(d, "fp4pin.so")
    subprocess.check_call([gxx, "-std=c++17", "-O1", "-fPIC", "-shared", "-I", CUDA_INC,
                           os.path.join(HERE, "pins", "fp4_codec.cpp"), "-o", so])
    lib = ctypes.CDLL(so)
    lib.pin_e2m1_decode.restype = ctypes.c_float
    lib.pin_e2m1_decode.argtypes = [ctypes.c_int]
    lib.pin_e2m1_encode.restype = ctypes.c_int
    lib.pin_e2m1_encode.argtypes = [ctypes.c_float]
    return lib


def test_e2m1_decode_every_code_matches_cuda(cuda_fp4):
    for c in range(16):
        want = cuda_fp4.pin_e2m1_decode(c)
        got = float(oracle.e2m1_to_f64(c)[()])
        assert got == want and math.copysign(1, got) == math.copysign(1, want), c
    # the value set: 0 and 0.5 .. 6, increasing with the code, largest 6
    mags = [float(oracle.e2m1_to_f64(c)[()]) for c in range(8)]
    assert mags == sorted(mags) and mags[0] == 0.0 and mags[1] == 0.5 and mags[-1] == 6.0


def test_e2m1_encode_matches_cuda_round_to_nearest_even(cuda_fp4):
    g = synth.rng(7)
    x = np.concatenate([
        synth.normal(g, 20000, 2.0),
        synth.uniform(g, 20000, -7.0, 7.0),
        # every midpoint between adjacent magnitudes, both signs, and just beside them
        np.array([m for a, b in zip([0, .5, 1, 1.5, 2, 3, 4], [.5, 1, 1.5, 2, 3, 4, 6])
                  for m in ((a + b) / 2, np.nextafter(np.float32((a + b) / 2), 0),
                            np.nextafter(np.float32((a + b) / 2), 10))], np.float32),
    ]).astype(np.float32)
    x = np.concatenate([x, -x, np.array([0.0, -0.0, 6.0, 6.5, 100.0, -100.0], np.float32)])
    got = oracle.f32_to_e2m1(x)
    want = np.array([cuda_fp4.pin_e2m1_encode(float(v)) for v in x], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_e2m1_round_trip_and_ties():
    for c in range(16):
        v = float(oracle.e2m1_to_f64(c)[()])
        if v == 0.0:
            continue                      # -0 encodes with its sign; 0 is code 0
        assert oracle.f32_to_e2m1(np.array([v], np.float32))[0] == c
    # ties go to the even code: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 2.5 -> 2, 5 -> 4
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    assert [float(oracle.e2m1_to_f64(c)[()]) for c in oracle.f32_to_e2m1(ties)] == [0, 1, 1, 2, 2, 4, 4]


def test_mxfp4_exponent_is_the_smallest_without_saturation():
    g = synth.rng(8)
    for a in np.abs(synth.normal(g, 2000, 1.0)) * np.exp(synth.uniform(g, 2000, -30, 30)):
        a = np.float32(a)
        e = oracle.mxfp4_exponent(a)
        assert float(a) <= 6.0 * 2.0 ** e
        assert float(a) > 6.0 * 2.0 ** (e - 1)
    assert oracle.mxfp4_exponent(6.0) == 0 and oracle.mxfp4_exponent(3.0) == -1
    assert oracle.mxfp4_exponent(0.0) == 0


def test_quantiser_packing_and_exact_grid_values():
    g = synth.rng(9)
    # values already on the grid (E2M1 value times a per-block power of two)
    # quantise exactly; element 2i sits in the low nibble of byte i
    codes = g.integers(0, 16, size=(5, 128)).astype(np.uint8)
    ex = g.integers(-20, 20, size=(5, 4))
    vals = oracle.e2m1_to_f64(codes) * np.repeat(2.0 ** ex, 32, axis=1)
    for r in range(5):
        for b in range(4):          # make each block's amax reach 6 * 2^e exactly
            vals[r, 32 * b] = 6.0 * 2.0 ** ex[r, b]
            codes[r, 32 * b] = 7
    data, sc = oracle.quant_idx_fp4_rows(vals.astype(np.float32))
    assert data.shape == (5, 64) and sc.shape == (5, 4)
    assert np.array_equal(sc.astype(np.int64) - 127, ex)
    unpacked = np.stack([data & 15, data >> 4], axis=-1).reshape(5, 128)
    zero = vals == 0.0
    assert np.array_equal(unpacked[~zero], codes[~zero])
    assert np.all((unpacked[zero] & 7) == 0)


def test_fp4_entry_and_page_bytes_match_the_pages():
    from test_oracle_schedule_bytes import golden_lines
    rows = [l for l in golden_lines("kv_bytes.txt") if l[0] == "fp4_block"]
    assert rows, "golden row missing"
    for _, name, entries, nbytes in rows:
        assert name == "c4_indexer"
        assert oracle.idx_fp4_entry_bytes(128) == int(nbytes)
        assert oracle.page_bytes(oracle.IDX_FP4_KIND) == int(entries) * int(nbytes)


def test_fp4_logits_equal_exact_logits_for_grid_keys():
    """Keys on the FP4 grid quantise exactly, so the FP4 logits equal the
    logits of the unquantised keys, computed here by a plain matrix product."""
    g = synth.rng(10)
    n, H = 150, 6
    codes = g.integers(0, 16, size=(n, 128)).astype(np.uint8)
    ex = g.integers(-6, 3, size=(n, 4))
    keys = oracle.e2m1_to_f64(codes) * np.repeat(2.0 ** ex, 32, axis=1)
    for r in range(n):
        for b in range(4):
            keys[r, 32 * b] = 6.0 * 2.0 ** ex[r, b]
    data, sc = oracle.quant_idx_fp4_rows(keys.astype(np.float32))
    bt = np.array([2, 0, 1], np.int32)
    cache = np.zeros(3 * oracle.page_bytes(oracle.IDX_FP4_KIND), np.uint8)
    oracle.page_write(oracle.IDX_FP4_KIND, cache, bt, data, sc, nope_dim=64)
    q = oracle.f32_to_e4m3(synth.normal(g, (H, 128)))
    w = synth.uniform(g, H)
    got = oracle.indexer_logits_fp4(q, w, cache, bt, n)
    qd = oracle.e4m3_to_f64(q)
    want = (np.maximum(qd @ keys.T, 0.0) * w[:, None].astype(np.float64)).sum(0)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # one head of weight 1 with every dot positive: the logit is the dot itself
    k1 = np.abs(keys[:10])
    d1, s1 = oracle.quant_idx_fp4_rows(k1.astype(np.float32))
    c1 = np.zeros(oracle.page_bytes(oracle.IDX_FP4_KIND), np.uint8)
    oracle.page_write(oracle.IDX_FP4_KIND, c1, np.array([0], np.int32), d1, s1, nope_dim=64)
    qpos = oracle.f32_to_e4m3(np.abs(synth.normal(g, (1, 128))) + 0.1)
    got1 = oracle.indexer_logits_fp4(qpos, np.ones(1, np.float32), c1, np.array([0], np.int32), 10)
    np.testing.assert_allclose(got1, oracle.e4m3_to_f64(qpos)[0] @ k1.T, rtol=1e-12)


def test_fp4_compress_stream_matches_the_fp8_path_before_quantisation():
    """The FP4 stream pools, normalises and rotates exactly as the FP8 one
    (same pre-quantisation vector); only the quantiser differs."""
    g = synth.rng(11)
    L = 64
    ks = oracle.f32_to_bf16(synth.normal(g, (L, 4 * 128)))
    ape = synth.normal(g, (4, 256), 0.1)
    w = synth.uniform(g, 128, 0.5, 1.5)
    cs = oracle.rope_table(L, 64)
    d4, s4 = oracle.compress_stream(oracle.IDX_FP4_KIND, 4, ks, ape, w, 1e-6, cs, nope_dim=64)
    assert d4.shape == (16, 64) and s4.shape == (16, 4)
    for j in range(16):
        p = 4 * j + 3
        z = oracle.rmsnorm(oracle.compress_pool(4, ks, ape, p), w, 1e-6)
        z[64:] = oracle.rope_gptj(z[64:], cs[(p // 4) * 4])
        dq, sq = oracle.quant_idx_fp4_rows(z[None])
        assert np.array_equal(d4[j], dq[0]) and np.array_equal(s4[j], sq[0])
