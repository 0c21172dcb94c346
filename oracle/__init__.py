"""CPU oracle for DeepSeek-V4 compressed sparse attention at decode.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The product path (the
CUDA library ``libdsv4.so`` and its binding) never imports, links or calls it,
and the two share no code.

This module is argument marshalling around the plain C reference in
``dsv4_oracle.c`` (numpy arrays in, numpy arrays out).  Each C function cites
the page and section it follows.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = ctypes.CDLL(build_oracle())

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)

_lib.or_bf16_to_f32.restype = ctypes.c_float
_lib.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
_lib.or_f32_to_bf16.restype = ctypes.c_uint16
_lib.or_f32_to_bf16.argtypes = [ctypes.c_float]
_lib.or_e4m3_to_f64.restype = ctypes.c_double
_lib.or_e4m3_to_f64.argtypes = [ctypes.c_uint8]
_lib.or_f32_to_e4m3.restype = ctypes.c_uint8
_lib.or_f32_to_e4m3.argtypes = [ctypes.c_float]
_lib.or_ue8m0_exponent.restype = ctypes.c_int
_lib.or_ue8m0_exponent.argtypes = [ctypes.c_float]
_lib.or_expf.restype = ctypes.c_float
_lib.or_expf.argtypes = [ctypes.c_float]
_lib.or_f32_to_e4m3_n.restype = None
_lib.or_f32_to_e4m3_n.argtypes = [ctypes.c_longlong, _f32p, _u8p]
_lib.or_f32_to_bf16_n.restype = None
_lib.or_f32_to_bf16_n.argtypes = [ctypes.c_longlong, _f32p, _u16p]
_lib.or_quant_mla_rows.restype = None
_lib.or_quant_mla_rows.argtypes = [ctypes.c_longlong, _f32p, ctypes.c_int, ctypes.c_int, _u8p,
                                   _u8p]
_lib.or_quant_idx_rows.restype = None
_lib.or_quant_idx_rows.argtypes = [ctypes.c_longlong, _f32p, ctypes.c_int, _u8p, _f32p]
_lib.or_layer_type.restype = ctypes.c_int
_lib.or_layer_type.argtypes = [ctypes.c_int]
_lib.or_index_schedule.restype = ctypes.c_int
_lib.or_index_schedule.argtypes = [_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_char_p, _u8p]
_lib.or_mla_entry_bytes.restype = ctypes.c_int
_lib.or_mla_entry_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
_lib.or_idx_entry_bytes.restype = ctypes.c_int
_lib.or_idx_entry_bytes.argtypes = [ctypes.c_int]
_lib.or_rope_table.restype = None
_lib.or_rope_table.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, _f32p]
_lib.or_compress_pool.restype = ctypes.c_int
_lib.or_compress_pool.argtypes = [ctypes.c_int, ctypes.c_int, _u16p, ctypes.c_longlong, _f32p,
                                  ctypes.c_int, _f32p]
_lib.or_rmsnorm.restype = None
_lib.or_rmsnorm.argtypes = [_f32p, ctypes.c_int, _f32p, ctypes.c_float, _f32p]
_lib.or_rope_gptj.restype = None
_lib.or_rope_gptj.argtypes = [_f32p, ctypes.c_int, _f32p]
_lib.or_quant_mla.restype = None
_lib.or_quant_mla.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, _u8p, _u8p]
_lib.or_quant_idx.restype = None
_lib.or_quant_idx.argtypes = [_f32p, ctypes.c_int, _u8p, _f32p]
_lib.or_compress_stream.restype = ctypes.c_int
_lib.or_compress_stream.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p,
                                    ctypes.c_longlong, _f32p, _f32p, ctypes.c_float, _f32p,
                                    ctypes.c_int, ctypes.c_int, _u8p, _u8p]
_lib.or_page_write.restype = None
_lib.or_page_write.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p,
                               ctypes.c_int, _u8p, _u8p, _u8p]
_lib.or_indexer_logits.restype = None
_lib.or_indexer_logits.argtypes = [_u8p, _f32p, ctypes.c_int, ctypes.c_int, _u8p, _i32p,
                                   ctypes.c_int, ctypes.c_int, _f64p]
_lib.or_topk.restype = ctypes.c_int
_lib.or_topk.argtypes = [_f64p, ctypes.c_int, ctypes.c_int, _i32p, _i32p]
_lib.or_dense_attention.restype = None
_lib.or_dense_attention.argtypes = [_f64p, ctypes.c_int, _f64p, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_double, _f64p, _f64p]
_lib.or_gather_keys.restype = ctypes.c_int
_lib.or_gather_keys.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _u8p, _i32p, _i32p,
                                ctypes.c_int, _u16p, _i32p, ctypes.c_int, ctypes.c_int, _f64p]
_lib.or_sparse_mla.restype = ctypes.c_int
_lib.or_sparse_mla.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               _u8p, _i32p, _i32p, ctypes.c_int, _u16p, _i32p, ctypes.c_int,
                               ctypes.c_int, ctypes.c_double, _f64p, _f64p]

_lib.or_e2m1_to_f64.restype = ctypes.c_double
_lib.or_e2m1_to_f64.argtypes = [ctypes.c_uint8]
_lib.or_f32_to_e2m1.restype = ctypes.c_uint8
_lib.or_f32_to_e2m1.argtypes = [ctypes.c_float]
_lib.or_mxfp4_exponent.restype = ctypes.c_int
_lib.or_mxfp4_exponent.argtypes = [ctypes.c_float]
_lib.or_quant_idx_fp4_rows.restype = None
_lib.or_quant_idx_fp4_rows.argtypes = [ctypes.c_longlong, _f32p, ctypes.c_int, _u8p, _u8p]
_lib.or_idx_fp4_entry_bytes.restype = ctypes.c_int
_lib.or_idx_fp4_entry_bytes.argtypes = [ctypes.c_int]
_lib.or_indexer_logits_fp4.restype = None
_lib.or_indexer_logits_fp4.argtypes = [_u8p, _f32p, ctypes.c_int, ctypes.c_int, _u8p, _i32p,
                                       ctypes.c_int, ctypes.c_int, _f64p]

_lib.or_dequant_gather.restype = None
_lib.or_dequant_gather.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u8p, _i32p,
                                   ctypes.c_int, ctypes.c_int, _u16p]
_lib.or_combine_topk_swa_indices.restype = ctypes.c_int
_lib.or_combine_topk_swa_indices.argtypes = [_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, _i32p]

_lib.or_sparse_mla_v4.restype = ctypes.c_int
_lib.or_sparse_mla_v4.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, _u8p, _i32p, _i32p, ctypes.c_int, _u8p,
                                  _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_double, _f64p, _f64p]
_lib.or_inv_rope_fp8_quant.restype = None
_lib.or_inv_rope_fp8_quant.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, _f32p, ctypes.c_int, _u8p, _f32p]

MLA_KIND = 0
IDX_KIND = 1
IDX_FP4_KIND = 2


def sparse_mla_v4(q_bf16, comp_cache, comp_bt_row, idx, length, swa_cache, swa_bt_row, p, scale, window=128,
                  page=64):
    """V4-native sparse decode attention (K = V over 512 dims, FP8 caches of
    584-byte rows): (out [H][512] double, lse [H])."""
    q = _c(q_bf16, np.uint16)
    n_heads = q.shape[0]
    out = np.empty((n_heads, 512), np.float64)
    lse = np.empty(n_heads, np.float64)
    cc = _c(comp_cache if comp_cache is not None else _EMPTY_U8, np.uint8)
    cbt = _c(comp_bt_row if comp_bt_row is not None else _EMPTY_I32, np.int32)
    ix = _c(idx if idx is not None and length else _EMPTY_I32, np.int32)
    _lib.or_sparse_mla_v4(_p(q, _u16p), n_heads, page, _p(cc, _u8p), _p(cbt, _i32p), _p(ix, _i32p), int(length),
                          _p(_c(swa_cache, np.uint8), _u8p), _p(_c(swa_bt_row, np.int32), _i32p), int(p), window,
                          float(scale), _p(out, _f64p), _p(lse, _f64p))
    return out, lse


def inv_rope_fp8_quant(o_bf16, pos, cos_sin, rope_dim=64):
    """o bf16 bits [H][512] -> (E4M3 codes [H][512], fp32 scales [H][4])."""
    o = _c(o_bf16, np.uint16)
    n_heads = o.shape[0]
    codes = np.empty((n_heads, 512), np.uint8)
    sc = np.empty((n_heads, 4), np.float32)
    _lib.or_inv_rope_fp8_quant(_p(o, _u16p), n_heads, int(pos), _p(_c(cos_sin, np.float32), _f32p), rope_dim,
                               _p(codes, _u8p), _p(sc, _f32p))
    return codes, sc


def dequant_gather(kind, cache, block_table_row, s0, n, nope_dim=512, rope_dim=64, page=64):
    """bf16 bits [n][nope + rope] of compressed slots (kind 0) or SWA tokens
    (kind 1) s0 .. s0 + n - 1 of one sequence."""
    cache = _c(cache, np.uint8) if kind == 0 else _c(cache, np.uint16).view(np.uint8)
    bt = _c(block_table_row, np.int32)
    out = np.zeros((max(n, 1), nope_dim + rope_dim), np.uint16)
    _lib.or_dequant_gather(kind, nope_dim, rope_dim, page, _p(cache, _u8p), _p(bt, _i32p), int(s0), int(n),
                           _p(out, _u16p))
    return out[:n]


def combine_topk_swa_indices(topk, topk_len, pos, seq_len, gather_len, window, n_comp):
    topk = _c(topk, np.int32)
    out = np.zeros(max(1, topk.size + window), np.int32)
    n = _lib.or_combine_topk_swa_indices(_p(topk, _i32p), int(topk_len), int(pos), int(seq_len),
                                         int(gather_len), int(window), int(n_comp), _p(out, _i32p))
    return None if n < 0 else out[:n]


def e2m1_to_f64(code):
    """E2M1 code(s) (low 4 bits) -> value(s), same shape."""
    code = np.asarray(code, np.uint8)
    table = np.array([_lib.or_e2m1_to_f64(c) for c in range(16)], np.float64)
    return table[code & 15]


def f32_to_e2m1(x):
    x = _c(x, np.float32)
    return np.array([_lib.or_f32_to_e2m1(float(v)) for v in x.ravel()], np.uint8).reshape(x.shape)


def mxfp4_exponent(amax: float) -> int:
    return int(_lib.or_mxfp4_exponent(float(np.float32(amax))))


def idx_fp4_entry_bytes(head_dim=128) -> int:
    return int(_lib.or_idx_fp4_entry_bytes(head_dim))


def quant_idx_fp4_rows(z):
    """Rows [n, d] fp32 -> (codes [n, d/2] u8 (two per byte, low nibble first),
    exponent bytes [n, d/32] u8)."""
    z = _c(z, np.float32)
    n, d = z.shape
    data = np.empty((n, d // 2), np.uint8)
    sc = np.empty((n, d // 32), np.uint8)
    _lib.or_quant_idx_fp4_rows(n, _p(z, _f32p), d, _p(data, _u8p), _p(sc, _u8p))
    return data, sc


def indexer_logits_fp4(q_fp8, w, cache, block_table_row, n_c, page=64):
    q = _c(q_fp8, np.uint8)
    n_heads, d = q.shape
    w = _c(w, np.float32)
    cache = _c(cache, np.uint8)
    bt = _c(block_table_row, np.int32)
    out = np.empty(max(n_c, 1), np.float64)
    _lib.or_indexer_logits_fp4(_p(q, _u8p), _p(w, _f32p), n_heads, d, _p(cache, _u8p),
                               _p(bt, _i32p), page, int(n_c), _p(out, _f64p))
    return out[:n_c]


def _p(a, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- number formats ------------------------------------------------------

def bf16_to_f32(h):
    h = _c(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _lib.or_f32_to_bf16_n(x.size, _p(x, _f32p), _p(out, _u16p))
    return out


def e4m3_to_f64(code):
    code = _c(code, np.uint8)
    table = np.array([_lib.or_e4m3_to_f64(c) for c in range(256)], np.float64)
    return table[code]


def f32_to_e4m3(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _lib.or_f32_to_e4m3_n(x.size, _p(x, _f32p), _p(out, _u8p))
    return out


def ue8m0_exponent(amax: float) -> int:
    return int(_lib.or_ue8m0_exponent(float(np.float32(amax))))


def expf(x: float) -> float:
    return float(_lib.or_expf(float(np.float32(x))))


# ---- layer type / schedule / bytes ----------------------------------------

def layer_type(ratio: int) -> int:
    return int(_lib.or_layer_type(int(ratio)))


def index_schedule(ratios, use_index_cache=True, freq=1, pattern=None):
    """Returns a uint8 array of skip_topk flags, or None for an invalid request."""
    r = _c(ratios, np.int32)
    skip = np.zeros(r.size, np.uint8)
    pat = pattern.encode() if pattern is not None else None
    rc = _lib.or_index_schedule(_p(r, _i32p), r.size, int(bool(use_index_cache)), int(freq),
                                pat, _p(skip, _u8p))
    return None if rc != 0 else skip


def mla_entry_bytes(nope_dim=512, rope_dim=64) -> int:
    return int(_lib.or_mla_entry_bytes(nope_dim, rope_dim))


def idx_entry_bytes(head_dim=128) -> int:
    return int(_lib.or_idx_entry_bytes(head_dim))


# ---- RoPE / compressor -----------------------------------------------------

def rope_table(max_pos: int, rope_dim: int = 64, theta: float = 10000.0):
    out = np.empty((max_pos, rope_dim), np.float32)
    _lib.or_rope_table(max_pos, rope_dim, float(theta), _p(out, _f32p))
    return out


def compress_pool(ratio, kv_score_bf16, ape, p):
    """Pre-norm pooled vector of the entry emitted at boundary p (None if p is not one)."""
    ks = _c(kv_score_bf16, np.uint16)
    coff = 2 if ratio == 4 else 1
    d = ks.shape[1] // (2 * coff)
    ape = _c(ape, np.float32)
    y = np.empty(d, np.float32)
    rc = _lib.or_compress_pool(ratio, d, _p(ks, _u16p), ks.shape[1], _p(ape, _f32p), int(p),
                               _p(y, _f32p))
    return None if rc != 0 else y


def rmsnorm(y, w, eps):
    y = _c(y, np.float32)
    w = _c(w, np.float32)
    z = np.empty_like(y)
    _lib.or_rmsnorm(_p(y, _f32p), y.size, _p(w, _f32p), float(np.float32(eps)), _p(z, _f32p))
    return z


def rope_gptj(x, cos_sin_row):
    x = _c(x, np.float32).copy()
    row = _c(cos_sin_row, np.float32)
    _lib.or_rope_gptj(_p(x, _f32p), x.size, _p(row, _f32p))
    return x


def quant_mla(z, nope_dim=512, rope_dim=64):
    z = _c(z, np.float32)
    data = np.empty(nope_dim + 2 * rope_dim, np.uint8)
    scales = np.empty(8, np.uint8)
    _lib.or_quant_mla(_p(z, _f32p), nope_dim, rope_dim, _p(data, _u8p), _p(scales, _u8p))
    return data, scales


def quant_idx(z):
    z = _c(z, np.float32)
    data = np.empty(z.size, np.uint8)
    s = np.empty(1, np.float32)
    _lib.or_quant_idx(_p(z, _f32p), z.size, _p(data, _u8p), _p(s, _f32p))
    return data, float(s[0])


def quant_mla_rows(z, nope_dim=512, rope_dim=64):
    """Rows [n, nope+rope] fp32 -> (data [n, nope+2*rope] u8, scales [n, 8] u8)."""
    z = _c(z, np.float32)
    n = z.shape[0]
    data = np.empty((n, nope_dim + 2 * rope_dim), np.uint8)
    scales = np.empty((n, 8), np.uint8)
    _lib.or_quant_mla_rows(n, _p(z, _f32p), nope_dim, rope_dim, _p(data, _u8p), _p(scales, _u8p))
    return data, scales


def quant_idx_rows(z):
    """Rows [n, d] fp32 -> (data [n, d] u8, scale [n] f32)."""
    z = _c(z, np.float32)
    n, d = z.shape
    data = np.empty((n, d), np.uint8)
    scale = np.empty(n, np.float32)
    _lib.or_quant_idx_rows(n, _p(z, _f32p), d, _p(data, _u8p), _p(scale, _f32p))
    return data, scale


def compress_stream(kind, ratio, kv_score_bf16, ape, rms_w, eps, cos_sin, nope_dim, rope_dim=64):
    """All compressed entries of one sequence's token stream, in slot order.

    Returns (data [n, data_bytes] uint8, scale [n, 8] uint8 (main), [n] float32
    (FP8 indexer) or [n, d/32] uint8 exponent bytes (FP4 indexer))."""
    ks = _c(kv_score_bf16, np.uint16)
    n_tok = ks.shape[0]
    n_out = n_tok // ratio
    d = nope_dim + rope_dim
    data_b = nope_dim + 2 * rope_dim if kind == MLA_KIND else (d if kind == IDX_KIND else d // 2)
    scale_b = 8 if kind == MLA_KIND else (4 if kind == IDX_KIND else d // 32)
    data = np.zeros((max(n_out, 1), data_b), np.uint8)
    scale = np.zeros((max(n_out, 1), scale_b), np.uint8)
    ape = _c(ape, np.float32)
    w = _c(rms_w, np.float32)
    cs = _c(cos_sin, np.float32)
    n = _lib.or_compress_stream(kind, ratio, n_tok, _p(ks, _u16p), ks.shape[1], _p(ape, _f32p),
                                _p(w, _f32p), float(np.float32(eps)), _p(cs, _f32p), rope_dim,
                                nope_dim, _p(data, _u8p), _p(scale, _u8p))
    assert n == n_out, (n, n_out)
    data, scale = data[:n_out], scale[:n_out]
    if kind == IDX_KIND:
        scale = scale.view(np.float32).reshape(n_out)
    return data, scale


def _nope(kind, nope_dim):
    return nope_dim if nope_dim is not None else (512 if kind == MLA_KIND else 64)


def page_bytes(kind, page=64, nope_dim=None, rope_dim=64):
    nope_dim = _nope(kind, nope_dim)
    if kind == MLA_KIND:
        return page * (nope_dim + 2 * rope_dim + 8)
    if kind == IDX_FP4_KIND:
        d = nope_dim + rope_dim
        return page * (d // 2 + d // 32)
    return page * (nope_dim + rope_dim + 4)


def page_write(kind, cache, block_table_row, data, scale, page=64, nope_dim=None, rope_dim=64):
    """Write a sequence's entries (slot order) into the paged byte array ``cache`` in place."""
    nope_dim = _nope(kind, nope_dim)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    bt = _c(block_table_row, np.int32)
    data = _c(data, np.uint8)
    sc = _c(scale, np.float32).view(np.uint8) if kind == IDX_KIND else _c(scale, np.uint8)
    _lib.or_page_write(kind, nope_dim, rope_dim, page, _p(bt, _i32p), data.shape[0],
                       _p(data, _u8p), _p(sc, _u8p), _p(cache, _u8p))


# ---- indexer / top-k ---------------------------------------------------------

def indexer_logits(q_fp8, w, cache, block_table_row, n_c, page=64):
    q = _c(q_fp8, np.uint8)
    n_heads, d = q.shape
    w = _c(w, np.float32)
    cache = _c(cache, np.uint8)
    bt = _c(block_table_row, np.int32)
    out = np.empty(max(n_c, 1), np.float64)
    _lib.or_indexer_logits(_p(q, _u8p), _p(w, _f32p), n_heads, d, _p(cache, _u8p),
                           _p(bt, _i32p), page, int(n_c), _p(out, _f64p))
    return out[:n_c]


def topk(logits, k):
    lg = _c(logits, np.float64)
    idx = np.empty(max(k, 1), np.int32)
    ln = np.zeros(1, np.int32)
    rc = _lib.or_topk(_p(lg, _f64p), lg.size, int(k), _p(idx, _i32p), _p(ln, _i32p))
    assert rc == 0
    return idx[:k], int(ln[0])


# ---- attention ------------------------------------------------------------------

def dense_attention(q, keys, dv, scale):
    q = _c(q, np.float64)
    keys = _c(keys, np.float64)
    n_heads, dk = q.shape
    out = np.empty((n_heads, dv), np.float64)
    lse = np.empty(n_heads, np.float64)
    _lib.or_dense_attention(_p(q, _f64p), n_heads, _p(keys, _f64p), keys.shape[0], dk, dv,
                            float(scale), _p(out, _f64p), _p(lse, _f64p))
    return out, lse


_EMPTY_U8 = np.zeros(1, np.uint8)
_EMPTY_I32 = np.zeros(1, np.int32)


def gather_keys(comp_cache, comp_bt_row, idx, length, swa_cache, swa_bt_row, p, window=128,
                page=64, nope_dim=512, rope_dim=64):
    dk = nope_dim + rope_dim
    cc = _c(comp_cache, np.uint8) if comp_cache is not None else _EMPTY_U8
    cbt = _c(comp_bt_row, np.int32) if comp_bt_row is not None else _EMPTY_I32
    ix = _c(idx, np.int32) if idx is not None else _EMPTY_I32
    sc = _c(swa_cache, np.uint16)
    sbt = _c(swa_bt_row, np.int32)
    keys = np.empty((length + window, dk), np.float64)
    n = _lib.or_gather_keys(nope_dim, rope_dim, page, _p(cc, _u8p), _p(cbt, _i32p),
                            _p(ix, _i32p), int(length), _p(sc, _u16p), _p(sbt, _i32p), int(p),
                            int(window), _p(keys, _f64p))
    return keys[:n]


def sparse_mla(q_bf16, comp_cache, comp_bt_row, idx, length, swa_cache, swa_bt_row, p, scale,
               window=128, page=64, nope_dim=512, rope_dim=64):
    """One query token: returns (out [H, nope] float64, lse [H] float64, n_keys)."""
    q = _c(q_bf16, np.uint16)
    n_heads = q.shape[0]
    cc = _c(comp_cache, np.uint8) if comp_cache is not None else _EMPTY_U8
    cbt = _c(comp_bt_row, np.int32) if comp_bt_row is not None else _EMPTY_I32
    ix = _c(idx, np.int32) if idx is not None else _EMPTY_I32
    sc = _c(swa_cache, np.uint16)
    sbt = _c(swa_bt_row, np.int32)
    out = np.empty((n_heads, nope_dim), np.float64)
    lse = np.empty(n_heads, np.float64)
    n = _lib.or_sparse_mla(_p(q, _u16p), n_heads, nope_dim, rope_dim, page, _p(cc, _u8p),
                           _p(cbt, _i32p), _p(ix, _i32p), int(length), _p(sc, _u16p),
                           _p(sbt, _i32p), int(p), int(window), float(scale), _p(out, _f64p),
                           _p(lse, _f64p))
    return out, lse, n
