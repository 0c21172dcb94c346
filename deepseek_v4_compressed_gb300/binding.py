"""Thin ctypes binding of libdsv4 (include/dsv4.h): argument marshalling only.

Every step of the decode path runs in the CUDA library; this module turns
torch tensors into device pointers and the current torch stream into a
cudaStream_t.  If the library is not built it raises: there is no fallback.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsv4.so")

SWAONLY, C4A, C128A = 1, 4, 128
CACHE_MLA, CACHE_IDX, CACHE_IDX_FP4, CACHE_V4 = 0, 1, 2, 3
IDX_FP8, IDX_FP4 = 0, 1
KV_576, KV_V4 = 0, 1

OK, ERR_INVALID, ERR_SHAPE, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_CHECK, ERR_TIMEOUT = range(7)
DEV_BAD_INDEX, DEV_BAD_PAGE, DEV_BAD_POSITION, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8

NOPE_DIM, ROPE_DIM, HEAD_DIM, V_DIM, IDX_DIM, PAGE, WINDOW = 512, 64, 576, 512, 128, 64, 128
MLA_PAGE_BYTES = 64 * 648
IDX_PAGE_BYTES = 64 * 132
IDX_FP4_PAGE_BYTES = 64 * 68
V4_NOPE_DIM, V4_HEAD_DIM = 448, 512
V4_PAGE_BYTES = 64 * 584
PAGE_BYTES = {CACHE_MLA: MLA_PAGE_BYTES, CACHE_IDX: IDX_PAGE_BYTES, CACHE_IDX_FP4: IDX_FP4_PAGE_BYTES,
              CACHE_V4: V4_PAGE_BYTES}
SWA_PAGE_BYTES = 64 * 576 * 2

EXPORTED = ["dsv4_version", "dsv4_status_string", "dsv4_layer_type_from_ratio",
            "dsv4_index_schedule", "dsv4_rope_table", "dsv4_read_device_status",
            "dsv4_plan_create", "dsv4_plan_destroy", "dsv4_plan_workspace_bytes",
            "dsv4_plan_get_info", "dsv4_compress_insert", "dsv4_cache_insert_rows",
            "dsv4_indexer_topk", "dsv4_sparse_mla_decode", "dsv4_selftest_bounded_wait",
            "dsv4_selftest_key_dequant", "dsv4_compress_insert_pair", "dsv4_plan_set_indexer_format",
            "dsv4_sparse_mla_prefill", "dsv4_dequant_gather", "dsv4_combine_topk_swa_indices",
            "dsv4_plan_set_kv_layout", "dsv4_inv_rope_fp8_quant", "dsv4_stream_gate"]
GATHER_COMP, GATHER_SWA = 0, 1


class Dsv4Error(RuntimeError):
    def __init__(self, status, what):
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))
        self.status = status


class Geom(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int), ("idx_heads", ctypes.c_int), ("window", ctypes.c_int),
                ("softmax_scale", ctypes.c_float)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("layer_type", ctypes.c_int), ("batch", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("idx_heads", ctypes.c_int), ("topk", ctypes.c_int), ("max_ctx", ctypes.c_int),
                ("max_slots", ctypes.c_int), ("idx_ctas_per_seq", ctypes.c_int),
                ("mla_splits", ctypes.c_int), ("mla_head_groups", ctypes.c_int),
                ("mla_keys_per_split", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
                ("launches_indexer", ctypes.c_int), ("launches_mla", ctypes.c_int)]


class CompressArgs(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("ratio", ctypes.c_int), ("num_tokens", ctypes.c_int),
                ("num_seqs", ctypes.c_int), ("one_token_per_seq", ctypes.c_int),
                ("kv_score_dev", ctypes.c_void_p), ("kv_score_stride", ctypes.c_longlong),
                ("positions_dev", ctypes.c_void_p), ("seq_dev", ctypes.c_void_p),
                ("ape_dev", ctypes.c_void_p), ("rms_weight_dev", ctypes.c_void_p),
                ("rms_eps", ctypes.c_float), ("cos_sin_dev", ctypes.c_void_p),
                ("max_pos", ctypes.c_int), ("state_dev", ctypes.c_void_p),
                ("cache_dev", ctypes.c_void_p), ("num_pages", ctypes.c_int),
                ("block_table_dev", ctypes.c_void_p), ("bt_stride", ctypes.c_int),
                ("status_dev", ctypes.c_void_p)]


class InsertRowsArgs(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("num_rows", ctypes.c_int), ("rows_dev", ctypes.c_void_p),
                ("seq_dev", ctypes.c_void_p), ("slot_dev", ctypes.c_void_p),
                ("cache_dev", ctypes.c_void_p), ("num_pages", ctypes.c_int),
                ("block_table_dev", ctypes.c_void_p), ("bt_stride", ctypes.c_int),
                ("num_seqs", ctypes.c_int), ("status_dev", ctypes.c_void_p)]


class IndexerArgs(ctypes.Structure):
    _fields_ = [("q_fp8_dev", ctypes.c_void_p), ("weights_dev", ctypes.c_void_p),
                ("idx_cache_dev", ctypes.c_void_p), ("num_pages", ctypes.c_int),
                ("block_table_dev", ctypes.c_void_p), ("bt_stride", ctypes.c_int),
                ("ctx_len_dev", ctypes.c_void_p), ("out_idx_dev", ctypes.c_void_p),
                ("out_stride", ctypes.c_int), ("out_len_dev", ctypes.c_void_p),
                ("status_dev", ctypes.c_void_p), ("row_seq_dev", ctypes.c_void_p), ("bt_rows", ctypes.c_int)]


class MlaArgs(ctypes.Structure):
    _fields_ = [("q_dev", ctypes.c_void_p), ("swa_cache_dev", ctypes.c_void_p),
                ("swa_num_pages", ctypes.c_int), ("swa_block_table_dev", ctypes.c_void_p),
                ("swa_bt_stride", ctypes.c_int), ("comp_cache_dev", ctypes.c_void_p),
                ("comp_num_pages", ctypes.c_int), ("comp_block_table_dev", ctypes.c_void_p),
                ("comp_bt_stride", ctypes.c_int), ("topk_idx_dev", ctypes.c_void_p),
                ("topk_stride", ctypes.c_int), ("topk_len_dev", ctypes.c_void_p),
                ("ctx_len_dev", ctypes.c_void_p), ("out_dev", ctypes.c_void_p),
                ("lse_dev", ctypes.c_void_p), ("status_dev", ctypes.c_void_p),
                ("row_seq_dev", ctypes.c_void_p), ("bt_rows", ctypes.c_int),
                ("out_codes_dev", ctypes.c_void_p), ("out_scales_dev", ctypes.c_void_p),
                ("cos_sin_dev", ctypes.c_void_p), ("max_pos", ctypes.c_int)]


class GatherArgs(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("cache_dev", ctypes.c_void_p), ("num_pages", ctypes.c_int),
                ("block_table_dev", ctypes.c_void_p), ("bt_stride", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("first_dev", ctypes.c_void_p), ("count_dev", ctypes.c_void_p), ("max_count", ctypes.c_int),
                ("out_dev", ctypes.c_void_p), ("out_rows", ctypes.c_int), ("out_offset", ctypes.c_int),
                ("status_dev", ctypes.c_void_p)]


class CombineArgs(ctypes.Structure):
    _fields_ = [("topk_dev", ctypes.c_void_p), ("topk_stride", ctypes.c_int), ("topk_len_dev", ctypes.c_void_p),
                ("pos_dev", ctypes.c_void_p), ("row_seq_dev", ctypes.c_void_p), ("seq_len_dev", ctypes.c_void_p),
                ("gather_len_dev", ctypes.c_void_p), ("num_tokens", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("window", ctypes.c_int), ("n_comp", ctypes.c_int), ("out_dev", ctypes.c_void_p),
                ("out_stride", ctypes.c_int), ("out_len_dev", ctypes.c_void_p), ("status_dev", ctypes.c_void_p)]


class InvRopeQuantArgs(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int), ("n_heads", ctypes.c_int), ("o_dev", ctypes.c_void_p),
                ("positions_dev", ctypes.c_void_p), ("cos_sin_dev", ctypes.c_void_p), ("max_pos", ctypes.c_int),
                ("codes_dev", ctypes.c_void_p), ("scales_dev", ctypes.c_void_p), ("status_dev", ctypes.c_void_p)]


class GateArgs(ctypes.Structure):
    _fields_ = [("flags_dev", ctypes.c_void_p * 4), ("timeout_us", ctypes.c_int), ("status_dev", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded libdsv4.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libdsv4.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    st = ctypes.c_int
    vp = ctypes.c_void_p
    L.dsv4_version.restype = ctypes.c_int
    L.dsv4_status_string.restype = ctypes.c_char_p
    L.dsv4_status_string.argtypes = [st]
    L.dsv4_layer_type_from_ratio.restype = st
    L.dsv4_layer_type_from_ratio.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    L.dsv4_index_schedule.restype = st
    L.dsv4_index_schedule.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_char_p, ctypes.POINTER(ctypes.c_ubyte)]
    L.dsv4_rope_table.restype = st
    L.dsv4_rope_table.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int, ctypes.c_int,
                                  ctypes.c_double]
    L.dsv4_read_device_status.restype = st
    L.dsv4_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    L.dsv4_plan_create.restype = st
    L.dsv4_plan_create.argtypes = [ctypes.c_int, ctypes.POINTER(Geom), ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.POINTER(vp)]
    L.dsv4_plan_destroy.restype = None
    L.dsv4_plan_destroy.argtypes = [vp]
    L.dsv4_plan_workspace_bytes.restype = ctypes.c_size_t
    L.dsv4_plan_workspace_bytes.argtypes = [vp]
    L.dsv4_plan_get_info.restype = st
    L.dsv4_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
    L.dsv4_compress_insert.restype = st
    L.dsv4_compress_insert.argtypes = [ctypes.POINTER(CompressArgs), vp]
    L.dsv4_cache_insert_rows.restype = st
    L.dsv4_cache_insert_rows.argtypes = [ctypes.POINTER(InsertRowsArgs), vp]
    L.dsv4_indexer_topk.restype = st
    L.dsv4_indexer_topk.argtypes = [vp, ctypes.POINTER(IndexerArgs), vp, ctypes.c_size_t, vp]
    L.dsv4_sparse_mla_decode.restype = st
    L.dsv4_sparse_mla_decode.argtypes = [vp, ctypes.POINTER(MlaArgs), vp, ctypes.c_size_t, vp]
    L.dsv4_selftest_bounded_wait.restype = st
    L.dsv4_selftest_bounded_wait.argtypes = [vp, ctypes.c_int, vp]
    L.dsv4_compress_insert_pair.restype = st
    L.dsv4_compress_insert_pair.argtypes = [ctypes.POINTER(CompressArgs), ctypes.POINTER(CompressArgs), vp]
    L.dsv4_selftest_key_dequant.restype = st
    L.dsv4_selftest_key_dequant.argtypes = [vp, vp]
    L.dsv4_plan_set_indexer_format.restype = st
    L.dsv4_plan_set_indexer_format.argtypes = [vp, ctypes.c_int]
    L.dsv4_sparse_mla_prefill.restype = st
    L.dsv4_sparse_mla_prefill.argtypes = [vp, ctypes.POINTER(MlaArgs), vp, ctypes.c_size_t, vp]
    L.dsv4_dequant_gather.restype = st
    L.dsv4_dequant_gather.argtypes = [ctypes.POINTER(GatherArgs), vp]
    L.dsv4_combine_topk_swa_indices.restype = st
    L.dsv4_combine_topk_swa_indices.argtypes = [ctypes.POINTER(CombineArgs), vp]
    L.dsv4_plan_set_kv_layout.restype = st
    L.dsv4_plan_set_kv_layout.argtypes = [vp, ctypes.c_int]
    L.dsv4_inv_rope_fp8_quant.restype = st
    L.dsv4_inv_rope_fp8_quant.argtypes = [ctypes.POINTER(InvRopeQuantArgs), vp]
    L.dsv4_stream_gate.restype = st
    L.dsv4_stream_gate.argtypes = [ctypes.POINTER(GateArgs), vp]
    _lib = L
    return L


def status_string(s):
    return lib().dsv4_status_string(int(s)).decode()


def _check(status, what):
    if status != OK:
        raise Dsv4Error(status, what)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _nbytes(t):
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def version():
    return lib().dsv4_version()


def layer_type_from_ratio(ratio):
    out = ctypes.c_int(0)
    _check(lib().dsv4_layer_type_from_ratio(int(ratio), ctypes.byref(out)), "layer_type_from_ratio")
    return out.value


def index_schedule(ratios, use_index_cache=True, freq=2, pattern=None):
    n = len(ratios)
    arr = (ctypes.c_int * max(n, 1))(*[int(r) for r in ratios])
    out = (ctypes.c_ubyte * max(n, 1))()
    _check(lib().dsv4_index_schedule(arr, n, int(bool(use_index_cache)), int(freq),
                                     pattern.encode() if pattern is not None else None, out),
           "index_schedule")
    return [int(out[i]) for i in range(n)]


def rope_table(max_pos, rope_dim=ROPE_DIM, theta=10000.0):
    """Host fp32 tensor [max_pos, rope_dim] (copy it to the GPU yourself)."""
    t = torch.empty((max_pos, rope_dim), dtype=torch.float32)
    _check(lib().dsv4_rope_table(ctypes.cast(t.data_ptr(), ctypes.POINTER(ctypes.c_float)), max_pos,
                                 rope_dim, float(theta)), "rope_table")
    return t


def read_device_status(status_dev, stream=None):
    bits = ctypes.c_int(0)
    st = lib().dsv4_read_device_status(_ptr(status_dev), _stream(stream), ctypes.byref(bits))
    return st, bits.value


def selftest_key_dequant(out_dev, stream=None):
    """Every (E4M3 code, UE8M0 scale byte) through the decode kernel's key
    conversion; out_dev: uint16 [65536] receives the bf16 bits."""
    _check(lib().dsv4_selftest_key_dequant(_ptr(out_dev), _stream(stream)), "selftest_key_dequant")


def selftest_bounded_wait(status_dev, spin_limit, stream=None):
    _check(lib().dsv4_selftest_bounded_wait(_ptr(status_dev), int(spin_limit), _stream(stream)),
           "selftest_bounded_wait")


class Plan:
    """One plan per layer type, reused by every layer of that type in a step."""

    def __init__(self, layer_type, n_heads, batch, topk, max_ctx, idx_heads=64, window=WINDOW,
                 softmax_scale=None, idx_format=IDX_FP8, kv_layout=KV_576):
        if softmax_scale is None:
            softmax_scale = (V4_HEAD_DIM if kv_layout == KV_V4 else HEAD_DIM) ** -0.5
        self.geom = Geom(int(n_heads), int(idx_heads), int(window), float(softmax_scale))
        h = ctypes.c_void_p()
        _check(lib().dsv4_plan_create(int(layer_type), ctypes.byref(self.geom), int(batch), int(topk),
                                      int(max_ctx), ctypes.byref(h)), "plan_create")
        self.handle = h
        self.layer_type = int(layer_type)
        self.idx_format = IDX_FP8
        if idx_format != IDX_FP8:
            _check(lib().dsv4_plan_set_indexer_format(self.handle, int(idx_format)), "plan_set_indexer_format")
            self.idx_format = int(idx_format)
        self.kv_layout = KV_576
        if kv_layout != KV_576:
            _check(lib().dsv4_plan_set_kv_layout(self.handle, int(kv_layout)), "plan_set_kv_layout")
            self.kv_layout = int(kv_layout)

    @property
    def comp_page_bytes(self):
        return V4_PAGE_BYTES if self.kv_layout == KV_V4 else MLA_PAGE_BYTES

    @property
    def swa_page_bytes(self):
        return V4_PAGE_BYTES if self.kv_layout == KV_V4 else SWA_PAGE_BYTES

    @property
    def idx_page_bytes(self):
        return IDX_FP4_PAGE_BYTES if self.idx_format == IDX_FP4 else IDX_PAGE_BYTES

    @property
    def workspace_bytes(self):
        return int(lib().dsv4_plan_workspace_bytes(self.handle))

    def info(self):
        i = PlanInfo()
        _check(lib().dsv4_plan_get_info(self.handle, ctypes.byref(i)), "plan_get_info")
        return {f: getattr(i, f) for f, _ in PlanInfo._fields_}

    def workspace(self, device="cuda"):
        return torch.empty(max(self.workspace_bytes, 1), dtype=torch.uint8, device=device)

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.dsv4_plan_destroy(self.handle)
            self.handle = None


def compress_insert(kind, ratio, kv_score, positions, seqs, ape, rms_weight, rms_eps, cos_sin,
                    state, cache, block_table, num_seqs, one_token_per_seq=True, status=None,
                    stream=None):
    """Compressor state update + compressed-cache insert for the tokens in kv_score
    (bf16 [T, 2*coff*d]); see dsv4_compress_insert."""
    a = CompressArgs(int(kind), int(ratio), int(kv_score.shape[0]), int(num_seqs),
                     int(bool(one_token_per_seq)), _ptr(kv_score), int(kv_score.stride(0)),
                     _ptr(positions), _ptr(seqs), _ptr(ape), _ptr(rms_weight), float(rms_eps),
                     _ptr(cos_sin), int(cos_sin.shape[0]), _ptr(state), _ptr(cache),
                     int(_nbytes(cache) // PAGE_BYTES[kind]),
                     _ptr(block_table), int(block_table.shape[1]), _ptr(status))
    _check(lib().dsv4_compress_insert(ctypes.byref(a), _stream(stream)), "compress_insert")


def _compress_args(kind, ratio, kv_score, positions, seqs, ape, rms_weight, rms_eps, cos_sin, state, cache,
                   block_table, num_seqs, one_token_per_seq, status):
    return CompressArgs(int(kind), int(ratio), int(kv_score.shape[0]), int(num_seqs),
                        int(bool(one_token_per_seq)), _ptr(kv_score), int(kv_score.stride(0)),
                        _ptr(positions), _ptr(seqs), _ptr(ape), _ptr(rms_weight), float(rms_eps),
                        _ptr(cos_sin), int(cos_sin.shape[0]), _ptr(state), _ptr(cache),
                        int(_nbytes(cache) // PAGE_BYTES[kind]),
                        _ptr(block_table), int(block_table.shape[1]), _ptr(status))


def compress_insert_pair(main, idx, stream=None):
    """Both compressor streams of a layer in one launch (decode: one token per
    sequence).  main / idx: dicts with the compress_insert arguments (kind,
    ratio, kv_score, positions, seqs, ape, rms_weight, rms_eps, cos_sin,
    state, cache, block_table, num_seqs, status); see dsv4_compress_insert_pair."""
    am = _compress_args(one_token_per_seq=True, **main)
    ai = _compress_args(one_token_per_seq=True, **idx)
    _check(lib().dsv4_compress_insert_pair(ctypes.byref(am), ctypes.byref(ai), _stream(stream)),
           "compress_insert_pair")


def cache_insert_rows(kind, rows, seqs, slots, cache, block_table, status=None, stream=None):
    a = InsertRowsArgs(int(kind), int(rows.shape[0]), _ptr(rows), _ptr(seqs), _ptr(slots),
                       _ptr(cache),
                       int(_nbytes(cache) // PAGE_BYTES[kind]),
                       _ptr(block_table), int(block_table.shape[1]), int(block_table.shape[0]),
                       _ptr(status))
    _check(lib().dsv4_cache_insert_rows(ctypes.byref(a), _stream(stream)), "cache_insert_rows")


def indexer_topk(plan, q_fp8, weights, idx_cache, block_table, ctx_len, out_idx, out_len, workspace,
                 status=None, stream=None, row_seq=None):
    """dsv4_indexer_topk; row_seq (int32 [rows]) maps each query row to its
    block-table row (prefill: one row per query token)."""
    a = IndexerArgs(_ptr(q_fp8), _ptr(weights), _ptr(idx_cache), int(_nbytes(idx_cache) // plan.idx_page_bytes),
                    _ptr(block_table), int(block_table.shape[1]), _ptr(ctx_len), _ptr(out_idx),
                    int(out_idx.shape[1]), _ptr(out_len), _ptr(status), _ptr(row_seq),
                    int(block_table.shape[0]))
    _check(lib().dsv4_indexer_topk(plan.handle, ctypes.byref(a), _ptr(workspace), _nbytes(workspace),
                                   _stream(stream)), "indexer_topk")


def sparse_mla_decode(plan, q, swa_cache, swa_block_table, ctx_len, out, workspace, comp_cache=None,
                      comp_block_table=None, topk_idx=None, topk_len=None, lse=None, status=None,
                      stream=None, row_seq=None, out_codes=None, out_scales=None, cos_sin=None):
    """dsv4_sparse_mla_decode; V4 plans may also ask for the quantised,
    inverse-rotated output (out_codes uint8 [B, H, 512], out_scales fp32
    [B, H, 4], cos_sin fp32 [max_pos, 64])."""
    a = MlaArgs(_ptr(q), _ptr(swa_cache), int(_nbytes(swa_cache) // plan.swa_page_bytes),
                _ptr(swa_block_table), int(swa_block_table.shape[1]), _ptr(comp_cache),
                int(_nbytes(comp_cache) // plan.comp_page_bytes) if comp_cache is not None else 0,
                _ptr(comp_block_table),
                int(comp_block_table.shape[1]) if comp_block_table is not None else 0,
                _ptr(topk_idx), int(topk_idx.shape[1]) if topk_idx is not None else 0,
                _ptr(topk_len), _ptr(ctx_len), _ptr(out), _ptr(lse), _ptr(status), _ptr(row_seq),
                int(swa_block_table.shape[0]), _ptr(out_codes), _ptr(out_scales), _ptr(cos_sin),
                int(cos_sin.shape[0]) if cos_sin is not None else 0)
    _check(lib().dsv4_sparse_mla_decode(plan.handle, ctypes.byref(a), _ptr(workspace),
                                        workspace.numel(), _stream(stream)), "sparse_mla_decode")


def indexer_topk_noalloc(plan, q_fp8, weights, idx_cache, block_table, ctx_len, out_idx, out_len,
                         status=None, stream=None):
    """dsv4_indexer_topk_noalloc: the indexer without a caller workspace (scratch in a
    4 MiB device array the library owns; overlapping calls race on it)."""
    f = lib().dsv4_indexer_topk_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.POINTER(IndexerArgs), ctypes.c_void_p]
    a = IndexerArgs(_ptr(q_fp8), _ptr(weights), _ptr(idx_cache), int(_nbytes(idx_cache) // plan.idx_page_bytes),
                    _ptr(block_table), int(block_table.shape[1]), _ptr(ctx_len), _ptr(out_idx),
                    int(out_idx.shape[1]), _ptr(out_len), _ptr(status))
    _check(f(plan.handle, ctypes.byref(a), _stream(stream)), "indexer_topk_noalloc")


def sparse_mla_prefill(plan, q, swa_cache, swa_block_table, ctx_len, row_seq, out, workspace, comp_cache=None,
                       comp_block_table=None, topk_idx=None, topk_len=None, lse=None, status=None, stream=None,
                       out_codes=None, out_scales=None, cos_sin=None):
    """dsv4_sparse_mla_prefill: one query row per prefill token (position
    ctx_len - 1), row_seq mapping each row to its block-table row; V4 plans
    may also ask for the quantised output as in sparse_mla_decode."""
    a = MlaArgs(_ptr(q), _ptr(swa_cache), int(_nbytes(swa_cache) // plan.swa_page_bytes),
                _ptr(swa_block_table), int(swa_block_table.shape[1]), _ptr(comp_cache),
                int(_nbytes(comp_cache) // plan.comp_page_bytes) if comp_cache is not None else 0,
                _ptr(comp_block_table),
                int(comp_block_table.shape[1]) if comp_block_table is not None else 0,
                _ptr(topk_idx), int(topk_idx.shape[1]) if topk_idx is not None else 0,
                _ptr(topk_len), _ptr(ctx_len), _ptr(out), _ptr(lse), _ptr(status), _ptr(row_seq),
                int(swa_block_table.shape[0]), _ptr(out_codes), _ptr(out_scales), _ptr(cos_sin),
                int(cos_sin.shape[0]) if cos_sin is not None else 0)
    _check(lib().dsv4_sparse_mla_prefill(plan.handle, ctypes.byref(a), _ptr(workspace), workspace.numel(),
                                         _stream(stream)), "sparse_mla_prefill")


def dequant_gather(kind, cache, block_table, first, count, max_count, out, out_offset=0, status=None, stream=None):
    """dsv4_dequant_gather: out[s][out_offset + i] = dequantised row first[s] + i, i < count[s]."""
    page_b = MLA_PAGE_BYTES if kind == GATHER_COMP else SWA_PAGE_BYTES
    a = GatherArgs(int(kind), _ptr(cache), int(_nbytes(cache) // page_b), _ptr(block_table),
                   int(block_table.shape[1]), int(block_table.shape[0]), _ptr(first), _ptr(count), int(max_count),
                   _ptr(out), int(out.shape[1]), int(out_offset), _ptr(status))
    _check(lib().dsv4_dequant_gather(ctypes.byref(a), _stream(stream)), "dequant_gather")


def combine_topk_swa_indices(topk, topk_len, pos, row_seq, seq_len, gather_len, window, n_comp, out, out_len,
                             status=None, stream=None):
    """dsv4_combine_topk_swa_indices: each prefill token's top-k slots, then its window rows."""
    a = CombineArgs(_ptr(topk), int(topk.shape[1]), _ptr(topk_len), _ptr(pos), _ptr(row_seq), _ptr(seq_len),
                    _ptr(gather_len), int(topk.shape[0]), int(seq_len.shape[0]), int(window), int(n_comp),
                    _ptr(out), int(out.shape[1]), _ptr(out_len), _ptr(status))
    _check(lib().dsv4_combine_topk_swa_indices(ctypes.byref(a), _stream(stream)), "combine_topk_swa_indices")


def inv_rope_fp8_quant(o, positions, cos_sin, codes, scales, status=None, stream=None):
    """dsv4_inv_rope_fp8_quant: o bf16 [T, H, 512] -> codes uint8 [T, H, 512]
    (E4M3) and scales fp32 [T, H, 4], R(-position) applied to dims 448..511."""
    a = InvRopeQuantArgs(int(o.shape[0]), int(o.shape[1]), _ptr(o), _ptr(positions), _ptr(cos_sin),
                         int(cos_sin.shape[0]), _ptr(codes), _ptr(scales), _ptr(status))
    _check(lib().dsv4_inv_rope_fp8_quant(ctypes.byref(a), _stream(stream)), "inv_rope_fp8_quant")


def stream_gate(flags, status=None, timeout_us=0, stream=None):
    """dsv4_stream_gate: wait until every flag (int32 CUDA tensors of one
    element, up to 4) is nonzero, clear them, and let the next kernel on the
    stream launch under programmatic dependent launch."""
    flags = list(flags)
    if not 1 <= len(flags) <= 4:
        raise ValueError("1 to 4 flags")
    a = GateArgs()
    for i, f in enumerate(flags):
        if f.dtype != torch.int32 or f.numel() != 1:
            raise ValueError("a flag is one int32 element")
        a.flags_dev[i] = _ptr(f)
    a.timeout_us = int(timeout_us)
    a.status_dev = _ptr(status)
    _check(lib().dsv4_stream_gate(ctypes.byref(a), _stream(stream)), "stream_gate")
