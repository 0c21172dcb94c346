"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and its host-side utilities and validation behave."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from deepseek_v4_compressed_gb300 import binding as B
from deepseek_v4_compressed_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dsv4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsv4_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B.LIB_PATH)
    syms = declared_symbols()
    assert len(syms) >= 15
    for s in syms:
        assert hasattr(lib, s), s
    assert set(B.EXPORTED) <= set(syms)
    assert B.version() == 1


def test_layer_type_from_ratio_matches_oracle():
    for r in [0, 1, 4, 128]:
        assert B.layer_type_from_ratio(r) == oracle.layer_type(r)
    for r in [2, 8, 64]:
        with pytest.raises(B.Dsv4Error) as e:
            B.layer_type_from_ratio(r)
        assert e.value.status == B.ERR_UNSUPPORTED


def test_index_schedule_matches_oracle():
    ratios = synth.mixed_stack_ratios()
    for use, freq, pat in [(True, 2, None), (True, 1, None), (False, 2, None), (True, 3, None),
                           (True, 2, "FSSF"), (True, 2, "F")]:
        assert B.index_schedule(ratios, use, freq, pat) == list(oracle.index_schedule(ratios, use, freq, pat))
    for pat in ["SF", "FX", ""]:
        with pytest.raises(B.Dsv4Error):
            B.index_schedule(ratios, True, 2, pat)


def test_rope_table_bitwise_equals_oracle():
    ours = B.rope_table(4096, 64, 10000.0).numpy()
    assert np.array_equal(ours, oracle.rope_table(4096, 64, 10000.0))


def test_plan_validation_and_info():
    p = B.Plan(B.C4A, n_heads=64, batch=32, topk=512, max_ctx=32768, idx_heads=64)
    info = p.info()
    assert info["max_slots"] == 8192 and info["topk"] == 512 and info["batch"] == 32
    assert p.workspace_bytes >= 32 * 8192 * 4
    assert p.workspace_bytes % 256 == 0
    assert B.Plan(B.SWAONLY, 8, 1, 0, 100).info()["max_slots"] == 0
    assert B.Plan(B.C128A, 64, 64, 512, 131072).info()["max_slots"] == 1024
    for kwargs, status in [(dict(n_heads=0), B.ERR_UNSUPPORTED), (dict(n_heads=129), B.ERR_UNSUPPORTED),
                           (dict(window=64), B.ERR_UNSUPPORTED), (dict(idx_heads=65), B.ERR_UNSUPPORTED),
                           (dict(topk=0), B.ERR_INVALID), (dict(batch=0), B.ERR_INVALID)]:
        args = dict(layer_type=B.C4A, n_heads=64, batch=4, topk=64, max_ctx=1024, idx_heads=64)
        args.update(kwargs)
        with pytest.raises(B.Dsv4Error) as e:
            B.Plan(**args)
        assert e.value.status == status, kwargs


def test_entry_points_reject_null_arguments_without_gpu():
    lib = B.lib()
    a = B.CompressArgs()
    a.kind, a.ratio, a.num_tokens, a.num_seqs = 0, 4, 1, 1
    assert lib.dsv4_compress_insert(ctypes.byref(a), None) == B.ERR_INVALID
    a.ratio = 8
    assert lib.dsv4_compress_insert(ctypes.byref(a), None) == B.ERR_UNSUPPORTED
    a.kind, a.ratio = 1, 128
    assert lib.dsv4_compress_insert(ctypes.byref(a), None) == B.ERR_UNSUPPORTED
    assert lib.dsv4_compress_insert(None, None) == B.ERR_INVALID
    assert lib.dsv4_compress_insert_pair(None, None, None) == B.ERR_INVALID
    m = B.CompressArgs()
    m.kind, m.ratio, m.num_tokens, m.num_seqs, m.one_token_per_seq = 0, 4, 0, 1, 1
    i = B.CompressArgs()
    i.kind, i.ratio, i.num_tokens, i.num_seqs, i.one_token_per_seq = 1, 4, 0, 1, 1
    assert lib.dsv4_compress_insert_pair(ctypes.byref(m), ctypes.byref(i), None) == B.OK      # nothing to do
    assert lib.dsv4_compress_insert_pair(ctypes.byref(i), ctypes.byref(m), None) == B.ERR_INVALID   # kinds swapped
    m.one_token_per_seq = 0
    assert lib.dsv4_compress_insert_pair(ctypes.byref(m), ctypes.byref(i), None) == B.ERR_INVALID
    p = B.Plan(B.C4A, 8, 1, 32, 512, idx_heads=4)
    ia = B.IndexerArgs()
    assert lib.dsv4_indexer_topk(p.handle, ctypes.byref(ia), None, 0, None) in (B.ERR_SHAPE, B.ERR_INVALID)
    ma = B.MlaArgs()
    assert lib.dsv4_sparse_mla_decode(p.handle, ctypes.byref(ma), None, 0, None) in (B.ERR_SHAPE, B.ERR_INVALID)
    sp = B.Plan(B.SWAONLY, 8, 1, 0, 512)
    assert lib.dsv4_indexer_topk(sp.handle, ctypes.byref(ia), None, 0, None) == B.ERR_SHAPE
    assert lib.dsv4_read_device_status(None, None, None) == B.ERR_INVALID
    assert B.status_string(B.ERR_TIMEOUT).startswith("device-side bounded wait")


@pytest.mark.parametrize("args,expect", [
    # (type, heads, batch, topk, max_ctx, idx_heads) -> plan choices on 152 SMs
    ((B.C4A, 64, 32, 512, 32768, 64), dict(idx_ctas_per_seq=4, launches_indexer=1, mla_splits=4, mla_head_groups=1)),
    ((B.C4A, 128, 4, 2048, 1048576, 64), dict(idx_ctas_per_seq=38, launches_indexer=2, mla_splits=8, mla_head_groups=2)),
    ((B.C4A, 64, 16, 512, 65536, 64), dict(idx_ctas_per_seq=9, launches_indexer=2, mla_splits=4, mla_head_groups=1)),
    ((B.C128A, 64, 64, 512, 131072, 64), dict(idx_ctas_per_seq=0, launches_indexer=0, mla_splits=2, mla_head_groups=1)),
    ((B.SWAONLY, 64, 16, 0, 65536, 64), dict(launches_indexer=0, mla_splits=4, launches_mla=1)),
])
def test_plan_choices_on_152_sms(args, expect):
    # indexer: floor(SMs / batch) CTAs per sequence, the top-k inside the logits
    # launch when they fit one cluster (<= 8 CTAs of <= 16 tiles), else a second
    # launch; attention: the largest cluster of 1, 2, 4 CTAs per (sequence,
    # 64-head group) that keeps every CTA on its own SM, 8 when 4 would leave
    # a CTA more than 256 keys (the 1M plan)
    import torch
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the expected choices are for 152 SMs")
    t, h, b, k, ctx, hi = args
    info = B.Plan(t, h, b, k, ctx, idx_heads=hi).info()
    for key, v in expect.items():
        assert info[key] == v, (key, info)


def test_fp4_format_and_prefill_entry_points_validate_on_the_host():
    lib = B.lib()
    p4 = B.Plan(B.C4A, 8, 2, 32, 4096, idx_heads=8)
    assert lib.dsv4_plan_set_indexer_format(p4.handle, B.IDX_FP4) == B.OK
    assert lib.dsv4_plan_set_indexer_format(p4.handle, 7) == B.ERR_INVALID
    pswa = B.Plan(B.SWAONLY, 8, 2, 0, 4096)
    assert lib.dsv4_plan_set_indexer_format(pswa.handle, B.IDX_FP4) == B.ERR_UNSUPPORTED
    # prefill attention needs the row -> sequence map
    a = B.MlaArgs()
    assert lib.dsv4_sparse_mla_prefill(p4.handle, ctypes.byref(a), None, 0, None) == B.ERR_INVALID
    # gather: unknown kind, output rows too few for offset + count
    g = B.GatherArgs(5, None, 1, None, 1, 1, None, None, 1, None, 1, 0, None)
    assert lib.dsv4_dequant_gather(ctypes.byref(g), None) == B.ERR_INVALID
    g = B.GatherArgs(B.GATHER_COMP, None, 1, None, 1, 1, None, None, 4, None, 3, 0, None)
    assert lib.dsv4_dequant_gather(ctypes.byref(g), None) == B.ERR_SHAPE
    # combine: a window of 0 is rejected; no tokens is a no-op
    c = B.CombineArgs(None, 0, None, None, None, None, None, 3, 1, 0, 0, None, 1, None, None)
    assert lib.dsv4_combine_topk_swa_indices(ctypes.byref(c), None) == B.ERR_SHAPE
    c = B.CombineArgs(None, 0, None, None, None, None, None, 0, 1, 128, 0, None, 1, None, None)
    assert lib.dsv4_combine_topk_swa_indices(ctypes.byref(c), None) == B.OK


def test_indexer_rejects_misaligned_buffers_on_the_host():
    """The indexer's cache and its workspace (the top-k bulk-copies logits rows
    out of it) must be 16-byte aligned; the call refuses before any launch."""
    lib = B.lib()
    p = B.Plan(B.C4A, 8, 1, 32, 512, idx_heads=4)
    ia = B.IndexerArgs()
    fake = 1 << 20
    for f in ("q_fp8_dev", "weights_dev", "idx_cache_dev", "block_table_dev", "ctx_len_dev", "out_idx_dev",
              "out_len_dev"):
        setattr(ia, f, fake)
    ia.num_pages, ia.bt_stride, ia.out_stride = 1, 1, 32
    ws_bytes = p.info()["workspace_bytes"]
    assert lib.dsv4_indexer_topk(p.handle, ctypes.byref(ia), ctypes.c_void_p(fake + 4), ws_bytes, None) == B.ERR_SHAPE
    ia.idx_cache_dev = fake + 8
    assert lib.dsv4_indexer_topk(p.handle, ctypes.byref(ia), ctypes.c_void_p(fake), ws_bytes, None) == B.ERR_SHAPE


def test_compress_rejects_a_misaligned_state_on_the_host():
    """The ring state is read by 16-byte bulk L2 prefetches at long windows:
    a state pointer off 16 bytes is refused before any launch."""
    lib = B.lib()
    a = B.CompressArgs()
    fake = 1 << 20
    a.kind, a.ratio, a.num_tokens, a.num_seqs, a.one_token_per_seq = B.CACHE_MLA, 128, 1, 1, 1
    for f in ("kv_score_dev", "positions_dev", "seq_dev", "ape_dev", "rms_weight_dev", "cos_sin_dev", "cache_dev",
              "block_table_dev"):
        setattr(a, f, fake)
    a.kv_score_stride, a.max_pos, a.num_pages, a.bt_stride = 2 * 576, 256, 1, 1
    a.state_dev = fake + 8
    assert lib.dsv4_compress_insert(ctypes.byref(a), None) == B.ERR_SHAPE


def test_stream_gate_validates_on_the_host():
    lib = B.lib()
    assert lib.dsv4_stream_gate(None, None) == B.ERR_INVALID
    a = B.GateArgs()
    assert lib.dsv4_stream_gate(ctypes.byref(a), None) == B.ERR_INVALID          # no flag
    a.flags_dev[1] = (1 << 20) + 2
    assert lib.dsv4_stream_gate(ctypes.byref(a), None) == B.ERR_SHAPE            # misaligned flag
    a.flags_dev[1] = 1 << 20
    a.timeout_us = -1
    assert lib.dsv4_stream_gate(ctypes.byref(a), None) == B.ERR_INVALID


def test_v4_layout_and_output_quant_validate_on_the_host():
    lib = B.lib()
    p = B.Plan(B.C4A, 8, 2, 32, 4096, idx_heads=8)
    assert lib.dsv4_plan_set_kv_layout(None, B.KV_V4) == B.ERR_INVALID
    assert lib.dsv4_plan_set_kv_layout(p.handle, 9) == B.ERR_INVALID
    assert lib.dsv4_plan_set_kv_layout(p.handle, B.KV_V4) == B.OK
    pv = B.Plan(B.SWAONLY, 8, 2, 0, 4096, kv_layout=B.KV_V4)
    assert pv.swa_page_bytes == B.V4_PAGE_BYTES == 37376 and abs(pv.geom.softmax_scale - 512 ** -0.5) < 1e-9
    # the V4 kind takes both ratios on the main stream; kind 4 does not exist
    a = B.CompressArgs()
    a.kind, a.ratio, a.num_tokens, a.num_seqs = B.CACHE_V4, 128, 0, 1
    assert lib.dsv4_compress_insert(ctypes.byref(a), None) == B.OK
    a.ratio = 8
    assert lib.dsv4_compress_insert(ctypes.byref(a), None) == B.ERR_UNSUPPORTED
    a.kind, a.ratio = 4, 4
    assert lib.dsv4_compress_insert(ctypes.byref(a), None) == B.ERR_INVALID
    m = B.CompressArgs()
    m.kind, m.ratio, m.num_tokens, m.num_seqs, m.one_token_per_seq = B.CACHE_V4, 4, 0, 1, 1
    i = B.CompressArgs()
    i.kind, i.ratio, i.num_tokens, i.num_seqs, i.one_token_per_seq = B.CACHE_IDX, 4, 0, 1, 1
    assert lib.dsv4_compress_insert_pair(ctypes.byref(m), ctypes.byref(i), None) == B.OK
    r = B.InsertRowsArgs(4, 1, None, None, None, None, 1, None, 1, 1, None)
    assert lib.dsv4_cache_insert_rows(ctypes.byref(r), None) == B.ERR_INVALID
    # output quant: NULL args, nothing to do, NULL buffers, misaligned codes
    assert lib.dsv4_inv_rope_fp8_quant(None, None) == B.ERR_INVALID
    q = B.InvRopeQuantArgs(0, 8, None, None, None, 16, None, None, None)
    assert lib.dsv4_inv_rope_fp8_quant(ctypes.byref(q), None) == B.OK
    q = B.InvRopeQuantArgs(2, 8, None, None, None, 16, None, None, None)
    assert lib.dsv4_inv_rope_fp8_quant(ctypes.byref(q), None) == B.ERR_INVALID
    q = B.InvRopeQuantArgs(2, 8, 4096, 4096, 4096, 16, 4100, 4096, None)
    assert lib.dsv4_inv_rope_fp8_quant(ctypes.byref(q), None) == B.ERR_SHAPE
    q = B.InvRopeQuantArgs(-1, 8, 4096, 4096, 4096, 16, 4096, 4096, None)
    assert lib.dsv4_inv_rope_fp8_quant(ctypes.byref(q), None) == B.ERR_INVALID
