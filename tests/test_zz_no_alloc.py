"""The allocation-free indexer entry point (dsv4_indexer_topk_noalloc), called
through the C ABI: its output must equal dsv4_indexer_topk's on the same
inputs, on two calls in a row.  Kept in a file collected last so that a run
stopping at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

from deepseek_v4_compressed_gb300 import binding as B

from _util import check_topk, make_decode_inputs, oracle_indexer

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    f = B.lib().dsv4_indexer_topk_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.POINTER(B.IndexerArgs), ctypes.c_void_p]
    return f


def _args(d, out_idx, out_len, status):
    return B.IndexerArgs(d.t["qi"].data_ptr(), d.t["w"].data_ptr(), d.t["idx"].data_ptr(),
                         d.t["idx"].numel() // B.IDX_PAGE_BYTES, d.t["idx_bt"].data_ptr(),
                         d.t["idx_bt"].shape[1], d.t["ctx"].data_ptr(), out_idx.data_ptr(),
                         out_idx.shape[1], out_len.data_ptr(), status.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice():
    ctx = np.array([32768, 20000, 7, 4099, 32768, 12345], np.int32)
    d = make_decode_inputs(4, len(ctx), ctx, 8, 64, 512, seed=61, with_comp=False)
    plan = B.Plan(B.C4A, 8, len(ctx), 512, 32768, idx_heads=64)
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    ref_idx = torch.full((len(ctx), 512), -5, dtype=torch.int32, device="cuda")
    ref_len = torch.full((len(ctx),), -5, dtype=torch.int32, device="cuda")
    ws = plan.workspace()
    rc = B.lib().dsv4_indexer_topk(plan.handle, ctypes.byref(_args(d, ref_idx, ref_len, status)),
                                   ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(stream))
    assert rc == B.OK

    f = _noalloc_fn()
    for call in range(2):
        out_idx = torch.full((len(ctx), 512), -9, dtype=torch.int32, device="cuda")
        out_len = torch.full((len(ctx),), -9, dtype=torch.int32, device="cuda")
        rc = f(plan.handle, ctypes.byref(_args(d, out_idx, out_len, status)), ctypes.c_void_p(stream))
        assert rc == B.OK, B.status_string(rc)
        torch.cuda.synchronize()
        st, bits = B.read_device_status(status)
        assert st == B.OK, bits
        got_idx, got_len = out_idx.cpu().numpy(), out_len.cpu().numpy()
        assert np.array_equal(got_len, ref_len.cpu().numpy()), call
        assert np.array_equal(got_idx, ref_idx.cpu().numpy()), call
        # and, like the workspace entry point, within the top-k rule of the oracle
        for b in range(len(ctx)):
            check_topk(got_idx[b], int(got_len[b]), oracle_indexer(d, b), 512)


def test_noalloc_rejects_plans_past_its_scratch():
    f = _noalloc_fn()
    big = B.Plan(B.C4A, 8, 64, 512, 131072, idx_heads=64)   # 64 x 32768 logits = 8 MiB
    a = B.IndexerArgs()
    rc = f(big.handle, ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == B.ERR_UNSUPPORTED


def test_noalloc_plan_at_exactly_the_scratch_size():
    """A plan whose workspace is exactly the 4 MiB of the array (batch 4 at
    context 1,048,576: 4 x 262,144 logits) is accepted and runs the separate
    long-row top-k through the array; its output equals the workspace entry
    point's, twice.  The actual contexts are short but one."""
    ctx = np.array([1048576, 5000, 70001, 3], np.int32)
    d = make_decode_inputs(4, len(ctx), ctx, 8, 64, 2048, seed=62, with_comp=False)
    plan = B.Plan(B.C4A, 8, len(ctx), 2048, 1048576, idx_heads=64)
    assert plan.workspace_bytes == 4 << 20
    assert plan.info()["launches_indexer"] == 2
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_idx = torch.full((len(ctx), 2048), -5, dtype=torch.int32, device="cuda")
    ref_len = torch.full((len(ctx),), -5, dtype=torch.int32, device="cuda")
    ws = plan.workspace()
    rc = B.lib().dsv4_indexer_topk(plan.handle, ctypes.byref(_args(d, ref_idx, ref_len, status)),
                                   ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(stream))
    assert rc == B.OK
    f = _noalloc_fn()
    for call in range(2):
        out_idx = torch.full((len(ctx), 2048), -9, dtype=torch.int32, device="cuda")
        out_len = torch.full((len(ctx),), -9, dtype=torch.int32, device="cuda")
        rc = f(plan.handle, ctypes.byref(_args(d, out_idx, out_len, status)), ctypes.c_void_p(stream))
        assert rc == B.OK, B.status_string(rc)
        torch.cuda.synchronize()
        st, bits = B.read_device_status(status)
        assert st == B.OK, bits
        assert np.array_equal(out_len.cpu().numpy(), ref_len.cpu().numpy()), call
        assert np.array_equal(out_idx.cpu().numpy(), ref_idx.cpu().numpy()), call
    got_idx, got_len = out_idx.cpu().numpy(), out_len.cpu().numpy()
    for b in range(len(ctx)):
        check_topk(got_idx[b], int(got_len[b]), oracle_indexer(d, b), 2048)
