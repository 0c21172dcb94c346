"""GPU parity of dsv4_sparse_mla_decode against the oracle (double): max-abs
2e-2, mean-abs 2e-3 and relative L2 1e-2 on the bf16 output."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_gb300 import binding as B

from _util import SCALE, check_attention, make_decode_inputs, synth

pytestmark = pytest.mark.gpu


def run_mla(d, idx=None, ln=None, max_ctx=None):
    lt = d.layer_type
    plan = B.Plan(lt, d.n_heads, d.batch, d.topk if lt != B.SWAONLY else 0, int(max_ctx or d.ctx.max()),
                  idx_heads=max(d.idx_heads, 1))
    ws = plan.workspace()
    out = torch.full((d.batch, d.n_heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((d.batch, d.n_heads), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = {}
    if lt != B.SWAONLY:
        kw = dict(comp_cache=d.t["comp"], comp_block_table=d.t["comp_bt"],
                  topk_idx=torch.from_numpy(idx).cuda(), topk_len=torch.from_numpy(ln).cuda())
    B.sparse_mla_decode(plan, d.t["q"], d.t["swa"], d.t["swa_bt"], d.t["ctx"], out, ws, lse=lse,
                        status=status, **kw)
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == B.OK, bits
    return out.float().cpu().numpy(), lse.cpu().numpy()


def oracle_mla(d, b, idx, ln):
    if d.layer_type == B.SWAONLY:
        return oracle.sparse_mla(d.q[b], None, None, None, 0, d.swa, d.swa_bt[b], int(d.p[b]), SCALE)
    return oracle.sparse_mla(d.q[b], d.comp, d.comp_bt[b], idx[b], int(ln[b]), d.swa, d.swa_bt[b],
                             int(d.p[b]), SCALE)


def random_indices(d, seed):
    g = synth.rng(seed)
    idx = np.full((d.batch, d.topk), -1, np.int32)
    ln = np.zeros(d.batch, np.int32)
    for b in range(d.batch):
        s = synth.sorted_sample(g, int(d.n_c[b]), d.topk)
        idx[b, :len(s)] = s
        ln[b] = len(s)
    return idx, ln


def check_batch(d, out, lse, idx, ln, seqs=None):
    worst = (0.0, 0.0, 0.0)
    for b in (range(d.batch) if seqs is None else seqs):
        ref, ref_lse, _ = oracle_mla(d, b, idx, ln)
        e = check_attention(out[b], ref, "seq %d" % b)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-3, atol=1e-3)
        worst = tuple(max(x, y) for x, y in zip(worst, e))
    return worst


def test_tiny_c4a():
    d = make_decode_inputs(4, 1, 512, 8, 4, 32, seed=0)
    idx, ln = random_indices(d, 100)
    out, lse = run_mla(d, idx, ln)
    check_batch(d, out, lse, idx, ln)


@pytest.mark.parametrize("peaky", [False, True])
def test_c4a_32k_batch32_full_size(peaky):
    d = make_decode_inputs(4, 32, 32768, 64, 0, 512, seed=1, peaky=peaky)
    idx, ln = random_indices(d, 101)
    out, lse = run_mla(d, idx, ln)
    print("worst (max abs, mean abs, rel L2):", check_batch(d, out, lse, idx, ln))


def test_c128a_128k_batch64_full_size():
    d = make_decode_inputs(128, 64, 131072, 64, 0, 512, seed=2)
    out, lse = run_mla(d, d.meta_idx, d.meta_len)
    check_batch(d, out, lse, d.meta_idx, d.meta_len)


def test_long_c4a_1m_heads128():
    d = make_decode_inputs(4, 4, 1048576, 128, 0, 2048, seed=4, comp_pool=4096)
    idx, ln = random_indices(d, 104)
    out, lse = run_mla(d, idx, ln)
    check_batch(d, out, lse, idx, ln)


def test_swaonly_and_short_windows():
    ctx = np.array([1, 70, 128, 129, 5000], np.int32)
    d = make_decode_inputs(1, len(ctx), ctx, 16, 0, 0, seed=5)
    out, lse = run_mla(d)
    check_batch(d, out, lse, None, None)


def test_ragged_lengths_and_padding():
    ctx = np.array([4, 40, 600, 2000, 3000], np.int32)   # n_c = 1, 10, 150, 500, 750 with k = 256
    d = make_decode_inputs(4, len(ctx), ctx, 24, 0, 256, seed=6)
    idx, ln = random_indices(d, 106)
    ln[4] = 100                                          # a shorter list than the row
    idx[4, 100:] = -1
    out, lse = run_mla(d, idx, ln)
    check_batch(d, out, lse, idx, ln)


def test_zero_output_fails_the_tolerance():
    d = make_decode_inputs(4, 2, 4096, 64, 0, 128, seed=7)
    idx, ln = random_indices(d, 107)
    out, _ = run_mla(d, idx, ln)
    ref, _, _ = oracle_mla(d, 0, idx, ln)
    check_attention(out[0], ref)
    with pytest.raises(AssertionError):
        check_attention(np.zeros_like(out[0]), ref)


def test_key_dequant_every_code_and_scale():
    """The decode kernel's key conversion (E4M3 code x 2^(s-127) -> bf16) for all
    256 codes and 256 scale bytes: bit-exact against the oracle's decode of the
    two formats wherever the result is a normal bf16, zero or infinite; results
    below the bf16 normal range only need the right sign and a magnitude below
    2^-126.  The two NaN codes are never written and are left out."""
    out = torch.zeros(65536, dtype=torch.int16, device="cuda")
    B.selftest_key_dequant(out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16).reshape(256, 256)
    vals = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    nan = np.isnan(vals)            # 0x7f / 0xff: never written (the quantiser saturates)
    assert nan.sum() == 2
    vals = np.where(nan, 0.0, vals)
    for s in range(256):
        v = vals * (2.0 ** (s - 127))
        small = ((v != 0) & (np.abs(v) < 2.0 ** -126)) | nan
        with np.errstate(over="ignore"):
            exp = oracle.f32_to_bf16(v.astype(np.float32))
        ok = (got[s] == exp) | small
        assert ok.all(), (s, np.nonzero(~ok)[0][:8], got[s][~ok][:8], exp[~ok][:8])
        tiny = small & ~nan
        if tiny.any():
            g = oracle.bf16_to_f32(got[s][tiny])
            assert np.all(np.abs(g) < 2.0 ** -126)
            assert np.all((np.signbit(g) == np.signbit(v[tiny])) | (g == 0))


def test_partial_second_head_group():
    # 96 heads: a full 64-head group and a 32-head one (rows past the heads
    # computed but never stored), ragged contexts
    ctx = np.array([5000, 130, 20000], np.int32)
    d = make_decode_inputs(4, len(ctx), ctx, 96, 0, 512, seed=8)
    idx, ln = random_indices(d, 108)
    out, lse = run_mla(d, idx, ln)
    check_batch(d, out, lse, idx, ln)
