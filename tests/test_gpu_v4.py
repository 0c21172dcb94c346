"""GPU parity of the V4-native geometry: sparse decode attention with K = V
over 512 dims and FP8 caches of 584-byte rows (compressed and SWA) against
the oracle in double (the attention tolerances of the 576 path), and the
inverse RoPE + FP8 output quantisation bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from deepseek_v4_compressed_gb300 import binding as B
from deepseek_v4_compressed_gb300 import synth

from _util import bits_tensor, check_attention, dev, make_v4_decode_inputs, oracle_v4

pytestmark = pytest.mark.gpu


def run_v4(d, max_ctx=None, cos_sin=None, expect=B.OK):
    """The V4 attention; with cos_sin also the output quantisation (returned
    as codes, scales, the plan's cluster size)."""
    lt = d.layer_type
    plan = B.Plan(lt, d.n_heads, d.batch, d.topk if lt != B.SWAONLY else 0, int(max_ctx or d.ctx.max()),
                  idx_heads=8, kv_layout=B.KV_V4)
    ws = plan.workspace()
    out = torch.full((d.batch, d.n_heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((d.batch, d.n_heads), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = {}
    if lt != B.SWAONLY:
        kw = dict(comp_cache=d.t["comp"], comp_block_table=d.t["comp_bt"], topk_idx=d.t["idx"],
                  topk_len=d.t["idx_len"])
    codes = scales = None
    if cos_sin is not None:
        codes = torch.full((d.batch, d.n_heads, 512), 0xAA, dtype=torch.uint8, device="cuda")
        scales = torch.full((d.batch, d.n_heads, 4), -1.0, dtype=torch.float32, device="cuda")
        kw.update(out_codes=codes, out_scales=scales, cos_sin=dev(cos_sin))
    B.sparse_mla_decode(plan, d.t["q"], d.t["swa"], d.t["swa_bt"], d.t["ctx"], out, ws, lse=lse, status=status,
                        **kw)
    torch.cuda.synchronize()
    st, bits = B.read_device_status(status)
    assert st == expect, bits
    res = (out.float().cpu().numpy(), lse.cpu().numpy())
    if cos_sin is not None:
        res += (codes.cpu().numpy(), scales.cpu().numpy(), plan.info()["mla_splits"])
    return res


def check_all(d, out, lse, seqs=None):
    worst = (0.0, 0.0, 0.0)
    for b in (range(d.batch) if seqs is None else seqs):
        ref, ref_lse = oracle_v4(d, b)
        e = check_attention(out[b], ref, "seq %d" % b)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-3, atol=1e-3)
        worst = tuple(max(x, y) for x, y in zip(worst, e))
    return worst


def test_v4_tiny_ragged_c4a():
    # contexts below the window, at page edges and past several tiles
    d = make_v4_decode_inputs(4, 6, [1, 63, 64, 200, 513, 1000], 8, 32, seed=3)
    out, lse = run_v4(d)
    check_all(d, out, lse)


def test_v4_value_carries_the_rope_dims():
    """Window-only keys (swaonly): the output's dims 448..511 are the
    attention-weighted RoPE values of the keys (K = V), not zeros."""
    d = make_v4_decode_inputs(1, 3, [5, 130, 300], 16, 0, seed=4)
    out, lse = run_v4(d)
    check_all(d, out, lse)
    ref = np.stack([oracle_v4(d, b)[0] for b in range(3)])
    assert np.abs(ref[:, :, 448:]).max() > 1e-3
    assert np.abs(out[:, :, 448:]).max() > 0.5 * np.abs(ref[:, :, 448:]).max()


@pytest.mark.parametrize("peaky", [False, True])
def test_v4_c4a_32k_batch32_full_size(peaky):
    d = make_v4_decode_inputs(4, 32, 32768, 64, 512, seed=5, peaky=peaky)
    out, lse = run_v4(d)
    print("worst (max abs, mean abs, rel L2):", check_all(d, out, lse))


def test_v4_c128a_128k_batch64_full_size():
    d = make_v4_decode_inputs(128, 64, 131072, 64, 512, seed=6)
    out, lse = run_v4(d)
    check_all(d, out, lse, seqs=range(0, 64, 7))


def test_v4_swaonly_and_two_head_groups():
    d = make_v4_decode_inputs(1, 5, [1, 2, 127, 128, 4097], 128, 0, seed=7)
    out, lse = run_v4(d)
    check_all(d, out, lse)


def test_v4_c4a_1m_batch4_sampled():
    d = make_v4_decode_inputs(4, 4, 1048576, 128, 2048, seed=8, comp_pool=4096)
    out, lse = run_v4(d)
    check_all(d, out, lse)


# ---- inverse RoPE + FP8 output quantisation ---------------------------------

def run_quant(o_bits, pos, cos_sin, status=None):
    T, H, _ = o_bits.shape
    codes = torch.full((T, H, 512), 0xAA, dtype=torch.uint8, device="cuda")
    scales = torch.full((T, H, 4), -1.0, dtype=torch.float32, device="cuda")
    B.inv_rope_fp8_quant(bits_tensor(o_bits), dev(np.asarray(pos, np.int32)), dev(cos_sin), codes, scales,
                         status=status)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("T,H", [(5, 64), (1, 128), (3, 3), (32, 64)])
def test_inv_rope_quant_bit_exact(T, H):
    g = synth.rng(60 + T * H)
    o = synth.normal(g, (T, H, 512), 0.05)
    o *= (10.0 ** g.uniform(-3, 2, size=(T, H, 1))).astype(np.float32)
    o[0, 0, 128:256] = 0.0                               # an all-zero block: scale 1
    o_bits = np.stack([oracle.f32_to_bf16(o[t]) for t in range(T)])
    max_pos = 70000
    cs = oracle.rope_table(max_pos, 64)
    pos = g.integers(0, max_pos, size=T)
    pos[0] = 0
    pos[-1] = max_pos - 1
    codes, sc = run_quant(o_bits, pos, cs)
    for t in range(T):
        wc, ws = oracle.inv_rope_fp8_quant(o_bits[t], int(pos[t]), cs)
        assert np.array_equal(codes[t], wc), "token %d codes" % t
        assert np.array_equal(sc[t].view(np.uint32), ws.view(np.uint32)), "token %d scales" % t


def test_inv_rope_quant_bad_position_is_flagged():
    g = synth.rng(70)
    o_bits = oracle.f32_to_bf16(synth.normal(g, (3 * 8, 512), 0.1)).reshape(3, 8, 512)
    cs = oracle.rope_table(100, 64)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, sc = run_quant(o_bits, [5, 100, -1], cs, status=status)
    st, bits = B.read_device_status(status)
    assert st == B.ERR_DEVICE_CHECK and bits & B.DEV_BAD_POSITION
    wc, ws = oracle.inv_rope_fp8_quant(o_bits[0], 5, cs)
    assert np.array_equal(codes[0], wc) and np.array_equal(sc[0], ws)
    assert np.all(codes[1:] == 0xAA) and np.all(sc[1:] == -1.0)


def test_v4_attention_then_output_quant():
    """The two kernels in sequence: the quantised, inverse-rotated output of
    the GPU attention equals the oracle's quantisation of that same bf16
    output bit for bit, and stays within the attention tolerance (plus FP8
    rounding) of the oracle's double output rotated by R(-p)."""
    d = make_v4_decode_inputs(4, 4, [300, 1000, 4096, 77], 64, 64, seed=9)
    out, _ = run_v4(d)
    out_bits = oracle.f32_to_bf16(out.reshape(-1, 512)).reshape(out.shape)
    cs = oracle.rope_table(4096, 64)
    codes, sc = run_quant(out_bits, d.p, cs)
    for b in range(d.batch):
        wc, ws = oracle.inv_rope_fp8_quant(out_bits[b], int(d.p[b]), cs)
        assert np.array_equal(codes[b], wc) and np.array_equal(sc[b], ws)
        ref = oracle_v4(d, b)[0]
        ref_rot = oracle.inv_rope_fp8_quant(oracle.f32_to_bf16(ref.astype(np.float32)), int(d.p[b]), cs)
        deq = oracle.e4m3_to_f64(codes[b]) * np.repeat(sc[b].astype(np.float64), 128, axis=1)
        deq_ref = oracle.e4m3_to_f64(ref_rot[0]) * np.repeat(ref_rot[1].astype(np.float64), 128, axis=1)
        amax = np.abs(deq_ref).max()
        assert np.abs(deq - deq_ref).max() <= 2e-2 + 2 * 2.0 ** -4 * amax


@pytest.mark.parametrize("shape", ["tiny_ragged", "c4a_32k_b32", "c128a_128k_b64", "c4a_1m_b4"])
def test_v4_attention_with_output_quant(shape):
    """dsv4_sparse_mla_decode asked for the quantised output (the call launches
    the quantisation kernel after the attention, positions from the context
    lengths): codes and scales equal the oracle's quantisation of the kernel's
    own bf16 output bit for bit, and the attention stays within its bars."""
    if shape == "tiny_ragged":
        d = make_v4_decode_inputs(4, 6, [1, 63, 64, 200, 513, 1000], 8, 32, seed=13)
    elif shape == "c4a_32k_b32":
        d = make_v4_decode_inputs(4, 32, 32768, 64, 512, seed=14)
    elif shape == "c128a_128k_b64":
        d = make_v4_decode_inputs(128, 64, 131072, 64, 512, seed=15)
    else:
        d = make_v4_decode_inputs(4, 4, 1048576, 128, 2048, seed=16, comp_pool=4096)
    cs = oracle.rope_table(int(d.ctx.max()), 64)
    out, lse, codes, scales, C = run_v4(d, cos_sin=cs)
    seqs = range(d.batch) if d.batch <= 32 else range(0, d.batch, 7)
    check_all(d, out, lse, seqs=seqs)
    out_bits = oracle.f32_to_bf16(out.reshape(-1, 512)).reshape(out.shape)
    for b in seqs:
        wc, ws = oracle.inv_rope_fp8_quant(out_bits[b], int(d.p[b]), cs)
        assert np.array_equal(codes[b], wc), "seq %d codes" % b
        assert np.array_equal(scales[b].view(np.uint32), ws.view(np.uint32)), "seq %d scales" % b


def test_v4_output_quant_bad_position():
    """A table too short for a row's position: the row is flagged and its
    codes left unwritten; the other rows are quantised."""
    d = make_v4_decode_inputs(4, 32, [32768] * 31 + [40000], 64, 512, seed=17)
    cs = oracle.rope_table(32768, 64)
    out, lse, codes, scales, C = run_v4(d, cos_sin=cs, expect=B.ERR_DEVICE_CHECK)
    assert np.all(codes[31] == 0xAA) and np.all(scales[31] == -1.0)
    out_bits = oracle.f32_to_bf16(out.reshape(-1, 512)).reshape(out.shape)
    wc, ws = oracle.inv_rope_fp8_quant(out_bits[0], int(d.p[0]), cs)
    assert np.array_equal(codes[0], wc) and np.array_equal(scales[0], ws)
