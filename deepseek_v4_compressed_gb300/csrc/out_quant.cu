// out_quant.cu -- inverse RoPE + FP8 quantisation of the V4-native attention
// output, ahead of the FP8 output projection.
//
// Follows 6.4 of "From MLA to CSA + HCA" (K = V sharing leaves the keys'
// absolute rotation R(j) in the output; R(-i) at the query position leaves
// only R(j - i); fused_inv_rope_fp8_quant feeds the FP8 einsum) and section 6
// of the V4 internals talk write-up ("Inverse RoPE + FP8 Quant" fused so the
// rotated output is never written to HBM on its own).
//
// One warp per 128-dim block of one (token, head) row, lane l owning dims
// 4l .. 4l + 3 of the block (8 bytes in, 4 code bytes out); the last block's
// upper half holds the 64 RoPE dims.  Pure streaming work: 1024 bytes read
// and 528 written per row, bound by HBM.
#include "dsv4_common.cuh"
#include "out_quant.h"

namespace dsv4 {

constexpr int kOutDim = DSV4_V4_HEAD_DIM;          // 512
constexpr int kOutNope = DSV4_V4_NOPE_DIM;         // 448
constexpr int kOqRowsPerCta = 2;                   // 8 warps: 2 rows x 4 blocks

struct InvRopeQuantParams {
    const uint16_t* o;
    const int* pos;
    int pos_minus;                 // subtracted from pos[t]: 1 when pos holds context lengths
    const float* cos_sin;
    int max_pos;
    int n_heads;
    long long rows;
    uint8_t* codes;
    float* scales;
    int* status;
};

__global__ void __launch_bounds__(32 * 4 * kOqRowsPerCta) inv_rope_fp8_quant_kernel(InvRopeQuantParams Q)
{
    // launched under programmatic dependent launch behind the kernel that
    // writes o: the next kernel may be scheduled now, and this one waits for
    // its predecessor before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kOqRowsPerCta + (warp >> 2);
    if (row >= Q.rows) return;
    const int blk = warp & 3;
    const int t = static_cast<int>(row / Q.n_heads);
    const int pos = Q.pos[t] - Q.pos_minus;
    if (pos < 0 || pos >= Q.max_pos) {
        if (lane == 0 && blk == 0) flag(Q.status, DSV4_DEV_BAD_POSITION);
        return;
    }
    const int c = blk * 128 + 4 * lane;
    const uint2 raw = *reinterpret_cast<const uint2*>(Q.o + row * kOutDim + c);
    const float2 a = bf16x2_to_f32x2(raw.x), b = bf16x2_to_f32x2(raw.y);
    float x[4] = {a.x, a.y, b.x, b.y};
    if (c >= kOutNope) {
        // R(-pos) on the GPT-J pairs (c, c + 1) and (c + 2, c + 3)
        const float* cs = Q.cos_sin + static_cast<long long>(pos) * kRope;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = (c - kOutNope) / 2 + j;
            const float co = cs[i], sn = cs[kRope / 2 + i];
            const float x0 = x[2 * j], x1 = x[2 * j + 1];
            x[2 * j] = __fadd_rn(__fmul_rn(x0, co), __fmul_rn(x1, sn));
            x[2 * j + 1] = __fsub_rn(__fmul_rn(x1, co), __fmul_rn(x0, sn));
        }
    }
    const float amax = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
    const float s = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
    const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
    const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s));
    *reinterpret_cast<uint32_t*>(Q.codes + row * kOutDim + c) = lo | (hi << 16);
    if (lane == 0) Q.scales[row * 4 + blk] = s;
}

cudaError_t launch_inv_rope_quant(const uint16_t* o, int num_tokens, int n_heads, const int* pos, bool pos_is_ctx,
                                  const float* cos_sin, int max_pos, uint8_t* codes, float* scales, int* status,
                                  cudaStream_t stream)
{
    InvRopeQuantParams Q;
    Q.o = o;
    Q.pos = pos;
    Q.pos_minus = pos_is_ctx ? 1 : 0;
    Q.cos_sin = cos_sin;
    Q.max_pos = max_pos;
    Q.n_heads = n_heads;
    Q.rows = static_cast<long long>(num_tokens) * n_heads;
    Q.codes = codes;
    Q.scales = scales;
    Q.status = status;
    if (Q.rows == 0) return cudaSuccess;
    const long long ctas = (Q.rows + kOqRowsPerCta - 1) / kOqRowsPerCta;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(32 * 4 * kOqRowsPerCta, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, inv_rope_fp8_quant_kernel, Q);
}

}  // namespace dsv4

using namespace dsv4;

extern "C" dsv4_status dsv4_inv_rope_fp8_quant(const dsv4_inv_rope_quant_args* a, dsv4_stream_t stream)
{
    if (a == nullptr) return DSV4_ERR_INVALID;
    if (a->num_tokens < 0 || a->n_heads < 0 || a->max_pos < 0) return DSV4_ERR_INVALID;
    if (a->num_tokens == 0 || a->n_heads == 0) return DSV4_OK;
    if (!a->o_dev || !a->positions_dev || !a->cos_sin_dev || !a->codes_dev || !a->scales_dev)
        return DSV4_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(a->o_dev) & 15) || (reinterpret_cast<uintptr_t>(a->codes_dev) & 15) ||
        (reinterpret_cast<uintptr_t>(a->scales_dev) & 3))
        return DSV4_ERR_SHAPE;
    const cudaError_t e = launch_inv_rope_quant(static_cast<const uint16_t*>(a->o_dev), a->num_tokens, a->n_heads,
                                                a->positions_dev, false, a->cos_sin_dev, a->max_pos,
                                                static_cast<uint8_t*>(a->codes_dev), a->scales_dev, a->status_dev,
                                                reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return DSV4_ERR_UNSUPPORTED;
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
