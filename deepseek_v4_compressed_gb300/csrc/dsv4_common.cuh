// dsv4_common.cuh -- device helpers shared by the libdsv4 kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "dsv4.h"

namespace dsv4 {

constexpr int kNope = DSV4_NOPE_DIM;     // 512 latent dims
constexpr int kRope = DSV4_ROPE_DIM;     // 64 rope dims
constexpr int kHead = DSV4_HEAD_DIM;     // 576
constexpr int kV = DSV4_V_DIM;           // 512
constexpr int kIdx = DSV4_IDX_DIM;       // 128
constexpr int kPage = DSV4_PAGE;         // 64
constexpr int kMlaData = kNope + 2 * kRope;   // 640 data bytes per compressed entry
constexpr int kMlaPage = DSV4_MLA_PAGE_BYTES;
constexpr int kIdxPage = DSV4_IDX_PAGE_BYTES;
constexpr int kIdxFp4Page = DSV4_IDX_FP4_PAGE_BYTES;
constexpr int kSwaPage = DSV4_SWA_PAGE_BYTES;

__device__ __forceinline__ void flag(int* status, int bits)
{
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h)
{
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t v)
{
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// FP8 E4M3, round to nearest even, saturating to +-448 (the hardware cvt).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi)
{
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE,
                                                          __NV_E4M3));
}

// E4M3 code -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint8_t c)
{
    __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
    return __half2float(__half(hr));
}

// Power of two 2^k as an fp32, k in [-126, 127].
__device__ __forceinline__ float exp2i(int k)
{
    return __int_as_float((k + 127) << 23);
}

// UE8M0 block exponent: the smallest e with amax <= 448 * 2^e, clamped to
// [-127, 127]; 0 for an all-zero block.  448 = 0.875 * 2^9, so with
// amax = m * 2^k (m in [0.5, 1)): e = k - 9 if m <= 0.875, else k - 8.
__device__ __forceinline__ int ue8m0_exponent(float amax)
{
    if (!(amax > 0.0f)) return 0;
    int k;
    float m = frexpf(amax, &k);
    int e = (m <= 0.875f) ? k - 9 : k - 8;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// The compressor's exp: Cody-Waite reduction x = n ln2 + r (ln2 split into a
// 16-significant-bit head and an fp32 tail), e^r by its degree-7 Taylor
// series in Horner form, times 2^n.  Every step an IEEE-rounded fp32
// operation with no contraction, so it gives the same bits wherever it runs.
// x < -87 gives 0; the compressor only calls it at score - max <= 0.
__device__ __forceinline__ float cw_expf(float x)
{
    if (x < -87.0f) return 0.0f;
    if (x > 88.0f) x = 88.0f;
    const float n = rintf(__fmul_rn(x, 1.44269504088896340736f));
    float r = __fsub_rn(x, __fmul_rn(n, 0.693145751953125f));
    r = __fsub_rn(r, __fmul_rn(n, 1.42860682030941723212e-6f));
    float p = 1.0f / 5040.0f;
    p = __fadd_rn(1.0f / 720.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f / 120.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f / 24.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f / 6.0f, __fmul_rn(r, p));
    p = __fadd_rn(0.5f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f, __fmul_rn(r, p));
    p = __fadd_rn(1.0f, __fmul_rn(r, p));
    return __fmul_rn(p, exp2i(static_cast<int>(n)));
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum_d(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Order-preserving map fp32 -> uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_order_key(float x)
{
    uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace dsv4
