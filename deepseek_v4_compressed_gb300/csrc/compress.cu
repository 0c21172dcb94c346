// compress.cu -- token-level Compressor -> RMSNorm -> RoPE -> FP8 -> paged insert.
//
// Follows DeepseekCompressor.forward / save_partial_states and "CSA layer
// Compressor" of the "DeepseekV4Attention" class walkthrough, "Compressor:
// ratio 4 vs 128" of "DeepSeek V4 attention in vLLM", and sections 5.1, 5.2,
// 6.3 of "From MLA to CSA + HCA".
//
// One CTA per token (ratio 128: a cluster, below), d/2 threads, thread i owns
// channels 2i and 2i+1
// (main cache d = 576: 288 threads = 9 warps, warp w < 8 owns nope block w of
// 64 dims, warp 8 the rope dims; V4-native main cache d = 512: 8 warps, warps
// 0-6 the 448 nope dims, warp 7 the rope dims; indexer d = 128: 64 threads).  The per-token
// state row is [kv block 0..coff-1 | score block 0..coff-1] in fp32; the
// window of a boundary token is read from the per-sequence ring (and, in a
// multi-token call, from this call's own inputs).  Work per entry is tiny and
// bound by the state reads; it runs on the CUDA cores, no contraction.
//
// Ratio 128 (the single-stream compressor of c128a layers): a boundary pools
// 128 ring rows, which one CTA per token reads only as fast as its one SM
// pulls them from L2.  There a token takes a cluster of G CTAs (3 for d = 576,
// 4 for d = 512), each owning whole 64-channel warps of the d/2 threads; the
// RMSNorm warp totals go to every CTA of the cluster and are added in the
// same ascending warp order, so the bytes are those of one CTA.
#include "dsv4_common.cuh"
#include "tc_common.cuh"
#include "tmap.h"

namespace dsv4 {

struct CompressParams {
    const uint16_t* kv_score;
    long long kv_stride;
    const int* positions;
    const int* seqs;
    const float* ape;
    const float* rms_w;
    float eps;
    const float* cos_sin;
    int max_pos;
    float* state;
    uint8_t* cache;
    int num_pages;
    const int* bt;
    int bt_stride;
    int num_tokens;
    int num_seqs;
    int* status;
};

// Per-block double reduction of the RMSNorm sum of squares, in the fixed
// association that defines the mean square: each thread's pair (channels 2i,
// 2i + 1) summed first, a butterfly over the 32 lanes of each warp (= one
// 64-channel group; at distance 16, 8, 4, 2, 1 lane l adds lane l ^ distance),
// then the warps' totals added to 0 in ascending warp order.  Double addition
// is commutative, so every lane of a warp holds the same total, and the
// result is the same bits wherever the order is followed.
// NWT warps in all, NWC of them in this CTA (rank `rank` of a cluster of G
// CTAs, global warp rank * NWC + local warp); with G > 1 each warp's total
// is stored into every CTA of the cluster before a cluster barrier.
template <int NWT, int NWC, int G>
__device__ __forceinline__ double block_sum_d(double v, double* red, int rank)
{
    v = warp_sum_d(v);
    const int gw = rank * NWC + static_cast<int>(threadIdx.x >> 5);
    if ((threadIdx.x & 31) == 0) {
        if constexpr (G == 1) {
            red[gw] = v;
        } else {
            const uint32_t a = tc::smem_u32(&red[gw]);
#pragma unroll
            for (int q = 0; q < G; ++q)
                asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(tc::map_to_rank(a, q)), "d"(v) : "memory");
        }
    }
    if constexpr (G == 1)
        __syncthreads();
    else
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    double s = 0.0;
#pragma unroll
    for (int i = 0; i < NWT; ++i) s += red[i];
    return s;
}

// CTAs per token of the compress kernel: the ratio-128 main streams split
// their 64-channel warps over a cluster (see the top of this file).
__host__ __device__ constexpr int compress_split(int D, int RATIO)
{
    return RATIO != 128 ? 1 : (D == 576 ? 3 : (D == 512 ? 4 : 1));
}

// Quantise the normalised, rotated vector (this thread's channels c0, c0+1)
// into a main-cache entry: E4M3 nope with one UE8M0 byte per 64 dims, bf16
// rope; with 448 nope dims the eighth scale byte is a zero pad.  Called by
// the (NOPE + 64) / 2 threads of the entry (one CTA, or the CTAs of a
// cluster): the 64-channel block and the lane follow from c0.
template <int NOPE>
__device__ __forceinline__ void store_mla_entry(float z0, float z1, int c0, uint8_t* data_row,
                                                uint8_t* scale_row)
{
    const int warp = c0 >> 6, lane = (c0 >> 1) & 31;
    if (NOPE < 512 && warp == NOPE / 64 && lane == 0) scale_row[7] = 0;
    if (warp < NOPE / 64) {
        const float amax = warp_max(fmaxf(fabsf(z0), fabsf(z1)));
        const int e = ue8m0_exponent(amax);
        const float mult = exp2i(-e);
        const uint16_t codes = f32x2_to_e4m3x2(__fmul_rn(z0, mult), __fmul_rn(z1, mult));
        *reinterpret_cast<uint16_t*>(data_row + c0) = codes;
        if (lane == 0) scale_row[warp] = static_cast<uint8_t>(e + 127);
    } else {
        const uint32_t pk = static_cast<uint32_t>(f32_to_bf16_bits(z0)) |
                            (static_cast<uint32_t>(f32_to_bf16_bits(z1)) << 16);
        *reinterpret_cast<uint32_t*>(data_row + NOPE + 2 * (c0 - NOPE)) = pk;
    }
}

constexpr int kV4Nope = DSV4_V4_NOPE_DIM;                 // 448
constexpr int kV4Data = kV4Nope + 2 * kRope;              // 576 data bytes per V4 row

// Model dimension of a cache kind's stream.
template <int KIND>
constexpr int kind_dim()
{
    return KIND == DSV4_CACHE_MLA ? kHead : (KIND == DSV4_CACHE_V4 ? DSV4_V4_HEAD_DIM : kIdx);
}

// Indexer entry: E4M3 of all 128 dims, one fp32 scale = amax / 448.
// Called by all 64 threads.
__device__ __forceinline__ void store_idx_entry(float z0, float z1, int c0, uint8_t* data_row,
                                                float* scale_ptr, float* red)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float amax = warp_max(fmaxf(fabsf(z0), fabsf(z1)));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = fmaxf(red[0], red[1]);
    const float s = (amax > 0.0f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
    const uint16_t codes = f32x2_to_e4m3x2(__fdiv_rn(z0, s), __fdiv_rn(z1, s));
    *reinterpret_cast<uint16_t*>(data_row + c0) = codes;
    if (threadIdx.x == 0) *scale_ptr = s;
}

// E2M1 code of v (FP4: 1 sign, 2 exponent, 1 mantissa bit): the nearest of
// 0, 0.5, 1, 1.5, 2, 3, 4, 6, ties to the even code, saturating at 6 (NaN
// gives the largest code).  Written out as the comparisons that rule implies.
__device__ __forceinline__ uint32_t f32_to_e2m1(float v)
{
    const float a = fabsf(v);
    uint32_t c;
    if (a <= 0.25f) c = 0;
    else if (a < 0.75f) c = 1;
    else if (a <= 1.25f) c = 2;
    else if (a < 1.75f) c = 3;
    else if (a <= 2.5f) c = 4;
    else if (a < 3.5f) c = 5;
    else if (a <= 5.0f) c = 6;
    else c = 7;
    return c | ((__float_as_uint(v) >> 31) << 3);
}

// FP4 indexer entry (MXFP4): blocks of 32 dims, each with a UE8M0 exponent e
// = the smallest with amax <= 6 * 2^e (6 = 0.75 * 2^3: with amax = m * 2^k,
// m in [0.5, 1), e = k - 3 if m <= 0.75, else k - 2), clamped to [-127, 127],
// 0 for an all-zero block; codes E2M1(z * 2^-e), two per byte (the low nibble
// the even dim).  Called by all 64 threads (16 threads per block).
__device__ __forceinline__ void store_idx_fp4_entry(float z0, float z1, int c0, uint8_t* data_row,
                                                    uint8_t* scale_row)
{
    float amax = fmaxf(fabsf(z0), fabsf(z1));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = 0;
    if (amax > 0.0f) {
        int k;
        const float m = frexpf(amax, &k);
        e = (m <= 0.75f) ? k - 3 : k - 2;
        e = e < -127 ? -127 : (e > 127 ? 127 : e);
    }
    // -e lies in [-126, 127] for every finite amax, so 2^-e is a normal fp32
    const float mult = exp2i(-e);
    const uint32_t lo = f32_to_e2m1(__fmul_rn(z0, mult)), hi = f32_to_e2m1(__fmul_rn(z1, mult));
    data_row[c0 >> 1] = static_cast<uint8_t>(lo | (hi << 4));
    if ((threadIdx.x & 15) == 0) scale_row[c0 >> 5] = static_cast<uint8_t>(e + 127);
}

// Bring [p, p + bytes) into L2 without waiting (p 16-byte aligned, bytes a
// multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes)
{
    asm volatile("{\n\t.reg .u64 g;\n\tcvta.to.global.u64 g, %0;\n\t"
                 "cp.async.bulk.prefetch.L2.global [g], %1;\n\t}" ::"l"(p), "r"(bytes)
                 : "memory");
}

// Resolve the page of logical slot j of sequence seq; nullptr (and a status
// bit) when the table entry is out of range.
template <int KIND>
__device__ __forceinline__ uint8_t* entry_page(const CompressParams& P, int seq, int j)
{
    const int pi = j / kPage;
    if (pi >= P.bt_stride) {
        flag(P.status, DSV4_DEV_BAD_PAGE);
        return nullptr;
    }
    const int pg = P.bt[static_cast<long long>(seq) * P.bt_stride + pi];
    if (pg < 0 || pg >= P.num_pages) {
        flag(P.status, DSV4_DEV_BAD_PAGE);
        return nullptr;
    }
    return P.cache + static_cast<long long>(pg) *
                         (KIND == DSV4_CACHE_MLA ? kMlaPage
                          : (KIND == DSV4_CACHE_V4 ? DSV4_V4_PAGE_BYTES
                             : (KIND == DSV4_CACHE_IDX ? kIdxPage : kIdxFp4Page)));
}

// The state values (kv, score + ape) of one token for this thread's two
// channels of block blk, straight from the projection input.
template <int D, int COFF>
__device__ __forceinline__ void token_values(const CompressParams& P, int t, int pos, int blk,
                                             int c0, float2& kv, float2& sc, int ratio)
{
    const uint16_t* row = P.kv_score + static_cast<long long>(t) * P.kv_stride;
    kv = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(row + blk * D + c0));
    const float2 s = bf16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(row + COFF * D + blk * D + c0));
    const float2 a = *reinterpret_cast<const float2*>(
        P.ape + static_cast<long long>(pos % ratio) * COFF * D + blk * D + c0);
    sc = make_float2(__fadd_rn(s.x, a.x), __fadd_rn(s.y, a.y));
}

// Compress kernel.  FUSED: each sequence has at most one token in the call;
// the token's state row is written here too.  Otherwise (multi-token calls)
// window rows inside the call come from the inputs and the ring is written
// by state_write_kernel afterwards.  G CTAs per token (a cluster; this one is
// rank `rank`, owning channels [rank d/G, (rank + 1) d/G)).
template <int D, int RATIO, int KIND, bool FUSED, int G = 1>
__device__ __forceinline__ void compress_token(const CompressParams& P, const int t, const int rank = 0)
{
    constexpr bool IDX = KIND == DSV4_CACHE_IDX || KIND == DSV4_CACHE_IDX_FP4;
    constexpr int COFF = (RATIO == 4) ? 2 : 1;
    constexpr int W = COFF * RATIO;
    constexpr int ROW = 2 * COFF * D;
    constexpr int NT = D / 2 / G;                      // threads of this CTA
    constexpr int NOPE = D - kRope;
    static_assert(D == kind_dim<KIND>(), "stream dimension of the cache kind");
    static_assert(NT % 32 == 0 && (G == 1 || !IDX), "a CTA owns whole 64-channel warps");
    __shared__ double red_d[D / 64];
    __shared__ float red_f[2];

    const int c0 = 2 * (static_cast<int>(threadIdx.x) + rank * NT);
    const int seq = P.seqs[t];
    const int p = P.positions[t];
    if (seq < 0 || seq >= P.num_seqs || p < 0) {
        if (threadIdx.x == 0) flag(P.status, DSV4_DEV_BAD_INDEX);
        return;
    }
    if (!FUSED && t > 0 && P.seqs[t - 1] == seq && P.positions[t - 1] != p - 1) {
        if (threadIdx.x == 0) flag(P.status, DSV4_DEV_BAD_POSITION);
        return;
    }
    float* ring = P.state + static_cast<long long>(seq) * W * ROW;

    // This token's own values (block coff-1 is the "new" block of a window).
    float2 own_kv[COFF], own_sc[COFF];
#pragma unroll
    for (int b = 0; b < COFF; ++b) token_values<D, COFF>(P, t, p, b, c0, own_kv[b], own_sc[b], RATIO);

    if (FUSED) {
        float* dst = ring + static_cast<long long>(p % W) * ROW;
#pragma unroll
        for (int b = 0; b < COFF; ++b) {
            *reinterpret_cast<float2*>(dst + b * D + c0) = own_kv[b];
            *reinterpret_cast<float2*>(dst + COFF * D + b * D + c0) = own_sc[b];
        }
    }
    if ((p + 1) % RATIO != 0) return;

    // Window rows s = p-W+1 .. p (s >= 0); block 0 for the old group of a
    // ratio-4 window (s <= p - 4), the last block otherwise.
    auto fetch = [&](int s, float2& kv, float2& sc) {
        const int blk = (COFF == 2 && s <= p - RATIO) ? 0 : COFF - 1;
        if (s == p) {
            kv = own_kv[COFF - 1];
            sc = own_sc[COFF - 1];
            return;
        }
        if (!FUSED) {
            const int ts = t - (p - s);
            if (ts >= 0 && P.seqs[ts] == seq && P.positions[ts] == s) {
                token_values<D, COFF>(P, ts, s, blk, c0, kv, sc, RATIO);
                return;
            }
        }
        const float* src = ring + static_cast<long long>(s % W) * ROW;
        kv = *reinterpret_cast<const float2*>(src + blk * D + c0);
        sc = *reinterpret_cast<const float2*>(src + COFF * D + blk * D + c0);
    };
    // Rows are fetched CH at a time (every load of a chunk in flight before
    // its values are used); the arithmetic and its order are the plain
    // two-pass ones: max, then sums in ascending s.
    constexpr int CH = W < 12 ? W : 12;
    const int s0 = (p - W + 1) < 0 ? 0 : p - W + 1;
    if constexpr (W >= 64) {
        // a long window: all of its ring rows into L2 at once (one bulk
        // prefetch per row, the rows dealt round-robin over the cluster), so
        // the two passes' chunks wait on L2, not HBM
        for (int s = s0 + rank + G * static_cast<int>(threadIdx.x); s < p; s += G * NT)
            prefetch_l2_bulk(ring + static_cast<long long>(s % W) * ROW, static_cast<uint32_t>(ROW * sizeof(float)));
    }
    float m0 = -INFINITY, m1 = -INFINITY;
    for (int sb = s0; sb <= p; sb += CH) {
        float2 kv[CH], sc[CH];
#pragma unroll
        for (int u = 0; u < CH; ++u)
            if (sb + u <= p) fetch(sb + u, kv[u], sc[u]);
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            if (sb + u <= p) {
                m0 = fmaxf(m0, sc[u].x);
                m1 = fmaxf(m1, sc[u].y);
            }
        }
    }
    float n0 = 0.f, n1 = 0.f, d0 = 0.f, d1 = 0.f;
    for (int sb = s0; sb <= p; sb += CH) {
        float2 kv[CH], sc[CH];
#pragma unroll
        for (int u = 0; u < CH; ++u)
            if (sb + u <= p) fetch(sb + u, kv[u], sc[u]);
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            if (sb + u <= p) {
                const float e0 = cw_expf(__fsub_rn(sc[u].x, m0));
                const float e1 = cw_expf(__fsub_rn(sc[u].y, m1));
                n0 = __fadd_rn(n0, __fmul_rn(e0, kv[u].x));
                n1 = __fadd_rn(n1, __fmul_rn(e1, kv[u].y));
                d0 = __fadd_rn(d0, e0);
                d1 = __fadd_rn(d1, e1);
            }
        }
    }
    const float y0 = __fdiv_rn(n0, d0), y1 = __fdiv_rn(n1, d1);

    // RMSNorm: mean square accumulated in double in the fixed order, rounded once.
    const double ss =
        block_sum_d<D / 64, NT / 32, G>(static_cast<double>(y0) * y0 + static_cast<double>(y1) * y1, red_d, rank);
    const float ms = __double2float_rn(ss / static_cast<double>(D));
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, P.eps)));
    const float2 w = *reinterpret_cast<const float2*>(P.rms_w + c0);
    float z0 = __fmul_rn(__fmul_rn(y0, inv), w.x);
    float z1 = __fmul_rn(__fmul_rn(y1, inv), w.y);

    // GPT-J RoPE on the last 64 dims at the slot's anchor position.
    if (c0 >= NOPE) {
        const int rp = (p / RATIO) * RATIO;
        const int pair = (c0 - NOPE) >> 1;
        if (rp < P.max_pos) {
            const float cs = P.cos_sin[static_cast<long long>(rp) * kRope + pair];
            const float sn = P.cos_sin[static_cast<long long>(rp) * kRope + kRope / 2 + pair];
            const float r0 = __fsub_rn(__fmul_rn(z0, cs), __fmul_rn(z1, sn));
            const float r1 = __fadd_rn(__fmul_rn(z0, sn), __fmul_rn(z1, cs));
            z0 = r0;
            z1 = r1;
        } else {
            flag(P.status, DSV4_DEV_BAD_POSITION);
        }
    }

    const int j = p / RATIO;
    uint8_t* page = entry_page<KIND>(P, seq, j);
    const int r = j % kPage;
    if (KIND == DSV4_CACHE_IDX_FP4) {
        if (page == nullptr) return;   // uniform across the CTA
        store_idx_fp4_entry(z0, z1, c0, page + r * (kIdx / 2), page + kPage * (kIdx / 2) + r * (kIdx / 32));
    } else if (IDX) {
        if (page == nullptr) return;   // uniform across the CTA
        store_idx_entry(z0, z1, c0, page + r * kIdx,
                        reinterpret_cast<float*>(page + kPage * kIdx) + r, red_f);
    } else if (KIND == DSV4_CACHE_V4) {
        if (page == nullptr) return;
        store_mla_entry<kV4Nope>(z0, z1, c0, page + r * kV4Data, page + kPage * kV4Data + r * 8);
    } else {
        if (page == nullptr) return;
        store_mla_entry<kNope>(z0, z1, c0, page + r * kMlaData, page + kPage * kMlaData + r * 8);
    }
}

// Multi-token calls: write the ring rows of the last W tokens of every
// sequence (earlier tokens of the call are never read again).
// A dependent kernel launched behind this one (programmatic dependent
// launch) may be scheduled at once; it waits for this grid before reading
// what it writes.
template <int D, int RATIO, int KIND, bool FUSED>
__global__ void __launch_bounds__(D / 2 / compress_split(D, RATIO)) compress_kernel(CompressParams P)
{
    constexpr int G = compress_split(D, RATIO);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // launched behind the previous kernel of the stream (clusters: under
    // programmatic dependent launch): touch nothing before it has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // G > 1: clusters of G consecutive blocks, one token each
    compress_token<D, RATIO, KIND, FUSED, G>(P, static_cast<int>(blockIdx.x) / G, static_cast<int>(blockIdx.x) % G);
}

// The main (d = 576, or 512 for the V4 row) and indexer (d = 128) streams of
// a layer in one launch, one token per sequence: blocks [0, main tokens) take
// the main entries, the rest the indexer entries with their first 64 threads.
template <int RATIO, int IDX_KIND, int MAIN_KIND>
__global__ void __launch_bounds__(kind_dim<MAIN_KIND>() / 2) compress_pair_kernel(CompressParams Pm,
                                                                                 CompressParams Pi)
{
    // the indexer of this layer, launched next, starts by reading the
    // sequence's indexer block-table row (a caller input): warm it in L2
    if (static_cast<int>(blockIdx.x) >= Pm.num_tokens && threadIdx.x < 32) {
        const int t = blockIdx.x - Pm.num_tokens;
        const int b = t < Pi.num_tokens ? __ldg(Pi.seqs + t) : -1;
        if (b >= 0 && b < Pi.num_seqs && static_cast<int>(threadIdx.x) * 32 < Pi.bt_stride)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(Pi.bt + static_cast<long long>(b) * Pi.bt_stride +
                                                          threadIdx.x * 32));
    }
    // The indexer launched next may be scheduled at once: it reads only
    // caller inputs and its cache's older slots before its own dependency
    // wait, and this kernel writes at most the newest entry of each sequence.
    // The kernel before this one may still be running: when it is the
    // library's attention, it let this kernel launch only after every one of
    // its CTAs had read its index rows and gathered its keys, and it writes
    // nothing the indexer reads (its output and lse), so the indexer's
    // writes (indices, logits) cannot race with it.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // launched behind the previous kernel of the stream (programmatic
    // dependent launch): its outputs may be this kernel's inputs
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (static_cast<int>(blockIdx.x) < Pm.num_tokens)
        compress_token<kind_dim<MAIN_KIND>(), RATIO, MAIN_KIND, true>(Pm, blockIdx.x);
    else if (threadIdx.x < kIdx / 2)
        compress_token<kIdx, 4, IDX_KIND, true>(Pi, blockIdx.x - Pm.num_tokens);
}

template <int D, int RATIO>
__global__ void __launch_bounds__(D / 2) state_write_kernel(CompressParams P)
{
    constexpr int COFF = (RATIO == 4) ? 2 : 1;
    constexpr int W = COFF * RATIO;
    constexpr int ROW = 2 * COFF * D;
    const int t = blockIdx.x;
    const int c0 = 2 * threadIdx.x;
    const int seq = P.seqs[t];
    const int p = P.positions[t];
    if (seq < 0 || seq >= P.num_seqs || p < 0) return;
    if (t + W < P.num_tokens && P.seqs[t + W] == seq) return;   // superseded in this call
    float* dst = P.state + (static_cast<long long>(seq) * W + p % W) * ROW;
#pragma unroll
    for (int b = 0; b < COFF; ++b) {
        float2 kv, sc;
        token_values<D, COFF>(P, t, p, b, c0, kv, sc, RATIO);
        *reinterpret_cast<float2*>(dst + b * D + c0) = kv;
        *reinterpret_cast<float2*>(dst + COFF * D + b * D + c0) = sc;
    }
}

// Quantise-and-insert of given fp32 rows (no pooling / norm / rope).
template <int D, int KIND>
__global__ void __launch_bounds__(D / 2) insert_rows_kernel(const float* rows, const int* seqs,
                                                            const int* slots, CompressParams P)
{
    __shared__ float red_f[2];
    const int i = blockIdx.x;
    const int c0 = 2 * threadIdx.x;
    const int seq = seqs[i], j = slots[i];
    if (seq < 0 || seq >= P.num_seqs || j < 0) {
        if (threadIdx.x == 0) flag(P.status, DSV4_DEV_BAD_INDEX);
        return;
    }
    const float2 z = *reinterpret_cast<const float2*>(rows + static_cast<long long>(i) * D + c0);
    uint8_t* page = entry_page<KIND>(P, seq, j);
    if (page == nullptr) return;
    const int r = j % kPage;
    if (KIND == DSV4_CACHE_IDX_FP4)
        store_idx_fp4_entry(z.x, z.y, c0, page + r * (kIdx / 2), page + kPage * (kIdx / 2) + r * (kIdx / 32));
    else if (KIND == DSV4_CACHE_IDX)
        store_idx_entry(z.x, z.y, c0, page + r * kIdx,
                        reinterpret_cast<float*>(page + kPage * kIdx) + r, red_f);
    else if (KIND == DSV4_CACHE_V4)
        store_mla_entry<kV4Nope>(z.x, z.y, c0, page + r * kV4Data, page + kPage * kV4Data + r * 8);
    else
        store_mla_entry<kNope>(z.x, z.y, c0, page + r * kMlaData, page + kPage * kMlaData + r * 8);
}

template <int D, int RATIO, int KIND, bool FUSED>
static cudaError_t launch_compress_kernel(const CompressParams& P, cudaStream_t st)
{
    constexpr int G = compress_split(D, RATIO);
    if (G == 1) {
        compress_kernel<D, RATIO, KIND, FUSED><<<P.num_tokens, D / 2, 0, st>>>(P);
        return cudaGetLastError();
    }
    if (static_cast<long long>(P.num_tokens) * G > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(P.num_tokens * G), 1, 1);
    cfg.blockDim = dim3(D / 2 / G, 1, 1);
    cfg.stream = st;
    // the small CTAs (d/2/G threads) fit beside an attention CTA, so when the
    // grid is at most one CTA per SM they launch while the previous attention
    // finishes (programmatic dependent launch; the kernel waits for it before
    // touching memory).  A larger grid keeps the plain launch: at 64 tokens
    // (192 CTAs) the early launch made a C128A 128K batch-64 step 1.1 us
    // slower, at 16 tokens it made the c128a layers 5% faster.
    const bool early = static_cast<long long>(P.num_tokens) * G <= sm_count();
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, compress_kernel<D, RATIO, KIND, FUSED>, P);
}

template <int D, int RATIO, int KIND>
static cudaError_t launch_compress(const CompressParams& P, bool fused, cudaStream_t st)
{
    if (P.num_tokens == 0) return cudaSuccess;
    if (fused) return launch_compress_kernel<D, RATIO, KIND, true>(P, st);
    cudaError_t e = launch_compress_kernel<D, RATIO, KIND, false>(P, st);
    if (e != cudaSuccess) return e;
    state_write_kernel<D, RATIO><<<P.num_tokens, D / 2, 0, st>>>(P);
    return cudaGetLastError();
}

}  // namespace dsv4

using namespace dsv4;

// Validate a call's arguments and fill the kernel parameters.
static dsv4_status compress_params(const dsv4_compress_args* a, CompressParams& P)
{
    if (a == nullptr) return DSV4_ERR_INVALID;
    if (a->num_tokens < 0 || a->num_seqs < 0 || a->bt_stride < 0 || a->num_pages < 0)
        return DSV4_ERR_INVALID;
    if (a->kind != DSV4_CACHE_MLA && a->kind != DSV4_CACHE_IDX && a->kind != DSV4_CACHE_IDX_FP4 &&
        a->kind != DSV4_CACHE_V4)
        return DSV4_ERR_INVALID;
    const bool main_kind = a->kind == DSV4_CACHE_MLA || a->kind == DSV4_CACHE_V4;
    if (a->ratio != 4 && a->ratio != 128) return DSV4_ERR_UNSUPPORTED;
    if (!main_kind && a->ratio != 4) return DSV4_ERR_UNSUPPORTED;
    if (a->num_tokens > 0 &&
        (!a->kv_score_dev || !a->positions_dev || !a->seq_dev || !a->ape_dev || !a->rms_weight_dev ||
         !a->cos_sin_dev || !a->state_dev || !a->cache_dev || !a->block_table_dev))
        return DSV4_ERR_INVALID;
    const int d = a->kind == DSV4_CACHE_MLA ? kHead : (a->kind == DSV4_CACHE_V4 ? DSV4_V4_HEAD_DIM : kIdx);
    const int coff = (a->ratio == 4) ? 2 : 1;
    if (a->num_tokens > 0 && (a->kv_score_stride < 2LL * coff * d || (a->kv_score_stride & 1)))
        return DSV4_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(a->kv_score_dev) & 3) || (reinterpret_cast<uintptr_t>(a->cache_dev) & 15) ||
        (reinterpret_cast<uintptr_t>(a->state_dev) & 15))
        return DSV4_ERR_SHAPE;
    P.kv_score = static_cast<const uint16_t*>(a->kv_score_dev);
    P.kv_stride = a->kv_score_stride;
    P.positions = a->positions_dev;
    P.seqs = a->seq_dev;
    P.ape = a->ape_dev;
    P.rms_w = a->rms_weight_dev;
    P.eps = a->rms_eps;
    P.cos_sin = a->cos_sin_dev;
    P.max_pos = a->max_pos;
    P.state = a->state_dev;
    P.cache = static_cast<uint8_t*>(a->cache_dev);
    P.num_pages = a->num_pages;
    P.bt = a->block_table_dev;
    P.bt_stride = a->bt_stride;
    P.num_tokens = a->num_tokens;
    P.num_seqs = a->num_seqs;
    P.status = a->status_dev;
    return DSV4_OK;
}

extern "C" dsv4_status dsv4_compress_insert(const dsv4_compress_args* a, dsv4_stream_t stream)
{
    CompressParams P;
    const dsv4_status s = compress_params(a, P);
    if (s != DSV4_OK) return s;
    if (a->num_tokens == 0) return DSV4_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool fused = a->one_token_per_seq != 0;
    cudaError_t e;
    if (a->kind == DSV4_CACHE_IDX)
        e = launch_compress<kIdx, 4, DSV4_CACHE_IDX>(P, fused, st);
    else if (a->kind == DSV4_CACHE_IDX_FP4)
        e = launch_compress<kIdx, 4, DSV4_CACHE_IDX_FP4>(P, fused, st);
    else if (a->kind == DSV4_CACHE_V4)
        e = a->ratio == 4 ? launch_compress<DSV4_V4_HEAD_DIM, 4, DSV4_CACHE_V4>(P, fused, st)
                          : launch_compress<DSV4_V4_HEAD_DIM, 128, DSV4_CACHE_V4>(P, fused, st);
    else if (a->ratio == 4)
        e = launch_compress<kHead, 4, DSV4_CACHE_MLA>(P, fused, st);
    else
        e = launch_compress<kHead, 128, DSV4_CACHE_MLA>(P, fused, st);
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

extern "C" dsv4_status dsv4_compress_insert_pair(const dsv4_compress_args* main_args,
                                                 const dsv4_compress_args* idx_args, dsv4_stream_t stream)
{
    CompressParams Pm, Pi;
    dsv4_status s = compress_params(main_args, Pm);
    if (s != DSV4_OK) return s;
    s = compress_params(idx_args, Pi);
    if (s != DSV4_OK) return s;
    if ((main_args->kind != DSV4_CACHE_MLA && main_args->kind != DSV4_CACHE_V4) ||
        (idx_args->kind != DSV4_CACHE_IDX && idx_args->kind != DSV4_CACHE_IDX_FP4))
        return DSV4_ERR_INVALID;
    if (!main_args->one_token_per_seq || !idx_args->one_token_per_seq) return DSV4_ERR_INVALID;
    const int n = Pm.num_tokens + Pi.num_tokens;
    if (n == 0) return DSV4_OK;
    // programmatic dependent launch: the CTAs may be scheduled while the
    // previous kernel drains; they wait for it before reading anything
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n, 1, 1);
    const bool v4 = main_args->kind == DSV4_CACHE_V4;
    cfg.blockDim = dim3((v4 ? DSV4_V4_HEAD_DIM : kHead) / 2, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool fp4 = idx_args->kind == DSV4_CACHE_IDX_FP4;
    const bool r4 = main_args->ratio == 4;
    cudaError_t e;
    if (v4) {
        if (r4)
            e = fp4 ? cudaLaunchKernelEx(&cfg, compress_pair_kernel<4, DSV4_CACHE_IDX_FP4, DSV4_CACHE_V4>, Pm, Pi)
                    : cudaLaunchKernelEx(&cfg, compress_pair_kernel<4, DSV4_CACHE_IDX, DSV4_CACHE_V4>, Pm, Pi);
        else
            e = fp4 ? cudaLaunchKernelEx(&cfg, compress_pair_kernel<128, DSV4_CACHE_IDX_FP4, DSV4_CACHE_V4>, Pm, Pi)
                    : cudaLaunchKernelEx(&cfg, compress_pair_kernel<128, DSV4_CACHE_IDX, DSV4_CACHE_V4>, Pm, Pi);
    } else {
        if (r4)
            e = fp4 ? cudaLaunchKernelEx(&cfg, compress_pair_kernel<4, DSV4_CACHE_IDX_FP4, DSV4_CACHE_MLA>, Pm, Pi)
                    : cudaLaunchKernelEx(&cfg, compress_pair_kernel<4, DSV4_CACHE_IDX, DSV4_CACHE_MLA>, Pm, Pi);
        else
            e = fp4 ? cudaLaunchKernelEx(&cfg, compress_pair_kernel<128, DSV4_CACHE_IDX_FP4, DSV4_CACHE_MLA>, Pm, Pi)
                    : cudaLaunchKernelEx(&cfg, compress_pair_kernel<128, DSV4_CACHE_IDX, DSV4_CACHE_MLA>, Pm, Pi);
    }
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

extern "C" dsv4_status dsv4_cache_insert_rows(const dsv4_insert_rows_args* a, dsv4_stream_t stream)
{
    if (a == nullptr) return DSV4_ERR_INVALID;
    if (a->num_rows < 0 || a->num_seqs < 0 || a->bt_stride < 0 || a->num_pages < 0)
        return DSV4_ERR_INVALID;
    if (a->kind != DSV4_CACHE_MLA && a->kind != DSV4_CACHE_IDX && a->kind != DSV4_CACHE_IDX_FP4 &&
        a->kind != DSV4_CACHE_V4)
        return DSV4_ERR_INVALID;
    if (a->num_rows == 0) return DSV4_OK;
    if (!a->rows_dev || !a->seq_dev || !a->slot_dev || !a->cache_dev || !a->block_table_dev)
        return DSV4_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(a->rows_dev) & 7) || (reinterpret_cast<uintptr_t>(a->cache_dev) & 15))
        return DSV4_ERR_SHAPE;
    CompressParams P{};
    P.cache = static_cast<uint8_t*>(a->cache_dev);
    P.num_pages = a->num_pages;
    P.bt = a->block_table_dev;
    P.bt_stride = a->bt_stride;
    P.num_seqs = a->num_seqs;
    P.status = a->status_dev;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (a->kind == DSV4_CACHE_IDX)
        insert_rows_kernel<kIdx, DSV4_CACHE_IDX><<<a->num_rows, kIdx / 2, 0, st>>>(a->rows_dev, a->seq_dev,
                                                                                 a->slot_dev, P);
    else if (a->kind == DSV4_CACHE_IDX_FP4)
        insert_rows_kernel<kIdx, DSV4_CACHE_IDX_FP4><<<a->num_rows, kIdx / 2, 0, st>>>(a->rows_dev, a->seq_dev,
                                                                                     a->slot_dev, P);
    else if (a->kind == DSV4_CACHE_V4)
        insert_rows_kernel<DSV4_V4_HEAD_DIM, DSV4_CACHE_V4><<<a->num_rows, DSV4_V4_HEAD_DIM / 2, 0, st>>>(
            a->rows_dev, a->seq_dev, a->slot_dev, P);
    else
        insert_rows_kernel<kHead, DSV4_CACHE_MLA><<<a->num_rows, kHead / 2, 0, st>>>(a->rows_dev, a->seq_dev,
                                                                                   a->slot_dev, P);
    return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
