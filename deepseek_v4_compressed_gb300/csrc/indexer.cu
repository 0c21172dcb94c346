// indexer.cu -- lightning indexer logits and per-query top-k.
//
// I_{t,s} = sum_j w_{t,j} ReLU(q_{t,j} . k_s) (SparseAttnIndexer formula in
// the "DeepseekV4Attention" class walkthrough; section 2 of the V4 internals
// talk write-up), with k_s = FP8 row * fp32 scale of the indexer cache, over
// the causal slots s < ctx_len / 4; then the k largest per query ("Indexer,
// C4A and C128A top-k", "DeepSeek V4 attention in vLLM").
#include "dsv4_common.cuh"
#include "plan.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace dsv4 {

// ---------------------------------------------------------------------------
// Logits on the tensor cores.  Per 128-slot tile (two 64-entry pages, each a
// contiguous 8 KB plane of FP8 rows), one tcgen05.mma kind::f8f6f4 chain
// D[128 slots x N heads] = K_tile[128 x 128] * Q^T[128 x N] (fp32 in TMEM),
// then each of 128 epilogue threads turns its slot's row of D into
// I_s = scale_s * sum_j w_j * max(D_sj, 0).
//   warp 4: TMA producer (query once, then two page loads per tile, 3-stage ring)
//   warp 5: MMA issuer (4 MMAs of K=32 per tile, double-buffered accumulator)
//   warps 0-3: epilogue (TMEM lane = slot row)
// Memory-bound: 132 bytes of cache per slot against 2 * 128 * N flops.
// ---------------------------------------------------------------------------
constexpr int kIdxTileSlots = 128;
constexpr int kIdxStages = 3;
constexpr int kIdxTileBytes = kIdxTileSlots * kIdx;       // 16 KB
constexpr int kIdxQBytes = 64 * kIdx;                     // query tile, N <= 64 rows
constexpr int kIdxThreads = 192;
constexpr int kIdxTmemCols = 128;                         // 2 accumulators x 64 columns
constexpr int kIdxScaleBytes = 2 * kPage * 4;                // scale planes of the tile's two pages
constexpr int kIdxSmem = kIdxStages * kIdxTileBytes + kIdxQBytes + kIdxStages * kIdxScaleBytes +
                         2048 /* barriers etc */ + 1024 /* align */;

struct IdxTcParams {
    const uint8_t* cache;
    int num_pages;
    const int* bt;
    int bt_stride;
    const int* ctx_len;
    const float* w;
    int H;
    int n_pad;
    float* logits;
    int logits_stride;
    int max_slots;
    int tiles_per_cta;
    int* status;
};

__global__ void __launch_bounds__(kIdxThreads, 1)
indexer_logits_tc(const __grid_constant__ CUtensorMap tm_cache, const __grid_constant__ CUtensorMap tm_q,
                  IdxTcParams P)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = tc::align1024_shared(smem_raw);
    uint8_t* a_tiles = smem;
    uint8_t* q_tile = smem + kIdxStages * kIdxTileBytes;
    float* scales_s = reinterpret_cast<float*>(q_tile + kIdxQBytes);   // [stage][128 slots]
    uint64_t* bars = reinterpret_cast<uint64_t*>(q_tile + kIdxQBytes + kIdxStages * kIdxScaleBytes);
    uint64_t* full = bars;                        // [kIdxStages]
    uint64_t* empty = bars + kIdxStages;          // [kIdxStages]
    uint64_t* acc_full = bars + 2 * kIdxStages;   // [2]
    uint64_t* acc_empty = acc_full + 2;           // [2]
    uint64_t* q_bar = acc_empty + 2;
    float* w_s = reinterpret_cast<float*>(q_bar + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(w_s + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int b = blockIdx.y;
    int n_c = P.ctx_len[b] / 4;
    if (n_c > P.max_slots) n_c = P.max_slots;
    if (n_c < 0) n_c = 0;
    const int n_tiles = (n_c + kIdxTileSlots - 1) / kIdxTileSlots;
    const int t_begin = blockIdx.x * P.tiles_per_cta;
    const int t_end = min(n_tiles, t_begin + P.tiles_per_cta);
    if (t_begin >= t_end) return;                 // uniform: nothing allocated yet
    const int n_my = t_end - t_begin;
    const int n_pages = (n_c + kPage - 1) / kPage;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kIdxStages; ++i) {
            tc::mbar_init(tc::smem_u32(&full[i]), 1);
            tc::mbar_init(tc::smem_u32(&empty[i]), 5);   // MMA commit + 4 epilogue warps (scales read)
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(tc::smem_u32(&acc_full[i]), 1);
            tc::mbar_init(tc::smem_u32(&acc_empty[i]), 4);
        }
        tc::mbar_init(tc::smem_u32(q_bar), 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (threadIdx.x < 64) w_s[threadIdx.x] = (threadIdx.x < P.H) ? P.w[static_cast<long long>(b) * P.H + threadIdx.x] : 0.f;
    if (warp == 0) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), kIdxTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    int issued = 0;   // tiles whose loads were issued (producer only)
    int consumed = 0; // tiles whose stage the MMA released (MMA thread only)

    if (warp == 4) {
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_cache);
            tc::prefetch_tensormap(&tm_q);
            tc::mbar_arrive_expect_tx(tc::smem_u32(q_bar), P.n_pad * kIdx);
            tc::tma_load_2d(tc::smem_u32(q_tile), &tm_q, tc::smem_u32(q_bar), 0, b * P.H);
            for (int i = 0; i < n_my; ++i) {
                const int st = i % kIdxStages;
                const uint32_t ph = (i / kIdxStages) & 1;
                if (i >= kIdxStages && !tc::mbar_wait(tc::smem_u32(&empty[st]), ph ^ 1, abort_flag, P.status)) break;
                const int tile = t_begin + i;
                int pg[2], spg[2];
                for (int h = 0; h < 2; ++h) {
                    const int pi = min(2 * tile + h, n_pages - 1);
                    int v = (pi < P.bt_stride) ? P.bt[static_cast<long long>(b) * P.bt_stride + pi] : -1;
                    spg[h] = v;
                    if (v < 0 || v >= P.num_pages) {
                        flag(P.status, DSV4_DEV_BAD_PAGE);
                        v = P.num_pages;          // out of the map: TMA fills zeros
                        spg[h] = 0;               // scales from a valid page (the row's data is zero)
                    }
                    pg[h] = v;
                }
                const uint32_t dst = tc::smem_u32(a_tiles + st * kIdxTileBytes);
                const uint32_t fb = tc::smem_u32(&full[st]);
                tc::mbar_arrive_expect_tx(fb, kIdxTileBytes + kIdxScaleBytes);
                tc::tma_load_3d(dst, &tm_cache, fb, 0, 0, pg[0]);
                tc::tma_load_3d(dst + kIdxTileBytes / 2, &tm_cache, fb, 0, 0, pg[1]);
                for (int h = 0; h < 2; ++h)
                    tc::bulk_load(tc::smem_u32(scales_s + st * 128 + h * kPage),
                                  P.cache + static_cast<long long>(spg[h]) * kIdxPage + kPage * kIdx, kPage * 4, fb);
                issued = i + 1;
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc(128, P.n_pad, tc::kFmtE4M3, tc::kFmtE4M3);
            const uint64_t b_desc = tc::desc_kmajor_sw128(tc::smem_u32(q_tile));
            if (tc::mbar_wait(tc::smem_u32(q_bar), 0, abort_flag, P.status)) {
                for (int i = 0; i < n_my; ++i) {
                    const int st = i % kIdxStages;
                    const uint32_t ph = (i / kIdxStages) & 1;
                    const int ab = i & 1;
                    const uint32_t aph = (i >> 1) & 1;
                    if (!tc::mbar_wait(tc::smem_u32(&full[st]), ph, abort_flag, P.status)) break;
                    if (i >= 2 && !tc::mbar_wait(tc::smem_u32(&acc_empty[ab]), aph ^ 1, abort_flag, P.status)) break;
                    tc::tc_fence_after();
                    const uint64_t a_desc = tc::desc_kmajor_sw128(tc::smem_u32(a_tiles + st * kIdxTileBytes));
                    const uint32_t d = tmem + ab * 64;
#pragma unroll
                    for (int k = 0; k < kIdx / 32; ++k)   // K = 32 FP8 (32 bytes) per instruction
                        tc::mma_f8f6f4(d, a_desc + 2 * k, b_desc + 2 * k, idesc, k > 0 ? 1u : 0u);
                    tc::mma_commit(tc::smem_u32(&empty[st]));
                    tc::mma_commit(tc::smem_u32(&acc_full[ab]));
                    consumed = i + 1;
                }
            }
        }
    } else {
        const int row = warp * 32 + lane;
        for (int i = 0; i < n_my; ++i) {
            const int ab = i & 1;
            const uint32_t aph = (i >> 1) & 1;
            if (!tc::mbar_wait(tc::smem_u32(&acc_full[ab]), aph, abort_flag, P.status)) break;
            tc::tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + ab * 64;
            float v0[32], v1[32];
            tc::tmem_ld32(taddr, v0);
            if (P.n_pad > 32) tc::tmem_ld32(taddr + 32, v1);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acc_empty[ab]));
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) acc += (j < P.H) ? w_s[j] * fmaxf(v0[j], 0.f) : 0.f;
            if (P.n_pad > 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j) acc += (j + 32 < P.H) ? w_s[j + 32] * fmaxf(v1[j], 0.f) : 0.f;
            }
            // the stage's scales: its full barrier cannot have moved on, since
            // the stage is only refilled after this warp releases it below
            const int st = i % kIdxStages;
            float scale = 0.f;
            if (tc::mbar_wait(tc::smem_u32(&full[st]), (i / kIdxStages) & 1, abort_flag, P.status))
                scale = scales_s[st * 128 + row];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&empty[st]));
            const int s = (t_begin + i) * kIdxTileSlots + row;
            if (s < n_c) P.logits[static_cast<long long>(b) * P.logits_stride + s] = acc * scale;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == 4 && lane == 0) {
        // let this CTA's own copies land before its shared memory is released
        for (int i = consumed > 0 ? consumed : 0; i < issued; ++i) {
            volatile int no_abort = 0;
            tc::mbar_wait(tc::smem_u32(&full[i % kIdxStages]), (i / kIdxStages) & 1, &no_abort, nullptr);
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kIdxTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Top-k: one CTA per query.  Keys are the order-preserving uint32 images of
// the logits, taken relative to their minimum so the radix digits start at the
// data's own range: up to three passes of 11-bit digits (2048-bin shared
// histograms) narrow the k-th largest key down to its bin; a pass stops early
// once the bin holding the k-th key is taken whole.  Keys equal to the final
// threshold are taken lowest slot first; an ordered compaction writes the k
// slots in ascending order.
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 512;
constexpr int kTopkBins = 2048;
constexpr int kTopkSmemKeys = 49152;   // keys staged in shared memory up to this many (192 KB)

// Exclusive scan of one int per thread over the CTA; also returns the total.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int& total)
{
    constexpr int NW = kTopkThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int t = (lane < NW) ? scratch[lane] : 0;
        int u = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, u, o);
            if (lane >= o) u += y;
        }
        scratch[lane] = u - t;
        if (lane == 31) scratch[32] = u;
    }
    __syncthreads();
    total = scratch[32];
    const int r = scratch[warp] + x - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(
    const float* __restrict__ logits, int row_stride, int max_slots, const int* __restrict__ ctx_len, int k,
    int* __restrict__ out_idx, int out_stride, int* __restrict__ out_len, int smem_keys)
{
    extern __shared__ uint32_t skeys[];
    __shared__ int hist[kTopkBins];
    __shared__ int scratch[33];
    __shared__ uint32_t s_min, s_prefix;
    __shared__ int s_lo, s_hi, s_rem, s_done;

    const int b = blockIdx.x;
    int n = ctx_len[b] / 4;
    n = n < 0 ? 0 : (n > max_slots ? max_slots : n);
    int* orow = out_idx + static_cast<long long>(b) * out_stride;
    const float* lrow = logits + static_cast<long long>(b) * row_stride;
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += blockDim.x) orow[i] = (i < n) ? i : -1;
        if (threadIdx.x == 0) out_len[b] = n;
        return;
    }
    const bool in_smem = n <= smem_keys;
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    // vectorised load (rows are 16-byte aligned: row_stride is a multiple of 4)
    const int n4 = n >> 2;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = reinterpret_cast<const float4*>(lrow)[i];
        const uint32_t k0 = f32_order_key(v.x), k1 = f32_order_key(v.y), k2 = f32_order_key(v.z),
                       k3 = f32_order_key(v.w);
        kmin = min(min(kmin, k0), min(min(k1, k2), k3));
        kmax = max(max(kmax, k0), max(max(k1, k2), k3));
        if (in_smem) reinterpret_cast<uint4*>(skeys)[i] = make_uint4(k0, k1, k2, k3);
    }
    for (int i = (n4 << 2) + threadIdx.x; i < n; i += blockDim.x) {
        const uint32_t kk = f32_order_key(lrow[i]);
        kmin = min(kmin, kk);
        kmax = max(kmax, kk);
        if (in_smem) skeys[i] = kk;
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if ((threadIdx.x & 31) == 0) {
        scratch[threadIdx.x >> 5] = static_cast<int>(kmin);
        hist[threadIdx.x >> 5] = static_cast<int>(kmax);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t mn = 0xffffffffu, mx = 0u;
        for (int w = 0; w < kTopkThreads / 32; ++w) {
            mn = min(mn, static_cast<uint32_t>(scratch[w]));
            mx = max(mx, static_cast<uint32_t>(hist[w]));
        }
        s_min = mn;
        const uint32_t range = mx - mn;
        s_hi = range ? 32 - __clz(range) : 0;   // offsets (key - min) fit in s_hi bits
        s_lo = s_hi;
        s_prefix = 0;
        s_rem = k;
        s_done = (range == 0);
    }
    __syncthreads();
    const uint32_t base = s_min;
    auto key_at = [&](int i) -> uint32_t { return in_smem ? skeys[i] : f32_order_key(lrow[i]); };

    while (!s_done) {
        const int hi = s_hi;
        const int lo = hi > 11 ? hi - 11 : 0;
        const uint32_t prefix = s_prefix;
        const int rem = s_rem;
        for (int i = threadIdx.x; i < kTopkBins; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint32_t off = key_at(i) - base;
            if (hi >= 32 || (off >> hi) == (prefix >> hi)) atomicAdd(&hist[(off >> lo) & (kTopkBins - 1)], 1);
        }
        __syncthreads();
        // bins from the top: thread t sums bins 2047-4t .. 2044-4t
        int c[4];
        int local = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            c[q] = hist[kTopkBins - 1 - 4 * threadIdx.x - q];
            local += c[q];
        }
        int tot;
        const int before = block_excl_scan(local, scratch, tot);
        if (before < rem && rem <= before + local) {
            int cum = before;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (cum + c[q] >= rem) {
                    const uint32_t d = kTopkBins - 1 - 4 * threadIdx.x - q;
                    s_prefix = prefix | (d << lo);
                    s_rem = rem - cum;
                    s_lo = lo;
                    s_hi = lo;
                    s_done = (lo == 0) || (cum + c[q] == rem);
                    break;
                }
                cum += c[q];
            }
        }
        __syncthreads();
    }
    const int lo = s_lo;
    const uint32_t thr = s_prefix >> lo;   // digit prefix of the threshold bin
    const int take_eq = s_rem;             // keys of the threshold bin to take, lowest slot first

    const int chunk = (n + blockDim.x - 1) / blockDim.x;
    const int i0 = threadIdx.x * chunk;
    const int i1 = min(n, i0 + chunk);
    int gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t d = (key_at(i) - base) >> lo;
        gt += d > thr;
        eq += d == thr;
    }
    int tot;
    const int gt_before = block_excl_scan(gt, scratch, tot);
    const int eq_before = block_excl_scan(eq, scratch, tot);
    int g = gt_before, e = eq_before;
    for (int i = i0; i < i1; ++i) {
        const uint32_t d = (key_at(i) - base) >> lo;
        if (d > thr) {
            orow[g + min(e, take_eq)] = i;
            ++g;
        } else if (d == thr) {
            if (e < take_eq) orow[g + e] = i;
            ++e;
        }
    }
    if (threadIdx.x == 0) out_len[b] = k;
}

}  // namespace dsv4

using namespace dsv4;

extern "C" dsv4_status dsv4_indexer_topk(const dsv4_plan* plan, const dsv4_indexer_args* a,
                                         void* workspace, size_t workspace_bytes, dsv4_stream_t stream)
{
    if (plan == nullptr || a == nullptr) return DSV4_ERR_INVALID;
    if (plan->type != DSV4_C4A) return DSV4_ERR_SHAPE;
    if (workspace_bytes < plan->ws_bytes || (workspace == nullptr && plan->ws_bytes)) return DSV4_ERR_SHAPE;
    if (!a->q_fp8_dev || !a->weights_dev || !a->idx_cache_dev || !a->block_table_dev ||
        !a->ctx_len_dev || !a->out_idx_dev || !a->out_len_dev)
        return DSV4_ERR_INVALID;
    if (a->out_stride < plan->topk || a->bt_stride < 1 || a->num_pages < 1) return DSV4_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(a->idx_cache_dev) & 15) return DSV4_ERR_SHAPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* logits = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan->ws_logits_off);
    const int B = plan->batch, H = plan->geom.idx_heads;
    if (plan->idx_ctas_per_seq > 0) {
        CUtensorMap tm_cache, tm_q;
        const uint64_t cdims[3] = {static_cast<uint64_t>(kIdx), static_cast<uint64_t>(kPage),
                                   static_cast<uint64_t>(a->num_pages)};
        const uint64_t cstr[2] = {static_cast<uint64_t>(kIdx), static_cast<uint64_t>(kIdxPage)};
        const uint32_t cbox[3] = {static_cast<uint32_t>(kIdx), static_cast<uint32_t>(kPage), 1};
        const int n_pad = H <= 16 ? 16 : (H + 15) / 16 * 16;
        const uint64_t qdims[2] = {static_cast<uint64_t>(kIdx), static_cast<uint64_t>(B) * H};
        const uint64_t qstr[1] = {static_cast<uint64_t>(kIdx)};
        const uint32_t qbox[2] = {static_cast<uint32_t>(kIdx), static_cast<uint32_t>(n_pad)};
        if (!encode_tmap(&tm_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a->idx_cache_dev, cdims, cstr, cbox,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a->q_fp8_dev, qdims, qstr, qbox,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return DSV4_ERR_CUDA;
        IdxTcParams P;
        P.cache = static_cast<const uint8_t*>(a->idx_cache_dev);
        P.num_pages = a->num_pages;
        P.bt = a->block_table_dev;
        P.bt_stride = a->bt_stride;
        P.ctx_len = a->ctx_len_dev;
        P.w = a->weights_dev;
        P.H = H;
        P.n_pad = n_pad;
        P.logits = logits;
        P.logits_stride = plan->logits_stride;
        P.max_slots = plan->max_slots;
        P.tiles_per_cta = plan->idx_tiles_per_cta;
        P.status = a->status_dev;
        static bool tc_attr = false;
        if (!tc_attr) {
            cudaFuncSetAttribute(indexer_logits_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kIdxSmem);
            tc_attr = true;
        }
        dim3 grid(plan->idx_ctas_per_seq, B);
        indexer_logits_tc<<<grid, kIdxThreads, kIdxSmem, st>>>(tm_cache, tm_q, P);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return DSV4_ERR_CUDA;
    }
    cudaError_t e;
    const int smem_keys = plan->max_slots <= kTopkSmemKeys ? plan->max_slots : 0;
    const size_t smem = static_cast<size_t>(smem_keys) * 4;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopkSmemKeys * 4);
        attr_set = true;
    }
    topk_kernel<<<B, kTopkThreads, smem, st>>>(logits, plan->logits_stride, plan->max_slots, a->ctx_len_dev,
                                               plan->topk, a->out_idx_dev, a->out_stride, a->out_len_dev,
                                               smem_keys);
    e = cudaGetLastError();
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
