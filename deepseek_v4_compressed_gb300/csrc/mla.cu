// mla.cu -- sparse absorbed-MQA decode over (selected compressed slots) ||
// (SWA window), one 576-dim latent KV head, value = the 512 latent dims.
//
// _forward_decode of the "DeepseekV4Attention" class walkthrough
// (flash_mla_with_kvcache over the SWA cache plus the compressed cache with
// their two index sets); KV_actual = selected history || recent window in
// section 2 of the V4 internals talk write-up; absorbed decode over the
// cached latent in section 2.2 of "From MLA to CSA + HCA".
#include "dsv4_common.cuh"
#include "plan.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace dsv4 {

struct MlaParams {
    const uint16_t* q;
    const uint8_t* swa;
    int swa_pages;
    const int* swa_bt;
    int swa_bt_stride;
    const uint8_t* comp;
    int comp_pages;
    const int* comp_bt;
    int comp_bt_stride;
    const int* idx;
    int idx_stride;
    const int* idx_len;
    const int* ctx_len;
    uint16_t* out;
    float* lse;
    int H;
    int window;
    float scale;
    int* status;
};

// Row pointer of key i of sequence b (compressed keys first, then the SWA
// window).  Returns false (and flags) for an out-of-range index or page.
struct KeyRef {
    const uint8_t* row;     // compressed: 640 data bytes; SWA: 576 bf16
    const uint8_t* scales;  // compressed only
    bool comp;
};

__device__ __forceinline__ bool key_ref(const MlaParams& P, int b, int i, int n_comp, int t0, KeyRef& k)
{
    if (i < n_comp) {
        const int slot = P.idx[static_cast<long long>(b) * P.idx_stride + i];
        const int pi = slot / kPage;
        if (slot < 0 || pi >= P.comp_bt_stride) {
            flag(P.status, DSV4_DEV_BAD_INDEX);
            return false;
        }
        const int pg = P.comp_bt[static_cast<long long>(b) * P.comp_bt_stride + pi];
        if (pg < 0 || pg >= P.comp_pages) {
            flag(P.status, DSV4_DEV_BAD_PAGE);
            return false;
        }
        const uint8_t* page = P.comp + static_cast<long long>(pg) * kMlaPage;
        const int r = slot % kPage;
        k.row = page + r * kMlaData;
        k.scales = page + kPage * kMlaData + r * 8;
        k.comp = true;
        return true;
    }
    const int t = t0 + (i - n_comp);
    const int pi = t / kPage;
    const int pg = (pi < P.swa_bt_stride) ? P.swa_bt[static_cast<long long>(b) * P.swa_bt_stride + pi] : -1;
    if (pg < 0 || pg >= P.swa_pages) {
        flag(P.status, DSV4_DEV_BAD_PAGE);
        return false;
    }
    k.row = P.swa + static_cast<long long>(pg) * kSwaPage + (t % kPage) * (kHead * 2);
    k.scales = nullptr;
    k.comp = false;
    return true;
}

// ---------------------------------------------------------------------------
// Tensor-core decode attention (tcgen05, TMEM accumulators).
//
// CTA = (rank r of a cluster of C CTAs, sequence b x 64-head group g).  The C
// CTAs of a cluster split the sequence's keys (selected compressed slots then
// the SWA window) into contiguous ranges, each CTA walks its range in 32-key
// tiles with an online softmax, and the partial results are merged through
// distributed shared memory -- no partials in HBM, no combine kernel.
//
//   S  = Q K^T     tcgen05.mma kind::f16, M = 64 head rows (row r lands in
//                  TMEM lane 32*(r/16) + r%16), N = 32 keys, K = 576 (36
//                  instructions); double-buffered in TMEM columns [0, 64).
//   O^T += V^T P^T M = 128 value dims (4 blocks cover the 512 latent dims),
//                  N = 64 heads, K = 32 keys; V^T is the same swizzled K tile
//                  read as an MN-major operand; O^T lives in TMEM [64, 320).
// Warps: 0-3 softmax (lanes 0-15 of each = 16 heads) and O^T correction (all lanes);
// 4-7 producers: gather and dequantise key rows (FP8 * 2^e -> bf16, exact) into
// the 128-byte-swizzled tile; 8 MMA issuer (and the Q load by TMA).
// ---------------------------------------------------------------------------
constexpr int kTcKeys = 32;
constexpr int kTcStages = 2;                               // bf16 key tiles (MMA operands)
constexpr int kTcRawStages = 2;                            // raw FP8 rows landing from TMA bulk copies
constexpr int kTcQChunk = 64 * 128;                        // 64 head rows x 64 dims (bf16)
constexpr int kTcQBytes = 9 * kTcQChunk;                   // 73728
constexpr int kTcKChunk = kTcKeys * 128;                   // 32 key rows x 64 dims
constexpr int kTcKBytes = 9 * kTcKChunk;                   // 36864 per stage
constexpr int kTcRawBytes = kTcKeys * kMlaData;            // 32 rows x 640 B
constexpr int kTcPBytes = 64 * 128;                        // 64 head rows x 32 keys (rows padded to 128 B)
constexpr int kTcMaxKeys = 1024;                           // keys one CTA can own (its pointer table)
constexpr int kTcThreads = 288;
constexpr int kTcTmemCols = 512;
constexpr int kTcOCol = 64;
constexpr int kOffQ = 0;
constexpr int kOffK = kTcQBytes;
constexpr int kOffRaw = kOffK + kTcStages * kTcKBytes;
constexpr int kOffP = kOffRaw + kTcRawStages * kTcRawBytes;
constexpr int kOffTab = kOffP + 2 * kTcPBytes;
constexpr int kOffMisc = kOffTab + kTcMaxKeys * 16;
constexpr int kMiscBytes = 4096;
constexpr int kTcSmem = kOffMisc + kMiscBytes + 1024;
constexpr int kStageO = 0;                                 // epilogue: fp32 [64 heads][512] (reuses Q/K space)
static_assert(64 * 512 * 4 <= kOffRaw, "staging must fit in the Q/K space");
static_assert(kTcSmem <= 232448, "shared memory budget");

struct MlaTcParams {
    MlaParams base;
    int head_groups;
    int cluster;
    int topk;
};

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16 FP8 E4M3 codes times 2^E -> 16 bf16.  Each code's 7 magnitude bits go to
// bit 20 of an fp32 word and its sign to bit 31: the word's value is the code's
// value times 2^-120 (exponent field 0 gives exactly the scaled subnormals).
// Two exact power-of-two multiplies restore 2^(E+120); the product has at most
// 4 significant bits, so its upper 16 bits are the bf16 (exact for every
// result in the normal range).  Integer and FMA pipes only.
__device__ __forceinline__ uint32_t code_f32_bits(uint32_t byte)
{
    return ((byte & 0x7fu) << 20) | ((byte & 0x80u) << 24);
}

__device__ __forceinline__ void dequant16(const uint4 w, uint32_t scale_byte, uint4& lo, uint4& hi)
{
    const int k = static_cast<int>(scale_byte) - 7;          // E + 120, E = byte - 127
    const int ka = k < 127 ? k : 127;
    const float ma = __int_as_float((ka + 127) << 23);        // 2^ka, ka in [-7, 127]
    const float mb = __int_as_float((k - ka + 127) << 23);    // 2^(k-ka) >= 1
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float f[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) f[c] = __uint_as_float(code_f32_bits((in[i] >> (8 * c)) & 0xffu)) * ma * mb;
        out[2 * i] = __byte_perm(__float_as_uint(f[0]), __float_as_uint(f[1]), 0x7632);
        out[2 * i + 1] = __byte_perm(__float_as_uint(f[2]), __float_as_uint(f[3]), 0x7632);
    }
    lo = make_uint4(out[0], out[1], out[2], out[3]);
    hi = make_uint4(out[4], out[5], out[6], out[7]);
}

__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

__global__ void __launch_bounds__(kTcThreads, 1)
mla_decode_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_swa, MlaTcParams T)
{
    const MlaParams& P = T.base;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q_s = smem + kOffQ;
    uint8_t* k_s = smem + kOffK;
    uint8_t* p_s = smem + kOffP;
    uint8_t* raw_s = smem + kOffRaw;
    uint4* table = reinterpret_cast<uint4*>(smem + kOffTab);   // per owned compressed row: pointer | flags, scales
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffMisc);
    uint64_t* kv_full = bars;          // [2] producers -> MMA (tile in its stage)
    uint64_t* kv_empty = bars + 2;     // [2] MMA -> producers (stage read by QK and PV)
    uint64_t* swa_full = bars + 4;     // [2] TMA tensor loads of a window tile landed
    uint64_t* s_full = bars + 6;       // [2] MMA -> softmax
    uint64_t* p_full = bars + 8;       // [2] softmax -> MMA (P written, S read, O^T corrected)
    uint64_t* pv_done = bars + 10;     // [2] MMA -> softmax
    uint64_t* q_full = bars + 12;
    uint64_t* sync4 = bars + 13;       // [2] the four softmax warps meet once per tile
    uint64_t* table_ready = bars + 15;
    float* sm_m = reinterpret_cast<float*>(bars + 32);   // [64] running max (log2 domain)
    float* sm_l = sm_m + 64;                              // [64] running sum
    float* sm_alpha = sm_l + 64;                          // [64] correction factors of this tile
    float* red_w = sm_alpha + 64;                         // [8][64] merge weights
    float* red_invl = red_w + 8 * 64;                     // [64]
    int* sm_any = reinterpret_cast<int*>(red_invl + 64);  // [2][4]
    volatile int* abort_flag = sm_any + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm_any + 9);

    const int rank = blockIdx.x;
    const int b = blockIdx.y / T.head_groups, g_head = blockIdx.y % T.head_groups;
    const int h0 = g_head * 64;
    const int nh = min(64, P.H - h0);
    const int p = P.ctx_len[b] - 1;
    const int n_comp = P.idx_len ? min(max(P.idx_len[b], 0), T.topk) : 0;
    const int t0 = max(0, p - P.window + 1);
    // Tiles of 32 keys: first the window, in 32-token-aligned blocks A0..A1
    // (rows outside [t0, p] masked), then the compressed keys in slot-list order
    // (rows past n_comp masked).  Tile g belongs to CTA g % C of the cluster,
    // so every CTA starts with its window tiles.
    const int C = T.cluster;
    const int A0 = t0 >> 5;
    const int n_swa_t = p >= 0 ? (p >> 5) - A0 + 1 : 0;
    const int n_comp_t = (n_comp + kTcKeys - 1) / kTcKeys;
    const int n_glob = n_swa_t + n_comp_t;
    const int n_swa_mine = n_swa_t > rank ? (n_swa_t - rank + C - 1) / C : 0;
    int n_tiles = n_glob > rank ? (n_glob - rank + C - 1) / C : 0;
    if (n_tiles - n_swa_mine > kTcMaxKeys / kTcKeys) {
        if (threadIdx.x == 0) flag(P.status, DSV4_DEV_BAD_INDEX);
        n_tiles = n_swa_mine + kTcMaxKeys / kTcKeys;
    }
    const int n_comp_mine = n_tiles - n_swa_mine;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float scale_log2 = P.scale * 1.4426950408889634f;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(tc::smem_u32(&kv_full[i]), 4);
            tc::mbar_init(tc::smem_u32(&kv_empty[i]), 1);
            tc::mbar_init(tc::smem_u32(&swa_full[i]), 1);
            tc::mbar_init(tc::smem_u32(&s_full[i]), 1);
            tc::mbar_init(tc::smem_u32(&p_full[i]), 4);
            tc::mbar_init(tc::smem_u32(&pv_done[i]), 1);
            tc::mbar_init(tc::smem_u32(&sync4[i]), 4);
        }
        tc::mbar_init(tc::smem_u32(q_full), 1);
        tc::mbar_init(tc::smem_u32(table_ready), 4);
        *abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (threadIdx.x < 64) {
        sm_m[threadIdx.x] = -INFINITY;
        sm_l[threadIdx.x] = 0.f;
    }
    if (warp == 0) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), kTcTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (n_tiles > 0) {
        if (warp == 8) {
            // ------------------------------------------------------------ MMA
            // S(t) = Q K(t)^T with M = 64 (the head rows; D row r in TMEM lane
            // 32*(r/16) + r%16) and O^T += V(u)^T P(u)^T, issued as soon as each
            // is ready: QK(t) needs tile t loaded and S buffer t%2 read out
            // (PV(t-2) issued); PV(u) needs P(u).
            if (lane == 0) {
                tc::prefetch_tensormap(&tm_q);
                tc::mbar_arrive_expect_tx(tc::smem_u32(q_full), kTcQBytes);
                for (int c = 0; c < 9; ++c)
                    tc::tma_load_2d(tc::smem_u32(q_s + c * kTcQChunk), &tm_q, tc::smem_u32(q_full), c * 64,
                                    b * P.H + h0);
                const uint32_t id_qk = tc::idesc(64, kTcKeys, tc::kFmtBF16, tc::kFmtBF16);
                const uint32_t id_pv = tc::idesc(128, 64, tc::kFmtBF16, tc::kFmtBF16, true, false);
                bool ok = tc::mbar_wait(tc::smem_u32(q_full), 0, abort_flag, P.status);
                int next_qk = 0, next_pv = 0;
                uint64_t t_idle = 0;
                while (ok && next_pv < n_tiles) {
                    bool did = false;
                    if (next_qk < n_tiles && next_qk <= next_pv + 1 &&
                        tc::mbar_test(tc::smem_u32(&kv_full[next_qk & 1]), (next_qk >> 1) & 1)) {
                        const int t = next_qk;
                        tc::tc_fence_after();
                        const uint32_t d = tmem + (t & 1) * kTcKeys;
                        const uint32_t kb = tc::smem_u32(k_s + (t & 1) * kTcKBytes);
#pragma unroll 1
                        for (int c = 0; c < 9; ++c) {
                            const uint64_t ad = tc::desc_kmajor_sw128(tc::smem_u32(q_s + c * kTcQChunk));
                            const uint64_t bd = tc::desc_kmajor_sw128(kb + c * kTcKChunk);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc::mma_f16(d, ad + 2 * k, bd + 2 * k, id_qk, (c | k) != 0 ? 1u : 0u);
                        }
                        tc::mma_commit(tc::smem_u32(&s_full[t & 1]));
                        ++next_qk;
                        did = true;
                    }
                    if (next_pv < next_qk &&
                        tc::mbar_test(tc::smem_u32(&p_full[next_pv & 1]), (next_pv >> 1) & 1)) {
                        const int u = next_pv;
                        tc::tc_fence_after();
                        const uint32_t kb = tc::smem_u32(k_s + (u & 1) * kTcKBytes);
                        const uint64_t pd = tc::desc_kmajor_sw128(tc::smem_u32(p_s + (u & 1) * kTcPBytes));
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int j = 0; j < 2; ++j)
                                tc::mma_f16(tmem + kTcOCol + i * 64,
                                            tc::desc_mnmajor_sw128(kb + 2 * i * kTcKChunk + j * 2048, kTcKChunk, 1024),
                                            pd + 2 * j, id_pv, (u > 0 || j > 0) ? 1u : 0u);
                        tc::mma_commit(tc::smem_u32(&kv_empty[u & 1]));
                        tc::mma_commit(tc::smem_u32(&pv_done[u & 1]));
                        ++next_pv;
                        did = true;
                    }
                    if (did) {
                        t_idle = 0;
                    } else if (*abort_flag) {
                        ok = false;
                    } else {
                        // with one event possible, sleep on it (the wait returns when
                        // it completes); with both possible, keep polling
                        const bool qk_possible = next_qk < n_tiles && next_qk <= next_pv + 1;
                        const bool pv_possible = next_pv < next_qk;
                        if (pv_possible && !qk_possible)
                            mbar_try_wait_hint(tc::smem_u32(&p_full[next_pv & 1]), (next_pv >> 1) & 1, 1000);
                        else if (qk_possible && !pv_possible)
                            mbar_try_wait_hint(tc::smem_u32(&kv_full[next_qk & 1]), (next_qk >> 1) & 1, 1000);
                        const uint64_t now = tc::global_timer_ns();
                        if (t_idle == 0) t_idle = now;
                        else if (now - t_idle > tc::kWaitNs) {
                            *abort_flag = 1;
                            flag(P.status, DSV4_DEV_TIMEOUT);
                            ok = false;
                        }
                    }
                }
            }
        } else if (warp >= 4) {
            // ------------------------------------------------------ producers
            const int pt = threadIdx.x - 128;
            const int pw = warp - 4;                           // producer warp: rows pw, pw + 4, ... of a tile
            const int n_ckeys = n_comp_mine * kTcKeys;
            // 1. pointer table of the owned compressed rows (row e: tile
            //    e / 32 of this CTA's compressed tiles, slot-list key 32 ct + e % 32);
            //    all index, block-table and scale loads of a phase issued together
            {
                constexpr int kPer = kTcMaxKeys / 128;
                int slot[kPer];
                int pg[kPer];
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int e = pt + 128 * i;
                    slot[i] = -1;
                    if (e < n_ckeys) {
                        const int ct = rank + (n_swa_mine + (e >> 5)) * C - n_swa_t;
                        const int key = ct * kTcKeys + (e & 31);
                        if (key < n_comp) slot[i] = P.idx[static_cast<long long>(b) * P.idx_stride + key];
                    }
                }
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    pg[i] = -1;
                    if (slot[i] >= 0 && (slot[i] >> 6) < P.comp_bt_stride)
                        pg[i] = P.comp_bt[static_cast<long long>(b) * P.comp_bt_stride + (slot[i] >> 6)];
                    else if (slot[i] != -1)
                        flag(P.status, DSV4_DEV_BAD_INDEX);
                }
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int e = pt + 128 * i;
                    if (e >= n_ckeys) continue;
                    uint64_t ent = 0;
                    uint2 sc = make_uint2(0, 0);
                    if (pg[i] >= 0 && pg[i] < P.comp_pages) {
                        const uint8_t* page = P.comp + static_cast<long long>(pg[i]) * kMlaPage;
                        const int r = slot[i] & (kPage - 1);
                        ent = reinterpret_cast<uint64_t>(page + r * kMlaData) | 3u;
                        sc = *reinterpret_cast<const uint2*>(page + kPage * kMlaData + r * 8);
                    } else if (slot[i] >= 0) {
                        flag(P.status, DSV4_DEV_BAD_PAGE);
                    }
                    table[e] = make_uint4(static_cast<uint32_t>(ent), static_cast<uint32_t>(ent >> 32), sc.x, sc.y);
                }
            }
            __threadfence_block();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(table_ready));
            bool ok = tc::mbar_wait(tc::smem_u32(table_ready), 0, abort_flag, P.status);
            // 2. compressed rows of tile jc: each lane copies its 16-byte units of
            //    its warp's rows (units lane and 32 + lane) into the raw stage,
            //    the same units it converts later (no cross-thread handoff)
            auto issue_comp = [&](int jc) {
                uint8_t* rbase = raw_s + (jc & 1) * kTcRawBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int r = pw + 4 * kk;
                    const uint4 e = table[jc * kTcKeys + r];
                    if ((e.x & 3u) != 3u) continue;
                    const uint8_t* src = reinterpret_cast<const uint8_t*>((static_cast<uint64_t>(e.y) << 32 | e.x) & ~uint64_t(15));
                    tc::cp_async16(tc::smem_u32(rbase + r * kMlaData + lane * 16), src + lane * 16);
                    if (lane < 8) tc::cp_async16(tc::smem_u32(rbase + r * kMlaData + kNope + lane * 16), src + kNope + lane * 16);
                }
                tc::cp_async_commit();
            };
            if (ok && n_comp_mine > 0) issue_comp(0);
            if (ok && n_comp_mine > 1) issue_comp(1);
            for (int i = 0; ok && i < n_tiles; ++i) {
                const int kst = i & 1;
                uint8_t* kp = k_s + kst * kTcKBytes;
                if (i >= kTcStages &&
                    !tc::mbar_wait(tc::smem_u32(&kv_empty[kst]), ((i >> 1) & 1) ^ 1, abort_flag, P.status))
                    break;
                if (i < n_swa_mine) {
                    // window tile: nine TMA tensor loads (64 dims x 32 tokens each)
                    // land it swizzled; nothing to convert
                    if (pt == 0) {
                        const int a = A0 + rank + i * C;
                        const int tok = a * kTcKeys;
                        int pg = ((tok >> 6) < P.swa_bt_stride) ? P.swa_bt[static_cast<long long>(b) * P.swa_bt_stride + (tok >> 6)] : -1;
                        if (pg < 0 || pg >= P.swa_pages) {
                            flag(P.status, DSV4_DEV_BAD_PAGE);
                            pg = -1;                               // outside the map: the load reads zeros
                        }
                        const uint32_t bar = tc::smem_u32(&swa_full[kst]);
                        tc::mbar_arrive_expect_tx(bar, kTcKBytes);
                        for (int c = 0; c < 9; ++c)
                            tc::tma_load_3d(tc::smem_u32(kp + c * kTcKChunk), &tm_swa, bar, c * 64, tok & 63, pg);
                    }
                    if (!tc::mbar_wait(tc::smem_u32(&swa_full[kst]), (i >> 1) & 1, abort_flag, P.status)) break;
                } else {
                    const int jc = i - n_swa_mine;
                    if (jc + 1 < n_comp_mine) asm volatile("cp.async.wait_group 1;" ::: "memory");
                    else asm volatile("cp.async.wait_group 0;" ::: "memory");
                    const uint8_t* rbase = raw_s + (jc & 1) * kTcRawBytes;
#pragma unroll 2
                    for (int kk = 0; kk < 8; ++kk) {
                        const int r = pw + 4 * kk;
                        const uint4 e = table[jc * kTcKeys + r];
                        const int sw = r & 7;
                        if ((e.x & 3u) == 3u) {
                            // lane: nope unit lane (dims 16 lane.., UE8M0 block lane/4);
                            // lanes 0-7: rope unit (bf16, copied)
                            const int blk = lane >> 2;
                            const uint32_t byte = (blk < 4 ? (e.z >> (8 * blk)) : (e.w >> (8 * (blk - 4)))) & 0xffu;
                            uint4 lo, hi;
                            dequant16(*reinterpret_cast<const uint4*>(rbase + r * kMlaData + lane * 16), byte, lo, hi);
                            const int w0 = 2 * (lane & 3);
                            uint8_t* row = kp + blk * kTcKChunk + r * 128;
                            *reinterpret_cast<uint4*>(row + ((w0 ^ sw) << 4)) = lo;
                            *reinterpret_cast<uint4*>(row + (((w0 + 1) ^ sw) << 4)) = hi;
                            if (lane < 8)
                                *reinterpret_cast<uint4*>(kp + 8 * kTcKChunk + r * 128 + ((lane ^ sw) << 4)) =
                                    *reinterpret_cast<const uint4*>(rbase + r * kMlaData + kNope + lane * 16);
                        } else {
                            // padding or unreadable row: zeros (masked in the softmax)
#pragma unroll
                            for (int q = 0; q < 3; ++q) {
                                const int w = lane + 32 * q;
                                if (w < 72)
                                    *reinterpret_cast<uint4*>(kp + (w >> 3) * kTcKChunk + r * 128 + (((w & 7) ^ sw) << 4)) =
                                        make_uint4(0, 0, 0, 0);
                            }
                        }
                    }
                    if (jc + 2 < n_comp_mine) issue_comp(jc + 2);
                    tc::fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&kv_full[kst]));
            }
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        } else {
            // ------------------------------------------- softmax + O correction
            const bool real = lane < 16;                  // S row h = 16*warp + lane sits in lane 32*warp + lane
            const int h = warp * 16 + (lane & 15);
            float m = -INFINITY, l = 0.f;
            for (int t = 0; t < n_tiles; ++t) {
                const int sb = t & 1;
                if (!tc::mbar_wait(tc::smem_u32(&s_full[sb]), (t >> 1) & 1, abort_flag, P.status)) break;
                tc::tc_fence_after();
                // rows of this tile that are keys of the query
                const int gt = rank + t * C;
                int lo_r, hi_r;
                if (gt < n_swa_t) {
                    const int tok0 = (A0 + gt) * kTcKeys;
                    lo_r = max(0, t0 - tok0);
                    hi_r = min(kTcKeys, p - tok0 + 1);
                } else {
                    lo_r = 0;
                    hi_r = min(kTcKeys, n_comp - (gt - n_swa_t) * kTcKeys);
                }
                float s[32];
                float mx = -INFINITY;
                tc::tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + sb * kTcKeys, s);
                tc::tmem_ld_wait();
                if (real) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        s[j] = (j >= lo_r && j < hi_r) ? s[j] * scale_log2 : -INFINITY;
                        mx = fmaxf(mx, s[j]);
                    }
                }
                const float m_new = fmaxf(m, mx);
                const bool need = real && (m_new > m + 8.0f);
                const float m_use = need ? m_new : m;
                uint32_t pk[16];
                float rowsum = 0.f;
                if (real) {
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float e0 = (j >= lo_r && j < hi_r) ? ex2_approx(s[j] - m_use) : 0.f;
                        const float e1 = (j + 1 >= lo_r && j + 1 < hi_r) ? ex2_approx(s[j + 1] - m_use) : 0.f;
                        const __nv_bfloat162 bb = __floats2bfloat162_rn(e0, e1);
                        const float2 rb = __bfloat1622float2(bb);
                        rowsum += rb.x + rb.y;
                        pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&bb);
                    }
                }
                if (t >= 1 && !tc::mbar_wait(tc::smem_u32(&pv_done[(t - 1) & 1]), ((t - 1) >> 1) & 1, abort_flag, P.status))
                    break;
                const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
                if (real) sm_alpha[h] = alpha;
                const int any_w = __any_sync(0xffffffffu, need);
                if (lane == 0) sm_any[sb * 4 + warp] = any_w;
                __threadfence_block();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sync4[sb]));
                if (!tc::mbar_wait(tc::smem_u32(&sync4[sb]), (t >> 1) & 1, abort_flag, P.status)) break;
                const bool any = (sm_any[sb * 4 + 0] | sm_any[sb * 4 + 1] | sm_any[sb * 4 + 2] | sm_any[sb * 4 + 3]) != 0;
                if (any && t >= 1) {
                    tc::tc_fence_after();
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
#pragma unroll 1
                        for (int half = 0; half < 2; ++half) {
                            const uint32_t ta = tmem + (static_cast<uint32_t>(warp * 32) << 16) + kTcOCol + i * 64 + half * 32;
                            float o[32];
                            tc::tmem_ld32(ta, o);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 32; ++j) o[j] *= sm_alpha[half * 32 + j];
                            tc::tmem_st32(ta, o);
                        }
                    }
                    tc::tmem_st_wait();
                }
                if (real) {
                    l = l * alpha + rowsum;
                    m = m_use;
                    uint8_t* prow = p_s + sb * kTcPBytes + h * 128;
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        *reinterpret_cast<uint4*>(prow + ((u ^ (h & 7)) << 4)) =
                            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                }
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&p_full[sb]));
            }
            if (real) {
                sm_m[h] = m;
                sm_l[h] = l;
            }
            tc::mbar_wait(tc::smem_u32(&pv_done[(n_tiles - 1) & 1]), ((n_tiles - 1) >> 1) & 1, abort_flag, P.status);
            tc::tc_fence_before();
        }
    }

    // ------------------------------------------------------------- epilogue
    __syncthreads();
    tc::tc_fence_after();
    float* stage_o = reinterpret_cast<float*>(smem + kStageO);    // [64 heads][512]
    if (n_tiles > 0 && !*abort_flag) {
        if (warp < 8) {
            const int q4 = warp & 3;
#pragma unroll 1
            for (int bi = 0; bi < 2; ++bi) {
                const int i = (warp >> 2) * 2 + bi;
                const int v = i * 128 + q4 * 32 + lane;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float o[32];
                    tc::tmem_ld32(tmem + (static_cast<uint32_t>(q4 * 32) << 16) + kTcOCol + i * 64 + half * 32, o);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) stage_o[(half * 32 + j) * 512 + v] = o[j];
                }
            }
        }
    } else {
        for (int i = threadIdx.x; i < 64 * 512; i += kTcThreads) stage_o[i] = 0.f;
        if (threadIdx.x < 64) {
            sm_m[threadIdx.x] = -INFINITY;
            sm_l[threadIdx.x] = 0.f;
        }
    }
    __syncthreads();
    tc::cluster_sync();
    if (threadIdx.x < 64) {
        const int hh = threadIdx.x;
        float mq[8], lq[8];
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            mq[q] = -INFINITY;
            lq[q] = 0.f;
            if (q < C) {
                mq[q] = tc::ld_cluster_f32(tc::map_to_rank(tc::smem_u32(sm_m + hh), q));
                lq[q] = tc::ld_cluster_f32(tc::map_to_rank(tc::smem_u32(sm_l + hh), q));
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) M = fmaxf(M, mq[q]);
        float L = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (q < C) {
                const float wq = (mq[q] == -INFINITY) ? 0.f : exp2f(mq[q] - M);
                red_w[q * 64 + hh] = wq;
                L += wq * lq[q];
            }
        }
        red_invl[hh] = L > 0.f ? 1.0f / L : 0.f;
        if (rank == 0 && hh < nh && P.lse)
            P.lse[static_cast<long long>(b) * P.H + h0 + hh] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    const int VS = kV / C;                  // value dims merged by this CTA
    const int per_h = VS / 4;
    for (int it = threadIdx.x; it < nh * per_h; it += kTcThreads) {
        const int hh = it / per_h;
        const int v = rank * VS + (it % per_h) * 4;
        const uint32_t local = tc::smem_u32(stage_o + hh * 512 + v);
        float4 x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)                   // all remote loads in flight together
            if (q < C) x[q] = tc::ld_cluster_v4(tc::map_to_rank(local, q));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (q < C) {
                const float wq = red_w[q * 64 + hh];
                acc.x += wq * x[q].x;
                acc.y += wq * x[q].y;
                acc.z += wq * x[q].z;
                acc.w += wq * x[q].w;
            }
        }
        const float il = red_invl[hh];
        const __nv_bfloat162 o01 = __floats2bfloat162_rn(acc.x * il, acc.y * il);
        const __nv_bfloat162 o23 = __floats2bfloat162_rn(acc.z * il, acc.w * il);
        uint2 pk2;
        pk2.x = *reinterpret_cast<const uint32_t*>(&o01);
        pk2.y = *reinterpret_cast<const uint32_t*>(&o23);
        *reinterpret_cast<uint2*>(P.out + (static_cast<long long>(b) * P.H + h0 + hh) * kV + v) = pk2;
    }
    tc::cluster_sync();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTcTmemCols);
    }
}

}  // namespace dsv4

using namespace dsv4;

extern "C" dsv4_status dsv4_sparse_mla_decode(const dsv4_plan* plan, const dsv4_mla_args* a,
                                              void* workspace, size_t workspace_bytes,
                                              dsv4_stream_t stream)
{
    if (plan == nullptr || a == nullptr) return DSV4_ERR_INVALID;
    if (workspace_bytes < plan->ws_bytes || (workspace == nullptr && plan->ws_bytes)) return DSV4_ERR_SHAPE;
    if (!a->q_dev || !a->swa_cache_dev || !a->swa_block_table_dev || !a->ctx_len_dev || !a->out_dev)
        return DSV4_ERR_INVALID;
    const bool sparse = plan->type != DSV4_SWAONLY;
    if (sparse && (!a->comp_cache_dev || !a->comp_block_table_dev || !a->topk_idx_dev || !a->topk_len_dev))
        return DSV4_ERR_INVALID;
    if (sparse && a->topk_stride < plan->topk) return DSV4_ERR_SHAPE;
    MlaParams P;
    P.q = static_cast<const uint16_t*>(a->q_dev);
    P.swa = static_cast<const uint8_t*>(a->swa_cache_dev);
    P.swa_pages = a->swa_num_pages;
    P.swa_bt = a->swa_block_table_dev;
    P.swa_bt_stride = a->swa_bt_stride;
    P.comp = sparse ? static_cast<const uint8_t*>(a->comp_cache_dev) : nullptr;
    P.comp_pages = a->comp_num_pages;
    P.comp_bt = sparse ? a->comp_block_table_dev : nullptr;
    P.comp_bt_stride = a->comp_bt_stride;
    P.idx = sparse ? a->topk_idx_dev : nullptr;
    P.idx_stride = a->topk_stride;
    P.idx_len = sparse ? a->topk_len_dev : nullptr;
    P.ctx_len = a->ctx_len_dev;
    P.out = static_cast<uint16_t*>(a->out_dev);
    P.lse = a->lse_dev;
    P.H = plan->geom.n_heads;
    P.window = plan->geom.window;
    P.scale = plan->geom.softmax_scale;
    P.status = a->status_dev;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MlaTcParams T;
    T.base = P;
    T.head_groups = plan->mla_head_groups;
    T.cluster = plan->mla_splits;
    T.topk = plan->topk;
    CUtensorMap tm_q;
    const uint64_t qdims[2] = {static_cast<uint64_t>(kHead), static_cast<uint64_t>(plan->batch) * P.H};
    const uint64_t qstr[1] = {static_cast<uint64_t>(kHead) * 2};
    const uint32_t qbox[2] = {64, 64};
    if ((reinterpret_cast<uintptr_t>(a->q_dev) & 15) || (reinterpret_cast<uintptr_t>(a->swa_cache_dev) & 15) ||
        (sparse && (reinterpret_cast<uintptr_t>(a->comp_cache_dev) & 15)))
        return DSV4_ERR_SHAPE;
    if (!encode_tmap(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->q_dev, qdims, qstr, qbox,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return DSV4_ERR_CUDA;
    CUtensorMap tm_swa;
    const uint64_t sdims[3] = {static_cast<uint64_t>(kHead), static_cast<uint64_t>(kPage),
                               static_cast<uint64_t>(a->swa_num_pages > 0 ? a->swa_num_pages : 1)};
    const uint64_t sstr[2] = {static_cast<uint64_t>(kHead) * 2, static_cast<uint64_t>(kSwaPage)};
    const uint32_t sbox[3] = {64, static_cast<uint32_t>(kTcKeys), 1};
    if (!encode_tmap(&tm_swa, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a->swa_cache_dev, sdims, sstr, sbox,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return DSV4_ERR_CUDA;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(mla_decode_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T.cluster, plan->batch * T.head_groups, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = kTcSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = T.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_decode_tc, tm_q, tm_swa, T);
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
