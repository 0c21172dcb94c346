// mla.cu -- sparse absorbed-MQA decode over (selected compressed slots) ||
// (SWA window), one 576-dim latent KV head, value = the 512 latent dims; and
// the V4-native variant: one 512-dim head (448 FP8 nope + 64 bf16 rope) that
// is both key and value, with the SWA window in the same FP8 row format.
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
#include "host_once.h"
#include "out_quant.h"

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
    // prefill rows: block-table row of query row b (NULL: b), bt_rows rows
    const int* row_seq;
    int bt_rows;
};

// ---------------------------------------------------------------------------
// Tensor-core decode attention (tcgen05, TMEM accumulators).
//
// CTA = (rank r of a cluster of C CTAs, sequence b x 64-head group g).  The
// keys of a sequence come as 64-key tiles: first the SWA window as whole
// 64-token cache pages (rows outside the window masked), then the selected
// compressed slots in list order (rows past the selection masked).  Tile j of
// that list belongs to CTA j mod C.  Each CTA runs an online softmax over its
// tiles; then every CTA pushes each 512/C-dim slice of its unnormalised O,
// with its running max and sum, into the shared memory of the CTA that owns
// the slice, which combines the C parts and stores the output -- no partials
// in HBM, no combine kernel.
//
//   S  = Q K^T      kind::f16, M = 64 head rows (row r in TMEM lane
//                   32*(r/16) + r%16), N = 64 keys, K = 576: 36 MMAs per
//                   tile, double-buffered in TMEM columns [0, 128).
//   O^T += V^T P^T  M = 128 value dims (4 blocks), N = 64 heads, K = 64 keys:
//                   V^T is the key tile read as an MN-major operand; O^T sits
//                   in TMEM columns [128, 384).
// A single thread issues one tcgen05.mma about every 20 ns whatever its shape
// (up to N = 64), so the tile is as wide as two bf16 tiles and Q fit in
// shared memory.  Once QK(t) is done the tile's RoPE chunk is free; P(t)
// (bf16, 64 heads x 64 keys) is written there, so P is double-buffered with
// the stages.
// Warps 0-3: softmax (lanes 0-15 = 16 heads each) and O^T correction; warps
// 4-11: producers (window pages by TMA; compressed rows loaded into registers
// one tile ahead and dequantised into the swizzled tile); warp 12: Q load and
// QK issue; warp 13: PV issue (two issuers keep PV(t) off QK(t+1)'s path).
//
// V4-native rows ([MLA-to-CSA] 5.5: K = V, FP8 SWA at 584 bytes): Q and K
// are 8 chunks of 64 dims (448 nope + 64 rope), the value is the whole key
// tile, so P(t) gets a buffer of its own (double-buffered, reused once PV(t-2)
// is complete); window tiles are FP8 rows too and go through the producers'
// register gather like the compressed ones.
// ---------------------------------------------------------------------------
constexpr int kTcKeys = 64;
constexpr int kTcStages = 2;
constexpr int kTcQChunk = 64 * 128;                        // 64 head rows x 64 dims (bf16)
constexpr int kTcQBytes = 9 * kTcQChunk;                   // 73728
constexpr int kTcKChunk = kTcKeys * 128;                   // 64 key rows x 64 dims
constexpr int kTcKBytes = 9 * kTcKChunk;                   // 73728 per stage
constexpr int kTcMaxCompTiles = 16;                        // compressed tiles one CTA can own
constexpr int kTcProdWarps = 8;
constexpr int kTcMmaWarp = 4 + kTcProdWarps;               // 12: Q load, QK issue
constexpr int kTcPvWarp = kTcMmaWarp + 1;                  // 13: PV issue
constexpr int kTcThreads = 32 * (kTcPvWarp + 1);           // 448
constexpr int kTcMaxTiles = 24;                            // per-tile PV completion barriers
constexpr int kTcTmemCols = 512;
constexpr int kTcOCol = 128;
constexpr int kOffQ = 0;
constexpr int kOffK = kTcQBytes;
constexpr int kOffMisc = kOffK + kTcStages * kTcKBytes;    // 221184
constexpr int kMiscBytes = 2048 + 4 * 1024;                   // + the compressed block-table row
constexpr int kBtSmem = 1024;                               // block-table entries kept in shared memory
constexpr int kTcSmem = kOffMisc + kMiscBytes + 1024;      // + alignment slack of the dynamic base
// epilogue buffers (in the Q / K space once the main loop is over): a slice
// is bf16 [512/C dims][64 heads] (16-byte head groups swizzled by dim) plus
// fp32 [64][2] running max and sum; receive slots [C], send slots [C], merge
// weights [8][64] and 1 / L [64]
constexpr int kOffRecv = 0;
constexpr int kEpiParts = 4;                               // a slice moves in 4 parts (by dim), merged as they land
constexpr int kOffSend = 64 * kV * 2 + 8 * 512;
constexpr int kOffWeights = 2 * kOffSend;
static_assert(kOffWeights + 9 * 64 * 4 <= kOffMisc, "epilogue buffers fit in the Q / K space");
static_assert(kTcSmem <= 232448, "shared memory budget");

// Shared-memory plan and cache-row geometry of the two variants.
template <bool V4>
struct AttnGeom {
    static constexpr int kChunks = V4 ? 8 : 9;                  // 64-dim chunks of Q and K
    static constexpr int kQBytes = kChunks * kTcQChunk;
    static constexpr int kKBytes = kChunks * kTcKChunk;         // per stage
    static constexpr int kOffK = kQBytes;
    static constexpr int kOffP = kOffK + kTcStages * kKBytes;   // V4: P(t) double buffer
    static constexpr int kPBytes = V4 ? 2 * kTcKChunk : 0;
    static constexpr int kOffMisc = kOffP + kPBytes;
    static constexpr int kSmem = kOffMisc + kMiscBytes + 1024;
    static constexpr int kRowBytes = V4 ? DSV4_V4_NOPE_DIM + 2 * kRope : kMlaData;   // data bytes of a row
    static constexpr int kNopeBytes = V4 ? DSV4_V4_NOPE_DIM : kNope;
    static constexpr int kPageBytes = V4 ? DSV4_V4_PAGE_BYTES : kMlaPage;
    static constexpr int kNopeLanes = kNopeBytes / 16;          // lanes holding a 16-code unit of a row
};
static_assert(AttnGeom<false>::kOffMisc == kOffMisc && AttnGeom<false>::kSmem == kTcSmem, "576 plan");
static_assert(AttnGeom<true>::kSmem <= 232448, "shared memory budget (V4)");
static_assert(kOffWeights + 9 * 64 * 4 <= AttnGeom<true>::kOffMisc, "epilogue buffers fit (V4)");

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

// 16 FP8 E4M3 codes times 2^E -> 16 bf16, E = scale_byte - 127 (UE8M0).
// Placing a code's 7 magnitude bits at bits 4-10 of a bf16 and its sign at
// bit 15 gives a bf16 whose value is the code's value times 2^-120 (exponent
// field 0 gives exactly the scaled subnormal codes).  Multiplying by 2^(E+120)
// in one or two exact power-of-two steps restores the value; results in the
// bf16 normal range are exact.  Integer and bf16x2 pipes only.
__device__ __forceinline__ __nv_bfloat162 e4m3_pair_scaled(uint32_t t)   // t: codes in bytes 1 and 3
{
    const uint32_t v = ((t >> 4) & 0x07f007f0u) | (t & 0x80008000u);
    return *reinterpret_cast<const __nv_bfloat162*>(&v);
}

__device__ __forceinline__ void dequant16(const uint4 w, uint32_t scale_byte, uint4& lo, uint4& hi)
{
    const int k = static_cast<int>(scale_byte) - 7;          // E + 120, in [-7, 248]
    const int ka = k < 127 ? k : 127;
    const uint32_t ba = static_cast<uint32_t>(ka + 127) << 7;        // bf16 2^ka
    const uint32_t bb = static_cast<uint32_t>(k - ka + 127) << 7;    // bf16 2^(k - ka)
    const uint32_t ma2 = ba | (ba << 16), mb2 = bb | (bb << 16);
    const __nv_bfloat162 ma = *reinterpret_cast<const __nv_bfloat162*>(&ma2);
    const __nv_bfloat162 mb = *reinterpret_cast<const __nv_bfloat162*>(&mb2);
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 x0 = __hmul2(e4m3_pair_scaled(__byte_perm(in[i], 0u, 0x1404)), ma);   // codes 0, 1
        __nv_bfloat162 x1 = __hmul2(e4m3_pair_scaled(__byte_perm(in[i], 0u, 0x3424)), ma);   // codes 2, 3
        if (k > 127) {
            x0 = __hmul2(x0, mb);
            x1 = __hmul2(x1, mb);
        }
        out[2 * i] = *reinterpret_cast<const uint32_t*>(&x0);
        out[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&x1);
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

// Loads that run only when `pred` holds and otherwise leave a default: the
// default and the load are one predicated sequence, so nothing that reads the
// result sits between one load and the next (a select after each load would
// wait for it and serialise the gather).  p is not dereferenced when pred is
// false.
__device__ __forceinline__ uint4 ldg_stream_v4_if(const uint8_t* p, bool pred)
{
    uint4 v;
    asm volatile("{\n\t.reg .pred q;\n\t"
                 "setp.ne.u32 q, %5, 0;\n\t"
                 "mov.u32 %0, 0;\n\tmov.u32 %1, 0;\n\tmov.u32 %2, 0;\n\tmov.u32 %3, 0;\n\t"
                 "@q ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
                 : "=&r"(v.x), "=&r"(v.y), "=&r"(v.z), "=&r"(v.w)
                 : "l"(p), "r"(static_cast<uint32_t>(pred)));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream_u8_if(const uint8_t* p, bool pred, uint32_t dflt)
{
    uint32_t v;
    asm volatile("{\n\t.reg .pred q;\n\t.reg .u16 h;\n\t"
                 "setp.ne.u32 q, %2, 0;\n\t"
                 "mov.u32 %0, %3;\n\t"
                 "@q ld.global.nc.L1::no_allocate.u8 h, [%1];\n\t"
                 "@q cvt.u32.u16 %0, h;\n\t}"
                 : "=&r"(v)
                 : "l"(p), "r"(static_cast<uint32_t>(pred)), "r"(dflt));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream_u32_if(const uint8_t* p, bool pred, uint32_t dflt)
{
    uint32_t v;
    asm volatile("{\n\t.reg .pred q;\n\t"
                 "setp.ne.u32 q, %2, 0;\n\t"
                 "mov.u32 %0, %3;\n\t"
                 "@q ld.global.nc.L1::no_allocate.u32 %0, [%1];\n\t}"
                 : "=&r"(v)
                 : "l"(p), "r"(static_cast<uint32_t>(pred)), "r"(dflt));
    return v;
}

// L2 load of an int written by the grid before this one, or dflt
__device__ __forceinline__ int ldcg_s32_if(const int* p, bool pred, int dflt)
{
    int v;
    asm volatile("{\n\t.reg .pred q;\n\t"
                 "setp.ne.u32 q, %2, 0;\n\t"
                 "mov.b32 %0, %3;\n\t"
                 "@q ld.global.cg.b32 %0, [%1];\n\t}"
                 : "=&r"(v)
                 : "l"(p), "r"(static_cast<uint32_t>(pred)), "r"(dflt));
    return v;
}

template <bool V4>
__global__ void __launch_bounds__(kTcThreads, 1)
mla_decode_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_swa, MlaTcParams T)
{
    using G = AttnGeom<V4>;
    const MlaParams& P = T.base;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = tc::align1024_shared(smem_raw);
    uint8_t* q_s = smem + kOffQ;
    uint8_t* k_s = smem + G::kOffK;
    uint8_t* p_s = smem + G::kOffP;    // V4 only
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::kOffMisc);
    uint64_t* kv_full = bars;          // [2] producers (8 warps; window tiles: + TMA bytes) -> MMA
    uint64_t* kv_empty = bars + 2;     // [2] MMA -> producers (stage read by QK and PV)
    uint64_t* s_full = bars + 4;       // [2] MMA -> softmax
    uint64_t* p_full = bars + 6;       // [2] softmax (4 warps) -> MMA: P written, S read, O^T corrected
    uint64_t* q_full = bars + 8;
    uint64_t* sync4 = bars + 9;        // [2] the four softmax warps meet once per tile
    uint64_t* recv_ml = bars + 11;     // epilogue: the C - 1 peers' running max and sum have landed (bytes)
    uint64_t* pv_done = bars + 12;     // [kTcMaxTiles] PV(u) complete (one phase each)
    uint64_t* recv_part = bars + 13 + kTcMaxTiles;                // [kEpiParts] epilogue: part p of the peer slices
    float* sm_m = reinterpret_cast<float*>(recv_part + kEpiParts); // [64] running max (log2 domain)
    float* sm_l = sm_m + 64;                              // [64] running sum
    float* sm_alpha = sm_l + 64;                          // [2][64] correction factors (by tile parity)
    int* sm_any = reinterpret_cast<int*>(sm_alpha + 128); // [2][4]
    volatile int* abort_flag = sm_any + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm_any + 9);
    int* bt_s = reinterpret_cast<int*>(smem + G::kOffMisc + 2048);  // [kBtSmem] this sequence's block-table row
    uint64_t* bt_ready = bars + 12 + kTcMaxTiles;                 // producers: bt_s loaded

    const int rank = blockIdx.x;                          // the cluster spans gridDim.x
    const int b = blockIdx.y / T.head_groups, g_head = blockIdx.y % T.head_groups;
    // the query row's block-table row (prefill rows map to their sequence's)
    int seq = b;
    if (P.row_seq) {
        seq = P.row_seq[b];
        if (seq < 0 || seq >= P.bt_rows) {
            if (threadIdx.x == 0) flag(P.status, DSV4_DEV_BAD_INDEX);
            seq = 0;
        }
    }
    const int h0 = g_head * 64;
    const int nh = min(64, P.H - h0);
    const int p = P.ctx_len[b] - 1;
    const int t0 = max(0, p - P.window + 1);
    const int C = T.cluster;
    const int pg0 = t0 >> 6;                              // first window page (64 tokens)
    const int n_swa_t = p >= 0 ? (p >> 6) - pg0 + 1 : 0;
    const int n_swa_mine = min(n_swa_t > rank ? (n_swa_t - rank + C - 1) / C : 0, kTcMaxTiles);
    // The selected slots come from the kernel launched before this one, which
    // this kernel may overlap (programmatic dependent launch): n_comp and the
    // tile counts are read after griddepcontrol.wait, by every thread once,
    // when it first needs them.  The window tiles need none of it.
    int n_comp = 0, n_tiles = n_swa_mine, n_comp_mine = 0;
    bool resolved = false;
    auto resolve = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // written by the grid before: L2 loads after the wait
        n_comp = P.idx_len ? min(max(__ldcg(P.idx_len + b), 0), T.topk) : 0;
        const int n_glob = n_swa_t + (n_comp + kTcKeys - 1) / kTcKeys;
        n_tiles = n_glob > rank ? (n_glob - rank + C - 1) / C : 0;
        if (n_tiles - n_swa_mine > kTcMaxCompTiles || n_tiles > kTcMaxTiles) {
            if (threadIdx.x == 0) flag(P.status, DSV4_DEV_BAD_INDEX);
            n_tiles = min(n_swa_mine + kTcMaxCompTiles, kTcMaxTiles);
        }
        n_comp_mine = n_tiles - n_swa_mine;
        resolved = true;
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float scale_log2 = P.scale * 1.4426950408889634f;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(tc::smem_u32(&kv_full[i]), kTcProdWarps);
            tc::mbar_init(tc::smem_u32(&kv_empty[i]), 1);
            tc::mbar_init(tc::smem_u32(&s_full[i]), 1);
            tc::mbar_init(tc::smem_u32(&sync4[i]), 4);
            tc::mbar_init(tc::smem_u32(&p_full[i]), 4);
        }
        for (int i = 0; i < kTcMaxTiles; ++i) tc::mbar_init(tc::smem_u32(&pv_done[i]), 1);
        tc::mbar_init(tc::smem_u32(bt_ready), kTcProdWarps);
        tc::mbar_init(tc::smem_u32(q_full), 1);
        tc::mbar_init(tc::smem_u32(recv_ml), 1);
        for (int i = 0; i < kEpiParts; ++i) tc::mbar_init(tc::smem_u32(&recv_part[i]), 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
        // the query's loads are in flight during the rest of the set-up
        tc::prefetch_tensormap(&tm_q);
        tc::mbar_arrive_expect_tx(tc::smem_u32(q_full), G::kQBytes);
        for (int c = 0; c < G::kChunks; ++c)
            tc::tma_load_2d(tc::smem_u32(q_s + c * kTcQChunk), &tm_q, tc::smem_u32(q_full), c * 64, b * P.H + h0);
    }
    if (threadIdx.x < 64) {
        sm_m[threadIdx.x] = -INFINITY;
        sm_l[threadIdx.x] = 0.f;
    }
    if (warp == kTcMmaWarp) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), kTcTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    {
        if (warp == kTcMmaWarp) {
            // ------------------------------------------------------- QK issue
            // QK(t) needs tile t loaded and S buffer t%2 read out by the
            // softmax (P(t-2) written).
            if (lane == 0) {
                tc::prefetch_tensormap(&tm_swa);
                constexpr uint32_t id_qk = tc::idesc(64, kTcKeys, tc::kFmtBF16, tc::kFmtBF16);
                bool ok = tc::mbar_wait(tc::smem_u32(q_full), 0, abort_flag, P.status);
                const uint64_t qd = tc::desc_kmajor_sw128(tc::smem_u32(q_s));
                for (int t = 0; ok; ++t) {
                    if (t == n_swa_mine) resolve();
                    if (t >= n_tiles) break;
                    ok = tc::mbar_wait(tc::smem_u32(&kv_full[t & 1]), (t >> 1) & 1, abort_flag, P.status);
                    if (ok && t >= 2)
                        ok = tc::mbar_wait(tc::smem_u32(&p_full[t & 1]), ((t - 2) >> 1) & 1, abort_flag, P.status);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint32_t d = tmem + (t & 1) * kTcKeys;
                    const uint64_t kd = tc::desc_kmajor_sw128(tc::smem_u32(k_s + (t & 1) * G::kKBytes));
#pragma unroll
                    for (int c = 0; c < G::kChunks; ++c)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc::mma_f16(d, qd + (c * kTcQChunk >> 4) + 2 * k, kd + (c * kTcKChunk >> 4) + 2 * k,
                                        id_qk, (c | k) != 0 ? 1u : 0u);
                    tc::mma_commit(tc::smem_u32(&s_full[t & 1]));
                }
            }
        } else if (warp == kTcPvWarp) {
            // ------------------------------------------------------- PV issue
            // O^T += V^T P^T once P(u) is written (in the RoPE chunk of tile u;
            // V4: in P buffer u % 2).
            if (lane == 0) {
                constexpr uint32_t id_pv = tc::idesc(128, 64, tc::kFmtBF16, tc::kFmtBF16, true, false);
                for (int u = 0;; ++u) {
                    if (u == n_swa_mine) resolve();
                    if (u >= n_tiles) break;
                    if (!tc::mbar_wait(tc::smem_u32(&p_full[u & 1]), (u >> 1) & 1, abort_flag, P.status)) break;
                    tc::tc_fence_after();
                    const uint32_t kb = tc::smem_u32(k_s + (u & 1) * G::kKBytes);
                    const uint64_t pd = tc::desc_kmajor_sw128(V4 ? tc::smem_u32(p_s + (u & 1) * kTcKChunk)
                                                                 : kb + 8 * kTcKChunk);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            tc::mma_f16(tmem + kTcOCol + i * 64,
                                        tc::desc_mnmajor_sw128(kb + 2 * i * kTcKChunk + j * 2048, kTcKChunk, 1024),
                                        pd + 2 * j, id_pv, (u > 0 || j > 0) ? 1u : 0u);
                    tc::mma_commit(tc::smem_u32(&kv_empty[u & 1]));
                    tc::mma_commit(tc::smem_u32(&pv_done[u]));
                }
            }
        } else if (warp >= 4) {
            // ------------------------------------------------------ producers (warps 4-11)
            // Producer warp pw owns rows pw + 8k (k = 0..7) of every tile.
            const int pw = warp - 4;
            // the sequence's compressed block-table row (a caller input) into
            // shared memory while the window tiles run
            const bool bt_smem = P.comp_bt != nullptr && P.comp_bt_stride <= kBtSmem;
            if (bt_smem)
                for (int i = threadIdx.x - 128; i < P.comp_bt_stride; i += 32 * kTcProdWarps)
                    bt_s[i] = P.comp_bt[static_cast<long long>(seq) * P.comp_bt_stride + i];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(bt_ready));
            // Row table, spread over the lanes: lane l holds row pw + 8 (l % 8) of
            // compressed tiles 4q + l / 8 (q = 0..3) as page * 64 + row (-1:
            // padding or unreadable).  Index loads, then block-table loads, each
            // issued together.
            int ent[4] = {-1, -1, -1, -1};
            // The slots of every key this CTA could own (keys below top-k, all
            // in bounds) are loaded before the count is known, so that the two
            // loads overlap; keys at or past the count are dropped once it is.
            int slot[4];
            auto load_slots = [&]() {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int jc = 4 * q + (lane >> 3);
                    const int key = (rank + (n_swa_mine + jc) * C - n_swa_t) * kTcKeys + pw + 8 * (lane & 7);
                    slot[q] = ldcg_s32_if(P.idx + static_cast<long long>(b) * P.idx_stride + key,
                                          P.idx_len != nullptr && key < T.topk, -1);
                }
            };
            auto build_table = [&]() {
                int pg[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int jc = 4 * q + (lane >> 3);
                    const int key = (rank + (n_swa_mine + jc) * C - n_swa_t) * kTcKeys + pw + 8 * (lane & 7);
                    if (jc >= n_comp_mine || key >= n_comp) slot[q] = -1;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    pg[q] = -2;
                    if (slot[q] >= 0 && (slot[q] >> 6) < P.comp_bt_stride)
                        pg[q] = bt_smem ? bt_s[slot[q] >> 6]
                                        : P.comp_bt[static_cast<long long>(seq) * P.comp_bt_stride + (slot[q] >> 6)];
                    else if (slot[q] != -1)
                        flag(P.status, DSV4_DEV_BAD_INDEX);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ent[q] = -1;
                    if (pg[q] != -2) {
                        if (pg[q] >= 0 && pg[q] < P.comp_pages) ent[q] = pg[q] * kPage + (slot[q] & (kPage - 1));
                        else flag(P.status, DSV4_DEV_BAD_PAGE);
                    }
                }
            };
            // raw data of one tile, loaded one tile ahead of its use: nope unit
            // `lane` (16 codes; V4: lanes below 28) of rows pw + 8k, rope unit
            // lane % 8 of rows pw + 8 (lane / 8) and pw + 8 (lane / 8 + 4), and
            // the scales: the 576 rows' byte lane / 4 of rows pw + 8k, one load
            // each; the V4 rows' bytes 4 (lane / 8) .. + 3 of row pw + 8 (lane % 8)
            // on lanes 0-15 (each nope lane takes its byte by a shuffle when it
            // converts; measured faster for V4, slower for the 576 rows).
            // ent_of(k): cache entry (page * 64 + row) of row pw + 8k, -1 for
            // none (the row then reads as zeros).
            uint4 rn[8];
            uint32_t rs[V4 ? 1 : 8];
            uint4 rr[2];
            auto fetch_rows = [&](const uint8_t* cache, auto&& ent_of) {
                const bool nope_lane = lane < G::kNopeLanes;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int e = ent_of(k);
                    const uint8_t* page = cache + static_cast<long long>(e >> 6) * G::kPageBytes;
                    rn[k] = ldg_stream_v4_if(page + (e & 63) * G::kRowBytes + lane * 16, e >= 0 && nope_lane);
                    if constexpr (!V4)
                        rs[k] = ldg_stream_u8_if(page + kPage * G::kRowBytes + (e & 63) * 8 + (lane >> 2),
                                                 e >= 0 && nope_lane, 127);
                }
                if constexpr (V4) {
                    const int e = ent_of(lane & 7);
                    rs[0] = ldg_stream_u32_if(cache + static_cast<long long>(e >> 6) * G::kPageBytes +
                                                  kPage * G::kRowBytes + (e & 63) * 8 + 4 * ((lane >> 3) & 1),
                                              e >= 0 && lane < 16, 0x7f7f7f7fu);
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int e = ent_of((lane >> 3) + 4 * hh);
                    rr[hh] = ldg_stream_v4_if(cache + static_cast<long long>(e >> 6) * G::kPageBytes +
                                                  (e & 63) * G::kRowBytes + G::kNopeBytes + (lane & 7) * 16,
                                              e >= 0);
                }
            };
            auto fetch = [&](int jc) {
                const int q = jc >> 2;
                const int e_src = q == 0 ? ent[0] : (q == 1 ? ent[1] : (q == 2 ? ent[2] : ent[3]));
                const int base = (jc & 3) * 8;
                fetch_rows(P.comp, [&](int k) { return __shfl_sync(0xffffffffu, e_src, base + k); });
            };
            // dequantise into the 128-byte-swizzled tile (row r, 16-byte unit u
            // of 64-dim chunk c at c * kTcKChunk + r * 128 + ((u ^ (r & 7)) << 4);
            // r & 7 == pw for every row of this warp).  Lanes of odd chunks store
            // their two units in the other order, which halves bank conflicts.
            auto convert = [&](uint8_t* kp) {
                const int w0 = 2 * (lane & 3);
                const int flip = (lane >> 2) & 1;
                // scale byte lane / 4 of row pw + 8k (V4: byte lane / 4 % 4 of the
                // word that lane k + 8 (lane / 16) loaded)
                uint32_t sb[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if constexpr (V4)
                        sb[k] = (__shfl_sync(0xffffffffu, rs[0], k + 8 * (lane >> 4)) >> (8 * ((lane >> 2) & 3))) &
                                0xffu;
                    else
                        sb[k] = rs[k];
                }
                if (lane < G::kNopeLanes) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int r = pw + 8 * k;
                        uint4 lo, hi;
                        dequant16(rn[k], sb[k], lo, hi);
                        uint8_t* row = kp + (lane >> 2) * kTcKChunk + r * 128;
                        const uint4 first = flip ? hi : lo;
                        const uint4 second = flip ? lo : hi;
                        *reinterpret_cast<uint4*>(row + (((w0 + flip) ^ pw) << 4)) = first;
                        *reinterpret_cast<uint4*>(row + (((w0 + 1 - flip) ^ pw) << 4)) = second;
                    }
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = pw + 8 * ((lane >> 3) + 4 * hh);
                    *reinterpret_cast<uint4*>(kp + (G::kChunks - 1) * kTcKChunk + r * 128 +
                                              (((lane & 7) ^ pw) << 4)) = rr[hh];
                }
            };
            // window pages first: they need nothing from the kernel before
            int i = 0;
            bool ok = true;
            if constexpr (V4) {
                // FP8 window rows through the register gather, one tile ahead;
                // rows outside [t0, p] read as zeros
                auto fetch_win = [&](int wi) {
                    const int lp = pg0 + rank + wi * C;
                    int pg = lp < P.swa_bt_stride ? P.swa_bt[static_cast<long long>(seq) * P.swa_bt_stride + lp] : -1;
                    if (pg < 0 || pg >= P.swa_pages) {
                        if (lane == 0) flag(P.status, DSV4_DEV_BAD_PAGE);
                        pg = -1;
                    }
                    fetch_rows(P.swa, [&](int k) {
                        const int tok = lp * kPage + pw + 8 * k;
                        return (pg >= 0 && tok >= t0 && tok <= p) ? pg * kPage + pw + 8 * k : -1;
                    });
                };
                if (n_swa_mine > 0) fetch_win(0);
                for (; i < n_swa_mine; ++i) {
                    const int kst = i & 1;
                    uint8_t* kp = k_s + kst * G::kKBytes;
                    if (i >= kTcStages &&
                        !tc::mbar_wait(tc::smem_u32(&kv_empty[kst]), ((i >> 1) & 1) ^ 1, abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    convert(kp);
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&kv_full[kst]));
                    if (i + 1 < n_swa_mine) fetch_win(i + 1);
                }
            }
            for (; !V4 && i < n_swa_mine; ++i) {
                const int kst = i & 1;
                uint8_t* kp = k_s + kst * G::kKBytes;
                if (i >= kTcStages &&
                    !tc::mbar_wait(tc::smem_u32(&kv_empty[kst]), ((i >> 1) & 1) ^ 1, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                // nine TMA tensor loads (64 dims x 64 tokens) land the page swizzled;
                // an unreadable page reads zeros (negative coordinate)
                if (pw == 0) {
                    if (lane == 0) {
                        const int lp = pg0 + rank + i * C;
                        int pg = lp < P.swa_bt_stride ? P.swa_bt[static_cast<long long>(seq) * P.swa_bt_stride + lp] : -1;
                        if (pg < 0 || pg >= P.swa_pages) {
                            flag(P.status, DSV4_DEV_BAD_PAGE);
                            pg = -1;
                        }
                        const uint32_t bar = tc::smem_u32(&kv_full[kst]);
                        tc::mbar_arrive_expect_tx(bar, kTcKBytes);
                        for (int c = 0; c < 9; ++c)
                            tc::tma_load_3d(tc::smem_u32(kp + c * kTcKChunk), &tm_swa, bar, c * 64, 0, pg);
                    }
                } else if (lane == 0) {
                    tc::mbar_arrive(tc::smem_u32(&kv_full[kst]));
                }
            }
            // then the selected slots: row table, first rows, compressed tiles
            asm volatile("griddepcontrol.wait;" ::: "memory");
            load_slots();
            resolve();
            if (ok) ok = tc::mbar_wait(tc::smem_u32(bt_ready), 0, abort_flag, P.status);
            if (ok) {
                build_table();
                if (n_comp_mine > 0) fetch(0);
            }
            for (; ok && i < n_tiles; ++i) {
                const int kst = i & 1;
                uint8_t* kp = k_s + kst * G::kKBytes;
                if (i >= kTcStages &&
                    !tc::mbar_wait(tc::smem_u32(&kv_empty[kst]), ((i >> 1) & 1) ^ 1, abort_flag, P.status))
                    break;
                const int jc = i - n_swa_mine;
                convert(kp);
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&kv_full[kst]));
                if (jc + 1 < n_comp_mine) fetch(jc + 1);
            }
            // every load of the selected rows is done: a kernel launched next
            // (programmatic dependent launch; the library's compressor, which
            // waits for this grid's completion before it reads or writes
            // anything) may now be scheduled while the last tile and the
            // merge run.  Every grid before this one is complete: the
            // producers passed griddepcontrol.wait.
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        } else {
            // ------------------------------------------- softmax + O correction
            // Head h = 16*warp + lane % 16 (S row in TMEM lane 32*warp + lane % 16);
            // lanes 0-15 take keys 0-31 of the tile, lanes 16-31 keys 32-63.
            const int half = lane >> 4;
            const int h = warp * 16 + (lane & 15);
            const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
            float m = -INFINITY, l = 0.f;
            for (int t = 0;; ++t) {
                if (t == n_swa_mine) resolve();
                if (t >= n_tiles) break;
                const int sb = t & 1;
                if (!tc::mbar_wait(tc::smem_u32(&s_full[sb]), (t >> 1) & 1, abort_flag, P.status)) break;
                tc::tc_fence_after();
                // rows of this tile that are keys of the query, relative to this half
                const int gt = rank + t * C;
                int lo_r, hi_r;
                if (gt < n_swa_t) {
                    const int tok0 = (pg0 + gt) * kPage;
                    lo_r = max(0, t0 - tok0);
                    hi_r = min(kTcKeys, p - tok0 + 1);
                } else {
                    lo_r = 0;
                    hi_r = min(kTcKeys, n_comp - (gt - n_swa_t) * kTcKeys);
                }
                lo_r -= 32 * half;
                hi_r -= 32 * half;
                float s[32];
                tc::tmem_ld16x2_32(tmem + lane_base + sb * kTcKeys, s);
                tc::tmem_ld_wait();
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = (j >= lo_r && j < hi_r) ? s[j] * scale_log2 : -INFINITY;
                    mx = fmaxf(mx, s[j]);
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m, mx);
                const bool need = m_new > m + 8.0f;
                const float m_use = need ? m_new : m;
                uint32_t pk[16];
                float rowsum = 0.f;
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float e0 = (j >= lo_r && j < hi_r) ? ex2_approx(s[j] - m_use) : 0.f;
                    const float e1 = (j + 1 >= lo_r && j + 1 < hi_r) ? ex2_approx(s[j + 1] - m_use) : 0.f;
                    const __nv_bfloat162 bb = __floats2bfloat162_rn(e0, e1);
                    const float2 rb = __bfloat1622float2(bb);
                    rowsum += rb.x + rb.y;
                    pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&bb);
                }
                rowsum += __shfl_xor_sync(0xffffffffu, rowsum, 16);
                const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
                if (half == 0) sm_alpha[sb * 64 + h] = alpha;
                const int any_w = __any_sync(0xffffffffu, need);
                if (lane == 0) sm_any[sb * 4 + warp] = any_w;
                __threadfence_block();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&sync4[sb]));
                if (!tc::mbar_wait(tc::smem_u32(&sync4[sb]), (t >> 1) & 1, abort_flag, P.status)) break;
                const bool any = (sm_any[sb * 4 + 0] | sm_any[sb * 4 + 1] | sm_any[sb * 4 + 2] | sm_any[sb * 4 + 3]) != 0;
                if (any && t >= 1) {
                    // rescale O^T once PV(t-1) (and so every earlier PV) is complete
                    if (!tc::mbar_wait(tc::smem_u32(&pv_done[t - 1]), 0, abort_flag, P.status)) break;
                    tc::tc_fence_after();
#pragma unroll 1
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t ta = tmem + lane_base + kTcOCol + i * 32;
                        float o[32];
                        tc::tmem_ld32(ta, o);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] *= sm_alpha[sb * 64 + (i & 1) * 32 + j];
                        tc::tmem_st32(ta, o);
                    }
                    tc::tmem_st_wait();
                }
                l = l * alpha + rowsum;
                m = m_use;
                // V4: P buffer t % 2 was last read by PV(t - 2)
                if (V4 && t >= 2) {
                    if (!tc::mbar_wait(tc::smem_u32(&pv_done[t - 2]), 0, abort_flag, P.status)) break;
                    tc::tc_fence_after();
                }
                uint8_t* prow = V4 ? p_s + sb * kTcKChunk + h * 128 : k_s + sb * G::kKBytes + 8 * kTcKChunk + h * 128;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4*>(prow + (((4 * half + u) ^ (h & 7)) << 4)) =
                        make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&p_full[sb]));
            }
            if (half == 0) {
                sm_m[h] = m;
                sm_l[h] = l;
            }
            if (n_tiles > 0) tc::mbar_wait(tc::smem_u32(&pv_done[n_tiles - 1]), 0, abort_flag, P.status);
            tc::tc_fence_before();
        }
    }
    if (!resolved) resolve();                                // lanes that ran no loop

    // ------------------------------------------------------------- epilogue
    // 1. every CTA is past its main loop (its shared memory is free to receive)
    __syncthreads();
    tc::tc_fence_after();
    const int DS = kV / C;                                  // value dims combined by each CTA
    const int slice = DS * 128 + 512;                       // bytes of one slice
    uint8_t* recv = smem + kOffRecv;                        // [C] slices from every CTA (own one written here)
    uint8_t* send = smem + kOffSend;                        // [C] slices for the peers
    float* mw = reinterpret_cast<float*>(smem + kOffWeights);   // [8][64] weights, then [64] 1 / L
    const int DP = DS / kEpiParts;                          // dims of one part
    if (threadIdx.x == 0) {
        tc::mbar_arrive_expect_tx(tc::smem_u32(recv_ml), static_cast<uint32_t>((C - 1) * 512));
        for (int i = 0; i < kEpiParts; ++i)
            tc::mbar_arrive_expect_tx(tc::smem_u32(&recv_part[i]), static_cast<uint32_t>((C - 1) * DP * 128));
    }
    __syncwarp();
    // ready to receive: every earlier access to the receive space has
    // completed (the last MMA reads were observed through pv_done), so the
    // arrival publishes nothing
    tc::cluster_arrive_relaxed();
    // 2. stage: O^T dim d (TMEM lane) belongs to CTA d / DS; the unnormalised
    // partial is rounded to bf16 (half the distributed shared memory traffic)
    const bool have = n_tiles > 0 && !*abort_flag;
    if (warp < 8) {
        const int q4 = warp & 3;
#pragma unroll 1
        for (int bi = 0; bi < 2; ++bi) {
            const int i = (warp >> 2) * 2 + bi;
            const int d = i * 128 + q4 * 32 + lane;
            const int dst = d / DS, dl = d - dst * DS;
            float o[64];
            if (have) {
                const uint32_t ta = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + kTcOCol + i * 64;
                tc::tmem_ld32(ta, *reinterpret_cast<float(*)[32]>(o));
                tc::tmem_ld32(ta + 32, *reinterpret_cast<float(*)[32]>(o + 32));
                tc::tmem_ld_wait();
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) o[j] = 0.f;
            }
            uint8_t* row = (dst == rank ? recv + rank * slice : send + dst * slice) + dl * 128;
#pragma unroll
            for (int hc = 0; hc < 8; ++hc) {
                uint32_t w[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[8 * hc + 2 * c], o[8 * hc + 2 * c + 1]);
                    w[c] = *reinterpret_cast<const uint32_t*>(&v2);
                }
                *reinterpret_cast<uint4*>(row + ((hc ^ (dl & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    } else if (warp < 10) {
        const int hh = threadIdx.x - 256;
        const float2 ml = have ? make_float2(sm_m[hh], sm_l[hh]) : make_float2(-INFINITY, 0.f);
        for (int q = 0; q < C; ++q)
            *reinterpret_cast<float2*>((q == rank ? recv + rank * slice : send + q * slice) + DS * 128 + hh * 8) = ml;
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    // 3. per peer: the running max and sum first, then the parts in order,
    // once every peer is past its main loop
    tc::cluster_wait_acquire();
    if (threadIdx.x < C && threadIdx.x != rank) {
        const int q = threadIdx.x;
        const uint32_t dst = tc::map_to_rank(tc::smem_u32(recv + rank * slice), q);
        const uint32_t src = tc::smem_u32(send + q * slice);
        tc::bulk_s2s(dst + DS * 128, src + DS * 128, 512u, tc::map_to_rank(tc::smem_u32(recv_ml), q));
        for (int i = 0; i < kEpiParts; ++i)
            tc::bulk_s2s(dst + i * DP * 128, src + i * DP * 128, static_cast<uint32_t>(DP * 128),
                         tc::map_to_rank(tc::smem_u32(&recv_part[i]), q));
    }
    // 4. warps 0-7 merge heads 8w .. 8w + 7 of this CTA's slice, part by part as
    // the parts land (bounded waits, also after an abort); the others only
    // wait for every part
    // (wait results are made warp-uniform: the cluster arrivals are per warp)
    bool got = __all_sync(0xffffffffu, tc::mbar_wait_cluster(tc::smem_u32(recv_ml), 0, P.status));
    if (warp < 8) {
        const int hc = warp;
        if (got && lane < 8) {
            const int hh = 8 * hc + lane;
            float mq[8], lq[8];
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                mq[q] = -INFINITY;
                lq[q] = 0.f;
                if (q < C) {
                    const float2 ml = *reinterpret_cast<const float2*>(recv + q * slice + DS * 128 + hh * 8);
                    mq[q] = ml.x;
                    lq[q] = ml.y;
                }
                M = fmaxf(M, mq[q]);
            }
            float L = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q < C) {
                    const float wq = (mq[q] == -INFINITY) ? 0.f : ex2_approx(mq[q] - M);
                    mw[q * 64 + hh] = wq;
                    L += wq * lq[q];
                }
            }
            mw[8 * 64 + hh] = L > 0.f ? 1.0f / L : 0.f;
            if (rank == 0 && hh < nh && P.lse)
                P.lse[static_cast<long long>(b) * P.H + h0 + hh] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
        }
        __syncwarp();
        float il[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) il[c] = mw[8 * 64 + 8 * hc + c];
        uint16_t* ob = P.out + (static_cast<long long>(b) * P.H + h0 + 8 * hc) * kV + rank * DS;
        bool arrived = false;
        for (int i = 0; got && i < kEpiParts; ++i) {
            got = __all_sync(0xffffffffu, tc::mbar_wait_cluster(tc::smem_u32(&recv_part[i]), 0, P.status));
            if (!got) break;
            if (i == kEpiParts - 1) {
                __syncwarp();
                tc::cluster_arrive_relaxed();               // the peers' copies into this CTA have landed
                arrived = true;
            }
            for (int dl = i * DP + lane; dl < (i + 1) * DP; dl += 32) {
                float acc[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[c] = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (q < C) {
                        const uint4 x = *reinterpret_cast<const uint4*>(recv + q * slice + dl * 128 + ((hc ^ (dl & 7)) << 4));
                        const float4 w0 = *reinterpret_cast<const float4*>(mw + q * 64 + 8 * hc);
                        const float4 w1 = *reinterpret_cast<const float4*>(mw + q * 64 + 8 * hc + 4);
                        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            acc[2 * c] += wv[2 * c] * __uint_as_float(xw[c] << 16);
                            acc[2 * c + 1] += wv[2 * c + 1] * __uint_as_float(xw[c] & 0xffff0000u);
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (8 * hc + c < nh) ob[c * kV + dl] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[c] * il[c]));
            }
        }
        __syncwarp();
        if (!arrived) tc::cluster_arrive_relaxed();         // after a failed wait
    } else {
        for (int i = 0; got && i < kEpiParts; ++i) got = tc::mbar_wait_cluster(tc::smem_u32(&recv_part[i]), 0, P.status);
        __syncwarp();
        tc::cluster_arrive_relaxed();
    }
    __syncwarp();
    tc::cluster_wait_acquire();                             // every peer has received this CTA's copies
    if (warp == kTcMmaWarp) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTcTmemCols);
    }
}

// Every (code, scale byte) pair through the key conversion of the decode
// kernel: out[s * 256 + c] = bf16 bits of code c times 2^(s - 127).
__global__ void key_dequant_selftest_kernel(uint16_t* out)
{
    const int s = blockIdx.x;                 // scale byte
    const int g = threadIdx.x;                // 16 groups of 16 codes
    uint32_t wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c0 = g * 16 + 4 * i;
        wv[i] = c0 | ((c0 + 1) << 8) | ((c0 + 2) << 16) | ((c0 + 3) << 24);
    }
    uint4 lo, hi;
    dequant16(make_uint4(wv[0], wv[1], wv[2], wv[3]), static_cast<uint32_t>(s), lo, hi);
    const uint32_t o[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        out[s * 256 + g * 16 + 2 * i] = static_cast<uint16_t>(o[i] & 0xffffu);
        out[s * 256 + g * 16 + 2 * i + 1] = static_cast<uint16_t>(o[i] >> 16);
    }
}

// ---------------------------------------------------------------------------
// Prefill helpers (_forward_prefill of the "DeepseekV4Attention" class
// walkthrough): dequantise-and-gather of cache rows into a dense bf16 buffer,
// and each prefill token's combined index list over that buffer.
// ---------------------------------------------------------------------------
struct GatherParams {
    int kind;
    const uint8_t* cache;
    int num_pages;
    const int* bt;
    int bt_stride;
    const int* first;
    const int* count;
    int max_count;
    uint8_t* out;
    int out_rows;
    int out_offset;
    int* status;
};

// One warp per gathered row: (row i of run s) -> out[s][out_offset + i].
// Compressed entries: lane l dequantises nope codes 16l .. 16l + 15 (as the
// decode kernel does), lanes 0-7 copy the bf16 rope dims; SWA rows are copied.
__global__ void __launch_bounds__(32) dequant_gather_kernel(GatherParams G)
{
    const int s = blockIdx.y, i = blockIdx.x, lane = threadIdx.x;
    int cnt = G.count[s];
    if (cnt > G.max_count || cnt < 0) {
        if (i == 0 && lane == 0) flag(G.status, DSV4_DEV_BAD_INDEX);
        cnt = min(max(cnt, 0), G.max_count);
    }
    if (i >= cnt) return;
    const int slot = G.first[s] + i;
    uint8_t* orow = G.out + (static_cast<long long>(s) * G.out_rows + G.out_offset + i) * (kHead * 2);
    int pg = -1;
    if (slot >= 0 && (slot >> 6) < G.bt_stride) {
        pg = G.bt[static_cast<long long>(s) * G.bt_stride + (slot >> 6)];
        if (pg < 0 || pg >= G.num_pages) pg = -1;
    }
    if (pg < 0) {
        if (lane == 0) flag(G.status, DSV4_DEV_BAD_PAGE);
        for (int u = lane; u < kHead * 2 / 16; u += 32) reinterpret_cast<uint4*>(orow)[u] = make_uint4(0, 0, 0, 0);
        return;
    }
    if (G.kind == DSV4_GATHER_COMP) {
        const uint8_t* page = G.cache + static_cast<long long>(pg) * kMlaPage;
        const uint8_t* row = page + (slot & 63) * kMlaData;
        const uint4 w = *reinterpret_cast<const uint4*>(row + lane * 16);
        const uint32_t sb = page[kPage * kMlaData + (slot & 63) * 8 + (lane >> 2)];
        uint4 lo, hi;
        dequant16(w, sb, lo, hi);
        reinterpret_cast<uint4*>(orow)[2 * lane] = lo;
        reinterpret_cast<uint4*>(orow)[2 * lane + 1] = hi;
        if (lane < 8)
            reinterpret_cast<uint4*>(orow + kNope * 2)[lane] = *reinterpret_cast<const uint4*>(row + kNope + lane * 16);
    } else {
        const uint4* row = reinterpret_cast<const uint4*>(G.cache + static_cast<long long>(pg) * kSwaPage +
                                                          (slot & 63) * (kHead * 2));
        for (int u = lane; u < kHead * 2 / 16; u += 32) reinterpret_cast<uint4*>(orow)[u] = row[u];
    }
}

struct CombineParams {
    const int* topk;
    int topk_stride;
    const int* topk_len;
    const int* pos;
    const int* row_seq;
    const int* seq_len;
    const int* gather_len;
    int num_seqs;
    int window;
    int n_comp;
    int* out;
    int out_stride;
    int* out_len;
    int* status;
};

// One warp per prefill token: the valid top-k entries in order (ballot
// compaction), then the window tokens as rows n_comp + (t - first gathered).
// A window token outside the gathered run, a bad sequence or too short an
// output row sets DSV4_DEV_BAD_INDEX and length -1.
__global__ void __launch_bounds__(32) combine_indices_kernel(CombineParams C)
{
    const int t = blockIdx.x, lane = threadIdx.x;
    int* orow = C.out + static_cast<long long>(t) * C.out_stride;
    const int s = C.row_seq[t];
    const int len = C.topk_len[t];
    const int pos = C.pos[t];
    bool bad = s < 0 || s >= C.num_seqs || len < 0 || len > C.topk_stride || pos < 0;
    int first = 0, seq_len = 0;
    if (!bad) {
        seq_len = C.seq_len[s];
        first = seq_len - C.gather_len[s];
        const int w0 = max(0, pos - C.window + 1);
        bad = pos >= seq_len || w0 < first || len + (pos - w0 + 1) > C.out_stride;
    }
    if (bad) {
        if (lane == 0) {
            flag(C.status, DSV4_DEV_BAD_INDEX);
            C.out_len[t] = -1;
        }
        return;
    }
    const int* krow = C.topk + static_cast<long long>(t) * C.topk_stride;
    int n = 0;
    for (int i0 = 0; i0 < len; i0 += 32) {
        const int v = i0 + lane < len ? krow[i0 + lane] : -1;
        const uint32_t m = __ballot_sync(0xffffffffu, v >= 0);
        if (v >= 0) orow[n + __popc(m & ((1u << lane) - 1u))] = v;
        n += __popc(m);
    }
    const int w0 = max(0, pos - C.window + 1);
    for (int tok = w0 + lane; tok <= pos; tok += 32) orow[n + tok - w0] = C.n_comp + (tok - first);
    n += pos - w0 + 1;
    for (int i = n + lane; i < C.out_stride; i += 32) orow[i] = -1;
    if (lane == 0) C.out_len[t] = n;
}

}  // namespace dsv4

using namespace dsv4;

extern "C" dsv4_status dsv4_dequant_gather(const dsv4_gather_args* a, dsv4_stream_t stream)
{
    if (a == nullptr) return DSV4_ERR_INVALID;
    if (a->kind != DSV4_GATHER_COMP && a->kind != DSV4_GATHER_SWA) return DSV4_ERR_INVALID;
    if (a->num_seqs < 0 || a->max_count < 0 || a->bt_stride < 1 || a->num_pages < 1 || a->out_offset < 0 ||
        a->out_rows < a->out_offset + a->max_count)
        return DSV4_ERR_SHAPE;
    if (a->num_seqs == 0 || a->max_count == 0) return DSV4_OK;
    if (!a->cache_dev || !a->block_table_dev || !a->first_dev || !a->count_dev || !a->out_dev)
        return DSV4_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(a->cache_dev) & 15) || (reinterpret_cast<uintptr_t>(a->out_dev) & 15))
        return DSV4_ERR_SHAPE;
    if (a->max_count > 65535 || a->num_seqs > 65535) return DSV4_ERR_UNSUPPORTED;
    GatherParams G{a->kind, static_cast<const uint8_t*>(a->cache_dev), a->num_pages, a->block_table_dev,
                   a->bt_stride, a->first_dev, a->count_dev, a->max_count, static_cast<uint8_t*>(a->out_dev),
                   a->out_rows, a->out_offset, a->status_dev};
    dequant_gather_kernel<<<dim3(a->max_count, a->num_seqs), 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(G);
    return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

extern "C" dsv4_status dsv4_combine_topk_swa_indices(const dsv4_combine_args* a, dsv4_stream_t stream)
{
    if (a == nullptr) return DSV4_ERR_INVALID;
    if (a->num_tokens < 0 || a->num_seqs < 1 || a->window < 1 || a->n_comp < 0 || a->topk_stride < 0 ||
        a->out_stride < 1)
        return DSV4_ERR_SHAPE;
    if (a->num_tokens == 0) return DSV4_OK;
    if ((a->topk_stride > 0 && !a->topk_dev) || !a->topk_len_dev || !a->pos_dev || !a->row_seq_dev ||
        !a->seq_len_dev || !a->gather_len_dev || !a->out_dev || !a->out_len_dev)
        return DSV4_ERR_INVALID;
    CombineParams C{a->topk_dev, a->topk_stride, a->topk_len_dev, a->pos_dev, a->row_seq_dev, a->seq_len_dev,
                    a->gather_len_dev, a->num_seqs, a->window, a->n_comp, a->out_dev, a->out_stride,
                    a->out_len_dev, a->status_dev};
    combine_indices_kernel<<<a->num_tokens, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(C);
    return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

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
    P.row_seq = a->row_seq_dev;
    P.bt_rows = a->bt_rows;
    if (P.row_seq && P.bt_rows < 1) return DSV4_ERR_INVALID;
    // the V4 output quantisation: a second launch after the attention (the
    // quantisation kernel, positions from the context lengths)
    const bool want_codes = a->out_codes_dev != nullptr;
    if (want_codes && (!plan->kv_v4 || !a->out_scales_dev || !a->cos_sin_dev || a->max_pos < 1))
        return DSV4_ERR_INVALID;
    if (want_codes && (reinterpret_cast<uintptr_t>(a->out_scales_dev) & 3)) return DSV4_ERR_SHAPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    MlaTcParams T;
    T.base = P;
    T.head_groups = plan->mla_head_groups;
    T.cluster = plan->mla_splits;
    T.topk = plan->topk;
    const bool v4 = plan->kv_v4 != 0;
    const int qdim = v4 ? DSV4_V4_HEAD_DIM : kHead;
    CUtensorMap tm_q;
    const uint64_t qdims[2] = {static_cast<uint64_t>(qdim), static_cast<uint64_t>(plan->batch) * P.H};
    const uint64_t qstr[1] = {static_cast<uint64_t>(qdim) * 2};
    const uint32_t qbox[2] = {64, 64};
    if ((reinterpret_cast<uintptr_t>(a->q_dev) & 15) || (reinterpret_cast<uintptr_t>(a->swa_cache_dev) & 15) ||
        (reinterpret_cast<uintptr_t>(a->out_dev) & 15) ||
        (sparse && (reinterpret_cast<uintptr_t>(a->comp_cache_dev) & 15)))
        return DSV4_ERR_SHAPE;
    if (!encode_tmap(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->q_dev, qdims, qstr, qbox,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return DSV4_ERR_CUDA;
    // the bf16 SWA pages by TMA (the V4 window rows are FP8 and gathered by
    // the producers: the Q map stands in for the unused parameter)
    CUtensorMap tm_swa = tm_q;
    if (!v4) {
        const uint64_t sdims[3] = {static_cast<uint64_t>(kHead), static_cast<uint64_t>(kPage),
                                   static_cast<uint64_t>(a->swa_num_pages > 0 ? a->swa_num_pages : 1)};
        const uint64_t sstr[2] = {static_cast<uint64_t>(kHead) * 2, static_cast<uint64_t>(kSwaPage)};
        const uint32_t sbox[3] = {64, static_cast<uint32_t>(kTcKeys), 1};
        if (!encode_tmap(&tm_swa, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a->swa_cache_dev, sdims, sstr, sbox,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return DSV4_ERR_CUDA;
    }
    static PerDeviceOnce attr_once, attr_once_v4;
    const bool attr_ok =
        v4 ? attr_once_v4.run([] {
                 return cudaFuncSetAttribute(mla_decode_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             AttnGeom<true>::kSmem) == cudaSuccess;
             })
           : attr_once.run([] {
                 return cudaFuncSetAttribute(mla_decode_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             AttnGeom<false>::kSmem) == cudaSuccess;
             });
    if (!attr_ok) return DSV4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T.cluster, plan->batch * T.head_groups, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = v4 ? AttnGeom<true>::kSmem : AttnGeom<false>::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = T.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: behind a kernel that allows it (the
    // top-k), the window tiles run while it finishes; the selected slots are
    // read after griddepcontrol.wait
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = v4 ? cudaLaunchKernelEx(&cfg, mla_decode_tc<true>, tm_q, tm_swa, T)
                       : cudaLaunchKernelEx(&cfg, mla_decode_tc<false>, tm_q, tm_swa, T);
    if (e == cudaSuccess && want_codes)
        e = launch_inv_rope_quant(static_cast<const uint16_t*>(a->out_dev), plan->batch, P.H, a->ctx_len_dev, true,
                                  a->cos_sin_dev, a->max_pos, static_cast<uint8_t*>(a->out_codes_dev),
                                  a->out_scales_dev, a->status_dev, st);
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}

// Sparse prefill attention: one query row per prefill token, each over its
// own top-k compressed slots and its own causal window, straight from the
// paged caches (the decode kernel with the rows mapped to their sequences).
extern "C" dsv4_status dsv4_sparse_mla_prefill(const dsv4_plan* plan, const dsv4_mla_args* a,
                                               void* workspace, size_t workspace_bytes, dsv4_stream_t stream)
{
    if (a == nullptr || a->row_seq_dev == nullptr) return DSV4_ERR_INVALID;
    return dsv4_sparse_mla_decode(plan, a, workspace, workspace_bytes, stream);
}

extern "C" dsv4_status dsv4_selftest_key_dequant(void* out_dev, dsv4_stream_t stream)
{
    if (out_dev == nullptr) return DSV4_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(out_dev) & 1) return DSV4_ERR_SHAPE;
    key_dequant_selftest_kernel<<<256, 16, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<uint16_t*>(out_dev));
    return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
