// indexer.cu -- lightning indexer logits and per-query top-k.
//
// I_{t,s} = sum_j w_{t,j} ReLU(q_{t,j} . k_s) (SparseAttnIndexer formula in
// the "DeepseekV4Attention" class walkthrough; section 2 of the V4 internals
// talk write-up), with k_s = FP8 row * fp32 scale of the indexer cache, over
// the causal slots s < ctx_len / 4; then the k largest per query ("Indexer,
// C4A and C128A top-k", "DeepSeek V4 attention in vLLM").
#include <cstddef>

#include "dsv4_common.cuh"
#include "plan.h"
#include "tc_common.cuh"
#include "tmap.h"
#include "host_once.h"

namespace dsv4 {

// ---------------------------------------------------------------------------
// Logits on the tensor cores.  Per 128-slot tile (two 64-entry pages, each a
// contiguous 8 KB plane of FP8 rows), one tcgen05.mma kind::f8f6f4 chain
// D[128 slots x N heads] = K_tile[128 x 128] * Q^T[128 x N] (fp32 in TMEM),
// then each of 128 epilogue threads turns its slot's row of D into
// I_s = scale_s * sum_j w_j * max(D_sj, 0).
//   warps 8, 10: TMA producers of the even / odd tiles (query once, then two
//            page loads per tile, 6-stage ring)
//   warp 9: MMA issuer (4 MMAs of K=32 per tile, 4 accumulators)
//   warps 0-3 / 4-7: epilogue of the even / odd tiles (TMEM lane = slot row)
// One CTA per SM: CTAs of kernels that allocate tensor memory start one
// after another on an SM, so the work of a sequence is split over at most
// SMs / batch CTAs that each stream many tiles.
// Memory-bound: 132 bytes of cache per slot against 2 * 128 * N flops.
// ---------------------------------------------------------------------------
constexpr int kIdxTileSlots = 128;
constexpr int kIdxStages = 6;
constexpr int kIdxAcc = 4;
constexpr int kIdxTileBytes = kIdxTileSlots * kIdx;       // 16 KB
constexpr int kIdxQBytes = 64 * kIdx;                     // query tile, N <= 64 rows
constexpr int kIdxThreads = 352;
constexpr int kIdxTmemCols = kIdxAcc * 64;                // 4 accumulators x 64 columns
constexpr int kIdxScaleBytes = 16;                           // the tile's two page ids (+ padding)
constexpr int kIdxSmem = kIdxStages * kIdxTileBytes + kIdxQBytes + kIdxStages * kIdxScaleBytes +
                         2048 /* barriers etc */ + 1024 /* align */;
// FP4 (MXFP4) indexer cache: each tile arrives as its two whole pages
// (4352 B each: 64 x 64 code bytes, then 64 x 4 exponent bytes; 1-D bulk
// copies) in a ring of its own after the FP8 layout.  The epilogue warps
// expand a tile into the E4M3 tile ring: a slot's 32-dim block b is stored as
// E2M1 value x 2^-(E - e_b), E the largest of the slot's four exponents,
// which E4M3 holds exactly while E - e_b <= 8; the epilogue then scales the
// one accumulator by 2^(E - 127), as the FP8 path scales by its fp32 scale.
// A slot with a wider exponent spread is scored exactly by the converter
// from the page bytes instead.  The converter, not the epilogue, releases a
// FP4 stage (with the MMA): the epilogue needs only the per-slot scale (or
// exact score) the converter leaves beside the tile.
constexpr int kIdxFp4PageB = DSV4_IDX_FP4_PAGE_BYTES;                       // 4352
constexpr int kIdxFp4Stage = 2 * kIdxFp4PageB;                              // 8704
constexpr int kIdxRawOff4 = (kIdxSmem - 1024 + 127) / 128 * 128;
constexpr int kIdxRowScaleOff4 = kIdxRawOff4 + kIdxStages * kIdxFp4Stage;  // [stage][128] 2^(E-127), < 0: exact path
constexpr int kIdxExactOff4 = kIdxRowScaleOff4 + kIdxStages * kIdxTileSlots * 4;    // [stage][128] exact logits
constexpr int kIdxSmem4 = kIdxExactOff4 + kIdxStages * kIdxTileSlots * 4 + 1024;

// ---------------------------------------------------------------------------
// Top-k inside the logits launch: the CTAs of a sequence form a cluster, CTA
// r holding the logits of its consecutive slots [s0, s1) in shared memory.
// The selection rule is the one of the single-CTA top-k below (keys relative
// to the row minimum; digit passes from the top until the bin of the k-th
// largest key is taken whole or is one key; keys equal to the threshold taken
// lowest slot first; slots written in ascending order), here with 8-bit
// digits and every count summed over the cluster: each CTA pushes its counts
// into every CTA's shared memory (asynchronous distributed shared memory
// stores that count their bytes on the receiving CTA's mbarrier), so a CTA
// waits only for the bytes it needs, reads them locally and takes the same
// decisions as the others -- no cluster-wide barrier.  A buffer that pass p
// fills is filled again in pass p + 2, which no CTA reaches before every CTA
// has pushed its pass p + 1 counts, i.e. finished reading pass p.
// ---------------------------------------------------------------------------
constexpr int kCtkSlots = 16 * kIdxTileSlots;                        // slots per CTA at most
constexpr int kCtkPer = (kCtkSlots + kIdxThreads - 1) / kIdxThreads;   // slots per thread (6)
constexpr int kCtkMaxCluster = 8;
// the decisions of a digit pass, shared by the CTA's threads (see ctk_decide)
struct CtkDecision {
    uint32_t prefix;
    int rem, done, decided, failed;
};
struct CtkScratch {
    uint64_t bar_mm;                        // every CTA's (min, max) has landed (bytes)
    uint64_t bar_h[2];                      // every CTA's histogram of the pass has landed, by pass parity
    uint32_t mm_in[kCtkMaxCluster][2];      // (min, max) key of CTA q's slots, pushed by q
    int cnt_in[kCtkMaxCluster][2];          // CTA q's keys above / at the threshold, from its histograms
    alignas(16) int hin[2][kCtkMaxCluster][256];   // CTA q's digit histogram, by pass parity, pushed by q
                                                   // (16-byte st.async pushes)
    alignas(16) int hist[2][256];                  // this CTA's histogram, by pass parity (read 16 B at a time)
    uint32_t mm[2];                         // this CTA's min, max
    CtkDecision dec;                        // the decisions, for the CTA's threads
    int scan[16];
};
static_assert(offsetof(CtkScratch, hin) % 16 == 0 && offsetof(CtkScratch, hist) % 16 == 0 &&
                  offsetof(CtkScratch, mm_in) % 8 == 0,
              "vector pushes and loads of the top-k scratch");
constexpr int kIdxSmemFused = kIdxSmem + kCtkSlots * 4 + static_cast<int>(sizeof(CtkScratch));
constexpr int kIdxSmem4Fused = kIdxSmem4 + kCtkSlots * 4 + static_cast<int>(sizeof(CtkScratch));
static_assert(kIdxSmem4Fused <= 232448, "shared memory budget");
static_assert((kIdxSmem - 1024 + kCtkSlots * 4) % 16 == 0 && (kIdxSmem4 - 1024 + kCtkSlots * 4) % 16 == 0,
              "the top-k scratch starts 16-byte aligned");

// E4M3 byte of the E2M1 magnitude with index c (0, 0.5, 1, 1.5, 2, 3, 4, 6)
// times 2^-k, k = 0..8: every such value is an E4M3 value (normal when its
// exponent is at least -6, else a multiple of 2^-9).
__host__ __device__ constexpr uint32_t e4m3_of_e2m1_shifted(int c, int k)
{
    constexpr int twice[8] = {0, 1, 2, 3, 4, 6, 8, 12};   // 2 x magnitude
    const int n = twice[c];                                // value = n * 2^(-1-k)
    if (n == 0) return 0;
    const int e = -1 - k;
    int p = 0;
    while ((2 << p) <= n) ++p;                             // 2^p <= n < 2^(p+1)
    const int ex = e + p;                                  // value = (n / 2^p) * 2^ex
    if (ex >= -6) return static_cast<uint32_t>(((ex + 7) << 3) | (((n * 8) >> p) - 8));
    return static_cast<uint32_t>(n << (9 + e));           // subnormal: m * 2^-9
}

__host__ __device__ constexpr uint32_t e2m1_lut_word(int k, int half)
{
    return e4m3_of_e2m1_shifted(4 * half, k) | (e4m3_of_e2m1_shifted(4 * half + 1, k) << 8) |
           (e4m3_of_e2m1_shifted(4 * half + 2, k) << 16) | (e4m3_of_e2m1_shifted(4 * half + 3, k) << 24);
}

// [k][2]: the byte-permute tables of shift k
__constant__ uint32_t c_e2m1_lut[9][2] = {
    {e2m1_lut_word(0, 0), e2m1_lut_word(0, 1)}, {e2m1_lut_word(1, 0), e2m1_lut_word(1, 1)},
    {e2m1_lut_word(2, 0), e2m1_lut_word(2, 1)}, {e2m1_lut_word(3, 0), e2m1_lut_word(3, 1)},
    {e2m1_lut_word(4, 0), e2m1_lut_word(4, 1)}, {e2m1_lut_word(5, 0), e2m1_lut_word(5, 1)},
    {e2m1_lut_word(6, 0), e2m1_lut_word(6, 1)}, {e2m1_lut_word(7, 0), e2m1_lut_word(7, 1)},
    {e2m1_lut_word(8, 0), e2m1_lut_word(8, 1)}};
static_assert(e2m1_lut_word(0, 0) == 0x3c383000u && e2m1_lut_word(0, 1) == 0x4c484440u, "E4M3 of the E2M1 values");

// Four E2M1 codes (the nibbles of the low 16 bits, the first in bits 0-3) as
// four E4M3 bytes (the first in byte 0), each magnitude scaled by the table's
// power of two: a byte permute picks the magnitude from the table (lo, hi), a
// second one in sign-replicate mode spreads each code's sign bit over its
// byte.
__device__ __forceinline__ uint32_t e2m1x4_to_e4m3x4(uint32_t n16, uint32_t lut_lo, uint32_t lut_hi)
{
    uint32_t mag, sgn;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(mag) : "r"(lut_lo), "r"(lut_hi), "r"(n16 & 0x7777u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(sgn) : "r"(n16 << 4), "r"(n16), "r"(0xd9c8u));
    return mag | (sgn & 0x80808080u);
}

// The decision of a digit pass of the cluster top-k, taken alike by one warp
// of every CTA once the pass's histograms of all C CTAs are in hin[q][256]:
// lane l sums digits 8l .. 8l + 7 over the cluster, a shuffle scan from the
// top gives the keys above each lane's digits, and the lane holding the digit
// of the rem-th largest key still in play writes the new prefix (that digit at
// bit lo), the keys of that bin still to take, whether the selection is
// complete (lo == 0, or the bin is taken whole) and decided = pass + 1.  After
// a failed wait (ok false) nothing is decided and `failed` is set.
__device__ __forceinline__ void ctk_decide(const int (*hin)[256], int C, bool ok, uint32_t prefix, int lo, int rem,
                                           int pass, CtkDecision* D)
{
    const int lane = threadIdx.x & 31;
    int g[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = 0;
    if (ok) {
        for (int q = 0; q < C; ++q) {
            const uint4 a = *reinterpret_cast<const uint4*>(&hin[q][8 * lane]);
            const uint4 c = *reinterpret_cast<const uint4*>(&hin[q][8 * lane + 4]);
            g[0] += a.x; g[1] += a.y; g[2] += a.z; g[3] += a.w;
            g[4] += c.x; g[5] += c.y; g[6] += c.z; g[7] += c.w;
        }
    }
    int tl = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) tl += g[j];
    int x = tl;                                      // keys in the digits from 8 lane up
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += y;
    }
    int above = x - tl;                              // keys in the digits above this lane's
#pragma unroll
    for (int j = 7; j >= 0; --j) {
        if (above < rem && rem <= above + g[j]) {
            D->prefix = prefix | (static_cast<uint32_t>(8 * lane + j) << lo);
            D->rem = rem - above;
            D->done = (lo == 0) || (g[j] == rem - above);
            D->decided = pass + 1;
        }
        above += g[j];
    }
    __syncwarp();
    if (lane == 0 && (!ok || D->decided != pass + 1)) D->failed = 1;
}

// Exclusive scan of one int per thread over the CTA (kIdxThreads threads).
__device__ __forceinline__ int ctk_excl_scan(int v, int* scan, int& total)
{
    constexpr int NW = kIdxThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scan[warp] = x;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const int t = scan[w];
        before += w < warp ? t : 0;
        total += t;
    }
    __syncthreads();
    return before + x - v;
}

// Called by every thread of every CTA of the cluster once the CTA's logits
// are in lg[0, s1 - s0), and after the cluster arrival that the kernel made
// when it started, with the scratch barriers initialised (this function waits
// for it before its first push).  Writes the row's k slots (or, with at most k
// slots, all of them and -1 past) and its length.  A wait that times out
// flags `status` and leaves the row unwritten.
__device__ void cluster_topk(const float* lg, int s0, int s1, int n_c, int k, int C, int rank, int* orow,
                             int* out_len, CtkScratch* S, int* status)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    tc::cluster_wait_acquire();                      // every CTA of the cluster has started
    if (n_c <= k) {
        for (int s = s0 + tid; s < s1; s += kIdxThreads) orow[s] = s;
        if (rank == 0) {
            for (int i = n_c + tid; i < k; i += kIdxThreads) orow[i] = -1;
            if (tid == 0) *out_len = n_c;
        }
        return;
    }
    // this thread's consecutive slots [i0, i0 + nv) of the CTA's range
    const int nl = max(0, s1 - s0);
    const int chunk = (nl + kIdxThreads - 1) / kIdxThreads;
    const int i0 = tid * chunk;
    const int nv = max(0, min(chunk, nl - i0));
    uint32_t key[kCtkPer];
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (int j = 0; j < kCtkPer; ++j) {
        key[j] = j < nv ? f32_order_key(lg[i0 + j]) : 0u;
        if (j < nv) {
            mn = min(mn, key[j]);
            mx = max(mx, key[j]);
        }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
        atomicMin(&S->mm[0], mn);
        atomicMax(&S->mm[1], mx);
    }
    if (tid < 256) {
        S->hist[0][tid] = 0;
        S->hist[1][tid] = 0;
    }
    __syncthreads();
    // (a) every CTA's min / max, in every CTA
    if (tid == 0) tc::mbar_arrive_expect_tx(tc::smem_u32(&S->bar_mm), static_cast<uint32_t>(C * 8));
    if (tid < C)
        tc::st_async_u32x2(tc::map_to_rank(tc::smem_u32(&S->mm_in[rank][0]), tid), S->mm[0], S->mm[1],
                           tc::map_to_rank(tc::smem_u32(&S->bar_mm), tid));
    if (warp == 0) {
        const bool ok = tc::mbar_wait_cluster(tc::smem_u32(&S->bar_mm), 0, status);
        if (lane == 0 && !ok) S->dec.failed = 1;
    }
    __syncthreads();
    if (S->dec.failed) return;
    uint32_t base = 0xffffffffu, top = 0u;
    for (int q = 0; q < C; ++q) {
        base = min(base, S->mm_in[q][0]);
        top = max(top, S->mm_in[q][1]);
    }
    const uint32_t range = top - base;
    const int shift = range ? 32 - __clz(range) : 0;     // (key - base) < 2^shift
    // digit passes: pass 0 takes bits [lo, shift) of every key, later passes
    // the next 8 bits of the keys still in the threshold bin
    int lo = shift > 8 ? shift - 8 : 0;
    int plo = 32;                                        // the bin is (key - base) >> plo == prefix >> plo
    uint32_t prefix = 0;
    int rem = k;
    // every CTA holds every CTA's histograms: warp q + 1 (q < rank) sums CTA
    // q's keys above each pass's threshold digit, and takes its count in the
    // final threshold bin, so the compaction needs no count exchange
    const int cq = warp - 1;
    const bool counts_peer = cq >= 0 && cq < rank;
    int gt_q = 0, eq_q = 0;
    for (int pass = 0;; ++pass) {
        const int p = pass & 1;
#pragma unroll
        for (int j = 0; j < kCtkPer; ++j) {
            const uint32_t o = key[j] - base;
            if (j < nv && (plo == 32 || (o >> plo) == (prefix >> plo))) atomicAdd(&S->hist[p][(o >> lo) & 255u], 1);
        }
        __syncthreads();
        if (tid == 0) tc::mbar_arrive_expect_tx(tc::smem_u32(&S->bar_h[p]), static_cast<uint32_t>(C * 1024));
        if (tid < 64) {
            const uint4 h4 = *reinterpret_cast<const uint4*>(&S->hist[p][4 * tid]);
            for (int q = 0; q < C; ++q)
                tc::st_async_u32x4(tc::map_to_rank(tc::smem_u32(&S->hin[p][rank][4 * tid]), q), h4,
                                   tc::map_to_rank(tc::smem_u32(&S->bar_h[p]), q));
        }
        if (tid < 256) S->hist[p ^ 1][tid] = 0;          // for the next pass (its last reader was the pass before)
        if (warp == 0) {
            const bool ok = tc::mbar_wait_cluster(tc::smem_u32(&S->bar_h[p]), (pass >> 1) & 1, status);
            ctk_decide(S->hin[p], C, ok, prefix, lo, rem, pass, &S->dec);
        }
        __syncthreads();
        if (S->dec.failed) return;
        prefix = S->dec.prefix;
        rem = S->dec.rem;
        if (counts_peer) {
            // hin[p] is rewritten only by pass p + 2, after this CTA's next push
            const uint32_t dd = (prefix >> lo) & 255u;
            int a = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t d = 8u * lane + u;
                a += d > dd ? S->hin[p][cq][d] : 0;
            }
            gt_q += __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(a));
            if (S->dec.done) eq_q = S->hin[p][cq][dd];
        }
        plo = lo;
        if (S->dec.done) break;
        lo = lo > 8 ? lo - 8 : 0;
    }
    if (counts_peer && lane == 0) {
        S->cnt_in[cq][0] = gt_q;
        S->cnt_in[cq][1] = eq_q;
    }
    // ordered compaction: keys above the threshold bin, and the first `rem`
    // in it (lowest slot first), at their positions in the whole row
    const uint32_t thr = prefix >> plo;
    int gtn = 0, eqn = 0;
#pragma unroll
    for (int j = 0; j < kCtkPer; ++j) {
        const uint32_t d = (key[j] - base) >> plo;
        gtn += j < nv && d > thr;
        eqn += j < nv && d == thr;
    }
    int tot;
    const int before = ctk_excl_scan((gtn << 16) | eqn, S->scan, tot);   // counts < 2^16; its barriers
                                                                          // also publish cnt_in
    int gpos = before >> 16, epos = before & 0xffff;
    for (int q = 0; q < rank; ++q) {
        gpos += S->cnt_in[q][0];
        epos += S->cnt_in[q][1];
    }
#pragma unroll
    for (int j = 0; j < kCtkPer; ++j) {
        const uint32_t d = (key[j] - base) >> plo;
        if (j < nv && d > thr) {
            orow[gpos + min(epos, rem)] = s0 + i0 + j;
            ++gpos;
        } else if (j < nv && d == thr) {
            if (epos < rem) orow[gpos + epos] = s0 + i0 + j;
            ++epos;
        }
    }
    if (rank == 0 && tid == 0) *out_len = k;
}

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
    // with the top-k in the launch: k, and the selection's rows
    int k;
    int* out_idx;
    int out_stride;
    int* out_len;
    // prefill rows: block-table row of query row b (NULL: b), bt_rows rows
    const int* row_seq;
    int bt_rows;
};

template <bool kFused, bool kFp4>
__global__ void __launch_bounds__(kIdxThreads, 1)
indexer_logits_tc(const __grid_constant__ CUtensorMap tm_cache, const __grid_constant__ CUtensorMap tm_q,
                  IdxTcParams P)
{
    constexpr int kAcc = kIdxAcc;                              // accumulators in flight
    constexpr int kAccCols = 64;                               // TMEM columns per accumulator
    constexpr int kTmemCols = kIdxTmemCols;
    constexpr int kTileIn = kFp4 ? kIdxFp4Stage : kIdxTileBytes;   // bytes a tile's copies bring in
    constexpr int kPageBytes = kFp4 ? kIdxFp4Page : kIdxPage;
    // the top-k kernel that follows may be scheduled now; it waits for this
    // grid's completion before reading the logits
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = tc::align1024_shared(smem_raw);
    uint8_t* a_tiles = smem;
    uint8_t* q_tile = smem + kIdxStages * kIdxTileBytes;
    int* stage_pages = reinterpret_cast<int*>(q_tile + kIdxQBytes);    // [stage][2] page ids of the tile
    uint64_t* bars = reinterpret_cast<uint64_t*>(q_tile + kIdxQBytes + kIdxStages * kIdxScaleBytes);
    uint64_t* full = bars;                        // [kIdxStages]
    uint64_t* empty = bars + kIdxStages;          // [kIdxStages]
    uint64_t* acc_full = bars + 2 * kIdxStages;   // [kIdxAcc]
    uint64_t* acc_empty = acc_full + kIdxAcc;     // [kIdxAcc]
    uint64_t* q_bar = acc_empty + kIdxAcc;
    uint64_t* conv = q_bar + 1;                   // [kIdxStages] FP4: the tile's E4M3 expansion written
    float* w_s = reinterpret_cast<float*>(bars + 32);            // [64], 16-byte aligned, zero past H
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(w_s + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint32_t* lut_s = tmem_slot + 4;              // FP4: [9][2] byte-permute tables by exponent shift
    uint8_t* raw_tiles = smem + kIdxRawOff4;      // FP4: [kIdxStages] the tiles' two pages
    float* row_scale = reinterpret_cast<float*>(smem + kIdxRowScaleOff4);   // FP4: [kIdxStages][128]
    float* exact_s = reinterpret_cast<float*>(smem + kIdxExactOff4);         // FP4: [kIdxStages][128]
    // with the top-k in the launch: this CTA's logits, then the top-k scratch
    float* lg_s = reinterpret_cast<float*>(smem + (kFp4 ? kIdxSmem4 : kIdxSmem) - 1024);
    CtkScratch* ctk = reinterpret_cast<CtkScratch*>(lg_s + kCtkSlots);

    const int b = blockIdx.y;
    int n_c = P.ctx_len[b] / 4;
    if (n_c > P.max_slots) n_c = P.max_slots;
    if (n_c < 0) n_c = 0;
    const int n_tiles = (n_c + kIdxTileSlots - 1) / kIdxTileSlots;
    const int t_begin = blockIdx.x * P.tiles_per_cta;
    const int t_end = min(n_tiles, t_begin + P.tiles_per_cta);
    if (!kFused && t_begin >= t_end) return;      // uniform: nothing allocated yet
    const int n_my = max(0, t_end - t_begin);
    const int n_pages = (n_c + kPage - 1) / kPage;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the query row's block-table row (prefill rows map to their sequence's)
    auto seq_of_row = [&]() {
        int sq = b;
        if (P.row_seq) {
            sq = P.row_seq[b];
            if (sq < 0 || sq >= P.bt_rows) {
                if (lane == 0) flag(P.status, DSV4_DEV_BAD_INDEX);
                sq = 0;
            }
        }
        return sq;
    };
    // lane l of a producer warp: page id of page l of the group of 16 tiles
    // starting at tile i, loaded by the lanes at once
    auto page_group = [&](int sq, int i) {
        int pg = -1;
        if (2 * i + lane < 2 * n_my) {
            const int pi = min(2 * (t_begin + i) + lane, n_pages - 1);
            pg = (pi < P.bt_stride) ? P.bt[static_cast<long long>(sq) * P.bt_stride + pi] : -1;
            if (pg < 0 || pg >= P.num_pages) {
                flag(P.status, DSV4_DEV_BAD_PAGE);
                pg = -1;
            }
        }
        return pg;
    };
    // tile i's loads into its stage (a whole producer warp; v: this lane's
    // page, lanes 0-1 the tile's two pages).  The tile's page ids go to
    // stage_pages (the epilogue reads the scales straight from those pages)
    // before the phase is armed.  FP8: TMA tensor loads (an unreadable page
    // is outside the map and reads zeros); FP4: the two whole pages by 1-D
    // bulk copies (an unreadable page, already flagged, is read as page 0).
    auto issue_tile = [&](int i, int v) {
        const int st = i % kIdxStages;
        const uint32_t fb = tc::smem_u32(&full[st]);
        if (lane < 2) stage_pages[st * 2 + lane] = v < 0 ? 0 : v;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_expect_tx(fb, kTileIn);
        __syncwarp();
        if (kFp4) {
            if (lane < 2)
                tc::bulk_g2s(tc::smem_u32(raw_tiles + st * kIdxFp4Stage + lane * kIdxFp4PageB),
                             P.cache + static_cast<long long>(v < 0 ? 0 : v) * kIdxFp4PageB, kIdxFp4PageB, fb);
        } else if (lane < 2) {
            tc::tma_load_3d(tc::smem_u32(a_tiles + st * kIdxTileBytes + lane * (kIdxTileBytes / 2)), &tm_cache,
                            fb, 0, 0, v < 0 ? P.num_pages : v);
        }
    };
    // This kernel may overlap the one before it (programmatic dependent
    // launch).  When that is the library's decode compressor, it writes at
    // most the newest entry of each sequence (slot n_c - 1, in the last tile),
    // and the kernel before it, when it may still run, is the library's
    // attention, which writes nothing read here and had read its index rows
    // before it let the compressor launch; a caller kernel in between does
    // not let this one start early.  So the tiles before the last are read
    // at once, and the wait for the previous grid (which completes only after
    // its own predecessors) comes right before the last tile's loads -- and
    // in every CTA, so that this grid completes only after it.
    //
    // Producer warp 8 sets up the barriers and, before the block-wide barrier,
    // issues the query's and the first kIdxStages tiles' loads (no stage has
    // been used yet), so that they are in flight during the set-up.
    const int n_early = min(n_my, kIdxStages);
    bool waited = false;
    if (warp == 8) {
        if (lane == 0) {
            for (int i = 0; i < kIdxStages; ++i) {
                tc::mbar_init(tc::smem_u32(&full[i]), 1);
                // MMA commit + 4 warps: the epilogue's (page ids read), FP4: the converter's (tile read)
                tc::mbar_init(tc::smem_u32(&empty[i]), 5);
                if (kFp4) tc::mbar_init(tc::smem_u32(&conv[i]), 4);   // the 4 warps of the tile's epilogue group
            }
            for (int i = 0; i < kAcc; ++i) {
                tc::mbar_init(tc::smem_u32(&acc_full[i]), 1);
                tc::mbar_init(tc::smem_u32(&acc_empty[i]), 4);
            }
            tc::mbar_init(tc::smem_u32(q_bar), 1);
            if (kFused) {
                // the top-k's, which the other CTAs of the cluster complete
                tc::mbar_init(tc::smem_u32(&ctk->bar_mm), 1);
                tc::mbar_init(tc::smem_u32(&ctk->bar_h[0]), 1);
                tc::mbar_init(tc::smem_u32(&ctk->bar_h[1]), 1);
            }
            *abort_flag = 0;
            tc::fence_barrier_init();
            tc::prefetch_tensormap(&tm_cache);
            tc::prefetch_tensormap(&tm_q);
            tc::mbar_arrive_expect_tx(tc::smem_u32(q_bar), P.n_pad * kIdx);
            tc::tma_load_2d(tc::smem_u32(q_tile), &tm_q, tc::smem_u32(q_bar), 0, b * P.H);
        }
        __syncwarp();
        const int pg0 = page_group(seq_of_row(), 0);
        for (int i = 0; i < n_early; ++i) {
            if (!waited && t_begin + i == n_tiles - 1) {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                waited = true;
            }
            issue_tile(i, __shfl_sync(0xffffffffu, pg0, 2 * i + (lane & 1)));
        }
    }
    if (kFused && threadIdx.x == 0) {
        ctk->mm[0] = 0xffffffffu;
        ctk->mm[1] = 0u;
        ctk->dec.failed = 0;
        ctk->dec.decided = 0;
    }
    if (warp == 0) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (kFused) tc::cluster_arrive_relaxed();   // this CTA has started (the top-k waits for every CTA)
    int issued = n_early;   // tiles whose loads were issued (producer only)
    int consumed = 0; // tiles whose stage the MMA released (MMA thread only)

    if (warp == 8 || warp == 10) {
        const int pgrp = warp == 8 ? 0 : 1;       // this producer's tiles: i = pgrp, pgrp + 2, ...
        const int seq = seq_of_row();
        int pgl = n_my > n_early ? page_group(seq, 0) : -1;
        for (int i = pgrp; i < n_my; i += 2) {
            if (!waited && t_begin + i == n_tiles - 1) {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                waited = true;
            }
            if (i < n_early) continue;                // issued before the block-wide barrier
            if (i >= 16 && (i & 15) < 2) pgl = page_group(seq, i & ~15);
            const int v = __shfl_sync(0xffffffffu, pgl, 2 * (i & 15) + (lane & 1));   // this lane's page
            const int st = i % kIdxStages;
            int go = 1;
            if (lane == 0) {
                const uint32_t ph = (i / kIdxStages) & 1;
                if (i >= kIdxStages && !tc::mbar_wait(tc::smem_u32(&empty[st]), ph ^ 1, abort_flag, P.status))
                    go = 0;
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            issue_tile(i, v);
            if (lane == 0) issued = i + 1;
        }
        if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");
    } else if (warp == 9) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc(128, P.n_pad, tc::kFmtE4M3, tc::kFmtE4M3);
            const uint64_t b_desc = tc::desc_kmajor_sw128(tc::smem_u32(q_tile));
            if (tc::mbar_wait(tc::smem_u32(q_bar), 0, abort_flag, P.status)) {
                for (int i = 0; i < n_my; ++i) {
                    const int st = i % kIdxStages;
                    const uint32_t ph = (i / kIdxStages) & 1;
                    const int ab = i % kAcc;
                    const uint32_t aph = (i / kAcc) & 1;
                    if (!tc::mbar_wait(tc::smem_u32(kFp4 ? &conv[st] : &full[st]), ph, abort_flag, P.status)) break;
                    if (i >= kAcc && !tc::mbar_wait(tc::smem_u32(&acc_empty[ab]), aph ^ 1, abort_flag, P.status)) break;
                    tc::tc_fence_after();
                    const uint64_t a_desc = tc::desc_kmajor_sw128(tc::smem_u32(a_tiles + st * kIdxTileBytes));
                    const uint32_t d = tmem + ab * kAccCols;
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
        // epilogue group (warps 0-3 or 4-7) takes every other tile; the scales it
        // reads come straight from the pages, and the last tile's may be written
        // by the kernel before this one (see the producers)
        // the head weights (FP4: and the byte-permute tables) into shared
        // memory, loaded here so that the block-wide barrier does not wait
        // for them; the 8 epilogue warps meet once before the first use
        if (threadIdx.x < 64) w_s[threadIdx.x] = (threadIdx.x < P.H) ? P.w[static_cast<long long>(b) * P.H + threadIdx.x] : 0.f;
        if (kFp4 && threadIdx.x >= 64 && threadIdx.x < 64 + 18) lut_s[threadIdx.x - 64] = (&c_e2m1_lut[0][0])[threadIdx.x - 64];
        asm volatile("bar.sync 1, 256;" ::: "memory");
        const int grp = warp >> 2;
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        // FP4 slot scored exactly from its page bytes (codes, exponent bytes)
        // and the FP8 query tile: sum over heads of w_j ReLU(sum_c q_jc k_c),
        // k_c = E2M1 x 2^(e_b - 127)
        auto exact_fp4 = [&](const uint8_t* codes, const uint8_t* exb) {
            constexpr float mags[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
            float acc = 0.f;
            for (int j = 0; j < P.H; ++j) {
                float dot = 0.f;
                for (int c = 0; c < kIdx; ++c) {
                    const uint32_t code = (codes[c >> 1] >> (4 * (c & 1))) & 15u;
                    const float kv = ldexpf((code & 8u) ? -mags[code & 7u] : mags[code & 7u],
                                            static_cast<int>(exb[c >> 5]) - 127);
                    const uint8_t qb = q_tile[j * 128 + ((((c >> 4) ^ (j & 7))) << 4) + (c & 15)];
                    dot = fmaf(e4m3_to_f32(qb), kv, dot);
                }
                acc += w_s[j] * fmaxf(dot, 0.f);
            }
            return acc;
        };
        // FP4: this group expands its tiles into the E4M3 tile ring two of its
        // tiles ahead of the epilogue (thread = tile row = slot).  Block b of a
        // slot becomes E2M1 x 2^-(E - e_b), E the slot's largest exponent; the
        // slot's 2^(E - 127) goes to row_scale, or -1 when a block lies more
        // than 8 binades below E (the epilogue then scores it exactly).  The
        // four 16-byte units of a row are read in a lane-rotated order, which
        // spreads them over the banks.
        auto convert4 = [&](int i) {
            const int st = i % kIdxStages;
            if (!tc::mbar_wait(tc::smem_u32(&full[st]), (i / kIdxStages) & 1, abort_flag, P.status)) return false;
            const uint8_t* pg = raw_tiles + st * kIdxFp4Stage + (row >> 6) * kIdxFp4PageB;
            const uint8_t* src = pg + (row & (kPage - 1)) * (kIdx / 2);
            const uint32_t ex = *reinterpret_cast<const uint32_t*>(pg + kPage * (kIdx / 2) + (row & (kPage - 1)) * 4);
            int eb[4], E = 0;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                eb[bb] = static_cast<int>((ex >> (8 * bb)) & 0xffu);
                E = max(E, eb[bb]);
            }
            bool exact = true;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) exact = exact && E - eb[bb] <= 8;
            row_scale[st * kIdxTileSlots + row] = !exact ? -1.0f : (E == 0 ? __int_as_float(0x00400000) : exp2i(E - 127));
            uint8_t* dst = a_tiles + st * kIdxTileBytes + row * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int u = (lane + k) & 3;
                const int sh = min(E - (u == 0 ? eb[0] : (u == 1 ? eb[1] : (u == 2 ? eb[2] : eb[3]))), 8);
                const uint32_t lo_t = lut_s[2 * sh], hi_t = lut_s[2 * sh + 1];
                const uint4 w = *reinterpret_cast<const uint4*>(src + u * 16);
                const uint4 lo = make_uint4(e2m1x4_to_e4m3x4(w.x & 0xffffu, lo_t, hi_t),
                                            e2m1x4_to_e4m3x4(w.x >> 16, lo_t, hi_t),
                                            e2m1x4_to_e4m3x4(w.y & 0xffffu, lo_t, hi_t),
                                            e2m1x4_to_e4m3x4(w.y >> 16, lo_t, hi_t));
                const uint4 hi = make_uint4(e2m1x4_to_e4m3x4(w.z & 0xffffu, lo_t, hi_t),
                                            e2m1x4_to_e4m3x4(w.z >> 16, lo_t, hi_t),
                                            e2m1x4_to_e4m3x4(w.w & 0xffffu, lo_t, hi_t),
                                            e2m1x4_to_e4m3x4(w.w >> 16, lo_t, hi_t));
                // 128-byte swizzle of the tile: unit v of row r at ((v ^ (r & 7)) << 4)
                *reinterpret_cast<uint4*>(dst + (((2 * u) ^ (row & 7)) << 4)) = lo;
                *reinterpret_cast<uint4*>(dst + (((2 * u + 1) ^ (row & 7)) << 4)) = hi;
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&conv[st]));
            if (!exact) exact_s[st * kIdxTileSlots + row] = exact_fp4(src, pg + kPage * (kIdx / 2) + (row & (kPage - 1)) * 4);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&empty[st]));   // the pages are read
            return true;
        };
        bool conv_ok = true;
        if (kFp4) {
            for (int i = grp; conv_ok && i < n_my && i < grp + 4; i += 2) conv_ok = convert4(i);
        }
        for (int i = grp; conv_ok && i < n_my; i += 2) {
            if (t_begin + i == n_tiles - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
            if (kFp4 && i + 4 < n_my && !convert4(i + 4)) break;
            const int ab = i % kAcc;
            const uint32_t aph = (i / kAcc) & 1;
            const int st = i % kIdxStages;
            // the tile's rows have landed: its page ids are known; this row's
            // scale (FP4: its four block exponents) comes straight from its
            // page (in flight during the MMA)
            float scale, exact_logit = 0.f;
            if (kFp4) {
                // the converter's per-slot scale (or exact score), beside the
                // tile until the converter of the stage's next tile
                scale = row_scale[st * kIdxTileSlots + row];
                if (scale < 0.f) exact_logit = exact_s[st * kIdxTileSlots + row];
            } else {
                if (!tc::mbar_wait(tc::smem_u32(&full[st]), (i / kIdxStages) & 1, abort_flag, P.status)) break;
                scale = *reinterpret_cast<const float*>(P.cache +
                                                        static_cast<long long>(stage_pages[st * 2 + (row >> 6)]) *
                                                            kPageBytes +
                                                        kPage * kIdx + (row & (kPage - 1)) * 4);
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(tc::smem_u32(&empty[st]));
            }
            if (!tc::mbar_wait(tc::smem_u32(&acc_full[ab]), aph, abort_flag, P.status)) break;
            tc::tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + ab * kAccCols;
            float v0[32], v1[32];
            tc::tmem_ld32(taddr, v0);
            if (P.n_pad > 32) tc::tmem_ld32(taddr + 32, v1);
            tc::tmem_ld_wait();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acc_empty[ab]));
            float acc = 0.f;
            if (P.n_pad == 64) {
                // weights past H are zero and every column is a real accumulator
                const float4* w4 = reinterpret_cast<const float4*>(w_s);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 a = w4[j], c = w4[j + 8];
                    acc += a.x * fmaxf(v0[4 * j], 0.f) + a.y * fmaxf(v0[4 * j + 1], 0.f) +
                           a.z * fmaxf(v0[4 * j + 2], 0.f) + a.w * fmaxf(v0[4 * j + 3], 0.f);
                    acc += c.x * fmaxf(v1[4 * j], 0.f) + c.y * fmaxf(v1[4 * j + 1], 0.f) +
                           c.z * fmaxf(v1[4 * j + 2], 0.f) + c.w * fmaxf(v1[4 * j + 3], 0.f);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) acc += (j < P.H) ? w_s[j] * fmaxf(v0[j], 0.f) : 0.f;
                if (P.n_pad > 32) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc += (j + 32 < P.H) ? w_s[j + 32] * fmaxf(v1[j], 0.f) : 0.f;
                }
            }
            const float lg = (kFp4 && scale < 0.f) ? exact_logit : acc * scale;
            const int s = (t_begin + i) * kIdxTileSlots + row;
            if (kFused) lg_s[i * kIdxTileSlots + row] = lg;
            else if (s < n_c) P.logits[static_cast<long long>(b) * P.logits_stride + s] = lg;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (*abort_flag && (warp == 8 || warp == 10) && lane == 0) {
        // let this CTA's own copies land before its shared memory is released
        for (int i = consumed > 0 ? consumed : 0; i < issued; ++i) {
            if ((i & 1) != (warp == 8 ? 0 : 1)) continue;
            volatile int no_abort = 0;
            tc::mbar_wait(tc::smem_u32(&full[i % kIdxStages]), (i / kIdxStages) & 1, &no_abort, nullptr);
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (kFused)
        cluster_topk(lg_s, t_begin * kIdxTileSlots, min(t_end * kIdxTileSlots, n_c), n_c, P.k, static_cast<int>(gridDim.x),
                     static_cast<int>(blockIdx.x), P.out_idx + static_cast<long long>(b) * P.out_stride,
                     P.out_len + b, ctk, P.status);
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
    const float* logits, int row_stride, int max_slots, const int* __restrict__ ctx_len, int k,
    int* __restrict__ out_idx, int out_stride, int* __restrict__ out_len, int smem_keys)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

    // ordered compaction: warp w owns slots [w R, (w + 1) R) and walks them 32
    // consecutive keys at a time (coalesced); one pass counts the keys above /
    // in the threshold bin per warp, the second writes each selected slot at
    // (keys above before it) + (keys of the bin taken before it)
    constexpr int NW = kTopkThreads / 32;
    __shared__ int wsum[NW][2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = ((n + NW - 1) / NW + 31) & ~31;
    const int w0 = warp * R, w1 = min(n, w0 + R);
    int wg = 0, we = 0;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t d = i < w1 ? (key_at(i) - base) >> lo : 0u;
        wg += __popc(__ballot_sync(0xffffffffu, i < w1 && d > thr));
        we += __popc(__ballot_sync(0xffffffffu, i < w1 && d == thr));
    }
    if (lane == 0) {
        wsum[warp][0] = wg;
        wsum[warp][1] = we;
    }
    __syncthreads();
    int g = 0, e = 0;
    for (int q = 0; q < warp; ++q) {
        g += wsum[q][0];
        e += wsum[q][1];
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t d = i < w1 ? (key_at(i) - base) >> lo : 0u;
        const uint32_t gb = __ballot_sync(0xffffffffu, i < w1 && d > thr);
        const uint32_t eb = __ballot_sync(0xffffffffu, i < w1 && d == thr);
        const int gr = g + __popc(gb & lt), er = e + __popc(eb & lt);
        if ((gb >> lane) & 1u) orow[gr + min(er, take_eq)] = i;
        else if (((eb >> lane) & 1u) && er < take_eq) orow[gr + er] = i;
        g += __popc(gb);
        e += __popc(eb);
    }
    if (threadIdx.x == 0) out_len[b] = k;
}

// Rows of at most 8192 slots, one CTA of 16 warps per row: warp w keeps
// slots 512 w + 32 j + lane (j = 0..15) in registers, so every step but
// three block-wide exchanges runs on warp votes.  An 11-bit digit pass over
// (key - row minimum) finds the bin of the k-th largest key; the keys of
// that bin (usually a handful) are ranked by one warp, or narrowed by 8-bit
// passes when there are more than 32; the slots above the threshold, and the
// lowest-slot ones equal to it, are written in ascending order.
constexpr int kTopkSmallPer = 16;
constexpr int kTopkSmallMax = kTopkThreads * kTopkSmallPer;   // 8192
constexpr int kTopkList = 2048;                                 // threshold-bin keys kept in a list

__global__ void __launch_bounds__(kTopkThreads, 1) topk_small_kernel(
    const float* logits, int row_stride, int max_slots, const int* __restrict__ ctx_len, int k,
    int* __restrict__ out_idx, int out_stride, int* __restrict__ out_len)
{
    constexpr int NW = kTopkThreads / 32;
    __shared__ int hist1[kTopkBins];
    __shared__ int hist2[256];
    __shared__ uint32_t list[kTopkList];
    __shared__ int scratch[33];
    __shared__ uint32_t s_min, s_max;
    __shared__ __align__(16) int s_wgt[NW];
    __shared__ __align__(16) int s_weq[NW];
    __shared__ uint32_t s_prefix;
    __shared__ int s_shift, s_rem, s_done, s_m, s_fill;

    // the attention kernel that follows may be scheduled now (it waits for
    // this grid before reading the selection); the logits were produced by
    // the previous kernel of this call
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int q = 0; q < kTopkBins / kTopkThreads; ++q) hist1[threadIdx.x * (kTopkBins / kTopkThreads) + q] = 0;
    if (threadIdx.x < 256) hist2[threadIdx.x] = 0;
    if (threadIdx.x == 0) {
        s_min = 0xffffffffu;
        s_max = 0u;
        s_fill = 0;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int b = blockIdx.x;
    const int base_slot = warp * 512 + lane;             // slot of row j: base_slot + 32 j
    const float* lrow = logits + static_cast<long long>(b) * row_stride;
    // the row is allocated up to max_slots: load it together with the length
    float v[kTopkSmallPer];
#pragma unroll
    for (int j = 0; j < kTopkSmallPer; ++j)   // written by the grid before: L2 loads, after the wait
        v[j] = (base_slot + 32 * j < max_slots) ? __ldcg(lrow + base_slot + 32 * j) : 0.f;
    int n = ctx_len[b] / 4;
    n = n < 0 ? 0 : (n > max_slots ? max_slots : n);
    int* orow = out_idx + static_cast<long long>(b) * out_stride;
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += blockDim.x) orow[i] = (i < n) ? i : -1;
        if (threadIdx.x == 0) out_len[b] = n;
        return;
    }
    uint32_t off[kTopkSmallPer];
    uint32_t vm = 0;                                     // bit j: slot of row j exists
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (int j = 0; j < kTopkSmallPer; ++j) {
        off[j] = f32_order_key(v[j]);
        if (base_slot + 32 * j < n) {
            vm |= 1u << j;
            mn = min(mn, off[j]);
            mx = max(mx, off[j]);
        }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
        atomicMin(&s_min, mn);
        atomicMax(&s_max, mx);
    }
    __syncthreads();                                                   // (1)
    const uint32_t base = s_min, top = s_max;
    const uint32_t range = top - base;
    int shift = range ? 32 - __clz(range) : 0;           // offsets fit in `shift` bits
    uint32_t prefix = 0;
    int rem = k;
    bool done = (range == 0);
#pragma unroll
    for (int j = 0; j < kTopkSmallPer; ++j) off[j] = ((vm >> j) & 1u) ? off[j] - base : 0u;

    // pass 1: 11-bit digits over the whole range
    int m = 0;                                           // keys in the threshold bin
    if (!done) {
        const int lo1 = shift > 11 ? shift - 11 : 0;
#pragma unroll
        for (int j = 0; j < kTopkSmallPer; ++j)
            if ((vm >> j) & 1u) atomicAdd(&hist1[off[j] >> lo1], 1);
        __syncthreads();                                               // (2)
        int c[4];
        int local = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            c[q] = hist1[kTopkBins - 1 - 4 * threadIdx.x - q];
            local += c[q];
        }
        int tot1;
        const int before = block_excl_scan(local, scratch, tot1);     // (3, 4, 5)
        if (before < rem && rem <= before + local) {
            int cum = before;
            bool found = false;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (!found && cum + c[q] >= rem) {
                    s_prefix = static_cast<uint32_t>(kTopkBins - 1 - 4 * threadIdx.x - q) << lo1;
                    s_rem = rem - cum;
                    s_shift = lo1;
                    s_done = (lo1 == 0) || (cum + c[q] == rem);
                    s_m = c[q];
                    found = true;
                }
                cum += c[q];
            }
        }
        __syncthreads();                                               // (6)
        prefix = s_prefix;
        rem = s_rem;
        shift = s_shift;
        done = s_done;
        m = s_m;
    }
    // the threshold bin's keys go to a list (warp-aggregated positions)
    if (!done && m <= kTopkList) {
#pragma unroll
        for (int j = 0; j < kTopkSmallPer; ++j) {
            const bool cand = ((vm >> j) & 1u) && (off[j] >> shift) == (prefix >> shift);
            const uint32_t bal = __ballot_sync(0xffffffffu, cand);
            if (bal) {
                int pos = 0;
                if (lane == 0) pos = atomicAdd(&s_fill, __popc(bal));
                pos = __shfl_sync(0xffffffffu, pos, 0) + __popc(bal & ((1u << lane) - 1u));
                if (cand) list[pos] = off[j];
            }
        }
        __syncthreads();
        if (m <= 32) {
            // one warp ranks the bin's keys: T = the rem-th largest, and how
            // many keys equal to T are taken
            if (warp == 0) {
                const uint32_t c = lane < m ? list[lane] : 0u;
                int gt = 0, eq = 0;
                for (int i = 0; i < m; ++i) {
                    const uint32_t o = __shfl_sync(0xffffffffu, c, i);
                    gt += o > c;
                    eq += o == c;
                }
                const bool is_t = lane < m && gt < rem && rem <= gt + eq;
                const uint32_t bal = __ballot_sync(0xffffffffu, is_t);
                if (lane == __ffs(bal) - 1) {
                    s_prefix = c;
                    s_rem = rem - gt;
                    s_shift = 0;
                    s_done = 1;
                }
            }
            __syncthreads();
            prefix = s_prefix;
            rem = s_rem;
            shift = s_shift;
            done = true;
        }
    }
    // more than 32 keys in the bin: 8-bit passes (over the list, or over the
    // registers when the bin holds more than the list)
    const bool use_list = m <= kTopkList;
    while (!done) {
        const int lo = shift > 8 ? shift - 8 : 0;
        if (use_list) {
            for (int i = threadIdx.x; i < m; i += kTopkThreads) {
                const uint32_t o = list[i];
                if ((o >> shift) == (prefix >> shift)) atomicAdd(&hist2[(o >> lo) & 255u], 1);
            }
        } else {
#pragma unroll
            for (int j = 0; j < kTopkSmallPer; ++j)
                if (((vm >> j) & 1u) && (off[j] >> shift) == (prefix >> shift)) atomicAdd(&hist2[(off[j] >> lo) & 255u], 1);
        }
        __syncthreads();
        // digit 255 - t for t < 256, scanned from the top
        const int cnt = threadIdx.x < 256 ? hist2[255 - threadIdx.x] : 0;
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31 && warp < 8) scratch[warp] = x;
        __syncthreads();
        if (threadIdx.x < 256) {
            hist2[255 - threadIdx.x] = 0;                 // every read of the histogram is done
            int before = x - cnt;
            for (int w = 0; w < warp; ++w) before += scratch[w];
            if (before < rem && rem <= before + cnt) {
                s_prefix = prefix | (static_cast<uint32_t>(255 - threadIdx.x) << lo);
                s_rem = rem - before;
                s_shift = lo;
                s_done = (lo == 0) || (before + cnt == rem);
            }
        }
        __syncthreads();
        prefix = s_prefix;
        rem = s_rem;
        shift = s_shift;
        done = s_done;
    }
    // ordered compaction: slot order is (warp, row, lane)
    const int lo = shift;
    const uint32_t thr = prefix >> lo;     // digit prefix of the threshold bin
    const int take_eq = rem;               // keys of that bin to take, lowest slot first
    uint32_t gtb[kTopkSmallPer], eqb[kTopkSmallPer];
    int gtw = 0, eqw = 0;
#pragma unroll
    for (int j = 0; j < kTopkSmallPer; ++j) {
        const bool valid = (vm >> j) & 1u;
        const uint32_t d = off[j] >> lo;
        gtb[j] = __ballot_sync(0xffffffffu, valid && d > thr);
        eqb[j] = __ballot_sync(0xffffffffu, valid && d == thr);
        gtw += __popc(gtb[j]);
        eqw += __popc(eqb[j]);
    }
    if (lane == 0) {
        s_wgt[warp] = gtw;
        s_weq[warp] = eqw;
    }
    __syncthreads();
    int g = 0, e = 0;
#pragma unroll
    for (int q = 0; q < NW / 4; ++q) {
        const int4 a4 = reinterpret_cast<const int4*>(s_wgt)[q];
        const int4 b4 = reinterpret_cast<const int4*>(s_weq)[q];
        g += (4 * q < warp ? a4.x : 0) + (4 * q + 1 < warp ? a4.y : 0) + (4 * q + 2 < warp ? a4.z : 0) +
             (4 * q + 3 < warp ? a4.w : 0);
        e += (4 * q < warp ? b4.x : 0) + (4 * q + 1 < warp ? b4.y : 0) + (4 * q + 2 < warp ? b4.z : 0) +
             (4 * q + 3 < warp ? b4.w : 0);
    }
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < kTopkSmallPer; ++j) {
        const int gr = g + __popc(gtb[j] & lt);
        const int er = e + __popc(eqb[j] & lt);
        if ((gtb[j] >> lane) & 1u) orow[gr + min(er, take_eq)] = base_slot + 32 * j;
        else if (((eqb[j] >> lane) & 1u) && er < take_eq) orow[gr + er] = base_slot + 32 * j;
        g += __popc(gtb[j]);
        e += __popc(eqb[j]);
    }
    if (threadIdx.x == 0) out_len[b] = k;
}

// ---------------------------------------------------------------------------
// Top-k of long rows (plans whose top-k is not in the logits launch): the row
// of a query is split over a cluster of C <= 16 CTAs, CTA r holding the keys of
// slots [r S, (r + 1) S) in shared memory.  The selection is the one of the
// cluster top-k above -- (min, max) keys, 8-bit digit passes from the top of
// the row's key range with every count summed over the cluster through
// st.async pushes on the receivers' mbarriers, keys equal to the threshold
// taken lowest slot first, slots written in ascending order -- with warp-
// private histograms (a pass over 32768 keys would otherwise serialise on the
// shared-memory atomics of its most crowded bins).  Clusters of up to 4 CTAs
// push every CTA's whole histogram to every CTA (one round, C KB in per CTA);
// larger ones sum a pass's histograms by a reduce-scatter and an all-gather:
// CTA q owns digits [q nb, q nb + nb), every CTA sends each owner its counts
// of the owner's digits, and each owner sends the cluster's sums of its digits
// to every CTA (two rounds of about 1 KB in and out per CTA).
//
// Candidate list: the second pass, which scans every key anyway, also writes
// the local index of each key at or above the first pass's threshold bin (the
// keys still in play and the ones already taken) into a per-warp list, warp w
// covering the w-th run of the CTA's slots in slot order.  Later passes and
// the compaction walk that list instead of all S keys; a CTA whose list would
// overflow its capacity keeps scanning all of its keys (every count is the
// same either way, so the CTAs of a cluster may differ in this).
// ---------------------------------------------------------------------------
constexpr int kTkcSlots = 32768;                 // keys per CTA at most
constexpr int kTkcWarps = kTopkThreads / 32;     // 16
constexpr int kTkcMaxCluster = 16;               // CTAs per query (above 8: a non-portable cluster size)
constexpr int kTkcA2aMax = 4;                   // largest cluster that exchanges whole histograms
// digits owned by each CTA of a cluster of C: a multiple of 4 (16-byte pushes)
__host__ __device__ constexpr int tkc_digits_per_owner(int C) { return ((256 + C - 1) / C + 3) & ~3; }
constexpr int tkc_rs_entries()
{
    int m = 0;
    for (int c = 1; c <= kTkcMaxCluster; ++c) m = m > c * tkc_digits_per_owner(c) ? m : c * tkc_digits_per_owner(c);
    return m;
}
struct TkcScratch {
    uint64_t bar_mm, bar_rs[2], bar_ag[2], bar_cnt;
    uint32_t mm_in[kTkcMaxCluster][2];
    int cnt_in[kTkcMaxCluster][2];
    alignas(16) int hin[2][kTkcA2aMax][256];     // CTA q's histogram (small clusters), by pass parity
    alignas(16) int rs_in[2][tkc_rs_entries()];  // CTA r's counts of this CTA's digits at r nb, by pass parity
    alignas(16) int ag_in[2][256];               // the cluster's count of every digit, by pass parity
    alignas(16) int seg[256];                    // the cluster's counts of this CTA's digits
    alignas(16) int whist[kTkcWarps][256];
    alignas(16) int hist[256];
    int wsum[kTkcWarps][2];
    int lcnt[kTkcWarps];                         // candidates found by each warp
    uint32_t mm[2];
    CtkDecision dec;
};
// entries of one warp's candidate list: the warp's whole run of slots up to
// 16384 keys per CTA, half of it above (the shared-memory budget)
__host__ __device__ constexpr int tkc_list_cap(int S)
{
    return S <= 16384 ? ((S + kTkcWarps - 1) / kTkcWarps + 31) & ~31
                      : (((S + kTkcWarps - 1) / kTkcWarps + 31) & ~31) / 2;
}
__host__ __device__ constexpr size_t tkc_smem_bytes(int S)
{
    return static_cast<size_t>(S) * 4 + static_cast<size_t>(kTkcWarps) * tkc_list_cap(S) * 2 + sizeof(TkcScratch);
}
static_assert(offsetof(TkcScratch, hin) % 16 == 0 && offsetof(TkcScratch, rs_in) % 16 == 0 &&
                  offsetof(TkcScratch, ag_in) % 16 == 0 && offsetof(TkcScratch, seg) % 16 == 0 &&
                  offsetof(TkcScratch, hist) % 16 == 0 && offsetof(TkcScratch, mm_in) % 8 == 0,
              "vector pushes and loads of the long-row top-k scratch");
static_assert(tkc_smem_bytes(kTkcSlots) <= 232448 && tkc_smem_bytes(16384) <= tkc_smem_bytes(kTkcSlots),
              "the largest S sets the shared-memory attribute");

__global__ void __launch_bounds__(kTopkThreads, 1) topk_cluster_kernel(
    const float* logits, int row_stride, int max_slots, const int* __restrict__ ctx_len, int k, int S,
    int* __restrict__ out_idx, int out_stride, int* __restrict__ out_len, int* status)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(16) uint32_t tkc_smem[];
    uint32_t* keys = tkc_smem;                                       // [S]
    const int LC = tkc_list_cap(S);                                  // a multiple of 32
    uint16_t* list = reinterpret_cast<uint16_t*>(tkc_smem + S);      // [kTkcWarps][LC]
    TkcScratch* T = reinterpret_cast<TkcScratch*>(list + kTkcWarps * LC);   // S is a multiple of 32
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = static_cast<int>(gridDim.x), rank = static_cast<int>(blockIdx.x), b = blockIdx.y;
    if (tid == 0) {
        tc::mbar_init(tc::smem_u32(&T->bar_mm), 1);
        tc::mbar_init(tc::smem_u32(&T->bar_rs[0]), 1);
        tc::mbar_init(tc::smem_u32(&T->bar_rs[1]), 1);
        tc::mbar_init(tc::smem_u32(&T->bar_ag[0]), 1);
        tc::mbar_init(tc::smem_u32(&T->bar_ag[1]), 1);
        tc::mbar_init(tc::smem_u32(&T->bar_cnt), 1);
        T->mm[0] = 0xffffffffu;
        T->mm[1] = 0u;
        T->dec.failed = 0;
        T->dec.decided = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    tc::cluster_arrive_relaxed();                    // this CTA's barriers are initialised
    int n = ctx_len[b] / 4;
    n = n < 0 ? 0 : (n > max_slots ? max_slots : n);
    int* orow = out_idx + static_cast<long long>(b) * out_stride;
    const int s0 = rank * S, s1 = min(n, s0 + S), nl = max(0, s1 - s0);
    // the logits come from the kernel launched before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    tc::cluster_wait_acquire();                      // every CTA of the cluster has started
    if (n <= k) {
        for (int s = s0 + tid; s < s1; s += kTopkThreads) orow[s] = s;
        if (rank == 0) {
            for (int i = n + tid; i < k; i += kTopkThreads) orow[i] = -1;
            if (tid == 0) out_len[b] = n;
        }
        return;
    }
    // keys of this CTA's slots (s0, the row stride and the workspace base are
    // 16-byte aligned)
    const float* lrow = logits + static_cast<long long>(b) * row_stride + s0;
    uint32_t mn = 0xffffffffu, mx = 0u;
    const int n4 = nl >> 2;                          // whole float4 groups, 4 loads in flight per thread
#pragma unroll 4
    for (int i = tid; i < n4; i += kTopkThreads) {
        const float4 v = reinterpret_cast<const float4*>(lrow)[i];
        const uint32_t k0 = f32_order_key(v.x), k1 = f32_order_key(v.y), k2 = f32_order_key(v.z),
                       k3 = f32_order_key(v.w);
        reinterpret_cast<uint4*>(keys)[i] = make_uint4(k0, k1, k2, k3);
        mn = min(min(mn, k0), min(min(k1, k2), k3));
        mx = max(max(mx, k0), max(max(k1, k2), k3));
    }
    for (int j = 4 * n4 + tid; j < nl; j += kTopkThreads) {
        const uint32_t kk = f32_order_key(lrow[j]);
        keys[j] = kk;
        mn = min(mn, kk);
        mx = max(mx, kk);
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
        atomicMin(&T->mm[0], mn);
        atomicMax(&T->mm[1], mx);
    }
    __syncthreads();
    // every CTA's min / max, in every CTA
    if (tid == 0) tc::mbar_arrive_expect_tx(tc::smem_u32(&T->bar_mm), static_cast<uint32_t>(C * 8));
    if (tid < C)
        tc::st_async_u32x2(tc::map_to_rank(tc::smem_u32(&T->mm_in[rank][0]), tid), T->mm[0], T->mm[1],
                           tc::map_to_rank(tc::smem_u32(&T->bar_mm), tid));
    if (warp == 0) {
        const bool ok = tc::mbar_wait_cluster(tc::smem_u32(&T->bar_mm), 0, status);
        if (lane == 0 && !ok) T->dec.failed = 1;
    }
    __syncthreads();
    if (T->dec.failed) return;
    uint32_t base = 0xffffffffu, top = 0u;
    for (int q = 0; q < C; ++q) {
        base = min(base, T->mm_in[q][0]);
        top = max(top, T->mm_in[q][1]);
    }
    const uint32_t range = top - base;
    const int shift = range ? 32 - __clz(range) : 0;
    int lo = shift > 8 ? shift - 8 : 0;
    int plo = 32;
    uint32_t prefix = 0;
    int rem = k;
    // warp w's run of this CTA's slots: [w0, w1)
    const int R = ((nl + kTkcWarps - 1) / kTkcWarps + 31) & ~31;
    const int w0 = min(nl, warp * R), w1 = min(nl, w0 + R);
    const uint32_t lt = (1u << lane) - 1u;
    uint16_t* wl = list + warp * LC;
    int wl_n = 0;                   // this warp's candidates (valid once use_list)
    bool use_list = false;          // the same in every thread of the CTA
    const bool a2a = C <= kTkcA2aMax;
    const int nb = tkc_digits_per_owner(C);
    const int my_nb = a2a ? 0 : max(0, min(256, (rank + 1) * nb) - rank * nb);   // digits this CTA owns
    for (int pass = 0;; ++pass) {
        const int p = pass & 1;
        const bool listed = use_list;
        const bool build = pass == 1;
        if (listed) {
            if (tid < 256) T->hist[tid] = 0;
        } else {
            for (int i = tid; i < kTkcWarps * 256; i += kTopkThreads) (&T->whist[0][0])[i] = 0;
        }
        __syncthreads();
        // keys in play: (key - base) >> plo == prefix >> plo, i.e. key - lo_key <
        // 2^plo with lo_key = base + the prefix's bits at and above plo (every
        // key in the first pass); their digit is (key - lo_key) >> lo.
        const uint32_t lo_key = base + (plo == 32 ? 0u : (prefix >> plo) << plo);
        const uint32_t span_m1 = plo == 32 ? 0xffffffffu : (1u << plo) - 1u;
        if (listed) {
            // few keys: one histogram for the CTA
            for (int j = lane; j < wl_n; j += 32) {
                const uint32_t o = keys[wl[j]] - lo_key;
                if (o <= span_m1) atomicAdd(&T->hist[(o >> lo) & 255u], 1);
            }
        } else if (build) {
            // the warp's run 128 keys at a time (slot order = 32 u + lane):
            // histogram of the keys in play, and every key >= lo_key appended
            // to the warp's list in slot order
            int* wh = T->whist[warp];
            int cnt = 0;
            for (int i0 = w0; i0 < w1; i0 += 128) {
                uint32_t kk[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + 32 * u + lane;
                    kk[u] = i < w1 ? keys[i] : 0u;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + 32 * u + lane;
                    const bool v = i < w1;
                    const uint32_t o = kk[u] - lo_key;
                    if (v && o <= span_m1) atomicAdd(&wh[(o >> lo) & 255u], 1);
                    const uint32_t bal = __ballot_sync(0xffffffffu, v && kk[u] >= lo_key);
                    if (bal) {
                        const int at = cnt + __popc(bal & lt);
                        if (((bal >> lane) & 1u) && at < LC) wl[at] = static_cast<uint16_t>(i);
                        cnt += __popc(bal);
                    }
                }
            }
            wl_n = cnt;
            if (lane == 0) T->lcnt[warp] = cnt;
        } else {
            // every key, four at a time (nl4 whole groups, then the tail)
            int* wh = T->whist[warp];
            const int nl4 = nl >> 2;
#pragma unroll 2
            for (int i4 = tid; i4 < nl4; i4 += kTopkThreads) {
                const uint4 kv = reinterpret_cast<const uint4*>(keys)[i4];
                const uint32_t o0 = kv.x - lo_key, o1 = kv.y - lo_key, o2 = kv.z - lo_key, o3 = kv.w - lo_key;
                if (o0 <= span_m1) atomicAdd(&wh[(o0 >> lo) & 255u], 1);
                if (o1 <= span_m1) atomicAdd(&wh[(o1 >> lo) & 255u], 1);
                if (o2 <= span_m1) atomicAdd(&wh[(o2 >> lo) & 255u], 1);
                if (o3 <= span_m1) atomicAdd(&wh[(o3 >> lo) & 255u], 1);
            }
            for (int i = 4 * nl4 + tid; i < nl; i += kTopkThreads) {
                const uint32_t o = keys[i] - lo_key;
                if (o <= span_m1) atomicAdd(&wh[(o >> lo) & 255u], 1);
            }
        }
        __syncthreads();
        if (build) {
            int mx_n = 0;
#pragma unroll
            for (int w = 0; w < kTkcWarps; ++w) mx_n = max(mx_n, T->lcnt[w]);
            use_list = mx_n <= LC;
        }
        if (!listed) {
            if (tid < 256) {
                int acc = 0;
#pragma unroll
                for (int w = 0; w < kTkcWarps; ++w) acc += T->whist[w][tid];
                T->hist[tid] = acc;
            }
            __syncthreads();
        }
        const uint32_t ph = (pass >> 1) & 1;
        if (a2a) {
            if (tid == 0) tc::mbar_arrive_expect_tx(tc::smem_u32(&T->bar_ag[p]), static_cast<uint32_t>(C * 1024));
            if (tid < 64) {
                const uint4 h4 = *reinterpret_cast<const uint4*>(&T->hist[4 * tid]);
                for (int q = 0; q < C; ++q)
                    tc::st_async_u32x4(tc::map_to_rank(tc::smem_u32(&T->hin[p][rank][4 * tid]), q), h4,
                                       tc::map_to_rank(tc::smem_u32(&T->bar_ag[p]), q));
            }
            if (warp == 0) {
                const bool ok = tc::mbar_wait_cluster(tc::smem_u32(&T->bar_ag[p]), ph, status);
                ctk_decide(T->hin[p], C, ok, prefix, lo, rem, pass, &T->dec);
            }
        } else {
            if (tid == 0 && my_nb > 0)
                tc::mbar_arrive_expect_tx(tc::smem_u32(&T->bar_rs[p]), static_cast<uint32_t>(C * my_nb * 4));
            if (tid == 32) tc::mbar_arrive_expect_tx(tc::smem_u32(&T->bar_ag[p]), 1024u);
            if (tid < 64) {
                // digits 4 tid .. 4 tid + 3 to their owner
                const int d0 = 4 * tid, q = d0 / nb;
                const uint4 h4 = *reinterpret_cast<const uint4*>(&T->hist[d0]);
                tc::st_async_u32x4(tc::map_to_rank(tc::smem_u32(&T->rs_in[p][rank * nb + d0 - q * nb]), q), h4,
                                   tc::map_to_rank(tc::smem_u32(&T->bar_rs[p]), q));
            }
            if (warp == 0) {
                bool ok = true;
                if (my_nb > 0) {
                    ok = __all_sync(0xffffffffu, tc::mbar_wait_cluster(tc::smem_u32(&T->bar_rs[p]), ph, status));
                    if (ok) {
                        // the cluster's counts of this CTA's digits (four peers' loads
                        // in flight at a time), to every CTA
                        const int* rs = T->rs_in[p];
                        for (int i = lane; i < my_nb; i += 32) {
                            int s0 = 0, s1 = 0, s2 = 0, s3 = 0, r = 0;
                            for (; r + 4 <= C; r += 4) {
                                s0 += rs[r * nb + i];
                                s1 += rs[(r + 1) * nb + i];
                                s2 += rs[(r + 2) * nb + i];
                                s3 += rs[(r + 3) * nb + i];
                            }
                            for (; r < C; ++r) s0 += rs[r * nb + i];
                            T->seg[i] = (s0 + s1) + (s2 + s3);
                        }
                        __syncwarp();
                        const int n4 = my_nb >> 2;
                        for (int j = lane; j < n4 * C; j += 32) {
                            const int dst = j / n4, part = j - dst * n4;
                            const uint4 v = *reinterpret_cast<const uint4*>(&T->seg[4 * part]);
                            tc::st_async_u32x4(tc::map_to_rank(tc::smem_u32(&T->ag_in[p][rank * nb + 4 * part]), dst),
                                               v, tc::map_to_rank(tc::smem_u32(&T->bar_ag[p]), dst));
                        }
                    }
                }
                ok = ok && tc::mbar_wait_cluster(tc::smem_u32(&T->bar_ag[p]), ph, status);
                ctk_decide(reinterpret_cast<const int (*)[256]>(T->ag_in[p]), 1, ok, prefix, lo, rem, pass, &T->dec);
            }
        }
        __syncthreads();
        if (T->dec.failed) return;
        prefix = T->dec.prefix;
        rem = T->dec.rem;
        plo = lo;
        if (T->dec.done) break;
        lo = lo > 8 ? lo - 8 : 0;
    }
    // ordered compaction: warp w walks its run of this CTA's slots (or its
    // candidate list, in the same order) 32 keys at a time; counts per warp,
    // per CTA (pushed to every CTA), then the writes
    const uint32_t thr = prefix >> plo;
    // ballots of 4 consecutive 32-key groups of the warp's run (their keys read
    // at once): gb[u] = lanes whose key lies above the threshold bin, eb[u] = in it
    auto groups4 = [&](int i0, uint32_t (&gb)[4], uint32_t (&eb)[4]) {
        uint32_t d[4];
        bool v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + 32 * u + lane;
            v[u] = i < w1;
            d[u] = v[u] ? (keys[i] - base) >> plo : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            gb[u] = __ballot_sync(0xffffffffu, v[u] && d[u] > thr);
            eb[u] = __ballot_sync(0xffffffffu, v[u] && d[u] == thr);
        }
    };
    // the same for one 32-entry group of the list: lane's slot in i
    auto group_l = [&](int j0, uint32_t& gb, uint32_t& eb, int& i) {
        const int j = j0 + lane;
        const bool v = j < wl_n;
        i = v ? static_cast<int>(wl[j]) : 0;
        const uint32_t d = v ? (keys[i] - base) >> plo : 0u;
        gb = __ballot_sync(0xffffffffu, v && d > thr);
        eb = __ballot_sync(0xffffffffu, v && d == thr);
    };
    int wg = 0, we = 0;
    if (use_list) {
        for (int j0 = 0; j0 < wl_n; j0 += 32) {
            uint32_t gb, eb;
            int i;
            group_l(j0, gb, eb, i);
            wg += __popc(gb);
            we += __popc(eb);
        }
    } else {
        for (int i0 = w0; i0 < w1; i0 += 128) {
            uint32_t gb[4], eb[4];
            groups4(i0, gb, eb);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                wg += __popc(gb[u]);
                we += __popc(eb[u]);
            }
        }
    }
    if (lane == 0) {
        T->wsum[warp][0] = wg;
        T->wsum[warp][1] = we;
    }
    __syncthreads();
    int cg = 0, ce = 0, g = 0, e = 0;
    for (int q = 0; q < kTkcWarps; ++q) {
        cg += T->wsum[q][0];
        ce += T->wsum[q][1];
        if (q < warp) {
            g += T->wsum[q][0];
            e += T->wsum[q][1];
        }
    }
    if (tid == 0) tc::mbar_arrive_expect_tx(tc::smem_u32(&T->bar_cnt), static_cast<uint32_t>(C * 8));
    if (tid < C)
        tc::st_async_u32x2(tc::map_to_rank(tc::smem_u32(&T->cnt_in[rank][0]), tid), static_cast<uint32_t>(cg),
                           static_cast<uint32_t>(ce), tc::map_to_rank(tc::smem_u32(&T->bar_cnt), tid));
    if (warp == 0) {
        const bool ok = tc::mbar_wait_cluster(tc::smem_u32(&T->bar_cnt), 0, status);
        if (lane == 0 && !ok) T->dec.failed = 1;
    }
    __syncthreads();
    if (T->dec.failed) return;
    for (int q = 0; q < rank; ++q) {
        g += T->cnt_in[q][0];
        e += T->cnt_in[q][1];
    }
    if (use_list) {
        for (int j0 = 0; j0 < wl_n; j0 += 32) {
            uint32_t gb, eb;
            int i;
            group_l(j0, gb, eb, i);
            const int gr = g + __popc(gb & lt), er = e + __popc(eb & lt);
            if ((gb >> lane) & 1u) orow[gr + min(er, rem)] = s0 + i;
            else if (((eb >> lane) & 1u) && er < rem) orow[gr + er] = s0 + i;
            g += __popc(gb);
            e += __popc(eb);
        }
    } else {
        for (int i0 = w0; i0 < w1; i0 += 128) {
            uint32_t gb[4], eb[4];
            groups4(i0, gb, eb);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + 32 * u + lane;
                const int gr = g + __popc(gb[u] & lt), er = e + __popc(eb[u] & lt);
                if ((gb[u] >> lane) & 1u) orow[gr + min(er, rem)] = s0 + i;
                else if (((eb[u] >> lane) & 1u) && er < rem) orow[gr + er] = s0 + i;
                g += __popc(gb[u]);
                e += __popc(eb[u]);
            }
        }
    }
    if (rank == 0 && tid == 0) out_len[b] = k;
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
    if (reinterpret_cast<uintptr_t>(workspace) & 15) return DSV4_ERR_SHAPE;
    if (a->row_seq_dev && a->bt_rows < 1) return DSV4_ERR_INVALID;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* logits = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan->ws_logits_off);
    const int B = plan->batch, H = plan->geom.idx_heads;
    if (plan->idx_ctas_per_seq > 0) {
        CUtensorMap tm_cache, tm_q;
        // the pages' data planes: FP8 rows of 128 bytes (128-byte swizzle,
        // the MMA's layout) or FP4 code rows of 64 bytes (expanded in the kernel)
        const bool fp4 = plan->idx_fp4 != 0;
        const uint32_t row_b = fp4 ? kIdx / 2 : kIdx;
        const uint64_t cdims[3] = {row_b, static_cast<uint64_t>(kPage), static_cast<uint64_t>(a->num_pages)};
        const uint64_t cstr[2] = {row_b, static_cast<uint64_t>(fp4 ? kIdxFp4Page : kIdxPage)};
        const uint32_t cbox[3] = {row_b, static_cast<uint32_t>(kPage), 1};
        const int n_pad = H <= 16 ? 16 : (H + 15) / 16 * 16;
        const uint64_t qdims[2] = {static_cast<uint64_t>(kIdx), static_cast<uint64_t>(B) * H};
        const uint64_t qstr[1] = {static_cast<uint64_t>(kIdx)};
        const uint32_t qbox[2] = {static_cast<uint32_t>(kIdx), static_cast<uint32_t>(n_pad)};
        if (!encode_tmap(&tm_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a->idx_cache_dev, cdims, cstr, cbox,
                         fp4 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B) ||
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
        P.k = plan->topk;
        P.out_idx = a->out_idx_dev;
        P.out_stride = a->out_stride;
        P.out_len = a->out_len_dev;
        P.row_seq = a->row_seq_dev;
        P.bt_rows = a->bt_rows;
        const bool fused = plan->idx_fused_topk != 0;
        static PerDeviceOnce tc_attr;
        const bool attr_ok = tc_attr.run([] {
            // the whole unified L1 as shared memory
            const auto set = [](const void* f, int smem) {
                return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
                       cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                            cudaSharedmemCarveoutMaxShared) == cudaSuccess;
            };
            return set(reinterpret_cast<const void*>(indexer_logits_tc<false, false>), kIdxSmem) &&
                   set(reinterpret_cast<const void*>(indexer_logits_tc<true, false>), kIdxSmemFused) &&
                   set(reinterpret_cast<const void*>(indexer_logits_tc<false, true>), kIdxSmem4) &&
                   set(reinterpret_cast<const void*>(indexer_logits_tc<true, true>), kIdxSmem4Fused);
        });
        if (!attr_ok) return DSV4_ERR_CUDA;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(plan->idx_ctas_per_seq, B, 1);
        cfg.blockDim = dim3(kIdxThreads, 1, 1);
        cfg.dynamicSmemBytes = fp4 ? (fused ? kIdxSmem4Fused : kIdxSmem4) : (fused ? kIdxSmemFused : kIdxSmem);
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        // with the top-k in the launch, a sequence's CTAs form one cluster
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = plan->idx_ctas_per_seq;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = fused ? 2 : 1;
        cudaError_t e =
            fp4 ? (fused ? cudaLaunchKernelEx(&cfg, indexer_logits_tc<true, true>, tm_cache, tm_q, P)
                         : cudaLaunchKernelEx(&cfg, indexer_logits_tc<false, true>, tm_cache, tm_q, P))
                : (fused ? cudaLaunchKernelEx(&cfg, indexer_logits_tc<true, false>, tm_cache, tm_q, P)
                         : cudaLaunchKernelEx(&cfg, indexer_logits_tc<false, false>, tm_cache, tm_q, P));
        if (e != cudaSuccess) return DSV4_ERR_CUDA;
        if (fused) return DSV4_OK;
    }
    cudaError_t e;
    if (plan->max_slots <= kTopkSmallMax) {
        // programmatic dependent launch: the top-k CTAs may be scheduled while the
        // logits kernel drains; they wait (griddepcontrol.wait) before reading it
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(B, 1, 1);
        cfg.blockDim = dim3(kTopkThreads, 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = plan->idx_ctas_per_seq > 0 ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, topk_small_kernel, static_cast<const float*>(logits), plan->logits_stride,
                               plan->max_slots, a->ctx_len_dev, plan->topk, a->out_idx_dev, a->out_stride,
                               a->out_len_dev);
        return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
    }
    {
        // long rows: a cluster of C CTAs per query (8192 keys or more each), S
        // keys each; clusters of more than 8 CTAs need the non-portable size,
        // and a launch the device refuses is retried with 8
        static PerDeviceOnce tkc_attr;
        if (!tkc_attr.run([] {
                return cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(tkc_smem_bytes(kTkcSlots))) == cudaSuccess &&
                       cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                            1) == cudaSuccess;
            }))
            return DSV4_ERR_CUDA;
        for (int cmax = kTkcMaxCluster; cmax >= kCtkMaxCluster; cmax /= 2) {
            const int Cq = min(cmax, (plan->max_slots + 8191) / 8192);
            const int S = ((plan->max_slots + Cq - 1) / Cq + 31) & ~31;
            if (S > kTkcSlots) break;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(Cq, B, 1);
            cfg.blockDim = dim3(kTopkThreads, 1, 1);
            cfg.dynamicSmemBytes = tkc_smem_bytes(S);
            cfg.stream = st;
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = plan->idx_ctas_per_seq > 0 ? 1 : 0;
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = Cq;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 2;
            e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel, static_cast<const float*>(logits), plan->logits_stride,
                                   plan->max_slots, a->ctx_len_dev, plan->topk, S, a->out_idx_dev, a->out_stride,
                                   a->out_len_dev, a->status_dev);
            if (e == cudaSuccess) return DSV4_OK;
            if (Cq <= kCtkMaxCluster) return DSV4_ERR_CUDA;
            (void)cudaGetLastError();                   // a refused cluster size: try the portable one
        }
    }
    const int smem_keys = plan->max_slots <= kTopkSmemKeys ? plan->max_slots : 0;
    const size_t smem = static_cast<size_t>(smem_keys) * 4;
    static PerDeviceOnce topk_attr;
    if (!topk_attr.run([] {
            return cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kTopkSmemKeys * 4) == cudaSuccess;
        }))
        return DSV4_ERR_CUDA;
    topk_kernel<<<B, kTopkThreads, smem, st>>>(logits, plan->logits_stride, plan->max_slots, a->ctx_len_dev,
                                               plan->topk, a->out_idx_dev, a->out_stride, a->out_len_dev,
                                               smem_keys);
    e = cudaGetLastError();
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
