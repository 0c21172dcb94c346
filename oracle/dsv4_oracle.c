/*
 * dsv4_oracle.c -- plain, slow CPU reference for DeepSeek-V4 compressed sparse
 * attention at decode.  TEST INFRASTRUCTURE ONLY (see dsv4_oracle.h): the
 * product path never includes, links or calls it.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no -ffast-math).
 * -ffp-contract=off matters: without it gcc on aarch64 fuses a*b+c and the fp32
 * operation sequence the cache bytes are defined by would change.
 *
 * Every function states the passage it follows.  Readings of passages that are
 * silent or ambiguous are marked "Reading:".
 */
#include "dsv4_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ========================================================================= */
/* Number formats                                                            */
/* ========================================================================= */

/* bf16 is the top half of an IEEE binary32; widening is exact. */
float or_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even (the usual IEEE rule).
 * [vLLM-classes] "CSA layer Compressor": the RoPE half of a cache entry is
 * stored as bfloat16. */
uint16_t or_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)            /* NaN stays NaN (quiet) */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;                                   /* may carry into inf: correct */
    return (uint16_t)keep;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, largest finite 448.  Normal codes are
 * (1 + m/8) * 2^(e-7); exponent field 0 gives the subnormals m * 2^-9.
 * [vLLM-classes] "CSA layer Compressor": the NoPE part is stored as FP8 E4M3. */
double or_e4m3_to_f64(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + (double)m, e - 10);
    return s ? -v : v;
}

/* Encode to E4M3: the nearest of the 127 non-negative finite codes, ties to
 * the even code, magnitudes past 448 saturate to 448 ("satfinite").  The
 * positive codes 0x00..0x7e increase monotonically in value, so the two
 * candidates are found by bisection: lo = the largest code not above |x|,
 * hi = lo + 1. */
uint8_t or_f32_to_e4m3(float x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    int lo = 0, hi = 0x7e;               /* invariant: value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (or_e4m3_to_f64((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - or_e4m3_to_f64((uint8_t)lo);
    double dhi = or_e4m3_to_f64((uint8_t)hi) - a;
    int best = (dlo < dhi) ? lo : (dhi < dlo) ? hi : ((lo & 1) == 0 ? lo : hi);
    return (uint8_t)(sign | best);
}

void or_f32_to_e4m3_n(long long n, const float* x, uint8_t* out)
{
    for (long long i = 0; i < n; ++i)
        out[i] = or_f32_to_e4m3(x[i]);
}

void or_f32_to_bf16_n(long long n, const float* x, uint16_t* out)
{
    for (long long i = 0; i < n; ++i)
        out[i] = or_f32_to_bf16(x[i]);
}

/* UE8M0 block scale: an unsigned power-of-two exponent stored as e + 127.
 * [vLLM-classes] "CSA layer Compressor" (cache block layout: UE8M0 scales) and
 * [MLA-to-CSA] 6.2 (UE8M0 FP8 quantisation).
 * Reading: the pages do not say how e is chosen.  We take the smallest power
 * of two that keeps the block's largest magnitude within E4M3's 448, so no
 * value saturates; e is clamped to [-127, 127] (the byte then lies in 0..254,
 * 255 being the format's NaN).  An all-zero block takes e = 0. */
int or_ue8m0_exponent(float amax)
{
    if (!(amax > 0.0f))
        return 0;
    int e = -127;
    while (e < 127 && (double)amax > 448.0 * ldexp(1.0, e))
        ++e;
    return e;
}

/* The compressor's exponential, fp32 in, fp32 out, with every operation an
 * IEEE-rounded fp32 add or multiply (no fused multiply-add):
 *   Cody & Waite argument reduction (W. J. Cody, W. Waite, "Software Manual
 *   for the Elementary Functions", 1980): n = rint(x / ln2),
 *   r = (x - n*LN2_HI) - n*LN2_LO with LN2_HI = ln2 cut to 16 significant bits
 *   (so n*LN2_HI is exact for |n| < 256) and LN2_LO = fp32(ln2 - LN2_HI);
 *   then e^r by its Taylor series to degree 7 in Horner form (|r| <= ln2/2,
 *   truncation error < 6e-9 relative), and the result scaled by 2^n.
 * Inputs below -87 return 0 (e^-87 is at the bottom of the normal range);
 * the compressor only evaluates it at score - max <= 0.
 * Reading: the pages fix a softmax over the window but not how exp is
 * evaluated; this definition is used so the FP8 bytes are defined exactly. */
float or_expf(float x)
{
    const float LOG2E = 1.44269504088896340736f;
    const float LN2_HI = 0.693145751953125f;          /* 45426 / 65536 */
    const float LN2_LO = 1.42860682030941723212e-6f;  /* ln2 - LN2_HI */
    const float C[8] = {1.0f, 1.0f, 0.5f, 1.0f / 6.0f, 1.0f / 24.0f, 1.0f / 120.0f,
                        1.0f / 720.0f, 1.0f / 5040.0f};
    if (x < -87.0f)
        return 0.0f;
    if (x > 88.0f)
        x = 88.0f;
    float t = x * LOG2E;
    float n = rintf(t);
    float nh = n * LN2_HI;
    float nl = n * LN2_LO;
    float r = x - nh;
    r = r - nl;
    float p = C[7];
    for (int k = 6; k >= 0; --k) {
        float rp = r * p;
        p = C[k] + rp;
    }
    int ni = (int)n;                      /* in [-126, 127] */
    uint32_t bits = (uint32_t)(ni + 127) << 23;
    float two_n;
    memcpy(&two_n, &bits, sizeof two_n);
    return p * two_n;
}

/* ========================================================================= */
/* Layer type and IndexCache schedule                                        */
/* ========================================================================= */

/* [vLLM-V4-attn] "compress_ratio: the three layer types": every layer reads
 * compress_ratios[layer], takes max(1, r); <= 1 is swaonly, 4 is c4a (overlap
 * compressor + indexer), 128 is c128a (compressor, top-k from metadata).  The
 * compressor asserts ratio in {4, 128}, so any other ratio is unsupported. */
int or_layer_type(int compress_ratio)
{
    int r = compress_ratio < 1 ? 1 : compress_ratio;
    if (r == 1 || r == 4 || r == 128)
        return r;
    return -1;
}

/* [IndexCache] section 2: for a c4 layer, indexer_seq_idx = number of c4
 * layers before it; skip_topk = indexer_seq_idx % freq != 0, only when
 * use_index_cache is on.  A pattern string, when given, takes precedence: its
 * first character must be 'F'; 'S' at the corresponding position means reuse;
 * layers past the end of the string compute.
 * Reading: "corresponding position" is the layer's indexer_seq_idx (its rank
 * among c4 layers), the same counter the frequency rule uses.
 * Returns 0, or -1 for an invalid frequency or pattern. */
int or_index_schedule(const int* ratios, int n_layers, int use_index_cache, int freq,
                      const char* pattern, uint8_t* skip_topk)
{
    if (n_layers < 0)
        return -1;
    if (pattern) {
        if (pattern[0] != 'F')
            return -1;
        for (const char* c = pattern; *c; ++c)
            if (*c != 'F' && *c != 'S')
                return -1;
    } else if (use_index_cache && freq < 1) {
        return -1;
    }
    int plen = pattern ? (int)strlen(pattern) : 0;
    int seq_idx = 0;
    for (int l = 0; l < n_layers; ++l) {
        int r = ratios[l] < 1 ? 1 : ratios[l];
        skip_topk[l] = 0;
        if (r == 4) {
            if (use_index_cache) {
                if (pattern)
                    skip_topk[l] = (seq_idx < plen && pattern[seq_idx] == 'S') ? 1 : 0;
                else
                    skip_topk[l] = (seq_idx % freq != 0) ? 1 : 0;
            }
            ++seq_idx;
        }
    }
    return 0;
}

/* ========================================================================= */
/* Cache byte accounting                                                     */
/* ========================================================================= */

/* [MLA-to-CSA] 5.5 (SWA cache format): nope fp8 bytes + rope bf16 bytes +
 * nope/64 UE8M0 scale bytes padded to 8 (448 + 128 + 7 + 1 = 584).  With the
 * 512-latent geometry the same rule gives 512 + 128 + 8 = 648. */
int or_mla_entry_bytes(int nope_dim, int rope_dim)
{
    int scale_bytes = (nope_dim / 64 + 7) / 8 * 8;
    return nope_dim + 2 * rope_dim + scale_bytes;
}

/* [vLLM-classes] DeepseekV4Indexer: head_dim + head_dim // quant_block * 4
 * bytes, quant_block = 128: 128 fp8 + one fp32 scale = 132. */
int or_idx_entry_bytes(int head_dim) { return head_dim + head_dim / 128 * 4; }

/* ========================================================================= */
/* RoPE table                                                                */
/* ========================================================================= */

/* [vLLM-classes] DeepseekCompressor.forward comment: cos_sin_cache is
 * [max_pos, rope_head_dim], first half cos, second half sin, one value per
 * rotated pair.  Angle of pair i at position pos: pos * theta^(-2i/rope_dim).
 * Built in double and rounded once to fp32. */
void or_rope_table(int max_pos, int rope_dim, double theta, float* out)
{
    int half = rope_dim / 2;
    for (int pos = 0; pos < max_pos; ++pos) {
        for (int i = 0; i < half; ++i) {
            double freq = pow(theta, -2.0 * (double)i / (double)rope_dim);
            double ang = (double)pos * freq;
            out[(long long)pos * rope_dim + i] = (float)cos(ang);
            out[(long long)pos * rope_dim + half + i] = (float)sin(ang);
        }
    }
}

/* ========================================================================= */
/* Compressor                                                                */
/* ========================================================================= */

/* Pooled (pre-norm) vector of the compressed entry emitted at boundary token p
 * of one sequence.
 *
 * kv_score holds, for positions 0..p of the sequence, the bf16 projection row
 * [kv block 0 | kv block 1 | score block 0 | score block 1] (coff blocks of d
 * each; [vLLM-classes] "CSA layer Compressor": "kv block0, kv block1, score
 * block0, score block1").  ape is [ratio][coff*d] fp32.
 *
 * Steps, following [vLLM-classes] DeepseekCompressor / save_partial_states and
 * "CSA layer Compressor", [vLLM-V4-attn] "Compressor: ratio 4 vs 128" and
 * [MLA-to-CSA] 5.1 / 5.2:
 *  - ratio 4 uses overlap (coff = 2): the window is the 8 tokens p-7..p; the
 *    old group p-7..p-4 contributes its block 0 (a), the new group p-3..p its
 *    block 1 (b) (the C_Comp formula's [Z_a + B_a; Z_b + B_b] stacking and the
 *    pos=3 / pos=7 table).  Ratio 128 has coff = 1: the window is the 128
 *    tokens p-127..p, block 0.
 *  - Tokens at negative positions are left out (pos >= 0 mask at the first
 *    boundary).
 *  - state values: kv = bf16 -> fp32 (exact); score = fp32(bf16 score +
 *    ape[t % ratio]) -- the APE addition fused into the state save.
 *  - per channel c, softmax over the window rows of the score, weights applied
 *    to the kv rows and summed ("Softmax_row(...)^T (.) C").
 * Reading: the softmax runs per channel across the window tokens.  fp32 ops
 * in this order: m = max score; e_t = or_expf(score_t - m); num += e_t * kv_t;
 * den += e_t (ascending t, each op rounded); y = num / den.
 * Returns 0, or -1 if p is not a boundary ((p + 1) % ratio != 0). */
int or_compress_pool(int ratio, int d, const uint16_t* kv_score, long long row_stride,
                     const float* ape, int p, float* y)
{
    if (ratio != 4 && ratio != 128)
        return -1;
    if ((p + 1) % ratio != 0)
        return -1;
    int coff = (ratio == 4) ? 2 : 1;
    int win = coff * ratio;
    for (int c = 0; c < d; ++c) {
        float sc[128], kv[128];
        int n = 0;
        for (int t = p - win + 1; t <= p; ++t) {
            if (t < 0)
                continue;
            int blk = (coff == 2 && t <= p - ratio) ? 0 : coff - 1;
            const uint16_t* row = kv_score + (long long)t * row_stride;
            float kvv = or_bf16_to_f32(row[blk * d + c]);
            float s = or_bf16_to_f32(row[coff * d + blk * d + c]);
            float a = ape[(long long)(t % ratio) * coff * d + blk * d + c];
            sc[n] = s + a;
            kv[n] = kvv;
            ++n;
        }
        float m = sc[0];
        for (int i = 1; i < n; ++i)
            if (sc[i] > m)
                m = sc[i];
        float num = 0.0f, den = 0.0f;
        for (int i = 0; i < n; ++i) {
            float diff = sc[i] - m;
            float e = or_expf(diff);
            float ek = e * kv[i];
            num = num + ek;
            den = den + e;
        }
        y[c] = num / den;
    }
    return 0;
}

/* RMSNorm over the d channels, weight w ([vLLM-classes] DeepseekCompressor:
 * self.norm = RMSNorm(head_dim, eps); "compress -> RMSNorm -> RoPE").
 * Reading (precision and summation order): the pages give the mean of the
 * squares but not how the sum is formed.  It is formed here in double in one
 * fixed association, so that every implementation following it gets the same
 * bits:
 *  - the squares of channels 2i and 2i+1 are added first (pair i);
 *  - the 32 pair sums of each group of 64 channels are combined by a
 *    butterfly of five levels: at distance 16, 8, 4, 2 and 1, element l
 *    becomes element l plus element (l xor distance); element 0 is then the
 *    group's total;
 *  - the group totals are added to 0 in ascending group order.
 * Every square of an fp32 value is exact in double, so this order alone
 * decides the rounding.  The sum is divided by d in double and rounded once
 * to fp32; then inv = 1 / sqrt(ms + eps) and z = (y * inv) * w, each an
 * IEEE-rounded fp32 operation.  d must be a multiple of 64. */
void or_rmsnorm(const float* y, int d, const float* w, float eps, float* z)
{
    double ss = 0.0;
    for (int g = 0; g < d / 64; ++g) {
        double v[32], nv[32];
        for (int l = 0; l < 32; ++l) {
            double a = (double)y[64 * g + 2 * l];
            double b = (double)y[64 * g + 2 * l + 1];
            double aa = a * a, bb = b * b;
            v[l] = aa + bb;
        }
        for (int dist = 16; dist >= 1; dist /= 2) {
            for (int l = 0; l < 32; ++l)
                nv[l] = v[l] + v[l ^ dist];
            memcpy(v, nv, sizeof v);
        }
        ss += v[0];
    }
    float ms = (float)(ss / (double)d);
    float root = sqrtf(ms + eps);
    float inv = 1.0f / root;
    for (int c = 0; c < d; ++c) {
        float t = y[c] * inv;
        z[c] = t * w[c];
    }
}

/* GPT-J style (interleaved pairs, not split-half) forward rotation of the
 * rope_dim values at x, pair i = (x[2i], x[2i+1]) with cos = row[i],
 * sin = row[rope_dim/2 + i]  ([vLLM-classes] DeepseekCompressor.forward RoPE
 * comment).  Each product and the sum/difference are separately rounded. */
void or_rope_gptj(float* x, int rope_dim, const float* cos_sin_row)
{
    int half = rope_dim / 2;
    for (int i = 0; i < half; ++i) {
        float x0 = x[2 * i], x1 = x[2 * i + 1];
        float c = cos_sin_row[i], s = cos_sin_row[half + i];
        float a = x0 * c, b = x1 * s, e = x0 * s, f = x1 * c;
        x[2 * i] = a - b;
        x[2 * i + 1] = e + f;
    }
}

/* Main (MLA) cache entry: FP8 E4M3 of the nope dims with one UE8M0 scale per
 * 64 dims, bf16 RoPE dims ([vLLM-classes] "CSA layer Compressor": nope -> FP8
 * quant blocks + scale, rope -> bf16; [MLA-to-CSA] 5.5 / 6.2).
 * data = nope fp8 codes then rope bf16 (little-endian); scales = 8 bytes
 * (nope/64 used, rest 0).  code = E4M3(z * 2^-e), the scaling exact. */
void or_quant_mla(const float* z, int nope_dim, int rope_dim, uint8_t* data, uint8_t* scales)
{
    memset(scales, 0, 8);
    for (int b = 0; b < nope_dim / 64; ++b) {
        float amax = 0.0f;
        for (int c = 0; c < 64; ++c) {
            float a = fabsf(z[b * 64 + c]);
            if (a > amax)
                amax = a;
        }
        int e = or_ue8m0_exponent(amax);
        float mult = (float)ldexp(1.0, -e);
        for (int c = 0; c < 64; ++c)
            data[b * 64 + c] = or_f32_to_e4m3(z[b * 64 + c] * mult);
        scales[b] = (uint8_t)(e + 127);
    }
    for (int i = 0; i < rope_dim; ++i) {
        uint16_t h = or_f32_to_bf16(z[nope_dim + i]);
        data[nope_dim + 2 * i] = (uint8_t)(h & 0xff);
        data[nope_dim + 2 * i + 1] = (uint8_t)(h >> 8);
    }
}

/* Indexer cache entry: all d (=128) dims in FP8 E4M3 with one fp32 scale
 * ([vLLM-classes] DeepseekV4Indexer: "128 fp8 + 4 fp32 scale = 132").
 * Reading: scale = amax / 448 (IEEE fp32 division; 1 if the row is all zero),
 * code = E4M3(z / scale). */
void or_quant_idx(const float* z, int d, uint8_t* data, float* scale)
{
    float amax = 0.0f;
    for (int c = 0; c < d; ++c) {
        float a = fabsf(z[c]);
        if (a > amax)
            amax = a;
    }
    float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    for (int c = 0; c < d; ++c)
        data[c] = or_f32_to_e4m3(z[c] / s);
    *scale = s;
}

/* ---- FP4 (MXFP4) indexer cache ------------------------------------------ */

/* OCP MX FP4 "E2M1": 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no
 * infinities or NaN.  Exponent field e > 0 gives (1 + m/2) * 2^(e-1);
 * e = 0 gives the subnormals m * 0.5.  The non-negative values are 0, 0.5,
 * 1, 1.5, 2, 3, 4, 6.  [V4-attn] eval note use_fp4_indexer_cache (the
 * indexer's K cache in MXFP4); [MLA-to-CSA] 6.1 (lightning-indexer K cache
 * FP4 / MXFP4). */
double or_e2m1_to_f64(uint8_t code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return s ? -v : v;
}

/* Encode to E2M1: the nearest of the 8 magnitudes, ties to the even code
 * (mantissa bit 0), magnitudes past 6 saturate to 6.  Same bisection as the
 * E4M3 encoder: the codes 0..7 increase in value. */
uint8_t or_f32_to_e2m1(float x)
{
    uint8_t sign = signbit(x) ? 0x8 : 0x0;
    double a = fabs((double)x);
    if (isnan(x) || a >= 6.0)
        return (uint8_t)(sign | 0x7);
    int lo = 0, hi = 7;                  /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (or_e2m1_to_f64((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - or_e2m1_to_f64((uint8_t)lo);
    double dhi = or_e2m1_to_f64((uint8_t)hi) - a;
    int best = (dlo < dhi) ? lo : (dhi < dlo) ? hi : ((lo & 1) == 0 ? lo : hi);
    return (uint8_t)(sign | best);
}

/* MX block exponent for FP4.
 * Reading: the pages name MXFP4 but not how its shared scale is chosen.  We
 * take the rule of the FP8 UE8M0 scales (or_ue8m0_exponent) with E2M1's
 * largest magnitude 6 in place of 448: the smallest e with amax <= 6 * 2^e,
 * so no value saturates; clamped to [-127, 127]; an all-zero block takes
 * e = 0.  Stored as the byte e + 127. */
int or_mxfp4_exponent(float amax)
{
    if (!(amax > 0.0f))
        return 0;
    int e = -127;
    while (e < 127 && (double)amax > 6.0 * ldexp(1.0, e))
        ++e;
    return e;
}

/* FP4 indexer entry of d (= 128) dims: E2M1 codes of blocks of 32 dims, each
 * block with its own UE8M0 exponent: code = E2M1(z * 2^-e), the scaling
 * exact.  data holds d/2 bytes, element 2i in the low nibble of byte i and
 * element 2i+1 in the high nibble; scales holds d/32 bytes e + 127.
 * Reading: 64 + 4 = 68 bytes per entry, the C4 indexer's 64 x 68 B FP4 block
 * of the V4 internals talk (the class walkthrough keeps the FP8 allocation of
 * 132 B and uses only part of it). */
void or_quant_idx_fp4(const float* z, int d, uint8_t* data, uint8_t* scales)
{
    memset(data, 0, (size_t)d / 2);
    for (int b = 0; b < d / 32; ++b) {
        float amax = 0.0f;
        for (int c = 0; c < 32; ++c) {
            float a = fabsf(z[b * 32 + c]);
            if (a > amax)
                amax = a;
        }
        int e = or_mxfp4_exponent(amax);
        float mult = (float)ldexp(1.0, -e);
        for (int c = 0; c < 32; ++c) {
            int i = b * 32 + c;
            uint8_t code = or_f32_to_e2m1(z[i] * mult);
            data[i / 2] |= (uint8_t)((i & 1) ? (code << 4) : code);
        }
        scales[b] = (uint8_t)(e + 127);
    }
}

void or_quant_idx_fp4_rows(long long n, const float* z, int d, uint8_t* data, uint8_t* scales)
{
    for (long long i = 0; i < n; ++i)
        or_quant_idx_fp4(z + i * d, d, data + i * (d / 2), scales + i * (d / 32));
}

int or_idx_fp4_entry_bytes(int head_dim) { return head_dim / 2 + head_dim / 32; }

/* Row-batched forms of or_quant_mla / or_quant_idx (n rows of d floats). */
void or_quant_mla_rows(long long n, const float* z, int nope_dim, int rope_dim, uint8_t* data,
                       uint8_t* scales)
{
    int d = nope_dim + rope_dim, db = nope_dim + 2 * rope_dim;
    for (long long i = 0; i < n; ++i)
        or_quant_mla(z + i * d, nope_dim, rope_dim, data + i * db, scales + i * 8);
}

void or_quant_idx_rows(long long n, const float* z, int d, uint8_t* data, float* scale)
{
    for (long long i = 0; i < n; ++i)
        or_quant_idx(z + i * d, d, data + i * d, scale + i);
}

/* Run the compressor over positions 0..n_tokens-1 of one sequence and emit
 * every compressed entry in slot order: slot j at boundary p = ratio*j +
 * ratio - 1 ([MLA-to-CSA] 6.3: is_valid = (pos + 1) % ratio == 0,
 * pos_after_compress = pos // ratio).  The pooled vector is RMS-normalised,
 * its last rope_dim dims rotated at position (p // ratio) * ratio
 * ([vLLM-V4-attn] "Compressor"; [MLA-to-CSA] 5.1: anchor 4j for slot j) and
 * quantised.
 * kind 0 = main cache (d = nope + rope; out_data rows of nope + 2*rope bytes,
 * out_scale rows of 8 bytes); kind 1 = indexer cache (d = nope + rope, usually
 * 64 + 64; out_data rows of d bytes, out_scale rows of one fp32); kind 2 =
 * FP4 indexer cache (out_data rows of d/2 bytes, out_scale rows of d/32
 * exponent bytes, or_quant_idx_fp4).
 * Returns the number of entries written, or -1. */
int or_compress_stream(int kind, int ratio, int n_tokens, const uint16_t* kv_score,
                       long long row_stride, const float* ape, const float* rms_w, float eps,
                       const float* cos_sin, int rope_dim, int nope_dim,
                       uint8_t* out_data, uint8_t* out_scale)
{
    int d = nope_dim + rope_dim;
    float* y = (float*)malloc(sizeof(float) * (size_t)d);
    float* z = (float*)malloc(sizeof(float) * (size_t)d);
    int n_out = 0;
    for (int p = 0; p < n_tokens; ++p) {
        if ((p + 1) % ratio != 0)
            continue;
        if (or_compress_pool(ratio, d, kv_score, row_stride, ape, p, y) != 0) {
            n_out = -1;
            break;
        }
        or_rmsnorm(y, d, rms_w, eps, z);
        int rope_pos = (p / ratio) * ratio;
        or_rope_gptj(z + nope_dim, rope_dim, cos_sin + (long long)rope_pos * rope_dim);
        if (kind == 0) {
            int eb = nope_dim + 2 * rope_dim;
            or_quant_mla(z, nope_dim, rope_dim, out_data + (long long)n_out * eb,
                         out_scale + (long long)n_out * 8);
        } else if (kind == 1) {
            float s;
            or_quant_idx(z, d, out_data + (long long)n_out * d, &s);
            memcpy(out_scale + (long long)n_out * 4, &s, 4);
        } else {
            or_quant_idx_fp4(z, d, out_data + (long long)n_out * (d / 2),
                             out_scale + (long long)n_out * (d / 32));
        }
        ++n_out;
    }
    free(y);
    free(z);
    return n_out;
}

/* Write entries 0..n_entries-1 (slot order) of one sequence into a paged
 * cache.  Slot j lives in page block_table[j / page], row j % page
 * ([MLA-to-CSA] 6.3 slot mapping).  Page layout ([vLLM-classes] "CSA layer
 * Compressor": data plane of page*entry bytes, then the scale plane):
 *   kind 0: [page][nope + 2*rope] data, then [page][8] UE8M0 scale bytes;
 *   kind 1: [page][d] fp8 data, then [page] fp32 scales (d = nope + rope);
 *   kind 2: [page][d/2] E2M1 codes, then [page][d/32] exponent bytes (the
 *           FP4 indexer cache: 64 x (64 + 4) bytes for d = 128). */
void or_page_write(int kind, int nope_dim, int rope_dim, int page, const int* block_table,
                   int n_entries, const uint8_t* data, const uint8_t* scale, uint8_t* cache)
{
    int d = nope_dim + rope_dim;
    int data_b = (kind == 0) ? nope_dim + 2 * rope_dim : (kind == 1 ? d : d / 2);
    int scale_b = (kind == 0) ? 8 : (kind == 1 ? 4 : d / 32);
    long long page_b = (long long)page * (data_b + scale_b);
    for (int j = 0; j < n_entries; ++j) {
        uint8_t* base = cache + (long long)block_table[j / page] * page_b;
        int r = j % page;
        memcpy(base + (long long)r * data_b, data + (long long)j * data_b, (size_t)data_b);
        memcpy(base + (long long)page * data_b + (long long)r * scale_b,
               scale + (long long)j * scale_b, (size_t)scale_b);
    }
}

/* ========================================================================= */
/* Lightning indexer and top-k                                               */
/* ========================================================================= */

/* I_s = sum_j w_j * ReLU(q_j . k_s) over the n_c causal compressed slots
 * ([vLLM-classes] SparseAttnIndexer formula; [V4-internals] section 2;
 * [MLA-to-CSA] 5.1).  One key per slot is shared by all heads.  The key is
 * the FP8 row times its fp32 scale; the scale is positive, so it factors out
 * of the ReLU: I_s = scale_s * sum_j w_j * ReLU(q_j . k8_s).
 * Reading: any per-head q scale is already folded into w by the caller.
 * FP8 products are exact in double, so are the 128-term dots. */
void or_indexer_logits(const uint8_t* q_fp8, const float* w, int n_heads, int d,
                       const uint8_t* cache, const int* block_table, int page, int n_c,
                       double* out)
{
    long long page_b = (long long)page * (d + 4);
    double* qd = (double*)malloc(sizeof(double) * (size_t)n_heads * (size_t)d);
    for (int i = 0; i < n_heads * d; ++i)
        qd[i] = or_e4m3_to_f64(q_fp8[i]);
    double kd[512];
    for (int s = 0; s < n_c; ++s) {
        const uint8_t* base = cache + (long long)block_table[s / page] * page_b;
        int r = s % page;
        const uint8_t* k = base + (long long)r * d;
        float scale;
        memcpy(&scale, base + (long long)page * d + (long long)r * 4, 4);
        for (int c = 0; c < d; ++c)
            kd[c] = or_e4m3_to_f64(k[c]);
        double acc = 0.0;
        for (int j = 0; j < n_heads; ++j) {
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += qd[(long long)j * d + c] * kd[c];
            acc += (double)w[j] * (dot > 0.0 ? dot : 0.0);
        }
        out[s] = (double)scale * acc;
    }
    free(qd);
}

/* Indexer logits over an FP4 indexer cache (kind 2 pages): the same
 * formula as or_indexer_logits with k[s][c] = E2M1(code) * 2^(byte_b - 127)
 * for the 32-dim block b of c, and no per-row fp32 scale.  The query stays
 * FP8 E4M3 ([V4-attn]: the FP4 option changes only the indexer's K cache).
 * Every product is exact in double, so are the 128-term dots. */
void or_indexer_logits_fp4(const uint8_t* q_fp8, const float* w, int n_heads, int d,
                           const uint8_t* cache, const int* block_table, int page, int n_c,
                           double* out)
{
    long long page_b = (long long)page * (d / 2 + d / 32);
    double* qd = (double*)malloc(sizeof(double) * (size_t)n_heads * (size_t)d);
    for (int i = 0; i < n_heads * d; ++i)
        qd[i] = or_e4m3_to_f64(q_fp8[i]);
    double kd[512];
    for (int s = 0; s < n_c; ++s) {
        const uint8_t* base = cache + (long long)block_table[s / page] * page_b;
        int r = s % page;
        const uint8_t* k = base + (long long)r * (d / 2);
        const uint8_t* sc = base + (long long)page * (d / 2) + (long long)r * (d / 32);
        for (int c = 0; c < d; ++c) {
            uint8_t code = (c & 1) ? (uint8_t)(k[c / 2] >> 4) : (uint8_t)(k[c / 2] & 15);
            kd[c] = or_e2m1_to_f64(code) * ldexp(1.0, (int)sc[c / 32] - 127);
        }
        double acc = 0.0;
        for (int j = 0; j < n_heads; ++j) {
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += qd[(long long)j * d + c] * kd[c];
            acc += (double)w[j] * (dot > 0.0 ? dot : 0.0);
        }
        out[s] = acc;
    }
    free(qd);
}

typedef struct { double v; int i; } or_scored;

static int cmp_score_desc(const void* a, const void* b)
{
    const or_scored* x = (const or_scored*)a;
    const or_scored* y = (const or_scored*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

static int cmp_int(const void* a, const void* b)
{
    int x = *(const int*)a, y = *(const int*)b;
    return (x > y) - (x < y);
}

/* Per-query top-k ([vLLM-V4-attn] "Indexer, C4A and C128A top-k";
 * [V4-internals] section 6: indices plus lengths).
 * Reading: order by score descending, lower slot first on equal scores; keep
 * min(k, n) slots; report them in ascending slot order, padded with -1;
 * length = min(k, n). */
int or_topk(const double* logits, int n, int k, int* out_idx, int* out_len)
{
    if (n < 0 || k < 0)
        return -1;
    or_scored* v = (or_scored*)malloc(sizeof(or_scored) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < n; ++i) {
        v[i].v = logits[i];
        v[i].i = i;
    }
    qsort(v, (size_t)n, sizeof(or_scored), cmp_score_desc);
    int len = n < k ? n : k;
    for (int i = 0; i < len; ++i)
        out_idx[i] = v[i].i;
    qsort(out_idx, (size_t)len, sizeof(int), cmp_int);
    for (int i = len; i < k; ++i)
        out_idx[i] = -1;
    *out_len = len;
    free(v);
    return 0;
}

/* ========================================================================= */
/* Attention                                                                 */
/* ========================================================================= */

/* Dense multi-query attention in double: every head attends to all n_keys
 * key rows (dk dims); the value is the first dv dims of the key row
 * ([MLA-to-CSA] 2.2 "matrix absorption": decode attends directly over the
 * cached latent vector, MQA-style).  s = scale * q.k; softmax over keys;
 * out = sum_t P_t * key_t[0:dv]; lse = max + log(sum exp(s - max)) (natural
 * log). */
void or_dense_attention(const double* q, int n_heads, const double* keys, int n_keys,
                        int dk, int dv, double scale, double* out, double* lse)
{
    double* s = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
    for (int h = 0; h < n_heads; ++h) {
        const double* qh = q + (long long)h * dk;
        double m = -INFINITY;
        for (int t = 0; t < n_keys; ++t) {
            double dot = 0.0;
            for (int c = 0; c < dk; ++c)
                dot += qh[c] * keys[(long long)t * dk + c];
            s[t] = scale * dot;
            if (s[t] > m)
                m = s[t];
        }
        double den = 0.0;
        for (int t = 0; t < n_keys; ++t) {
            s[t] = exp(s[t] - m);
            den += s[t];
        }
        for (int v = 0; v < dv; ++v) {
            double acc = 0.0;
            for (int t = 0; t < n_keys; ++t)
                acc += s[t] * keys[(long long)t * dk + v];
            out[(long long)h * dv + v] = (n_keys > 0) ? acc / den : 0.0;
        }
        if (lse)
            lse[h] = (n_keys > 0) ? m + log(den) : -INFINITY;
    }
    free(s);
}

/* Key rows a decode query attends to, dequantised to double
 * ([vLLM-V4-attn] "Indexer, C4A and C128A top-k": FlashMLA takes the SWA
 * indices and the compressed top-k indices together; [V4-internals] section
 * 2: KV_actual = selected history || recent window):
 *  1. the compressed slots idx[0..len) of this sequence (logical slot ids,
 *     mapped through comp_bt); value = fp8 * 2^(scale byte - 127) for the
 *     nope dims, bf16 for the rope dims;
 *  2. the raw SWA tokens max(0, p - window + 1) .. p, bf16 rows of
 *     nope + rope values, mapped through swa_bt (pages of `page` tokens).
 * Reading: no de-duplication between the two sets.  comp_cache may be NULL
 * when len == 0 (swaonly).  Returns the number of key rows. */
int or_gather_keys(int nope_dim, int rope_dim, int page,
                   const uint8_t* comp_cache, const int* comp_bt, const int* idx, int len,
                   const uint16_t* swa_cache, const int* swa_bt, int p, int window,
                   double* keys)
{
    int dk = nope_dim + rope_dim;
    int data_b = nope_dim + 2 * rope_dim;
    long long cpage_b = (long long)page * (data_b + 8);
    int n = 0;
    for (int i = 0; i < len; ++i) {
        int slot = idx[i];
        const uint8_t* base = comp_cache + (long long)comp_bt[slot / page] * cpage_b;
        int r = slot % page;
        const uint8_t* row = base + (long long)r * data_b;
        const uint8_t* sc = base + (long long)page * data_b + (long long)r * 8;
        double* k = keys + (long long)n * dk;
        for (int c = 0; c < nope_dim; ++c)
            k[c] = or_e4m3_to_f64(row[c]) * ldexp(1.0, (int)sc[c / 64] - 127);
        for (int i2 = 0; i2 < rope_dim; ++i2) {
            uint16_t h = (uint16_t)(row[nope_dim + 2 * i2] | (row[nope_dim + 2 * i2 + 1] << 8));
            k[nope_dim + i2] = (double)or_bf16_to_f32(h);
        }
        ++n;
    }
    int t0 = p - window + 1 < 0 ? 0 : p - window + 1;
    for (int t = t0; t <= p; ++t) {
        const uint16_t* row = swa_cache + ((long long)swa_bt[t / page] * page + t % page) * dk;
        double* k = keys + (long long)n * dk;
        for (int c = 0; c < dk; ++c)
            k[c] = (double)or_bf16_to_f32(row[c]);
        ++n;
    }
    return n;
}

/* ---- V4-native geometry: K = V over 512 dims, FP8 SWA, inverse RoPE ------ */

/* One V4 cache row of 584 bytes ([MLA-to-CSA] 5.5: 448 NoPE fp8 + 128 RoPE
 * bf16 + 7 UE8M0 scales + 1 pad; pages of 64: data plane then scale plane),
 * dequantised to double: dims 0..447 = fp8 * 2^(scale_b - 127) (64-dim blocks),
 * dims 448..511 = the bf16 RoPE values. */
static void or_v4_row(const uint8_t* cache, const int* bt, int page, int s, double* k)
{
    const int nope = 448, rope = 64, data_b = 576;
    long long page_b = (long long)page * (data_b + 8);
    const uint8_t* base = cache + (long long)bt[s / page] * page_b;
    const uint8_t* row = base + (long long)(s % page) * data_b;
    const uint8_t* sc = base + (long long)page * data_b + (long long)(s % page) * 8;
    for (int c = 0; c < nope; ++c)
        k[c] = or_e4m3_to_f64(row[c]) * ldexp(1.0, (int)sc[c / 64] - 127);
    for (int i = 0; i < rope; ++i) {
        uint16_t h = (uint16_t)(row[nope + 2 * i] | (row[nope + 2 * i + 1] << 8));
        k[nope + i] = (double)or_bf16_to_f32(h);
    }
}

/* Sparse decode attention in the V4-native geometry ([MLA-to-CSA] 5.5 and 6.4:
 * K and V share one 512-dim vector; the SWA cache is FP8 like the compressed
 * one): keys = the compressed slots idx[0..len) (logical ids through comp_bt)
 * followed by the window tokens max(0, p - window + 1) .. p (through swa_bt),
 * both caches of 584-byte rows; s = scale * q.k over the 512 dims; the value
 * is the same 512-dim row.  q bf16 [n_heads][512]; out double [n_heads][512]
 * (the output still carries the keys' rotation: see or_inv_rope_fp8_quant). */
int or_sparse_mla_v4(const uint16_t* q, int n_heads, int page, const uint8_t* comp_cache,
                     const int* comp_bt, const int* idx, int len, const uint8_t* swa_cache,
                     const int* swa_bt, int p, int window, double scale, double* out, double* lse)
{
    const int d = 512;
    int t0 = p - window + 1 < 0 ? 0 : p - window + 1;
    int n = len + (p - t0 + 1);
    double* keys = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * d);
    double* qd = (double*)malloc(sizeof(double) * (size_t)n_heads * d);
    for (int i = 0; i < n_heads * d; ++i)
        qd[i] = (double)or_bf16_to_f32(q[i]);
    int m = 0;
    for (int i = 0; i < len; ++i)
        or_v4_row(comp_cache, comp_bt, page, idx[i], keys + (long long)(m++) * d);
    for (int t = t0; t <= p; ++t)
        or_v4_row(swa_cache, swa_bt, page, t, keys + (long long)(m++) * d);
    or_dense_attention(qd, n_heads, keys, m, d, d, scale, out, lse);
    free(keys);
    free(qd);
    return m;
}

/* Inverse RoPE and FP8 quantisation of the attention output
 * ([MLA-to-CSA] 6.4, fused_inv_rope_fp8_quant; [V4-internals] section 6:
 * Inverse RoPE + FP8 Quant after Flash MLA).  Per head: the 64 RoPE dims
 * (448..511) rotated by R(-pos) -- GPT-J pairs, cos / sin of the query
 * position from the table: x0' = x0 c + x1 s, x1' = x1 c - x0 s, each
 * product and sum rounded to fp32 -- so that R(-i) R(j) k = R(j - i) k; then
 * every 128-dim block quantised as the indexer cache is: scale = amax / 448
 * (fp32; 1 for an all-zero block), code = E4M3(x / scale).
 * Reading: the pages name the fused operator and its inputs (o, positions,
 * cos_sin_cache, groups, nope / rope dims) but not the quantisation grain;
 * 128-dim blocks with fp32 scales (the indexer cache's rule) are taken.
 * o: bf16 bits [n_heads][512]; codes [n_heads][512]; scales [n_heads][4]. */
void or_inv_rope_fp8_quant(const uint16_t* o, int n_heads, int pos, const float* cos_sin, int rope_dim,
                           uint8_t* codes, float* scales)
{
    const int d = 512, nope = 448;
    float x[512];
    for (int h = 0; h < n_heads; ++h) {
        for (int c = 0; c < d; ++c)
            x[c] = or_bf16_to_f32(o[(long long)h * d + c]);
        const float* row = cos_sin + (long long)pos * rope_dim;
        for (int i = 0; i < rope_dim / 2; ++i) {
            float x0 = x[nope + 2 * i], x1 = x[nope + 2 * i + 1];
            float c = row[i], sn = row[rope_dim / 2 + i];
            float a = x0 * c, b = x1 * sn, e = x1 * c, f = x0 * sn;
            x[nope + 2 * i] = a + b;
            x[nope + 2 * i + 1] = e - f;
        }
        for (int blk = 0; blk < d / 128; ++blk) {
            float sc;
            or_quant_idx(x + blk * 128, 128, codes + (long long)h * d + blk * 128, &sc);
            scales[h * (d / 128) + blk] = sc;
        }
    }
}

/* ---- prefill helpers ----------------------------------------------------- */

/* Dequantise-and-gather of cache rows into a dense bf16 buffer ([vLLM-classes]
 * _forward_prefill, dequantize_and_gather_k_cache: the compressed cache into
 * kv[:, 0:N], the SWA cache into kv[:, N : N + gather_len]).
 * kind 0: compressed entries of logical slots s0 .. s0 + n - 1 of a sequence
 * (block table bt, 64-entry pages of nope + 2*rope data bytes then 8 scale
 * bytes): row = FP8 * 2^(scale - 127) for the nope dims, the bf16 rope dims;
 * kind 1: SWA rows of tokens s0 .. s0 + n - 1 (bf16, nope + rope per token).
 * out: bf16 [n][nope + rope], each value rounded to bf16 (exact for the
 * dequantised FP8 values in bf16's normal range). */
void or_dequant_gather(int kind, int nope_dim, int rope_dim, int page, const uint8_t* cache,
                       const int* bt, int s0, int n, uint16_t* out)
{
    int d = nope_dim + rope_dim;
    int data_b = nope_dim + 2 * rope_dim;
    long long cpage_b = (long long)page * (data_b + 8);
    for (int i = 0; i < n; ++i) {
        int s = s0 + i;
        uint16_t* o = out + (long long)i * d;
        if (kind == 0) {
            const uint8_t* base = cache + (long long)bt[s / page] * cpage_b;
            const uint8_t* row = base + (long long)(s % page) * data_b;
            const uint8_t* sc = base + (long long)page * data_b + (long long)(s % page) * 8;
            for (int c = 0; c < nope_dim; ++c)
                o[c] = or_f32_to_bf16((float)(or_e4m3_to_f64(row[c]) * ldexp(1.0, (int)sc[c / 64] - 127)));
            for (int c = 0; c < rope_dim; ++c)
                o[nope_dim + c] = (uint16_t)(row[nope_dim + 2 * c] | (row[nope_dim + 2 * c + 1] << 8));
        } else {
            const uint16_t* row = (const uint16_t*)cache + ((long long)bt[s / page] * page + s % page) * d;
            memcpy(o, row, sizeof(uint16_t) * (size_t)d);
        }
    }
}

/* Key index list of one prefill query token over the gathered buffer
 * ([vLLM-classes] _forward_prefill, combine_topk_swa_indices): its top-k
 * compressed slots (indices 0..N-1 of the buffer: slot j at j) followed by its
 * causal window, the raw tokens max(0, pos - window + 1) .. pos, which the
 * buffer holds from index N on for tokens seq_len - gather_len .. seq_len - 1.
 * Reading: the top-k entries past topk_len (or -1) are dropped; the window
 * follows the compressed entries in token order; a window token outside the
 * gathered range is an error (returns -1).  Returns the list's length. */
int or_combine_topk_swa_indices(const int* topk, int topk_len, int pos, int seq_len, int gather_len,
                                int window, int n_comp, int* out)
{
    int n = 0;
    for (int i = 0; i < topk_len; ++i)
        if (topk[i] >= 0)
            out[n++] = topk[i];
    int first = seq_len - gather_len;
    int t0 = pos - window + 1 < 0 ? 0 : pos - window + 1;
    for (int t = t0; t <= pos; ++t) {
        if (t < first || t >= seq_len)
            return -1;
        out[n++] = n_comp + (t - first);
    }
    return n;
}

/* Sparse absorbed-MQA decode for one query token at position p: gather the
 * key set (or_gather_keys) and attend densely over it with the 576-dim key,
 * the value being its first nope_dim dims (the latent)
 * ([vLLM-classes] _forward_decode; [MLA-to-CSA] 2.2, 5.1).
 * q is bf16 [n_heads][nope + rope]; out is [n_heads][nope] in double.
 * Returns the number of keys attended. */
int or_sparse_mla(const uint16_t* q, int n_heads, int nope_dim, int rope_dim, int page,
                  const uint8_t* comp_cache, const int* comp_bt, const int* idx, int len,
                  const uint16_t* swa_cache, const int* swa_bt, int p, int window,
                  double scale, double* out, double* lse)
{
    int dk = nope_dim + rope_dim;
    int max_keys = len + window;
    double* keys = (double*)malloc(sizeof(double) * (size_t)max_keys * (size_t)dk);
    double* qd = (double*)malloc(sizeof(double) * (size_t)n_heads * (size_t)dk);
    for (int i = 0; i < n_heads * dk; ++i)
        qd[i] = (double)or_bf16_to_f32(q[i]);
    int n = or_gather_keys(nope_dim, rope_dim, page, comp_cache, comp_bt, idx, len, swa_cache,
                           swa_bt, p, window, keys);
    or_dense_attention(qd, n_heads, keys, n, dk, nope_dim, scale, out, lse);
    free(keys);
    free(qd);
    return n;
}
