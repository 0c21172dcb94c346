// plan.h -- the per-layer-type plan (host object) and its workspace layout.
#pragma once

#include <stddef.h>

#include "dsv4.h"

struct dsv4_plan {
    dsv4_layer_type type;
    dsv4_geom geom;
    int batch;
    int topk;
    int max_ctx;
    int max_slots;           // compressed slots per sequence at max_ctx
    int max_keys;            // topk + window
    int idx_ctas_per_seq;    // indexer split over slots
    int idx_tiles_per_cta;   // 128-slot tiles per indexer CTA
    int idx_fused_topk;      // the top-k runs inside the logits launch (one cluster per sequence)
    int idx_fp4;             // the indexer cache is MXFP4 (68-byte entries), not FP8 (132-byte)
    int kv_v4;               // V4-native attention rows (512 dims, K = V, FP8 SWA)
    int mla_head_groups;     // ceil(n_heads / 64)
    int mla_splits;          // key splits per (sequence, head group)
    int mla_keys_per_split;
    int logits_stride;       // floats per logits row (max_slots rounded up to 4)
    size_t ws_logits_off;    // fp32 [batch][logits_stride] indexer logits
    size_t ws_partial_off;   // fp32 attention partials
    size_t ws_partial_bytes;
    size_t ws_bytes;
};

namespace dsv4 {
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
}
