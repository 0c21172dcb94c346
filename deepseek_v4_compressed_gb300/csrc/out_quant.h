// out_quant.h -- the inverse RoPE + FP8 output quantisation as an internal
// launch (used by the attention entry point when its merge does not quantise).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dsv4 {

// rows = tokens x heads of bf16 [512] outputs; pos[t] is the token's position,
// or (pos_is_ctx) its context length, the position plus one.
cudaError_t launch_inv_rope_quant(const uint16_t* o, int num_tokens, int n_heads, const int* pos, bool pos_is_ctx,
                                  const float* cos_sin, int max_pos, uint8_t* codes, float* scales, int* status,
                                  cudaStream_t stream);

}  // namespace dsv4
