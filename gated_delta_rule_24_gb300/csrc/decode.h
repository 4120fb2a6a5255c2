// Internal interface between the C-ABI host code (api.cpp) and the decode-step kernel
// (decode.cu).  Not part of the public ABI.
#pragma once
#include <cuda_runtime_api.h>
#include <stdint.h>

namespace gdn {

// One decode step: every batch row b (one token) updates its state slot in place.
struct DecodeParams {
  const void* q;  // [B, H_qk, 128] bf16; strides in elements
  int64_t q_sb, q_sh;
  const void* k;  // [B, H_qk, 128] bf16
  int64_t k_sb, k_sh;
  const void* v;  // [B, H_v, 128] bf16
  int64_t v_sb, v_sh;
  const void* g;  // [B, H] or null
  int64_t g_sb, g_sh;
  const void* beta;  // [B, H] or null
  int64_t b_sb, b_sh;
  void* state;       // [slots, H, 128, 128], updated in place
  int64_t st_slot, st_head, st_slots;
  const void* state_idx;  // [B] or null (slot b)
  void* out;              // [B, H, 128] bf16
  int64_t o_sb, o_sh;
  int32_t* dev_err;
  int32_t B, H, H_qk, H_v;
  int32_t g_dtype, b_dtype, st_dtype, idx_dtype;
  float scale;
  int32_t l2norm;
  int32_t in_f16;  // q/k/v/output fp16 instead of bf16
};

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);

}  // namespace gdn
