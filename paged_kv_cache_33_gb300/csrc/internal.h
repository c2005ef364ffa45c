// Host-side declarations shared by the C ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

struct kv_pool {
  int device = 0;
  int sm_count = 0;
  int64_t num_blocks = 0;
  int32_t block_size = 0, n_kv_heads = 0, head_dim = 0;
  kv_dtype dtype = KV_BF16;
  void* base = nullptr;        // device pool memory
  uint64_t bytes = 0;
  float* scales = nullptr;     // device [2][Hkv]: K scales then V scales
  uint32_t* err = nullptr;     // device error word
  CUtensorMap tmap;            // pool viewed as [NB*Hkv][2][BS][D] for TMA
  int32_t partition_blocks = 0;  // 0 = automatic
  cudaEvent_t ev_start = nullptr, ev_stop = nullptr;  // optional timing hook
};

namespace pkv {

// Arguments of the split-K decode and its reduce, shared by all variants.
struct DecodeParams {
  const void* q;                // bf16 [B][Hq][D]
  const int32_t* block_tables;  // [B][mbs]
  const int32_t* context_lens;  // [B]
  float* out;                   // [B][Hq][D]
  float* part_o;                // [B][Hq][max_parts][D]  unnormalised partial outputs
  float* part_ml;               // [B][Hq][max_parts][2]  (running max in log2 units, sum)
  uint32_t* err;
  const float* k_scale;         // fp8: [Hkv]
  const float* v_scale;
  int64_t num_blocks;
  int32_t mbs, batch, n_q_heads, n_kv_heads, group;
  int32_t max_ctx, window, part_blocks, max_parts;
  float scale_log2;             // softmax scale * log2(e)
  uint64_t wait_limit_ns;
};

// Geometry of the split-K launch for one call.
struct DecodePlan {
  int32_t part_blocks;   // blocks per partition
  int32_t max_parts;     // partitions of the longest sequence
  size_t workspace_bytes;
};

DecodePlan plan_decode(const kv_pool* pool, int32_t batch, int32_t n_q_heads,
                       int32_t max_context_len, int32_t sliding_window);

cudaError_t launch_kv_write(const kv_pool* pool, const void* k, const void* v,
                            const int64_t* slots, int64_t num_tokens, cudaStream_t stream);

cudaError_t launch_decode(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream);

cudaError_t launch_reduce(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream);

}  // namespace pkv
