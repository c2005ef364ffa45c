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
  uint8_t* vexp = nullptr;     // bf16 pools: [NB][Hkv][BS], the largest exponent field of each
                               // V row as paged_kv_write stored it (0: not known)
  CUtensorMap tmap;            // pool viewed as [NB*Hkv][2][BS][D] for TMA
  CUtensorMap tmap_rows;       // bf16 / FP8 pools: the same view, boxes of one tile (K or V);
                               // FP4 pools: each (block, head)'s records as rows of 128 bytes
  int32_t partition_blocks = 0;  // 0 = automatic
  uint64_t wait_limit_ns = 1000000000ull;  // bound of every wait in the kernels
  uint32_t stall_tx = 0;       // test hook (kv_pool_set_test_stall)
  cudaEvent_t ev_start = nullptr, ev_stop = nullptr;  // optional timing hook
};

namespace pkv {

// Sequences per decode launch: every CTA keeps a table of the batch in shared
// memory.  Larger batches are split into several launches by the host.
constexpr int kMaxDecodeBatch = 512;
// Query heads per KV head the decode accepts; groups above 8 run as passes
// of at most 8 heads.
constexpr int kMaxDecodeGroup = 64;

// Arguments of the stream-K decode, shared by all variants.
//
// The work of one call is the sequence of "units" (sequence b, KV head h,
// k-th run of BPU attended blocks of b), ordered by b, then h, then k, cut into
// segments: `num_workers` static shares of its first part, then fixed-size
// chunks of the rest handed out through `ticket`.  A (b, h) pair inside one
// segment is finished by the warp that holds it; a pair cut between segments
// leaves one partial per segment in slot (segment + pair index), merged by
// the reduce kernel.
struct DecodeParams {
  const void* q;                // bf16 [B][Hq][D]
  const int32_t* block_tables;  // [B][mbs]
  const int32_t* context_lens;  // [B]
  float* out;                   // [B][Hq][D]
  float* part_o;                // [slots][g][D]  unnormalised partial outputs
  float* part_ml;               // [slots][g][2]  (max in log2 units, sum)
  int2* pair_meta;              // [B*Hkv]  (first segment, number of segments) per pair
  int32_t* ticket;              // next dynamic chunk; zero at launch
  uint32_t* err;
  const uint8_t* pool;          // pool base (FP4 records are staged with bulk copies)
  const float* k_scale;         // fp8 / fp4: [Hkv]
  const float* v_scale;
  int64_t num_blocks;
  int32_t mbs, batch, n_q_heads, n_kv_heads, group;
  int32_t group_stride;         // query heads per KV head in q and out (>= group: a call
                                // with more than 8 runs as passes of <= 8 heads, q and out
                                // offset to the pass's first head)
  int32_t max_ctx, window, num_workers;
  int64_t num_slots;            // partial slots in the workspace (bounds the reduce's reads)
  float scale_log2;             // softmax scale * log2(e)
  uint64_t wait_limit_ns;
  uint32_t stall_tx;            // test hook: extra bytes expected by worker 0's first copy
};

// Geometry of one call.
struct DecodePlan {
  int32_t ctas;          // persistent CTAs of the decode kernel
  int32_t workers;       // warps sharing the work (ctas * warps per CTA)
  int32_t batch;         // sequences per launch (<= kMaxDecodeBatch)
  size_t part_o_bytes, part_ml_bytes, meta_bytes;
  size_t workspace_bytes;
  int64_t num_slots;
};

DecodePlan plan_decode(const kv_pool* pool, int32_t batch, int32_t n_q_heads,
                       int32_t max_context_len, int32_t sliding_window);

// Warps per CTA, resident CTAs per SM, and pool blocks staged per work unit
// of the decode variant the pool uses.
int decode_warps_per_cta(const kv_pool* pool);
int decode_ctas_per_sm(const kv_pool* pool);
int decode_blocks_per_unit(const kv_pool* pool);
// Most dynamic chunks a launch of at most `max_units` units can hand out.
int64_t decode_max_chunks(int64_t max_units);

// The KV write; with `zero_word` it also clears that int (the decode's ticket
// counter) and lets a programmatic dependent launch early.
// bf16 pools: recompute the V exponent map from the pool's V rows.
cudaError_t launch_refresh_exponent_map(const kv_pool* pool, cudaStream_t stream);
cudaError_t launch_kv_write(const kv_pool* pool, const void* k, const void* v,
                            const int64_t* slots, int64_t num_tokens, cudaStream_t stream,
                            int32_t* zero_word = nullptr);

// The decode kernel; `dependent`: launch as a programmatic dependent of the
// kernel before it on the stream (the KV write of the same step).
cudaError_t launch_decode(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream,
                          bool dependent);

// Bytes of one physical block ([Hkv][2][BS][D] elements, or the FP4 records
// of its Hkv x BS/16 sub-tiles).
int64_t block_bytes(const kv_pool* pool);

// Whole-block copies of host-validated (src, dst) pairs, with the result of
// applying them in order.
cudaError_t launch_copy_blocks(const kv_pool* pool, const int32_t* pairs, int64_t n,
                               cudaStream_t stream);

// Arguments of the paged prefill (extend) attention.
struct PrefillParams {
  const void* q;                // bf16 [T][Hq][D], the new tokens of every sequence
  const int32_t* cu_q_lens;     // [B + 1]
  const int32_t* block_tables;  // [B][mbs]
  const int32_t* context_lens;  // [B]
  float* out;                   // [T][Hq][D]
  uint32_t* err;
  const uint8_t* vexp;          // bf16: the pool's V exponent map (kv_pool::vexp)
  const float* k_scale;         // FP8: [Hkv]
  const float* v_scale;
  int64_t num_blocks;
  int32_t mbs, batch, n_q_heads, n_kv_heads, group, group_pow2;
  int32_t max_ctx, window;
  uint32_t q_sign;              // xor into every word of q: 0x80008000 negates it (the
                                // kernels work with |scale|)
  float scale_log2;             // |softmax scale| * log2(e), at least 1e-30
  uint64_t wait_limit_ns;
};

// Dynamic shared memory of the prefill kernel, and its launch.
int prefill_smem_bytes();
cudaError_t launch_prefill(const kv_pool* pool, const PrefillParams& p, int32_t max_q_len,
                           cudaStream_t stream);
// The same over an FP8 (E4M3) pool, with E4M3 tensor-core products.
cudaError_t launch_prefill_fp8(const kv_pool* pool, const PrefillParams& p, int32_t max_q_len,
                               cudaStream_t stream);
// The same over an FP4 pool, its values dequantised exactly into f16.
cudaError_t launch_prefill_fp4(const kv_pool* pool, const PrefillParams& p, int32_t max_q_len,
                               cudaStream_t stream);

// The merge of cut pairs, launched as a programmatic dependent of the decode.
cudaError_t launch_reduce(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream);

}  // namespace pkv
