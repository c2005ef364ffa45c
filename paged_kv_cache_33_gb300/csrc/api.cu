// C ABI of the paged KV cache decode path: pool lifetime, argument checks,
// split-K planning and kernel launches.  Declarations and the contract of
// every entry point are in include/pagedkv.h.

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "common.cuh"
#include "internal.h"

namespace {


// Make the pool's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1, want;
  explicit DeviceGuard(int d) : want(d) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != want) cudaSetDevice(want);
  }
  ~DeviceGuard() {
    if (prev >= 0 && prev != want) cudaSetDevice(prev);
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// The pool as a 4-D tensor (D, BS, 2, NB*Hkv) with a box of one (block, head)
// K+V pair: 64 bf16 columns (head_dim 128 takes two boxes) or 128 E4M3
// columns, 16 token rows, both K and V; 128-byte swizzle in shared memory.
bool encode_pool_map(kv_pool* p) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  if (p->dtype == KV_FP4_E2M1) {
    // The decode stages FP4 records with plain bulk copies; the prefill takes
    // the records of one (block, head), contiguous, as rows of 128 bytes, all
    // of them in one box, verbatim (no swizzle).
    const uint64_t rec = static_cast<uint64_t>(p->block_size / 16) * pkv::kFp4SubBytes;
    cuuint64_t dims[3] = {128, rec / 128, static_cast<cuuint64_t>(p->num_blocks) * p->n_kv_heads};
    cuuint64_t strides[2] = {128, rec};
    cuuint32_t box[3] = {128, static_cast<cuuint32_t>(rec / 128), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return encode(&p->tmap_rows, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p->base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
  }
  const uint64_t esz = p->dtype == KV_BF16 ? 2 : 1;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(p->head_dim),
                        static_cast<cuuint64_t>(p->block_size), 2,
                        static_cast<cuuint64_t>(p->num_blocks) * p->n_kv_heads};
  cuuint64_t strides[3] = {p->head_dim * esz, p->block_size * p->head_dim * esz,
                           2 * p->block_size * p->head_dim * esz};
  // one box: 128 bytes of every K row and every V row of one (block, head)
  // (FP8: the transposed V tile is read as block_size rows of 128 bytes)
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(p->block_size),
                       2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(&p->tmap,
                      p->dtype == KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                      4, p->base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  // the prefill gathers the K rows and the V rows of a block separately: one
  // box is the 128 bytes of every row of one tile (bf16: half a row)
  cuuint32_t box_rows[4] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(p->block_size),
                            1, 1};
  r = encode(&p->tmap_rows,
             p->dtype == KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
             p->base, dims, strides, box_rows, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int32_t blocks_for(int64_t tokens, int32_t bs) { return static_cast<int32_t>((tokens + bs - 1) / bs); }

// Most units one (sequence, KV head) pair can have in a launch.
int64_t max_units_per_pair(const kv_pool* p, int32_t max_context_len, int32_t sliding_window) {
  const int32_t bs = p->block_size;
  int64_t nblk = blocks_for(max_context_len, bs);
  if (sliding_window > 0) nblk = std::min<int64_t>(nblk, (sliding_window - 1) / bs + 2);
  const int bpu = pkv::decode_blocks_per_unit(p);
  return std::max<int64_t>(1, (nblk + bpu - 1) / bpu);
}

}  // namespace

namespace pkv {

DecodePlan plan_decode(const kv_pool* pool, int32_t batch, int32_t n_q_heads,
                       int32_t max_context_len, int32_t sliding_window) {
  DecodePlan plan{};
  plan.batch = std::min(batch, kMaxDecodeBatch);
  const int nw = decode_warps_per_cta(pool);
  // A persistent grid: every SM holds as many CTAs as fit at once.
  const int64_t max_ctas = static_cast<int64_t>(std::max(pool->sm_count, 1)) *
                           decode_ctas_per_sm(pool);
  const int64_t t_max = static_cast<int64_t>(plan.batch) * pool->n_kv_heads *
                        max_units_per_pair(pool, max_context_len, sliding_window);
  int64_t ctas = max_ctas;
  if (pool->partition_blocks > 0) {
    // about `partition_blocks` units per warp for the longest possible launch
    const int64_t workers = (t_max + pool->partition_blocks - 1) / pool->partition_blocks;
    ctas = std::max<int64_t>(1, std::min<int64_t>(max_ctas, (workers + nw - 1) / nw));
  }
  plan.ctas = static_cast<int32_t>(ctas);
  plan.workers = static_cast<int32_t>(ctas * nw);
  const int64_t g = std::min<int64_t>(n_q_heads / pool->n_kv_heads, 8);  // heads per pass
  const int64_t pairs = static_cast<int64_t>(plan.batch) * pool->n_kv_heads;
  // partial slot of (segment s, pair p) is s + p: segments + pairs slots
  const int64_t slots = plan.workers + decode_max_chunks(t_max) + pairs;
  plan.num_slots = slots;
  auto round256 = [](size_t x) { return (x + 255) / 256 * 256; };
  plan.part_o_bytes = round256(static_cast<size_t>(slots * g * pool->head_dim) * sizeof(float));
  plan.part_ml_bytes = round256(static_cast<size_t>(slots * g * 2) * sizeof(float));
  plan.meta_bytes = round256(static_cast<size_t>(pairs) * 2 * sizeof(int32_t) + 16);
  plan.workspace_bytes = plan.part_o_bytes + plan.part_ml_bytes + plan.meta_bytes;
  return plan;
}

}  // namespace pkv

extern "C" {

const char* kv_status_str(kv_status s) {
  switch (s) {
    case KV_OK: return "KV_OK";
    case KV_ERR_INVALID_ARG: return "KV_ERR_INVALID_ARG";
    case KV_ERR_OOM: return "KV_ERR_OOM";
    case KV_ERR_CUDA: return "KV_ERR_CUDA";
    case KV_ERR_UNSUPPORTED: return "KV_ERR_UNSUPPORTED";
    case KV_ERR_BAD_BLOCK_ID: return "KV_ERR_BAD_BLOCK_ID";
    case KV_ERR_TIMEOUT: return "KV_ERR_TIMEOUT";
    case KV_ERR_DRAIN_TIMEOUT: return "KV_ERR_DRAIN_TIMEOUT";
    case KV_ERR_BAD_SLOT: return "KV_ERR_BAD_SLOT";
    case KV_ERR_BAD_CONTEXT: return "KV_ERR_BAD_CONTEXT";
    case KV_ERR_STALE_EXPONENT_MAP: return "KV_ERR_STALE_EXPONENT_MAP";
  }
  return "KV_ERR_UNKNOWN";
}

kv_status kv_pool_create(int64_t num_blocks, int32_t block_size, int32_t n_kv_heads,
                         int32_t head_dim, kv_dtype dtype, kv_pool** out) {
  if (!out) return KV_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks <= 0 || n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
    return KV_ERR_INVALID_ARG;
  if (dtype != KV_BF16 && dtype != KV_FP8_E4M3 && dtype != KV_FP4_E2M1) return KV_ERR_INVALID_ARG;
  if (block_size != 16 && block_size != 32) return KV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return KV_ERR_UNSUPPORTED;
  if (dtype != KV_BF16 && head_dim != 128) return KV_ERR_UNSUPPORTED;
  if (num_blocks * n_kv_heads >= (int64_t(1) << 31)) return KV_ERR_UNSUPPORTED;

  kv_pool* p = new (std::nothrow) kv_pool;
  if (!p) return KV_ERR_OOM;
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->n_kv_heads = n_kv_heads;
  p->head_dim = head_dim;
  p->dtype = dtype;
  std::memset(&p->tmap, 0, sizeof p->tmap);
  std::memset(&p->tmap_rows, 0, sizeof p->tmap_rows);
  p->bytes = static_cast<uint64_t>(num_blocks) * pkv::block_bytes(p);
  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) !=
          cudaSuccess) {
    cudaGetLastError();
    delete p;
    return KV_ERR_CUDA;
  }
  if (cudaMalloc(&p->base, p->bytes) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return KV_ERR_OOM;
  }
  float ones[2 * 256];
  const int ns = 2 * n_kv_heads;
  bool ok = cudaMalloc(reinterpret_cast<void**>(&p->scales), ns * sizeof(float)) == cudaSuccess &&
            cudaMalloc(reinterpret_cast<void**>(&p->err), sizeof(uint32_t)) == cudaSuccess;
  if (ok) {
    for (int i = 0; i < ns && i < 512; ++i) ones[i] = 1.0f;
    for (int i = 0; i < ns && ok; i += 512)
      ok = cudaMemcpy(p->scales + i, ones, std::min(512, ns - i) * sizeof(float),
                      cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemset(p->err, 0, sizeof(uint32_t)) == cudaSuccess;
  }
  ok = ok && encode_pool_map(p);
  if (ok && dtype == KV_BF16) {
    const size_t n = static_cast<size_t>(num_blocks) * n_kv_heads * block_size;
    ok = cudaMalloc(reinterpret_cast<void**>(&p->vexp), n) == cudaSuccess &&
         cudaMemset(p->vexp, 0, n) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();
    cudaFree(p->base);
    cudaFree(p->scales);
    cudaFree(p->err);
    cudaFree(p->vexp);
    delete p;
    return KV_ERR_CUDA;
  }
  *out = p;
  return KV_OK;
}

kv_status kv_pool_destroy(kv_pool* p) {
  if (!p) return KV_ERR_INVALID_ARG;
  DeviceGuard guard(p->device);
  cudaError_t e = cudaDeviceSynchronize();
  cudaFree(p->base);
  cudaFree(p->scales);
  cudaFree(p->err);
  cudaFree(p->vexp);
  delete p;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kv_status kv_pool_exponent_map(const kv_pool* p, void** map_dev, int64_t* bytes) {
  if (!p || !map_dev || !bytes) return KV_ERR_INVALID_ARG;
  *map_dev = p->vexp;
  *bytes = p->vexp ? p->num_blocks * p->n_kv_heads * p->block_size : 0;
  return KV_OK;
}

kv_status kv_pool_refresh_exponent_map(kv_pool* p, void* stream) {
  if (!p) return KV_ERR_INVALID_ARG;
  if (!p->vexp) return KV_OK;
  DeviceGuard guard(p->device);
  if (pkv::launch_refresh_exponent_map(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return KV_OK;
}

kv_status kv_pool_info(const kv_pool* p, kv_pool_desc* out) {
  if (!p || !out) return KV_ERR_INVALID_ARG;
  out->base_dev = p->base;
  out->num_blocks = p->num_blocks;
  out->block_size = p->block_size;
  out->n_kv_heads = p->n_kv_heads;
  out->head_dim = p->head_dim;
  out->dtype = p->dtype;
  out->strides[4] = 1;
  out->strides[3] = p->head_dim;
  out->strides[2] = static_cast<int64_t>(p->block_size) * p->head_dim;
  out->strides[1] = 2 * out->strides[2];
  out->strides[0] = static_cast<int64_t>(p->n_kv_heads) * out->strides[1];
  out->bytes = p->bytes;
  out->device = p->device;
  out->scales_dev = p->scales;
  out->v_layout = p->dtype == KV_FP8_E4M3 ? 1 : p->dtype == KV_FP4_E2M1 ? 2 : 0;
  if (p->dtype == KV_FP4_E2M1)
    for (int i = 0; i < 5; ++i) out->strides[i] = 0;
  return KV_OK;
}

kv_status kv_pool_set_scales(kv_pool* p, const float* k_scale, const float* v_scale,
                             void* stream) {
  if (!p || !k_scale || !v_scale) return KV_ERR_INVALID_ARG;
  DeviceGuard guard(p->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t n = p->n_kv_heads * sizeof(float);
  if (cudaMemcpyAsync(p->scales, k_scale, n, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(p->scales + p->n_kv_heads, v_scale, n, cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return KV_OK;
}

kv_status paged_kv_write(kv_pool* p, const void* k, const void* v, const int64_t* slots,
                         int64_t num_tokens, void* stream) {
  if (!p || num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  if (!k || !v || !slots || !aligned16(k) || !aligned16(v)) return KV_ERR_INVALID_ARG;
  if (num_tokens > (int64_t(1) << 40)) return KV_ERR_INVALID_ARG;
  DeviceGuard guard(p->device);
  cudaError_t e = pkv::launch_kv_write(p, k, v, slots, num_tokens, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kv_status paged_kv_copy_blocks(kv_pool* p, const int32_t* pairs, int64_t num_pairs,
                               void* stream) {
  if (!p || num_pairs < 0 || (num_pairs > 0 && !pairs)) return KV_ERR_INVALID_ARG;
  for (int64_t i = 0; i < 2 * num_pairs; ++i)
    if (pairs[i] < 0 || pairs[i] >= p->num_blocks) return KV_ERR_INVALID_ARG;
  if (num_pairs == 0) return KV_OK;
  DeviceGuard guard(p->device);
  const cudaError_t e = pkv::launch_copy_blocks(p, pairs, num_pairs, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

size_t paged_decode_workspace_bytes(const kv_pool* p, int32_t batch, int32_t n_q_heads,
                                    int32_t max_context_len, int32_t sliding_window) {
  if (!p || batch < 0 || n_q_heads <= 0 || max_context_len < 0) return 0;
  return pkv::plan_decode(p, batch, n_q_heads, max_context_len, sliding_window).workspace_bytes;
}

}  // extern "C"

namespace {

// The new tokens a fused step writes before its attention.
struct StepWrite {
  const void* k;
  const void* v;
  const int64_t* slots;
  int64_t num_tokens;
};

kv_status decode_call(kv_pool* p, const StepWrite* w, const void* q, int32_t n_q_heads,
                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                      const int32_t* context_lens, int32_t batch, int32_t max_context_len,
                      float scale, int32_t sliding_window, float* out, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!p || batch < 0 || n_q_heads <= 0) return KV_ERR_INVALID_ARG;
  if (n_q_heads % p->n_kv_heads != 0) return KV_ERR_INVALID_ARG;
  const int32_t g = n_q_heads / p->n_kv_heads;
  if (g > pkv::kMaxDecodeGroup) return KV_ERR_UNSUPPORTED;
  if (w) {
    if (w->num_tokens < 0 || w->num_tokens > (int64_t(1) << 40)) return KV_ERR_INVALID_ARG;
    if (w->num_tokens > 0 && (!w->k || !w->v || !w->slots || !aligned16(w->k) || !aligned16(w->v)))
      return KV_ERR_INVALID_ARG;
  }
  if (batch == 0) {
    if (!w || w->num_tokens == 0) return KV_OK;
    DeviceGuard guard(p->device);
    return pkv::launch_kv_write(p, w->k, w->v, w->slots, w->num_tokens,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KV_OK
               : KV_ERR_CUDA;
  }
  if (!q || !block_tables || !context_lens || !out || !aligned16(q) || !aligned16(out))
    return KV_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || max_context_len < 0 ||
      static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * p->block_size)
    return KV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KV_ERR_INVALID_ARG;
  if (batch > 65535 || p->n_kv_heads > 65535) return KV_ERR_UNSUPPORTED;

  DeviceGuard guard(p->device);
  const pkv::DecodePlan plan = pkv::plan_decode(p, batch, n_q_heads, max_context_len, sliding_window);
  if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned16(workspace))
    return KV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(plan.batch) * p->n_kv_heads *
          max_units_per_pair(p, max_context_len, sliding_window) >= (int64_t(1) << 30))
    return KV_ERR_UNSUPPORTED;  // unit indices are 32-bit

  pkv::DecodeParams d{};
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  d.part_o = reinterpret_cast<float*>(ws);
  d.part_ml = reinterpret_cast<float*>(ws + plan.part_o_bytes);
  d.pair_meta = reinterpret_cast<int2*>(ws + plan.part_o_bytes + plan.part_ml_bytes);
  d.ticket = reinterpret_cast<int32_t*>(ws + plan.part_o_bytes + plan.part_ml_bytes +
                                        plan.meta_bytes - 16);
  d.err = p->err;
  d.pool = static_cast<const uint8_t*>(p->base);
  d.k_scale = p->scales;
  d.v_scale = p->scales + p->n_kv_heads;
  d.num_blocks = p->num_blocks;
  d.mbs = max_blocks_per_seq;
  d.n_q_heads = n_q_heads;
  d.n_kv_heads = p->n_kv_heads;
  d.group_stride = g;
  d.max_ctx = max_context_len;
  d.window = sliding_window > 0 ? sliding_window : 0;
  d.num_workers = plan.workers;
  d.num_slots = plan.num_slots;
  d.stall_tx = p->stall_tx;
  d.scale_log2 = scale * 1.4426950408889634f;
  d.wait_limit_ns = p->wait_limit_ns;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool timed = p->ev_start != nullptr;
  // batches beyond one launch's table run as consecutive launches, and a
  // group of more than 8 query heads per KV head as passes over 8 of them
  // at a time (each pass reads the K/V again)
  for (int32_t b0 = 0; b0 < batch; b0 += plan.batch)
  for (int32_t h0 = 0; h0 < g; h0 += 8) {
    const int32_t nb = std::min(plan.batch, batch - b0);
    const int64_t first = static_cast<int64_t>(b0) * n_q_heads + h0;  // the pass's first q row
    d.q = static_cast<const uint16_t*>(q) + first * p->head_dim;
    d.block_tables = block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq;
    d.context_lens = context_lens + b0;
    d.out = out + first * p->head_dim;
    d.batch = nb;
    d.group = std::min(8, g - h0);
    // The fused step's write kernel clears the ticket and lets the first
    // decode launch start while it runs; otherwise a memset clears it.
    const bool fused = w != nullptr && b0 == 0 && h0 == 0;
    if (fused) {
      if (pkv::launch_kv_write(p, w->k, w->v, w->slots, w->num_tokens, s, d.ticket) != cudaSuccess)
        return KV_ERR_CUDA;
    } else if (cudaMemsetAsync(d.ticket, 0, sizeof(int32_t), s) != cudaSuccess) {
      return KV_ERR_CUDA;
    }
    if (timed && cudaEventRecord(p->ev_start, s) != cudaSuccess) return KV_ERR_CUDA;
    if (pkv::launch_decode(p, d, s, fused && !timed) != cudaSuccess) return KV_ERR_CUDA;
    if (timed && cudaEventRecord(p->ev_stop, s) != cudaSuccess) return KV_ERR_CUDA;
    if (pkv::launch_reduce(p, d, s) != cudaSuccess) return KV_ERR_CUDA;
  }
  return KV_OK;
}

}  // namespace

extern "C" {

kv_status paged_decode_attention(kv_pool* p, const void* q, int32_t n_q_heads,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, int32_t batch,
                                 int32_t max_context_len, float scale, int32_t sliding_window,
                                 float* out, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  return decode_call(p, nullptr, q, n_q_heads, block_tables, max_blocks_per_seq, context_lens,
                     batch, max_context_len, scale, sliding_window, out, workspace,
                     workspace_bytes, stream);
}

kv_status paged_decode_step(kv_pool* p, const void* k, const void* v,
                            const int64_t* slot_mapping, int64_t num_tokens, const void* q,
                            int32_t n_q_heads, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* context_lens,
                            int32_t batch, int32_t max_context_len, float scale,
                            int32_t sliding_window, float* out, void* workspace,
                            size_t workspace_bytes, void* stream) {
  const StepWrite w{k, v, slot_mapping, num_tokens};
  return decode_call(p, &w, q, n_q_heads, block_tables, max_blocks_per_seq, context_lens, batch,
                     max_context_len, scale, sliding_window, out, workspace, workspace_bytes,
                     stream);
}

kv_status paged_prefill_attention(kv_pool* p, const void* q, int32_t n_q_heads,
                                  const int32_t* cu_q_lens, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t batch, int32_t max_q_len, int32_t max_context_len,
                                  float scale, int32_t sliding_window, float* out, void* stream) {
  if (!p || batch < 0 || n_q_heads <= 0 || max_q_len < 0 || max_context_len < 0)
    return KV_ERR_INVALID_ARG;
  if (n_q_heads % p->n_kv_heads != 0) return KV_ERR_INVALID_ARG;
  const int32_t g = n_q_heads / p->n_kv_heads;
  // a query tile holds 128 (token, head) rows: groups up to 128 heads
  if (g > 128 || p->head_dim != 128) return KV_ERR_UNSUPPORTED;
  if (batch == 0 || max_q_len == 0) return KV_OK;
  if (!q || !cu_q_lens || !block_tables || !context_lens || !out || !aligned16(q) || !aligned16(out))
    return KV_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || max_q_len > max_context_len ||
      static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * p->block_size)
    return KV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KV_ERR_INVALID_ARG;
  if (batch > 65535 || p->n_kv_heads > 65535) return KV_ERR_UNSUPPORTED;
  int32_t gp = 1;
  while (gp < g) gp <<= 1;
  const int64_t tiles = (static_cast<int64_t>(max_q_len) * gp + 127) / 128;
  if (tiles > (int64_t(1) << 31) - 1) return KV_ERR_UNSUPPORTED;
  DeviceGuard guard(p->device);
  pkv::PrefillParams d{};
  d.q = q;
  d.cu_q_lens = cu_q_lens;
  d.block_tables = block_tables;
  d.context_lens = context_lens;
  d.out = out;
  d.err = p->err;
  d.vexp = p->vexp;
  d.k_scale = p->scales;
  d.v_scale = p->scales + p->n_kv_heads;
  d.num_blocks = p->num_blocks;
  d.mbs = max_blocks_per_seq;
  d.batch = batch;
  d.n_q_heads = n_q_heads;
  d.n_kv_heads = p->n_kv_heads;
  d.group = g;
  d.group_pow2 = gp;
  d.max_ctx = max_context_len;
  d.window = sliding_window > 0 ? sliding_window : 0;
  // The kernels take the row maximum of the unscaled scores and mask with
  // -inf, so they need a positive scale: a negative one negates q instead,
  // and zero (equal weights) becomes a scale too small to change any weight.
  d.q_sign = scale < 0.f ? 0x80008000u : 0u;
  d.scale_log2 = std::max(std::fabs(scale) * 1.4426950408889634f, 1e-30f);
  d.wait_limit_ns = p->wait_limit_ns;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = p->dtype == KV_FP8_E4M3   ? pkv::launch_prefill_fp8(p, d, max_q_len, s)
                        : p->dtype == KV_FP4_E2M1 ? pkv::launch_prefill_fp4(p, d, max_q_len, s)
                                                  : pkv::launch_prefill(p, d, max_q_len, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return KV_OK;
}

kv_status kv_pool_set_partition_blocks(kv_pool* p, int32_t blocks_per_partition) {
  if (!p) return KV_ERR_INVALID_ARG;
  if (blocks_per_partition != 0 &&
      (blocks_per_partition < 4 || blocks_per_partition > 1024 || blocks_per_partition % 4 != 0))
    return KV_ERR_INVALID_ARG;
  p->partition_blocks = blocks_per_partition;
  return KV_OK;
}

kv_status kv_pool_set_timing_events(kv_pool* p, void* start_event, void* stop_event) {
  if (!p || (!start_event) != (!stop_event)) return KV_ERR_INVALID_ARG;
  p->ev_start = static_cast<cudaEvent_t>(start_event);
  p->ev_stop = static_cast<cudaEvent_t>(stop_event);
  return KV_OK;
}

kv_status kv_pool_set_wait_limit(kv_pool* p, uint64_t limit_ns) {
  if (!p || limit_ns < 100000ull || limit_ns > 10000000000ull) return KV_ERR_INVALID_ARG;
  p->wait_limit_ns = limit_ns;
  return KV_OK;
}

kv_status kv_pool_set_test_stall(kv_pool* p, int32_t enable) {
  if (!p) return KV_ERR_INVALID_ARG;
  p->stall_tx = enable ? 16u : 0u;
  return KV_OK;
}

kv_status kv_pool_check_status(kv_pool* p, void* stream) {
  if (!p) return KV_ERR_INVALID_ARG;
  DeviceGuard guard(p->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, p->err, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemsetAsync(p->err, 0, sizeof word, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  if (word & pkv::kErrDrainTimeout) return KV_ERR_DRAIN_TIMEOUT;
  if (word & pkv::kErrTimeout) return KV_ERR_TIMEOUT;
  if (word & pkv::kErrBadBlock) return KV_ERR_BAD_BLOCK_ID;
  if (word & pkv::kErrBadSlot) return KV_ERR_BAD_SLOT;
  if (word & pkv::kErrBadContext) return KV_ERR_BAD_CONTEXT;
  if (word & pkv::kErrStaleMap) return KV_ERR_STALE_EXPONENT_MAP;
  return KV_OK;
}

}  // extern "C"
