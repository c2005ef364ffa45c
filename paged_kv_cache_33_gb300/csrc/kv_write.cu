// Paged KV write: scatter each new token's K and V rows into its slot.
//
// "Optimizing KV Cache Memory Management in vLLM with PagedAttention and
// Dynamic Block Allocation", sections "The Prefill Phase" and "The Decode
// Phase": the kernel writes the computed key/value states into the physical
// blocks; in decode the new token goes to the free slot of the last block.
// Slot s names physical block s / block_size and offset s mod block_size
// (section "PagedAttention: Virtual Memory for LLMs").
//
// Pool layout: [num_blocks][Hkv][2][block_size][D], D contiguous (FP8 pools
// keep each V tile transposed, in [D][16] sub-tiles; FP4 pools hold one
// packed record per 16-token sub-tile, see fp4_*_offset).  For bf16 and FP8
// one thread moves 16 bytes of destination; consecutive threads cover one
// destination row, so every store is a full, coalesced 16-byte vector.

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

// In the fused decode step this kernel is launched as a programmatic dependent
// of the kernel before it on the stream (the previous step's reduce, in a loop
// of steps): it may be scheduled while that kernel runs, and waits for it to
// complete -- and its results to be visible -- before it reads its inputs or
// writes anything.  The early launch hides the launch latency; the wait keeps
// every input (k, v, slots, produced by any earlier kernel) and the previous
// decode's partials safe.  Outside such a launch the wait returns at once.
__device__ __forceinline__ void wait_for_prerequisites() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lane-wise maximum of two pairs of unsigned 16-bit halves.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The largest exponent field of a bf16 row held 16 bytes per thread by
// kChunks consecutive lanes (all in `lanes`), at least 1 (0 marks a row the
// exponent map has no entry for).
template <int kChunks>
__device__ __forceinline__ uint32_t row_exponent(const uint4 val, uint32_t lanes) {
  constexpr uint32_t kE = 0x7F807F80u;
  uint32_t m = max_u16x2(max_u16x2(val.x & kE, val.y & kE), max_u16x2(val.z & kE, val.w & kE));
  m = max(m & 0xFFFFu, m >> 16) >> 7;
#pragma unroll
  for (int o = 1; o < kChunks; o <<= 1) m = max(m, __shfl_xor_sync(lanes, m, o));
  return max(m, 1u);
}

// BF16 pool: bit copy.  Thread i handles chunk c of row (t, h, kv).  The
// threads of a V row also record the row's largest exponent field in the
// pool's exponent map (at least 1: 0 stands for a row never written here),
// which the prefill reads to scale its f16 copy of V.
template <int D>
__global__ void __launch_bounds__(256) kv_write_bf16_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
    int64_t num_tokens, int hkv, int bs, int64_t num_slots, uint4* __restrict__ pool,
    uint8_t* __restrict__ vexp, uint32_t* __restrict__ err, int32_t* __restrict__ zero_word) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  // Once the kernels before this one are complete, a decode launched as this
  // kernel's programmatic dependent may start (it reads its inputs at once,
  // and waits for this grid to complete before it reads the pool).
  wait_for_prerequisites();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (zero_word && blockIdx.x == 0 && threadIdx.x == 0) *zero_word = 0;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = num_tokens * hkv * 2 * kChunks;
  if (i >= total) return;
  const int c = static_cast<int>(i % kChunks);
  int64_t rest = i / kChunks;
  const int kv = static_cast<int>(rest % 2);
  rest /= 2;
  const int h = static_cast<int>(rest % hkv);
  const int64_t t = rest / hkv;
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= num_slots) {
    if (c == 0 && kv == 0 && h == 0) atomicOr(err, kErrBadSlot);
    return;
  }
  const int64_t blk = s / bs;
  const int off = static_cast<int>(s % bs);
  const uint4 val = (kv ? v : k)[(t * hkv + h) * kChunks + c];
  const int64_t row = ((blk * hkv + h) * 2 + kv) * bs + off;
  pool[row * kChunks + c] = val;
  if (kv && vexp) {
    // the kChunks threads of the row are consecutive lanes, all present
    const uint32_t m = row_exponent<kChunks>(val, __activemask());
    if (c == 0) vexp[(blk * hkv + h) * bs + off] = static_cast<uint8_t>(m);
  }
}

// bf16 pools: every V row's exponent-map entry again, from the pool itself
// (after V was written other than through paged_kv_write).  Thread i reads
// chunk c of V row r = i / kChunks of the pool.
template <int D>
__global__ void __launch_bounds__(256) refresh_exponent_map_kernel(const uint4* __restrict__ pool,
                                                                   int64_t rows, int bs,
                                                                   uint8_t* __restrict__ vexp) {
  constexpr int kChunks = D / 8;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * kChunks) return;
  const int64_t r = i / kChunks;  // (block, head) * bs + offset
  const int c = static_cast<int>(i % kChunks);
  const int64_t bh = r / bs;
  const int off = static_cast<int>(r % bs);
  const uint4 val = pool[((bh * 2 + 1) * bs + off) * kChunks + c];
  const uint32_t m = row_exponent<kChunks>(val, __activemask());
  if (c == 0) vexp[r] = static_cast<uint8_t>(m);
}

// Byte position of token `off` (0..15) inside a row of a transposed FP8 V
// sub-tile: tokens 2t, 2t+1, 2t+8, 2t+9 sit at codes 4t..4t+3, the order in
// which the decode kernel's probabilities arrive after their transpose.
__device__ __forceinline__ int vt_slot(int off) {
  return 4 * ((off & 7) >> 1) + (off & 1) + 2 * (off >> 3);
}

// FP8 pool: code = E4M3(float(x) / scale[h]) with round-to-nearest-even and
// saturation to +-448 (the cvt.rn.satfinite conversion).  Thread i makes 16
// codes from 16 bf16 inputs: one 16-byte store into a K row, or 16 byte
// stores down one column of the transposed V tile ([D][16] codes).
template <int D>
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
    int64_t num_tokens, int hkv, int bs, int64_t num_slots, const float* __restrict__ scales,
    uint4* __restrict__ pool, uint32_t* __restrict__ err, int32_t* __restrict__ zero_word) {
  constexpr int kChunks = D / 16;  // 16-code chunks per row
  wait_for_prerequisites();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (zero_word && blockIdx.x == 0 && threadIdx.x == 0) *zero_word = 0;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = num_tokens * hkv * 2 * kChunks;
  if (i >= total) return;
  const int c = static_cast<int>(i % kChunks);
  int64_t rest = i / kChunks;
  const int kv = static_cast<int>(rest % 2);
  rest /= 2;
  const int h = static_cast<int>(rest % hkv);
  const int64_t t = rest / hkv;
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= num_slots) {
    if (c == 0 && kv == 0 && h == 0) atomicOr(err, kErrBadSlot);
    return;
  }
  const float sc = scales[kv * hkv + h];
  const uint4* src = (kv ? v : k) + ((t * hkv + h) * D) / 8 + 2 * c;
  const uint4 x0 = src[0], x1 = src[1];
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  uint32_t packed[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t pair = w[2 * q + e];
      const float a = __fdiv_rn(bf16_lo(pair), sc);
      const float b = __fdiv_rn(bf16_hi(pair), sc);
      const __nv_fp8x2_storage_t two =
          __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
      word |= static_cast<uint32_t>(two) << (16 * e);
    }
    packed[q] = word;
  }
  const int64_t blk = s / bs;
  const int off = static_cast<int>(s % bs);
  const int64_t tile = (blk * hkv + h) * 2 + kv;  // K or V tile of (block, head)
  if (kv == 0) {
    pool[(tile * bs + off) * kChunks + c] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  } else {
    // sub-tile off / 16 of the transposed V tile: [D][16] codes
    uint8_t* vt = reinterpret_cast<uint8_t*>(pool) + tile * bs * D + (off >> 4) * 16 * D;
    const int col = vt_slot(off & 15);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      vt[(16 * c + i) * 16 + col] = static_cast<uint8_t>(packed[i >> 2] >> (8 * (i & 3)));
  }
}

// E2M1 code of q (low four bits S.EE.M): round to nearest, ties to the even
// code, saturating at +-6; NaN stores +0.  The representable magnitudes are
// 0, 0.5, 1, 1.5, 2, 3, 4, 6: the code counts the decision points below |q|,
// a tie going to the even neighbour (>= where the upper code is even).
__device__ __forceinline__ uint32_t e2m1_code(float q) {
  if (isnan(q)) return 0u;
  const float a = fabsf(q);
  const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.0f);
  return m | (signbit(q) ? 8u : 0u);
}

// FP4 pool: E2M1 codes with one E4M3 scale per 16 elements of a row, under the
// per-KV-head fp32 scale G (NVIDIA's NVFP4 arrangement):
//   sc = E4M3(amax / (6 G)), S = value(sc) * G, code = E2M1(x / S) (+0 if S = 0),
// every step one binary32 operation rounded to nearest even.  One warp per
// (token, KV head, K or V) row of 128 elements; lane l holds elements
// 4l .. 4l+3, so the four lanes of a 16-element group agree on its maximum
// with two shuffles.  The row goes to the decode layout of its 16-token
// sub-tile record (fp4_*_offset): K codes as bytes of two consecutive
// dimensions, V codes as bytes of two consecutive tokens, which a warp of
// this kernel shares with its neighbour token, so V nibbles are merged into
// their word with atomic AND / OR.
__global__ void __launch_bounds__(256) kv_write_fp4_kernel(
    const uint2* __restrict__ k, const uint2* __restrict__ v, const int64_t* __restrict__ slots,
    int64_t num_tokens, int hkv, int bs, int64_t num_slots, const float* __restrict__ scales,
    uint8_t* __restrict__ pool, uint32_t* __restrict__ err, int32_t* __restrict__ zero_word) {
  constexpr int D = 128;
  wait_for_prerequisites();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (zero_word && blockIdx.x == 0 && threadIdx.x == 0) *zero_word = 0;
  const int lane = threadIdx.x & 31;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= num_tokens * hkv * 2) return;
  const int kv = static_cast<int>(row & 1);
  const int h = static_cast<int>((row >> 1) % hkv);
  const int64_t t = (row >> 1) / hkv;
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= num_slots) {
    if (lane == 0 && kv == 0 && h == 0) atomicOr(err, kErrBadSlot);
    return;
  }
  const float G = scales[kv * hkv + h];
  const uint2 raw = (kv ? v : k)[((t * hkv + h) * D) / 4 + lane];
  const float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(x[i]));  // fmaxf drops a NaN operand
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const float r = __fdiv_rn(amax, __fmul_rn(6.0f, G));
  const uint32_t sc = static_cast<uint32_t>(__nv_cvt_float_to_fp8(r, __NV_SATFINITE, __NV_E4M3));
  const float S = __fmul_rn(__half2float(__ushort_as_half(
                                static_cast<unsigned short>(e4m3x2_to_f16x2(sc) & 0xFFFFu))),
                            G);
  uint32_t code[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) code[i] = S == 0.f ? 0u : e2m1_code(__fdiv_rn(x[i], S));

  const int64_t blk = s / bs;
  const int off = static_cast<int>(s % bs);
  uint8_t* rec = pool + ((blk * hkv + h) * (bs / 16) + off / 16) * kFp4SubBytes;
  const int r16 = off & 15;  // token row inside the 16-token sub-tile
  const int d0 = 4 * lane;
  if (kv == 0) {
    rec[fp4_k_code_offset(r16, d0)] = static_cast<uint8_t>(code[0] | (code[1] << 4));
    rec[fp4_k_code_offset(r16, d0 + 2)] = static_cast<uint8_t>(code[2] | (code[3] << 4));
    if ((lane & 3) == 0) rec[fp4_k_scale_offset(r16, d0 / 16)] = static_cast<uint8_t>(sc);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int o = fp4_v_code_offset(r16, d0 + i);  // byte of tokens (r16 & ~1, r16 | 1)
      uint32_t* word = reinterpret_cast<uint32_t*>(rec + (o & ~3));
      const int shift = 8 * (o & 3) + 4 * (r16 & 1);
      atomicAnd(word, ~(0xFu << shift));
      atomicOr(word, code[i] << shift);
    }
    if ((lane & 3) == 0) rec[fp4_v_scale_offset(r16, d0 / 16)] = static_cast<uint8_t>(sc);
  }
}

}  // namespace

// The fused step's write (the one that clears the decode's counters) is
// launched as a programmatic dependent of whatever kernel precedes it on the
// stream; the kernels wait for their prerequisites before they do anything.
template <typename Kernel, typename... Args>
cudaError_t launch_write(Kernel kernel, int64_t blocks, cudaStream_t stream, bool dependent,
                         Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_refresh_exponent_map(const kv_pool* pool, cudaStream_t stream) {
  const int64_t rows = pool->num_blocks * pool->n_kv_heads * pool->block_size;
  const int64_t total = rows * (pool->head_dim / 8);
  const int64_t blocks = (total + 255) / 256;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (pool->head_dim == 128)
    refresh_exponent_map_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(pool->base), rows, pool->block_size, pool->vexp);
  else
    refresh_exponent_map_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(pool->base), rows, pool->block_size, pool->vexp);
  return cudaGetLastError();
}

cudaError_t launch_kv_write(const kv_pool* pool, const void* k, const void* v,
                            const int64_t* slots, int64_t num_tokens, cudaStream_t stream,
                            int32_t* zero_word) {
  const int hkv = pool->n_kv_heads;
  const int64_t num_slots = pool->num_blocks * pool->block_size;
  const int threads = 256;
  const bool dependent = zero_word != nullptr;
  if (pool->dtype == KV_BF16) {
    const int64_t total = num_tokens * hkv * 2 * (pool->head_dim / 8);
    const int64_t blocks = std::max<int64_t>(1, (total + threads - 1) / threads);
    if (pool->head_dim == 128)
      return launch_write(kv_write_bf16_kernel<128>, blocks, stream, dependent,
                          static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
                          num_tokens, hkv, pool->block_size, num_slots,
                          static_cast<uint4*>(pool->base), pool->vexp, pool->err, zero_word);
    return launch_write(kv_write_bf16_kernel<64>, blocks, stream, dependent,
                        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
                        num_tokens, hkv, pool->block_size, num_slots,
                        static_cast<uint4*>(pool->base), pool->vexp, pool->err, zero_word);
  }
  if (pool->dtype == KV_FP4_E2M1) {
    const int64_t total = num_tokens * hkv * 2 * 32;  // one warp per row
    const int64_t blocks = std::max<int64_t>(1, (total + threads - 1) / threads);
    return launch_write(kv_write_fp4_kernel, blocks, stream, dependent,
                        static_cast<const uint2*>(k), static_cast<const uint2*>(v), slots,
                        num_tokens, hkv, pool->block_size, num_slots,
                        static_cast<const float*>(pool->scales), static_cast<uint8_t*>(pool->base),
                        pool->err, zero_word);
  }
  const int64_t total = num_tokens * hkv * 2 * (pool->head_dim / 16);
  const int64_t blocks = std::max<int64_t>(1, (total + threads - 1) / threads);
  return launch_write(kv_write_fp8_kernel<128>, blocks, stream, dependent,
                      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
                      num_tokens, hkv, pool->block_size, num_slots,
                      static_cast<const float*>(pool->scales), static_cast<uint4*>(pool->base),
                      pool->err, zero_word);
}

}  // namespace pkv
