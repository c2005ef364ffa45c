// Batched whole-block copy inside one pool, for copy-on-write.
//
// "Optimizing KV Cache Memory Management in vLLM with PagedAttention and
// Dynamic Block Allocation", section "Copy-on-Write (CoW) for Parallel
// Sampling and Prefix Caching": before a sequence writes into a block it
// shares, the block's K/V states are copied device to device into a fresh
// block that the sequence then owns.
//
// A physical block is one contiguous run of the pool ([Hkv][2][BS][D], or
// [Hkv][BS/16] FP4 records), so a copy is a flat move of block_bytes (plus,
// for bf16 pools, its Hkv x BS bytes of the V exponent map).  The (src, dst) pairs come from the
// host block manager; the host cuts them into waves in which no block is
// both read and written, so every wave runs fully parallel and the result is
// that of applying the pairs one after another.  Each wave's pairs travel in
// the kernel's parameter space (no device staging buffer, no extra copy).
// HBM-bound: 2 * block_bytes per pair (read + write), 16-byte vector accesses,
// four loads in flight per thread before the stores.

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;                       // 16-byte chunks per thread
constexpr int kChunksPerCta = kCopyThreads * kCopyUnroll;
constexpr int kMaxWave = 2048;                       // pairs per launch (16 KB of parameters)

struct CopyWave {
  int2 pairs[kMaxWave];  // (src, dst) block ids, validated on the host
};

__global__ void __launch_bounds__(kCopyThreads) kv_copy_blocks_kernel(
    const __grid_constant__ CopyWave wave, int slices, int64_t chunks_per_block,
    uint4* __restrict__ pool, uint4* __restrict__ map, int map_chunks) {
  const int pair = blockIdx.x / slices;
  const int slice = blockIdx.x - pair * slices;
  const int2 pr = wave.pairs[pair];
  // bf16 pools: the block's rows of the V exponent map move with it
  if (slice == 0)
    for (int m = threadIdx.x; m < map_chunks; m += kCopyThreads)
      map[static_cast<int64_t>(pr.y) * map_chunks + m] = map[static_cast<int64_t>(pr.x) * map_chunks + m];
  const uint4* src = pool + static_cast<int64_t>(pr.x) * chunks_per_block;
  uint4* dst = pool + static_cast<int64_t>(pr.y) * chunks_per_block;
  const int64_t base = static_cast<int64_t>(slice) * kChunksPerCta + threadIdx.x;
  uint4 v[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t c = base + u * kCopyThreads;
    if (c < chunks_per_block) v[u] = src[c];
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t c = base + u * kCopyThreads;
    if (c < chunks_per_block) dst[c] = v[u];
  }
}

}  // namespace

int64_t block_bytes(const kv_pool* pool) {
  if (pool->dtype == KV_FP4_E2M1)
    return static_cast<int64_t>(pool->n_kv_heads) * (pool->block_size / 16) * kFp4SubBytes;
  const int64_t elem = pool->dtype == KV_BF16 ? 2 : 1;
  return static_cast<int64_t>(pool->n_kv_heads) * 2 * pool->block_size * pool->head_dim * elem;
}

cudaError_t launch_copy_blocks(const kv_pool* pool, const int32_t* pairs, int64_t n,
                               cudaStream_t stream) {
  const int64_t chunks = block_bytes(pool) / 16;
  // exponent-map bytes per block: Hkv x block_size, a multiple of 16
  const int map_chunks = pool->vexp ? pool->n_kv_heads * pool->block_size / 16 : 0;
  const int slices = static_cast<int>((chunks + kChunksPerCta - 1) / kChunksPerCta);
  static thread_local CopyWave wave;
  int count = 0;
  // Blocks read / written by the pairs of the current wave: a block is in
  // the set when its stamp equals the wave's number (no clearing per wave).
  static thread_local std::vector<uint32_t> read_stamp, write_stamp;
  static thread_local uint32_t wave_id = 0;
  if (read_stamp.size() < static_cast<size_t>(pool->num_blocks)) {
    read_stamp.assign(pool->num_blocks, 0u);
    write_stamp.assign(pool->num_blocks, 0u);
    wave_id = 0;
  }
  auto next_wave = [&]() {
    if (++wave_id == 0) {  // wrapped: forget every stamp
      std::fill(read_stamp.begin(), read_stamp.end(), 0u);
      std::fill(write_stamp.begin(), write_stamp.end(), 0u);
      wave_id = 1;
    }
  };
  next_wave();
  auto flush = [&]() -> cudaError_t {
    if (count == 0) return cudaSuccess;
    kv_copy_blocks_kernel<<<count * slices, kCopyThreads, 0, stream>>>(
        wave, slices, chunks, static_cast<uint4*>(pool->base), reinterpret_cast<uint4*>(pool->vexp),
        map_chunks);
    count = 0;
    next_wave();
    return cudaGetLastError();
  };
  for (int64_t i = 0; i < n; ++i) {
    const int32_t s = pairs[2 * i], d = pairs[2 * i + 1];
    if (s == d) continue;
    // A pair that reads a block this wave writes, or writes a block this
    // wave reads or writes, must see the wave's result: start a new wave.
    if (count == kMaxWave || write_stamp[s] == wave_id || write_stamp[d] == wave_id ||
        read_stamp[d] == wave_id) {
      const cudaError_t e = flush();
      if (e != cudaSuccess) return e;
    }
    wave.pairs[count++] = make_int2(s, d);
    read_stamp[s] = wave_id;
    write_stamp[d] = wave_id;
  }
  return flush();
}

}  // namespace pkv
