// Split-K paged decode attention for sm_103a, and its reduce.
//
// What it computes ("Optimizing KV Cache Memory Management in vLLM with
// PagedAttention and Dynamic Block Allocation", section "PagedAttention:
// Virtual Memory for LLMs"; GQA from "The Math of the KV Cache Bottleneck";
// the window rule from "How the block pool manages KV memory", "Hybrid models
// get groups"): for sequence b and query head hq of KV head h,
//     out[b, hq] = sum_t softmax_t(scale * q . K_t) V_t,  t in [lo, ctx),
// where token t is found in physical block table[b][t / 16] at offset t % 16.
//
// How (GB300 design):
//  * Grid (partition, KV head, sequence).  A partition is a run of
//    `part_blocks` consecutive logical blocks; one CTA per (b, h, partition)
//    reads each K/V block once for all g = Hq/Hkv query heads of the group.
//  * Every warp walks its own share of the partition's blocks (block i goes to
//    warp i mod NW) through a private ring of STAGES shared-memory stages.
//    Lane 0 resolves the physical block from the table and issues one TMA
//    tensor copy per (block, head) (two for bf16 with head_dim 128), landing
//    the K tile and the V tile with the 128-byte swizzle so that every
//    ldmatrix below is bank-conflict free.  Completion is an mbarrier with a
//    transaction count; every wait is bounded in wall time.
//  * Scores S^T[16 tokens x 8 heads] = K Q^T on the tensor cores
//    (mma.sync m16n8k16, fp32 accumulate), the online softmax in the exp2
//    domain with warp shuffles over the token rows, and O^T[D x 8 heads] +=
//    V^T P^T again on the tensor cores.  P^T is formed from the score
//    accumulator by movmatrix.  For bf16 KV, P is split into a bf16 high part
//    and a bf16 remainder so the product keeps ~16 bits of P; for FP8 KV,
//    K and V are widened exactly from E4M3 to f16 and P is f16.
//  * Masking uses selects: scores of positions outside [lo, ctx) become -inf
//    and their V rows are zeroed before the product, so stale or NaN slots
//    of a partly filled block never reach the result.
//  * The warps of a CTA merge their (max, sum, O) in shared memory; a
//    sequence with one partition writes its output directly, otherwise the
//    partition's unnormalised partial goes to the workspace and the reduce
//    kernel combines the partitions.

#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr uint64_t kShortWaitNs = 200000;  // wait bound once some warp has timed out

struct SeqRange {
  int32_t lo, ctx, first_blk, nblk;
  bool bad;
};

// Attended positions [lo, ctx) of sequence b and the blocks that hold them.
__device__ __forceinline__ SeqRange seq_range(const DecodeParams& p, int b) {
  int32_t ctx = p.context_lens[b];
  const bool bad = ctx < 0 || ctx > p.max_ctx || ctx > p.mbs * kBlockSize;
  if (bad) ctx = 0;
  SeqRange r;
  r.ctx = ctx;
  r.bad = bad;
  r.lo = p.window > 0 ? max(0, ctx - p.window) : 0;
  r.first_blk = r.lo / kBlockSize;
  r.nblk = ctx > r.lo ? (ctx - 1) / kBlockSize - r.first_blk + 1 : 0;
  return r;
}

template <int D, bool FP8>
struct Geometry {
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kRowBytes = 128;                  // one swizzled smem row
  static constexpr int kBoxes = FP8 ? 1 : D / 64;        // TMA boxes per (block, head)
  static constexpr int kBoxBytes = 2 * kBlockSize * kRowBytes;  // K rows, then V rows
  static constexpr int kStageBytes = kBoxes * kBoxBytes;
  static constexpr int kSteps = D / 16;                  // mma k-steps (QK) = m-tiles (PV)
  static_assert(kStageBytes == 2 * kBlockSize * D * kElem, "stage holds one K and one V tile");
  static_assert(!FP8 || D == 128, "FP8 rows are one 128-byte swizzle row");
};

template <int D, bool FP8, int NW, int STAGES>
constexpr int decode_smem_bytes() {
  return NW * STAGES * Geometry<D, FP8>::kStageBytes + NW * STAGES * 8 + 1024;
}

template <int D, bool FP8, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32) paged_decode_kernel(const __grid_constant__ CUtensorMap tmap,
                                                               const DecodeParams p) {
  using G = Geometry<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the stage buffers keeps the 128-byte swizzle
  // pattern equal to (row mod 8).
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int part = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const SeqRange r = seq_range(p, b);
  if (r.bad && part == 0 && threadIdx.x == 0) atomicOr(p.err, kErrBadContext);
  const int nparts = (r.nblk + p.part_blocks - 1) / p.part_blocks;
  if (part >= max(nparts, 1)) return;  // uniform over the CTA

  const int g = p.group;
  const int64_t row0 = static_cast<int64_t>(b) * p.n_q_heads + static_cast<int64_t>(h) * g;
  if (r.nblk == 0) {  // nothing to attend to: zeros
    for (int i = threadIdx.x; i < g * D; i += NW * 32) p.out[row0 * D + i] = 0.f;
    return;
  }
  const int blk_begin = r.first_blk + part * p.part_blocks;
  const int blk_end = min(blk_begin + p.part_blocks, r.first_blk + r.nblk);
  const int my_first = blk_begin + warp;
  const int my_n = my_first < blk_end ? (blk_end - my_first + NW - 1) / NW : 0;

  uint8_t* ring = smem + warp * STAGES * G::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * STAGES * G::kStageBytes) + warp * STAGES;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int32_t* table = p.block_tables + static_cast<int64_t>(b) * p.mbs;

  // Lane 0: stage logical block (my_first + it * NW) into ring slot it % STAGES.
  auto issue = [&](int it) {
    const int lb = my_first + it * NW;
    int phys = table[lb];
    if (phys < 0 || phys >= p.num_blocks) {
      atomicOr(p.err, kErrBadBlock);
      phys = 0;  // a valid address; every position of this block is masked below
    }
    const int s = it % STAGES;
    const uint32_t bar = smem_addr(&bars[s]);
    const uint32_t dst = smem_addr(ring + s * G::kStageBytes);
    mbar_arrive_expect_tx(bar, G::kStageBytes);
#pragma unroll
    for (int bx = 0; bx < G::kBoxes; ++bx)
      tma_load_4d(dst + bx * G::kBoxBytes, &tmap, bar, bx * 64, 0, 0, phys * p.n_kv_heads + h);
  };
  if (lane == 0) {
    const int pre = min(STAGES, my_n);
    for (int it = 0; it < pre; ++it) issue(it);
  }

  // ---- query fragments: B operand of S^T = K Q^T (k = head_dim, n = query head)
  const int n = lane >> 2;  // query head of the group this lane feeds (n < 8)
  const int j = lane & 3;
  uint32_t qf[G::kSteps][2];
  float score_scale = p.scale_log2;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + row0 * D;
  if constexpr (!FP8) {
    const uint32_t* qr = reinterpret_cast<const uint32_t*>(qg + n * D);
#pragma unroll
    for (int ks = 0; ks < G::kSteps; ++ks) {
      qf[ks][0] = n < g ? qr[(ks * 16 + 2 * j) >> 1] : 0u;
      qf[ks][1] = n < g ? qr[(ks * 16 + 8 + 2 * j) >> 1] : 0u;
    }
  } else {
    // f16 operands: bring the group's queries into (-1, 1) by an exact power
    // of two and fold that power back into the score scale.
    float amax = 0.f;
    for (int i = lane; i < g * D; i += 32) amax = fmaxf(amax, fabsf(__bfloat162float(qg[i])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    int e = 0;
    if (amax > 0.f) frexpf(amax, &e);
    const float qs = ldexpf(1.f, -e);
    score_scale = p.scale_log2 * p.k_scale[h] * ldexpf(1.f, e);
    // k-slot order matching the widened E4M3 fragments: slots 2j, 2j+1 hold
    // d = 16c + 4j + {0, 1}; slots 2j+8, 2j+9 hold d = 16c + 4j + {2, 3}.
#pragma unroll
    for (int c = 0; c < G::kSteps; ++c) {
      float v4[4] = {0.f, 0.f, 0.f, 0.f};
      if (n < g) {
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) v4[e4] = __bfloat162float(qg[n * D + 16 * c + 4 * j + e4]) * qs;
      }
      qf[c][0] = pack_f16x2(v4[0], v4[1]);
      qf[c][1] = pack_f16x2(v4[2], v4[3]);
    }
  }

  // ---- running state for query heads 2j and 2j+1
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float acc[G::kSteps][4];
#pragma unroll
  for (int i = 0; i < G::kSteps; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  const int trow_k = (lane & 7) + (((lane >> 3) & 1) << 3);  // ldmatrix row for the K operand
  const int swz = lane & 7;                                    // 128B-swizzle phase of that row
  bool timed_out = false;
  int it = 0;
  for (; it < my_n; ++it) {
    const int s = it % STAGES;
    const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), (it / STAGES) & 1, p.wait_limit_ns,
                                      p.err, kErrTimeout, kShortWaitNs);
    if (!__all_sync(kFull, ok)) {
      timed_out = true;
      break;
    }
    const int lb = my_first + it * NW;
    const int phys = table[lb];
    const bool blk_ok = phys >= 0 && phys < p.num_blocks;
    const int t0 = lb * kBlockSize;
    const bool full = blk_ok && t0 >= r.lo && t0 + kBlockSize <= r.ctx;
    auto tok_ok = [&](int tr) {
      const int pos = t0 + tr;
      return full || (blk_ok && pos >= r.lo && pos < r.ctx);
    };
    const uint32_t st = smem_addr(ring + s * G::kStageBytes);

    // ---- S^T = K Q^T : rows = 16 tokens, cols = 8 query heads
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (!FP8) {
#pragma unroll
      for (int ks = 0; ks < G::kSteps; ++ks) {
        const int chunk = ((ks & 3) << 1) + (lane >> 4);
        const uint32_t addr = st + (ks >> 2) * G::kBoxBytes + trow_k * G::kRowBytes +
                              ((chunk ^ swz) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
        if (ks & 1)
          mma_bf16(sb, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
        else
          mma_bf16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
      }
    } else {
#pragma unroll
      for (int cp = 0; cp < G::kSteps; cp += 2) {
        const int chunk = cp + (lane >> 4);
        const uint32_t addr = st + trow_k * G::kRowBytes + ((chunk ^ swz) << 4);
        uint32_t r0, r1, r2, r3;
        ldsm_x4(addr, r0, r1, r2, r3);
        mma_f16(sa, e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                e4m3x2_to_f16x2(r1 >> 16), qf[cp][0], qf[cp][1]);
        mma_f16(sb, e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                e4m3x2_to_f16x2(r3 >> 16), qf[cp + 1][0], qf[cp + 1][1]);
      }
    }

    // ---- online softmax (log2 domain); this lane holds tokens n, n+8 of heads 2j, 2j+1
    const bool v0 = tok_ok(n), v1 = tok_ok(n + 8);
    const float s0 = v0 ? (sa[0] + sb[0]) * score_scale : -INFINITY;
    const float s1 = v0 ? (sa[1] + sb[1]) * score_scale : -INFINITY;
    const float s2 = v1 ? (sa[2] + sb[2]) * score_scale : -INFINITY;
    const float s3 = v1 ? (sa[3] + sb[3]) * score_scale : -INFINITY;
    float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, o));
      bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, o));
    }
    const float mn0 = fmaxf(m_run[0], bm0), mn1 = fmaxf(m_run[1], bm1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(m_run[0] - mu0), al1 = fast_exp2(m_run[1] - mu1);
    const float p0 = fast_exp2(s0 - mu0), p1 = fast_exp2(s1 - mu1);
    const float p2 = fast_exp2(s2 - mu0), p3 = fast_exp2(s3 - mu1);
    l_run[0] = l_run[0] * al0 + p0 + p2;
    l_run[1] = l_run[1] * al1 + p1 + p3;
    m_run[0] = mn0;
    m_run[1] = mn1;
#pragma unroll
    for (int i = 0; i < G::kSteps; ++i) {
      acc[i][0] *= al0;
      acc[i][1] *= al1;
      acc[i][2] *= al0;
      acc[i][3] *= al1;
    }

    // ---- O^T += V^T P^T : rows = head_dim, cols = 8 query heads, k = 16 tokens
    if constexpr (!FP8) {
      const uint32_t x01 = pack_bf16x2(p0, p1), x23 = pack_bf16x2(p2, p3);
      const uint32_t y01 = pack_bf16x2(p0 - bf16_lo(x01), p1 - bf16_hi(x01));
      const uint32_t y23 = pack_bf16x2(p2 - bf16_lo(x23), p3 - bf16_hi(x23));
      const uint32_t bh0 = movmatrix_trans(x01), bh1 = movmatrix_trans(x23);
      const uint32_t bl0 = movmatrix_trans(y01), bl1 = movmatrix_trans(y23);
      // this lane's V^T fragment covers tokens 2j, 2j+1 (a0, a1) and 2j+8, 2j+9 (a2, a3)
      uint32_t mlo = kFull, mhi = kFull;
      if (!full) {
        mlo = (tok_ok(2 * j) ? 0x0000ffffu : 0u) | (tok_ok(2 * j + 1) ? 0xffff0000u : 0u);
        mhi = (tok_ok(2 * j + 8) ? 0x0000ffffu : 0u) | (tok_ok(2 * j + 9) ? 0xffff0000u : 0u);
      }
      const int trow_v = kBlockSize + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
      for (int mt = 0; mt < G::kSteps; ++mt) {
        const int chunk = ((mt & 3) << 1) + ((lane >> 3) & 1);
        const uint32_t addr = st + (mt >> 2) * G::kBoxBytes + trow_v * G::kRowBytes +
                              ((chunk ^ swz) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(addr, a0, a1, a2, a3);
        a0 &= mlo;
        a1 &= mlo;
        a2 &= mhi;
        a3 &= mhi;
        mma_bf16(acc[mt], a0, a1, a2, a3, bh0, bh1);
        mma_bf16(acc[mt], a0, a1, a2, a3, bl0, bl1);
      }
    } else {
      const uint32_t b0 = movmatrix_trans(pack_f16x2(p0, p1));
      const uint32_t b1 = movmatrix_trans(pack_f16x2(p2, p3));
#pragma unroll
      for (int cp = 0; cp < G::kSteps; cp += 2) {
        const int chunk = cp + (lane >> 4);
        const uint32_t addr = st + (kBlockSize + trow_k) * G::kRowBytes + ((chunk ^ swz) << 4);
        uint32_t r0, r1, r2, r3;  // V[token n or n+8][16 codes of chunk cp or cp+1]
        ldsm_x4(addr, r0, r1, r2, r3);
        if (!v0) r0 = r2 = 0u;
        if (!v1) r1 = r3 = 0u;
        mma_f16(acc[cp], movmatrix_trans(e4m3x2_to_f16x2(r0)),
                movmatrix_trans(e4m3x2_to_f16x2(r0 >> 16)), movmatrix_trans(e4m3x2_to_f16x2(r1)),
                movmatrix_trans(e4m3x2_to_f16x2(r1 >> 16)), b0, b1);
        mma_f16(acc[cp + 1], movmatrix_trans(e4m3x2_to_f16x2(r2)),
                movmatrix_trans(e4m3x2_to_f16x2(r2 >> 16)), movmatrix_trans(e4m3x2_to_f16x2(r3)),
                movmatrix_trans(e4m3x2_to_f16x2(r3 >> 16)), b0, b1);
      }
    }

    __syncwarp();
    if (lane == 0 && it + STAGES < my_n) {
      fence_proxy_async_smem();  // this stage's reads happen before the next copy lands
      issue(it + STAGES);
    }
  }

  if (timed_out) {
    if (lane == 0) {
      atomicOr(p.err, kErrTimeout);
      const int issued = min(my_n, it + STAGES);
      for (int k = it; k < issued; ++k)
        mbar_wait_bounded(smem_addr(&bars[k % STAGES]), (k / STAGES) & 1, p.wait_limit_ns, p.err,
                          kErrTimeout, kShortWaitNs);
    }
    __syncwarp();
  }

#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l_run[0] += __shfl_xor_sync(kFull, l_run[0], o);
    l_run[1] += __shfl_xor_sync(kFull, l_run[1], o);
  }

  // ---- merge the warps of this CTA in shared memory (the rings are idle now)
  __syncthreads();
  float* mbuf = reinterpret_cast<float*>(smem);  // [NW][8 max | 8 sum]
  float* obuf = mbuf + NW * 16;                   // [NW][8 heads][D]
  if (lane < 4) {
    mbuf[warp * 16 + 2 * lane] = m_run[0];
    mbuf[warp * 16 + 2 * lane + 1] = m_run[1];
    mbuf[warp * 16 + 8 + 2 * lane] = l_run[0];
    mbuf[warp * 16 + 8 + 2 * lane + 1] = l_run[1];
  }
  float* ow = obuf + warp * 8 * D;
#pragma unroll
  for (int i = 0; i < G::kSteps; ++i) {
    int da, db;  // head_dim rows of accumulator entries {0,1} and {2,3}
    if constexpr (!FP8) {
      da = 16 * i + n;
      db = da + 8;
    } else {
      da = 16 * i + 4 * (n >> 1) + (n & 1);
      db = da + 2;
    }
    ow[(2 * j) * D + da] = acc[i][0];
    ow[(2 * j + 1) * D + da] = acc[i][1];
    ow[(2 * j) * D + db] = acc[i][2];
    ow[(2 * j + 1) * D + db] = acc[i][3];
  }
  __syncthreads();

  const bool single = nparts == 1;
  const float vsc = FP8 ? p.v_scale[h] : 1.f;
  for (int idx = threadIdx.x; idx < g * D; idx += NW * 32) {
    const int hd = idx / D;
    const int d = idx - hd * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mbuf[w * 16 + hd]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = fast_exp2(mbuf[w * 16 + hd] - M);
        L += f * mbuf[w * 16 + 8 + hd];
        O += f * obuf[(w * 8 + hd) * D + d];
      }
    }
    O *= vsc;
    if (single) {
      p.out[(row0 + hd) * D + d] = L > 0.f ? O / L : 0.f;
    } else {
      const int64_t pi = (row0 + hd) * p.max_parts + part;
      p.part_o[pi * D + d] = O;
      if (d == 0) {
        p.part_ml[2 * pi] = M;
        p.part_ml[2 * pi + 1] = L;
      }
    }
  }
}

// Combine the partitions of one (sequence, query head):
//   out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p.
template <int D>
__global__ void __launch_bounds__(D) paged_decode_reduce_kernel(const DecodeParams p) {
  const int hq = blockIdx.x;
  const int b = blockIdx.y;
  const SeqRange r = seq_range(p, b);
  const int np = (r.nblk + p.part_blocks - 1) / p.part_blocks;
  if (np <= 1) return;  // the decode kernel wrote this row itself
  const int64_t base = (static_cast<int64_t>(b) * p.n_q_heads + hq) * p.max_parts;
  const float* ml = p.part_ml + 2 * base;
  float M = -INFINITY;
  for (int i = 0; i < np; ++i) M = fmaxf(M, ml[2 * i]);
  float L = 0.f, O = 0.f;
  const int d = threadIdx.x;
  if (M != -INFINITY) {
    for (int i = 0; i < np; ++i) {
      const float f = fast_exp2(ml[2 * i] - M);
      L += f * ml[2 * i + 1];
      O += f * p.part_o[(base + i) * D + d];
    }
  }
  p.out[(static_cast<int64_t>(b) * p.n_q_heads + hq) * D + d] = L > 0.f ? O / L : 0.f;
}

template <int D, bool FP8, int NW, int STAGES>
cudaError_t launch_variant(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = decode_smem_bytes<D, FP8, NW, STAGES>();
  auto kernel = paged_decode_kernel<D, FP8, NW, STAGES>;
  static bool attr_set = false;  // per instantiation; setting it again is harmless
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(p.max_parts, p.n_kv_heads, p.batch);
  kernel<<<grid, NW * 32, smem, stream>>>(pool->tmap, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream) {
  if (pool->dtype == KV_FP8_E4M3) return launch_variant<128, true, 4, 4>(pool, p, stream);
  if (pool->head_dim == 128) return launch_variant<128, false, 4, 3>(pool, p, stream);
  return launch_variant<64, false, 4, 4>(pool, p, stream);
}

cudaError_t launch_reduce(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(p.n_q_heads, p.batch);
  if (pool->head_dim == 128)
    paged_decode_reduce_kernel<128><<<grid, 128, 0, stream>>>(p);
  else
    paged_decode_reduce_kernel<64><<<grid, 64, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
