// Paged prefill / extend attention over an FP4 pool (E2M1 codes, one E4M3
// scale per 16 elements of a row, a per-KV-head fp32 scale), on the
// 5th-generation tensor cores with f16 operands.
//
// What it computes is the bf16 prefill's ("Optimizing KV Cache Memory
// Management in vLLM with PagedAttention and Dynamic Block Allocation", "The
// Prefill Phase"; prefix caching from "PagedAttention", "Walking through two
// requests"), every key and value being e2m1 code x E4M3 group scale x the
// KV head's scale: new token i of sequence b sits at position
// pos = ctx - q_len + i and attends causally to [lo, pos], lo = max(0,
// pos + 1 - W) under a window W, keys resolved through the block table;
// query head hq reads KV head hq / g.
//
// How.  The CTA geometry, barriers and the alternation of two 128-row query
// tiles over shared key tiles are those of the bf16 kernel.
//  * An E2M1 value times an E4M3 scale has at most 5 significant bits and
//    lies in [2^-10, 2688], so it is exact in f16: K and V enter the tensor
//    cores as f16 (kind::f16), the head scales applied in fp32.  The query
//    rows are f16 too, each scaled by a power of two that puts its largest
//    magnitude below 2^15 (every bf16 value of the row stays exact), the
//    power folded into the exponent's coefficient with the K head scale.
//  * The pool's records (2304 bytes per 16-token sub-tile: K codes, V codes,
//    K and V group scales, permuted for the decode's fragments) are copied
//    verbatim, one TMA box per block, into a 2-stage ring.  A converter
//    warpgroup turns each key tile into an f16 K tile (thread = key: its 64
//    code bytes are four 16-byte rows whose byte c holds dims 8c + 2i, +1 of
//    row i; 128-byte swizzled, K-major, one stage), and at the same time two
//    more warps turn it into an f16 V tile (thread = two dims: per 16 tokens
//    four code words and four scale words, tokens in natural order; K-major
//    without swizzle, 2 stages), zeros for tokens past the sequence's end and
//    for blocks not loaded.  K feeds the S products, which wait on it, so
//    the converter warpgroup's four warps convert K alone.
//  * S = Q K^T, O += P V with P one f16 per weight (relative rounding
//    2^-11); out = O v_scale / l.
//  * Registers: the two softmax warpgroups take 192 per thread, the others
//    give theirs up to 64.
//  * Every wait is bounded in wall time; on a timeout the CTA records
//    KV_ERR_TIMEOUT, drains what it issued and frees its tensor memory.

#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;           // query rows per tile (M)
constexpr int kTiles = 2;            // query tiles per CTA, alternating over the same keys
constexpr int kKv = 128;             // keys per key tile (N of S, K of P V)
constexpr int kSub = 16;             // tokens per FP4 record
constexpr int kRawStages = 2;        // ring of the records as copied
constexpr int kV16Stages = 2;        // V ring converted (f16 sub-tiles); K has one f16 stage
constexpr int kSoftmax = kTiles * kRows;
constexpr int kRawWarp = kSoftmax / 32, kMmaWarp = kRawWarp + 2;
constexpr int kVCvtWarpA = kRawWarp + 1, kVCvtWarpB = kRawWarp + 3;  // V converters
constexpr int kVCvt = 64;
constexpr int kCvtWarp = kRawWarp + 4;       // K converter warpgroup
constexpr int kCvt = 128;
constexpr int kThreads = kSoftmax + 128 + kCvt;
constexpr int kLaunchRegs = 65536 / kThreads;
constexpr int kSoftmaxRegs = 192, kOtherRegs = 64;
static_assert(2 * kSoftmaxRegs + 2 * kOtherRegs <= 4 * kLaunchRegs,
              "register increases must be covered by the decreases");
constexpr float kLazy = 8.f;         // rescale O when a row maximum grows by more than this (log2)
constexpr uint64_t kShortWaitNs = 200000;

// Shared memory (offsets from a 1024-aligned base).  The f16 V ring sits
// right after Q, so every byte its descriptor can address stays inside the
// allocation.
constexpr int kQTile = 2 * kRows * 128;               // 2 column halves x [128 rows][64] f16
constexpr int kK16 = kKv * kD * 2;                    // 2 column halves x [128 keys][64] f16
constexpr int kV16Stage = kKv * kD * 2;               // 8 sub-tiles x 2 x [128 dims][8 f16]
constexpr int kV16Sub = kSub * kD * 2;                // 4 KB per 16 tokens
constexpr int kRawStage = (kKv / kSub) * kFp4SubBytes;  // 8 records
constexpr int kQ = 0;
constexpr int kV16 = kQ + kTiles * kQTile;
constexpr int kKt = kV16 + kV16Stages * kV16Stage;
constexpr int kRaw = kKt + kK16;
constexpr int kRs = kRaw + kRawStages * kRawStage;     // float [kTiles][kRows]: 2^-(row power)
constexpr int kRawMask = kRs + kTiles * kRows * 4;     // uint32 [kRawStages]: blocks each stage holds
constexpr int kBars = kRawMask + 16;
constexpr int kNumBars = 2 * kRawStages + 2 + 2 * kV16Stages + 4 * kTiles + 2;
constexpr int kTmemSlot = kBars + kNumBars * 8;
constexpr int kSmemBytes = kTmemSlot + 16 + 1024;     // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");
static_assert(kRawStages * 4 <= 16, "the raw stages' block masks fit");
static_assert(kRawStage % 128 == 0 && kRaw % 1024 == 0, "TMA destinations stay 128-byte aligned");
static_assert(kTiles * kRows * 256 <= kTiles * kQTile, "output staging fits in the Q buffers");
// tensor memory per query tile: S [0,128) (P as f16 pairs over columns [0,64)), O [128,256)
constexpr uint32_t kOCol = kKv;
constexpr uint32_t kTmemTile = 256;
constexpr uint32_t kTmemCols = kTiles * kTmemTile;

__device__ __forceinline__ int swz128(int row, int chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// f16 pair word of tokens (2k, 2k+1) with the tokens from `nv` on zeroed.
__device__ __forceinline__ uint32_t keep_tokens(uint32_t w, int k, int nv) {
  return 2 * k + 1 < nv ? w : (2 * k < nv ? (w & 0xFFFFu) : 0u);
}

// a * b on two f16 lanes held as raw bits.
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  return half2_as_u32(__hmul2(u32_as_half2(a), u32_as_half2(b)));
}

// Tiled 3-D tensor copy global -> shared; completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1) paged_prefill_fp4_kernel(
    const __grid_constant__ CUtensorMap tmap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA order as in the bf16 kernel: (sequence, KV head) pairs sixteen at a
  // time, the query tiles with the most keys first inside a group.
  constexpr int kGroupPairs = 16;
  const int pairs = p.n_kv_heads * p.batch;
  const int nx = static_cast<int>(gridDim.x) / pairs;
  const int grp = static_cast<int>(blockIdx.x) / (kGroupPairs * nx);
  const int rb = static_cast<int>(blockIdx.x) - grp * kGroupPairs * nx;
  const int kc = min(kGroupPairs, pairs - grp * kGroupPairs);
  const int qx = nx - 1 - rb / kc;
  const int hb = grp * kGroupPairs + rb % kc;
  const int b = hb / p.n_kv_heads, h = hb - b * p.n_kv_heads;
  const int Gp = p.group_pow2, g = p.group;
  const int log2_gp = __ffs(Gp) - 1;
  const int tpt = kRows / Gp;  // query tokens per tile

  const int32_t q0 = p.cu_q_lens[b];
  const int32_t qn = p.cu_q_lens[b + 1] - q0;
  const int32_t ctx = p.context_lens[b];
  if (qn < 0 || qn > ctx || ctx > p.max_ctx || static_cast<int64_t>(ctx) > static_cast<int64_t>(p.mbs) * BS) {
    if (qn != 0 && qx == 0 && h == 0 && tid == 0) atomicOr(p.err, kErrBadContext);
    return;
  }
  const int tok0 = qx * (kTiles * tpt);
  if (tok0 >= qn) return;
  const int pos_base = ctx - qn;
  const int kv_begin = p.window > 0 ? max(0, pos_base + tok0 + 1 - p.window) : 0;
  const int jt0 = kv_begin / kKv;
  const int ntok0 = min(tpt, qn - tok0), ntok1 = max(0, min(tpt, qn - tok0 - tpt));
  const int last0 = pos_base + tok0 + ntok0 - 1;
  const int last1 = pos_base + tok0 + tpt + ntok1 - 1;
  const int n_kv0 = last0 / kKv - jt0 + 1;
  const int n_kv1 = ntok1 > 0 ? last1 / kKv - jt0 + 1 : 0;
  const int kv_end = (ntok1 > 0 ? last1 : last0) + 1;
  const int n_tiles = max(n_kv0, n_kv1);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBars);
  const uint32_t bar0 = smem_addr(bars);
  auto raw_full = [&](int s) { return bar0 + 8u * s; };
  auto raw_empty = [&](int s) { return bar0 + 8u * (kRawStages + s); };
  const uint32_t k16_full = bar0 + 8u * (2 * kRawStages);
  const uint32_t k16_empty = k16_full + 8;
  constexpr int kB16 = 2 * kRawStages + 2, kBT = kB16 + 2 * kV16Stages;
  auto v16_full = [&](int s) { return bar0 + 8u * (kB16 + s); };
  auto v16_empty = [&](int s) { return bar0 + 8u * (kB16 + kV16Stages + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (kBT + 4 * t); };
  auto p_full = [&](int t) { return bar0 + 8u * (kBT + 4 * t + 1); };
  auto pv_done = [&](int t) { return bar0 + 8u * (kBT + 4 * t + 2); };
  auto o_final = [&](int t) { return bar0 + 8u * (kBT + 4 * t + 3); };
  const uint32_t q_full = bar0 + 8u * (kBT + 4 * kTiles);
  const uint32_t mma_done = q_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlot);
  float* row_rs = reinterpret_cast<float*>(smem + kRs);
  uint32_t* raw_mask = reinterpret_cast<uint32_t*>(smem + kRawMask);

  if (tid == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(raw_full(s), 1);
      mbar_init(raw_empty(s), kCvt + kVCvt);
    }
    mbar_init(k16_full, kCvt);
    mbar_init(k16_empty, 1);
    for (int s = 0; s < kV16Stages; ++s) {
      mbar_init(v16_full(s), kVCvt);
      mbar_init(v16_empty(s), 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), kRows);
      mbar_init(pv_done(t), 1);
      mbar_init(o_final(t), 1);
    }
    mbar_init(q_full, kSoftmax);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto wait = [&](uint32_t bar, uint32_t parity) {
    return mbar_wait_bounded(bar, parity, p.wait_limit_ns, p.err, kErrTimeout, kShortWaitNs);
  };
  const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.mbs;
  auto needed = [&](int jt, int i) {
    const int k0 = (jt0 + jt) * kKv + i * BS;
    return k0 + BS > kv_begin && k0 < kv_end;
  };

  if (warp < kRawWarp) {
    warpgroup_regs_inc<kSoftmaxRegs>();
    // ====== softmax warps: warps 4t..4t+3 serve query tile t, one row per thread
    const int t = warp >> 2;
    const int r = tid & (kRows - 1);
    const int tq = r / Gp, jh = r - tq * Gp;
    const bool row_ok = tq < (t ? ntok1 : ntok0) && jh < g;
    const int tok = tok0 + t * tpt + tq;
    const int pos = pos_base + tok;
    const int lo = p.window > 0 ? max(0, pos + 1 - p.window) : 0;
    // Q of both tiles -> f16 in shared memory, 16 threads per row (one
    // 16-byte chunk of bf16 each), the row's power of two from a maximum
    // over those 16 lanes
    {
      const uint4* qg = static_cast<const uint4*>(p.q);
      constexpr int kChunks = kD / 8;
#pragma unroll 2
      for (int it = 0; it < kTiles * kRows * kChunks / kSoftmax; ++it) {
        const int idx = it * kSoftmax + tid;
        const int row = idx / kChunks, ch = idx % kChunks;
        const int tt = row / kRows, rr = row % kRows;
        const int tq2 = rr >> log2_gp, jh2 = rr & (Gp - 1);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tq2 < (tt ? ntok1 : ntok0) && jh2 < g)
          v = qg[(static_cast<int64_t>(q0 + tok0 + tt * tpt + tq2) * p.n_q_heads + h * g + jh2) *
                     kChunks + ch];
        const uint32_t w[4] = {v.x ^ p.q_sign, v.y ^ p.q_sign, v.z ^ p.q_sign, v.w ^ p.q_sign};
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
#pragma unroll
        for (int o = 1; o < kChunks; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        // amax in [2^e, 2^(e+1)); the row is scaled by 2^(14 - e), below 2^15
        int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
        e = amax > 0.f ? max(-100, min(100, e)) : 0;
        const float qs = __uint_as_float(static_cast<uint32_t>(127 + 14 - e) << 23);
        uint4 hv;
        hv.x = pack_f16x2(bf16_lo(w[0]) * qs, bf16_hi(w[0]) * qs);
        hv.y = pack_f16x2(bf16_lo(w[1]) * qs, bf16_hi(w[1]) * qs);
        hv.z = pack_f16x2(bf16_lo(w[2]) * qs, bf16_hi(w[2]) * qs);
        hv.w = pack_f16x2(bf16_lo(w[3]) * qs, bf16_hi(w[3]) * qs);
        *reinterpret_cast<uint4*>(smem + kQ + tt * kQTile + (ch >> 3) * (kRows * 128) +
                                  swz128(rr, ch & 7)) = hv;
        if (ch == 0) row_rs[tt * kRows + rr] = __uint_as_float(static_cast<uint32_t>(127 - 14 + e) << 23);
      }
      fence_proxy_async_smem();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(q_full) : "memory");
      asm volatile("bar.sync 1, %0;" ::"n"(kSoftmax) : "memory");  // the row powers
    }
    const uint32_t lane_base = tmem + t * kTmemTile + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    // coefficient of the exponent: softmax scale (log2) x k_scale x the row's power
    const float coef = p.scale_log2 * p.k_scale[h] * row_rs[t * kRows + r];
    constexpr uint32_t kAllBlocks = (1u << (kKv / BS)) - 1u;
    float m_raw = -INFINITY, l_run = 0.f;  // running maximum in raw score units
    bool ok = true;
    const int nt = t ? n_kv1 : n_kv0;
    int next[kKv / BS];
    auto fetch = [&](int jt) {
#pragma unroll
      for (int i = 0; i < kKv / BS; ++i)
        next[i] = needed(jt, i) ? trow[((jt0 + jt) * kKv + i * BS) / BS] : -1;
    };
    if (nt > 0) fetch(0);
    for (int jt = 0; jt < nt && ok; ++jt) {
      uint32_t mask = 0;
#pragma unroll
      for (int i = 0; i < kKv / BS; ++i)
        if (next[i] >= 0 && next[i] < p.num_blocks) mask |= 1u << i;
      if (jt + 1 < nt) fetch(jt + 1);
      ok = wait(s_full(t), jt & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const int key0 = (jt0 + jt) * kKv;
      // the row of S, two loads of 64 columns (an instruction may not name
      // more registers than the launch gives a thread) and one wait
      uint32_t x[kKv];
      tmem_ld64_nowait(lane_base, *reinterpret_cast<uint32_t(*)[64]>(&x[0]));
      tmem_ld64_nowait(lane_base + 64, *reinterpret_cast<uint32_t(*)[64]>(&x[64]));
      tmem_wait_ld();
      if (!__all_sync(0xffffffffu, row_ok && key0 >= lo && key0 + kKv - 1 <= pos &&
                                       mask == kAllBlocks)) {
#pragma unroll
        for (int c = 0; c < kKv; ++c) {
          const int key = key0 + c;
          const bool valid = row_ok && key >= lo && key <= pos && ((mask >> (c / BS)) & 1u);
          if (!valid) x[c] = __float_as_uint(-INFINITY);
        }
      }
      float mt4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kKv; ++c) mt4[c & 3] = fmaxf(mt4[c & 3], __uint_as_float(x[c]));
      const float mt_raw = fmaxf(fmaxf(mt4[0], mt4[1]), fmaxf(mt4[2], mt4[3]));
      // The running maximum is kept in raw score units (coef > 0 keeps the
      // order), so the lazy rescale and, for large scores, the exponents come
      // from exact differences of raw scores.
      const bool rescale = m_raw != -INFINITY && mt_raw != -INFINITY && (mt_raw - m_raw) * coef > kLazy;
      const float m_old = m_raw;
      if (m_raw == -INFINITY || rescale) m_raw = mt_raw;
      const float mr = m_raw == -INFINITY ? 0.f : m_raw;
      float mu = mr * coef;
      // The exponent (x - m) coef is at most kLazy (p <= 256), taken as one
      // FMA against m coef.  Once |m coef| reaches 2^13 fp32 holds it only
      // to within 2^-11 (scores of no real model get there): such warps
      // first subtract m from their raw scores, exactly near the maximum,
      // and use no offset.
      if (__any_sync(0xffffffffu, fabsf(mu) >= 0x1p13f)) {
        const float2 nmr2 = make_float2(-mr, -mr);
#pragma unroll
        for (int c = 0; c < kKv; c += 2) {
          const float2 d = fadd2(make_float2(__uint_as_float(x[c]), __uint_as_float(x[c + 1])), nmr2);
          x[c] = __float_as_uint(d.x);
          x[c + 1] = __float_as_uint(d.y);
        }
        mu = 0.f;
      }
      const float2 sc2 = make_float2(coef, coef), nmu2 = make_float2(-mu, -mu);
      // P as f16 pairs over the first 64 columns of S, a quarter of the keys
      // per store
      float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      {
        constexpr int kQuarter = kKv / 8;  // f16 pairs per quarter of the keys
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          uint32_t wp[kQuarter];
#pragma unroll
          for (int i = 0; i < kQuarter; ++i) {
            const int e2 = kq * kQuarter + i;
            const float2 a = ffma2(make_float2(__uint_as_float(x[2 * e2]), __uint_as_float(x[2 * e2 + 1])),
                                   sc2, nmu2);
            const float2 pe = make_float2(fast_exp2(a.x), fast_exp2(a.y));
            l2[i & 1] = fadd2(l2[i & 1], pe);
            wp[i] = pack_f16x2(pe.x, pe.y);
          }
          tmem_st16_nowait(lane_base + kq * kQuarter, wp);
        }
      }
      tmem_wait_st();
      if (__any_sync(0xffffffffu, rescale)) {
        const float alpha = rescale ? fast_exp2((m_old - m_raw) * coef) : 1.f;
        l_run *= alpha;
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + kOCol + c0, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(lane_base + kOCol + c0, o);
        }
      }
      l_run += (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(p_full(t)) : "memory");
    }
    if (ok && nt > 0) ok = __all_sync(0xffffffffu, wait(o_final(t), 0));
    if (ok && nt > 0) {
      tc_fence_after();
      const float inv = l_run > 0.f ? p.v_scale[h] / l_run : 0.f;
      // O v_scale / l -> out through a per-warp staging area in the tile's Q
      // buffer (free once the tile's last product is done), whole rows per store
      uint8_t* stg = smem + kQ + t * kQTile + (warp & 3) * (32 * 256);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + kOCol + hh * 64 + c0, o);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const int ch = (c0 + i) >> 2;
            *reinterpret_cast<float4*>(stg + lane * 256 + ((ch ^ (lane & 15)) << 4)) =
                make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                            __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
          }
        }
        __syncwarp();
#pragma unroll 4
        for (int rr = 0; rr < 32; rr += 2) {
          const int row = rr + (lane >> 4), ch = lane & 15;
          const int r_t = 32 * (warp & 3) + row;
          const int tq2 = r_t >> log2_gp, jh2 = r_t & (Gp - 1);
          if (tq2 < (t ? ntok1 : ntok0) && jh2 < g) {
            const float4 v = *reinterpret_cast<const float4*>(stg + row * 256 + ((ch ^ (row & 15)) << 4));
            *reinterpret_cast<float4*>(
                p.out + (static_cast<int64_t>(q0 + tok0 + t * tpt + tq2) * p.n_q_heads + h * g + jh2) * kD +
                hh * 64 + ch * 4) = v;
          }
        }
        __syncwarp();
      }
    }
  } else if (warp >= kCvtWarp) {
    warpgroup_regs_dec<kOtherRegs>();
    // ====== K converters: from each stage of records, the f16 K tile
    // (thread ct = key ct of the tile)
    const int ct = tid - kCvtWarp * 32;
    bool ok = true;
    for (int jt = 0; jt < n_tiles && ok; ++jt) {
      const int sr = jt % kRawStages;
      ok = wait(raw_full(sr), (jt / kRawStages) & 1);
      if (ok && jt >= 1) ok = wait(k16_empty, (jt - 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const uint32_t mask = raw_mask[sr];  // the blocks the stage holds (from the producer)
      const int key0 = (jt0 + jt) * kKv;
      const uint8_t* raw = smem + kRaw + sr * kRawStage;
      // -- K: key ct, token r of record st
      {
        const int st = ct >> 4, r = ct & 15;
        const bool kvalid = ((mask >> ((kSub * st) / BS)) & 1u) && key0 + ct < ctx;
        uint8_t* krow = smem + kKt;
        if (!kvalid) {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            *reinterpret_cast<uint4*>(krow + (c >> 3) * (kKv * 128) + swz128(ct, c & 7)) =
                make_uint4(0u, 0u, 0u, 0u);
        } else {
          const uint8_t* rec = raw + st * kFp4SubBytes;
          // the token's 64 code bytes: row i (16 bytes), byte c = dims 8c + 2i, 8c + 2i + 1
          const uint4* kc4 = reinterpret_cast<const uint4*>(rec + (r >> 3) * 512 + 64 * (r & 7));
          const uint2 scw = *reinterpret_cast<const uint2*>(rec + 2048 + 8 * r);  // 8 group scales
          uint32_t sg[4];  // f16 pairs of the group scales: groups (2m, 2m+1) in sg[m]
          e4m3x4_to_f16x2(scw.x, sg[0], sg[1]);
          e4m3x4_to_f16x2(scw.y, sg[2], sg[3]);
          const uint4 q[4] = {kc4[0], kc4[1], kc4[2], kc4[3]};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // word k of each row: bytes 4k..4k+3, i.e. chunks c = 4k + m, pair i from row i
            uint32_t f[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t w = k == 0 ? q[i].x : k == 1 ? q[i].y : k == 2 ? q[i].z : q[i].w;
              fp4x8_to_f16x2(w, f[i]);
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int c = 4 * k + m;
              // group c / 2: the low or high half of sg[c / 4], on both lanes
              const uint32_t pair = sg[c >> 2];
              const uint32_t sc = ((c >> 1) & 1) ? __byte_perm(pair, 0, 0x3232) : __byte_perm(pair, 0, 0x1010);
              *reinterpret_cast<uint4*>(krow + (c >> 3) * (kKv * 128) + swz128(ct, c & 7)) =
                  make_uint4(hmul2_bits(f[0][m], sc), hmul2_bits(f[1][m], sc),
                             hmul2_bits(f[2][m], sc), hmul2_bits(f[3][m], sc));
            }
          }
        }
      }
      fence_proxy_async_smem();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(k16_full) : "memory");
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(raw_empty(sr)) : "memory");
    }
  } else {
    warpgroup_regs_dec<kOtherRegs>();
    if (warp == kRawWarp) {
      // ======================= producer: each block's records (K and V codes
      // and scales of its 16-token sub-tiles) by one TMA box, verbatim
      if (lane == 0) {
        int next[kKv / BS];
        auto fetch = [&](int jt) {
#pragma unroll
          for (int i = 0; i < kKv / BS; ++i)
            next[i] = needed(jt, i) ? trow[((jt0 + jt) * kKv + i * BS) / BS] : 0;
        };
        if (n_tiles > 0) fetch(0);
        int issued = 0;
        for (int jt = 0; jt < n_tiles; ++jt) {
          const int s = jt % kRawStages;
          int cur[kKv / BS];
#pragma unroll
          for (int i = 0; i < kKv / BS; ++i) cur[i] = next[i];
          if (jt + 1 < n_tiles) fetch(jt + 1);
          if (jt >= kRawStages && !wait(raw_empty(s), ((jt / kRawStages) - 1) & 1)) break;
          uint32_t mask = 0;
          int phys[kKv / BS];
#pragma unroll
          for (int i = 0; i < kKv / BS; ++i) {
            phys[i] = -1;
            if (!needed(jt, i)) continue;
            const int e = cur[i];
            if (e < 0 || e >= p.num_blocks) {
              atomicOr(p.err, kErrBadBlock);
              continue;
            }
            phys[i] = e;
            mask |= 1u << i;
          }
          const uint32_t bar = raw_full(s);
          const int nblk = __popc(mask);
          raw_mask[s] = mask;  // for the converters (published by the arrive below)
          if (nblk == 0) {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
          } else {
            constexpr int kBlockBytes = (BS / kSub) * kFp4SubBytes;
            mbar_arrive_expect_tx(bar, nblk * kBlockBytes);
            const uint32_t st = smem_addr(smem + kRaw + s * kRawStage);
#pragma unroll
            for (int i = 0; i < kKv / BS; ++i) {
              if (phys[i] < 0) continue;
              const int64_t tile = static_cast<int64_t>(phys[i]) * p.n_kv_heads + h;
              tma_load_3d(st + i * kBlockBytes, &tmap, bar, 0, 0, static_cast<int>(tile));
            }
          }
          ++issued;
        }
        for (int jt = max(0, issued - kRawStages); jt < issued; ++jt)
          if (!wait(raw_full(jt % kRawStages), (jt / kRawStages) & 1)) atomicOr(p.err, kErrDrainTimeout);
      }
      __syncwarp();
    } else if (warp == kVCvtWarpA || warp == kVCvtWarpB) {
      // ================== V converters: from each stage of records, the f16
      // V tile (thread vc makes dims vc and vc + 64)
      const int vc = lane + (warp == kVCvtWarpB ? 32 : 0);
      bool ok = true;
      for (int jt = 0; jt < n_tiles && ok; ++jt) {
        const int sr = jt % kRawStages, s16 = jt % kV16Stages;
        ok = wait(raw_full(sr), (jt / kRawStages) & 1);
        if (ok && jt >= kV16Stages) ok = wait(v16_empty(s16), ((jt / kV16Stages) - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const uint32_t mask = raw_mask[sr];
        const int key0 = (jt0 + jt) * kKv;
        const uint8_t* raw = smem + kRaw + sr * kRawStage;
        // dim d of every record; tokens 2k, 2k+1 (word A_k) and 2k+8, 2k+9
        // (word B_k) of record st
        for (int d = vc; d < kD; d += kVCvt) {
          uint8_t* dst = smem + kV16 + s16 * kV16Stage + d * 16;
          const int code_base = 1024 + 16 * ((d >> 6) * 32 + 4 * (d & 7)) + 4 * ((d >> 4) & 3);
          const int byte0 = 2 * ((d & 15) >> 3);  // byte of tokens (2k, 2k+1); +1: (2k+8, 2k+9)
          const int scale_base = 2176 + 4 * (d >> 4);
#pragma unroll 2
          for (int st = 0; st < kKv / kSub; ++st) {
            const int nv = ((mask >> ((kSub * st) / BS)) & 1u) ? min(kSub, max(0, ctx - (key0 + kSub * st))) : 0;
            uint4 a = make_uint4(0u, 0u, 0u, 0u), c = make_uint4(0u, 0u, 0u, 0u);
            if (nv > 0) {
              const uint8_t* rec = raw + st * kFp4SubBytes;
              uint32_t av[4], bv[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint32_t cw = *reinterpret_cast<const uint32_t*>(rec + code_base + 16 * k);
                const uint32_t sw = *reinterpret_cast<const uint32_t*>(rec + scale_base + 32 * k);
                uint32_t slo, shi;  // scales of tokens (2k, 2k+1) and (2k+8, 2k+9)
                e4m3x4_to_f16x2(sw, slo, shi);
                uint32_t f[4];
                fp4x8_to_f16x2(cw >> (8 * byte0), f);  // f[0]: tokens 2k, 2k+1; f[1]: 2k+8, 2k+9
                av[k] = hmul2_bits(f[0], slo);
                bv[k] = hmul2_bits(f[1], shi);
              }
              a = make_uint4(av[0], av[1], av[2], av[3]);
              c = make_uint4(bv[0], bv[1], bv[2], bv[3]);
              if (nv < kSub) {
                a = make_uint4(keep_tokens(a.x, 0, nv), keep_tokens(a.y, 1, nv), keep_tokens(a.z, 2, nv),
                               keep_tokens(a.w, 3, nv));
                c = make_uint4(keep_tokens(c.x, 4, nv), keep_tokens(c.y, 5, nv), keep_tokens(c.z, 6, nv),
                               keep_tokens(c.w, 7, nv));
              }
            }
            *reinterpret_cast<uint4*>(dst + st * kV16Sub) = a;
            *reinterpret_cast<uint4*>(dst + st * kV16Sub + kV16Sub / 2) = c;
          }
        }
        fence_proxy_async_smem();
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(v16_full(s16)) : "memory");
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(raw_empty(sr)) : "memory");
      }
    } else if (warp == kMmaWarp) {
      // ===================== MMA issuer, in the bf16 kernel's order: per key
      // tile and query tile, P V of the previous key tile, then S
      if (lane == 0) {
        constexpr uint32_t idS = umma_idesc_f16(kRows, kKv, false);
        constexpr uint32_t idO = umma_idesc_f16(kRows, kD, false);
        const uint64_t q_desc = umma_desc_sw128(smem_addr(smem + kQ), 16, 1024);
        const uint64_t k_desc = umma_desc_sw128(smem_addr(smem + kKt), 16, 1024);
        // f16 V: core matrices 8 dims x 8 tokens; 128 bytes to the next 8
        // dims, 2 KB to the next 8 tokens
        const uint64_t v_desc = umma_desc_noswz(smem_addr(smem + kV16), kV16Sub / 2, 128);
        const uint32_t q_lo = static_cast<uint32_t>(q_desc), q_hi = static_cast<uint32_t>(q_desc >> 32);
        const uint32_t k_lo = static_cast<uint32_t>(k_desc), k_hi = static_cast<uint32_t>(k_desc >> 32);
        const uint32_t v_lo = static_cast<uint32_t>(v_desc), v_hi = static_cast<uint32_t>(v_desc >> 32);
        bool ok = wait(q_full, 0);
        if (ok) tc_fence_after();
        auto issue_s = [&](int t) {
          const uint32_t qa = q_lo + t * (kQTile >> 4);
          const uint32_t d = tmem + t * kTmemTile;
          // S = Q K^T, 16 dims per product
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            umma_bf16_w(d, qa + (((k >> 2) * (kRows * 128) + (k & 3) * 32) >> 4), q_hi,
                        k_lo + (((k >> 2) * (kKv * 128) + (k & 3) * 32) >> 4), k_hi, idS, k > 0);
          umma_commit(s_full(t));
        };
        auto issue_pv = [&](int t, int jt) {
          const uint32_t va = v_lo + (jt % kV16Stages) * (kV16Stage >> 4);
          const uint32_t pt = tmem + t * kTmemTile;
          const uint32_t d = pt + kOCol;
          // O += P V, 16 keys (one record, eight columns of P) per product
#pragma unroll
          for (int k = 0; k < kKv / 16; ++k)
            umma_bf16_ta_w(d, pt + k * 8, va + ((k * kV16Sub) >> 4), v_hi, idO, (jt > 0 || k > 0) ? 1u : 0u);
        };
        for (int jt = 0; ok && jt <= n_tiles; ++jt) {
          bool v_ready = false, k_ready = false;
          for (int t = 0; t < kTiles && ok; ++t) {
            const int nt = t ? n_kv1 : n_kv0;
            if (jt > 0 && jt - 1 < nt) {
              if (!v_ready) {
                ok = wait(v16_full((jt - 1) % kV16Stages), ((jt - 1) / kV16Stages) & 1);
                if (!ok) break;
                tc_fence_after();
                v_ready = true;
              }
              ok = wait(p_full(t), (jt - 1) & 1);
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, jt - 1);
              umma_commit(jt == nt ? o_final(t) : pv_done(t));
            }
            if (jt < nt) {
              // S of this key tile overwrites the P the previous product reads
              // (products with different accumulators are not ordered)
              if (jt > 0) {
                ok = wait(pv_done(t), (jt - 1) & 1);
                if (!ok) break;
                tc_fence_after();
              }
              if (!k_ready) {
                ok = wait(k16_full, jt & 1);
                if (!ok) break;
                tc_fence_after();
                k_ready = true;
              }
              issue_s(t);
            }
          }
          if (!ok) break;
          if (k_ready) umma_commit(k16_empty);
          if (v_ready) umma_commit(v16_empty((jt - 1) % kV16Stages));
        }
        umma_commit(mma_done);
        if (!wait(mma_done, 0)) atomicOr(p.err, kErrDrainTimeout);
      }
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int BS>
int smem_opt_in() {
  static int done = -1;
  if (done < 0)
    done = cudaFuncSetAttribute(paged_prefill_fp4_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes) == cudaSuccess ? 1 : 0;
  return done;
}

}  // namespace

cudaError_t launch_prefill_fp4(const kv_pool* pool, const PrefillParams& p, int32_t max_q_len,
                               cudaStream_t stream) {
  const int tok_per_cta = kTiles * (kRows / p.group_pow2);
  const int64_t ntiles = (max_q_len + tok_per_cta - 1) / tok_per_cta;
  const int64_t ctas = ntiles * p.n_kv_heads * p.batch;
  if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ctas));
  if (pool->block_size == 32) {
    if (!smem_opt_in<32>()) return cudaErrorInvalidValue;
    paged_prefill_fp4_kernel<32><<<grid, kThreads, kSmemBytes, stream>>>(pool->tmap_rows, p);
  } else {
    if (!smem_opt_in<16>()) return cudaErrorInvalidValue;
    paged_prefill_fp4_kernel<16><<<grid, kThreads, kSmemBytes, stream>>>(pool->tmap_rows, p);
  }
  return cudaGetLastError();
}

}  // namespace pkv
