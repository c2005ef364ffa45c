// Paged prefill / extend attention on the 5th-generation tensor cores.
//
// What it computes ("Optimizing KV Cache Memory Management in vLLM with
// PagedAttention and Dynamic Block Allocation", "The Prefill Phase"; prefix
// caching from "PagedAttention", "Walking through two requests"): the q_len
// new tokens of sequence b are the last positions of its context_lens[b]
// tokens, their K/V already in the pool; token i at position
// pos = ctx - q_len + i attends causally to [lo, pos] of the sequence, with
// lo = max(0, pos + 1 - W) under a window W, else 0, resolving every key
// through the block table.  GQA: query head hq reads KV head hq / g.
//
// How (GB300 design), one CTA per (two 128-row query tiles, KV head, sequence):
//  * Rows of the tile are (new token, query head of the group) pairs, the
//    group padded to a power of two Gp: 128 / Gp tokens x Gp heads.  Q is
//    staged once in shared memory (128-byte swizzled, K-major), read with
//    whole rows per load instruction.
//  * Keys run in tiles of 128 tokens (8 or 4 pool blocks).  Two producer
//    warps gather each tile's K rows and V rows with one TMA box per block
//    and column half, K into a 2-stage ring and V into a 3-stage ring: a K
//    stage is refilled as soon as the S products of its tile are done, a V
//    stage once its P V products are.  Blocks outside the attended range or
//    with a bad id are left out and their rows masked.
//  * S = Q K^T on kind::f16 with bf16 operands (128 x 128, fp32 in tensor
//    memory).  P V on kind::f16 with f16 operands: P is one f16 per weight
//    (relative rounding 2^-12 on average, where one bf16 P, 2^-9, would put
//    the output ~1e-3 off the exact attention), so V is converted to f16 in
//    place in its stage by a converter warpgroup, scaled by a power of two
//    2^-e: every bf16 value at least 2^-31 times the largest V the CTA has
//    seen is exact in f16 then.  e is set from the first key tile's largest
//    exponent and raised when a later tile would overflow; the largest
//    exponent of a tile comes from the pool's V exponent map (one byte per
//    V row, kept by paged_kv_write), read a tile ahead, not from a pass over
//    the tile.  The softmax warps rescale O by a change of e, and the output
//    by 2^e.  Rows past the sequence's end and of blocks not loaded become
//    zeros.
//    128-key products run the tensor pipe at its full rate; 64-key ones
//    reach two thirds of it.
//  * Two query tiles share every key tile and alternate on the tensor pipe:
//    the products of one tile run while the softmax warps of the other do.
//    Each tile has one S buffer: S of the next key tile is issued once the
//    P V product that reads P from it has completed (products with different
//    accumulators are not ordered), so a finished S also means O is stable.
//  * Four softmax warps per query tile own one row each per thread: two
//    tensor-memory loads of the row of S (128 columns), masking (causal,
//    window, sequence end, missing blocks), online softmax in the exp2
//    domain with a lazy maximum (O in tensor memory is rescaled only when a
//    row's maximum grows by more than 2^8), P as f16 pairs back over the
//    first 64 columns of S.  The epilogue divides O by the row sum and
//    stores the valid rows through a per-warp staging area in the tile's
//    (then unused) Q buffer, so that every store instruction writes whole
//    rows.
//  * Registers: the two softmax warpgroups take 192 per thread, the
//    producer / issuer and converter warpgroups give theirs up to 64.
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
constexpr int kKStages = 2;          // K ring
constexpr int kVStages = 3;          // V ring (bf16 as copied, then f16 in place)
constexpr int kSoftmax = kTiles * kRows;      // one softmax thread per query row
constexpr int kKWarp = kSoftmax / 32, kVWarp = kKWarp + 1, kMmaWarp = kVWarp + 1;
constexpr int kCvtWarp = kKWarp + 4;          // converter warpgroup (warp kKWarp + 3 is idle)
constexpr int kCvt = 128;
constexpr int kThreads = kSoftmax + 128 + kCvt;
constexpr int kLaunchRegs = 65536 / kThreads;
constexpr int kSoftmaxRegs = 192, kOtherRegs = 64;
static_assert(2 * kSoftmaxRegs + 2 * kOtherRegs <= 4 * kLaunchRegs,
              "register increases must be covered by the decreases");
constexpr float kLazy = 8.f;         // rescale O when a row maximum grows by more than this (log2)
// V's power of two: e = E - kVBias for a largest biased bf16 exponent E puts
// the largest magnitude in [2^14, 2^15)
constexpr int kVBias = 141, kVMin = -126, kVMax = 113;
constexpr uint64_t kShortWaitNs = 200000;

// Shared memory (offsets from a 1024-aligned base).
constexpr int kQ = 0;                                 // tiles x 2 halves x [128][64] bf16
constexpr int kQTile = 2 * kRows * 128;
constexpr int kKvStage = 2 * kKv * 128;               // 2 column halves x [128 keys][64] bf16
constexpr int kK = kQ + kTiles * kQTile;
constexpr int kV = kK + kKStages * kKvStage;
constexpr int kVe = kV + kVStages * kKvStage;         // int32 [kVStages]: each stage's e
constexpr int kVMask = kVe + 16;                      // uint32 [kVStages]: blocks each V stage holds
constexpr int kBars = kVMask + 16;
static_assert(kVStages * 4 <= 16, "the V stages' exponents and block masks fit");
// barriers: k_full[2], k_empty[2], v_full[3], v_empty[3], v16_full[3], per tile
// s_full, p_full, pv_done, o_final; q_full, mma_done
constexpr int kNumBars = 2 * kKStages + 3 * kVStages + 4 * kTiles + 2;
constexpr int kTmemSlot = kBars + kNumBars * 8;
constexpr int kSmemBytes = kTmemSlot + 16 + 1024;     // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");
// tensor memory per query tile: S [0,128) (P as f16 pairs over its first 64 columns),
// O [128,256)
constexpr uint32_t kOCol = kKv;
constexpr uint32_t kTmemTile = 256;
constexpr uint32_t kTmemCols = kTiles * kTmemTile;

__device__ __forceinline__ int swz128(int row, int chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// a * b on two fp32 lanes at once.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(reinterpret_cast<const uint64_t&>(a)), "l"(reinterpret_cast<const uint64_t&>(b)));
  return reinterpret_cast<const float2&>(d);
}

// The two bf16 of a word, times s, as an f16 pair (exact while the products
// are normal in f16).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float2 s) {
  const float2 f = fmul2(make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)), s);
  return pack_f16x2(f.x, f.y);
}

// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

template <int BS>
__global__ void __launch_bounds__(kThreads, 1) paged_prefill_kernel(
    const __grid_constant__ CUtensorMap tmap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Heavy tiles first, in groups: the 1-D grid takes the (sequence, KV head)
  // pairs sixteen at a time and, inside a group, walks the query-tile index
  // from the last (the most keys under the causal mask) down with the pairs
  // fastest.  The block scheduler then starts every group's longest CTAs
  // first, so short CTAs fill the end of the grid, while the CTAs running at
  // once still share the K/V of only a few pairs in L2.
  constexpr int kGroupPairs = 16;
  const int pairs = p.n_kv_heads * p.batch;
  const int nx = static_cast<int>(gridDim.x) / pairs;
  const int grp = static_cast<int>(blockIdx.x) / (kGroupPairs * nx);
  const int r = static_cast<int>(blockIdx.x) - grp * kGroupPairs * nx;
  const int kc = min(kGroupPairs, pairs - grp * kGroupPairs);  // pairs in this group
  const int qx = nx - 1 - r / kc;
  const int hb = grp * kGroupPairs + r % kc;
  const int b = hb / p.n_kv_heads, h = hb - b * p.n_kv_heads;
  const int Gp = p.group_pow2, g = p.group;
  const int log2_gp = __ffs(Gp) - 1;
  const int tpt = kRows / Gp;  // query tokens per tile

  // ---- the CTA's queries and the keys they need (uniform over the CTA)
  const int32_t q0 = p.cu_q_lens[b];
  const int32_t qn = p.cu_q_lens[b + 1] - q0;
  const int32_t ctx = p.context_lens[b];
  if (qn < 0 || qn > ctx || ctx > p.max_ctx || static_cast<int64_t>(ctx) > static_cast<int64_t>(p.mbs) * BS) {
    if (qn != 0 && qx == 0 && h == 0 && tid == 0) atomicOr(p.err, kErrBadContext);
    return;
  }
  const int tok0 = qx * (kTiles * tpt);
  if (tok0 >= qn) return;
  const int pos_base = ctx - qn;  // position of new token 0
  // tile t holds tokens tok0 + t * tpt .. (ntok[t] of them; tile 1 may be empty)
  static_assert(kTiles == 2, "two query tiles alternating");
  const int kv_begin = p.window > 0 ? max(0, pos_base + tok0 + 1 - p.window) : 0;
  const int jt0 = kv_begin / kKv;
  const int ntok0 = min(tpt, qn - tok0), ntok1 = max(0, min(tpt, qn - tok0 - tpt));
  const int last0 = pos_base + tok0 + ntok0 - 1;               // last position of tile 0
  const int last1 = pos_base + tok0 + tpt + ntok1 - 1;         // (tile 1, when not empty)
  const int n_kv0 = last0 / kKv - jt0 + 1;                     // key tiles of each query tile
  const int n_kv1 = ntok1 > 0 ? last1 / kKv - jt0 + 1 : 0;
  const int kv_end = (ntok1 > 0 ? last1 : last0) + 1;
  const int n_tiles = max(n_kv0, n_kv1);                       // key tiles of the CTA

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBars);
  const uint32_t bar0 = smem_addr(bars);
  auto k_full = [&](int s) { return bar0 + 8u * s; };
  auto k_empty = [&](int s) { return bar0 + 8u * (kKStages + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (2 * kKStages + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (2 * kKStages + kVStages + s); };
  auto v16_full = [&](int s) { return bar0 + 8u * (2 * kKStages + 2 * kVStages + s); };
  constexpr int kTileBars = 2 * kKStages + 3 * kVStages;
  auto s_full = [&](int t) { return bar0 + 8u * (kTileBars + 4 * t); };
  auto p_full = [&](int t) { return bar0 + 8u * (kTileBars + 4 * t + 1); };
  auto pv_done = [&](int t) { return bar0 + 8u * (kTileBars + 4 * t + 2); };
  auto o_final = [&](int t) { return bar0 + 8u * (kTileBars + 4 * t + 3); };
  const uint32_t q_full = bar0 + 8u * (kTileBars + 4 * kTiles);
  const uint32_t mma_done = q_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlot);
  int* v_e = reinterpret_cast<int*>(smem + kVe);
  uint32_t* v_mask = reinterpret_cast<uint32_t*>(smem + kVMask);

  if (tid == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(v16_full(s), kCvt);
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
  // Which blocks of key tile jt are loaded (inside [kv_begin, kv_end), a
  // table entry inside the pool): the rule every role applies.
  const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.mbs;
  auto needed = [&](int jt, int i) {
    const int k0 = (jt0 + jt) * kKv + i * BS;
    return k0 + BS > kv_begin && k0 < kv_end;
  };

  if (warp < kKWarp) {
    warpgroup_regs_inc<kSoftmaxRegs>();
    // ====== softmax warps: warps 4t..4t+3 serve query tile t, one row per thread
    const int t = warp >> 2;
    const int r = tid & (kRows - 1);
    const int tq = r / Gp, jh = r - tq * Gp;
    const bool row_ok = tq < (t ? ntok1 : ntok0) && jh < g;
    const int tok = tok0 + t * tpt + tq;
    const int pos = pos_base + tok;
    const int lo = p.window > 0 ? max(0, pos + 1 - p.window) : 0;
    // Q of both tiles -> shared memory (zeros for padding rows), coalesced:
    // 16 threads per row, so one load instruction reads two whole 256-byte
    // rows of q
    {
      const uint4* qg = static_cast<const uint4*>(p.q);
      constexpr int kChunks = kD / 8;  // 16-byte chunks per row
#pragma unroll
      for (int it = 0; it < kTiles * kRows * kChunks / kSoftmax; ++it) {
        const int idx = it * kSoftmax + tid;
        const int row = idx / kChunks, ch = idx % kChunks;
        const int tt = row / kRows, rr = row % kRows;
        const int tq2 = rr >> log2_gp, jh2 = rr & (Gp - 1);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tq2 < (tt ? ntok1 : ntok0) && jh2 < g) {
          v = qg[(static_cast<int64_t>(q0 + tok0 + tt * tpt + tq2) * p.n_q_heads + h * g + jh2) *
                     kChunks + ch];
          v = make_uint4(v.x ^ p.q_sign, v.y ^ p.q_sign, v.z ^ p.q_sign, v.w ^ p.q_sign);
        }
        *reinterpret_cast<uint4*>(smem + kQ + tt * kQTile + (ch >> 3) * (kRows * 128) +
                                  swz128(rr, ch & 7)) = v;
      }
      fence_proxy_async_smem();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(q_full) : "memory");
    }
    const uint32_t lane_base = tmem + t * kTmemTile + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const float coef = p.scale_log2;
    constexpr uint32_t kAllBlocks = (1u << (kKv / BS)) - 1u;
    float m_raw = -INFINITY, l_run = 0.f;  // running maximum in raw score units
    int ve = 0;                            // V's power of two in the products so far
    bool ok = true;
    const int nt = t ? n_kv1 : n_kv0;
    // Which blocks of a key tile hold keys: the same rule the producers use
    // (inside [kv_begin, kv_end), a table entry inside the pool), from the
    // table entries read one key tile ahead, so the softmax never waits for
    // the V copy it does not read.
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
      // rows of this warp that see every key of the tile need no mask;
      // masked keys become -inf (the scale is applied in the exp)
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
      // A row with nothing accumulated yet (O's row is zero) takes the new
      // maximum; others keep theirs unless it grew by more than 2^kLazy.  The
      // maximum is kept in raw score units (the scale is positive), so the
      // rescale and, for large scores, the exponents come from exact
      // differences of raw scores.
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
      // V's power of two for this key tile (its P V product cannot be issued
      // before the conversion anyway); a raised one scales what O holds down
      const int sv = jt % kVStages;
      ok = wait(v16_full(sv), (jt / kVStages) & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const int ve_j = v_e[sv];
      const bool vchange = jt > 0 && ve_j != ve;
      if (__any_sync(0xffffffffu, rescale) || vchange) {  // tensor-memory access is warp-wide
        const float alpha = rescale ? fast_exp2((m_old - m_raw) * coef) : 1.f;
        l_run *= alpha;
        const float f = vchange ? alpha * pow2i(max(ve - ve_j, kVMin)) : alpha;
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + kOCol + c0, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(lane_base + kOCol + c0, o);
        }
      }
      ve = ve_j;
      l_run += (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(p_full(t)) : "memory");
    }
    if (ok && nt > 0) ok = __all_sync(0xffffffffu, wait(o_final(t), 0));
    if (ok && nt > 0) {
      tc_fence_after();
      const float inv = l_run > 0.f ? pow2i(ve) / l_run : 0.f;
      // O 2^e / l -> out, coalesced: each warp stages its 32 rows, 64 columns
      // at a time, in shared memory (the tile's Q buffer, free once the tile's
      // last product is done; 16-byte chunk c of row r at slot c ^ (r & 15)),
      // then stores two whole 256-byte row halves per instruction.
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
          const int r_t = 32 * (warp & 3) + row;  // row of the tile
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
    // ====== converters: each V stage, bf16 as copied, into f16 in place.
    // Thread ct takes the 16-byte chunks ct + 128 i (i < 16) of the stage's
    // two column halves: key row ct / 8 + 16 (i mod 8), a whole 512-byte run
    // of the stage per warp and instruction.  The largest exponent of the
    // rows that hold keys comes from the pool's exponent map: lane l reads
    // the entries of keys 4l .. 4l + 3, loaded a key tile ahead (the table
    // entry two tiles ahead), and every warp reads all 128 and comes to the
    // same answer.  Then the conversion, scaled by the power of two that
    // keeps it exact; rows without a key are zeroed.
    const int ct = tid - kCvtWarp * 32;
    const int mblk = (4 * lane) / BS, moff = (4 * lane) % BS;
    auto table_entry = [&](int jt) -> int {
      return jt < n_tiles && needed(jt, mblk) ? trow[((jt0 + jt) * kKv) / BS + mblk] : -1;
    };
    auto map_word = [&](int phys) -> uint32_t {
      if (phys < 0 || phys >= p.num_blocks) return 0u;
      return __ldg(reinterpret_cast<const uint32_t*>(
          p.vexp + (static_cast<int64_t>(phys) * p.n_kv_heads + h) * BS + moff));
    };
    int tab1 = table_entry(1);
    uint32_t map0 = map_word(table_entry(0));
    int e = 0;
    bool ok = true;
    for (int jt = 0; jt < n_tiles && ok; ++jt) {
      const int tab2 = table_entry(jt + 2);
      const uint32_t map1 = map_word(tab1);
      const int s = jt % kVStages;
      ok = wait(v_full(s), (jt / kVStages) & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const uint32_t mask = v_mask[s];  // the blocks the stage holds, left by the V producer
      const int key0 = (jt0 + jt) * kKv;
      constexpr uint32_t kAllBlocks = (1u << (kKv / BS)) - 1u;
      const bool full = mask == kAllBlocks && key0 + kKv <= ctx;
      auto row_ok = [&](int key) { return full || (((mask >> (key / BS)) & 1u) && key0 + key < ctx); };
      uint32_t E = 0;
      bool stale = false;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t x = (map0 >> (8 * b)) & 0xFFu;
        if (row_ok(4 * lane + b)) {
          stale = stale || x == 0u;
          E = max(E, x);
        }
      }
      if (stale && warp == kCvtWarp) atomicOr(p.err, kErrStaleMap);
      E = __reduce_max_sync(0xffffffffu, E);
      map0 = map1;
      tab1 = tab2;
      // the first tile sets e; later tiles only raise it, when they would
      // overflow
      const int need = static_cast<int>(E) - kVBias;
      if (jt == 0)
        e = min(max(need, kVMin), kVMax);
      else if (need > e)
        e = min(need, kVMax);
      const float2 sc = make_float2(pow2i(-e), pow2i(-e));
      const uint32_t st = smem_addr(smem + kV + s * kKvStage) + 16 * ct;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (row_ok((ct >> 3) + 16 * (i & 7))) {
          const uint4 v = lds128(st + 2048 * i);
          o = make_uint4(bf16x2_to_f16x2(v.x, sc), bf16x2_to_f16x2(v.y, sc), bf16x2_to_f16x2(v.z, sc),
                         bf16x2_to_f16x2(v.w, sc));
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(st + 2048 * i), "r"(o.x), "r"(o.y),
                     "r"(o.z), "r"(o.w) : "memory");
      }
      if (ct == 0) v_e[s] = e;
      fence_proxy_async_smem();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(v16_full(s)) : "memory");
    }
  } else {
    warpgroup_regs_dec<kOtherRegs>();
    if (warp == kKWarp || warp == kVWarp) {
      // ========================= producers: the K rows (one warp) and the V
      // rows (the other) of each key tile, each into its own ring
      if (lane == 0) {
        const bool is_v = warp == kVWarp;
        const int stages = is_v ? kVStages : kKStages;
        const int rows = is_v ? 1 : 0;  // the pool's K / V index
        uint8_t* ring = smem + (is_v ? kV : kK);
        auto full = [&](int s) { return is_v ? v_full(s) : k_full(s); };
        auto empty = [&](int s) { return is_v ? v_empty(s) : k_empty(s); };
        // The block-table entries of a key tile are read one tile ahead, so
        // their global-memory latency overlaps the wait for a free stage.
        int next[kKv / BS];
        auto fetch = [&](int jt) {
#pragma unroll
          for (int i = 0; i < kKv / BS; ++i)
            next[i] = needed(jt, i) ? trow[((jt0 + jt) * kKv + i * BS) / BS] : 0;
        };
        if (n_tiles > 0) fetch(0);
        int issued = 0;
        for (int jt = 0; jt < n_tiles; ++jt) {
          const int s = jt % stages;
          int cur[kKv / BS];
#pragma unroll
          for (int i = 0; i < kKv / BS; ++i) cur[i] = next[i];
          if (jt + 1 < n_tiles) fetch(jt + 1);
          if (jt >= stages && !wait(empty(s), ((jt / stages) - 1) & 1)) break;
          uint32_t mask = 0;
          int phys[kKv / BS];
#pragma unroll
          for (int i = 0; i < kKv / BS; ++i) {
            phys[i] = -1;
            if (!needed(jt, i)) continue;
            const int e = cur[i];
            if (e < 0 || e >= p.num_blocks) {
              if (!is_v) atomicOr(p.err, kErrBadBlock);
              continue;
            }
            phys[i] = e;
            mask |= 1u << i;
          }
          const uint32_t bar = full(s);
          const int nblk = __popc(mask);
          if (is_v) v_mask[s] = mask;  // for the converters (published by the arrive below)
          if (nblk == 0) {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
          } else {
            mbar_arrive_expect_tx(bar, nblk * 2 * BS * 128);
            const uint32_t st = smem_addr(ring + s * kKvStage);
#pragma unroll
            for (int i = 0; i < kKv / BS; ++i) {
              if (phys[i] < 0) continue;
              const int tile = phys[i] * p.n_kv_heads + h;
#pragma unroll
              for (int half = 0; half < 2; ++half)
                tma_load_4d(st + half * (kKv * 128) + i * BS * 128, &tmap, bar, half * 64, 0, rows,
                            tile);
            }
          }
          ++issued;
        }
        // leave no copy in flight: wait (bounded) for the stages not yet consumed
        for (int jt = max(0, issued - stages); jt < issued; ++jt)
          if (!wait(full(jt % stages), (jt / stages) & 1)) atomicOr(p.err, kErrDrainTimeout);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ========================= MMA issuer.  Key tile jt: for each query
      // tile, the P V product of key tile jt - 1 (which reads P from the S
      // buffer), then S of key tile jt into that buffer.
      if (lane == 0) {
        constexpr uint32_t idS = umma_idesc_bf16(kRows, kKv, false);
        constexpr uint32_t idO = umma_idesc_f16(kRows, kD, true);
        // Descriptors as 32-bit halves, computed once: a stage or k-step moves
        // only the start address (16-byte units, low half).
        const uint64_t q_desc = umma_desc_sw128(smem_addr(smem + kQ), 16, 1024);
        const uint64_t k_desc = umma_desc_sw128(smem_addr(smem + kK), 16, 1024);
        const uint64_t v_desc = umma_desc_sw128(smem_addr(smem + kV), kKv * 128, 1024);
        const uint32_t q_lo = static_cast<uint32_t>(q_desc), q_hi = static_cast<uint32_t>(q_desc >> 32);
        const uint32_t k_lo = static_cast<uint32_t>(k_desc), k_hi = static_cast<uint32_t>(k_desc >> 32);
        const uint32_t v_lo = static_cast<uint32_t>(v_desc), v_hi = static_cast<uint32_t>(v_desc >> 32);
        constexpr uint32_t kStageUnits = kKvStage >> 4;
        bool ok = wait(q_full, 0);
        if (ok) tc_fence_after();
        auto issue_s = [&](int t, int jt) {
          const uint32_t ka = k_lo + (jt % kKStages) * kStageUnits;
          const uint32_t qa = q_lo + t * (kQTile >> 4);
          const uint32_t d = tmem + t * kTmemTile;
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            umma_bf16_w(d, qa + (((k >> 2) * (kRows * 128) + (k & 3) * 32) >> 4), q_hi,
                        ka + (((k >> 2) * (kKv * 128) + (k & 3) * 32) >> 4), k_hi, idS, k > 0);
          umma_commit(s_full(t));
        };
        auto issue_pv = [&](int t, int jt) {
          const uint32_t va = v_lo + (jt % kVStages) * kStageUnits;
          const uint32_t pt = tmem + t * kTmemTile;  // P over the S columns
          const uint32_t d = tmem + t * kTmemTile + kOCol;
          // O += P V, 16 keys (eight columns of P) per product
#pragma unroll
          for (int k = 0; k < kKv / 16; ++k)
            umma_bf16_ta_w(d, pt + k * 8, va + ((k * 16 * 128) >> 4), v_hi, idO, (jt > 0 || k > 0) ? 1u : 0u);
        };
        for (int jt = 0; ok && jt <= n_tiles; ++jt) {
          bool v_ready = false, k_ready = false;
          for (int t = 0; t < kTiles && ok; ++t) {
            const int nt = t ? n_kv1 : n_kv0;
            if (jt > 0 && jt - 1 < nt) {
              if (!v_ready) {
                ok = wait(v16_full((jt - 1) % kVStages), ((jt - 1) / kVStages) & 1);
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
              // tcgen05 products with different accumulators are not ordered:
              // S of this key tile overwrites the P the previous product reads,
              // and the softmax rescales O once this S is done, so that product
              // must have completed first (the tensor pipe is busy with it
              // meanwhile)
              if (jt > 0) {
                ok = wait(pv_done(t), (jt - 1) & 1);
                if (!ok) break;
                tc_fence_after();
              }
              if (!k_ready) {
                ok = wait(k_full(jt % kKStages), (jt / kKStages) & 1);
                if (!ok) break;
                tc_fence_after();
                k_ready = true;
              }
              issue_s(t, jt);
            }
          }
          if (!ok) break;
          if (k_ready) umma_commit(k_empty(jt % kKStages));  // free once these products are done
          if (v_ready) umma_commit(v_empty((jt - 1) % kVStages));
        }
        // every product issued has completed before the tensor memory is freed
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
    done = cudaFuncSetAttribute(paged_prefill_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes) == cudaSuccess ? 1 : 0;
  return done;
}

}  // namespace

int prefill_smem_bytes() { return kSmemBytes; }

cudaError_t launch_prefill(const kv_pool* pool, const PrefillParams& p, int32_t max_q_len,
                           cudaStream_t stream) {
  const int tok_per_cta = kTiles * (kRows / p.group_pow2);
  const int64_t ntiles = (max_q_len + tok_per_cta - 1) / tok_per_cta;
  const int64_t ctas = ntiles * p.n_kv_heads * p.batch;
  if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ctas));
  if (pool->block_size == 32) {
    if (!smem_opt_in<32>()) return cudaErrorInvalidValue;
    paged_prefill_kernel<32><<<grid, kThreads, kSmemBytes, stream>>>(pool->tmap_rows, p);
  } else {
    if (!smem_opt_in<16>()) return cudaErrorInvalidValue;
    paged_prefill_kernel<16><<<grid, kThreads, kSmemBytes, stream>>>(pool->tmap_rows, p);
  }
  return cudaGetLastError();
}

}  // namespace pkv
