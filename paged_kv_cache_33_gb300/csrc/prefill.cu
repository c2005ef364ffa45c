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
//  * One thread issues tcgen05.mma: S = Q K^T (128 x 128, fp32 in tensor
//    memory), then O += P_hi V + P_lo V (128 x 128, fp32 in tensor memory)
//    with P read from tensor memory and V read MN-major straight from its
//    pool rows.  P is a bf16 high part plus the bf16 rounding of its
//    remainder: one bf16 P alone (2^-9 relative per weight) would put the
//    output ~1e-3 (relative) off the exact attention.
//    128-key products run the tensor pipe at its full rate; 64-key ones
//    reach two thirds of it.
//  * Two query tiles share every key tile and alternate on the tensor pipe:
//    the products of one tile run while the softmax warps of the other do.
//    Each tile has one S buffer: S of the next key tile is issued once the
//    P V product that reads P from it has completed (products with different
//    accumulators are not ordered), so a finished S also means O is stable.
//  * Four softmax warps per query tile own one row each per thread: one
//    tensor-memory load of the row of S (128 columns), masking (causal, window, sequence end, missing blocks),
//    online softmax in the exp2 domain with a lazy maximum (O in tensor
//    memory is rescaled only when a row's maximum grows by more than 2^8),
//    P's two bf16 parts back over the columns of S (P never touches shared
//    memory, whose bandwidth the products' operand reads use), and zeros into
//    the V rows the product must not see (slots past the sequence's end,
//    blocks not loaded).  The epilogue divides O by the row sum and stores
//    the valid rows through a per-warp staging area in the tile's (then
//    unused) Q buffer, so that every store instruction writes whole rows.
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
constexpr int kVStages = 3;          // V ring
constexpr int kSoftmax = kTiles * kRows;      // one softmax thread per query row
constexpr int kThreads = kSoftmax + 96;       // + K producer, V producer, MMA warps
constexpr int kKWarp = kSoftmax / 32, kVWarp = kKWarp + 1, kMmaWarp = kVWarp + 1;
constexpr float kLazy = 8.f;         // rescale O when a row maximum grows by more than this (log2)
constexpr uint64_t kShortWaitNs = 200000;

// Shared memory (offsets from a 1024-aligned base).
constexpr int kQ = 0;                                 // tiles x 2 halves x [128][64] bf16
constexpr int kQTile = 2 * kRows * 128;
constexpr int kKvStage = 2 * kKv * 128;               // 2 column halves x [128 keys][64] bf16
constexpr int kK = kQ + kTiles * kQTile;
constexpr int kV = kK + kKStages * kKvStage;
constexpr int kBars = kV + kVStages * kKvStage;
// barriers: k_full[2], k_empty[2], v_full[3], v_empty[3], per tile s_full, p_full,
// pv_done, o_final; q_full, mma_done
constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 4 * kTiles + 2;
constexpr int kTmemSlot = kBars + kNumBars * 8;
constexpr int kSmemBytes = kTmemSlot + 16 + 1024;     // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");
// tensor memory per query tile: S [0,128) (P_hi over its first 64 columns, P_lo over
// the last 64), O [128,256)
constexpr uint32_t kOCol = kKv;
constexpr uint32_t kTmemTile = 256;
constexpr uint32_t kTmemCols = kTiles * kTmemTile;

__device__ __forceinline__ int swz128(int row, int chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

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
  constexpr int kTileBars = 2 * kKStages + 2 * kVStages;
  auto s_full = [&](int t) { return bar0 + 8u * (kTileBars + 4 * t); };
  auto p_full = [&](int t) { return bar0 + 8u * (kTileBars + 4 * t + 1); };
  auto pv_done = [&](int t) { return bar0 + 8u * (kTileBars + 4 * t + 2); };
  auto o_final = [&](int t) { return bar0 + 8u * (kTileBars + 4 * t + 3); };
  const uint32_t q_full = bar0 + 8u * (kTileBars + 4 * kTiles);
  const uint32_t mma_done = q_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlot);

  if (tid == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
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

  if (warp < kKWarp) {
    // ====== softmax warps: warps 4t..4t+3 serve query tile t, one row per thread
    const int t = warp >> 2;
    const int r = tid & (kRows - 1);
    const int tq = r / Gp, jh = r - tq * Gp;
    const bool row_ok = tq < (t ? ntok1 : ntok0) && jh < g;
    const int tok = tok0 + t * tpt + tq;
    const int pos = pos_base + tok;
    const int lo = p.window > 0 ? max(0, pos + 1 - p.window) : 0;
    const int hq = h * g + jh;
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
    constexpr uint32_t kAllBlocks = (1u << (kKv / BS)) - 1u;
    float m_raw = -INFINITY, l_run = 0.f;  // running maximum in raw score units
    bool ok = true;
    const int nt = t ? n_kv1 : n_kv0;
    // Which blocks of a key tile hold keys: the same rule the producers use
    // (inside [kv_begin, kv_end), a table entry inside the pool), from the
    // table entries read one key tile ahead, so the softmax never waits for
    // the V copy it does not read.
    const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.mbs;
    auto needed = [&](int jt, int i) {
      const int k0 = (jt0 + jt) * kKv + i * BS;
      return k0 + BS > kv_begin && k0 < kv_end;
    };
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
      const int sv = jt % kVStages;
      ok = wait(s_full(t), jt & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const int key0 = (jt0 + jt) * kKv;
      // the row of S: one tensor-memory load of all kKv columns
      uint32_t x[kKv];
      tmem_ld128(lane_base, x);
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
      const float coef = p.scale_log2;
      const bool rescale = m_raw != -INFINITY && mt_raw != -INFINITY && (mt_raw - m_raw) * coef > kLazy;
      const float m_old = m_raw;
      if (m_raw == -INFINITY || rescale) m_raw = mt_raw;
      const float mr = m_raw == -INFINITY ? 0.f : m_raw;
      float mu = mr * coef;
      // The exponent (x - m) coef is at most kLazy, taken as one FMA against
      // m coef.  Once |m coef| reaches 2^13 fp32 holds it only to within
      // 2^-11 (scores of no real model get there): such warps first subtract
      // m from their raw scores, exactly near the maximum, and use no offset.
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
      // the exponentials; P as a bf16 high part (pairs over the first kKv/2
      // columns of S) and the bf16 rounding of its remainder (the last kKv/2
      // columns), so ~16 significant bits of every weight reach the products.
      // Each quarter of the keys is stored as soon as it is done (its S
      // columns were read into registers above), which keeps few registers
      // live; one wait covers the stores.
      float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      constexpr int kQuarter = kKv / 8;  // bf16 pairs per quarter of the keys
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        uint32_t wh[kQuarter], wl[kQuarter];
#pragma unroll
        for (int i = 0; i < kQuarter; ++i) {
          const int e = kq * kQuarter + i;
          const float2 arg = ffma2(make_float2(__uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1])),
                                   sc2, nmu2);
          const float2 pe = make_float2(fast_exp2(arg.x), fast_exp2(arg.y));
          l2[i & 1] = fadd2(l2[i & 1], pe);
          wh[i] = pack_bf16x2(pe.x, pe.y);
          const float2 rem = fsub2(pe, make_float2(bf16_lo(wh[i]), bf16_hi(wh[i])));
          wl[i] = pack_bf16x2(rem.x, rem.y);
        }
        tmem_st16_nowait(lane_base + kq * kQuarter, wh);
        tmem_st16_nowait(lane_base + kKv / 2 + kq * kQuarter, wl);
      }
      tmem_wait_st();
      // O is stable: S of this key tile was issued only after the tile's
      // previous P V product had completed
      if (__any_sync(0xffffffffu, rescale)) {  // tensor-memory access is warp-wide
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
      // V rows the products must not see: slots past the sequence's end and
      // blocks that were not loaded (stale or never-written shared memory).
      // The first query tile that uses this key tile does it before handing
      // its P over; the product of the other tile is issued after that.
      const int zero_tile = jt < n_kv0 ? 0 : 1;
      if (t == zero_tile && (mask != kAllBlocks || key0 + kKv > ctx)) {
        // the V stage of this key tile cannot be refilled before this tile's
        // P of it is consumed, so its phase is safe to wait on here
        ok = wait(v_full(sv), (jt / kVStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        for (int idx = r; idx < kKv * 2 * 8; idx += kRows) {
          const int key = idx >> 4, half = (idx >> 3) & 1, chunk = idx & 7;
          if (key0 + key >= ctx || !((mask >> (key / BS)) & 1u))
            *reinterpret_cast<uint4*>(smem + kV + sv * kKvStage + half * (kKv * 128) + key * 128 +
                                      chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(p_full(t)) : "memory");
    }
    if (ok && nt > 0) ok = __all_sync(0xffffffffu, wait(o_final(t), 0));
    if (ok && nt > 0) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      // O / l -> out, coalesced: each warp stages its 32 rows, 64 columns at a
      // time, in shared memory (the tile's Q buffer, free once the tile's last
      // product is done; 16-byte chunk c of row r at slot c ^ (r & 15)), then
      // stores two whole 256-byte row halves per instruction.
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
  } else if (warp == kKWarp || warp == kVWarp) {
    // =========================== producers: the K rows (one warp) and the V
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
      const int32_t* trow = p.block_tables + static_cast<int64_t>(b) * p.mbs;
      auto needed = [&](int jt, int i) {
        const int k0 = (jt0 + jt) * kKv + i * BS;
        return k0 + BS > kv_begin && k0 < kv_end;
      };
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
  } else {
    // =========================== MMA issuer.  Key tile jt: for each query
    // tile, the P V product of key tile jt - 1 (which reads P from the S
    // buffer), then S of key tile jt into that buffer.
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc_bf16(kRows, kKv, false);
      constexpr uint32_t idO = umma_idesc_bf16(kRows, kD, true);
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
        // O += P_hi V, then O += P_lo V (the remainders, kKv/2 columns on)
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int k = 0; k < kKv / 16; ++k)
            umma_bf16_ta_w(d, pt + part * (kKv / 2) + k * 8, va + ((k * 16 * 128) >> 4), v_hi, idO,
                           (jt > 0 || part > 0 || k > 0) ? 1u : 0u);
      };
      for (int jt = 0; ok && jt <= n_tiles; ++jt) {
        bool v_ready = false, k_ready = false;
        for (int t = 0; t < kTiles && ok; ++t) {
          const int nt = t ? n_kv1 : n_kv0;
          if (jt > 0 && jt - 1 < nt) {
            if (!v_ready) {
              ok = wait(v_full((jt - 1) % kVStages), ((jt - 1) / kVStages) & 1);
              if (!ok) break;
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
