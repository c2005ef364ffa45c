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
//    staged once in shared memory (128-byte swizzled, K-major).
//  * Keys run in tiles of 64 tokens (4 or 2 pool blocks).  A producer warp
//    gathers each tile's K and V rows with one TMA box per block and column
//    half into a 4-stage ring; blocks outside the attended range or with a
//    bad id are left out and their rows masked.
//  * One thread issues tcgen05.mma: S = Q K^T (128 x 64, fp32 in tensor
//    memory, double-buffered so S of the next tile runs while the softmax of
//    this one does), then O += P V (128 x 128, fp32 in tensor memory), P
//    from tensor memory and V read MN-major straight from its pool rows.
//  * Two query tiles share every key tile: the tensor cores work on one
//    tile's products while the softmax warps of the other run, which hides
//    the latency chain of each (S ready -> softmax -> P -> product).
//  * Four softmax warps per query tile own one row each per thread: tcgen05.ld the row of
//    S, mask (causal, window, sequence end, missing blocks), online softmax
//    in the exp2 domain with a lazy maximum (O in tensor memory is rescaled
//    only when a row's maximum grows by more than 2^8), P in bf16 back into
//    the tensor-memory columns of its S (the P V product reads its A operand
//    from there, so P never touches shared memory, whose bandwidth the
//    products' operand reads already use up), and zeros into the V rows the
//    product must not see (slots past the sequence's end, blocks not loaded).  The epilogue divides O by the
//    row sum and stores the valid rows.
//  * Every wait is bounded in wall time; on a timeout the CTA records
//    KV_ERR_TIMEOUT, drains what it issued and frees its tensor memory.

#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;           // query rows per tile (M)
constexpr int kTiles = 2;            // query tiles per CTA, in ping-pong over the same keys
constexpr int kKv = 64;              // keys per tile (N of S, K of P V)
#ifndef PKV_PF_STAGES
#define PKV_PF_STAGES 4
#endif
constexpr int kStages = PKV_PF_STAGES;  // K/V ring
constexpr int kSoftmax = kTiles * kRows;      // one softmax thread per query row
constexpr int kThreads = kSoftmax + 64;       // + producer warp + MMA warp
constexpr int kProducerWarp = kSoftmax / 32, kMmaWarp = kProducerWarp + 1;
constexpr float kLazy = 8.f;         // rescale O when a row maximum grows by more than this (log2)
constexpr uint64_t kShortWaitNs = 200000;

// Shared memory (offsets from a 1024-aligned base).
constexpr int kQ = 0;                                 // tiles x 2 halves x [128][64] bf16
constexpr int kQTile = 2 * kRows * 128;
constexpr int kK = kQ + kTiles * kQTile;              // stages x 2 halves x [64][64]
constexpr int kV = kK + kStages * 2 * kKv * 128;
constexpr int kBars = kV + kStages * 2 * kKv * 128;
// barriers: kv_full[3], kv_empty[3], then per tile s_full[2], p_full, o_done; q_full, mma_done
constexpr int kNumBars = 2 * kStages + 4 * kTiles + 2;
constexpr int kTileMask = kBars + kNumBars * 8;       // uint32 [kStages]
constexpr int kTmemSlot = kTileMask + kStages * 4;
constexpr int kSmemBytes = kTmemSlot + 16 + 1024;     // + alignment slack
// tensor memory per query tile: S0 [0,64) S1 [64,128) O [128,256); the
// softmax overwrites the first 32 columns of S_i with P (bf16 pairs)
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
  // pairs four at a time and, inside a group, walks the query-tile index
  // from the last (the most keys under the causal mask) down with the pairs
  // fastest.  The block scheduler then starts every group's longest CTAs
  // first, so short CTAs fill the end of the grid, while the CTAs running at
  // once still share the K/V of only a few pairs in L2.
  constexpr int kGroupPairs = 4;
  const int pairs = p.n_kv_heads * p.batch;
  const int nx = static_cast<int>(gridDim.x) / pairs;
  const int grp = static_cast<int>(blockIdx.x) / (kGroupPairs * nx);
  const int r = static_cast<int>(blockIdx.x) - grp * kGroupPairs * nx;
  const int kc = min(kGroupPairs, pairs - grp * kGroupPairs);  // pairs in this group
  const int qx = nx - 1 - r / kc;
  const int hb = grp * kGroupPairs + r % kc;
  const int b = hb / p.n_kv_heads, h = hb - b * p.n_kv_heads;
  const int Gp = p.group_pow2, g = p.group;
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
  static_assert(kTiles == 2, "two query tiles in ping-pong");
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
  auto kv_full = [&](int s) { return bar0 + 8u * s; };
  auto kv_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto s_full = [&](int t, int i) { return bar0 + 8u * (2 * kStages + 4 * t + i); };
  auto p_full = [&](int t) { return bar0 + 8u * (2 * kStages + 4 * t + 2); };
  auto o_done = [&](int t) { return bar0 + 8u * (2 * kStages + 4 * t + 3); };
  const uint32_t q_full = bar0 + 8u * (2 * kStages + 4 * kTiles);
  const uint32_t mma_done = q_full + 8;
  uint32_t* tile_mask = reinterpret_cast<uint32_t*>(smem + kTileMask);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlot);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(s_full(t, 0), 1);
      mbar_init(s_full(t, 1), 1);
      mbar_init(p_full(t), kRows);
      mbar_init(o_done(t), 1);
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

  if (warp < kProducerWarp) {
    // ====== softmax warps: warps 4t..4t+3 serve query tile t, one row per thread
    const int t = warp >> 2;
    const int r = tid & (kRows - 1);
    const int tq = r / Gp, jh = r - tq * Gp;
    const bool row_ok = tq < (t ? ntok1 : ntok0) && jh < g;
    const int tok = tok0 + t * tpt + tq;
    const int pos = pos_base + tok;
    const int lo = p.window > 0 ? max(0, pos + 1 - p.window) : 0;
    const int hq = h * g + jh;
    // Q row r of tile t -> shared memory (zeros for padding rows)
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(p.q) +
          (static_cast<int64_t>(q0 + tok) * p.n_q_heads + hq) * kD);
      uint8_t* qt = smem + kQ + t * kQTile;
#pragma unroll
      for (int c = 0; c < kD / 8; ++c) {
        const uint4 v = row_ok ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(qt + (c >> 3) * (kRows * 128) + swz128(r, c & 7)) = v;
      }
      fence_proxy_async_smem();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(q_full) : "memory");
    }
    const uint32_t lane_base = tmem + t * kTmemTile + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    const int nt = t ? n_kv1 : n_kv0;
    for (int jt = 0; jt < nt && ok; ++jt) {
      const int s = jt % kStages, sb = jt & 1;
      ok = wait(s_full(t, sb), (jt >> 1) & 1) && wait(kv_full(s), (jt / kStages) & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t mask = tile_mask[s];
      const int key0 = (jt0 + jt) * kKv;
      // raw scores; masked keys become -inf (the scale is applied in the exp)
      float x[kKv];
      float mt4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      {
        uint32_t raw[2][32];
        tmem_ld32x2(lane_base + sb * kKv, lane_base + sb * kKv + 32, raw[0], raw[1]);
        // rows of this warp that see every key of the tile need no mask
        const bool whole = row_ok && key0 >= lo && key0 + kKv - 1 <= pos &&
                           mask == (1u << (kKv / BS)) - 1u;
        if (__all_sync(0xffffffffu, whole)) {
#pragma unroll
          for (int c = 0; c < kKv; ++c) {
            x[c] = __uint_as_float(raw[c >> 5][c & 31]);
            mt4[c & 3] = fmaxf(mt4[c & 3], x[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kKv; ++c) {
            const int key = key0 + c;
            const bool valid = row_ok && key >= lo && key <= pos && ((mask >> (c / BS)) & 1u);
            x[c] = valid ? __uint_as_float(raw[c >> 5][c & 31]) : -INFINITY;
            mt4[c & 3] = fmaxf(mt4[c & 3], x[c]);
          }
        }
      }
      // row maximum in the exp2 domain (scale > 0)
      const float mt_raw = fmaxf(fmaxf(mt4[0], mt4[1]), fmaxf(mt4[2], mt4[3]));
      const float mt = mt_raw == -INFINITY ? -INFINITY : mt_raw * p.scale_log2;
      // The new running maximum needs no tensor memory: a row with nothing
      // accumulated yet (O's row is zero) takes it; others keep theirs unless
      // it grew by more than 2^kLazy.  The exponentials and the store of P
      // (into the other S buffer) proceed while the previous P V product of
      // this tile may still run; the rescale of O waits for it.
      const float m_new = fmaxf(m_run, mt);
      const bool rescale = m_run != -INFINITY && m_new > m_run + kLazy;
      const float m_old = m_run;
      if (m_run == -INFINITY || rescale) m_run = m_new;
      const float mu = m_run == -INFINITY ? 0.f : m_run;
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nmu2 = make_float2(-mu, -mu);
      float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t w[kKv / 2];  // the P row, bf16 pairs
#pragma unroll
      for (int e = 0; e < kKv / 2; ++e) {
        const float2 arg = ffma2(make_float2(x[2 * e], x[2 * e + 1]), sc2, nmu2);
        const float2 pe = make_float2(fast_exp2(arg.x), fast_exp2(arg.y));
        l2[e & 1] = fadd2(l2[e & 1], pe);
        w[e] = pack_bf16x2(pe.x, pe.y);
      }
      // P row (bf16 pairs) over the S columns just read: the product of key
      // tile jt takes its A operand from there, and S of key tile jt + 2,
      // the next writer of these columns, is issued after that product
      tmem_st32(lane_base + sb * kKv, w);
      // The previous product of this tile: O is stable once it is done.  The
      // wait is taken every key tile, so the barrier's phases stay in step
      // with jt (its parity then names exactly one product).
      if (jt > 0) {
        ok = wait(o_done(t), (jt - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {  // tensor-memory access is warp-wide
        const float alpha = rescale ? fast_exp2(m_old - m_new) : 1.f;
        l_run *= alpha;
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + 2 * kKv + c0, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(lane_base + 2 * kKv + c0, o);
        }
      }
      l_run += (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
      // V rows the products must not see: slots past the sequence's end and
      // blocks that were not loaded (stale or never-written shared memory).
      // The first query tile that uses this key tile does it before handing
      // its P over; the products of the other tile are issued after that.
      const int zero_tile = jt < n_kv0 ? 0 : 1;
      if (t == zero_tile && (mask != (1u << (kKv / BS)) - 1u || key0 + kKv > ctx)) {
        for (int idx = r; idx < kKv * 2 * 8; idx += kRows) {
          const int key = idx >> 4, half = (idx >> 3) & 1, chunk = idx & 7;
          if (key0 + key >= ctx || !((mask >> (key / BS)) & 1u))
            *reinterpret_cast<uint4*>(smem + kV + s * (2 * kKv * 128) + half * (kKv * 128) +
                                      key * 128 + chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(p_full(t)) : "memory");
    }
    if (ok && nt > 0) ok = __all_sync(0xffffffffu, wait(o_done(t), (nt - 1) & 1));
    if (ok && nt > 0) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      float* dst = p.out + (static_cast<int64_t>(q0 + tok) * p.n_q_heads + hq) * kD;
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(lane_base + 2 * kKv + c0, o);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + c0 + i) =
                make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                            __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
        }
      }
    }
  } else if (warp == kProducerWarp) {
    // =========================== producer: K and V rows of each key tile
    if (lane == 0) {
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
        const int s = jt % kStages;
        int cur[kKv / BS];
#pragma unroll
        for (int i = 0; i < kKv / BS; ++i) cur[i] = next[i];
        if (jt + 1 < n_tiles) fetch(jt + 1);
        if (jt >= kStages && !wait(kv_empty(s), ((jt / kStages) - 1) & 1)) break;
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
        tile_mask[s] = mask;
        const uint32_t bar = kv_full(s);
        const int nblk = __popc(mask);
        if (nblk == 0) {
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
        } else {
          mbar_arrive_expect_tx(bar, nblk * 2 * 2 * BS * 128);
          const uint32_t ks = smem_addr(smem + kK + s * (2 * kKv * 128));
          const uint32_t vs = smem_addr(smem + kV + s * (2 * kKv * 128));
#pragma unroll
          for (int i = 0; i < kKv / BS; ++i) {
            if (phys[i] < 0) continue;
            const int tile = phys[i] * p.n_kv_heads + h;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t off = half * (kKv * 128) + i * BS * 128;
              tma_load_4d(ks + off, &tmap, bar, half * 64, 0, 0, tile);
              tma_load_4d(vs + off, &tmap, bar, half * 64, 0, 1, tile);
            }
          }
        }
        ++issued;
      }
      // leave no copy in flight: wait (bounded) for the stages not yet consumed
      for (int jt = max(0, issued - kStages); jt < issued; ++jt)
        wait(kv_full(jt % kStages), (jt / kStages) & 1);
    }
    __syncwarp();
  } else {
    // =========================== MMA issuer: for every key tile, S of both
    // query tiles, then the P V products of the previous key tile
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
      constexpr uint32_t kStageUnits = (2 * kKv * 128) >> 4;
      bool ok = wait(q_full, 0);
      if (ok) tc_fence_after();
      auto issue_s = [&](int t, int jt) {
        const uint32_t ka = k_lo + (jt % kStages) * kStageUnits;
        const uint32_t qa = q_lo + t * (kQTile >> 4);
        const uint32_t d = tmem + t * kTmemTile + (jt & 1) * kKv;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)
          umma_bf16_w(d, qa + (((k >> 2) * (kRows * 128) + (k & 3) * 32) >> 4), q_hi,
                      ka + (((k >> 2) * (kKv * 128) + (k & 3) * 32) >> 4), k_hi, idS, k > 0);
        umma_commit(s_full(t, jt & 1));
      };
      auto issue_pv = [&](int t, int jt) {
        const uint32_t va = v_lo + (jt % kStages) * kStageUnits;
        const uint32_t pt = tmem + t * kTmemTile + (jt & 1) * kKv;  // P in tensor memory
        const uint32_t d = tmem + t * kTmemTile + 2 * kKv;
#pragma unroll
        for (int k = 0; k < kKv / 16; ++k)
          umma_bf16_ta_w(d, pt + k * 8, va + ((k * 16 * 128) >> 4), v_hi, idO,
                         (jt > 0 || k > 0) ? 1u : 0u);
        umma_commit(o_done(t));
      };
      // P V of key tile jt for every query tile that has it; then the stage is free
      auto issue_pvs = [&](int jt) {
        for (int t = 0; t < kTiles && ok; ++t) {
          if (jt >= (t ? n_kv1 : n_kv0)) continue;
          ok = wait(p_full(t), jt & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(t, jt);
        }
        if (ok) umma_commit(kv_empty(jt % kStages));
      };
      for (int jt = 0; ok && jt < n_tiles; ++jt) {
        ok = wait(kv_full(jt % kStages), (jt / kStages) & 1);
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < kTiles; ++t)
          if (jt < (t ? n_kv1 : n_kv0)) issue_s(t, jt);
        if (jt > 0) issue_pvs(jt - 1);
      }
      if (ok) issue_pvs(n_tiles - 1);
      // every product issued has completed before the tensor memory is freed
      umma_commit(mma_done);
      wait(mma_done, 0);
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
