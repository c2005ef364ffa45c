// Stream-K paged decode attention for sm_103a, and its reduce.
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
//  * Work is the list of units (b, h, k-th attended block of b), ordered by
//    b, then h, then k; one unit is one K tile and one V tile, read once for
//    the g = Hq/Hkv query heads of its KV head.  Every CTA first builds a
//    table of the batch in shared memory (context lengths and the prefix of
//    units per sequence), so any unit is located by a binary search.
//  * A persistent grid splits the list into segments: each warp streams a
//    static share of the first ~75% of the units, then takes chunks of the
//    rest from an atomic ticket counter, smaller and smaller towards the end.  SMs do not all stream at the same rate; the dynamic tail lets
//    fast warps absorb the difference, so the grid finishes together.
//  * Each warp streams its segments through a private ring of STAGES shared
//    memory stages without draining between them: lane 0 resolves the next
//    unit's physical block from the table (read one issue ahead; a bad id is
//    recorded and the block masked), writes the unit's coordinates into the
//    stage's info slot and issues one or two 4-D TMA tensor copies, landing
//    K and V with the 128-byte swizzle so every ldmatrix is free of bank
//    conflicts.  Completion is an mbarrier with a transaction count; every
//    wait is bounded in wall time.  A stage with no unit carries a sentinel.
//  * S^T[16 tokens x 8 heads] = K Q^T on the tensor cores (mma.sync m16n8k16,
//    fp32 accumulate); the V fragments are then moved to registers and the
//    stage refilled at once; online softmax in the exp2 domain with warp
//    shuffles over the token rows; O^T[D x 8 heads] += V^T P^T on the tensor
//    cores.  P^T comes from the score accumulator by movmatrix.  For bf16 KV,
//    P is a bf16 high part plus a bf16 remainder (two products) so ~16 bits
//    of P survive.  For FP8 KV the codes go to the tensor cores untouched
//    (mma.sync m16n8k32 on E4M3): the query and P are each split into an
//    E4M3 high code and the E4M3 code of the remainder (~8 bits together),
//    and the V tile is stored transposed in the pool so that its rows are
//    the A operand of V^T P^T with no conversion or transpose on the SM.
//  * Masking uses selects: scores outside [lo, ctx) become -inf and the V
//    rows of masked positions are zeroed before the product, so stale or NaN
//    slots of a partly filled block never reach the result.
//  * A (b, h) pair inside one segment is normalised and written by its warp.
//    A pair cut between segments leaves one unnormalised partial per segment
//    in slot (segment + pair index) -- unique, because segments and pairs are
//    both contiguous ranges of the same list -- and the warp holding the
//    pair's first unit records (first segment, number of segments).  The
//    reduce kernel, launched as a programmatic dependent of the decode
//    kernel so that its CTAs are already resident, merges them.
//  * Sequences with nothing to attend to get zeros from the CTAs' opening
//    pass, which also reports context lengths out of bounds.

#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr uint64_t kShortWaitNs = 200000;  // wait bound once some warp has timed out
#ifndef PKV_DYN_PCT
#define PKV_DYN_PCT 25
#endif
// The dynamic part is cut into four regions of decreasing chunk size: the
// first three take kPlan.pct of it, the last region the rest.
#ifndef PKV_C0
#define PKV_C0 16
#define PKV_C1 8
#define PKV_C2 4
#define PKV_C3 4
#endif
#ifndef PKV_P0
#define PKV_P0 60
#define PKV_P1 30
#define PKV_P2 10
#endif
#ifndef PKV_FP4_MINB
#define PKV_FP4_MINB 3  // FP4 decode CTAs per SM the registers must allow
#endif
#ifndef PKV_RIF
#define PKV_RIF 4
#define PKV_RMB 1
#endif
// The reduce: threads per CTA and the CTAs per SM its registers must allow.
constexpr int kReduceThreads = 512, kReduceCtas = PKV_RMB;
constexpr int kDynNum = PKV_DYN_PCT, kDynDen = 100;  // dynamic share of the units
struct ChunkPlan {
  int c[4];    // units per chunk in each region
  int pct[3];  // share of the dynamic units in regions 0..2
};
constexpr ChunkPlan kPlan = {{PKV_C0, PKV_C1, PKV_C2, PKV_C3}, {PKV_P0, PKV_P1, PKV_P2}};
constexpr int kC0 = kPlan.c[0], kC1 = kPlan.c[1], kC2 = kPlan.c[2], kC3 = kPlan.c[3];

struct SeqRange {
  int32_t lo, ctx, first_blk, nblk, nunit;
};

// Attended positions [lo, ctx) of a sequence, the blocks of BS tokens that
// hold them, and the units (runs of BPU consecutive blocks) that cover them.
template <int BS, int BPU>
__device__ __forceinline__ SeqRange seq_from_ctx(int32_t ctx, int32_t window) {
  SeqRange r;
  r.ctx = ctx;
  r.lo = window > 0 ? max(0, ctx - window) : 0;
  r.first_blk = r.lo / BS;
  r.nblk = ctx > r.lo ? (ctx - 1) / BS - r.first_blk + 1 : 0;
  r.nunit = (r.nblk + BPU - 1) / BPU;
  return r;
}

// A context length is usable when 0 <= ctx <= both bounds; others count as 0.
template <int BS>
__device__ __forceinline__ bool ctx_ok(const DecodeParams& p, int32_t ctx) {
  return ctx >= 0 && ctx <= p.max_ctx && static_cast<int64_t>(ctx) <= static_cast<int64_t>(p.mbs) * BS;
}

// Shared-memory image of one unit: BPU blocks of BS tokens, each as TMA
// boxes of 128-byte rows with the 128-byte swizzle:
// bf16: D/64 boxes of [K rows | V rows] x 64 columns;
// FP8: one box of [K rows (128 codes) | the transposed V tile seen as BS
//      rows of 128 bytes: BS/16 sub-tiles of [D][16] codes].
// The compute side walks the unit in sub-tiles of 16 tokens.
// Element formats of the pool.
constexpr int kBf16 = 0, kFp8 = 1, kFp4 = 2;

template <int D, int KIND, int BS, int BPU>
struct Geometry {
  static constexpr bool FP8 = KIND == kFp8, FP4 = KIND == kFp4;
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kRowBytes = 128;                         // one swizzled smem row
  static constexpr int kBoxes = FP8 ? 1 : D / 64;               // TMA boxes per block
  static constexpr int kBoxBytes = 2 * BS * kRowBytes;
  static constexpr int kSubPerBlock = BS / 16;
  // FP4: the block's BS/16 sub-tile records, one bulk copy
  static constexpr int kBlockBytes = FP4 ? kSubPerBlock * kFp4SubBytes : kBoxes * kBoxBytes;
  static constexpr int kStageBytes = BPU * kBlockBytes;
  static constexpr int kSub = BPU * kSubPerBlock;               // 16-token sub-tiles per unit
  static constexpr int kSteps = D / 16;                         // k-steps (QK) = m-tiles (PV)
  static_assert(FP4 || kBlockBytes == 2 * BS * D * kElem, "a block is one K and one V tile");
  static_assert(KIND == kBf16 || D == 128, "FP8 rows are one 128-byte swizzle row; FP4 records hold D = 128");
  static_assert(kStageBytes % 16 == 0, "bulk copies land on 16-byte boundaries");
  static_assert(kBoxBytes % 1024 == 0, "boxes keep the 1024-byte swizzle alignment");
  // byte offsets inside a stage of sub-tile `sub`: K row 0 of box 0, and
  // (bf16) V row 0 of box 0 or (FP8) the first row of the transposed V
  // sub-tile; all are multiples of 8 rows, so a row's swizzle phase is its
  // row index from there, mod 8
  __device__ static constexpr int k_off(int sub) {
    return (sub / kSubPerBlock) * kBlockBytes + (sub % kSubPerBlock) * 16 * kRowBytes;
  }
  __device__ static constexpr int v_off(int sub) {
    return FP8 ? (sub / kSubPerBlock) * kBlockBytes + BS * kRowBytes + (sub % kSubPerBlock) * 16 * D
               : k_off(sub) + BS * kRowBytes;
  }
  // FP4: the record of sub-tile `sub`
  __device__ static constexpr int rec_off(int sub) {
    return (sub / kSubPerBlock) * kBlockBytes + (sub % kSubPerBlock) * kFp4SubBytes;
  }
};

// Coordinates of the unit held by one ring stage (u < 0: no unit).
struct StageInfo {
  int32_t u, b, h, k, seg_end, seg;
};

template <int D, int KIND, int BS, int BPU, int NW, int STAGES>
struct Smem {
  static constexpr int kRing = NW * STAGES * Geometry<D, KIND, BS, BPU>::kStageBytes;
  static constexpr int kBars = kRing;                          // uint64 [NW][STAGES]
  static constexpr int kInfo = kBars + NW * STAGES * 8;        // StageInfo [NW][STAGES]
  static constexpr int kCtx = kInfo + NW * STAGES * 24;        // int32 [kMaxDecodeBatch]
  static constexpr int kPre = kCtx + kMaxDecodeBatch * 4;      // int32 [kMaxDecodeBatch + 1]
  static constexpr int kScan = kPre + (kMaxDecodeBatch + 1) * 4 + 4;  // int32 [NW]
  static constexpr int kBytes = kScan + NW * 4 + 1024;         // + alignment slack
};

// Position of one unit: sequence b, KV head h, k-th attended block of b.
struct Cursor {
  int b, h, k;
  SeqRange r;
};

// The segments of one launch.  Static shares are [floor(w Ts / Ps),
// floor((w+1) Ts / Ps)) for w < Ps; then chunk region r starts at unit
// start[r] (start[0] = Ts) with chunks of kC<r> units, its first chunk being
// ticket[r] (ticket[0] = 0).  Segment ids: shares 0..Ps-1, then Ps + ticket.
struct Split {
  int T, Ts, Ps, Nc;
  int start1, start2, start3;     // first units of chunk regions 1..3
  int ticket1, ticket2, ticket3;  // first tickets of regions 1..3

  __device__ void init(int total, int P) {
    T = total;
    const int Td = T >= 8 * P ? static_cast<int>(static_cast<int64_t>(T) * kDynNum / kDynDen) : 0;
    Ts = T - Td;
    Ps = min(P, Ts);
    const int r0 = Td * kPlan.pct[0] / 100 / kC0 * kC0;
    const int r1 = Td * kPlan.pct[1] / 100 / kC1 * kC1;
    const int r2 = Td * kPlan.pct[2] / 100 / kC2 * kC2;
    start1 = Ts + r0;
    start2 = start1 + r1;
    start3 = start2 + r2;
    ticket1 = r0 / kC0;
    ticket2 = ticket1 + r1 / kC1;
    ticket3 = ticket2 + r2 / kC2;
    Nc = ticket3 + (T - start3 + kC3 - 1) / kC3;
  }
  __device__ int seg_of(int u) const {
    if (u < Ts) return static_cast<int>((static_cast<int64_t>(u + 1) * Ps - 1) / Ts);
    if (u < start1) return Ps + (u - Ts) / kC0;
    if (u < start2) return Ps + ticket1 + (u - start1) / kC1;
    if (u < start3) return Ps + ticket2 + (u - start2) / kC2;
    return Ps + ticket3 + (u - start3) / kC3;
  }
  // [first, end) units of dynamic chunk `t` (t < Nc)
  __device__ void chunk(int t, int& first, int& end) const {
    if (t < ticket1) {
      first = Ts + t * kC0;
      end = min(start1, first + kC0);
    } else if (t < ticket2) {
      first = start1 + (t - ticket1) * kC1;
      end = min(start2, first + kC1);
    } else if (t < ticket3) {
      first = start2 + (t - ticket2) * kC2;
      end = min(start3, first + kC2);
    } else {
      first = start3 + (t - ticket3) * kC3;
      end = min(T, first + kC3);
    }
  }
};

template <int D, int KIND, int BS, int BPU, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32, (NW <= 2 ? 6 : (KIND == kFp4 ? PKV_FP4_MINB : 3))) paged_decode_kernel(
    const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
  using G = Geometry<D, KIND, BS, BPU>;
  using S = Smem<D, KIND, BS, BPU, NW, STAGES>;
  constexpr bool FP8 = G::FP8, FP4 = G::FP4;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the stage buffers keeps the 128-byte swizzle
  // pattern equal to (row mod 8).
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  int32_t* s_ctx = reinterpret_cast<int32_t*>(smem + S::kCtx);
  int32_t* s_pre = reinterpret_cast<int32_t*>(smem + S::kPre);
  int32_t* s_scan = reinterpret_cast<int32_t*>(smem + S::kScan);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int worker = blockIdx.x * NW + warp;
  // the reduce kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Pull the block tables into L2 (one line per thread across the grid), so
  // that the first table entries every warp reads, right after the batch
  // table below, do not wait on DRAM.
  {
    const char* tb = reinterpret_cast<const char*>(p.block_tables);
    const int64_t tbytes = static_cast<int64_t>(p.batch) * p.mbs * 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * (NW * 32) * 128;
    for (int64_t off = (static_cast<int64_t>(blockIdx.x) * (NW * 32) + threadIdx.x) * 128;
         off < tbytes; off += stride)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(tb + off));
  }

  // ---- the batch table: usable context lengths and units before each sequence
  {
    constexpr int kThreads = NW * 32;
    constexpr int kPer = kMaxDecodeBatch / kThreads + 1;
    const int per = (p.batch + kThreads - 1) / kThreads;  // consecutive sequences per thread
    const int b0 = threadIdx.x * per;
    int32_t local[kPer];
    int32_t sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      local[i] = 0;
      const int b = b0 + i;
      if (i < per && b < p.batch) {
        int32_t ctx = p.context_lens[b];
        if (!ctx_ok<BS>(p, ctx)) {
          if (blockIdx.x == 0) atomicOr(p.err, kErrBadContext);
          ctx = 0;
        }
        s_ctx[b] = ctx;
        local[i] = seq_from_ctx<BS, BPU>(ctx, p.window).nunit * p.n_kv_heads;
        sum += local[i];
      }
    }
    // exclusive scan of the per-thread sums over the CTA
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    int base = incl - sum;
    for (int w = 0; w < warp; ++w) base += s_scan[w];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int b = b0 + i;
      if (i < per && b < p.batch) s_pre[b] = base;
      base += local[i];
    }
    if (threadIdx.x == kThreads - 1) s_pre[p.batch] = base;
    __syncthreads();
    // zero the outputs of sequences with nothing to attend to (CTA-strided;
    // this call's heads of every KV head)
    for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
      if (s_pre[b + 1] == s_pre[b]) {
        float* o = p.out + static_cast<int64_t>(b) * p.n_q_heads * D;
        const int per_kv = p.group * D;
        for (int x = threadIdx.x; x < p.n_kv_heads * per_kv; x += kThreads) {
          const int hk = x / per_kv;
          o[static_cast<int64_t>(hk) * p.group_stride * D + (x - hk * per_kv)] = 0.f;
        }
      }
    }
  }

  // ---- the split of this call's units into segments
  Split sp;
  sp.init(s_pre[p.batch], p.num_workers);
  if (sp.T == 0) return;

  uint8_t* ring = smem + warp * STAGES * G::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBars) + warp * STAGES;
  StageInfo* info = reinterpret_cast<StageInfo*>(smem + S::kInfo) + warp * STAGES;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Cursor of unit u (u < T): binary search of the batch table.
  auto locate = [&](int u) {
    int lo = 0, hi = p.batch - 1;  // largest b with s_pre[b] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= u) lo = mid; else hi = mid - 1;
    }
    Cursor c;
    c.b = lo;
    c.r = seq_from_ctx<BS, BPU>(s_ctx[lo], p.window);
    const int off = u - s_pre[lo];
    c.h = off / c.r.nunit;
    c.k = off - c.h * c.r.nunit;
    return c;
  };
  // Table entries of the unit's blocks (-1 past the sequence's last block).
  auto table_entries = [&](const Cursor& c, int (&phys)[BPU]) {
    const int32_t* row = p.block_tables + static_cast<int64_t>(c.b) * p.mbs + c.r.first_blk;
#pragma unroll
    for (int i = 0; i < BPU; ++i) {
      const int kb = c.k * BPU + i;
      phys[i] = kb < c.r.nblk ? row[kb] : -1;
    }
  };

  // ---- issue side (lane 0): the next unit to stage, in segment order
  Cursor ic{};
  int iu = 0, iu_end = 0, iseg = 0;
  bool idone = false;
  int next_phys[BPU];
  uint32_t bad_stages = 0, tma_stages = 0;  // bad: bit s * BPU + i for block i of stage s
  // test hook: the first copy of worker 0 expects more bytes than it brings,
  // so its (bounded) wait runs out
  uint32_t stall = worker == 0 ? p.stall_tx : 0u;
  uint32_t stall_bar = 0;  // the barrier that expects the extra bytes
  auto next_segment = [&]() {
    const int t = atomicAdd(p.ticket, 1);
    if (t >= sp.Nc) {
      idone = true;
      return;
    }
    sp.chunk(t, iu, iu_end);
    iseg = sp.Ps + t;
    ic = locate(iu);
    table_entries(ic, next_phys);
  };
  auto issue = [&](int s) {
    const uint32_t bar = smem_addr(&bars[s]);
    if (idone) {  // sentinel: no unit, the phase completes on the arrival alone
      info[s].u = -1;
      tma_stages &= ~(1u << s);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
      return;
    }
    uint32_t bad = 0;
    int nload = 0;
    int phys[BPU];
#pragma unroll
    for (int i = 0; i < BPU; ++i) {
      phys[i] = next_phys[i];
      if (ic.k * BPU + i >= ic.r.nblk) {
        phys[i] = -2;  // past the sequence: nothing to load
        continue;
      }
      if (phys[i] < 0 || phys[i] >= p.num_blocks) {
        atomicOr(p.err, kErrBadBlock);
        bad |= 1u << i;
        phys[i] = 0;  // a valid address; every position of this block is masked
      }
      ++nload;
    }
    const uint32_t smask = ((1u << BPU) - 1u) << (s * BPU);
    bad_stages = (bad_stages & ~smask) | (bad << (s * BPU));
    tma_stages |= 1u << s;
    info[s] = StageInfo{iu, ic.b, ic.h, ic.k, iu_end, iseg};
    const uint32_t dst = smem_addr(ring + s * G::kStageBytes);
    mbar_arrive_expect_tx(bar, nload * G::kBlockBytes + stall);
    if (stall) stall_bar = bar;
    stall = 0;
#pragma unroll
    for (int i = 0; i < BPU; ++i) {
      if (phys[i] == -2) continue;
      const int tile = phys[i] * p.n_kv_heads + ic.h;
      const uint32_t bdst = dst + i * G::kBlockBytes;
      if constexpr (FP4) {
        bulk_load(bdst, p.pool + static_cast<int64_t>(tile) * G::kBlockBytes, G::kBlockBytes, bar);
      } else {
#pragma unroll
        for (int bx = 0; bx < G::kBoxes; ++bx)
          tma_load_4d(bdst + bx * G::kBoxBytes, &tmap, bar, bx * 64, 0, 0, tile);
      }
    }
    // step to the next unit: within the segment, or the next chunk
    if (++iu < iu_end) {
      if (++ic.k == ic.r.nunit) {
        ic.k = 0;
        if (++ic.h == p.n_kv_heads) {
          ic.h = 0;
          do {
            ++ic.b;
            ic.r = seq_from_ctx<BS, BPU>(s_ctx[ic.b], p.window);
          } while (ic.r.nunit == 0);
        }
      }
      table_entries(ic, next_phys);
    } else {
      next_segment();
    }
  };
  // A static share's first unit and its table entries come from inputs of
  // the call alone, so they are resolved before the wait below.
  if (lane == 0 && worker < sp.Ps) {
    iu = static_cast<int>(static_cast<int64_t>(sp.Ts) * worker / sp.Ps);
    iu_end = static_cast<int>(static_cast<int64_t>(sp.Ts) * (worker + 1) / sp.Ps);
    iseg = worker;
    ic = locate(iu);
    table_entries(ic, next_phys);
  }

  // Launched after the KV write of the same step as its programmatic
  // dependent, this kernel has built its table and found its first units
  // while the write ran (the write lets it start only once every kernel
  // before the write has completed, so the tables and lengths are final);
  // the pool and the ticket counter are touched only after the write has
  // completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("fence.proxy.async;" ::: "memory");
  if (lane == 0) {
    if (worker >= sp.Ps) next_segment();
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issue(s);
  }

  // ---- compute side
  const int n = lane >> 2;  // query head (within the group) this lane feeds, and token row
  const int j = lane & 3;
  const int g = p.group;
  const int trow_k = (lane & 7) + (((lane >> 3) & 1) << 3);  // ldmatrix row of K
  const int swz = lane & 7;                                    // swizzle phase of that row

  uint32_t qf[G::kSteps][2];
  float score_scale = p.scale_log2;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float acc[G::kSteps][4];
  int prev_u = -2;
  bool timed_out = false;
  int it = 0;
  for (;; ++it) {
    const int s = it % STAGES;
    const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), (it / STAGES) & 1, p.wait_limit_ns,
                                      p.err, kErrTimeout, kShortWaitNs);
    if (!__all_sync(kFull, ok)) {
      timed_out = true;
      break;
    }
    const StageInfo si = info[s];
    if (si.u < 0) break;
    const SeqRange r = seq_from_ctx<BS, BPU>(s_ctx[si.b], p.window);
    const int64_t row0 = static_cast<int64_t>(si.b) * p.n_q_heads +
                         static_cast<int64_t>(si.h) * p.group_stride;
    if (si.u != prev_u + 1 || si.k == 0) {
      // ---- a new piece of a (b, h) pair: its query fragments, a fresh state
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + row0 * D;
      if constexpr (KIND == kBf16) {
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(qg + n * D);
#pragma unroll
        for (int ks = 0; ks < G::kSteps; ++ks) {
          qf[ks][0] = n < g ? qr[(ks * 16 + 2 * j) >> 1] : 0u;
          qf[ks][1] = n < g ? qr[(ks * 16 + 8 + 2 * j) >> 1] : 0u;
        }
      } else if constexpr (FP4) {
        // f16 operands (the dequantised FP4 keys are exact in f16): scale the
        // group's queries by a power of two that puts the largest below
        // 2^15, which keeps every bf16 query exact, and fold it back into the
        // score scale with the head's K scale.
        float amax = 0.f;
        for (int i = lane; i < g * D; i += 32) amax = fmaxf(amax, fabsf(__bfloat162float(qg[i])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        int e = 0;
        if (amax > 0.f) frexpf(amax, &e);
        const float qs = ldexpf(1.f, 15 - e);  // amax * qs < 2^15
        score_scale = p.scale_log2 * p.k_scale[si.h] * ldexpf(1.f, e - 15);
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(qg + n * D);
#pragma unroll
        for (int ks = 0; ks < G::kSteps; ++ks) {
          const uint32_t w0 = n < g ? qr[(ks * 16 + 2 * j) >> 1] : 0u;
          const uint32_t w1 = n < g ? qr[(ks * 16 + 8 + 2 * j) >> 1] : 0u;
          qf[ks][0] = pack_f16x2(bf16_lo(w0) * qs, bf16_hi(w0) * qs);
          qf[ks][1] = pack_f16x2(bf16_lo(w1) * qs, bf16_hi(w1) * qs);
        }
      } else {
        // E4M3 operands: scale the group's queries by an exact power of two
        // below 256, split each into a high code and the code of its
        // remainder (~8 significant bits together), and fold the power back
        // into the score scale.  qf[c] holds the high codes of k-step c
        // (dims 32c + 4j.. and 32c + 16 + 4j..), qf[4 + c] the remainders.
        float amax = 0.f;
        for (int i = lane; i < g * D; i += 32) amax = fmaxf(amax, fabsf(__bfloat162float(qg[i])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        int e = 0;
        if (amax > 0.f) frexpf(amax, &e);
        const float qs = ldexpf(1.f, 8 - e);  // amax * qs < 256
        score_scale = p.scale_log2 * p.k_scale[si.h] * ldexpf(1.f, e - 8);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v4[4] = {0.f, 0.f, 0.f, 0.f};
            if (n < g) {
#pragma unroll
              for (int e4 = 0; e4 < 4; ++e4)
                v4[e4] = __bfloat162float(qg[n * D + 32 * c + 16 * half + 4 * j + e4]) * qs;
            }
            const uint32_t h01 = f32x2_to_e4m3x2(v4[0], v4[1]);
            const uint32_t h23 = f32x2_to_e4m3x2(v4[2], v4[3]);
            const __half2 b01 = u32_as_half2(e4m3x2_to_f16x2(h01));
            const __half2 b23 = u32_as_half2(e4m3x2_to_f16x2(h23));
            const uint32_t l01 = f32x2_to_e4m3x2(v4[0] - __low2float(b01), v4[1] - __high2float(b01));
            const uint32_t l23 = f32x2_to_e4m3x2(v4[2] - __low2float(b23), v4[3] - __high2float(b23));
            qf[c][half] = h01 | (h23 << 16);
            qf[D / 32 + c][half] = l01 | (l23 << 16);
          }
        }
      }
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
#pragma unroll
      for (int i = 0; i < G::kSteps; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    }
    prev_u = si.u;

    const uint32_t bad_blocks = __shfl_sync(kFull, bad_stages, 0) >> (s * BPU);
    const int unit_t0 = (r.first_blk + si.k * BPU) * BS;  // first token of the unit
    const uint32_t st = smem_addr(ring + s * G::kStageBytes);

#pragma unroll
    for (int sub = 0; sub < G::kSub; ++sub) {
      const int t0 = unit_t0 + 16 * sub;
      const bool blk_ok = ((bad_blocks >> (sub / G::kSubPerBlock)) & 1u) == 0;
      // a sub-tile wholly outside [lo, ctx) (before the window, or past the
      // sequence's end in its last unit) is skipped; the warp agrees on it
      const bool live = t0 < r.ctx && t0 + 16 > r.lo;
      const bool full = blk_ok && t0 >= r.lo && t0 + 16 <= r.ctx;
      auto tok_ok = [&](int tr) {
        const int pos = t0 + tr;
        return full || (blk_ok && pos >= r.lo && pos < r.ctx);
      };
      const uint32_t sk = st + G::k_off(sub), sv = st + G::v_off(sub);

      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t vf[G::kSteps][4];
      uint4 vq[4];  // FP4: this lane's V code words (m-tiles 0-3, 4-7) and V scale words
      if (live) {
        // ---- S^T = K Q^T : rows = 16 tokens, cols = 8 query heads
        if constexpr (FP4) {
          // Dequantise the lane's K fragments exactly into f16: code value
          // times its E4M3 block scale (a k-step's 16 dimensions are one
          // scale group).  Tokens n and n + 8; the record puts each lane's
          // bytes in one 16-byte vector per token.
          const uint32_t rec = st + G::rec_off(sub);
          const uint4 kc0 = lds128(rec + 16 * lane), kc1 = lds128(rec + 512 + 16 * lane);
          const uint2 kq0 = lds64(rec + 2048 + 8 * n), kq1 = lds64(rec + 2048 + 64 + 8 * n);
          const uint32_t kw[2][4] = {{kc0.x, kc0.y, kc0.z, kc0.w}, {kc1.x, kc1.y, kc1.z, kc1.w}};
          const uint32_t kq[2][2] = {{kq0.x, kq0.y}, {kq1.x, kq1.y}};
          // scale pairs (groups 2i, 2i+1) of tokens n and n + 8
          uint32_t ksp[2][4];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            e4m3x4_to_f16x2(kq[t][0], ksp[t][0], ksp[t][1]);
            e4m3x4_to_f16x2(kq[t][1], ksp[t][2], ksp[t][3]);
          }
#pragma unroll
          for (int i = 0; i < G::kSteps / 2; ++i) {
            // word i of a token's chunk: k-steps 2i and 2i+1, each the bytes
            // of dims (2j, 2j+1) and (2j+8, 2j+9)
            uint32_t c0[4], c1[4];
            fp4x8_to_f16x2(kw[0][i], c0);
            fp4x8_to_f16x2(kw[1][i], c1);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int ks = 2 * i + e;
              const __half2 p0 = u32_as_half2(ksp[0][i]), p1 = u32_as_half2(ksp[1][i]);
              const __half2 s0 = e ? __high2half2(p0) : __low2half2(p0);
              const __half2 s1 = e ? __high2half2(p1) : __low2half2(p1);
              const uint32_t a0 = half2_as_u32(__hmul2(u32_as_half2(c0[2 * e]), s0));
              const uint32_t a2 = half2_as_u32(__hmul2(u32_as_half2(c0[2 * e + 1]), s0));
              const uint32_t a1 = half2_as_u32(__hmul2(u32_as_half2(c1[2 * e]), s1));
              const uint32_t a3 = half2_as_u32(__hmul2(u32_as_half2(c1[2 * e + 1]), s1));
              if (ks & 1)
                mma_f16(sb, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
              else
                mma_f16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            }
          }
          // V code and scale words, kept raw until the product
          vq[0] = lds128(rec + 1024 + 16 * lane);
          vq[1] = lds128(rec + 1536 + 16 * lane);
          vq[2] = lds128(rec + 2176 + 32 * j);
          vq[3] = lds128(rec + 2176 + 32 * j + 16);
        } else if constexpr (!FP8) {
#pragma unroll
          for (int ks = 0; ks < G::kSteps; ++ks) {
            const int chunk = ((ks & 3) << 1) + (lane >> 4);
            const uint32_t addr = sk + (ks >> 2) * G::kBoxBytes + trow_k * G::kRowBytes +
                                  ((chunk ^ swz) << 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(addr, a0, a1, a2, a3);
            if (ks & 1)
              mma_bf16(sb, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            else
              mma_bf16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
          }
        } else {
          // K codes go to the tensor cores as they are: k-step c covers dims
          // 32c..32c+31 (swizzled chunks 2c and 2c+1 of each K row)
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            const int chunk = 2 * c + (lane >> 4);
            const uint32_t addr = sk + trow_k * G::kRowBytes + ((chunk ^ swz) << 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(addr, a0, a1, a2, a3);
            mma_e4m3(sa, a0, a1, a2, a3, qf[c][0], qf[c][1]);
            mma_e4m3(sb, a0, a1, a2, a3, qf[D / 32 + c][0], qf[D / 32 + c][1]);
          }
        }
        // ---- V fragments to registers
        if constexpr (FP4) {
        } else if constexpr (!FP8) {
          const int trow_v = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
          for (int mt = 0; mt < G::kSteps; ++mt) {
            const int chunk = ((mt & 3) << 1) + ((lane >> 3) & 1);
            const uint32_t addr = sv + (mt >> 2) * G::kBoxBytes + trow_v * G::kRowBytes +
                                  ((chunk ^ swz) << 4);
            ldsm_x4_trans(addr, vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3]);
          }
        } else {
          // transposed V: dimension d's 16 codes are chunk d % 8 of smem row
          // d / 8 (swizzled); ldmatrix i takes dims 32i..32i+31, i.e. rows g
          // and g+8 of m-tiles 2i and 2i+1
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            const int row = 4 * i + (lane >> 3);
            ldsm_x4(sv + row * G::kRowBytes + (((lane & 7) ^ (row & 7)) << 4), vf[i][0], vf[i][1],
                    vf[i][2], vf[i][3]);
          }
        }
      }
      // after the unit's last reads from the stage, refill it at once so the
      // ring stays full while the softmax and V^T P^T run
      if (sub == G::kSub - 1) {
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async_smem();  // this stage's reads happen before the next copy lands
          issue(s);
        }
      }
      if (!live) continue;

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
      const float p0 = fast_exp2(s0 - mu0), p1 = fast_exp2(s1 - mu1);
      const float p2 = fast_exp2(s2 - mu0), p3 = fast_exp2(s3 - mu1);
      // rescale the running state only when some running maximum moved
      if (__any_sync(kFull, mn0 != m_run[0] || mn1 != m_run[1])) {
        const float al0 = fast_exp2(m_run[0] - mu0), al1 = fast_exp2(m_run[1] - mu1);
        l_run[0] *= al0;
        l_run[1] *= al1;
#pragma unroll
        for (int i = 0; i < G::kSteps; ++i) {
          acc[i][0] *= al0;
          acc[i][1] *= al1;
          acc[i][2] *= al0;
          acc[i][3] *= al1;
        }
      }
      l_run[0] += p0 + p2;
      l_run[1] += p1 + p3;
      m_run[0] = mn0;
      m_run[1] = mn1;

      // ---- O^T += V^T P^T : rows = head_dim, cols = 8 query heads, k = 16 tokens
      if constexpr (FP4) {
        // P in f16 (11 significant bits).  The A fragments are the V codes as
        // exact f16 values; each token's E4M3 group scale of m-tile mt goes
        // into its P entry instead (word mt of the lane's scale words holds
        // tokens 2j, 2j+1, 2j+8, 2j+9: the tokens of b0 and b1), so a
        // fragment costs two conversions of codes and none of scales.
        // Masked tokens get a zero scale: stale slots contribute nothing.
        const __half2 b0 = u32_as_half2(movmatrix_trans(pack_f16x2(p0, p1)));
        const __half2 b1 = u32_as_half2(movmatrix_trans(pack_f16x2(p2, p3)));
        const uint32_t vw[8] = {vq[0].x, vq[0].y, vq[0].z, vq[0].w, vq[1].x, vq[1].y, vq[1].z, vq[1].w};
        uint32_t sw[8] = {vq[2].x, vq[2].y, vq[2].z, vq[2].w, vq[3].x, vq[3].y, vq[3].z, vq[3].w};
        if (!full) {
          const uint32_t m = (tok_ok(2 * j) ? 0x000000ffu : 0u) | (tok_ok(2 * j + 1) ? 0x0000ff00u : 0u) |
                             (tok_ok(2 * j + 8) ? 0x00ff0000u : 0u) | (tok_ok(2 * j + 9) ? 0xff000000u : 0u);
#pragma unroll
          for (int mt = 0; mt < G::kSteps; ++mt) sw[mt] &= m;
        }
#pragma unroll
        for (int mt = 0; mt < G::kSteps; ++mt) {
          uint32_t slo, shi, a[4];
          e4m3x4_to_f16x2(sw[mt], slo, shi);
          fp4x8_to_f16x2(vw[mt], a);
          const uint32_t bb0 = half2_as_u32(__hmul2(b0, u32_as_half2(slo)));
          const uint32_t bb1 = half2_as_u32(__hmul2(b1, u32_as_half2(shi)));
          // bytes 0..3: tokens (2j, 2j+1) / (2j+8, 2j+9) at dim n, then dim n + 8
          mma_f16(acc[mt], a[0], a[2], a[1], a[3], bb0, bb1);
        }
      } else if constexpr (!FP8) {
        const uint32_t x01 = pack_bf16x2(p0, p1), x23 = pack_bf16x2(p2, p3);
        const uint32_t y01 = pack_bf16x2(p0 - bf16_lo(x01), p1 - bf16_hi(x01));
        const uint32_t y23 = pack_bf16x2(p2 - bf16_lo(x23), p3 - bf16_hi(x23));
        const uint32_t bh0 = movmatrix_trans(x01), bh1 = movmatrix_trans(x23);
        const uint32_t bl0 = movmatrix_trans(y01), bl1 = movmatrix_trans(y23);
        // this lane's V^T fragment covers tokens 2j, 2j+1 (a0, a1) and 2j+8, 2j+9 (a2, a3)
        if (!full) {
          const uint32_t mlo = (tok_ok(2 * j) ? 0x0000ffffu : 0u) | (tok_ok(2 * j + 1) ? 0xffff0000u : 0u);
          const uint32_t mhi = (tok_ok(2 * j + 8) ? 0x0000ffffu : 0u) | (tok_ok(2 * j + 9) ? 0xffff0000u : 0u);
#pragma unroll
          for (int mt = 0; mt < G::kSteps; ++mt) {
            vf[mt][0] &= mlo;
            vf[mt][1] &= mlo;
            vf[mt][2] &= mhi;
            vf[mt][3] &= mhi;
          }
        }
#pragma unroll
        for (int mt = 0; mt < G::kSteps; ++mt) {
          mma_bf16(acc[mt], vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3], bh0, bh1);
          mma_bf16(acc[mt], vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3], bl0, bl1);
        }
      } else {
        // P^T as E4M3 codes of 256 p: after the transpose this lane holds head
        // n at tokens 2j, 2j+1 (tX) and 2j+8, 2j+9 (tY) -- the tokens the
        // transposed V tile keeps at codes 4j..4j+3 of every row.  k 0..15 of
        // the product take the high codes, k 16..31 the codes of the
        // remainders against the same V codes, so P keeps ~8 bits.
        const uint32_t tX = movmatrix_trans(pack_f16x2(p0 * 256.f, p1 * 256.f));
        const uint32_t tY = movmatrix_trans(pack_f16x2(p2 * 256.f, p3 * 256.f));
        const uint32_t bhi = f16x2x2_to_e4m3x4(tX, tY);
        uint32_t dX, dY;
        e4m3x4_to_f16x2(bhi, dX, dY);
        const uint32_t blo = f16x2x2_to_e4m3x4(hsub2_bits(tX, dX), hsub2_bits(tY, dY));
        if (!full) {
          const uint32_t vmask = (tok_ok(2 * j) ? 0x000000ffu : 0u) | (tok_ok(2 * j + 1) ? 0x0000ff00u : 0u) |
                                 (tok_ok(2 * j + 8) ? 0x00ff0000u : 0u) | (tok_ok(2 * j + 9) ? 0xff000000u : 0u);
#pragma unroll
          for (int i = 0; i < D / 32; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) vf[i][e] &= vmask;
        }
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          mma_e4m3(acc[2 * i], vf[i][0], vf[i][1], vf[i][0], vf[i][1], bhi, blo);
          mma_e4m3(acc[2 * i + 1], vf[i][2], vf[i][3], vf[i][2], vf[i][3], bhi, blo);
        }
      }
    }

    // ---- end of this piece of pair (b, h): write it out
    if (si.k == r.nunit - 1 || si.u + 1 == si.seg_end) {
      float l0 = l_run[0], l1 = l_run[1];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, o);
        l1 += __shfl_xor_sync(kFull, l1, o);
      }
      const int pair = si.b * p.n_kv_heads + si.h;
      const int pair_start = si.u - si.k;
      const int first_seg = sp.seg_of(pair_start);
      const int cnt = sp.seg_of(pair_start + r.nunit - 1) - first_seg + 1;
      const bool whole = cnt == 1;
      // FP8: P was 256 p; FP4: the head's V scale is not in the dequantised values
      const float vsc = FP8 ? p.v_scale[si.h] * (1.f / 256.f) : FP4 ? p.v_scale[si.h] : 1.f;
      const int h0 = 2 * j, h1 = 2 * j + 1;  // query heads of this lane's columns
      const float f0 = whole ? (l0 > 0.f ? vsc / l0 : 0.f) : vsc;
      const float f1 = whole ? (l1 > 0.f ? vsc / l1 : 0.f) : vsc;
      float* dst = whole ? p.out + row0 * D
                         : p.part_o + (static_cast<int64_t>(si.seg) + pair) * g * D;
#pragma unroll
      for (int i = 0; i < G::kSteps; ++i) {
        const int da = 16 * i + n, db = da + 8;  // head_dim rows of entries {0,1}, {2,3}
        if (h0 < g) {
          dst[h0 * D + da] = acc[i][0] * f0;
          dst[h0 * D + db] = acc[i][2] * f0;
        }
        if (h1 < g) {
          dst[h1 * D + da] = acc[i][1] * f1;
          dst[h1 * D + db] = acc[i][3] * f1;
        }
      }
      if (!whole && n == 0) {
        float* ml = p.part_ml + (static_cast<int64_t>(si.seg) + pair) * g * 2;
        if (h0 < g) {
          ml[2 * h0] = m_run[0];
          ml[2 * h0 + 1] = l0;
        }
        if (h1 < g) {
          ml[2 * h1] = m_run[1];
          ml[2 * h1 + 1] = l1;
        }
      }
      if (lane == 0 && si.seg == first_seg) p.pair_meta[pair] = make_int2(first_seg, cnt);
    }
  }

  if (timed_out && lane == 0) {
    // leave no copy in flight: wait (bounded) for every stage holding one.
    // Under the test stall the missing bytes are supplied here, so that the
    // stalled stage completes once its real copy has landed.
    atomicOr(p.err, kErrTimeout);
    if (stall_bar) mbar_complete_tx(stall_bar, p.stall_tx);
    for (int k = it; k < it + STAGES; ++k)
      if ((tma_stages >> (k % STAGES)) & 1u &&
          !mbar_wait_bounded(smem_addr(&bars[k % STAGES]), (k / STAGES) & 1, p.wait_limit_ns,
                             p.err, kErrTimeout, kShortWaitNs))
        atomicOr(p.err, kErrDrainTimeout);
  }
}

// Merge the partials of pairs cut between segments:
//   out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k,  M = max_k m_k.
// One CTA per (sequence, KV head) pair; thread = (k-slice, query head, 4
// columns).  Each k-slice folds every KS-th partial with a running maximum,
// then slice 0 combines the slices in shared memory.  Launched as a
// programmatic dependent of the decode kernel: everything before
// griddepcontrol.wait reads only inputs of the call.
template <int D, int BS>
__global__ void __launch_bounds__(kReduceThreads, kReduceCtas) paged_decode_reduce_kernel(
    const DecodeParams p) {
  constexpr int kGroups = D / 4;  // float4 column groups per head
  constexpr int kInFlight = PKV_RIF;  // partials loaded at once per thread
  __shared__ float4 s_o[kReduceThreads];
  __shared__ float2 s_ml[kReduceThreads];
  const int pair = blockIdx.x;
  const int b = pair / p.n_kv_heads;
  const int h = pair - b * p.n_kv_heads;
  const int g = p.group;
  const int lanes = g * kGroups;  // threads of one k-slice
  const int KS = blockDim.x / lanes;
  const int ks = threadIdx.x / lanes;
  const int idx = threadIdx.x - ks * lanes;
  const int hd = idx / kGroups;
  const int c4 = idx - hd * kGroups;
  int32_t ctx = p.context_lens[b];
  if (!ctx_ok<BS>(p, ctx)) ctx = 0;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The decode is complete: the next kernel on the stream may be scheduled
  // (the next step's KV write, a programmatic dependent, waits for this grid
  // to complete before it reads or writes anything).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (ctx == 0) return;  // nothing attended: zeroed by the decode kernel
  const int2 meta = p.pair_meta[pair];
  const int cnt = meta.y;
  if (cnt <= 1) return;  // finished by the one warp that held it
  const int64_t slot0 = static_cast<int64_t>(meta.x) + pair;
  // a pair whose record was never written (its first segment's warp gave up
  // on a wait) can hold anything: stay inside the workspace
  if (meta.x < 0 || slot0 + cnt > p.num_slots) return;
  // partial k of this thread's head: ml at pm + 2 g k, its columns at po + g D k
  const float* pm = p.part_ml + (slot0 * g + hd) * 2;
  const float* po = p.part_o + (slot0 * g + hd) * D + 4 * c4;
  const int sm = 2 * g, so = g * D;
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = ks; k0 < cnt; k0 += kInFlight * KS) {
    float2 ml[kInFlight];
    float4 o[kInFlight];
#pragma unroll
    for (int i = 0; i < kInFlight; ++i) {
      const int k = k0 + i * KS;
      const int kk = k < cnt ? k : k0;
      ml[i] = *reinterpret_cast<const float2*>(pm + kk * sm);
      o[i] = *reinterpret_cast<const float4*>(po + kk * so);
      if (k >= cnt) ml[i].x = -INFINITY;
    }
    float mb = M;
#pragma unroll
    for (int i = 0; i < kInFlight; ++i) mb = fmaxf(mb, ml[i].x);
    if (mb == -INFINITY) continue;
    const float a = fast_exp2(M - mb);  // rescale what was folded so far
    L *= a;
    O.x *= a;
    O.y *= a;
    O.z *= a;
    O.w *= a;
#pragma unroll
    for (int i = 0; i < kInFlight; ++i) {
      const float f = fast_exp2(ml[i].x - mb);
      L += f * ml[i].y;
      O.x += f * o[i].x;
      O.y += f * o[i].y;
      O.z += f * o[i].z;
      O.w += f * o[i].w;
    }
    M = mb;
  }
  s_o[threadIdx.x] = O;
  s_ml[threadIdx.x] = make_float2(M, L);
  __syncthreads();
  if (ks != 0) return;
  float Mt = -INFINITY;
  for (int q = 0; q < KS; ++q) Mt = fmaxf(Mt, s_ml[q * lanes + idx].x);
  float Lt = 0.f;
  float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
  if (Mt != -INFINITY) {
    for (int q = 0; q < KS; ++q) {
      const float2 ml = s_ml[q * lanes + idx];
      const float4 o = s_o[q * lanes + idx];
      const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - Mt);
      Lt += f * ml.y;
      Ot.x += f * o.x;
      Ot.y += f * o.y;
      Ot.z += f * o.z;
      Ot.w += f * o.w;
    }
  }
  const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
  float4* dst = reinterpret_cast<float4*>(
      p.out + (static_cast<int64_t>(b) * p.n_q_heads + static_cast<int64_t>(h) * p.group_stride + hd) * D) + c4;
  *dst = make_float4(Ot.x * inv, Ot.y * inv, Ot.z * inv, Ot.w * inv);
}

template <int D, int KIND, int BS, int BPU, int NW, int STAGES>
struct Variant {
  static constexpr int kSmem = Smem<D, KIND, BS, BPU, NW, STAGES>::kBytes;
  static constexpr int kWarps = NW;
  static constexpr int kBlocksPerUnit = BPU;

  // Opt in to the dynamic shared memory once; report resident CTAs per SM.
  static int ctas_per_sm() {
    static int ctas = -1;
    if (ctas < 0) {
      auto kernel = paged_decode_kernel<D, KIND, BS, BPU, NW, STAGES>;
      int n = 0;
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, NW * 32, kSmem) !=
              cudaSuccess) {
        cudaGetLastError();
        return 1;
      }
      ctas = n > 0 ? n : 1;
    }
    return ctas;
  }

  static cudaError_t launch(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream,
                            bool dependent) {
    ctas_per_sm();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.num_workers + NW - 1) / NW);
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, KIND, BS, BPU, NW, STAGES>, pool->tmap,
                              p);
  }
};

// Warps per CTA and ring stages per warp of each variant.
#ifndef PKV_BF16_WARPS
#define PKV_BF16_WARPS 4
#endif
#ifndef PKV_BF16_STAGES
#define PKV_BF16_STAGES 2
#endif
#ifndef PKV_FP8_WARPS
#define PKV_FP8_WARPS 4
#endif
#ifndef PKV_FP8_STAGES
#define PKV_FP8_STAGES 2
#endif
#ifndef PKV_FP8_BPU
#define PKV_FP8_BPU 2
#endif
#ifndef PKV_BS32_WARPS
#define PKV_BS32_WARPS 2
#endif

// 16-token blocks: bf16 stages one block per unit; FP8 stages two, so a unit
// carries 32 tokens (8 KB) and the per-unit work is spread over twice the
// bytes.  32-token blocks: one block per unit (two 16-token sub-tiles).
#ifndef PKV_BF16_BPU
#define PKV_BF16_BPU 1
#endif
using Bf16D128 = Variant<128, kBf16, 16, PKV_BF16_BPU, PKV_BF16_WARPS, PKV_BF16_STAGES>;
using Bf16D64 = Variant<64, kBf16, 16, 1, 4, 4>;
using Fp8D128 = Variant<128, kFp8, 16, PKV_FP8_BPU, PKV_FP8_WARPS, PKV_FP8_STAGES>;
using Bf16D128B32 = Variant<128, kBf16, 32, 1, PKV_BS32_WARPS, 2>;
using Bf16D64B32 = Variant<64, kBf16, 32, 1, 4, 2>;
using Fp8D128B32 = Variant<128, kFp8, 32, 1, PKV_FP8_WARPS, 2>;
// FP4 records are 2304 bytes per 16 tokens: units of three 16-token blocks
// (one 32-token block) keep ~14 KB of ring per warp, as the other variants.
#ifndef PKV_FP4_BPU
#define PKV_FP4_BPU 3
#define PKV_FP4_STAGES 2
#endif
using Fp4D128 = Variant<128, kFp4, 16, PKV_FP4_BPU, 4, PKV_FP4_STAGES>;
using Fp4D128B32 = Variant<128, kFp4, 32, 1, 4, 3>;

// Call f with the variant type the pool uses.
template <typename F>
auto with_variant(const kv_pool* pool, F&& f) {
  if (pool->block_size == 32) {
    if (pool->dtype == KV_FP4_E2M1) return f(Fp4D128B32{});
    if (pool->dtype == KV_FP8_E4M3) return f(Fp8D128B32{});
    if (pool->head_dim == 128) return f(Bf16D128B32{});
    return f(Bf16D64B32{});
  }
  if (pool->dtype == KV_FP4_E2M1) return f(Fp4D128{});
  if (pool->dtype == KV_FP8_E4M3) return f(Fp8D128{});
  if (pool->head_dim == 128) return f(Bf16D128{});
  return f(Bf16D64{});
}

}  // namespace

int decode_warps_per_cta(const kv_pool* pool) {
  return with_variant(pool, [](auto v) { return decltype(v)::kWarps; });
}

int decode_ctas_per_sm(const kv_pool* pool) {
  return with_variant(pool, [](auto v) { return decltype(v)::ctas_per_sm(); });
}

int decode_blocks_per_unit(const kv_pool* pool) {
  return with_variant(pool, [](auto v) { return decltype(v)::kBlocksPerUnit; });
}

// Upper bound of Split::Nc over every launch of at most `max_units` units:
// each region's chunk count grows with the dynamic part, and the last region
// also takes what the rounding of the first two left over.
int64_t decode_max_chunks(int64_t max_units) {
  const int64_t td = max_units * kDynNum / kDynDen;
  const int64_t r0 = td * kPlan.pct[0] / 100 / kC0 * kC0;
  const int64_t r1 = td * kPlan.pct[1] / 100 / kC1 * kC1;
  const int64_t r2 = td * kPlan.pct[2] / 100 / kC2 * kC2;
  const int64_t rest = td * (100 - kPlan.pct[0] - kPlan.pct[1] - kPlan.pct[2]) / 100 + kC0 + kC1 + kC2;
  return r0 / kC0 + r1 / kC1 + r2 / kC2 + (rest + kC3 - 1) / kC3 + 1;
}

cudaError_t launch_decode(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream,
                          bool dependent) {
  return with_variant(pool, [&](auto v) { return decltype(v)::launch(pool, p, stream, dependent); });
}

cudaError_t launch_reduce(const kv_pool* pool, const DecodeParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.n_kv_heads);
  const int lanes = p.group * pool->head_dim / 4;  // threads per k-slice
  cfg.blockDim = dim3(lanes * std::max(1, std::min(4, kReduceThreads / lanes)));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pool->block_size == 32) {
    if (pool->head_dim == 128) return cudaLaunchKernelEx(&cfg, paged_decode_reduce_kernel<128, 32>, p);
    return cudaLaunchKernelEx(&cfg, paged_decode_reduce_kernel<64, 32>, p);
  }
  if (pool->head_dim == 128) return cudaLaunchKernelEx(&cfg, paged_decode_reduce_kernel<128, 16>, p);
  return cudaLaunchKernelEx(&cfg, paged_decode_reduce_kernel<64, 16>, p);
}

}  // namespace pkv
