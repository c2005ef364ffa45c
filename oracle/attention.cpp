// Oracle: number formats, host KV pool, paged KV write and fp64 paged decode
// attention.  TEST INFRASTRUCTURE ONLY -- see oracle.h.
//
// Sources restated here (by page title and section):
//  * "PagedAttention" (zhangchitc.github.io/posts/paged-attention), section
//    "What a physical block looks like": one layer's pool is num_blocks blocks,
//    each a tensor [2, block_size, num_kv_heads, head_dim] holding K and V.
//  * "Optimizing KV Cache Memory Management in vLLM with PagedAttention and
//    Dynamic Block Allocation", section "PagedAttention: Virtual Memory for
//    LLMs": token i of a sequence lives in logical block floor(i/B) at offset
//    i mod B; the block table gives the physical block.  Section "The Decode
//    Phase": the new token's K/V go to the free slot of the last block.
//    Section "The Math of the KV Cache Bottleneck": GQA, fewer KV heads than
//    query heads; 2 bytes per element for BF16, 1 byte for FP8.
//  * "How the block pool manages KV memory", section "Hybrid models get
//    groups": a sliding-window layer needs only the blocks inside the last
//    window.
//  * Number formats: bfloat16 is the upper 16 bits of an IEEE-754 binary32;
//    FP8 E4M3 follows the OCP 8-bit floating point specification (1 sign,
//    4 exponent bits with bias 7, 3 mantissa bits, no infinities, NaN is
//    S.1111.111, largest finite magnitude 448, subnormal step 2^-9).  FP4
//    E2M1 is the element format of the OCP Microscaling (MX) specification
//    (1 sign, 2 exponent bits with bias 1, 1 mantissa bit, no infinities or
//    NaN; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6).
//
// Readings where the pages are silent (each one is listed in the design
// notes): the query attends to positions [lo, ctx) with ctx counting the
// token just written and lo = max(0, ctx - W) when a window W > 0 is given;
// query head hq uses KV head floor(hq / (Hq/Hkv)); a sequence with nothing to
// attend to yields zeros; FP8 values carry one fp32 scale per KV head for K and
// one for V, with value = code * scale and code = E4M3(float(x) / scale).
// FP4 (the pages name it only as a format on its way to becoming standard)
// takes NVIDIA's NVFP4 arrangement: every 16 consecutive head_dim elements of
// a token's K or V row share one E4M3 block scale, on top of the per-KV-head
// fp32 scale G; see oracle_fp4_quantize_row.

#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

// ---------------------------------------------------------------- formats --

extern "C" double oracle_bf16_to_double(uint16_t bits) {
  // bfloat16 keeps the sign, the 8 exponent bits and the top 7 fraction bits
  // of a binary32, so widening is a 16-bit shift.
  uint32_t w = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &w, sizeof f);
  return static_cast<double>(f);
}

extern "C" double oracle_e4m3_to_double(uint8_t code) {
  const int s = code >> 7;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  if (e == 0xF && m == 0x7) return std::nan("");
  // normal: (1 + m/8) * 2^(e-7) = (8 + m) * 2^(e-10); subnormal: m * 2^-9.
  double v = (e == 0) ? std::ldexp(static_cast<double>(m), -9)
                      : std::ldexp(static_cast<double>(8 + m), e - 10);
  return s ? -v : v;
}

// Round a non-negative value to the nearest integer, ties to even.
static long round_half_even(double q) {
  double f = std::floor(q);
  double r = q - f;
  long n = static_cast<long>(f);
  if (r > 0.5) return n + 1;
  if (r < 0.5) return n;
  return (n % 2 == 0) ? n : n + 1;
}

extern "C" uint8_t oracle_e4m3_from_float(float x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(x));
  // Saturating conversion: every magnitude at or above the largest finite
  // value (including infinity) maps to 448 = S.1111.110.
  if (a >= 448.0) return sign | 0x7E;
  if (a < std::ldexp(1.0, -6)) {
    // Subnormal range: integer multiples of 2^-9.  A count of 8 is exactly
    // the smallest normal, whose code is also 8 (exponent 1, mantissa 0).
    long m = round_half_even(a * 512.0);
    return sign | static_cast<uint8_t>(m);
  }
  int e2;
  std::frexp(a, &e2);                 // a = f * 2^e2, f in [0.5, 1)
  int unbiased = e2 - 1;              // a = (1 + frac) * 2^unbiased
  double frac8 = (std::ldexp(a, -unbiased) - 1.0) * 8.0;  // exact
  long m = round_half_even(frac8);
  int biased = unbiased + 7;
  if (m == 8) { m = 0; biased += 1; }
  return sign | static_cast<uint8_t>((biased << 3) | m);
}

extern "C" uint8_t oracle_e4m3_quantize(uint16_t bf16_bits, float scale) {
  uint32_t w = static_cast<uint32_t>(bf16_bits) << 16;
  float x;
  std::memcpy(&x, &w, sizeof x);
  float q = x / scale;  // one IEEE binary32 division, round to nearest even
  return oracle_e4m3_from_float(q);
}

extern "C" double oracle_e2m1_to_double(uint8_t code) {
  const int s = (code >> 3) & 1;
  const int e = (code >> 1) & 0x3;
  const int m = code & 0x1;
  // normal: (1 + m/2) * 2^(e-1) = (2 + m) * 2^(e-2); subnormal (e = 0): m * 0.5.
  double v = (e == 0) ? 0.5 * m : std::ldexp(static_cast<double>(2 + m), e - 2);
  return s ? -v : v;
}

extern "C" uint8_t oracle_e2m1_from_float(float x) {
  if (std::isnan(x)) return 0x0;  // the format has no NaN: a NaN input stores +0
  const uint8_t sign = std::signbit(x) ? 0x8 : 0x0;
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 6.0) return sign | 0x7;  // saturate (infinity included)
  // The representable magnitudes are 0.5 * n for n = 0..4 (codes 0..3 and
  // code 4 = 2.0) and then 3, 4, 6.  Below 2 the grid step is 0.5, from 2 to 4
  // it is 1, from 4 to 6 it is 2; round to nearest, ties to the even code.
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double dc = std::fabs(a - mag[c]), db = std::fabs(a - mag[best]);
    if (dc < db || (dc == db && (c % 2) == 0 && (best % 2) != 0)) best = c;
  }
  return sign | static_cast<uint8_t>(best);
}

// One token's K or V row of n elements (n a multiple of 16) under the per-KV-
// head scale G: for each group of 16 consecutive elements,
//   amax  = max |x| over the group (NaN elements count as 0),
//   sc    = E4M3(amax / (6 * G))            (binary32: t = 6 * G, then amax / t),
//   S     = value(sc) * G                   (one binary32 product),
//   code  = E2M1(x / S)                     (binary32 division), or +0 when S is 0,
// so the stored value of x is e2m1(code) * e4m3(sc) * G.  6 is the largest
// E2M1 magnitude: the group's largest element lands at the top of the grid.
extern "C" void oracle_fp4_quantize_row(const uint16_t* x_bf16, int32_t n, float G,
                                        uint8_t* codes, uint8_t* scales) {
  for (int g0 = 0; g0 < n; g0 += 16) {
    float x[16];
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      const uint32_t w = static_cast<uint32_t>(x_bf16[g0 + i]) << 16;
      std::memcpy(&x[i], &w, sizeof(float));
      if (!std::isnan(x[i])) amax = std::max(amax, std::fabs(x[i]));
    }
    const float t = 6.0f * G;
    const uint8_t sc = oracle_e4m3_from_float(amax / t);
    const float S = static_cast<float>(oracle_e4m3_to_double(sc)) * G;
    scales[g0 / 16] = sc;
    for (int i = 0; i < 16; ++i) codes[g0 + i] = (S == 0.0f) ? 0 : oracle_e2m1_from_float(x[i] / S);
  }
}

// ------------------------------------------------------------------- pool --

struct oracle_pool {
  int64_t nb;
  int32_t bs, hkv, d, dtype;
  std::vector<uint8_t> data;          // bf16 bits, E4M3 codes or E2M1 codes (one per byte)
  std::vector<uint8_t> block_scales;  // FP4: E4M3 scale of every 16 elements of a row
  std::vector<float> k_scale, v_scale;
};

static inline size_t elem_bytes(const oracle_pool* p) { return p->dtype == 0 ? 2 : 1; }

// Element (blk, kv, off, h, d) of the pages' block shape [2, BS, Hkv, D].
static inline uint64_t pool_index(const oracle_pool* p, int64_t blk, int kv, int off, int h,
                                  int d) {
  return ((((static_cast<uint64_t>(blk) * 2 + kv) * p->bs + off) * p->hkv + h) * p->d) + d;
}

extern "C" oracle_pool* oracle_pool_create(int64_t num_blocks, int32_t block_size,
                                           int32_t n_kv_heads, int32_t head_dim, int32_t dtype) {
  if (num_blocks <= 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0) return nullptr;
  if (dtype != 0 && dtype != 1 && dtype != 2) return nullptr;
  if (dtype == 2 && head_dim % 16 != 0) return nullptr;
  oracle_pool* p = new oracle_pool;
  p->nb = num_blocks;
  p->bs = block_size;
  p->hkv = n_kv_heads;
  p->d = head_dim;
  p->dtype = dtype;
  p->data.assign(static_cast<size_t>(num_blocks) * 2 * block_size * n_kv_heads * head_dim *
                     elem_bytes(p),
                 0);
  if (dtype == 2)
    p->block_scales.assign(static_cast<size_t>(num_blocks) * 2 * block_size * n_kv_heads *
                               (head_dim / 16), 0);
  p->k_scale.assign(n_kv_heads, 1.0f);
  p->v_scale.assign(n_kv_heads, 1.0f);
  return p;
}

extern "C" void oracle_pool_destroy(oracle_pool* p) { delete p; }
extern "C" void* oracle_pool_data(oracle_pool* p) { return p->data.data(); }
extern "C" uint64_t oracle_pool_bytes(const oracle_pool* p) { return p->data.size(); }
extern "C" void* oracle_pool_block_scales(oracle_pool* p) {
  return p->block_scales.empty() ? nullptr : p->block_scales.data();
}

// Block scale of row (blk, kv, off, h), elements 16 * j .. 16 * j + 15.
static inline uint64_t scale_index(const oracle_pool* p, int64_t blk, int kv, int off, int h,
                                   int j) {
  return ((((static_cast<uint64_t>(blk) * 2 + kv) * p->bs + off) * p->hkv + h) * (p->d / 16)) + j;
}

extern "C" int oracle_pool_set_scales(oracle_pool* p, const float* k_scale, const float* v_scale) {
  for (int h = 0; h < p->hkv; ++h) {
    if (!(k_scale[h] > 0.0f) || !(v_scale[h] > 0.0f)) return 1;
    p->k_scale[h] = k_scale[h];
    p->v_scale[h] = v_scale[h];
  }
  return 0;
}

// ------------------------------------------------------------ block copy --
// Copy-on-write copies a whole physical block ("Optimizing KV Cache Memory
// Management in vLLM with PagedAttention and Dynamic Block Allocation",
// section "Copy-on-Write (CoW) for Parallel Sampling and Prefix Caching"):
// every element (kv, off, h, d) of block src is copied to block dst.

extern "C" int oracle_pool_copy_blocks(oracle_pool* p, const int32_t* pairs, int64_t n) {
  for (int64_t i = 0; i < 2 * n; ++i)
    if (pairs[i] < 0 || pairs[i] >= p->nb) return 1;
  const size_t eb = elem_bytes(p);
  for (int64_t i = 0; i < n; ++i) {
    const int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    for (int kv = 0; kv < 2; ++kv)
      for (int off = 0; off < p->bs; ++off)
        for (int h = 0; h < p->hkv; ++h)
          for (int d = 0; d < p->d; ++d)
            std::memcpy(&p->data[pool_index(p, dst, kv, off, h, d) * eb],
                        &p->data[pool_index(p, src, kv, off, h, d) * eb], eb);
    if (p->dtype == 2)
      for (int kv = 0; kv < 2; ++kv)
        for (int off = 0; off < p->bs; ++off)
          for (int h = 0; h < p->hkv; ++h)
            for (int j = 0; j < p->d / 16; ++j)
              p->block_scales[scale_index(p, dst, kv, off, h, j)] =
                  p->block_scales[scale_index(p, src, kv, off, h, j)];
  }
  return 0;
}

// ------------------------------------------------------------- KV write --
// Token t with slot s goes to physical block s / BS at offset s mod BS; a
// negative slot marks a padded token and is skipped.

extern "C" int oracle_kv_write(oracle_pool* p, const uint16_t* k, const uint16_t* v,
                               const int64_t* slot_mapping, int64_t num_tokens) {
  const int64_t nslots = p->nb * p->bs;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= nslots) return 5;
    const int64_t blk = s / p->bs;
    const int off = static_cast<int>(s % p->bs);
    for (int kv = 0; kv < 2; ++kv) {
      const uint16_t* src = (kv == 0 ? k : v) + static_cast<uint64_t>(t) * p->hkv * p->d;
      for (int h = 0; h < p->hkv; ++h) {
        const float sc = (kv == 0 ? p->k_scale : p->v_scale)[h];
        if (p->dtype == 2) {
          std::vector<uint8_t> codes(p->d), scales(p->d / 16);
          oracle_fp4_quantize_row(src + h * p->d, p->d, sc, codes.data(), scales.data());
          for (int d = 0; d < p->d; ++d) p->data[pool_index(p, blk, kv, off, h, d)] = codes[d];
          for (int j = 0; j < p->d / 16; ++j)
            p->block_scales[scale_index(p, blk, kv, off, h, j)] = scales[j];
          continue;
        }
        for (int d = 0; d < p->d; ++d) {
          const uint16_t x = src[h * p->d + d];
          const uint64_t idx = pool_index(p, blk, kv, off, h, d);
          if (p->dtype == 0) {
            std::memcpy(&p->data[idx * 2], &x, 2);
          } else {
            p->data[idx] = oracle_e4m3_quantize(x, sc);
          }
        }
      }
    }
  }
  return 0;
}

// Exact value of pool element (blk, kv, off, h, d), scale applied for FP8.
static inline double pool_value(const oracle_pool* p, int64_t blk, int kv, int off, int h, int d) {
  const uint64_t idx = pool_index(p, blk, kv, off, h, d);
  if (p->dtype == 0) {
    uint16_t x;
    std::memcpy(&x, &p->data[idx * 2], 2);
    return oracle_bf16_to_double(x);
  }
  const double sc = static_cast<double>((kv == 0 ? p->k_scale : p->v_scale)[h]);
  if (p->dtype == 2)
    return oracle_e2m1_to_double(p->data[idx]) *
           oracle_e4m3_to_double(p->block_scales[scale_index(p, blk, kv, off, h, d / 16)]) * sc;
  return oracle_e4m3_to_double(p->data[idx]) * sc;
}

// ------------------------------------------------------ decode attention --
// For sequence b and query head hq (KV head h = hq / g):
//   s_t = scale * sum_d q[d] * K_t[d]          for t in [lo, ctx)
//   o   = sum_t softmax(s)_t * V_t
// evaluated in fp64 with the maximum subtracted before exponentiation.

extern "C" int oracle_paged_decode(const oracle_pool* p, const uint16_t* q, int32_t n_q_heads,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t batch, double scale,
                                   int32_t window, const int32_t* seqs, int32_t n_seqs,
                                   float* out) {
  if (n_q_heads <= 0 || n_q_heads % p->hkv != 0) return 1;
  const int g = n_q_heads / p->hkv;
  const int D = p->d;
  const int n = seqs ? n_seqs : batch;
  std::vector<double> qd(static_cast<size_t>(g) * D);
  std::vector<double> kd(D), vd(D);
  for (int i = 0; i < n; ++i) {
    const int b = seqs ? seqs[i] : i;
    if (b < 0 || b >= batch) return 1;
    const int64_t ctx = context_lens[b];
    if (ctx < 0 || ctx > static_cast<int64_t>(max_blocks_per_seq) * p->bs) return 1;
    const int64_t lo = (window > 0) ? std::max<int64_t>(0, ctx - window) : 0;
    const int32_t* table = block_tables + static_cast<int64_t>(b) * max_blocks_per_seq;
    for (int h = 0; h < p->hkv; ++h) {
      // query vectors of the g heads sharing KV head h
      for (int j = 0; j < g; ++j) {
        const uint16_t* qrow = q + (static_cast<int64_t>(b) * n_q_heads + h * g + j) * D;
        for (int d = 0; d < D; ++d) qd[j * D + d] = oracle_bf16_to_double(qrow[d]);
      }
      const int64_t n_att = ctx - lo;
      std::vector<double> s(static_cast<size_t>(g) * (n_att > 0 ? n_att : 0));
      for (int64_t t = lo; t < ctx; ++t) {
        const int64_t blk = table[t / p->bs];
        const int off = static_cast<int>(t % p->bs);
        if (blk < 0 || blk >= p->nb) return 5;
        for (int d = 0; d < D; ++d) kd[d] = pool_value(p, blk, 0, off, h, d);
        for (int j = 0; j < g; ++j) {
          double acc = 0.0;
          for (int d = 0; d < D; ++d) acc += qd[j * D + d] * kd[d];
          s[j * n_att + (t - lo)] = scale * acc;
        }
      }
      if (n_att <= 0) {
        for (int j = 0; j < g; ++j) {
          float* orow = out + (static_cast<int64_t>(b) * n_q_heads + h * g + j) * D;
          for (int d = 0; d < D; ++d) orow[d] = 0.0f;
        }
        continue;
      }
      // softmax weights w[j][t] = exp(s - max) / sum exp(s - max)
      std::vector<double> w(static_cast<size_t>(g) * n_att);
      for (int j = 0; j < g; ++j) {
        double m = -INFINITY;
        for (int64_t t = 0; t < n_att; ++t) m = std::max(m, s[j * n_att + t]);
        double l = 0.0;
        for (int64_t t = 0; t < n_att; ++t) {
          w[j * n_att + t] = std::exp(s[j * n_att + t] - m);
          l += w[j * n_att + t];
        }
        for (int64_t t = 0; t < n_att; ++t) w[j * n_att + t] /= l;
      }
      // o[j] = sum_t w[j][t] * V_t
      std::vector<double> o(static_cast<size_t>(g) * D, 0.0);
      for (int64_t t = lo; t < ctx; ++t) {
        const int64_t blk = table[t / p->bs];
        const int off = static_cast<int>(t % p->bs);
        for (int d = 0; d < D; ++d) vd[d] = pool_value(p, blk, 1, off, h, d);
        for (int j = 0; j < g; ++j) {
          const double wt = w[j * n_att + (t - lo)];
          for (int d = 0; d < D; ++d) o[j * D + d] += wt * vd[d];
        }
      }
      for (int j = 0; j < g; ++j) {
        float* orow = out + (static_cast<int64_t>(b) * n_q_heads + h * g + j) * D;
        for (int d = 0; d < D; ++d) orow[d] = static_cast<float>(o[j * D + d]);
      }
    }
  }
  return 0;
}

// -------------------------------------------------------- paged prefill --
// "Optimizing KV Cache Memory Management in vLLM with PagedAttention and
// Dynamic Block Allocation", "The Prefill Phase": the prompt's key/value
// states are computed in one parallel step and written into the physical
// blocks; with prefix caching ("PagedAttention", "Walking through two
// requests") only the uncached tail of the prompt is computed.  Each new
// query token attends, causally, to every cached or new position up to its
// own: token i of the q_len new tokens of sequence b sits at position
// pos = ctx - q_len + i and attends to [lo, pos], lo = max(0, pos + 1 - W)
// under a window W > 0, else 0 -- the decode rule applied with a context of
// pos + 1.  fp64 throughout; outputs rounded to float.

extern "C" int oracle_paged_prefill(const oracle_pool* p, const uint16_t* q, int32_t n_q_heads,
                                    const int32_t* cu_q_lens, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                                    int32_t batch, double scale, int32_t window, float* out) {
  if (n_q_heads <= 0 || n_q_heads % p->hkv != 0) return 1;
  const int g = n_q_heads / p->hkv;
  const int D = p->d;
  std::vector<double> qd(D), kd(D), vd(D), o(D);
  for (int b = 0; b < batch; ++b) {
    const int64_t q0 = cu_q_lens[b], qn = cu_q_lens[b + 1] - cu_q_lens[b];
    const int64_t ctx = context_lens[b];
    if (qn < 0 || qn > ctx || ctx > static_cast<int64_t>(max_blocks_per_seq) * p->bs) return 1;
    const int32_t* table = block_tables + static_cast<int64_t>(b) * max_blocks_per_seq;
    for (int64_t i = 0; i < qn; ++i) {
      const int64_t pos = ctx - qn + i;
      const int64_t lo = window > 0 ? std::max<int64_t>(0, pos + 1 - window) : 0;
      for (int hq = 0; hq < n_q_heads; ++hq) {
        const int h = hq / g;
        const uint16_t* qrow = q + ((q0 + i) * n_q_heads + hq) * D;
        for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_double(qrow[d]);
        // scores over [lo, pos], then softmax with the maximum subtracted
        std::vector<double> s(pos - lo + 1);
        for (int64_t t = lo; t <= pos; ++t) {
          const int64_t blk = table[t / p->bs];
          if (blk < 0 || blk >= p->nb) return 5;
          const int off = static_cast<int>(t % p->bs);
          double acc = 0.0;
          for (int d = 0; d < D; ++d) acc += qd[d] * pool_value(p, blk, 0, off, h, d);
          s[t - lo] = scale * acc;
        }
        double m = -INFINITY;
        for (double x : s) m = std::max(m, x);
        double l = 0.0;
        for (double& x : s) {
          x = std::exp(x - m);
          l += x;
        }
        std::fill(o.begin(), o.end(), 0.0);
        for (int64_t t = lo; t <= pos; ++t) {
          const int64_t blk = table[t / p->bs];
          const int off = static_cast<int>(t % p->bs);
          const double wt = s[t - lo] / l;
          for (int d = 0; d < D; ++d) o[d] += wt * pool_value(p, blk, 1, off, h, d);
        }
        float* orow = out + ((q0 + i) * n_q_heads + hq) * D;
        for (int d = 0; d < D; ++d) orow[d] = static_cast<float>(o[d]);
      }
    }
  }
  return 0;
}
