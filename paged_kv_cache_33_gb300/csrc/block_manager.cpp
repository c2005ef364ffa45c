// Host block manager of one KV block pool (C ABI in include/kv_block_manager.h).
//
// The bookkeeping the pages assign to the block pool, made fast enough to run
// every scheduler step next to the GPU:
//  * "PagedAttention" (zhangchitc.github.io/posts/paged-attention), sections
//    "What a physical block looks like", "Two lookup structures", "Walking
//    through two requests", "When a request finishes", "Picking freed blocks
//    back up", "Block hash": per-block reference count, hash and free-queue
//    links; a hash map from block hash to block; touch on a hit; misses from
//    the queue head; frees to the tail in reverse order; lazy eviction of the
//    hash when a cached block is handed out again; chained block hashes.
//  * "How the block pool manages KV memory", "Finding a prefix again": only
//    full blocks are hashed, salt and extra keys enter the hash, lookup stops
//    at the first miss.
//  * "The memory behind the next token", chapter 2, "How vLLM recognizes a
//    reusable prefix": a full hit still computes the prompt's last token.
//  * "Why the KV cache is a pool of 16-token blocks", "When memory runs out":
//    preempt the newest running request.
//  * "Optimizing KV Cache Memory Management in vLLM with PagedAttention and
//    Dynamic Block Allocation", "Copy-on-Write (CoW) for Parallel Sampling and
//    Prefix Caching": forks share blocks; a write into a shared block first
//    moves the writer to a fresh block whose contents the device copies.
//
// Data structures: blocks as parallel arrays with intrusive free-queue links
// (O(1) unlink / push / pop), an unordered map keyed by the 32-byte digest,
// requests in an unordered map holding only what later hashing needs (the
// last chain hash and the tokens of the partly filled block), and an ordered
// set of admission numbers for O(log n) preemption of the newest request.

#include <algorithm>
#include <array>
#include <climits>
#include <cstring>
#include <new>
#include <set>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/kv_block_manager.h"

namespace {

using Digest = std::array<uint8_t, 32>;

// ---------------------------------------------------------------- SHA-256 --
// FIPS 180-4.  The round constants and initial hash value are the leading 32
// fraction bits of the cube roots of the first 64 primes and of the square
// roots of the first 8 primes; they are derived here with exact integer
// roots instead of being tabulated.

uint64_t icbrt(unsigned __int128 n) {  // floor(cbrt(n)), n < 2^110
  uint64_t lo = 0, hi = uint64_t(1) << 37;
  while (hi - lo > 1) {
    const uint64_t mid = lo + (hi - lo) / 2;
    const unsigned __int128 m = mid;
    if (m * m * m <= n) lo = mid; else hi = mid;
  }
  return lo;
}

uint64_t isqrt(unsigned __int128 n) {  // floor(sqrt(n)), n < 2^74
  uint64_t lo = 0, hi = uint64_t(1) << 38;
  while (hi - lo > 1) {
    const uint64_t mid = lo + (hi - lo) / 2;
    const unsigned __int128 m = mid;
    if (m * m <= n) lo = mid; else hi = mid;
  }
  return lo;
}

struct ShaConstants {
  uint32_t k[64];
  uint32_t h0[8];
  ShaConstants() {
    int found = 0;
    for (uint32_t p = 2; found < 64; ++p) {
      bool prime = true;
      for (uint32_t d = 2; d * d <= p; ++d)
        if (p % d == 0) { prime = false; break; }
      if (!prime) continue;
      // floor(cbrt(p) * 2^32) = floor(cbrt(p * 2^96)); keep the fraction bits
      k[found] = static_cast<uint32_t>(icbrt(static_cast<unsigned __int128>(p) << 96));
      if (found < 8) h0[found] = static_cast<uint32_t>(isqrt(static_cast<unsigned __int128>(p) << 64));
      ++found;
    }
  }
};

const ShaConstants& sha_constants() {
  static const ShaConstants c;
  return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

class Sha256 {
 public:
  Sha256() : c_(sha_constants()) { std::memcpy(h_, c_.h0, sizeof h_); }

  void update(const void* data, size_t len) {
    const uint8_t* p = static_cast<const uint8_t*>(data);
    total_ += len;
    while (len > 0) {
      const size_t take = std::min(len, sizeof buf_ - fill_);
      std::memcpy(buf_ + fill_, p, take);
      fill_ += take;
      p += take;
      len -= take;
      if (fill_ == sizeof buf_) {
        compress(buf_);
        fill_ = 0;
      }
    }
  }

  Digest finish() {
    const uint64_t bits = total_ * 8;
    const uint8_t one = 0x80, zero = 0;
    update(&one, 1);
    while (fill_ != 56) update(&zero, 1);
    uint8_t len_be[8];
    for (int i = 0; i < 8; ++i) len_be[i] = static_cast<uint8_t>(bits >> (56 - 8 * i));
    update(len_be, 8);
    Digest d;
    for (int i = 0; i < 8; ++i)
      for (int j = 0; j < 4; ++j) d[4 * i + j] = static_cast<uint8_t>(h_[i] >> (24 - 8 * j));
    return d;
  }

 private:
  void compress(const uint8_t* blk) {
    uint32_t w[64];
    for (int t = 0; t < 16; ++t)
      w[t] = (uint32_t(blk[4 * t]) << 24) | (uint32_t(blk[4 * t + 1]) << 16) |
             (uint32_t(blk[4 * t + 2]) << 8) | uint32_t(blk[4 * t + 3]);
    for (int t = 16; t < 64; ++t) {
      const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
      const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
      w[t] = w[t - 16] + s0 + w[t - 7] + s1;
    }
    uint32_t a = h_[0], b = h_[1], c = h_[2], d = h_[3], e = h_[4], f = h_[5], g = h_[6],
             h = h_[7];
    for (int t = 0; t < 64; ++t) {
      const uint32_t t1 = h + (rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25)) + ((e & f) ^ (~e & g)) +
                          c_.k[t] + w[t];
      const uint32_t t2 = (rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22)) + ((a & b) ^ (a & c) ^ (b & c));
      h = g;
      g = f;
      f = e;
      e = d + t1;
      d = c;
      c = b;
      b = a;
      a = t1 + t2;
    }
    h_[0] += a; h_[1] += b; h_[2] += c; h_[3] += d;
    h_[4] += e; h_[5] += f; h_[6] += g; h_[7] += h;
  }

  const ShaConstants& c_;
  uint32_t h_[8];
  uint8_t buf_[64];
  size_t fill_ = 0;
  uint64_t total_ = 0;
};

struct DigestHash {
  size_t operator()(const Digest& d) const {
    uint64_t x;
    std::memcpy(&x, d.data(), sizeof x);  // a SHA-256 prefix is already uniform
    return static_cast<size_t>(x);
  }
};

// Chain hash of one full block: parent, token ids (int32 little-endian),
// extra keys, then the salt for block 0 only.
Digest block_digest(const Digest& parent, const int32_t* toks, int32_t bs,
                    const std::string& extra, const std::string* salt) {
  Sha256 s;
  s.update(parent.data(), parent.size());
  uint8_t le[4 * 64];
  for (int32_t i = 0; i < bs;) {
    const int32_t n = std::min<int32_t>(64, bs - i);
    for (int32_t j = 0; j < n; ++j) {
      const uint32_t u = static_cast<uint32_t>(toks[i + j]);
      le[4 * j] = static_cast<uint8_t>(u);
      le[4 * j + 1] = static_cast<uint8_t>(u >> 8);
      le[4 * j + 2] = static_cast<uint8_t>(u >> 16);
      le[4 * j + 3] = static_cast<uint8_t>(u >> 24);
    }
    s.update(le, 4 * static_cast<size_t>(n));
    i += n;
  }
  s.update(extra.data(), extra.size());
  if (salt) s.update(salt->data(), salt->size());
  return s.finish();
}

struct Request {
  std::vector<int32_t> blocks;   // logical -> physical
  std::vector<int32_t> partial;  // token ids of the partly filled last block
  Digest last_hash{};            // chain hash of the last hashed block
  int64_t num_hashed = 0;        // leading full blocks hashed so far
  int64_t num_tokens = 0;
  bool content_known = false;
  std::string salt, extra;
  uint64_t order = 0;            // admission (or fork) number
};

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

struct kv_block_manager {
  int32_t nb = 0, bs = 0;
  std::vector<int32_t> ref, prev, next;
  std::vector<uint8_t> queued, hashed;
  std::vector<Digest> hash;
  int32_t head = -1, tail = -1;
  int64_t nfree = 0;
  std::unordered_map<Digest, int32_t, DigestHash> map;
  std::unordered_map<int64_t, Request> reqs;
  std::set<std::pair<uint64_t, int64_t>> by_order;  // (order, request id)
  std::vector<int32_t> copies;                      // pending (src, dst) pairs, flattened
  uint64_t counter = 0;
  kv_bm_stats st{};

  void unlink(int32_t id) {
    const int32_t p = prev[id], n = next[id];
    if (p >= 0) next[p] = n; else head = n;
    if (n >= 0) prev[n] = p; else tail = p;
    prev[id] = next[id] = -1;
    queued[id] = 0;
    --nfree;
  }
  void push_back(int32_t id) {
    prev[id] = tail;
    next[id] = -1;
    if (tail >= 0) next[tail] = id; else head = id;
    tail = id;
    queued[id] = 1;
    ++nfree;
  }
  void touch(int32_t id) {
    if (ref[id] == 0 && queued[id]) unlink(id);
    ++ref[id];
  }
  // Hand out the queue's head; its old hash leaves the map only now.
  int32_t pop() {
    const int32_t id = head;
    unlink(id);
    if (hashed[id]) {
      auto it = map.find(hash[id]);
      if (it != map.end() && it->second == id) map.erase(it);
      hashed[id] = 0;
      ++st.evictions;
    }
    ref[id] = 1;
    return id;
  }
  void set_hash(int32_t id, const Digest& h) {
    hash[id] = h;
    hashed[id] = 1;
    map.emplace(h, id);  // the first block registered under a hash stays
  }
  void release(Request& r) {
    for (auto it = r.blocks.rbegin(); it != r.blocks.rend(); ++it)
      if (--ref[*it] == 0) push_back(*it);
    r.blocks.clear();
  }
};

extern "C" {

kv_status kv_bm_create(int64_t num_blocks, int32_t block_size, kv_block_manager** out) {
  if (!out) return KV_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks <= 0 || num_blocks >= (int64_t(1) << 31) || block_size <= 0)
    return KV_ERR_INVALID_ARG;
  kv_block_manager* m = new (std::nothrow) kv_block_manager;
  if (!m) return KV_ERR_OOM;
  m->nb = static_cast<int32_t>(num_blocks);
  m->bs = block_size;
  m->ref.assign(m->nb, 0);
  m->prev.assign(m->nb, -1);
  m->next.assign(m->nb, -1);
  m->queued.assign(m->nb, 0);
  m->hashed.assign(m->nb, 0);
  m->hash.assign(m->nb, Digest{});
  for (int32_t i = 0; i < m->nb; ++i) m->push_back(i);  // initial queue in id order
  *out = m;
  return KV_OK;
}

kv_status kv_bm_destroy(kv_block_manager* bm) {
  if (!bm) return KV_ERR_INVALID_ARG;
  delete bm;
  return KV_OK;
}

kv_status kv_bm_admit(kv_block_manager* bm, int64_t req_id, const int32_t* tokens,
                      int64_t num_tokens, const uint8_t* salt, int32_t salt_len,
                      const uint8_t* extra, int32_t extra_len, int64_t* cached_tokens) {
  if (!bm || num_tokens < 0 || salt_len < 0 || extra_len < 0 || bm->reqs.count(req_id))
    return KV_ERR_INVALID_ARG;
  const int32_t bs = bm->bs;
  const int64_t nblocks = cdiv(num_tokens, bs);
  Request r;
  r.num_tokens = num_tokens;
  r.content_known = tokens != nullptr;
  if (salt && salt_len > 0) r.salt.assign(reinterpret_cast<const char*>(salt), salt_len);
  if (extra && extra_len > 0) r.extra.assign(reinterpret_cast<const char*>(extra), extra_len);

  // Chain hashes of the full blocks; the longest run of leading hits, leaving
  // at least the last token to be computed.
  std::vector<Digest> digests;
  std::vector<int32_t> hits;
  if (r.content_known) {
    const int64_t nfull = num_tokens / bs;
    digests.reserve(nfull);
    Digest parent{};
    for (int64_t i = 0; i < nfull; ++i) {
      parent = block_digest(parent, tokens + i * bs, bs, r.extra, i == 0 ? &r.salt : nullptr);
      digests.push_back(parent);
    }
    const int64_t cap = num_tokens > 0 ? (num_tokens - 1) / bs : 0;
    const int64_t probes = std::min(nfull, cap);
    for (int64_t i = 0; i < probes; ++i) {
      ++bm->st.prefix_queries;
      auto it = bm->map.find(digests[i]);
      if (it == bm->map.end()) break;
      hits.push_back(it->second);
      ++bm->st.prefix_hits;
    }
  }
  // Hit blocks nobody uses still sit in the free queue and leave it.
  int64_t idle = 0;
  for (int32_t id : hits) idle += bm->ref[id] == 0 ? 1 : 0;
  const int64_t need = nblocks - static_cast<int64_t>(hits.size());
  if (bm->nfree - idle < need) return KV_ERR_OOM;

  r.blocks.reserve(nblocks);
  for (int32_t id : hits) {
    bm->touch(id);
    r.blocks.push_back(id);
  }
  for (int64_t i = static_cast<int64_t>(hits.size()); i < nblocks; ++i) {
    const int32_t id = bm->pop();
    r.blocks.push_back(id);
    if (i < static_cast<int64_t>(digests.size())) bm->set_hash(id, digests[i]);
  }
  if (r.content_known) {
    r.num_hashed = static_cast<int64_t>(digests.size());
    if (!digests.empty()) r.last_hash = digests.back();
    r.partial.assign(tokens + r.num_hashed * bs, tokens + num_tokens);
  }
  r.order = ++bm->counter;
  if (cached_tokens) *cached_tokens = static_cast<int64_t>(hits.size()) * bs;
  bm->by_order.emplace(r.order, req_id);
  bm->reqs.emplace(req_id, std::move(r));
  ++bm->st.running;
  return KV_OK;
}

kv_status kv_bm_append(kv_block_manager* bm, int64_t req_id, const int32_t* tokens, int64_t n) {
  if (!bm || n < 0) return KV_ERR_INVALID_ARG;
  auto it = bm->reqs.find(req_id);
  if (it == bm->reqs.end()) return KV_ERR_INVALID_ARG;
  Request& r = it->second;
  const int32_t bs = bm->bs;
  const bool cow = n > 0 && r.num_tokens % bs != 0 && bm->ref[r.blocks.back()] > 1;
  const int64_t need = cdiv(r.num_tokens + n, bs) - cdiv(r.num_tokens, bs) + (cow ? 1 : 0);
  if (bm->nfree < need) return KV_ERR_OOM;
  if (cow) {
    const int32_t old_id = r.blocks.back();
    const int32_t new_id = bm->pop();
    bm->copies.push_back(old_id);
    bm->copies.push_back(new_id);
    ++bm->st.cow_copies;
    --bm->ref[old_id];  // the other sharers still hold it
    r.blocks.back() = new_id;
  }
  if (!tokens) {
    r.content_known = false;  // no more hashes for this request
    r.partial.clear();
  }
  for (int64_t i = 0; i < n; ++i) {
    if (r.num_tokens % bs == 0) r.blocks.push_back(bm->pop());
    ++r.num_tokens;
    if (!r.content_known) continue;
    r.partial.push_back(tokens[i]);
    if (r.num_tokens % bs == 0) {  // the block just filled: chain its hash
      const int64_t bi = r.num_tokens / bs - 1;
      if (r.num_hashed == bi) {
        r.last_hash = block_digest(bi ? r.last_hash : Digest{}, r.partial.data(), bs, r.extra,
                                   bi == 0 ? &r.salt : nullptr);
        r.num_hashed = bi + 1;
        bm->set_hash(r.blocks[bi], r.last_hash);
      }
      r.partial.clear();
    }
  }
  return KV_OK;
}

kv_status kv_bm_fork(kv_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return KV_ERR_INVALID_ARG;
  auto it = bm->reqs.find(parent);
  if (it == bm->reqs.end() || bm->reqs.count(child)) return KV_ERR_INVALID_ARG;
  Request r = it->second;
  for (int32_t id : r.blocks) bm->touch(id);
  r.order = ++bm->counter;
  bm->by_order.emplace(r.order, child);
  bm->reqs.emplace(child, std::move(r));
  ++bm->st.running;
  return KV_OK;
}

kv_status kv_bm_free(kv_block_manager* bm, int64_t req_id) {
  if (!bm) return KV_ERR_INVALID_ARG;
  auto it = bm->reqs.find(req_id);
  if (it == bm->reqs.end()) return KV_ERR_INVALID_ARG;
  bm->release(it->second);
  bm->by_order.erase({it->second.order, req_id});
  bm->reqs.erase(it);
  --bm->st.running;
  return KV_OK;
}

kv_status kv_bm_preempt_newest(kv_block_manager* bm, int64_t* req_id) {
  if (!bm) return KV_ERR_INVALID_ARG;
  if (bm->by_order.empty()) return KV_ERR_OOM;
  const int64_t id = bm->by_order.rbegin()->second;
  if (req_id) *req_id = id;
  kv_bm_free(bm, id);
  ++bm->st.preemptions;
  return KV_OK;
}

int64_t kv_bm_take_copies(kv_block_manager* bm, int32_t* pairs, int64_t cap) {
  if (!bm) return -1;
  const int64_t n = static_cast<int64_t>(bm->copies.size() / 2);
  if (pairs && cap > 0)
    std::copy(bm->copies.begin(), bm->copies.begin() + 2 * std::min(n, cap), pairs);
  if (n <= cap) bm->copies.clear();
  return n;
}

int64_t kv_bm_pending_copies(const kv_block_manager* bm, int32_t* pairs, int64_t cap) {
  if (!bm) return -1;
  const int64_t n = static_cast<int64_t>(bm->copies.size() / 2);
  if (pairs && cap > 0)
    std::copy(bm->copies.begin(), bm->copies.begin() + 2 * std::min(n, cap), pairs);
  return n;
}

kv_status kv_bm_block_table(const kv_block_manager* bm, int64_t req_id, int32_t* out,
                            int64_t cap, int64_t* n) {
  if (!bm) return KV_ERR_INVALID_ARG;
  auto it = bm->reqs.find(req_id);
  if (it == bm->reqs.end()) return KV_ERR_INVALID_ARG;
  const auto& b = it->second.blocks;
  if (n) *n = static_cast<int64_t>(b.size());
  if (out && cap > 0) std::copy(b.begin(), b.begin() + std::min<int64_t>(cap, b.size()), out);
  return KV_OK;
}

kv_status kv_bm_slot_mapping(const kv_block_manager* bm, int64_t req_id, int64_t first_pos,
                             int64_t n, int64_t* slots) {
  if (!bm || first_pos < 0 || n < 0 || (n > 0 && !slots)) return KV_ERR_INVALID_ARG;
  auto it = bm->reqs.find(req_id);
  if (it == bm->reqs.end() || first_pos + n > it->second.num_tokens) return KV_ERR_INVALID_ARG;
  const auto& b = it->second.blocks;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t pos = first_pos + i;
    slots[i] = static_cast<int64_t>(b[pos / bm->bs]) * bm->bs + pos % bm->bs;
  }
  return KV_OK;
}

kv_status kv_bm_decode_inputs(const kv_block_manager* bm, const int64_t* req_ids, int32_t batch,
                              int32_t max_blocks_per_seq, int32_t* block_tables,
                              int32_t* context_lens, int64_t* slot_mapping) {
  if (!bm || batch < 0 || max_blocks_per_seq <= 0) return KV_ERR_INVALID_ARG;
  if (batch > 0 && (!req_ids || !block_tables || !context_lens || !slot_mapping))
    return KV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < batch; ++i) {
    auto it = bm->reqs.find(req_ids[i]);
    if (it == bm->reqs.end()) return KV_ERR_INVALID_ARG;
    const Request& r = it->second;
    if (r.num_tokens == 0 || r.num_tokens > INT32_MAX ||
        static_cast<int64_t>(r.blocks.size()) > max_blocks_per_seq)
      return KV_ERR_INVALID_ARG;
    int32_t* row = block_tables + static_cast<int64_t>(i) * max_blocks_per_seq;
    std::copy(r.blocks.begin(), r.blocks.end(), row);
    std::fill(row + r.blocks.size(), row + max_blocks_per_seq, -1);
    context_lens[i] = static_cast<int32_t>(r.num_tokens);
    const int64_t last = r.num_tokens - 1;
    slot_mapping[i] = static_cast<int64_t>(r.blocks[last / bm->bs]) * bm->bs + last % bm->bs;
  }
  return KV_OK;
}

int64_t kv_bm_num_tokens(const kv_block_manager* bm, int64_t req_id) {
  if (!bm) return -1;
  auto it = bm->reqs.find(req_id);
  return it == bm->reqs.end() ? -1 : it->second.num_tokens;
}

int64_t kv_bm_num_free(const kv_block_manager* bm) { return bm ? bm->nfree : -1; }

int64_t kv_bm_free_queue(const kv_block_manager* bm, int32_t* out, int64_t cap) {
  if (!bm) return -1;
  int64_t n = 0;
  for (int32_t id = bm->head; id >= 0; id = bm->next[id]) {
    if (out && n < cap) out[n] = id;
    ++n;
  }
  return n;
}

kv_status kv_bm_block_info(const kv_block_manager* bm, int32_t block_id, int32_t* ref_cnt,
                           int32_t* has_hash, uint8_t hash[32]) {
  if (!bm || block_id < 0 || block_id >= bm->nb) return KV_ERR_INVALID_ARG;
  if (ref_cnt) *ref_cnt = bm->ref[block_id];
  if (has_hash) *has_hash = bm->hashed[block_id];
  if (hash) std::memcpy(hash, bm->hash[block_id].data(), 32);
  return KV_OK;
}

int32_t kv_bm_lookup(const kv_block_manager* bm, const uint8_t hash[32]) {
  if (!bm || !hash) return -1;
  Digest d;
  std::memcpy(d.data(), hash, 32);
  auto it = bm->map.find(d);
  return it == bm->map.end() ? -1 : it->second;
}

int64_t kv_bm_map_entries(const kv_block_manager* bm, uint8_t* hashes, int32_t* ids,
                          int64_t cap) {
  if (!bm) return -1;
  int64_t n = 0;
  for (const auto& kv : bm->map) {
    if (n < cap) {
      if (hashes) std::memcpy(hashes + 32 * n, kv.first.data(), 32);
      if (ids) ids[n] = kv.second;
    }
    ++n;
  }
  return n;
}

kv_status kv_bm_get_stats(const kv_block_manager* bm, kv_bm_stats* out) {
  if (!bm || !out) return KV_ERR_INVALID_ARG;
  *out = bm->st;
  return KV_OK;
}

}  // extern "C"
