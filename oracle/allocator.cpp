// Oracle: host-side block pool bookkeeping.  TEST INFRASTRUCTURE ONLY.
//
// Restated from the pages (by title and section):
//  * "PagedAttention" (zhangchitc.github.io/posts/paged-attention):
//    - "What a physical block looks like": a KVCacheBlock has block_id,
//      ref_cnt, the block hash and prev/next links of the doubly linked
//      free_block_queue; blocks are taken from the queue and returned to it.
//    - "Two lookup structures": BlockHashToBlockMap (one global map from hash
//      to block) and req_to_blocks (each request's blocks, in order).
//    - "Walking through two requests" / "When a request finishes" / "Picking
//      freed blocks back up": a hit adds one to ref_cnt (a block with ref_cnt
//      0 is pulled out of the free queue first); misses take blocks from the
//      front of the queue; a freed block keeps its hash and its map entry; the
//      entry is dropped only when the block is handed out again.  Freed blocks
//      go to the end of the queue.
//    - "Block hash": hash of block n = H(hash of block n-1, tokens of block n).
//  * "How the block pool manages KV memory":
//    - "Finding a prefix again": only full blocks are hashed; the hash also
//      covers LoRA adapter, images and an optional per-request salt; lookup
//      stops at the first miss.
//    - "Eviction": the head of the free list is the block unused the longest.
//  * "The memory behind the next token" (deepmox chapter 2):
//    - "Sharing requires explicit ownership": touch removes a ref_cnt-0 block
//      from the free queue before incrementing; a finished request's blocks
//      are released in reverse order.
//    - "How vLLM recognizes a reusable prefix": append-only block tables may
//      hold a duplicate of a cached hash for a while; even a full prompt hit
//      must leave the last token to be computed; cache_salt is mixed into the
//      first block's identity.
//  * "Why the KV cache is a pool of 16-token blocks", section "When memory
//    runs out": with no free block, the newest running request is preempted
//    and all of its blocks are freed.
//  * "Optimizing KV Cache Memory Management in vLLM with PagedAttention and
//    Dynamic Block Allocation", sections "Copy-on-Write (CoW) for Parallel
//    Sampling and Prefix Caching" and "Simulating vLLM's Block Manager in
//    Python": a fork maps the child's logical blocks to the parent's physical
//    blocks and raises their reference counts; a sequence about to write a
//    token into a block whose count is above one gets a new block, the old
//    block's contents are copied into it on the device, the old block loses a
//    reference and the table entry is switched to the new block.
//
// Readings where the pages leave details open: the hash input of block i is
// parent_hash (32 bytes, all zero for block 0) || the block's token ids as
// little-endian int32 || extra keys || (block 0 only) the salt; the map keeps
// the first block registered under a hash (insert if absent); a full-hit cap
// of floor((len-1)/BS) blocks; admit and append are all-or-nothing.

#include "oracle.h"

#include <algorithm>
#include <array>
#include <map>
#include <string>
#include <vector>

namespace {

using Hash = std::array<uint8_t, 32>;

struct Block {
  int32_t id = 0;
  int32_t ref_cnt = 0;
  bool has_hash = false;
  Hash hash{};
  int32_t prev_free = -1;  // links of the doubly linked free queue
  int32_t next_free = -1;
  bool in_free = false;
};

struct Request {
  std::vector<int32_t> blocks;  // req_to_blocks entry: logical -> physical
  std::vector<int32_t> tokens;  // token ids (empty when content is unknown)
  bool content_known = false;
  std::string salt, extra;
  std::vector<Hash> hashes;     // chain hashes of its full blocks
  int64_t num_tokens = 0;
  uint64_t admit_order = 0;
};

}  // namespace

struct oracle_alloc {
  int32_t nb = 0, bs = 0;
  std::vector<Block> blocks;
  int32_t head = -1, tail = -1, nfree = 0;
  std::map<Hash, int32_t> hash_to_block;
  std::map<int64_t, Request> reqs;
  std::vector<std::pair<int32_t, int32_t>> copies;  // pending copy-on-write (src, dst)
  uint64_t admit_counter = 0;
  int64_t queries = 0, hits = 0, evictions = 0, preemptions = 0;
};

namespace {

void queue_unlink(oracle_alloc* a, int32_t id) {
  Block& b = a->blocks[id];
  if (b.prev_free >= 0) a->blocks[b.prev_free].next_free = b.next_free; else a->head = b.next_free;
  if (b.next_free >= 0) a->blocks[b.next_free].prev_free = b.prev_free; else a->tail = b.prev_free;
  b.prev_free = b.next_free = -1;
  b.in_free = false;
  a->nfree--;
}

void queue_push_back(oracle_alloc* a, int32_t id) {
  Block& b = a->blocks[id];
  b.prev_free = a->tail;
  b.next_free = -1;
  if (a->tail >= 0) a->blocks[a->tail].next_free = id; else a->head = id;
  a->tail = id;
  b.in_free = true;
  a->nfree++;
}

// Hash of one full block: SHA-256(parent || tokens (int32 LE) || extra || salt).
Hash block_hash(const Hash& parent, const int32_t* toks, int32_t bs, const std::string& extra,
                const std::string* salt) {
  std::vector<uint8_t> buf(parent.begin(), parent.end());
  for (int32_t i = 0; i < bs; ++i) {
    uint32_t u = static_cast<uint32_t>(toks[i]);
    for (int k = 0; k < 4; ++k) buf.push_back(uint8_t(u >> (8 * k)));
  }
  buf.insert(buf.end(), extra.begin(), extra.end());
  if (salt) buf.insert(buf.end(), salt->begin(), salt->end());
  Hash h;
  oracle_sha256(buf.data(), buf.size(), h.data());
  return h;
}

// Touch: a hit block with no users leaves the free queue before its count rises.
void touch(oracle_alloc* a, int32_t id) {
  Block& b = a->blocks[id];
  if (b.ref_cnt == 0 && b.in_free) queue_unlink(a, id);
  b.ref_cnt++;
}

// Take the block at the head of the free queue.  Its old hash entry (if the
// map still points at it) is dropped only now: lazy eviction.
int32_t pop_free(oracle_alloc* a) {
  int32_t id = a->head;
  queue_unlink(a, id);
  Block& b = a->blocks[id];
  if (b.has_hash) {
    auto it = a->hash_to_block.find(b.hash);
    if (it != a->hash_to_block.end() && it->second == id) a->hash_to_block.erase(it);
    b.has_hash = false;
    a->evictions++;
  }
  b.ref_cnt = 1;
  return id;
}

void register_hash(oracle_alloc* a, int32_t id, const Hash& h) {
  Block& b = a->blocks[id];
  b.hash = h;
  b.has_hash = true;
  a->hash_to_block.emplace(h, id);  // insert if absent: duplicates stay unmapped
}

// Release every block of a request, last logical block first.
void release(oracle_alloc* a, Request& r) {
  for (auto it = r.blocks.rbegin(); it != r.blocks.rend(); ++it) {
    Block& b = a->blocks[*it];
    b.ref_cnt--;
    if (b.ref_cnt == 0) queue_push_back(a, *it);
  }
  r.blocks.clear();
}

int64_t blocks_for(int64_t tokens, int32_t bs) { return (tokens + bs - 1) / bs; }

}  // namespace

extern "C" oracle_alloc* oracle_alloc_create(int32_t num_blocks, int32_t block_size) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  oracle_alloc* a = new oracle_alloc;
  a->nb = num_blocks;
  a->bs = block_size;
  a->blocks.resize(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) {
    a->blocks[i].id = i;
    queue_push_back(a, i);  // initial queue in block id order
  }
  return a;
}

extern "C" void oracle_alloc_destroy(oracle_alloc* a) { delete a; }

extern "C" int oracle_alloc_admit(oracle_alloc* a, int64_t req_id, const int32_t* tokens,
                                  int64_t num_tokens, const uint8_t* salt, int32_t salt_len,
                                  const uint8_t* extra, int32_t extra_len,
                                  int64_t* cached_tokens) {
  if (num_tokens < 0 || a->reqs.count(req_id)) return 1;
  Request r;
  r.num_tokens = num_tokens;
  r.content_known = tokens != nullptr;
  if (salt && salt_len > 0) r.salt.assign(reinterpret_cast<const char*>(salt), salt_len);
  if (extra && extra_len > 0) r.extra.assign(reinterpret_cast<const char*>(extra), extra_len);
  const int32_t bs = a->bs;
  const int64_t nblocks = blocks_for(num_tokens, bs);

  // Chain hashes of the full prompt blocks, then the longest run of hits.
  std::vector<int32_t> hit_blocks;
  if (r.content_known) {
    r.tokens.assign(tokens, tokens + num_tokens);
    Hash parent{};
    const int64_t nfull = num_tokens / bs;
    for (int64_t i = 0; i < nfull; ++i) {
      Hash h = block_hash(parent, tokens + i * bs, bs, r.extra, i == 0 ? &r.salt : nullptr);
      r.hashes.push_back(h);
      parent = h;
    }
    const int64_t cap = num_tokens > 0 ? (num_tokens - 1) / bs : 0;  // last token is computed
    const int64_t lookups = std::min<int64_t>(nfull, cap);
    for (int64_t i = 0; i < lookups; ++i) {
      a->queries++;
      auto it = a->hash_to_block.find(r.hashes[i]);
      if (it == a->hash_to_block.end()) break;
      hit_blocks.push_back(it->second);
      a->hits++;
    }
  }

  // Capacity: hit blocks with no users sit in the free queue and leave it.
  int64_t idle_hits = 0;
  for (int32_t id : hit_blocks) idle_hits += (a->blocks[id].ref_cnt == 0) ? 1 : 0;
  const int64_t need = nblocks - static_cast<int64_t>(hit_blocks.size());
  if (a->nfree - idle_hits < need) return 2;

  for (int32_t id : hit_blocks) {
    touch(a, id);
    r.blocks.push_back(id);
  }
  for (int64_t i = static_cast<int64_t>(hit_blocks.size()); i < nblocks; ++i) {
    int32_t id = pop_free(a);
    r.blocks.push_back(id);
    if (r.content_known && i < static_cast<int64_t>(r.hashes.size())) register_hash(a, id, r.hashes[i]);
  }
  r.admit_order = ++a->admit_counter;
  if (cached_tokens) *cached_tokens = static_cast<int64_t>(hit_blocks.size()) * bs;
  a->reqs.emplace(req_id, std::move(r));
  return 0;
}

extern "C" int oracle_alloc_append(oracle_alloc* a, int64_t req_id, const int32_t* tokens,
                                   int64_t n) {
  auto it = a->reqs.find(req_id);
  if (it == a->reqs.end() || n < 0) return 1;
  Request& r = it->second;
  const int32_t bs = a->bs;
  // The first new token lands in a partly filled last block shared with
  // another request: that block must be copied before it is written.
  const bool cow = n > 0 && r.num_tokens % bs != 0 && a->blocks[r.blocks.back()].ref_cnt > 1;
  const int64_t need = blocks_for(r.num_tokens + n, bs) - blocks_for(r.num_tokens, bs) + (cow ? 1 : 0);
  if (a->nfree < need) return 2;
  if (cow) {
    const int32_t old_id = r.blocks.back();
    const int32_t new_id = pop_free(a);
    a->copies.emplace_back(old_id, new_id);
    a->blocks[old_id].ref_cnt--;  // still >= 1: the other sharers keep it
    r.blocks.back() = new_id;
  }
  if (!tokens) r.content_known = false;  // content unknown from here on: no more hashes
  for (int64_t i = 0; i < n; ++i) {
    // The sequence reached a block boundary: it needs a new block.
    if (r.num_tokens % bs == 0) r.blocks.push_back(pop_free(a));
    if (r.content_known) r.tokens.push_back(tokens[i]);
    r.num_tokens++;
    // A block that just filled gets its chain hash.
    if (r.content_known && r.num_tokens % bs == 0) {
      const int64_t bi = r.num_tokens / bs - 1;
      if (static_cast<int64_t>(r.hashes.size()) == bi) {
        Hash parent = bi ? r.hashes[bi - 1] : Hash{};
        Hash h = block_hash(parent, r.tokens.data() + bi * bs, bs, r.extra,
                            bi == 0 ? &r.salt : nullptr);
        r.hashes.push_back(h);
        register_hash(a, r.blocks[bi], h);
      }
    }
  }
  return 0;
}

extern "C" int oracle_alloc_fork(oracle_alloc* a, int64_t parent, int64_t child) {
  auto it = a->reqs.find(parent);
  if (it == a->reqs.end() || a->reqs.count(child)) return 1;
  Request r = it->second;  // same tokens, hashes, salt and extra keys
  for (int32_t id : r.blocks) touch(a, id);
  r.admit_order = ++a->admit_counter;
  a->reqs.emplace(child, std::move(r));
  return 0;
}

extern "C" int64_t oracle_alloc_copies(oracle_alloc* a, int32_t* pairs, int64_t cap,
                                       int32_t take) {
  const int64_t n = static_cast<int64_t>(a->copies.size());
  for (int64_t i = 0; i < n && i < cap; ++i) {
    pairs[2 * i] = a->copies[i].first;
    pairs[2 * i + 1] = a->copies[i].second;
  }
  if (take) a->copies.clear();
  return n;
}

extern "C" int oracle_alloc_free(oracle_alloc* a, int64_t req_id) {
  auto it = a->reqs.find(req_id);
  if (it == a->reqs.end()) return 1;
  release(a, it->second);
  a->reqs.erase(it);
  return 0;
}

extern "C" int oracle_alloc_preempt_newest(oracle_alloc* a, int64_t* req_id) {
  auto newest = a->reqs.end();
  for (auto it = a->reqs.begin(); it != a->reqs.end(); ++it)
    if (newest == a->reqs.end() || it->second.admit_order > newest->second.admit_order) newest = it;
  if (newest == a->reqs.end()) return 2;
  if (req_id) *req_id = newest->first;
  release(a, newest->second);
  a->reqs.erase(newest);
  a->preemptions++;
  return 0;
}

extern "C" int oracle_alloc_table(const oracle_alloc* a, int64_t req_id, int32_t* out, int64_t cap,
                                  int64_t* n) {
  auto it = a->reqs.find(req_id);
  if (it == a->reqs.end()) return 1;
  const auto& bl = it->second.blocks;
  if (n) *n = static_cast<int64_t>(bl.size());
  for (int64_t i = 0; i < static_cast<int64_t>(bl.size()) && i < cap; ++i) out[i] = bl[i];
  return 0;
}

extern "C" int64_t oracle_alloc_num_tokens(const oracle_alloc* a, int64_t req_id) {
  auto it = a->reqs.find(req_id);
  return it == a->reqs.end() ? -1 : it->second.num_tokens;
}

extern "C" int32_t oracle_alloc_num_free(const oracle_alloc* a) { return a->nfree; }

extern "C" int32_t oracle_alloc_free_queue(const oracle_alloc* a, int32_t* out, int32_t cap) {
  int32_t n = 0;
  for (int32_t id = a->head; id >= 0; id = a->blocks[id].next_free) {
    if (n < cap) out[n] = id;
    ++n;
  }
  return n;
}

extern "C" int oracle_alloc_block_info(const oracle_alloc* a, int32_t id, int32_t* ref_cnt,
                                       int32_t* has_hash, uint8_t hash[32]) {
  if (id < 0 || id >= a->nb) return 1;
  const Block& b = a->blocks[id];
  if (ref_cnt) *ref_cnt = b.ref_cnt;
  if (has_hash) *has_hash = b.has_hash ? 1 : 0;
  if (hash) std::copy(b.hash.begin(), b.hash.end(), hash);
  return 0;
}

extern "C" int32_t oracle_alloc_lookup(const oracle_alloc* a, const uint8_t hash[32]) {
  Hash h;
  std::copy(hash, hash + 32, h.begin());
  auto it = a->hash_to_block.find(h);
  return it == a->hash_to_block.end() ? -1 : it->second;
}

extern "C" int32_t oracle_alloc_map_size(const oracle_alloc* a) {
  return static_cast<int32_t>(a->hash_to_block.size());
}

extern "C" int32_t oracle_alloc_map_entries(const oracle_alloc* a, uint8_t* hashes, int32_t* ids,
                                            int32_t cap) {
  int32_t n = 0;
  for (const auto& kv : a->hash_to_block) {
    if (n < cap) {
      std::copy(kv.first.begin(), kv.first.end(), hashes + 32 * n);
      ids[n] = kv.second;
    }
    ++n;
  }
  return n;
}

extern "C" void oracle_alloc_stats(const oracle_alloc* a, int64_t out[5]) {
  out[0] = a->queries;
  out[1] = a->hits;
  out[2] = a->evictions;
  out[3] = a->preemptions;
  out[4] = static_cast<int64_t>(a->reqs.size());
}
