/*
 * kv_block_manager.h -- C ABI of the host-side block manager that owns the
 * bookkeeping of one KV block pool: which physical blocks each request
 * holds, the free queue, reference counts, the prefix-cache hash map,
 * preemption, fork and copy-on-write.  It runs on the CPU and emits what the
 * device calls of pagedkv.h consume: block tables, context lengths, slot
 * mappings, and (src, dst) block pairs for paged_kv_copy_blocks.
 *
 * What it follows (sources by page title and section):
 *  - "PagedAttention" (zhangchitc.github.io/posts/paged-attention):
 *      "What a physical block looks like" -- a block has an id, a reference
 *      count, a hash and the links of the doubly linked free queue;
 *      "Two lookup structures" -- one map from block hash to block, and each
 *      request's ordered list of blocks;
 *      "Walking through two requests", "When a request finishes", "Picking
 *      freed blocks back up" -- a cache hit raises the block's count (taking
 *      it out of the free queue first when the count was 0); misses take
 *      blocks from the queue's head; a finished request's blocks go back to
 *      the tail, last block first, and keep their hash until the block is
 *      handed out again;
 *      "Block hash" -- the hash of block n chains the hash of block n-1 with
 *      the block's tokens.
 *  - "How the block pool manages KV memory", "Finding a prefix again" and
 *    "Eviction": only full blocks are hashed; salt and extra keys separate
 *    otherwise equal prefixes; lookup stops at the first miss; the queue's
 *    head is the least recently used block.
 *  - "The memory behind the next token" (chapter 2), "How vLLM recognizes a
 *    reusable prefix": a full hit still leaves the last prompt token to be
 *    computed, so at most floor((len - 1) / block_size) blocks hit.
 *  - "Why the KV cache is a pool of 16-token blocks", "When memory runs out":
 *    the newest running request is preempted and all its blocks freed.
 *  - "Optimizing KV Cache Memory Management in vLLM with PagedAttention and
 *    Dynamic Block Allocation", "Copy-on-Write (CoW) for Parallel Sampling
 *    and Prefix Caching": forked sequences share physical blocks; a write
 *    into a shared block first moves the writer to a fresh copy.
 *
 * Choices where the pages leave details open (the same readings as this
 * project's test oracle): the hash of block i is SHA-256 over the parent hash
 * (32 zero bytes for block 0), the block's token ids as little-endian int32,
 * the extra keys, and (block 0 only) the salt; the map keeps the first block
 * registered under a hash; admit and append change nothing when they fail.
 *
 * Conventions: every pointer is HOST memory owned by the caller.  Calls on
 * one manager are not thread-safe; use one manager per pool and serialise.
 * Status codes are pagedkv.h's kv_status: KV_ERR_OOM means "not enough free
 * blocks" (nothing changed), KV_ERR_INVALID_ARG an unknown or duplicate
 * request id or a bad size.
 */
#ifndef KV_BLOCK_MANAGER_H
#define KV_BLOCK_MANAGER_H

#include <stddef.h>
#include <stdint.h>

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kv_block_manager kv_block_manager; /* opaque */

typedef struct {
  int64_t prefix_queries;  /* full blocks looked up at admission            */
  int64_t prefix_hits;     /* of which found in the hash map                */
  int64_t evictions;       /* cached blocks whose hash was dropped on reuse */
  int64_t preemptions;
  int64_t running;         /* requests currently holding blocks             */
  int64_t cow_copies;      /* copy-on-write pairs produced so far           */
} kv_bm_stats;

/* kv_bm_create -- a manager of num_blocks blocks (ids 0..num_blocks-1, all
 * free, queued in id order) of block_size tokens.  num_blocks in [1, 2^31),
 * block_size >= 1. */
kv_status kv_bm_create(int64_t num_blocks, int32_t block_size, kv_block_manager** out);
kv_status kv_bm_destroy(kv_block_manager* bm);

/* kv_bm_admit -- a new request of num_tokens tokens.  With `tokens` (int32
 * ids) its full blocks are hashed and the longest cached prefix is reused;
 * NULL means the content is unknown (no lookup, no hashes).  salt goes into
 * block 0's hash only, extra into every block's.  *cached_tokens (optional)
 * receives the number of tokens found in the cache (a multiple of
 * block_size); their K/V need not be written again. */
kv_status kv_bm_admit(kv_block_manager* bm, int64_t req_id, const int32_t* tokens,
                      int64_t num_tokens, const uint8_t* salt, int32_t salt_len,
                      const uint8_t* extra, int32_t extra_len, int64_t* cached_tokens);

/* kv_bm_append -- grow a request by n tokens (ids, or NULL when unknown: no
 * hashes from then on).  A block is taken whenever a token starts a new
 * block; a block that fills gets its chain hash.  When the first new token
 * falls into a partly filled block shared with another request, that block
 * is copied on write: the request moves to a fresh block and the pair (old,
 * new) joins the pending copies (kv_bm_take_copies), which the caller must
 * run on the device (paged_kv_copy_blocks) before writing the new tokens. */
kv_status kv_bm_append(kv_block_manager* bm, int64_t req_id, const int32_t* tokens, int64_t n);

/* kv_bm_fork -- request `child` shares every block of `parent` (parallel
 * sampling): one more reference each, same tokens and hashes, admitted as the
 * newest request.  No device work is needed. */
kv_status kv_bm_fork(kv_block_manager* bm, int64_t parent, int64_t child);

/* kv_bm_free -- release a finished request's blocks, last block first. */
kv_status kv_bm_free(kv_block_manager* bm, int64_t req_id);

/* kv_bm_preempt_newest -- free every block of the newest running request
 * (by admission or fork order) and report its id; KV_ERR_OOM if none runs. */
kv_status kv_bm_preempt_newest(kv_block_manager* bm, int64_t* req_id);

/* kv_bm_take_copies -- the pending copy-on-write pairs, oldest first, as
 * pairs[2*i] = src, pairs[2*i+1] = dst.  Returns their number; the list is
 * cleared only when it fit (count <= cap). */
int64_t kv_bm_take_copies(kv_block_manager* bm, int32_t* pairs, int64_t cap);
/* kv_bm_pending_copies -- the same pairs without clearing the list. */
int64_t kv_bm_pending_copies(const kv_block_manager* bm, int32_t* pairs, int64_t cap);

/* kv_bm_block_table -- the request's physical block ids in logical order;
 * *n receives their number, at most cap are written. */
kv_status kv_bm_block_table(const kv_block_manager* bm, int64_t req_id, int32_t* out,
                            int64_t cap, int64_t* n);

/* kv_bm_slot_mapping -- slots of positions [first_pos, first_pos + n) of a
 * request (slot = block * block_size + offset), for paged_kv_write. */
kv_status kv_bm_slot_mapping(const kv_block_manager* bm, int64_t req_id, int64_t first_pos,
                             int64_t n, int64_t* slots);

/* kv_bm_decode_inputs -- the host arrays of one decode step for `batch`
 * requests: block_tables [batch][max_blocks_per_seq] int32 (entries past a
 * request's blocks are -1), context_lens [batch] (token counts) and
 * slot_mapping [batch] int64 (slot of each request's last token, i.e. the
 * token just appended).  KV_ERR_INVALID_ARG if a request is unknown, empty,
 * or holds more than max_blocks_per_seq blocks. */
kv_status kv_bm_decode_inputs(const kv_block_manager* bm, const int64_t* req_ids, int32_t batch,
                              int32_t max_blocks_per_seq, int32_t* block_tables,
                              int32_t* context_lens, int64_t* slot_mapping);

/* Inspection (tests, metrics). */
int64_t kv_bm_num_tokens(const kv_block_manager* bm, int64_t req_id); /* -1 if unknown */
int64_t kv_bm_num_free(const kv_block_manager* bm);
/* the free queue from head (next to be handed out) to tail; returns its length */
int64_t kv_bm_free_queue(const kv_block_manager* bm, int32_t* out, int64_t cap);
kv_status kv_bm_block_info(const kv_block_manager* bm, int32_t block_id, int32_t* ref_cnt,
                           int32_t* has_hash, uint8_t hash[32]);
/* block registered under a hash, or -1 */
int32_t kv_bm_lookup(const kv_block_manager* bm, const uint8_t hash[32]);
/* (hash, block) entries of the map in no particular order; returns their number */
int64_t kv_bm_map_entries(const kv_block_manager* bm, uint8_t* hashes, int32_t* ids, int64_t cap);
kv_status kv_bm_get_stats(const kv_block_manager* bm, kv_bm_stats* out);

#ifdef __cplusplus
}
#endif

#endif /* KV_BLOCK_MANAGER_H */
