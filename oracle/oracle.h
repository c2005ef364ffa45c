/*
 * Oracle for the paged KV cache decode path -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of what the pages describe:
 *   - the bf16, FP8-E4M3 and FP4-E2M1 number formats, from their definitions;
 *   - the paged KV write (each new token's K/V scattered to its slot);
 *   - paged decode attention, evaluated in fp64 by walking the block table;
 *   - the host block pool: LRU free queue, ref_cnt, touch, reverse-order
 *     free, chained SHA-256 block hashes, lazy eviction, preemption.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the bench
 * may load this library.  It shares no source, header, table or helper with
 * the CUDA library, and its pool uses the pages' own block shape
 * [2, block_size, num_kv_heads, head_dim] rather than the GPU pool layout.
 *
 * Return codes: 0 ok, 1 invalid argument, 2 out of blocks, 5 bad block id.
 */
#ifndef PAGEDKV_ORACLE_H
#define PAGEDKV_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ------------------------------------------------------ */
double  oracle_bf16_to_double(uint16_t bits);
double  oracle_e4m3_to_double(uint8_t code);
uint8_t oracle_e4m3_from_float(float x);                 /* RNE, saturate to +-448 */
uint8_t oracle_e4m3_quantize(uint16_t bf16_bits, float scale); /* e4m3(float(x)/scale) */
double  oracle_e2m1_to_double(uint8_t code);             /* low 4 bits: S.EE.M */
uint8_t oracle_e2m1_from_float(float x);                 /* RNE, saturate to +-6, NaN -> +0 */
/* FP4 row quantization (NVFP4 arrangement): E4M3 scale per 16 elements under
 * the per-head fp32 scale G; codes[n] (one E2M1 code per byte), scales[n/16]. */
void    oracle_fp4_quantize_row(const uint16_t* x_bf16, int32_t n, float G,
                                uint8_t* codes, uint8_t* scales);

/* ---- host KV pool in the pages' block shape ----------------------------- */
/* element (blk, kv, off, h, d) lives at ((((blk*2+kv)*BS+off)*Hkv+h)*D+d)  */
/* FP4 block scale (blk, kv, off, h, j) at ((((blk*2+kv)*BS+off)*Hkv+h)*(D/16)+j) */
typedef struct oracle_pool oracle_pool;
oracle_pool* oracle_pool_create(int64_t num_blocks, int32_t block_size,
                                int32_t n_kv_heads, int32_t head_dim,
                                int32_t dtype /* 0 bf16, 1 e4m3, 2 e2m1 + block scales */);
void     oracle_pool_destroy(oracle_pool* p);
void*    oracle_pool_data(oracle_pool* p);
uint64_t oracle_pool_bytes(const oracle_pool* p);
void*    oracle_pool_block_scales(oracle_pool* p);       /* FP4 only, else NULL */
int      oracle_pool_set_scales(oracle_pool* p, const float* k_scale, const float* v_scale);

/* Copy every K and V row of block pairs[2i] into block pairs[2i+1] (both
 * must be in [0, num_blocks)); pairs are applied in order.  1 on a bad id
 * (nothing copied). */
int oracle_pool_copy_blocks(oracle_pool* p, const int32_t* pairs, int64_t n);

/* k, v: [T, Hkv, D] bf16 bits; slot < 0 = padded token (skipped). */
int oracle_kv_write(oracle_pool* p, const uint16_t* k, const uint16_t* v,
                    const int64_t* slot_mapping, int64_t num_tokens);

/* q: [B, Hq, D] bf16 bits; block_tables: [B, max_blocks_per_seq];
 * out: [B, Hq, D] float.  Only the sequences listed in `seqs` are computed
 * (all of them when seqs == NULL).  window <= 0 disables the sliding window. */
int oracle_paged_decode(const oracle_pool* p, const uint16_t* q, int32_t n_q_heads,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, int32_t batch,
                        double scale, int32_t window,
                        const int32_t* seqs, int32_t n_seqs, float* out);

/* Paged prefill / extend attention: q is [T, Hq, D] bf16 bits with the new
 * tokens of sequence b at rows cu_q_lens[b] .. cu_q_lens[b+1]-1 (the last
 * positions of its context_lens[b] tokens, already written to the pool);
 * each attends causally to positions [lo, pos] of its sequence.
 * out: [T, Hq, D] float. */
int oracle_paged_prefill(const oracle_pool* p, const uint16_t* q, int32_t n_q_heads,
                         const int32_t* cu_q_lens, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         int32_t batch, double scale, int32_t window, float* out);

/* ---- SHA-256 (FIPS 180-4) ------------------------------------------------ */
void oracle_sha256(const uint8_t* msg, uint64_t len, uint8_t digest[32]);

/* ---- block pool bookkeeping --------------------------------------------- */
typedef struct oracle_alloc oracle_alloc;
oracle_alloc* oracle_alloc_create(int32_t num_blocks, int32_t block_size);
void    oracle_alloc_destroy(oracle_alloc* a);
/* Admit a request.  tokens may be NULL (content unknown: no prefix lookup and
 * no hashes).  salt goes into block 0's hash only; extra into every block's. */
int     oracle_alloc_admit(oracle_alloc* a, int64_t req_id, const int32_t* tokens,
                           int64_t num_tokens, const uint8_t* salt, int32_t salt_len,
                           const uint8_t* extra, int32_t extra_len,
                           int64_t* cached_tokens);
/* Grow a request by n tokens (tokens may be NULL). All-or-nothing.  When the
 * first new token falls into a partly filled last block that other requests
 * share (ref_cnt > 1), that block is copied on write first: a fresh block
 * replaces it in this request's table, the pair (old, new) joins the pending
 * copies, and the old block loses one reference. */
int     oracle_alloc_append(oracle_alloc* a, int64_t req_id, const int32_t* tokens, int64_t n);
/* Fork: `child` shares every block of `parent` (one more reference each) and
 * takes its token count, token ids, hashes, salt and extra keys; it counts as
 * the newest admission.  1 if parent is unknown or child exists. */
int     oracle_alloc_fork(oracle_alloc* a, int64_t parent, int64_t child);
/* Pending copy-on-write pairs (src, dst), oldest first, into pairs[2*cap];
 * returns their number; take != 0 clears the list. */
int64_t oracle_alloc_copies(oracle_alloc* a, int32_t* pairs, int64_t cap, int32_t take);
int     oracle_alloc_free(oracle_alloc* a, int64_t req_id);
int     oracle_alloc_preempt_newest(oracle_alloc* a, int64_t* req_id);
int     oracle_alloc_table(const oracle_alloc* a, int64_t req_id, int32_t* out,
                           int64_t cap, int64_t* n);
int64_t oracle_alloc_num_tokens(const oracle_alloc* a, int64_t req_id);
int32_t oracle_alloc_num_free(const oracle_alloc* a);
int32_t oracle_alloc_free_queue(const oracle_alloc* a, int32_t* out, int32_t cap);
int     oracle_alloc_block_info(const oracle_alloc* a, int32_t id, int32_t* ref_cnt,
                                int32_t* has_hash, uint8_t hash[32]);
int32_t oracle_alloc_lookup(const oracle_alloc* a, const uint8_t hash[32]);
int32_t oracle_alloc_map_size(const oracle_alloc* a);
int32_t oracle_alloc_map_entries(const oracle_alloc* a, uint8_t* hashes, int32_t* ids, int32_t cap);
/* stats: [0] prefix queries (blocks looked up), [1] prefix hits (blocks),
 *        [2] evictions, [3] preemptions, [4] running requests */
void    oracle_alloc_stats(const oracle_alloc* a, int64_t out[5]);

#ifdef __cplusplus
}
#endif
#endif
