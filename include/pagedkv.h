/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV cache decode path.
 *
 * What it computes (sources by page title and section):
 *  - "PagedAttention" (zhangchitc.github.io/posts/paged-attention), "What a
 *    physical block looks like": one preallocated pool per layer, split into
 *    num_blocks physical blocks of block_size tokens, each holding K and V for
 *    every KV head.
 *  - "Optimizing KV Cache Memory Management in vLLM with PagedAttention and
 *    Dynamic Block Allocation":
 *      "PagedAttention: Virtual Memory for LLMs" -- token i of a sequence is in
 *      logical block floor(i / block_size) at offset i mod block_size; the
 *      sequence's block table maps logical to physical blocks; the kernel
 *      resolves K_i and V_i through the table.
 *      "The Decode Phase" -- each step writes the new token's K/V into the
 *      free slot of the last block; one query token per sequence attends.
 *      "The Math of the KV Cache Bottleneck" -- GQA: several query heads per
 *      KV head; BF16 (2 bytes) or FP8 (1 byte) elements.
 *  - "How the block pool manages KV memory", "Hybrid models get groups": a
 *    sliding-window layer needs only the blocks inside the last window.
 *
 * Conventions used by every call:
 *  - Pointers named *_dev, and all tensor arguments, are DEVICE pointers on
 *    the pool's device, owned by the caller, unless stated otherwise.
 *  - The per-step inputs of paged_kv_write, paged_decode_attention,
 *    paged_decode_step and paged_decode_attention_noalloc (k, v,
 *    slot_mapping, q, block_tables, context_lens) may instead be pinned host
 *    memory the device can address (cudaHostAlloc, or cudaHostRegister with
 *    cudaHostRegisterMapped, under unified addressing), like out_dev: the
 *    kernels then read them in place over the host link (NVLink-C2C on
 *    Grace-Blackwell), with no separate copy.  The host must not modify them
 *    until the call's work on `stream` has completed.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls that
 *    take a stream are asynchronous: they validate their host-side arguments,
 *    enqueue kernels and return.  Device-side problems (a table entry outside
 *    [0, num_blocks), a slot outside the pool, a context length above the
 *    bound, a wait that ran out) never trap: the kernel records them in the
 *    pool's error word and skips the offending work; kv_pool_check_status()
 *    reports and clears that word.
 *  - A query attends to positions [lo, ctx) of its sequence, where ctx =
 *    context_lens[b] counts the token written this step and lo = max(0, ctx -
 *    sliding_window) when sliding_window > 0, else 0.  A sequence with ctx = 0
 *    gets an all-zero output row.
 *  - Pool layout (this library's, not the pages'): elements are stored as
 *    [num_blocks][n_kv_heads][2 (K, V)][block_size][head_dim], head_dim
 *    contiguous, so the K tile and the V tile of one (block, KV head) are one
 *    contiguous run (8 KB for bf16, head_dim 128).  The base is 256-byte
 *    aligned; every row is 16-byte aligned.  FP8 pools store each V tile
 *    transposed instead ([head_dim][block_size] codes: one 16-byte row per
 *    dimension), with token t of the block at code position
 *    4 * ((t % 8) / 2) + t % 2 + 2 * (t / 8) of every row; kv_pool_desc's
 *    v_layout says which.
 *  - FP4 pools (KV_FP4_E2M1, head_dim 128) hold E2M1 codes with one E4M3
 *    scale per 16 consecutive elements of a token's K or V row, under the
 *    per-KV-head fp32 scale (NVIDIA's NVFP4 arrangement; the pages name FP4
 *    only as a format coming into use, "Optimizing KV Cache ...",
 *    "Conclusion").  Each 16-token sub-tile of a (block, KV head) is one
 *    2304-byte record, [num_blocks][n_kv_heads][block_size / 16][2304]:
 *    bytes [0, 1024) K codes, [1024, 2048) V codes, [2048, 2176) K scales,
 *    [2176, 2304) V scales, permuted inside each part into the order the
 *    decode kernel's fragments consume (v_layout 2).  Byte offsets, for token
 *    r of the sub-tile and element d (or 16-element group b):
 *      K codes  (r / 8) * 512 + 16 * (4 * (r % 8) + (d % 8) / 2) + 2 * (d / 16)
 *               + (d % 16) / 8, low nibble for even d;
 *      V codes  1024 + 16 * (32 * (d / 64) + 4 * (d % 8) + (r % 8) / 2)
 *               + 4 * ((d / 16) % 4) + r / 8 + 2 * ((d % 16) / 8), low
 *               nibble for even r;
 *      K scales 2048 + 8 * r + b;   V scales 2176 + 32 * ((r % 8) / 2) + 4 * b
 *               + r % 2 + 2 * (r / 8).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = 1,   /* a host-side argument is out of range          */
  KV_ERR_OOM = 2,           /* device memory allocation failed               */
  KV_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed          */
  KV_ERR_UNSUPPORTED = 4,   /* valid, but a shape this build does not cover  */
  KV_ERR_BAD_BLOCK_ID = 5,  /* device: a block-table entry outside the pool  */
  KV_ERR_TIMEOUT = 6,       /* device: a bounded wait on a copy ran out      */
  KV_ERR_BAD_SLOT = 7,      /* device: a slot_mapping entry outside the pool */
  KV_ERR_BAD_CONTEXT = 8,   /* device: context_lens[b] < 0 or above a bound  */
  KV_ERR_DRAIN_TIMEOUT = 9, /* device: a kernel gave up waiting for its own   */
                            /* copies while leaving; treat the context as     */
                            /* suspect (see kv_pool_check_status)             */
  KV_ERR_STALE_EXPONENT_MAP = 10 /* device: a bf16 prefill read a V row the      */
                            /* exponent map has no entry for (written other   */
                            /* than by paged_kv_write; see kv_pool_exponent_map) */
} kv_status;

typedef enum { KV_BF16 = 0, KV_FP8_E4M3 = 1, KV_FP4_E2M1 = 2 } kv_dtype;

typedef struct kv_pool kv_pool; /* opaque */

typedef struct {
  void* base_dev;         /* device address of element (0,0,0,0,0)                  */
  int64_t num_blocks;
  int32_t block_size, n_kv_heads, head_dim;
  int32_t dtype;          /* kv_dtype                                                */
  int64_t strides[5];     /* element strides of [num_blocks][Hkv][2][block_size][D]  */
  uint64_t bytes;         /* total pool bytes                                        */
  int32_t device;         /* CUDA device ordinal the pool lives on                   */
  float* scales_dev;      /* fp8: device float[2 * Hkv], K scales then V scales      */
  int32_t v_layout;       /* 0: V tiles as K ([block_size][D]); 1: transposed (FP8); */
                          /* 2: FP4 sub-tile records (strides not meaningful)        */
} kv_pool_desc;

/*
 * kv_pool_create -- allocate one layer's block pool on the current device.
 *   num_blocks > 0, block_size 16 or 32 (the pages' default and the larger
 *   size "Optimizing KV Cache ...", "Trade-offs of Block Size Tuning",
 *   recommends for very long contexts), n_kv_heads >= 1, head_dim in {64, 128}
 *   (FP8 and FP4: head_dim 128).  The pool owns its memory (cudaMalloc here, cudaFree
 *   in kv_pool_destroy); its contents start undefined.  FP8 scales start at
 *   1.0.  Returns KV_ERR_INVALID_ARG / KV_ERR_UNSUPPORTED for bad shapes,
 *   KV_ERR_OOM when the allocation fails, KV_ERR_CUDA when no device works.
 */
kv_status kv_pool_create(int64_t num_blocks, int32_t block_size, int32_t n_kv_heads,
                         int32_t head_dim, kv_dtype dtype, kv_pool** out);

/* kv_pool_destroy -- synchronise the pool's device, free its memory and the handle. */
kv_status kv_pool_destroy(kv_pool* pool);

/* kv_pool_info -- describe the pool (a test or a framework can view its memory). */
kv_status kv_pool_info(const kv_pool* pool, kv_pool_desc* out);

/*
 * kv_pool_exponent_map -- bf16 pools keep, next to the blocks, one byte per
 * (block, KV head, token): the largest biased exponent field of the token's
 * V row as paged_kv_write stored it (at least 1), 0 for a row no write has
 * recorded.  Layout [num_blocks][n_kv_heads][block_size] uint8, owned by the
 * pool.  paged_kv_write sets it, paged_kv_copy_blocks moves it with the
 * blocks, and paged_prefill_attention reads it to scale its f16 copy of V
 * without a pass over each key tile.  V rows changed by other means (the
 * memory kv_pool_info describes) keep their old entries, or 0: call
 * kv_pool_refresh_exponent_map afterwards.  A prefill that attends to a row
 * whose entry is 0 records KV_ERR_STALE_EXPONENT_MAP (its output is then
 * undefined); an entry below the row's true exponent makes its f16 copy of V
 * overflow.
 *   map_dev, bytes: out; the map's device address and size (NULL and 0 for
 *                   FP8 and FP4 pools).
 */
kv_status kv_pool_exponent_map(const kv_pool* pool, void** map_dev, int64_t* bytes);

/*
 * kv_pool_refresh_exponent_map -- bf16 pools: recompute every entry from the
 * V rows the pool holds (one pass over the pool), ordered on `stream`; a
 * no-op for FP8 and FP4 pools.
 */
kv_status kv_pool_refresh_exponent_map(kv_pool* pool, void* stream);

/*
 * kv_pool_set_scales -- FP8 and FP4 pools: copy per-KV-head scales (device
 * float[Hkv] each) into the pool, ordered on `stream`.  A stored FP8 code c of
 * KV head h stands for c * k_scale[h] (K) or c * v_scale[h] (V); the write
 * quantises x to E4M3(float(x) / scale) with round-to-nearest-even and
 * saturation to +-448.  FP4: with G the head's scale, each 16-element group
 * of a row gets the E4M3 scale sc = E4M3(amax / (6 G)) (amax over the
 * group's non-NaN |x|) and every element the code E2M1(x / S), S = value(sc)
 * * G (+0 when S = 0; NaN stores +0; round to nearest even, saturation to
 * +-6; each step one binary32 operation), standing for e2m1 * value(sc) * G.
 * Scales must be finite and > 0 (not checked on the device).
 */
kv_status kv_pool_set_scales(kv_pool* pool, const float* k_scale_dev, const float* v_scale_dev,
                             void* stream);

/*
 * paged_kv_write -- scatter new tokens' K/V into their slots ("The Decode
 * Phase" / "The Prefill Phase": the kernel writes the computed states into
 * the physical blocks).
 *   k_dev, v_dev:        bf16 [num_tokens][n_kv_heads][head_dim], 16-byte aligned.
 *   slot_mapping_dev:    int64 [num_tokens]; slot = physical_block * block_size
 *                        + offset; slot < 0 marks a padded token (skipped);
 *                        slot >= num_blocks * block_size sets KV_ERR_BAD_SLOT.
 * BF16 pools receive a bit copy, and each written V row's largest exponent
 * field goes into the pool's exponent map (see kv_pool_exponent_map); FP8 and
 * FP4 pools the quantised codes (see kv_pool_set_scales).  Two tokens with the
 * same slot in one call is undefined.  num_tokens == 0 is a no-op.
 */
kv_status paged_kv_write(kv_pool* pool, const void* k_dev, const void* v_dev,
                         const int64_t* slot_mapping_dev, int64_t num_tokens, void* stream);

/*
 * paged_kv_copy_blocks -- copy whole physical blocks inside the pool, for
 * copy-on-write ("Optimizing KV Cache Memory Management in vLLM with
 * PagedAttention and Dynamic Block Allocation", "Copy-on-Write (CoW) for
 * Parallel Sampling and Prefix Caching": the shared block's K/V states are
 * copied device to device into the writer's new block).
 *   pairs:      HOST int32 [num_pairs][2] of (src, dst) block ids, e.g. from
 *               kv_bm_take_copies; every id in [0, num_blocks), else
 *               KV_ERR_INVALID_ARG before any work.  src == dst is a no-op.
 * The result is that of applying the pairs one after another (chains, a
 * block written twice, a block read after it is written all behave so): the
 * host cuts the list into waves without conflicts, one kernel per wave, the
 * pairs passed in the launch parameters.  A bf16 block's rows of the V
 * exponent map move with it.  `pairs` may be reused when the call returns.
 * Asynchronous on `stream`.
 */
kv_status paged_kv_copy_blocks(kv_pool* pool, const int32_t* pairs, int64_t num_pairs,
                               void* stream);

/*
 * paged_decode_workspace_bytes -- bytes of device scratch that
 * paged_decode_attention needs for these sizes (split-K partial results).
 * Depends on the pool's partition setting; 0 for invalid arguments.
 */
size_t paged_decode_workspace_bytes(const kv_pool* pool, int32_t batch, int32_t n_q_heads,
                                    int32_t max_context_len, int32_t sliding_window);

/*
 * paged_decode_attention -- one decode step of attention over the pool.
 *   q_dev:               bf16 [batch][n_q_heads][head_dim]; query head hq uses
 *                        KV head hq / (n_q_heads / n_kv_heads); n_q_heads must
 *                        be a multiple of n_kv_heads with a group of at most
 *                        64 (KV_ERR_UNSUPPORTED above).  A group of more than
 *                        8 runs as passes over 8 query heads at a time, each
 *                        reading the attended K/V again.
 *   block_tables_dev:    int32 [batch][max_blocks_per_seq]; only entries of
 *                        blocks holding an attended position are read.
 *   context_lens_dev:    int32 [batch]; each in [0, max_context_len] and
 *                        <= max_blocks_per_seq * block_size.
 *   max_context_len:     host-side upper bound of context_lens (sizes the grid).
 *   scale:               softmax scale applied to q.k.
 *   sliding_window:      <= 0 disables the window.
 *   out_dev:             fp32 [batch][n_q_heads][head_dim], softmax(scale q K^T) V;
 *                        16-byte aligned.  Device memory, or pinned host memory
 *                        the device can address (cudaHostAlloc, or
 *                        cudaHostRegister with cudaHostRegisterMapped, under
 *                        unified addressing): the kernels then write the result
 *                        into host memory directly, with no separate copy.
 *   workspace_dev:       at least paged_decode_workspace_bytes(...) bytes,
 *                        16-byte aligned; contents need no initialisation.
 * Work is split evenly over a persistent grid (stream-K over the list of
 * (sequence, KV head, block) units); a (sequence, KV head) pair cut between
 * warps leaves partial results that a reduce kernel merges.  On `stream`:
 * the decode kernel, then the reduce kernel as its programmatic dependent.
 * Calls that share a workspace must not overlap in time.
 */
kv_status paged_decode_attention(kv_pool* pool, const void* q_dev, int32_t n_q_heads,
                                 const int32_t* block_tables_dev, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens_dev, int32_t batch,
                                 int32_t max_context_len, float scale, int32_t sliding_window,
                                 float* out_dev, void* workspace_dev, size_t workspace_bytes,
                                 void* stream);

/*
 * paged_decode_step -- one decode step of a layer: paged_kv_write of the
 * step's new tokens, then paged_decode_attention over the pool that now holds
 * them ("The Decode Phase": the new token's K/V go into the last block, then
 * the query attends over every cached token including it).
 *   Arguments: those of paged_kv_write (k_dev, v_dev, slot_mapping_dev,
 *   num_tokens), then those of paged_decode_attention, with the same meaning,
 *   layout and checks; context_lens must already count the new tokens.
 *   Results are those of the two calls made one after the other.  The decode
 *   kernel is launched as a programmatic dependent of the write kernel: it
 *   reads its sequence table while the write runs and waits for the write to
 *   complete before it reads the pool.  The write kernel is itself launched as
 *   a programmatic dependent of the kernel before it on the stream: it may be
 *   scheduled while that kernel runs and waits for it to complete before it
 *   reads or writes anything (so inputs produced by any earlier kernel are
 *   safe).  batch == 0 performs the write alone.  The call neither
 *   synchronises nor allocates: with the pool, the workspace and the output
 *   in place it can be captured into a CUDA graph (stream capture), whose
 *   replays read whatever the captured input buffers then hold.
 */
kv_status paged_decode_step(kv_pool* pool, const void* k_dev, const void* v_dev,
                            const int64_t* slot_mapping_dev, int64_t num_tokens,
                            const void* q_dev, int32_t n_q_heads,
                            const int32_t* block_tables_dev, int32_t max_blocks_per_seq,
                            const int32_t* context_lens_dev, int32_t batch,
                            int32_t max_context_len, float scale, int32_t sliding_window,
                            float* out_dev, void* workspace_dev, size_t workspace_bytes,
                            void* stream);

/*
 * paged_decode_attention_noalloc -- paged_decode_attention for callers that
 * cannot allocate device memory when they run decode, e.g. a serving runtime
 * that gave all free memory to its KV pool at start-up and allows no later
 * cudaMalloc, or a plugin interface with no workspace argument.  (The pages
 * have no counterpart to this entry point.)
 *   Same arguments and results as paged_decode_attention, without the
 *   workspace: the split-K partials go to one static device array of
 *   PAGED_DECODE_STATIC_SCRATCH_BYTES that this library holds on every GPU
 *   that loads it, until the process exits.  The call itself allocates
 *   nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *   out_dev may be pinned host memory, as for paged_decode_attention.
 *   Returns KV_ERR_INVALID_ARG when paged_decode_workspace_bytes() for these
 *   sizes exceeds PAGED_DECODE_STATIC_SCRATCH_BYTES (use a larger partition,
 *   kv_pool_set_partition_blocks, or the workspace entry point then), else
 *   what paged_decode_attention returns for the same arguments.
 *   The first call on a device looks up the array's device address (once
 *   per device and CUDA context, with that device current; again after the
 *   context was destroyed and made anew, e.g. by cudaDeviceReset); make that
 *   first call before any stream capture.  All calls on a device share the
 *   array: calls that may overlap on the GPU (different streams, no ordering
 *   between them) race on it.
 */
#define PAGED_DECODE_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
kv_status paged_decode_attention_noalloc(kv_pool* pool, const void* q_dev, int32_t n_q_heads,
                                         const int32_t* block_tables_dev,
                                         int32_t max_blocks_per_seq,
                                         const int32_t* context_lens_dev, int32_t batch,
                                         int32_t max_context_len, float scale,
                                         int32_t sliding_window, float* out_dev, void* stream);

/*
 * paged_prefill_attention -- prefill / extend attention over the pool
 * ("Optimizing KV Cache Memory Management in vLLM with PagedAttention and
 * Dynamic Block Allocation", "The Prefill Phase": the prompt's states are
 * computed in one parallel step; with prefix caching ("PagedAttention",
 * "Walking through two requests") only the uncached tail is computed).
 *   q_dev:             bf16 [T][n_q_heads][128]: the new tokens of all
 *                      sequences, sequence b at rows cu_q_lens[b] ..
 *                      cu_q_lens[b+1]-1; their K/V already written to the
 *                      pool (paged_kv_write) at the last q_len positions.
 *   cu_q_lens_dev:     int32 [batch + 1], cu_q_lens[0] = 0, non-decreasing.
 *   block_tables_dev, max_blocks_per_seq, context_lens_dev: as for decode;
 *                      context_lens counts the new tokens.
 *   max_q_len:         host bound of cu_q_lens[b+1] - cu_q_lens[b] (sizes the grid).
 *   max_context_len:   host bound of context_lens.
 *   out_dev:           fp32 [T][n_q_heads][128]; token i of sequence b (at
 *                      position pos = ctx - q_len + i) gets
 *                      softmax(scale q K^T) V over positions [lo, pos], lo =
 *                      max(0, pos + 1 - sliding_window) when the window is on.
 * bf16, FP8 and FP4 pools with head_dim 128 and a query group of at most
 * 128 heads per KV head (a query tile's 128 rows are (token, head) pairs with
 * the group padded to a power of two; other shapes: KV_ERR_UNSUPPORTED).  Runs on the tcgen05
 * tensor cores.  bf16: Q K^T on bf16 operands; P V on f16 ones, P rounded
 * once to f16 and V converted to f16 scaled by a power of two (set from the
 * largest V of the key tiles seen so far, as the pool's exponent map
 * records it, raised when a later tile would overflow), which keeps every V
 * value exact whose magnitude is at least 2^-31 times that largest one
 * (smaller ones are off by at most 2^-39 of it); the result meets the
 * decode's bf16 accuracy.  FP8: Q K^T
 * takes E4M3 operands -- the K codes as stored, each query row scaled by a
 * power of two and split into an E4M3 code and the code of its remainder --
 * and P V f16 ones (P rounded once to f16, the V codes converted exactly),
 * with k_scale and v_scale applied in fp32.  FP4: keys and values
 * dequantised exactly into f16 (an E2M1 value times an E4M3 group scale),
 * each query row scaled by a power of two into f16, P one f16 per weight,
 * the head scales applied in fp32; the result meets the decode's bf16
 * accuracy.  Scores of any magnitude are handled (the softmax maximum is
 * kept in raw score units).  A sequence with q_len > context_len or a
 * context above a bound sets KV_ERR_BAD_CONTEXT and is skipped.
 * Asynchronous on `stream`; no workspace.
 */
kv_status paged_prefill_attention(kv_pool* pool, const void* q_dev, int32_t n_q_heads,
                                  const int32_t* cu_q_lens_dev, const int32_t* block_tables_dev,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens_dev,
                                  int32_t batch, int32_t max_q_len, int32_t max_context_len,
                                  float scale, int32_t sliding_window, float* out_dev,
                                  void* stream);

/*
 * kv_pool_set_partition_blocks -- split-K granularity: aim for about this
 * many blocks per warp (a multiple of 4, 4..1024) for the longest possible
 * call, using fewer warps than the full persistent grid when that needs
 * fewer; 0 restores the automatic choice (the full grid).  Tuning and tests
 * only: results are the same for every setting up to rounding.
 */
kv_status kv_pool_set_partition_blocks(kv_pool* pool, int32_t blocks_per_partition);

/*
 * kv_pool_set_timing_events -- instrumentation: when both are non-NULL, each
 * paged_decode_attention / paged_decode_step records `start_event` just
 * before each decode kernel launch and `stop_event` just after it, on its
 * stream, so that the pair brackets the decode kernel alone.  While they are
 * set, paged_decode_step launches its decode kernel after the write has
 * completed instead of overlapping its start with it.
 * The events (cudaEvent_t) stay owned by the caller; NULL, NULL turns it off.
 */
kv_status kv_pool_set_timing_events(kv_pool* pool, void* start_event, void* stop_event);

/*
 * kv_pool_set_wait_limit -- bound, in nanoseconds of wall time, of every wait
 * the pool's kernels make on a copy or on another warp (default 1 s; 1e5 ..
 * 1e10).  A wait that runs out records KV_ERR_TIMEOUT, the kernel drains
 * what it issued and returns; nothing traps.  The drain is bounded too: if a
 * wait for one of its own copies (or, in the prefill, for its tensor-core
 * products) also runs out, the kernel records KV_ERR_DRAIN_TIMEOUT and exits
 * with that work possibly still in flight.
 *
 * kv_pool_set_test_stall -- test instrumentation for the timeout path: while
 * enabled, the first copy of worker 0 in each decode launch expects 16 more
 * bytes than it brings, so that warp's bounded wait runs out and the call
 * reports KV_ERR_TIMEOUT (its outputs are then undefined).  Having recorded
 * the timeout, the kernel supplies the 16 bytes itself, so its drain
 * completes: no copy is left in flight and the context stays usable.
 * 0 disables it (the default).
 */
kv_status kv_pool_set_wait_limit(kv_pool* pool, uint64_t limit_ns);
kv_status kv_pool_set_test_stall(kv_pool* pool, int32_t enable);

/*
 * kv_pool_check_status -- synchronise `stream`, read and clear the pool's
 * device error word.  Returns KV_OK, or the first recorded problem in the
 * order KV_ERR_DRAIN_TIMEOUT, KV_ERR_TIMEOUT, KV_ERR_BAD_BLOCK_ID,
 * KV_ERR_BAD_SLOT, KV_ERR_BAD_CONTEXT, KV_ERR_STALE_EXPONENT_MAP; KV_ERR_CUDA if the stream itself
 * failed.  After KV_ERR_TIMEOUT the context stays usable (every copy the
 * kernel issued was seen to land).  After KV_ERR_DRAIN_TIMEOUT it is not
 * known to be: copies may still have been writing shared memory when the
 * kernel exited, so the caller should stop issuing work on it, synchronise
 * and tear the context down rather than keep using it.
 */
kv_status kv_pool_check_status(kv_pool* pool, void* stream);

/* kv_status_str -- static, human-readable name of a status code. */
const char* kv_status_str(kv_status status);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
