/*
 * paged_kv.h -- C ABI of the GB300 paged KV-cache decode library (libpagedkv.so).
 *
 * One decode step of one layer is
 *     kv_step (host)  ->  kv_append (GPU)  ->  paged_decode_attention (GPU)
 * i.e. the new token's K/V is appended to the cache first and the new query
 * then attends over the whole cache, including itself ("Transformer
 * attention mask and KV cache inference", section "Prefill and decode
 * phases").  paged_decode_step does the two GPU parts in one launch pair;
 * paged_decode is its general form (shared-prefix chunks, early inputs).
 *
 * Conventions shared by every entry point
 *   - Every function returns an int status: KV_OK (0) or a negative KV_ERR_*.
 *     Nothing throws across this boundary.
 *   - Device buffers are plain device pointers owned by the caller; the
 *     library never allocates, frees or retains device memory.  Host
 *     buffers are plain host pointers, also caller-owned.  The per-step
 *     buffers of the decode entry points (q, k_new, v_new, block_tables,
 *     context_lens, prefix tables, out) may also be pinned host memory that
 *     the device can address (cudaHostAlloc / cudaHostRegister with unified
 *     addressing): the kernels then read and write them in place, over the
 *     coherent NVLink-C2C link of a Grace-Blackwell node, with no copy.  The
 *     caches and the workspace must be device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  GPU entry points only enqueue work and return; a launch
 *     failure is reported as KV_ERR_CUDA.  Faults found by the kernels'
 *     own bounds checks (a slot or block id outside the pool, a context
 *     longer than its block-table row) do not abort: the offending access
 *     is skipped (or reads zeros) and a sticky device flag is set that
 *     kv_get_device_error() returns.
 *   - Cache layout, per layer: k_cache and v_cache are each
 *     [num_blocks][num_kv_heads][16][head_dim] elements of kv_dtype,
 *     row-major.  One (block, head) tile is 16*head_dim*elem_bytes
 *     contiguous bytes.  The 16-token block is the page of "KV Cache, Flash
 *     Attention and inference optimization", section "PagedAttention", and
 *     the [heads, seq, head_dim] order inside it is the tensor shape of "KV
 *     Cache" (heepie.pages.dev), section "Tensor".
 *   - Supported shapes: head_dim 64 or 128; num_q_heads a multiple of
 *     num_kv_heads with group size G = num_q_heads / num_kv_heads
 *     ("KV cache complete guide", section "(2) GQA": MHA G=1, GQA, and MQA,
 *     one KV head for all query heads).  G may be 1..16, or up to 128 when
 *     G / 2^k <= 16 for some k <= 3 divides evenly (e.g. 24, 32, 64, 128;
 *     not 17 or 34: KV_ERR_UNSUPPORTED).  Query head h reads KV head h / G.
 *     Groups above 8 rows run the two-row-tile kernel; groups above 16 are
 *     cut into 2^k sub-groups that each read the KV head's tiles (the
 *     repeats are served mostly from L2).  Prefix chunks need G <= 8.
 */
#ifndef PAGED_KV_H
#define PAGED_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define KV_OK 0
#define KV_ERR_INVALID_ARG (-1)   /* bad pointer, size, shape or id */
#define KV_ERR_OUT_OF_BLOCKS (-2) /* the block pool cannot satisfy the request */
#define KV_ERR_UNSUPPORTED (-3)   /* valid but not implemented (head_dim, group size) */
#define KV_ERR_CUDA (-4)          /* a CUDA runtime call or launch failed */
#define KV_ERR_NOT_FOUND (-5)     /* unknown sequence id */
#define KV_ERR_EXISTS (-6)        /* sequence id already present */
#define KV_ERR_TOO_LARGE (-7)     /* the request exceeds a fixed size limit of the library */

/* --------------------------------------------------------------- data types */
#define KV_DTYPE_BF16 0     /* bfloat16 */
#define KV_DTYPE_FP8_E4M3 1 /* OCP E4M3 ("fn"), per-tensor scale: x = code * scale */
#define KV_DTYPE_F32 2      /* float32 (attention output only) */

#define KV_BLOCK_SIZE 16

/* Device error flags reported by kv_get_device_error(). */
#define KV_DEVERR_SLOT_OUT_OF_RANGE 1     /* kv_append: slot >= num_blocks*16 */
#define KV_DEVERR_BLOCK_OUT_OF_RANGE 2    /* a block-table entry outside [0, num_blocks) */
#define KV_DEVERR_CONTEXT_TOO_LONG 4      /* context_lens[s] > 16*max_blocks_per_seq, or < 0 */
#define KV_DEVERR_PIPELINE_TIMEOUT 8      /* a bulk copy never arrived (a bug, never expected) */
#define KV_DEVERR_BAD_PREFIX 16           /* a prefix chunk table entry is inconsistent */

/* ------------------------------------------------------------------ sizing */

/* Bytes of K plus V for a whole model:
 *     2 (K and V) * layers * batch * kv_heads * seq * head_dim * dtype_bytes
 * ("KV cache complete guide" (techblog.paldyn.com), section "KV cache memory
 * size calculation"; "Transformer attention mask and KV cache inference",
 * section "Cache shape and memory calculation").  Returns -1 if any argument
 * is negative or the product overflows int64. */
int64_t kv_bytes(int layers, int batch, int kv_heads, int64_t seq, int head_dim, int dtype_bytes);

/* --------------------------------------------------- host block allocator */

/* Library-owned host object: a pool of num_blocks 16-token blocks with a
 * free list and per-block reference counts, plus the sequences that own
 * blocks ("KV Cache, Flash Attention and inference optimization", section
 * "PagedAttention" and exercise 3: fixed 16-token blocks, a free list, blocks
 * returned to the pool when a sequence ends; "KV cache complete guide",
 * section "(4) PagedAttention": requests with a common prefix share physical
 * blocks, copy-on-write).  Not thread-safe: one caller thread at a time. */
typedef struct kv_alloc kv_alloc_t;

/* Create an allocator.  block_size must be 16; num_kv_heads, head_dim and
 * kv_dtype are recorded for kv_alloc_stats and checks.  *out receives the
 * handle (NULL on failure).  The caller allocates the device caches itself
 * ([num_blocks][num_kv_heads][16][head_dim] per layer, K and V). */
int kv_cache_alloc(kv_alloc_t** out, int num_blocks, int num_kv_heads, int head_dim,
                   int block_size, int kv_dtype);

/* Destroy an allocator (NULL is ignored). */
void kv_alloc_destroy(kv_alloc_t* a);

/* Register sequence seq_id holding `len` prefilled tokens: takes
 * ceil(len/16) blocks from the free list.  KV_ERR_EXISTS if the id is in use,
 * KV_ERR_OUT_OF_BLOCKS (and no change) if the pool is too small. */
int kv_seq_add(kv_alloc_t* a, int64_t seq_id, int64_t len);

/* New sequence `child` that shares the first ceil(shared_len/16) blocks of
 * `parent` (reference counts incremented, no copy) and has length
 * shared_len <= len(parent).  A later append into a shared partial block
 * copies it first (see kv_step).  Beam/parallel-sample branching and
 * common-prefix reuse both use this. */
int kv_seq_fork(kv_alloc_t* a, int64_t parent, int64_t child, int64_t shared_len);

/* End a sequence: drop one reference from each of its blocks; blocks that
 * reach zero return to the free list.  KV_ERR_NOT_FOUND for unknown ids. */
int kv_seq_free(kv_alloc_t* a, int64_t seq_id);

/* Plan one decode step for n sequences (the append contract of
 * "Transformer attention mask and KV cache inference", section "Position ID
 * and append contract": the new token goes at position == current length).
 * For row i (sequence seq_ids[i], current length pos):
 *   - if pos % 16 == 0 a fresh block is taken from the free list;
 *   - else if the tail block is shared (refcount > 1) a fresh block is taken,
 *     the pair (old, new) is reported in cow_src/cow_dst so the caller can
 *     copy its contents on the GPU (kv_copy_blocks) before appending, and the
 *     old block loses one reference;
 *   - slot_mapping[i] = block_table[pos / 16] * 16 + pos % 16;
 *   - the sequence length becomes pos + 1 and context_lens[i] = pos + 1;
 *   - block_tables[i*max_blocks ...] receives the sequence's block ids, the
 *     rest of the row is filled with -1.
 * All outputs are host arrays: slot_mapping[n] int64, block_tables
 * [n][max_blocks] int32, context_lens[n] int32, cow_src/cow_dst[cow_cap]
 * int32, *n_cow.  The step is all-or-nothing: on KV_ERR_OUT_OF_BLOCKS,
 * KV_ERR_NOT_FOUND, a repeated id, a row longer than max_blocks or
 * cow_cap < needed copies (KV_ERR_INVALID_ARG) nothing changes. */
int kv_step(kv_alloc_t* a, const int64_t* seq_ids, int n, int64_t* slot_mapping,
            int32_t* block_tables, int max_blocks, int32_t* context_lens, int32_t* cow_src,
            int32_t* cow_dst, int cow_cap, int* n_cow);

/* Reorder the KV state of a batch of live sequences (beam search selection
 * or batch-row reuse): after the call, sequence seq_ids[i] holds the length
 * and blocks that sequence seq_ids[src_index[i]] held before it, e.g. rows
 * [A0, A1, B0] with src_index [2, 1, 0] become [B0, A1, A0] ("Transformer
 * attention mask and KV cache inference", section "Batch and beam reorder":
 * the cache must follow the same permutation as the rows).  With paging this
 * moves no K/V data: block tables are permuted and shared through reference
 * counts, so a src_index with repeats (beam duplication) makes the duplicates
 * share every block, and the next kv_step copies a shared tail block before
 * appending.  Blocks no row keeps return to the free list.  seq_ids must be
 * distinct and live; 0 <= src_index[i] < n; on an error nothing changes. */
int kv_seq_reorder(kv_alloc_t* a, const int64_t* seq_ids, const int32_t* src_index, int n);

/* Read a sequence's state: *len (may be NULL), and its block ids into
 * row[max_blocks] (may be NULL; -1 padded).  *nblocks (may be NULL) gets
 * the number of blocks it holds.  KV_ERR_INVALID_ARG if row is too short. */
int kv_seq_info(kv_alloc_t* a, int64_t seq_id, int64_t* len, int32_t* row, int max_blocks,
                int* nblocks);

/* Pool statistics: free blocks, blocks in use, live sequences, and the
 * reference count of one block (block < 0: skipped). */
int kv_alloc_stats(kv_alloc_t* a, int* free_blocks, int* used_blocks, int* num_seqs,
                   int block, int* refcount);

/* The allocator's shape: pool blocks, KV heads, head dim and cache dtype, so
 * that a trace can state the per-layer cache shape
 * [num_blocks][num_kv_heads][16][head_dim].  Any pointer may be NULL. */
int kv_alloc_shape(kv_alloc_t* a, int* num_blocks, int* num_kv_heads, int* head_dim,
                   int* kv_dtype);

/* Debug trace of the cache state: the fields that "Transformer attention mask
 * and KV cache inference", section "Implementation and verification
 * procedure", wants a trace to keep, so that a wrong output can be narrowed
 * down to a broken state contract.  One row
 * of KV_TRACE_FIELDS int64 per sequence, fields indexed by KV_TRACE_*:
 *   SEQ_ID         the request id;
 *   SLOT           its batch row in the last kv_step or kv_seq_reorder that
 *                  named it (-1: none yet);
 *   LEN            current length (tokens held);
 *   POSITION       position offset the next appended token takes (equal to
 *                  LEN: a paged sequence holds no padding);
 *   BLOCKS         blocks held;
 *   SHARED_BLOCKS  of those, blocks whose reference count is above 1;
 *   CACHE_BYTES    K + V bytes of the held blocks for one layer
 *                  (BLOCKS * 2 * 16 * num_kv_heads * head_dim * element size);
 *   REORDER_SRC    the src_index its row had in the last kv_seq_reorder that
 *                  named it, i.e. the reorder permutation (-1: never).
 * A decode step has no mask tensor: each row attends to LEN keys (mask shape
 * [1, LEN]).  seq_ids != NULL: rows for those n sequences in that order
 * (KV_ERR_NOT_FOUND for an unknown id).  seq_ids == NULL: every live
 * sequence in ascending id order; n is the capacity of rows in sequences and
 * KV_ERR_INVALID_ARG if fewer than the live count.  rows is a host array of
 * [n][KV_TRACE_FIELDS] int64; *count (may be NULL) gets the rows written.
 * Reads only; nothing changes. */
#define KV_TRACE_FIELDS 8
#define KV_TRACE_SEQ_ID 0
#define KV_TRACE_SLOT 1
#define KV_TRACE_LEN 2
#define KV_TRACE_POSITION 3
#define KV_TRACE_BLOCKS 4
#define KV_TRACE_SHARED_BLOCKS 5
#define KV_TRACE_CACHE_BYTES 6
#define KV_TRACE_REORDER_SRC 7
int kv_alloc_trace(kv_alloc_t* a, const int64_t* seq_ids, int n, int64_t* rows, int* count);

/* Slot of position positions[i] of sequence row i of block_tables (host):
 *     slot = block_tables[i][pos / 16] * 16 + pos % 16
 * ("KV Cache, Flash Attention and inference optimization", section
 * "PagedAttention": the page table maps a logical position to a physical
 * block).  A negative position gives slot -1 (a padding token).
 * KV_ERR_INVALID_ARG if pos / 16 >= max_blocks or the entry is negative. */
int kv_slot_mapping(const int32_t* block_tables, int max_blocks, const int64_t* positions,
                    int n, int64_t* slot_mapping);

/* ------------------------------------------------------------- GPU: append */

/* Write each token's K and V into its cache slot (device pointers):
 *   k, v:          [num_tokens][num_kv_heads][head_dim] bfloat16
 *   slot_mapping:  [num_tokens] int64, slot = block * 16 + offset; a slot < 0
 *                  skips the token (padding); a slot >= num_blocks*16 is
 *                  skipped and flags KV_DEVERR_SLOT_OUT_OF_RANGE
 *   k_cache, v_cache: the layer's caches (layout above)
 *   kv_dtype:      KV_DTYPE_BF16 (bit copy) or KV_DTYPE_FP8_E4M3: code =
 *                  E4M3(x / scale), quotient in binary32, round to nearest
 *                  even, saturating to +-448 ("KV cache complete guide",
 *                  section "(1) FP8 quantization": an FP8 KV cache halves its
 *                  memory).  k_scale / v_scale must be finite and > 0.
 * Tokens with equal slots race (last writer wins, unspecified). */
int kv_append(const void* k, const void* v, void* k_cache, void* v_cache,
              const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
              int num_blocks, int kv_dtype, float k_scale, float v_scale, void* stream);

/* Copy whole blocks (all KV heads, K and V) src[i] -> dst[i] inside the
 * caches; src/dst are device int32 arrays of n ids.  Used for the
 * copy-on-write pairs reported by kv_step ("KV cache complete guide",
 * section "(4) PagedAttention": shared blocks are copy-on-write).  Ids
 * outside [0, num_blocks) are skipped and flag KV_DEVERR_BLOCK_OUT_OF_RANGE.
 * A dst that is also some src in the same call gives an unspecified result. */
int kv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int n,
                   int num_kv_heads, int head_dim, int num_blocks, int kv_dtype, void* stream);

/* --------------------------------------------------- GPU: decode attention */

/* Workspace bytes paged_decode_attention / paged_decode_step need on the
 * current device for this shape: split-KV partial outputs with their (max,
 * sum) terms, and a small per-(sequence, KV head) table.  Queries the device;
 * KV_ERR_CUDA without one.  The workspace needs no initialisation and carries
 * nothing from one call to the next; calls that overlap on the GPU need
 * separate workspaces. */
int paged_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int kv_dtype, size_t* bytes);

/* One decode step of attention over a paged cache (all device pointers):
 *   out:           [num_seqs][num_q_heads][head_dim], out_dtype KV_DTYPE_BF16
 *                  (rounded to nearest even) or KV_DTYPE_F32
 *   q:             [num_seqs][num_q_heads][head_dim] bfloat16
 *   k_cache, v_cache: layout above, kv_dtype; fp8 values are code * k_scale
 *                  (K) and code * v_scale (V).  Base addresses 16-byte aligned.
 *   num_blocks:    blocks in the pool (block ids must lie in [0, num_blocks))
 *   block_tables:  [num_seqs][max_blocks_per_seq] int32; only the first
 *                  ceil(context_lens[s]/16) entries of row s are read
 *   context_lens:  [num_seqs] int32, the number of cached tokens each query
 *                  attends over (after this step's append)
 *   scale:         the softmax scale, normally 1/sqrt(head_dim)
 *   workspace:     device buffer of paged_decode_workspace_bytes(...) bytes,
 *                  16-byte aligned
 * Computes, for query head h of sequence s and KV head hk = h / G,
 *     out[s][h] = sum_j softmax_j(scale * q[s][h] . K[s][hk][j]) V[s][hk][j]
 * over key positions j < context_lens[s] (the length mask of "Transformer
 * attention mask and KV cache inference", section "Padding mask and batch
 * length"; the formula of "KV Cache" (heepie), section "Self-Attention").
 * The softmax runs as an online (running max, running sum) pass over 16-token
 * blocks, split evenly across the warps of one persistent launch; warps that
 * share a (sequence, KV head) leave partial results that a second, small
 * kernel merges with the log-sum-exp rule ("KV Cache, Flash Attention and
 * inference optimization", section "Numerical trick": the running (max, sum)
 * makes the tiled result exact).  A sequence with context_lens[s] == 0 gets
 * zeros.  Bad table entries never fault: a block id outside [0, num_blocks)
 * is not read (its sequence's output is then unspecified) and a context
 * length outside [0, 16*max_blocks_per_seq] is clamped into that range; each
 * raises its KV_DEVERR_* flag (kv_get_device_error, the first bad value as
 * the detail).  Both kernels use programmatic dependent launch: each may start
 * while the previous kernel on the stream drains, and waits on the device for
 * it to finish before reading or writing any buffer.  Deterministic: the same
 * inputs on the same device give bit-identical outputs, whatever the physical
 * block ids.  The split of the work over warps, and so the rounding order,
 * follows the device's SM count and max_blocks_per_seq (a narrow table lets
 * short sequences spread over more warps); results agree within the
 * tolerance across either.  `out` must be 16-byte aligned. */
int paged_decode_attention(void* out, int out_dtype, const void* q, const void* k_cache,
                           const void* v_cache, int kv_dtype, float k_scale, float v_scale,
                           int num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, float scale, void* workspace,
                           size_t workspace_bytes, void* stream);

/* The same operation, recording caller-created CUDA events (cudaEvent_t
 * passed as void*, each may be NULL) on `stream` immediately before the
 * split-KV kernel, after it, and after the merge kernel, so that a caller can
 * time the library's own launches on the stream they run on.  This is a
 * measurement hook of this implementation (the pages have no counterpart). */
int paged_decode_attention_timed(void* out, int out_dtype, const void* q, const void* k_cache,
                                 const void* v_cache, int kv_dtype, float k_scale, float v_scale,
                                 int num_blocks, const int32_t* block_tables,
                                 int max_blocks_per_seq, const int32_t* context_lens,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 float scale, void* workspace, size_t workspace_bytes,
                                 void* stream, void* ev_begin, void* ev_split_end, void* ev_end);

/* A whole decode step of one layer: append each sequence's new
 * token, then attend (the order of "Transformer attention mask and KV cache
 * inference", section "Prefill and decode phases").  Same arguments as
 * paged_decode_attention, plus
 *   k_new, v_new:  [num_seqs][num_kv_heads][head_dim] bfloat16 (device), the
 *                  new token's K and V of every sequence;
 *   k_cache, v_cache are written: the new token of sequence s is stored at
 *                  position context_lens[s]-1, i.e. slot
 *                  block_tables[s][(L-1)/16]*16 + (L-1)%16 (the append
 *                  contract of the same page, section "Position ID and append
 *                  contract"), with the same bits as kv_append (bf16 copy or
 *                  E4M3(x/scale)), and is attended to in the same launch.
 * context_lens are the lengths after the append (as for
 * paged_decode_attention).  The block receiving a new token must be private
 * to its sequence (kv_step's copy-on-write guarantees it); sequences with
 * context_lens[s] == 0 append nothing.  Equivalent to kv_append with
 * slot_mapping = kv_slot_mapping(block_tables, context_lens-1) followed by
 * paged_decode_attention. */
int paged_decode_step(void* out, int out_dtype, const void* q, const void* k_new,
                      const void* v_new, void* k_cache, void* v_cache, int kv_dtype,
                      float k_scale, float v_scale, int num_blocks, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, float scale,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free variant of paged_decode_attention for callers that cannot
 * allocate device memory: code running inside a host framework that owns the
 * device memory pool and forbids its plugins to allocate, or a
 * latency-critical path that must not call into the driver's allocator.
 * Such a caller cannot provide the `workspace` buffer, so this entry point
 * takes none and uses scratch that the library itself holds: a file-scope
 * device array of KV_NOALLOC_WORKSPACE_BYTES (16 MiB) that every GPU loading
 * the library keeps until the process exits.  It calls no cudaMalloc,
 * cudaFree or allocating library routine.  (This is an interface of this
 * implementation; the pages have no counterpart.)
 *   - Arguments, layouts and results are those of paged_decode_attention
 *     (the caller still passes every input and the output).
 *   - A shape whose scratch (paged_decode_workspace_bytes) exceeds
 *     KV_NOALLOC_WORKSPACE_BYTES is rejected with KV_ERR_TOO_LARGE before
 *     anything is launched.
 *   - The first call on each device performs a one-time set-up on that device
 *     (it looks up the device address of the array and configures the
 *     kernels); make that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents (nothing in it has to start at zero: each call rewrites
 *     what it reads).  Calls that overlap on the GPU -- concurrent streams,
 *     or host threads launching at once -- race on it and give undefined
 *     results; serialise them, or use paged_decode_attention with separate
 *     workspaces. */
#define KV_NOALLOC_WORKSPACE_BYTES (16u << 20)
int paged_decode_attention_noalloc(void* out, int out_dtype, const void* q, const void* k_cache,
                                   const void* v_cache, int kv_dtype, float k_scale,
                                   float v_scale, int num_blocks, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   float scale, void* stream);

/* --------------------------------------------------- shared-prefix decoding */

/* Requests that share a system prompt share its KV blocks ("KV cache complete
 * guide", sections "(3) Prefix Caching" and "(4) PagedAttention": the same
 * physical blocks, copy-on-write).  The entry points below read each shared
 * (block, KV head) tile once for a whole chunk of sequences instead of once
 * per sequence.  (An interface of this implementation; the pages describe
 * the sharing, not a kernel for it.)
 *
 * A prefix chunk is a set of 2..KV_PREFIX_MAX_ROWS/G sequences (G = query
 * heads per KV head) whose block-table rows start with the same P block ids,
 * all P blocks lying wholly before each member's new token (16*P <=
 * context_lens[s] - 1).  Chunk table: int32 [num_chunks][KV_PREFIX_CHUNK_INTS],
 * row c = {P, m, member_0, ..., member_{m-1}, -1 ...}; the shared blocks are
 * read from member_0's block-table row.  seq_chunk: int32 [num_seqs],
 * (c << 4) | (index of s among chunk c's members), or -1 for a sequence in no
 * chunk.  Each chunk's query rows (m * G <= 16) are attended together over
 * its P blocks; every sequence then attends alone from block P (0 without a
 * chunk) on, and the two partial results are combined by their log-sum-exp
 * weights.  The result equals paged_decode_attention / paged_decode_step on
 * the same inputs up to floating-point summation order. */
#define KV_PREFIX_MAX_ROWS 16
#define KV_PREFIX_MAX_MEMBERS 16
#define KV_PREFIX_CHUNK_INTS (2 + KV_PREFIX_MAX_MEMBERS)

/* Build a chunk table from block tables (host memory, plain C):
 *   - sequences whose rows begin with the same block id and have at least
 *     min_blocks full blocks before their new token form a group;
 *   - each member's shared run is the number of leading block ids it has in
 *     common with the group's leader -- its member with the most full blocks
 *     before the new token, the first such -- capped by both members' full
 *     blocks before their new tokens;
 *   - members are ordered by shared run (longest first, then by index) and
 *     cut into chunks of up to KV_PREFIX_MAX_ROWS / group_size sequences;
 *     a chunk's P is its shortest member run; chunks with fewer than two
 *     members or P < min_blocks are dropped (their sequences get -1).
 * chunks must hold num_seqs / 2 rows (the most chunks possible); seq_chunk
 * num_seqs entries.  group_size = num_q_heads / num_kv_heads (1..8: a chunk
 * packs at least two members' rows into one 16-row tile).
 * Returns KV_OK and *num_chunks, or KV_ERR_INVALID_ARG. */
int kv_prefix_chunks(const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs, int group_size, int min_blocks,
                     int32_t* chunks, int32_t* seq_chunk, int* num_chunks);

/* kv_prefix_chunks with the decision whether the chunks pay (host memory):
 * returns the chunk table kv_prefix_chunks builds (group_size = num_q_heads /
 * num_kv_heads, min_blocks 1) when its chunks save a large enough fraction f
 * of the blocks the step reads for the step's P = num_seqs * num_kv_heads
 * (sequence, KV head) pairs against the split-KV kernel's W resident warps:
 * f >= 6 % when 5 P >= 2 W, f >= 30 % when W <= 5 P < 2 W, never when
 * 5 P < W.  Otherwise *num_chunks = 0 and seq_chunk all -1, i.e. plain
 * decoding.  (Measured crossovers of this implementation: below these bounds
 * the shared-prefix kernel, which carries two row tiles of state, is slower
 * than reading the shared blocks once per sequence -- which, with few pairs,
 * mostly hit L2 anyway.)  resident_warps: W, or <= 0 to query the current
 * device (152 SMs x 2 CTAs x 4 warps = 1216 on GB300 at d128).  Groups of more
 * than 8 query heads per KV head always get plain decoding.  chunks:
 * num_seqs / 2 rows; seq_chunk: num_seqs entries.  Returns KV_OK,
 * KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED (shape) or KV_ERR_CUDA (device
 * query). */
int kv_prefix_plan(const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                   int head_dim, int kv_dtype, int resident_warps, int32_t* chunks,
                   int32_t* seq_chunk, int* num_chunks);

/* Workspace bytes paged_decode needs with num_chunks prefix chunks (as
 * paged_decode_workspace_bytes, which is the num_chunks == 0 case). */
int paged_decode_prefix_workspace_bytes(int num_seqs, int num_chunks, int num_q_heads,
                                        int num_kv_heads, int head_dim, int kv_dtype,
                                        size_t* bytes);

/* Flags of paged_decode. */
#define KV_DECODE_EARLY_INPUTS 1u   /* read block_tables, context_lens, the prefix
                                       tables and the caches early (below) */

/* One decode step, general form (an interface of this implementation):
 * arguments as paged_decode_step, plus
 *   - k_new and v_new may both be NULL: then nothing is appended (as
 *     paged_decode_attention) and k_cache / v_cache are only read;
 *   - chunks, seq_chunk, num_chunks: device copies of a prefix chunk table
 *     (above; num_chunks == 0 gives plain decoding, the tables may then be
 *     NULL).  A chunk entry that breaks the rules above (P out of range, a
 *     member index outside [0, num_seqs), a shared block reaching a member's
 *     new token, a seq_chunk entry naming another chunk) flags
 *     KV_DEVERR_BAD_PREFIX; every access stays in bounds, the results of the
 *     sequences concerned are undefined.  The chunk table must describe
 *     blocks that really are shared: the kernel reads them from member_0's
 *     row;
 *   - flags: 0 or KV_DECODE_EARLY_INPUTS.  Every kernel of this library
 *     starts while the kernel before it on the stream drains (programmatic
 *     dependent launch) and, by default, reads nothing until that kernel has
 *     completed.  With KV_DECODE_EARLY_INPUTS the split kernel reads
 *     context_lens, block_tables, the prefix tables and the cache tiles as
 *     soon as it starts, overlapping the previous kernel's end (q, k_new,
 *     v_new, the outputs and the workspace still wait for it).  The caller
 *     guarantees that the kernel launched immediately before this call on
 *     the stream writes none of those inputs, unless it is a call of this
 *     library (whose last kernel allows dependent launches only once the
 *     call's appends are complete).  Inputs written by copies, or by work on
 *     other streams joined to this one by events, are fine.  It removes ~2 us
 *     from each step of a decode loop. */
int paged_decode(void* out, int out_dtype, const void* q, const void* k_new, const void* v_new,
                 void* k_cache, void* v_cache, int kv_dtype, float k_scale, float v_scale,
                 int num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                 const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                 int head_dim, float scale, const int32_t* chunks, const int32_t* seq_chunk,
                 int num_chunks, unsigned flags, void* workspace, size_t workspace_bytes,
                 void* stream);

/* The same step as paged_decode, with events recorded on the stream before
 * the split-KV kernel, after it, and after the merge kernel (each may be
 * NULL), so that a caller can time the split kernel inside a loop of
 * consecutive decode steps in the mode it normally runs in (fused append,
 * KV_DECODE_EARLY_INPUTS).  A measurement hook of this implementation (the
 * pages have no counterpart); an event record between the two kernels may
 * delay the merge kernel's start by a launch latency. */
int paged_decode_timed(void* out, int out_dtype, const void* q, const void* k_new,
                       const void* v_new, void* k_cache, void* v_cache, int kv_dtype,
                       float k_scale, float v_scale, int num_blocks,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, float scale, const int32_t* chunks,
                       const int32_t* seq_chunk, int num_chunks, unsigned flags,
                       void* workspace, size_t workspace_bytes, void* stream, void* ev_begin,
                       void* ev_split_end, void* ev_end);

/* Read-only bandwidth ceiling (a measurement hook; the pages have no
 * counterpart): streams `bytes` of device memory at `buf` into shared memory
 * with bulk copies and no arithmetic, in the decode kernel's own pattern (a
 * persistent grid, per-warp rings of 3 x 8 KB stages, equal contiguous ranges
 * per warp, L2 evict-first), so its bandwidth bounds what the decode kernel
 * can reach.  buf: device, 16-byte aligned; bytes: a positive multiple of 16;
 * sink: device, 2 words the caller zeroes -- sink[0] receives an XOR of the
 * data read, sink[1] becomes 1 if a copy never arrived (bounded wait).
 * Asynchronous on `stream`.  Returns KV_OK, KV_ERR_INVALID_ARG or KV_ERR_CUDA. */
int kv_read_ceiling(const void* buf, size_t bytes, unsigned* sink, void* stream);

/* ------------------------------------------------------------- diagnostics */

/* Test hook (no counterpart in the pages): while `cycles` > 0, every warp of
 * the split-KV kernels launched afterwards makes the first wait of its range
 * on a barrier that nothing arrives on, gives up after `cycles` SM clocks
 * and takes the time-out path -- KV_DEVERR_PIPELINE_TIMEOUT raised, the bulk
 * copies it has issued waited for at the normal limit, the warp stops, so
 * that call's output is undefined.  In the wide-group kernel (groups of more
 * than 32 rows, bf16 cache, head_dim 128) the score-MMA warp of every CTA does so on its first wait, and every
 * role of the CTA then stops (copies and MMAs in flight are waited for and
 * tensor memory is freed before the CTA ends).  It lets a test see the flag without a
 * copy that really never arrives.  0 (the default) turns it off; a value
 * outside [0, 2^31] returns KV_ERR_INVALID_ARG.  Process-wide. */
int kv_test_pipeline_stall(long long cycles);

/* Read (synchronously, on the current device) and clear the sticky device
 * error flags (KV_DEVERR_* bits) set by the kernels' bounds checks; *detail
 * receives the first offending value (slot, block id or length), or -1. */
int kv_get_device_error(int* flags, int64_t* detail);

/* Library version string, e.g. "pagedkv 0.1 sm_103a". */
const char* kv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H */
