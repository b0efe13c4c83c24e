/*
 * pagedkv.h -- C ABI of libpagedkv, a GB300 (sm_103a) library for the decode
 * hot path of paged KV-cache attention.
 *
 * Pages the operations follow (title and section):
 *   P1 = "KV Cache与PagedAttention深度解析：vLLM内存管理革命" (iopencloud.com)
 *   P2 = "KV Cache从原理到实战：大模型推理内存管理演进与优化" (xnwp.cn/news/16711)
 *   P3 = PagedAttention + prefix caching via nano-vllm (zwxr.cn/news/317362)
 *   P4 = "大模型 (LLM) 推理加速核心技术解析：从 KV Cache 到 PagedAttention 实战"
 *        (jsqmd.com/news/745991)
 *
 * Conventions shared by every call
 * --------------------------------
 * Layout.  The KV pool is [num_blocks][2][num_kv_heads][block_size][head_dim]
 *   (P1 §4.3 and §5.1, with num_kv_heads for grouped-query models, P2 §5.3).
 *   Calls take the K half and the V half as two base pointers plus the stride,
 *   in elements, between consecutive physical blocks: for the packed pool
 *   k_cache = pool, v_cache = pool + num_kv_heads*block_size*head_dim and
 *   block_stride_elems = 2*num_kv_heads*block_size*head_dim.  Within a block,
 *   row (h, offset) of K starts at k_cache + blk*block_stride_elems +
 *   (h*block_size + offset)*head_dim.
 * Slots.  Slot s names block s / block_size, offset s % block_size (P1 §5.3).
 * Heads.  Query head hq reads KV head hq / (num_q_heads / num_kv_heads).
 * Types.  dtype is fp16 or bf16 for q, K, V and out; accumulation is fp32.
 *   head_dim is 64 or 128; block_size is 8, 16 or 32.  Others: PKV_ERR_UNSUPPORTED.
 * Memory.  Every pointer argument is a DEVICE pointer owned by the caller,
 *   except where a call says HOST (pkv_slot_mapping_host, the outputs of
 *   pkv_get_device_error and the block manager's arrays).  Tensor base
 *   pointers must be 16-byte aligned and block strides a multiple of 8
 *   elements.  No call allocates memory; the library's only state is one
 *   device status word per device (see pkv_get_device_error), the fixed
 *   scratch array of pkv_paged_attention_decode_static_scratch, and cached
 *   device attributes.
 * Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).  Every
 *   call only enqueues work on it and returns; results are ready when the
 *   stream reaches that point.
 * Errors.  Arguments that can be checked on the host are checked before any
 *   launch: PKV_ERR_INVALID_ARG (nothing enqueued).  Values that live in device
 *   memory (slots, block-table entries, context lengths, copy pairs) are
 *   checked by the kernels: a bad value is skipped, never dereferenced, and
 *   raises a flag in the device status word.  A failed launch returns
 *   PKV_ERR_CUDA.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* host-checkable argument out of contract      */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not built (dtype, head_dim, bs)    */
    PKV_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed         */
    PKV_ERR_DEVICE = 4,        /* pkv_get_device_error found flags raised      */
    PKV_ERR_SCRATCH_LIMIT = 5, /* split-context scratch needed exceeds
                                  PKV_STATIC_SCRATCH_BYTES (static-scratch decode) */
    PKV_ERR_OUT_OF_BLOCKS = 6  /* block manager: the free pool cannot cover the request */
} pkv_status;

/* PKV_INT8 names an INT8 cache; only pkv_copy_blocks takes it as `dtype` (the
 * INT8 entry points below take the query / new-row dtype, fp16 or bf16). */
typedef enum pkv_dtype { PKV_F16 = 0, PKV_BF16 = 1, PKV_INT8 = 2 } pkv_dtype;

/* Flags of the device status word (bitwise OR of what the kernels saw). */
#define PKV_DEVERR_SLOT        0x1u  /* slot_mapping entry >= num_blocks*block_size  */
#define PKV_DEVERR_BLOCK_TABLE 0x2u  /* block_tables entry outside [0, num_blocks)    */
#define PKV_DEVERR_CONTEXT_LEN 0x4u  /* context_lens entry < 0, > max_context_len or
                                        > max_blocks_per_seq*block_size (clamped)      */
#define PKV_DEVERR_COPY_PAIR   0x8u  /* copy pair entry outside [0, num_blocks)       */
#define PKV_DEVERR_TIMEOUT     0x10u /* a bounded wait on an async copy gave up       */

/*
 * pkv_reshape_and_cache -- write each new token's K and V rows into its slot.
 * (P1 §2.2: compute only K_t, V_t and append them; P1 §5.3: the write goes to
 * offset t % block_size of the sequence's last block.)
 *
 *   k_new, v_new   [num_tokens][num_kv_heads][head_dim], contiguous, dtype.
 *   slot_mapping   [num_tokens] int64; slot < 0 means "skip this token"
 *                  (padding); slot >= num_blocks*block_size raises
 *                  PKV_DEVERR_SLOT and the token is skipped.  Two tokens must
 *                  not share a slot (the result would be either row).
 *   k_cache/v_cache, num_blocks, block_stride_elems: the pool, as above.
 * The copy is bit-exact.  num_tokens == 0 is a no-op.
 */
PKV_API pkv_status pkv_reshape_and_cache(const void *k_new, const void *v_new,
                                         const int64_t *slot_mapping, int64_t num_tokens,
                                         void *k_cache, void *v_cache, int64_t num_blocks,
                                         int64_t block_stride_elems, int num_kv_heads,
                                         int head_dim, int block_size, pkv_dtype dtype,
                                         void *stream);

/*
 * pkv_slot_mapping -- the slot each new token's K/V rows are written to, i.e.
 * the slot_mapping input of pkv_reshape_and_cache (P1 §5.3: logical position t
 * of a sequence lies in its table entry t / block_size at offset
 * t % block_size; the flat slot is entry * block_size + offset; P1 §4.2's worked
 * table [7, 2, 9, 1, 5, 8, 3] puts position 99 in slot 3*16 + 3).
 *
 *   block_tables   [num_table_rows][max_blocks_per_seq] int32, device.
 *   token_rows     [num_tokens] int64, device: the table row of each token's
 *                  sequence; NULL means token i uses row i (then
 *                  num_table_rows >= num_tokens).
 *   positions      [num_tokens] int64, device: each token's logical position;
 *                  a negative position is padding and gets slot -1.
 *   num_blocks     pool size, for the range check of table entries.
 *   slot_mapping   [num_tokens] int64, device output.
 * A position past the table (>= max_blocks_per_seq * block_size) or a token row
 * outside the table raises PKV_DEVERR_SLOT, a table entry outside
 * [0, num_blocks) raises PKV_DEVERR_BLOCK_TABLE; such a token gets slot -1.
 * Enqueued on `stream`; num_tokens == 0 is a no-op.
 */
PKV_API pkv_status pkv_slot_mapping(const int32_t *block_tables, int64_t num_table_rows,
                                    int max_blocks_per_seq, const int64_t *token_rows,
                                    const int64_t *positions, int64_t num_tokens, int block_size,
                                    int64_t num_blocks, int64_t *slot_mapping, void *stream);

/*
 * pkv_slot_mapping_host -- pkv_slot_mapping on HOST arrays, computed on the
 * calling thread (no CUDA call), for callers that keep their block tables in
 * host memory.  Same rule and outputs; instead of device flags it returns
 * PKV_ERR_INVALID_ARG when any token had a bad position, row or table entry
 * (every slot is still written, those tokens' as -1).
 */
PKV_API pkv_status pkv_slot_mapping_host(const int32_t *block_tables, int64_t num_table_rows,
                                         int max_blocks_per_seq, const int64_t *token_rows,
                                         const int64_t *positions, int64_t num_tokens,
                                         int block_size, int64_t num_blocks,
                                         int64_t *slot_mapping);

/*
 * pkv_decode_workspace_bytes -- device scratch that pkv_paged_attention_decode
 * needs for a split-context (partitioned) call: fp32 partial outputs plus the
 * running maximum and sum of every (sequence, query head, partition).
 * partition_size 0 means "the library's choice" and returns the size for the
 * partition count that choice gives on the current device.  Returns 0 when
 * no split is needed and (size_t)-1 for arguments out of contract.
 */
PKV_API size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, int max_context_len,
                                          int partition_size);

/*
 * pkv_paged_attention_decode -- one query token per sequence attends over its
 * paged KV cache:  out[i, hq] = softmax(scale * q[i, hq] . K_i^T) V_i
 * (P1 §2.1), where K_i, V_i are the first context_lens[i] tokens of sequence i
 * reached through block_tables[i] (P1 §4.2-4.3), accumulated with the running
 * maximum / running sum rescaling of P1 §7.2 in fp32.
 *
 *   q             [num_seqs][num_q_heads][head_dim], contiguous, dtype.
 *   block_tables  [num_seqs][max_blocks_per_seq] int32, physical block ids.
 *   context_lens  [num_seqs] int32, tokens to attend over (the new token
 *                 included); 0 gives a zero output row.
 *   max_context_len  host-side upper bound of context_lens (sizes the grid; a
 *                 larger device value raises PKV_DEVERR_CONTEXT_LEN and is
 *                 clamped).
 *   scale         softmax scale, normally 1/sqrt(head_dim).
 *   out           [num_seqs][num_q_heads][head_dim], contiguous, dtype; each
 *                 value rounded once (to nearest even) from fp32.
 *   workspace     device scratch of workspace_bytes (>= the value of
 *                 pkv_decode_workspace_bytes for the same arguments); may be
 *                 NULL when that value is 0.  Contents need no initialisation.
 *   partition_size  tokens per split-context partition, a multiple of
 *                 block_size; 0 = library's choice.  Each (sequence, KV head,
 *                 partition) is processed independently and merged by a second
 *                 kernel (log-sum-exp merge) when a sequence spans >1 partition.
 * The reduction order depends only on logical positions, so the result is
 * bitwise independent of where blocks sit in the pool.
 */
PKV_API pkv_status pkv_paged_attention_decode(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    int64_t block_stride_elems, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, float scale, void *out, void *workspace,
    size_t workspace_bytes, int partition_size, pkv_dtype dtype, void *stream);

/*
 * pkv_copy_blocks -- copy-on-write block copies (P1 §8.3; P3 §2.3 and §5.5).
 * For each pair p, the K half and the V half of block src_dst_pairs[2p] are
 * copied bit-exactly over those of block src_dst_pairs[2p+1].  dtype is the
 * cache's: PKV_F16, PKV_BF16 or PKV_INT8.
 *
 *   src_dst_pairs  [num_pairs][2] int64, device.  Destinations must be
 *                  distinct and must not also appear as sources (otherwise the
 *                  result depends on the order the GPU runs the copies).  An
 *                  entry outside [0, num_blocks) raises PKV_DEVERR_COPY_PAIR
 *                  and that pair is skipped.
 * num_pairs == 0 is a no-op.
 */
PKV_API pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, int64_t num_blocks,
                                   int64_t block_stride_elems, int num_kv_heads, int head_dim,
                                   int block_size, const int64_t *src_dst_pairs,
                                   int64_t num_pairs, pkv_dtype dtype, void *stream);

/* ------------------------------------------------------------------------
 * INT8 KV cache with per-channel scales (P2 §5.2: storing the cache in INT8
 * halves its bytes, and with it the bytes a decode step reads; per-channel
 * scales, computed separately for K and V, are the variant that page
 * recommends).  The pool keeps the layout above with one signed byte per
 * element: [num_blocks][2][num_kv_heads][block_size][head_dim] int8, block
 * strides and offsets counted in elements (= bytes) and a multiple of 16.
 * Scales are caller-owned device arrays k_scale, v_scale of
 * [num_kv_heads][head_dim] fp32, each > 0 and finite (calibrated offline;
 * the library never changes them), 16-byte aligned.
 * A value x (fp16 / bf16) of KV head h, channel c is stored as
 *     code = round_half_even(clamp(x / s[h][c], -127, 127))
 * with the division in IEEE single precision (a NaN input stores -127), and
 * read back as code * s[h][c].
 * ------------------------------------------------------------------------ */

/*
 * pkv_reshape_and_cache_int8 -- pkv_reshape_and_cache into an INT8 cache:
 * each element of the new rows k_new / v_new ([num_tokens][num_kv_heads]
 * [head_dim], dtype = fp16 or bf16) is quantised with its channel's scale and
 * stored at its slot.  Slot rules and errors as pkv_reshape_and_cache.
 */
PKV_API pkv_status pkv_reshape_and_cache_int8(const void *k_new, const void *v_new,
                                              const int64_t *slot_mapping, int64_t num_tokens,
                                              int8_t *k_cache, int8_t *v_cache, int64_t num_blocks,
                                              int64_t block_stride_elems, int num_kv_heads,
                                              int head_dim, int block_size, const float *k_scale,
                                              const float *v_scale, pkv_dtype dtype, void *stream);

/* Workspace of pkv_paged_attention_decode_int8 (same contract as
 * pkv_decode_workspace_bytes). */
PKV_API size_t pkv_decode_int8_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                               int head_dim, int block_size, int max_context_len,
                                               int partition_size);

/*
 * pkv_paged_attention_decode_int8 -- pkv_paged_attention_decode over an INT8
 * cache: the same softmax attention with K_i[t][c] = code * k_scale[h][c] and
 * V_i[t][c] = code * v_scale[h][c].  q and out are `dtype` (fp16 or bf16);
 * accumulation is fp32.  The K scales are folded into the query and the V
 * scales applied once per output channel, so the kernel reads only the codes.
 * Every other argument and the errors are those of pkv_paged_attention_decode;
 * the automatic split is pkv_decode_int8_plan's.
 */
PKV_API pkv_status pkv_paged_attention_decode_int8(
    const void *q, const int8_t *k_cache, const int8_t *v_cache, const float *k_scale,
    const float *v_scale, int64_t num_blocks, int64_t block_stride_elems,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, float scale, void *out, void *workspace, size_t workspace_bytes,
    int partition_size, pkv_dtype dtype, void *stream);

/*
 * pkv_shared_prefix_workspace_bytes -- workspace of
 * pkv_paged_attention_decode_shared_prefix for these arguments on the current
 * device ((size_t)-1 if they are out of contract).
 */
PKV_API size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                                 int head_dim, int block_size, int prefix_len,
                                                 int max_context_len, int partition_size);

/*
 * pkv_paged_attention_decode_shared_prefix -- the same result as
 * pkv_paged_attention_decode for a batch whose sequences all start with the
 * same prefix_len tokens held in the blocks prefix_block_table[0 ..
 * prefix_len/block_size) (prefix caching: P1 §8.2, P3 §2.3 / §3), computed as
 * a cascade: (1) all num_seqs * G query rows of each KV head attend to the
 * prefix together as dense tensor-core tiles, so each prefix block is read once
 * per 128 query rows instead of once per sequence; (2) each sequence attends
 * to its own tokens [prefix_len, context_len); (3) a log-sum-exp merge.
 *
 *   prefix_block_table  [prefix_len / block_size] int32, device.
 *   prefix_len          > 0, a multiple of block_size, <= max_context_len.
 *                       Every context_lens[i] must be >= prefix_len (a shorter
 *                       one raises PKV_DEVERR_CONTEXT_LEN), and every
 *                       block_tables[i] must start with the prefix's blocks
 *                       (or blocks holding the same data).
 *   workspace           >= pkv_shared_prefix_workspace_bytes(...); required.
 * Other arguments as pkv_paged_attention_decode.  head_dim 128 only (else
 * PKV_ERR_UNSUPPORTED).
 */
PKV_API pkv_status pkv_paged_attention_decode_shared_prefix(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    int64_t block_stride_elems, const int32_t *prefix_block_table, int prefix_len,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, float scale, void *out, void *workspace, size_t workspace_bytes,
    int partition_size, pkv_dtype dtype, void *stream);

/*
 * pkv_prefill_workspace_bytes -- workspace of pkv_paged_attention_prefill for
 * these arguments on the current device: 0 when the KV range is not split,
 * (size_t)-1 for arguments out of contract.  kv_splits as in
 * pkv_paged_attention_prefill.
 */
PKV_API size_t pkv_prefill_workspace_bytes(int num_rows, int num_seqs, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size,
                                           int max_query_len, int max_context_len, int kv_splits);

/*
 * pkv_paged_attention_prefill -- chunked prefill attention over the paged
 * cache (P4 §2: with a cache, the new tokens' queries attend to the cached
 * tokens and causally to each other; P2 §2.3 / §5.4: a whole prompt, or a long
 * prompt in chunks).  Sequence i has context_lens[i] = L_i tokens in the
 * cache, the last C_i = query_start[i+1] - query_start[i] of which are its
 * chunk (already written, e.g. by pkv_reshape_and_cache with the chunk's
 * slots).  Chunk row j -- global query row query_start[i] + j, at position
 * p = L_i - C_i + j -- attends to tokens 0 .. p (the causal rule on absolute
 * positions):
 *     out[row, hq] = softmax_t<=p(scale * q[row, hq] . k_t) V,
 * accumulated in fp32 on the tensor cores (tcgen05, 128 query rows x 128
 * tokens per tile; the group's heads of each token share the K/V tiles).
 *
 *   q, out         [num_rows][num_q_heads][head_dim], contiguous, dtype; the
 *                  chunks of all sequences back to back.
 *   query_start    [num_seqs + 1] int32, device: non-decreasing chunk offsets,
 *                  query_start[num_seqs] <= num_rows.
 *   context_lens   [num_seqs] int32, device: L_i >= C_i.
 *   max_query_len, max_context_len   host bounds of C_i and L_i (size the grid;
 *                  a sequence outside them, or with query_start out of order,
 *                  raises PKV_DEVERR_CONTEXT_LEN and its rows are not written).
 *   kv_splits      0 = library's choice; n > 0 splits each row tile's KV range
 *                  into about n pieces of whole 128-token tiles, merged by a
 *                  log-sum-exp pass (workspace needed when the plan splits).
 * Other arguments as pkv_paged_attention_decode; head_dim 128 only (else
 * PKV_ERR_UNSUPPORTED).  A chunk of one token per sequence computes the same
 * attention as pkv_paged_attention_decode.
 */
PKV_API pkv_status pkv_paged_attention_prefill(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    int64_t block_stride_elems, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *query_start, const int32_t *context_lens, int num_rows, int max_query_len,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, float scale, void *out, void *workspace, size_t workspace_bytes,
    int kv_splits, pkv_dtype dtype, void *stream);

/* Size of the library's built-in decode scratch array (per device). */
#define PKV_STATIC_SCRATCH_BYTES (32u << 20) /* 32 MiB */

/*
 * pkv_paged_attention_decode_static_scratch -- pkv_paged_attention_decode for
 * callers that cannot allocate device memory.  The pages have no counterpart:
 * this is a deployment convenience, not part of the method.
 *
 * Who needs it: a caller that has no device memory to give the decode call
 * its split-context workspace -- e.g. a serving engine that reserved nearly
 * all free device memory for its KV block pool up front, or a plug-in whose
 * host framework hands it tensor pointers but no allocator it may call.
 *
 * Arguments and results are those of pkv_paged_attention_decode without the
 * workspace pair; the scratch comes from a PKV_STATIC_SCRATCH_BYTES array
 * inside the library that every device loading the library keeps until the
 * process exits.  The call allocates nothing (no cudaMalloc/cudaFree, no
 * allocating library routine).
 *   - A plan whose scratch (pkv_decode_workspace_bytes for the same
 *     arguments) exceeds PKV_STATIC_SCRATCH_BYTES is rejected with
 *     PKV_ERR_SCRATCH_LIMIT before anything is enqueued; pass a larger
 *     partition_size (fewer partitions) or use the workspace entry point.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents.  Nothing in it needs clearing (every value is written before
 *     it is read), but calls that overlap on the GPU -- e.g. on two streams
 *     with no ordering between them -- race on it and must be serialised by
 *     the caller.
 */
PKV_API pkv_status pkv_paged_attention_decode_static_scratch(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    int64_t block_stride_elems, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, float scale, void *out, int partition_size,
    pkv_dtype dtype, void *stream);

/*
 * pkv_get_device_error -- synchronise `stream`, read the current device's
 * status word into *flags (PKV_DEVERR_* bits; may be NULL) and clear it.
 * Returns PKV_OK when no flag was set, PKV_ERR_DEVICE when one was, and
 * PKV_ERR_CUDA if the read failed.
 */
PKV_API pkv_status pkv_get_device_error(void *stream, uint32_t *flags);

/* Static description of a status code. */
PKV_API const char *pkv_status_string(pkv_status status);

/* Kernel launches this process has made through the library (all calls). */
PKV_API uint64_t pkv_launch_count(void);

/*
 * pkv_decode_plan -- the launch decision pkv_paged_attention_decode makes,
 * as a pure host function (no CUDA call): given the shape and the SM count it
 * writes the partition size, partitions per sequence, query heads handled per
 * block and whether the merge kernel runs.  Returns PKV_OK or the status the
 * decode call would return for these arguments.  A block serves the largest
 * of 16 (head_dim 128), 8, 4, 2, 1 query heads dividing the group.  With
 * partition_size 0 the split aims at eight waves of the kernel form's resident
 * blocks per SM (two for the per-lane form and for 16 heads per block, three
 * for the warp-MMA form of 4 or 8 heads per block), with partitions of at
 * least 256 tokens whose K/V bytes are at least 32 times their partial
 * outputs.  For the forms with two resident blocks per SM, when those floors
 * leave fewer than eight waves, the partition count per max_context_len
 * sequence is the smallest in [n/2, n] (n: the floors' count) whose blocks
 * fill whole waves within 0.15 of the best count in that range.
 */
PKV_API pkv_status pkv_decode_plan(int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, int max_context_len,
                                   int partition_size, int sm_count, int *out_partition_size,
                                   int *out_num_partitions, int *out_heads_per_block,
                                   int *out_needs_merge);

/*
 * pkv_decode_int8_plan -- pkv_decode_plan for pkv_paged_attention_decode_int8
 * (the same rules, with at most 8 heads per block; the INT8 forms keep six
 * (per-lane) or four (warp MMAs) blocks resident per SM, and a token's K/V is
 * half the bytes).
 */
PKV_API pkv_status pkv_decode_int8_plan(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_context_len,
                                        int partition_size, int sm_count, int *out_partition_size,
                                        int *out_num_partitions, int *out_heads_per_block,
                                        int *out_needs_merge);

/*
 * pkv_debug_wait_timeout -- failure-detection self test.  Launches one block
 * that waits, with the library's bounded wait, on an mbarrier that nothing
 * completes; after timeout_ns nanoseconds the wait gives up, raises
 * PKV_DEVERR_TIMEOUT in the status word and the kernel returns normally.
 * timeout_ns must be in (0, 10^10].
 */
PKV_API pkv_status pkv_debug_wait_timeout(uint64_t timeout_ns, void *stream);

/* ------------------------------------------------------------------------
 * Host block manager (no GPU involved): the bookkeeping that produces the
 * inputs of the calls above -- block tables, context lengths, slot mappings
 * and copy-on-write pairs.  P1 §5.2-5.3: a free pool of physical blocks; when
 * token t is appended the sequence needs ceil((t+1)/block_size) blocks, a new
 * block comes from the pool when its table is short, and the token's slot is
 * offset t % block_size of the last block.  P1 §6.2 / §8.2-8.3: finished
 * sequences return their blocks; shared blocks carry a reference count and are
 * freed at zero.  P3 §2.3 / §5.5: a sequence about to write into a block that
 * another sequence references first gets a private copy (a copy-on-write pair
 * for pkv_copy_blocks).  Blocks are handed out 0, 1, 2, ... from a fresh pool
 * and reused last-freed-first.  One manager per thread (not thread-safe).
 * ------------------------------------------------------------------------ */
typedef struct pkv_block_manager pkv_block_manager;

/* NULL on bad sizes (num_blocks in [1, 2^31), block_size >= 1, max_blocks_per_seq >= 1). */
PKV_API pkv_block_manager *pkv_bm_create(int64_t num_blocks, int block_size,
                                         int max_blocks_per_seq);
PKV_API void pkv_bm_destroy(pkv_block_manager *bm);
PKV_API int64_t pkv_bm_num_free(const pkv_block_manager *bm);
/* Reference count of a physical block (0 = free); -1 for a bad block id. */
PKV_API int32_t pkv_bm_refcount(const pkv_block_manager *bm, int64_t block);
/* New empty sequence; PKV_ERR_INVALID_ARG if the id exists. */
PKV_API pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id);
/* New sequence child_id sharing every block of parent_id (reference counts +1),
 * e.g. a beam-search branch. */
PKV_API pkv_status pkv_bm_fork(pkv_block_manager *bm, int64_t parent_id, int64_t child_id);
/* Prefix caching: the empty sequence dst_id starts with src_id's first
 * num_tokens tokens (a multiple of block_size) by sharing their blocks. */
PKV_API pkv_status pkv_bm_share_prefix(pkv_block_manager *bm, int64_t src_id, int64_t dst_id,
                                       int64_t num_tokens);
/* Append one token: *slot receives its slot.  If the sequence's last block was
 * shared, it is replaced by a fresh copy and (*cow_src, *cow_dst) name the copy
 * to perform before the cache write; otherwise both are -1.
 * PKV_ERR_OUT_OF_BLOCKS when a block is needed and the pool is empty (nothing
 * changes); PKV_ERR_INVALID_ARG for an unknown id or a full table. */
PKV_API pkv_status pkv_bm_append_token(pkv_block_manager *bm, int64_t seq_id, int64_t *slot,
                                       int64_t *cow_src, int64_t *cow_dst);
/* Drop a sequence; its blocks' reference counts fall and blocks at zero return
 * to the pool. */
PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id);
/* Tokens held by a sequence (-1 if unknown). */
PKV_API int64_t pkv_bm_seq_len(const pkv_block_manager *bm, int64_t seq_id);
/* Copy a sequence's block table (host int32) into out[capacity]; *num_entries
 * gets its length (also when capacity is too small, which returns
 * PKV_ERR_INVALID_ARG). */
PKV_API pkv_status pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *out,
                                      int capacity, int *num_entries);
/* One decode step for a batch of distinct sequences, all host buffers: appends
 * one token to each and writes slot_mapping[num_seqs], block_tables
 * [num_seqs][max_blocks_per_seq] (unused entries 0), context_lens[num_seqs]
 * (the new token included) and up to num_seqs copy-on-write pairs
 * cow_pairs[*num_cow_pairs][2] -- exactly the inputs of pkv_copy_blocks,
 * pkv_reshape_and_cache and pkv_paged_attention_decode for this step, run in
 * that order.  The pool is checked for the whole step first: on
 * PKV_ERR_OUT_OF_BLOCKS nothing changes. */
PKV_API pkv_status pkv_bm_decode_step(pkv_block_manager *bm, const int64_t *seq_ids,
                                      int num_seqs, int64_t *slot_mapping,
                                      int32_t *block_tables, int32_t *context_lens,
                                      int64_t *cow_pairs, int64_t *num_cow_pairs);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
