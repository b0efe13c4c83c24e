// decode.cu -- the pkv_paged_attention_decode entry point: argument checks,
// the split-context plan, workspace layout, and the launch.
#include <algorithm>
#include <cmath>

#include "decode_launch.cuh"

namespace pkv {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// 3-D view of one half (K or V) of the pool: (head_dim, num_kv_heads*block_size
// rows, num_blocks) with the caller's block stride; boxes are box_rows rows of one
// head (0: a whole block's), 64 columns wide, 128-byte swizzled.
bool encode_half_map(CUtensorMap *map, const void *base, int64_t num_blocks,
                     int64_t block_stride_elems, int num_kv_heads, int block_size, pkv_dtype dt,
                     int box_rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(num_kv_heads) * block_size,
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(block_stride_elems) * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows > 0 ? box_rows : block_size), 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return fn(map, dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
              3, const_cast<void *>(base), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of one half (K or V) of an INT8 pool with head_dim 128: (128 codes,
// num_kv_heads*block_size rows, num_blocks) with the caller's block stride;
// boxes are one block's rows of one head (128 bytes each), 128-byte swizzled.
bool encode_i8_half_map(CUtensorMap *map, const void *base, int64_t num_blocks,
                        int64_t block_stride_elems, int num_kv_heads, int block_size) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(num_kv_heads) * block_size,
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(block_stride_elems)};
    const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(block_size), 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of the prefill queries [num_rows][num_q_heads][128]: boxes of
// `tokens` tokens x `group` heads x 64 columns, 128-byte swizzled, so a box
// lands as tokens * group consecutive 128-byte rows (token-major).
bool encode_query_map(CUtensorMap *map, const void *q, int num_rows, int num_q_heads, int group,
                      int tokens, pkv_dtype dt) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(num_q_heads),
                                static_cast<cuuint64_t>(num_rows)};
    const cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(num_q_heads) * 128 * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tokens)};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return fn(map, dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
              3, const_cast<void *>(q), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pkv

namespace {

constexpr int kTargetWaves = 8;        // CTA waves the automatic split aims for
constexpr int kMinAutoPartition = 256; // tokens: below this the per-CTA set-up dominates
constexpr int kMergeShare = 32;        // a partition's K/V bytes >= this x its partial bytes
constexpr double kFillSlack = 0.15;    // wave fill given up for fewer, longer partitions (two-per-SM forms)

// Decode CTAs resident per SM for each kernel form (their stage budgets and
// register counts): 16-bit per-lane loops two, 16-bit warp MMAs three (two with
// 16 heads per block), INT8 per-lane loops six, INT8 warp MMAs four.
int resident_ctas_per_sm(bool int8_kv, int heads_per_block) {
    if (int8_kv) return heads_per_block >= 4 ? 4 : 6;
    if (heads_per_block == 16) return 2;
    return heads_per_block >= 4 ? 3 : 2;
}
// Query heads per CTA: the largest of 16 (16-bit caches at head_dim 128), 8, 4, 2, 1
// dividing the group (4 to 16 run the products as warp-level MMAs, 1 or 2 as
// per-lane loops).
int heads_per_block_for(int group, bool int8_kv, int head_dim) {
    if (!int8_kv && head_dim == 128 && group % 16 == 0) return 16;
    if (group % 8 == 0) return 8;
    if (group % 4 == 0) return 4;
    if (group % 2 == 0) return 2;
    return 1;
}

size_t workspace_for(int num_seqs, int num_q_heads, int head_dim, int num_partitions) {
    if (num_partitions <= 1) return 0;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * num_partitions;
    return rows * (static_cast<size_t>(head_dim) + 2) * sizeof(float);
}

// The launch plan of a decode call over a 16-bit or an INT8 cache.
// `resident` overrides the form's resident CTAs per SM in the automatic split
// (0: the form's own count).
pkv_status plan_decode(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int max_context_len, int partition_size, int sm_count,
                       bool int8_kv, int *out_partition_size, int *out_num_partitions,
                       int *out_heads_per_block, int *out_needs_merge, int resident = 0) {
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0 ||
        partition_size < 0 || sm_count <= 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
    if (partition_size % block_size) return PKV_ERR_INVALID_ARG;
    const int max_partition = pkv::DecodeGeom<128, 16>::kMaxTableEntries * block_size;
    if (partition_size > max_partition) return PKV_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    const int gh = heads_per_block_for(group, int8_kv, head_dim);
    const int64_t grid_y = static_cast<int64_t>(num_kv_heads) * (group / gh);
    if (grid_y > 65535 || num_seqs > 65535) return PKV_ERR_INVALID_ARG;

    int part = partition_size;
    if (part == 0) {
        // Enough CTAs for kTargetWaves waves of the form's resident CTAs over every
        // SM, but partitions no shorter than kMinAutoPartition tokens, nor so short
        // that the partial outputs (GH rows of head_dim + 2 floats, written and read
        // back by the merge) pass 1 / kMergeShare of the partition's K/V bytes.
        const int64_t units = std::max<int64_t>(1, static_cast<int64_t>(num_seqs) * grid_y);
        const int64_t slots = static_cast<int64_t>(sm_count) *
                              (resident > 0 ? resident : resident_ctas_per_sm(int8_kv, gh));
        const int64_t target = slots * kTargetWaves;
        const int64_t want = std::max<int64_t>(1, (target + units - 1) / units);
        const int64_t len = max_context_len;
        int64_t p = (len + want - 1) / want;
        const int64_t kv_per_token = 2LL * head_dim * (int8_kv ? 1 : 2);
        const int64_t partial = 2LL * gh * (head_dim + 2) * 4;
        p = std::max<int64_t>(p, kMinAutoPartition);
        p = std::max<int64_t>(p, (kMergeShare * partial + kv_per_token - 1) / kv_per_token);
        p = (p + block_size - 1) / block_size * block_size;
        p = std::min<int64_t>(p, max_partition);
        // When the floors leave fewer than kTargetWaves waves of a form with two
        // resident CTAs per SM, the CTAs of sequences at max_context_len run in a few
        // rounds: a last round that fills few slots idles most SMs, and each CTA's
        // start-up costs its SM half its streams.  Take the fewest partitions in
        // [n / 2, n] whose CTAs fill whole waves within kFillSlack of the best count.
        const int64_t n = len > 0 ? (len + p - 1) / p : 1;
        if (n > 1 && units * n < target && slots <= 2LL * sm_count) {
            auto fill = [&](int64_t parts) {  // CTAs / (rounds x slots)
                const int64_t ctas = units * parts;
                return static_cast<double>(ctas) / static_cast<double>((ctas + slots - 1) / slots * slots);
            };
            auto part_for = [&](int64_t k) {  // tokens per partition for k partitions
                return ((len + k - 1) / k + block_size - 1) / block_size * block_size;
            };
            double best = fill(n);
            for (int64_t k = (n + 1) / 2; k < n; ++k)
                if (part_for(k) <= max_partition) best = std::max(best, fill((len + part_for(k) - 1) / part_for(k)));
            for (int64_t k = (n + 1) / 2; k < n; ++k) {
                const int64_t pk = part_for(k);
                if (pk <= max_partition && fill((len + pk - 1) / pk) >= best - kFillSlack) {
                    p = pk;
                    break;
                }
            }
        }
        part = static_cast<int>(p);
    }
    const int nparts = max_context_len > 0 ? (max_context_len + part - 1) / part : 1;
    if (out_partition_size) *out_partition_size = part;
    if (out_num_partitions) *out_num_partitions = nparts;
    if (out_heads_per_block) *out_heads_per_block = gh;
    if (out_needs_merge) *out_needs_merge = nparts > 1 ? 1 : 0;
    return PKV_OK;
}

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_context_len, int partition_size, bool int8_kv) {
    const int sm = partition_size > 0 ? 1 : pkv::current_sm_count();
    if (sm <= 0) return static_cast<size_t>(-1);
    int part = 0, nparts = 0, gh = 0, merge = 0;
    if (plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                    partition_size, sm, int8_kv, &part, &nparts, &gh, &merge) != PKV_OK)
        return static_cast<size_t>(-1);
    return workspace_for(num_seqs, num_q_heads, head_dim, nparts);
}

// Tensor maps of the swizzled warp-MMA staging: INT8 boxes of one block's token
// rows (128 codes each); 16-bit boxes of one stage's token rows (min(block_size,
// 16)) by 64 channels.
bool encode_decode_maps(pkv::DecodeMaps *maps, const void *k_cache, const void *v_cache,
                        bool int8_kv, int64_t num_blocks, int64_t block_stride_elems,
                        int num_kv_heads, int block_size, pkv_dtype dtype) {
    if (int8_kv)
        return pkv::encode_i8_half_map(&maps->k, k_cache, num_blocks, block_stride_elems, num_kv_heads,
                                       block_size) &&
               pkv::encode_i8_half_map(&maps->v, v_cache, num_blocks, block_stride_elems, num_kv_heads,
                                       block_size);
    const int rows = std::min(block_size, 16);
    return pkv::encode_half_map(&maps->k, k_cache, num_blocks, block_stride_elems, num_kv_heads,
                                block_size, dtype, rows) &&
           pkv::encode_half_map(&maps->v, v_cache, num_blocks, block_stride_elems, num_kv_heads,
                                block_size, dtype, rows);
}

// Decode over a 16-bit cache (k_scale == v_scale == nullptr) or an INT8 cache
// with per-channel scales.  Element strides and offsets count cache elements.
pkv_status decode_impl(const void *q, const void *k_cache, const void *v_cache,
                       const float *k_scale, const float *v_scale, bool int8_kv,
                       int64_t num_blocks, int64_t block_stride_elems,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, int max_context_len, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       float scale, void *out, void *workspace, size_t workspace_bytes,
                       int partition_size, pkv_dtype dtype, void *stream) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0 ||
        static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size ||
        !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    const int64_t half_elems = static_cast<int64_t>(num_kv_heads) * block_size * head_dim;
    // block starts 16-byte aligned: 8 16-bit elements or 16 INT8 codes
    if (block_stride_elems < half_elems || block_stride_elems % (int8_kv ? 16 : 8))
        return PKV_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    if (int8_kv && (!k_scale || !v_scale || !pkv::aligned16(k_scale) || !pkv::aligned16(v_scale)))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !out || !block_tables || !context_lens || !pkv::aligned16(q) || !pkv::aligned16(out))
        return PKV_ERR_INVALID_ARG;

    int part = 0, nparts = 0, gh = 0, merge = 0;
    // Validate the shape first (no CUDA call), then plan for the real SM count.
    pkv_status plan = plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                  max_context_len, partition_size, 1, int8_kv, &part, &nparts, &gh,
                                  &merge);
    if (plan != PKV_OK) return plan;
    if (partition_size == 0) {
        const int sm = pkv::current_sm_count();
        if (sm <= 0) return PKV_ERR_CUDA;
        plan = plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_context_len, 0, sm, int8_kv, &part, &nparts, &gh, &merge);
        if (plan != PKV_OK) return plan;
    }
    const size_t need = workspace_for(num_seqs, num_q_heads, head_dim, nparts);
    if (need > 0 && (!workspace || workspace_bytes < need || !pkv::aligned16(workspace)))
        return PKV_ERR_INVALID_ARG;
    unsigned int *status = pkv::status_word_ptr();
    if (!status) return PKV_ERR_CUDA;

    const int group = num_q_heads / num_kv_heads;
    pkv::DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.out = out;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * nparts;
    p.ws_o = need ? static_cast<float *>(workspace) : nullptr;
    p.ws_m = need ? p.ws_o + rows * head_dim : nullptr;
    p.ws_l = need ? p.ws_m + rows : nullptr;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.status = status;
    p.num_blocks = num_blocks;
    p.block_stride = block_stride_elems;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.len_cap = max_context_len;  // <= max_blocks_per_seq * block_size (checked above)
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.group = group;
    p.subgroups = group / gh;
    p.items_y = num_kv_heads * p.subgroups;
    p.partition_size = part;
    p.num_partitions = nparts;
    p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)

    const int merge_rows = merge ? num_seqs * num_q_heads : 0;
    p.trigger_dependents = merge_rows > 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid(static_cast<unsigned>(nparts), static_cast<unsigned>(num_kv_heads * p.subgroups),
                    static_cast<unsigned>(num_seqs));
    // The warp-MMA forms at head_dim 128 (4, 8 or 16 heads per block) stage K/V tiles by
    // tiled TMA copies with a 128-byte swizzle
    pkv::DecodeMaps maps{};
    if (head_dim == 128 && gh >= 4 &&
        !encode_decode_maps(&maps, k_cache, v_cache, int8_kv, num_blocks, block_stride_elems,
                            num_kv_heads, block_size, dtype))
        return PKV_ERR_CUDA;
    if (int8_kv)
        return dtype == PKV_F16
                   ? pkv::launch_decode_i8_f16(p, maps, head_dim, block_size, gh, grid, merge_rows, s)
                   : pkv::launch_decode_i8_bf16(p, maps, head_dim, block_size, gh, grid, merge_rows, s);
    return dtype == PKV_F16
               ? pkv::launch_decode_f16(p, maps, head_dim, block_size, gh, grid, merge_rows, s)
               : pkv::launch_decode_bf16(p, maps, head_dim, block_size, gh, grid, merge_rows, s);
}

}  // namespace

extern "C" {

PKV_API pkv_status pkv_decode_plan(int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, int max_context_len,
                                   int partition_size, int sm_count, int *out_partition_size,
                                   int *out_num_partitions, int *out_heads_per_block,
                                   int *out_needs_merge) {
    return plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       max_context_len, partition_size, sm_count, false, out_partition_size,
                       out_num_partitions, out_heads_per_block, out_needs_merge);
}

PKV_API pkv_status pkv_decode_int8_plan(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_context_len,
                                        int partition_size, int sm_count, int *out_partition_size,
                                        int *out_num_partitions, int *out_heads_per_block,
                                        int *out_needs_merge) {
    return plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       max_context_len, partition_size, sm_count, true, out_partition_size,
                       out_num_partitions, out_heads_per_block, out_needs_merge);
}

PKV_API size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, int max_context_len,
                                          int partition_size) {
    return decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                  max_context_len, partition_size, false);
}

PKV_API pkv_status pkv_paged_attention_decode(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    int64_t block_stride_elems, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, float scale, void *out, void *workspace,
    size_t workspace_bytes, int partition_size, pkv_dtype dtype, void *stream) {
    return decode_impl(q, k_cache, v_cache, nullptr, nullptr, false, num_blocks,
                       block_stride_elems, block_tables, max_blocks_per_seq, context_lens,
                       max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       scale, out, workspace, workspace_bytes, partition_size, dtype, stream);
}

PKV_API size_t pkv_decode_int8_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                               int head_dim, int block_size, int max_context_len,
                                               int partition_size) {
    return decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                  max_context_len, partition_size, true);
}

PKV_API pkv_status pkv_paged_attention_decode_int8(
    const void *q, const int8_t *k_cache, const int8_t *v_cache, const float *k_scale,
    const float *v_scale, int64_t num_blocks, int64_t block_stride_elems,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, float scale, void *out, void *workspace, size_t workspace_bytes,
    int partition_size, pkv_dtype dtype, void *stream) {
    return decode_impl(q, k_cache, v_cache, k_scale, v_scale, true, num_blocks,
                       block_stride_elems, block_tables, max_blocks_per_seq, context_lens,
                       max_context_len, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       scale, out, workspace, workspace_bytes, partition_size, dtype, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Shared-prefix (cascade) decode.
// ---------------------------------------------------------------------------
namespace {

#ifndef PKV_PREFIX_SM_SHARE
#define PKV_PREFIX_SM_SHARE 5
#endif
constexpr int kPrefixSmShare = PKV_PREFIX_SM_SHARE;  // prefix CTAs ~ SMs / this
constexpr int kCascadeSuffixResident = 2;            // suffix split: see plan_cascade

struct CascadePlan {
    int rows = 0;          // num_seqs * group
    int row_tiles = 0;     // of 128 query rows
    int splits = 0;        // prefix splits (workspace slots 0 .. splits-1)
    int split_tokens = 0;  // multiple of 128
    int suffix_part = 0;   // suffix partition size
    int suffix_parts = 0;  // suffix partitions of the longest sequence
    int gh = 0;            // suffix kernel's heads per block
};

pkv_status plan_cascade(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int prefix_len, int max_context_len, int partition_size,
                        int sm_count, CascadePlan *cp) {
    if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
        prefix_len <= 0 || prefix_len % block_size || prefix_len > max_context_len ||
        sm_count <= 0)
        return PKV_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    cp->rows = num_seqs * group;
    cp->row_tiles = (cp->rows + 127) / 128;
    if (cp->row_tiles > 0x7fffffff / 2 || num_kv_heads > 65535) return PKV_ERR_INVALID_ARG;
    // The prefix CTAs (one per SM: their shared memory fills it) run beside the
    // suffix decode, which overlaps them: split the prefix, in whole 128-token
    // tiles, only as far as about sm_count / kPrefixSmShare CTAs, so the suffix
    // keeps most SMs and each prefix CTA runs enough tiles to amortise its set-up.
    const int tiles = (prefix_len + 127) / 128;
    const int64_t units = static_cast<int64_t>(cp->row_tiles) * num_kv_heads;
    const int64_t want = std::max(1, sm_count / kPrefixSmShare);
    int splits = static_cast<int>(std::min<int64_t>(tiles, std::max<int64_t>(1, (want + units - 1) / units)));
    const int tiles_per_split = (tiles + splits - 1) / splits;
    cp->split_tokens = tiles_per_split * 128;
    cp->splits = (prefix_len + cp->split_tokens - 1) / cp->split_tokens;
    if (cp->splits > 65535) return PKV_ERR_INVALID_ARG;
    // the suffix: the decode plan over the longest suffix, its split sized as for
    // two resident CTAs per SM (the prefix tiles hold some SMs meanwhile; measured
    // faster than the form's own three)
    const int span = max_context_len - prefix_len;
    int part = 0, nparts = 0, gh = 0, merge = 0;
    const pkv_status st = plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                      std::max(span, 1), partition_size, sm_count, false, &part,
                                      &nparts, &gh, &merge, kCascadeSuffixResident);
    if (st != PKV_OK) return st;
    cp->suffix_part = part;
    cp->suffix_parts = nparts;
    cp->gh = gh;
    return PKV_OK;
}

}  // namespace

extern "C" {

PKV_API size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                                 int head_dim, int block_size, int prefix_len,
                                                 int max_context_len, int partition_size) {
    const int sm = pkv::current_sm_count();
    if (sm <= 0) return static_cast<size_t>(-1);
    CascadePlan cp;
    if (plan_cascade(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, prefix_len,
                     max_context_len, partition_size, sm, &cp) != PKV_OK)
        return static_cast<size_t>(-1);
    const size_t slots = static_cast<size_t>(cp.splits + cp.suffix_parts);
    return static_cast<size_t>(num_seqs) * num_q_heads * slots * (head_dim + 2) * sizeof(float);
}

PKV_API pkv_status pkv_paged_attention_decode_shared_prefix(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    int64_t block_stride_elems, const int32_t *prefix_block_table, int prefix_len,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, float scale, void *out, void *workspace, size_t workspace_bytes,
    int partition_size, pkv_dtype dtype, void *stream) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_seqs <= 0 || num_blocks <= 0 || num_blocks > 0x7fffffffLL || max_blocks_per_seq <= 0 ||
        max_context_len < 0 ||
        static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size ||
        !std::isfinite(scale) || partition_size < 0 || partition_size % block_size)
        return PKV_ERR_INVALID_ARG;
    const int64_t half_elems = static_cast<int64_t>(num_kv_heads) * block_size * head_dim;
    if (num_kv_heads <= 0 || block_stride_elems < half_elems || block_stride_elems % 8)
        return PKV_ERR_INVALID_ARG;
    if (!q || !out || !k_cache || !v_cache || !block_tables || !context_lens || !prefix_block_table ||
        !workspace || !pkv::aligned16(q) || !pkv::aligned16(out) || !pkv::aligned16(k_cache) ||
        !pkv::aligned16(v_cache) || !pkv::aligned16(workspace))
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || num_q_heads % num_kv_heads || prefix_len <= 0 ||
        prefix_len % block_size || prefix_len > max_context_len)
        return PKV_ERR_INVALID_ARG;
    const int sm = pkv::current_sm_count();
    if (sm <= 0) return PKV_ERR_CUDA;
    CascadePlan cp;
    pkv_status st = plan_cascade(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 prefix_len, max_context_len, partition_size, sm, &cp);
    if (st != PKV_OK) return st;
    const int slots = cp.splits + cp.suffix_parts;
    const size_t need = static_cast<size_t>(num_seqs) * num_q_heads * slots * (head_dim + 2) * sizeof(float);
    if (workspace_bytes < need) return PKV_ERR_INVALID_ARG;
    unsigned int *status = pkv::status_word_ptr();
    if (!status) return PKV_ERR_CUDA;
    CUtensorMap tk, tv;
    if (!pkv::encode_half_map(&tk, k_cache, num_blocks, block_stride_elems, num_kv_heads, block_size, dtype, 0) ||
        !pkv::encode_half_map(&tv, v_cache, num_blocks, block_stride_elems, num_kv_heads, block_size, dtype, 0))
        return PKV_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int group = num_q_heads / num_kv_heads;
    const size_t rows_ws = static_cast<size_t>(num_seqs) * num_q_heads * slots;
    float *ws_o = static_cast<float *>(workspace);
    float *ws_m = ws_o + rows_ws * head_dim;
    float *ws_l = ws_m + rows_ws;

    // 1. every query row of a KV head over the shared prefix (dense, tensor cores)
    pkv::PrefixParams pp{};
    pp.q = q;
    pp.ws_o = ws_o;
    pp.ws_m = ws_m;
    pp.ws_l = ws_l;
    pp.prefix_table = prefix_block_table;
    pp.context_lens = context_lens;
    pp.status = status;
    pp.num_blocks = num_blocks;
    pp.num_seqs = num_seqs;
    pp.num_q_heads = num_q_heads;
    pp.group = group;
    pp.rows = cp.rows;
    pp.prefix_len = prefix_len;
    pp.split_tokens = cp.split_tokens;
    pp.num_partitions = slots;
    pp.scale_log2 = scale * 1.4426950408889634f;
    const dim3 pgrid(static_cast<unsigned>(cp.row_tiles), static_cast<unsigned>(num_kv_heads),
                     static_cast<unsigned>(cp.splits));
    st = dtype == PKV_F16 ? pkv::launch_prefix_tc_f16(pp, tk, tv, block_size, pgrid, s)
                          : pkv::launch_prefix_tc_bf16(pp, tk, tv, block_size, pgrid, s);
    if (st != PKV_OK) return st;

    // 2. each sequence's own tokens after the prefix, into the following slots: a
    //    programmatic dependent launch that runs beside step 1 on the SMs it leaves
    //    free (the two write disjoint slots); the grid completes only after step 1
    // 3. the log-sum-exp merge of all slots, behind step 2
    pkv::DecodeParams p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.out = out;
    p.ws_o = ws_o;
    p.ws_m = ws_m;
    p.ws_l = ws_l;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.status = status;
    p.num_blocks = num_blocks;
    p.block_stride = block_stride_elems;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.len_cap = max_context_len;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.group = group;
    p.subgroups = group / cp.gh;
    p.items_y = num_kv_heads * p.subgroups;
    p.partition_size = cp.suffix_part;
    p.num_partitions = slots;
    p.scale_log2 = pp.scale_log2;
    p.tok_begin = prefix_len;
    p.slot_base = cp.splits;
    p.always_partial = 1;
    p.wait_prior_grid = 1;  // overlaps the prefix tiles; the merge still follows both
    p.trigger_dependents = 1;
    const int merge_rows = num_seqs * num_q_heads;
    const dim3 grid(static_cast<unsigned>(cp.suffix_parts), static_cast<unsigned>(p.items_y),
                    static_cast<unsigned>(num_seqs));
    pkv::DecodeMaps maps{};
    if (cp.gh >= 4 && !encode_decode_maps(&maps, k_cache, v_cache, false, num_blocks, block_stride_elems,
                                          num_kv_heads, block_size, dtype))
        return PKV_ERR_CUDA;
    return dtype == PKV_F16
               ? pkv::launch_decode_f16(p, maps, head_dim, block_size, cp.gh, grid, merge_rows, s)
               : pkv::launch_decode_bf16(p, maps, head_dim, block_size, cp.gh, grid, merge_rows, s);
}

}  // extern "C"
