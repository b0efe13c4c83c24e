// prefill.cu -- the pkv_paged_attention_prefill entry point (chunked prefill
// attention over the paged cache): argument checks, the row-tile and KV-split
// plan, and the launches of the persistent paged_prefill_tc_kernel and its
// merge.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "prefill_tc_kernel.cuh"
#include "pkv_host.h"

namespace {

constexpr int kMinSplitTokens = 512;  // a KV split covers at least 4 tiles

struct PrefillPlan {
    int tile_tokens = 0;   // chunk tokens per row tile: 128 / group
    int row_tiles = 0;     // row tiles of the longest chunk
    int splits = 0;
    int split_tokens = 0;  // multiple of 128
    int items = 0;         // row_tiles * num_kv_heads * num_seqs * splits
};

pkv_status plan_prefill(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int max_query_len, int max_context_len, int kv_splits,
                        int sm_count, PrefillPlan *pp) {
    if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
        max_query_len < 0 || max_context_len < max_query_len || kv_splits < 0 || sm_count <= 0 ||
        num_kv_heads > 65535)
        return PKV_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    if (group > 128) return PKV_ERR_UNSUPPORTED;  // a row tile holds at least one token
    pp->tile_tokens = 128 / group;
    const int64_t row_tiles = (static_cast<int64_t>(max_query_len) + pp->tile_tokens - 1) / pp->tile_tokens;
    pp->row_tiles = static_cast<int>(row_tiles);
    const int64_t ctx_tiles = std::max<int64_t>(1, (max_context_len + 127) / 128);
    int64_t want = kv_splits;
    if (want == 0) {
        // split the KV range only when the row tiles alone leave SMs idle
        const int64_t units = std::max<int64_t>(1, row_tiles * num_kv_heads * num_seqs);
        want = units >= sm_count ? 1 : (sm_count + units - 1) / units;
        want = std::min<int64_t>(want, std::max<int64_t>(1, max_context_len / kMinSplitTokens));
    }
    want = std::min<int64_t>(want, ctx_tiles);
    const int64_t tiles_per_split = (ctx_tiles + want - 1) / want;
    pp->split_tokens = static_cast<int>(tiles_per_split * 128);
    pp->splits = static_cast<int>((ctx_tiles + tiles_per_split - 1) / tiles_per_split);
    if (static_cast<int64_t>(num_seqs) * pp->splits > 65535) return PKV_ERR_INVALID_ARG;
    const int64_t items = row_tiles * num_kv_heads * num_seqs * pp->splits;  // < 2^63
    if (items > 0x7fffffff) return PKV_ERR_INVALID_ARG;
    pp->items = static_cast<int>(items);
    return PKV_OK;
}

size_t prefill_workspace(int num_rows, int num_q_heads, int splits) {
    if (splits <= 1) return 0;
    return static_cast<size_t>(num_rows) * num_q_heads * splits * (128 + 2) * sizeof(float);
}

template <typename T, int BS, int ORDER>
pkv_status launch_prefill_one(const pkv::PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                              const CUtensorMap &tv, const CUtensorMap &to, int grid, cudaStream_t stream) {
    static std::atomic<uint64_t> configured_devices{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured_devices.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(pkv::paged_prefill_tc_kernel<T, BS, ORDER>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 pkv::PrefillLayout::kSmemBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_devices.fetch_or(bit, std::memory_order_acq_rel);
    }
    pkv::paged_prefill_tc_kernel<T, BS, ORDER>
        <<<grid, pkv::PrefillLayout::kThreads, pkv::PrefillLayout::kSmemBytes, stream>>>(tq, tk, tv, to, p);
    pkv::count_launch();
    return pkv::launch_status();
}

template <typename T, int BS>
pkv_status launch_prefill_bs(const pkv::PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const CUtensorMap &to, int grid, cudaStream_t s) {
    if (p.order == pkv::kOrderSortedGroups)
        return launch_prefill_one<T, BS, pkv::kOrderSortedGroups>(p, tq, tk, tv, to, grid, s);
    if (p.order == pkv::kOrderPairs) return launch_prefill_one<T, BS, pkv::kOrderPairs>(p, tq, tk, tv, to, grid, s);
    return launch_prefill_one<T, BS, pkv::kOrderRowTiles>(p, tq, tk, tv, to, grid, s);
}

template <typename T>
pkv_status launch_prefill(const pkv::PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                          const CUtensorMap &tv, const CUtensorMap &to, int block_size, int grid,
                          int max_query_len, cudaStream_t s) {
    pkv_status st = PKV_ERR_UNSUPPORTED;
    if (block_size == 8) st = launch_prefill_bs<T, 8>(p, tq, tk, tv, to, grid, s);
    else if (block_size == 16) st = launch_prefill_bs<T, 16>(p, tq, tk, tv, to, grid, s);
    else if (block_size == 32) st = launch_prefill_bs<T, 32>(p, tq, tk, tv, to, grid, s);
    if (st != PKV_OK || p.splits == 1) return st;
    const int64_t rows = static_cast<int64_t>(max_query_len) * p.num_q_heads;
    const dim3 mgrid(static_cast<unsigned>((rows + 3) / 4), static_cast<unsigned>(p.num_seqs));
    pkv::paged_prefill_merge_kernel<T><<<mgrid, 128, 0, s>>>(p);
    pkv::count_launch();
    return pkv::launch_status();
}

}  // namespace

extern "C" {

PKV_API size_t pkv_prefill_workspace_bytes(int num_rows, int num_seqs, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size,
                                           int max_query_len, int max_context_len, int kv_splits) {
    const int sm = kv_splits > 0 ? 1 : pkv::current_sm_count();
    if (sm <= 0 || num_rows < 0) return static_cast<size_t>(-1);
    PrefillPlan pp;
    if (plan_prefill(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_query_len,
                     max_context_len, kv_splits, sm, &pp) != PKV_OK)
        return static_cast<size_t>(-1);
    return prefill_workspace(num_rows, num_q_heads, pp.splits);
}

PKV_API pkv_status pkv_paged_attention_prefill(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    int64_t block_stride_elems, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *query_start, const int32_t *context_lens, int num_rows, int max_query_len,
    int max_context_len, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, float scale, void *out, void *workspace, size_t workspace_bytes,
    int kv_splits, pkv_dtype dtype, void *stream) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_rows < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads || num_blocks <= 0 || num_blocks > 0x7fffffffLL ||
        max_blocks_per_seq <= 0 || max_query_len < 0 || max_context_len < max_query_len ||
        static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size ||
        kv_splits < 0 || !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    const int64_t half_elems = static_cast<int64_t>(num_kv_heads) * block_size * head_dim;
    if (block_stride_elems < half_elems || block_stride_elems % 8) return PKV_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_rows == 0 || max_query_len == 0) return PKV_OK;
    if (!q || !out || !block_tables || !query_start || !context_lens || !pkv::aligned16(q) ||
        !pkv::aligned16(out))
        return PKV_ERR_INVALID_ARG;
    PrefillPlan pp;
    // shape first (no CUDA call), then the plan for the real SM count
    pkv_status st = plan_prefill(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_query_len, max_context_len, kv_splits, 1, &pp);
    if (st != PKV_OK) return st;
    int sm = 0;
    if (kv_splits == 0) {
        sm = pkv::current_sm_count();
        if (sm <= 0) return PKV_ERR_CUDA;
        st = plan_prefill(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_query_len,
                          max_context_len, 0, sm, &pp);
        if (st != PKV_OK) return st;
    }
    const size_t need = prefill_workspace(num_rows, num_q_heads, pp.splits);
    if (need > 0 && (!workspace || workspace_bytes < need || !pkv::aligned16(workspace)))
        return PKV_ERR_INVALID_ARG;
    unsigned int *status = pkv::status_word_ptr();
    if (!status) return PKV_ERR_CUDA;
    if (sm == 0) sm = pkv::current_sm_count();
    if (sm <= 0) return PKV_ERR_CUDA;
    const int group = num_q_heads / num_kv_heads;
    // the output has the queries' shape: full row tiles leave through the same boxes
    CUtensorMap tq, tk, tv, to;
    if (!pkv::encode_query_map(&tq, q, num_rows, num_q_heads, group, pp.tile_tokens, dtype) ||
        !pkv::encode_query_map(&to, out, num_rows, num_q_heads, group, pp.tile_tokens, dtype) ||
        !pkv::encode_half_map(&tk, k_cache, num_blocks, block_stride_elems, num_kv_heads, block_size,
                              dtype, 0) ||
        !pkv::encode_half_map(&tv, v_cache, num_blocks, block_stride_elems, num_kv_heads, block_size,
                              dtype, 0))
        return PKV_ERR_CUDA;

    pkv::PrefillParams p{};
    p.q = q;
    p.out = out;
    const size_t slots = static_cast<size_t>(num_rows) * num_q_heads * pp.splits;
    p.ws_o = need ? static_cast<float *>(workspace) : nullptr;
    p.ws_m = need ? p.ws_o + slots * head_dim : nullptr;
    p.ws_l = need ? p.ws_m + slots : nullptr;
    p.block_tables = block_tables;
    p.query_start = query_start;
    p.context_lens = context_lens;
    p.status = status;
    p.num_blocks = num_blocks;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.len_cap = max_context_len;
    p.qlen_cap = max_query_len;
    p.num_rows = num_rows;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = group;
    p.tile_tokens = pp.tile_tokens;
    p.tile_rows = pp.tile_tokens * group;
    p.row_tiles = pp.row_tiles;
    p.num_items = pp.items;
    p.splits = pp.splits;
    p.split_tokens = pp.split_tokens;
    p.div_row_tiles = pkv::make_fast_div(p.row_tiles);
    p.div_kv_heads = pkv::make_fast_div(num_kv_heads);
    p.div_group = pkv::make_fast_div(group);
    p.div_splits = pkv::make_fast_div(p.splits);
    p.div_per_tile = pkv::make_fast_div(num_kv_heads * num_seqs * p.splits);
    // item order (prefill_item): whole prompts of one length (every chunk
    // max_query_len tokens on an empty cache) in row-tile pairs, a few sequences of
    // different lengths by (sequence, KV head) sorted by length, both for L2 reuse
    // of each (sequence, KV head)'s K/V tiles; otherwise row tiles, heaviest first
    const bool whole_prompts = num_rows == static_cast<int64_t>(num_seqs) * max_query_len &&
                               max_context_len == max_query_len;
    p.order = pp.splits != 1 ? pkv::kOrderRowTiles
              : whole_prompts ? pkv::kOrderPairs
              : num_seqs <= pkv::kSortedGroupsMaxSeqs ? pkv::kOrderSortedGroups
                                                      : pkv::kOrderRowTiles;
    p.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    // persistent: one CTA per SM (or per item when there are fewer)
    const int grid = std::min(pp.items, sm);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == PKV_F16
               ? launch_prefill<__half>(p, tq, tk, tv, to, block_size, grid, max_query_len, s)
               : launch_prefill<__nv_bfloat16>(p, tq, tk, tv, to, block_size, grid, max_query_len, s);
}

}  // extern "C"
