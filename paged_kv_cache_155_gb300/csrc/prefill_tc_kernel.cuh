// prefill_tc_kernel.cuh -- chunked prefill attention over the paged cache.
//
// "大模型 (LLM) 推理加速核心技术解析" §2 (causal self-attention with a cache):
// the new tokens' K and V join the cache, then each new token's query attends
// to the cached tokens and, causally, to the new tokens up to itself; "KV Cache
// 从原理到实战" §2.3 / §5.4: a whole prompt at once (prefill), or a long prompt
// in pieces (chunked prefill).  Sequence i holds L_i tokens in the cache, the
// last C_i of which are its chunk; chunk row j (global query row
// query_start[i] + j) sits at position L_i - C_i + j and attends to tokens
// 0 .. that position.
//
// Work item: the query rows of one row tile of one sequence and one KV head --
// row r of the sequence's rows is chunk token r / G, query head r % G of the
// group, so a KV tile is shared by the G heads of every token in the tile; a
// row tile holds 128 / G whole tokens (R = G * (128 / G) <= 128 rows) -- over
// one split of the KV range (all of it unless the row tiles alone would leave
// SMs idle).  The KV range ends at the causal limit of the tile's last row;
// inside a tile a row's columns past its own position are masked.  Same
// machinery as the shared-prefix tile kernel: tcgen05 MMAs with M = 128 rows,
// N = 128 tokens, K = 128; S triple-buffered in TMEM, O accumulated in TMEM; a
// row's softmax is local to one thread pair (its scores are read from TMEM once
// per tile); the row's reference maximum moves only when a tile exceeds it by
// more than kRescaleLog2.  The row sum l adds the fp32 weights whose bf16/fp16
// roundings feed the PV MMA (unbiased rounding, relative error 2^-9 per weight
// at most).  With one split the kernel writes the normalised output; with
// several it writes (o, m, l) partials that paged_prefill_merge_kernel
// combines.
//
// Persistent CTAs, one per SM: CTA c takes items c, c + grid, ... of a static
// order with the heaviest row tiles (longest causal range) first, which
// balances the SMs without a shared counter.  Every role walks the same item
// list and counts tiles across items, so the rings and barriers run on from
// one item to the next: the queries of the next item (a TMA load into the Q
// buffer as soon as the last QK^T of the current item has read it) and its
// first K/V tiles and S = QK^T are in flight while the softmax warps still
// write out the current item.  With one Q buffer the K and V rings hold three
// tiles each (measured: faster than two Q buffers with two-slot rings).
//
// Warps: 0 / 10 TMA producers of the K / V rings (PrefillLayout::kKS / kVS
// slots; warp 0 also loads each item's Q tile), 1 TMEM owner + QK^T issuer,
// 11 PV issuer, 2-9 softmax in pairs: warps w and w + 4 share TMEM lane
// quarter w & 3 (the same 32 query rows) and take tile columns 0-63 and
// 64-127.  A pair exchanges its partial row maxima each tile through two
// columns of the tile's own S buffer whose scores are already read (an
// mbarrier with a bounded wait orders them), so both warps hold the same
// reference maximum; each rescales, writes P for and outputs its own half.
// P goes back into TMEM over the scores it came from (16-bit values packed two
// per column) and the PV MMA takes it from there, so P is triple-buffered with
// S: QK^T(j + 3) waits only for PV(j), and the softmax of tile j + 1 runs
// while PV(j) does.
#pragma once

#include "prefix_tc_kernel.cuh"

namespace pkv {

// Division of a non-negative int by a fixed positive divisor through one multiplication
// (Granlund and Montgomery, "Division by Invariant Integers using Multiplication", 1994,
// the form with a 33-bit add): l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, and
// n / d = (umulhi(m, n) + n) >> l for 0 <= n < 2^31 (umulhi(m, n) < n, so the add does
// not wrap).  The item arithmetic divides by the same few launch constants in every role.
struct FastDiv {
    uint32_t m, l;
};
inline FastDiv make_fast_div(int d) {
    if (d < 1) d = 1;  // no launch divides by less (empty launches return before)
    uint32_t l = 0;
    while ((1ull << l) < static_cast<uint64_t>(d)) ++l;
    const uint64_t m = (1ull << 32) * ((1ull << l) - static_cast<uint64_t>(d)) / static_cast<uint64_t>(d) + 1;
    return FastDiv{static_cast<uint32_t>(m), l};
}
__device__ __forceinline__ int fast_div(int n, FastDiv f) {
    return static_cast<int>((__umulhi(static_cast<uint32_t>(n), f.m) + static_cast<uint32_t>(n)) >> f.l);
}

struct PrefillParams {
    const void *q;                 // [num_rows][num_q_heads][128]
    void *out;                     // [num_rows][num_q_heads][128]
    float *ws_o;                   // [num_rows * num_q_heads][splits][128] (splits > 1)
    float *ws_m;                   // [num_rows * num_q_heads][splits] (log2 units)
    float *ws_l;
    const int32_t *block_tables;   // [num_seqs][max_blocks_per_seq]
    const int32_t *query_start;    // [num_seqs + 1]
    const int32_t *context_lens;   // [num_seqs], chunk included
    unsigned int *status;
    int64_t num_blocks;
    int max_blocks_per_seq;
    int len_cap;       // host bound of context_lens (<= max_blocks_per_seq * block_size)
    int qlen_cap;      // host bound of the chunk lengths
    int num_rows;      // query_start[num_seqs] as given by the host
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int tile_tokens;   // chunk tokens per row tile: 128 / group
    int tile_rows;     // query rows per row tile: tile_tokens * group
    int row_tiles;     // row tiles of the longest chunk
    int num_items;     // row_tiles * num_kv_heads * num_seqs * splits
    int splits;        // KV splits per row tile
    int split_tokens;  // tokens per split, a multiple of 128
    int order;         // item order: kOrderRowTiles, kOrderPairs or kOrderSortedGroups
    FastDiv div_row_tiles, div_kv_heads, div_group, div_splits, div_per_tile;  // make_fast_div of
                       // row_tiles, num_kv_heads, group, splits, num_kv_heads * num_seqs * splits
    float scale_log2;
};

// Item orders (PrefillParams::order), see prefill_item.
constexpr int kOrderRowTiles = 0, kOrderPairs = 1, kOrderSortedGroups = 2;
constexpr int kSortedGroupsMaxSeqs = 32;  // sequences a block ranks by length itself

// One sequence's chunk start, chunk end and context length, as read from the
// device arrays.
struct PrefillSeqVals {
    int q0, q1, len;
};

// The sequence of item i (no global-memory access).  by_len: the sequences by
// context length, longest first (sorted-groups order only).
// ORDER: the item order (each compiled apart, so no order's code is shaped by the
// others').
template <int ORDER>
__device__ __forceinline__ int prefill_item_seq(const PrefillParams &p, int i, const unsigned char *by_len) {
    if constexpr (ORDER == kOrderSortedGroups)
        return by_len[fast_div(fast_div(i, p.div_row_tiles), p.div_kv_heads)];
    if constexpr (ORDER == kOrderPairs) return fast_div(fast_div(i, p.div_row_tiles), p.div_kv_heads);
    const int per_tile = p.num_kv_heads * p.num_seqs * p.splits;
    const int rem = i - fast_div(i, p.div_per_tile) * per_tile;
    return fast_div(fast_div(rem, p.div_kv_heads), p.div_splits);
}

// Loads item i's sequence values (zeros past the item count).
template <int ORDER>
__device__ __forceinline__ PrefillSeqVals prefill_seq_vals(const PrefillParams &p, int i,
                                                          const unsigned char *by_len) {
    PrefillSeqVals v{0, 0, 0};
    if (i < p.num_items) {
        const int seq = prefill_item_seq<ORDER>(p, i, by_len);
        v.q0 = p.query_start[seq];
        v.q1 = p.query_start[seq + 1];
        v.len = p.context_lens[seq];
    }
    return v;
}

// Checks one sequence's (chunk start, chunk length, context length); false when
// they are out of contract.
__device__ __forceinline__ bool prefill_seq(const PrefillParams &p, const PrefillSeqVals &v, int &q0,
                                            int &chunk, int &len) {
    q0 = v.q0;
    chunk = v.q1 - v.q0;
    len = v.len;
    return q0 >= 0 && chunk >= 0 && v.q1 <= p.num_rows && chunk <= p.qlen_cap && len >= chunk &&
           len <= p.len_cap;
}

struct PrefillItem {
    int q0, chunk, len;  // the sequence's chunk start row, chunk length, context length
    int kvh, split, row_tile;
    int rows;            // the sequence's query rows of one KV head: chunk * group
    int row0;            // first of the item's rows: row_tile * tile_rows
    int base_pos;        // position of chunk token 0
    int tok_lo, tok_hi;  // the item's KV tokens
    int ntiles;          // 128-token KV tiles
    int seq;
};

// Item i of the static order.
// - Row tiles (default): row tiles from the last (longest causal range) down, then
//   sequence and split, then KV head, so that CTA c's items c, c + grid, ... are
//   heaviest first.
// - Pairs (whole prompts of one length, one split): (sequence, KV head) major, and
//   within it the row tiles as last, first, second to last, second, ..., taken two
//   at a time by a CTA (prefill_slot_item), so that every CTA's pair of row tiles
//   carries the same causal work.
// - Sorted groups (one split, at most kSortedGroupsMaxSeqs sequences of different
//   lengths): (sequence, KV head) major with the sequences by context length,
//   longest first (by_len), and within a group the row tiles from the last down;
//   the CTAs take the items in rounds of one each, every other round in reverse
//   (prefill_slot_item), which spreads the long and short items evenly.
// In the last two the CTAs that run together share the K/V tiles of a few
// (sequence, KV head) pairs in L2.  False when the item holds no work: a row tile
// past the chunk, a split past the tile's causal limit, or a sequence out of
// contract (flagged once when `flag`).
template <int ORDER>
__device__ __forceinline__ bool prefill_item(const PrefillParams &p, int i, const PrefillSeqVals &sv,
                                             bool flag, PrefillItem &it, const unsigned char *by_len) {
    if constexpr (ORDER == kOrderSortedGroups) {
        const int g = fast_div(i, p.div_row_tiles);
        const int pos = i - g * p.row_tiles;
        const int rank = fast_div(g, p.div_kv_heads);
        it.seq = by_len[rank];
        it.kvh = g - rank * p.num_kv_heads;
        it.split = 0;
        it.row_tile = p.row_tiles - 1 - pos;
    } else if constexpr (ORDER == kOrderPairs) {
        const int g = fast_div(i, p.div_row_tiles);
        const int pos = i - g * p.row_tiles;
        it.seq = fast_div(g, p.div_kv_heads);
        it.kvh = g - it.seq * p.num_kv_heads;
        it.split = 0;
        it.row_tile = (pos & 1) ? pos >> 1 : p.row_tiles - 1 - (pos >> 1);
    } else {
        const int per_tile = p.num_kv_heads * p.num_seqs * p.splits;
        const int rt_rev = fast_div(i, p.div_per_tile);
        const int rem = i - rt_rev * per_tile;
        const int ss = fast_div(rem, p.div_kv_heads);
        it.kvh = rem - ss * p.num_kv_heads;
        it.seq = fast_div(ss, p.div_splits);
        it.split = ss - it.seq * p.splits;
        it.row_tile = p.row_tiles - 1 - rt_rev;
    }
    if (!prefill_seq(p, sv, it.q0, it.chunk, it.len)) {
        if (flag && it.row_tile == 0 && it.kvh == 0 && it.split == 0)
            raise_flag(p.status, PKV_DEVERR_CONTEXT_LEN);
        return false;
    }
    it.rows = it.chunk * p.group;
    it.row0 = it.row_tile * p.tile_rows;
    if (it.row0 >= it.rows) return false;
    const int last_row = min(it.rows, it.row0 + p.tile_rows) - 1;
    it.base_pos = it.len - it.chunk;
    const int pos_max = it.base_pos + fast_div(last_row, p.div_group);
    it.tok_lo = it.split * p.split_tokens;
    it.tok_hi = min(min(it.len, pos_max + 1), it.tok_lo + p.split_tokens);
    it.ntiles = (it.tok_hi - it.tok_lo + 127) / 128;
    return it.tok_hi > it.tok_lo;
}

// The k-th item of this CTA: items blockIdx.x + k * grid in the row-tile order,
// the pairs (2 q, 2 q + 1) for q = blockIdx.x + (k / 2) * grid in pair order, and
// item blockIdx.x of round k (counted from the end in odd rounds) in sorted-groups
// order.
template <int ORDER>
__device__ __forceinline__ int prefill_slot_item(const PrefillParams &p, int k) {
    if constexpr (ORDER == kOrderSortedGroups)
        return k * gridDim.x + ((k & 1) ? gridDim.x - 1 - blockIdx.x : blockIdx.x);
    if constexpr (ORDER == kOrderPairs) return 2 * (blockIdx.x + (k >> 1) * gridDim.x) + (k & 1);
    return blockIdx.x + k * gridDim.x;
}

// Items whose O tile leaves through the output tensor map, staged in the item's
// last V slot (one split, and every row of the row tile inside the chunk, so the
// box holds no other sequence's rows); the others store row by row.
__device__ __forceinline__ bool prefill_staged(const PrefillParams &p, const PrefillItem &it) {
    return p.splits == 1 && it.row0 + p.tile_rows <= it.rows;
}

// Shared memory: the Q tile(s) of consecutive items, K and V rings of
// 128-token tiles, and the barriers (rings, Q, S / O double buffers, the
// softmax pairs).
// P lives in TMEM.
struct PrefillLayout {
    static constexpr int kTile = 128;
    static constexpr int kHalf = 128 * 128;           // 128 rows x 128 B
    static constexpr int kPanel = 2 * kHalf;          // 128 rows x 128 16-bit values
    static constexpr int kQB = 1;                     // Q buffers
    static constexpr int kKS = 3, kVS = 3;            // K slots, V slots
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQB * kPanel;
    static constexpr int kOffV = kOffK + kKS * kPanel;
    static constexpr int kOffBar = kOffV + kVS * kPanel;
    static constexpr int kSB = 3;                     // S buffers (P over S) in TMEM
    static constexpr int kNumBars = 2 * kKS + 2 * kVS + 2 * kQB + 4 * kSB + 2 + 8 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffSum = kOffMisc + 16;     // row-sum exchange: [2 halves][128 rows] fp32
    static constexpr int kOffByLen = kOffSum + 2 * 128 * 4;  // sequences by length (sorted-groups order)
    static constexpr int kBytes = kOffByLen + kSortedGroupsMaxSeqs;
    static constexpr int kSmemBytes = kBytes + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 512;        // S[3] at 0 / 128 / 256 (P[b] over S[b]), O at 384
    static constexpr uint32_t kOCol = 384;
    static constexpr float kRescaleLog2 = 8.f;
    static constexpr int kThreads = 384;
    static_assert(kSmemBytes <= 232448, "dynamic shared memory per block");
};

template <typename T, int BS, int ORDER>
__global__ void __launch_bounds__(384, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                            const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v,
                            const __grid_constant__ CUtensorMap tmap_o, const PrefillParams p) {
    using L = PrefillLayout;
    constexpr int TILE = L::kTile, D = 128;
    constexpr bool kBF16 = !std::is_same<T, __half>::value;
    static_assert(TILE / BS <= 32, "one table entry per producer lane");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = p.tile_rows;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm =
        smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u);
    constexpr int KS = L::kKS, VS = L::kVS, QB = L::kQB;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
    uint64_t *k_full = bars, *k_empty = k_full + KS, *v_full = k_empty + KS, *v_empty = v_full + VS;
    uint64_t *q_full = v_empty + VS, *q_empty = q_full + QB;
    constexpr int SB = L::kSB;
    uint64_t *s_full = q_empty + QB, *s_empty = s_full + SB, *p_full = s_full + 2 * SB, *o_done = s_full + 3 * SB;
    uint64_t *drain_bar = s_full + 4 * SB;  // QK^T issuer's drain on exit
    uint64_t *drain_pv = drain_bar + 1;     // PV issuer's drain on exit
    uint64_t *pair_bar = drain_pv + 1;     // [quarter][parity]
    uint64_t *o_staged = pair_bar + 8;     // an item's O tile is in its last V slot
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffMisc + 4);
    unsigned char *by_len = sm + L::kOffByLen;  // sorted-groups order: sequences by length
    const uint32_t smem_base = static_cast<uint32_t>(__cvta_generic_to_shared(sm));

    if (threadIdx.x == 0) {
        for (int i = 0; i < KS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < VS; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < QB; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 1);
            mbar_init(&p_full[i], 8);
            mbar_init(&o_done[i], 1);
        }
        for (int i = 0; i < 8; ++i) mbar_init(&pair_bar[i], 2);
        mbar_init(o_staged, 8);
        mbar_init(drain_bar, 1);
        mbar_init(drain_pv, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::kTmemCols);
        tc::tmem_relinquish();
    }
    // Q rows R .. 127 are never loaded (a row tile holds whole tokens): zero
    // them once so the MMA reads finite values there
    if (R < 128) {
        for (int i = threadIdx.x; i < QB * 2 * (128 - R) * 8; i += blockDim.x) {
            const int c16 = i & 7, rr = R + (i >> 3) % (128 - R), h = (i >> 3) / (128 - R);
            *reinterpret_cast<uint4 *>(sm + L::kOffQ + h * L::kHalf + rr * 128 + c16 * 16) =
                make_uint4(0, 0, 0, 0);
        }
    }
    if (ORDER == kOrderSortedGroups && warp == 2) {
        // rank the (at most 32) sequences by context length, longest first, ties by index
        const int len = lane < p.num_seqs ? p.context_lens[lane] : 0;
        int rank = 0;
        for (int j = 0; j < p.num_seqs; ++j) {
            const int lj = __shfl_sync(0xffffffffu, len, j);
            rank += (lj > len || (lj == len && j < lane)) ? 1 : 0;
        }
        if (lane < p.num_seqs) by_len[rank] = static_cast<unsigned char>(lane);
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tensormap(&tmap_q);
        tc::prefetch_tensormap(&tmap_k);
        tc::prefetch_tensormap(&tmap_v);
        tc::prefetch_tensormap(&tmap_o);
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == 10) {
        // ===================== TMA producers: K (warp 0), V (warp 10) =====================
        // Separate producers so a K tile never waits behind a V slot that its PV still
        // holds; each reads the next tile's table entries while it waits for a slot.
        // The K producer also loads each item's Q tile into Q buffer n % kQB once
        // the QK^T of item n - kQB is done, without holding back the item's K tiles.
        const int kv = warp == 10;
        const int nst = kv ? VS : KS;
        uint64_t *full = kv ? v_full : k_full;
        uint64_t *empty = kv ? v_empty : k_empty;
        const CUtensorMap *map = kv ? &tmap_v : &tmap_k;
        unsigned char *ring = sm + (kv ? L::kOffV : L::kOffK);
        const uint64_t policy = l2_policy_evict_last();  // every row tile of the sequence reads it
        const uint64_t q_policy = l2_policy_evict_first();
        int last_issue[4] = {-1, -1, -1, -1};
        static_assert(L::kKS <= 4 && L::kVS <= 4 && L::kQB <= 2, "drain bookkeeping");
        int q_issue[2] = {-1, -1};
        bool ok = true;
        int jt = 0, n = 0;  // tiles and items so far
        for (int ki = 0, item = prefill_slot_item<ORDER>(p, 0); item < p.num_items && ok; item = prefill_slot_item<ORDER>(p, ++ki)) {
            PrefillItem it;
            if (!prefill_item<ORDER>(p, item, prefill_seq_vals<ORDER>(p, item, by_len), kv == 0, it, by_len)) continue;
            const int32_t *trow = p.block_tables + static_cast<int64_t>(it.seq) * p.max_blocks_per_seq;
            auto entry = [&](int j) -> int {  // this lane's block of tile j (-1: none or bad)
                const int t0 = it.tok_lo + j * TILE;
                const int nblk = (min(TILE, it.tok_hi - t0) + BS - 1) / BS;
                int e = -1;
                if (lane < nblk) {
                    e = trow[t0 / BS + lane];
                    if (e < 0 || e >= p.num_blocks) {
                        if (kv == 0) raise_flag(p.status, PKV_DEVERR_BLOCK_TABLE);
                        e = -1;
                    }
                }
                return e;
            };
            int e_next = entry(0);
            // The K producer loads the item's Q tile as soon as Q buffer n % kQB is free
            // (the QK^T of item n - kQB done), while it already streams the item's K
            // tiles: lane 0 polls that buffer whenever it waits for a K slot, and waits
            // for it at the latest after the item's last K tile.
            const int qb = n % QB;
            const uint32_t q_par = ((n / QB) & 1) ^ 1;
            bool q_pending = kv == 0;  // lane 0's state
            auto issue_q = [&]() {
                // boxes of tile_tokens tokens x group heads x 64 columns; rows of tokens
                // past the query array arrive as zeros and count as bytes
                mbar_arrive_expect_tx(&q_full[qb], 256u * R);
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    tc::tma_load_3d(sm + L::kOffQ + qb * L::kPanel + c * L::kHalf, &tmap_q, c * 64,
                                    it.kvh * p.group, it.q0 + it.row_tile * p.tile_tokens, &q_full[qb], q_policy);
                q_issue[qb] = n;
                q_pending = false;
                // the next item's Q box into L2 now, so its load does not wait for HBM
                PrefillItem nx;
                for (int k2 = ki + 1, i2 = prefill_slot_item<ORDER>(p, k2); i2 < p.num_items; i2 = prefill_slot_item<ORDER>(p, ++k2)) {
                    if (!prefill_item<ORDER>(p, i2, prefill_seq_vals<ORDER>(p, i2, by_len), false, nx, by_len)) continue;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        tc::tma_prefetch_3d(&tmap_q, c * 64, nx.kvh * p.group, nx.q0 + nx.row_tile * p.tile_tokens);
                    break;
                }
            };
            // lane 0: bounded wait for `bar`, issuing the pending Q load when its buffer
            // frees up meanwhile
            auto wait_slot = [&](uint64_t *bar, uint32_t par) -> bool {
                if (!q_pending) return tc_wait(bar, par, abort_flag, p.status);
                const uint64_t t0 = global_timer_ns();
                while (true) {
                    if (q_pending && mbar_test_wait(&q_empty[qb], q_par)) issue_q();
                    if (mbar_test_wait(bar, par)) return true;
                    if (!q_pending) return tc_wait(bar, par, abort_flag, p.status);
                    if (*abort_flag) return false;
                    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                        raise_flag(p.status, PKV_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                        return false;
                    }
                }
            };
            for (int j = 0; j < it.ntiles; ++j, ++jt) {
                const int e = e_next;
                if (j + 1 < it.ntiles) e_next = entry(j + 1);  // in flight while this tile waits
                const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, e >= 0)) * BS * 256u;
                const int s = jt % nst;
                int go = 1;
                if (lane == 0) {
                    go = wait_slot(&empty[s], ((jt / nst) & 1) ^ 1);
                    if (go) {
                        if (bytes) mbar_arrive_expect_tx(&full[s], bytes);
                        else mbar_arrive(&full[s]);
                        last_issue[s] = jt;
                    }
                }
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
                if (e >= 0) {
                    unsigned char *slot = ring + s * L::kPanel;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        tc::tma_load_3d(slot + c * L::kHalf + lane * BS * 128, map, c * 64, it.kvh * BS, e,
                                        &full[s], policy);
                }
                __syncwarp();
            }
            if (ok && kv == 0) {
                int go = 1;
                if (lane == 0 && q_pending) {
                    go = tc_wait(&q_empty[qb], q_par, abort_flag, p.status);
                    if (go) issue_q();
                }
                if (!__shfl_sync(0xffffffffu, go, 0)) ok = false;
            }
            ++n;
        }
        if (!ok && lane == 0) {
            // copies still in flight land before the CTA exits
            for (int s = 0; s < nst; ++s)
                if (last_issue[s] >= 0)
                    mbar_wait_bounded(&full[s], (last_issue[s] / nst) & 1, kDrainTimeoutNs);
            for (int b = 0; b < QB; ++b)
                if (q_issue[b] >= 0) mbar_wait_bounded(&q_full[b], (q_issue[b] / QB) & 1, kDrainTimeoutNs);
        }
    } else if (warp == 1) {
        // ===================== QK^T issuer =====================
        // QK^T of each tile as soon as its K landed and its S buffer is free; PV is
        // issued by warp 11, so a ready PV never waits behind a QK^T batch (a batch
        // of MMAs holds its issuing thread for its whole execution).
        constexpr uint32_t idesc_qk = tc::idesc_f16_f32acc(kBF16, 128, 128, false, false);
        bool ok = true;
        int jt = 0, n = 0;
        for (int ki = 0, item = prefill_slot_item<ORDER>(p, 0); item < p.num_items && ok; item = prefill_slot_item<ORDER>(p, ++ki)) {
            PrefillItem it;
            if (!prefill_item<ORDER>(p, item, prefill_seq_vals<ORDER>(p, item, by_len), false, it, by_len)) continue;
            const int qb = n % QB;
            int go = 1;
            if (lane == 0) go = tc_wait(&q_full[qb], (n / QB) & 1, abort_flag, p.status);
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            for (int j = 0; j < it.ntiles; ++j, ++jt) {
                if (lane == 0)
                    go = tc_wait(&k_full[jt % KS], (jt / KS) & 1, abort_flag, p.status) &&
                         tc_wait(&s_empty[jt % SB], ((jt / SB) & 1) ^ 1, abort_flag, p.status);
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int b = jt % SB;
                    tc::fence_after_sync();
                    const uint32_t qa = smem_base + L::kOffQ + qb * L::kPanel;
                    const uint32_t ka = smem_base + L::kOffK + (jt % KS) * L::kPanel;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t a = tc::smem_desc_sw128(qa + (k / 4) * L::kHalf + (k % 4) * 32, 16, 1024);
                        const uint64_t bd = tc::smem_desc_sw128(ka + (k / 4) * L::kHalf + (k % 4) * 32, 16, 1024);
                        tc::mma_f16_ss(tmem + 128 * b, a, bd, idesc_qk, k > 0);
                    }
                    tc::mma_commit(&s_full[b]);
                    tc::mma_commit(&k_empty[jt % KS]);
                    if (j + 1 == it.ntiles) tc::mma_commit(&q_empty[qb]);  // Q buffer free
                }
                __syncwarp();
            }
            ++n;
        }
        if (lane == 0) {
            // this thread's MMAs complete before TMEM is released
            tc::mma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, kDrainTimeoutNs);
        }
        __syncwarp();
    } else if (warp == 11) {
        // ===================== PV issuer =====================
        constexpr uint32_t idesc_pv = tc::idesc_f16_f32acc(kBF16, 128, 128, false, true);
        bool ok = true;
        int jt = 0, n_staged = 0;
        for (int ki = 0, item = prefill_slot_item<ORDER>(p, 0); item < p.num_items && ok; item = prefill_slot_item<ORDER>(p, ++ki)) {
            PrefillItem it;
            if (!prefill_item<ORDER>(p, item, prefill_seq_vals<ORDER>(p, item, by_len), false, it, by_len)) continue;
            const bool staged = prefill_staged(p, it);
            for (int j = 0; j < it.ntiles; ++j, ++jt) {
                int go = 1;
                if (lane == 0)
                    go = tc_wait(&p_full[jt % SB], (jt / SB) & 1, abort_flag, p.status) &&
                         tc_wait(&v_full[jt % VS], (jt / VS) & 1, abort_flag, p.status);
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int b = jt % SB;
                    tc::fence_after_sync();
                    const uint32_t va = smem_base + L::kOffV + (jt % VS) * L::kPanel;
#pragma unroll
                    for (int k = 0; k < TILE / 16; ++k) {
                        const uint64_t bd = tc::smem_desc_sw128(va + k * 2048, L::kHalf, 1024);
                        // P from TMEM (16 tokens = 8 columns per step); the item's first
                        // tile starts O afresh
                        tc::mma_f16_ts(tmem + L::kOCol, tmem + 128 * b + 8 * k, bd, idesc_pv, j > 0 || k > 0);
                    }
                    tc::mma_commit(&o_done[b]);
                    tc::mma_commit(&s_empty[b]);  // S[b] / P[b] free for QK^T(jt + SB)
                    // a staged item's last V slot receives its O tile: freed below
                    if (!(staged && j + 1 == it.ntiles)) tc::mma_commit(&v_empty[jt % VS]);
                }
                __syncwarp();
                if (staged && j + 1 == it.ntiles) {
                    // the softmax warps have written the normalised O tile into this V
                    // slot (after PV(jt) completed): store it with the queries' boxes,
                    // then free the slot once the copies have read it
                    if (lane == 0) {
                        go = tc_wait(o_staged, n_staged & 1, abort_flag, p.status);
                        if (go) {
                            unsigned char *slot = sm + L::kOffV + (jt % VS) * L::kPanel;
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                tc::tma_store_3d(&tmap_o, c * 64, it.kvh * p.group,
                                                 it.q0 + it.row_tile * p.tile_tokens, slot + c * L::kHalf);
                            tc::bulk_commit_group();
                            tc::bulk_wait_read_all();
                            mbar_arrive(&v_empty[jt % VS]);
                        }
                    }
                    ++n_staged;
                    if (!__shfl_sync(0xffffffffu, go, 0)) {
                        ok = false;
                        break;
                    }
                }
            }
        }
        if (lane == 0) {
            tc::bulk_wait_all();  // output tiles written before the CTA exits
            tc::mma_commit(drain_pv);
            mbar_wait_bounded(drain_pv, 0, kDrainTimeoutNs);
        }
        __syncwarp();
    } else {
        // ===================== softmax (warps 2..9): thread = query row, 64 columns =====================
        const int quarter = warp & 3;
        const int half = warp >= 6 ? 1 : 0;  // tile columns 64*half .. +63
        const int c0 = half * 64;
        const int r = quarter * 32 + lane;   // row within the tile = TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        float *sum_x = reinterpret_cast<float *>(sm + L::kOffSum);  // [half][row]
        bool ok = true;
        int jt = 0, xs = 0;  // tiles and pair exchanges so far
        // One value per row between the two warps of the pair, ordered by the pair's
        // mbarrier (phase s & 1 of barrier [quarter][s & 1] for exchange step s).
        // A tile's partial maxima travel in S[b] itself, in columns whose scores their
        // writer has already read and that nothing overwrites before the partner has
        // read them: half 0 writes column 32 (half 1's P lands there only after half 1
        // has read it), half 1 column 64 (no P store reaches it; QK^T(jt + SB) rewrites
        // S[b] only after PV(jt), which waits for both warps).  An item's row sums go
        // through shared memory; a slot is rewritten only after the next tile's
        // exchange, which the partner reaches after reading it.
        auto pair_sync = [&](int step) -> bool {
            __syncwarp();
            uint64_t *pb = &pair_bar[quarter * 2 + (step & 1)];
            if (lane == 0) mbar_arrive(pb);
            return tc_wait_warp(pb, (step >> 1) & 1, abort_flag, p.status);
        };
        auto exchange_max = [&](int step, int b, float mine, float &other) -> bool {
            const uint32_t sb = lane_base + 128 * b;
            tc::tmem_st_x1(sb + (half ? 64 : 32), mine);
            tc::tmem_st_wait();
            tc::fence_before_sync();
            if (!pair_sync(step)) return false;
            tc::fence_after_sync();
            other = tc::tmem_ld_x1(sb + (half ? 32 : 64));
            tc::tmem_ld_wait();
            return true;
        };
        auto exchange_sum = [&](int step, float mine, float &other) -> bool {
            sum_x[half * 128 + r] = mine;
            if (!pair_sync(step)) return false;
            other = sum_x[(1 - half) * 128 + r];
            return true;
        };
        for (int ki = 0, item = prefill_slot_item<ORDER>(p, 0); item < p.num_items && ok; item = prefill_slot_item<ORDER>(p, ++ki)) {
            PrefillItem it;
            if (!prefill_item<ORDER>(p, item, prefill_seq_vals<ORDER>(p, item, by_len), false, it, by_len)) continue;
            const int row = it.row0 + r;
            const bool live = r < R && row < it.rows;
            const int jtok = live ? fast_div(row, p.div_group) : 0;
            const int pos = it.base_pos + jtok;  // this row sees tokens 0 .. pos
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < it.ntiles && ok; ++j, ++jt) {
                const int b = jt % SB;
                const int t0 = it.tok_lo + j * TILE;
                const int valid = min(TILE, it.tok_hi - t0);                    // columns loaded
                const int vr = live ? max(0, min(valid, pos + 1 - t0)) : 0;  // columns this row sees
                const int vh = max(0, min(64, vr - c0));                     // ... in this half
                if (!tc_wait_warp(&s_full[b], (jt / SB) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                // this row's 64 scores of the half, read from TMEM once
                float x[64];
#pragma unroll
                for (int c = 0; c < 64; c += 16) tc::tmem_ld_x16(lane_base + 128 * b + c0 + c, x + c);
                tc::tmem_ld_wait();
                // tiles every row of the warp sees completely skip the per-column masks
                const bool full = __all_sync(0xffffffffu, vr == TILE);
                // partial maximum of the visible scaled scores: the extreme raw score times
                // the scale (the maximum for a positive scale, the minimum otherwise)
                float pmax = -INFINITY;
                if (vh > 0) {
                    const bool pos_scale = p.scale_log2 > 0.f;
                    float ext = x[0];
                    if (full) {
#pragma unroll
                        for (int i = 1; i + 1 < 64; i += 2)
                            ext = pos_scale ? fmax3(ext, x[i], x[i + 1]) : fmin3(ext, x[i], x[i + 1]);
                        ext = pos_scale ? fmaxf(ext, x[63]) : fminf(ext, x[63]);
                    } else {
#pragma unroll
                        for (int i = 1; i < 64; ++i)
                            if (i < vh) ext = pos_scale ? fmaxf(ext, x[i]) : fminf(ext, x[i]);
                    }
                    pmax = ext * p.scale_log2;
                }
                float pmax_other;
                if (!exchange_max(xs++, b, pmax, pmax_other)) {
                    ok = false;
                    break;
                }
                const float tmax = fmaxf(pmax, pmax_other);
                // the reference maximum moves only by more than kRescaleLog2 (a row that sees
                // nothing keeps -inf and alpha 1); both warps of the pair take the same
                // decision for a row; TMEM loads and stores are warp-wide, so the warp
                // rescales its half of O if any of its rows must
                const float new_ref = tmax > m_ref + L::kRescaleLog2 ? tmax : m_ref;
                const float alpha = new_ref == m_ref ? 1.f : fast_exp2(m_ref - new_ref);
                if (__any_sync(0xffffffffu, new_ref != m_ref)) {
                    if (j > 0) {
                        // O holds tiles < j: wait for PV(j-1), rescale this half of O in TMEM
                        if (!tc_wait_warp(&o_done[(jt - 1) % SB], ((jt - 1) / SB) & 1, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
#pragma unroll
                        for (int c = 0; c < 64; c += 16) {
                            float o[16];
                            tc::tmem_ld_x16(lane_base + L::kOCol + c0 + c, o);
                            tc::tmem_ld_wait();
                            uint32_t w[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(o[i] * alpha);
                            asm volatile(
                                "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, "
                                "%8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(lane_base + L::kOCol + c0 + c),
                                "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                                "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]),
                                "r"(w[13]), "r"(w[14]), "r"(w[15])
                                : "memory");
                        }
                        tc::tmem_st_wait();
                    }
                    l *= alpha;
                    m_ref = new_ref;
                }
                // P = 2^(s - m_ref) on visible columns (0 elsewhere), rounded to T and packed
                // two per 32-bit column over the first 64 columns of S[b] (tokens 64 half ..
                // +63 -> columns 32 half .. +31; both warps of the pair have read their
                // scores, the exchange above orders it), where the PV MMA reads it; the row
                // sum l adds the fp32 values
                const uint32_t pcol = lane_base + 128 * b + 32 * half;
                float l0 = 0.f, l1 = 0.f;
                // two copies of the loop, so fully visible tiles carry no per-column mask
                auto weights = [&](auto masked) {
#pragma unroll
                    for (int c16 = 0; c16 < 2; ++c16) {
                        uint32_t packed[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int t = c16 * 32 + 2 * i;
                            // s * scale - m for two columns in one packed FMA
                            float e0 = -m_ref, e1 = -m_ref;
                            fma_f32x2(e0, e1, x[t], x[t + 1], p.scale_log2, p.scale_log2);
                            float p0 = fast_exp2(e0);
                            float p1 = fast_exp2(e1);
                            if constexpr (decltype(masked)::value) {
                                p0 = t < vh ? p0 : 0.f;
                                p1 = t + 1 < vh ? p1 : 0.f;
                            }
                            add_f32x2(l0, l1, p0, p1);
                            packed[i] = Elem<T>::pack2(p0, p1);
                        }
                        tc::tmem_st_x16(pcol + 16 * c16, packed);
                    }
                };
                if (full) weights(std::false_type{});
                else weights(std::true_type{});
                l += l0 + l1;
                if (valid < TILE) {
                    // V rows past the loaded range: zero this half so 0 * stale never reaches
                    // the MMA.  The parity wait cannot alias an older phase of the slot: S(jt)
                    // exists only once PV(jt - kSB) has completed, so V(jt - kVS), the slot's
                    // previous tile, has landed when kVS >= kSB.  With more S buffers than V
                    // slots the wait could pass on V(jt - kVS)'s phase and zero rows that a
                    // pending PV still reads.
                    static_assert(L::kVS >= L::kSB, "V slots >= S buffers");
                    if (!tc_wait_warp(&v_full[jt % VS], (jt / VS) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    if (r >= valid) {
                        uint4 *vrow = reinterpret_cast<uint4 *>(sm + L::kOffV + (jt % VS) * L::kPanel + half * L::kHalf +
                                                                r * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i) vrow[i] = make_uint4(0, 0, 0, 0);
                    }
                }
                tc::tmem_st_wait();
                tc::fence_before_sync();   // P and the O rescale's TMEM stores precede PV(j)
                fence_proxy_async_smem();  // zeroed V rows visible to the MMA
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }
            // the pair's row sum, then this half of the O row -> out (one split) or its
            // partial slot.  TMEM loads are warp-wide: every lane loads, only live rows store.
            float l_other = 0.f;
            if (ok) ok = exchange_sum(xs++, l, l_other);
            const float lt = l + l_other;
            if (ok) ok = tc_wait_warp(&o_done[(jt - 1) % SB], ((jt - 1) / SB) & 1, abort_flag, p.status);
            if (ok && prefill_staged(p, it)) {
                // normalised O rows into the item's last V slot (free since PV(jt - 1)
                // completed), laid out as the queries' boxes land: two half panels of
                // 128-byte rows, 16-byte chunk c of row r at chunk c ^ (r & 7); the PV
                // issuer stores them with the output tensor map
                tc::fence_after_sync();
                unsigned char *orow_s = sm + L::kOffV + ((jt - 1) % VS) * L::kPanel + half * L::kHalf + r * 128;
                const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
                for (int c = 0; c < 64; c += 16) {
                    float o[16];
                    tc::tmem_ld_x16(lane_base + L::kOCol + c0 + c, o);
                    tc::tmem_ld_wait();
                    if (!live) continue;
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[i] = Elem<T>::pack2(o[2 * i] * inv_l, o[2 * i + 1] * inv_l);
                    const int k0 = c / 8;  // chunks k0, k0 + 1 of the row
                    *reinterpret_cast<uint4 *>(orow_s + (((k0) ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(orow_s + (((k0 + 1) ^ (r & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                fence_proxy_async_smem();  // visible to the tensor store
                __syncwarp();
                if (lane == 0) mbar_arrive(o_staged);
            } else if (ok) {
                tc::fence_after_sync();
                const int g = live ? row - jtok * p.group : 0;
                const int64_t orow = (static_cast<int64_t>(it.q0) + jtok) * p.num_q_heads + it.kvh * p.group + g;
                const bool direct = p.splits == 1;
                const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
                for (int c = 0; c < 64; c += 16) {
                    float o[16];
                    tc::tmem_ld_x16(lane_base + L::kOCol + c0 + c, o);
                    tc::tmem_ld_wait();
                    if (!live) continue;
                    if (direct) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[i] = Elem<T>::pack2(o[2 * i] * inv_l, o[2 * i + 1] * inv_l);
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + orow * D + c0 + c);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    } else {
                        float *dst = p.ws_o + (orow * p.splits + it.split) * D + c0 + c;
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
                    }
                }
                if (live && !direct && half == 0) {
                    p.ws_m[orow * p.splits + it.split] = m_ref;
                    p.ws_l[orow * p.splits + it.split] = lt;
                }
            }
        }
    }

    // ---- tear-down: both issuers drained their MMAs; TMEM is freed
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, L::kTmemCols);
    }
}

// Log-sum-exp merge of a prefill's KV splits: one warp per (chunk row, query
// head); the row at position pos has partials in splits 0 .. pos / split_tokens.
template <typename T>
__global__ void __launch_bounds__(128) paged_prefill_merge_kernel(const PrefillParams p) {
    constexpr int D = 128, PER_LANE = D / 32;
    const int seq = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int idx = blockIdx.x * 4 + (threadIdx.x >> 5);  // (chunk token, query head)
    int q0, chunk, len;
    const PrefillSeqVals sv{p.query_start[seq], p.query_start[seq + 1], p.context_lens[seq]};
    if (!prefill_seq(p, sv, q0, chunk, len)) return;     // flagged by the main kernel
    const int jtok = idx / p.num_q_heads, hq = idx - jtok * p.num_q_heads;
    if (jtok >= chunk) return;
    const int pos = len - chunk + jtok;
    const int nsp = min(p.splits, pos / p.split_tokens + 1);
    const int64_t orow = (static_cast<int64_t>(q0) + jtok) * p.num_q_heads + hq;
    const int64_t base = orow * p.splits;
    float mmax = -INFINITY;
    for (int s = 0; s < nsp; ++s) mmax = fmaxf(mmax, p.ws_m[base + s]);
    float lsum = 0.f, o[PER_LANE] = {};
    for (int s = 0; s < nsp; ++s) {
        const float ms = p.ws_m[base + s];
        const float w = ms == -INFINITY ? 0.f : fast_exp2(ms - mmax);
        lsum += w * p.ws_l[base + s];
        const float *src = p.ws_o + (base + s) * D + lane * PER_LANE;
#pragma unroll
        for (int e = 0; e < PER_LANE; ++e) o[e] += w * src[e];
    }
    T *dst = static_cast<T *>(p.out) + orow * D + lane * PER_LANE;
#pragma unroll
    for (int e = 0; e < PER_LANE; ++e) dst[e] = Elem<T>::from_f32(lsum > 0.f ? o[e] / lsum : 0.f);
}

}  // namespace pkv
