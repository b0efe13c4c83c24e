// decode_tc_kernel.cuh -- paged decode attention on the 5th-generation tensor
// cores for grouped-query attention with head_dim 128 and 4, 8 or 16 query
// heads per KV head.
//
// What it computes is the same as paged_decode_kernel ("KV Cache与PagedAttention
// 深度解析" §2.1 definition, §4.2-4.3 block-table addressing, §7.2 running
// max / running sum): per (sequence, KV head, context partition) and for the
// GH query heads of the group,  o = sum_t exp(s_t - m) V_t,  l = sum_t exp(s_t - m),
// s_t = scale * q . K_t, all accumulated in fp32.
//
// With GH >= 4 query heads sharing each K/V tile, the products are dense
// tiles, so they run as tcgen05 MMAs (M = 128):
//   S^T[128 tokens x 16]  = K_tile[128 x 128 d] . Q^T[128 d x 16]      (K-major A and B)
//   O^T[128 d x 16]       = V_tile^T[128 d x 128 tokens] . P^T[128 x 16]  (MN-major A)
// The 16 columns hold the GH heads (zero padded).  P is rounded to the input
// type for the second MMA; l is summed from the same rounded values so
// numerator and denominator use identical weights.
//
// Structure (one persistent CTA per SM, 8 warps):
//   warps 0, 6  TMA producers of K and of V: per 128-token tile, one 3-D tiled
//               bulk-tensor copy per (block, 64-column half), 128-byte swizzled,
//               into separate rings of 32 KiB K slots and 32 KiB V slots (a K
//               slot is refilled as soon as QK^T has read it; K never waits
//               behind a V slot).
//   warp 1      TMEM owner and QK^T issuer (one thread); warp 7 issues PV, so a
//               ready PV never waits behind a QK^T batch (a batch of MMAs holds
//               its issuing thread for its whole execution).
//   warps 2-5   softmax and accumulation, one TMEM lane quarter each: a thread
//               owns a token row of S and a head-dim row of O^T; the tile max is
//               exchanged through shared memory; o stays in registers.
// Work items (sequence, KV head, partition) are enumerated in order and dealt
// round-robin to the CTAs; a CTA's pipeline runs straight across its items.
// Every wait is bounded; a timeout raises PKV_DEVERR_TIMEOUT, all roles stop,
// in-flight copies and MMAs are drained and TMEM is freed.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "decode_kernel.cuh"
#include "pkv_tc.cuh"

namespace pkv {

struct TcLayout {
    static constexpr int kTile = 128;          // tokens per MMA tile
    static constexpr int kD = 128;             // head_dim
    static constexpr int kN = 16;              // MMA N (query heads, padded)
    // K and V tiles have separate rings: a K slot is free again as soon as
    // QK^T has read it, a V slot only after PV.
    static constexpr int kKStages = 2;
    static constexpr int kVStages = 4;
    static constexpr int kHalfBytes = 128 * 128;        // 128 rows x 64 columns x 2 B
    static constexpr int kKVBytes = 2 * kHalfBytes;     // K (or V) tile: 32 KiB
    static constexpr int kPanelBytes = 4096;            // 16 x 128 x 2 B (Q or P)
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kKStages * kKVBytes;
    static constexpr int kOffQ = kOffV + kVStages * kKVBytes;
    static constexpr int kOffP = kOffQ + 2 * kPanelBytes;
    static constexpr int kOffRed = kOffP + 2 * kPanelBytes;           // float [2][4][16] + [4][16]
    static constexpr int kOffBar = kOffRed + 3 * 4 * 16 * 4;
    static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 * 5 + 2 + 1 + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;           // tmem slot, abort flag
    static constexpr int kMaxStagedSeqs = 1024;                      // context lengths kept in smem
    static constexpr int kOffLens = kOffMisc + 16;
    static constexpr int kBytes = kOffLens + 4 * kMaxStagedSeqs;
    static constexpr int kSmemBytes = kBytes + 1024;                  // + alignment slack
    static constexpr uint32_t kTmemCols = 64;  // S[2] at 0/16, O[2] at 32/48
};

// Walks the work items of a launch in order: item r -> (sequence, y, partition).
// Items of sequence s are nparts(s) * Y consecutive indices.  A CTA's items
// are gridDim.x apart, so a step may cross several sequences; the lengths come
// from the shared-memory copy `s_len` when the batch fits it, so that walk
// costs no global-memory round trips.
struct ItemWalker {
    int seq = 0;
    int64_t first = 0;  // index of the first item of `seq`
    int nparts = -1;
    int len = 0;
    __device__ bool seek(const DecodeParams &p, const int *s_len, int64_t r, int &y, int &part) {
        while (seq < p.num_seqs) {
            if (nparts < 0) {
                int l = s_len ? s_len[seq] : p.context_lens[seq];
                l = l < 0 ? 0 : (l > p.len_cap ? p.len_cap : l);
                len = l;
                nparts = partitions_of(p, l);
            }
            const int64_t count = static_cast<int64_t>(nparts) * p.items_y;
            if (r < first + count) {
                const int64_t local = r - first;
                y = static_cast<int>(local % p.items_y);
                part = static_cast<int>(local / p.items_y);
                return true;
            }
            first += count;
            ++seq;
            nparts = -1;
        }
        return false;
    }
};

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                        unsigned int *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
            raise_flag(status, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// tc_wait for a whole warp: every lane waits, and the warp continues only if
// every lane's wait succeeded, so no lane leaves a loop that the others stay in
// (the warp-wide shuffles and TMEM accesses that follow need all 32 lanes).
__device__ __forceinline__ bool tc_wait_warp(uint64_t *bar, uint32_t parity,
                                             volatile int *abort_flag, unsigned int *status) {
    const bool ok = tc_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

template <typename T, int BS, int GH>
__global__ void __launch_bounds__(256, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
    using L = TcLayout;
    constexpr int TILE = L::kTile, D = L::kD;
    constexpr int BLOCKS_PER_TILE = TILE / BS;
    constexpr bool kBF16 = sizeof(T) == 2 && !std::is_same<T, __half>::value;
    static_assert(GH == 4 || GH == 8 || GH == 16, "tensor-core path serves 4, 8 or 16 heads");
    static_assert(BLOCKS_PER_TILE <= 32, "one table entry per producer lane");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm =
        smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
    constexpr int KS = L::kKStages, VS = L::kVStages;
    uint64_t *k_full = bars;              // [KS] K tile landed -> MMA
    uint64_t *k_empty = k_full + KS;      // [KS] QK^T done -> TMA
    uint64_t *v_full = k_empty + KS;      // [VS] V tile landed -> MMA
    uint64_t *v_empty = v_full + VS;      // [VS] PV done -> TMA
    uint64_t *s_full = v_empty + VS;      // [2] QK done -> softmax
    uint64_t *s_empty = s_full + 2;       // [2] S read -> MMA
    uint64_t *p_full = s_full + 4;        // [2] P written -> MMA
    uint64_t *o_full = s_full + 6;        // [2] PV done -> softmax
    uint64_t *o_empty = s_full + 8;       // [2] O read -> MMA
    uint64_t *max_bar = s_full + 10;      // [2] softmax tile-max exchange
    uint64_t *lsum_bar = s_full + 12;     // softmax l exchange
    uint64_t *drain_bar = s_full + 13;    // MMA drain on exit
    uint64_t *drain_pv = s_full + 14;     // PV issuer's drain on exit
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffMisc + 4);
    float *red_max = reinterpret_cast<float *>(sm + L::kOffRed);            // [2][4][16]
    float *red_l = red_max + 2 * 4 * 16;                                       // [4][16]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t smem_base = static_cast<uint32_t>(__cvta_generic_to_shared(sm));

    // ---- set-up: zero the Q / P panels (padding rows stay zero), barriers, TMEM
    for (int i = threadIdx.x; i < 4 * L::kPanelBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(sm + L::kOffQ)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < KS; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < VS; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], 4);
            mbar_init(&p_full[b], 4);
            mbar_init(&o_full[b], 1);
            mbar_init(&o_empty[b], 4);
            mbar_init(&max_bar[b], 4);
        }
        mbar_init(lsum_bar, 4);
        mbar_init(drain_bar, 1);
        mbar_init(drain_pv, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tensormap(&tmap_k);
        tc::prefetch_tensormap(&tmap_v);
    }
    const bool staged = p.num_seqs <= L::kMaxStagedSeqs;
    int *s_len = staged ? reinterpret_cast<int *>(sm + L::kOffLens) : nullptr;
    if (staged) {
        bool bad = false;
        for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
            const int l = p.context_lens[i];
            bad |= (l < 0 || l > p.len_cap);
            s_len[i] = l < 0 ? 0 : (l > p.len_cap ? p.len_cap : l);
        }
        if (bad && blockIdx.x == 0) raise_flag(p.status, PKV_DEVERR_CONTEXT_LEN);
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == 6) {
        // ===================== TMA producers: K (warp 0), V (warp 6) =====================
        // Separate producers so a K tile never waits behind a V slot that its PV still
        // holds; each loads the next tile's table entries while it waits for a slot.
        const int kv = warp == 6;
        const int nst = kv ? VS : KS;
        uint64_t *full = kv ? v_full : k_full;
        uint64_t *empty = kv ? v_empty : k_empty;
        const CUtensorMap *map = kv ? &tmap_v : &tmap_k;
        unsigned char *ring = sm + (kv ? L::kOffV : L::kOffK);
        const uint64_t policy = l2_policy_evict_first();
        // the CTA's tiles in order: item (sequence, KV head, partition), tile offset
        struct Cursor {
            ItemWalker walk;
            int64_t r;
            int tok0 = 0, ntok = 0, t0 = 0, kvh = 0;
            bool valid = false;
        } cur;
        cur.r = blockIdx.x;
        auto next_item = [&](Cursor &c) {
            int y, part;
            while (c.walk.seek(p, s_len, c.r, y, part)) {
                c.r += gridDim.x;
                c.tok0 = p.tok_begin + part * p.partition_size;
                c.ntok = max(0, min(c.walk.len, c.tok0 + p.partition_size) - c.tok0);
                if (c.ntok > 0) {
                    c.t0 = 0;
                    c.kvh = y / p.subgroups;
                    c.valid = true;
                    return;
                }
            }
            c.valid = false;
        };
        auto entry = [&](const Cursor &c) -> int {  // this lane's block of the tile (-1: none / bad)
            const int nblk = (min(TILE, c.ntok - c.t0) + BS - 1) / BS;
            int e = -1;
            if (lane < nblk) {
                e = p.block_tables[static_cast<int64_t>(c.walk.seq) * p.max_blocks_per_seq +
                                   (c.tok0 + c.t0) / BS + lane];
                if (e < 0 || e >= p.num_blocks) {
                    if (kv == 0) raise_flag(p.status, PKV_DEVERR_BLOCK_TABLE);
                    e = -1;
                }
            }
            return e;
        };
        next_item(cur);
        int e_next = cur.valid ? entry(cur) : -1;
        int last_issue[8];
        for (int i = 0; i < 8; ++i) last_issue[i] = -1;
        bool ok = true;
        for (uint32_t g = 0; cur.valid && ok; ++g) {
            const int e = e_next;
            const int kvh = cur.kvh;
            cur.t0 += TILE;
            if (cur.t0 >= cur.ntok) next_item(cur);
            if (cur.valid) e_next = entry(cur);  // in flight while this tile waits
            const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, e >= 0)) * BS * 256u;
            const int s = g % nst;
            int go = 1;
            if (lane == 0) {
                go = tc_wait(&empty[s], ((g / nst) & 1) ^ 1, abort_flag, p.status);
                if (go) {
                    if (bytes) mbar_arrive_expect_tx(&full[s], bytes);
                    else mbar_arrive(&full[s]);
                    last_issue[s] = static_cast<int>(g);
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) {
                ok = false;
                break;
            }
            if (e >= 0) {
                unsigned char *slot = ring + s * L::kKVBytes;
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    tc::tma_load_3d(slot + c * L::kHalfBytes + lane * BS * 128, map, c * 64, kvh * BS, e,
                                    &full[s], policy);
            }
            __syncwarp();
        }
        if (!ok && lane == 0) {
            // let every copy this warp issued land before the CTA exits
            for (int s = 0; s < nst; ++s)
                if (last_issue[s] >= 0)
                    mbar_wait_bounded(&full[s], (last_issue[s] / nst) & 1, kDrainTimeoutNs);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        // QK^T of each tile in order, as soon as its K landed and its S buffer is
        // free (PV is issued by warp 7).
        constexpr uint32_t idesc_qk = tc::idesc_f16_f32acc(kBF16, 128, L::kN, false, false);
        // Queries of the next item that has tiles, loaded into registers one
        // item ahead so no global load sits in front of an item's first MMA.
        constexpr int QCHUNKS = (GH * 16 + 31) / 32;  // 16-byte chunks per lane
        ItemWalker ahead;
        int64_t r_ahead = blockIdx.x;
        uint4 qreg[QCHUNKS];
        auto load_next_q = [&]() {
            int ya, pa;
            while (ahead.seek(p, s_len, r_ahead, ya, pa)) {
                r_ahead += gridDim.x;
                const int t0a = p.tok_begin + pa * p.partition_size;
                if (min(ahead.len, t0a + p.partition_size) - t0a <= 0) continue;
                const int hqa = (ya / p.subgroups) * p.group + (ya % p.subgroups) * GH;
                const T *qsrc = static_cast<const T *>(p.q) +
                                (static_cast<int64_t>(ahead.seq) * p.num_q_heads + hqa) * D;
#pragma unroll
                for (int c = 0; c < QCHUNKS; ++c) {
                    const int i = lane + c * 32;
                    if (i < GH * 16)
                        qreg[c] = *reinterpret_cast<const uint4 *>(qsrc + (i >> 4) * D + (i & 15) * 8);
                }
                return;
            }
        };
        load_next_q();

        // tiles in QK^T order: the current item and the tile offset within it
        ItemWalker walk;
        int64_t r = blockIdx.x;
        int tok0 = 0, ntok = 0, t0 = 0;
        auto next_item = [&]() -> bool {
            int y, part;
            while (walk.seek(p, s_len, r, y, part)) {
                r += gridDim.x;
                tok0 = p.tok_begin + part * p.partition_size;
                ntok = max(0, min(walk.len, tok0 + p.partition_size) - tok0);
                if (ntok > 0) {
                    t0 = 0;
                    return true;
                }
            }
            return false;
        };
        bool have_tile = next_item();
        uint32_t n_qk = 0;   // tiles whose QK^T has been issued
        uint32_t items = 0;  // items whose queries went to a panel
        bool ok = true;
        while (ok && have_tile) {
            int go = 1;
            if (lane == 0)
                go = tc_wait(&k_full[n_qk % KS], (n_qk / KS) & 1, abort_flag, p.status) &&
                     tc_wait(&s_empty[n_qk & 1], ((n_qk >> 1) & 1) ^ 1, abort_flag, p.status);
            if (!__shfl_sync(0xffffffffu, go, 0)) {
                ok = false;
                break;
            }
            const int qb = (items - (t0 == 0 ? 0 : 1)) & 1;  // panel of this tile's item
            if (t0 == 0) {
                // this item's queries -> Q panel qb (K-major, 128-byte swizzle).  The
                // QK^T that last read this panel (two items back) has completed: the
                // s_empty wait above showed S of tile n_qk-2 was consumed.
                unsigned char *panel = sm + L::kOffQ + qb * L::kPanelBytes;
#pragma unroll
                for (int c = 0; c < QCHUNKS; ++c) {
                    const int i = lane + c * 32;
                    if (i < GH * 16) {
                        const int row = i >> 4, c8 = i & 15;
                        const uint32_t off = ((c8 >> 3) * 2 + (row >> 3)) * 1024 + (row & 7) * 128 +
                                             (((c8 & 7) ^ (row & 7)) << 4);
                        *reinterpret_cast<uint4 *>(panel + off) = qreg[c];
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                ++items;
            }
            if (lane == 0) {
                const uint32_t g = n_qk;
                const int b = g & 1;
                tc::fence_after_sync();
                const uint32_t k_addr = smem_base + L::kOffK + (g % KS) * L::kKVBytes;
                const uint32_t q_addr = smem_base + L::kOffQ + qb * L::kPanelBytes;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t a = tc::smem_desc_sw128(
                        k_addr + (k / 4) * L::kHalfBytes + (k % 4) * 32, 16, 1024);
                    const uint64_t bd =
                        tc::smem_desc_sw128(q_addr + (k / 4) * 2048 + (k % 4) * 32, 16, 1024);
                    tc::mma_f16_ss(tmem + 16 * b, a, bd, idesc_qk, k > 0);
                }
                tc::mma_commit(&s_full[b]);
                tc::mma_commit(&k_empty[g % KS]);
            }
            __syncwarp();
            if (t0 == 0) load_next_q();
            ++n_qk;
            t0 += TILE;
            if (t0 >= ntok) have_tile = next_item();
        }
        if (lane == 0) {
            // all MMAs of this CTA complete before TMEM is released
            tc::mma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, kDrainTimeoutNs);
        }
        __syncwarp();
    } else if (warp == 7) {
        // ===================== PV issuer =====================
        // PV of tile t as soon as P(t) is written (and V(t) landed, O(t) of two
        // tiles back read): a second issuing thread, so a PV never waits behind the
        // QK^T batch of the next tile (an MMA batch holds its issuing thread for
        // its whole execution).
        constexpr uint32_t idesc_pv = tc::idesc_f16_f32acc(kBF16, 128, L::kN, true, false);
        ItemWalker walk;
        uint32_t t = 0;
        bool ok = true;
        for (int64_t r = blockIdx.x; ok; r += gridDim.x) {
            int y, part;
            if (!walk.seek(p, s_len, r, y, part)) break;
            const int tok0 = p.tok_begin + part * p.partition_size;
            const int ntok = max(0, min(walk.len, tok0 + p.partition_size) - tok0);
            for (int t0 = 0; t0 < ntok; t0 += TILE, ++t) {
                int go = 1;
                if (lane == 0)
                    go = tc_wait(&p_full[t & 1], (t >> 1) & 1, abort_flag, p.status) &&
                         tc_wait(&o_empty[t & 1], ((t >> 1) & 1) ^ 1, abort_flag, p.status) &&
                         tc_wait(&v_full[t % VS], (t / VS) & 1, abort_flag, p.status);
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int b = t & 1;
                    tc::fence_after_sync();
                    const uint32_t v_addr = smem_base + L::kOffV + (t % VS) * L::kKVBytes;
                    const uint32_t p_addr = smem_base + L::kOffP + b * L::kPanelBytes;
#pragma unroll
                    for (int k = 0; k < TILE / 16; ++k) {
                        const uint64_t a = tc::smem_desc_sw128(v_addr + k * 2048, L::kHalfBytes, 1024);
                        const uint64_t bd =
                            tc::smem_desc_sw128(p_addr + (k / 4) * 2048 + (k % 4) * 32, 16, 1024);
                        tc::mma_f16_ss(tmem + 32 + 16 * b, a, bd, idesc_pv, k > 0);
                    }
                    tc::mma_commit(&o_full[b]);
                    tc::mma_commit(&v_empty[t % VS]);
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            // this thread's MMAs complete before TMEM is released
            tc::mma_commit(drain_pv);
            mbar_wait_bounded(drain_pv, 0, kDrainTimeoutNs);
        }
        __syncwarp();
    } else {
        // ===================== softmax / accumulate (warps 2..5) =====================
        // The PV of a tile is folded into o after the softmax of the next tile,
        // also across work items: an item's last tile, its cross-warp l sum and its
        // write-out happen after the next item's first tile, so the warps never
        // wait for the tail of an item's MMAs before starting the next one.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // token row of S, head-dim row of O^T
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);

        struct Item {
            int64_t qrow0;  // (sequence, first query head) row of the output
            int part, nparts;
            float m[GH], lp[GH], o[GH];
        };
        Item cur, pend;   // the item being worked on; the finished one awaiting its last PV
        bool pend_valid = false;
        float alpha_prev[GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) alpha_prev[h] = 0.f;
        ItemWalker walk;
        uint32_t g = 0;
        uint32_t epilogues = 0;
        bool ok = true;
        bool flagged_len = false;

        auto accumulate = [&](uint32_t t, Item &it) -> bool {
            const int b = t & 1;
            if (!tc_wait_warp(&o_full[b], (t >> 1) & 1, abort_flag, p.status)) return false;
            tc::fence_after_sync();
            float pv[GH];
            tc::tmem_ld<GH>(lane_base + 32 + 16 * b, pv);
            tc::tmem_ld_wait();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[b]);
#pragma unroll
            for (int h = 0; h < GH; ++h) it.o[h] = fmaf(it.o[h], alpha_prev[h], pv[h]);
            return true;
        };
        // l = sum over the 128 token rows; then the item's output (row = head-dim index)
        auto epilogue = [&](Item &it) -> bool {
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                float v = it.lp[h];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                it.lp[h] = v;
            }
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < GH; ++h) red_l[quarter * 16 + h] = it.lp[h];
                mbar_arrive(lsum_bar);
            }
            if (!tc_wait_warp(lsum_bar, epilogues & 1, abort_flag, p.status)) return false;
            ++epilogues;
#pragma unroll
            for (int h = 0; h < GH; ++h)
                it.lp[h] = red_l[h] + red_l[16 + h] + red_l[32 + h] + red_l[48 + h];
            if (it.nparts == 1 && !p.always_partial) {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const float res = it.lp[h] > 0.f ? it.o[h] / it.lp[h] : 0.f;
                    static_cast<T *>(p.out)[(it.qrow0 + h) * D + row] = Elem<T>::from_f32(res);
                }
            } else {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const int64_t pr = (it.qrow0 + h) * p.num_partitions + p.slot_base + it.part;
                    p.ws_o[pr * D + row] = it.o[h];
                    if (row == 0) {
                        p.ws_m[pr] = it.m[h];
                        p.ws_l[pr] = it.lp[h];
                    }
                }
            }
            return true;
        };

        for (int64_t r = blockIdx.x; ok; r += gridDim.x) {
            int y, part;
            if (!walk.seek(p, s_len, r, y, part)) break;
            if (!staged && !flagged_len && warp == 2 && lane == 0) {
                const int raw = p.context_lens[walk.seq];
                if (raw < 0 || raw > p.len_cap) {
                    raise_flag(p.status, PKV_DEVERR_CONTEXT_LEN);
                    flagged_len = true;
                }
            }
            const int tok0 = p.tok_begin + part * p.partition_size;
            const int ntok = max(0, min(walk.len, tok0 + p.partition_size) - tok0);
            const int kvh = y / p.subgroups;
            const int64_t qrow0 = static_cast<int64_t>(walk.seq) * p.num_q_heads + kvh * p.group +
                                  (y % p.subgroups) * GH;
            if (ntok == 0) {
                // no tokens (empty context or empty range): a zero result, nothing to wait for
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    if (walk.nparts == 1 && !p.always_partial) {
                        static_cast<T *>(p.out)[(qrow0 + h) * D + row] = Elem<T>::from_f32(0.f);
                    } else {
                        const int64_t pr = (qrow0 + h) * p.num_partitions + p.slot_base + part;
                        p.ws_o[pr * D + row] = 0.f;
                        if (row == 0) {
                            p.ws_m[pr] = -INFINITY;
                            p.ws_l[pr] = 0.f;
                        }
                    }
                }
                continue;
            }
            cur.qrow0 = qrow0;
            cur.part = part;
            cur.nparts = walk.nparts;
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                cur.m[h] = -INFINITY;
                cur.lp[h] = 0.f;
                cur.o[h] = 0.f;
            }
            for (int t0 = 0; t0 < ntok; t0 += TILE, ++g) {
                const int tile_ntok = min(TILE, ntok - t0);
                const int b = g & 1;
                if (!tc_wait_warp(&s_full[b], (g >> 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                float sv[GH];
                tc::tmem_ld<GH>(lane_base + 16 * b, sv);
                tc::tmem_ld_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[b]);

                const bool valid = row < tile_ntok;
                float mx[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    sv[h] = valid ? sv[h] * p.scale_log2 : -INFINITY;
                    float v = sv[h];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                    mx[h] = v;
                }
                float *red = red_max + (g & 1) * 64;
                if (lane == 0) {
#pragma unroll
                    for (int h = 0; h < GH; ++h) red[quarter * 16 + h] = mx[h];
                    mbar_arrive(&max_bar[g & 1]);
                }
                if (!tc_wait_warp(&max_bar[g & 1], (g >> 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                float alpha[GH];
                unsigned char *panel = sm + L::kOffP + b * L::kPanelBytes;
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const float tmax = fmaxf(fmaxf(red[h], red[16 + h]), fmaxf(red[32 + h], red[48 + h]));
                    const float m_new = fmaxf(cur.m[h], tmax);
                    alpha[h] = fast_exp2(cur.m[h] - m_new);  // 0 on the first tile (m = -inf)
                    cur.m[h] = m_new;
                    const float pf = valid ? fast_exp2(sv[h] - m_new) : 0.f;
                    const T p16 = Elem<T>::from_f32(pf);
                    cur.lp[h] = fmaf(cur.lp[h], alpha[h], static_cast<float>(p16));
                    const uint32_t off = ((row >> 6) * 2 + (h >> 3)) * 1024 + tc::sw128_offset(h & 7, row & 63);
                    *reinterpret_cast<T *>(panel + off) = p16;
                }
                if (tile_ntok < TILE) {
                    // rows past the context: zero their V so 0 * stale never reaches the MMA
                    const int s = g % VS;
                    if (!tc_wait_warp(&v_full[s], (g / VS) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    if (!valid) {
                        unsigned char *vrow = sm + L::kOffV + s * L::kKVBytes + row * 128;
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                reinterpret_cast<uint4 *>(vrow + c * L::kHalfBytes)[i] = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
                // fold in the previous tile: the last tile of the pending item, or this item's
                if (t0 == 0 && pend_valid) {
                    if (!accumulate(g - 1, pend) || !epilogue(pend)) {
                        ok = false;
                        break;
                    }
                    pend_valid = false;
                } else if (t0 > 0 && !accumulate(g - 1, cur)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int h = 0; h < GH; ++h) alpha_prev[h] = alpha[h];
            }
            if (!ok) break;
            pend = cur;  // its last tile (g - 1) is folded in after the next tile
            pend_valid = true;
        }
        if (ok && pend_valid) {
            if (accumulate(g - 1, pend)) epilogue(pend);
        }
    }

    // ---- tear-down: every role is done with TMEM and shared memory
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace pkv
