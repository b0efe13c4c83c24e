// prefix_tc_kernel.cuh -- the shared-prefix half of a cascade decode.
//
// When every sequence of a batch starts with the same prefix blocks (prefix
// caching: "KV Cache与PagedAttention深度解析" §8.2, the nano-vllm article
// (zwxr.cn) §2.3 / §3), the decode of all B*G query rows of a KV head over the
// prefix is one dense attention: S = Q K_prefix^T for a [B*G x prefix] tile,
// then P V_prefix.  Reading the prefix once per 128 query rows instead of once
// per sequence removes the prefix's repeated reads.  This kernel computes, for
// a tile of 128 query rows of one KV head and one split of the prefix, the
// partial (o, m, l) of each row (same definition as the decode kernels:
// P1 §2.1, running max / running sum of §7.2) and writes it to a workspace
// slot; the suffix of each sequence is decoded by the usual kernels into the
// following slots and the log-sum-exp merge combines them.
//
// tcgen05 MMAs, M = 128 query rows, N = 128 tokens, K = 128 (head_dim):
//   S  = Q . K^T      A = Q tile (K-major), B = K tile (K-major)
//   O += P . V        A = P from TMEM, B = V tile (MN-major: head_dim contiguous)
// S is double-buffered in TMEM (2 x 128 columns), O accumulates in TMEM (128
// columns); P is written back over its scores (two 16-bit values per column),
// so shared memory holds only Q and three-slot K and V rings, whose depth
// covers the load latency while the suffix decode keeps HBM busy.  A row's softmax belongs to one pair of threads (TMEM lane = query
// row), each taking 64 of the tile's 128 columns; the pair exchanges its
// partial row maxima through spare TMEM columns, so both halves use one
// reference maximum.  That maximum is raised only when a tile's maximum
// exceeds it by more than kRescaleLog2 (then O and l are rescaled in place),
// so P <= 2^kRescaleLog2.  P is rounded to the input type for the MMA; l adds
// the fp32 values (unbiased rounding, relative error 2^-9 per weight at most).
//
// Warps: 0 / 10 TMA producers of the K ring and the V ring (3 slots each, 3-D
// tiled copies with 128-byte swizzle), 1 TMEM owner + QK^T issuer, 11 PV issuer,
// 2-9 softmax in pairs (warps w and w + 4 share TMEM lane quarter w & 3).
#pragma once

#include <cuda.h>

#include <type_traits>

#include "decode_kernel.cuh"
#include "pkv_tc.cuh"

namespace pkv {

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

struct PrefixParams {
    const void *q;
    float *ws_o;
    float *ws_m;
    float *ws_l;
    const int32_t *prefix_table;  // [prefix_len / block_size] physical blocks
    const int32_t *context_lens;
    unsigned int *status;
    int64_t num_blocks;
    int num_seqs;
    int num_q_heads;
    int group;            // query heads per KV head
    int rows;             // num_seqs * group
    int prefix_len;       // tokens, a multiple of block_size
    int split_tokens;     // tokens per prefix split, a multiple of 128
    int num_partitions;   // workspace slots per (sequence, query head)
    float scale_log2;
};

struct PrefixLayout {
    static constexpr int kThreads = 384;               // 12 warps (roles below)
    static constexpr int kTile = 128;
    static constexpr int kHalf = 128 * 128;            // 128 rows x 128 B
    static constexpr int kPanel = 2 * kHalf;           // 128 rows x 128 16-bit values
    static constexpr int kOffQ = 0;
    static constexpr int kKS = 3, kVS = 3;             // K / V ring slots
    static constexpr int kOffK = kOffQ + kPanel;
    static constexpr int kOffV = kOffK + kKS * kPanel;
    static constexpr int kOffBar = kOffV + kVS * kPanel;
    static constexpr int kNumBars = 2 * kKS + 2 * kVS + 8 + 2 + 8;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kSmemBytes = kBytes + 1024;
    static constexpr uint32_t kTmemCols = 512;           // S[2] (P[b] over S[b]) at 0 / 128, O at 256, exchange 384
    static constexpr uint32_t kXchgCol = 384;            // spare TMEM columns for the pairs
    static constexpr float kRescaleLog2 = 8.f;
};

template <typename T, int BS>
__global__ void __launch_bounds__(PrefixLayout::kThreads, 1)
    paged_prefix_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const PrefixParams p) {
    using L = PrefixLayout;
    constexpr int TILE = L::kTile, D = 128, kThreads = L::kThreads, KS = L::kKS, VS = L::kVS;
    static_assert(VS >= 2, "V slots >= S buffers (2): see the V-row zeroing wait");
    constexpr bool kBF16 = !std::is_same<T, __half>::value;
    static_assert(TILE / BS <= 32, "one table entry per producer lane");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm =
        smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
    uint64_t *k_full = bars, *k_empty = k_full + KS, *v_full = k_empty + KS, *v_empty = v_full + VS;
    uint64_t *s_full = v_empty + VS, *s_empty = s_full + 2, *p_full = s_empty + 2, *o_done = p_full + 2;
    uint64_t *drain_bar = o_done + 2;    // [QK issuer, PV issuer]
    uint64_t *pair_bar = drain_bar + 2;  // [quarter][parity]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffMisc + 4);

    // the suffix decode, launched behind this kernel, may start on the SMs this grid
    // leaves free (its last CTA waits for this grid before it exits)
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_tile = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
    const int tok_lo = split * p.split_tokens;
    const int tok_hi = min(p.prefix_len, tok_lo + p.split_tokens);
    const int ntiles = tok_hi > tok_lo ? (tok_hi - tok_lo + TILE - 1) / TILE : 0;
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 1);  // committed by PV(j): P[b] lives over S[b]
            mbar_init(&p_full[i], 8);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(&drain_bar[0], 1);
        mbar_init(&drain_bar[1], 1);
        for (int i = 0; i < 8; ++i) mbar_init(&pair_bar[i], 2);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::kTmemCols);
        tc::tmem_relinquish();
    }
    // query rows of this tile -> Q panel (K-major, 128-byte swizzle); rows past the
    // batch are zero.  Every thread issues all of its loads before its first store,
    // so the panel costs about one global-memory latency, not one per vector.
    {
        constexpr int kItems = 128 * 16, kPer = (kItems + kThreads - 1) / kThreads;
        uint4 v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int i = threadIdx.x + u * kThreads;
            const int r = i >> 4, c8 = i & 15;
            const int grow = row_tile * 128 + r;
            v[u] = make_uint4(0, 0, 0, 0);
            if (i < kItems && grow < p.rows) {
                const int seq = grow / p.group, g = grow - seq * p.group;
                const T *src = static_cast<const T *>(p.q) +
                               (static_cast<int64_t>(seq) * p.num_q_heads + kvh * p.group + g) * D;
                v[u] = *reinterpret_cast<const uint4 *>(src + c8 * 8);
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int i = threadIdx.x + u * kThreads;
            const int r = i >> 4, c8 = i & 15;
            if (i < kItems)
                *reinterpret_cast<uint4 *>(sm + L::kOffQ + (c8 >> 3) * L::kHalf + r * 128 +
                                           (((c8 & 7) ^ (r & 7)) << 4)) = v[u];
        }
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tensormap(&tmap_k);
        tc::prefetch_tensormap(&tmap_v);
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == 10) {
        // ===================== TMA producers: K (warp 0), V (warp 10) =====================
        // Separate producers so a K tile never waits behind a V slot that its PV still
        // holds; each loads the next tile's table entries while it waits for a slot.
        const int kv = warp == 10;
        uint64_t *full = kv ? v_full : k_full;
        uint64_t *empty = kv ? v_empty : k_empty;
        const int nst = kv ? VS : KS;
        const CUtensorMap *map = kv ? &tmap_v : &tmap_k;
        unsigned char *ring = sm + (kv ? L::kOffV : L::kOffK);
        const uint64_t policy = l2_policy_evict_last();  // the prefix is read by every row tile
        auto entry = [&](int j) -> int {  // this lane's block of tile j (-1: none or bad)
            const int t0 = tok_lo + j * TILE;
            const int nblk = (min(TILE, tok_hi - t0) + BS - 1) / BS;
            int e = -1;
            if (lane < nblk) {
                e = p.prefix_table[t0 / BS + lane];
                if (e < 0 || e >= p.num_blocks) {
                    if (kv == 0) raise_flag(p.status, PKV_DEVERR_BLOCK_TABLE);
                    e = -1;
                }
            }
            return e;
        };
        int last_issue[3] = {-1, -1, -1};
        bool ok = true;
        int e_next = ntiles > 0 ? entry(0) : -1;
        for (int j = 0; j < ntiles && ok; ++j) {
            const int e = e_next;
            if (j + 1 < ntiles) e_next = entry(j + 1);  // in flight while this tile waits
            const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, e >= 0)) * BS * 256u;
            const int s = j % nst;
            int go = 1;
            if (lane == 0) {
                go = tc_wait(&empty[s], ((j / nst) & 1) ^ 1, abort_flag, p.status);
                if (go) {
                    if (bytes) mbar_arrive_expect_tx(&full[s], bytes);
                    else mbar_arrive(&full[s]);
                    last_issue[s] = j;
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
                    tc::tma_load_3d(slot + c * L::kHalf + lane * BS * 128, map, c * 64, kvh * BS, e,
                                    &full[s], policy);
            }
            __syncwarp();
        }
        if (!ok && lane == 0) {
            for (int s = 0; s < nst; ++s)
                if (last_issue[s] >= 0)
                    mbar_wait_bounded(&full[s], (last_issue[s] / nst) & 1, kDrainTimeoutNs);
        }
    } else if (warp == 1) {
        // ===================== QK^T issuer =====================
        // QK^T of each tile as soon as its K landed and its S buffer is free; PV is
        // issued by warp 11, so a ready PV never waits behind a QK^T batch (a batch of
        // MMAs holds its issuing thread for its whole execution).
        constexpr uint32_t idesc_qk = tc::idesc_f16_f32acc(kBF16, 128, 128, false, false);
        for (int j = 0; j < ntiles; ++j) {
            int go = 1;
            if (lane == 0)
                go = tc_wait(&k_full[j % KS], (j / KS) & 1, abort_flag, p.status) &&
                     tc_wait(&s_empty[j & 1], ((j >> 1) & 1) ^ 1, abort_flag, p.status);
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            if (lane == 0) {
                const int b = j & 1;
                tc::fence_after_sync();
                const uint32_t qa = smem_base + L::kOffQ;
                const uint32_t ka = smem_base + L::kOffK + (j % KS) * L::kPanel;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t a = tc::smem_desc_sw128(qa + (k / 4) * L::kHalf + (k % 4) * 32, 16, 1024);
                    const uint64_t bd = tc::smem_desc_sw128(ka + (k / 4) * L::kHalf + (k % 4) * 32, 16, 1024);
                    tc::mma_f16_ss(tmem + 128 * b, a, bd, idesc_qk, k > 0);
                }
                tc::mma_commit(&s_full[b]);
                tc::mma_commit(&k_empty[j % KS]);
            }
            __syncwarp();
        }
        if (lane == 0) {
            // this thread's MMAs complete before TMEM is released
            tc::mma_commit(&drain_bar[0]);
            mbar_wait_bounded(&drain_bar[0], 0, kDrainTimeoutNs);
        }
        __syncwarp();
    } else if (warp == 11) {
        // ===================== PV issuer =====================
        constexpr uint32_t idesc_pv = tc::idesc_f16_f32acc(kBF16, 128, 128, false, true);
        for (int j = 0; j < ntiles; ++j) {
            int go = 1;
            if (lane == 0)
                go = tc_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, p.status) &&
                     tc_wait(&v_full[j % VS], (j / VS) & 1, abort_flag, p.status);
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            if (lane == 0) {
                const int b = j & 1;
                tc::fence_after_sync();
                const uint32_t va = smem_base + L::kOffV + (j % VS) * L::kPanel;
#pragma unroll
                for (int k = 0; k < TILE / 16; ++k) {
                    const uint64_t bd = tc::smem_desc_sw128(va + k * 2048, L::kHalf, 1024);
                    // P from TMEM: 16 tokens = 8 packed columns per step
                    tc::mma_f16_ts(tmem + 256, tmem + 128 * b + 8 * k, bd, idesc_pv, j > 0 || k > 0);
                }
                tc::mma_commit(&o_done[b]);
                tc::mma_commit(&s_empty[b]);  // S[b] / P[b] free for QK^T(j + 2)
                tc::mma_commit(&v_empty[j % VS]);
            }
            __syncwarp();
        }
        if (lane == 0) {
            tc::mma_commit(&drain_bar[1]);
            mbar_wait_bounded(&drain_bar[1], 0, kDrainTimeoutNs);
        }
        __syncwarp();
    } else {
        // ===================== softmax (warps 2..9): thread = query row, 64 columns =====================
        const int quarter = warp & 3;
        const int half = warp >= 6 ? 1 : 0;  // tile columns 64 half .. +63
        const int c0 = half * 64;
        const int r = quarter * 32 + lane;   // row within the tile = TMEM lane
        const int grow = row_tile * 128 + r;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t xchg = lane_base + L::kXchgCol;
        // One value per row between the two warps of the pair: step s writes column
        // 2 (s & 1) + half and reads the partner's; a warp reuses a column two steps
        // later, after the partner has passed the step in between.
        auto exchange = [&](int step, float mine, float &other) -> bool {
            const int par = step & 1;
            tc::tmem_st_x1(xchg + 2 * par + half, mine);
            tc::tmem_st_wait();
            tc::fence_before_sync();
            __syncwarp();
            uint64_t *pb = &pair_bar[quarter * 2 + par];
            if (lane == 0) mbar_arrive(pb);
            if (!tc_wait_warp(pb, (step >> 1) & 1, abort_flag, p.status)) return false;
            tc::fence_after_sync();
            other = tc::tmem_ld_x1(xchg + 2 * par + (1 - half));
            tc::tmem_ld_wait();
            return true;
        };
        const bool pos_scale = p.scale_log2 > 0.f;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        int xs = 0;  // pair exchanges so far
        for (int j = 0; j < ntiles && ok; ++j) {
            const int b = j & 1;
            const int t0 = tok_lo + j * TILE;
            const int valid = min(TILE, tok_hi - t0);  // >= 1: column 0 is always in the prefix
            const int vh = max(0, min(64, valid - c0));  // ... of this half
            if (!tc_wait_warp(&s_full[b], (j >> 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            // this row's 64 scores of the half, read from TMEM once; the half's extreme
            // raw score (max for a positive scale, min otherwise; a half past the prefix
            // end contributes the neutral infinity)
            float x[64];
#pragma unroll
            for (int c = 0; c < 64; c += 16) tc::tmem_ld_x16(lane_base + 128 * b + c0 + c, x + c);
            tc::tmem_ld_wait();
            const bool full = vh == 64;  // uniform over the warp
            float ext;
            if (full) {
                ext = x[0];
#pragma unroll
                for (int i = 1; i + 1 < 64; i += 2)
                    ext = pos_scale ? fmax3(ext, x[i], x[i + 1]) : fmin3(ext, x[i], x[i + 1]);
                ext = pos_scale ? fmaxf(ext, x[63]) : fminf(ext, x[63]);
            } else {
                ext = pos_scale ? -INFINITY : INFINITY;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i < vh) ext = pos_scale ? fmaxf(ext, x[i]) : fminf(ext, x[i]);
            }
            float ext_other;
            if (!exchange(xs++, ext, ext_other)) {
                ok = false;
                break;
            }
            // both threads of the pair derive the same tile maximum and reference
            const float tmax = (pos_scale ? fmaxf(ext, ext_other) : fminf(ext, ext_other)) * p.scale_log2;
            // the reference maximum moves only by more than kRescaleLog2; TMEM loads and
            // stores are warp-wide, so the warp rescales if any of its rows must (the
            // two warps of a pair see the same rows, so they decide alike)
            const float new_ref = tmax > m_ref + L::kRescaleLog2 ? tmax : m_ref;
            const float alpha = fast_exp2(m_ref - new_ref);  // 1 if unchanged, 0 on the first tile
            if (__any_sync(0xffffffffu, new_ref != m_ref)) {
                if (j > 0) {
                    // O holds tiles < j: wait for PV(j-1), rescale this half of O in TMEM
                    if (!tc_wait_warp(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
#pragma unroll
                    for (int c = 0; c < 64; c += 16) {
                        float o[16];
                        tc::tmem_ld_x16(lane_base + 256 + c0 + c, o);
                        tc::tmem_ld_wait();
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(o[i] * alpha);
                        tc::tmem_st_x16(lane_base + 256 + c0 + c, w);
                    }
                    tc::tmem_st_wait();
                }
                l *= alpha;
                m_ref = new_ref;
            }
            // P = 2^(s - m_ref) (0 past the prefix end), rounded to T and packed two per
            // 32-bit column over the first 64 columns of S[b] (tokens 64 half .. +63 ->
            // columns 32 half .. +31; both threads of the pair have read their scores,
            // the exchange above orders it), where the PV MMA reads it; the row sum l
            // adds the fp32 values.  S[b] was free for QK^T(j) only after PV(j-2).
            const uint32_t pcol = lane_base + 128 * b + 32 * half;
            float l0 = 0.f, l1 = 0.f;
            // two copies of the loop, so full halves carry no per-column mask
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
                // rows of V past the prefix end: zero them (this thread: row r, this
                // half's 64 channels) so 0 * stale never reaches the MMA.  The parity
                // wait cannot pass on an older phase of the slot: S(j) exists only once
                // PV(j-2) has completed (two S buffers), and with VS >= 2 the slot's
                // previous tile, V(j - VS), was consumed by then.
                if (!tc_wait_warp(&v_full[j % VS], (j / VS) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                if (r >= valid) {
                    uint4 *vrow = reinterpret_cast<uint4 *>(sm + L::kOffV + (j % VS) * L::kPanel + half * L::kHalf +
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
        // final: the pair's row sum, then this half of the O row -> workspace slot
        // `split` of the row's (sequence, query head).  TMEM loads are warp-wide:
        // every lane loads, only rows of the batch store.
        if (ntiles > 0) {
            float l_other = 0.f;
            if (ok) ok = exchange(xs++, l, l_other);
            if (ok) ok = tc_wait_warp(&o_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, abort_flag, p.status);
            if (ok) {
                tc::fence_after_sync();
                const bool mine = grow < p.rows;
                int64_t prow_ws = 0;
                if (mine) {
                    const int seq = grow / p.group, g = grow - seq * p.group;
                    prow_ws = (static_cast<int64_t>(seq) * p.num_q_heads + kvh * p.group + g) *
                                  p.num_partitions + split;
                }
#pragma unroll
                for (int c = 0; c < 64; c += 16) {
                    float o[16];
                    tc::tmem_ld_x16(lane_base + 256 + c0 + c, o);
                    tc::tmem_ld_wait();
                    if (mine) {
                        float *dst = p.ws_o + prow_ws * D + c0 + c;
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
                    }
                }
                if (mine && half == 0) {
                    p.ws_m[prow_ws] = m_ref;
                    p.ws_l[prow_ws] = l + l_other;
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

}  // namespace pkv
