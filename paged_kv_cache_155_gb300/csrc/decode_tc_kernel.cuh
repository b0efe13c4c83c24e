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
// Structure (one persistent CTA per SM, 6 warps):
//   warp 0      TMA producer: per 128-token tile, one 3-D tiled bulk-tensor copy
//               per (block, 64-column half) for K and for V, 128-byte swizzled,
//               into a 3-stage ring of 64 KiB stages; block-table entries are
//               read one tile ahead.
//   warp 1      TMEM owner and MMA issuer (one thread): QK^T of tile i+1 is
//               issued before PV of tile i so the softmax of tile i overlaps it.
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
    static constexpr int kStages = 3;
    static constexpr int kHalfBytes = 128 * 128;        // 128 rows x 64 columns x 2 B
    static constexpr int kKVBytes = 2 * kHalfBytes;     // K (or V) tile: 32 KiB
    static constexpr int kStageBytes = 2 * kKVBytes;    // K + V: 64 KiB
    static constexpr int kPanelBytes = 4096;            // 16 x 128 x 2 B (Q or P)
    static constexpr int kOffQ = kStages * kStageBytes;
    static constexpr int kOffP = kOffQ + 2 * kPanelBytes;
    static constexpr int kOffRed = kOffP + 2 * kPanelBytes;           // float [2][4][16] + [4][16]
    static constexpr int kOffBar = kOffRed + 3 * 4 * 16 * 4;
    static constexpr int kNumBars = 3 + 3 + 2 * 5 + 2 + 1 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;           // tmem slot, abort flag
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kSmemBytes = kBytes + 1024;                  // + alignment slack
    static constexpr uint32_t kTmemCols = 64;  // S[2] at 0/16, O[2] at 32/48
};

// Walks the work items of a launch in order: item r -> (sequence, y, partition).
// Items of sequence s are nparts(s) * Y consecutive indices.
struct ItemWalker {
    int seq = 0;
    int64_t first = 0;  // index of the first item of `seq`
    int nparts = -1;
    int len = 0;
    __device__ bool seek(const DecodeParams &p, int64_t r, int &y, int &part) {
        while (seq < p.num_seqs) {
            if (nparts < 0) {
                int l = p.context_lens[seq];
                l = l < 0 ? 0 : (l > p.len_cap ? p.len_cap : l);
                len = l;
                nparts = l > 0 ? (l + p.partition_size - 1) / p.partition_size : 1;
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

template <typename T, int BS, int GH>
__global__ void __launch_bounds__(192, 1)
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
    uint64_t *full = bars;            // [3] TMA -> MMA
    uint64_t *empty = bars + 3;       // [3] MMA -> TMA
    uint64_t *s_full = bars + 6;      // [2] QK done -> softmax
    uint64_t *s_empty = bars + 8;     // [2] S read -> MMA
    uint64_t *p_full = bars + 10;     // [2] P written -> MMA
    uint64_t *o_full = bars + 12;     // [2] PV done -> softmax
    uint64_t *o_empty = bars + 14;    // [2] O read -> MMA
    uint64_t *max_bar = bars + 16;    // [2] softmax tile-max exchange
    uint64_t *lsum_bar = bars + 18;   // softmax l exchange
    uint64_t *drain_bar = bars + 19;  // MMA drain on exit
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
        for (int s = 0; s < 3; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
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
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ===================== TMA producer =====================
        const uint64_t policy = l2_policy_evict_first();
        ItemWalker walk;
        uint32_t g = 0;  // global tile counter
        int last_issue[3] = {-1, -1, -1};
        bool ok = true;
        for (int64_t r = blockIdx.x; ok; r += gridDim.x) {
            int y, part;
            if (!walk.seek(p, r, y, part)) break;
            const int tok0 = part * p.partition_size;
            const int ntok = max(0, min(walk.len, tok0 + p.partition_size) - tok0);
            const int kvh = y / p.subgroups;
            const int32_t *trow = p.block_tables + static_cast<int64_t>(walk.seq) * p.max_blocks_per_seq;
            for (int t0 = 0; t0 < ntok && ok; t0 += TILE, ++g) {
                const int tile_ntok = min(TILE, ntok - t0);
                const int nblk = (tile_ntok + BS - 1) / BS;
                const int blk0 = (tok0 + t0) / BS;
                int e = -1;
                if (lane < nblk) {
                    e = trow[blk0 + lane];
                    if (e < 0 || e >= p.num_blocks) {
                        raise_flag(p.status, PKV_DEVERR_BLOCK_TABLE);
                        e = -1;
                    }
                }
                const unsigned valid = __ballot_sync(0xffffffffu, e >= 0);
                const int s = g % 3;
                int go = 1;
                if (lane == 0) {
                    go = tc_wait(&empty[s], ((g / 3) & 1) ^ 1, abort_flag, p.status);
                    if (go) {
                        const uint32_t bytes = __popc(valid) * BS * 512u;
                        if (bytes) mbar_arrive_expect_tx(&full[s], bytes);
                        else mbar_arrive(&full[s]);
                        last_issue[s] = static_cast<int>(g);
                    }
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
                if (e >= 0) {
                    unsigned char *stage = sm + s * L::kStageBytes;
                    const int row = lane * BS;
                    for (int c = 0; c < 2; ++c) {
                        tc::tma_load_3d(stage + c * L::kHalfBytes + row * 128, &tmap_k, c * 64,
                                        kvh * BS, e, &full[s], policy);
                        tc::tma_load_3d(stage + L::kKVBytes + c * L::kHalfBytes + row * 128, &tmap_v,
                                        c * 64, kvh * BS, e, &full[s], policy);
                    }
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            // let every copy this warp issued land before the CTA exits
            for (int s = 0; s < 3; ++s)
                if (last_issue[s] >= 0)
                    mbar_wait_bounded(&full[s], (last_issue[s] / 3) & 1, kDrainTimeoutNs);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        constexpr uint32_t idesc_qk = tc::idesc_f16_f32acc(kBF16, 128, L::kN, false, false);
        constexpr uint32_t idesc_pv = tc::idesc_f16_f32acc(kBF16, 128, L::kN, true, false);
        ItemWalker walk;
        uint32_t g = 0;
        uint32_t items_with_tiles = 0;
        bool ok = true;
        bool have_prev = false;

        auto issue_pv = [&](uint32_t t) -> bool {
            const int b = t & 1;
            int go = 1;
            if (lane == 0) {
                go = tc_wait(&p_full[b], (t >> 1) & 1, abort_flag, p.status) &&
                     tc_wait(&o_empty[b], ((t >> 1) & 1) ^ 1, abort_flag, p.status);
                if (go) {
                    tc::fence_after_sync();
                    const unsigned char *stage = sm + (t % 3) * L::kStageBytes;
                    const uint32_t v_addr = smem_base + static_cast<uint32_t>(stage - sm) + L::kKVBytes;
                    const uint32_t p_addr = smem_base + L::kOffP + b * L::kPanelBytes;
#pragma unroll
                    for (int k = 0; k < TILE / 16; ++k) {
                        const uint64_t a = tc::smem_desc_sw128(v_addr + k * 2048, L::kHalfBytes, 1024);
                        const uint64_t bd =
                            tc::smem_desc_sw128(p_addr + (k / 4) * 2048 + (k % 4) * 32, 16, 1024);
                        tc::mma_f16_ss(tmem + 32 + 16 * b, a, bd, idesc_pv, k > 0);
                    }
                    tc::mma_commit(&o_full[b]);
                    tc::mma_commit(&empty[t % 3]);
                }
            }
            return __shfl_sync(0xffffffffu, go, 0) != 0;
        };

        for (int64_t r = blockIdx.x; ok; r += gridDim.x) {
            int y, part;
            if (!walk.seek(p, r, y, part)) break;
            const int tok0 = part * p.partition_size;
            const int ntok = max(0, min(walk.len, tok0 + p.partition_size) - tok0);
            if (ntok == 0) continue;
            const int kvh = y / p.subgroups;
            const int hq0 = kvh * p.group + (y % p.subgroups) * GH;
            const int qb = items_with_tiles & 1;
            ++items_with_tiles;
            for (int t0 = 0; t0 < ntok; t0 += TILE, ++g) {
                const int b = g & 1;
                int go = 1;
                if (lane == 0) {
                    go = tc_wait(&full[g % 3], (g / 3) & 1, abort_flag, p.status) &&
                         tc_wait(&s_empty[b], ((g >> 1) & 1) ^ 1, abort_flag, p.status);
                }
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
                if (t0 == 0) {
                    // this item's queries -> Q panel qb (K-major, 128-byte swizzle)
                    const T *qsrc = static_cast<const T *>(p.q) +
                                    (static_cast<int64_t>(walk.seq) * p.num_q_heads + hq0) * D;
                    unsigned char *panel = sm + L::kOffQ + qb * L::kPanelBytes;
                    for (int i = lane; i < GH * 16; i += 32) {
                        const int row = i >> 4, c8 = i & 15;
                        const uint4 v = *reinterpret_cast<const uint4 *>(qsrc + row * D + c8 * 8);
                        const uint32_t off = ((c8 >> 3) * 2 + (row >> 3)) * 1024 + (row & 7) * 128 +
                                             (((c8 & 7) ^ (row & 7)) << 4);
                        *reinterpret_cast<uint4 *>(panel + off) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    tc::fence_after_sync();
                    const uint32_t k_addr = smem_base + (g % 3) * L::kStageBytes;
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
                }
                __syncwarp();
                if (have_prev && !issue_pv(g - 1)) {
                    ok = false;
                    break;
                }
                have_prev = true;
            }
        }
        if (ok && have_prev) issue_pv(g - 1);
        if (lane == 0) {
            // all MMAs of this CTA complete before TMEM is released
            tc::mma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, kDrainTimeoutNs);
        }
        __syncwarp();
    } else {
        // ===================== softmax / accumulate (warps 2..5) =====================
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // token row of S, head-dim row of O^T
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        ItemWalker walk;
        uint32_t g = 0;
        uint32_t items_with_tiles = 0;
        bool ok = true;
        bool flagged_len = false;

        for (int64_t r = blockIdx.x; ok; r += gridDim.x) {
            int y, part;
            if (!walk.seek(p, r, y, part)) break;
            if (!flagged_len && warp == 2 && lane == 0) {
                const int raw = p.context_lens[walk.seq];
                if (raw < 0 || raw > p.len_cap) {
                    raise_flag(p.status, PKV_DEVERR_CONTEXT_LEN);
                    flagged_len = true;
                }
            }
            const int tok0 = part * p.partition_size;
            const int ntok = max(0, min(walk.len, tok0 + p.partition_size) - tok0);
            const int nparts = walk.nparts;
            const int kvh = y / p.subgroups;
            const int hq0 = kvh * p.group + (y % p.subgroups) * GH;
            float m[GH], lp[GH], o[GH], alpha_prev[GH];
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                m[h] = -INFINITY;
                lp[h] = 0.f;
                o[h] = 0.f;
                alpha_prev[h] = 0.f;
            }

            auto accumulate = [&](uint32_t t) -> bool {
                const int b = t & 1;
                if (!tc_wait(&o_full[b], (t >> 1) & 1, abort_flag, p.status)) return false;
                tc::fence_after_sync();
                float pv[GH];
                tc::tmem_ld<GH>(lane_base + 32 + 16 * b, pv);
                tc::tmem_ld_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&o_empty[b]);
#pragma unroll
                for (int h = 0; h < GH; ++h) o[h] = fmaf(o[h], alpha_prev[h], pv[h]);
                return true;
            };

            if (ntok > 0) ++items_with_tiles;
            bool have_prev = false;
            for (int t0 = 0; t0 < ntok; t0 += TILE, ++g) {
                const int tile_ntok = min(TILE, ntok - t0);
                const int b = g & 1;
                if (!tc_wait(&s_full[b], (g >> 1) & 1, abort_flag, p.status)) {
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
                if (!tc_wait(&max_bar[g & 1], (g >> 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                float alpha[GH];
                unsigned char *panel = sm + L::kOffP + b * L::kPanelBytes;
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const float tmax = fmaxf(fmaxf(red[h], red[16 + h]), fmaxf(red[32 + h], red[48 + h]));
                    const float m_new = fmaxf(m[h], tmax);
                    alpha[h] = fast_exp2(m[h] - m_new);  // 0 on the first tile (m = -inf)
                    m[h] = m_new;
                    const float pf = valid ? fast_exp2(sv[h] - m_new) : 0.f;
                    const T p16 = Elem<T>::from_f32(pf);
                    lp[h] = fmaf(lp[h], alpha[h], static_cast<float>(p16));
                    const uint32_t off = ((row >> 6) * 2 + (h >> 3)) * 1024 + tc::sw128_offset(h & 7, row & 63);
                    *reinterpret_cast<T *>(panel + off) = p16;
                }
                if (tile_ntok < TILE) {
                    // rows past the context: zero their V so 0 * stale never reaches the MMA
                    const int s = g % 3;
                    if (!tc_wait(&full[s], (g / 3) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    if (!valid) {
                        unsigned char *vrow = sm + s * L::kStageBytes + L::kKVBytes + row * 128;
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
                if (have_prev && !accumulate(g - 1)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int h = 0; h < GH; ++h) alpha_prev[h] = alpha[h];
                have_prev = true;
            }
            if (!ok) break;
            if (have_prev && !accumulate(g - 1)) {
                ok = false;
                break;
            }
            // l = sum over the 128 token rows of the per-row partial sums
            if (ntok > 0) {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    float v = lp[h];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    lp[h] = v;
                }
                if (lane == 0) {
#pragma unroll
                    for (int h = 0; h < GH; ++h) red_l[quarter * 16 + h] = lp[h];
                    mbar_arrive(lsum_bar);
                }
                if (!tc_wait(lsum_bar, (items_with_tiles - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int h = 0; h < GH; ++h) lp[h] = red_l[h] + red_l[16 + h] + red_l[32 + h] + red_l[48 + h];
            }
            // ---- write this item's result (row = head-dim index)
            const int64_t qrow0 = static_cast<int64_t>(walk.seq) * p.num_q_heads + hq0;
            if (nparts == 1) {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const float res = lp[h] > 0.f ? o[h] / lp[h] : 0.f;
                    static_cast<T *>(p.out)[(qrow0 + h) * D + row] = Elem<T>::from_f32(res);
                }
            } else {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const int64_t pr = (qrow0 + h) * p.num_partitions + part;
                    p.ws_o[pr * D + row] = o[h];
                    if (row == 0) {
                        p.ws_m[pr] = m[h];
                        p.ws_l[pr] = lp[h];
                    }
                }
            }
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
