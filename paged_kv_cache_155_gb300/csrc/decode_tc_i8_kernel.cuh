// decode_tc_i8_kernel.cuh -- paged decode attention over an INT8 cache on the
// tensor cores, for grouped-query attention with head_dim 128 and 4, 8 or 16
// query heads per KV head.
//
// Same result as paged_decode_kernel<T, int8_t, ...>: the INT8 cache of "KV
// Cache从原理到实战" §5.2 with per-channel scales (value = code * scale[h][c]),
// attended with the definition of "KV Cache与PagedAttention深度解析" §2.1 through
// the block tables of §4.2-4.3 and the running max / running sum of §7.2.
//
// With G >= 4 heads per KV head the CUDA cores would spend G FMAs per code;
// here the products run as tcgen05 MMAs (kind::f16, fp32 accumulate, M = 128,
// N = 16) exactly as in paged_decode_tc_kernel, on 16-bit copies of the codes:
//   * codes in [-127, 127] are exact in fp16, so converter warps widen each
//     staged INT8 tile into the 128-byte-swizzled fp16 layout the MMA reads;
//   * the per-channel K scale is folded into the query: q'[h][c] = q[h][c] *
//     k_scale[c] * 2^-e_h, rounded once to fp16, where 2^e_h (a power of two,
//     so the scaling is exact) brings the row's largest |q * k_scale| into
//     [1/2, 1) -- any fp32-representable query fits fp16 this way;
//     s = (q' . code) * 2^e_h * scale;
//   * P is rounded to fp16 for the second MMA (p <= 1), O^T = codes^T . P^T,
//     and the V scale multiplies each output channel once at the end.
//
// Warps (352 threads, one persistent CTA per SM):
//   0 / 6  K / V producers: 1-D bulk copies of each block's code rows
//          (block_size x 128 bytes per head) into INT8 staging rings;
//   1      TMEM owner and MMA issuer (event-driven, PV first), writes the
//          scaled fp16 query panels and each item's score scales;
//   2-5    softmax and accumulation (as paged_decode_tc_kernel);
//   7-8    K converters, 9-10 V converters: staged codes -> fp16 ring slots.
// K and V move through separate producers, staging rings and converters, so
// a V slot still waiting for its PV never holds back the next tile's K.
// Every wait is bounded; a timeout raises PKV_DEVERR_TIMEOUT and all roles stop.
#pragma once

#include "decode_tc_kernel.cuh"

namespace pkv {

struct TcI8Layout {
    static constexpr int kTile = 128, kD = 128, kN = 16;
    static constexpr int kStageK = 2, kStageV = 2;       // INT8 staging slots
    static constexpr int kKStages = 2, kVStages = 2;     // fp16 ring slots
    static constexpr int kStageBytes = 128 * 128;        // 128 tokens x 128 codes
    static constexpr int kHalfBytes = 128 * 128;         // 128 rows x 64 fp16
    static constexpr int kKVBytes = 2 * kHalfBytes;      // fp16 K (or V) tile
    static constexpr int kPanelBytes = 4096;             // 16 x 128 fp16 (Q or P)
    static constexpr int kQsRing = 4;                    // per-item score scales in flight
    static constexpr int kOffSK = 0;
    static constexpr int kOffSV = kOffSK + kStageK * kStageBytes;
    static constexpr int kOffK = kOffSV + kStageV * kStageBytes;
    static constexpr int kOffV = kOffK + kKStages * kKVBytes;
    static constexpr int kOffQ = kOffV + kVStages * kKVBytes;
    static constexpr int kOffP = kOffQ + 2 * kPanelBytes;
    static constexpr int kOffRed = kOffP + 2 * kPanelBytes;          // float [2][4][16] + [4][16]
    static constexpr int kOffQs = kOffRed + 3 * 4 * 16 * 4;          // float [kQsRing][16]
    static constexpr int kOffBar = kOffQs + kQsRing * 16 * 4;
    static constexpr int kNumBars = 2 * kStageK + 2 * kStageV + 2 * kKStages + 2 * kVStages + 13 +
                                    kQsRing + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kMaxStagedSeqs = 1024;
    static constexpr int kOffLens = kOffMisc + 16;
    static constexpr int kBytes = kOffLens + 4 * kMaxStagedSeqs;
    static constexpr int kSmemBytes = kBytes + 1024;
    static constexpr uint32_t kTmemCols = 64;  // S[2] at 0/16, O[2] at 32/48
    static constexpr int kThreads = 352;
    static_assert(kSmemBytes <= 232448, "dynamic shared memory per block");
};

template <typename T, int BS, int GH>
__global__ void __launch_bounds__(352, 1) paged_decode_tc_i8_kernel(const DecodeParams p) {
    using L = TcI8Layout;
    constexpr int TILE = L::kTile, D = L::kD;
    constexpr int BLOCKS_PER_TILE = TILE / BS;
    constexpr int STK = L::kStageK, STV = L::kStageV, KS = L::kKStages, VS = L::kVStages;
    static_assert(GH == 4 || GH == 8 || GH == 16, "tensor-core path serves 4, 8 or 16 heads");
    static_assert(BLOCKS_PER_TILE <= 32, "one table entry per producer lane");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm =
        smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
    uint64_t *sk_full = bars;             // [STK] codes of K landed -> K converters
    uint64_t *sk_empty = sk_full + STK;   // [STK] K codes converted -> K producer
    uint64_t *sv_full = sk_empty + STK;   // [STV]
    uint64_t *sv_empty = sv_full + STV;   // [STV]
    uint64_t *k_full = sv_empty + STV;    // [KS] fp16 K tile written -> MMA
    uint64_t *k_empty = k_full + KS;      // [KS] QK^T done -> converters
    uint64_t *v_full = k_empty + KS;      // [VS]
    uint64_t *v_empty = v_full + VS;      // [VS] PV done -> converters
    uint64_t *s_full = v_empty + VS;      // [2] QK done -> softmax
    uint64_t *s_empty = s_full + 2;       // [2] S read -> MMA
    uint64_t *p_full = s_full + 4;        // [2] P written -> MMA
    uint64_t *o_full = s_full + 6;        // [2] PV done -> softmax
    uint64_t *o_empty = s_full + 8;       // [2] O read -> MMA
    uint64_t *max_bar = s_full + 10;      // [2] softmax tile-max exchange
    uint64_t *lsum_bar = s_full + 12;     // softmax l exchange
    uint64_t *qs_bar = s_full + 13;       // [kQsRing] an item's score scales written
    uint64_t *drain_bar = qs_bar + L::kQsRing;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::kOffMisc + 4);
    float *red_max = reinterpret_cast<float *>(sm + L::kOffRed);  // [2][4][16]
    float *red_l = red_max + 2 * 4 * 16;                             // [4][16]
    float *qs_ring = reinterpret_cast<float *>(sm + L::kOffQs);     // [kQsRing][16]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t smem_base = static_cast<uint32_t>(__cvta_generic_to_shared(sm));

    // ---- set-up: zero the Q / P panels (padding rows stay zero), barriers, TMEM
    for (int i = threadIdx.x; i < 4 * L::kPanelBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(sm + L::kOffQ)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STK; ++s) {
            mbar_init(&sk_full[s], 1);
            mbar_init(&sk_empty[s], 2);  // the two K converter warps
        }
        for (int s = 0; s < STV; ++s) {
            mbar_init(&sv_full[s], 1);
            mbar_init(&sv_empty[s], 2);
        }
        for (int s = 0; s < KS; ++s) {
            mbar_init(&k_full[s], 2);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < VS; ++s) {
            mbar_init(&v_full[s], 2);
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
        for (int i = 0; i < L::kQsRing; ++i) mbar_init(&qs_bar[i], 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::kTmemCols);
        tc::tmem_relinquish();
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
        // ===================== producers: INT8 code rows -> staging (K: warp 0, V: warp 6)
        const int kv = warp == 6;
        const int nst = kv ? STV : STK;
        const uint64_t policy = l2_policy_evict_first();
        const int8_t *base = static_cast<const int8_t *>(kv ? p.v_cache : p.k_cache);
        uint64_t *full = kv ? sv_full : sk_full;
        uint64_t *empty = kv ? sv_empty : sk_empty;
        unsigned char *stage0 = sm + (kv ? L::kOffSV : L::kOffSK);
        ItemWalker walk;
        uint32_t g = 0;  // global tile counter
        int last_issue[3] = {-1, -1, -1};
        static_assert(L::kStageK <= 3 && L::kStageV <= 3, "drain bookkeeping");
        bool ok = true;
        for (int64_t r = blockIdx.x; ok; r += gridDim.x) {
            int y, part;
            if (!walk.seek(p, s_len, r, y, part)) break;
            const int tok0 = p.tok_begin + part * p.partition_size;
            const int ntok = max(0, min(walk.len, tok0 + p.partition_size) - tok0);
            const int kvh = y / p.subgroups;
            const int32_t *trow = p.block_tables + static_cast<int64_t>(walk.seq) * p.max_blocks_per_seq;
            for (int t0 = 0; t0 < ntok && ok; t0 += TILE, ++g) {
                const int nblk = (min(TILE, ntok - t0) + BS - 1) / BS;
                const int blk0 = (tok0 + t0) / BS;
                int e = -1;
                if (lane < nblk) {
                    e = trow[blk0 + lane];
                    if (e < 0 || e >= p.num_blocks) {
                        raise_flag(p.status, PKV_DEVERR_BLOCK_TABLE);
                        e = -1;
                    }
                }
                const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, e >= 0)) * BS * 128u;
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
                if (e >= 0)
                    bulk_copy_g2s(stage0 + s * L::kStageBytes + lane * BS * D,
                                  base + static_cast<int64_t>(e) * p.block_stride +
                                      static_cast<int64_t>(kvh) * BS * D,
                                  BS * D, &full[s], policy);
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            for (int s = 0; s < nst; ++s)
                if (last_issue[s] >= 0)
                    mbar_wait_bounded(&full[s], (last_issue[s] / nst) & 1, kDrainTimeoutNs);
        }
    } else if (warp >= 7) {
        // ===================== converters: staged codes -> fp16 ring slots =====================
        // K: warps 7-8, V: warps 9-10.  Thread c (0..63) widens 16-code groups
        // c, c + 64, ...: row = idx / 8 (token), columns 16 * (idx % 8) .. + 15,
        // written as two swizzled 16-byte chunks.
        const int kv = warp >= 9;
        const int c = threadIdx.x - (kv ? 288 : 224);
        const int nsg = kv ? STV : STK;   // staging slots
        const int nst = kv ? VS : KS;     // ring slots
        uint64_t *sfull0 = kv ? sv_full : sk_full;
        uint64_t *sempty0 = kv ? sv_empty : sk_empty;
        uint64_t *rfull0 = kv ? v_full : k_full;
        uint64_t *rempty0 = kv ? v_empty : k_empty;
        const unsigned char *src0 = sm + (kv ? L::kOffSV : L::kOffSK);
        unsigned char *dst0 = sm + (kv ? L::kOffV : L::kOffK);
        ItemWalker walk;
        uint32_t g = 0;
        bool ok = true;
        for (int64_t r = blockIdx.x; ok; r += gridDim.x) {
            int y, part;
            if (!walk.seek(p, s_len, r, y, part)) break;
            const int tok0 = p.tok_begin + part * p.partition_size;
            const int ntok = max(0, min(walk.len, tok0 + p.partition_size) - tok0);
            for (int t0 = 0; t0 < ntok; t0 += TILE, ++g) {
                const int s = g % nsg, slot = g % nst;
                if (!tc_wait_warp(&sfull0[s], (g / nsg) & 1, abort_flag, p.status) ||
                    !tc_wait_warp(&rempty0[slot], ((g / nst) & 1) ^ 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const unsigned char *src = src0 + s * L::kStageBytes;
                unsigned char *dst = dst0 + slot * L::kKVBytes;
#pragma unroll 4
                for (int i = 0; i < 16; ++i) {
                    const int idx = c + 64 * i;
                    const int row = idx >> 3, grp = idx & 7;
                    const uint4 w = *reinterpret_cast<const uint4 *>(src + row * 128 + grp * 16);
                    uint4 a, b;
                    codes_to_f16x4(w.x, a.x, a.y);
                    codes_to_f16x4(w.y, a.z, a.w);
                    codes_to_f16x4(w.z, b.x, b.y);
                    codes_to_f16x4(w.w, b.z, b.w);
                    // columns 16*grp .. +15 -> half grp / 4, 8-column chunks 2*(grp%4), +1
                    unsigned char *half = dst + (grp >> 2) * L::kHalfBytes + row * 128;
                    const int ch = (grp & 3) * 2;
                    *reinterpret_cast<uint4 *>(half + ((ch ^ (row & 7)) << 4)) = a;
                    *reinterpret_cast<uint4 *>(half + (((ch + 1) ^ (row & 7)) << 4)) = b;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&rfull0[slot]);
                    mbar_arrive(&sempty0[s]);
                }
            }
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        // Event-driven: lane 0 polls the barriers and issues whichever MMA is
        // ready, PV first (it frees a V slot), else the next tile's QK^T.  A
        // fixed order would make PV of one tile wait for the next tile's K.
        constexpr uint32_t idesc_qk = tc::idesc_f16_f32acc(false, 128, L::kN, false, false);
        constexpr uint32_t idesc_pv = tc::idesc_f16_f32acc(false, 128, L::kN, true, false);
        // Queries of the next item that has tiles, prepared in registers one item
        // ahead: q * k_scale per channel, the row's power-of-two exponent e (the 16
        // lanes of a head reduce its largest magnitude), and q * k_scale * 2^-e
        // rounded to fp16.
        constexpr int QCHUNKS = (GH * 16 + 31) / 32;  // 16-byte chunks per lane
        ItemWalker ahead;
        int64_t r_ahead = blockIdx.x;
        uint4 qreg[QCHUNKS];
        int qexp[QCHUNKS];
        auto load_next_q = [&]() {
            int ya, pa;
            while (ahead.seek(p, s_len, r_ahead, ya, pa)) {
                r_ahead += gridDim.x;
                const int t0a = p.tok_begin + pa * p.partition_size;
                if (min(ahead.len, t0a + p.partition_size) - t0a <= 0) continue;
                const int kvha = ya / p.subgroups;
                const int hqa = kvha * p.group + (ya % p.subgroups) * GH;
                const T *qsrc = static_cast<const T *>(p.q) +
                                (static_cast<int64_t>(ahead.seq) * p.num_q_heads + hqa) * D;
#pragma unroll
                for (int c = 0; c < QCHUNKS; ++c) {
                    const int i = lane + c * 32;  // GH * 16 is a multiple of 32
                    const uint4 u = *reinterpret_cast<const uint4 *>(qsrc + (i >> 4) * D + (i & 15) * 8);
                    const float4 *ks = reinterpret_cast<const float4 *>(p.k_scale + kvha * D + (i & 15) * 8);
                    const float4 k0 = ks[0], k1 = ks[1];
                    float f[8];
                    Elem<T>::to_f32x8(u, f);
                    f[0] *= k0.x; f[1] *= k0.y; f[2] *= k0.z; f[3] *= k0.w;
                    f[4] *= k1.x; f[5] *= k1.y; f[6] *= k1.z; f[7] *= k1.w;
                    float mx = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(f[j]));
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    const int e = row_exponent(mx);
                    const float down = exp2_int(-e);
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const __half2 h2 = __floats2half2_rn(f[2 * j] * down, f[2 * j + 1] * down);
                        w[j] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                    qreg[c] = make_uint4(w[0], w[1], w[2], w[3]);
                    qexp[c] = e;
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
        uint32_t n_qk = 0, n_pv = 0;  // tiles whose QK^T / PV have been issued
        uint32_t items = 0;           // items whose queries went to a panel
        bool ok = true;
        uint64_t idle_since = 0;
        while (ok && (have_tile || n_pv < n_qk)) {
            int act = 0;  // 1 = PV, 2 = QK
            if (lane == 0) {
                if (n_pv < n_qk && mbar_test_wait(&p_full[n_pv & 1], (n_pv >> 1) & 1) &&
                    mbar_test_wait(&o_empty[n_pv & 1], ((n_pv >> 1) & 1) ^ 1) &&
                    mbar_test_wait(&v_full[n_pv % VS], (n_pv / VS) & 1))
                    act = 1;
                else if (have_tile && mbar_test_wait(&k_full[n_qk % KS], (n_qk / KS) & 1) &&
                         mbar_test_wait(&s_empty[n_qk & 1], ((n_qk >> 1) & 1) ^ 1))
                    act = 2;
                if (act) {
                    idle_since = 0;
                } else {
                    const uint64_t now = global_timer_ns();
                    if (!idle_since) idle_since = now;
                    if (*abort_flag) {
                        act = -1;
                    } else if (now - idle_since > kWaitTimeoutNs) {
                        raise_flag(p.status, PKV_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                        act = -1;
                    }
                }
            }
            act = __shfl_sync(0xffffffffu, act, 0);
            if (act < 0) {
                ok = false;
                break;
            }
            if (act == 1) {
                if (lane == 0) {
                    const uint32_t t = n_pv;
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
                ++n_pv;
            } else if (act == 2) {
                const int qb = (items - (t0 == 0 ? 0 : 1)) & 1;  // panel of this tile's item
                if (t0 == 0) {
                    // this item's queries -> Q panel qb (K-major, 128-byte swizzle).  The
                    // QK^T that last read this panel (two items back) has completed: the
                    // s_empty wait above showed S of tile n_qk-2 was consumed.
                    unsigned char *panel = sm + L::kOffQ + qb * L::kPanelBytes;
                    const int qslot = items % L::kQsRing;
#pragma unroll
                    for (int c = 0; c < QCHUNKS; ++c) {
                        const int i = lane + c * 32;
                        const int row = i >> 4, c8 = i & 15;
                        const uint32_t off = ((c8 >> 3) * 2 + (row >> 3)) * 1024 + (row & 7) * 128 +
                                             (((c8 & 7) ^ (row & 7)) << 4);
                        *reinterpret_cast<uint4 *>(panel + off) = qreg[c];
                        if (c8 == 0) qs_ring[qslot * 16 + row] = exp2_int(qexp[c]) * p.scale_log2;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    // the softmax of this item reads its score scales after this arrive;
                    // slot qslot was last read kQsRing items ago, before S of this
                    // item's first tile could be issued
                    if (lane == 0) mbar_arrive(&qs_bar[qslot]);
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
        }
        if (lane == 0) {
            // all MMAs of this CTA complete before TMEM is released
            tc::mma_commit(drain_bar);
            mbar_wait_bounded(drain_bar, 0, kDrainTimeoutNs);
        }
        __syncwarp();
    } else {
        // ===================== softmax / accumulate (warps 2..5) =====================
        // (scores scaled per head by the item's 2^e_h * scale * log2(e); P in fp16)
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
            float vs;       // V scale of this thread's output channel
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
        uint32_t nitem = 0;  // items with tiles, in the MMA warp's panel order
        float qsc[GH];
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
                    const float res = it.lp[h] > 0.f ? it.o[h] * it.vs / it.lp[h] : 0.f;
                    static_cast<T *>(p.out)[(it.qrow0 + h) * D + row] = Elem<T>::from_f32(res);
                }
            } else {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const int64_t pr = (it.qrow0 + h) * p.num_partitions + p.slot_base + it.part;
                    p.ws_o[pr * D + row] = it.o[h] * it.vs;
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
            cur.vs = p.v_scale[kvh * D + row];
            {   // this item's score scales 2^e_h * scale * log2(e)
                const int qslot = nitem % L::kQsRing;
                if (!tc_wait_warp(&qs_bar[qslot], (nitem / L::kQsRing) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int h = 0; h < GH; ++h) qsc[h] = qs_ring[qslot * 16 + h];
                ++nitem;
            }
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
                    sv[h] = valid ? sv[h] * qsc[h] : -INFINITY;
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
                    const __half p16 = __float2half_rn(pf);
                    cur.lp[h] = fmaf(cur.lp[h], alpha[h], __half2float(p16));
                    const uint32_t off = ((row >> 6) * 2 + (h >> 3)) * 1024 + tc::sw128_offset(h & 7, row & 63);
                    *reinterpret_cast<__half *>(panel + off) = p16;
                }
                // (V rows past the context need no zeroing: widened codes are finite)
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
