// decode_kernel.cuh -- paged decode attention, one CTA per
// (partition of the context, KV head [x query-head subgroup], sequence).
//
// What it computes ("KV Cache与PagedAttention深度解析" §2.1 definition, §4.2-4.3
// block-table addressing, §7.2 running-max / running-sum form): for every query
// head hq of the CTA's group, over the partition's tokens t,
//     s_t = scale * q[hq] . K[t],   m = max s_t,   l = sum exp(s_t - m),
//     o = sum exp(s_t - m) V[t]
// in fp32.  A sequence that fits in one partition gets out = o / l directly;
// otherwise (o, m, l) go to the workspace and the merge kernel combines the
// partitions.  Scores are kept in log2 units (q is pre-multiplied by
// scale * log2(e)) so every exponential is one ex2.
//
// GB300 design:
//  * K/V are read in place from the paged pool ("gather then compute" would
//    cost an extra pass over HBM): the per-(block, head) K and V tiles are
//    contiguous, so each warp streams them with 1-D bulk copies on the TMA
//    engine into its own ring of shared-memory stages, tracked by one
//    mbarrier per stage.  Each warp is its own producer and consumer: no
//    CTA-wide barrier in the main loop.  Tiles are marked evict-first in L2.
//  * Lane layout: a token row of head_dim 16-bit values is LPT = head_dim/8
//    lanes x one 16-byte vector (INT8: head_dim/16 lanes x 16 codes for one or
//    two heads per block, else head_dim/8 lanes x 8 codes), so TPG = 32/LPT
//    tokens are in flight per warp instruction and shared-memory reads are
//    conflict-free.  The QK partial
//    sums are reduced across the LPT lanes with xor shuffles; the PV update is
//    lane-local (each lane owns 8 output dims of every head of the group).
//  * GQA: all GH query heads of the group share each K/V tile, so a tile is
//    read from HBM once per group, not once per query head.
//  * The chunk-to-warp assignment and every merge are fixed by logical token
//    position, so the output does not depend on the physical placement.
//  * INT8 cache ("KV Cache从原理到实战" §5.2, per-channel scales): the storage
//    type KT is int8_t.  The per-channel K scale is folded into the query once
//    (s_t = sum_j (q_j k_scale_j) code_j) and the V scale multiplies each output
//    channel once at the end, so the inner loop reads only codes.  It runs on
//    fp16 operands with fp32 sums: the folded query is rounded once to fp16
//    after a per-head power-of-two scaling (its largest magnitude in [1/2, 1)),
//    a byte permute turns two codes into the exact fp16 values code + 1152,
//    and mixed-precision FMAs (fp16 x fp16 + fp32) accumulate.  The offset
//    leaves known sums: a dot product starts from -1152 times the lane's query
//    sum, and the output removes 1152 times the weight sum, whose terms are the
//    weights rounded to fp16 exactly as they meet V.
//  * 4, 8 or 16 query heads per block (grouped-query attention): the lane loops
//    would spend GH FMAs per cache element, so both products run as warp-level
//    MMAs (m16n8k16, fp32 accumulators) on register fragments, 16 tokens per
//    step, and each warp still streams its own ring with no hand-off to other
//    warps.  The k indices of QK^T are mapped to channels so that a lane's
//    16-byte vector of a token row holds whole k pairs.
//    - 16-bit cache: S = Q K^T with the heads as the 16 rows (rows past GH are
//      zero; with 16 heads a lane holds heads g and g + 8) and the tokens as
//      columns; the K words go straight in as the B fragment, and the S
//      accumulators of a row are the A fragment of P V after the softmax.  V's
//      B fragment pairs two tokens of one channel with one byte permute.
//    - INT8 cache: S^T = K Q^T with the tokens as rows and the heads as
//      columns, on the fp16 values code + 1152 widened in registers (one byte
//      permute per pair); P moves into the B layout of O^T = (V + 1152)^T P^T
//      by two 8 x 8 transposes, and V's A fragment pairs two tokens of a
//      channel with a byte permute and one three-input logic op.  No padded
//      head rows: half the MMAs and accumulators, so four CTAs fit an SM.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_tc.cuh"

namespace pkv {

struct DecodeParams {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    void *out;
    float *ws_o;  // [num_seqs][num_q_heads][num_partitions][head_dim]
    float *ws_m;  // [num_seqs][num_q_heads][num_partitions] (log2 units)
    float *ws_l;  // [num_seqs][num_q_heads][num_partitions]
    const float *k_scale;  // INT8 cache: [num_kv_heads][head_dim] per-channel scales
    const float *v_scale;
    const int32_t *block_tables;
    const int32_t *context_lens;
    unsigned int *status;
    int64_t num_blocks;
    int64_t block_stride;  // elements between consecutive physical blocks
    int max_blocks_per_seq;
    int len_cap;     // min(max_context_len, max_blocks_per_seq * block_size)
    int num_seqs;
    int num_q_heads;
    int items_y;     // num_kv_heads * subgroups (work items per sequence partition)
    int group;       // num_q_heads / num_kv_heads
    int subgroups;   // group / heads_per_block
    int partition_size;
    int num_partitions;  // workspace partition slots per (sequence, query head)
    float scale_log2;    // scale * log2(e)
    // Token range and workspace slots of this launch: attention runs over tokens
    // [tok_begin, context_len) split into partitions of partition_size, whose
    // partials go to slots slot_base + partition.  always_partial keeps even a
    // single-partition result in the workspace for a later merge.  The plain
    // decode uses 0 / 0 / 0; the shared-prefix decode runs the suffix with
    // tok_begin = prefix length and slot_base = number of prefix splits.
    int tok_begin;
    int slot_base;
    int always_partial;
    // Set when this launch overlaps the kernel before it in the stream
    // (programmatic dependent launch, the shared-prefix decode): the CTA with the
    // last block index waits for that kernel before it exits, so this grid -- and
    // whatever the stream runs after it -- completes only after that kernel.
    int wait_prior_grid;
    // Set when the library's merge kernel follows as a programmatic dependent: the
    // CTAs signal at their start that it may be placed.  Without it the next kernel
    // of the stream starts only when this grid has completed.
    int trigger_dependents;
};

// Tensor maps of the two pool halves for the forms that stage by tiled TMA
// copies (zero-filled otherwise).
struct DecodeMaps {
    CUtensorMap k;
    CUtensorMap v;
};

// Partitions of a sequence of `len` tokens in a launch (at least one, possibly empty).
__device__ __forceinline__ int partitions_of(const DecodeParams &p, int len) {
    const int span = len - p.tok_begin;
    return span > 0 ? (span + p.partition_size - 1) / p.partition_size : 1;
}

// Values per lane vector of the CUDA-core kernel (see DecodeGeom).
template <typename KT, int GH>
__host__ __device__ constexpr int decode_lane_values() {
    return (sizeof(KT) == 1 && GH <= 2) ? 16 : 8;
}

// One lane's VL consecutive cache values of a row in shared memory -> fp32.
template <typename KT, int VL>
__device__ __forceinline__ void load_lane(const KT *src, float *f) {
    if constexpr (sizeof(KT) == 2) {
        static_assert(VL == 8, "16-bit caches use 8 values per lane");
        Elem<KT>::to_f32x8(*reinterpret_cast<const uint4 *>(src), f);
    } else if constexpr (VL == 8) {
        Elem<KT>::to_f32x8(*reinterpret_cast<const uint2 *>(src), f);
    } else {
        const uint4 u = *reinterpret_cast<const uint4 *>(src);
        Elem<KT>::to_f32x8(make_uint2(u.x, u.y), f);
        Elem<KT>::to_f32x8(make_uint2(u.z, u.w), f + 8);
    }
}

// One lane's VL consecutive INT8 codes of a row in shared memory -> VL / 2
// words of two exact fp16 values code + kCodeOffset each (codes 2i and 2i + 1
// in word i).
template <int VL>
__device__ __forceinline__ void load_codes_f16(const int8_t *src, uint32_t *h) {
    if constexpr (VL == 8) {
        const uint2 u = *reinterpret_cast<const uint2 *>(src);
        codes_to_f16x4_offset(u.x, h[0], h[1]);
        codes_to_f16x4_offset(u.y, h[2], h[3]);
    } else {
        static_assert(VL == 16, "8 or 16 codes per lane");
        const uint4 u = *reinterpret_cast<const uint4 *>(src);
        codes_to_f16x4_offset(u.x, h[0], h[1]);
        codes_to_f16x4_offset(u.y, h[2], h[3]);
        codes_to_f16x4_offset(u.z, h[4], h[5]);
        codes_to_f16x4_offset(u.w, h[6], h[7]);
    }
}

// Decode-kernel geometry for one (head_dim, block_size, cache element bytes,
// values per lane vector).  16-bit caches use 8 values (16 bytes) per lane;
// the INT8 cache uses 16 codes (16 bytes) per lane when a block serves at most
// two query heads (fewer lanes per token row: shorter shuffle reductions and
// fewer per-row steps per byte), else 8 codes (register budget).  The stage
// budget per warp sets how many CTAs share an SM: INT8 lane loops 8 KiB (six at
// 80 registers), INT8 warp MMAs 12 KiB (four), 16-bit lane loops 24 KiB (two),
// 16-bit warp MMAs 16 KiB (three), and 24 KiB for sixteen heads per block, whose
// registers allow two CTAs per SM (a CTA's bytes in flight bound its rate).
template <int D, int BS, int EB = 2, int VL = 8, bool kMmaForm = false, bool kWide = false>
struct DecodeGeom {
    static constexpr int kWarps = 4;
    static constexpr int kMaxTile = 32 / EB;             // 4 KiB K tiles at head_dim 128
    static constexpr int kTile = BS < kMaxTile ? BS : kMaxTile;  // tokens per stage
    static constexpr int kVec = VL;                      // values per lane vector
    static constexpr int kLanesPerToken = D / kVec;      // LPT
    static constexpr int kTokenGroups = 32 / kLanesPerToken;  // TPG
    static constexpr int kIters = kTile / kTokenGroups;  // token rows per lane per stage
    static constexpr int kTileBytes = kTile * D * EB;    // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kBudget = EB == 1 ? (kMmaForm ? 12288 : 8192) : (kMmaForm && !kWide ? 16384 : 24576);
    static constexpr int kStagesRaw = kBudget / kStageBytes;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kMaxTableEntries = 1024;        // table slice per partition
    // Warp-MMA forms at head_dim 128: K/V tiles arrive by tiled TMA copies with a
    // 128-byte swizzle (16-bit tiles as two 64-channel half panels), whose 8-row
    // atoms need 1024-byte-aligned stages
    static constexpr bool kSwizzled = kMmaForm && D == 128;
    static constexpr int kAlignPad = kSwizzled ? 1024 : 0;
    static constexpr int kSmemBytes = kWarps * kStages * kStageBytes +
                                      kWarps * kStages * 8 + kMaxTableEntries * 4 + kAlignPad;
    static_assert(kIters >= 1, "tile smaller than a warp's token groups");
};

// T: query / output type; KT: cache storage type (T, or int8_t for the INT8 cache).
// tmap_k / tmap_v: tiled tensor maps of the pool halves (box: TILE token rows of
// one head, 128 bytes each -- all 128 INT8 codes, or 64 16-bit values -- with a
// 128-byte swizzle), used by the warp-MMA forms at head_dim 128; the other forms
// ignore them.
template <typename T, typename KT, int D, int BS, int GH>
__global__ void __launch_bounds__(128, (GH >= 4 && sizeof(KT) == 2) ? (GH == 16 ? 2 : 3) : 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                              const __grid_constant__ CUtensorMap tmap_v,
                                                              const DecodeParams p) {
    constexpr bool kQuant = sizeof(KT) == 1;
    // 4, 8 or 16 query heads per block: the products run as warp-level MMAs (the per-lane
    // loops would spend GH FMAs per element), INT8 codes on exact fp16 copies
    constexpr bool kMma = GH >= 4;
    constexpr bool kMmaBF16 = std::is_same<KT, __nv_bfloat16>::value;  // MMA operand type
    constexpr int VL = decode_lane_values<KT, GH>();  // values per lane vector
    using G = DecodeGeom<D, BS, sizeof(KT), VL, (GH >= 4), (GH == 16)>;
    constexpr int NW = G::kWarps, S = G::kStages, TILE = G::kTile, LPT = G::kLanesPerToken,
                  TPG = G::kTokenGroups, ITERS = G::kIters;
    // token rows processed between two online-softmax updates (bounds registers)
    constexpr int IT_STEP = (ITERS * GH <= 32) ? ITERS : (32 / GH > 0 ? 32 / GH : 1);
    static_assert(ITERS % IT_STEP == 0, "step must divide the stage");
    static_assert(GH * (D + 4) * 4 <= S * G::kStageBytes, "merge scratch must fit a warp's stages");

    // the merge kernel, launched behind this one, may be placed as this grid's CTAs run
    if (p.trigger_dependents) pdl_trigger();
    if (p.wait_prior_grid && blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 &&
        blockIdx.z == gridDim.z - 1)
        pdl_wait();  // uniform over the CTA; normally dispatched last, when nothing is left to wait for

    // warp-MMA forms at head_dim 128: stages filled by swizzled tiled TMA copies
    constexpr bool kSwz = G::kSwizzled;
    constexpr int kHalfBytes = TILE * 128;  // 16-bit swizzled tiles: one 64-channel half panel
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_raw;
    if constexpr (kSwz)
        smem += (1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u;
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * S * G::kStageBytes);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + NW * S * G::kStageBytes + NW * S * 8);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int part = blockIdx.x;
    const int seq = blockIdx.z;
    const int kvh = blockIdx.y / p.subgroups;
    const int hq0 = kvh * p.group + (blockIdx.y % p.subgroups) * GH;

    // ---- the partition's first table entries are fetched together with the context
    //      length (where the partition starts does not depend on it), so the first
    //      tile copies wait for one global-memory round trip, not two
    const int tok0 = p.tok_begin + part * p.partition_size;
    const int blk0 = tok0 / BS;
    const int32_t *trow = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq + blk0;
    int first_entry = 0;  // entry threadIdx.x of the slice, if the table has it
    if (static_cast<int>(threadIdx.x) < min(p.max_blocks_per_seq - blk0, p.partition_size / BS))
        first_entry = trow[threadIdx.x];

    // ---- context length (device value, range-checked) and partition bounds
    int len = p.context_lens[seq];
    if (len < 0 || len > p.len_cap) {
        if (threadIdx.x == 0 && part == 0 && blockIdx.y == 0)
            raise_flag(p.status, PKV_DEVERR_CONTEXT_LEN);
        len = len < 0 ? 0 : p.len_cap;
    }
    const int nparts = partitions_of(p, len);
    if (part >= nparts) return;  // uniform over the CTA
    const int tok1 = min(len, tok0 + p.partition_size);
    const int ntok = max(0, tok1 - tok0);
    const int nchunks = (ntok + TILE - 1) / TILE;
    const int nblk = (ntok + BS - 1) / BS;  // <= partition_size / BS, within the table

    // ---- table slice of this partition -> shared memory (bad entries -> -1)
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
        int b = i < static_cast<int>(blockDim.x) ? first_entry : trow[i];
        if (b < 0 || b >= p.num_blocks) {
            raise_flag(p.status, PKV_DEVERR_BLOCK_TABLE);
            b = -1;
        }
        tbl[i] = b;
    }
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[warp * S + s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const KT *kc = static_cast<const KT *>(p.k_cache);
    const KT *vc = static_cast<const KT *>(p.v_cache);
    unsigned char *my_stages = stages + warp * S * G::kStageBytes;
    uint64_t *my_bars = bars + warp * S;
    const uint64_t policy = l2_policy_evict_first();

    // chunk c (partition-local, TILE tokens) -> stage s of this warp
    auto issue = [&](int c, int s) {
        const int row = c * TILE;                   // partition-local token index
        const int b = tbl[row / BS];
        const int r0 = row % BS;
        if (b < 0) {  // flagged entry: complete the phase without data
            mbar_arrive(&my_bars[s]);
            return;
        }
        const int64_t off = static_cast<int64_t>(b) * p.block_stride +
                            (static_cast<int64_t>(kvh) * BS + r0) * D;
        unsigned char *dst = my_stages + s * G::kStageBytes;
        mbar_arrive_expect_tx(&my_bars[s], G::kStageBytes);
        if constexpr (kSwz && kQuant) {
            // token row t of the tile lands as 128 bytes whose 16-byte chunk c sits at
            // chunk c ^ (t & 7)
            tc::tma_load_3d(dst, &tmap_k, 0, kvh * BS + r0, b, &my_bars[s], policy);
            tc::tma_load_3d(dst + G::kTileBytes, &tmap_v, 0, kvh * BS + r0, b, &my_bars[s], policy);
        } else if constexpr (kSwz) {
            // 16-bit: channels 64 c .. 64 c + 63 of token row t land in half panel c
            // as 128 bytes whose 16-byte chunk j sits at chunk j ^ (t & 7)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                tc::tma_load_3d(dst + c * kHalfBytes, &tmap_k, 64 * c, kvh * BS + r0, b, &my_bars[s], policy);
                tc::tma_load_3d(dst + G::kTileBytes + c * kHalfBytes, &tmap_v, 64 * c, kvh * BS + r0, b,
                                &my_bars[s], policy);
            }
        } else {
            bulk_copy_g2s(dst, kc + off, G::kTileBytes, &my_bars[s], policy);
            bulk_copy_g2s(dst + G::kTileBytes, vc + off, G::kTileBytes, &my_bars[s], policy);
        }
    };

    const int my_chunks = nchunks > warp ? (nchunks - warp + NW - 1) / NW : 0;
    if (lane == 0) {
        for (int i = 0; i < S && i < my_chunks; ++i) issue(warp + i * NW, i);
    }

    // ---- per-lane query slice (pre-scaled) and accumulators
    const int sub = lane % LPT;   // which VL dims
    const int grp = lane / LPT;   // which token row of a TPG-row step
    float qf[GH][VL];
    if constexpr (!kMma) {
        const T *qb = static_cast<const T *>(p.q) +
                      (static_cast<int64_t>(seq) * p.num_q_heads + hq0) * D + sub * VL;
#pragma unroll
        for (int g = 0; g < GH; ++g) {
#pragma unroll
            for (int v = 0; v < VL; v += 8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(qb + g * D + v);
                Elem<T>::to_f32x8(u, qf[g] + v);
            }
#pragma unroll
            for (int e = 0; e < VL; ++e) qf[g][e] *= p.scale_log2;
        }
        if constexpr (kQuant) {  // K dequantisation folded into the query
            const float4 *ks = reinterpret_cast<const float4 *>(p.k_scale + kvh * D + sub * VL);
#pragma unroll
            for (int v = 0; v < VL / 4; ++v) {
                const float4 a = ks[v];
#pragma unroll
                for (int g = 0; g < GH; ++g) {
                    qf[g][4 * v] *= a.x;
                    qf[g][4 * v + 1] *= a.y;
                    qf[g][4 * v + 2] *= a.z;
                    qf[g][4 * v + 3] *= a.w;
                }
            }
        }
    }
    // INT8 cache: the query goes to fp16 with one power-of-two exponent per head
    // (its largest magnitude lands in [0.5, 1)), so each code pair meets it in two
    // mixed-precision FMAs (fp16 operands, fp32 sums).  The codes enter as the
    // exact fp16 values code + kCodeOffset; a dot product starts from minus the
    // offset times this lane's query sum, and the value sums shed the offset
    // times the weight sum at the end.
    uint32_t qh[GH][VL / 2];
    float qs[GH];  // 2^exponent: the scale of the fp16 query's dot products
    float qo[GH];  // kCodeOffset * (sum of this lane's fp16 query values)
    if constexpr (kQuant && !kMma) {
#pragma unroll
        for (int g = 0; g < GH; ++g) {
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < VL; ++e) amax = fmaxf(amax, fabsf(qf[g][e]));
#pragma unroll
            for (int o = LPT / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const int qe = row_exponent(amax);
            qs[g] = exp2_int(qe);
            const float down = exp2_int(-qe);
            float qsum = 0.f;
#pragma unroll
            for (int e = 0; e < VL; e += 2) {
                const __half2 h = __floats2half2_rn(qf[g][e] * down, qf[g][e + 1] * down);
                qh[g][e / 2] = *reinterpret_cast<const uint32_t *>(&h);
                qsum += __low2float(h) + __high2float(h);
            }
            qo[g] = kCodeOffset * qsum;
        }
    }
    // Warp-MMA forms (m16n8k16, fp32 accumulators), lane (mg, mt) = (lane / 4, lane % 4),
    // per step of 16 tokens, k of QK^T running over channels in chunks of 16:
    //  - INT8: S^T = K Q^T with the tokens as the 16 rows and the query heads as the 8
    //    columns (columns >= GH zero), then O^T = V^T P^T with channels as rows;
    //  - 16-bit: S = Q K^T with the heads as the 16 rows (rows >= GH zero) and two
    //    8-token column tiles, then O = P V.
    // The k indices of QK^T are mapped to channels so that a lane reads its part of a
    // token row as 16-byte vectors: INT8 k-chunk kc = 4 j + w pairs channels
    // 64 j + 16 t + 4 w + {0, 1} / {2, 3} of lane t with k 2t, 2t+1 / 2t+8, 2t+9; a
    // 16-bit cache packs two channels per word, so chunk kc = 2 j + p takes channels
    // 32 j + 8 t + 4 p + {0, 1} / {2, 3}.  Either way a lane's values run in
    // RUN-channel groups and chunk kc takes its values 4 kc .. 4 kc + 3.  The query of head mg (the B operand of S^T,
    // the A operand of S) sits in lanes (mg, .) with exactly those channels.
    constexpr int KC = D / 16;                   // k-chunks of QK^T
    constexpr int MT = D / 16;                   // INT8: m-tiles of O^T (16 channels each)
    constexpr int NT = D / 8;                    // 16-bit: n-tiles of O (8 channels each)
    constexpr int STEP = TILE < 16 ? TILE : 16;  // tokens per MMA step
    const int mg = lane >> 2, mt = lane & 3;
    uint32_t qa[KC][2];
    // 16-bit warp MMAs with 16 heads per block: a lane also holds head mg + 8, the
    // MMA rows 8..15 that fewer heads leave zero
    constexpr bool kRows16 = kMma && !kQuant && GH == 16;
    uint32_t qb[kRows16 ? KC : 1][2];
    constexpr int RUN = kQuant ? 16 : 8;         // a lane's contiguous channels (16 bytes)
    float mqs = 1.f, mqb = 0.f;  // row mg's score scale 2^e and code-offset bias
    // swizzled INT8 staging reads lane t's K chunks 2 t and 2 t + 1 (conflict-free
    // under the swizzle), so its channels are 2 RUN t + RUN j + (0 .. RUN - 1), j = 0, 1
    constexpr int kLaneStride = kSwz ? 2 * RUN : RUN;  // channel offset of lane t's first vector
    constexpr int kVecStride = kSwz ? RUN : 4 * RUN;   // ... between its vectors j and j + 1
    if constexpr (kMma) {
        const T *qrow = static_cast<const T *>(p.q) +
                        (static_cast<int64_t>(seq) * p.num_q_heads + hq0 + mg) * D + kLaneStride * mt;
        if constexpr (kQuant) {
            // the query times scale * log2(e) and the K scale, then one power-of-two
            // exponent per head (its largest magnitude into [1/2, 1)) before fp16
            float f[D / 4];
#pragma unroll
            for (int e = 0; e < D / 4; ++e) f[e] = 0.f;
            if (mg < GH) {
#pragma unroll
                for (int j = 0; j < D / (4 * RUN); ++j) {
#pragma unroll
                    for (int v = 0; v < RUN; v += 8)
                        Elem<T>::to_f32x8(*reinterpret_cast<const uint4 *>(qrow + kVecStride * j + v), f + RUN * j + v);
                    const float *ksr = p.k_scale + kvh * D + kVecStride * j + kLaneStride * mt;
#pragma unroll
                    for (int v = 0; v < RUN / 4; ++v) {
                        const float4 a = reinterpret_cast<const float4 *>(ksr)[v];
                        f[RUN * j + 4 * v] *= a.x * p.scale_log2;
                        f[RUN * j + 4 * v + 1] *= a.y * p.scale_log2;
                        f[RUN * j + 4 * v + 2] *= a.z * p.scale_log2;
                        f[RUN * j + 4 * v + 3] *= a.w * p.scale_log2;
                    }
                }
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < D / 4; ++e) amax = fmaxf(amax, fabsf(f[e]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int qe = row_exponent(amax);
            const float down = exp2_int(-qe);
            float qsum = 0.f;
#pragma unroll
            for (int kc = 0; kc < KC; ++kc) {
                float r0, r1, r2, r3;
                qa[kc][0] = pack_mma2<false>(f[4 * kc] * down, f[4 * kc + 1] * down, r0, r1);
                qa[kc][1] = pack_mma2<false>(f[4 * kc + 2] * down, f[4 * kc + 3] * down, r2, r3);
                qsum += (r0 + r1) + (r2 + r3);
            }
            qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
            qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
            mqs = exp2_int(qe);
            mqb = mqs * (kCodeOffset * qsum);
        } else {
            // 16-bit cache: the query enters unchanged (the cache's type), the
            // scores take scale * log2(e) in fp32.  Swizzled staging: lane t's vector
            // j holds channels 64 (j / 2) + 16 t + 8 (j % 2) .. + 7, chunk 2 t + j % 2
            // of half panel j / 2, like its K vectors
#pragma unroll
            for (int j = 0; j < D / (4 * RUN); ++j) {
                const int qofs = kSwz ? 64 * (j >> 1) + 8 * (j & 1) : 4 * RUN * j;
                const uint4 u = mg < GH ? *reinterpret_cast<const uint4 *>(qrow + qofs) : make_uint4(0, 0, 0, 0);
                qa[2 * j][0] = u.x;
                qa[2 * j][1] = u.y;
                qa[2 * j + 1][0] = u.z;
                qa[2 * j + 1][1] = u.w;
                if constexpr (kRows16) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(qrow + 8 * D + qofs);  // head mg + 8
                    qb[2 * j][0] = w.x;
                    qb[2 * j][1] = w.y;
                    qb[2 * j + 1][0] = w.z;
                    qb[2 * j + 1][1] = w.w;
                }
            }
            mqs = p.scale_log2;
        }
    }
    // MMA accumulators of O.  INT8 (O^T = (V + 1152)^T P^T, heads as columns): m-tile j
    // holds channels (D / 8) mg + 2 j (d0, d1) and + 1 (d2, d3) of heads 2 mt (d0, d2)
    // and 2 mt + 1 (d1, d3).  16-bit (O = P V, heads as rows): n-tile nt holds head mg
    // (d0, d1; d2, d3 rows 8..15) at channels (D / 8) (2 mt) + nt and (D / 8) (2 mt + 1) + nt.
    float oacc[NT][4];
    float mh[2] = {-INFINITY, -INFINITY}, lh[2] = {0.f, 0.f};  // INT8: heads 2 mt, 2 mt + 1
    float hqs[2] = {1.f, 1.f}, hqb[2] = {0.f, 0.f};            // their score scales / biases
    float mrow = -INFINITY, lrow = 0.f;                        // 16-bit: head mg
    float mrow2 = -INFINITY, lrow2 = 0.f;                      // ... and head mg + 8 (16 heads)
    if constexpr (kMma) {
#pragma unroll
        for (int j = 0; j < NT; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            hqs[e] = __shfl_sync(0xffffffffu, mqs, 4 * (2 * mt + e));
            hqb[e] = __shfl_sync(0xffffffffu, mqb, 4 * (2 * mt + e));
        }
    }
    float acc[GH][VL];
    float m[GH], l[GH];
#pragma unroll
    for (int g = 0; g < GH; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < VL; ++e) acc[g][e] = 0.f;
    }

    bool aborted = false;
    for (int i = 0; i < my_chunks; ++i) {
        const int s = i % S;
        const uint32_t parity = (i / S) & 1;
        const bool ok = mbar_wait_bounded(&my_bars[s], parity, kWaitTimeoutNs);
        if (__any_sync(0xffffffffu, !ok)) {
            // give up: flag it, let this warp's copies still in flight land, stop
            if (lane == 0) {
                raise_flag(p.status, PKV_DEVERR_TIMEOUT);
                for (int k = i; k < my_chunks && k < i + S; ++k)
                    mbar_wait_bounded(&my_bars[k % S], (k / S) & 1, kDrainTimeoutNs);
            }
            __syncwarp();
            aborted = true;
            break;
        }
        const int c = warp + i * NW;
        const int valid = min(TILE, ntok - c * TILE);  // >= 1
        if (tbl[(c * TILE) / BS] >= 0) {
            const KT *ks = reinterpret_cast<const KT *>(my_stages + s * G::kStageBytes);
            const KT *vs = ks + TILE * D;
            if constexpr (kMma && kQuant) {
                // INT8 cache: S^T = K Q^T with the tokens as the 16 rows and the heads as
                // the 8 columns, O^T = (V + 1152)^T P^T with the channels as rows; P moves
                // from the S^T accumulators into the B layout by 8 x 8 transposes.  No
                // padded head rows: half the MMAs and accumulators of the heads-as-rows form.
                const unsigned char *kt = reinterpret_cast<const unsigned char *>(ks);
                const unsigned char *vt = reinterpret_cast<const unsigned char *>(vs);
#pragma unroll
                for (int tb = 0; tb < TILE; tb += STEP) {
                    if (tb >= valid) break;  // warp-uniform: the step holds no context token
                    // S^T for the step: A rows mg and mg + 8 are tokens tb + mg and tb + 8 + mg,
                    // read by lanes (mg, .) as 16-byte vectors; two accumulators (even / odd
                    // k-chunks) halve the MMA chains
                    float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sodd[4] = {0.f, 0.f, 0.f, 0.f};
                    const unsigned char *krow0 = kt + (tb + mg) * D;
                    const unsigned char *krow1 = krow0 + 8 * D;
#pragma unroll
                    for (int j = 0; j < D / (4 * RUN); ++j) {
                        // this lane's vector j of rows tb + mg and tb + 8 + mg (both = mg mod 8)
                        const int kofs = kSwz ? ((((2 * mt + j) ^ mg) & 7) << 4) : RUN * mt + 64 * j;
                        const uint4 u0 = *reinterpret_cast<const uint4 *>(krow0 + kofs);
                        uint4 u1 = make_uint4(0, 0, 0, 0);
                        if constexpr (STEP == 16) u1 = *reinterpret_cast<const uint4 *>(krow1 + kofs);
                        const uint32_t w0[4] = {u0.x, u0.y, u0.z, u0.w};
                        const uint32_t w1[4] = {u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                        for (int w = 0; w < 4; ++w) {  // four codes -> the two k pairs of one chunk
                            uint32_t lo0, hi0, lo1 = 0u, hi1 = 0u;
                            codes_to_f16x4_offset(w0[w], lo0, hi0);
                            if constexpr (STEP == 16) codes_to_f16x4_offset(w1[w], lo1, hi1);
                            mma_16816<false>(w & 1 ? sodd : sacc, lo0, lo1, hi0, hi1, qa[4 * j + w][0],
                                             qa[4 * j + w][1]);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[e] += sodd[e];
                    // scores in log2 units: d0, d1 = token tb + mg, heads 2 mt, 2 mt + 1; d2, d3 =
                    // token tb + 8 + mg; tokens past the context -> -inf
                    float sc[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sc[e] = tb + mg + 8 * (e >> 1) < valid ? fmaf(sacc[e], hqs[e & 1], -hqb[e & 1]) : -INFINITY;
                    // per head, the maximum over the step's tokens (the eight lanes with this
                    // mt hold them): finite, as token tb is in the context
                    float mx[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float v = fmaxf(sc[e], sc[2 + e]);
#pragma unroll
                        for (int o = 4; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                        mx[e] = v;
                    }
                    const bool grow0 = mx[0] > mh[0], grow1 = mx[1] > mh[1];
                    if (__any_sync(0xffffffffu, grow0 || grow1)) {
                        const float a0 = grow0 ? fast_exp2(mh[0] - mx[0]) : 1.f;  // 0 when m = -inf
                        const float a1 = grow1 ? fast_exp2(mh[1] - mx[1]) : 1.f;
                        lh[0] *= a0;
                        lh[1] *= a1;
#pragma unroll
                        for (int j = 0; j < MT; ++j) {
                            oacc[j][0] *= a0;
                            oacc[j][2] *= a0;
                            oacc[j][1] *= a1;
                            oacc[j][3] *= a1;
                        }
                        if (grow0) mh[0] = mx[0];
                        if (grow1) mh[1] = mx[1];
                    }
                    // P^T rounded to the MMA type (the row sums add the rounded values), moved
                    // into the B layout of O^T += V^T P^T (k = tokens, columns = heads) by 8 x 8
                    // transposes
                    float r[4];
                    const uint32_t p0 = pack_mma2<false>(fast_exp2(sc[0] - mh[0]), fast_exp2(sc[1] - mh[1]), r[0], r[1]);
                    const uint32_t p1 = pack_mma2<false>(fast_exp2(sc[2] - mh[0]), fast_exp2(sc[3] - mh[1]), r[2], r[3]);
                    lh[0] += r[0] + r[2];
                    lh[1] += r[1] + r[3];
                    const uint32_t pb0 = movmatrix_trans(p0);
                    const uint32_t pb1 = STEP == 16 ? movmatrix_trans(p1) : 0u;
                    // O^T += (V + 1152)^T P^T: A rows mg / mg + 8 of m-tile j are channels
                    // (D / 8) mg + 2 j / + 1; lane (mg, mt) reads tokens tb + 2 mt, +1 (k 2t, 2t+1)
                    // and tb + 8 + 2 mt, +1 (k 2t+8, 2t+9) at its D / 8 channels and pairs them per
                    // channel (byte permute + lop3, code + 1152)
                    constexpr int VW = D / 32;  // 32-bit words of a lane's channels in a row
                    uint32_t x[STEP / 4][VW];
#pragma unroll
                    for (int rr = 0; rr < STEP / 4; ++rr) {
                        const int vr = tb + 2 * mt + (rr >> 1) * 8 + (rr & 1);  // token row
                        // its D / 8 channels at (D / 8) mg: chunk mg, at chunk mg ^ (row & 7) swizzled
                        const unsigned char *src = vt + vr * D + (kSwz ? (((mg ^ vr) & 7) << 4) : (D / 8) * mg);
                        if constexpr (VW == 4) {
                            const uint4 u = *reinterpret_cast<const uint4 *>(src);
                            x[rr][0] = u.x;
                            x[rr][1] = u.y;
                            x[rr][2] = u.z;
                            x[rr][3] = u.w;
                        } else {
                            const uint2 u = *reinterpret_cast<const uint2 *>(src);
                            x[rr][0] = u.x;
                            x[rr][1] = u.y;
                        }
                    }
#pragma unroll
                    for (int w = 0; w < VW; ++w) {  // channels 4 w + e: m-tile 2 w + e / 2, row half e % 2
                        uint32_t a[4], c[4] = {0u, 0u, 0u, 0u};
                        a[0] = token_pair_f16_offset<0>(x[0][w], x[1][w]);
                        a[1] = token_pair_f16_offset<1>(x[0][w], x[1][w]);
                        a[2] = token_pair_f16_offset<2>(x[0][w], x[1][w]);
                        a[3] = token_pair_f16_offset<3>(x[0][w], x[1][w]);
                        if constexpr (STEP == 16) {
                            c[0] = token_pair_f16_offset<0>(x[2][w], x[3][w]);
                            c[1] = token_pair_f16_offset<1>(x[2][w], x[3][w]);
                            c[2] = token_pair_f16_offset<2>(x[2][w], x[3][w]);
                            c[3] = token_pair_f16_offset<3>(x[2][w], x[3][w]);
                        }
                        mma_16816<false>(oacc[2 * w], a[0], a[1], c[0], c[1], pb0, pb1);
                        mma_16816<false>(oacc[2 * w + 1], a[2], a[3], c[2], c[3], pb0, pb1);
                    }
                }
            } else if constexpr (kMma) {
                // 16-bit cache: S = Q K^T with the heads as the 16 rows (rows >= GH are
                // zero) and two 8-token column tiles; O = P V with P taken straight from
                // the S accumulators (the A fragment of a row is its S fragment)
                const unsigned char *kt = reinterpret_cast<const unsigned char *>(ks);
                const unsigned char *vt = reinterpret_cast<const unsigned char *>(vs);
#pragma unroll
                for (int tb = 0; tb < TILE; tb += STEP) {
                    if (tb >= valid) break;  // warp-uniform: the step holds no context token
                    // n-tile h = tokens tb + 8 h + (0..7); B column mg of it is token
                    // tb + 8 h + mg, read by lanes (mg, .) as 16-byte vectors (two channels
                    // per word, so one vector holds two k-chunks); two accumulators per
                    // n-tile (even / odd k-chunks) halve the MMA chains
                    float sacc[STEP / 8][4], sodd[STEP / 8][4];
#pragma unroll
                    for (int h = 0; h < STEP / 8; ++h) {
                        sacc[h][0] = sacc[h][1] = sacc[h][2] = sacc[h][3] = 0.f;
                        sodd[h][0] = sodd[h][1] = sodd[h][2] = sodd[h][3] = 0.f;
                        const int kr = tb + 8 * h + mg;  // token row (= mg mod 8)
                        const unsigned char *krow = kt + (kr * D + RUN * mt) * 2;
#pragma unroll
                        for (int j = 0; j < D / (4 * RUN); ++j) {
                            // swizzled: chunk 2 mt + j % 2 of half panel j / 2, at chunk ^ mg
                            const unsigned char *kp =
                                kSwz ? kt + (j >> 1) * kHalfBytes + kr * 128 + ((((2 * mt + (j & 1)) ^ mg) & 7) << 4)
                                     : krow + 64 * j;
                            const uint4 u = *reinterpret_cast<const uint4 *>(kp);
                            if constexpr (kRows16) {
                                mma_16816<kMmaBF16>(sacc[h], qa[2 * j][0], qb[2 * j][0], qa[2 * j][1], qb[2 * j][1],
                                                    u.x, u.y);
                                mma_16816<kMmaBF16>(sodd[h], qa[2 * j + 1][0], qb[2 * j + 1][0], qa[2 * j + 1][1],
                                                    qb[2 * j + 1][1], u.z, u.w);
                            } else {
                                mma_16816<kMmaBF16>(sacc[h], qa[2 * j][0], 0u, qa[2 * j][1], 0u, u.x, u.y);
                                mma_16816<kMmaBF16>(sodd[h], qa[2 * j + 1][0], 0u, qa[2 * j + 1][1], 0u, u.z, u.w);
                            }
                        }
                        sacc[h][0] += sodd[h][0];
                        sacc[h][1] += sodd[h][1];
                        if constexpr (kRows16) {
                            sacc[h][2] += sodd[h][2];
                            sacc[h][3] += sodd[h][3];
                        }
                    }
                    // row mg's scores in log2 units (d0, d1: tokens 2 mt, 2 mt + 1 of the
                    // n-tile); tokens past the context -> -inf
                    float sc[STEP / 4];
#pragma unroll
                    for (int h = 0; h < STEP / 8; ++h)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            sc[2 * h + e] = tb + 8 * h + 2 * mt + e < valid ? sacc[h][e] * mqs : -INFINITY;
                    // ... and row mg + 8's (d2, d3) with 16 heads per block
                    float sc2[kRows16 ? STEP / 4 : 1];
                    if constexpr (kRows16) {
#pragma unroll
                        for (int h = 0; h < STEP / 8; ++h)
#pragma unroll
                            for (int e = 0; e < 2; ++e)
                                sc2[2 * h + e] = tb + 8 * h + 2 * mt + e < valid ? sacc[h][2 + e] * mqs : -INFINITY;
                    }
                    float mx = sc[0], mx2 = kRows16 ? sc2[0] : -INFINITY;
#pragma unroll
                    for (int e = 1; e < STEP / 4; ++e) {
                        mx = fmaxf(mx, sc[e]);
                        if constexpr (kRows16) mx2 = fmaxf(mx2, sc2[e]);
                    }
                    // over the row's four lanes: finite, as token tb is in the context
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    if constexpr (kRows16) {
                        mx2 = fmaxf(mx2, __shfl_xor_sync(0xffffffffu, mx2, 1));
                        mx2 = fmaxf(mx2, __shfl_xor_sync(0xffffffffu, mx2, 2));
                    }
                    const bool grow = mx > mrow, grow2 = kRows16 && mx2 > mrow2;
                    if (__any_sync(0xffffffffu, grow || grow2)) {
                        const float alpha = grow ? fast_exp2(mrow - mx) : 1.f;  // 0 when mrow = -inf
                        lrow *= alpha;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            oacc[nt][0] *= alpha;
                            oacc[nt][1] *= alpha;
                        }
                        if (grow) mrow = mx;
                        if constexpr (kRows16) {
                            const float alpha2 = grow2 ? fast_exp2(mrow2 - mx2) : 1.f;
                            lrow2 *= alpha2;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                oacc[nt][2] *= alpha2;
                                oacc[nt][3] *= alpha2;
                            }
                            if (grow2) mrow2 = mx2;
                        }
                    }
                    // the weights meet V rounded to the cache type (as the A fragment of P V,
                    // rows and k indices those of S); the row sum adds the rounded values
                    uint32_t pa[STEP / 8], pb[STEP / 8];
#pragma unroll
                    for (int h = 0; h < STEP / 8; ++h) {
                        float r0, r1;
                        pa[h] = pack_mma2<kMmaBF16>(fast_exp2(sc[2 * h] - mrow), fast_exp2(sc[2 * h + 1] - mrow),
                                                    r0, r1);
                        lrow += r0 + r1;
                        pb[h] = 0u;
                        if constexpr (kRows16) {
                            pb[h] = pack_mma2<kMmaBF16>(fast_exp2(sc2[2 * h] - mrow2),
                                                        fast_exp2(sc2[2 * h + 1] - mrow2), r0, r1);
                            lrow2 += r0 + r1;
                        }
                    }
                    // O += P V: B column mg of n-tile nt is channel (D / 8) mg + nt; lane
                    // (mg, mt) reads tokens tb + 2 mt, +1 (b0) and tb + 8 + 2 mt, +1 (b1) at its
                    // D / 8 channels and pairs them per channel with one byte permute
                    constexpr int VW = D / 16;  // 32-bit words of a lane's channels in a row
                    uint32_t x[STEP / 4][VW];
                    const unsigned char *vrow = vt + ((tb + 2 * mt) * D + (D / 8) * mg) * 2;
#pragma unroll
                    for (int r = 0; r < STEP / 4; ++r) {
                        if constexpr (kSwz) {
                            // this lane's channels 16 mg .. + 15 are chunks 2 mg, 2 mg + 1 (mod 8) of
                            // half panel mg / 4, at chunk ^ (row & 7); odd mg read the second
                            // chunk first, which keeps the eight lanes of a quarter-warp on
                            // eight different chunks
                            const int vr = tb + 2 * mt + (r >> 1) * 8 + (r & 1);
                            const unsigned char *vp = vt + (mg >> 2) * kHalfBytes + vr * 128;
                            const int odd = mg & 1;
                            const uint4 a = *reinterpret_cast<const uint4 *>(vp + ((((2 * mg + odd) ^ vr) & 7) << 4));
                            const uint4 c = *reinterpret_cast<const uint4 *>(vp + ((((2 * mg + 1 - odd) ^ vr) & 7) << 4));
                            const uint4 lo = odd ? c : a, hi = odd ? a : c;
                            x[r][0] = lo.x;
                            x[r][1] = lo.y;
                            x[r][2] = lo.z;
                            x[r][3] = lo.w;
                            x[r][4] = hi.x;
                            x[r][5] = hi.y;
                            x[r][6] = hi.z;
                            x[r][7] = hi.w;
                        } else {
                            const uint4 *src = reinterpret_cast<const uint4 *>(vrow + ((r >> 1) * 8 + (r & 1)) * D * 2);
#pragma unroll
                            for (int v = 0; v < VW / 4; ++v) {
                                const uint4 u = src[v];
                                x[r][4 * v] = u.x;
                                x[r][4 * v + 1] = u.y;
                                x[r][4 * v + 2] = u.z;
                                x[r][4 * v + 3] = u.w;
                            }
                        }
                    }
                    if (tb + STEP > valid) {  // warp-uniform: a step that ends past the context
                        // rows past the context are unwritten slots of the last block; their
                        // weight is 0, but 0 * NaN or 0 * Inf would still poison O, so the
                        // rows themselves are zeroed before they reach the MMA
#pragma unroll
                        for (int r = 0; r < STEP / 4; ++r) {
                            if (tb + (r >> 1) * 8 + 2 * mt + (r & 1) >= valid) {
#pragma unroll
                                for (int w = 0; w < VW; ++w) x[r][w] = 0u;
                            }
                        }
                    }
#pragma unroll
                    for (int w = 0; w < VW; ++w) {
                        uint32_t b0[2], b1[2] = {0u, 0u};
                        b0[0] = __byte_perm(x[0][w], x[1][w], 0x5410);  // low halves: channel 2 w
                        b0[1] = __byte_perm(x[0][w], x[1][w], 0x7632);  // high halves: 2 w + 1
                        if constexpr (STEP == 16) {
                            b1[0] = __byte_perm(x[2][w], x[3][w], 0x5410);
                            b1[1] = __byte_perm(x[2][w], x[3][w], 0x7632);
                        }
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            mma_16816<kMmaBF16>(oacc[2 * w + e], pa[0], pb[0], STEP == 16 ? pa[STEP / 8 - 1] : 0u,
                                                STEP == 16 ? pb[STEP / 8 - 1] : 0u, b0[e], b1[e]);
                    }
                }
            } else {
#pragma unroll
                for (int it0 = 0; it0 < ITERS; it0 += IT_STEP) {
                    // QK: partial dot products over this lane's 8 dims
                    float sc[IT_STEP][GH];
#pragma unroll
                    for (int it = 0; it < IT_STEP; ++it) {
                        const int t = (it0 + it) * TPG + grp;
                        if constexpr (kQuant) {
                            uint32_t kh[VL / 2];
                            load_codes_f16<VL>(ks + t * D + sub * VL, kh);
#pragma unroll
                            for (int g = 0; g < GH; ++g) {
                                float a0 = -qo[g], a1 = 0.f;
#pragma unroll
                                for (int e = 0; e < VL / 2; ++e) fma_f16x2_f32(qh[g][e], kh[e], a0, a1);
                                sc[it][g] = (a0 + a1) * qs[g];
                            }
                        } else {
                            float kf[VL];
                            load_lane<KT, VL>(ks + t * D + sub * VL, kf);
#pragma unroll
                            for (int g = 0; g < GH; ++g) {
                                float a = 0.f;
#pragma unroll
                                for (int e = 0; e < VL; ++e) a = fmaf(qf[g][e], kf[e], a);
                                sc[it][g] = a;
                            }
                        }
                    }
                    // full dot products: sum over the LPT lanes of each token row
#pragma unroll
                    for (int it = 0; it < IT_STEP; ++it)
#pragma unroll
                        for (int g = 0; g < GH; ++g)
#pragma unroll
                            for (int o = LPT / 2; o > 0; o >>= 1)
                                sc[it][g] += __shfl_xor_sync(0xffffffffu, sc[it][g], o);
                    // mask rows past the end of the context
#pragma unroll
                    for (int it = 0; it < IT_STEP; ++it) {
                        const int t = (it0 + it) * TPG + grp;
                        if (t >= valid) {
#pragma unroll
                            for (int g = 0; g < GH; ++g) sc[it][g] = -INFINITY;
                        }
                    }
                    // online softmax update (P1 §7.2), m warp-uniform
#pragma unroll
                    for (int g = 0; g < GH; ++g) {
                        float mx = sc[0][g];
#pragma unroll
                        for (int it = 1; it < IT_STEP; ++it) mx = fmaxf(mx, sc[it][g]);
#pragma unroll
                        for (int o = LPT; o < 32; o <<= 1)
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                        if (mx > m[g]) {  // warp-uniform branch
                            const float alpha = fast_exp2(m[g] - mx);  // 0 when m was -inf
                            l[g] *= alpha;
#pragma unroll
                            for (int e = 0; e < VL; ++e) acc[g][e] *= alpha;
                            m[g] = mx;
                        }
#pragma unroll
                        for (int it = 0; it < IT_STEP; ++it) {
                            sc[it][g] = fast_exp2(sc[it][g] - m[g]);  // masked rows -> 0
                            // INT8: the weight meets V in fp16; the sum adds the rounded value
                            if constexpr (kQuant) sc[it][g] = __half2float(__float2half_rn(sc[it][g]));
                            l[g] += sc[it][g];
                        }
                    }
                    // PV: lane-local, each lane owns 8 dims of every head
#pragma unroll
                    for (int it = 0; it < IT_STEP; ++it) {
                        const int t = (it0 + it) * TPG + grp;
                        if (t < valid) {
                            if constexpr (kQuant) {
                                uint32_t vh[VL / 2];
                                load_codes_f16<VL>(vs + t * D + sub * VL, vh);
#pragma unroll
                                for (int g = 0; g < GH; ++g) {
                                    const __half2 w2 = __float2half2_rn(sc[it][g]);  // exact: rounded above
                                    const uint32_t w = *reinterpret_cast<const uint32_t *>(&w2);
#pragma unroll
                                    for (int e = 0; e < VL / 2; ++e)
                                        fma_f16x2_f32(w, vh[e], acc[g][2 * e], acc[g][2 * e + 1]);
                                }
                            } else {
                                float vf[VL];
                                load_lane<KT, VL>(vs + t * D + sub * VL, vf);
#pragma unroll
                                for (int g = 0; g < GH; ++g) {
#pragma unroll
                                    for (int e = 0; e < VL; ++e) acc[g][e] = fmaf(sc[it][g], vf[e], acc[g][e]);
                                }
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && i + S < my_chunks) {
            fence_proxy_async_smem();
            issue(warp + (i + S) * NW, s);
        }
    }

    // ---- merge the token groups of this warp (same m across the warp); in the
    //      MMA form the row sums of a head's four lanes
    if constexpr (kMma && kQuant) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], o);
            if (aborted) {
                mh[e] = -INFINITY;
                lh[e] = 0.f;
            }
        }
    } else if constexpr (kMma) {
        lrow += __shfl_xor_sync(0xffffffffu, lrow, 1);
        lrow += __shfl_xor_sync(0xffffffffu, lrow, 2);
        lrow2 += __shfl_xor_sync(0xffffffffu, lrow2, 1);
        lrow2 += __shfl_xor_sync(0xffffffffu, lrow2, 2);
        if (aborted) {
            mrow = mrow2 = -INFINITY;
            lrow = lrow2 = 0.f;
        }
    } else {
#pragma unroll
        for (int g = 0; g < GH; ++g) {
#pragma unroll
            for (int o = LPT; o < 32; o <<= 1) {
                l[g] += __shfl_xor_sync(0xffffffffu, l[g], o);
#pragma unroll
                for (int e = 0; e < VL; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);
            }
        }
        if (aborted) {
#pragma unroll
            for (int g = 0; g < GH; ++g) {
                m[g] = -INFINITY;
                l[g] = 0.f;
            }
        }
    }

    // ---- merge the warps through shared memory (each warp reuses its own
    //      stage buffers: all of its copies have landed)
    float *mine = reinterpret_cast<float *>(my_stages);  // [GH][D + 2]
    if constexpr (kMma && kQuant) {
        // lane (mg, mt): heads 2 mt, 2 mt + 1 at channels (D / 8) mg + 2 j (+ 1)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * mt + e;
            if (h >= GH) continue;
            float *row = mine + h * (D + 4) + (D / 8) * mg;
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                row[2 * j] = oacc[j][e];
                row[2 * j + 1] = oacc[j][2 + e];
            }
            if (mg == 0) {
                mine[h * (D + 4) + D] = mh[e];
                mine[h * (D + 4) + D + 1] = lh[e];
            }
        }
    } else if constexpr (kMma) {
        // d0 / d1 of n-tile nt: head mg, channels (D / 8) (2 mt) + nt / (D / 8) (2 mt + 1) + nt;
        // d2 / d3: head mg + 8 (16 heads per block)
        if (mg < GH) {
            float *row = mine + mg * (D + 4);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                row[(D / 8) * (2 * mt) + nt] = oacc[nt][0];
                row[(D / 8) * (2 * mt + 1) + nt] = oacc[nt][1];
            }
            if (mt == 0) {
                row[D] = mrow;
                row[D + 1] = lrow;
            }
        }
        if constexpr (kRows16) {
            float *row = mine + (mg + 8) * (D + 4);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                row[(D / 8) * (2 * mt) + nt] = oacc[nt][2];
                row[(D / 8) * (2 * mt + 1) + nt] = oacc[nt][3];
            }
            if (mt == 0) {
                row[D] = mrow2;
                row[D + 1] = lrow2;
            }
        }
    } else {
        if (grp == 0) {
#pragma unroll
            for (int g = 0; g < GH; ++g) {
                float4 *dst = reinterpret_cast<float4 *>(mine + g * (D + 4) + sub * VL);
#pragma unroll
                for (int v = 0; v < VL / 4; ++v)
                    dst[v] = make_float4(acc[g][4 * v], acc[g][4 * v + 1], acc[g][4 * v + 2], acc[g][4 * v + 3]);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int g = 0; g < GH; ++g) {
                mine[g * (D + 4) + D] = m[g];
                mine[g * (D + 4) + D + 1] = l[g];
            }
        }
    }
    __syncthreads();

    const bool single = nparts == 1 && !p.always_partial;
    for (int idx = threadIdx.x; idx < GH * D; idx += blockDim.x) {
        const int g = idx / D;
        const int j = idx - g * D;
        float mw[NW];
        float mmax = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float *src = reinterpret_cast<const float *>(stages + w * S * G::kStageBytes);
            mw[w] = src[g * (D + 4) + D];
            mmax = fmaxf(mmax, mw[w]);
        }
        float lsum = 0.f, osum = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float *src = reinterpret_cast<const float *>(stages + w * S * G::kStageBytes);
            const float wgt = mw[w] == -INFINITY ? 0.f : fast_exp2(mw[w] - mmax);
            lsum += wgt * src[g * (D + 4) + D + 1];
            osum += wgt * src[g * (D + 4) + j];
        }
        // V: the value sums carry kCodeOffset per unit of weight; then dequantise
        if constexpr (kQuant) osum = (osum - kCodeOffset * lsum) * p.v_scale[kvh * D + j];
        const int hq = hq0 + g;
        const int64_t row = static_cast<int64_t>(seq) * p.num_q_heads + hq;
        if (single) {
            const float r = lsum > 0.f ? osum / lsum : 0.f;
            static_cast<T *>(p.out)[row * D + j] = Elem<T>::from_f32(r);
        } else {
            const int64_t pr = row * p.num_partitions + p.slot_base + part;
            p.ws_o[pr * D + j] = osum;
            if (j == 0) {
                p.ws_m[pr] = mmax;
                p.ws_l[pr] = lsum;
            }
        }
    }
}

// Log-sum-exp merge of the partitions of each (sequence, query head):
//   M = max_p m_p,  L = sum_p l_p 2^(m_p - M),  out = sum_p o_p 2^(m_p - M) / L.
// WPR warps per (sequence, query head): one (four rows per block) for a few
// partitions, four (one row per block) for many, warp w taking partitions w,
// w + 4, ... and the four results combined through shared memory as they would
// be partitions (the same formula over M_w, L_w, O_w).  Sequences that fit one
// partition were written by the main kernel and are skipped.  In a warp, lane q
// reads its q-th partition's m and l, so the maximum and the weights take one
// round of loads and shuffles; the partial outputs (D / 32 values per lane and
// partition) are then read kMergeUnroll partitions at a time, all in flight
// together.  Launched behind the decode kernel (programmatic dependent launch):
// it waits for that grid's partials before reading any.
constexpr int kMergeUnroll = 8;
constexpr int kMergeWideFrom = 32;  // partitions per row from which four warps share a row

template <typename T, int D, int WPR>
__global__ void __launch_bounds__(128) paged_decode_merge_kernel(const DecodeParams p,
                                                                 int num_rows) {
    static_assert(WPR == 1 || WPR == 4, "one or four warps per row");
    pdl_wait();
    constexpr int PER_LANE = D / 32;
    using Part = typename std::conditional<PER_LANE == 4, float4, float2>::type;
    static_assert(PER_LANE == 4 || PER_LANE == 2, "head_dim 128 or 64");
    __shared__ float comb[WPR == 4 ? 4 : 1][D + 2];  // four warps' (o, m, l) of one row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * (4 / WPR) + warp / WPR;  // uniform over a block when WPR == 4
    const int share = warp % WPR;                          // this warp takes partitions share + WPR i
    if (row >= num_rows) return;
    const int seq = row / p.num_q_heads;
    int len = p.context_lens[seq];  // clamped exactly as the main kernel does
    if (p.tok_begin > 0 && len < p.tok_begin && lane == 0 && share == 0 && (row % p.num_q_heads) == 0)
        raise_flag(p.status, PKV_DEVERR_CONTEXT_LEN);  // shorter than the shared prefix
    if (len < 0) len = 0;
    if (len > p.len_cap) len = p.len_cap;
    const int nparts = p.slot_base + partitions_of(p, len);  // slots holding partials
    if (nparts <= 1 && !p.always_partial) return;           // written by the decode kernel
    const int mine = nparts > share ? (nparts - share + WPR - 1) / WPR : 0;  // this warp's partitions
    const int64_t base = static_cast<int64_t>(row) * p.num_partitions;
    auto slot = [&](int i) { return share + WPR * i; };  // the slot of this warp's i-th partition
    float mmax = -INFINITY;
    for (int q = lane; q < mine; q += 32) mmax = fmaxf(mmax, p.ws_m[base + slot(q)]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    float lsum = 0.f;
    float o[PER_LANE];
#pragma unroll
    for (int e = 0; e < PER_LANE; ++e) o[e] = 0.f;
    const Part *parts = reinterpret_cast<const Part *>(p.ws_o + base * D) + lane;  // slot q at q * 32
    for (int q0 = 0; q0 < mine; q0 += 32) {
        const int cnt = min(32, mine - q0);
        float w = 0.f;  // this lane's partition q0 + lane
        if (lane < cnt) {
            const float mq = p.ws_m[base + slot(q0 + lane)];
            w = mq == -INFINITY ? 0.f : fast_exp2(mq - mmax);
            lsum += w * p.ws_l[base + slot(q0 + lane)];
        }
        for (int j0 = 0; j0 < cnt; j0 += kMergeUnroll) {
            Part v[kMergeUnroll];
#pragma unroll
            for (int u = 0; u < kMergeUnroll; ++u)
                if (j0 + u < cnt) v[u] = parts[static_cast<int64_t>(slot(q0 + j0 + u)) * 32];
#pragma unroll
            for (int u = 0; u < kMergeUnroll; ++u) {
                const float wu = __shfl_sync(0xffffffffu, w, (j0 + u) & 31);
                if (j0 + u < cnt) {
                    const float *f = reinterpret_cast<const float *>(&v[u]);
#pragma unroll
                    for (int e = 0; e < PER_LANE; ++e) o[e] = fmaf(wu, f[e], o[e]);
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if constexpr (WPR == 4) {
        // the four warps' results, relative to their own maxima, combined in warp 0
#pragma unroll
        for (int e = 0; e < PER_LANE; ++e) comb[share][lane * PER_LANE + e] = o[e];
        if (lane == 0) {
            comb[share][D] = mmax;
            comb[share][D + 1] = lsum;
        }
        __syncthreads();
        if (share != 0) return;
        float mw[4], mall = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            mw[w] = comb[w][D];
            mall = fmaxf(mall, mw[w]);
        }
        lsum = 0.f;
#pragma unroll
        for (int e = 0; e < PER_LANE; ++e) o[e] = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float sw = mw[w] == -INFINITY ? 0.f : fast_exp2(mw[w] - mall);
            lsum += sw * comb[w][D + 1];
#pragma unroll
            for (int e = 0; e < PER_LANE; ++e) o[e] = fmaf(sw, comb[w][lane * PER_LANE + e], o[e]);
        }
    }
    T *dst = static_cast<T *>(p.out) + static_cast<int64_t>(row) * D + lane * PER_LANE;
#pragma unroll
    for (int e = 0; e < PER_LANE; ++e) dst[e] = Elem<T>::from_f32(lsum > 0.f ? o[e] / lsum : 0.f);
}

}  // namespace pkv
