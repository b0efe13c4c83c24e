/*
 * pagedkv_oracle.c -- plain, slow CPU oracle for paged-KV-cache decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference legs may load this code.  The product
 * (the CUDA library and its Python binding) never links, imports or calls it,
 * and this file includes nothing from the product.
 *
 * Pages this follows (cited by title and section):
 *   P1 = "KV Cache与PagedAttention深度解析：vLLM内存管理革命" (iopencloud.com)
 *   P2 = "KV Cache从原理到实战：大模型推理内存管理演进与优化" (xnwp.cn/news/16711)
 *   P3 = PagedAttention + prefix caching via nano-vllm (zwxr.cn/news/317362)
 *   P4 = "大模型 (LLM) 推理加速核心技术解析：从 KV Cache 到 PagedAttention 实战"
 *        (jsqmd.com/news/745991)
 *
 * Arithmetic: every floating-point value is carried in IEEE double (fp64).
 * The 16-bit inputs are decoded exactly from their bit patterns by this file's
 * own decoders (no compiler half/bfloat16 type is used).  exp() is libm's.
 *
 * Physical cache layout (P1 §4.3 and §5.1, with num_kv_heads in place of
 * num_heads): pool[num_blocks][2][num_kv_heads][block_size][head_dim]; the K
 * half of physical block b, head h, in-block offset o, element j sits at
 *     k_cache[b * block_stride + (h * block_size + o) * head_dim + j]
 * and the V half at the same index of v_cache.  For the packed pool
 * block_stride = 2 * num_kv_heads * block_size * head_dim and
 * v_cache = k_cache + num_kv_heads * block_size * head_dim.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);               /* subnormal: frac * 2^(1-15-10) */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/2^10) * 2^(expo-15) */
    return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xff;
    int frac = bits & 0x7f;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -133);               /* subnormal: frac * 2^(1-127-7) */
    else if (expo == 255)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + frac), expo - 134); /* (1 + frac/2^7) * 2^(expo-127) */
    return sign ? -mag : mag;
}

static double decode16(uint16_t bits, int dtype) {
    return dtype == ORACLE_BF16 ? oracle_bf16_to_f64(bits) : oracle_f16_to_f64(bits);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Slot of logical position t of a sequence (P1 §5.3: the new token goes to
 * the last block of the table at offset t % block_size; the block holding
 * position t is table[t / block_size]). */
int64_t oracle_slot_for_position(const int32_t *table_row, int64_t t, int block_size) {
    return (int64_t)table_row[t / block_size] * block_size + t % block_size;
}

/* Blocks a sequence needs once it holds token t (P1 §5.3: ceil((t+1)/block_size)). */
int64_t oracle_blocks_needed(int64_t t, int block_size) {
    return (t + 1 + block_size - 1) / block_size;
}

/*
 * Decode attention, direct definition (P1 §2.1: softmax(Q K^T / sqrt(d_k)) V,
 * with one query row per sequence and head).  For sequence i and query head
 * hq the KV head is h = hq / G with G = num_q_heads / num_kv_heads (grouped
 * query attention, P2 §5.3; heads of a group are contiguous).  Token t of the
 * sequence lives in physical block block_tables[i][t / bs] at offset t % bs
 * (P1 §4.2 and §4.3).  Two passes: scores and their maximum M, then
 * w_t = exp(s_t - M), Z = sum w_t, out = sum w_t v_t / Z.  A sequence with no
 * tokens gets a zero row (P1 §4.3 starts the output at zeros).
 *
 * q: [num_seqs][num_q_heads][head_dim] 16-bit values; out: same shape, fp64.
 */
void oracle_paged_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         int64_t block_stride, const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, double scale, int dtype,
                         double *out) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t pairs = (int64_t)num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pair = 0; pair < pairs; ++pair) {
        const int i = (int)(pair / num_q_heads);
        const int hq = (int)(pair % num_q_heads);
        const int h = hq / group;
        const int64_t len = context_lens[i];
        const uint16_t *qrow = q + ((int64_t)i * num_q_heads + hq) * head_dim;
        double *orow = out + ((int64_t)i * num_q_heads + hq) * head_dim;
        for (int j = 0; j < head_dim; ++j) orow[j] = 0.0;
        if (len <= 0) continue;

        double *qv = (double *)malloc(sizeof(double) * head_dim);
        double *score = (double *)malloc(sizeof(double) * len);
        for (int j = 0; j < head_dim; ++j) qv[j] = decode16(qrow[j], dtype);

        /* pass 1: s_t = scale * q . k_t, and the maximum score */
        double smax = -INFINITY;
        for (int64_t t = 0; t < len; ++t) {
            const int64_t phys = block_tables[(int64_t)i * max_blocks_per_seq + t / block_size];
            const int64_t off = t % block_size;
            const uint16_t *krow = k_cache + phys * block_stride + ((int64_t)h * block_size + off) * head_dim;
            double dot = 0.0;
            for (int j = 0; j < head_dim; ++j) dot += qv[j] * decode16(krow[j], dtype);
            score[t] = scale * dot;
            if (score[t] > smax) smax = score[t];
        }
        /* pass 2: w_t = exp(s_t - max), Z = sum w_t, out = sum w_t v_t / Z */
        double z = 0.0;
        for (int64_t t = 0; t < len; ++t) {
            const int64_t phys = block_tables[(int64_t)i * max_blocks_per_seq + t / block_size];
            const int64_t off = t % block_size;
            const uint16_t *vrow = v_cache + phys * block_stride + ((int64_t)h * block_size + off) * head_dim;
            const double w = exp(score[t] - smax);
            z += w;
            for (int j = 0; j < head_dim; ++j) orow[j] += w * decode16(vrow[j], dtype);
        }
        for (int j = 0; j < head_dim; ++j) orow[j] /= z;
        free(score);
        free(qv);
    }
}

/*
 * Decode attention in the online (running max / running sum) form that P1
 * §7.2 gives for its block-table-aware flash kernel: per logical block, scores
 * of the block, m_new = max(m, max scores), alpha = exp(m - m_new),
 * l = l * alpha + sum exp(scores - m_new), acc = acc * alpha + exp(scores - m_new) V,
 * and the result is acc / l.  Mathematically equal to oracle_paged_decode;
 * kept so tests can check the rescaling algebra the GPU kernel relies on.
 */
void oracle_paged_flash_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                               int64_t block_stride, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               double scale, int dtype, double *out) {
    const int group = num_q_heads / num_kv_heads;
    double *qv = (double *)malloc(sizeof(double) * head_dim);
    double *sblk = (double *)malloc(sizeof(double) * block_size);
    for (int i = 0; i < num_seqs; ++i) {
        for (int hq = 0; hq < num_q_heads; ++hq) {
            const int h = hq / group;
            const int64_t len = context_lens[i];
            const uint16_t *qrow = q + ((int64_t)i * num_q_heads + hq) * head_dim;
            double *orow = out + ((int64_t)i * num_q_heads + hq) * head_dim;
            for (int j = 0; j < head_dim; ++j) {
                orow[j] = 0.0;
                qv[j] = decode16(qrow[j], dtype);
            }
            if (len <= 0) continue;
            double m = -INFINITY, l = 0.0;
            const int64_t nblocks = (len + block_size - 1) / block_size;
            for (int64_t b = 0; b < nblocks; ++b) {
                const int64_t phys = block_tables[(int64_t)i * max_blocks_per_seq + b];
                const int64_t ntok = (b + 1) * block_size <= len ? block_size : len - b * block_size;
                double bmax = -INFINITY;
                for (int64_t o = 0; o < ntok; ++o) {
                    const uint16_t *krow = k_cache + phys * block_stride + ((int64_t)h * block_size + o) * head_dim;
                    double dot = 0.0;
                    for (int j = 0; j < head_dim; ++j) dot += qv[j] * decode16(krow[j], dtype);
                    sblk[o] = scale * dot;
                    if (sblk[o] > bmax) bmax = sblk[o];
                }
                const double m_new = m > bmax ? m : bmax;
                const double alpha = exp(m - m_new);
                l *= alpha;
                for (int j = 0; j < head_dim; ++j) orow[j] *= alpha;
                for (int64_t o = 0; o < ntok; ++o) {
                    const double p = exp(sblk[o] - m_new);
                    const uint16_t *vrow = v_cache + phys * block_stride + ((int64_t)h * block_size + o) * head_dim;
                    l += p;
                    for (int j = 0; j < head_dim; ++j) orow[j] += p * decode16(vrow[j], dtype);
                }
                m = m_new;
            }
            for (int j = 0; j < head_dim; ++j) orow[j] /= l;
        }
    }
    free(sblk);
    free(qv);
}

/*
 * Cache write for the new tokens (P1 §2.2: compute K_t, V_t and append them;
 * P1 §5.3: write them at offset t % block_size of the sequence's last block).
 * Token n's head h row of k_new/v_new ([num_tokens][num_kv_heads][head_dim])
 * is copied byte for byte to slot s = slot_mapping[n], i.e. block s / bs,
 * offset s % bs.  A negative slot means "no write" (padding).
 */
void oracle_reshape_and_cache(const uint16_t *k_new, const uint16_t *v_new,
                              const int64_t *slot_mapping, int64_t num_tokens, uint16_t *k_cache,
                              uint16_t *v_cache, int64_t block_stride, int num_kv_heads,
                              int head_dim, int block_size) {
    for (int64_t n = 0; n < num_tokens; ++n) {
        const int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        const int64_t blk = slot / block_size;
        const int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t dst = blk * block_stride + ((int64_t)h * block_size + off) * head_dim;
            const int64_t src = (n * num_kv_heads + h) * (int64_t)head_dim;
            memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * head_dim);
            memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * head_dim);
        }
    }
}

/*
 * Copy-on-write block copies (P1 §8.3 and P3 §2.3 / §5.5: a sequence about
 * to write into a shared block first gets a private copy).  For each pair
 * (src, dst) in src_dst ([num_pairs][2]) the K half and the V half of
 * physical block src are copied byte for byte over those of block dst.
 */
void oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, int64_t block_stride,
                        int64_t block_elems, const int64_t *src_dst, int64_t num_pairs) {
    for (int64_t p = 0; p < num_pairs; ++p) {
        const int64_t src = src_dst[2 * p], dst = src_dst[2 * p + 1];
        memcpy(k_cache + dst * block_stride, k_cache + src * block_stride, sizeof(uint16_t) * block_elems);
        memcpy(v_cache + dst * block_stride, v_cache + src * block_stride, sizeof(uint16_t) * block_elems);
    }
}

/* ------------------------------------------------------------------------
 * INT8 KV cache with per-channel scales (P2 §5.2: storing the cache as INT8
 * halves its bytes; scales computed per channel, separately for K and V, is
 * the INT8 variant that page recommends over per-tensor scales).  Channel c of
 * KV head h owns one K scale and one V scale, scale[h * head_dim + c] > 0.
 *
 * Quantise (the page does not fix the rounding; the readings used here):
 * x is the 16-bit input, widened exactly to IEEE single precision;
 * r = x / s in single precision; r is clamped to [-127, 127] (symmetric
 * range, -128 unused) and rounded to the nearest integer, ties to even.
 * The division is done in single precision because the code is an integer
 * decided by floating point: both implementations must take that decision in
 * the same precision.  (A NaN input clamps to -127: fmaxf returns the
 * non-NaN operand.)
 * Dequantise: x' = code * s (exact in fp64).  Attention then follows the
 * same definition as oracle_paged_decode on the dequantised K and V.
 * ------------------------------------------------------------------------ */
int oracle_quantize_int8(uint16_t bits, int dtype, float scale) {
    const float x = (float)decode16(bits, dtype); /* exact: 16-bit values fit in binary32 */
    float r = x / scale;
    r = fmaxf(r, -127.0f);
    r = fminf(r, 127.0f);
    return (int)nearbyintf(r); /* default rounding mode: to nearest, ties to even */
}

/* Element i of x uses scale[i % scale_period] (x laid out [..][heads][head_dim]
 * with scale [heads][head_dim] gives scale_period = heads * head_dim). */
void oracle_quantize_int8_array(const uint16_t *x, int64_t n, const float *scale,
                                int64_t scale_period, int dtype, int8_t *codes) {
    for (int64_t i = 0; i < n; ++i)
        codes[i] = (int8_t)oracle_quantize_int8(x[i], dtype, scale[i % scale_period]);
}

/* Cache write into an INT8 pool: token n's head h row is quantised channel by
 * channel with that head's scales and stored at slot s = slot_mapping[n]
 * (block s / bs, offset s % bs), exactly as oracle_reshape_and_cache places a
 * 16-bit row.  A negative slot means "no write". */
void oracle_reshape_and_cache_int8(const uint16_t *k_new, const uint16_t *v_new,
                                   const int64_t *slot_mapping, int64_t num_tokens,
                                   int8_t *k_cache, int8_t *v_cache, int64_t block_stride,
                                   int num_kv_heads, int head_dim, int block_size,
                                   const float *k_scale, const float *v_scale, int dtype) {
    for (int64_t n = 0; n < num_tokens; ++n) {
        const int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        const int64_t blk = slot / block_size;
        const int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t dst = blk * block_stride + ((int64_t)h * block_size + off) * head_dim;
            const int64_t src = (n * num_kv_heads + h) * (int64_t)head_dim;
            for (int j = 0; j < head_dim; ++j) {
                k_cache[dst + j] = (int8_t)oracle_quantize_int8(k_new[src + j], dtype, k_scale[h * head_dim + j]);
                v_cache[dst + j] = (int8_t)oracle_quantize_int8(v_new[src + j], dtype, v_scale[h * head_dim + j]);
            }
        }
    }
}

/* Decode attention over an INT8 pool: the direct two-pass definition of
 * oracle_paged_decode with k_t[j] = code * k_scale[h][j] and
 * v_t[j] = code * v_scale[h][j].  q is 16-bit; out is fp64. */
void oracle_paged_decode_int8(const uint16_t *q, const int8_t *k_cache, const int8_t *v_cache,
                              const float *k_scale, const float *v_scale, int64_t block_stride,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int num_seqs, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size, double scale,
                              int dtype, double *out) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t pairs = (int64_t)num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t pair = 0; pair < pairs; ++pair) {
        const int i = (int)(pair / num_q_heads);
        const int hq = (int)(pair % num_q_heads);
        const int h = hq / group;
        const int64_t len = context_lens[i];
        const uint16_t *qrow = q + ((int64_t)i * num_q_heads + hq) * head_dim;
        const float *ks = k_scale + (int64_t)h * head_dim;
        const float *vs = v_scale + (int64_t)h * head_dim;
        double *orow = out + ((int64_t)i * num_q_heads + hq) * head_dim;
        for (int j = 0; j < head_dim; ++j) orow[j] = 0.0;
        if (len <= 0) continue;

        double *qv = (double *)malloc(sizeof(double) * head_dim);
        double *score = (double *)malloc(sizeof(double) * len);
        for (int j = 0; j < head_dim; ++j) qv[j] = decode16(qrow[j], dtype);

        double smax = -INFINITY;
        for (int64_t t = 0; t < len; ++t) {
            const int64_t phys = block_tables[(int64_t)i * max_blocks_per_seq + t / block_size];
            const int64_t off = t % block_size;
            const int8_t *krow = k_cache + phys * block_stride + ((int64_t)h * block_size + off) * head_dim;
            double dot = 0.0;
            for (int j = 0; j < head_dim; ++j) dot += qv[j] * ((double)krow[j] * (double)ks[j]);
            score[t] = scale * dot;
            if (score[t] > smax) smax = score[t];
        }
        double z = 0.0;
        for (int64_t t = 0; t < len; ++t) {
            const int64_t phys = block_tables[(int64_t)i * max_blocks_per_seq + t / block_size];
            const int64_t off = t % block_size;
            const int8_t *vrow = v_cache + phys * block_stride + ((int64_t)h * block_size + off) * head_dim;
            const double w = exp(score[t] - smax);
            z += w;
            for (int j = 0; j < head_dim; ++j) orow[j] += w * ((double)vrow[j] * (double)vs[j]);
        }
        for (int j = 0; j < head_dim; ++j) orow[j] /= z;
        free(score);
        free(qv);
    }
}

/* copy-on-write block copies on a pool of any element size: the K and V
 * halves of block src, block_bytes each, copied byte for byte over block dst's. */
void oracle_copy_blocks_bytes(unsigned char *k_cache, unsigned char *v_cache,
                              int64_t block_stride_bytes, int64_t block_bytes,
                              const int64_t *src_dst, int64_t num_pairs) {
    for (int64_t p = 0; p < num_pairs; ++p) {
        const int64_t src = src_dst[2 * p], dst = src_dst[2 * p + 1];
        memcpy(k_cache + dst * block_stride_bytes, k_cache + src * block_stride_bytes, block_bytes);
        memcpy(v_cache + dst * block_stride_bytes, v_cache + src * block_stride_bytes, block_bytes);
    }
}

/* ------------------------------------------------------------------------
 * Chunked prefill attention over the paged cache.  P4 §2 (causal
 * self-attention with a cache): the new tokens' K and V are appended to the
 * cache, then each new token's query attends to the cached tokens and,
 * causally, to the new tokens up to itself; P2 §2.3 (prefill handles a whole
 * prompt at once) and §5.4 (chunked prefill splits a long prompt into pieces).
 * The page's mask is a square lower triangle over the new tokens only; with
 * cached tokens in front, the reading used here is the same rule on absolute
 * positions: query at position p sees tokens 0 .. p.
 *
 * Sequence i holds context_lens[i] = L_i tokens in the cache, of which its
 * chunk is the last C_i = query_start[i+1] - query_start[i] (positions
 * L_i - C_i .. L_i - 1; the chunk's K and V are already in the cache).  Query
 * row j of the chunk is global row query_start[i] + j of q
 * ([num_rows][num_q_heads][head_dim]); at position p = L_i - C_i + j it gives
 *     out = sum_{t <= p} exp(s_t - M) v_t / sum_{t <= p} exp(s_t - M),
 *     s_t = scale * q . k_t,  M = max_{t <= p} s_t,
 * the two-pass direct definition of oracle_paged_decode over tokens 0 .. p.
 * ------------------------------------------------------------------------ */
void oracle_paged_prefill(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          int64_t block_stride, const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *query_start, const int32_t *context_lens, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          double scale, int dtype, double *out) {
    const int group = num_q_heads / num_kv_heads;
    const int64_t num_rows = query_start[num_seqs];
    const int64_t pairs = num_rows * num_q_heads;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t pair = 0; pair < pairs; ++pair) {
        const int64_t row = pair / num_q_heads;
        const int hq = (int)(pair % num_q_heads);
        const int h = hq / group;
        int i = 0;
        while (query_start[i + 1] <= row) ++i;            /* the row's sequence */
        const int64_t chunk = query_start[i + 1] - query_start[i];
        const int64_t pos = context_lens[i] - chunk + (row - query_start[i]);
        const int64_t len = pos + 1;                      /* tokens this row sees */
        const uint16_t *qrow = q + (row * num_q_heads + hq) * head_dim;
        double *orow = out + (row * num_q_heads + hq) * head_dim;
        for (int j = 0; j < head_dim; ++j) orow[j] = 0.0;
        if (len <= 0) continue;

        double *qv = (double *)malloc(sizeof(double) * head_dim);
        double *score = (double *)malloc(sizeof(double) * len);
        for (int j = 0; j < head_dim; ++j) qv[j] = decode16(qrow[j], dtype);
        double smax = -INFINITY;
        for (int64_t t = 0; t < len; ++t) {
            const int64_t phys = block_tables[(int64_t)i * max_blocks_per_seq + t / block_size];
            const int64_t off = t % block_size;
            const uint16_t *krow = k_cache + phys * block_stride + ((int64_t)h * block_size + off) * head_dim;
            double dot = 0.0;
            for (int j = 0; j < head_dim; ++j) dot += qv[j] * decode16(krow[j], dtype);
            score[t] = scale * dot;
            if (score[t] > smax) smax = score[t];
        }
        double z = 0.0;
        for (int64_t t = 0; t < len; ++t) {
            const int64_t phys = block_tables[(int64_t)i * max_blocks_per_seq + t / block_size];
            const int64_t off = t % block_size;
            const uint16_t *vrow = v_cache + phys * block_stride + ((int64_t)h * block_size + off) * head_dim;
            const double w = exp(score[t] - smax);
            z += w;
            for (int j = 0; j < head_dim; ++j) orow[j] += w * decode16(vrow[j], dtype);
        }
        for (int j = 0; j < head_dim; ++j) orow[j] /= z;
        free(score);
        free(qv);
    }
}
