// cache_ops.cu -- the cache-side ops of the paged KV cache:
//   pkv_reshape_and_cache: scatter each new token's K/V rows into its slot
//     ("KV Cache与PagedAttention深度解析" §2.2 append step, §5.3 slot rule);
//   pkv_reshape_and_cache_int8: the same placement into an INT8 cache, each
//     value quantised with its channel's scale ("KV Cache从原理到实战" §5.2);
//   pkv_copy_blocks: copy-on-write copies of whole blocks (same page §8.3;
//     zwxr.cn nano-vllm article §2.3, §5.5);
//   pkv_slot_mapping / pkv_slot_mapping_host: the slot each new token is
//     written to (same page §5.3), on the device or on host arrays.
// The 16-bit write and the copy move 16-byte vectors and are bit-exact; the
// INT8 write's codes are those of the quantiser in pkv_device.cuh.
// Device-resident indices are range-checked before use; a bad one raises a
// status flag and is skipped.
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace {

// One CTA per new token; threads walk the token's (head, 16-byte chunk) pairs
// for K and V.  row_vecs = head_dim * elem_bytes / 16.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int64_t *__restrict__ slot_mapping, char *__restrict__ k_cache,
    char *__restrict__ v_cache, int64_t num_slots, int64_t block_stride_bytes, int num_kv_heads,
    int row_vecs, int block_size, unsigned int *status) {
    const int64_t n = blockIdx.x;
    const int64_t slot = slot_mapping[n];
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        if (threadIdx.x == 0) pkv::raise_flag(status, PKV_DEVERR_SLOT);
        return;
    }
    const int64_t blk = slot / block_size;
    const int off = static_cast<int>(slot % block_size);
    const int per_token = num_kv_heads * row_vecs;
    for (int i = threadIdx.x; i < per_token; i += blockDim.x) {
        const int h = i / row_vecs;
        const int c = i - h * row_vecs;
        const int64_t dst = blk * block_stride_bytes +
                            ((static_cast<int64_t>(h) * block_size + off) * row_vecs + c) * 16;
        const uint4 kv = k_new[n * per_token + i];
        const uint4 vv = v_new[n * per_token + i];
        *reinterpret_cast<uint4 *>(k_cache + dst) = kv;
        *reinterpret_cast<uint4 *>(v_cache + dst) = vv;
    }
}

// INT8 cache write ("KV Cache从原理到实战" §5.2, per-channel scales): one CTA
// per new token; a thread quantises 8 channels of one head of K and of V
// (one 16-byte input vector -> 8 codes) with those channels' scales.
template <typename T>
__global__ void __launch_bounds__(256) reshape_and_cache_int8_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int64_t *__restrict__ slot_mapping, int8_t *__restrict__ k_cache,
    int8_t *__restrict__ v_cache, const float *__restrict__ k_scale,
    const float *__restrict__ v_scale, int64_t num_slots, int64_t block_stride, int num_kv_heads,
    int head_dim, int block_size, unsigned int *status) {
    const int64_t n = blockIdx.x;
    const int64_t slot = slot_mapping[n];
    if (slot < 0) return;  // padding token
    if (slot >= num_slots) {
        if (threadIdx.x == 0) pkv::raise_flag(status, PKV_DEVERR_SLOT);
        return;
    }
    const int64_t blk = slot / block_size;
    const int off = static_cast<int>(slot % block_size);
    const int chunks = head_dim / 8;
    const int per_token = num_kv_heads * chunks;
    for (int i = threadIdx.x; i < per_token; i += blockDim.x) {
        const int h = i / chunks;
        const int c = i - h * chunks;
        const int64_t dst = blk * block_stride + (static_cast<int64_t>(h) * block_size + off) * head_dim + c * 8;
        const int sc = h * head_dim + c * 8;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint4 x = (half ? v_new : k_new)[n * per_token + i];
            const float4 *s4 = reinterpret_cast<const float4 *>((half ? v_scale : k_scale) + sc);
            const float4 sa = s4[0], sb = s4[1];
            const float s[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
            float f[8];
            pkv::Elem<T>::to_f32x8(x, f);
            uint32_t w[2] = {0u, 0u};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                w[e / 4] |= (static_cast<uint32_t>(pkv::quantize_int8(f[e], s[e])) & 0xffu) << (8 * (e % 4));
            *reinterpret_cast<uint2 *>((half ? v_cache : k_cache) + dst) = make_uint2(w[0], w[1]);
        }
    }
}

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

// grid.x = pair, grid.y = chunk of kCopyThreads*kCopyUnroll vectors, grid.z = K (0) / V (1).
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    char *__restrict__ k_cache, char *__restrict__ v_cache, int64_t num_blocks,
    int64_t block_stride_bytes, int64_t slice_vecs, const int64_t *__restrict__ pairs,
    unsigned int *status) {
    const int64_t p = blockIdx.x;
    const int64_t src = pairs[2 * p];
    const int64_t dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
            pkv::raise_flag(status, PKV_DEVERR_COPY_PAIR);
        return;
    }
    char *base = blockIdx.z ? v_cache : k_cache;
    const uint4 *s = reinterpret_cast<const uint4 *>(base + src * block_stride_bytes);
    uint4 *d = reinterpret_cast<uint4 *>(base + dst * block_stride_bytes);
    const int64_t first = static_cast<int64_t>(blockIdx.y) * kCopyThreads * kCopyUnroll + threadIdx.x;
    uint4 buf[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = first + u * kCopyThreads;
        if (i < slice_vecs) buf[u] = s[i];
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = first + u * kCopyThreads;
        if (i < slice_vecs) d[i] = buf[u];
    }
}

// Slot rule of "KV Cache与PagedAttention深度解析" §5.3 for one token: position t
// of a sequence lies in the table entry t / block_size at offset t % block_size,
// and the flat slot is entry * block_size + offset.  A negative position is
// padding (slot -1).  Returns the PKV_DEVERR_* flag of a bad input (its slot is
// -1 too) or 0.  Shared by the device kernel and the host entry point.
__host__ __device__ inline unsigned int slot_of(const int32_t *table_row, int max_blocks_per_seq,
                                                int64_t pos, int block_size, int64_t num_blocks,
                                                int64_t *slot) {
    *slot = -1;
    if (pos < 0) return 0;
    const int64_t entry = pos / block_size;
    if (entry >= max_blocks_per_seq) return PKV_DEVERR_SLOT;
    const int64_t blk = table_row[entry];
    if (blk < 0 || blk >= num_blocks) return PKV_DEVERR_BLOCK_TABLE;
    *slot = blk * block_size + pos % block_size;
    return 0;
}

// One thread per token; token i reads table row token_rows[i] (or row i).
__global__ void __launch_bounds__(256) slot_mapping_kernel(
    const int32_t *__restrict__ block_tables, int64_t num_table_rows, int max_blocks_per_seq,
    const int64_t *__restrict__ token_rows, const int64_t *__restrict__ positions,
    int64_t num_tokens, int block_size, int64_t num_blocks, int64_t *__restrict__ slot_mapping,
    unsigned int *status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= num_tokens) return;
    const int64_t row = token_rows ? token_rows[i] : i;
    int64_t slot = -1;
    unsigned int flag = PKV_DEVERR_SLOT;  // a token row outside the table
    if (row >= 0 && row < num_table_rows)
        flag = slot_of(block_tables + row * max_blocks_per_seq, max_blocks_per_seq, positions[i],
                       block_size, num_blocks, &slot);
    if (flag) pkv::raise_flag(status, flag);
    slot_mapping[i] = slot;
}

bool supported_shape(int head_dim, int block_size) {
    return (head_dim == 64 || head_dim == 128) &&
           (block_size == 8 || block_size == 16 || block_size == 32);
}

}  // namespace

extern "C" {

PKV_API pkv_status pkv_reshape_and_cache(const void *k_new, const void *v_new,
                                         const int64_t *slot_mapping, int64_t num_tokens,
                                         void *k_cache, void *v_cache, int64_t num_blocks,
                                         int64_t block_stride_elems, int num_kv_heads,
                                         int head_dim, int block_size, pkv_dtype dtype,
                                         void *stream) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (!supported_shape(head_dim, block_size)) return PKV_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    const int64_t half_elems = static_cast<int64_t>(num_kv_heads) * block_size * head_dim;
    if (block_stride_elems < half_elems || block_stride_elems % 8) return PKV_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !pkv::aligned16(k_new) || !pkv::aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_INVALID_ARG;
    unsigned int *status = pkv::status_word_ptr();
    if (!status) return PKV_ERR_CUDA;
    const int row_vecs = head_dim * 2 / 16;
    const int per_token = num_kv_heads * row_vecs;
    const int threads = per_token < 256 ? ((per_token + 31) / 32) * 32 : 256;
    reshape_and_cache_kernel<<<static_cast<unsigned>(num_tokens), threads, 0,
                               static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping,
        static_cast<char *>(k_cache), static_cast<char *>(v_cache), num_blocks * block_size,
        block_stride_elems * 2, num_kv_heads, row_vecs, block_size, status);
    pkv::count_launch();
    return pkv::launch_status();
}

PKV_API pkv_status pkv_reshape_and_cache_int8(const void *k_new, const void *v_new,
                                              const int64_t *slot_mapping, int64_t num_tokens,
                                              int8_t *k_cache, int8_t *v_cache, int64_t num_blocks,
                                              int64_t block_stride_elems, int num_kv_heads,
                                              int head_dim, int block_size, const float *k_scale,
                                              const float *v_scale, pkv_dtype dtype, void *stream) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (!supported_shape(head_dim, block_size)) return PKV_ERR_UNSUPPORTED;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    const int64_t half_elems = static_cast<int64_t>(num_kv_heads) * block_size * head_dim;
    if (block_stride_elems < half_elems || block_stride_elems % 16) return PKV_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_scale || !v_scale || !pkv::aligned16(k_new) ||
        !pkv::aligned16(v_new) || !pkv::aligned16(k_scale) || !pkv::aligned16(v_scale) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_INVALID_ARG;
    unsigned int *status = pkv::status_word_ptr();
    if (!status) return PKV_ERR_CUDA;
    const int per_token = num_kv_heads * (head_dim / 8);
    const int threads = per_token < 256 ? ((per_token + 31) / 32) * 32 : 256;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned grid = static_cast<unsigned>(num_tokens);
    if (dtype == PKV_F16)
        reshape_and_cache_int8_kernel<__half><<<grid, threads, 0, s>>>(
            static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping,
            k_cache, v_cache, k_scale, v_scale, num_blocks * block_size, block_stride_elems,
            num_kv_heads, head_dim, block_size, status);
    else
        reshape_and_cache_int8_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(
            static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping,
            k_cache, v_cache, k_scale, v_scale, num_blocks * block_size, block_stride_elems,
            num_kv_heads, head_dim, block_size, status);
    pkv::count_launch();
    return pkv::launch_status();
}

PKV_API pkv_status pkv_slot_mapping(const int32_t *block_tables, int64_t num_table_rows,
                                    int max_blocks_per_seq, const int64_t *token_rows,
                                    const int64_t *positions, int64_t num_tokens, int block_size,
                                    int64_t num_blocks, int64_t *slot_mapping, void *stream) {
    if (num_tokens < 0 || num_table_rows < 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (!token_rows && num_table_rows < num_tokens) return PKV_ERR_INVALID_ARG;
    if ((num_tokens + 255) / 256 > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!block_tables || !positions || !slot_mapping) return PKV_ERR_INVALID_ARG;
    unsigned int *status = pkv::status_word_ptr();
    if (!status) return PKV_ERR_CUDA;
    slot_mapping_kernel<<<static_cast<unsigned>((num_tokens + 255) / 256), 256, 0,
                          static_cast<cudaStream_t>(stream)>>>(
        block_tables, num_table_rows, max_blocks_per_seq, token_rows, positions, num_tokens,
        block_size, num_blocks, slot_mapping, status);
    pkv::count_launch();
    return pkv::launch_status();
}

PKV_API pkv_status pkv_slot_mapping_host(const int32_t *block_tables, int64_t num_table_rows,
                                         int max_blocks_per_seq, const int64_t *token_rows,
                                         const int64_t *positions, int64_t num_tokens,
                                         int block_size, int64_t num_blocks,
                                         int64_t *slot_mapping) {
    if (num_tokens < 0 || num_table_rows < 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (!token_rows && num_table_rows < num_tokens) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!block_tables || !positions || !slot_mapping) return PKV_ERR_INVALID_ARG;
    bool bad = false;
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t row = token_rows ? token_rows[i] : i;
        int64_t slot = -1;
        if (row >= 0 && row < num_table_rows) {
            if (slot_of(block_tables + row * max_blocks_per_seq, max_blocks_per_seq, positions[i],
                        block_size, num_blocks, &slot))
                bad = true;
        } else {
            bad = true;
        }
        slot_mapping[i] = slot;
    }
    return bad ? PKV_ERR_INVALID_ARG : PKV_OK;
}

PKV_API pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, int64_t num_blocks,
                                   int64_t block_stride_elems, int num_kv_heads, int head_dim,
                                   int block_size, const int64_t *src_dst_pairs,
                                   int64_t num_pairs, pkv_dtype dtype, void *stream) {
    if (dtype != PKV_F16 && dtype != PKV_BF16 && dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
    if (!supported_shape(head_dim, block_size)) return PKV_ERR_UNSUPPORTED;
    if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (num_pairs > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    const int elem_bytes = dtype == PKV_INT8 ? 1 : 2;
    const int64_t half_elems = static_cast<int64_t>(num_kv_heads) * block_size * head_dim;
    if (block_stride_elems < half_elems || (block_stride_elems * elem_bytes) % 16)
        return PKV_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!src_dst_pairs || (reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u))
        return PKV_ERR_INVALID_ARG;
    unsigned int *status = pkv::status_word_ptr();
    if (!status) return PKV_ERR_CUDA;
    const int64_t slice_vecs = half_elems * elem_bytes / 16;
    const int64_t chunks = (slice_vecs + kCopyThreads * kCopyUnroll - 1) / (kCopyThreads * kCopyUnroll);
    if (chunks > 65535) return PKV_ERR_INVALID_ARG;
    dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(chunks), 2);
    copy_blocks_kernel<<<grid, kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<char *>(k_cache), static_cast<char *>(v_cache), num_blocks,
        block_stride_elems * elem_bytes, slice_vecs, src_dst_pairs, status);
    pkv::count_launch();
    return pkv::launch_status();
}

}  // extern "C"
