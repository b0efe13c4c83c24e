// cache_ops.cu -- the two byte-moving ops of the paged KV cache:
//   pkv_reshape_and_cache: scatter each new token's K/V rows into its slot
//     ("KV Cache与PagedAttention深度解析" §2.2 append step, §5.3 slot rule);
//   pkv_copy_blocks: copy-on-write copies of whole blocks (same page §8.3;
//     zwxr.cn nano-vllm article §2.3, §5.5).
// Both move 16-byte vectors and are bit-exact.  Device-resident indices are
// range-checked before use; a bad one raises a status flag and is skipped.
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

PKV_API pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, int64_t num_blocks,
                                   int64_t block_stride_elems, int num_kv_heads, int head_dim,
                                   int block_size, const int64_t *src_dst_pairs,
                                   int64_t num_pairs, pkv_dtype dtype, void *stream) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (!supported_shape(head_dim, block_size)) return PKV_ERR_UNSUPPORTED;
    if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (num_pairs > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
    const int64_t half_elems = static_cast<int64_t>(num_kv_heads) * block_size * head_dim;
    if (block_stride_elems < half_elems || block_stride_elems % 8) return PKV_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !pkv::aligned16(k_cache) || !pkv::aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    if (!src_dst_pairs || (reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u))
        return PKV_ERR_INVALID_ARG;
    unsigned int *status = pkv::status_word_ptr();
    if (!status) return PKV_ERR_CUDA;
    const int64_t slice_vecs = half_elems * 2 / 16;
    const int64_t chunks = (slice_vecs + kCopyThreads * kCopyUnroll - 1) / (kCopyThreads * kCopyUnroll);
    if (chunks > 65535) return PKV_ERR_INVALID_ARG;
    dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(chunks), 2);
    copy_blocks_kernel<<<grid, kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<char *>(k_cache), static_cast<char *>(v_cache), num_blocks,
        block_stride_elems * 2, slice_vecs, src_dst_pairs, status);
    pkv::count_launch();
    return pkv::launch_status();
}

}  // extern "C"
