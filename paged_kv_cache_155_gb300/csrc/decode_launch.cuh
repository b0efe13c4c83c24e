// decode_launch.cuh -- host-side dispatch from runtime (head_dim, block_size,
// heads per block) to the decode kernel instantiations of one element type.
// Included by decode_f16.cu and decode_bf16.cu so the two element types
// compile as separate translation units.
#pragma once

#include <atomic>
#include <utility>

#include "decode_kernel.cuh"
#include "prefix_tc_kernel.cuh"
#include "pkv_host.h"

namespace pkv {

// Launch `kernel` on `stream`; with `overlap`, as a programmatic dependent launch:
// it may start while the kernel before it in the stream still runs, once every
// CTA of that kernel has executed pdl_trigger (and must order itself after that
// kernel with pdl_wait where it needs to).
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool overlap, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename T, typename KT, int D, int BS, int GH>
pkv_status launch_decode_one(const DecodeParams &p, const DecodeMaps &maps, dim3 grid, cudaStream_t stream,
                             bool overlap) {
    using G = DecodeGeom<D, BS, sizeof(KT), decode_lane_values<KT, GH>(), (GH >= 4), (GH == 16)>;
    static std::atomic<uint64_t> configured_devices{0};  // bit per device ordinal
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured_devices.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(paged_decode_kernel<T, KT, D, BS, GH>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 G::kSmemBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_devices.fetch_or(bit, std::memory_order_acq_rel);
    }
    if (launch_kernel(paged_decode_kernel<T, KT, D, BS, GH>, grid, dim3(G::kWarps * 32),
                      G::kSmemBytes, stream, overlap, maps.k, maps.v, p) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    count_launch();
    return launch_status();
}

template <typename T, typename KT, int D, int BS>
pkv_status launch_decode_gh(const DecodeParams &p, const DecodeMaps &m, int gh, dim3 grid,
                            cudaStream_t s, bool overlap) {
    switch (gh) {
        case 1: return launch_decode_one<T, KT, D, BS, 1>(p, m, grid, s, overlap);
        case 2: return launch_decode_one<T, KT, D, BS, 2>(p, m, grid, s, overlap);
        case 4: return launch_decode_one<T, KT, D, BS, 4>(p, m, grid, s, overlap);
        case 8: return launch_decode_one<T, KT, D, BS, 8>(p, m, grid, s, overlap);
        case 16:
            // 16 heads per block: the 16-bit warp-MMA form at head_dim 128
            if constexpr (sizeof(KT) == 2 && D == 128) return launch_decode_one<T, KT, D, BS, 16>(p, m, grid, s, overlap);
            break;
    }
    return PKV_ERR_UNSUPPORTED;
}

// T: query / output type; KT: cache storage type (T, or int8_t).  The decode
// kernel overlaps the kernel before it when p.wait_prior_grid is set; the merge
// (when merge_rows > 0) always starts behind the decode kernel as its
// programmatic dependent and waits for its partials.
template <typename T, typename KT = T>
pkv_status launch_decode_typed(const DecodeParams &p, const DecodeMaps &m, int head_dim,
                               int block_size, int gh, dim3 grid, int merge_rows, cudaStream_t s) {
    pkv_status st = PKV_ERR_UNSUPPORTED;
    const bool overlap = p.wait_prior_grid != 0;
    if (head_dim == 128) {
        if (block_size == 8) st = launch_decode_gh<T, KT, 128, 8>(p, m, gh, grid, s, overlap);
        else if (block_size == 16) st = launch_decode_gh<T, KT, 128, 16>(p, m, gh, grid, s, overlap);
        else if (block_size == 32) st = launch_decode_gh<T, KT, 128, 32>(p, m, gh, grid, s, overlap);
    } else if (head_dim == 64) {
        if (block_size == 8) st = launch_decode_gh<T, KT, 64, 8>(p, m, gh, grid, s, overlap);
        else if (block_size == 16) st = launch_decode_gh<T, KT, 64, 16>(p, m, gh, grid, s, overlap);
        else if (block_size == 32) st = launch_decode_gh<T, KT, 64, 32>(p, m, gh, grid, s, overlap);
    }
    if (st != PKV_OK || merge_rows == 0) return st;
    // four warps share a row once a row has many partitions (their loads in flight
    // together instead of one warp's rounds of them)
    const bool wide = p.num_partitions >= kMergeWideFrom;
    const unsigned blocks = static_cast<unsigned>(wide ? merge_rows : (merge_rows + 3) / 4);
    cudaError_t err;
    if (head_dim == 128)
        err = wide ? launch_kernel(paged_decode_merge_kernel<T, 128, 4>, dim3(blocks), dim3(128), 0, s, true, p, merge_rows)
                   : launch_kernel(paged_decode_merge_kernel<T, 128, 1>, dim3(blocks), dim3(128), 0, s, true, p, merge_rows);
    else
        err = wide ? launch_kernel(paged_decode_merge_kernel<T, 64, 4>, dim3(blocks), dim3(128), 0, s, true, p, merge_rows)
                   : launch_kernel(paged_decode_merge_kernel<T, 64, 1>, dim3(blocks), dim3(128), 0, s, true, p, merge_rows);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    count_launch();
    return launch_status();
}

template <typename T, int BS>
pkv_status launch_prefix_tc_one(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                                dim3 grid, cudaStream_t stream) {
    static std::atomic<uint64_t> configured_devices{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured_devices.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(paged_prefix_tc_kernel<T, BS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PrefixLayout::kSmemBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_devices.fetch_or(bit, std::memory_order_acq_rel);
    }
    paged_prefix_tc_kernel<T, BS><<<grid, PrefixLayout::kThreads, PrefixLayout::kSmemBytes, stream>>>(tk, tv, p);
    count_launch();
    return launch_status();
}

template <typename T>
pkv_status launch_prefix_tc_typed(const PrefixParams &p, const CUtensorMap &tk,
                                  const CUtensorMap &tv, int block_size, dim3 grid, cudaStream_t s) {
    if (block_size == 8) return launch_prefix_tc_one<T, 8>(p, tk, tv, grid, s);
    if (block_size == 16) return launch_prefix_tc_one<T, 16>(p, tk, tv, grid, s);
    if (block_size == 32) return launch_prefix_tc_one<T, 32>(p, tk, tv, grid, s);
    return PKV_ERR_UNSUPPORTED;
}

// Defined in decode_f16.cu / decode_bf16.cu (16-bit caches) and
// decode_i8.cu (INT8 cache, fp16 or bf16 queries).
pkv_status launch_decode_f16(const DecodeParams &p, const DecodeMaps &m, int head_dim,
                             int block_size, int gh, dim3 grid, int merge_rows, cudaStream_t s);
pkv_status launch_decode_i8_f16(const DecodeParams &p, const DecodeMaps &m, int head_dim,
                                int block_size, int gh, dim3 grid, int merge_rows, cudaStream_t s);
pkv_status launch_decode_i8_bf16(const DecodeParams &p, const DecodeMaps &m, int head_dim,
                                 int block_size, int gh, dim3 grid, int merge_rows, cudaStream_t s);
pkv_status launch_decode_bf16(const DecodeParams &p, const DecodeMaps &m, int head_dim,
                              int block_size, int gh, dim3 grid, int merge_rows, cudaStream_t s);
pkv_status launch_prefix_tc_f16(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                                int block_size, dim3 grid, cudaStream_t s);
pkv_status launch_prefix_tc_bf16(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                                 int block_size, dim3 grid, cudaStream_t s);

}  // namespace pkv
