// decode_tc_i8.cu -- launches of the INT8-cache tensor-core decode kernel
// (fp16 and bf16 queries; block size 8, 16, 32; 4, 8 or 16 heads per KV head).
#include <atomic>

#include "decode_tc_i8_kernel.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

template <typename T, int BS, int GH>
pkv_status launch_one(const DecodeParams &p, int grid, cudaStream_t stream) {
    static std::atomic<uint64_t> configured_devices{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured_devices.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(paged_decode_tc_i8_kernel<T, BS, GH>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcI8Layout::kSmemBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_devices.fetch_or(bit, std::memory_order_acq_rel);
    }
    paged_decode_tc_i8_kernel<T, BS, GH>
        <<<grid, TcI8Layout::kThreads, TcI8Layout::kSmemBytes, stream>>>(p);
    count_launch();
    return launch_status();
}

template <typename T, int BS>
pkv_status launch_gh(const DecodeParams &p, int gh, int grid, cudaStream_t s) {
    switch (gh) {
        case 4: return launch_one<T, BS, 4>(p, grid, s);
        case 8: return launch_one<T, BS, 8>(p, grid, s);
        case 16: return launch_one<T, BS, 16>(p, grid, s);
    }
    return PKV_ERR_UNSUPPORTED;
}

template <typename T>
pkv_status launch_typed(const DecodeParams &p, int block_size, int gh, int grid, int merge_rows,
                        cudaStream_t s) {
    pkv_status st = PKV_ERR_UNSUPPORTED;
    if (block_size == 8) st = launch_gh<T, 8>(p, gh, grid, s);
    else if (block_size == 16) st = launch_gh<T, 16>(p, gh, grid, s);
    else if (block_size == 32) st = launch_gh<T, 32>(p, gh, grid, s);
    if (st != PKV_OK || merge_rows == 0) return st;
    const unsigned blocks = static_cast<unsigned>((merge_rows + 3) / 4);
    paged_decode_merge_kernel<T, 128><<<blocks, 128, 0, s>>>(p, merge_rows);
    count_launch();
    return launch_status();
}

}  // namespace

pkv_status launch_decode_tc_i8(const DecodeParams &p, pkv_dtype dtype, int block_size, int gh,
                               int grid, int merge_rows, cudaStream_t s) {
    return dtype == PKV_F16 ? launch_typed<__half>(p, block_size, gh, grid, merge_rows, s)
                            : launch_typed<__nv_bfloat16>(p, block_size, gh, grid, merge_rows, s);
}

}  // namespace pkv
