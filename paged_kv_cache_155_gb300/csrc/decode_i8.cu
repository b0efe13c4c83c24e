// decode_i8.cu -- instantiations of the paged decode kernels over an
// INT8 cache (per-channel scales), for fp16 and bf16 queries.
#include "decode_launch.cuh"

namespace pkv {
pkv_status launch_decode_i8_f16(const DecodeParams &p, const DecodeMaps &m, int head_dim, int block_size, int gh,
                                dim3 grid, int merge_rows, cudaStream_t s) {
    return launch_decode_typed<__half, int8_t>(p, m, head_dim, block_size, gh, grid, merge_rows, s);
}
pkv_status launch_decode_i8_bf16(const DecodeParams &p, const DecodeMaps &m, int head_dim, int block_size, int gh,
                                 dim3 grid, int merge_rows, cudaStream_t s) {
    return launch_decode_typed<__nv_bfloat16, int8_t>(p, m, head_dim, block_size, gh, grid,
                                                      merge_rows, s);
}
}  // namespace pkv
