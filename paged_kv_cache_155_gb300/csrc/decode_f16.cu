// decode_f16.cu -- fp16 instantiations of the paged decode kernels.
#include "decode_launch.cuh"

namespace pkv {
pkv_status launch_decode_f16(const DecodeParams &p, const DecodeMaps &m, int head_dim, int block_size, int gh,
                             dim3 grid, int merge_rows, cudaStream_t s) {
    return launch_decode_typed<__half>(p, m, head_dim, block_size, gh, grid, merge_rows, s);
}
pkv_status launch_prefix_tc_f16(const PrefixParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                                int block_size, dim3 grid, cudaStream_t s) {
    return launch_prefix_tc_typed<__half>(p, tk, tv, block_size, grid, s);
}
}  // namespace pkv
