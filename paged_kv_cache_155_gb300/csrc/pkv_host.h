// pkv_host.h -- host-side helpers shared by the libpagedkv translation units
// (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// Device address of the current device's status word (nullptr on failure).
unsigned int *status_word_ptr();

// Streaming-multiprocessor count of the current device (0 on failure).
int current_sm_count();

// Count one kernel launch made through the library.
void count_launch();

// Tiled tensor map of one half (K or V) of a 16-bit pool for 3-D TMA loads:
// dims (head_dim 128, num_kv_heads * block_size rows, num_blocks), boxes of
// box_rows rows of one head (0: a whole block's), 64 columns wide, 128-byte
// swizzled.  False if the driver entry point is missing or the encode fails.
bool encode_half_map(CUtensorMap *map, const void *base, int64_t num_blocks,
                     int64_t block_stride_elems, int num_kv_heads, int block_size, pkv_dtype dt,
                     int box_rows);

// Tiled tensor map of one half (K or V) of an INT8 pool with head_dim 128 for
// 3-D TMA loads: dims (128 codes, num_kv_heads * block_size rows, num_blocks),
// boxes of one block's rows of one head (128 bytes each), 128-byte swizzled.
bool encode_i8_half_map(CUtensorMap *map, const void *base, int64_t num_blocks,
                        int64_t block_stride_elems, int num_kv_heads, int block_size);

// Tiled tensor map of the prefill queries [num_rows][num_q_heads][128] for
// 3-D TMA loads: boxes of `tokens` tokens x `group` query heads x 64 columns,
// 128-byte swizzled (group <= 256, tokens <= 256).
bool encode_query_map(CUtensorMap *map, const void *q, int num_rows, int num_q_heads, int group,
                      int tokens, pkv_dtype dt);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline pkv_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
