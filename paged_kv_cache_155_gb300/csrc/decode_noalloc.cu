// decode_noalloc.cu -- paged decode for callers that cannot allocate device
// memory.
//
// pkv_paged_attention_decode needs a caller-provided workspace whenever a
// sequence is split into several context partitions.  Some callers have no
// way to provide one: a serving engine that reserved (nearly) all free device
// memory for its KV block pool at start-up has nothing left to hand out per
// call, and a plug-in that its host framework gives only tensor pointers has
// no device allocator it is allowed to call.  This entry point serves them: it
// takes its split-context scratch from a fixed array inside the library.
//
// The array is a file-scope __device__ array of PKV_STATIC_SCRATCH_BYTES.  Every
// device that loads the library holds one for the life of the process.  Host
// code cannot use the array's name as a device address, so the first call on
// each device (with that device current) looks up the real address with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls on a device share the one array and it keeps whatever
// the last call left there: the decode kernels write every scratch value before
// they read it, so nothing needs clearing between calls, but two calls that
// run at the same time on the GPU (different streams, no ordering between
// them) race on it.
#include <mutex>

#include "pkv_host.h"

namespace {

__device__ __align__(256) unsigned char g_static_decode_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices];

// Device address of the current device's scratch array (nullptr on failure).
void *static_scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *addr = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&addr, g_static_decode_scratch);
        if (err != cudaSuccess || !addr) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_addr[dev] = addr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

PKV_API pkv_status pkv_paged_attention_decode_static_scratch(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    int64_t block_stride_elems, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, float scale, void *out, int partition_size,
    pkv_dtype dtype, void *stream) {
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                   head_dim, block_size, max_context_len,
                                                   partition_size);
    void *scratch = nullptr;
    if (need != static_cast<size_t>(-1)) {
        if (need > PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_SCRATCH_LIMIT;
        if (need > 0) {
            scratch = static_scratch_address();
            if (!scratch) return PKV_ERR_CUDA;
        }
    }
    // Arguments that failed the size query are rejected by the call below with
    // the same status the workspace-taking entry point gives them.
    return pkv_paged_attention_decode(q, k_cache, v_cache, num_blocks, block_stride_elems,
                                      block_tables, max_blocks_per_seq, context_lens,
                                      max_context_len, num_seqs, num_q_heads, num_kv_heads,
                                      head_dim, block_size, scale, out, scratch,
                                      scratch ? PKV_STATIC_SCRATCH_BYTES : 0, partition_size,
                                      dtype, stream);
}

}  // extern "C"
