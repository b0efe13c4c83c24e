// api.cu -- library-wide state and the small entry points of libpagedkv:
// the device status word, its read-back, status strings, the launch counter,
// device-attribute caches and the bounded-wait self test.
#include <atomic>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace {

// One status word per device (a __device__ variable has one instance per
// device context).  Kernels OR PKV_DEVERR_* flags into it.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned int *g_status_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];
std::atomic<uint64_t> g_launches{0};

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

__global__ void wait_timeout_kernel(uint64_t timeout_ns, unsigned int *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        pkv::mbar_init(&bar, 1);
        pkv::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the wait must run out and report it.
        if (!pkv::mbar_wait_bounded(&bar, 0, timeout_ns)) pkv::raise_flag(status, PKV_DEVERR_TIMEOUT);
    }
}

}  // namespace

namespace pkv {

unsigned int *status_word_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    return g_status_ptr[dev];
}

int current_sm_count() {
    const int dev = current_device();
    if (dev < 0) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace pkv

extern "C" {

PKV_API pkv_status pkv_get_device_error(void *stream, uint32_t *flags) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int *word = pkv::status_word_ptr();
    if (!word) return PKV_ERR_CUDA;
    unsigned int value = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyAsync(&value, word, sizeof(value), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(word, 0, sizeof(value), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (flags) *flags = value;
    return value ? PKV_ERR_DEVICE : PKV_OK;
}

PKV_API const char *pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or block_size";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_DEVICE: return "a kernel raised a device status flag";
        case PKV_ERR_SCRATCH_LIMIT:
            return "split-context scratch needed exceeds the library's static scratch array";
        case PKV_ERR_OUT_OF_BLOCKS: return "out of KV cache blocks";
    }
    return "unknown status";
}

PKV_API uint64_t pkv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

PKV_API pkv_status pkv_debug_wait_timeout(uint64_t timeout_ns, void *stream) {
    if (timeout_ns == 0 || timeout_ns > 10000000000ull) return PKV_ERR_INVALID_ARG;
    unsigned int *word = pkv::status_word_ptr();
    if (!word) return PKV_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns, word);
    pkv::count_launch();
    return pkv::launch_status();
}

}  // extern "C"
