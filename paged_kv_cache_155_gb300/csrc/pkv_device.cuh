// pkv_device.cuh -- device-side building blocks shared by the libpagedkv kernels:
// inline-PTX mbarrier and bulk-copy (TMA engine) wrappers, a wait with a time
// limit, and 16-bit <-> fp32 conversions.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// Upper bound of any wait on an asynchronous copy in the hot kernels.  A
// legitimate copy finishes in microseconds; after this the kernel raises
// PKV_DEVERR_TIMEOUT and returns instead of spinning forever.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
constexpr uint64_t kDrainTimeoutNs = 200000000ull;  // 0.2 s, for the clean-up waits

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same buffers.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking probe of phase `parity` (for event loops that poll several
// barriers: a try_wait may hold the thread for a while on an incomplete phase,
// delaying the check of a barrier that is already complete).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after timeout_ns.
// Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// L2 policy for data read once (the streamed KV tiles).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for data several CTAs read (a shared prefix).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk (non-tensor) copy global -> this CTA's shared memory on the TMA engine;
// completion is signalled as `bytes` of transaction count on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch.  pdl_trigger: this CTA no longer holds back
// the next kernel of the stream if that kernel was launched with programmatic
// stream serialisation (it may start on free SMs while this grid runs).
// pdl_wait: block until the grids this one was launched behind have completed
// and their memory is visible.  Both are no-ops without such a launch.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) / min(a, b, c) in one instruction (sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (d0, d1) = (a0, a1) * (b0, b1) + (d0, d1) as one packed fp32 FMA (sm_100 and later).
__device__ __forceinline__ void fma_f32x2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rd, {%0, %1};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (a0, a1) += (b0, b1) as one packed fp32 add (sm_100 and later).
__device__ __forceinline__ void add_f32x2(float &a0, float &a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%0, %1};\n\t"
        "mov.b64 rb, {%2, %3};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}

__device__ __forceinline__ void raise_flag(unsigned int *status, unsigned int flag) {
    atomicOr(status, flag);
}

// Element traits: eight packed values (one Vec) -> fp32.
template <typename T>
struct Elem;

template <>
struct Elem<__half> {
    using Vec = uint4;
    static __device__ __forceinline__ void to_f32x8(const uint4 &u, float f[8]) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = __half22float2(h[i]);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
    static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
    // two values rounded to nearest even, packed low / high (one conversion)
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
};

template <>
struct Elem<__nv_bfloat16> {
    using Vec = uint4;
    // bf16 is the high half of an fp32 pattern: widening is a shift / mask.
    static __device__ __forceinline__ void to_f32x8(const uint4 &u, float f[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) {
        return __float2bfloat16_rn(x);
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
};

// INT8 codes of the quantised cache: eight codes (8 bytes) -> fp32, exactly.
// Each code, biased by 128 into [1, 255], is placed in the low mantissa bits
// of 2^23 (a byte permute) and the float 2^23 + 128 subtracted: two ALU ops
// per value instead of a conversion-unit I2F.
template <>
struct Elem<int8_t> {
    using Vec = uint2;
    static __device__ __forceinline__ void to_f32x8(const uint2 &u, float f[8]) {
        const uint32_t w[2] = {u.x ^ 0x80808080u, u.y ^ 0x80808080u};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                f[4 * i + j] = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7440u + j));
            // minus 2^23 + 128, two values per packed add (exact: integers below 2^24)
            add_f32x2(f[4 * i], f[4 * i + 1], -8388736.f, -8388736.f);
            add_f32x2(f[4 * i + 2], f[4 * i + 3], -8388736.f, -8388736.f);
        }
    }
};

// Four INT8 codes (one word) -> four exact fp16 values code + 1152 (two words):
// each code, biased by 128, goes into the low mantissa byte of 1024.0 (0x64xx).
// Sums over these values remove the offset once, as kCodeOffset times the sum
// of the other operand.
constexpr float kCodeOffset = 1152.f;
__device__ __forceinline__ void codes_to_f16x4_offset(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t b = w ^ 0x80808080u;
    lo = __byte_perm(b, 0x64646464u, 0x4140u);
    hi = __byte_perm(b, 0x64646464u, 0x4342u);
}

// Byte E of x and byte E of y (two INT8 codes of one channel in two token rows)
// -> the exact fp16 pair (x_E + 1152, y_E + 1152): a byte permute puts the two
// codes in the low bytes of the two halves, and one three-input logic op flips
// their sign bits (code + 128) and sets both high bytes to 0x64.
template <int E>
__device__ __forceinline__ uint32_t token_pair_f16_offset(uint32_t x, uint32_t y) {
    constexpr uint32_t sel = E | (E << 4) | ((E + 4) << 8) | ((E + 4) << 12);
    const uint32_t r = __byte_perm(x, y, sel);
    uint32_t out;
    // bits of 0x647F647F pass r, bits of 0x64806480 invert it, both set -> 1
    asm("lop3.b32 %0, %1, %2, %3, 0xCA;" : "=r"(out) : "r"(r), "r"(0x647F647Fu), "r"(0x64806480u));
    return out;
}

// Warp-level MMA m16n8k16, fp16 (or bf16) operands, fp32 accumulators (d += a b):
// a0 / a2 = row g, k 2t..2t+1 / 2t+8..2t+9; a1 / a3 the same for row g + 8;
// b0 / b1 = k 2t..2t+1 / 2t+8..2t+9 of column g; d0, d1 = row g, columns
// 2t, 2t+1; d2, d3 = row g + 8 (g = lane / 4, t = lane % 4).
template <bool kBF16 = false>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    if constexpr (kBF16)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8 x 8 matrix of 16-bit values held by a warp: lane i holds
// row i / 4, columns 2 (i % 4) and 2 (i % 4) + 1 (low half first), before and after.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// Two floats -> one word of two fp16 (or bf16) values, the first in the low half;
// ra / rb receive the two rounded values.
template <bool kBF16>
__device__ __forceinline__ uint32_t pack_mma2(float a, float b, float &ra, float &rb) {
    if constexpr (kBF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        ra = __low2float(h);
        rb = __high2float(h);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        ra = __low2float(h);
        rb = __high2float(h);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

// Exponent e with |m| * 2^-e in [1/2, 1) for a finite m > 0 (e = 0 otherwise),
// clamped so that 2^e and 2^-e are normal floats.
__device__ __forceinline__ int row_exponent(float m) {
    if (!(m > 0.f) || !(m < INFINITY)) return 0;
    const int biased = static_cast<int>((__float_as_uint(m) >> 23) & 0xffu);
    const int e = (biased == 0 ? 1 : biased) - 126;
    return e < -125 ? -125 : (e > 126 ? 126 : e);
}

__device__ __forceinline__ float exp2_int(int e) {  // 2^e, e in [-126, 127]
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// (d0, d1) += (a.lo * b.lo, a.hi * b.hi) for two fp16 pairs, fp32 accumulators:
// mixed-precision FMAs (fp16 operands, fp32 addend and result, one rounding;
// the product of two fp16 values is exact in fp32).
__device__ __forceinline__ void fma_f16x2_f32(uint32_t a, uint32_t b, float &d0, float &d1) {
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(a), "r"(b));
}

// Per-channel INT8 quantiser ("KV Cache从原理到实战" §5.2): x / s in IEEE single
// precision (correctly rounded division), clamped to [-127, 127] -- a NaN
// quotient clamps to -127, since fmaxf returns the non-NaN operand -- then
// rounded to the nearest integer, ties to even.
__device__ __forceinline__ int quantize_int8(float x, float s) {
    float r = __fdiv_rn(x, s);
    r = fmaxf(r, -127.f);
    r = fminf(r, 127.f);
    return __float2int_rn(r);
}

}  // namespace pkv
