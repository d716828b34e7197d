// Device-side helpers shared by the Talker kernels: PTX wrappers for mbarriers,
// bulk (TMA) copies and programmatic dependent launch, bf16 unpacking, warp
// reductions and the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace talker_dev {

// Bits of the device status word (talker_sync_status reports them).
enum : int {
    ST_BAD_POSITION = 1 << 0,   // a cache row at or past max_seq_len was requested
    ST_WAIT_TIMEOUT = 1 << 1,   // an mbarrier wait gave up after its time limit
    ST_NAN_LOGIT = 1 << 2,      // argmax met a NaN logit
    ST_BAD_ARG = 1 << 3,        // a kernel met arguments it cannot handle
};

constexpr int kPage = 64;                          // KV cache positions per page
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s bound on every mbarrier wait
// Bound for waits timed with the SM clock (reading %globaltimer costs ~800 cycles, so
// hot wait loops count SM cycles instead): 2^31 cycles, about 1 s at 2 GHz.
constexpr long long kWaitLimitCycles = 1ll << 31;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- programmatic dependent launch (no-ops when launched without the attribute)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// kWaitLimitNs. Returns false (and sets ST_WAIT_TIMEOUT) on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, ST_WAIT_TIMEOUT);
            return false;
        }
    }
}

// ---- bulk copies (the TMA engine, 1-D form): 16-byte aligned, size % 16 == 0
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---- loads
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---- explicit shared-memory loads (32-bit shared addresses), so the hot loops
// never fall back to generic addressing when pointers cross function boundaries
__device__ __forceinline__ uint4 lds_u4(uint32_t a) {
    uint4 v;
    asm("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
    unsigned short v;
    asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds_u2(uint32_t a) {
    uint2 v;
    asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

// ---- bf16 / f32 element helpers
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPerVec = 4;   // elements per 16-byte vector
    __device__ static __forceinline__ float round(float v) { return v; }
    __device__ static __forceinline__ float load(const float *p, size_t i) { return p[i]; }
    __device__ static __forceinline__ void store(float *p, size_t i, float v) { p[i] = v; }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ static __forceinline__ float round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
    __device__ static __forceinline__ float load(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
    __device__ static __forceinline__ void store(__nv_bfloat16 *p, size_t i, float v) {
        p[i] = __float2bfloat16_rn(v);
    }
};

__device__ __forceinline__ float warp_max_abs(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Q8_0 block (ggml layout, the talker's quantized KV storage): 32 values held one per lane of a
// warp (lane = position in the block). d = max|x| / 127, code = x * (1/d) rounded half away from
// zero (0 for an all-zero block); codes at t + code_off + lane, d as fp16 at t + scale_off.
__device__ __forceinline__ void q8_store_block(unsigned char *t, int code_off, int scale_off, float x, int lane) {
    const float amax = warp_max_abs(fabsf(x));
    const float d = amax / 127.0f;
    const float id = d > 0.f ? 1.0f / d : 0.f;
    reinterpret_cast<int8_t *>(t)[code_off + lane] = (int8_t)roundf(x * id);
    if (lane == 0) *reinterpret_cast<__half *>(t + scale_off) = __float2half_rn(d);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace talker_dev
