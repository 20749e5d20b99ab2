// Device-side helpers shared by the kernels of libbi (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bi.h"

namespace bi {

// ---------------------------------------------------------------------------
// bf16 <-> fp32.  bf16 -> fp32 is exact (a shift); fp32 -> bf16 rounds to
// nearest even (cuda_bf16's conversion).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t packed) {
    return __uint_as_float(packed << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t packed) {
    return __uint_as_float(packed & 0xffff0000u);
}
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(f32_to_bf16(lo)) | (static_cast<uint32_t>(f32_to_bf16(hi)) << 16);
}

// ---------------------------------------------------------------------------
// Device status word: the first nonzero code wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Upper bound for any device-side wait (nanoseconds).  Every legitimate wait
// in these kernels is microseconds to a few milliseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------------------
// Loads that bypass L1 allocation for streamed data.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------------------
// Greedy argmax as a 64-bit key ("temperature=0 means deterministic").
// (value, index) pairs are totally ordered: a NaN beats every number, a
// larger number beats a smaller one, and between equal values (-0 equals +0)
// or two NaNs the lower index wins.  argmax_key maps a pair to an unsigned
// key whose minimum over a row is the winner, so the winner can be taken
// with atomicMin in any order and still be unique.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long argmax_key(float v, int32_t idx) {
    uint32_t hi = 0u;  // NaN
    if (!isnan(v)) {
        uint32_t b = __float_as_uint(v);
        if (b == 0x80000000u) b = 0u;
        const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);  // grows with v
        hi = ~ord;  // in [1, 0xfffffffe] for every number
    }
    return (static_cast<unsigned long long>(hi) << 32) | static_cast<uint32_t>(idx);
}
constexpr unsigned long long kArgmaxKeyNone = ~0ull;  // worse than every candidate

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of this library is launched so
// that it may start while the kernel before it in the stream is finishing:
// pdl_trigger() lets the next kernel start its own prologue, pdl_wait() blocks
// until every kernel ordered before this one has completed with its writes
// visible.  Each kernel runs pdl_wait() in every thread before it reads or
// writes global memory that another kernel touches, and before it exits, so
// completion of a kernel still implies completion of all earlier ones.  Both
// are no-ops when the launch carries no such dependency.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

}  // namespace bi
