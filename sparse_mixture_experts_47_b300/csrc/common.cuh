// Shared device helpers of the MoE layer library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Device error word: set by a kernel whose bounded wait gave up or that met
// an out-of-range index; read and cleared by moe_device_status().  The
// library is one translation unit (moe_api.cu includes every kernel file),
// so this definition is the only one.
__device__ int g_error_word;

constexpr int kErrTimeout = 1;

// Iteration limit of every spin wait (an mbarrier try_wait loop); about
// seconds of polling at most, far beyond any legitimate wait.
constexpr uint32_t kSpinLimit = 1u << 26;

__device__ __forceinline__ void flag_error(int code) { atomicOr(&g_error_word, code); }

// Host-side count of kernels launched by the library (moe_kernel_launches).
inline long long g_kernel_launches = 0;
inline void note_launch() { __atomic_add_fetch(&g_kernel_launches, 1, __ATOMIC_RELAXED); }

template <typename T> struct Vec;   // 16-byte vector of T
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

// Load 16 bytes (N elements) starting at p and widen to fp32.
__device__ __forceinline__ void load16_f32(const float *p, float *v) {
    float4 a = *reinterpret_cast<const float4 *>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void load16_f32(const __nv_bfloat16 *p, float *v) {
    uint4 a = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ float to_f32(float a) { return a; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 a) { return __bfloat162float(a); }

template <typename T> __device__ __forceinline__ T from_f32(float a);
template <> __device__ __forceinline__ float from_f32<float>(float a) { return a; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float a) {
    return __float2bfloat16_rn(a);
}

__device__ __forceinline__ float silu(float a) { return a / (1.0f + __expf(-a)); }

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace moe
