// common.cuh -- internal helpers shared by the library's translation units:
// status/message plumbing, argument checks, device status words and the
// number-format conversions the kernels use.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>

#include "moe_gb300.h"

namespace moe {

// ---------------------------------------------------------------- host side

// Sets the thread-local message of the last non-OK status and returns `s`.
moe_status fail(moe_status s, const char *fmt, ...);

inline cudaStream_t to_cuda(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Launch-error check after a kernel launch.
moe_status check_launch(const char *what);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline double mib(double bytes) { return bytes / (1024.0 * 1024.0); }

// Round up to a multiple of 256 bytes (workspace sub-allocation).
inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

#define MOE_REQUIRE(cond, ...)                                                 \
    do {                                                                       \
        if (!(cond)) return ::moe::fail(MOE_ERR_INVALID_ARG, __VA_ARGS__);     \
    } while (0)

#define MOE_CUDA_TRY(call)                                                               \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess)                                                           \
            return ::moe::fail(MOE_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_));   \
    } while (0)

// Number of SMs of the current device (cached per device).
int sm_count();

// ---------------------------------------------------------------- device side

// First error wins: a status word is only written while it is still 0.
__device__ __forceinline__ void set_status(int32_t *st, int32_t code)
{
    if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Round-to-nearest-even fp32 -> bf16 (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return uint16_t((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

__device__ __forceinline__ float fp16_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

}  // namespace moe
