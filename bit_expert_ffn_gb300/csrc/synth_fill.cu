// synth_fill.cu -- device side of the seeded input generator (built into
// libmoe_synth.so, not into the product library).  It holds none of the
// layer's arithmetic: it only draws the synthetic codes, scales, weights and
// activations that the multi-gigabyte workloads need, with the same
// counter-based definition as bit_expert_ffn_gb300/synth.py:
//
//   mix64(z): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
//             z *= 0x94D049BB133111EB; z ^= z >> 31     (SplitMix64 output,
//             Steele, Lea and Flood, OOPSLA 2014)
//   u64(key, i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
//   code(i)     = top `bits` bits of u64(key, i)
//   normal(i)   = f32(S - 262140) * scale, S the sum of the eight 16-bit
//                 halves of u64(key, 2i) and u64(key, 2i+1) (Irwin-Hall),
//                 one fp32 multiply with round-to-nearest-even; the host
//                 passes `scale` so both sides use the identical constant.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t u64(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull); }

__device__ __forceinline__ float normal(uint64_t key, uint64_t i, float scale)
{
    uint64_t a = u64(key, 2 * i), b = u64(key, 2 * i + 1);
    int s = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) s += (int)((a >> (16 * j)) & 0xFFFF) + (int)((b >> (16 * j)) & 0xFFFF);
    return __fmul_rn(__int2float_rn(s - 262140), scale);
}

__device__ __forceinline__ uint16_t bf16_rne(float f)
{
    uint32_t u = __float_as_uint(f);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

__global__ void codes_kernel(uint64_t key, uint64_t start, int64_t n, int bits, uint8_t *out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)(u64(key, start + i) >> (64 - bits));
}

// kind 0: fp32 N(0, sigma); 1: bf16 N(0, sigma); 2: fp16 |N(0, sigma)|
__global__ void normal_kernel(uint64_t key, uint64_t start, int64_t n, float scale, float sigma, int kind, void *out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float v = __fmul_rn(normal(key, start + i, scale), sigma);
        if (kind == 0) static_cast<float *>(out)[i] = v;
        else if (kind == 1) static_cast<uint16_t *>(out)[i] = bf16_rne(v);
        else static_cast<uint16_t *>(out)[i] = __half_as_ushort(__float2half_rn(fabsf(v)));
    }
}

int grid_for(int64_t n)
{
    int64_t b = (n + 255) / 256;
    return (int)(b < 65536 ? (b > 0 ? b : 1) : 65536);
}

}  // namespace

extern "C" int moe_synth_codes(uint64_t key, uint64_t start, int64_t n, int bits, uint8_t *out, cudaStream_t s)
{
    if (n <= 0) return 0;
    codes_kernel<<<grid_for(n), 256, 0, s>>>(key, start, n, bits, out);
    return (int)cudaGetLastError();
}

extern "C" int moe_synth_normal(uint64_t key, uint64_t start, int64_t n, float scale, float sigma, int kind, void *out,
                                cudaStream_t s)
{
    if (n <= 0) return 0;
    normal_kernel<<<grid_for(n), 256, 0, s>>>(key, start, n, scale, sigma, kind, out);
    return (int)cudaGetLastError();
}
