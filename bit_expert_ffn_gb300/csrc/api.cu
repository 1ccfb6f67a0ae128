// api.cu -- status plumbing, size queries and small helpers of the C ABI.
#include <mutex>

#include "common.cuh"

namespace moe {

static thread_local char g_msg[1024] = "";

moe_status fail(moe_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    int n = snprintf(g_msg, sizeof g_msg, "%s: ", moe_status_name(s));
    if (n < 0) n = 0;
    if (n < (int)sizeof g_msg) vsnprintf(g_msg + n, sizeof g_msg - n, fmt, ap);
    va_end(ap);
    return s;
}

moe_status check_launch(const char *what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "launch of %s failed: %s", what, cudaGetErrorString(e));
    return MOE_OK;
}

int sm_count()
{
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

__global__ void f32_to_bf16_kernel(const float *__restrict__ in, uint16_t *__restrict__ out, int64_t n)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (; i < n; i += stride) out[i] = f32_to_bf16(in[i]);
}

// One CTA per token: x / sqrt(mean(x^2) + eps) rounded to bf16.  The sum of
// squares is taken in a fixed order (per-thread strided sums, a warp tree,
// then the warps in order), the same order the fused decode kernel uses.
__global__ void rms_norm_bf16_kernel(const float *__restrict__ x, uint16_t *__restrict__ out, int H, float eps)
{
    __shared__ float wsum[32];
    const float *xr = x + (int64_t)blockIdx.x * H;
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane_id() == 0) wsum[warp_id()] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += wsum[w];
    float inv = 1.0f / sqrtf(tot / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x) out[(int64_t)blockIdx.x * H + i] = f32_to_bf16(xr[i] * inv);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_last_error(void) { return g_msg; }

const char *moe_status_name(moe_status s)
{
    switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_NONFINITE: return "MOE_ERR_NONFINITE";
    case MOE_ERR_BOUNDS: return "MOE_ERR_BOUNDS";
    case MOE_ERR_RANGE: return "MOE_ERR_RANGE";
    }
    return "MOE_ERR_UNKNOWN";
}

moe_status moe_check_status(int32_t *dev_status, int reset, moe_stream_t stream)
{
    MOE_REQUIRE(dev_status, "dev_status is NULL");
    int32_t v = 0;
    MOE_CUDA_TRY(cudaMemcpyAsync(&v, dev_status, sizeof v, cudaMemcpyDeviceToHost, to_cuda(stream)));
    MOE_CUDA_TRY(cudaStreamSynchronize(to_cuda(stream)));
    if (reset && v) {
        MOE_CUDA_TRY(cudaMemsetAsync(dev_status, 0, sizeof v, to_cuda(stream)));
        MOE_CUDA_TRY(cudaStreamSynchronize(to_cuda(stream)));
    }
    if (v == 0) return MOE_OK;
    moe_status s = (v >= 1 && v <= 8) ? (moe_status)v : MOE_ERR_CUDA;
    return fail(s, "a kernel reported %s through the device status word", moe_status_name(s));
}

moe_status moe_packed_size(int bits, int64_t rows, int64_t cols, size_t *code_bytes, size_t *scale_bytes)
{
    MOE_REQUIRE(bits == 2 || bits == 3, "bits must be 2 or 3 (got %d)", bits);
    MOE_REQUIRE(rows >= 0 && cols > 0 && cols % 32 == 0,
                "rows >= 0 and cols a positive multiple of 32 (got rows=%lld cols=%lld)", (long long)rows,
                (long long)cols);
    int64_t rb = bits == 2 ? cols / 4 : cols / 4 + cols / 8;
    if (code_bytes) *code_bytes = (size_t)(rows * rb);
    if (scale_bytes) *scale_bytes = (size_t)(rows * (cols / 32) * 2);
    return MOE_OK;
}

moe_status moe_f32_to_bf16(const float *in_f32, uint16_t *out_bf16, int64_t n, moe_stream_t stream)
{
    MOE_REQUIRE(n >= 0, "n must be >= 0");
    if (n == 0) return MOE_OK;
    MOE_REQUIRE(in_f32 && out_bf16, "NULL pointer");
    int64_t blocks = (n + 255) / 256;
    int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    f32_to_bf16_kernel<<<(unsigned)blocks, 256, 0, to_cuda(stream)>>>(in_f32, out_bf16, n);
    return check_launch("f32_to_bf16");
}

moe_status moe_rms_norm_bf16(const float *x, uint16_t *out, int T, int H, float eps, moe_stream_t stream)
{
    MOE_REQUIRE(T >= 0 && H > 0, "T >= 0 and H > 0 (got T=%d H=%d)", T, H);
    MOE_REQUIRE(eps >= 0.f, "eps must be >= 0");
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x && out, "NULL pointer");
    rms_norm_bf16_kernel<<<T, 256, 0, to_cuda(stream)>>>(x, out, H, eps);
    return check_launch("rms_norm_bf16");
}

}  // extern "C"
