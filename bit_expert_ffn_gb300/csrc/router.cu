// router.cu -- moe_router_topk / moe_topk_from_logits.
//
// logits[t][e] = bias[e] + sum_i W[e][i] x[t][i] in fp32, then top-k with
// ties to the lower id and the renormalised softmax weights of the kept
// experts.  The pages: a router per layer keeps 10 of 512 experts for each
// token ("Strata Open-Source Runtime: Running a 125B-Parameter Qwen3 Model on
// a 12GB GPU", section "The Model Itself").
#include "common.cuh"
#include "dense_tc.cuh"

namespace moe {

constexpr int kTopkMaxK = 16;
constexpr int kMaxE = 1024;

// ------------------------------------------------------------------ GEMV
// Small T: one warp per expert row, the whole of x staged in shared memory
// as fp32.  W is streamed with 128-bit loads.
template <int TT>
__global__ void __launch_bounds__(256) router_gemv_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                          const float *__restrict__ W,
                                                          const float *__restrict__ bias, int E,
                                                          float *__restrict__ logits)
{
    extern __shared__ float xs[];  // [TT][H]
    for (int i = threadIdx.x; i < TT * H; i += blockDim.x) {
        int t = i / H;
        xs[i] = t < T ? bf16_to_f32(x[i]) : 0.f;
    }
    __syncthreads();
    int e = blockIdx.x * (blockDim.x >> 5) + warp_id();
    if (e >= E) return;
    int lane = lane_id();
    const float4 *wrow = reinterpret_cast<const float4 *>(W + (int64_t)e * H);
    float acc[TT];
#pragma unroll
    for (int t = 0; t < TT; t++) acc[t] = 0.f;
    int n4 = H >> 2;
    for (int c = lane; c < n4; c += 32) {
        float4 w = __ldg(wrow + c);
#pragma unroll
        for (int t = 0; t < TT; t++) {
            float4 xv = *reinterpret_cast<const float4 *>(xs + t * H + 4 * c);
            acc[t] = fmaf(w.x, xv.x, acc[t]);
            acc[t] = fmaf(w.y, xv.y, acc[t]);
            acc[t] = fmaf(w.z, xv.z, acc[t]);
            acc[t] = fmaf(w.w, xv.w, acc[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < TT; t++) {
#pragma unroll
        for (int o = 16; o; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    }
    if (lane == 0) {
        float b = bias ? bias[e] : 0.f;
        for (int t = 0; t < T && t < TT; t++) logits[(int64_t)t * E + e] = acc[t] + b;
    }
}

// ------------------------------------------------------------------ GEMM
// Large T: 64 tokens x 64 experts per CTA, 256 threads with a 4x4 register
// tile each, K staged 32 at a time (x converted from bf16 on the way in).
constexpr int RG_BM = 64, RG_BN = 64, RG_BK = 32;

__global__ void __launch_bounds__(256) router_gemm_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                          const float *__restrict__ W,
                                                          const float *__restrict__ bias, int E,
                                                          float *__restrict__ logits)
{
    __shared__ float xs[RG_BK][RG_BM + 4];
    __shared__ float ws[RG_BK][RG_BN + 4];
    int t0 = blockIdx.x * RG_BM, e0 = blockIdx.y * RG_BN;
    int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < H; k0 += RG_BK) {
        for (int i = threadIdx.x; i < RG_BM * RG_BK; i += 256) {
            int r = i / RG_BK, c = i % RG_BK;
            int t = t0 + r;
            xs[c][r] = (t < T) ? bf16_to_f32(x[(int64_t)t * H + k0 + c]) : 0.f;
            int e = e0 + r;
            ws[c][r] = (e < E) ? W[(int64_t)e * H + k0 + c] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < RG_BK; c++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = xs[c][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = ws[c][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int e = e0 + tx * 4 + j;
            if (e < E) logits[(int64_t)t * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
        }
    }
}

// ------------------------------------------------------------------ top-k
// One warp per token.  Lane l holds experts l, l+32, ...; k rounds of a warp
// arg-max under the order (logit descending, id ascending).
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}

__global__ void topk_kernel(const float *__restrict__ logits, int T, int E, int k, int32_t *__restrict__ ids,
                            float *__restrict__ wout, int32_t *status)
{
    int t = blockIdx.x * (blockDim.x >> 5) + warp_id();
    if (t >= T) return;
    int lane = lane_id();
    const float *l = logits + (int64_t)t * E;
    float v[kMaxE / 32];
    uint32_t avail = 0;
    bool nan = false;
#pragma unroll
    for (int q = 0; q < kMaxE / 32; q++) {
        int e = lane + 32 * q;
        v[q] = e < E ? l[e] : 0.f;
        if (e < E) {
            avail |= 1u << q;
            nan |= isnan(v[q]);
        }
    }
    nan = __any_sync(0xffffffffu, nan);
    if (nan) {
        set_status(status, MOE_ERR_NONFINITE);
        if (lane < k) {
            ids[(int64_t)t * k + lane] = lane;
            wout[(int64_t)t * k + lane] = 1.f / (float)k;
        }
        return;
    }
    float my_v = 0.f;  // lane j keeps the j-th selected logit
    int my_id = 0;
    for (int j = 0; j < k; j++) {
        float bv = 0.f;
        int bi = INT32_MAX;
#pragma unroll
        for (int q = 0; q < kMaxE / 32; q++) {
            if (avail & (1u << q)) {
                int e = lane + 32 * q;
                if (bi == INT32_MAX || ranks_before(v[q], e, bv, bi)) {
                    bv = v[q];
                    bi = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != INT32_MAX && (bi == INT32_MAX || ranks_before(ov, oi, bv, bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
        if (lane == j) {
            my_v = bv;
            my_id = bi;
        }
    }
    // renormalised softmax of the kept logits; the top-1 logit is the maximum
    float m = __shfl_sync(0xffffffffu, my_v, 0);
    float p = 0.f;
    if (lane < k) {
        if (isinf(m)) p = (my_v == m) ? 1.f : 0.f;
        else p = expf(my_v - m);
    }
    float z = p;
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < k) {
        ids[(int64_t)t * k + lane] = my_id;
        wout[(int64_t)t * k + lane] = p / z;
    }
}

static moe_status launch_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w, int32_t *st,
                              cudaStream_t s)
{
    int warps = 8;
    int blocks = (T + warps - 1) / warps;
    topk_kernel<<<blocks, warps * 32, 0, s>>>(logits, T, E, k, ids, w, st);
    return check_launch("topk");
}

static moe_status check_topk_args(int T, int E, int k)
{
    MOE_REQUIRE(T >= 0, "T must be >= 0 (got %d)", T);
    MOE_REQUIRE(E >= 1 && E <= kMaxE, "E must be in [1, %d] (got %d)", kMaxE, E);
    MOE_REQUIRE(k >= 1 && k <= E && k <= kTopkMaxK, "k must be in [1, min(E, %d)] (got k=%d, E=%d)", kTopkMaxK, k, E);
    return MOE_OK;
}

template <int TT>
static moe_status launch_router_gemv(const uint16_t *x, int T, int H, const float *W, const float *bias, int E,
                                     float *logits, cudaStream_t s)
{
    int warps = 8;
    int blocks = (E + warps - 1) / warps;
    size_t smem = (size_t)TT * H * sizeof(float);
    if (smem > 200 * 1024)
        return fail(MOE_ERR_UNSUPPORTED, "H=%d too large for the decode router (%zu bytes of shared memory)", H, smem);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(router_gemv_kernel<TT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "router smem attribute: %s", cudaGetErrorString(e));
    }
    router_gemv_kernel<TT><<<blocks, warps * 32, smem, s>>>(x, T, H, W, bias, E, logits);
    return check_launch("router_gemv");
}

// W = W1 + W2 + W3 with each piece bf16 (round to nearest even of what the
// previous pieces leave; each difference is exact in fp32), stored side by
// side: Ws[e][j*H + i] = piece j of W[e][i].  Three pieces carry 24
// significant bits, so x . (W1 + W2 + W3) with exact bf16 products and fp32
// sums keeps the fp32 router's accuracy.
__global__ void split_router_kernel(const float *__restrict__ W, int64_t n, int H, uint16_t *__restrict__ Ws)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t e = i / H, c = i - e * H;
        float w = W[i];
        uint16_t a = f32_to_bf16(w);
        float r1 = w - bf16_to_f32(a);
        uint16_t b = f32_to_bf16(r1);
        float r2 = r1 - bf16_to_f32(b);
        uint16_t d = f32_to_bf16(r2);
        uint16_t *row = Ws + e * 3 * H;
        row[c] = a;
        row[H + c] = b;
        row[2 * H + c] = d;
    }
}

static bool router_tc_shape(int T, int H) { return T > 8 && H % 64 == 0; }

static size_t router_ws_bytes(int T, int H, int E, int logits_given)
{
    size_t b = logits_given ? 0 : align256((size_t)T * E * sizeof(float));
    if (router_tc_shape(T, H)) b += align256((size_t)E * 3 * H * sizeof(uint16_t));
    return b;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_topk_from_logits(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                                           int32_t *dev_status, moe_stream_t stream)
{
    moe_status st = check_topk_args(T, E, k);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && ids && w, "NULL pointer");
    return launch_topk(logits, T, E, k, ids, w, dev_status, to_cuda(stream));
}

extern "C" moe_status moe_router_workspace_size(int T, int H, int E, int logits_given, size_t *bytes)
{
    MOE_REQUIRE(bytes, "bytes is NULL");
    MOE_REQUIRE(T >= 0 && H > 0 && E >= 1, "T >= 0, H > 0 and E >= 1");
    *bytes = router_ws_bytes(T, H, E, logits_given);
    return MOE_OK;
}

extern "C" moe_status moe_router_topk(const uint16_t *x_bf16, int T, int H, const float *w_router, const float *bias,
                                      int E, int k, float *logits_out, int32_t *topk_ids, float *topk_w, void *ws,
                                      size_t ws_bytes, int32_t *dev_status, moe_stream_t stream)
{
    moe_status st = check_topk_args(T, E, k);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(H > 0 && H % 32 == 0, "H must be a positive multiple of 32 (got %d)", H);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x_bf16 && w_router && topk_ids && topk_w, "NULL pointer");
    MOE_REQUIRE(aligned16(w_router), "w_router must be 16-byte aligned");
    size_t need = router_ws_bytes(T, H, E, logits_out != nullptr);
    if (need && (!ws || ws_bytes < need))
        return fail(MOE_ERR_WORKSPACE, "router (T=%d) needs %zu bytes (%.2f MiB) of workspace, got %zu", T, need,
                    mib((double)need), ws ? ws_bytes : (size_t)0);
    MOE_REQUIRE(!need || aligned16(ws), "workspace must be 16-byte aligned");
    char *wsp = static_cast<char *>(ws);
    float *logits = logits_out;
    if (!logits) {
        logits = reinterpret_cast<float *>(wsp);
        wsp += align256((size_t)T * E * sizeof(float));
    }
    cudaStream_t s = to_cuda(stream);
    if (T <= 8) {
        if (T == 1) st = launch_router_gemv<1>(x_bf16, T, H, w_router, bias, E, logits, s);
        else if (T == 2) st = launch_router_gemv<2>(x_bf16, T, H, w_router, bias, E, logits, s);
        else if (T <= 4) st = launch_router_gemv<4>(x_bf16, T, H, w_router, bias, E, logits, s);
        else st = launch_router_gemv<8>(x_bf16, T, H, w_router, bias, E, logits, s);
    } else {
        DenseGemm g = {};
        uint16_t *wsplit = reinterpret_cast<uint16_t *>(wsp);
        g.A = x_bf16;
        g.a_cols = H;
        g.B0 = wsplit;
        g.b_cols = 3 * H;
        g.M = T;
        g.N = E;
        g.K = 3 * H;
        g.bias = bias;
        g.out = logits;
        g.status = dev_status;
        if (router_tc_shape(T, H) && dense_tc_supported(g, DENSE_OUT)) {
            int64_t n = (int64_t)E * H;
            int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
            split_router_kernel<<<blocks, 256, 0, s>>>(w_router, n, H, wsplit);
            st = check_launch("split_router");
            if (st == MOE_OK) st = dense_tc_gemm(g, DENSE_OUT, s);
        } else {
            dim3 grid((T + RG_BM - 1) / RG_BM, (E + RG_BN - 1) / RG_BN);
            router_gemm_kernel<<<grid, 256, 0, s>>>(x_bf16, T, H, w_router, bias, E, logits);
            st = check_launch("router_gemm");
        }
    }
    if (st != MOE_OK) return st;
    return launch_topk(logits, T, E, k, topk_ids, topk_w, dev_status, s);
}
