// shared_expert.cu -- moe_shared_expert: the always-on bf16 SwiGLU expert.
//
// The pages: one shared expert runs beside the routed ones in every layer
// ("Strata Open-Source Runtime: Running a 125B-Parameter Qwen3 Model on a 12GB
// GPU", section "The Model Itself").  T <= 8 runs the dense-mode GEMV of
// gemv.cuh (fp32 maths on exact bf16 weights); larger T a tiled GEMM.
#include "common.cuh"
#include "dense_tc.cuh"
#include "gemv.cuh"

namespace moe {

moe_status launch_bf16_gemv(bool swiglu, const GemvArgs &a, int nvmax, cudaStream_t s);

// out[i] = (acc ? out[i] : 0) + y[i]
__global__ void add_out_kernel(const float *__restrict__ y, int64_t n, void *out, int out_bf16, int accumulate)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    if (out_bf16) {
        uint16_t *o = static_cast<uint16_t *>(out);
        o[i] = f32_to_bf16((accumulate ? bf16_to_f32(o[i]) : 0.f) + y[i]);
    } else {
        float *o = static_cast<float *>(out);
        o[i] = (accumulate ? o[i] : 0.f) + y[i];
    }
}

// C[t][r] = sum_i A[t][i] B[r][i]; A bf16 or fp32, B bf16 [rows][K].
// SWIGLU: B holds the gate rows and Bu the up rows; C = silu(g) * u.
constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 32;

template <bool SWIGLU>
__global__ void __launch_bounds__(256) dense_bf16_gemm_kernel(const uint16_t *__restrict__ Abf,
                                                              const float *__restrict__ Af, int T, int K,
                                                              const uint16_t *__restrict__ B,
                                                              const uint16_t *__restrict__ Bu, int rows,
                                                              float *__restrict__ C)
{
    __shared__ float as[SG_BK][SG_BM + 4];
    __shared__ float bs[SG_BK][SG_BN + 4];
    __shared__ float gs[SWIGLU ? SG_BM : 1][SWIGLU ? SG_BN + 1 : 1];
    int t0 = blockIdx.x * SG_BM, nt = blockIdx.y;
    int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += SG_BK) {
        for (int i = threadIdx.x; i < SG_BM * SG_BK; i += 256) {
            int r = i / SG_BK, c = i % SG_BK;
            int t = t0 + r;
            float v = 0.f;
            if (t < T) v = Abf ? bf16_to_f32(Abf[(int64_t)t * K + k0 + c]) : Af[(int64_t)t * K + k0 + c];
            as[c][r] = v;
            int rr;
            const uint16_t *src = B;
            if (SWIGLU) {
                rr = nt * (SG_BN / 2) + (r % (SG_BN / 2));
                if (r >= SG_BN / 2) src = Bu;
            } else {
                rr = nt * SG_BN + r;
            }
            bs[c][r] = rr < rows ? bf16_to_f32(src[(int64_t)rr * K + k0 + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < SG_BK; kk++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = as[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    if (SWIGLU) {
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) gs[ty * 4 + i][tx * 4 + j] = acc[i][j];
        __syncthreads();
        for (int i = threadIdx.x; i < SG_BM * (SG_BN / 2); i += 256) {
            int r = i / (SG_BN / 2), c = i % (SG_BN / 2);
            int t = t0 + r, row = nt * (SG_BN / 2) + c;
            if (t < T && row < rows) C[(int64_t)t * rows + row] = silu(gs[r][c]) * gs[r][c + SG_BN / 2];
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            int t = t0 + ty * 4 + i;
            if (t >= T) continue;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                int row = nt * SG_BN + tx * 4 + j;
                if (row < rows) C[(int64_t)t * rows + row] = acc[i][j];
            }
        }
    }
}

static size_t shared_ws_bytes(int H, int I, int T)
{
    return align256((size_t)T * I * sizeof(float)) + align256((size_t)T * H * sizeof(float));
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_shared_expert_workspace_size(int H, int I, int T, size_t *bytes)
{
    MOE_REQUIRE(bytes, "bytes is NULL");
    MOE_REQUIRE(H > 0 && I > 0 && T >= 0, "H, I > 0 and T >= 0");
    *bytes = shared_ws_bytes(H, I, T);
    return MOE_OK;
}

extern "C" moe_status moe_shared_expert(const uint16_t *wg, const uint16_t *wu, const uint16_t *wd, int H, int I,
                                        const uint16_t *x_bf16, int T, void *out, moe_dtype out_dtype, int accumulate,
                                        void *ws, size_t ws_bytes, int32_t *dev_status, moe_stream_t stream)
{
    MOE_REQUIRE(H > 0 && H % 32 == 0 && I > 0 && I % 32 == 0, "H and I must be positive multiples of 32 (got H=%d I=%d)",
                H, I);
    MOE_REQUIRE(T >= 0, "T must be >= 0");
    MOE_REQUIRE(out_dtype == MOE_F32 || out_dtype == MOE_BF16, "out_dtype must be MOE_F32 or MOE_BF16");
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(wg && wu && wd && x_bf16 && out, "NULL pointer");
    MOE_REQUIRE(aligned16(wg) && aligned16(wu) && aligned16(wd) && aligned16(x_bf16),
                "weights and x must be 16-byte aligned");
    size_t need = shared_ws_bytes(H, I, T);
    if (!ws || ws_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "shared_expert (T=%d) needs %zu bytes (%.2f MiB) of workspace, got %zu", T, need,
                    mib((double)need), ws ? ws_bytes : (size_t)0);
    MOE_REQUIRE(aligned16(ws), "workspace must be 16-byte aligned");
    cudaStream_t s = to_cuda(stream);
    float *h = static_cast<float *>(ws);
    float *y = reinterpret_cast<float *>(static_cast<char *>(ws) + align256((size_t)T * I * sizeof(float)));
    moe_status st;
    if (T <= 8) {
        GemvArgs a = {};
        a.mode = GEMV_DENSE;
        a.T = T;
        a.codes = reinterpret_cast<const uint8_t *>(wg);
        a.row_bytes = (int64_t)H * 2;
        a.up_delta = (int64_t)(reinterpret_cast<const char *>(wu) - reinterpret_cast<const char *>(wg));
        a.up_sdelta = 0;
        a.vec_bf16 = x_bf16;
        a.out = h;
        st = gemv_plan(a, H, I, 1);
        if (st != MOE_OK) return st;
        st = launch_bf16_gemv(true, a, T, s);
        if (st != MOE_OK) return st;
        GemvArgs b = a;
        b.codes = reinterpret_cast<const uint8_t *>(wd);
        b.row_bytes = (int64_t)I * 2;
        b.up_delta = 0;
        b.vec_bf16 = nullptr;
        b.vec_f32 = h;
        b.out = y;
        st = gemv_plan(b, I, H, 1);
        if (st != MOE_OK) return st;
        st = launch_bf16_gemv(false, b, T, s);
        if (st != MOE_OK) return st;
    } else {
        // tensor cores: gate/up with exact bf16 products, h = h_hi + h_lo in
        // two bf16 halves, down projection over [h_hi | h_lo] against the down
        // weights read twice, accumulated straight into out
        DenseGemm gu = {};
        uint16_t *hs = static_cast<uint16_t *>(ws);
        gu.A = x_bf16;
        gu.a_cols = H;
        gu.B0 = wg;
        gu.B1 = wu;
        gu.b_cols = H;
        gu.M = T;
        gu.N = I;
        gu.K = H;
        gu.hsplit = hs;
        gu.status = dev_status;
        DenseGemm gd = {};
        gd.A = hs;
        gd.a_cols = 2 * I;
        gd.B0 = wd;
        gd.b_cols = I;
        gd.M = T;
        gd.N = H;
        gd.K = 2 * I;
        gd.out = out;
        gd.out_bf16 = out_dtype == MOE_BF16;
        gd.accumulate = accumulate;
        gd.status = dev_status;
        if (dense_tc_supported(gu, DENSE_SWIGLU_SPLIT) && dense_tc_supported(gd, DENSE_OUT)) {
            st = dense_tc_gemm(gu, DENSE_SWIGLU_SPLIT, s);
            if (st != MOE_OK) return st;
            return dense_tc_gemm(gd, DENSE_OUT, s);
        }
        dim3 g1((T + SG_BM - 1) / SG_BM, (I + SG_BN / 2 - 1) / (SG_BN / 2));
        dense_bf16_gemm_kernel<true><<<g1, 256, 0, s>>>(x_bf16, nullptr, T, H, wg, wu, I, h);
        st = check_launch("shared_gateup");
        if (st != MOE_OK) return st;
        dim3 g2((T + SG_BM - 1) / SG_BM, (H + SG_BN - 1) / SG_BN);
        dense_bf16_gemm_kernel<false><<<g2, 256, 0, s>>>(nullptr, h, T, I, wd, nullptr, H, y);
        st = check_launch("shared_down");
        if (st != MOE_OK) return st;
    }
    int64_t n = (int64_t)T * H;
    add_out_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(y, n, out, out_dtype == MOE_BF16, accumulate);
    return check_launch("shared_add");
}
