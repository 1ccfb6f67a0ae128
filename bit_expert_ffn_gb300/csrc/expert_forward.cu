// expert_forward.cu -- moe_expert_forward: the routed experts of one layer.
//
// DECODE (T <= 8): grouped dequant GEMVs (gemv.cuh) for gate/up -> h and
// down -> y, then an atomic-free combine that sums each token's k slots in
// slot order.  PREFILL: grouped GEMM (expert_prefill.cu).
//
// The combine follows the pages' statement that the finished expert vectors
// are summed on the GPU ("How Strata runs a 125-billion-parameter model on a
// single 12 GB to 24 GB graphics card", Step 2, "Dynamic PCIe and CPU
// co-execution").
#include "common.cuh"
#include "gemv.cuh"
#include "prefill.cuh"

namespace moe {

// out[t][o] = (acc ? out[t][o] : 0) + sum_j w[t][j] * y[inv[t*k+j]][o]
__global__ void combine_kernel(const float *__restrict__ y, const float *__restrict__ w,
                               const int32_t *__restrict__ inv, int T, int k, int H, void *out, int out_bf16,
                               int accumulate)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)T * H) return;
    int t = (int)(i / H), o = (int)(i - (int64_t)t * H);
    float s = 0.f;
    for (int j = 0; j < k; j++) {
        int p = inv[t * k + j];
        if (p >= 0) s = fmaf(w[t * k + j], y[(int64_t)p * H + o], s);
    }
    if (out_bf16) {
        uint16_t *ob = static_cast<uint16_t *>(out);
        float base = accumulate ? bf16_to_f32(ob[i]) : 0.f;
        ob[i] = f32_to_bf16(base + s);
    } else {
        float *of = static_cast<float *>(out);
        of[i] = (accumulate ? of[i] : 0.f) + s;
    }
}

moe_status launch_combine(const float *y, const float *w, const int32_t *inv, int T, int k, int H, void *out,
                          moe_dtype dt, int accumulate, cudaStream_t s)
{
    int64_t n = (int64_t)T * H;
    combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(y, w, inv, T, k, H, out, dt == MOE_BF16, accumulate);
    return check_launch("combine");
}

// As combine_kernel for fp16 rows of y (the prefill GEMM's output): eight
// consecutive outputs per thread, 16-byte loads of y; same slot order.
__global__ void combine_f16_kernel(const uint16_t *__restrict__ y, const float *__restrict__ w,
                                   const int32_t *__restrict__ inv, int T, int k, int H, void *out, int out_bf16,
                                   int accumulate)
{
    const int H8 = H / 8;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)T * H8) return;
    const int t = (int)(i / H8), o = 8 * (int)(i - (int64_t)t * H8);
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; j++) {
        const int p = inv[t * k + j];
        if (p < 0) continue;
        const float wj = w[t * k + j];
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(y + (int64_t)p * H + o));
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&qw[m]));
            s[2 * m] = fmaf(wj, f.x, s[2 * m]);
            s[2 * m + 1] = fmaf(wj, f.y, s[2 * m + 1]);
        }
    }
    const int64_t b = (int64_t)t * H + o;
    if (out_bf16) {
        uint16_t *ob = static_cast<uint16_t *>(out) + b;
#pragma unroll
        for (int m = 0; m < 8; m++) ob[m] = f32_to_bf16((accumulate ? bf16_to_f32(ob[m]) : 0.f) + s[m]);
    } else {
        float *of = static_cast<float *>(out) + b;  // the caller's buffer: no alignment beyond 4 bytes assumed
#pragma unroll
        for (int m = 0; m < 8; m++) of[m] = (accumulate ? of[m] : 0.f) + s[m];
    }
}

moe_status launch_combine_f16(const uint16_t *y, const float *w, const int32_t *inv, int T, int k, int H, void *out,
                              moe_dtype dt, int accumulate, cudaStream_t s)
{
    int64_t n = (int64_t)T * (H / 8);
    combine_f16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(y, w, inv, T, k, H, out, dt == MOE_BF16,
                                                                     accumulate);
    return check_launch("combine_f16");
}

template <class W, bool SWIGLU>
static moe_status launch_gemv(const GemvArgs &a, int groups, int nvmax, cudaStream_t s)
{
    unsigned grid = (unsigned)(groups * a.tasks_per_group);
    if (nvmax <= 1) gemv_kernel<W, SWIGLU, 1><<<grid, kGemvThreads, 0, s>>>(a);
    else if (nvmax <= 2) gemv_kernel<W, SWIGLU, 2><<<grid, kGemvThreads, 0, s>>>(a);
    else gemv_kernel<W, SWIGLU, 4><<<grid, kGemvThreads, 0, s>>>(a);
    return check_launch("gemv");
}

moe_status launch_quant_gemv(int bits, bool swiglu, const GemvArgs &a, int groups, int nvmax, cudaStream_t s)
{
    if (bits == 2)
        return swiglu ? launch_gemv<QuantW<2>, true>(a, groups, nvmax, s) : launch_gemv<QuantW<2>, false>(a, groups, nvmax, s);
    return swiglu ? launch_gemv<QuantW<3>, true>(a, groups, nvmax, s) : launch_gemv<QuantW<3>, false>(a, groups, nvmax, s);
}

moe_status launch_bf16_gemv(bool swiglu, const GemvArgs &a, int nvmax, cudaStream_t s)
{
    return swiglu ? launch_gemv<Bf16W, true>(a, 1, nvmax, s) : launch_gemv<Bf16W, false>(a, 1, nvmax, s);
}

static int64_t row_bytes_of(int bits, int cols) { return bits == 2 ? cols / 4 : cols / 4 + cols / 8; }

struct DecodeWs {
    float *h, *y;
    size_t bytes;
};

static DecodeWs decode_ws(const moe_expert_arena &A, int T, int k, void *base)
{
    DecodeWs d;
    size_t n = (size_t)T * k;
    size_t hb = align256(n * A.I * sizeof(float)), yb = align256(n * A.H * sizeof(float));
    d.bytes = hb + yb;
    d.h = static_cast<float *>(base);
    d.y = base ? reinterpret_cast<float *>(static_cast<char *>(base) + hb) : nullptr;
    return d;
}

static moe_status decode_forward(const moe_expert_arena &A, const uint16_t *x, int T, const int32_t *ids,
                                 const float *w, int k, const int32_t *offsets, const int32_t *perm,
                                 const int32_t *inv, void *out, moe_dtype dt, int accumulate, void *ws,
                                 cudaStream_t s)
{
    DecodeWs d = decode_ws(A, T, k, ws);
    int groups = std::min(T * k, A.E);
    int nvmax = T;  // a group holds at most one pair per token
    GemvArgs a = {};
    a.mode = GEMV_ROUTED;
    a.k = k;
    a.T = T;
    a.ids = ids;
    a.perm = perm;
    a.offsets = offsets;
    a.E = A.E;
    // gate/up: rows = I row pairs, K = H, vectors = x[token]
    a.codes = A.gu_codes;
    a.scales = A.gu_scales;
    a.row_bytes = row_bytes_of(A.bits, A.H);
    a.scale_row = A.H / 32;
    a.codes_expert_stride = (int64_t)2 * A.I * a.row_bytes;
    a.scales_expert_stride = (int64_t)2 * A.I * a.scale_row;
    a.up_delta = (int64_t)A.I * a.row_bytes;
    a.up_sdelta = (int64_t)A.I * a.scale_row;
    a.vec_bf16 = x;
    a.vec_f32 = nullptr;
    a.vec_by_token = 1;
    a.out = d.h;
    moe_status st = gemv_plan(a, A.H, A.I, groups);
    if (st != MOE_OK) return st;
    st = launch_quant_gemv(A.bits, true, a, groups, nvmax, s);
    if (st != MOE_OK) return st;
    // down: rows = H, K = I, vectors = h[pair]
    GemvArgs b = a;
    b.codes = A.d_codes;
    b.scales = A.d_scales;
    b.row_bytes = row_bytes_of(A.bits, A.I);
    b.scale_row = A.I / 32;
    b.codes_expert_stride = (int64_t)A.H * b.row_bytes;
    b.scales_expert_stride = (int64_t)A.H * b.scale_row;
    b.up_delta = 0;
    b.up_sdelta = 0;
    b.vec_bf16 = nullptr;
    b.vec_f32 = d.h;
    b.vec_by_token = 0;
    b.out = d.y;
    st = gemv_plan(b, A.I, A.H, groups);
    if (st != MOE_OK) return st;
    st = launch_quant_gemv(A.bits, false, b, groups, nvmax, s);
    if (st != MOE_OK) return st;
    return launch_combine(d.y, w, inv, T, k, A.H, out, dt, accumulate, s);
}

static moe_status check_arena(const moe_expert_arena *A)
{
    MOE_REQUIRE(A, "arena is NULL");
    MOE_REQUIRE(A->bits == 2 || A->bits == 3, "arena bits must be 2 or 3 (got %d)", A->bits);
    MOE_REQUIRE(A->H > 0 && A->H % 32 == 0 && A->I > 0 && A->I % 32 == 0,
                "H and I must be positive multiples of 32 (got H=%d I=%d)", A->H, A->I);
    MOE_REQUIRE(A->E >= 1 && A->E <= 1024, "E must be in [1, 1024] (got %d)", A->E);
    MOE_REQUIRE(A->gu_codes && A->gu_scales && A->d_codes && A->d_scales, "arena pointer is NULL");
    MOE_REQUIRE(aligned16(A->gu_codes) && aligned16(A->gu_scales) && aligned16(A->d_codes) && aligned16(A->d_scales),
                "arena pointers must be 16-byte aligned");
    return MOE_OK;
}

static moe_path resolve_path(moe_path p, int T)
{
    return p == MOE_PATH_AUTO ? (T <= 8 ? MOE_PATH_DECODE : MOE_PATH_PREFILL) : p;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_expert_forward_workspace_size(const moe_expert_arena *arena, int T, int k, moe_path path,
                                                        size_t *bytes)
{
    moe_status st = check_arena(arena);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(bytes, "bytes is NULL");
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= 16, "T >= 0 and 1 <= k <= 16");
    moe_path p = resolve_path(path, T);
    MOE_REQUIRE(p == MOE_PATH_DECODE || p == MOE_PATH_PREFILL || p == MOE_PATH_PREFILL_FP8, "unknown path %d",
                (int)path);
    if (p == MOE_PATH_PREFILL_FP8 && !prefill_fp8_supported(*arena))
        return fail(MOE_ERR_UNSUPPORTED, "the FP8 prefill takes 2-bit arenas with H and I multiples of 128 "
                    "(got bits=%d H=%d I=%d)", arena->bits, arena->H, arena->I);
    if (p == MOE_PATH_DECODE) *bytes = decode_ws(*arena, T, k, nullptr).bytes;
    else if (p == MOE_PATH_PREFILL_FP8) *bytes = prefill_fp8_workspace_bytes(*arena, T, k);
    else *bytes = prefill_workspace_bytes(*arena, T, k);
    return MOE_OK;
}

extern "C" moe_status moe_expert_forward(const moe_expert_arena *arena, const uint16_t *x_bf16, int T,
                                         const int32_t *ids, const float *w, int k, const int32_t *offsets,
                                         const int32_t *perm, const int32_t *inv_perm, void *out, moe_dtype out_dtype,
                                         int accumulate, moe_path path, void *ws, size_t ws_bytes,
                                         int32_t *dev_status, moe_stream_t stream)
{
    moe_status st = check_arena(arena);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(T >= 0, "T must be >= 0");
    MOE_REQUIRE(k >= 1 && k <= 16 && k <= arena->E, "k must be in [1, min(E, 16)] (got %d)", k);
    MOE_REQUIRE(out_dtype == MOE_F32 || out_dtype == MOE_BF16, "out_dtype must be MOE_F32 or MOE_BF16");
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x_bf16 && ids && w && offsets && perm && inv_perm && out, "NULL pointer");
    MOE_REQUIRE(aligned16(x_bf16), "x_bf16 must be 16-byte aligned");
    moe_path p = resolve_path(path, T);
    MOE_REQUIRE(p == MOE_PATH_DECODE || p == MOE_PATH_PREFILL || p == MOE_PATH_PREFILL_FP8, "unknown path %d",
                (int)path);
    if (p == MOE_PATH_DECODE)
        MOE_REQUIRE(T <= 8, "the decode path takes at most 8 tokens (got %d); use MOE_PATH_PREFILL", T);
    if (p == MOE_PATH_PREFILL_FP8 && !prefill_fp8_supported(*arena))
        return fail(MOE_ERR_UNSUPPORTED, "the FP8 prefill takes 2-bit arenas with H and I multiples of 128 "
                    "(got bits=%d H=%d I=%d)", arena->bits, arena->H, arena->I);
    size_t need = p == MOE_PATH_DECODE        ? decode_ws(*arena, T, k, nullptr).bytes
                  : p == MOE_PATH_PREFILL_FP8 ? prefill_fp8_workspace_bytes(*arena, T, k)
                                              : prefill_workspace_bytes(*arena, T, k);
    if (need && (!ws || ws_bytes < need))
        return fail(MOE_ERR_WORKSPACE, "expert_forward (%s, T=%d) needs %zu bytes (%.2f MiB) of workspace, got %zu",
                    p == MOE_PATH_DECODE ? "decode" : p == MOE_PATH_PREFILL_FP8 ? "fp8 prefill" : "prefill", T,
                    need, mib((double)need), ws ? ws_bytes : (size_t)0);
    MOE_REQUIRE(!ws || aligned16(ws), "workspace must be 16-byte aligned");
    cudaStream_t s = to_cuda(stream);
    if (p == MOE_PATH_DECODE)
        return decode_forward(*arena, x_bf16, T, ids, w, k, offsets, perm, inv_perm, out, out_dtype, accumulate, ws, s);
    if (p == MOE_PATH_PREFILL_FP8)
        return prefill_fp8_forward(*arena, x_bf16, T, w, k, offsets, perm, inv_perm, out, out_dtype, accumulate, ws,
                                   dev_status, s);
    return prefill_forward(*arena, x_bf16, T, ids, w, k, offsets, perm, inv_perm, out, out_dtype, accumulate, ws,
                           dev_status, s);
}
