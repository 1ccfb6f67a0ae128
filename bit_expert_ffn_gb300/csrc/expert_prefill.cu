// expert_prefill.cu -- the prefill path of moe_expert_forward: grouped GEMMs
// over the experts' token lists, then the slot-ordered combine.
//
//   gate/up:  h[p][r] = silu(sum_i dq(Wg_e[r][i]) x[tok(p)][i]) * (same with Wu_e)
//   down:     y[p][o] = sum_r dq(Wd_e[o][r]) h[p][r]
//   combine:  out[t][o] = sum_j w[t][j] y[inv[t*k+j]][o]
// where p runs over the sorted pairs of expert e (offsets[e] .. offsets[e+1])
// and tok(p) = perm[p] / k.
//
// The tile kernel here is the CUDA-core form (fp32 FFMA on weights
// dequantised exactly into shared memory, 64 x 64 tiles); it serves shapes
// the tensor-core form (prefill_tc.cu) does not take.
#include "common.cuh"
#include "prefill.cuh"

namespace moe {

constexpr int PF_BM = 64;  // pairs per tile
constexpr int PF_BN = 64;  // weight rows per tile (SWIGLU: 32 gate + 32 up)
constexpr int PF_BK = 32;  // one quantisation block

__global__ void __launch_bounds__(1024) tile_prefix_kernel(const int32_t *__restrict__ offsets, int E, int bm,
                                                           int32_t *__restrict__ mt_prefix)
{
    __shared__ int32_t warp_tot[32];
    int e = threadIdx.x;
    int v = 0;
    if (e < E) {
        int n = offsets[e + 1] - offsets[e];
        v = (n + bm - 1) / bm;
    }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane_id() >= o) incl += y;
    }
    if (lane_id() == 31) warp_tot[warp_id()] = incl;
    __syncthreads();
    if (warp_id() == 0) {
        int wt = warp_tot[lane_id()];
        int wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane_id() >= o) wi += y;
        }
        warp_tot[lane_id()] = wi - wt;
    }
    __syncthreads();
    int excl = incl - v + warp_tot[warp_id()];
    if (e < E) mt_prefix[e] = excl;
    if (e == E - 1) mt_prefix[E] = excl + v;
}

struct PfArgs {
    const uint8_t *codes;
    const uint16_t *scales;
    int64_t codes_expert_stride, scales_expert_stride, row_bytes, scale_row;
    int K, rows, up_offset;
    const uint16_t *vec_bf16;  // gate/up: x [T][K]
    const float *vec_f32;      // down: h [n][K]
    const int32_t *perm, *offsets, *mt_prefix;
    int E, k;
    float *out;  // [n][rows]
};

__device__ __forceinline__ int hi_bit(int i) { return (i & 7) | ((i & 8) << 1) | ((i & 16) >> 1); }

// Dequantise 8 consecutive weights (kk0..kk0+7 of block b) of one row.
template <int BITS>
__device__ __forceinline__ void dq8(const uint8_t *rowc, int64_t scale_row, const uint16_t *rows_, int b, int kk0,
                                    float (&o)[8])
{
    uint32_t lo = *reinterpret_cast<const uint16_t *>(rowc + 8 * b + kk0 / 4);  // 8 codes = 16 bits
    uint32_t hi = 0;
    if (BITS == 3) hi = *reinterpret_cast<const uint32_t *>(rowc + scale_row * 8 + 4 * b);
    float s = fp16_to_f32(rows_[b]);
    constexpr float mid = BITS == 2 ? 1.5f : 3.5f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        int c = (lo >> (2 * j)) & 3;
        if (BITS == 3) c |= ((hi >> hi_bit(kk0 + j)) & 1) << 2;
        o[j] = ((float)c - mid) * s;
    }
}

template <int BITS, bool SWIGLU>
__global__ void __launch_bounds__(256) prefill_ffma_kernel(PfArgs a, int n_tiles_n)
{
    __shared__ float xs[PF_BK][PF_BM + 4];
    __shared__ float wsm[PF_BK][PF_BN + 4];
    __shared__ float gs[SWIGLU ? PF_BM : 1][SWIGLU ? PF_BN + 1 : 1];
    int total = a.mt_prefix[a.E] * n_tiles_n;
    int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16 threads, 4 x 4 outputs each
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int mt = tile / n_tiles_n, nt = tile % n_tiles_n;
        int e = expert_of_tile(a.mt_prefix, a.E, mt);
        int p_begin = a.offsets[e] + (mt - a.mt_prefix[e]) * PF_BM;
        int p_end = min(a.offsets[e + 1], p_begin + PF_BM);
        const uint8_t *codes = a.codes + (int64_t)e * a.codes_expert_stride;
        const uint16_t *scales = a.scales + (int64_t)e * a.scales_expert_stride;
        float acc[4][4] = {};
        for (int k0 = 0; k0 < a.K; k0 += PF_BK) {
            // activations: 64 pairs x 32 k
            for (int i = threadIdx.x; i < PF_BM * PF_BK / 8; i += 256) {
                int r = i / (PF_BK / 8), q = i % (PF_BK / 8);
                int p = p_begin + r;
                float v[8];
                if (p < p_end) {
                    if (SWIGLU) {
                        int tok = a.perm[p] / a.k;
                        uint4 u = *reinterpret_cast<const uint4 *>(a.vec_bf16 + (int64_t)tok * a.K + k0 + 8 * q);
                        uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            v[2 * j] = __uint_as_float(ww[j] << 16);
                            v[2 * j + 1] = __uint_as_float(ww[j] & 0xffff0000u);
                        }
                    } else {
                        const float4 *f = reinterpret_cast<const float4 *>(a.vec_f32 + (int64_t)p * a.K + k0 + 8 * q);
                        float4 f0 = f[0], f1 = f[1];
                        v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w;
                        v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; j++) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 8; j++) xs[8 * q + j][r] = v[j];
            }
            // weights: 64 rows x 32 k, dequantised exactly
            for (int i = threadIdx.x; i < PF_BN * PF_BK / 8; i += 256) {
                int c = i / (PF_BK / 8), q = i % (PF_BK / 8);
                int rr, row;
                if (SWIGLU) {
                    rr = nt * (PF_BN / 2) + (c % (PF_BN / 2));
                    row = rr + (c >= PF_BN / 2 ? a.up_offset : 0);
                } else {
                    rr = nt * PF_BN + c;
                    row = rr;
                }
                float v[8];
                if (rr < a.rows)
                    dq8<BITS>(codes + (int64_t)row * a.row_bytes, a.scale_row, scales + (int64_t)row * a.scale_row,
                              k0 / 32, 8 * q, v);
                else
#pragma unroll
                    for (int j = 0; j < 8; j++) v[j] = 0.f;
#pragma unroll
                for (int j = 0; j < 8; j++) wsm[8 * q + j][c] = v[j];
            }
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < PF_BK; kk++) {
                float xa[4], wb[4];
#pragma unroll
                for (int i = 0; i < 4; i++) xa[i] = xs[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; j++) wb[j] = wsm[kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int j = 0; j < 4; j++) acc[i][j] = fmaf(xa[i], wb[j], acc[i][j]);
            }
            __syncthreads();
        }
        if (SWIGLU) {
            // columns tx*4..tx*4+3: tx < 8 hold gate rows, tx >= 8 the matching up rows
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) gs[ty * 4 + i][tx * 4 + j] = acc[i][j];
            __syncthreads();
            for (int i = threadIdx.x; i < PF_BM * (PF_BN / 2); i += 256) {
                int r = i / (PF_BN / 2), c = i % (PF_BN / 2);
                int p = p_begin + r, row = nt * (PF_BN / 2) + c;
                if (p < p_end && row < a.rows) a.out[(int64_t)p * a.rows + row] = silu(gs[r][c]) * gs[r][c + PF_BN / 2];
            }
            __syncthreads();
        } else {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                int p = p_begin + ty * 4 + i;
                if (p >= p_end) continue;
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    int row = nt * PF_BN + tx * 4 + j;
                    if (row < a.rows) a.out[(int64_t)p * a.rows + row] = acc[i][j];
                }
            }
        }
    }
}

static int64_t rb_of(int bits, int cols) { return bits == 2 ? cols / 4 : cols / 4 + cols / 8; }

struct PfWs {
    int32_t *mt_prefix;
    float *h, *y;
    size_t bytes;
};

static PfWs pf_ws(const moe_expert_arena &A, int T, int k, void *base)
{
    PfWs d;
    size_t n = (size_t)T * k;
    size_t tb = align256((A.E + 1) * sizeof(int32_t));
    size_t hb = align256(n * A.I * sizeof(float));
    size_t yb = align256(n * A.H * sizeof(float));
    char *b = static_cast<char *>(base);
    d.mt_prefix = reinterpret_cast<int32_t *>(b);
    d.h = b ? reinterpret_cast<float *>(b + tb) : nullptr;
    d.y = b ? reinterpret_cast<float *>(b + tb + hb) : nullptr;
    d.bytes = tb + hb + yb;
    return d;
}

size_t prefill_workspace_bytes(const moe_expert_arena &A, int T, int k)
{
    if (prefill_tc_supported(A)) return prefill_tc_workspace_bytes(A, T, k);
    return pf_ws(A, T, k, nullptr).bytes;
}

template <int BITS>
static moe_status run_prefill(const moe_expert_arena &A, const uint16_t *x, int T, const float *w, int k,
                              const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out, moe_dtype dt,
                              int accumulate, const PfWs &d, cudaStream_t s)
{
    tile_prefix_kernel<<<1, 1024, 0, s>>>(offsets, A.E, PF_BM, d.mt_prefix);
    moe_status st = check_launch("tile_prefix");
    if (st != MOE_OK) return st;
    int64_t n = (int64_t)T * k;
    int64_t mt_bound = (n + PF_BM - 1) / PF_BM + A.E;
    int64_t cap = (int64_t)sm_count() * 4;
    PfArgs a = {};
    a.perm = perm;
    a.offsets = offsets;
    a.mt_prefix = d.mt_prefix;
    a.E = A.E;
    a.k = k;
    // gate/up
    a.codes = A.gu_codes;
    a.scales = A.gu_scales;
    a.row_bytes = rb_of(BITS, A.H);
    a.scale_row = A.H / 32;
    a.codes_expert_stride = 2LL * A.I * a.row_bytes;
    a.scales_expert_stride = 2LL * A.I * a.scale_row;
    a.K = A.H;
    a.rows = A.I;
    a.up_offset = A.I;
    a.vec_bf16 = x;
    a.out = d.h;
    int ntn = (A.I + PF_BN / 2 - 1) / (PF_BN / 2);
    int64_t grid = std::min<int64_t>(mt_bound * ntn, cap);
    prefill_ffma_kernel<BITS, true><<<(unsigned)grid, 256, 0, s>>>(a, ntn);
    st = check_launch("prefill_gateup");
    if (st != MOE_OK) return st;
    // down
    PfArgs b = a;
    b.codes = A.d_codes;
    b.scales = A.d_scales;
    b.row_bytes = rb_of(BITS, A.I);
    b.scale_row = A.I / 32;
    b.codes_expert_stride = (int64_t)A.H * b.row_bytes;
    b.scales_expert_stride = (int64_t)A.H * b.scale_row;
    b.K = A.I;
    b.rows = A.H;
    b.up_offset = 0;
    b.vec_bf16 = nullptr;
    b.vec_f32 = d.h;
    b.out = d.y;
    ntn = (A.H + PF_BN - 1) / PF_BN;
    grid = std::min<int64_t>(mt_bound * ntn, cap);
    prefill_ffma_kernel<BITS, false><<<(unsigned)grid, 256, 0, s>>>(b, ntn);
    st = check_launch("prefill_down");
    if (st != MOE_OK) return st;
    return launch_combine(d.y, w, inv, T, k, A.H, out, dt, accumulate, s);
}

moe_status prefill_forward(const moe_expert_arena &A, const uint16_t *x, int T, const int32_t *ids, const float *w,
                           int k, const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out,
                           moe_dtype dt, int accumulate, void *ws, int32_t *dev_status, cudaStream_t s)
{
    (void)ids;
    if (prefill_tc_supported(A))
        return prefill_tc_forward(A, x, T, w, k, offsets, perm, inv, out, dt, accumulate, ws, dev_status, s);
    PfWs d = pf_ws(A, T, k, ws);
    if (A.bits == 2) return run_prefill<2>(A, x, T, w, k, offsets, perm, inv, out, dt, accumulate, d, s);
    return run_prefill<3>(A, x, T, w, k, offsets, perm, inv, out, dt, accumulate, d, s);
}

}  // namespace moe
