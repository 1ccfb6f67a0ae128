// gemv.cuh -- grouped, dequant-fused GEMV for decode-sized batches (CUDA
// cores, fp32 arithmetic).
//
// One launch computes, for every group g of vectors that share a weight
// matrix (a routed expert and the tokens that picked it, or the shared
// expert and all tokens):
//     out[p][r] = sum_i W_g[r][i] * v_p[i]            (PLAIN)
//     out[p][r] = silu(G_g[r] . v_p) * (U_g[r] . v_p) (SWIGLU)
//
// Work split.  A row of K weights is cut into 32-weight chunks (one
// quantisation block).  Each lane owns one chunk position and keeps the
// matching 32 entries of every vector of the group in registers; a warp
// covers up to 32 chunks and `wpr` warps split longer rows.  Rows are handed
// out in tasks of R consecutive rows of one group, one task per CTA, and a
// warp loads several rows before using any, so that enough bytes are in
// flight to cover the memory latency.  The per-row sum is a fixed butterfly
// over the lanes of the row, then a fixed sum over the warps that split the
// row, so a vector's result never depends on the other vectors in its group
// (decode is batch-invariant).
//
// Dequantisation (2-bit shown; 3-bit is the same with 3 code bits).  Pairs
// of codes (m, m+8) of a 16-code word are moved to the top two mantissa bits
// of the two halves of an fp16x2 whose exponent is that of 1.0, giving the
// exact values 1 + c/4; then per block, with X = sum_i v_i,
//     sum_i (c_i - 1.5) v_i = 4 * sum_i (1 + c_i/4) v_i - 5.5 * X,
// and the block's fp16 scale multiplies the result.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvMaxR = 64;  // rows per task (upper bound)
constexpr int kGemvNV = 4;     // most vectors per register batch
constexpr int kGemvRB = 4;     // row steps in flight per warp (fewer for wide chunks)

enum GemvMode { GEMV_ROUTED = 0, GEMV_DENSE = 1 };

struct GemvArgs {
    // weights of group 0; group g adds e * expert stride (ROUTED mode)
    const uint8_t *codes;          // packed codes, or bf16 weights
    const uint16_t *scales;        // fp16 block scales (quantised only)
    int64_t codes_expert_stride;   // bytes
    int64_t scales_expert_stride;  // elements
    int64_t row_bytes;             // bytes of one row of codes (or bf16 row)
    int64_t scale_row;             // scales per row (K/32)
    int64_t up_delta;              // SWIGLU: bytes from a gate row to the matching up row
    int64_t up_sdelta;             // SWIGLU: scale elements from a gate row to the up row
    int rows;                      // output rows per group
    int K;                         // reduction length
    int lpr;                       // lanes per row (power of two, 4..32)
    int wpr;                       // warps per row
    int R;                         // rows per task
    int tasks_per_group;
    // vectors
    const uint16_t *vec_bf16;  // [.][K] bf16 (x) or NULL
    const float *vec_f32;      // [.][K] fp32 (h) or NULL
    // grouping
    int mode;
    int k;                   // ROUTED: slots per token
    int T;                   // DENSE: number of vectors
    const int32_t *ids;      // ROUTED: [T][k]
    const int32_t *perm;     // ROUTED: [T*k]
    const int32_t *offsets;  // ROUTED: [E+1]
    int E;
    int vec_by_token;        // ROUTED: vector index = perm[p]/k (x) instead of p (h)
    // output
    float *out;              // [pair or token][rows]
};

// Group g of a ROUTED launch: the g-th distinct expert in sorted pair order,
// found by one warp from perm/ids.  Returns false when g is past the last one.
__device__ __forceinline__ bool find_group(const GemvArgs &a, int g, int &e, int &p0, int &n)
{
    int nvalid = a.offsets[a.E];
    int lane = lane_id();
    int seen = 0;
    for (int base = 0; base < nvalid; base += 32) {
        int p = base + lane;
        bool start = false;
        if (p < nvalid) {
            int ep = a.ids[a.perm[p]];
            start = (p == 0) || (a.ids[a.perm[p - 1]] != ep);
        }
        unsigned m = __ballot_sync(0xffffffffu, start);
        int c = __popc(m);
        if (g < seen + c) {
            int want = g - seen;
            unsigned mm = m;
            for (int i = 0; i < want; i++) mm &= mm - 1;
            p0 = base + __ffs(mm) - 1;
            e = a.ids[a.perm[p0]];
            int end = p0 + 1;
            while (end < nvalid && a.ids[a.perm[end]] == e) end++;
            n = end - p0;
            return true;
        }
        seen += c;
    }
    return false;
}

// ------------------------------------------------------------ chunk dots

__device__ __forceinline__ float2 h2_to_f2(uint32_t bits)
{
    __half2 h = *reinterpret_cast<__half2 *>(&bits);
    return __half22float2(h);
}

template <int S>
__device__ __forceinline__ uint32_t shl(uint32_t w)
{
    if constexpr (S > 0) return w << S;
    else if constexpr (S < 0) return w >> (-S);
    else return w;
}

// sum_i (1 + c_i/4) v[i] for the 16 codes of word w, codes m and m+8 paired.
template <int NV>
__device__ __forceinline__ void dot16_q2(uint32_t w, const float (&v)[NV][32], int off, float (&acc)[NV][2])
{
#define MOE_Q2_PAIR(M)                                                                 \
    {                                                                                  \
        float2 f = h2_to_f2((shl<8 - 2 * (M)>(w) & 0x03000300u) | 0x3C003C00u);       \
        _Pragma("unroll") for (int t = 0; t < NV; t++) {                               \
            acc[t][0] = fmaf(f.x, v[t][off + (M)], acc[t][0]);                         \
            acc[t][1] = fmaf(f.y, v[t][off + (M) + 8], acc[t][1]);                     \
        }                                                                              \
    }
    MOE_Q2_PAIR(0) MOE_Q2_PAIR(1) MOE_Q2_PAIR(2) MOE_Q2_PAIR(3)
    MOE_Q2_PAIR(4) MOE_Q2_PAIR(5) MOE_Q2_PAIR(6) MOE_Q2_PAIR(7)
#undef MOE_Q2_PAIR
}

// sum_i (1 + c_i/8) v[i] for 16 3-bit codes: low bits from w, high bits from
// hw, positioned so code m's high bit is at bit m and code m+8's at m+16.
template <int NV>
__device__ __forceinline__ void dot16_q3(uint32_t w, uint32_t hw, const float (&v)[NV][32], int off,
                                         float (&acc)[NV][2])
{
#define MOE_Q3_PAIR(M)                                                                         \
    {                                                                                          \
        uint32_t b = (shl<7 - 2 * (M)>(w) & 0x01800180u) | (shl<9 - (M)>(hw) & 0x02000200u)    \
                     | 0x3C003C00u;                                                            \
        float2 f = h2_to_f2(b);                                                                \
        _Pragma("unroll") for (int t = 0; t < NV; t++) {                                       \
            acc[t][0] = fmaf(f.x, v[t][off + (M)], acc[t][0]);                                 \
            acc[t][1] = fmaf(f.y, v[t][off + (M) + 8], acc[t][1]);                             \
        }                                                                                      \
    }
    MOE_Q3_PAIR(0) MOE_Q3_PAIR(1) MOE_Q3_PAIR(2) MOE_Q3_PAIR(3)
    MOE_Q3_PAIR(4) MOE_Q3_PAIR(5) MOE_Q3_PAIR(6) MOE_Q3_PAIR(7)
#undef MOE_Q3_PAIR
}

// Weight policies: load one row chunk, then accumulate its dot with NV vectors.
template <int BITS>
struct QuantW {
    static constexpr bool kQuant = true;
    struct Chunk {
        uint32_t lo0, lo1, hi;
        uint16_t s;
    };
    __device__ __forceinline__ static Chunk load(const GemvArgs &a, const uint8_t *rowc, const uint16_t *rows,
                                                 int chunk)
    {
        Chunk c;
        if (BITS == 2) {
            uint2 lo = __ldg(reinterpret_cast<const uint2 *>(rowc + 8 * chunk));
            c.lo0 = lo.x;
            c.lo1 = lo.y;
            c.hi = 0;
        } else {  // 3-bit rows are 12*(K/32) bytes: only 4-byte alignment is guaranteed
            const uint32_t *lo = reinterpret_cast<const uint32_t *>(rowc + 8 * chunk);
            c.lo0 = __ldg(lo);
            c.lo1 = __ldg(lo + 1);
            c.hi = __ldg(reinterpret_cast<const uint32_t *>(rowc + a.scale_row * 8 + 4 * chunk));
        }
        c.s = __ldg(rows + chunk);
        return c;
    }
    template <int NV>
    __device__ __forceinline__ static void dot(const Chunk &c, const float (&v)[NV][32], const float (&X)[NV],
                                               float (&part)[NV])
    {
        float acc[NV][2];
#pragma unroll
        for (int t = 0; t < NV; t++) acc[t][0] = acc[t][1] = 0.f;
        if (BITS == 2) {
            dot16_q2<NV>(c.lo0, v, 0, acc);
            dot16_q2<NV>(c.lo1, v, 16, acc);
        } else {
            // word 0 pairs (m, m+8): high bits at m and m+16, as stored;
            // word 1 pairs (16+m, 24+m): high bits at m+8 and m+24 -> shift by 8
            dot16_q3<NV>(c.lo0, c.hi, v, 0, acc);
            dot16_q3<NV>(c.lo1, c.hi >> 8, v, 16, acc);
        }
        float s = fp16_to_f32(c.s);
        constexpr float kMul = BITS == 2 ? 4.f : 8.f;
        constexpr float kOff = BITS == 2 ? 5.5f : 11.5f;  // 2^B + (2^B - 1)/2
#pragma unroll
        for (int t = 0; t < NV; t++) {
            float bsum = acc[t][0] + acc[t][1];
            part[t] = fmaf(s, fmaf(kMul, bsum, -kOff * X[t]), part[t]);
        }
    }
};

struct Bf16W {
    static constexpr bool kQuant = false;
    struct Chunk {
        uint4 q[4];
    };
    __device__ __forceinline__ static Chunk load(const GemvArgs &, const uint8_t *rowc, const uint16_t *, int chunk)
    {
        Chunk c;
        const uint4 *p = reinterpret_cast<const uint4 *>(rowc + 64 * chunk);
#pragma unroll
        for (int i = 0; i < 4; i++) c.q[i] = __ldg(p + i);
        return c;
    }
    template <int NV>
    __device__ __forceinline__ static void dot(const Chunk &c, const float (&v)[NV][32], const float (&)[NV],
                                               float (&part)[NV])
    {
        float acc[NV][2];
#pragma unroll
        for (int t = 0; t < NV; t++) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint32_t w[4] = {c.q[i].x, c.q[i].y, c.q[i].z, c.q[i].w};
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
                int idx = 8 * i + 2 * j;
#pragma unroll
                for (int t = 0; t < NV; t++) {
                    acc[t][0] = fmaf(lo, v[t][idx], acc[t][0]);
                    acc[t][1] = fmaf(hi, v[t][idx + 1], acc[t][1]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NV; t++) part[t] += acc[t][0] + acc[t][1];
    }
};

// This lane's 32 vector entries for NV vectors, and their block sums.
template <int NV>
__device__ __forceinline__ void load_vectors(const GemvArgs &a, const int (&vidx)[kGemvNV], int chunk, bool active,
                                             float (&v)[NV][32], float (&X)[NV])
{
#pragma unroll
    for (int t = 0; t < NV; t++) {
        X[t] = 0.f;
        if (!active) {
#pragma unroll
            for (int i = 0; i < 32; i++) v[t][i] = 0.f;
            continue;
        }
        if (a.vec_bf16) {
            const uint4 *p = reinterpret_cast<const uint4 *>(a.vec_bf16 + (int64_t)vidx[t] * a.K + 32 * chunk);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                uint4 u = __ldg(p + q);
                uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    v[t][8 * q + 2 * j] = __uint_as_float(w[j] << 16);
                    v[t][8 * q + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
                }
            }
        } else {
            const float4 *p = reinterpret_cast<const float4 *>(a.vec_f32 + (int64_t)vidx[t] * a.K + 32 * chunk);
#pragma unroll
            for (int q = 0; q < 8; q++) {
                float4 f = __ldg(p + q);
                v[t][4 * q] = f.x;
                v[t][4 * q + 1] = f.y;
                v[t][4 * q + 2] = f.z;
                v[t][4 * q + 3] = f.w;
            }
        }
#pragma unroll
        for (int i = 0; i < 32; i++) X[t] += v[t][i];
    }
}

// Rows [r0, r0+R) of one group for vectors vidx[0..NV).  The partial row sums
// of each K-warp land in `part` (shared), indexed [kw][row][mat][t].
template <class W, int NV, bool SWIGLU>
__device__ __forceinline__ void gemv_rows(const GemvArgs &a, const uint8_t *gcodes, const uint16_t *gscales,
                                          const int (&vidx)[kGemvNV], int r0, int R, float *part)
{
    constexpr int NM = SWIGLU ? 2 : 1;
    constexpr int RB = (NV >= 3 || !W::kQuant) ? 2 : kGemvRB;
    int warp = warp_id(), lane = lane_id();
    int kw = warp % a.wpr;                 // K-warp index
    int slot = warp / a.wpr;               // row-slot group
    int slots = kGemvWarps / a.wpr;
    int rpw = 32 / a.lpr;                  // rows per warp step
    int sub = lane / a.lpr;                // row within the warp step
    int chunk = kw * 32 + (lane % a.lpr);  // this lane's 32-weight chunk
    bool active = chunk < a.K / 32;
    float v[NV][32];
    float X[NV];
    load_vectors<NV>(a, vidx, chunk, active, v, X);
    int step = slots * rpw;
    for (int rb = slot * rpw; rb < R; rb += step * RB) {
        typename W::Chunk c[RB][NM];
        bool ok[RB];
#pragma unroll
        for (int b = 0; b < RB; b++) {
            int rr = rb + b * step + sub;
            ok[b] = active && rr < R && (r0 + rr) < a.rows;
#pragma unroll
            for (int m = 0; m < NM; m++) {
                if (ok[b]) {
                    int64_t row = r0 + rr;
                    c[b][m] = W::load(a, gcodes + row * a.row_bytes + (m ? a.up_delta : 0),
                                      gscales + row * a.scale_row + (m ? a.up_sdelta : 0), chunk);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < RB; b++) {
            if (rb + b * step >= R) break;  // warp-uniform
            int rr = rb + b * step + sub;
            float p[NM][NV];
#pragma unroll
            for (int m = 0; m < NM; m++) {
#pragma unroll
                for (int t = 0; t < NV; t++) p[m][t] = 0.f;
                if (ok[b]) W::template dot<NV>(c[b][m], v, X, p[m]);
            }
#pragma unroll
            for (int m = 0; m < NM; m++)
#pragma unroll
                for (int t = 0; t < NV; t++)
                    for (int o = a.lpr >> 1; o; o >>= 1) p[m][t] += __shfl_xor_sync(0xffffffffu, p[m][t], o);
            if ((lane % a.lpr) == 0 && rr < R) {
#pragma unroll
                for (int m = 0; m < NM; m++)
#pragma unroll
                    for (int t = 0; t < NV; t++) part[((kw * kGemvMaxR + rr) * NM + m) * kGemvNV + t] = p[m][t];
            }
        }
    }
}

template <class W, bool SWIGLU, int NVMAX>
__global__ void __launch_bounds__(kGemvThreads, NVMAX == 1 ? 2 : 1) gemv_kernel(GemvArgs a)
{
    constexpr int NM = SWIGLU ? 2 : 1;
    __shared__ float part[kGemvWarps * kGemvMaxR * 2 * kGemvNV];
    __shared__ int s_group[3];
    int g = blockIdx.x / a.tasks_per_group;
    int task = blockIdx.x % a.tasks_per_group;
    int r0 = task * a.R;
    if (r0 >= a.rows) return;
    int R = min(a.R, a.rows - r0);
    int e = 0, p0 = 0, n = a.T;
    if (a.mode == GEMV_ROUTED) {
        if (warp_id() == 0) {
            int ee = -1, pp = 0, nn = 0;
            bool found = find_group(a, g, ee, pp, nn);
            if (lane_id() == 0) {
                s_group[0] = found ? ee : -1;
                s_group[1] = pp;
                s_group[2] = nn;
            }
        }
        __syncthreads();
        e = s_group[0];
        p0 = s_group[1];
        n = s_group[2];
        if (e < 0) return;
    } else if (g > 0) {
        return;
    }
    const uint8_t *gcodes = a.codes + (int64_t)e * a.codes_expert_stride;
    const uint16_t *gscales = W::kQuant ? a.scales + (int64_t)e * a.scales_expert_stride : nullptr;
    for (int v0 = 0; v0 < n; v0 += NVMAX) {
        int nv = min(NVMAX, n - v0);
        int vidx[kGemvNV];
#pragma unroll
        for (int t = 0; t < kGemvNV; t++) {
            int q = v0 + min(t, nv - 1);
            if (a.mode == GEMV_ROUTED) vidx[t] = a.vec_by_token ? a.perm[p0 + q] / a.k : p0 + q;
            else vidx[t] = q;
        }
        if (NVMAX == 1 || nv == 1) gemv_rows<W, 1, SWIGLU>(a, gcodes, gscales, vidx, r0, R, part);
        else if (NVMAX == 2 || nv == 2) gemv_rows<W, (NVMAX >= 2 ? 2 : 1), SWIGLU>(a, gcodes, gscales, vidx, r0, R, part);
        else if (nv == 3) gemv_rows<W, (NVMAX >= 3 ? 3 : 1), SWIGLU>(a, gcodes, gscales, vidx, r0, R, part);
        else gemv_rows<W, NVMAX, SWIGLU>(a, gcodes, gscales, vidx, r0, R, part);
        __syncthreads();
        // sum the K-warps in order, apply the epilogue, store
        for (int i = threadIdx.x; i < R * nv; i += blockDim.x) {
            int rr = i / nv, t = i % nv;
            float acc[NM];
#pragma unroll
            for (int m = 0; m < NM; m++) {
                acc[m] = 0.f;
                for (int kw = 0; kw < a.wpr; kw++) acc[m] += part[((kw * kGemvMaxR + rr) * NM + m) * kGemvNV + t];
            }
            float res = SWIGLU ? silu(acc[0]) * acc[NM - 1] : acc[0];
            int orow = (a.mode == GEMV_ROUTED) ? p0 + v0 + t : v0 + t;
            a.out[(int64_t)orow * a.rows + r0 + rr] = res;
        }
        __syncthreads();
    }
}

// Host: the split parameters for a reduction length K and row count.
inline moe_status gemv_plan(GemvArgs &a, int K, int rows, int groups_max)
{
    int C = K / 32;
    if (C <= 32) {
        int l = 4;  // at least 4 lanes per row keeps a step within kGemvMaxR rows
        while (l < C) l <<= 1;
        a.lpr = l;
        a.wpr = 1;
    } else {
        a.lpr = 32;
        a.wpr = (C + 31) / 32;
        if (a.wpr > kGemvWarps || (kGemvWarps % a.wpr) != 0)
            return fail(MOE_ERR_UNSUPPORTED, "decode GEMV supports reduction lengths up to %d in steps of 1024 above "
                        "1024 (got %d)", 32 * 32 * kGemvWarps, K);
    }
    a.K = K;
    a.rows = rows;
    int rows_per_step = (kGemvWarps / a.wpr) * (32 / a.lpr);
    // aim for about two CTAs per SM over all groups
    int target = 2 * sm_count();
    int tasks = (target + groups_max - 1) / groups_max;
    int R = (rows + tasks - 1) / tasks;
    R = ((R + rows_per_step - 1) / rows_per_step) * rows_per_step;
    if (R > kGemvMaxR) R = (kGemvMaxR / rows_per_step) * rows_per_step;
    if (R < rows_per_step) R = rows_per_step;
    a.R = R;
    a.tasks_per_group = (rows + R - 1) / R;
    return MOE_OK;
}

}  // namespace moe
