// decode_fused.cu -- moe_decode_forward: a stack of MoE layers for up to four
// tokens in one persistent cooperative kernel.
//
// Per layer, with a residual stream x (fp32) and xb = bf16(x):
//   phase A  router logits W_r xb + b, shared gate/up h_s = silu(Wg xb)*(Wu xb)
//   -- grid barrier --
//   phase B  top-k + renormalised softmax (every CTA, redundantly, from the
//            logits), grouping of the (token, slot) pairs by expert, routed
//            gate/up h_p = silu(dq(Wg_e) xb_t) * dq(Wu_e) xb_t
//   -- grid barrier --
//   phase C  routed down dq(Wd_e) h_p and shared down Wd_s h_s for this CTA's
//            output rows, then x[t][o] += sum_j w_tj y_j[o] + S[o] (slot order)
//   -- grid barrier --
// The pages put a router, ten of 512 experts and an always-on shared expert
// in each of 48 layers ("Strata Open-Source Runtime: Running a 125B-Parameter
// Qwen3 Model on a 12GB GPU", section "The Model Itself") and sum the expert
// vectors on the GPU ("How Strata runs a 125-billion-parameter model ...",
// Step 2); verify windows hold up to four tokens ("Strata serves a 125B MoE
// ...", section "Six billion active parameters per token").
//
// Every CTA is resident (cooperative launch); the barriers are a counter in
// the workspace with acquire/release ordering and a %globaltimer deadline
// after which the kernel records MOE_ERR_TIMEOUT and returns.  A token's
// result is computed with a fixed split and reduction order that does not
// depend on the other tokens of the call.
#include "common.cuh"

namespace moe {
namespace fused {

constexpr int kMaxLayers = 64;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxT = 4;
constexpr int kMaxK = 16;
constexpr int kMaxPairs = kMaxT * kMaxK;
constexpr int kMaxCand = 512;  // k lanes x 32 values per lane at most
constexpr int kRB = 4;         // units per phase-B batch
constexpr int kRowBlock = 8;   // rows per phase-C item
constexpr unsigned long long kBarrierTimeoutNs = 2000000000ull;
constexpr unsigned kAbort = 0x80000000u;

struct Layer {
    const uint8_t *gu_codes;
    const uint16_t *gu_scales;
    const uint8_t *d_codes;
    const uint16_t *d_scales;
    const float *w_router;
    const float *bias;
    const uint16_t *swg, *swu, *swd;
};

struct Args {
    Layer L[kMaxLayers];
    int n_layers, T, H, I, E, k, Is, bits;
    int rows_per_cta;
    float rms_eps;     // < 0: no normalisation in front of each layer
    float *x;          // [T][H] residual stream, in/out
    float *logits;     // [T][E]
    float *h;          // [T*k][I] routed h in sorted pair order
    float *hs;         // [T][Is] shared h
    unsigned *bar;     // barrier counter (zero at launch)
    int32_t *ids_out;  // [n_layers][T][k] or NULL
    float *w_out;
    int32_t *status;
};

struct Routing {
    int ids[kMaxPairs];
    float w[kMaxPairs];
    int perm[kMaxPairs];  // sorted position -> flat t*k+j
    int inv[kMaxPairs];   // flat -> sorted position
    int g_e[kMaxPairs], g_p0[kMaxPairs], g_n[kMaxPairs];
    int ngroups;
    float cand_v[kMaxT][kMaxCand];
    int cand_i[kMaxT][kMaxCand];
    float sel_v[kMaxT][kMaxK];
    int sel_i[kMaxT][kMaxK];
    float team[kWarps][kRB][2][kMaxT];  // phase-B partials of each warp
    float wsum[kMaxT][kWarps];
    float inv_rms[kMaxT];
    int abort;
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Grid-wide barrier: every CTA adds one to *bar and waits until it reaches
// `target`.  Gives up after timeout_ns (recording MOE_ERR_TIMEOUT and setting
// the abort bit so the other CTAs stop waiting too).  Returns false when the
// barrier failed; `flag` is a shared-memory word for the CTA-wide answer.
__device__ bool barrier_wait(unsigned *bar, unsigned target, unsigned long long timeout_ns, int32_t *status,
                             int &flag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add(bar, 1u);
        unsigned long long t0 = globaltimer();
        int ab = 0;
        for (;;) {
            unsigned v = ld_acquire(bar);
            if (v & kAbort) { ab = 1; break; }
            if (v >= target) break;
            if (globaltimer() - t0 > timeout_ns) {
                set_status(status, MOE_ERR_TIMEOUT);
                atomicOr(bar, kAbort);
                ab = 1;
                break;
            }
        }
        flag = ab;
    }
    __syncthreads();
    return flag == 0;
}

// Barrier number n (1-based) of the decode kernel.
__device__ __forceinline__ bool grid_barrier(const Args &a, Routing &R, unsigned n)
{
    return barrier_wait(a.bar, n * gridDim.x, kBarrierTimeoutNs, a.status, R.abort);
}

// Self-test of the barrier's time limit: one barrier whose target exceeds the
// number of CTAs by `extra`, so for extra > 0 it can only end by timing out.
__global__ void barrier_probe_kernel(unsigned *bar, unsigned extra, unsigned long long timeout_ns, int32_t *status,
                                     int32_t *passed)
{
    __shared__ int flag;
    bool ok = barrier_wait(bar, gridDim.x + extra, timeout_ns, status, flag);
    if (ok && threadIdx.x == 0) atomicAdd(passed, 1);
}

__device__ __forceinline__ bool before(float av, int ai, float bv, int bi)
{
    return av > bv || (av == bv && ai < bi);
}

// Top-k of one token's logits by one warp.  The k-th best of the 32 lane
// maxima bounds the k-th best overall, so only values ranking at or before
// it are candidates; candidates are ranked exactly among themselves.
__device__ void topk_warp(const float *__restrict__ l, int E, int k, Routing &R, int t, int32_t *status)
{
    int lane = lane_id();
    int nq = (E + 31) >> 5;
    float mv = 0.f;
    int mi = INT32_MAX;
    bool nan = false;
    for (int q = 0; q < nq; q++) {
        int e = lane + 32 * q;
        if (e < E) {
            float v = __ldcg(l + e);
            nan |= isnan(v);
            if (mi == INT32_MAX || before(v, e, mv, mi)) {
                mv = v;
                mi = e;
            }
        }
    }
    if (__any_sync(0xffffffffu, nan)) {
        if (lane == 0) set_status(status, MOE_ERR_NONFINITE);
        if (lane < k) {
            R.sel_i[t][lane] = lane;
            R.sel_v[t][lane] = 0.f;
        }
        __syncwarp();
        return;
    }
    // rank of this lane's maximum among the lane maxima
    int rank = 0;
    for (int s = 0; s < 32; s++) {
        float ov = __shfl_sync(0xffffffffu, mv, s);
        int oi = __shfl_sync(0xffffffffu, mi, s);
        if (oi != INT32_MAX && mi != INT32_MAX && before(ov, oi, mv, mi)) rank++;
    }
    unsigned who = __ballot_sync(0xffffffffu, mi != INT32_MAX && rank == k - 1);
    int src = __ffs(who) - 1;  // min(E, 32) >= k valid lane maxima, so exactly one lane has rank k-1
    float tv = __shfl_sync(0xffffffffu, mv, src);
    int ti = __shfl_sync(0xffffffffu, mi, src);
    // candidates: values at or before the threshold (tv, ti)
    int base = 0;
    for (int q = 0; q < nq; q++) {
        int e = lane + 32 * q;
        bool c = false;
        float v = 0.f;
        if (e < E) {
            v = __ldcg(l + e);
            c = before(v, e, tv, ti) || (v == tv && e == ti);
        }
        unsigned m = __ballot_sync(0xffffffffu, c);
        if (c) {
            int pos = base + __popc(m & ((1u << lane) - 1u));
            R.cand_v[t][pos] = v;
            R.cand_i[t][pos] = e;
        }
        base += __popc(m);
    }
    __syncwarp();
    int C = base;
    for (int c = lane; c < C; c += 32) {
        float v = R.cand_v[t][c];
        int e = R.cand_i[t][c];
        int r = 0;
        for (int d = 0; d < C; d++) r += before(R.cand_v[t][d], R.cand_i[t][d], v, e) ? 1 : 0;
        if (r < k) {
            R.sel_v[t][r] = v;
            R.sel_i[t][r] = e;
        }
    }
    __syncwarp();
}

// Renormalised softmax of the k kept logits of token t (lane j = slot j).
__device__ void topk_weights(Routing &R, int t, int k, bool nan_token)
{
    int lane = lane_id();
    float m = R.sel_v[t][0];
    float p = 0.f;
    float v = lane < k ? R.sel_v[t][lane] : 0.f;
    if (lane < k) {
        if (nan_token) p = 1.f;
        else if (isinf(m)) p = (v == m) ? 1.f : 0.f;
        else p = expf(v - m);
    }
    float z = p;
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < k) {
        R.ids[t * k + lane] = R.sel_i[t][lane];
        R.w[t * k + lane] = p / z;
    }
}

// Sort the T*k pairs by (expert, flat index) and cut them into groups.
__device__ void build_groups(Routing &R, int n)
{
    int lane = lane_id();
    for (int f = lane; f < n; f += 32) {
        int e = R.ids[f], r = 0;
        for (int g = 0; g < n; g++) {
            int eg = R.ids[g];
            r += (eg < e || (eg == e && g < f)) ? 1 : 0;
        }
        R.perm[r] = f;
        R.inv[f] = r;
    }
    __syncwarp();
    int seen = 0;
    for (int b = 0; b < n; b += 32) {
        int p = b + lane;
        bool start = false;
        int e = 0;
        if (p < n) {
            e = R.ids[R.perm[p]];
            start = p == 0 || R.ids[R.perm[p - 1]] != e;
        }
        unsigned m = __ballot_sync(0xffffffffu, start);
        if (start) {
            int g = seen + __popc(m & ((1u << lane) - 1u));
            R.g_e[g] = e;
            R.g_p0[g] = p;
        }
        seen += __popc(m);
    }
    __syncwarp();
    for (int g = lane; g < seen; g += 32) R.g_n[g] = (g + 1 < seen ? R.g_p0[g + 1] : n) - R.g_p0[g];
    if (lane == 0) R.ngroups = seen;
    __syncwarp();
}

// ------------------------------------------------------------ chunk dots
// (exact dequantisation through fp16x2 words with exponent of 1.0; see the
// block-sum identity in gemv.cuh: sum (c - mid) v = 2^B sum (1 + c/2^B) v - (2^B + mid) sum v)

__device__ __forceinline__ float2 h2f(uint32_t b)
{
    __half2 h = *reinterpret_cast<__half2 *>(&b);
    return __half22float2(h);
}

template <int S>
__device__ __forceinline__ uint32_t sh(uint32_t w)
{
    if constexpr (S > 0) return w << S;
    else if constexpr (S < 0) return w >> (-S);
    else return w;
}

template <int NV, int BITS>
__device__ __forceinline__ void dot_word(uint32_t w, uint32_t hw, const float (&v)[NV][32], int off,
                                         float (&acc)[NV][2])
{
#define MOE_F_PAIR(M)                                                                                  \
    {                                                                                                  \
        uint32_t b;                                                                                    \
        if (BITS == 2) b = (sh<8 - 2 * (M)>(w) & 0x03000300u) | 0x3C003C00u;                           \
        else b = (sh<7 - 2 * (M)>(w) & 0x01800180u) | (sh<9 - (M)>(hw) & 0x02000200u) | 0x3C003C00u;  \
        float2 f = h2f(b);                                                                             \
        _Pragma("unroll") for (int t = 0; t < NV; t++) {                                               \
            acc[t][0] = fmaf(f.x, v[t][off + (M)], acc[t][0]);                                         \
            acc[t][1] = fmaf(f.y, v[t][off + (M) + 8], acc[t][1]);                                     \
        }                                                                                              \
    }
    MOE_F_PAIR(0) MOE_F_PAIR(1) MOE_F_PAIR(2) MOE_F_PAIR(3)
    MOE_F_PAIR(4) MOE_F_PAIR(5) MOE_F_PAIR(6) MOE_F_PAIR(7)
#undef MOE_F_PAIR
}

struct QChunk {
    uint32_t lo0, lo1, hi;
    uint16_t s;
};

template <int BITS>
__device__ __forceinline__ QChunk qload(const uint8_t *rowc, const uint16_t *rows, int cols, int chunk)
{
    QChunk c;
    if (BITS == 2) {
        uint2 lo = __ldg(reinterpret_cast<const uint2 *>(rowc + 8 * chunk));
        c.lo0 = lo.x;
        c.lo1 = lo.y;
        c.hi = 0;
    } else {
        const uint32_t *lo = reinterpret_cast<const uint32_t *>(rowc + 8 * chunk);
        c.lo0 = __ldg(lo);
        c.lo1 = __ldg(lo + 1);
        c.hi = __ldg(reinterpret_cast<const uint32_t *>(rowc + (cols / 4) + 4 * chunk));
    }
    c.s = __ldg(rows + chunk);
    return c;
}

template <int NV, int BITS>
__device__ __forceinline__ void qdot(const QChunk &c, const float (&v)[NV][32], const float (&X)[NV], float (&part)[NV])
{
    float acc[NV][2];
#pragma unroll
    for (int t = 0; t < NV; t++) acc[t][0] = acc[t][1] = 0.f;
    dot_word<NV, BITS>(c.lo0, c.hi, v, 0, acc);
    dot_word<NV, BITS>(c.lo1, c.hi >> 8, v, 16, acc);
    float s = fp16_to_f32(c.s);
    constexpr float kMul = BITS == 2 ? 4.f : 8.f;
    constexpr float kOff = BITS == 2 ? 5.5f : 11.5f;
#pragma unroll
    for (int t = 0; t < NV; t++) part[t] = fmaf(s, fmaf(kMul, acc[t][0] + acc[t][1], -kOff * X[t]), part[t]);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf16_round(float f) { return bf16_to_f32(f32_to_bf16(f)); }

// ------------------------------------------------------------ phase A
template <int T>
__device__ void phase_a(const Args &a, const Layer &L, const float *xs)
{
    int lane = lane_id();
    int gw = blockIdx.x * kWarps + warp_id(), nw = gridDim.x * kWarps;
    int H = a.H;
    int units = a.E + (L.swg ? a.Is : 0);
    for (int u = gw; u < units; u += nw) {
        if (u < a.E) {
            const float4 *wr = reinterpret_cast<const float4 *>(L.w_router + (int64_t)u * H);
            float acc[T];
#pragma unroll
            for (int t = 0; t < T; t++) acc[t] = 0.f;
            int n4 = H >> 2;
#pragma unroll 8
            for (int c = lane; c < n4; c += 32) {
                float4 w = __ldg(wr + c);
#pragma unroll
                for (int t = 0; t < T; t++) {
                    float4 xv = *reinterpret_cast<const float4 *>(xs + t * H + 4 * c);
                    acc[t] = fmaf(w.x, xv.x, acc[t]);
                    acc[t] = fmaf(w.y, xv.y, acc[t]);
                    acc[t] = fmaf(w.z, xv.z, acc[t]);
                    acc[t] = fmaf(w.w, xv.w, acc[t]);
                }
            }
            float b = L.bias ? L.bias[u] : 0.f;
#pragma unroll
            for (int t = 0; t < T; t++) {
                float s = warp_sum(acc[t]);
                if (lane == 0) a.logits[t * a.E + u] = s + b;
            }
        } else {
            int r = u - a.E;
            const uint4 *wg = reinterpret_cast<const uint4 *>(L.swg + (int64_t)r * H);
            const uint4 *wu = reinterpret_cast<const uint4 *>(L.swu + (int64_t)r * H);
            float g[T], uu[T];
#pragma unroll
            for (int t = 0; t < T; t++) g[t] = uu[t] = 0.f;
            int n8 = H >> 3;
#pragma unroll 4
            for (int c = lane; c < n8; c += 32) {
                uint4 qg = __ldg(wg + c), qu = __ldg(wu + c);
                uint32_t G[4] = {qg.x, qg.y, qg.z, qg.w}, U[4] = {qu.x, qu.y, qu.z, qu.w};
#pragma unroll
                for (int t = 0; t < T; t++) {
                    const float4 *xp = reinterpret_cast<const float4 *>(xs + t * H + 8 * c);
                    float4 x0 = xp[0], x1 = xp[1];
                    float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        g[t] = fmaf(__uint_as_float(G[j] << 16), xv[2 * j], g[t]);
                        g[t] = fmaf(__uint_as_float(G[j] & 0xffff0000u), xv[2 * j + 1], g[t]);
                        uu[t] = fmaf(__uint_as_float(U[j] << 16), xv[2 * j], uu[t]);
                        uu[t] = fmaf(__uint_as_float(U[j] & 0xffff0000u), xv[2 * j + 1], uu[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < T; t++) {
                float gs = warp_sum(g[t]), us = warp_sum(uu[t]);
                if (lane == 0) a.hs[t * a.Is + r] = silu(gs) * us;
            }
        }
    }
}

// ------------------------------------------------------------ phase B
// Routed gate/up.  A team of `team` warps shares each row (team = ceil(H/1024)
// so that one 32-weight chunk per lane covers the row); units (group, row r)
// are handed out in contiguous ranges per team, in batches of one group.
template <int T, int BITS>
__device__ void phase_b(const Args &a, const Layer &L, const float *xsw, Routing &R)
{
    int lane = lane_id(), warp = warp_id();
    int H = a.H, I = a.I;
    int C = H / 32;
    int team = (C + 31) / 32;
    int kw = warp % team;
    int teams_per_cta = kWarps / team;
    int tid_team = warp / team;
    int gteam = blockIdx.x * teams_per_cta + tid_team, nteams = gridDim.x * teams_per_cta;
    int chunk = kw * 32 + lane;
    bool active = chunk < C;
    int64_t rb = BITS == 2 ? H / 4 : H / 4 + H / 8;
    int64_t expert_codes = 2LL * I * rb, expert_scales = 2LL * I * (H / 32);
    int total = R.ngroups * I;
    int per = (total + nteams - 1) / nteams;
    int u0 = gteam * per, u1 = min(total, u0 + per);
    int bar_id = 1 + tid_team;
    int cur_g = -1;
    float v[T][32];
    float X[T];
    for (int u = u0; u < u1;) {
        int g = u / I;
        int r0 = u % I;
        int nb = min(kRB, min(u1 - u, I - r0));  // stay inside one group
        int n = R.g_n[g], p0 = R.g_p0[g], e = R.g_e[g];
        if (g != cur_g) {
            cur_g = g;
#pragma unroll
            for (int t = 0; t < T; t++) {
                X[t] = 0.f;
                int tok = t < n ? R.perm[p0 + t] / a.k : 0;
#pragma unroll
                for (int i = 0; i < 32; i++) v[t][i] = (active && t < n) ? xsw[tok * H + i * C + chunk] : 0.f;
#pragma unroll
                for (int i = 0; i < 32; i++) X[t] += v[t][i];
            }
        }
        const uint8_t *codes = L.gu_codes + (int64_t)e * expert_codes;
        const uint16_t *scales = L.gu_scales + (int64_t)e * expert_scales;
        QChunk c[kRB][2];
#pragma unroll
        for (int b = 0; b < kRB; b++) {
            if (b < nb && active) {
                int r = r0 + b;
                c[b][0] = qload<BITS>(codes + (int64_t)r * rb, scales + (int64_t)r * (H / 32), H, chunk);
                c[b][1] = qload<BITS>(codes + (int64_t)(I + r) * rb, scales + (int64_t)(I + r) * (H / 32), H, chunk);
            }
        }
#pragma unroll
        for (int b = 0; b < kRB; b++) {
            if (b >= nb) break;
#pragma unroll
            for (int m = 0; m < 2; m++) {
                float p[T];
#pragma unroll
                for (int t = 0; t < T; t++) p[t] = 0.f;
                if (active) qdot<T, BITS>(c[b][m], v, X, p);
#pragma unroll
                for (int t = 0; t < T; t++) {
                    float s = warp_sum(p[t]);
                    if (lane == 0) R.team[warp][b][m][t] = s;
                }
            }
        }
        if (team > 1) asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(team * 32) : "memory");
        else __syncwarp();
        if (kw == 0 && lane < nb * T) {
            int b = lane / T, t = lane % T;
            if (t < n) {
                float gs = 0.f, us = 0.f;
                for (int q = 0; q < team; q++) {
                    gs += R.team[warp + q][b][0][t];
                    us += R.team[warp + q][b][1][t];
                }
                a.h[(int64_t)(p0 + t) * I + r0 + b] = silu(gs) * us;
            }
        }
        if (team > 1) asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(team * 32) : "memory");
        else __syncwarp();
        u += nb;
    }
}

// ------------------------------------------------------------ phase C
// Down projections for this CTA's output rows.  Items are (unit, block of
// kRowBlock rows); unit g < ngroups is a routed group (its pairs' h in
// registers), unit ngroups is the shared expert (all tokens' h_s).
template <int T, int BITS>
__device__ void phase_c(const Args &a, const Layer &L, Routing &R, float *part, int o0, int nrows)
{
    int lane = lane_id(), warp = warp_id();
    int H = a.H, I = a.I;
    int np = a.T * a.k;
    int pstride = np + a.T;
    int units = R.ngroups + (L.swg ? 1 : 0);
    int nblk = (nrows + kRowBlock - 1) / kRowBlock;
    int64_t rb = BITS == 2 ? I / 4 : I / 4 + I / 8;
    int64_t expert_codes = (int64_t)H * rb, expert_scales = (int64_t)H * (I / 32);
    for (int it = warp; it < units * nblk; it += kWarps) {
        int unit = it / nblk, blk = it % nblk;
        int rr0 = blk * kRowBlock, rr1 = min(nrows, rr0 + kRowBlock);
        float v[T][32];
        float X[T];
        if (unit < R.ngroups) {
            int n = R.g_n[unit], p0 = R.g_p0[unit], e = R.g_e[unit];
            bool active = lane < I / 32;
#pragma unroll
            for (int t = 0; t < T; t++) {
                X[t] = 0.f;
                if (active && t < n) {
                    const float4 *hp = reinterpret_cast<const float4 *>(a.h + (int64_t)(p0 + t) * I + 32 * lane);
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        float4 f = __ldcg(hp + q);
                        v[t][4 * q] = f.x; v[t][4 * q + 1] = f.y; v[t][4 * q + 2] = f.z; v[t][4 * q + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i++) v[t][i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 32; i++) X[t] += v[t][i];
            }
            const uint8_t *codes = L.d_codes + (int64_t)e * expert_codes;
            const uint16_t *scales = L.d_scales + (int64_t)e * expert_scales;
            QChunk c[kRowBlock];
#pragma unroll
            for (int b = 0; b < kRowBlock; b++)
                if (rr0 + b < rr1 && active) {
                    int o = o0 + rr0 + b;
                    c[b] = qload<BITS>(codes + (int64_t)o * rb, scales + (int64_t)o * (I / 32), I, lane);
                }
#pragma unroll
            for (int b = 0; b < kRowBlock; b++) {
                if (rr0 + b >= rr1) break;
                float p[T];
#pragma unroll
                for (int t = 0; t < T; t++) p[t] = 0.f;
                if (active) qdot<T, BITS>(c[b], v, X, p);
#pragma unroll
                for (int t = 0; t < T; t++) {
                    float s = warp_sum(p[t]);
                    if (lane == 0 && t < n) part[(rr0 + b) * pstride + p0 + t] = s;
                }
            }
        } else {
            int Is = a.Is;
            bool active = lane < Is / 32;
#pragma unroll
            for (int t = 0; t < T; t++) {
                if (active) {
                    const float4 *hp = reinterpret_cast<const float4 *>(a.hs + (int64_t)t * Is + 32 * lane);
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        float4 f = __ldcg(hp + q);
                        v[t][4 * q] = f.x; v[t][4 * q + 1] = f.y; v[t][4 * q + 2] = f.z; v[t][4 * q + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; i++) v[t][i] = 0.f;
                }
            }
            for (int b0 = rr0; b0 < rr1; b0 += 2) {
                uint4 q[2][4];
#pragma unroll
                for (int b = 0; b < 2; b++)
                    if (b0 + b < rr1 && active) {
                        const uint4 *wp = reinterpret_cast<const uint4 *>(L.swd + (int64_t)(o0 + b0 + b) * Is + 32 * lane);
#pragma unroll
                        for (int j = 0; j < 4; j++) q[b][j] = __ldg(wp + j);
                    }
#pragma unroll
                for (int b = 0; b < 2; b++) {
                    if (b0 + b >= rr1) break;
                    float p[T];
#pragma unroll
                    for (int t = 0; t < T; t++) p[t] = 0.f;
                    if (active) {
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            uint32_t w4[4] = {q[b][j].x, q[b][j].y, q[b][j].z, q[b][j].w};
#pragma unroll
                            for (int i = 0; i < 4; i++) {
                                float lo = __uint_as_float(w4[i] << 16), hi = __uint_as_float(w4[i] & 0xffff0000u);
#pragma unroll
                                for (int t = 0; t < T; t++) {
                                    p[t] = fmaf(lo, v[t][8 * j + 2 * i], p[t]);
                                    p[t] = fmaf(hi, v[t][8 * j + 2 * i + 1], p[t]);
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < T; t++) {
                        float s = warp_sum(p[t]);
                        if (lane == 0) part[(b0 + b) * pstride + np + t] = s;
                    }
                }
            }
        }
    }
}

template <int T, int BITS>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ Args a)
{
    extern __shared__ __align__(16) float dyn[];
    __shared__ Routing R;
    float *xs = dyn;                    // [T][H] bf16(x) as fp32
    float *xsw = dyn + T * a.H;         // [T][32][H/32]: the same, chunk-interleaved for phase B
    float *part = dyn + 2 * T * a.H;    // [rows_per_cta][T*k + T]
    int C = a.H / 32;
    int o0 = blockIdx.x * a.rows_per_cta;
    int nrows = max(0, min(a.H, o0 + a.rows_per_cta) - o0);
    int np = T * a.k;
    unsigned nbar = 0;
    for (int l = 0; l < a.n_layers; l++) {
        const Layer &L = a.L[l];
        // layer input: bf16(x / rms(x)) (or bf16(x)), as fp32 in shared memory.
        // Per-token sum of squares in a fixed order: strided per thread, a warp
        // tree, then the warps in order (independent of the other tokens).
        if (a.rms_eps >= 0.f) {
            for (int t = 0; t < T; t++) {
                float ss = 0.f;
                for (int i = threadIdx.x; i < a.H; i += kThreads) {
                    float v = __ldcg(a.x + (int64_t)t * a.H + i);
                    ss = fmaf(v, v, ss);
                }
                ss = warp_sum(ss);
                if (lane_id() == 0) R.wsum[t][warp_id()] = ss;
            }
            __syncthreads();
            if (threadIdx.x < T) {
                float tot = 0.f;
                for (int w = 0; w < kWarps; w++) tot += R.wsum[threadIdx.x][w];
                R.inv_rms[threadIdx.x] = 1.0f / sqrtf(tot / (float)a.H + a.rms_eps);
            }
            __syncthreads();
        } else if (threadIdx.x < T) {
            R.inv_rms[threadIdx.x] = 1.0f;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < T * a.H; i += kThreads) {
            float v = bf16_round(__ldcg(a.x + i) * R.inv_rms[i / a.H]);
            int t = i / a.H, r = i - t * a.H;
            xs[i] = v;
            xsw[t * a.H + (r & 31) * C + (r >> 5)] = v;
        }
        __syncthreads();
        phase_a<T>(a, L, xs);
        if (!grid_barrier(a, R, ++nbar)) return;
        // routing, redundantly in every CTA
        int w = warp_id();
        bool nan_token = false;
        if (w < T) {
            topk_warp(a.logits + w * a.E, a.E, a.k, R, w, a.status);
            nan_token = false;
            for (int e = lane_id(); e < a.E; e += 32) nan_token |= isnan(__ldcg(a.logits + w * a.E + e));
            nan_token = __any_sync(0xffffffffu, nan_token);
            topk_weights(R, w, a.k, nan_token);
        }
        __syncthreads();
        if (w == 0) build_groups(R, np);
        __syncthreads();
        if (blockIdx.x == 0 && a.ids_out && threadIdx.x < np) {
            a.ids_out[(int64_t)l * np + threadIdx.x] = R.ids[threadIdx.x];
            a.w_out[(int64_t)l * np + threadIdx.x] = R.w[threadIdx.x];
        }
        phase_b<T, BITS>(a, L, xsw, R);
        if (!grid_barrier(a, R, ++nbar)) return;
        phase_c<T, BITS>(a, L, R, part, o0, nrows);
        __syncthreads();
        int pstride = np + T;
        for (int i = threadIdx.x; i < nrows * T; i += kThreads) {
            int rr = i / T, t = i % T;
            float s = 0.f;
            for (int j = 0; j < a.k; j++) s = fmaf(R.w[t * a.k + j], part[rr * pstride + R.inv[t * a.k + j]], s);
            if (L.swg) s += part[rr * pstride + np + t];
            float *xp = a.x + (int64_t)t * a.H + o0 + rr;
            *xp = __ldcg(xp) + s;
        }
        if (!grid_barrier(a, R, ++nbar)) return;
    }
}

template <int T, int BITS>
static cudaError_t launch(const Args &a, int grid, size_t smem, cudaStream_t s)
{
    auto fn = decode_kernel<T, BITS>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {const_cast<Args *>(&a)};
    return cudaLaunchCooperativeKernel((const void *)fn, dim3(grid), dim3(kThreads), args, smem, s);
}

template <int T, int BITS>
static cudaError_t occupancy(int *blocks, size_t smem)
{
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, decode_kernel<T, BITS>, kThreads, smem);
}

struct Ws {
    size_t bar, logits, h, hs, total;
};

static Ws ws_layout(int T, int H, int I, int E, int k, int Is)
{
    Ws w;
    w.bar = 0;
    w.logits = 256;
    w.h = w.logits + align256((size_t)T * E * 4);
    w.hs = w.h + align256((size_t)T * k * I * 4);
    w.total = w.hs + align256((size_t)T * std::max(Is, 1) * 4);
    return w;
}

}  // namespace fused
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_decode_workspace_size(int T, int H, int I, int E, int k, int shared_I, size_t *bytes)
{
    MOE_REQUIRE(bytes, "bytes is NULL");
    MOE_REQUIRE(T >= 1 && T <= fused::kMaxT, "T must be in [1, %d] (got %d)", fused::kMaxT, T);
    MOE_REQUIRE(H > 0 && I > 0 && E > 0 && k > 0 && shared_I >= 0, "positive shapes required");
    *bytes = fused::ws_layout(T, H, I, E, k, shared_I).total;
    return MOE_OK;
}

extern "C" moe_status moe_decode_forward(const moe_layer_weights *layers, int n_layers, float *x, int T, int k,
                                         float rms_eps, int32_t *ids_out, float *w_out, void *ws, size_t ws_bytes,
                                         int32_t *dev_status, moe_stream_t stream)
{
    using namespace fused;
    MOE_REQUIRE(layers && n_layers >= 0, "layers is NULL or n_layers < 0");
    MOE_REQUIRE(n_layers <= kMaxLayers, "at most %d layers per call (got %d)", kMaxLayers, n_layers);
    MOE_REQUIRE(T >= 1 && T <= kMaxT, "T must be in [1, %d] (got %d)", kMaxT, T);
    if (n_layers == 0) return MOE_OK;
    const moe_expert_arena &A0 = layers[0].experts;
    int H = A0.H, I = A0.I, E = A0.E, bits = A0.bits, Is = layers[0].shared_I;
    MOE_REQUIRE(bits == 2 || bits == 3, "bits must be 2 or 3 (got %d)", bits);
    MOE_REQUIRE(H % 32 == 0 && H >= 32 && (H <= 1024 || H == 2048 || H == 4096),
                "the fused decode takes H a multiple of 32 up to 1024, or 2048 or 4096 (got %d)", H);
    MOE_REQUIRE(I % 32 == 0 && I >= 32 && I <= 1024, "the fused decode takes I a multiple of 32 up to 1024 (got %d)", I);
    MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= kMaxK && k <= E, "1 <= k <= min(E, 16), E <= 1024");
    MOE_REQUIRE(Is >= 0 && Is % 32 == 0 && Is <= 1024, "shared_I must be a multiple of 32 up to 1024 (got %d)", Is);
    MOE_REQUIRE(x && aligned16(x), "x must be a 16-byte aligned device pointer");
    MOE_REQUIRE(!ids_out == !w_out, "ids_out and w_out must both be given or both be NULL");
    Args a;
    memset(&a, 0, sizeof a);
    for (int l = 0; l < n_layers; l++) {
        const moe_layer_weights &W = layers[l];
        const moe_expert_arena &A = W.experts;
        MOE_REQUIRE(A.H == H && A.I == I && A.E == E && A.bits == bits && W.shared_I == Is,
                    "layer %d has a different shape from layer 0", l);
        MOE_REQUIRE(A.gu_codes && A.gu_scales && A.d_codes && A.d_scales && W.w_router,
                    "layer %d: NULL weight pointer", l);
        MOE_REQUIRE(aligned16(A.gu_codes) && aligned16(A.gu_scales) && aligned16(A.d_codes) && aligned16(A.d_scales) &&
                    aligned16(W.w_router), "layer %d: weight pointers must be 16-byte aligned", l);
        MOE_REQUIRE(!Is || (W.shared_wg && W.shared_wu && W.shared_wd && aligned16(W.shared_wg) &&
                            aligned16(W.shared_wu) && aligned16(W.shared_wd)),
                    "layer %d: shared expert pointers must be 16-byte aligned and non-NULL", l);
        a.L[l] = {A.gu_codes, A.gu_scales, A.d_codes, A.d_scales, W.w_router, W.bias,
                  Is ? W.shared_wg : nullptr, Is ? W.shared_wu : nullptr, Is ? W.shared_wd : nullptr};
    }
    Ws lay = ws_layout(T, H, I, E, k, Is);
    if (!ws || ws_bytes < lay.total)
        return fail(MOE_ERR_WORKSPACE, "moe_decode_forward needs %zu bytes (%.2f MiB) of workspace, got %zu", lay.total,
                    mib((double)lay.total), ws ? ws_bytes : (size_t)0);
    MOE_REQUIRE(aligned16(ws), "workspace must be 16-byte aligned");
    char *wb = static_cast<char *>(ws);
    a.n_layers = n_layers;
    a.T = T;
    a.H = H;
    a.I = I;
    a.E = E;
    a.k = k;
    a.Is = Is;
    a.bits = bits;
    a.x = x;
    a.rms_eps = rms_eps;
    a.logits = reinterpret_cast<float *>(wb + lay.logits);
    a.h = reinterpret_cast<float *>(wb + lay.h);
    a.hs = reinterpret_cast<float *>(wb + lay.hs);
    a.bar = reinterpret_cast<unsigned *>(wb + lay.bar);
    a.ids_out = ids_out;
    a.w_out = w_out;
    a.status = dev_status;
    int grid = sm_count();
    a.rows_per_cta = (H + grid - 1) / grid;
    size_t smem = (2 * (size_t)T * H + (size_t)a.rows_per_cta * (T * k + T)) * sizeof(float);
    int per_sm = 0;
    cudaError_t e = cudaSuccess;
#define MOE_F_DISPATCH(FN, ...)                                           \
    switch (T * 10 + bits) {                                              \
    case 12: e = FN<1, 2>(__VA_ARGS__); break;                            \
    case 13: e = FN<1, 3>(__VA_ARGS__); break;                            \
    case 22: e = FN<2, 2>(__VA_ARGS__); break;                            \
    case 23: e = FN<2, 3>(__VA_ARGS__); break;                            \
    case 32: e = FN<3, 2>(__VA_ARGS__); break;                            \
    case 33: e = FN<3, 3>(__VA_ARGS__); break;                            \
    case 42: e = FN<4, 2>(__VA_ARGS__); break;                            \
    default: e = FN<4, 3>(__VA_ARGS__); break;                            \
    }
    MOE_F_DISPATCH(occupancy, &per_sm, smem)
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "decode occupancy query: %s", cudaGetErrorString(e));
    if (per_sm < 1)
        return fail(MOE_ERR_UNSUPPORTED, "the fused decode kernel does not fit on an SM (%zu bytes of shared memory)",
                    smem);
    cudaStream_t s = to_cuda(stream);
    MOE_CUDA_TRY(cudaMemsetAsync(a.bar, 0, sizeof(unsigned), s));
    MOE_F_DISPATCH(launch, a, grid, smem, s)
#undef MOE_F_DISPATCH
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cooperative launch of the fused decode: %s", cudaGetErrorString(e));
    return MOE_OK;
}

extern "C" moe_status moe_selftest_barrier(unsigned extra_arrivals, int timeout_ms, void *ws, size_t ws_bytes,
                                           int32_t *dev_status, moe_stream_t stream)
{
    MOE_REQUIRE(timeout_ms >= 1 && timeout_ms <= 5000, "timeout_ms must be in [1, 5000] (got %d)", timeout_ms);
    MOE_REQUIRE(ws && ws_bytes >= 8 && aligned16(ws), "the self-test needs 8 bytes of 16-byte aligned workspace");
    MOE_REQUIRE(extra_arrivals < 0x10000000u, "extra_arrivals too large");
    unsigned *bar = static_cast<unsigned *>(ws);
    int32_t *passed = reinterpret_cast<int32_t *>(bar + 1);
    cudaStream_t s = to_cuda(stream);
    MOE_CUDA_TRY(cudaMemsetAsync(ws, 0, 8, s));
    int grid = sm_count();
    unsigned extra = extra_arrivals;
    unsigned long long tns = (unsigned long long)timeout_ms * 1000000ull;
    void *args[] = {&bar, &extra, &tns, &dev_status, &passed};
    MOE_CUDA_TRY(cudaLaunchCooperativeKernel((const void *)fused::barrier_probe_kernel, dim3(grid), dim3(128), args, 0, s));
    return MOE_OK;
}
