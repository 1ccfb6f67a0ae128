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
constexpr int kMaxWarps = 16;  // warps per CTA: 16 for one token, 8 for more
template <int T>
__host__ __device__ constexpr int warps_for() { return T == 1 ? 16 : 8; }
constexpr int kMaxT = 4;
constexpr int kMaxK = 16;
constexpr int kMaxPairs = kMaxT * kMaxK;
constexpr int kMaxCand = 512;  // k lanes x 32 values per lane at most
constexpr int kRB = 4;         // units per phase-B batch (team partial sums)
constexpr int kMaxChunks = 128;  // phase-B / phase-C chunk list entries per CTA
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
    float team[kMaxWarps][kRB][2][kMaxT];  // phase-B partials of each warp
    float wsum[kMaxT][kMaxWarps];
    float wmax_v[kMaxWarps];
    int wmax_i[kMaxWarps];
    float tau_v;
    int tau_i, tau_all, ncand;
    float inv_rms[kMaxT];
    int b_g[kMaxChunks], b_r[kMaxChunks], b_n[kMaxChunks], nb;  // phase-B chunks: group, first row, rows
    int c_g[kMaxChunks], c_n[kMaxChunks], nc;                   // phase-C chunks: first group, groups
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

// ------------------------------------------------------------ async copies
// Every thread copies its share of a contiguous range in 16-byte pieces
// (cp.async, L2-only); a commit group then covers one logical transfer.
__device__ __forceinline__ void cp16(void *dst, const void *src)
{
    uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp8(void *dst, const void *src)
{
    uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp4(void *dst, const void *src)
{
    uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}

// Pieces of 16, 8 or 4 bytes, the largest that the addresses and length allow
// (the host only admits shapes whose rows are multiples of 4 bytes).
__device__ __forceinline__ void copy_range(void *dst, const void *src, uint32_t bytes)
{
    char *d = static_cast<char *>(dst);
    const char *s = static_cast<const char *>(src);
    uint32_t al = (uint32_t)(reinterpret_cast<uintptr_t>(d) | reinterpret_cast<uintptr_t>(s) | bytes);
    if ((al & 15u) == 0) {
        for (uint32_t off = threadIdx.x * 16u; off < bytes; off += blockDim.x * 16u) cp16(d + off, s + off);
    } else if ((al & 7u) == 0) {
        for (uint32_t off = threadIdx.x * 8u; off < bytes; off += blockDim.x * 8u) cp8(d + off, s + off);
    } else {
        for (uint32_t off = threadIdx.x * 4u; off < bytes; off += blockDim.x * 4u) cp4(d + off, s + off);
    }
}

__device__ __forceinline__ void commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until commit group number `gi` (0-based, in commit order) has landed,
// given that `ncommit` groups have been committed.  Waiting for more groups
// than needed is always safe, so larger distances are clamped.
__device__ __forceinline__ void wait_group_index(int gi, int ncommit)
{
    int n = ncommit - 1 - gi;
    if (n <= 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
    else if (n == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else if (n == 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
    else if (n == 3) asm volatile("cp.async.wait_group 3;" ::: "memory");
    else if (n == 4) asm volatile("cp.async.wait_group 4;" ::: "memory");
    else if (n == 5) asm volatile("cp.async.wait_group 5;" ::: "memory");
    else if (n == 6) asm volatile("cp.async.wait_group 6;" ::: "memory");
    else asm volatile("cp.async.wait_group 7;" ::: "memory");
}

__device__ __forceinline__ void wait_all_copies() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ------------------------------------------------------------ routing

// Top-k of one token's logits by one warp.  Every logit is loaded once into
// registers.  The k-th best of the 32 lane maxima bounds the k-th best
// overall, so only values at or before it are candidates, and candidates are
// ranked exactly among themselves.  Returns true for a NaN logit.
__device__ bool topk_warp(const float *__restrict__ l, int E, int k, Routing &R, int t)
{
    int lane = lane_id();
    float v[32];
#pragma unroll
    for (int q = 0; q < 32; q++) {
        int e = lane + 32 * q;
        v[q] = (e < E) ? __ldcg(l + e) : 0.f;
    }
    float mv = 0.f;
    int mi = INT32_MAX;
    bool nan = false;
#pragma unroll
    for (int q = 0; q < 32; q++) {
        int e = lane + 32 * q;
        if (e < E) {
            nan |= isnan(v[q]);
            if (mi == INT32_MAX || before(v[q], e, mv, mi)) {
                mv = v[q];
                mi = e;
            }
        }
    }
    if (__any_sync(0xffffffffu, nan)) {
        if (lane < k) {
            R.sel_i[t][lane] = lane;
            R.sel_v[t][lane] = 0.f;
        }
        __syncwarp();
        return true;
    }
    int rank = 0;
    for (int s = 0; s < 32; s++) {
        float ov = __shfl_sync(0xffffffffu, mv, s);
        int oi = __shfl_sync(0xffffffffu, mi, s);
        if (oi != INT32_MAX && mi != INT32_MAX && before(ov, oi, mv, mi)) rank++;
    }
    unsigned who = __ballot_sync(0xffffffffu, mi != INT32_MAX && rank == k - 1);
    int src = __ffs(who) - 1;  // min(E, 32) >= k valid lane maxima: exactly one has rank k-1
    float tv = __shfl_sync(0xffffffffu, mv, src);
    int ti = __shfl_sync(0xffffffffu, mi, src);
    int base = 0;
#pragma unroll
    for (int q = 0; q < 32; q++) {
        int e = lane + 32 * q;
        bool c = e < E && (before(v[q], e, tv, ti) || (v[q] == tv && e == ti));
        unsigned m = __ballot_sync(0xffffffffu, c);
        if (c) {
            int pos = base + __popc(m & ((1u << lane) - 1u));
            R.cand_v[t][pos] = v[q];
            R.cand_i[t][pos] = e;
        }
        base += __popc(m);
    }
    __syncwarp();
    int C = base;
    for (int c = lane; c < C; c += 32) {
        float cv = R.cand_v[t][c];
        int ce = R.cand_i[t][c];
        int r = 0;
        for (int d = 0; d < C; d++) r += before(R.cand_v[t][d], R.cand_i[t][d], cv, ce) ? 1 : 0;
        if (r < k) {
            R.sel_v[t][r] = cv;
            R.sel_i[t][r] = ce;
        }
    }
    __syncwarp();
    return false;
}

// Top-k of a single token's logits by the whole CTA (T = 1).  Each thread
// holds up to two logits.  With at least k warps holding logits, the k-th
// best warp maximum bounds the k-th best logit, so only logits at or before
// it are candidates (otherwise every logit is); candidates are ranked exactly
// among themselves.  Returns true for a NaN logit.
__device__ bool topk_block(const float *__restrict__ l, int E, int k, Routing &R)
{
    int tid = threadIdx.x, lane = lane_id(), warp = warp_id(), nw = blockDim.x >> 5, nthr = blockDim.x;
    int e0 = tid, e1 = tid + nthr;
    bool h0 = e0 < E, h1 = e1 < E;
    float v0 = h0 ? __ldcg(l + e0) : 0.f, v1 = h1 ? __ldcg(l + e1) : 0.f;
    bool nan = (h0 && isnan(v0)) || (h1 && isnan(v1));
    if (__syncthreads_or(nan)) {
        if (tid < k) {
            R.sel_i[0][tid] = tid;
            R.sel_v[0][tid] = 0.f;
        }
        __syncthreads();
        return true;
    }
    float mv = 0.f;
    int mi = INT32_MAX;
    if (h0) { mv = v0; mi = e0; }
    if (h1 && (mi == INT32_MAX || before(v1, e1, mv, mi))) { mv = v1; mi = e1; }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, mv, o);
        int oi = __shfl_xor_sync(0xffffffffu, mi, o);
        if (oi != INT32_MAX && (mi == INT32_MAX || before(ov, oi, mv, mi))) { mv = ov; mi = oi; }
    }
    if (lane == 0) {
        R.wmax_v[warp] = mv;
        R.wmax_i[warp] = mi;
    }
    if (tid == 0) R.ncand = 0;
    __syncthreads();
    if (warp == 0) {
        float wv = lane < nw ? R.wmax_v[lane] : 0.f;
        int wi = lane < nw ? R.wmax_i[lane] : INT32_MAX;
        int r = 0;
        for (int q = 0; q < nw; q++) {
            int oi = R.wmax_i[q];
            if (oi != INT32_MAX && wi != INT32_MAX && before(R.wmax_v[q], oi, wv, wi)) r++;
        }
        unsigned valid = __ballot_sync(0xffffffffu, wi != INT32_MAX);
        unsigned who = __ballot_sync(0xffffffffu, wi != INT32_MAX && r == k - 1);
        int src = who ? __ffs(who) - 1 : 0;
        float tv = __shfl_sync(0xffffffffu, wv, src);
        int ti = __shfl_sync(0xffffffffu, wi, src);
        if (lane == 0) {
            R.tau_all = __popc(valid) < k;
            R.tau_v = tv;
            R.tau_i = ti;
        }
    }
    __syncthreads();
    float tv = R.tau_v;
    int ti = R.tau_i;
    bool all = R.tau_all;
    float *cv = &R.cand_v[0][0];
    int *ci = &R.cand_i[0][0];
    if (h0 && (all || before(v0, e0, tv, ti) || (v0 == tv && e0 == ti))) {
        int pos = atomicAdd(&R.ncand, 1);
        cv[pos] = v0;
        ci[pos] = e0;
    }
    if (h1 && (all || before(v1, e1, tv, ti) || (v1 == tv && e1 == ti))) {
        int pos = atomicAdd(&R.ncand, 1);
        cv[pos] = v1;
        ci[pos] = e1;
    }
    __syncthreads();
    int C = R.ncand;
    for (int c = tid; c < C; c += nthr) {
        float x = cv[c];
        int e = ci[c], r = 0;
        for (int d = 0; d < C; d++) r += before(cv[d], ci[d], x, e) ? 1 : 0;
        if (r < k) {
            R.sel_v[0][r] = x;
            R.sel_i[0][r] = e;
        }
    }
    __syncthreads();
    return false;
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
// (exact dequantisation through fp16x2 words with exponent of 1.0, then the
// block-sum identity sum (c - mid) v = 2^B sum (1 + c/2^B) v - (2^B + mid) sum v)

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

// One 32-weight chunk of a packed row that sits in shared memory.
template <int BITS>
__device__ __forceinline__ QChunk qload_s(const uint8_t *rowc, const uint16_t *rows, int cols, int chunk)
{
    QChunk c;
    if (BITS == 2) {
        uint2 lo = *reinterpret_cast<const uint2 *>(rowc + 8 * chunk);
        c.lo0 = lo.x;
        c.lo1 = lo.y;
        c.hi = 0;
    } else {
        const uint32_t *lo = reinterpret_cast<const uint32_t *>(rowc + 8 * chunk);
        c.lo0 = lo[0];
        c.lo1 = lo[1];
        c.hi = *reinterpret_cast<const uint32_t *>(rowc + (cols / 4) + 4 * chunk);
    }
    c.s = rows[chunk];
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

// ------------------------------------------------------------ per-CTA plan
// Shapes and shared-memory layout, computed on the host and passed in Args.
struct Plan {
    int rb_gu, sb_gu, rb_d, sb_d;  // bytes per row: codes / scales of gate||up and down
    int C;                         // chunks of 32 along H
    int xsw_stride;                // C + 1 (padding keeps the interleaved copy conflict-free)
    int uB;                        // bytes of one phase-B unit (gate+up row codes and scales)
    int chB;                       // phase-B units per ring buffer
    int gC;                        // bytes of one group's phase-C rows
    int chC;                       // groups per phase-C ring buffer
    int sC;                        // bytes of the shared expert's phase-C rows
    int off_xsw, off_part, off_xown, off_ab, off_c, off_h;  // byte offsets in dynamic shared memory
    int regAB, regC;
    int stage_h;  // 1: phase C reads h and h_s from a padded shared-memory copy
};

// Balanced contiguous split of n items over the grid.
__device__ __forceinline__ void split_range(int n, int c, int G, int &lo, int &hi)
{
    lo = (int)((int64_t)n * c / G);
    hi = (int)((int64_t)n * (c + 1) / G);
}

// Phase A units: router rows [0, E) then shared gate/up row pairs [E, E+Is).
__device__ void issue_a(const Args &a, const Plan &P, const Layer &L, char *ab)
{
    int lo, hi;
    split_range(a.E + (L.swg ? a.Is : 0), blockIdx.x, gridDim.x, lo, hi);
    int r0 = min(lo, a.E), r1 = min(hi, a.E);
    uint32_t rbytes = (uint32_t)(r1 - r0) * a.H * 4u;
    if (r1 > r0) copy_range(ab, L.w_router + (int64_t)r0 * a.H, rbytes);
    int q0 = max(lo, a.E) - a.E, q1 = max(hi, a.E) - a.E;
    if (q1 > q0) {
        uint32_t qb = (uint32_t)(q1 - q0) * a.H * 2u;
        copy_range(ab + rbytes, L.swg + (int64_t)q0 * a.H, qb);
        copy_range(ab + rbytes + qb, L.swu + (int64_t)q0 * a.H, qb);
    }
    commit();
}

// Phase C shared-expert rows [o0, o0+nrows) of Wd_s.
__device__ void issue_cs(const Args &a, const Plan &P, const Layer &L, char *cregion, int o0, int nrows)
{
    if (L.swg && nrows > 0) copy_range(cregion, L.swd + (int64_t)o0 * a.Is, (uint32_t)nrows * a.Is * 2u);
    commit();
}

template <int T>
__device__ void phase_a(const Args &a, const Plan &P, const Layer &L, const float *xs, const char *ab)
{
    int lane = lane_id(), warp = warp_id();
    int lo, hi;
    split_range(a.E + (L.swg ? a.Is : 0), blockIdx.x, gridDim.x, lo, hi);
    int H = a.H;
    int r1 = min(hi, a.E), r0 = min(lo, a.E);
    const char *qbase = ab + (size_t)(r1 - r0) * H * 4;
    int nq = max(hi, a.E) - max(lo, a.E);
    for (int u = lo + warp; u < hi; u += (int)(blockDim.x >> 5)) {
        if (u < a.E) {
            const float4 *wr = reinterpret_cast<const float4 *>(ab + (size_t)(u - r0) * H * 4);
            float acc[T];
#pragma unroll
            for (int t = 0; t < T; t++) acc[t] = 0.f;
#pragma unroll 4
            for (int c = lane; c < (H >> 2); c += 32) {
                float4 w = wr[c];
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
            int q = u - max(lo, a.E);
            int r = u - a.E;
            const uint4 *wg = reinterpret_cast<const uint4 *>(qbase + (size_t)q * H * 2);
            const uint4 *wu = reinterpret_cast<const uint4 *>(qbase + (size_t)(nq + q) * H * 2);
            float g[T], uu[T];
#pragma unroll
            for (int t = 0; t < T; t++) g[t] = uu[t] = 0.f;
#pragma unroll 2
            for (int c = lane; c < (H >> 3); c += 32) {
                uint4 qg = wg[c], qu = wu[c];
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

// Phase-B chunk list: the CTA's range of (group, row) units cut at group
// boundaries and at chB units.
__device__ void plan_b(const Args &a, const Plan &P, Routing &R)
{
    if (threadIdx.x != 0) return;
    int lo, hi;
    split_range(R.ngroups * a.I, blockIdx.x, gridDim.x, lo, hi);
    int n = 0;
    for (int u = lo; u < hi && n < kMaxChunks;) {
        int g = u / a.I, r = u % a.I;
        int nr = min(P.chB, min(hi - u, a.I - r));
        R.b_g[n] = g;
        R.b_r[n] = r;
        R.b_n[n] = nr;
        n++;
        u += nr;
    }
    R.nb = n;
    int covered = n ? (R.b_g[n - 1] * a.I + R.b_r[n - 1] + R.b_n[n - 1]) : lo;
    int nc = 0, gdone = 0;
    for (int g = 0; g < R.ngroups && nc < kMaxChunks; g += P.chC) {
        R.c_g[nc] = g;
        R.c_n[nc] = min(P.chC, R.ngroups - g);
        gdone = g + R.c_n[nc];
        nc++;
    }
    R.nc = nc;
    if (covered < hi || gdone < R.ngroups) set_status(a.status, MOE_ERR_UNSUPPORTED);  // never drop work silently
}

template <int BITS>
__device__ void issue_b(const Args &a, const Plan &P, const Layer &L, const Routing &R, int i, char *ab)
{
    char *buf = ab + (size_t)(i & 1) * (P.regAB / 2);
    int e = R.g_e[R.b_g[i]], r = R.b_r[i], nr = R.b_n[i];
    const uint8_t *codes = L.gu_codes + (int64_t)e * 2 * a.I * P.rb_gu;
    const char *scales = reinterpret_cast<const char *>(L.gu_scales) + (int64_t)e * 2 * a.I * P.sb_gu;
    uint32_t cb = (uint32_t)nr * P.rb_gu, sb = (uint32_t)nr * P.sb_gu;
    copy_range(buf, codes + (int64_t)r * P.rb_gu, cb);
    copy_range(buf + cb, codes + (int64_t)(a.I + r) * P.rb_gu, cb);
    copy_range(buf + 2 * cb, scales + (int64_t)r * P.sb_gu, sb);
    copy_range(buf + 2 * cb + sb, scales + (int64_t)(a.I + r) * P.sb_gu, sb);
    commit();
}

template <int BITS>
__device__ void issue_cr(const Args &a, const Plan &P, const Layer &L, const Routing &R, int j, char *cregion,
                         int o0, int nrows)
{
    char *buf = cregion + P.sC + (size_t)(j & 1) * P.chC * P.gC;
    if (nrows > 0) {
        for (int q = 0; q < R.c_n[j]; q++) {
            int e = R.g_e[R.c_g[j] + q];
            const uint8_t *codes = L.d_codes + (int64_t)e * a.H * P.rb_d + (int64_t)o0 * P.rb_d;
            const char *scales = reinterpret_cast<const char *>(L.d_scales) + (int64_t)e * a.H * P.sb_d + (int64_t)o0 * P.sb_d;
            char *d = buf + (size_t)q * P.gC;
            copy_range(d, codes, (uint32_t)nrows * P.rb_d);
            copy_range(d + (size_t)nrows * P.rb_d, scales, (uint32_t)nrows * P.sb_d);
        }
    }
    commit();
}

// Phase B on one chunk in shared memory: rows r..r+nr of group g, gate and up.
// A team of `team` warps shares each row (one 32-weight chunk per lane).
template <int T, int BITS, int CPL>
__device__ void phase_b_chunk(const Args &a, const Plan &P, const float *xsw, Routing &R, int i, const char *ab,
                              float (&v)[CPL][T][32], float (&X)[CPL][T], int &cur_g)
{
    int lane = lane_id(), warp = warp_id();
    int team = (P.C + 32 * CPL - 1) / (32 * CPL);
    int kw = warp % team, tid_team = warp / team, nteams = (int)(blockDim.x >> 5) / team;
    const char *buf = ab + (size_t)(i & 1) * (P.regAB / 2);
    int g = R.b_g[i], r0 = R.b_r[i], nr = R.b_n[i];
    int n = R.g_n[g], p0 = R.g_p0[g];
    if (g != cur_g) {
        cur_g = g;
#pragma unroll
        for (int c = 0; c < CPL; c++) {
            int chunk = (kw + team * c) * 32 + lane;
            bool active = chunk < P.C;
#pragma unroll
            for (int t = 0; t < T; t++) {
                X[c][t] = 0.f;
                int tok = t < n ? R.perm[p0 + t] / a.k : 0;
                const float *xb = xsw + tok * 32 * P.xsw_stride + chunk;
#pragma unroll
                for (int q = 0; q < 32; q++) v[c][t][q] = (active && t < n) ? xb[q * P.xsw_stride] : 0.f;
#pragma unroll
                for (int q = 0; q < 32; q++) X[c][t] += v[c][t][q];
            }
        }
    }
    const uint8_t *gc = reinterpret_cast<const uint8_t *>(buf);
    const uint8_t *uc = gc + (size_t)nr * P.rb_gu;
    const uint16_t *gs = reinterpret_cast<const uint16_t *>(uc + (size_t)nr * P.rb_gu);
    const uint16_t *us = gs + (size_t)nr * (P.sb_gu / 2);
    int bar_id = 1 + tid_team;
    for (int u0 = tid_team * kRB; u0 < nr; u0 += nteams * kRB) {
        int nbt = min(kRB, nr - u0);
#pragma unroll 1
        for (int b = 0; b < kRB; b++) {
            if (b >= nbt) break;
            int row = u0 + b;
            float pg[T], pu[T];
#pragma unroll
            for (int t = 0; t < T; t++) pg[t] = pu[t] = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; c++) {
                int chunk = (kw + team * c) * 32 + lane;
                if (chunk < P.C) {
                    QChunk cg = qload_s<BITS>(gc + (size_t)row * P.rb_gu, gs + (size_t)row * (P.sb_gu / 2), a.H, chunk);
                    QChunk cu = qload_s<BITS>(uc + (size_t)row * P.rb_gu, us + (size_t)row * (P.sb_gu / 2), a.H, chunk);
                    qdot<T, BITS>(cg, v[c], X[c], pg);
                    qdot<T, BITS>(cu, v[c], X[c], pu);
                }
            }
#pragma unroll
            for (int t = 0; t < T; t++) {
                float sg = warp_sum(pg[t]), su = warp_sum(pu[t]);
                if (lane == 0) {
                    R.team[warp][b][0][t] = sg;
                    R.team[warp][b][1][t] = su;
                }
            }
        }
        if (team > 1) asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(team * 32) : "memory");
        else __syncwarp();
        if (kw == 0 && lane < nbt * T) {
            int b = lane / T, t = lane % T;
            if (t < n) {
                float sg = 0.f, su = 0.f;
                for (int q = 0; q < team; q++) {
                    sg += R.team[warp + q][b][0][t];
                    su += R.team[warp + q][b][1][t];
                }
                a.h[(int64_t)(p0 + t) * a.I + r0 + u0 + b] = silu(sg) * su;
            }
        }
        if (team > 1) asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(team * 32) : "memory");
        else __syncwarp();
    }
}

// Phase C for one chunk of routed groups (weights in shared memory): each
// warp takes whole groups, keeps their h in registers and runs all rows.
// h vectors for phase C: a padded copy in shared memory ([vector][chunk][36]
// floats, conflict-free 16-byte reads) or the workspace in L2.
__device__ __forceinline__ float4 h_load(const Plan &P, const float *hsm, const float *hg, int vec, int K, int lane,
                                         int i)
{
    if (P.stage_h) return *reinterpret_cast<const float4 *>(hsm + ((size_t)vec * (K / 32) + lane) * 36 + 4 * i);
    return __ldcg(reinterpret_cast<const float4 *>(hg + (int64_t)vec * K + 32 * lane) + i);
}

template <int T, int BITS>
__device__ void phase_c_chunk(const Args &a, const Plan &P, Routing &R, int j, const char *cregion, float *part,
                              int nrows, const float *hsm)
{
    int lane = lane_id(), warp = warp_id();
    int np = a.T * a.k, pstride = np + a.T;
    const char *buf = cregion + P.sC + (size_t)(j & 1) * P.chC * P.gC;
    bool active = lane < a.I / 32;
    int half = (nrows + 1) / 2;
    int nw = (int)(blockDim.x >> 5);
    for (int it = warp; it < 2 * R.c_n[j]; it += nw) {
        int q = it >> 1;
        int rr0 = (it & 1) ? half : 0, rr1 = (it & 1) ? nrows : half;
        int g = R.c_g[j] + q;
        int n = R.g_n[g], p0 = R.g_p0[g];
        float v[T][32];
        float X[T];
#pragma unroll
        for (int t = 0; t < T; t++) {
            X[t] = 0.f;
            if (active && t < n) {
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    float4 f = h_load(P, hsm, a.h, p0 + t, a.I, lane, i);
                    v[t][4 * i] = f.x; v[t][4 * i + 1] = f.y; v[t][4 * i + 2] = f.z; v[t][4 * i + 3] = f.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; i++) v[t][i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 32; i++) X[t] += v[t][i];
        }
        const uint8_t *codes = reinterpret_cast<const uint8_t *>(buf + (size_t)q * P.gC);
        const uint16_t *scales = reinterpret_cast<const uint16_t *>(codes + (size_t)nrows * P.rb_d);
        for (int rr = rr0; rr < rr1; rr++) {
            float p[T];
#pragma unroll
            for (int t = 0; t < T; t++) p[t] = 0.f;
            if (active) {
                QChunk c = qload_s<BITS>(codes + (size_t)rr * P.rb_d, scales + (size_t)rr * (P.sb_d / 2), a.I, lane);
                qdot<T, BITS>(c, v, X, p);
            }
#pragma unroll
            for (int t = 0; t < T; t++) {
                float s = warp_sum(p[t]);
                if (lane == 0 && t < n) part[rr * pstride + p0 + t] = s;
            }
        }
    }
}

// Phase C for the shared expert: rows of Wd_s in shared memory, h_s from L2.
template <int T>
__device__ void phase_c_shared(const Args &a, const Plan &P, const char *cregion, float *part, int nrows,
                               const float *hsm_s)
{
    int lane = lane_id(), warp = warp_id();
    int np = a.T * a.k, pstride = np + a.T;
    int Is = a.Is;
    bool active = lane < Is / 32;
    float v[T][32];
#pragma unroll
    for (int t = 0; t < T; t++) {
        if (active) {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                float4 f = h_load(P, hsm_s, a.hs, t, Is, lane, i);
                v[t][4 * i] = f.x; v[t][4 * i + 1] = f.y; v[t][4 * i + 2] = f.z; v[t][4 * i + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; i++) v[t][i] = 0.f;
        }
    }
    for (int rr = warp; rr < nrows; rr += (int)(blockDim.x >> 5)) {
        float p[T];
#pragma unroll
        for (int t = 0; t < T; t++) p[t] = 0.f;
        if (active) {
            const uint4 *wp = reinterpret_cast<const uint4 *>(cregion + (size_t)rr * Is * 2) + 4 * lane;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                uint4 q = wp[j];
                uint32_t w4[4] = {q.x, q.y, q.z, q.w};
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
            if (lane == 0) part[rr * pstride + np + t] = s;
        }
    }
}

template <int T, int BITS>
__global__ void __launch_bounds__(warps_for<T>() * 32, 1) decode_kernel(const __grid_constant__ Args a,
                                                                         const __grid_constant__ Plan P)
{
    constexpr int NW = warps_for<T>();
    constexpr int NT = NW * 32;
    // activations of phase B held per lane: two chunks when they fit, else one chunk and a warp team
    constexpr int CPL = T == 1 ? 2 : 1;
    extern __shared__ __align__(128) char dyn[];
    __shared__ Routing R;
    float *xs = reinterpret_cast<float *>(dyn);                 // [T][H] layer input as fp32
    float *xsw = reinterpret_cast<float *>(dyn + P.off_xsw);    // [T][32][C+1] the same, chunk-interleaved
    float *part = reinterpret_cast<float *>(dyn + P.off_part);  // [rows][T*k + T]
    float *xown = reinterpret_cast<float *>(dyn + P.off_xown);  // [T][rows] this CTA's rows of x
    char *ab = dyn + P.off_ab;                                  // phase A data / phase B ring
    char *cregion = dyn + P.off_c;                              // phase C shared rows + ring
    int o0 = blockIdx.x * a.rows_per_cta;
    int nrows = max(0, min(a.H, o0 + a.rows_per_cta) - o0);
    int np = T * a.k, pstride = np + T;
    int H = a.H;
    unsigned nbar = 0;
    int ncommit = 0;
    for (int i = threadIdx.x; i < T * nrows; i += NT) {
        int t = i / nrows, rr = i % nrows;
        xown[t * nrows + rr] = __ldcg(a.x + (int64_t)t * H + o0 + rr);
    }
    issue_a(a, P, a.L[0], ab);
    int gi_a = ncommit++;
    issue_cs(a, P, a.L[0], cregion, o0, nrows);
    int gi_cs = ncommit++;
    for (int l = 0; l < a.n_layers; l++) {
        const Layer &L = a.L[l];
        // -- layer input: bf16(x / rms(x)) per token; sums of squares in a fixed order
        for (int t = 0; t < T; t++) {
            float ss = 0.f;
            const float4 *xp = reinterpret_cast<const float4 *>(a.x + (int64_t)t * H);
            for (int i = threadIdx.x; i < (H >> 2); i += NT) {
                float4 v = __ldcg(xp + i);
                ss = fmaf(v.x, v.x, ss);
                ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss);
                ss = fmaf(v.w, v.w, ss);
            }
            ss = warp_sum(ss);
            if (lane_id() == 0) R.wsum[t][warp_id()] = ss;
        }
        __syncthreads();
        if (threadIdx.x < T) {
            float inv = 1.0f;
            if (a.rms_eps >= 0.f) {
                float tot = 0.f;
                for (int w = 0; w < NW; w++) tot += R.wsum[threadIdx.x][w];
                inv = 1.0f / sqrtf(tot / (float)H + a.rms_eps);
            }
            R.inv_rms[threadIdx.x] = inv;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < T * (H >> 2); i += NT) {
            int t = i / (H >> 2), c4 = i % (H >> 2);
            float4 v = __ldcg(reinterpret_cast<const float4 *>(a.x + (int64_t)t * H) + c4);
            float inv = R.inv_rms[t];
            float4 o = make_float4(bf16_round(v.x * inv), bf16_round(v.y * inv), bf16_round(v.z * inv),
                                   bf16_round(v.w * inv));
            reinterpret_cast<float4 *>(xs + t * H)[c4] = o;
            int r = 4 * c4;
            float *dst = xsw + t * 32 * P.xsw_stride;
            dst[((r + 0) & 31) * P.xsw_stride + ((r + 0) >> 5)] = o.x;
            dst[((r + 1) & 31) * P.xsw_stride + ((r + 1) >> 5)] = o.y;
            dst[((r + 2) & 31) * P.xsw_stride + ((r + 2) >> 5)] = o.z;
            dst[((r + 3) & 31) * P.xsw_stride + ((r + 3) >> 5)] = o.w;
        }
        // -- phase A from the prefetched rows
        wait_group_index(gi_a, ncommit);
        __syncthreads();
        phase_a<T>(a, P, L, xs, ab);
        if (!grid_barrier(a, R, ++nbar)) { wait_all_copies(); return; }
        // -- routing, redundantly in every CTA
        int w = warp_id();
        if (T == 1) {
            bool nan_token = topk_block(a.logits, a.E, a.k, R);
            if (nan_token && threadIdx.x == 0) set_status(a.status, MOE_ERR_NONFINITE);
            if (w == 0) topk_weights(R, 0, a.k, nan_token);
        } else if (w < T) {
            bool nan_token = topk_warp(a.logits + w * a.E, a.E, a.k, R, w);
            if (nan_token && lane_id() == 0) set_status(a.status, MOE_ERR_NONFINITE);
            topk_weights(R, w, a.k, nan_token);
        }
        __syncthreads();
        if (w == 0) build_groups(R, np);
        __syncthreads();
        if (blockIdx.x == 0 && a.ids_out && threadIdx.x < np) {
            a.ids_out[(int64_t)l * np + threadIdx.x] = R.ids[threadIdx.x];
            a.w_out[(int64_t)l * np + threadIdx.x] = R.w[threadIdx.x];
        }
        plan_b(a, P, R);
        __syncthreads();
        // -- prefetch phase B chunks 0,1 and phase C routed chunks 0,1
        int gi_b[2] = {-1, -1}, gi_c[2] = {-1, -1};
        for (int i = 0; i < 2 && i < R.nb; i++) {
            issue_b<BITS>(a, P, L, R, i, ab);
            gi_b[i] = ncommit++;
        }
        for (int j = 0; j < 2 && j < R.nc; j++) {
            issue_cr<BITS>(a, P, L, R, j, cregion, o0, nrows);
            gi_c[j] = ncommit++;
        }
        // -- phase B
        {
            float v[CPL][T][32];
            float X[CPL][T];
            int cur_g = -1;
            for (int i = 0; i < R.nb; i++) {
                wait_group_index(gi_b[i & 1], ncommit);
                __syncthreads();
                phase_b_chunk<T, BITS, CPL>(a, P, xsw, R, i, ab, v, X, cur_g);
                __syncthreads();
                if (i + 2 < R.nb) {
                    issue_b<BITS>(a, P, L, R, i + 2, ab);
                    gi_b[i & 1] = ncommit++;
                }
            }
        }
        // -- prefetch the next layer's phase A rows (the ring is free now)
        if (l + 1 < a.n_layers) {
            issue_a(a, P, a.L[l + 1], ab);
            gi_a = ncommit++;
        }
        if (!grid_barrier(a, R, ++nbar)) { wait_all_copies(); return; }
        // -- phase C: stage h and h_s (one coalesced pass), then the down projections
        float *hsm = reinterpret_cast<float *>(dyn + P.off_h);
        float *hsm_s = hsm + (size_t)np * (a.I / 32) * 36;
        if (P.stage_h) {
            int n4 = np * (a.I / 4), ns4 = L.swg ? T * (a.Is / 4) : 0;
            for (int i = threadIdx.x; i < n4 + ns4; i += NT) {
                bool sh_ = i >= n4;
                int ii = sh_ ? i - n4 : i;
                int K = sh_ ? a.Is : a.I;
                int vec = ii / (K / 4), e4 = ii % (K / 4);
                float4 f = __ldcg(reinterpret_cast<const float4 *>(sh_ ? a.hs : a.h) + ii);
                float *dst = (sh_ ? hsm_s : hsm) + ((size_t)vec * (K / 32) + (e4 >> 3)) * 36 + 4 * (e4 & 7);
                *reinterpret_cast<float4 *>(dst) = f;
            }
        }
        wait_group_index(gi_cs, ncommit);
        __syncthreads();
        if (L.swg) phase_c_shared<T>(a, P, cregion, part, nrows, hsm_s);
        for (int j = 0; j < R.nc; j++) {
            wait_group_index(gi_c[j & 1], ncommit);
            __syncthreads();
            phase_c_chunk<T, BITS>(a, P, R, j, cregion, part, nrows, hsm);
            __syncthreads();
            if (j + 2 < R.nc) {
                issue_cr<BITS>(a, P, L, R, j + 2, cregion, o0, nrows);
                gi_c[j & 1] = ncommit++;
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nrows * T; i += NT) {
            int rr = i / T, t = i % T;
            float s = 0.f;
            for (int j = 0; j < a.k; j++) s = fmaf(R.w[t * a.k + j], part[rr * pstride + R.inv[t * a.k + j]], s);
            if (L.swg) s += part[rr * pstride + np + t];
            float nx = xown[t * nrows + rr] + s;
            xown[t * nrows + rr] = nx;
            a.x[(int64_t)t * H + o0 + rr] = nx;
        }
        __syncthreads();
        if (l + 1 < a.n_layers) {
            issue_cs(a, P, a.L[l + 1], cregion, o0, nrows);
            gi_cs = ncommit++;
        }
        if (!grid_barrier(a, R, ++nbar)) { wait_all_copies(); return; }
    }
    wait_all_copies();
}

template <int T, int BITS>
static cudaError_t launch(const Args &a, const Plan &P, int grid, size_t smem, cudaStream_t s)
{
    auto fn = decode_kernel<T, BITS>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {const_cast<Args *>(&a), const_cast<Plan *>(&P)};
    return cudaLaunchCooperativeKernel((const void *)fn, dim3(grid), dim3(warps_for<T>() * 32), args, smem, s);
}

template <int T, int BITS>
static cudaError_t occupancy(int *blocks, size_t smem, size_t *static_smem)
{
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, decode_kernel<T, BITS>);
    if (e != cudaSuccess) return e;
    *static_smem = fa.sharedSizeBytes;
    e = cudaFuncSetAttribute(decode_kernel<T, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, decode_kernel<T, BITS>, warps_for<T>() * 32, smem);
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

static size_t al128(size_t n) { return (n + 127) & ~size_t(127); }

// Shared-memory plan; returns false if the shapes do not fit.
static bool make_plan(Plan &P, int T, int H, int I, int E, int k, int Is, int bits, int grid, int rows_per_cta,
                      size_t budget)
{
    P.rb_gu = bits == 2 ? H / 4 : H / 4 + H / 8;
    P.sb_gu = H / 16;
    P.rb_d = bits == 2 ? I / 4 : I / 4 + I / 8;
    P.sb_d = I / 16;
    P.C = H / 32;
    P.xsw_stride = P.C + 1;
    P.uB = 2 * (P.rb_gu + P.sb_gu);
    P.gC = (rows_per_cta * (P.rb_d + P.sb_d) + 15) & ~15;  // ring slots stay 16-byte aligned
    P.sC = (int)al128((size_t)rows_per_cta * Is * 2);
    int unitsA = (E + Is + grid - 1) / grid;
    size_t regA = al128((size_t)unitsA * H * 4);
    size_t fixed = al128((size_t)T * H * 4) + al128((size_t)T * 32 * P.xsw_stride * 4) +
                   al128((size_t)rows_per_cta * (T * k + T) * 4) + al128((size_t)T * rows_per_cta * 4);
    if (fixed + regA >= budget) return false;
    size_t hbytes = al128(((size_t)T * k * (I / 32) + (size_t)T * (Is / 32)) * 36 * 4);
    P.stage_h = fixed + regA + hbytes + (64u << 10) <= budget;  // keep at least 64 KiB for the rings
    if (P.stage_h) fixed += hbytes;
    size_t left = budget - fixed;
    // phase C: shared rows + two ring buffers of up to 8 groups; phase A/B: the rest
    int chC = 8;
    while (chC > 1 && (size_t)P.sC + 2 * (size_t)chC * P.gC > left / 3) chC--;
    size_t regC = al128((size_t)P.sC + 2 * (size_t)chC * P.gC);
    if (regC + regA > left) return false;
    size_t regAB = std::max(regA, (size_t)2 * P.uB);
    regAB = std::min(left - regC, std::max(regAB, (size_t)2 * 32 * P.uB));  // room for 32 units per ring half
    regAB &= ~size_t(255);
    if (regAB < regA || regAB < (size_t)2 * P.uB) return false;
    P.chB = (int)std::min<size_t>((regAB / 2) / P.uB, (size_t)1 << 20);
    P.chC = chC;
    P.regAB = (int)regAB;
    P.regC = (int)regC;
    P.off_xsw = (int)al128((size_t)T * H * 4);
    P.off_part = P.off_xsw + (int)al128((size_t)T * 32 * P.xsw_stride * 4);
    P.off_xown = P.off_part + (int)al128((size_t)rows_per_cta * (T * k + T) * 4);
    P.off_ab = P.off_xown + (int)al128((size_t)T * rows_per_cta * 4);
    P.off_c = P.off_ab + P.regAB;
    P.off_h = P.off_c + P.regC;
    return true;
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
    MOE_REQUIRE(H % 64 == 0 && H >= 64 && (H <= 1024 || H == 2048 || H == 4096),
                "the fused decode takes H a multiple of 64 up to 1024, or 2048 or 4096 (got %d)", H);
    MOE_REQUIRE(I % 64 == 0 && I >= 64 && I <= 1024, "the fused decode takes I a multiple of 64 up to 1024 (got %d)", I);
    MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= kMaxK && k <= E, "1 <= k <= min(E, 16), E <= 1024");
    MOE_REQUIRE(Is >= 0 && Is % 64 == 0 && Is <= 1024, "shared_I must be a multiple of 64 up to 1024 (got %d)", Is);
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
    int per_sm = 0;
    size_t static_smem = 0;
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
    MOE_F_DISPATCH(occupancy, &per_sm, 0, &static_smem)
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "decode kernel attributes: %s", cudaGetErrorString(e));
    int dev = 0, optin = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    size_t budget = (size_t)optin > static_smem + 1024 ? (size_t)optin - static_smem - 1024 : 0;
    Plan P;
    if (!make_plan(P, T, H, I, E, k, Is, bits, grid, a.rows_per_cta, budget))
        return fail(MOE_ERR_UNSUPPORTED, "the fused decode's buffers do not fit in %zu bytes of shared memory "
                    "(T=%d H=%d I=%d E=%d k=%d shared_I=%d)", budget, T, H, I, E, k, Is);
    size_t smem = (size_t)P.off_h + (P.stage_h ? al128(((size_t)T * k * (I / 32) + (size_t)T * (Is / 32)) * 36 * 4) : 0);
    MOE_F_DISPATCH(occupancy, &per_sm, smem, &static_smem)
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "decode occupancy query: %s", cudaGetErrorString(e));
    if (per_sm < 1)
        return fail(MOE_ERR_UNSUPPORTED, "the fused decode kernel does not fit on an SM (%zu bytes of shared memory)",
                    smem);
    cudaStream_t s = to_cuda(stream);
    MOE_CUDA_TRY(cudaMemsetAsync(a.bar, 0, sizeof(unsigned), s));
    MOE_F_DISPATCH(launch, a, P, grid, smem, s)
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
