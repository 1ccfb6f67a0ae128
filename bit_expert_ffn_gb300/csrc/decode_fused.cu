// decode_fused.cu -- moe_decode_forward: a stack of MoE layers for up to four
// tokens in one persistent cooperative kernel (one CTA per SM).
//
// Per layer, with a residual stream x (fp32) and u = bf16(x / rms(x)):
//   gather   every CTA reads the whole x (tagged words written by the owners
//            of its rows in the previous layer), normalises it and keeps u in
//            shared memory, both in natural order and as MMA operand pairs
//   A        router logits W_r u + b of this CTA's router rows -> tagged words
//   A'       shared gate/up h_s = silu(Wg u) * (Wu u) of this CTA's rows
//   routing  every CTA reads all logits (tagged words), takes the top-k of
//            each token, the renormalised softmax weights and the groups of
//            (token, slot) pairs that share an expert
//   B        routed gate/up: this CTA's share of the (group, 16-row tile)
//            units, h = silu(dq(Wg_e) u) * dq(Wu_e) u, on the tensor cores
//   -- h counter barrier (also covers h_s) --
//   C        shared down Wd_s h_s (while every pair's h comes into shared
//            memory by one bulk copy), then routed down dq(Wd_e) h of this
//            CTA's output rows, then x[t][o] += sum_j w_tj y_j[o] + S[o]
// The pages put a router, ten of 512 experts and an always-on shared expert
// in each of 48 layers ("Strata Open-Source Runtime: Running a 125B-Parameter
// Qwen3 Model on a 12GB GPU", section "The Model Itself") and sum the expert
// vectors on the GPU ("How Strata runs a 125-billion-parameter model ...",
// Step 2); verify windows hold up to four tokens ("Strata serves a 125B MoE
// ...", section "Six billion active parameters per token").
//
// Weights move by bulk asynchronous copies (TMA; each copy one contiguous run
// of code rows or of their scales) completing on mbarriers; the next layer's
// router and shared-expert rows are fetched while this layer finishes.  Routed products
// run on mma.sync fp16 tensor-core instructions: a 2-/3-bit code c is turned
// into the exact fp16 value c - mid (one LOP3 + one HFMA2 per pair), the
// MMA sums (c - mid)*u exactly per 32-weight block (one block per
// accumulator column), and the block scale is applied in fp32.  The down
// projection's fp32 h enters as two fp16 parts (h = hi + lo to 2^-22), and u
// (bf16) converts to fp16 exactly down to 2^-17, so no operand is rounded
// beyond fp32 accumulation (below 2^-17 by at most 2^-25).  Every wait (mbarrier, counter,
// tagged word) gives up after about 2 s, records MOE_ERR_TIMEOUT and raises an
// abort flag that the other CTAs check.  A token's result is computed by the
// same instruction sequence whatever the other tokens of the call are.
#include "common.cuh"
#include "dequant.cuh"
#include "tc.cuh"

namespace moe {
namespace fused {

constexpr int kMaxLayers = 64;
constexpr int kMaxT = 4;
constexpr int kMaxK = 16;
constexpr int kMaxPairs = kMaxT * kMaxK;
constexpr int kMaxCand = 64;   // top-k logits ranked by one warp
constexpr int kMaxChunks = 4;  // top-k: E <= 1024 logits over >= 256 threads
constexpr int kMaxUnitSlots = 16;
constexpr int kMaxDownSlots = kMaxPairs;
constexpr int kRedV = 256;  // fixed number of partial sums in the RMS reduction
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr unsigned kAbort = 0x80000000u;

// Sixteen warps per CTA whatever the number of tokens: with more than one
// token the tensor-core items run one token at a time (the one-token item's
// 128 registers), so the warps keep enough work in flight.
template <int T>
__host__ __device__ constexpr int warps_for() { return 16; }

// Phase trace for development builds, compiled out unless MOE_DECODE_TRACE is
// defined: thread 0 of every CTA stamps the global timer at the phase
// boundaries of every layer (moe_decode_trace_read copies the stamps out).
#ifdef MOE_DECODE_TRACE
constexpr int kTracePhases = 12;
__device__ unsigned long long g_decode_trace[kMaxLayers][160][kTracePhases];
#define MOE_TRACE(P)                                                                     \
    do {                                                                                 \
        if (threadIdx.x == 0 && blockIdx.x < 160) g_decode_trace[l][blockIdx.x][P] = tc::now_ns(); \
    } while (0)
#else
#define MOE_TRACE(P) \
    do {             \
    } while (0)
#endif

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
    int rpc;           // output rows per CTA (even, <= 16)
    float rms_eps;     // < 0: no normalisation in front of each layer
    float *x;          // [T][H] residual stream, in/out (read at layer 0, written after the last)
    uint64_t *xll;     // [2][T][H] tagged x between layers
    uint64_t *lgll;    // [2][T][E] tagged router logits
    uint32_t *hop;     // [T*k][I/32][2][16] routed h as fp16 operand pairs (high, low parts), sorted pair order
    float *hs;         // [T][Is] shared h
    unsigned *cnt;     // [0] h (and h_s) counter, [2] abort word
    int32_t *ids_out;  // [n_layers][T][k] or NULL
    float *w_out;
    int32_t *status;
    int tail_skip;          // route-tail skip from this rank on (0: off)
    const uint32_t *hot;    // [n_layers][(E + 31) / 32] hot-expert bit masks, or NULL (no cache hints)
};

// Shared-memory plan (host-computed): strides, slot sizes, byte offsets.
struct Plan {
    int cb_gu, sb_gu;                // gate/up code and scale row bytes
    int cb_d, sb_d;                  // down code and scale row bytes
    int unitB, nsu;                  // bytes per unit slot (16 gate + 16 up rows), number of slots
    int downB, nsd;                  // bytes per down slot (16 code rows + scales), number of slots
    int NST, NSD2;                   // gate/up super-tiles (256 wide), down super-tiles (128 wide)
    int rA, sA;                      // max router rows, max shared rows per CTA
    int xp_stride;                   // bytes per block of operand pairs (80: conflict-free 16-byte reads)
    int off_xb, off_xp, off_lg, off_r1, off_r2, off_r3, off_hs, off_pgu, off_pd, off_xown, off_hop;
    int stage_h;                     // h's operand words staged in shared memory for the down items
    int r1B, smem;
};

struct Routing {
    int ids[kMaxPairs];
    float w[kMaxPairs];
    int perm[kMaxPairs];  // sorted position -> flat t*k+j
    int inv[kMaxPairs];   // flat -> sorted position
    int key[kMaxPairs];   // expert of each pair, INT32_MAX for a pair the route-tail skip leaves out
    int g_e[kMaxPairs], g_p0[kMaxPairs], g_n[kMaxPairs];
    int tok_of[kMaxPairs];  // sorted position -> token
    int ngroups;
    int sel_i[kMaxT][kMaxK];
    float sel_v[kMaxT][kMaxK];
    uint32_t lmax[32];              // top-k: maximum of each 32-logit list
    uint32_t cand_k[kMaxCand];      // top-k: logits at or above the threshold
    int cand_i[kMaxCand];
    int ncand;
    float inv_rms[kMaxT];
    float wred[kMaxT][8];
    int u0, nu;                     // this CTA's units [u0, u0 + nu)
    int fills_u[kMaxUnitSlots];     // completed fills per unit slot before this layer
    int fills_d[kMaxDownSlots];
    int ucnt[kMaxUnitSlots];        // finished items of the unit in each slot
    int dcnt[kMaxDownSlots];
    int fillsA, fillsS;             // fills of the router/shared-rows and shared-down barriers
    int abort;
    uint64_t fullU[kMaxUnitSlots];
    uint64_t fullD[kMaxDownSlots];
    uint64_t fullA, fullS, fullH;   // router/shared rows, shared down rows, staged h
};

// ------------------------------------------------------------ memory helpers

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

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t *p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t tagged(float v, unsigned tag)
{
    return (uint64_t)__float_as_uint(v) | ((uint64_t)tag << 32);
}

// One bulk asynchronous copy global -> shared completing on `bar` (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     tc::smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
                 : "memory");
}

// The same copy with an L2 eviction-priority hint (a policy from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            tc::smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(tc::smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// A weight copy: with hot-expert masks given, marked experts' weights carry an
// L2 evict-last hint (they stay in L2 from one decode step to the next) and
// every other weight an evict-first hint; without masks, a plain copy.
// OPT: the kernel variant that honours the options (route-tail skip, hot
// masks); the plain variant compiles them away.
template <bool OPT>
__device__ __forceinline__ void weight_g2s(const Args &a, bool hot, void *dst, const void *src, uint32_t bytes,
                                           uint64_t *bar)
{
    if (!OPT || a.hot == nullptr) bulk_g2s(dst, src, bytes, bar);
    else bulk_g2s_hint(dst, src, bytes, bar, hot ? policy_evict_last() : policy_evict_first());
}

template <bool OPT>
__device__ __forceinline__ bool is_hot(const Args &a, int l, int e)
{
    return OPT && a.hot != nullptr && ((a.hot[(size_t)l * ((a.E + 31) >> 5) + (e >> 5)] >> (e & 31)) & 1u);
}

__device__ __forceinline__ bool aborted(const Args &a) { return (ld_acquire(a.cnt + 2) & kAbort) != 0; }

__device__ __forceinline__ void raise_abort(const Args &a)
{
    set_status(a.status, MOE_ERR_TIMEOUT);
    atomicOr(a.cnt + 2, kAbort);
}

// Wait (one thread) until *c >= target; false on timeout or abort.
__device__ bool wait_counter(const Args &a, const unsigned *c, unsigned target)
{
    unsigned long long t0 = tc::now_ns();
    for (;;) {
        if (ld_acquire(c) >= target) return true;
        if (ld_acquire(a.cnt + 2) & kAbort) return false;
        if (tc::now_ns() - t0 > kTimeoutNs) {
            raise_abort(a);
            return false;
        }
    }
}

// Wait for a tagged word; false on timeout or abort (checked every 64 polls).
__device__ __noinline__ bool wait_word(const Args &a, const uint64_t *p, unsigned tag, uint32_t &v)
{
    unsigned long long t0 = tc::now_ns();
    for (int it = 1;; it++) {
        const uint64_t w = ld_relaxed_u64(p);
        if ((unsigned)(w >> 32) == tag) {
            v = (uint32_t)w;
            return true;
        }
        if ((it & 63) == 0) {
            if (ld_acquire(a.cnt + 2) & kAbort) return false;
            if (tc::now_ns() - t0 > kTimeoutNs) {
                raise_abort(a);
                return false;
            }
        }
    }
}

// Wait until the n words p[0], p[stride], ... all carry `tag` (the slow
// path of a batched poll: the caller then reads them again).
__device__ __noinline__ bool wait_tags(const Args &a, const uint64_t *p, int n, int stride, unsigned tag)
{
#pragma unroll 1
    for (int j = 0; j < n; j++) {
        uint32_t v;
        if (!wait_word(a, p + (size_t)j * stride, tag, v)) return false;
    }
    return true;
}

// Barrier-style self-test used by moe_selftest_barrier: one counter barrier
// whose target exceeds the number of CTAs by `extra`.
__global__ void barrier_probe_kernel(unsigned *bar, unsigned extra, unsigned long long timeout_ns, int32_t *status,
                                     int32_t *passed)
{
    __shared__ int flag;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add(bar, 1u);
        unsigned long long t0 = tc::now_ns();
        int ab = 0;
        for (;;) {
            unsigned v = ld_acquire(bar);
            if (v & kAbort) { ab = 1; break; }
            if (v >= gridDim.x + extra) break;
            if (tc::now_ns() - t0 > timeout_ns) {
                set_status(status, MOE_ERR_TIMEOUT);
                atomicOr(bar, kAbort);
                ab = 1;
                break;
            }
        }
        flag = ab;
    }
    __syncthreads();
    if (flag == 0 && threadIdx.x == 0) atomicAdd(passed, 1);
}

__device__ __forceinline__ bool before(float av, int ai, float bv, int bi)
{
    return av > bv || (av == bv && ai < bi);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------ routing

// Order-preserving 32-bit key of a logit (a larger key is a larger logit;
// -0 counts as +0; every logit's key is >= 0x007FFFFF, so 0 means "none").
__device__ __forceinline__ uint32_t order_key(float v)
{
    if (v == 0.f) v = 0.f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one token's logits (in shared memory) by the whole CTA.  The
// logits fall into 32-entry lists (one per warp and chunk of `threads`
// logits).  The k-th largest list maximum tau is a lower bound of the k-th
// largest logit (the k lists holding the k largest maxima hold k distinct
// logits >= tau), so only logits >= tau can be kept.  When at most
// kMaxCand of them remain, one warp ranks them by (value desc, id asc);
// otherwise every warp pops the k best of each of its lists in order (max
// of the keys; among equal keys the lowest lane, which is the lowest id) and
// one warp merges the sorted lists (max of the heads; among equal heads the
// lowest id).  `ck`, `ci` hold ceil(E/threads) x warps x k entries.  Needs
// E <= 32 * 32 lists.  Returns true for a NaN logit (the token then gets ids
// 0..k-1).
__device__ __noinline__ bool topk_cta(const float *l, int E, int k, Routing &R, int t, uint32_t *ck, int *ci)
{
    const int tid = threadIdx.x, nthr = blockDim.x, lane = lane_id(), warp = warp_id(), nw = nthr >> 5;
    const int nch = (E + nthr - 1) / nthr, nl = nch * nw;
    bool nan = false;
    uint32_t key[kMaxChunks];
#pragma unroll
    for (int c = 0; c < kMaxChunks; c++) {
        key[c] = 0u;
        if (c < nch) {
            const int e = c * nthr + tid;
            if (e < E) {
                const float v = l[e];
                nan |= isnan(v);
                key[c] = order_key(v);
            }
            const uint32_t m = __reduce_max_sync(0xffffffffu, key[c]);
            if (lane == 0) R.lmax[c * nw + warp] = m;
        }
    }
    if (tid == 0) R.ncand = 0;
    if (__syncthreads_or(nan)) {
        if (tid < k) {
            R.sel_i[t][tid] = tid;
            R.sel_v[t][tid] = 0.f;
        }
        __syncthreads();
        return true;
    }
    // tau: the list maximum of rank k-1 under (key desc, list asc); 1 (every
    // logit) when there are fewer than k lists
    uint32_t tau = 1u;
    if (nl >= k) {
        const uint32_t mj = lane < nl ? R.lmax[lane] : 0u;
        int rank = 0;
#pragma unroll 4
        for (int i = 0; i < nl; i++) {
            const uint32_t mi = R.lmax[i];
            rank += (mi > mj) || (mi == mj && i < lane);
        }
        const unsigned at = __ballot_sync(0xffffffffu, lane < nl && rank == k - 1);
        tau = max(__shfl_sync(0xffffffffu, mj, __ffs(at) - 1), 1u);
    }
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int c = 0; c < kMaxChunks; c++) {
        if (c < nch) {
            const bool p = key[c] >= tau;
            const unsigned b = __ballot_sync(0xffffffffu, p);
            if (b) {
                int base = 0;
                if (lane == 0) base = atomicAdd(&R.ncand, __popc(b));
                base = __shfl_sync(0xffffffffu, base, 0);
                const int pos = base + __popc(b & below);
                if (p && pos < kMaxCand) {
                    R.cand_k[pos] = key[c];
                    R.cand_i[pos] = c * nthr + tid;
                }
            }
        }
    }
    __syncthreads();
    const int N = R.ncand;
    if (N <= kMaxCand) {
        if (warp == 0) {
            const bool va = lane < N, vb = lane + 32 < N;
            const uint32_t ka = va ? R.cand_k[lane] : 0u, kb = vb ? R.cand_k[lane + 32] : 0u;
            const int ia = va ? R.cand_i[lane] : INT32_MAX, ib = vb ? R.cand_i[lane + 32] : INT32_MAX;
            int ra = 0, rb = 0;
#pragma unroll 4
            for (int i = 0; i < N; i++) {
                const uint32_t ki = R.cand_k[i];
                const int ii = R.cand_i[i];
                ra += (ki > ka) || (ki == ka && ii < ia);
                rb += (ki > kb) || (ki == kb && ii < ib);
            }
            if (va && ra < k) {
                R.sel_i[t][ra] = ia;
                R.sel_v[t][ra] = l[ia];
            }
            if (vb && rb < k) {
                R.sel_i[t][rb] = ib;
                R.sel_v[t][rb] = l[ib];
            }
        }
        __syncthreads();
        return false;
    }
#pragma unroll
    for (int c = 0; c < kMaxChunks; c++) {
        if (c < nch) {
            uint32_t kc = key[c];
            const int list = c * nw + warp;
#pragma unroll 1
            for (int r = 0; r < k; r++) {
                const uint32_t m = __reduce_max_sync(0xffffffffu, kc);
                const unsigned who = __ballot_sync(0xffffffffu, kc == m && m != 0u);
                const int w = who ? __ffs(who) - 1 : 0;
                if (lane == w) kc = 0u;
                if (lane == 0) {
                    ck[list * k + r] = m;
                    ci[list * k + r] = who ? c * nthr + warp * 32 + w : INT32_MAX;
                }
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        int p = 0;
#pragma unroll 1
        for (int r = 0; r < k; r++) {
            const bool live = lane < nl && p < k;
            const uint32_t hk = live ? ck[lane * k + p] : 0u;
            const int hi = live ? ci[lane * k + p] : INT32_MAX;
            const uint32_t m = __reduce_max_sync(0xffffffffu, hk);
            const int idx = (int)__reduce_min_sync(0xffffffffu, (unsigned)(hk == m ? hi : INT32_MAX));
            if (hk == m && hi == idx) p++;
            if (lane == 0) {
                R.sel_i[t][r] = idx;
                R.sel_v[t][r] = l[idx];
            }
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

// Sort the T*k pairs by (key, flat index) and cut the kept ones (key below
// INT32_MAX) into groups of one expert each (one warp; n <= 64 pairs, two per
// lane, ranks by shuffles).  The pairs left out sort after every kept one.
template <bool OPT>
__device__ void build_groups(Routing &R, int n)
{
    const int lane = lane_id();
    const int *key = OPT ? R.key : R.ids;
    const int e0 = lane < n ? key[lane] : INT32_MAX, e1 = lane + 32 < n ? key[lane + 32] : INT32_MAX;
    const int nk = OPT ? __popc(__ballot_sync(0xffffffffu, lane < n && e0 != INT32_MAX)) +
                             __popc(__ballot_sync(0xffffffffu, lane + 32 < n && e1 != INT32_MAX))
                       : n;
    int r0 = 0, r1 = 0;
    const int n0 = n < 32 ? n : 32;
#pragma unroll 4
    for (int g = 0; g < n0; g++) {
        const int eg = __shfl_sync(0xffffffffu, e0, g);
        r0 += (eg < e0 || (eg == e0 && g < lane)) ? 1 : 0;
        r1 += (eg <= e1) ? 1 : 0;  // g < lane + 32 always
    }
    if (n > 32) {
#pragma unroll 4
        for (int g = 0; g < n - 32; g++) {
            const int eg = __shfl_sync(0xffffffffu, e1, g);
            r0 += (eg < e0) ? 1 : 0;  // g + 32 > lane always
            r1 += (eg < e1 || (eg == e1 && g < lane)) ? 1 : 0;
        }
    }
    if (lane < n) {
        R.perm[r0] = lane;
        R.inv[lane] = r0;
    }
    if (lane + 32 < n) {
        R.perm[r1] = lane + 32;
        R.inv[lane + 32] = r1;
    }
    __syncwarp();
    int seen = 0;
#pragma unroll 1
    for (int b = 0; b < nk; b += 32) {
        const int p = b + lane;
        bool start = false;
        int e = 0;
        if (p < nk) {
            e = key[R.perm[p]];
            start = p == 0 || key[R.perm[p - 1]] != e;
        }
        const unsigned m = __ballot_sync(0xffffffffu, start);
        if (start) {
            const int g = seen + __popc(m & ((1u << lane) - 1u));
            R.g_e[g] = e;
            R.g_p0[g] = p;
        }
        seen += __popc(m);
    }
    __syncwarp();
#pragma unroll 1
    for (int g = lane; g < seen; g += 32) R.g_n[g] = (g + 1 < seen ? R.g_p0[g + 1] : nk) - R.g_p0[g];
    if (lane == 0) R.ngroups = seen;
    __syncwarp();
}

// The expert key of every pair (one warp): its expert id, or INT32_MAX when
// the route-tail skip leaves it out.  From rank a.tail_skip on, a pair is
// left out when no token of the call keeps its expert at a lower rank and the
// expert is not marked hot ("How Strata runs a 125-billion-parameter model
// ...", Step 2, "Verify-window route tail skip": an expert every token of a
// verify window ranks at the tail of its top-10 contributes almost nothing,
// and every expert resident in the fast tier is kept).  The kept pairs'
// weights are left as they are (not renormalised).
__device__ void mark_pairs(const Args &a, Routing &R, int n, int k, int l)
{
    for (int i = lane_id(); i < n; i += 32) {
        const int e = R.ids[i];
        bool drop = false;
        if (a.tail_skip > 0 && i % k >= a.tail_skip && !is_hot<true>(a, l, e)) {
            drop = true;
#pragma unroll 1
            for (int q = 0; q < n; q++)
                if (q % k < a.tail_skip && R.ids[q] == e) drop = false;
        }
        R.key[i] = drop ? INT32_MAX : e;
    }
    __syncwarp();
}

// Token of each sorted pair (k pairs per token).
__device__ void pair_tokens(Routing &R, int n, int k)
{
#pragma unroll 1
    for (int p = lane_id(); p < n; p += 32) R.tok_of[p] = R.perm[p] / k;
    __syncwarp();
}

// ------------------------------------------------------------ tensor-core pieces

// D += A * B for one m16n8k16 tile, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float2 h2f2(uint32_t b)
{
    __half2 h = *reinterpret_cast<__half2 *>(&b);
    return __half22float2(h);
}

__device__ __forceinline__ uint32_t pack16(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

__device__ __forceinline__ uint16_t f16_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ float f16_val(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// B operands of one 256-wide super-tile for the n tokens of a group: word
// i = 8w+m of block 8s+gid as fp16 pairs (16w+m, 16w+m+8).  For T <= 2 two
// copies, one per B register of the MMA, each zero in the lanes that do not
// supply it (loaded from a zero area, so no per-MMA masking); for more tokens
// one copy, masked per MMA.
template <int T>
struct GuOps {
    static constexpr bool kPre = T <= 2;
    uint32_t A[kPre ? T : 1][16], B[kPre ? T : 1][16];
    uint32_t X[kPre ? 1 : T][16];
};

template <int T>
__device__ __forceinline__ void gu_load_ops(GuOps<T> &O, int s, int n, const int (&tok)[kMaxT], const char *xp, int H,
                                            int xp_stride, const uint32_t *zero16)
{
    const int lane = lane_id(), gid = lane >> 2, tig = lane & 3;
    const bool isA = gid == 2 * tig, isB = gid == 2 * tig + 1;
#pragma unroll
    for (int t = 0; t < T; t++) {
        if (t < n) {
            const char *src = xp + ((size_t)tok[t] * (H / 32) + 8 * s + gid) * xp_stride;
            if constexpr (GuOps<T>::kPre) {
                const uint4 *pa = reinterpret_cast<const uint4 *>(isA ? src : reinterpret_cast<const char *>(zero16));
                const uint4 *pb = reinterpret_cast<const uint4 *>(isB ? src : reinterpret_cast<const char *>(zero16));
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const uint4 va = pa[j], vb = pb[j];
                    O.A[t][4 * j] = va.x; O.A[t][4 * j + 1] = va.y; O.A[t][4 * j + 2] = va.z; O.A[t][4 * j + 3] = va.w;
                    O.B[t][4 * j] = vb.x; O.B[t][4 * j + 1] = vb.y; O.B[t][4 * j + 2] = vb.z; O.B[t][4 * j + 3] = vb.w;
                }
            } else {
                const uint4 *px = reinterpret_cast<const uint4 *>(src);
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const uint4 v = px[j];
                    O.X[t][4 * j] = v.x; O.X[t][4 * j + 1] = v.y; O.X[t][4 * j + 2] = v.z; O.X[t][4 * j + 3] = v.w;
                }
            }
        }
    }
}

// One gate/up work item: matrix `mtx` (0 gate, 1 up) of the unit in `slot`,
// super-tile s (columns 256s .. 256s+255), for the n tokens of the unit's
// group.  MMA k-pair j (j < 4) carries block 8s+2j and k-pair j+4 block
// 8s+2j+1, so a thread's A operand is one 16-byte read per row; accumulator
// column c sums block 8s+c.  Writes per-row partial sums (over the
// super-tile's 8 blocks) of s_block * sum_i (c_i - mid) u_i to `pgu`
// [2][NST][16][T].
template <int T, int BITS, int TS = T>
__device__ __forceinline__ void gu_item(const Plan &P, const char *slot, int mtx, int s, int n, const GuOps<T> &O,
                                        int H, float *pgu, int t_off = 0)
{
    const int lane = lane_id(), gid = lane >> 2, tig = lane & 3;
    const int cbr = P.cb_gu;
    const uint8_t *cb = reinterpret_cast<const uint8_t *>(slot) + (size_t)mtx * 16 * cbr;
    const char *sb = slot + 32 * cbr + (size_t)mtx * 16 * P.sb_gu;
    const int bA = 8 * s + 2 * tig;  // blocks bA (k-pair tig) and bA + 1 (k-pair tig + 4)
    const uint4 q0 = *reinterpret_cast<const uint4 *>(cb + (size_t)gid * cbr + bA * 8);
    const uint4 q1 = *reinterpret_cast<const uint4 *>(cb + (size_t)(gid + 8) * cbr + bA * 8);
    uint2 hq0 = make_uint2(0u, 0u), hq1 = make_uint2(0u, 0u);
    if constexpr (BITS == 3) {
        hq0 = *reinterpret_cast<const uint2 *>(cb + (size_t)gid * cbr + H / 4 + bA * 4);
        hq1 = *reinterpret_cast<const uint2 *>(cb + (size_t)(gid + 8) * cbr + H / 4 + bA * 4);
    }
    // operand column gid is block 8s+gid: held by the lane whose k-pair carries that block
    const uint32_t mA = gid == 2 * tig ? 0xffffffffu : 0u, mB = gid == 2 * tig + 1 ? 0xffffffffu : 0u;
    float acc[T][2][4];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int w = 0; w < 2; w++) acc[t][w][0] = acc[t][w][1] = acc[t][w][2] = acc[t][w][3] = 0.f;
#define MOE_GU_STEP(Wn, Mn)                                                                               \
    {                                                                                                     \
        const uint32_t a0 = dq_pair<Mn, BITS, Wn>(D0, H0);                                                \
        const uint32_t a1 = dq_pair<Mn, BITS, Wn>(D1, H1);                                                \
        const uint32_t a2 = dq_pair<Mn, BITS, Wn>(D2, H2);                                                \
        const uint32_t a3 = dq_pair<Mn, BITS, Wn>(D3, H3);                                                \
        _Pragma("unroll") for (int t = 0; t < T; t++) if (t < n) {                                        \
            if constexpr (GuOps<T>::kPre)                                                                 \
                mma16816(acc[t][Wn], a0, a1, a2, a3, O.A[t][8 * Wn + Mn], O.B[t][8 * Wn + Mn]);           \
            else                                                                                          \
                mma16816(acc[t][Wn], a0, a1, a2, a3, O.X[t][8 * Wn + Mn] & mA, O.X[t][8 * Wn + Mn] & mB); \
        }                                                                                                 \
    }
#define MOE_GU_WORD(Wn, X0, X1, X2, X3)                                                                   \
    {                                                                                                     \
        const DqWord<BITS> D0 = dq_word<BITS>(X0), D1 = dq_word<BITS>(X1);                                \
        const DqWord<BITS> D2 = dq_word<BITS>(X2), D3 = dq_word<BITS>(X3);                                \
        const uint32_t H0 = hq0.x, H1 = hq1.x, H2 = hq0.y, H3 = hq1.y;                                    \
        MOE_GU_STEP(Wn, 0) MOE_GU_STEP(Wn, 1) MOE_GU_STEP(Wn, 2) MOE_GU_STEP(Wn, 3)                        \
        MOE_GU_STEP(Wn, 4) MOE_GU_STEP(Wn, 5) MOE_GU_STEP(Wn, 6) MOE_GU_STEP(Wn, 7)                        \
    }
    MOE_GU_WORD(0, q0.x, q1.x, q0.z, q1.z)
    MOE_GU_WORD(1, q0.y, q1.y, q0.w, q1.w)
#undef MOE_GU_WORD
#undef MOE_GU_STEP
    const int bs = 8 * s + 2 * tig;
    const float2 sa = h2f2(*reinterpret_cast<const uint32_t *>(sb + (size_t)gid * P.sb_gu + bs * 2));
    const float2 sc = h2f2(*reinterpret_cast<const uint32_t *>(sb + (size_t)(gid + 8) * P.sb_gu + bs * 2));
#pragma unroll
    for (int t = 0; t < T; t++) {
        if (t < n) {
            const float c0 = acc[t][0][0] + acc[t][1][0], c1 = acc[t][0][1] + acc[t][1][1];
            const float c2 = acc[t][0][2] + acc[t][1][2], c3 = acc[t][0][3] + acc[t][1][3];
            float p0 = sa.x * c0;
            p0 = fmaf(sa.y, c1, p0);
            float p1 = sc.x * c2;
            p1 = fmaf(sc.y, c3, p1);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
            if (tig == 0) {
                const int NST = H / 256;
                pgu[((mtx * NST + s) * 16 + gid) * TS + t_off + t] = p0;
                pgu[((mtx * NST + s) * 16 + gid + 8) * TS + t_off + t] = p1;
            }
        }
    }
}

// One down work item: super-tile s2 (columns 128 s2 .. 128 s2 + 127 of h) of
// the group in `slot` (16 code rows of Wd_e, the CTA's output rows, and their
// scales), for the n tokens of the group.  Accumulator columns are (part,
// block): 0..3 the fp16 high parts of h in the super-tile's four blocks, 4..7
// the low parts, so both parts share one dequantised A operand.  h's operand
// words come from `hop` (shared memory if `staged`, else global).  Writes
// per-row partial sums to pd[(p0 + t) * NSD2 + s2][16].
template <int T, int BITS>
__device__ __forceinline__ void down_item(const Plan &P, const char *slot, int s2, int n, int p0, const uint32_t *hop,
                                          bool staged, const uint32_t *zero16, int I, float *pd)
{
    const int lane = lane_id(), gid = lane >> 2, tig = lane & 3;
    const uint8_t *cb = reinterpret_cast<const uint8_t *>(slot);
    const char *sb = slot + 16 * P.cb_d;
    const int bt = 4 * s2 + tig;  // the block of this thread's A operand
    const uint2 q0 = *reinterpret_cast<const uint2 *>(cb + (size_t)gid * P.cb_d + bt * 8);
    const uint2 q1 = *reinterpret_cast<const uint2 *>(cb + (size_t)(gid + 8) * P.cb_d + bt * 8);
    uint32_t hw0 = 0, hw1 = 0;
    if constexpr (BITS == 3) {
        hw0 = *reinterpret_cast<const uint32_t *>(cb + (size_t)gid * P.cb_d + I / 4 + bt * 4);
        hw1 = *reinterpret_cast<const uint32_t *>(cb + (size_t)(gid + 8) * P.cb_d + I / 4 + bt * 4);
    }
    const bool isA = gid == tig, isB = gid == tig + 4;
    const uint32_t mA = isA ? 0xffffffffu : 0u, mB = isB ? 0xffffffffu : 0u;
    // B operands: the high (isA lanes) or low (isB lanes) fp16 part of h over
    // block bt as pairs (16w+m, 16w+m+8), made by the gate/up epilogue
    constexpr bool kPre = T <= 2;
    uint32_t BA[kPre ? T : 1][16], BB[kPre ? T : 1][16], BX[kPre ? 1 : T][16];
#pragma unroll
    for (int t = 0; t < T; t++) {
        if (t < n) {
            const size_t pb = (size_t)(p0 + t) * (I / 32) + bt;
            const uint32_t *wa = hop + pb * 32, *wb = wa + 16;
            if (kPre && staged) {
                const uint4 *pa = reinterpret_cast<const uint4 *>(isA ? wa : zero16);
                const uint4 *pq = reinterpret_cast<const uint4 *>(isB ? wb : zero16);
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const uint4 va = pa[j], vb = pq[j];
                    BA[kPre ? t : 0][4 * j] = va.x; BA[kPre ? t : 0][4 * j + 1] = va.y;
                    BA[kPre ? t : 0][4 * j + 2] = va.z; BA[kPre ? t : 0][4 * j + 3] = va.w;
                    BB[kPre ? t : 0][4 * j] = vb.x; BB[kPre ? t : 0][4 * j + 1] = vb.y;
                    BB[kPre ? t : 0][4 * j + 2] = vb.z; BB[kPre ? t : 0][4 * j + 3] = vb.w;
                }
            } else {
                uint32_t v[16];
#pragma unroll
                for (int i = 0; i < 16; i++) v[i] = 0u;
                if (isA || isB) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(isB ? wb : wa);
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint4 q = staged ? src[j] : __ldcg(src + j);
                        v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
                    }
                }
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    if constexpr (kPre) {
                        BA[t][i] = v[i] & mA;
                        BB[t][i] = v[i] & mB;
                    } else {
                        BX[kPre ? 0 : t][i] = v[i];
                    }
                }
            }
        }
    }
    float acc[T][2][4];
#pragma unroll
    for (int t = 0; t < T; t++)
#pragma unroll
        for (int w = 0; w < 2; w++) acc[t][w][0] = acc[t][w][1] = acc[t][w][2] = acc[t][w][3] = 0.f;
#define MOE_D_STEP(Wn, Mn)                                                                                \
    {                                                                                                     \
        const uint32_t a0 = dq_pair<Mn, BITS, Wn>(D0, hw0);                                               \
        const uint32_t a1 = dq_pair<Mn, BITS, Wn>(D1, hw1);                                               \
        _Pragma("unroll") for (int t = 0; t < T; t++) if (t < n) {                                        \
            if constexpr (kPre)                                                                           \
                mma16816(acc[t][Wn], a0, a1, a0, a1, BA[t][8 * Wn + Mn], BB[t][8 * Wn + Mn]);             \
            else                                                                                          \
                mma16816(acc[t][Wn], a0, a1, a0, a1, BX[t][8 * Wn + Mn] & mA, BX[t][8 * Wn + Mn] & mB);   \
        }                                                                                                 \
    }
#define MOE_D_WORD(Wn)                                                                                    \
    {                                                                                                     \
        const DqWord<BITS> D0 = dq_word<BITS>(Wn ? q0.y : q0.x), D1 = dq_word<BITS>(Wn ? q1.y : q1.x);      \
        MOE_D_STEP(Wn, 0) MOE_D_STEP(Wn, 1) MOE_D_STEP(Wn, 2) MOE_D_STEP(Wn, 3)                            \
        MOE_D_STEP(Wn, 4) MOE_D_STEP(Wn, 5) MOE_D_STEP(Wn, 6) MOE_D_STEP(Wn, 7)                            \
    }
    MOE_D_WORD(0)
    MOE_D_WORD(1)
#undef MOE_D_WORD
#undef MOE_D_STEP
    const int bb = 4 * s2 + 2 * (tig & 1);  // blocks of accumulator columns 2 tig, 2 tig + 1
    const float2 sa = h2f2(*reinterpret_cast<const uint32_t *>(sb + (size_t)gid * P.sb_d + bb * 2));
    const float2 sc = h2f2(*reinterpret_cast<const uint32_t *>(sb + (size_t)(gid + 8) * P.sb_d + bb * 2));
    const int NSD2 = I / 128;
#pragma unroll
    for (int t = 0; t < T; t++) {
        if (t < n) {
            const float c0 = acc[t][0][0] + acc[t][1][0], c1 = acc[t][0][1] + acc[t][1][1];
            const float c2 = acc[t][0][2] + acc[t][1][2], c3 = acc[t][0][3] + acc[t][1][3];
            float r0 = sa.x * c0;
            r0 = fmaf(sa.y, c1, r0);
            float r1 = sc.x * c2;
            r1 = fmaf(sc.y, c3, r1);
            r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
            r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
            r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
            r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
            if (tig == 0) {
                pd[((size_t)(p0 + t) * NSD2 + s2) * 16 + gid] = r0;
                pd[((size_t)(p0 + t) * NSD2 + s2) * 16 + gid + 8] = r1;
            }
        }
    }
}

// ------------------------------------------------------------ copies (warp-collective issue)

__device__ __forceinline__ void split_range(int n, int c, int G, int &lo, int &hi)
{
    lo = (int)((int64_t)n * c / G);
    hi = (int)((int64_t)n * (c + 1) / G);
}

// Router rows and shared gate/up rows of layer L into region r1 (one thread).
template <bool OPT>
__device__ void issue_a(const Args &a, const Plan &P, const Layer &L, char *r1, uint64_t *bar)
{
    int r0, rh, q0, qh;
    split_range(a.E, blockIdx.x, gridDim.x, r0, rh);
    split_range(a.Is, blockIdx.x, gridDim.x, q0, qh);
    if (!L.swg) qh = q0;
    uint32_t rb = (uint32_t)(rh - r0) * a.H * 4u, qb = (uint32_t)(qh - q0) * a.H * 2u;
    tc::mbar_arrive_expect_tx(bar, rb + 2 * qb);
    if (rb) weight_g2s<OPT>(a, false, r1, L.w_router + (size_t)r0 * a.H, rb, bar);
    if (qb) {
        weight_g2s<OPT>(a, false, r1 + rb, L.swg + (size_t)q0 * a.H, qb, bar);
        weight_g2s<OPT>(a, false, r1 + rb + qb, L.swu + (size_t)q0 * a.H, qb, bar);
    }
}

// Shared down rows [o0, o0 + nrows) of layer L into region r3 (one thread).
template <bool OPT>
__device__ void issue_s(const Args &a, const Layer &L, char *r3, int o0, int nrows, uint64_t *bar)
{
    uint32_t b = (L.swg && nrows > 0) ? (uint32_t)nrows * a.Is * 2u : 0u;
    tc::mbar_arrive_expect_tx(bar, b);
    if (b) weight_g2s<OPT>(a, false, r3, L.swd + (size_t)o0 * a.Is, b, bar);
}

// Unit u (group u / (I/16), rows 16 rt .. 16 rt + 15 of gate and of up) into
// a unit slot, as four contiguous copies: gate codes, up codes (16 rows each),
// gate scales, up scales.  One thread.  l: the layer (for the hot-expert mask).
template <bool OPT>
__device__ void issue_unit(const Args &a, const Plan &P, const Layer &L, const Routing &R, int l, int u, char *slot,
                           uint64_t *bar)
{
    const int tiles = a.I / 16;
    const int g = u / tiles, rt = u % tiles, e = R.g_e[g];
    const size_t rg = (size_t)e * 2 * a.I + 16 * (size_t)rt, ru = rg + a.I;  // first gate row, first up row
    const uint32_t cb = 16u * P.cb_gu, sb = 16u * P.sb_gu;
    const char *sc = reinterpret_cast<const char *>(L.gu_scales);
    tc::fence_proxy_async_smem();
    const bool hot = is_hot<OPT>(a, l, e);
    tc::mbar_arrive_expect_tx(bar, 2 * (cb + sb));
    weight_g2s<OPT>(a, hot, slot, L.gu_codes + rg * P.cb_gu, cb, bar);
    weight_g2s<OPT>(a, hot, slot + cb, L.gu_codes + ru * P.cb_gu, cb, bar);
    weight_g2s<OPT>(a, hot, slot + 2 * cb, sc + rg * P.sb_gu, sb, bar);
    weight_g2s<OPT>(a, hot, slot + 2 * cb + sb, sc + ru * P.sb_gu, sb, bar);
}

// Down rows [o0, o0 + nrows) of group g's expert into a down slot: the code
// rows (contiguous) and their scales, two copies.  One thread.
template <bool OPT>
__device__ void issue_down(const Args &a, const Plan &P, const Layer &L, const Routing &R, int l, int g, int o0,
                           int nrows, char *slot, uint64_t *bar)
{
    const size_t row0 = (size_t)R.g_e[g] * a.H + o0;
    const bool hot = is_hot<OPT>(a, l, R.g_e[g]);
    tc::fence_proxy_async_smem();
    tc::mbar_arrive_expect_tx(bar, (uint32_t)nrows * (P.cb_d + P.sb_d));
    weight_g2s<OPT>(a, hot, slot, L.d_codes + row0 * P.cb_d, (uint32_t)nrows * P.cb_d, bar);
    weight_g2s<OPT>(a, hot, slot + 16 * P.cb_d, reinterpret_cast<const char *>(L.d_scales) + row0 * P.sb_d,
               (uint32_t)nrows * P.sb_d, bar);
}

// The number of fills a ring slot s receives when n items go through nslot slots.
__device__ __forceinline__ int fills_of(int s, int n, int nslot) { return s < n ? (n - 1 - s) / nslot + 1 : 0; }


// h = silu(g) * u for the 16 rows of unit row tile rt (n tokens, sorted pairs
// p0..p0+n-1) from its per-super-tile partial sums, stored as the down
// projection's operand words: fp16 high and low parts paired (16w+m,
// 16w+m+8) in block rt/2, word half w = rt&1.  One warp.
template <int T>
__device__ __forceinline__ void finalize_unit(const Args &a, const float *pslot, int n, int p0, int rt, int I, int NST)
{
    const int lane = lane_id();
    for (int tb = 0; tb < n; tb += 2) {
        const int t = tb + (lane >> 4), r = lane & 15;
        float hv = 0.f;
        if (t < n) {
            float gs = 0.f, us = 0.f;
            for (int s2 = 0; s2 < NST; s2++) {
                gs += pslot[((size_t)s2 * 16 + r) * T + t];
                us += pslot[((size_t)(NST + s2) * 16 + r) * T + t];
            }
            hv = silu(gs) * us;
        }
        if (t < n && !(fabsf(hv) < 65520.f)) set_status(a.status, MOE_ERR_RANGE);  // no finite fp16 part
        const uint16_t hi = f16_bits(hv);
        const uint16_t lo = f16_bits(hv - f16_val(hi));
        const uint16_t hi8 = (uint16_t)__shfl_down_sync(0xffffffffu, (unsigned)hi, 8);
        const uint16_t lo8 = (uint16_t)__shfl_down_sync(0xffffffffu, (unsigned)lo, 8);
        if (t < n) {
            const size_t pb = (size_t)(p0 + t) * (I / 32) + (rt >> 1);
            if (r < 8) {
                __stcg(a.hop + pb * 32 + 8 * (rt & 1) + r, pack16(hi, hi8));
                __stcg(a.hop + pb * 32 + 16 + 8 * (rt & 1) + r, pack16(lo, lo8));
            }
        }
    }
}

// ------------------------------------------------------------ the kernel

template <int T, int BITS, bool OPT>
__global__ void __launch_bounds__(warps_for<T>() * 32, 1) decode_kernel(const __grid_constant__ Args a,
                                                                         const __grid_constant__ Plan P)
{
    constexpr int NW = warps_for<T>();
    constexpr int NT = NW * 32;
    constexpr int kQ = 10;  // H / 256 <= 9 (at most 16 output rows per CTA)
    extern __shared__ __align__(128) char dyn[];
    __shared__ Routing R;
    __shared__ __align__(16) uint32_t zero16[16];  // B operands of lanes that supply none
    __shared__ int iss_u[kMaxUnitSlots], iss_d[kMaxDownSlots], iss_a, iss_s, iss_h;  // fills issued per barrier
    const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
    const int G = gridDim.x, cta = blockIdx.x;
    const int H = a.H, I = a.I, E = a.E, k = a.k, Is = a.Is;
    const int o0 = cta * a.rpc, nrows = max(0, min(H, o0 + a.rpc) - o0);
    const int NST = H / 256, NSD2 = I / 128, tiles = I / 16, per_unit = 2 * NST;
    uint16_t *xb = reinterpret_cast<uint16_t *>(dyn + P.off_xb);  // [T][H] u (bf16)
    char *xp = dyn + P.off_xp;                                     // [T][H/32] blocks of operand pairs
    float *lg = reinterpret_cast<float *>(dyn + P.off_lg);         // [T][E] logits
    char *r1 = dyn + P.off_r1;                                     // router/shared rows, then unit slots
    char *r2 = dyn + P.off_r2;                                     // down slots
    char *r3 = dyn + P.off_r3;                                     // shared down rows
    float *hsm = reinterpret_cast<float *>(dyn + P.off_hs);        // [T][Is] shared h
    float *pgu = reinterpret_cast<float *>(dyn + P.off_pgu);       // [nsu][2][NST][16][T]
    float *pd = reinterpret_cast<float *>(dyn + P.off_pd);         // [T*k][NSD2][16]
    float *xown = reinterpret_cast<float *>(dyn + P.off_xown);     // [T][16] own rows of x
    float *sdn = xown + T * 16;                                    // [T][16] shared down outputs

    if (tid < 16) zero16[tid] = 0u;
    if (tid == 0) {
        for (int s = 0; s < P.nsu; s++) {
            tc::mbar_init(&R.fullU[s], 1);
            R.fills_u[s] = 0;
            R.ucnt[s] = 0;
            iss_u[s] = 0;
        }
        for (int s = 0; s < P.nsd; s++) {
            tc::mbar_init(&R.fullD[s], 1);
            R.fills_d[s] = 0;
            R.dcnt[s] = 0;
            iss_d[s] = 0;
        }
        tc::mbar_init(&R.fullA, 1);
        tc::mbar_init(&R.fullS, 1);
        tc::mbar_init(&R.fullH, 1);
        tc::fence_mbar_init();
        issue_a<OPT>(a, P, a.L[0], r1, &R.fullA);
        issue_s<OPT>(a, a.L[0], r3, o0, nrows, &R.fullS);
        iss_a = 1;
        iss_s = 1;
        iss_h = 0;
    }
    __syncthreads();
    int fillsA = 0, fillsS = 0, fillsH = 0;
    bool ok = true;
    for (int l = 0; l < a.n_layers; l++) {
        const Layer &L = a.L[l];
        bool fail = false;
        MOE_TRACE(0);
        int r0, rh, q0, qh;
        split_range(E, cta, G, r0, rh);
        split_range(Is, cta, G, q0, qh);
        if (!L.swg) qh = q0;
        // the bias of router row r0 + warp, requested now and used in phase A
        const float bias_w = (L.bias && warp < rh - r0) ? __ldg(L.bias + r0 + warp) : 0.f;
        // ---- gather x_l (every CTA, all of it), u = bf16(x * inv_rms)
        const int nq = H / 256;
        float xr[T][kQ];
        if (tid < kRedV) {
            // all of this thread's words are requested before any is checked
            // (one round trip when they are ready), then late ones are polled
            if (l == 0) {
#pragma unroll
                for (int t = 0; t < T; t++)
#pragma unroll
                    for (int q = 0; q < kQ; q++)
                        xr[t][q] = q < nq ? __ldcg(a.x + (size_t)t * H + tid + 256 * q) : 0.f;
            } else {
                const uint64_t *src = a.xll + (size_t)(l & 1) * T * H + tid;
                uint64_t wv[T][kQ];
#pragma unroll 1
                for (;;) {  // read every word; while one is late, wait for it and read them all again
#pragma unroll
                    for (int t = 0; t < T; t++)
#pragma unroll
                        for (int q = 0; q < kQ; q++)
                            wv[t][q] = q < nq ? ld_relaxed_u64(src + (size_t)t * H + 256 * q) : 0;
                    const uint64_t *lp = nullptr;
#pragma unroll
                    for (int t = 0; t < T; t++)
#pragma unroll
                        for (int q = 0; q < kQ; q++)
                            if (!lp && q < nq && (unsigned)(wv[t][q] >> 32) != (unsigned)l) lp = src + (size_t)t * H + 256 * q;
                    if (!lp) break;
                    if (!wait_tags(a, lp, 1, 0, (unsigned)l)) {
                        fail = true;
                        break;
                    }
                }
#pragma unroll
                for (int t = 0; t < T; t++)
#pragma unroll
                    for (int q = 0; q < kQ; q++) xr[t][q] = q < nq ? __uint_as_float((unsigned)wv[t][q]) : 0.f;
            }
#pragma unroll
            for (int t = 0; t < T; t++) {
                float ss = 0.f;
#pragma unroll
                for (int q = 0; q < kQ; q++) {
                    if (q < nq) {
                        const int idx = tid + 256 * q;
                        if (idx >= o0 && idx < o0 + nrows) xown[t * 16 + idx - o0] = xr[t][q];
                        ss = fmaf(xr[t][q], xr[t][q], ss);
                    }
                }
                ss = warp_sum(ss);
                if (lane == 0) R.wred[t][warp] = ss;
            }
        }
        if (__syncthreads_or(fail)) { ok = false; break; }
        MOE_TRACE(1);
        if (tid < T) {
            float inv = 1.0f;
            if (a.rms_eps >= 0.f) {
                float tot = 0.f;
                for (int w = 0; w < kRedV / 32; w++) tot += R.wred[tid][w];
                inv = 1.0f / sqrtf(tot / (float)H + a.rms_eps);
            }
            R.inv_rms[tid] = inv;
        }
        __syncthreads();
        if (tid < kRedV) {
            // warp w holds block 8q+w of every token for each q: u and its MMA
            // operand pairs (16w+m, 16w+m+8) straight from here
#pragma unroll
            for (int t = 0; t < T; t++)
#pragma unroll
                for (int q = 0; q < kQ; q++)
                    if (q < nq) {
                        const int b = 8 * q + warp;
                        const uint16_t uv = f32_to_bf16(xr[t][q] * R.inv_rms[t]);
                        xb[(size_t)t * H + tid + 256 * q] = uv;
                        const float uf = bf16_to_f32(uv);
                        if (!(fabsf(uf) < 65520.f)) set_status(a.status, MOE_ERR_RANGE);  // no finite fp16
                        const uint16_t uh = f16_bits(uf);  // exact for 2^-17 <= |u| < 65520
                        const uint16_t up = (uint16_t)__shfl_down_sync(0xffffffffu, (unsigned)uh, 8);
                        if ((lane & 8) == 0)
                            reinterpret_cast<uint32_t *>(xp + ((size_t)t * (H / 32) + b) * P.xp_stride)
                                [8 * (lane >> 4) + (lane & 7)] = pack16(uh, up);
                    }
        }
        // ---- A: router rows (fp32 weights) -> tagged logits
        bool okA = tc::mbar_wait(&R.fullA, (uint32_t)(fillsA & 1), kTimeoutNs);
        fillsA++;
        if (__syncthreads_or(!okA)) {
            if (tid == 0) raise_abort(a);
            ok = false;
            break;
        }
        MOE_TRACE(2);
        // items: this CTA's router rows, then its shared gate/up rows (A'),
        // spread over the warps; A' overlaps the wait for the other CTAs' logits,
        // and the h counter after phase B also covers h_s
        const int nra = rh - r0, nqa = qh - q0;
        for (int item = warp; item < nra + nqa; item += NW) {
            if (item < nra) {
                const float4 *wr = reinterpret_cast<const float4 *>(r1 + (size_t)item * H * 4);
                float acc[T];
#pragma unroll
                for (int t = 0; t < T; t++) acc[t] = 0.f;
#pragma unroll 4
                for (int cc = lane; cc < (H >> 2); cc += 32) {
                    const float4 w = wr[cc];
#pragma unroll
                    for (int t = 0; t < T; t++) {
                        const uint2 ub = *reinterpret_cast<const uint2 *>(xb + (size_t)t * H + 4 * cc);
                        acc[t] = fmaf(w.x, __uint_as_float(ub.x << 16), acc[t]);
                        acc[t] = fmaf(w.y, __uint_as_float(ub.x & 0xffff0000u), acc[t]);
                        acc[t] = fmaf(w.z, __uint_as_float(ub.y << 16), acc[t]);
                        acc[t] = fmaf(w.w, __uint_as_float(ub.y & 0xffff0000u), acc[t]);
                    }
                }
                const float b = item < NW ? bias_w : (L.bias ? L.bias[r0 + item] : 0.f);
#pragma unroll
                for (int t = 0; t < T; t++) {
                    const float sv = warp_sum(acc[t]);
                    if (lane == 0)
                        st_relaxed_u64(a.lgll + ((size_t)(l & 1) * T + t) * E + r0 + item,
                                       tagged(sv + b, (unsigned)(l + 1)));
                }
            } else {
                const int q = item - nra;
                const char *qg = r1 + (size_t)nra * H * 4;
                const uint4 *wg = reinterpret_cast<const uint4 *>(qg + (size_t)q * H * 2);
                const uint4 *wu = reinterpret_cast<const uint4 *>(qg + (size_t)(nqa + q) * H * 2);
                float gg[T], uu[T];
#pragma unroll
                for (int t = 0; t < T; t++) gg[t] = uu[t] = 0.f;
#pragma unroll 2
                for (int cc = lane; cc < (H >> 3); cc += 32) {
                    const uint4 Gv = wg[cc], Uv = wu[cc];
                    const uint32_t Gw[4] = {Gv.x, Gv.y, Gv.z, Gv.w}, Uw[4] = {Uv.x, Uv.y, Uv.z, Uv.w};
#pragma unroll
                    for (int t = 0; t < T; t++) {
                        const uint4 Xv = *reinterpret_cast<const uint4 *>(xb + (size_t)t * H + 8 * cc);
                        const uint32_t Xw[4] = {Xv.x, Xv.y, Xv.z, Xv.w};
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            const float x0 = __uint_as_float(Xw[j] << 16), x1 = __uint_as_float(Xw[j] & 0xffff0000u);
                            gg[t] = fmaf(__uint_as_float(Gw[j] << 16), x0, gg[t]);
                            gg[t] = fmaf(__uint_as_float(Gw[j] & 0xffff0000u), x1, gg[t]);
                            uu[t] = fmaf(__uint_as_float(Uw[j] << 16), x0, uu[t]);
                            uu[t] = fmaf(__uint_as_float(Uw[j] & 0xffff0000u), x1, uu[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < T; t++) {
                    const float gs = warp_sum(gg[t]), us = warp_sum(uu[t]);
                    if (lane == 0) __stcg(a.hs + (size_t)t * Is + q0 + q, silu(gs) * us);
                }
            }
        }
        __syncthreads();  // poll only once this CTA's own rows are done (fewer spinning requests in L2)
        MOE_TRACE(3);
        // ---- routing: all logits, top-k per token, groups of pairs
        {
            // all requests first (one round trip when the logits are ready), then late ones
            constexpr int kL = (kMaxT * 1024 + NT - 1) / NT;
            const uint64_t *src = a.lgll + (size_t)(l & 1) * T * E;
            uint64_t wv[kL];
#pragma unroll 1
            for (;;) {  // read every word; while one is late, wait for it and read them all again
#pragma unroll
                for (int j = 0; j < kL; j++) {
                    const int i = tid + NT * j;
                    wv[j] = i < T * E ? ld_relaxed_u64(src + i) : 0;
                }
                const uint64_t *lp = nullptr;
#pragma unroll
                for (int j = 0; j < kL; j++)
                    if (!lp && tid + NT * j < T * E && (unsigned)(wv[j] >> 32) != (unsigned)(l + 1)) lp = src + tid + NT * j;
                if (!lp) break;
                if (!wait_tags(a, lp, 1, 0, (unsigned)(l + 1))) {
                    fail = true;
                    break;
                }
            }
#pragma unroll
            for (int j = 0; j < kL; j++) {
                const int i = tid + NT * j;
                if (i < T * E) lg[i] = __uint_as_float((unsigned)wv[j]);
            }
        }
        if (__syncthreads_or(fail)) { ok = false; break; }
        MOE_TRACE(4);
        unsigned nan_mask = 0;
        for (int t = 0; t < T; t++)
            if (topk_cta(lg + (size_t)t * E, E, k, R, t, reinterpret_cast<uint32_t *>(r1),
                         reinterpret_cast<int *>(r1) + ((E + 255) / 256) * 16 * kMaxK))
                nan_mask |= 1u << t;
        if (nan_mask && tid == 0) set_status(a.status, MOE_ERR_NONFINITE);
        if (warp < T) topk_weights(R, warp, k, (nan_mask >> warp) & 1u);
        if (T > 1) __syncthreads();
        if (warp == 0) {
            __syncwarp();
            if constexpr (OPT) mark_pairs(a, R, T * k, k, l);
            build_groups<OPT>(R, T * k);
            pair_tokens(R, T * k, k);
        }
        __syncthreads();
        if (cta == 0 && a.ids_out && tid < T * k) {
            a.ids_out[(size_t)l * T * k + tid] = R.ids[tid];
            a.w_out[(size_t)l * T * k + tid] = R.w[tid];
        }
        MOE_TRACE(5);
        const int ng = R.ngroups, NU = ng * tiles;
        int u0, u1;
        split_range(NU, cta, G, u0, u1);
        const int nu = u1 - u0;
        if (warp == 0) {  // one lane per unit slot and per down slot
            const int nui = min(nu, P.nsu), ndi = nrows > 0 ? min(ng, P.nsd) : 0;
            for (int j = lane; j < nui + ndi; j += 32) {
                if (j < nui) {
                    issue_unit<OPT>(a, P, L, R, l, u0 + j, r1 + (size_t)j * P.unitB, &R.fullU[j]);
                    iss_u[j]++;
                } else {
                    const int g = j - nui;
                    issue_down<OPT>(a, P, L, R, l, g, o0, nrows, r2 + (size_t)g * P.downB, &R.fullD[g]);
                    iss_d[g]++;
                }
            }
        }
        // ---- B: routed gate/up on the tensor cores
        const bool ring = nu > P.nsu;
        // item j = ul * per_unit + it for j = warp, warp + NW, ...: the unit ul
        // (its slot, fill, group and row tile) and the item it advance by
        // counting, without divisions
        int ul = 0, it = warp, slot = 0, fq = 0, g = u0 / tiles, rt = u0 % tiles;
        while (it >= per_unit) {
            it -= per_unit;
            ul++;
            if (++slot == P.nsu) { slot = 0; fq++; }
            if (++rt == tiles) { rt = 0; g++; }
        }
        for (; ul < nu;) {
            const int mtx = it >= NST, s = it - mtx * NST;
            const int fill = R.fills_u[slot] + fq;
            if (!tc::mbar_wait(&R.fullU[slot], (uint32_t)(fill & 1), kTimeoutNs)) {
                fail = true;
                break;
            }
            const int u = u0 + ul;
            const int n = R.g_n[g], p0 = R.g_p0[g];
            int tok[kMaxT];
#pragma unroll
            for (int t = 0; t < kMaxT; t++) tok[t] = t < n ? R.tok_of[p0 + t] : 0;
            float *pslot = pgu + (size_t)slot * per_unit * 16 * T;
            if constexpr (T == 1) {
                GuOps<T> ops;
                gu_load_ops<T>(ops, s, n, tok, xp, H, P.xp_stride, zero16);
                gu_item<T, BITS>(P, r1 + (size_t)slot * P.unitB, mtx, s, n, ops, H, pslot);
            } else {
#pragma unroll 1
                for (int t = 0; t < n; t++) {  // one token at a time: the one-token item's registers
                    const int tk[kMaxT] = {tok[t], 0, 0, 0};
                    GuOps<1> ops;
                    gu_load_ops<1>(ops, s, 1, tk, xp, H, P.xp_stride, zero16);
                    gu_item<1, BITS, T>(P, r1 + (size_t)slot * P.unitB, mtx, s, 1, ops, H, pslot, t);
                }
            }
            if (ring) {  // slots are reused: the last item of a unit finalises it and refills the slot
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();
                    last = atomicAdd(&R.ucnt[slot], 1) == per_unit - 1;
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence_block();
                    finalize_unit<T>(a, pslot, n, p0, rt, I, NST);
                    __syncwarp();
                    if (lane == 0) {
                        atomicExch(&R.ucnt[slot], 0);
                        if (ul + P.nsu < nu) {
                            issue_unit<OPT>(a, P, L, R, l, u + P.nsu, r1 + (size_t)slot * P.unitB, &R.fullU[slot]);
                            iss_u[slot]++;
                        }
                    }
                }
            }
            for (it += NW; it >= per_unit;) {
                it -= per_unit;
                ul++;
                if (++slot == P.nsu) { slot = 0; fq++; }
                if (++rt == tiles) { rt = 0; g++; }
            }
        }
        if (!ring) {  // every unit had its own slot: finalise them all once every item is done
            if (__syncthreads_or(fail)) {
                if (tid == 0) raise_abort(a);
                ok = false;
                break;
            }
            for (int ul = warp; ul < nu; ul += NW) {
                const int u = u0 + ul, g = u / tiles;
                finalize_unit<T>(a, pgu + (size_t)ul * per_unit * 16 * T, R.g_n[g], R.g_p0[g], u % tiles, I, NST);
            }
        }
        if (__syncthreads_or(fail)) {
            if (tid == 0) raise_abort(a);
            ok = false;
            break;
        }
        MOE_TRACE(6);
        if (tid == 0) {
            for (int s = 0; s < P.nsu; s++) R.fills_u[s] += fills_of(s, nu, P.nsu);
            red_release_add(a.cnt + 0, 1u);
            if (l + 1 < a.n_layers) {
                tc::fence_proxy_async_smem();
                issue_a<OPT>(a, P, a.L[l + 1], r1, &R.fullA);
                iss_a++;
            }
        }
        // ---- every CTA's h (and h_s): the routed h's operand words come by one
        // bulk copy into shared memory when they fit (else each down item reads
        // them from global memory), in flight during the shared down rows; h_s
        // by plain loads
        if (tid == 0) {
            fail = !wait_counter(a, a.cnt + 0, (unsigned)(l + 1) * (unsigned)G);
            if (!fail && P.stage_h && nrows > 0) {
                tc::fence_proxy_async_global();  // the other CTAs' h, acquired above, before the copy reads it
                tc::fence_proxy_async_smem();    // the last layer's reads of the staging area before the copy writes it
                tc::mbar_arrive_expect_tx(&R.fullH, (uint32_t)(T * k * I * 4));
                bulk_g2s(dyn + P.off_hop, a.hop, (uint32_t)(T * k * I * 4), &R.fullH);
                iss_h++;
            }
        }
        if (__syncthreads_or(fail)) { ok = false; break; }
        MOE_TRACE(7);
        const uint32_t *hop = P.stage_h ? reinterpret_cast<const uint32_t *>(dyn + P.off_hop) : a.hop;
        if (L.swg && nrows > 0)
            for (int i = tid; i < T * Is; i += NT) hsm[i] = __ldcg(a.hs + i);
        const bool okS = tc::mbar_wait(&R.fullS, (uint32_t)(fillsS & 1), kTimeoutNs);
        fillsS++;
        if (__syncthreads_or(!okS)) {
            if (tid == 0) raise_abort(a);
            ok = false;
            break;
        }
        MOE_TRACE(8);
        // ---- shared down rows, one per warp, while the staged h is in flight
        if (L.swg) {
            for (int rr = warp; rr < nrows; rr += NW) {
                const uint4 *wd = reinterpret_cast<const uint4 *>(r3 + (size_t)rr * Is * 2);
                float p[T];
#pragma unroll
                for (int t = 0; t < T; t++) p[t] = 0.f;
                for (int cc = lane; cc < Is / 8; cc += 32) {
                    const uint4 Wv = wd[cc];
                    const uint32_t Ww[4] = {Wv.x, Wv.y, Wv.z, Wv.w};
#pragma unroll
                    for (int t = 0; t < T; t++) {
                        const float4 h0 = *reinterpret_cast<const float4 *>(hsm + (size_t)t * Is + 8 * cc);
                        const float4 h1 = *reinterpret_cast<const float4 *>(hsm + (size_t)t * Is + 8 * cc + 4);
                        const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            p[t] = fmaf(__uint_as_float(Ww[j] << 16), hv[2 * j], p[t]);
                            p[t] = fmaf(__uint_as_float(Ww[j] & 0xffff0000u), hv[2 * j + 1], p[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < T; t++) {
                    const float sv = warp_sum(p[t]);
                    if (lane == 0) sdn[t * 16 + rr] = sv;
                }
            }
        }
        if (P.stage_h && nrows > 0) {
            if (!tc::mbar_wait(&R.fullH, (uint32_t)(fillsH & 1), kTimeoutNs)) fail = true;
            fillsH++;
        }
        MOE_TRACE(9);
        // ---- C: routed down on the tensor cores
        if (nrows > 0 && !fail) {
            int g = 0, s2 = warp, slot = 0, fq = 0;
            while (s2 >= NSD2) {
                s2 -= NSD2;
                g++;
                if (++slot == P.nsd) { slot = 0; fq++; }
            }
            for (; g < ng;) {
                const int fill = R.fills_d[slot] + fq;
                if (!tc::mbar_wait(&R.fullD[slot], (uint32_t)(fill & 1), kTimeoutNs)) {
                    fail = true;
                    break;
                }
                if constexpr (T == 1) {
                    down_item<T, BITS>(P, r2 + (size_t)slot * P.downB, s2, R.g_n[g], R.g_p0[g], hop, P.stage_h != 0,
                                       zero16, I, pd);
                } else {
#pragma unroll 1
                    for (int t = 0; t < R.g_n[g]; t++)
                        down_item<1, BITS>(P, r2 + (size_t)slot * P.downB, s2, 1, R.g_p0[g] + t, hop, P.stage_h != 0,
                                           zero16, I, pd);
                }
                if (ng > P.nsd) {  // slots are reused: the last item of a group refills its slot
                    __syncwarp();
                    int last = 0;
                    if (lane == 0) {
                        __threadfence_block();
                        last = atomicAdd(&R.dcnt[slot], 1) == NSD2 - 1;
                    }
                    last = __shfl_sync(0xffffffffu, last, 0);
                    if (last && lane == 0) {
                        atomicExch(&R.dcnt[slot], 0);
                        if (g + P.nsd < ng) {
                            issue_down<OPT>(a, P, L, R, l, g + P.nsd, o0, nrows, r2 + (size_t)slot * P.downB, &R.fullD[slot]);
                            iss_d[slot]++;
                        }
                    }
                }
                for (s2 += NW; s2 >= NSD2;) {
                    s2 -= NSD2;
                    g++;
                    if (++slot == P.nsd) { slot = 0; fq++; }
                }
            }
        }
        if (__syncthreads_or(fail)) {
            if (tid == 0) raise_abort(a);
            ok = false;
            break;
        }
        MOE_TRACE(10);
        if (tid == 0 && l + 1 < a.n_layers) {  // the shared down rows are consumed: fetch the next layer's
            tc::fence_proxy_async_smem();
            issue_s<OPT>(a, a.L[l + 1], r3, o0, nrows, &R.fullS);
            iss_s++;
        }
        // ---- combine in slot order, residual update, x_{l+1} out
        for (int i = tid; i < T * k * nrows; i += NT) {  // y of pair p, row rr: its super-tiles in order
            const int p = i / nrows, rr = i % nrows;
            float y = 0.f;
#pragma unroll 8
            for (int s2 = 0; s2 < NSD2; s2++) y += pd[((size_t)p * NSD2 + s2) * 16 + rr];
            pd[(size_t)p * NSD2 * 16 + rr] = y;
        }
        __syncthreads();
        for (int i = tid; i < nrows * T; i += NT) {
            const int rr = i / T, t = i % T;
            // every slot's weight and partial first (independent loads), then the sum in slot order
            float wj[kMaxK], yj[kMaxK];
#pragma unroll
            for (int j = 0; j < kMaxK; j++) {
                wj[j] = 0.f;
                yj[j] = 0.f;
                if (j < k) {
                    wj[j] = R.w[t * k + j];
                    if (!OPT || R.key[t * k + j] != INT32_MAX) yj[j] = pd[(size_t)R.inv[t * k + j] * NSD2 * 16 + rr];
                }
            }
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxK; j++)
                if (j < k) sum = fmaf(wj[j], yj[j], sum);
            if (L.swg) sum += sdn[t * 16 + rr];
            const float nx = xown[t * 16 + rr] + sum;
            if (l + 1 < a.n_layers)
                st_relaxed_u64(a.xll + ((size_t)((l + 1) & 1) * T + t) * H + o0 + rr, tagged(nx, (unsigned)(l + 1)));
            else
                a.x[(size_t)t * H + o0 + rr] = nx;
        }
        if (tid == NT - 1 && nrows > 0)  // (a thread that has no row to combine)
            for (int s = 0; s < P.nsd; s++) R.fills_d[s] += fills_of(s, ng, P.nsd);
        __syncthreads();
        MOE_TRACE(11);
    }
    // ---- on an early exit, let every copy in flight land before the CTA ends
    if (!ok && tid == 0) {
        constexpr unsigned long long kDrainNs = 100000000ull;
        for (int s = 0; s < P.nsu; s++)
            if (iss_u[s]) tc::mbar_wait(&R.fullU[s], (uint32_t)((iss_u[s] - 1) & 1), kDrainNs);
        for (int s = 0; s < P.nsd; s++)
            if (iss_d[s]) tc::mbar_wait(&R.fullD[s], (uint32_t)((iss_d[s] - 1) & 1), kDrainNs);
        tc::mbar_wait(&R.fullA, (uint32_t)((iss_a - 1) & 1), kDrainNs);
        tc::mbar_wait(&R.fullS, (uint32_t)((iss_s - 1) & 1), kDrainNs);
        if (iss_h) tc::mbar_wait(&R.fullH, (uint32_t)((iss_h - 1) & 1), kDrainNs);
    }
}

// ------------------------------------------------------------ host side

template <int T, int BITS, bool OPT>
static cudaError_t launch(const Args &a, const Plan &P, int grid, cudaStream_t s)
{
    auto fn = decode_kernel<T, BITS, OPT>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, P.smem);
    if (e != cudaSuccess) return e;
    void *args[] = {const_cast<Args *>(&a), const_cast<Plan *>(&P)};
    return cudaLaunchCooperativeKernel((const void *)fn, dim3(grid), dim3(warps_for<T>() * 32), args, (size_t)P.smem, s);
}

template <int T, int BITS, bool OPT>
static cudaError_t attributes(size_t *static_smem)
{
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, decode_kernel<T, BITS, OPT>);
    if (e == cudaSuccess) *static_smem = fa.sharedSizeBytes;
    return e;
}

template <int T, int BITS, bool OPT>
static cudaError_t occupancy(int *blocks, int smem)
{
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, BITS, OPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, decode_kernel<T, BITS, OPT>, warps_for<T>() * 32, smem);
}

struct Ws {
    size_t cnt, xll, lgll, hop, hs, zero_end, total;
};

static Ws ws_layout(int T, int H, int I, int E, int k, int Is)
{
    Ws w;
    w.cnt = 0;  // counters and tagged words: zeroed before each launch
    w.xll = 256;
    w.lgll = w.xll + align256((size_t)2 * T * H * 8);
    w.zero_end = w.lgll + align256((size_t)2 * T * E * 8);
    w.hop = w.zero_end;
    w.hs = w.hop + align256((size_t)T * k * I * 4);
    w.total = w.hs + align256((size_t)T * std::max(Is, 1) * 4);
    return w;
}

static int al128(long n) { return (int)((n + 127) & ~127L); }

// Shared-memory plan; false if the shapes do not fit in `budget` bytes.
static bool make_plan(Plan &P, int T, int H, int I, int E, int k, int Is, int bits, int G, int rpc, long budget,
                      bool stage_h)
{
    memset(&P, 0, sizeof P);
    P.cb_gu = bits == 2 ? H / 4 : 3 * H / 8;
    P.sb_gu = H / 16;
    P.cb_d = bits == 2 ? I / 4 : 3 * I / 8;
    P.sb_d = I / 16;
    P.unitB = al128(32L * (P.cb_gu + P.sb_gu));
    P.downB = al128(16L * (P.cb_d + P.sb_d));
    P.NST = H / 256;
    P.NSD2 = I / 128;
    P.rA = (E + G - 1) / G;
    P.sA = (Is + G - 1) / G;
    P.xp_stride = 80;
    const int np = T * k;
    const long aBytes = std::max((long)P.rA * H * 4 + 2L * P.sA * H * 2,
                                 8L * ((E + 255) / 256) * 16 * kMaxK);  // also the top-k lists
    long off = 0;
    P.off_xb = (int)off;   off += al128((long)T * H * 2);
    P.off_xp = (int)off;   off += al128((long)T * (H / 32) * P.xp_stride);
    P.off_lg = (int)off;   off += al128((long)T * E * 4);
    P.off_hs = (int)off;   off += al128((long)T * std::max(Is, 1) * 4);
    P.off_pd = (int)off;   off += al128((long)np * P.NSD2 * 16 * 4);
    P.off_xown = (int)off; off += al128((long)2 * T * 16 * 4);
    P.off_r3 = (int)off;   off += al128((long)rpc * std::max(Is, 1) * 2);
    P.stage_h = stage_h;
    if (stage_h) {
        P.off_hop = (int)off;  off += al128((long)np * I * 4);
    }
    const long fixed = off;
    const long pguPer = (long)2 * P.NST * 16 * T * 4;
    const int nsuMax = std::min(kMaxUnitSlots, std::max(1, (np * (I / 16) + G - 1) / G));
    const int nsdMax = np;
    // the most unit slots that still leave room for min(np, 4) down slots
    for (int nsu = nsuMax; nsu >= 1; nsu--) {
        const long r1 = al128(std::max(aBytes, (long)nsu * P.unitB));
        const long base = fixed + al128(nsu * pguPer) + r1;
        if (base > budget) continue;
        const int nsd = (int)std::min<long>(nsdMax, (budget - base) / P.downB);
        if (nsd < std::min(nsdMax, 4)) continue;
        P.nsu = nsu;
        P.nsd = nsd;
        P.r1B = (int)r1;
        P.off_pgu = (int)off;
        off += al128(nsu * pguPer);
        P.off_r1 = (int)off;
        off += r1;
        P.off_r2 = (int)off;
        off += (long)nsd * P.downB;
        P.smem = (int)off;
        return true;
    }
    return false;
}

}  // namespace fused
}  // namespace moe

using namespace moe;

// Shape checks shared by the workspace query and the launch.
static moe_status decode_shapes_ok(int T, int H, int I, int E, int k, int Is)
{
    using namespace fused;
    MOE_REQUIRE(T >= 1 && T <= kMaxT, "T must be in [1, %d] (got %d)", kMaxT, T);
    MOE_REQUIRE(H >= 256 && H % 256 == 0, "the fused decode takes H a multiple of 256 (got %d)", H);
    MOE_REQUIRE(I >= 128 && I % 128 == 0 && I <= 4096, "the fused decode takes I a multiple of 128 up to 4096 (got %d)",
                I);
    MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= kMaxK && k <= E, "1 <= k <= min(E, 16), E <= 1024");
    MOE_REQUIRE(Is >= 0 && Is % 64 == 0 && Is <= 4096, "shared_I must be a multiple of 64 up to 4096 (got %d)", Is);
    return MOE_OK;
}

extern "C" moe_status moe_decode_workspace_size(int T, int H, int I, int E, int k, int shared_I, size_t *bytes)
{
    MOE_REQUIRE(bytes, "bytes is NULL");
    moe_status st = decode_shapes_ok(T, H, I, E, k, shared_I);
    if (st != MOE_OK) return st;
    *bytes = fused::ws_layout(T, H, I, E, k, shared_I).total;
    return MOE_OK;
}

extern "C" moe_status moe_decode_forward_ex(const moe_layer_weights *layers, int n_layers, float *x, int T, int k,
                                            float rms_eps, const moe_decode_options *opts, int32_t *ids_out,
                                            float *w_out, void *ws, size_t ws_bytes, int32_t *dev_status,
                                            moe_stream_t stream)
{
    using namespace fused;
    MOE_REQUIRE(layers && n_layers >= 0, "layers is NULL or n_layers < 0");
    MOE_REQUIRE(n_layers <= kMaxLayers, "at most %d layers per call (got %d)", kMaxLayers, n_layers);
    MOE_REQUIRE(T >= 1 && T <= kMaxT, "T must be in [1, %d] (got %d)", kMaxT, T);
    if (n_layers == 0) return MOE_OK;
    const moe_expert_arena &A0 = layers[0].experts;
    const int H = A0.H, I = A0.I, E = A0.E, bits = A0.bits, Is = layers[0].shared_I;
    MOE_REQUIRE(bits == 2 || bits == 3, "bits must be 2 or 3 (got %d)", bits);
    moe_status st = decode_shapes_ok(T, H, I, E, k, Is);
    if (st != MOE_OK) return st;
    MOE_REQUIRE(x && aligned16(x), "x must be a 16-byte aligned device pointer");
    MOE_REQUIRE(!ids_out == !w_out, "ids_out and w_out must both be given or both be NULL");
    const int tail_skip = opts ? opts->route_tail_skip : 0;
    const uint32_t *hot = opts ? opts->hot_experts : nullptr;
    MOE_REQUIRE(tail_skip >= 0 && tail_skip <= k, "route_tail_skip must be in [0, k] (got %d)", tail_skip);
    MOE_REQUIRE(!hot || (reinterpret_cast<uintptr_t>(hot) & 3u) == 0, "hot_experts must be 4-byte aligned");
    Args a;
    memset(&a, 0, sizeof a);
    a.tail_skip = tail_skip;
    a.hot = hot;
    for (int l = 0; l < n_layers; l++) {
        const moe_layer_weights &W = layers[l];
        const moe_expert_arena &A = W.experts;
        MOE_REQUIRE(A.H == H && A.I == I && A.E == E && A.bits == bits && W.shared_I == Is,
                    "layer %d has a different shape from layer 0", l);
        MOE_REQUIRE(A.gu_codes && A.gu_scales && A.d_codes && A.d_scales && W.w_router,
                    "layer %d: NULL weight pointer", l);
        MOE_REQUIRE(aligned16(A.gu_codes) && aligned16(A.gu_scales) && aligned16(A.d_codes) && aligned16(A.d_scales) &&
                        aligned16(W.w_router),
                    "layer %d: weight pointers must be 16-byte aligned", l);
        MOE_REQUIRE(!Is || (W.shared_wg && W.shared_wu && W.shared_wd && aligned16(W.shared_wg) &&
                            aligned16(W.shared_wu) && aligned16(W.shared_wd)),
                    "layer %d: shared expert pointers must be 16-byte aligned and non-NULL", l);
        a.L[l] = {A.gu_codes, A.gu_scales, A.d_codes, A.d_scales, W.w_router, W.bias,
                  Is ? W.shared_wg : nullptr, Is ? W.shared_wu : nullptr, Is ? W.shared_wd : nullptr};
    }
    const Ws lay = ws_layout(T, H, I, E, k, Is);
    if (!ws || ws_bytes < lay.total)
        return fail(MOE_ERR_WORKSPACE, "moe_decode_forward needs %zu bytes (%.2f MiB) of workspace, got %zu", lay.total,
                    mib((double)lay.total), ws ? ws_bytes : (size_t)0);
    MOE_REQUIRE(aligned16(ws), "workspace must be 16-byte aligned");
    const int grid = sm_count();
    int rpc = (H + grid - 1) / grid;
    rpc += rpc & 1;
    if (rpc > 16)
        return fail(MOE_ERR_UNSUPPORTED, "the fused decode gives each of the %d SMs at most 16 output rows (H=%d)", grid,
                    H);
    char *wb = static_cast<char *>(ws);
    a.n_layers = n_layers;
    a.T = T;
    a.H = H;
    a.I = I;
    a.E = E;
    a.k = k;
    a.Is = Is;
    a.bits = bits;
    a.rpc = rpc;
    a.rms_eps = rms_eps;
    a.x = x;
    a.cnt = reinterpret_cast<unsigned *>(wb + lay.cnt);
    a.xll = reinterpret_cast<uint64_t *>(wb + lay.xll);
    a.lgll = reinterpret_cast<uint64_t *>(wb + lay.lgll);
    a.hop = reinterpret_cast<uint32_t *>(wb + lay.hop);
    a.hs = reinterpret_cast<float *>(wb + lay.hs);
    a.ids_out = ids_out;
    a.w_out = w_out;
    a.status = dev_status;
    cudaError_t e = cudaSuccess;
    size_t static_smem = 0;
    const bool opt = tail_skip > 0 || hot != nullptr;
#define MOE_F_DISPATCH(FN, ...)                                \
    switch (T * 100 + bits * 10 + (opt ? 1 : 0)) {             \
    case 120: e = FN<1, 2, false>(__VA_ARGS__); break;         \
    case 121: e = FN<1, 2, true>(__VA_ARGS__); break;          \
    case 130: e = FN<1, 3, false>(__VA_ARGS__); break;         \
    case 131: e = FN<1, 3, true>(__VA_ARGS__); break;          \
    case 220: e = FN<2, 2, false>(__VA_ARGS__); break;         \
    case 221: e = FN<2, 2, true>(__VA_ARGS__); break;          \
    case 230: e = FN<2, 3, false>(__VA_ARGS__); break;         \
    case 231: e = FN<2, 3, true>(__VA_ARGS__); break;          \
    case 320: e = FN<3, 2, false>(__VA_ARGS__); break;         \
    case 321: e = FN<3, 2, true>(__VA_ARGS__); break;          \
    case 330: e = FN<3, 3, false>(__VA_ARGS__); break;         \
    case 331: e = FN<3, 3, true>(__VA_ARGS__); break;          \
    case 420: e = FN<4, 2, false>(__VA_ARGS__); break;         \
    case 421: e = FN<4, 2, true>(__VA_ARGS__); break;          \
    case 430: e = FN<4, 3, false>(__VA_ARGS__); break;         \
    default: e = FN<4, 3, true>(__VA_ARGS__); break;           \
    }
    MOE_F_DISPATCH(attributes, &static_smem)
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "decode kernel attributes: %s", cudaGetErrorString(e));
    int dev = 0, optin = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    const long budget = (long)optin - (long)static_smem - 1024;
    Plan P;
    if (!make_plan(P, T, H, I, E, k, Is, bits, grid, rpc, budget, true) &&
        !make_plan(P, T, H, I, E, k, Is, bits, grid, rpc, budget, false))
        return fail(MOE_ERR_UNSUPPORTED,
                    "the fused decode's buffers do not fit in %ld bytes of shared memory "
                    "(T=%d H=%d I=%d E=%d k=%d shared_I=%d)",
                    budget, T, H, I, E, k, Is);
    int per_sm = 0;
    MOE_F_DISPATCH(occupancy, &per_sm, P.smem)
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "decode occupancy query: %s", cudaGetErrorString(e));
    if (per_sm < 1)
        return fail(MOE_ERR_UNSUPPORTED, "the fused decode kernel does not fit on an SM (%d bytes of shared memory)",
                    P.smem);
    cudaStream_t s = to_cuda(stream);
    MOE_CUDA_TRY(cudaMemsetAsync(ws, 0, lay.zero_end, s));
    MOE_F_DISPATCH(launch, a, P, grid, s)
#undef MOE_F_DISPATCH
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cooperative launch of the fused decode: %s", cudaGetErrorString(e));
    return MOE_OK;
}

#ifdef MOE_DECODE_TRACE
extern "C" int moe_decode_trace_read(unsigned long long *host)
{
    if (cudaDeviceSynchronize() != cudaSuccess) return 1;
    return cudaMemcpyFromSymbol(host, fused::g_decode_trace, sizeof(fused::g_decode_trace)) != cudaSuccess;
}
#endif

extern "C" moe_status moe_decode_forward(const moe_layer_weights *layers, int n_layers, float *x, int T, int k,
                                         float rms_eps, int32_t *ids_out, float *w_out, void *ws, size_t ws_bytes,
                                         int32_t *dev_status, moe_stream_t stream)
{
    return moe_decode_forward_ex(layers, n_layers, x, T, k, rms_eps, nullptr, ids_out, w_out, ws, ws_bytes, dev_status,
                                 stream);
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
