// permute.cu -- moe_permute: stable counting sort of the T*k (token, slot)
// pairs by expert id.  All integer work, bit-exact and deterministic: counts
// may be gathered with atomics (integer sums do not depend on order), but
// every position comes from ordered scans.
//
// The pages group the tokens of a verify window that share an expert
// ("Strata serves a 125B MoE at 94 tokens/s from a 12 GB card and 64 GB of
// RAM", section "Six billion active parameters per token").
#include "common.cuh"

namespace moe {

constexpr int kPermChunk = 2048;     // pairs per chunk in the multi-CTA path
constexpr int kPermSmallMax = 4096;  // single-CTA path up to this many pairs

// Warp-serial stable placement of pairs [f0, f1) starting from per-expert
// cursors `cur` (shared memory).  Lanes take 32 pairs at a time in order.
__device__ void place_pairs(const int32_t *__restrict__ ids, int64_t f0, int64_t f1, int E, int32_t *cur,
                            int32_t *__restrict__ perm, int32_t *__restrict__ inv)
{
    int lane = lane_id();
    unsigned lt = (1u << lane) - 1u;
    for (int64_t base = f0; base < f1; base += 32) {
        int64_t f = base + lane;
        bool in = f < f1;
        int id = in ? ids[f] : -1;
        bool valid = in && id >= 0 && id < E;
        int key = valid ? id : (in ? -1 : -2);  // invalid lanes never match a valid id
        unsigned m = __match_any_sync(0xffffffffu, key);
        if (valid) {
            int pos = cur[id] + __popc(m & lt);
            perm[pos] = (int32_t)f;
            inv[f] = pos;
        } else if (in) {
            inv[f] = -1;
        }
        __syncwarp();
        if (valid && (m & lt) == 0) cur[id] += __popc(m);
        __syncwarp();
    }
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int32_t *warp_tot, int &total)
{
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane_id() >= o) incl += y;
    }
    if (lane_id() == 31) warp_tot[warp_id()] = incl;
    __syncthreads();
    if (warp_id() == 0) {
        int nw = blockDim.x >> 5;
        int wt = lane_id() < nw ? warp_tot[lane_id()] : 0;
        int wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane_id() >= o) wi += y;
        }
        if (lane_id() < nw) warp_tot[lane_id()] = wi - wt;
        if (lane_id() == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    int excl = incl - v + warp_tot[warp_id()];
    total = warp_tot[32];
    __syncthreads();
    return excl;
}

// Single CTA (1024 threads): count, scan, place.
__global__ void __launch_bounds__(1024) permute_small_kernel(const int32_t *__restrict__ ids, int n, int E,
                                                             int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                                                             int32_t *__restrict__ inv, int32_t *status)
{
    __shared__ int32_t cnt[1024];
    __shared__ int32_t warp_tot[33];
    int tid = threadIdx.x;
    if (tid < E) cnt[tid] = 0;
    __syncthreads();
    for (int f = tid; f < n; f += blockDim.x) {
        int id = ids[f];
        if (id >= 0 && id < E) atomicAdd(&cnt[id], 1);
        else if (id != MOE_ID_NOT_LOCAL) set_status(status, MOE_ERR_BOUNDS);
    }
    __syncthreads();
    int v = tid < E ? cnt[tid] : 0;
    int total = 0;
    int excl = block_exclusive_scan(v, warp_tot, total);
    if (tid < E) {
        offsets[tid] = excl;
        cnt[tid] = excl;  // becomes the placement cursor
    }
    if (tid == 0) offsets[E] = total;
    for (int p = total + tid; p < n; p += blockDim.x) perm[p] = -1;
    __syncthreads();
    if (warp_id() == 0) place_pairs(ids, 0, n, E, cnt, perm, inv);
}

// Multi-CTA pass 1: per-chunk histograms -> counts[chunk][E].
__global__ void permute_count_kernel(const int32_t *__restrict__ ids, int64_t n, int E, int32_t *__restrict__ counts,
                                     int32_t *status)
{
    __shared__ int32_t h[1024];
    for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
    __syncthreads();
    int64_t f0 = (int64_t)blockIdx.x * kPermChunk;
    int64_t f1 = min(n, f0 + kPermChunk);
    for (int64_t f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
        int id = ids[f];
        if (id >= 0 && id < E) atomicAdd(&h[id], 1);
        else if (id != MOE_ID_NOT_LOCAL) set_status(status, MOE_ERR_BOUNDS);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(int64_t)blockIdx.x * E + e] = h[e];
}

// Multi-CTA pass 2 (one CTA of 1024 threads): offsets and per-chunk bases.
__global__ void __launch_bounds__(1024) permute_scan_kernel(const int32_t *__restrict__ counts, int n_chunks, int E,
                                                            int64_t n, int32_t *__restrict__ base,
                                                            int32_t *__restrict__ offsets, int32_t *__restrict__ perm)
{
    __shared__ int32_t warp_tot[33];
    int tid = threadIdx.x;
    int v = 0;
    if (tid < E)
        for (int c = 0; c < n_chunks; c++) v += counts[(int64_t)c * E + tid];
    int total = 0;
    int excl = block_exclusive_scan(v, warp_tot, total);
    if (tid < E) {
        offsets[tid] = excl;
        int run = excl;
        for (int c = 0; c < n_chunks; c++) {
            base[(int64_t)c * E + tid] = run;
            run += counts[(int64_t)c * E + tid];
        }
    }
    if (tid == 0) offsets[E] = total;
    for (int64_t p = total + tid; p < n; p += blockDim.x) perm[p] = -1;
}

// Multi-CTA pass 3: one warp per chunk places its pairs in order.
__global__ void permute_place_kernel(const int32_t *__restrict__ ids, int64_t n, int E,
                                     const int32_t *__restrict__ base, int32_t *__restrict__ perm,
                                     int32_t *__restrict__ inv)
{
    __shared__ int32_t cur[1024];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cur[e] = base[(int64_t)blockIdx.x * E + e];
    __syncthreads();
    int64_t f0 = (int64_t)blockIdx.x * kPermChunk;
    int64_t f1 = min(n, f0 + kPermChunk);
    if (warp_id() == 0) place_pairs(ids, f0, f1, E, cur, perm, inv);
}

static int64_t n_chunks_for(int64_t n) { return (n + kPermChunk - 1) / kPermChunk; }

// local[i] = ids[i] - e0 for ids in [e0, e0 + e_count), MOE_ID_NOT_LOCAL otherwise.
__global__ void shard_ids_kernel(const int32_t *__restrict__ ids, int64_t n, int e0, int e_count,
                                 int32_t *__restrict__ local)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int id = ids[i];
        local[i] = (id >= e0 && id - e0 < e_count) ? id - e0 : MOE_ID_NOT_LOCAL;
    }
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_shard_ids(const int32_t *ids, int64_t n, int e0, int e_count, int32_t *local_ids,
                                    moe_stream_t stream)
{
    MOE_REQUIRE(n >= 0, "n must be >= 0");
    MOE_REQUIRE(e0 >= 0 && e_count >= 1 && e_count <= 1024, "e0 >= 0 and 1 <= e_count <= 1024 (got %d, %d)", e0,
                e_count);
    if (n == 0) return MOE_OK;
    MOE_REQUIRE(ids && local_ids, "NULL pointer");
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
    shard_ids_kernel<<<(unsigned)blocks, 256, 0, to_cuda(stream)>>>(ids, n, e0, e_count, local_ids);
    return check_launch("shard_ids");
}

extern "C" moe_status moe_permute_workspace_size(int T, int k, int E, size_t *bytes)
{
    MOE_REQUIRE(bytes, "bytes is NULL");
    MOE_REQUIRE(T >= 0 && k >= 1 && E >= 1 && E <= 1024, "T >= 0, k >= 1, 1 <= E <= 1024");
    int64_t n = (int64_t)T * k;
    if (n <= kPermSmallMax) {
        *bytes = 0;
        return MOE_OK;
    }
    int64_t c = n_chunks_for(n);
    *bytes = 2 * align256((size_t)c * E * sizeof(int32_t));
    return MOE_OK;
}

extern "C" moe_status moe_permute(const int32_t *ids, int T, int k, int E, int32_t *offsets, int32_t *perm,
                                  int32_t *inv_perm, void *ws, size_t ws_bytes, int32_t *dev_status,
                                  moe_stream_t stream)
{
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= 16, "T >= 0 and 1 <= k <= 16 (got T=%d k=%d)", T, k);
    MOE_REQUIRE(E >= 1 && E <= 1024, "E must be in [1, 1024] (got %d)", E);
    MOE_REQUIRE(offsets, "offsets is NULL");
    int64_t n = (int64_t)T * k;
    MOE_REQUIRE(n <= INT32_MAX, "T*k too large");
    cudaStream_t s = to_cuda(stream);
    if (n == 0) {
        MOE_CUDA_TRY(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s));
        return MOE_OK;
    }
    MOE_REQUIRE(ids && perm && inv_perm, "NULL pointer");
    if (n <= kPermSmallMax) {
        permute_small_kernel<<<1, 1024, 0, s>>>(ids, (int)n, E, offsets, perm, inv_perm, dev_status);
        return check_launch("permute_small");
    }
    int64_t c = n_chunks_for(n);
    size_t part = align256((size_t)c * E * sizeof(int32_t));
    if (!ws || ws_bytes < 2 * part)
        return fail(MOE_ERR_WORKSPACE, "permute needs %zu bytes (%.2f MiB) of workspace, got %zu", 2 * part,
                    mib(2.0 * part), ws ? ws_bytes : (size_t)0);
    int32_t *counts = static_cast<int32_t *>(ws);
    int32_t *base = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + part);
    permute_count_kernel<<<(unsigned)c, 256, 0, s>>>(ids, n, E, counts, dev_status);
    moe_status st = check_launch("permute_count");
    if (st != MOE_OK) return st;
    permute_scan_kernel<<<1, 1024, 0, s>>>(counts, (int)c, E, n, base, offsets, perm);
    st = check_launch("permute_scan");
    if (st != MOE_OK) return st;
    permute_place_kernel<<<(unsigned)c, 32, 0, s>>>(ids, n, E, base, perm, inv_perm);
    return check_launch("permute_place");
}

// --------------------------------------------------------------------------
// moe_permute_noalloc: the three-pass sort above with its scratch in a fixed
// device array of this library instead of a caller workspace.
// --------------------------------------------------------------------------
#include <cuda.h>

#include <mutex>

namespace moe {

// Per-chunk counts and per-chunk bases, kNoAllocScratchInts int32 each.
constexpr int64_t kNoAllocScratchInts = 32768;  // chunks * E <= 32768 -> 2 x 128 KiB
static __device__ __align__(256) int32_t g_permute_scratch[2 * kNoAllocScratchInts];

// The current CUDA context through the driver's cuCtxGetCurrent, found by
// the runtime's entry-point query (no link against the driver library).
static CUcontext current_context()
{
    using Fn = CUresult (*)(CUcontext *);
    static Fn fn = []() -> Fn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<Fn>(p);
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of g_permute_scratch on the current device, looked up with
// that device current and cached together with the context it belongs to: a
// new context on the device (after cudaDeviceReset, say, which unloads the
// library's device code) finds the cached context changed and looks the
// address up again.
static moe_status permute_scratch_address(int32_t **out)
{
    static std::mutex mu;
    static int32_t *addr[64] = {nullptr};
    static CUcontext ctx[64] = {nullptr};
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    const CUcontext cur = current_context();  // NULL before the runtime has made one current
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || !cur || cur != ctx[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);  // makes the primary context current
        if (e != cudaSuccess)
            return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(g_permute_scratch) on device %d: %s", dev,
                        cudaGetErrorString(e));
        addr[dev] = static_cast<int32_t *>(p);
        ctx[dev] = current_context();
    }
    *out = addr[dev];
    return MOE_OK;
}

}  // namespace moe

extern "C" moe_status moe_permute_noalloc(const int32_t *ids, int T, int k, int E, int32_t *offsets, int32_t *perm,
                                          int32_t *inv_perm, int32_t *dev_status, moe_stream_t stream)
{
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= 16, "T >= 0 and 1 <= k <= 16 (got T=%d k=%d)", T, k);
    MOE_REQUIRE(E >= 1 && E <= 1024, "E must be in [1, 1024] (got %d)", E);
    MOE_REQUIRE(offsets, "offsets is NULL");
    int64_t n = (int64_t)T * k;
    int64_t c = n_chunks_for(n);
    if (c * E > kNoAllocScratchInts)
        return fail(MOE_ERR_INVALID_ARG,
                    "moe_permute_noalloc holds at most %lld (chunks x experts) counters in its fixed scratch: "
                    "T*k=%lld pairs form %lld chunks of %d, times E=%d is %lld; use moe_permute with a workspace",
                    (long long)kNoAllocScratchInts, (long long)n, (long long)c, kPermChunk, E, (long long)(c * E));
    cudaStream_t s = to_cuda(stream);
    if (n == 0) {
        MOE_CUDA_TRY(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s));
        return MOE_OK;
    }
    MOE_REQUIRE(ids && perm && inv_perm, "NULL pointer");
    int32_t *scratch = nullptr;
    moe_status st = permute_scratch_address(&scratch);
    if (st != MOE_OK) return st;
    int32_t *counts = scratch;                      // every cell read below is written
    int32_t *base = scratch + kNoAllocScratchInts;  // earlier in the same call
    permute_count_kernel<<<(unsigned)c, 256, 0, s>>>(ids, n, E, counts, dev_status);
    st = check_launch("permute_count (no-alloc)");
    if (st != MOE_OK) return st;
    permute_scan_kernel<<<1, 1024, 0, s>>>(counts, (int)c, E, n, base, offsets, perm);
    st = check_launch("permute_scan (no-alloc)");
    if (st != MOE_OK) return st;
    permute_place_kernel<<<(unsigned)c, 32, 0, s>>>(ids, n, E, base, perm, inv_perm);
    return check_launch("permute_place (no-alloc)");
}
