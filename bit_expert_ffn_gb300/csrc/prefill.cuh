// prefill.cuh -- the prefill (grouped GEMM) path: host entry points and the
// tile bookkeeping both of its kernels share.
//
// The work of one GEMM is a list of (expert, M tile of sorted pairs, N tile
// of weight rows) items.  tile_prefix_kernel turns the per-expert pair
// counts into a prefix of M tiles, so a CTA maps a flat tile index to its
// expert with a binary search (expert_of_tile).
#pragma once

#include "common.cuh"

namespace moe {

// mt_prefix[e] = M tiles (of bm pairs) of experts < e; mt_prefix[E] = total.
// One CTA of 1024 threads, E <= 1024.
__global__ void tile_prefix_kernel(const int32_t *__restrict__ offsets, int E, int bm, int32_t *__restrict__ mt_prefix);

// Largest e with mt_prefix[e] <= mt (experts with zero tiles are skipped).
__device__ __forceinline__ int expert_of_tile(const int32_t *mt_prefix, int E, int mt)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (mt_prefix[mid] <= mt) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

size_t prefill_workspace_bytes(const moe_expert_arena &A, int T, int k);

moe_status prefill_forward(const moe_expert_arena &A, const uint16_t *x, int T, const int32_t *ids, const float *w,
                           int k, const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out,
                           moe_dtype dt, int accumulate, void *ws, int32_t *dev_status, cudaStream_t s);

// Tensor-core form (prefill_tc.cu): H and I multiples of 64.
bool prefill_tc_supported(const moe_expert_arena &A);
size_t prefill_tc_workspace_bytes(const moe_expert_arena &A, int T, int k);
moe_status prefill_tc_forward(const moe_expert_arena &A, const uint16_t *x, int T, const float *w, int k,
                              const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out, moe_dtype dt,
                              int accumulate, void *ws, int32_t *dev_status, cudaStream_t s);

// FP8 variant (prefill_tc.cu): 2-bit arenas, H and I multiples of 128.
bool prefill_fp8_supported(const moe_expert_arena &A);
size_t prefill_fp8_workspace_bytes(const moe_expert_arena &A, int T, int k);
moe_status prefill_fp8_forward(const moe_expert_arena &A, const uint16_t *x, int T, const float *w, int k,
                               const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out,
                               moe_dtype dt, int accumulate, void *ws, int32_t *dev_status, cudaStream_t s);

moe_status launch_combine(const float *y, const float *w, const int32_t *inv, int T, int k, int H, void *out,
                          moe_dtype dt, int accumulate, cudaStream_t s);
// fp16 rows of y (16-byte aligned, H a multiple of 8).
moe_status launch_combine_f16(const uint16_t *y, const float *w, const int32_t *inv, int T, int k, int H, void *out,
                              moe_dtype dt, int accumulate, cudaStream_t s);

}  // namespace moe
