// prefill.cuh -- host entry points of the prefill (grouped GEMM) path.
#pragma once

#include "common.cuh"

namespace moe {

size_t prefill_workspace_bytes(const moe_expert_arena &A, int T, int k);

moe_status prefill_forward(const moe_expert_arena &A, const uint16_t *x, int T, const int32_t *ids, const float *w,
                           int k, const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out,
                           moe_dtype dt, int accumulate, void *ws, int32_t *dev_status, cudaStream_t s);

moe_status launch_combine(const float *y, const float *w, const int32_t *inv, int T, int k, int H, void *out,
                          moe_dtype dt, int accumulate, cudaStream_t s);

}  // namespace moe
