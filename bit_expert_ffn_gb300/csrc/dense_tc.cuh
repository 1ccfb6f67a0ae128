// dense_tc.cuh -- dense bf16 GEMMs on the tcgen05 tensor cores (sm_103a) and
// the TMA tensor-map helper the tensor-core kernels share.
//
//   D[m][n] = sum_{kb} A[m][kA(kb)] * B[n][kB(kb)]       fp32 accumulation
//
// K runs in blocks of 64; block kb reads A at column (64 kb) mod a_cols and
// B at (64 kb) mod b_cols, so an operand can be repeated along K without
// being stored twice.  Two uses of that:
//   * the fp32 router: logits = x . W with W = W1 + W2 + W3 split into three
//     bf16 planes laid side by side ([E][3H]) and x read three times;
//   * the shared expert's down projection: h = h_hi + h_lo (two bf16 halves
//     side by side, [T][2I]) against the down weights read twice.
// In both, every product of the tensor cores is exact and the sum is fp32,
// so the results keep fp32-level accuracy with bf16 operands.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

enum DenseEpi {
    // B0 = gate rows, B1 = up rows (N each): h = silu(g) * u, written as two
    // bf16 halves hsplit[m][0..N) = bf16(h), hsplit[m][N..2N) = bf16(h - hi).
    DENSE_SWIGLU_SPLIT = 0,
    // out[m][n] = (accumulate ? out[m][n] : 0) + D[m][n] (+ bias[n]), fp32 or bf16.
    DENSE_OUT = 1,
};

struct DenseGemm {
    const uint16_t *A;  // [M][a_cols] bf16
    int a_cols;
    const uint16_t *B0, *B1;  // [N][b_cols] bf16; B1 only for DENSE_SWIGLU_SPLIT
    int b_cols;
    int M, N, K;  // K a multiple of 64
    uint16_t *hsplit;
    const float *bias;
    void *out;
    int out_bf16, accumulate;
    int32_t *status;
};

// True when the shapes and pointers suit the tensor-core kernel: a_cols,
// b_cols and K multiples of 64, every operand 16-byte aligned.
bool dense_tc_supported(const DenseGemm &g, DenseEpi epi);

moe_status dense_tc_gemm(const DenseGemm &g, DenseEpi epi, cudaStream_t s);

// Row-major 2D tensor map with a (box_cols x box_rows) box.
moe_status make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, int64_t rows,
                        int64_t cols, int box_cols, int box_rows,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

}  // namespace moe
