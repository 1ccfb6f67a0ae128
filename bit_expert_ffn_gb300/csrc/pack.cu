// pack.cu -- moe_pack_experts / moe_unpack_experts: logical codes (one per
// byte) <-> the packed block format of moe_gb300.h.  One thread per 32-weight
// block; every access stays inside the block's own bytes.
#include "common.cuh"

namespace moe {

// Bit of the 3-bit high-plane word that holds weight i (0..31) of a block.
__device__ __forceinline__ int hi_pos(int i) { return (i & 7) | ((i & 8) << 1) | ((i & 16) >> 1); }

template <int BITS>
__global__ void pack_kernel(int64_t n_blocks, int64_t blocks_per_row, int64_t row_bytes,
                            const uint8_t *__restrict__ codes, const uint16_t *__restrict__ scales,
                            uint8_t *__restrict__ packed, uint16_t *packed_scales, bool copy_scales,
                            int32_t *status)
{
    int64_t gb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gb >= n_blocks) return;
    int64_t row = gb / blocks_per_row;
    int64_t b = gb - row * blocks_per_row;
    const uint4 *src = reinterpret_cast<const uint4 *>(codes + gb * 32);
    uint4 q0 = src[0], q1 = src[1];
    uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    uint32_t lo0 = 0, lo1 = 0, hi = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        uint32_t c = (w[i >> 2] >> (8 * (i & 3))) & 0xffu;
        bad |= c >= (1u << BITS);
        uint32_t l = c & 3u;
        if (i < 16) lo0 |= l << (2 * i);
        else lo1 |= l << (2 * (i - 16));
        if (BITS == 3) hi |= ((c >> 2) & 1u) << hi_pos(i);
    }
    uint8_t *prow = packed + row * row_bytes;
    uint32_t *lo = reinterpret_cast<uint32_t *>(prow + 8 * b);
    lo[0] = lo0;
    lo[1] = lo1;
    if (BITS == 3) *reinterpret_cast<uint32_t *>(prow + blocks_per_row * 8 + 4 * b) = hi;
    uint16_t s = scales[gb];
    if ((s & 0x7c00u) == 0x7c00u) bad = true;  // fp16 Inf or NaN
    if (copy_scales) packed_scales[gb] = s;
    if (bad) set_status(status, MOE_ERR_INVALID_ARG);
}

template <int BITS>
__global__ void unpack_kernel(int64_t n_blocks, int64_t blocks_per_row, int64_t row_bytes,
                              const uint8_t *__restrict__ packed, uint8_t *__restrict__ codes)
{
    int64_t gb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gb >= n_blocks) return;
    int64_t row = gb / blocks_per_row;
    int64_t b = gb - row * blocks_per_row;
    const uint8_t *prow = packed + row * row_bytes;
    const uint32_t *lo = reinterpret_cast<const uint32_t *>(prow + 8 * b);
    uint32_t lo0 = lo[0], lo1 = lo[1];
    uint32_t hi = BITS == 3 ? *reinterpret_cast<const uint32_t *>(prow + blocks_per_row * 8 + 4 * b) : 0u;
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; q++) w[q] = 0;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        uint32_t c = ((i < 16 ? lo0 >> (2 * i) : lo1 >> (2 * (i - 16)))) & 3u;
        if (BITS == 3) c |= ((hi >> hi_pos(i)) & 1u) << 2;
        w[i >> 2] |= c << (8 * (i & 3));
    }
    uint4 *dst = reinterpret_cast<uint4 *>(codes + gb * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

static moe_status check_pack_args(int bits, int64_t n_mats, int64_t rows, int64_t cols)
{
    MOE_REQUIRE(bits == 2 || bits == 3, "bits must be 2 or 3 (got %d)", bits);
    MOE_REQUIRE(n_mats >= 0 && rows >= 0, "n_mats and rows must be >= 0");
    MOE_REQUIRE(cols > 0 && cols % 32 == 0, "cols must be a positive multiple of 32 (got %lld)", (long long)cols);
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_pack_experts(int bits, int64_t n_mats, int64_t rows, int64_t cols, const uint8_t *codes,
                                       const uint16_t *scales, uint8_t *packed_codes, uint16_t *packed_scales,
                                       int32_t *dev_status, moe_stream_t stream)
{
    moe_status st = check_pack_args(bits, n_mats, rows, cols);
    if (st != MOE_OK) return st;
    int64_t n_blocks = n_mats * rows * (cols / 32);
    if (n_blocks == 0) return MOE_OK;
    MOE_REQUIRE(codes && scales && packed_codes && packed_scales, "NULL pointer");
    MOE_REQUIRE(aligned16(codes), "codes must be 16-byte aligned");
    MOE_REQUIRE(((uintptr_t)packed_codes & 3u) == 0, "packed_codes must be 4-byte aligned");
    int64_t rb = bits == 2 ? cols / 4 : cols / 4 + cols / 8;
    int64_t blocks = (n_blocks + 255) / 256;
    MOE_REQUIRE(blocks <= INT32_MAX, "too many blocks");
    bool copy = packed_scales != scales;
    if (bits == 2)
        pack_kernel<2><<<(unsigned)blocks, 256, 0, to_cuda(stream)>>>(n_blocks, cols / 32, rb, codes, scales,
                                                                      packed_codes, packed_scales, copy, dev_status);
    else
        pack_kernel<3><<<(unsigned)blocks, 256, 0, to_cuda(stream)>>>(n_blocks, cols / 32, rb, codes, scales,
                                                                      packed_codes, packed_scales, copy, dev_status);
    return check_launch("pack");
}

extern "C" moe_status moe_unpack_experts(int bits, int64_t n_mats, int64_t rows, int64_t cols,
                                         const uint8_t *packed_codes, uint8_t *codes, moe_stream_t stream)
{
    moe_status st = check_pack_args(bits, n_mats, rows, cols);
    if (st != MOE_OK) return st;
    int64_t n_blocks = n_mats * rows * (cols / 32);
    if (n_blocks == 0) return MOE_OK;
    MOE_REQUIRE(codes && packed_codes, "NULL pointer");
    MOE_REQUIRE(aligned16(codes), "codes must be 16-byte aligned");
    MOE_REQUIRE(((uintptr_t)packed_codes & 3u) == 0, "packed_codes must be 4-byte aligned");
    int64_t rb = bits == 2 ? cols / 4 : cols / 4 + cols / 8;
    int64_t blocks = (n_blocks + 255) / 256;
    MOE_REQUIRE(blocks <= INT32_MAX, "too many blocks");
    if (bits == 2)
        unpack_kernel<2><<<(unsigned)blocks, 256, 0, to_cuda(stream)>>>(n_blocks, cols / 32, rb, packed_codes, codes);
    else
        unpack_kernel<3><<<(unsigned)blocks, 256, 0, to_cuda(stream)>>>(n_blocks, cols / 32, rb, packed_codes, codes);
    return check_launch("unpack");
}
