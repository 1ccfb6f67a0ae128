// prefill_tc.cu -- the prefill path of moe_expert_forward on the tcgen05
// tensor cores (sm_103a): grouped GEMMs over the experts' token lists with
// the 2-/3-bit weights dequantised to fp16 in shared memory.
//
//   gate/up:  D[p][r] = sum_i x[tok(p)][i] * dq(W_e[r][i])  for the gate rows r
//             and the matching up rows, then h[p][r] = silu(g) * u   (fp16)
//   down:     y[p][o] = sum_r h[p][r] * dq(Wd_e[o][r])                (fp32)
//   combine:  out[t][o] = sum_j w[t][j] y[inv[t*k+j]][o]   (slot order)
//
// One CTA per SM runs a persistent loop over tiles (expert, 128 sorted
// pairs) x (256 weight rows): warp 0 loads the token tile with TMA (128-byte
// swizzle), warps 8..15 dequantise the weight tile straight into the same
// swizzled K-major layout, warp 1 issues tcgen05.mma (M=128, N=256, K=16,
// fp16 operands, fp32 accumulators in TMEM, two accumulator buffers) and
// warps 4..7 read TMEM and write the epilogue.  Operands are fp16: x (bf16)
// converts exactly, the weights (c - mid) * s round once to fp16, h rounds
// to fp16 between the two GEMMs.
//
// Inside every 16-element group of the reduction dimension the operands are
// stored in the order 0,8,1,9,...,7,15 (both x/h and the weights, so the
// product is unchanged): a 2-bit code word then dequantises with one shift
// and one mask per pair of weights.
//
// The pages place the routed experts' FFN on the GPU and add their outputs
// ("How Strata runs a 125-billion-parameter model on a single 12 GB to 24 GB
// graphics card", Step 2) and read long prompts in chunks of tokens
// ("Strata Open-Source Runtime ...", section "Prefill and Long Context").
#include <cuda.h>

#include "common.cuh"
#include "dense_tc.cuh"
#include "prefill.cuh"
#include "tc.cuh"

namespace moe {
namespace ptc {

constexpr int BM = 128;          // pairs (tokens) per tile: MMA M
constexpr int BN = 256;          // weight rows per tile: MMA N (gate/up: 128 + 128)
constexpr int BK = 64;           // reduction per stage (one 128-byte swizzle row of fp16)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KiB
constexpr int B_BYTES = BN * BK * 2;  // 32 KiB
constexpr int THREADS = 512;
constexpr int DQ_WARP0 = 8;      // warps 8..15 dequantise (one weight row per thread)
constexpr int EPI_WARP0 = 4;     // warps 4..7 run the epilogue (TMEM lane quadrants 0..3)
constexpr unsigned long long kWaitNs = 2000000000ull;

struct Args {
    const uint8_t *codes;
    const uint16_t *scales;
    int64_t codes_expert_stride, scales_expert_stride;
    int row_bytes, scale_row;  // per weight row
    int K;                     // reduction length (H or I)
    int rows;                  // output rows of one matrix (I for gate/up, H for down)
    int up_rows;               // SWIGLU: offset of the up matrix (I), else 0
    int tiles_n;               // N tiles per M tile
    const int32_t *offsets, *mt_prefix;
    int E;
    uint16_t *h_out;           // SWIGLU: fp16 [pairs][I]
    float *y_out;              // down: fp32 [pairs][H]
    int32_t *status;
};

struct Shared {
    uint64_t afull[STAGES], bfull[STAGES], empty[STAGES];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem;
    volatile int abort;
};

// Stored position, inside its 16-element group, of element m.
__host__ __device__ __forceinline__ int perm16(int m) { return m < 8 ? 2 * m : 2 * (m - 8) + 1; }

template <int S>
__device__ __forceinline__ uint32_t shx(uint32_t w)
{
    if constexpr (S > 0) return w << S;
    else if constexpr (S < 0) return w >> (-S);
    else return w;
}

// Four fp16x2 words (k pairs (m, m+8), m = M0..M0+3) of one 16-code word:
// values (c - mid) * s.
template <int BITS, int M0>
__device__ __forceinline__ void dq_chunk(uint32_t w, uint32_t hw, __half2 s2, uint32_t (&o)[4])
{
    const __half2 off = BITS == 2 ? __halves2half2(__ushort_as_half(0x6003), __ushort_as_half(0x6003))   // 513.5
                                  : __halves2half2(__ushort_as_half(0x6007), __ushort_as_half(0x6007));  // 515.5
#define MOE_DQ(J)                                                                                       \
    {                                                                                                   \
        constexpr int m = M0 + (J);                                                                     \
        uint32_t b = (shx<1 - 2 * m>(w) & 0x00060006u) | 0x60006000u;                                   \
        if (BITS == 3) b |= shx<3 - m>(hw) & 0x00080008u;                                               \
        __half2 v = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&b), off), s2);                        \
        o[J] = *reinterpret_cast<uint32_t *>(&v);                                                       \
    }
    MOE_DQ(0) MOE_DQ(1) MOE_DQ(2) MOE_DQ(3)
#undef MOE_DQ
}

// 16 bytes of 2-bit codes of one row: 64 weights.  A 3-bit row (3K/8 bytes)
// is only 8-byte aligned, so it is read as two halves.
template <int BITS>
__device__ __forceinline__ uint4 load_codes(const uint8_t *p)
{
    if constexpr (BITS == 2) {
        return __ldg(reinterpret_cast<const uint4 *>(p));
    } else {
        uint2 lo = __ldg(reinterpret_cast<const uint2 *>(p)), hi = __ldg(reinterpret_cast<const uint2 *>(p + 8));
        return make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
}

// Dequantise 64 weights (one stage of one row) into the 128-byte swizzled row.
template <int BITS>
__device__ __forceinline__ void dq_row(const uint32_t (&w)[4], const uint32_t (&hw)[2], uint32_t sc, char *rowp, int r)
{
    __half2 s0 = __half2half2(__ushort_as_half((uint16_t)(sc & 0xffffu)));
    __half2 s1 = __half2half2(__ushort_as_half((uint16_t)(sc >> 16)));
#pragma unroll
    for (int g = 0; g < 4; g++) {
        __half2 s2 = g < 2 ? s0 : s1;
        uint32_t hword = BITS == 3 ? ((g & 1) ? hw[g >> 1] >> 8 : hw[g >> 1]) : 0u;
        uint32_t lo4[4], hi4[4];
        dq_chunk<BITS, 0>(w[g], hword, s2, lo4);
        dq_chunk<BITS, 4>(w[g], hword, s2, hi4);
        int c0 = 2 * g, c1 = 2 * g + 1;  // 16-byte chunks of the row
        *reinterpret_cast<uint4 *>(rowp + ((c0 ^ (r & 7)) << 4)) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
        *reinterpret_cast<uint4 *>(rowp + ((c1 ^ (r & 7)) << 4)) = make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
    }
}

template <int BITS, bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1) tc_gemm_kernel(const __grid_constant__ Args a,
                                                             const __grid_constant__ CUtensorMap tmap)
{
    extern __shared__ __align__(1024) char dyn_raw[];
    // 1024-byte alignment of the operand tiles (the swizzle atoms)
    char *dyn = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    char *sA = dyn;
    char *sB = dyn + STAGES * A_BYTES;
    __shared__ Shared S;
    int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            tc::mbar_init(&S.afull[s], 1);
            tc::mbar_init(&S.bfull[s], 256);
            tc::mbar_init(&S.empty[s], 1);
        }
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&S.acc_full[i], 1);
            tc::mbar_init(&S.acc_empty[i], 4);
        }
        tc::mbar_init(&S.mma_done, 1);
        S.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 2) tc::tmem_alloc(&S.tmem, 512);
    if (warp == 0 && lane == 0) tc::tma_prefetch_desc(&tmap);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;
    const int total = a.mt_prefix[a.E] * a.tiles_n;
    const int nk = a.K / BK;
    const int nrow_tile = SWIGLU ? BN / 2 : BN;

    if (warp == 0) {
        // ---------------- TMA producer: token tiles
        if (lane == 0) {
            int it = 0;
            for (int tile = blockIdx.x; tile < total && !S.abort; tile += gridDim.x) {
                int mt = tile / a.tiles_n;
                int e = expert_of_tile(a.mt_prefix, a.E, mt);
                int p0 = a.offsets[e] + (mt - a.mt_prefix[e]) * BM;
                for (int kb = 0; kb < nk; kb++, it++) {
                    int s = it % STAGES, u = it / STAGES;
                    if (u > 0 && !tc::mbar_wait(&S.empty[s], (u - 1) & 1, kWaitNs)) {
                        set_status(a.status, MOE_ERR_TIMEOUT);
                        S.abort = 1;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&S.afull[s], A_BYTES);
                    tc::tma_load_2d(sA + s * A_BYTES, &tmap, kb * BK, p0, &S.afull[s]);
                }
            }
            // no copy may still be in flight when the CTA leaves (after a timeout elsewhere)
            for (int s = 0; s < STAGES && s < it; s++) {
                int u = (s + STAGES * ((it - 1 - s) / STAGES)) / STAGES;
                if (!tc::mbar_wait(&S.afull[s], u & 1, kWaitNs)) set_status(a.status, MOE_ERR_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16_f32(BM, BN);
            int it = 0, j = 0;
            for (int tile = blockIdx.x; tile < total && !S.abort; tile += gridDim.x, j++) {
                int acc = j & 1, v = j >> 1;
                if (v > 0 && !tc::mbar_wait(&S.acc_empty[acc], (v - 1) & 1, kWaitNs)) {
                    set_status(a.status, MOE_ERR_TIMEOUT);
                    S.abort = 1;
                    break;
                }
                tc::tc_fence_after();
                uint32_t d = tmem + (uint32_t)(acc * BN);
                bool ok = true;
                for (int kb = 0; kb < nk; kb++, it++) {
                    int s = it % STAGES, u = it / STAGES;
                    if (!tc::mbar_wait(&S.afull[s], u & 1, kWaitNs) || !tc::mbar_wait(&S.bfull[s], u & 1, kWaitNs)) {
                        set_status(a.status, MOE_ERR_TIMEOUT);
                        S.abort = 1;
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    uint32_t abase = tc::smem_u32(sA + s * A_BYTES), bbase = tc::smem_u32(sB + s * B_BYTES);
#pragma unroll
                    for (int k16 = 0; k16 < BK / 16; k16++) {
                        uint64_t ad = tc::desc_kmajor_sw128(abase + k16 * 32);
                        uint64_t bd = tc::desc_kmajor_sw128(bbase + k16 * 32);
                        tc::mma_f16_ss(d, ad, bd, idesc, (kb | k16) ? 1u : 0u);
                    }
                    tc::mma_commit(&S.empty[s]);
                }
                if (!ok) break;
                tc::mma_commit(&S.acc_full[acc]);
            }
            // every MMA of this CTA has finished before TMEM is released
            tc::mma_commit(&S.mma_done);
            if (!tc::mbar_wait(&S.mma_done, 0, kWaitNs)) set_status(a.status, MOE_ERR_TIMEOUT);
        }
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + 4) {
        // ---------------- epilogue: TMEM -> registers -> global
        int q = warp - EPI_WARP0;  // lane quadrant
        int m = q * 32 + lane;     // row of the tile (pair)
        int j = 0;
        for (int tile = blockIdx.x; tile < total && !S.abort; tile += gridDim.x, j++) {
            int acc = j & 1, v = j >> 1;
            if (!tc::mbar_wait(&S.acc_full[acc], v & 1, kWaitNs)) {
                if (lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
                S.abort = 1;
                break;
            }
            tc::tc_fence_after();
            int mt = tile / a.tiles_n, nt = tile % a.tiles_n;
            int e = expert_of_tile(a.mt_prefix, a.E, mt);
            int p0 = a.offsets[e] + (mt - a.mt_prefix[e]) * BM;
            int pend = min(a.offsets[e + 1], p0 + BM);
            int p = p0 + m;
            bool valid = p < pend;
            uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            int n0 = nt * nrow_tile;
            if (SWIGLU) {
                for (int c = 0; c < BN / 2; c += 32) {
                    uint32_t g[32], u[32];
                    __syncwarp();
                    tc::tmem_ld_32x32b_x32(tbase + c, g);
                    tc::tmem_ld_32x32b_x32(tbase + BN / 2 + c, u);
                    tc::tmem_ld_wait();
                    int r0 = n0 + c;
                    if (valid && r0 < a.rows) {
                        uint32_t o[16];
#pragma unroll
                        for (int gi = 0; gi < 2; gi++)
#pragma unroll
                            for (int mm = 0; mm < 8; mm++) {
                                float x0 = __uint_as_float(g[16 * gi + mm]), y0 = __uint_as_float(u[16 * gi + mm]);
                                float x1 = __uint_as_float(g[16 * gi + mm + 8]), y1 = __uint_as_float(u[16 * gi + mm + 8]);
                                __half2 hv = __floats2half2_rn(silu(x0) * y0, silu(x1) * y1);
                                o[8 * gi + mm] = *reinterpret_cast<uint32_t *>(&hv);
                            }
                        uint4 *dst = reinterpret_cast<uint4 *>(a.h_out + (int64_t)p * a.rows + r0);
                        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                        dst[2] = make_uint4(o[8], o[9], o[10], o[11]);
                        dst[3] = make_uint4(o[12], o[13], o[14], o[15]);
                    }
                }
            } else {
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r[32];
                    __syncwarp();
                    tc::tmem_ld_32x32b_x32(tbase + c, r);
                    tc::tmem_ld_wait();
                    int o0 = n0 + c;
                    if (valid && o0 < a.rows) {
                        float4 *dst = reinterpret_cast<float4 *>(a.y_out + (int64_t)p * a.rows + o0);
#pragma unroll
                        for (int i = 0; i < 8; i++)
                            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.acc_empty[acc]);
        }
    } else if (warp >= DQ_WARP0) {
        // ---------------- dequantisation: one weight row of the tile per thread
        int d = threadIdx.x - DQ_WARP0 * 32;  // 0..255
        int it = 0;
        for (int tile = blockIdx.x; tile < total && !S.abort; tile += gridDim.x) {
            int mt = tile / a.tiles_n, nt = tile % a.tiles_n;
            int e = expert_of_tile(a.mt_prefix, a.E, mt);
            int rr = SWIGLU ? nt * (BN / 2) + (d & (BN / 2 - 1)) : nt * BN + d;
            bool valid = rr < a.rows;
            int64_t mrow = SWIGLU && d >= BN / 2 ? (int64_t)a.up_rows + rr : rr;
            const uint8_t *rowc = a.codes + (int64_t)e * a.codes_expert_stride + mrow * a.row_bytes;
            const uint16_t *rows_ = a.scales + (int64_t)e * a.scales_expert_stride + mrow * a.scale_row;
            // software pipeline: codes and scales of the next stage are loaded ahead
            uint4 cw = make_uint4(0, 0, 0, 0), nw = cw;
            uint2 hw = make_uint2(0, 0), nhw = hw;
            uint32_t sc = 0, nsc = 0;
            if (valid) {
                cw = load_codes<BITS>(rowc);
                if (BITS == 3) hw = __ldg(reinterpret_cast<const uint2 *>(rowc + a.K / 4));
                sc = __ldg(reinterpret_cast<const uint32_t *>(rows_));
            }
            for (int kb = 0; kb < nk; kb++, it++) {
                int s = it % STAGES, u = it / STAGES;
                if (valid && kb + 1 < nk) {
                    nw = load_codes<BITS>(rowc + (kb + 1) * 16);
                    if (BITS == 3) nhw = __ldg(reinterpret_cast<const uint2 *>(rowc + a.K / 4 + (kb + 1) * 8));
                    nsc = __ldg(reinterpret_cast<const uint32_t *>(rows_ + 2 * (kb + 1)));
                }
                if (u > 0 && !tc::mbar_wait(&S.empty[s], (u - 1) & 1, kWaitNs)) {
                    if (lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
                    S.abort = 1;
                    break;
                }
                char *rowp = sB + s * B_BYTES + d * 128;
                if (valid) {
                    uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
                    uint32_t h2[2] = {hw.x, hw.y};
                    dq_row<BITS>(w4, h2, sc, rowp, d);
                } else {
#pragma unroll
                    for (int c = 0; c < 8; c++) *reinterpret_cast<uint4 *>(rowp + 16 * c) = make_uint4(0, 0, 0, 0);
                }
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(&S.bfull[s]);
                cw = nw;
                hw = nhw;
                sc = nsc;
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// x_g[p][16g + perm16(m)] = fp16(x[tok(p)][16g + m]) for the valid pairs.
__global__ void gather_x_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ perm,
                                const int32_t *__restrict__ offsets, int E, int k, int H, uint16_t *__restrict__ xg)
{
    int n = offsets[E];
    int groups = H / 16;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)n * groups;
         i += (int64_t)gridDim.x * blockDim.x) {
        int p = (int)(i / groups), g = (int)(i % groups);
        int tok = perm[p] / k;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)tok * H + 16 * g);
        uint4 a0 = src[0], a1 = src[1];
        uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float f[16];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            f[2 * j] = __uint_as_float(w[j] << 16);
            f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
        uint32_t o[8];
#pragma unroll
        for (int mm = 0; mm < 8; mm++) {
            __half2 hv = __floats2half2_rn(f[mm], f[mm + 8]);
            o[mm] = *reinterpret_cast<uint32_t *>(&hv);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(xg + (int64_t)p * H + 16 * g);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// ---------------------------------------------------------------- host
// Tensor map over a row-major fp16 matrix [rows][cols]: 64 x 128 boxes, 128-byte swizzle.
static moe_status make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols)
{
    return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows, cols, BK, BM);
}

static size_t smem_bytes() { return (size_t)STAGES * (A_BYTES + B_BYTES) + 1024; }

template <int BITS, bool SWIGLU>
static moe_status launch_gemm(const Args &a, const CUtensorMap &map, int grid, cudaStream_t s)
{
    auto fn = tc_gemm_kernel<BITS, SWIGLU>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes());
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "tc gemm attribute: %s", cudaGetErrorString(e));
    fn<<<grid, THREADS, smem_bytes(), s>>>(a, map);
    return check_launch(SWIGLU ? "tc_gemm_gateup" : "tc_gemm_down");
}

}  // namespace ptc

struct PtcWs {
    int32_t *mt_prefix;
    uint16_t *xg, *h;
    float *y;
    size_t bytes;
};

static PtcWs ptc_ws(const moe_expert_arena &A, int T, int k, void *base)
{
    PtcWs w;
    size_t n = (size_t)T * k;
    size_t tb = align256((A.E + 1) * sizeof(int32_t));
    size_t xb = align256(n * A.H * 2), hb = align256(n * A.I * 2), yb = align256(n * A.H * 4);
    char *b = static_cast<char *>(base);
    w.mt_prefix = reinterpret_cast<int32_t *>(b);
    w.xg = b ? reinterpret_cast<uint16_t *>(b + tb) : nullptr;
    w.h = b ? reinterpret_cast<uint16_t *>(b + tb + xb) : nullptr;
    w.y = b ? reinterpret_cast<float *>(b + tb + xb + hb) : nullptr;
    w.bytes = tb + xb + hb + yb;
    return w;
}

bool prefill_tc_supported(const moe_expert_arena &A) { return A.H % 64 == 0 && A.I % 64 == 0 && A.H >= 64 && A.I >= 64; }

size_t prefill_tc_workspace_bytes(const moe_expert_arena &A, int T, int k) { return ptc_ws(A, T, k, nullptr).bytes; }

template <int BITS>
static moe_status run_tc(const moe_expert_arena &A, const uint16_t *x, int T, const float *w, int k,
                         const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out, moe_dtype dt,
                         int accumulate, const PtcWs &d, int32_t *status, cudaStream_t s)
{
    using namespace ptc;
    int64_t n = (int64_t)T * k;
    tile_prefix_kernel<<<1, 1024, 0, s>>>(offsets, A.E, BM, d.mt_prefix);
    moe_status st = check_launch("tile_prefix");
    if (st != MOE_OK) return st;
    int64_t gthreads = n * (A.H / 16);
    int gblocks = (int)std::min<int64_t>((gthreads + 255) / 256, (int64_t)sm_count() * 16);
    gather_x_kernel<<<gblocks, 256, 0, s>>>(x, perm, offsets, A.E, k, A.H, d.xg);
    st = check_launch("gather_x");
    if (st != MOE_OK) return st;
    int rbH = BITS == 2 ? A.H / 4 : A.H / 4 + A.H / 8;
    int rbI = BITS == 2 ? A.I / 4 : A.I / 4 + A.I / 8;
    int grid = sm_count();
    // gate/up
    CUtensorMap mx, mh;
    st = make_map(&mx, d.xg, n, A.H);
    if (st != MOE_OK) return st;
    Args a = {};
    a.codes = A.gu_codes;
    a.scales = A.gu_scales;
    a.row_bytes = rbH;
    a.scale_row = A.H / 32;
    a.codes_expert_stride = (int64_t)2 * A.I * rbH;
    a.scales_expert_stride = (int64_t)2 * A.I * (A.H / 32);
    a.K = A.H;
    a.rows = A.I;
    a.up_rows = A.I;
    a.tiles_n = (A.I + BN / 2 - 1) / (BN / 2);
    a.offsets = offsets;
    a.mt_prefix = d.mt_prefix;
    a.E = A.E;
    a.h_out = d.h;
    a.status = status;
    st = launch_gemm<BITS, true>(a, mx, grid, s);
    if (st != MOE_OK) return st;
    // down
    st = make_map(&mh, d.h, n, A.I);
    if (st != MOE_OK) return st;
    Args b = a;
    b.codes = A.d_codes;
    b.scales = A.d_scales;
    b.row_bytes = rbI;
    b.scale_row = A.I / 32;
    b.codes_expert_stride = (int64_t)A.H * rbI;
    b.scales_expert_stride = (int64_t)A.H * (A.I / 32);
    b.K = A.I;
    b.rows = A.H;
    b.up_rows = 0;
    b.tiles_n = (A.H + BN - 1) / BN;
    b.h_out = nullptr;
    b.y_out = d.y;
    st = launch_gemm<BITS, false>(b, mh, grid, s);
    if (st != MOE_OK) return st;
    return launch_combine(d.y, w, inv, T, k, A.H, out, dt, accumulate, s);
}

moe_status prefill_tc_forward(const moe_expert_arena &A, const uint16_t *x, int T, const float *w, int k,
                              const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out, moe_dtype dt,
                              int accumulate, void *ws, int32_t *dev_status, cudaStream_t s)
{
    PtcWs d = ptc_ws(A, T, k, ws);
    if (A.bits == 2) return run_tc<2>(A, x, T, w, k, offsets, perm, inv, out, dt, accumulate, d, dev_status, s);
    return run_tc<3>(A, x, T, w, k, offsets, perm, inv, out, dt, accumulate, d, dev_status, s);
}

}  // namespace moe
