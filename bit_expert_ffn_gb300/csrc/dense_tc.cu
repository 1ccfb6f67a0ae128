// dense_tc.cu -- persistent tcgen05 GEMM for bf16 operands that are both in
// global memory (the router and the shared expert at prefill sizes).
//
// One CTA per SM walks (128-row M tile, 256-column N tile) items.  Warp 0
// loads both operands with TMA (128-byte swizzle, four 48 KiB stages),
// warp 1 issues tcgen05.mma (M=128, N=256, K=16, bf16 x bf16 -> fp32 in
// TMEM, two accumulator buffers so the epilogue of one tile overlaps the
// next tile's MMAs), warp 2 owns the TMEM allocation and waits on the
// barriers for warp 1 (a named barrier hands each ready step over, so the
// issuing thread does no mbarrier waits of its own), and warps 4..7 move
// the accumulators out (one TMEM lane quadrant each).  Every wait is
// bounded: after about 2 s the CTA records MOE_ERR_TIMEOUT and stops.
#include "dense_tc.cuh"
#include "tc.cuh"

namespace moe {
namespace dtc {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
constexpr int THREADS = 256;
constexpr int EPI_WARP0 = 4;
constexpr unsigned long long kWaitNs = 2000000000ull;

struct Params {
    int M, N, nk, a_kb, b_kb, tiles_n, total;
    uint16_t *hsplit;
    const float *bias;
    void *out;
    int out_bf16, accumulate, vec;
    int32_t *status;
};

struct Shared {
    uint64_t full[STAGES], empty[STAGES];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem;
    volatile int abort;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    return (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1) dense_kernel(const __grid_constant__ Params p,
                                                           const __grid_constant__ CUtensorMap ma,
                                                           const __grid_constant__ CUtensorMap mb0,
                                                           const __grid_constant__ CUtensorMap mb1)
{
    extern __shared__ __align__(1024) char dyn_raw[];
    char *dyn = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    char *sA = dyn;
    char *sB = dyn + STAGES * A_BYTES;
    __shared__ Shared S;
    const int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            tc::mbar_init(&S.full[s], 1);
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
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch_desc(&ma);
        tc::tma_prefetch_desc(&mb0);
        if (EPI == DENSE_SWIGLU_SPLIT) tc::tma_prefetch_desc(&mb1);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int it = 0;
            for (int tile = blockIdx.x; tile < p.total && !S.abort; tile += gridDim.x) {
                int mt = tile / p.tiles_n, nt = tile % p.tiles_n;
                for (int kb = 0; kb < p.nk; kb++, it++) {
                    int s = it % STAGES, u = it / STAGES;
                    if (u > 0 && !tc::mbar_wait(&S.empty[s], (u - 1) & 1, kWaitNs)) {
                        set_status(p.status, MOE_ERR_TIMEOUT);
                        S.abort = 1;
                        break;
                    }
                    int ka = (kb % p.a_kb) * BK, kbb = (kb % p.b_kb) * BK;
                    tc::mbar_arrive_expect_tx(&S.full[s], A_BYTES + B_BYTES);
                    char *b = sB + s * B_BYTES;
                    tc::tma_load_2d(sA + s * A_BYTES, &ma, ka, mt * BM, &S.full[s]);
                    if (EPI == DENSE_SWIGLU_SPLIT) {
                        tc::tma_load_2d(b, &mb0, kbb, nt * (BN / 2), &S.full[s]);
                        tc::tma_load_2d(b + B_BYTES / 2, &mb1, kbb, nt * (BN / 2), &S.full[s]);
                    } else {
                        tc::tma_load_2d(b, &mb0, kbb, nt * BN, &S.full[s]);
                        tc::tma_load_2d(b + B_BYTES / 2, &mb0, kbb, nt * BN + BN / 2, &S.full[s]);
                    }
                }
            }
            // no copy may still be in flight when the CTA leaves
            for (int s = 0; s < STAGES && s < it; s++) {
                int u = (s + STAGES * ((it - 1 - s) / STAGES)) / STAGES;
                if (!tc::mbar_wait(&S.full[s], u & 1, kWaitNs)) set_status(p.status, MOE_ERR_TIMEOUT);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA: warp 2 waits on the barriers, lane 0 of warp 1 issues; they meet
        // at named barrier 3 every step, so the issuing thread never waits on
        // an mbarrier behind its own queued MMAs.  The OR over the barrier
        // makes every stop decision common to both warps.
        const bool issuer = warp == 1;
        const uint32_t idesc = tc::idesc_f16_f32(BM, BN, true);
        int it = 0, j = 0;
        bool stop = false;
        for (int tile = blockIdx.x; tile < p.total; tile += gridDim.x, j++) {
            int acc = j & 1, v = j >> 1;
            bool fail = false;
            if (!issuer && lane == 0)
                fail = S.abort || (v > 0 && !tc::mbar_wait(&S.acc_empty[acc], (v - 1) & 1, kWaitNs));
            if (tc::named_sync_or(3, 64, fail)) {
                stop = true;
                break;
            }
            uint32_t d = tmem + (uint32_t)(acc * BN);
            for (int kb = 0; kb < p.nk; kb++, it++) {
                int s = it % STAGES, u = it / STAGES;
                fail = false;
                if (!issuer && lane == 0) fail = !tc::mbar_wait(&S.full[s], u & 1, kWaitNs);
                if (tc::named_sync_or(3, 64, fail)) {
                    stop = true;
                    break;
                }
                if (issuer && lane == 0) {
                    tc::tc_fence_after();
                    uint32_t abase = tc::smem_u32(sA + s * A_BYTES), bbase = tc::smem_u32(sB + s * B_BYTES);
#pragma unroll
                    for (int k16 = 0; k16 < BK / 16; k16++)
                        tc::mma_f16_ss(d, tc::desc_kmajor_sw128(abase + k16 * 32), tc::desc_kmajor_sw128(bbase + k16 * 32),
                                       idesc, (kb | k16) ? 1u : 0u);
                    tc::mma_commit(&S.empty[s]);
                }
            }
            if (stop) break;
            if (issuer && lane == 0) tc::mma_commit(&S.acc_full[acc]);
        }
        if (stop && !issuer && lane == 0) {
            set_status(p.status, MOE_ERR_TIMEOUT);
            S.abort = 1;
        }
        if (issuer && lane == 0) {
            tc::mma_commit(&S.mma_done);
            if (!tc::mbar_wait(&S.mma_done, 0, kWaitNs)) set_status(p.status, MOE_ERR_TIMEOUT);
        }
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + 4) {
        // ---------------- epilogue
        const int q = warp - EPI_WARP0;
        int j = 0;
        for (int tile = blockIdx.x; tile < p.total && !S.abort; tile += gridDim.x, j++) {
            int acc = j & 1, v = j >> 1;
            if (!tc::mbar_wait(&S.acc_full[acc], v & 1, kWaitNs)) {
                if (lane == 0) set_status(p.status, MOE_ERR_TIMEOUT);
                S.abort = 1;
                break;
            }
            tc::tc_fence_after();
            int mt = tile / p.tiles_n, nt = tile % p.tiles_n;
            int row = mt * BM + q * 32 + lane;
            bool valid = row < p.M;
            uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if (EPI == DENSE_SWIGLU_SPLIT) {
                for (int c = 0; c < BN / 2; c += 32) {
                    int r0 = nt * (BN / 2) + c;
                    if (r0 >= p.N) break;  // warp-uniform
                    uint32_t g[32], u[32];
                    __syncwarp();
                    tc::tmem_ld_32x32b_x32(tbase + c, g);
                    tc::tmem_ld_32x32b_x32(tbase + BN / 2 + c, u);
                    tc::tmem_ld_wait();
                    if (valid) {
                        uint32_t hi[16], lo[16];
#pragma unroll
                        for (int i = 0; i < 16; i++) {
                            float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                            float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                            uint16_t a0 = f32_to_bf16(h0), a1 = f32_to_bf16(h1);
                            hi[i] = (uint32_t)a0 | ((uint32_t)a1 << 16);
                            lo[i] = pack_bf16x2(h0 - bf16_to_f32(a0), h1 - bf16_to_f32(a1));
                        }
                        uint4 *dh = reinterpret_cast<uint4 *>(p.hsplit + (int64_t)row * 2 * p.N + r0);
                        uint4 *dl = reinterpret_cast<uint4 *>(p.hsplit + (int64_t)row * 2 * p.N + p.N + r0);
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            dh[i] = make_uint4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]);
                            dl[i] = make_uint4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]);
                        }
                    }
                }
            } else {
                for (int c = 0; c < BN; c += 32) {
                    int c0 = nt * BN + c;
                    if (c0 >= p.N) break;  // warp-uniform
                    uint32_t r[32];
                    __syncwarp();
                    tc::tmem_ld_32x32b_x32(tbase + c, r);
                    tc::tmem_ld_wait();
                    if (valid) {
                    float v32[32];
#pragma unroll
                    for (int i = 0; i < 32; i++) v32[i] = __uint_as_float(r[i]);
                    bool full = p.vec && c0 + 32 <= p.N;
                    if (p.bias) {
                        if (full) {
                            const float4 *b4 = reinterpret_cast<const float4 *>(p.bias + c0);
#pragma unroll
                            for (int i = 0; i < 8; i++) {
                                float4 bb = __ldg(b4 + i);
                                v32[4 * i] += bb.x;
                                v32[4 * i + 1] += bb.y;
                                v32[4 * i + 2] += bb.z;
                                v32[4 * i + 3] += bb.w;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                if (c0 + i < p.N) v32[i] += p.bias[c0 + i];
                        }
                    }
                    int64_t o = (int64_t)row * p.N + c0;
                    if (p.out_bf16) {
                        uint16_t *ob = static_cast<uint16_t *>(p.out) + o;
                        if (full) {
                            uint4 *o4 = reinterpret_cast<uint4 *>(ob);
#pragma unroll
                            for (int i = 0; i < 4; i++) {
                                uint4 old = make_uint4(0, 0, 0, 0);
                                if (p.accumulate) old = o4[i];
                                uint32_t ow[4] = {old.x, old.y, old.z, old.w}, nw[4];
#pragma unroll
                                for (int e = 0; e < 4; e++)
                                    nw[e] = pack_bf16x2(bf16_to_f32((uint16_t)(ow[e] & 0xffffu)) + v32[8 * i + 2 * e],
                                                        bf16_to_f32((uint16_t)(ow[e] >> 16)) + v32[8 * i + 2 * e + 1]);
                                o4[i] = make_uint4(nw[0], nw[1], nw[2], nw[3]);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                if (c0 + i < p.N) ob[i] = f32_to_bf16((p.accumulate ? bf16_to_f32(ob[i]) : 0.f) + v32[i]);
                        }
                    } else {
                        float *of = static_cast<float *>(p.out) + o;
                        if (full) {
                            float4 *o4 = reinterpret_cast<float4 *>(of);
#pragma unroll
                            for (int i = 0; i < 8; i++) {
                                float4 old = p.accumulate ? o4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                                o4[i] = make_float4(old.x + v32[4 * i], old.y + v32[4 * i + 1], old.z + v32[4 * i + 2],
                                                    old.w + v32[4 * i + 3]);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                if (c0 + i < p.N) of[i] = (p.accumulate ? of[i] : 0.f) + v32[i];
                        }
                    }
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.acc_empty[acc]);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

static size_t smem_bytes() { return (size_t)STAGES * (A_BYTES + B_BYTES) + 1024; }

}  // namespace dtc

// ---------------------------------------------------------------- host
typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static moe_status encode_fn(EncodeTiled *fn)
{
    // resolved once (thread-safe static initialisation); the runtime hands
    // out the driver's entry point, so nothing links against libcuda
    static EncodeTiled cached = []() -> EncodeTiled {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) return nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    if (!cached) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    *fn = cached;
    return MOE_OK;
}

moe_status make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes, int64_t rows,
                        int64_t cols, int box_cols, int box_rows, CUtensorMapSwizzle swizzle)
{
    EncodeTiled enc;
    moe_status st = encode_fn(&enc);
    if (st != MOE_OK) return st;
    if (rows < 1 || cols < 1 || !aligned16(base) || (cols * elem_bytes) % 16 != 0)
        return fail(MOE_ERR_INVALID_ARG, "tensor map: %lld x %lld elements of %d bytes at %p", (long long)rows,
                    (long long)cols, elem_bytes, base);
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * elem_bytes)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t elem[2] = {1, 1};
    CUresult r = enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return MOE_OK;
}

bool dense_tc_supported(const DenseGemm &g, DenseEpi epi)
{
    if (g.M < 1 || g.N < 1 || g.K < 64 || g.K % 64 || g.a_cols % 64 || g.b_cols % 64) return false;
    if (!aligned16(g.A) || !aligned16(g.B0)) return false;
    if (epi == DENSE_SWIGLU_SPLIT) return g.B1 && aligned16(g.B1) && g.hsplit && aligned16(g.hsplit) && g.N % 32 == 0;
    return g.out != nullptr;
}

moe_status dense_tc_gemm(const DenseGemm &g, DenseEpi epi, cudaStream_t s)
{
    using namespace dtc;
    if (!dense_tc_supported(g, epi)) return fail(MOE_ERR_UNSUPPORTED, "dense tensor-core GEMM: unsupported shape");
    CUtensorMap ma, mb0, mb1;
    int b_rows = g.N;
    moe_status st = make_tmap_2d(&ma, g.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.M, g.a_cols, BK, BM);
    if (st == MOE_OK) st = make_tmap_2d(&mb0, g.B0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b_rows, g.b_cols, BK, BN / 2);
    if (st == MOE_OK && epi == DENSE_SWIGLU_SPLIT)
        st = make_tmap_2d(&mb1, g.B1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b_rows, g.b_cols, BK, BN / 2);
    else
        mb1 = mb0;
    if (st != MOE_OK) return st;
    Params p = {};
    p.M = g.M;
    p.N = g.N;
    p.nk = g.K / BK;
    p.a_kb = g.a_cols / BK;
    p.b_kb = g.b_cols / BK;
    p.tiles_n = epi == DENSE_SWIGLU_SPLIT ? (g.N + BN / 2 - 1) / (BN / 2) : (g.N + BN - 1) / BN;
    int64_t total = (int64_t)((g.M + BM - 1) / BM) * p.tiles_n;
    if (total > INT32_MAX) return fail(MOE_ERR_UNSUPPORTED, "dense GEMM: %lld tiles", (long long)total);
    p.total = (int)total;
    p.hsplit = g.hsplit;
    p.bias = g.bias;
    p.out = g.out;
    p.out_bf16 = g.out_bf16;
    p.accumulate = g.accumulate;
    p.vec = aligned16(g.out) && (g.bias == nullptr || aligned16(g.bias)) && g.N % 8 == 0;
    p.status = g.status;
    int grid = (int)std::min<int64_t>(total, sm_count());
    auto fn = epi == DENSE_SWIGLU_SPLIT ? dense_kernel<DENSE_SWIGLU_SPLIT> : dense_kernel<DENSE_OUT>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes());
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "dense GEMM attribute: %s", cudaGetErrorString(e));
    fn<<<grid, THREADS, smem_bytes(), s>>>(p, ma, mb0, mb1);
    return check_launch(epi == DENSE_SWIGLU_SPLIT ? "dense_tc_swiglu" : "dense_tc_out");
}

}  // namespace moe
