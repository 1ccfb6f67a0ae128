// prefill_tc.cu -- the prefill path of moe_expert_forward on the tcgen05
// tensor cores (sm_103a): grouped GEMMs over the experts' token lists with
// the 2-/3-bit weights dequantised to fp16 in shared memory.
//
//   gate/up:  D[r][p] = sum_i dq(W_e[r][i]) * x[tok(p)][i]   for 64 gate rows r
//             and the 64 matching up rows, then h[p][r] = silu(g) * u   (fp16)
//   down:     y[p][o] = sum_r dq(Wd_e[o][r]) * h[p][r]                  (fp32)
//   combine:  out[t][o] = sum_j w[t][j] y[inv[t*k+j]][o]   (slot order)
//
// The weights are the MMA's M operand (128 rows per tile) and an expert's
// sorted pairs its N operand (up to 256 per tile, in steps of 32, so an
// expert with few pairs costs few columns).  One CTA per SM runs a
// persistent loop over (expert, up to 256 pairs) x (128 weight rows) tiles:
//   warp 0      TMA: the packed codes of each 64-wide K step and the pairs'
//               fp16 rows (128-byte swizzle);
//   warps 8-15  dequantise the codes into the swizzled K-major fp16 tile
//               (two threads per row, one 32-weight block each);
//   warp 1      tcgen05.mma M=128, N=32..256, K=16 into TMEM (two
//               accumulator buffers: the epilogue of one tile overlaps the
//               next tile's MMAs);
//   warp 2      owns the TMEM allocation;
//   warps 4-7   epilogue: TMEM -> registers, transposed through shared
//               memory, written by TMA stores (the gate/up epilogue first
//               hands the up rows' values to the gate rows' warps).
// Operands are fp16: x (bf16) converts exactly, the weights (c - mid) * s
// round once to fp16, h rounds to fp16 between the two GEMMs.  Every wait is
// bounded: after about 2 s the CTA records MOE_ERR_TIMEOUT and stops.
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

constexpr int BM = 128;  // weight rows per tile (MMA M); gate/up: 64 gate + 64 up rows
constexpr int BT = 256;  // sorted pairs per tile at most (MMA N, multiples of 32)
constexpr int BK = 64;   // reduction per stage: one 128-byte swizzle row of fp16
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK * 2;   // dequantised weights
constexpr int B_BYTES = BT * BK * 2;   // pairs' rows
constexpr int C_BYTES = BM * 16;       // 2-bit (low) codes of one stage: 16 B per row
constexpr int HI_BYTES = BM * 16;      // 3-bit high planes of two stages: 16 B per row
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + C_BYTES + HI_BYTES;
constexpr int XCH_BYTES = 32 * 64 * 4;  // up values: 32 pairs x 64 rows, fp32
constexpr int STG_BYTES = 32 * 32 * 4;  // one 32 x 32 output block
constexpr int OFF_XCH = STAGES * STAGE_BYTES;
constexpr int OFF_STG = OFF_XCH + 2 * XCH_BYTES;
constexpr int SMEM_BYTES = OFF_STG + 8 * STG_BYTES + 1024;
constexpr int THREADS = 512;
constexpr int DQ_WARP0 = 8;
constexpr int EPI_WARP0 = 4;
constexpr unsigned long long kWaitNs = 2000000000ull;
static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0 && OFF_STG % 1024 == 0, "1024-byte aligned areas");

struct Args {
    const uint16_t *scales;
    int64_t scales_expert_stride;  // elements
    int64_t code_rows;             // rows of the code tensor per expert (2I or H)
    int scale_row;                 // K / 32
    int K, rows, up_rows;          // rows: output rows (I or H); up_rows: where the up rows start (I)
    int rtiles;                    // weight-row tiles per pair tile
    int hi_x;                      // byte offset of the 3-bit high plane inside a code row
    const int32_t *offsets, *mt_prefix;
    int E;
    uint16_t *h_out;  // gate/up: fp16 [pairs][I] (columns permuted within 16-groups)
    float *y_out;     // down: fp32 [pairs][H]
    int32_t *status;
};

struct Shared {
    uint64_t tfull[STAGES], cfull[STAGES], wfull[STAGES], empty[STAGES];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem;
    volatile int abort;
};

struct Tile {
    int e, p0, cnt, rt, n32;  // n32: 32-pair chunks (MMA N = 32 n32)
};

__device__ __forceinline__ Tile decode_tile(const Args &a, int tile)
{
    Tile t;
    int tt = tile / a.rtiles;
    t.rt = tile - tt * a.rtiles;
    t.e = expert_of_tile(a.mt_prefix, a.E, tt);
    t.p0 = a.offsets[t.e] + (tt - a.mt_prefix[t.e]) * BT;
    t.cnt = min(BT, a.offsets[t.e + 1] - t.p0);
    t.n32 = (t.cnt + 31) >> 5;
    return t;
}

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
// values (c - mid) * s.  The code lands in mantissa bits 1-2 (and bit 3 for
// the 3-bit high plane) of 512.0, so 512 + c is exact; subtracting 512 + mid
// is exact too and the product with s rounds once.
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

// One 32-weight block (codes c0: weights 0-15, c1: 16-31; 3-bit high plane
// word hw; fp16 scale bits sc) into the four 16-byte chunks 4*half .. 4*half+3
// of swizzled row r.
template <int BITS>
__device__ __forceinline__ void dq_block(uint32_t c0, uint32_t c1, uint32_t hw, uint32_t sc, char *rowp, int r,
                                         int half)
{
    __half2 s2 = __half2half2(__ushort_as_half((uint16_t)sc));
#pragma unroll
    for (int g = 0; g < 2; g++) {
        uint32_t w = g ? c1 : c0;
        uint32_t hword = BITS == 3 ? (g ? hw >> 8 : hw) : 0u;
        uint32_t lo4[4], hi4[4];
        dq_chunk<BITS, 0>(w, hword, s2, lo4);
        dq_chunk<BITS, 4>(w, hword, s2, hi4);
        int c = 4 * half + 2 * g;
        *reinterpret_cast<uint4 *>(rowp + ((c ^ (r & 7)) << 4)) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
        *reinterpret_cast<uint4 *>(rowp + (((c + 1) ^ (r & 7)) << 4)) = make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
    }
}

// Shared-memory reads of what TMA wrote: ordered after the mbarrier wait by
// that wait's memory clobber.
__device__ __forceinline__ uint32_t lds32(const void *p) { return *reinterpret_cast<const uint32_t *>(p); }

template <int BITS, bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1) tc_gemm_kernel(const __grid_constant__ Args a,
                                                             const __grid_constant__ CUtensorMap tok_map,
                                                             const __grid_constant__ CUtensorMap code_map,
                                                             const __grid_constant__ CUtensorMap out_map)
{
    extern __shared__ __align__(1024) char dyn_raw[];
    char *dyn = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Shared S;
    const int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            tc::mbar_init(&S.tfull[s], 1);
            tc::mbar_init(&S.cfull[s], 1);
            tc::mbar_init(&S.wfull[s], 8);
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
        tc::tma_prefetch_desc(&tok_map);
        tc::tma_prefetch_desc(&code_map);
        tc::tma_prefetch_desc(&out_map);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;
    const int total = a.mt_prefix[a.E] * a.rtiles;
    const int nk = a.K / BK;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: codes and the pairs' rows
            int it = 0;
            for (int tile = blockIdx.x; tile < total && !S.abort; tile += gridDim.x) {
                Tile t = decode_tile(a, tile);
                int64_t base = (int64_t)t.e * a.code_rows;
                int r0 = (int)(base + (SWIGLU ? t.rt * 64 : t.rt * 128));
                int r1 = SWIGLU ? (int)(base + a.up_rows + t.rt * 64) : r0 + 64;
                for (int kb = 0; kb < nk; kb++, it++) {
                    int s = it % STAGES, u = it / STAGES;
                    if (u > 0 && !tc::mbar_wait(&S.empty[s], (u - 1) & 1, kWaitNs)) {
                        set_status(a.status, MOE_ERR_TIMEOUT);
                        S.abort = 1;
                        break;
                    }
                    char *st = dyn + s * STAGE_BYTES;
                    char *cs = st + A_BYTES + B_BYTES;
                    bool hi = BITS == 3 && !(kb & 1);
                    tc::mbar_arrive_expect_tx(&S.cfull[s], C_BYTES + (hi ? HI_BYTES : 0));
                    tc::tma_load_2d(cs, &code_map, kb * 16, r0, &S.cfull[s]);
                    tc::tma_load_2d(cs + C_BYTES / 2, &code_map, kb * 16, r1, &S.cfull[s]);
                    if (hi) {
                        tc::tma_load_2d(cs + C_BYTES, &code_map, a.hi_x + (kb >> 1) * 16, r0, &S.cfull[s]);
                        tc::tma_load_2d(cs + C_BYTES + HI_BYTES / 2, &code_map, a.hi_x + (kb >> 1) * 16, r1,
                                        &S.cfull[s]);
                    }
                    tc::mbar_arrive_expect_tx(&S.tfull[s], t.n32 * 32 * BK * 2);
                    for (int i = 0; i < t.n32; i++)
                        tc::tma_load_2d(st + A_BYTES + i * 32 * BK * 2, &tok_map, kb * BK, t.p0 + 32 * i, &S.tfull[s]);
                }
            }
            // no copy may still be in flight when the CTA leaves (after a timeout elsewhere)
            for (int s = 0; s < STAGES && s < it; s++) {
                int u = (s + STAGES * ((it - 1 - s) / STAGES)) / STAGES;
                if (!tc::mbar_wait(&S.cfull[s], u & 1, kWaitNs) || !tc::mbar_wait(&S.tfull[s], u & 1, kWaitNs))
                    set_status(a.status, MOE_ERR_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int it = 0, j = 0;
            for (int tile = blockIdx.x; tile < total && !S.abort; tile += gridDim.x, j++) {
                Tile t = decode_tile(a, tile);
                const uint32_t idesc = tc::idesc_f16_f32(BM, 32 * t.n32);
                int acc = j & 1, v = j >> 1;
                if (v > 0 && !tc::mbar_wait(&S.acc_empty[acc], (v - 1) & 1, kWaitNs)) {
                    set_status(a.status, MOE_ERR_TIMEOUT);
                    S.abort = 1;
                    break;
                }
                tc::tc_fence_after();
                uint32_t d = tmem + (uint32_t)(acc * BT);
                bool ok = true;
                for (int kb = 0; kb < nk; kb++, it++) {
                    int s = it % STAGES, u = it / STAGES;
                    if (!tc::mbar_wait(&S.wfull[s], u & 1, kWaitNs) || !tc::mbar_wait(&S.tfull[s], u & 1, kWaitNs)) {
                        set_status(a.status, MOE_ERR_TIMEOUT);
                        S.abort = 1;
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    char *st = dyn + s * STAGE_BYTES;
                    uint32_t abase = tc::smem_u32(st), bbase = tc::smem_u32(st + A_BYTES);
#pragma unroll
                    for (int k16 = 0; k16 < BK / 16; k16++)
                        tc::mma_f16_ss(d, tc::desc_kmajor_sw128(abase + k16 * 32), tc::desc_kmajor_sw128(bbase + k16 * 32),
                                       idesc, (kb | k16) ? 1u : 0u);
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
        // ---------------- epilogue: TMEM -> registers -> shared (transposed) -> TMA store
        const int q = warp - EPI_WARP0;  // TMEM lane quadrant: weight rows 32q .. 32q+31 of the tile
        float *xch = reinterpret_cast<float *>(dyn + OFF_XCH);
        int nstore = 0;
        int j = 0;
        // the gate/up warps meet at named barriers, so they decide together
        // whether to stop (the OR over the four warps); the down warps alone
        for (int tile = blockIdx.x; tile < total && (SWIGLU || !S.abort); tile += gridDim.x, j++) {
            int acc = j & 1, v = j >> 1;
            bool stop = !tc::mbar_wait(&S.acc_full[acc], v & 1, kWaitNs);
            if (stop) {
                if (lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
                S.abort = 1;
            }
            stop = stop || S.abort;
            if (SWIGLU) stop = tc::named_sync_or(2, 128, stop);
            if (stop) break;
            tc::tc_fence_after();
            Tile t = decode_tile(a, tile);
            uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BT);
            for (int ch = 0; ch < t.n32; ch++) {
                uint32_t r[32];
                __syncwarp();
                tc::tmem_ld_32x32b_x32(tbase + ch * 32, r);
                tc::tmem_ld_wait();
                int tok0 = ch * 32;
                bool full = tok0 + 32 <= t.cnt;
                int nv = min(32, t.cnt - tok0);
                if (SWIGLU) {
                    float *xb = xch + (ch & 1) * (XCH_BYTES / 4);
                    if (q >= 2) {
                        // up rows: hand the values to the warps holding the gate rows
#pragma unroll
                        for (int i = 0; i < 32; i++) xb[i * 64 + (q - 2) * 32 + lane] = __uint_as_float(r[i]);
                    }
                    tc::named_sync(1, 128);
                    int orow0 = t.rt * 64 + q * 32;  // first output row of this warp
                    if (q < 2 && orow0 < a.rows) {
                        int pos = (lane & ~15) + perm16(lane & 15);  // stored column within the warp's 32
                        uint16_t hv[32];
#pragma unroll
                        for (int i = 0; i < 32; i++) {
                            float g = __uint_as_float(r[i]);
                            hv[i] = __half_as_ushort(__float2half_rn(silu(g) * xb[i * 64 + q * 32 + lane]));
                        }
                        if (full) {
                            uint16_t *sb = reinterpret_cast<uint16_t *>(dyn + OFF_STG + (q * 2 + (nstore & 1)) * STG_BYTES);
                            if (lane == 0) tc::bulk_wait_read<1>();
                            __syncwarp();
#pragma unroll
                            for (int i = 0; i < 32; i++) sb[i * 32 + pos] = hv[i];
                            tc::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tc::tma_store_2d(&out_map, orow0, t.p0 + tok0, sb);
                                tc::bulk_commit();
                            }
                            nstore++;
                        } else {
                            uint16_t *dst = a.h_out + (int64_t)(t.p0 + tok0) * a.rows + orow0 + pos;
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                if (i < nv) dst[(int64_t)i * a.rows] = hv[i];
                        }
                    }
                } else {
                    int o0 = t.rt * 128 + q * 32;
                    if (o0 < a.rows) {
                        if (full) {
                            float *sb = reinterpret_cast<float *>(dyn + OFF_STG + (q * 2 + (nstore & 1)) * STG_BYTES);
                            if (lane == 0) tc::bulk_wait_read<1>();
                            __syncwarp();
#pragma unroll
                            for (int i = 0; i < 32; i++) sb[i * 32 + lane] = __uint_as_float(r[i]);
                            tc::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tc::tma_store_2d(&out_map, o0, t.p0 + tok0, sb);
                                tc::bulk_commit();
                            }
                            nstore++;
                        } else {
                            float *dst = a.y_out + (int64_t)(t.p0 + tok0) * a.rows + o0 + lane;
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                if (i < nv) dst[(int64_t)i * a.rows] = __uint_as_float(r[i]);
                        }
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.acc_empty[acc]);
        }
        if (lane == 0) tc::bulk_wait_all();
        __syncwarp();
    } else if (warp >= DQ_WARP0) {
        // ---------------- dequantisation: thread = (row r of the tile, 32-weight half of the stage)
        const int d = threadIdx.x - DQ_WARP0 * 32;
        const int r = d & (BM - 1), half = d >> 7;
        const bool vec_scales = (a.K & 255) == 0;  // rows of scales 16-byte aligned: 8 blocks per load
        int it = 0;
        for (int tile = blockIdx.x; tile < total && !S.abort; tile += gridDim.x) {
            Tile t = decode_tile(a, tile);
            int orow = SWIGLU ? t.rt * 64 + (r & 63) : t.rt * 128 + r;
            bool valid = orow < a.rows;
            int64_t mrow = SWIGLU && r >= 64 ? (int64_t)a.up_rows + orow : orow;
            const uint16_t *sp = a.scales + (int64_t)t.e * a.scales_expert_stride + mrow * a.scale_row;
            uint4 cur4 = make_uint4(0, 0, 0, 0), nxt4 = cur4;
            if (valid && vec_scales) nxt4 = __ldg(reinterpret_cast<const uint4 *>(sp));
            uint32_t hw_next = 0;
            bool aborted = false;
            for (int kb = 0; kb < nk; kb++, it++) {
                int s = it % STAGES, u = it / STAGES;
                uint32_t sc = 0;
                if (valid) {
                    if (vec_scales) {
                        if ((kb & 3) == 0) {
                            cur4 = nxt4;
                            if (kb + 4 < nk) nxt4 = __ldg(reinterpret_cast<const uint4 *>(sp + 8 * ((kb >> 2) + 1)));
                        }
                        int wsel = kb & 3;
                        uint32_t w2 = wsel == 0 ? cur4.x : wsel == 1 ? cur4.y : wsel == 2 ? cur4.z : cur4.w;
                        sc = half ? w2 >> 16 : w2 & 0xffffu;
                    } else {
                        sc = __ldg(sp + 2 * kb + half);
                    }
                }
                if ((u > 0 && !tc::mbar_wait(&S.empty[s], (u - 1) & 1, kWaitNs)) ||
                    !tc::mbar_wait(&S.cfull[s], u & 1, kWaitNs)) {
                    if (lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
                    S.abort = 1;
                    aborted = true;
                    break;
                }
                char *st = dyn + s * STAGE_BYTES;
                const char *cs = st + A_BYTES + B_BYTES;
                char *rowp = st + r * 128;
                if (valid) {
                    uint2 cw = *reinterpret_cast<const uint2 *>(cs + r * 16 + half * 8);
                    uint32_t hw = 0;
                    if (BITS == 3) {
                        if (!(kb & 1)) {
                            hw = lds32(cs + C_BYTES + r * 16 + half * 4);
                            hw_next = lds32(cs + C_BYTES + r * 16 + 8 + half * 4);
                        } else {
                            hw = hw_next;
                        }
                    }
                    dq_block<BITS>(cw.x, cw.y, hw, sc, rowp, r, half);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        *reinterpret_cast<uint4 *>(rowp + (((4 * half + c) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&S.wfull[s]);
            }
            if (aborted) break;
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

template <int BITS, bool SWIGLU>
static moe_status launch_gemm(const Args &a, const CUtensorMap &tok, const CUtensorMap &codes,
                              const CUtensorMap &out, int grid, cudaStream_t s)
{
    auto fn = tc_gemm_kernel<BITS, SWIGLU>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "tc gemm attribute: %s", cudaGetErrorString(e));
    fn<<<grid, THREADS, SMEM_BYTES, s>>>(a, tok, codes, out);
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

// Code rows must be 16-byte multiples for the TMA copies of the codes:
// 2-bit rows are K/4 bytes (K a multiple of 64), 3-bit rows 3K/8 bytes (K a
// multiple of 128).
bool prefill_tc_supported(const moe_expert_arena &A)
{
    int q = A.bits == 2 ? 64 : 128;
    return A.H % q == 0 && A.I % q == 0 && A.H >= 64 && A.I >= 64 && (int64_t)A.E * 2 * A.I < INT32_MAX &&
           (int64_t)A.E * A.H < INT32_MAX;
}

size_t prefill_tc_workspace_bytes(const moe_expert_arena &A, int T, int k) { return ptc_ws(A, T, k, nullptr).bytes; }

template <int BITS>
static moe_status run_tc(const moe_expert_arena &A, const uint16_t *x, int T, const float *w, int k,
                         const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out, moe_dtype dt,
                         int accumulate, const PtcWs &d, int32_t *status, cudaStream_t s)
{
    using namespace ptc;
    int64_t n = (int64_t)T * k;
    tile_prefix_kernel<<<1, 1024, 0, s>>>(offsets, A.E, BT, d.mt_prefix);
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
    const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // gate/up: codes [E * 2I][rbH], pairs' rows xg [n][H] -> h [n][I]
    CUtensorMap mtok, mcode, mout;
    st = make_tmap_2d(&mtok, d.xg, F16, 2, n, A.H, BK, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK)
        st = make_tmap_2d(&mcode, A.gu_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (int64_t)A.E * 2 * A.I, rbH, 16, 64,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st == MOE_OK) st = make_tmap_2d(&mout, d.h, F16, 2, n, A.I, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != MOE_OK) return st;
    Args a = {};
    a.scales = A.gu_scales;
    a.scales_expert_stride = (int64_t)2 * A.I * (A.H / 32);
    a.code_rows = (int64_t)2 * A.I;
    a.scale_row = A.H / 32;
    a.K = A.H;
    a.rows = A.I;
    a.up_rows = A.I;
    a.rtiles = (A.I + 63) / 64;
    a.hi_x = A.H / 4;
    a.offsets = offsets;
    a.mt_prefix = d.mt_prefix;
    a.E = A.E;
    a.h_out = d.h;
    a.status = status;
    st = launch_gemm<BITS, true>(a, mtok, mcode, mout, grid, s);
    if (st != MOE_OK) return st;
    // down: codes [E * H][rbI], h [n][I] -> y [n][H]
    st = make_tmap_2d(&mtok, d.h, F16, 2, n, A.I, BK, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK)
        st = make_tmap_2d(&mcode, A.d_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (int64_t)A.E * A.H, rbI, 16, 64,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st == MOE_OK)
        st = make_tmap_2d(&mout, d.y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, n, A.H, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != MOE_OK) return st;
    Args b = a;
    b.scales = A.d_scales;
    b.scales_expert_stride = (int64_t)A.H * (A.I / 32);
    b.code_rows = A.H;
    b.scale_row = A.I / 32;
    b.K = A.I;
    b.rows = A.H;
    b.up_rows = 0;
    b.rtiles = (A.H + 127) / 128;
    b.hi_x = A.I / 4;
    b.h_out = nullptr;
    b.y_out = d.y;
    st = launch_gemm<BITS, false>(b, mtok, mcode, mout, grid, s);
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
