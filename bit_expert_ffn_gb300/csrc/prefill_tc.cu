// prefill_tc.cu -- the prefill path of moe_expert_forward on the tcgen05
// tensor cores (sm_103a): grouped GEMMs over the experts' token lists with
// the 2-/3-bit weights dequantised to fp16 in shared memory.
//
//   gate/up:  D[r][p] = sum_i dq(W_e[r][i]) * x[tok(p)][i]   for 64 gate rows r
//             and the 64 matching up rows, then h[p][r] = silu(g) * u   (fp16)
//   down:     y[p][o] = sum_r dq(Wd_e[o][r]) * h[p][r]   (fp32 accumulate, stored fp16)
//   combine:  out[t][o] = sum_j w[t][j] y[inv[t*k+j]][o]   (slot order)
//
// The weights are the MMA's M operand (128 rows per tile) and an expert's
// sorted pairs its N operand (up to 192 per tile, in steps of 32, so an
// expert with few pairs costs few columns).  One CTA per SM runs a
// persistent loop over (expert, up to 192 pairs) x (128 weight rows) tiles,
// streaming the reduction dimension in 64-wide steps through three rings,
// each as deep as its producer's latency asks:
//   warp 3      TMA: packed codes and scales of each step into the code
//               ring (shared memory, several steps ahead);
//   warp 0      TMA: the pairs' fp16 (FP8: e4m3) rows of each step into the
//               pair ring (shared memory, 128-byte swizzle);
//   warps 16-17 wait for free slots of the pair and code rings and hand
//               them to the two TMA warps (an mbarrier call right after
//               queued copies would stall the issuing thread);
//   warps 8-15  dequantise codes straight into the weight ring in TMEM
//               (tcgen05.st; a warp per lane quadrant, two warps per
//               quadrant taking every other step: more warps only add
//               issue-slot contention with the MMA and epilogue warps);
//   warp 1      tcgen05.mma M=128, N=32..192, K=16 with the weights read
//               from TMEM and the pairs from shared memory, into two TMEM
//               accumulator buffers (the epilogue of one tile overlaps the
//               next tile's MMAs);
//   warp 2      owns the TMEM allocation and waits on the rings' barriers
//               for warp 1, handing each ready step over by a named barrier;
//   warps 4-7   epilogue: TMEM -> registers, transposed through shared
//               memory, written by TMA stores (the gate/up epilogue first
//               hands the up rows' values to the gate rows' warps); the
//               FP8 kernels add warps 18-21, a second set that takes the
//               odd 32-pair chunks of each tile.
// Keeping the weights out of shared memory leaves its bandwidth to the
// pairs' rows, which the tensor cores read there.
// Operands are fp16: x (bf16) converts exactly while 2^-14 <= |x| <= 65504
// (smaller values keep fewer bits, down to 2^-24, and bf16 values of 65536 or
// more have no finite fp16), the weights (c - mid) * s round once to fp16, h
// rounds to fp16 between the two GEMMs, and each pair's down output y (fp32
// accumulated) is stored as fp16 for the combine, which halves the bytes of
// the layer's largest intermediate.  A value that leaves fp16's finite range
// on the way (|x|, |(c - mid) s|, |h| or |y| rounding to 65520 or more, or a
// non-finite one) sets MOE_ERR_RANGE; the kernels still write every output
// (such entries become infinite).  Every wait is bounded: after about 2 s the
// CTA records MOE_ERR_TIMEOUT and stops.
//
// Inside every 16-element group of the reduction dimension the operands are
// stored in the order 0,8,1,9,...,7,15 (both x/h and the weights, so the
// product is unchanged): a code word then dequantises with one LOP3 and one
// fp16 FMA per pair of weights.
//
// The FP8 variant (MOE_PATH_PREFILL_FP8, 2-bit codes) runs the same kernel
// on e4m3 operands (tcgen05.mma kind::f8f6f4, K = 32 per instruction): a
// step still moves 128 bytes of every pair row and fills 32 TMEM columns per
// weight row, but covers 128 reduction elements.  Every operand carries a
// power-of-two scaling -- one exponent per weight row (from the row's largest
// block scale), per pair for x and per pair for h -- which the epilogue
// undoes on the fp32 accumulators.  A 32-weight block decodes through a
// four-entry byte table of its e4m3 values (one conversion per block) and
// byte selects, which put the even elements of each 16-group before the odd
// ones; x and h are stored in that order too.
//
// The pages place the routed experts' FFN on the GPU and add their outputs
// ("How Strata runs a 125-billion-parameter model on a single 12 GB to 24 GB
// graphics card", Step 2) and read long prompts in chunks of tokens
// ("Strata Open-Source Runtime ...", section "Prefill and Long Context").
#include <cuda.h>

#include "common.cuh"
#include "dense_tc.cuh"
#include "dequant.cuh"
#include "prefill.cuh"
#include "tc.cuh"

namespace moe {
namespace ptc {

constexpr int BM = 128;  // weight rows per tile (MMA M); gate/up: 64 gate + 64 up rows
constexpr int BT = 192;  // sorted pairs per tile at most (MMA N, multiples of 32)
constexpr int BK = 64;   // reduction per step: one 128-byte swizzle row of fp16
constexpr int B_BYTES = BT * BK * 2;   // one step of the pairs' rows
constexpr int C_LO = 0;                // code entry: low codes, 16 B (FP8: 32 B) per row, then scales of
                                       //   four (FP8: two) steps, then 3-bit high planes of two (FP8: one)
                                       //   steps, 16 B per row each (offsets in Cfg)
constexpr int NA = 4, NB = 6;          // weight ring (TMEM), pair ring (shared memory)
// TMEM columns: two accumulators of BT fp32 columns, then the weight ring
// (a 64-wide fp16 step is 32 columns).
constexpr int TM_A = 2 * BT;
static_assert(TM_A + NA * 32 <= 512, "TMEM columns");
constexpr int XCH_BYTES = 32 * 64 * 4;  // up values of one 32-pair chunk: 64 rows, fp32
// Epilogue area.  Every storing warp has two fp16 32 x 32 staging blocks used
// in turn, so one chunk's TMA store can still be reading a block while the
// next chunk fills the other.  down: eight warps x two blocks; gate/up: the
// four gate warps x two blocks, then one exchange buffer per warp set.
constexpr int STG = 32 * 32 * 2;
constexpr int OFF_XCH = 4 * 2 * STG;
constexpr int EPI_BYTES = OFF_XCH + 2 * XCH_BYTES > 8 * 2 * STG ? OFF_XCH + 2 * XCH_BYTES : 8 * 2 * STG;
// 22 warps: 0-3, 16-17 producers and MMA, 4-7 epilogue, 8-15 dequantisation,
// 18-21 the FP8 variant's second epilogue set (the fp16 kernels launch 18 warps)
constexpr int DQ_WARP0 = 8;  // warps 8..15 dequantise: two threads per weight row, each every other step
constexpr int DQ_WARPS = 8;
constexpr int RING_WARP = 16;  // waits for free pair slots for the pair TMA issuer
constexpr int CODE_WARP = 17;  // waits for free code slots for the code TMA issuer
constexpr int EPI_WARP0 = 4;   // epilogue warps 4..7 and, for FP8, 18..21 (the odd 32-pair chunks);
constexpr int EPI_WARP1 = 18;  // a warp reads TMEM lane quadrant warp % 4
constexpr int NC_MAX = 8;
constexpr unsigned long long kWaitNs = 2000000000ull;
// fp32 values of this magnitude or more (and NaN) round to a non-finite fp16
constexpr float kF16Limit = 65520.f;

// Shared-memory plan per bit width and operand type: the code entry carries
// the 3-bit high planes only for 3 bits, which leaves room for fewer entries.
// A step of the FP8 variant covers 128 elements of the reduction: 32 bytes
// of low codes per row, four block scales, and (3 bits) 16 bytes of high bits.
template <int BITS, bool FP8 = false>
struct Cfg {
    static constexpr int BKE = FP8 ? 128 : BK;          // reduction elements per step (128 bytes of a pair row)
    static constexpr int CODE_STEP = FP8 ? 32 : 16;     // low-code bytes per weight row and step
    static constexpr int C_SC = BM * CODE_STEP;         // offset of the scales in a code entry
    static constexpr int C_HI = C_SC + BM * 16;         // offset of the 3-bit high planes (16 B per row)
    static constexpr int C_BYTES = C_SC + BM * 16 + (BITS == 3 ? BM * 16 : 0);
    // code-ring entries (an FP8 entry covers twice the reduction; with 3 bits five leave room for the
    // static spreading table)
    static constexpr int NC = BITS == 2 ? 8 : (FP8 ? 5 : 6);
    // epilogue warp sets: the FP8 tiles' MMAs are short enough that a second set of four
    // epilogue warps pays; with fp16 operands the extra warps only take issue slots
    static constexpr int NSET = FP8 ? 2 : 1;
    static constexpr int THREADS = FP8 ? 704 : 576;
    static constexpr int OFF_B = 0;
    static constexpr int OFF_C = OFF_B + NB * B_BYTES;
    static constexpr int OFF_E = OFF_C + NC * C_BYTES;
    static constexpr int SMEM = OFF_E + EPI_BYTES + 1024;
    static_assert(OFF_C % 1024 == 0 && OFF_E % 1024 == 0 && B_BYTES % 1024 == 0, "1024-byte aligned areas");
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
    static_assert(NC <= NC_MAX, "code ring");
};

struct Args {
    const uint16_t *scales;
    int64_t scales_expert_stride;  // elements
    int64_t code_rows;             // rows of the code tensor per expert (2I or H)
    int scale_row;                 // K / 32
    int K, rows, up_rows;          // rows: output rows (I or H); up_rows: where the up rows start (I)
    int rtiles;                    // weight-row tiles per pair tile
    int hi_x;                      // byte offset of the 3-bit high plane inside a code row
    int scale_tma;                 // scales come by TMA (rows of K/32 scales are 16-byte multiples)
    const int4 *table;          // per pair tile: expert, first pair, pair count
    const int32_t *ntt;         // number of pair tiles
    uint16_t *h_out;  // gate/up: fp16 [pairs][I] (columns permuted within 16-groups)
    uint16_t *y_out;  // down: fp16 [pairs][H]
    int32_t *status;
    // FP8 variant: the power-of-two exponents of the operands' scalings
    const int8_t *kw;       // per weight row, [E][code_rows]
    const int32_t *pexp;    // per pair: x's (gate/up) or h's (down)
};

struct Shared {
    uint64_t afull[NA], aempty[NA], bfull[NB], bempty[NB], cfull[NC_MAX], cempty[NC_MAX];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem;
    volatile int abort;
};

struct Tile {
    int e, p0, cnt, rt, n32;  // n32: 32-pair chunks (MMA N = 32 n32)
};

// A tile's entry of the pair-tile table; loaded one tile ahead of its use,
// so the load's latency hides behind the current tile's work.
__device__ __forceinline__ int4 tile_entry(const Args &a, int tile, int total)
{
    return tile < total ? __ldg(&a.table[tile / a.rtiles]) : make_int4(0, 0, 0, 0);
}

__device__ __forceinline__ Tile make_tile(const Args &a, int4 e, int tile)
{
    Tile t;
    t.e = e.x;
    t.p0 = e.y;
    t.cnt = e.z;
    t.rt = tile % a.rtiles;
    t.n32 = (t.cnt + 31) >> 5;
    return t;
}

// table[mt_prefix[e] + j] = (e, offsets[e] + j*BT, pairs of that tile): one thread per expert.
__global__ void tile_table_kernel(const int32_t *__restrict__ offsets, const int32_t *__restrict__ mt_prefix, int E,
                                  int bt, int4 *__restrict__ table)
{
    int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    int n = offsets[e + 1] - offsets[e], base = mt_prefix[e];
    for (int j = 0; j * bt < n; j++) table[base + j] = make_int4(e, offsets[e] + j * bt, min(bt, n - j * bt), 0);
}

// Ring slot and phase parity of step `it` in a ring of n entries.
struct Slot {
    int s;
    uint32_t par;
    bool reuse;  // the slot held an earlier step: wait until it is free
};
__device__ __forceinline__ Slot slot_of(int it, int n)
{
    int u = it / n;
    return Slot{it - u * n, (uint32_t)(u & 1), u > 0};
}

// Stored position, inside its 16-element group, of element m.
__host__ __device__ __forceinline__ int perm16(int m) { return m < 8 ? 2 * m : 2 * (m - 8) + 1; }

// One 16-weight group (codes w, 3-bit high bits hw already aligned to the
// group, fp16 scale bits sc) as eight fp16x2 words: word m holds the stored
// positions 2m and 2m+1 of the group (true elements m and m+8), the values
// (c - mid) * s.  The centred codes come out exact (one LOP3 and one fp16 FMA
// per word, see dq_pair); the product with s rounds once.
template <int BITS>
__device__ __forceinline__ void dq_group(uint32_t w, uint32_t hw, uint32_t sc, uint32_t (&v)[8])
{
    const __half2 s2 = __half2half2(__ushort_as_half((uint16_t)sc));
    const DqWord<BITS> d = dq_word<BITS>(w);
#define MOE_DQ(M)                                                                                       \
    {                                                                                                   \
        uint32_t c = dq_pair<M, BITS, 0>(d, hw);                                                        \
        __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&c), s2);                                      \
        v[M] = *reinterpret_cast<uint32_t *>(&r);                                                       \
    }
    MOE_DQ(0) MOE_DQ(1) MOE_DQ(2) MOE_DQ(3) MOE_DQ(4) MOE_DQ(5) MOE_DQ(6) MOE_DQ(7)
#undef MOE_DQ
}

// ---- FP8 variant ------------------------------------------------------------
// Stored position, inside its 16-element group, of element m in the FP8
// operands: the even elements first, then the odd ones (the order in which
// lut_word below decodes a code word).
__host__ __device__ __forceinline__ int pos8(int m) { return (m >> 1) | ((m & 1) << 3); }

// 2^e as an fp32 for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// The exponent that scales a set of magnitudes with maximum amax (>= 0,
// finite) into [128, 256): 7 - floor(log2 amax), clamped to [-64, 64]; 0 for
// amax = 0.  fp32 subnormal maxima clamp to 64.
__device__ __forceinline__ int fp8_exponent(float amax)
{
    if (amax == 0.f) return 0;
    const int be = (__float_as_int(amax) >> 23) & 0xff;
    const int k = be == 0 ? 64 : 7 - (be - 127);
    return k < -64 ? -64 : (k > 64 ? 64 : k);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// e4m3 bytes of two fp32 values, rounded to nearest (ties to even) with
// saturation: the low byte is lo's, the high byte hi's.
__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo)
{
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return h;
}

// The four e4m3 values a 2-bit block with scale S = s 2^kw stands for, one
// byte per code: e4m3((c - 1.5) S) for c = 0..3.  Each is rounded once from
// its exact value (1.5 S and 0.5 S are exact in fp32), and e4m3 rounding is
// symmetric, so the negative entries are the positive ones with the sign bit.
__device__ __forceinline__ uint32_t lut_2bit(float S)
{
    const uint32_t h = e4m3x2(1.5f * S, 0.5f * S);  // byte 0: 0.5 S, byte 1: 1.5 S
    return prmt(h, 0u, 0x1001u) ^ 0x8080u;          // bytes: -1.5 S, -0.5 S, 0.5 S, 1.5 S
}

// A word of sixteen 2-bit codes (weight j at bits 2j..2j+1) as sixteen e4m3
// bytes, one byte select per four weights: o[0] holds weights 0, 2, 4, 6,
// o[1] 8, 10, 12, 14, o[2] 1, 3, 5, 7 and o[3] 9, 11, 13, 15 (pos8 order).
__device__ __forceinline__ void lut_word(uint32_t w, uint32_t lut, uint32_t *o)
{
    const uint32_t ev = w & 0x33333333u, od = (w >> 2) & 0x33333333u;  // one code per nibble
    o[0] = prmt(lut, 0u, ev);
    o[1] = prmt(lut, 0u, ev >> 16);
    o[2] = prmt(lut, 0u, od);
    o[3] = prmt(lut, 0u, od >> 16);
}

// The eight e4m3 values a 3-bit block with scale S stands for, e4m3((c - 3.5) S):
// hi holds codes 4..7 (0.5 S .. 3.5 S, each rounded once from its exact
// value), lo codes 0..3 (the same magnitudes in reverse order, sign bit set).
__device__ __forceinline__ void lut_3bit(float S, uint32_t &lo, uint32_t &hi)
{
    hi = e4m3x2(1.5f * S, 0.5f * S) | (e4m3x2(3.5f * S, 2.5f * S) << 16);
    lo = prmt(hi, 0u, 0x0123u) ^ 0x80808080u;
}

// Byte b's bit j (the high bit of the j-th weight of a gathered byte: the
// even or odd weights 0, 2, 4, 6 of a 16-weight word at j = 0, 2, 4, 6 and
// 8, 10, 12, 14 at j = 1, 3, 5, 7) moved to bit 2 of the nibble that
// lut_word's byte select gives that weight.
__host__ __device__ __forceinline__ uint32_t spread_byte(int b)
{
    uint32_t v = 0;
    for (int j = 0; j < 8; j++)
        if ((b >> j) & 1) v |= 1u << (4 * ((j & 1) ? 4 + (j >> 1) : j >> 1) + 2);
    return v;
}

// A word of sixteen 3-bit codes: low bits w (weight j at bits 2j..2j+1),
// high bits hw as laid out for the word's half of the block (weights 0-7 at
// bits 0-7, 8-15 at bits 16-23); output as lut_word's.
__device__ __forceinline__ void lut_word3(uint32_t w, uint32_t hw, uint32_t lo, uint32_t hi, const uint32_t *spread,
                                          uint32_t *o)
{
    const uint32_t be = (hw & 0x55u) | ((hw >> 15) & 0xAAu);         // high bits of the even weights
    const uint32_t bo = ((hw >> 1) & 0x55u) | ((hw >> 16) & 0xAAu);  // and of the odd ones
    const uint32_t ev = (w & 0x33333333u) | spread[be], od = ((w >> 2) & 0x33333333u) | spread[bo];
    o[0] = prmt(lo, hi, ev);
    o[1] = prmt(lo, hi, ev >> 16);
    o[2] = prmt(lo, hi, od);
    o[3] = prmt(lo, hi, od >> 16);
}

// silu with a fast division: h is rounded to fp16 right after, far coarser
// than the approximation's couple of fp32 ulps.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Shared-memory reads of what TMA wrote: ordered after the mbarrier wait by
// that wait's memory clobber.
__device__ __forceinline__ uint32_t lds32(const void *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Waits for the last phase each slot of a ring was filled in (its copies
// have landed); used before the CTA leaves, so no copy is still in flight.
__device__ __forceinline__ void drain_ring(uint64_t *full, int n, int issued, int32_t *status)
{
    for (int s = 0; s < n && s < issued; s++) {
        int last = s + n * ((issued - 1 - s) / n);
        if (!tc::mbar_wait(&full[s], (uint32_t)((last / n) & 1), kWaitNs)) set_status(status, MOE_ERR_TIMEOUT);
    }
}

template <int BITS, bool SWIGLU, bool FP8>
__global__ void __launch_bounds__(Cfg<BITS, FP8>::THREADS, 1) tc_gemm_kernel(const __grid_constant__ Args a,
                                                             const __grid_constant__ CUtensorMap tok_map,
                                                             const __grid_constant__ CUtensorMap tok_full_map,
                                                             const __grid_constant__ CUtensorMap code_map,
                                                             const __grid_constant__ CUtensorMap scale_map,
                                                             const __grid_constant__ CUtensorMap out_map,
                                                             const __grid_constant__ CUtensorMap hi_map)
{
    using C = Cfg<BITS, FP8>;
    // FP8 with 3-bit codes: the high bits of eight weights (a byte) spread to bit 2 of the nibbles of
    // their byte-select word
    __shared__ uint32_t spread8[(FP8 && BITS == 3) ? 256 : 1];
    if constexpr (FP8 && BITS == 3)
        for (int i = threadIdx.x; i < 256; i += blockDim.x) spread8[i] = spread_byte(i);
    extern __shared__ __align__(1024) char dyn_raw[];
    char *dyn = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Shared S;
    const int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        for (int s = 0; s < NA; s++) {
            tc::mbar_init(&S.afull[s], 4);  // the four lane-quadrant warps of a step
            tc::mbar_init(&S.aempty[s], 1);
        }
        for (int s = 0; s < NB; s++) {
            tc::mbar_init(&S.bfull[s], 1);
            tc::mbar_init(&S.bempty[s], 1);
        }
        for (int s = 0; s < C::NC; s++) {
            tc::mbar_init(&S.cfull[s], 1);
            tc::mbar_init(&S.cempty[s], 4);
        }
        for (int i = 0; i < 2; i++) {
            tc::mbar_init(&S.acc_full[i], 1);
            tc::mbar_init(&S.acc_empty[i], 4 * C::NSET);
        }
        tc::mbar_init(&S.mma_done, 1);
        S.abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 2) tc::tmem_alloc(&S.tmem, 512);
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch_desc(&tok_map);
        tc::tma_prefetch_desc(&tok_full_map);
        tc::tma_prefetch_desc(&code_map);
        if (a.scale_tma) tc::tma_prefetch_desc(&scale_map);
        tc::tma_prefetch_desc(&out_map);
        if (FP8 && BITS == 3) tc::tma_prefetch_desc(&hi_map);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = S.tmem;
    const int total = *a.ntt * a.rtiles;
    const int nk = a.K / C::BKE;

    if (warp == 0 || warp == 3 || warp == RING_WARP || warp == CODE_WARP) {
        // ---------------- TMA: warps 16 and 17 wait for free pair and code slots and
        // post the expected bytes; they hand each step over by named barriers 4
        // (pair rows, issued by warp 0) and 5 (codes and scales, issued by warp 3),
        // so the issuing threads make no mbarrier calls between their copies.
        // The two rings run independently, each as far ahead as its own slots
        // allow.  The OR over each barrier makes the stop decision common to a
        // waiter and its issuer.
        // roles: 0 pair waiter, 1 pair issuer, 2 code issuer, 3 code waiter
        const int role = warp == RING_WARP ? 0 : warp == 0 ? 1 : warp == 3 ? 2 : 3;
        const uint32_t cbytes = BM * C::CODE_STEP + (BITS == 3 ? BM * 16 : 0) + (a.scale_tma ? BM * 16 : 0);
        int it = 0;
        bool stop = false;
        int4 nxt = tile_entry(a, blockIdx.x, total);
        for (int tile = blockIdx.x; tile < total && !stop; tile += gridDim.x) {
            Tile t = make_tile(a, nxt, tile);
            nxt = tile_entry(a, tile + gridDim.x, total);
            int64_t base = (int64_t)t.e * a.code_rows;
            int r0 = (int)(base + (SWIGLU ? t.rt * 64 : t.rt * 128));
            int r1 = SWIGLU ? (int)(base + a.up_rows + t.rt * 64) : r0 + 64;
            for (int kb = 0; kb < nk; kb++, it++) {
                Slot b = slot_of(it, NB), c = slot_of(it, C::NC);
                if (role <= 1) {
                    bool fail = false;
                    if (role == 0 && lane == 0) {
                        fail = S.abort || (b.reuse && !tc::mbar_wait_sleep(&S.bempty[b.s], b.par ^ 1, kWaitNs));
                        if (!fail) tc::mbar_arrive_expect_tx(&S.bfull[b.s], t.n32 * 32 * BK * 2);
                    }
                    if (tc::named_sync_or(4, 64, fail)) {
                        stop = true;
                        break;
                    }
                    if (role == 1 && lane == 0) {
                        char *bs = dyn + C::OFF_B + b.s * B_BYTES;
                        if (t.n32 * 32 == BT) {  // a full tile: one box of BT rows
                            tc::tma_load_2d(bs, &tok_full_map, kb * C::BKE, t.p0, &S.bfull[b.s]);
                        } else {
                            for (int i = 0; i < t.n32; i++)
                                tc::tma_load_2d(bs + i * 32 * BK * 2, &tok_map, kb * C::BKE, t.p0 + 32 * i,
                                                &S.bfull[b.s]);
                        }
                    }
                }
                if (role >= 2) {
                    bool fail = false;
                    if (role == 3 && lane == 0) {
                        fail = S.abort || (c.reuse && !tc::mbar_wait_sleep(&S.cempty[c.s], c.par ^ 1, kWaitNs));
                        if (!fail) tc::mbar_arrive_expect_tx(&S.cfull[c.s], cbytes);
                    }
                    if (tc::named_sync_or(5, 64, fail)) {
                        stop = true;
                        break;
                    }
                    if (role == 2 && lane == 0) {
                        char *cs = dyn + C::OFF_C + c.s * C::C_BYTES;
                        tc::tma_load_2d(cs + C_LO, &code_map, kb * C::CODE_STEP, r0, &S.cfull[c.s]);
                        tc::tma_load_2d(cs + C_LO + 64 * C::CODE_STEP, &code_map, kb * C::CODE_STEP, r1,
                                        &S.cfull[c.s]);
                        if (a.scale_tma) {  // 16 B of scales per row: four steps (FP8: two)
                            const int sx = (FP8 ? kb >> 1 : kb >> 2) * 8;
                            tc::tma_load_2d(cs + C::C_SC, &scale_map, sx, r0, &S.cfull[c.s]);
                            tc::tma_load_2d(cs + C::C_SC + 64 * 16, &scale_map, sx, r1, &S.cfull[c.s]);
                        }
                        if (BITS == 3) {  // 16 B of high bits per row: two steps (FP8: one)
                            const CUtensorMap *hm = FP8 ? &hi_map : &code_map;
                            const int hx = a.hi_x + (FP8 ? kb : kb >> 1) * 16;
                            tc::tma_load_2d(cs + C::C_HI, hm, hx, r0, &S.cfull[c.s]);
                            tc::tma_load_2d(cs + C::C_HI + 64 * 16, hm, hx, r1,
                                            &S.cfull[c.s]);
                        }
                    }
                }
            }
        }
        if (stop && (role == 0 || role == 3) && lane == 0) {
            set_status(a.status, MOE_ERR_TIMEOUT);
            S.abort = 1;
        }
        // no copy may still be in flight when the CTA leaves (after a timeout elsewhere);
        // the waiter posted the bytes of every step it handed over, so each slot's
        // last phase completes once its copies land
        if (role == 1 && lane == 0) drain_ring(S.bfull, NB, it, a.status);
        if (role == 2 && lane == 0) drain_ring(S.cfull, C::NC, it, a.status);
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA: warp 2 waits on the rings' barriers, lane 0 of warp 1 issues.
        // They meet at named barrier 3 every step, so the issuing thread never
        // waits on an mbarrier behind its own queued MMAs (such a wait takes
        // longer than a step's MMAs).  The OR over the barrier makes every
        // stop decision common to both warps.
        const bool issuer = warp == 1;
        int it = 0, j = 0;
        bool stop = false;
        int4 nxt = tile_entry(a, blockIdx.x, total);
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, j++) {
            Tile t = make_tile(a, nxt, tile);
            nxt = tile_entry(a, tile + gridDim.x, total);
            int acc = j & 1, v = j >> 1;
            bool fail = false;
            if (!issuer && lane == 0)
                fail = S.abort || (v > 0 && !tc::mbar_wait(&S.acc_empty[acc], (v - 1) & 1, kWaitNs));
            if (tc::named_sync_or(3, 64, fail)) {
                stop = true;
                break;
            }
            const uint32_t idesc = tc::idesc_f16_f32(BM, 32 * t.n32);
            uint32_t d = tmem + (uint32_t)(acc * BT);
            // two steps per hand-over (one named barrier for eight MMAs)
            for (int kb = 0; kb < nk; kb += 2) {
                const int ns = kb + 1 < nk ? 2 : 1;
                fail = false;
                if (!issuer && lane == 0) {
                    for (int j = 0; j < ns && !fail; j++) {
                        const Slot sa = slot_of(it + j, NA), sb = slot_of(it + j, NB);
                        fail = !tc::mbar_wait(&S.afull[sa.s], sa.par, kWaitNs) ||
                               !tc::mbar_wait(&S.bfull[sb.s], sb.par, kWaitNs);
                    }
                }
                if (tc::named_sync_or(3, 64, fail)) {
                    stop = true;
                    break;
                }
                if (issuer && lane == 0) {
                    tc::tc_fence_after();
                    for (int j = 0; j < ns; j++) {
                        const Slot sa = slot_of(it + j, NA), sb = slot_of(it + j, NB);
                        const uint32_t abase = tmem + (uint32_t)(TM_A + sa.s * 32);
                        // the step's B descriptor once; each instruction's 32 bytes of K advance its start
                        // address field (bytes / 16) by 2, which stays inside the 14-bit field
                        const uint64_t bdesc = tc::desc_kmajor_sw128(tc::smem_u32(dyn + C::OFF_B + sb.s * B_BYTES));
                        const uint32_t acc0 = (kb + j) ? 1u : 0u;
#pragma unroll
                        for (int k16 = 0; k16 < BK / 16; k16++) {  // 32 bytes of K per instruction
                            if constexpr (FP8)
                                tc::mma_f8_ts(d, abase + k16 * 8, bdesc + (uint64_t)(2 * k16), idesc, k16 ? 1u : acc0);
                            else
                                tc::mma_f16_ts(d, abase + k16 * 8, bdesc + (uint64_t)(2 * k16), idesc, k16 ? 1u : acc0);
                        }
                        tc::mma_commit(&S.aempty[sa.s]);
                        tc::mma_commit(&S.bempty[sb.s]);
                    }
                }
                it += ns;
            }
            if (stop) break;
            if (issuer && lane == 0) tc::mma_commit(&S.acc_full[acc]);
        }
        if (stop && !issuer && lane == 0) {
            set_status(a.status, MOE_ERR_TIMEOUT);
            S.abort = 1;
        }
        if (issuer && lane == 0) {
            // every MMA of this CTA has finished before TMEM is released
            tc::mma_commit(&S.mma_done);
            if (!tc::mbar_wait(&S.mma_done, 0, kWaitNs)) set_status(a.status, MOE_ERR_TIMEOUT);
        }
    } else if ((warp >= EPI_WARP0 && warp < EPI_WARP0 + 4) ||
               (C::NSET == 2 && warp >= EPI_WARP1 && warp < EPI_WARP1 + 4)) {
        // ---------------- epilogue: TMEM -> registers -> shared (transposed) -> TMA store.  With two
        // sets of four warps (one per TMEM lane quadrant each) they take the even and the odd
        // 32-pair chunks of a tile, so two chunks drain at once.
        const int q = warp & 3;  // TMEM lane quadrant: weight rows 32q .. 32q+31 of the tile
        const int set = warp >= EPI_WARP1 ? 1 : 0;
        const int xbar = set ? 6 : 1;  // the set's named barrier for the gate/up exchange
        float *xch = reinterpret_cast<float *>(dyn + C::OFF_E + OFF_XCH);
        // this warp's two staging blocks (gate/up: only the gate warps store)
        char *stg = dyn + C::OFF_E + (SWIGLU ? set * 2 + (q & 1) : set * 4 + q) * 2 * STG;
        bool out_of_range = false;  // an h or y value that has no finite fp16
        int j = 0, nst = 0;         // nst: TMA stores this warp issued (block nst & 1 is next)
        // the gate/up warps meet at named barriers, so they decide together
        // whether to stop (the OR over the eight warps); the down warps alone
        int4 nxt = tile_entry(a, blockIdx.x, total);
        for (int tile = blockIdx.x; tile < total && (SWIGLU || !S.abort); tile += gridDim.x, j++) {
            int acc = j & 1, v = j >> 1;
            Tile t = make_tile(a, nxt, tile);
            nxt = tile_entry(a, tile + gridDim.x, total);
            // FP8: the exponents this tile needs are loaded before the accumulator wait (and each
            // chunk's pair exponents one chunk ahead), so their latency hides behind the wait
            int kwr = 0, pe_next = 0;
            if constexpr (FP8) {
                const int orow = SWIGLU ? t.rt * 64 + (q & 1) * 32 + lane : t.rt * 128 + q * 32 + lane;
                const int64_t mrow = SWIGLU && q >= 2 ? (int64_t)a.up_rows + orow : orow;
                if (orow < a.rows) kwr = __ldg(a.kw + (int64_t)t.e * a.code_rows + mrow);
                if (set * 32 + lane < t.cnt) pe_next = __ldg(a.pexp + t.p0 + set * 32 + lane);
            }
            bool stop = !tc::mbar_wait_sleep(&S.acc_full[acc], v & 1, kWaitNs);
            stop = __any_sync(0xffffffffu, stop);  // the warp's TMEM loads need all its lanes
            if (stop) {
                if (lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
                S.abort = 1;
            }
            stop = stop || S.abort;
            if (SWIGLU) stop = tc::named_sync_or(2, 128 * C::NSET, stop);
            if (stop) break;
            tc::tc_fence_after();
            uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BT);
            const float frow = exp2i(-kwr);  // FP8: 2^-kw of this lane's weight row (kw lies in [-9, 31])
            for (int ch = set; ch < t.n32; ch += C::NSET) {
                uint32_t r[32];
                __syncwarp();
                tc::tmem_ld_32x32b_x32(tbase + ch * 32, r);
                int tok0 = ch * 32;
                bool full = tok0 + 32 <= t.cnt;
                int nv = min(32, t.cnt - tok0);
                int pe = 0;
                if constexpr (FP8) {
                    pe = pe_next;
                    if (tok0 + 64 + lane < t.cnt) pe_next = __ldg(a.pexp + t.p0 + tok0 + 64 + lane);  // FP8: 2 sets
                }
                tc::tmem_ld_wait();
                if constexpr (FP8) {
                    // undo the operands' scalings: 2^-kw of the weight row, then 2^-e of pair i (e in
                    // [-64, 64]); the two factors are exact, so their order does not matter while the
                    // product stays a normal fp32
                    const float fpair = exp2i(-pe);
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        r[i] = __float_as_uint(__uint_as_float(r[i]) * frow * __shfl_sync(0xffffffffu, fpair, i));
                }
                if (SWIGLU) {
                    // up rows: hand the values to the warps holding the gate rows.  One set alternates
                    // two exchange buffers (a barrier per chunk); with two sets each has one buffer and
                    // waits, before writing it, for its gate warps to have read the previous chunk.
                    float *xb = xch + (C::NSET == 2 ? set : (ch & 1)) * (XCH_BYTES / 4);
                    if (C::NSET == 2) tc::named_sync(xbar, 128);
                    if (q >= 2) {
#pragma unroll
                        for (int i = 0; i < 32; i++) xb[i * 64 + (q - 2) * 32 + lane] = __uint_as_float(r[i]);
                    }
                    tc::named_sync(xbar, 128);
                    int orow0 = t.rt * 64 + q * 32;  // first output row of this warp
                    if (q < 2 && orow0 < a.rows) {
                        // stored column within the warp's 32
                        int pos = (lane & ~15) + (FP8 ? pos8(lane & 15) : perm16(lane & 15));
                        uint16_t hv[32];
#pragma unroll
                        for (int i = 0; i < 32; i++) {
                            float g = __uint_as_float(r[i]);
                            const float hf = silu_fast(g) * xb[i * 64 + q * 32 + lane];
                            out_of_range |= i < nv && !(fabsf(hf) < kF16Limit);
                            hv[i] = __half_as_ushort(__float2half_rn(hf));
                        }
                        if (full) {
                            // the block's previous store (two stores back) has finished reading it
                            uint16_t *sb = reinterpret_cast<uint16_t *>(stg + (nst & 1) * STG);
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
                            nst++;
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
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            out_of_range |= i < nv && !(fabsf(__uint_as_float(r[i])) < kF16Limit);
                        if (full) {
                            uint16_t *sb = reinterpret_cast<uint16_t *>(stg + (nst & 1) * STG);
                            if (lane == 0) tc::bulk_wait_read<1>();
                            __syncwarp();
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                sb[i * 32 + lane] = __half_as_ushort(__float2half_rn(__uint_as_float(r[i])));
                            tc::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tc::tma_store_2d(&out_map, o0, t.p0 + tok0, sb);
                                tc::bulk_commit();
                            }
                            nst++;
                        } else {
                            uint16_t *dst = a.y_out + (int64_t)(t.p0 + tok0) * a.rows + o0 + lane;
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                if (i < nv) dst[(int64_t)i * a.rows] = __half_as_ushort(__float2half_rn(__uint_as_float(r[i])));
                        }
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.acc_empty[acc]);
        }
        if (lane == 0) tc::bulk_wait_all();
        if (__any_sync(0xffffffffu, out_of_range) && lane == 0) set_status(a.status, MOE_ERR_RANGE);
        __syncwarp();
    } else if (warp >= DQ_WARP0 && warp < DQ_WARP0 + DQ_WARPS) {
        // ---------------- dequantisation into TMEM: warp = (lane quadrant qd, step group jg); the
        // four warps of group jg take every other step, each a whole step of its 32 rows
        // (one 16-byte read of the row's codes, four 16-weight groups, one store wait per step)
        const int dw = warp - DQ_WARP0;
        const int qd = warp & 3, jg = dw >> 2;
        const int r = qd * 32 + lane;  // weight row of the tile = TMEM lane
        const uint32_t tq = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)TM_A;
        int base = 0;  // steps of the earlier tiles
        bool aborted = false, scale_out_of_range = false;
        int4 nxt = tile_entry(a, blockIdx.x, total);
        for (int tile = blockIdx.x; tile < total && !S.abort && !aborted; tile += gridDim.x) {
            Tile t = make_tile(a, nxt, tile);
            nxt = tile_entry(a, tile + gridDim.x, total);
            int orow = SWIGLU ? t.rt * 64 + (r & 63) : t.rt * 128 + r;
            bool valid = orow < a.rows;
            int64_t mrow = SWIGLU && r >= 64 ? (int64_t)a.up_rows + orow : orow;
            // scales from global memory only when they cannot come by TMA
            const uint16_t *sp = a.scales + (int64_t)t.e * a.scales_expert_stride + mrow * a.scale_row;
            float p2kw = 1.f;  // FP8: 2^kw, the scaling of this weight row (kw in [-9, 31])
            if constexpr (FP8)
                if (valid) p2kw = exp2i(__ldg(a.kw + (int64_t)t.e * a.code_rows + mrow));
            // the steps of this tile that belong to group jg: global step index = jg (mod 2)
            for (int kb = (jg - base) & 1; kb < nk; kb += 2) {
                const int it = base + kb;
                Slot c = slot_of(it, C::NC), sa = slot_of(it, NA);
                uint32_t sc = 0;  // the step's two block scales (low half: first block)
                uint2 sc4 = make_uint2(0u, 0u);  // FP8: the step's four block scales
                if (valid && !a.scale_tma) {
                    if constexpr (FP8) sc4 = __ldg(reinterpret_cast<const uint2 *>(sp + 4 * kb));
                    else sc = (uint32_t)__ldg(sp + 2 * kb) | ((uint32_t)__ldg(sp + 2 * kb + 1) << 16);
                }
                // the warp moves as one (its TMEM stores need all lanes): lane 0 waits
                bool ok = lane == 0 ? tc::mbar_wait(&S.cfull[c.s], c.par, kWaitNs) : true;
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    aborted = true;
                    break;
                }
                // codes of this step into registers, then the code slot is free
                const char *cs = dyn + C::OFF_C + c.s * C::C_BYTES;
                uint4 cw = make_uint4(0u, 0u, 0u, 0u), cw1 = make_uint4(0u, 0u, 0u, 0u);
                uint2 hw = make_uint2(0u, 0u);
                uint4 hw4 = make_uint4(0u, 0u, 0u, 0u);  // FP8, 3 bits: one high-bit word per block
                if (valid) {
                    cw = *reinterpret_cast<const uint4 *>(cs + C_LO + r * C::CODE_STEP);
                    if constexpr (FP8) {
                        cw1 = *reinterpret_cast<const uint4 *>(cs + C_LO + r * C::CODE_STEP + 16);
                        if (a.scale_tma) sc4 = *reinterpret_cast<const uint2 *>(cs + C::C_SC + r * 16 + (kb & 1) * 8);
                    } else {
                        if (a.scale_tma) sc = lds32(cs + C::C_SC + r * 16 + (kb & 3) * 4);
                    }
                    if constexpr (BITS == 3) {
                        if constexpr (FP8) hw4 = *reinterpret_cast<const uint4 *>(cs + C::C_HI + r * 16);
                        else hw = *reinterpret_cast<const uint2 *>(cs + C::C_HI + r * 16 + (kb & 1) * 8);
                    }
                }
                if (valid) {
                    if constexpr (FP8) {
                        // the e4m3 scaling takes any finite scale
                        const float2 s01 = __half22float2(*reinterpret_cast<const __half2 *>(&sc4.x));
                        const float2 s23 = __half22float2(*reinterpret_cast<const __half2 *>(&sc4.y));
                        scale_out_of_range |= !isfinite(s01.x) || !isfinite(s01.y) || !isfinite(s23.x) ||
                                              !isfinite(s23.y);
                    } else {
                        // (c - mid) s leaves fp16's range when |s| max|c - mid| rounds past 65504
                        const float2 sf = __half22float2(*reinterpret_cast<const __half2 *>(&sc));
                        constexpr float kMaxCode = BITS == 2 ? 1.5f : 3.5f;
                        scale_out_of_range |=
                            !(fabsf(sf.x) * kMaxCode < kF16Limit) || !(fabsf(sf.y) * kMaxCode < kF16Limit);
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&S.cempty[c.s]);
                ok = lane == 0 && sa.reuse ? tc::mbar_wait_sleep(&S.aempty[sa.s], sa.par ^ 1, kWaitNs) : true;  // usually ahead
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    aborted = true;
                    break;
                }
                tc::tc_fence_after();
                if constexpr (FP8) {
                    // 128 weights: four 32-weight blocks, each a byte table of its four e4m3 values
                    // and two code words decoded by byte selects into eight TMEM columns
                    const uint32_t words[8] = {cw.x, cw.y, cw.z, cw.w, cw1.x, cw1.y, cw1.z, cw1.w};
                    const uint32_t hws[4] = {hw4.x, hw4.y, hw4.z, hw4.w};
#pragma unroll
                    for (int b = 0; b < 4; b++) {
                        uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                        if (valid) {
                            const uint32_t sw = b < 2 ? sc4.x : sc4.y;
                            const uint16_t sh = (uint16_t)((b & 1) ? sw >> 16 : sw & 0xffffu);
                            const float S = __half2float(__ushort_as_half(sh)) * p2kw;
                            if constexpr (BITS == 2) {
                                const uint32_t lut = lut_2bit(S);
                                lut_word(words[2 * b], lut, v);
                                lut_word(words[2 * b + 1], lut, v + 4);
                            } else {
                                uint32_t lo, hi;
                                lut_3bit(S, lo, hi);
                                lut_word3(words[2 * b], hws[b], lo, hi, spread8, v);
                                lut_word3(words[2 * b + 1], hws[b] >> 8, lo, hi, spread8, v + 4);
                            }
                        }
                        tc::tmem_st_32x32b_x8(tq + (uint32_t)(sa.s * 32 + b * 8), v);
                    }
                } else {
                    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int gq = 0; gq < 4; gq++) {  // 16-weight group gq of block gq / 2
                        uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                        const uint32_t hb = gq < 2 ? hw.x : hw.y;
                        if (valid)
                            dq_group<BITS>(words[gq], (gq & 1) ? hb >> 8 : hb, gq < 2 ? sc & 0xffffu : sc >> 16, v);
                        tc::tmem_st_32x32b_x8(tq + (uint32_t)(sa.s * 32 + gq * 8), v);
                    }
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&S.afull[sa.s]);
            }
            base += nk;
        }
        if (aborted) {
            if (lane == 0) set_status(a.status, MOE_ERR_TIMEOUT);
            S.abort = 1;
        }
        if (__any_sync(0xffffffffu, scale_out_of_range) && lane == 0) set_status(a.status, MOE_ERR_RANGE);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// x_g[p][16g + perm16(m)] = fp16(x[t][16g + m]) for every pair p = inv[t*k + j]
// of token t (pairs with inv < 0 are not in this call); an x without a
// finite fp16 sets MOE_ERR_RANGE.  One warp per token: its row is read once
// (in token order, so each x row comes from memory once) and written to each
// of its pair rows; lanes take the row's 16-element groups, 16-byte accesses.
__global__ void gather_x_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ inv, int T, int k,
                                int H, uint16_t *__restrict__ xg, int32_t *__restrict__ status)
{
    bool out_of_range = false;
    const int groups = H / 16, lane = lane_id();
    const int warps = (int)(gridDim.x * blockDim.x >> 5);
    for (int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); t < T; t += warps) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t * H);
        for (int g0 = 0; g0 < groups; g0 += 4 * 32) {
            uint4 a[4][2];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int g = g0 + u * 32 + lane;
                if (g < groups) {
                    a[u][0] = __ldg(src + 2 * g);
                    a[u][1] = __ldg(src + 2 * g + 1);
                }
            }
            uint4 o[4][2];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int g = g0 + u * 32 + lane;
                if (g >= groups) continue;
                const uint32_t w[8] = {a[u][0].x, a[u][0].y, a[u][0].z, a[u][0].w,
                                       a[u][1].x, a[u][1].y, a[u][1].z, a[u][1].w};
                float f[16];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    f[2 * j] = __uint_as_float(w[j] << 16);
                    f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
                }
#pragma unroll
                for (int mm = 0; mm < 16; mm++) out_of_range |= !(fabsf(f[mm]) < kF16Limit);
                uint32_t h[8];
#pragma unroll
                for (int mm = 0; mm < 8; mm++) {
                    __half2 hv = __floats2half2_rn(f[mm], f[mm + 8]);
                    h[mm] = *reinterpret_cast<uint32_t *>(&hv);
                }
                o[u][0] = make_uint4(h[0], h[1], h[2], h[3]);
                o[u][1] = make_uint4(h[4], h[5], h[6], h[7]);
            }
            for (int j = 0; j < k; j++) {
                const int p = __ldg(inv + (int64_t)t * k + j);
                if (p < 0) continue;
                uint4 *dst = reinterpret_cast<uint4 *>(xg + (int64_t)p * H);
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const int g = g0 + u * 32 + lane;
                    if (g < groups) {
                        dst[2 * g] = o[u][0];
                        dst[2 * g + 1] = o[u][1];
                    }
                }
            }
        }
    }
    if (out_of_range) set_status(status, MOE_ERR_RANGE);
}

template <int BITS, bool SWIGLU, bool FP8 = false>
static moe_status launch_gemm(const Args &a, const CUtensorMap &tok, const CUtensorMap &tok_full,
                              const CUtensorMap &codes, const CUtensorMap &scales, const CUtensorMap &out, int grid,
                              cudaStream_t s, const CUtensorMap *hi = nullptr)
{
    auto fn = tc_gemm_kernel<BITS, SWIGLU, FP8>;
    const int smem = Cfg<BITS, FP8>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "tc gemm attribute: %s", cudaGetErrorString(e));
    fn<<<grid, Cfg<BITS, FP8>::THREADS, smem, s>>>(a, tok, tok_full, codes, scales, out, hi ? *hi : codes);
    return check_launch(SWIGLU ? (FP8 ? "tc_gemm_gateup_fp8" : "tc_gemm_gateup")
                               : (FP8 ? "tc_gemm_down_fp8" : "tc_gemm_down"));
}

// ---- FP8 variant: the operands' exponents and e4m3 copies -------------------

// kw[e][row] = the exponent of weight row `row` of expert e, from the largest
// magnitude a code of the row can stand for (maxc = max|c - mid|, 1.5 or 3.5,
// times its largest |s|), for the experts that have pairs (the others are
// never read).  A non-finite scale sets MOE_ERR_RANGE.
__global__ void fp8_row_exponent_kernel(const uint16_t *__restrict__ scales, const int32_t *__restrict__ offsets,
                                        int E, int rows, int blocks, float maxc, int8_t *__restrict__ kw,
                                        int32_t *__restrict__ status)
{
    bool bad = false;
    const int64_t n = (int64_t)E * rows;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int e = (int)(i / rows);
        if (offsets[e + 1] == offsets[e]) continue;
        const uint16_t *sp = scales + i * blocks;
        uint32_t mx = 0;  // largest |s| as fp16 bits (magnitudes order like the bits; inf and NaN above all)
        if (blocks % 8 == 0) {
            for (int b = 0; b < blocks; b += 8) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(sp + b));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; j++) mx = max(mx, max(w[j] & 0x7fffu, (w[j] >> 16) & 0x7fffu));
            }
        } else {
            for (int b = 0; b < blocks; b++) mx = max(mx, (uint32_t)__ldg(sp + b) & 0x7fffu);
        }
        bad |= mx >= 0x7c00u;
        kw[i] = (int8_t)(mx >= 0x7c00u ? 0 : fp8_exponent(maxc * __half2float(__ushort_as_half((uint16_t)mx))));
    }
    if (bad) set_status(status, MOE_ERR_RANGE);
}

// x8[p][16g + pos8(m)] = e4m3(x[t][16g + m] 2^ex[p]) for every pair p =
// inv[t*k + j] of token t (pairs with inv < 0 are not in this call), ex the
// exponent of the token's largest |x|.  One warp per token: the row is read
// once (rows of up to 2,048 elements are kept in registers between the
// maximum and the conversion), converted once, and written to each of its pair
// rows.  A non-finite x, or a row whose largest |x| still exceeds e4m3's range
// after the largest down-scaling (2^-64), sets MOE_ERR_RANGE.
__global__ void gather_x_fp8_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ inv, int T, int k,
                                    int H, uint8_t *__restrict__ x8, int32_t *__restrict__ pexp,
                                    int32_t *__restrict__ status)
{
    bool out_of_range = false;
    const int groups = H / 16, lane = lane_id();
    const int warps = (int)(gridDim.x * blockDim.x >> 5);
    const bool held = groups <= 4 * 32;
    for (int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); t < T; t += warps) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t * H);
        uint4 a[4][2];
        uint32_t mx = 0;  // largest |x| as bf16 bits
        if (held) {
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int g = u * 32 + lane;
                a[u][0] = a[u][1] = make_uint4(0u, 0u, 0u, 0u);
                if (g < groups) {
                    a[u][0] = __ldg(src + 2 * g);
                    a[u][1] = __ldg(src + 2 * g + 1);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const uint32_t w[8] = {a[u][0].x, a[u][0].y, a[u][0].z, a[u][0].w,
                                       a[u][1].x, a[u][1].y, a[u][1].z, a[u][1].w};
#pragma unroll
                for (int j = 0; j < 8; j++) mx = max(mx, max(w[j] & 0x7fffu, (w[j] >> 16) & 0x7fffu));
            }
        } else {
            for (int g = lane; g < groups; g += 32) {
                const uint4 a0 = __ldg(src + 2 * g), a1 = __ldg(src + 2 * g + 1);
                const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int j = 0; j < 8; j++) mx = max(mx, max(w[j] & 0x7fffu, (w[j] >> 16) & 0x7fffu));
            }
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        const float amax = __uint_as_float(mx << 16);
        const int ex = mx >= 0x7f80u ? 0 : fp8_exponent(amax);
        out_of_range |= mx >= 0x7f80u || amax * exp2i(ex) >= 464.f;
        const float sc = exp2i(ex);
        // stored bytes 0-3: elements 0, 2, 4, 6; 4-7: 8, 10, 12, 14; 8-11: 1, 3, 5, 7; 12-15: 9, 11, 13, 15
        auto conv = [&](const uint4 &a0, const uint4 &a1) {
            const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float f[16];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                f[2 * j] = __uint_as_float(w[j] << 16) * sc;
                f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u) * sc;
            }
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int m0 = (q & 1) * 8 + (q >> 1);  // element at the word's first byte
                o[q] = e4m3x2(f[m0 + 2], f[m0]) | (e4m3x2(f[m0 + 6], f[m0 + 4]) << 16);
            }
            return make_uint4(o[0], o[1], o[2], o[3]);
        };
        if (held) {
            uint4 c[4];
#pragma unroll
            for (int u = 0; u < 4; u++) c[u] = conv(a[u][0], a[u][1]);
            for (int j = 0; j < k; j++) {
                const int p = __ldg(inv + (int64_t)t * k + j);
                if (p < 0) continue;
                if (lane == 0) pexp[p] = ex;
                uint4 *dst = reinterpret_cast<uint4 *>(x8 + (int64_t)p * H);
#pragma unroll
                for (int u = 0; u < 4; u++)
                    if (u * 32 + lane < groups) dst[u * 32 + lane] = c[u];
            }
        } else {
            for (int j = 0; j < k; j++) {
                const int p = __ldg(inv + (int64_t)t * k + j);
                if (p < 0) continue;
                if (lane == 0) pexp[p] = ex;
                uint4 *dst = reinterpret_cast<uint4 *>(x8 + (int64_t)p * H);
                for (int g = lane; g < groups; g += 32) dst[g] = conv(__ldg(src + 2 * g), __ldg(src + 2 * g + 1));
            }
        }
    }
    if (out_of_range) set_status(status, MOE_ERR_RANGE);
}

// h8[p][i] = e4m3(h[p][i] 2^eh[p]), eh[p] the exponent of the pair's largest
// |h|; positions stay as the gate/up epilogue stored them.  One warp per pair
// row.  (An h past fp16's range was reported by that epilogue.)
__global__ void quantise_h_kernel(const uint16_t *__restrict__ h, const int32_t *__restrict__ offsets, int E, int I,
                                  uint8_t *__restrict__ h8, int32_t *__restrict__ pexp)
{
    const int n = offsets[E];
    const int chunks = I / 8, lane = lane_id();
    const int warps = (int)(gridDim.x * blockDim.x >> 5);
    for (int p = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); p < n; p += warps) {
        const uint4 *src = reinterpret_cast<const uint4 *>(h + (int64_t)p * I);
        // rows of up to 128 chunks of eight stay in registers between the two passes
        const bool held = chunks <= 4 * 32;
        uint4 v[4];
        uint32_t mx = 0;  // largest |h| as fp16 bits
        auto amax = [&](const uint4 &c) {
            const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int j = 0; j < 4; j++) mx = max(mx, max(w[j] & 0x7fffu, (w[j] >> 16) & 0x7fffu));
        };
        if (held) {
#pragma unroll
            for (int u = 0; u < 4; u++) {
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (u * 32 + lane < chunks) v[u] = src[u * 32 + lane];
            }
#pragma unroll
            for (int u = 0; u < 4; u++) amax(v[u]);
        } else {
            for (int c = lane; c < chunks; c += 32) amax(src[c]);
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        const int eh = mx >= 0x7c00u ? 0 : fp8_exponent(__half2float(__ushort_as_half((uint16_t)mx)));
        if (lane == 0) pexp[p] = eh;
        const float sc = exp2i(eh);
        uint2 *dst = reinterpret_cast<uint2 *>(h8 + (int64_t)p * I);
        auto put = [&](const uint4 &c, int i) {
            const uint32_t w[4] = {c.x, c.y, c.z, c.w};
            uint32_t o[2];
#pragma unroll
            for (int j = 0; j < 2; j++) {
                const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&w[2 * j]));
                const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&w[2 * j + 1]));
                o[j] = e4m3x2(a.y * sc, a.x * sc) | (e4m3x2(b.y * sc, b.x * sc) << 16);
            }
            dst[i] = make_uint2(o[0], o[1]);
        };
        if (held) {
#pragma unroll
            for (int u = 0; u < 4; u++)
                if (u * 32 + lane < chunks) put(v[u], u * 32 + lane);
        } else {
            for (int c = lane; c < chunks; c += 32) put(src[c], c);
        }
    }
}

}  // namespace ptc

struct PtcWs {
    int32_t *mt_prefix;
    int4 *table;
    uint16_t *xg, *h, *y;
    // FP8 variant
    uint8_t *x8, *h8;
    int32_t *ex, *eh;
    int8_t *kw_gu, *kw_d;
    size_t bytes;
};

// Workspace carve-up (256-byte aligned pieces): tile prefix and table, then
// the pairs' x rows (fp16, or e4m3 for FP8), h (fp16), y (fp16), and for FP8
// the e4m3 h, the per-pair exponents and the per-row exponents.
static PtcWs ptc_ws(const moe_expert_arena &A, int T, int k, void *base, bool fp8 = false)
{
    PtcWs w = {};
    size_t n = (size_t)T * k;
    char *b = static_cast<char *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = b ? b + off : nullptr;
        off += align256(bytes);
        return p;
    };
    w.mt_prefix = reinterpret_cast<int32_t *>(take((A.E + 1) * sizeof(int32_t)));
    w.table = reinterpret_cast<int4 *>(take((n / ptc::BT + A.E + 1) * sizeof(int4)));  // at most n/BT + one partial per expert
    if (fp8) w.x8 = reinterpret_cast<uint8_t *>(take(n * A.H));
    else w.xg = reinterpret_cast<uint16_t *>(take(n * A.H * 2));
    w.h = reinterpret_cast<uint16_t *>(take(n * A.I * 2));
    w.y = reinterpret_cast<uint16_t *>(take(n * A.H * 2));
    if (fp8) {
        w.h8 = reinterpret_cast<uint8_t *>(take(n * A.I));
        w.ex = reinterpret_cast<int32_t *>(take(n * sizeof(int32_t)));
        w.eh = reinterpret_cast<int32_t *>(take(n * sizeof(int32_t)));
        w.kw_gu = reinterpret_cast<int8_t *>(take((size_t)A.E * 2 * A.I));
        w.kw_d = reinterpret_cast<int8_t *>(take((size_t)A.E * A.H));
    }
    w.bytes = off;
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

// The FP8 variant takes arenas whose H and I are multiples of 128 (a step
// reduces over 128 elements).
bool prefill_fp8_supported(const moe_expert_arena &A)
{
    return (A.bits == 2 || A.bits == 3) && prefill_tc_supported(A) && A.H % 128 == 0 && A.I % 128 == 0;
}

size_t prefill_fp8_workspace_bytes(const moe_expert_arena &A, int T, int k)
{
    return ptc_ws(A, T, k, nullptr, true).bytes;
}

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
    tile_table_kernel<<<(A.E + 255) / 256, 256, 0, s>>>(offsets, d.mt_prefix, A.E, BT, d.table);
    st = check_launch("tile_table");
    if (st != MOE_OK) return st;
    const int tblocks = std::max(1, std::min((T + 7) / 8, sm_count() * 16));  // 8 tokens per CTA
    gather_x_kernel<<<tblocks, 256, 0, s>>>(x, inv, T, k, A.H, d.xg, status);
    st = check_launch("gather_x");
    if (st != MOE_OK) return st;
    int rbH = BITS == 2 ? A.H / 4 : A.H / 4 + A.H / 8;
    int rbI = BITS == 2 ? A.I / 4 : A.I / 4 + A.I / 8;
    int grid = sm_count();
    const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // gate/up: codes [E * 2I][rbH], pairs' rows xg [n][H] -> h [n][I]
    CUtensorMap mtok, mtokf, mcode, mscale, mout;
    st = make_tmap_2d(&mtok, d.xg, F16, 2, n, A.H, BK, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK) st = make_tmap_2d(&mtokf, d.xg, F16, 2, n, A.H, BK, BT, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK)
        st = make_tmap_2d(&mcode, A.gu_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (int64_t)A.E * 2 * A.I, rbH, 16, 64,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st == MOE_OK) st = make_tmap_2d(&mout, d.h, F16, 2, n, A.I, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    bool sc_gu = A.H % 256 == 0;  // scale rows (H/32 fp16) are 16-byte multiples
    mscale = mcode;
    if (st == MOE_OK && sc_gu)
        st = make_tmap_2d(&mscale, A.gu_scales, F16, 2, (int64_t)A.E * 2 * A.I, A.H / 32, 8, 64,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != MOE_OK) return st;
    Args a = {};
    a.scale_tma = sc_gu;
    a.scales = A.gu_scales;
    a.scales_expert_stride = (int64_t)2 * A.I * (A.H / 32);
    a.code_rows = (int64_t)2 * A.I;
    a.scale_row = A.H / 32;
    a.K = A.H;
    a.rows = A.I;
    a.up_rows = A.I;
    a.rtiles = (A.I + 63) / 64;
    a.hi_x = A.H / 4;
    a.table = d.table;
    a.ntt = d.mt_prefix + A.E;
    a.h_out = d.h;
    a.status = status;
    st = launch_gemm<BITS, true>(a, mtok, mtokf, mcode, mscale, mout, grid, s);
    if (st != MOE_OK) return st;
    // down: codes [E * H][rbI], h [n][I] -> y [n][H]
    st = make_tmap_2d(&mtok, d.h, F16, 2, n, A.I, BK, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK) st = make_tmap_2d(&mtokf, d.h, F16, 2, n, A.I, BK, BT, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK)
        st = make_tmap_2d(&mcode, A.d_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (int64_t)A.E * A.H, rbI, 16, 64,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st == MOE_OK)
        st = make_tmap_2d(&mout, d.y, F16, 2, n, A.H, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    bool sc_d = A.I % 256 == 0;
    mscale = mcode;
    if (st == MOE_OK && sc_d)
        st = make_tmap_2d(&mscale, A.d_scales, F16, 2, (int64_t)A.E * A.H, A.I / 32, 8, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != MOE_OK) return st;
    Args b = a;
    b.scale_tma = sc_d;
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
    st = launch_gemm<BITS, false>(b, mtok, mtokf, mcode, mscale, mout, grid, s);
    if (st != MOE_OK) return st;
    return launch_combine_f16(d.y, w, inv, T, k, A.H, out, dt, accumulate, s);
}

// The FP8 variant: the weights' row exponents, the pairs' e4m3 x rows, the
// gate/up GEMM (h in fp16), h to e4m3, the down GEMM, the combine.
template <int BITS>
static moe_status run_fp8(const moe_expert_arena &A, const uint16_t *x, int T, const float *w, int k,
                          const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out, moe_dtype dt,
                          int accumulate, const PtcWs &d, int32_t *status, cudaStream_t s)
{
    using namespace ptc;
    using C = Cfg<BITS, true>;
    const float maxc = BITS == 2 ? 1.5f : 3.5f;
    int64_t n = (int64_t)T * k;
    tile_prefix_kernel<<<1, 1024, 0, s>>>(offsets, A.E, BT, d.mt_prefix);
    moe_status st = check_launch("tile_prefix");
    if (st != MOE_OK) return st;
    tile_table_kernel<<<(A.E + 255) / 256, 256, 0, s>>>(offsets, d.mt_prefix, A.E, BT, d.table);
    st = check_launch("tile_table");
    if (st != MOE_OK) return st;
    const int sms = sm_count();
    fp8_row_exponent_kernel<<<sms * 4, 256, 0, s>>>(A.gu_scales, offsets, A.E, 2 * A.I, A.H / 32, maxc, d.kw_gu,
                                                     status);
    st = check_launch("fp8_row_exponent");
    if (st != MOE_OK) return st;
    fp8_row_exponent_kernel<<<sms * 4, 256, 0, s>>>(A.d_scales, offsets, A.E, A.H, A.I / 32, maxc, d.kw_d, status);
    st = check_launch("fp8_row_exponent");
    if (st != MOE_OK) return st;
    const int gblocks = (int)std::max<int64_t>(1, std::min<int64_t>((n + 7) / 8, (int64_t)sms * 16));  // 8 rows per CTA
    const int tblocks = std::max(1, std::min((T + 7) / 8, sms * 16));  // 8 tokens per CTA
    gather_x_fp8_kernel<<<tblocks, 256, 0, s>>>(x, inv, T, k, A.H, d.x8, d.ex, status);
    st = check_launch("gather_x_fp8");
    if (st != MOE_OK) return st;
    const int rbH = BITS == 2 ? A.H / 4 : A.H / 4 + A.H / 8, rbI = BITS == 2 ? A.I / 4 : A.I / 4 + A.I / 8;
    const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // gate/up: codes [E * 2I][rbH], pairs' e4m3 rows x8 [n][H] -> h [n][I] (fp16); for 3 bits the high
    // planes come through a map of 16-byte boxes
    CUtensorMap mtok, mtokf, mcode, mscale, mout, mhi;
    st = make_tmap_2d(&mtok, d.x8, U8, 1, n, A.H, C::BKE, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK) st = make_tmap_2d(&mtokf, d.x8, U8, 1, n, A.H, C::BKE, BT, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK)
        st = make_tmap_2d(&mcode, A.gu_codes, U8, 1, (int64_t)A.E * 2 * A.I, rbH, C::CODE_STEP, 64,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    mhi = mcode;
    if (st == MOE_OK && BITS == 3)
        st = make_tmap_2d(&mhi, A.gu_codes, U8, 1, (int64_t)A.E * 2 * A.I, rbH, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st == MOE_OK) st = make_tmap_2d(&mout, d.h, F16, 2, n, A.I, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    const bool sc_gu = A.H % 256 == 0;  // scale rows (H/32 fp16) are 16-byte multiples
    mscale = mcode;
    if (st == MOE_OK && sc_gu)
        st = make_tmap_2d(&mscale, A.gu_scales, F16, 2, (int64_t)A.E * 2 * A.I, A.H / 32, 8, 64,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != MOE_OK) return st;
    Args a = {};
    a.scale_tma = sc_gu;
    a.scales = A.gu_scales;
    a.scales_expert_stride = (int64_t)2 * A.I * (A.H / 32);
    a.code_rows = (int64_t)2 * A.I;
    a.scale_row = A.H / 32;
    a.K = A.H;
    a.rows = A.I;
    a.up_rows = A.I;
    a.rtiles = (A.I + 63) / 64;
    a.hi_x = A.H / 4;
    a.table = d.table;
    a.ntt = d.mt_prefix + A.E;
    a.h_out = d.h;
    a.status = status;
    a.kw = d.kw_gu;
    a.pexp = d.ex;
    st = launch_gemm<BITS, true, true>(a, mtok, mtokf, mcode, mscale, mout, sms, s, &mhi);
    if (st != MOE_OK) return st;
    quantise_h_kernel<<<gblocks, 256, 0, s>>>(d.h, offsets, A.E, A.I, d.h8, d.eh);
    st = check_launch("quantise_h");
    if (st != MOE_OK) return st;
    // down: codes [E * H][rbI], e4m3 h8 [n][I] -> y [n][H] (fp16)
    st = make_tmap_2d(&mtok, d.h8, U8, 1, n, A.I, C::BKE, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK) st = make_tmap_2d(&mtokf, d.h8, U8, 1, n, A.I, C::BKE, BT, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st == MOE_OK)
        st = make_tmap_2d(&mcode, A.d_codes, U8, 1, (int64_t)A.E * A.H, rbI, C::CODE_STEP, 64,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    mhi = mcode;
    if (st == MOE_OK && BITS == 3)
        st = make_tmap_2d(&mhi, A.d_codes, U8, 1, (int64_t)A.E * A.H, rbI, 16, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st == MOE_OK) st = make_tmap_2d(&mout, d.y, F16, 2, n, A.H, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    const bool sc_d = A.I % 256 == 0;
    mscale = mcode;
    if (st == MOE_OK && sc_d)
        st = make_tmap_2d(&mscale, A.d_scales, F16, 2, (int64_t)A.E * A.H, A.I / 32, 8, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != MOE_OK) return st;
    Args b = a;
    b.scale_tma = sc_d;
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
    b.kw = d.kw_d;
    b.pexp = d.eh;
    st = launch_gemm<BITS, false, true>(b, mtok, mtokf, mcode, mscale, mout, sms, s, &mhi);
    if (st != MOE_OK) return st;
    return launch_combine_f16(d.y, w, inv, T, k, A.H, out, dt, accumulate, s);
}

moe_status prefill_fp8_forward(const moe_expert_arena &A, const uint16_t *x, int T, const float *w, int k,
                               const int32_t *offsets, const int32_t *perm, const int32_t *inv, void *out,
                               moe_dtype dt, int accumulate, void *ws, int32_t *dev_status, cudaStream_t s)
{
    PtcWs d = ptc_ws(A, T, k, ws, true);
    if (A.bits == 2) return run_fp8<2>(A, x, T, w, k, offsets, perm, inv, out, dt, accumulate, d, dev_status, s);
    return run_fp8<3>(A, x, T, w, k, offsets, perm, inv, out, dt, accumulate, d, dev_status, s);
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
