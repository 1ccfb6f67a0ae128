// dequant.cuh -- exact dequantisation of packed 2-/3-bit codes to centred
// fp16 values (c - mid), shared by the decode and prefill kernels.
//
// The routed experts are 2-bit ("Q2_0") or 3-bit block-quantised ("How Strata
// runs a 125-billion-parameter model on a single 12 GB to 24 GB graphics
// card", introduction and the Step 1 byte-census table); the pages give no
// bit layout, so the mapping of a code c to (c - 1.5) s (2 bits) or
// (c - 3.5) s (3 bits), one fp16 scale s per 32-weight block, and the bit
// positions inside a word are this library's own (those of moe_pack_experts).
#pragma once
#include <cstdint>

namespace moe {

__device__ __forceinline__ uint32_t hfma2_f16(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// (a & b) | c in one instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Codes of a 16-weight word: weight j at bits 2j..2j+1 (low plane).  Pair M
// (weights M and M+8, bits 2M and 2M+16) becomes the fp16x2 of the centred
// codes (c_M - mid, c_{M+8} - mid) exactly: the codes are OR-ed into the
// mantissa of 1024.0 at bit 2M' with M' in 1..4 (2 bits) or 1..3 (3 bits),
// giving 1024 + c*4^M' (< 2048, so exact), and one fma with 4^-M' and
// -(1024*4^-M' + mid) (both fp16 values) yields c - mid, also exact.  Which
// shift of the word puts pair M at M' is in dq_src; for 3 bits the high bit
// of each weight (word `hw`, bits M+8w and M+8w+16 for word w of the block)
// joins at bit 2M'+2.
template <int BITS>
struct DqWord {
    uint32_t w0, wl2, wr;   // the word, << 2, >> 8 (2 bits) or >> 6 (3 bits)
    uint32_t wr12;          // >> 12 (3 bits)
};

template <int BITS>
__device__ __forceinline__ DqWord<BITS> dq_word(uint32_t w)
{
    DqWord<BITS> d;
    d.w0 = w;
    d.wl2 = w << 2;
    d.wr = w >> (BITS == 2 ? 8 : 6);
    d.wr12 = BITS == 2 ? 0u : w >> 12;
    return d;
}

template <int M, int BITS, int W>
__device__ __forceinline__ uint32_t dq_pair(const DqWord<BITS> &d, uint32_t hw)
{
    // pair M sits at bit 2*MP of: the word (M 1..4 | 1..3), the word << 2 (M 0), the word >> 8 (M 5..7, 2 bits),
    // >> 6 (M 4..6, 3 bits), >> 12 (M 7, 3 bits)
    constexpr int MP = M == 0 ? 1 : (BITS == 2 ? (M <= 4 ? M : M - 4) : (M <= 3 ? M : (M <= 6 ? M - 3 : 1)));
    const uint32_t src = M == 0 ? d.wl2
                                : (BITS == 2 ? (M <= 4 ? d.w0 : d.wr) : (M <= 3 ? d.w0 : (M <= 6 ? d.wr : d.wr12)));
    uint32_t v = and_or(src, 0x00030003u << (2 * MP), 0x64006400u);
    if constexpr (BITS == 3) {
        constexpr int SH = 8 * W + M - 2 * MP - 2;  // bring bit (8W+M) to bit 2MP+2
        const uint32_t hb = SH >= 0 ? (hw >> (SH >= 0 ? SH : 0)) : (hw << (SH < 0 ? -SH : 0));
        v = and_or(hb, 0x00010001u << (2 * MP + 2), v);
    }
    // 4^-MP and -(1024 * 4^-MP + mid) as fp16 pairs, MP = 1..4
    constexpr uint32_t kMul[5] = {0u, 0x34003400u, 0x2C002C00u, 0x24002400u, 0x1C001C00u};
    constexpr uint32_t kAdd2[5] = {0u, 0xDC06DC06u, 0xD418D418u, 0xCC60CC60u, 0xC580C580u};  // mid 1.5
    constexpr uint32_t kAdd3[4] = {0u, 0xDC0EDC0Eu, 0xD438D438u, 0xCCE0CCE0u};               // mid 3.5
    return hfma2_f16(v, kMul[MP], BITS == 2 ? kAdd2[MP] : kAdd3[MP < 4 ? MP : 1]);
}

}  // namespace moe
