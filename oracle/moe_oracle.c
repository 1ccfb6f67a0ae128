/*
 * moe_oracle.c -- the oracle for the routed-expert MoE layer with 2-/3-bit
 * block-quantised experts.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU statement of what the GPU path computes.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load it.  It shares no
 * code, header, table or constant with the CUDA library, and never calls it.
 *
 * Every floating-point quantity is carried in double (fp64).  The one place
 * where floating point decides an integer -- which experts a token keeps --
 * takes that decision on fp32 logits, exactly as the GPU does, so that both
 * sides decide in the same precision.
 *
 * What the pages fix, and where:
 *   - a router per layer keeps the top 10 of 512 experts for every token, and
 *     one always-on shared expert runs beside them:
 *       "How Strata runs a 125-billion-parameter model on a single 12 GB to
 *        24 GB graphics card", introduction;
 *       "Strata Open-Source Runtime: Running a 125B-Parameter Qwen3 Model on a
 *        12GB GPU", section "The Model Itself: The Compute-Storage Gap in
 *        Sparse MoE";
 *   - the routed experts are stored at 2 bits per weight ("Q2_0") and a token
 *     reads 0.66 GB of the 34.0 GB of them: the Step 1 byte-census table of
 *     the first page and Table 1 ("Where the weights live") of
 *     "Strata serves a 125B MoE at 94 tokens/s from a 12 GB card and 64 GB
 *      of RAM";
 *   - the finished expert vectors are summed on the GPU: first page, Step 2,
 *     "Dynamic PCIe and CPU co-execution".
 *
 * What the pages leave open, and the reading taken here (each one is also
 * listed with the design notes):
 *   - block format: 32 consecutive weights of one row along the reduction
 *     (input) dimension share one fp16 scale s; a 2-bit code c in {0..3}
 *     stands for (c - 1.5) * s, a 3-bit code c in {0..7} for (c - 3.5) * s;
 *   - expert network: SwiGLU, h_r = silu(g_r) * u_r with silu(g) = g/(1+e^-g),
 *     y = W_down h;
 *   - routing: softmax over all E logits, keep the k largest logits (ties to
 *     the lower expert id), renormalise the kept probabilities to sum to 1;
 *   - the shared expert is added with weight 1 (no gate);
 *   - bit layout of the packed codes (the pages give none), see oracle_pack;
 *   - the FP8 variant of the routed experts (oracle_expert_ffn_fp8): the pages
 *     run no 8-bit arithmetic, so its scheme -- e4m3 operands with one
 *     power-of-two scale per weight row, per token and per h vector -- is this
 *     library's own approximation of oracle_expert_ffn, stated there.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status numbers of the library's C ABI, restated here so the oracle needs
 * none of the library's headers. */
#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG 1
#define ORACLE_ERR_NONFINITE 6
#define ORACLE_ERR_BOUNDS 7

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16 bit pattern -> exact double. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)man, -24); /* subnormal: man * 2^-14 * 2^-10 */
    } else if (exp == 31) {
        v = man ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + man), exp - 25); /* (1 + man/1024) * 2^(exp-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 bit pattern -> exact double (bf16 is the top half of an fp32). */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Nearest binary16 value to v, ties to the even mantissa; magnitudes that
 * round past the largest finite value (65504) give +-inf, NaN stays NaN. */
double oracle_fp16_round(double v)
{
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    double a = fabs(v);
    int e;
    frexp(a, &e);                           /* a = m 2^e, 1/2 <= m < 1: floor(log2 a) = e - 1 */
    int E = e - 1 < -14 ? -14 : e - 1;      /* below 2^-14 the spacing stays 2^-24 */
    double q = ldexp(1.0, E - 10);          /* spacing of the values in [2^E, 2^(E+1)) */
    double r = nearbyint(a / q) * q;        /* default rounding mode: nearest, ties to even */
    if (r > 65504.0) r = INFINITY;
    return copysign(r, v);
}

/*
 * e4m3, the 8-bit float of the FP8 variant: sign, 4 exponent bits (bias 7),
 * 3 mantissa bits.  Exponent field 0 holds the subnormals m * 2^-9; exponent
 * field 15 with mantissa 7 is NaN; there are no infinities, so the largest
 * finite magnitude is 1.75 * 2^8 = 448.
 */
double oracle_e4m3_to_double(uint8_t b)
{
    int sign = b >> 7, exp = (b >> 3) & 15, man = b & 7;
    if (exp == 15 && man == 7) return NAN;
    double v = exp == 0 ? ldexp((double)man, -9) : ldexp((double)(8 + man), exp - 10);
    return sign ? -v : v;
}

/* Nearest e4m3 value to v, ties to the even mantissa; magnitudes past 448
 * give +-448 (saturation), NaN stays NaN. */
double oracle_e4m3_round(double v)
{
    if (isnan(v) || v == 0.0) return v;
    if (isinf(v)) return copysign(448.0, v);
    double a = fabs(v);
    int e;
    frexp(a, &e);
    int E = e - 1 < -6 ? -6 : e - 1;        /* below 2^-6 the spacing stays 2^-9 */
    double q = ldexp(1.0, E - 3);
    double r = nearbyint(a / q) * q;
    if (r > 448.0) r = 448.0;
    return copysign(r, v);
}

void oracle_fp16_round_array(int64_t n, const double *in, double *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_fp16_round(in[i]);
}

void oracle_e4m3_round_array(int64_t n, const double *in, double *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_round(in[i]);
}

/*
 * The power-of-two exponent that brings a set of values whose largest
 * magnitude is amax into e4m3's range: amax * 2^e lands in [128, 256), so
 * e = 7 - floor(log2 amax), clamped to [-64, 64]; e = 0 when amax is 0 (or
 * not finite, which the callers report).
 */
int oracle_fp8_exponent(double amax)
{
    if (amax == 0.0 || !isfinite(amax)) return 0;
    int e;
    frexp(amax, &e);
    int k = 7 - (e - 1);
    return k < -64 ? -64 : (k > 64 ? 64 : k);
}

/* The value a code stands for: (c - (2^bits - 1)/2) * s.  Exact in double. */
double oracle_dequant(int bits, int code, uint16_t scale_fp16)
{
    double mid = (bits == 3) ? 3.5 : 1.5;
    return ((double)code - mid) * oracle_fp16_to_double(scale_fp16);
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------------------ */
/* Packed block format                                                      */
/* ------------------------------------------------------------------------ */

/*
 * Byte length of one packed row of `cols` codes.
 * 2-bit: cols/4 bytes.  3-bit: a 2-bit plane of the low bits (cols/4 bytes)
 * followed by a 1-bit plane of the high bits (cols/8 bytes).
 */
int64_t oracle_packed_row_bytes(int bits, int64_t cols)
{
    if (bits == 2) return cols / 4;
    if (bits == 3) return cols / 4 + cols / 8;
    return -1;
}

/* Position, inside the 32-bit high-bit word of a 3-bit block, of the high
 * bit of weight i (0..31) of that block: weights 0-7 -> bits 0-7, 8-15 ->
 * bits 16-23, 16-23 -> bits 8-15, 24-31 -> bits 24-31. */
static int hi_bit_pos(int i) { return (i & 7) | ((i & 8) << 1) | ((i & 16) >> 1); }

/*
 * Pack a [rows][cols] matrix of logical codes (one code per byte).
 * Row r of the result starts at byte r * oracle_packed_row_bytes(bits, cols).
 * Low plane: weight i of the row sits in byte i/4 at bits 2*(i%4)..2*(i%4)+1
 * (its two low bits for 3-bit codes).  High plane (3-bit only): the high bit
 * of weight 32*b + i is bit hi_bit_pos(i) of the little-endian 32-bit word at
 * byte cols/4 + 4*b of the row.
 * Returns ORACLE_ERR_INVALID_ARG for a code that does not fit in `bits`.
 */
int oracle_pack(int bits, int64_t rows, int64_t cols, const uint8_t *codes, uint8_t *packed)
{
    if ((bits != 2 && bits != 3) || cols % 32 != 0 || rows < 0) return ORACLE_ERR_INVALID_ARG;
    int64_t rb = oracle_packed_row_bytes(bits, cols);
    int maxc = (1 << bits) - 1;
    memset(packed, 0, (size_t)(rows * rb));
    for (int64_t r = 0; r < rows; r++) {
        uint8_t *prow = packed + r * rb;
        for (int64_t i = 0; i < cols; i++) {
            int c = codes[r * cols + i];
            if (c > maxc) return ORACLE_ERR_INVALID_ARG;
            prow[i / 4] |= (uint8_t)((c & 3) << (2 * (i % 4)));
            if (bits == 3 && (c >> 2)) {
                int64_t b = i / 32;
                int pos = hi_bit_pos((int)(i % 32));
                prow[cols / 4 + 4 * b + pos / 8] |= (uint8_t)(1u << (pos % 8));
            }
        }
    }
    return ORACLE_OK;
}

/* Inverse of oracle_pack. */
int oracle_unpack(int bits, int64_t rows, int64_t cols, const uint8_t *packed, uint8_t *codes)
{
    if ((bits != 2 && bits != 3) || cols % 32 != 0 || rows < 0) return ORACLE_ERR_INVALID_ARG;
    int64_t rb = oracle_packed_row_bytes(bits, cols);
    for (int64_t r = 0; r < rows; r++) {
        const uint8_t *prow = packed + r * rb;
        for (int64_t i = 0; i < cols; i++) {
            int c = (prow[i / 4] >> (2 * (i % 4))) & 3;
            if (bits == 3) {
                int64_t b = i / 32;
                int pos = hi_bit_pos((int)(i % 32));
                c |= ((prow[cols / 4 + 4 * b + pos / 8] >> (pos % 8)) & 1) << 2;
            }
            codes[r * cols + i] = (uint8_t)c;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Router                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * logits[t][e] = bias[e] + sum_i W[e][i] * x[t][i], summed in double in
 * index order.  x is bf16 [T][H], W fp32 [E][H] row-major, bias fp32 [E] or
 * NULL.
 */
void oracle_router_logits(int T, int H, int E, const uint16_t *x_bf16, const float *w,
                          const float *bias, double *logits)
{
    for (int t = 0; t < T; t++)
        for (int e = 0; e < E; e++) {
            double acc = bias ? (double)bias[e] : 0.0;
            for (int i = 0; i < H; i++)
                acc += (double)w[(int64_t)e * H + i] * oracle_bf16_to_double(x_bf16[(int64_t)t * H + i]);
            logits[(int64_t)t * E + e] = acc;
        }
}

/* a ranks before b: larger logit first, equal logits (+0 == -0) by lower id. */
static int ranks_before(float la, int a, float lb, int b)
{
    if (la > lb) return 1;
    if (la < lb) return 0;
    return a < b;
}

/*
 * Top-k selection on fp32 logits and the routing weights.
 *   ids[t][j]: the j-th expert in the order (logit descending, id ascending);
 *   w[t][j] = p(ids[t][j]) / sum_j' p(ids[t][j']), p = softmax over all E.
 * The selection is k passes of "best remaining expert".  A NaN logit makes
 * the call return ORACLE_ERR_NONFINITE.  When the largest logit is infinite
 * the softmax is taken in its limit: p is uniform over the experts that hold
 * that value and zero elsewhere.
 */
int oracle_topk(int T, int E, int k, const float *logits, int32_t *ids, double *w)
{
    if (T < 0 || E < 1 || k < 1 || k > E) return ORACLE_ERR_INVALID_ARG;
    char *taken = (char *)malloc((size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    int status = ORACLE_OK;
    for (int t = 0; t < T && status == ORACLE_OK; t++) {
        const float *l = logits + (int64_t)t * E;
        for (int e = 0; e < E; e++)
            if (isnan(l[e])) status = ORACLE_ERR_NONFINITE;
        if (status != ORACLE_OK) break;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
        }
        /* softmax over all E experts, in double */
        double m = -INFINITY;
        for (int e = 0; e < E; e++)
            if ((double)l[e] > m) m = (double)l[e];
        double z = 0.0;
        for (int e = 0; e < E; e++) {
            if (isinf(m)) p[e] = ((double)l[e] == m) ? 1.0 : 0.0;
            else p[e] = exp((double)l[e] - m);
            z += p[e];
        }
        double zs = 0.0;
        for (int j = 0; j < k; j++) zs += p[ids[(int64_t)t * k + j]] / z;
        for (int j = 0; j < k; j++) w[(int64_t)t * k + j] = (p[ids[(int64_t)t * k + j]] / z) / zs;
    }
    free(taken);
    free(p);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Token -> expert permutation                                              */
/* ------------------------------------------------------------------------ */

/*
 * Stable counting sort of the T*k (token, slot) pairs by expert id.
 *   offsets[e] = number of pairs with id < e (offsets[E] = T*k);
 *   perm[p]    = flat index t*k + j of the p-th pair in (expert, flat) order;
 *   inv_perm[perm[p]] = p.
 * An id outside [0, E) returns ORACLE_ERR_BOUNDS.
 */
int oracle_permute(int T, int k, int E, const int32_t *ids, int32_t *offsets, int32_t *perm,
                   int32_t *inv_perm)
{
    int64_t n = (int64_t)T * k;
    for (int64_t f = 0; f < n; f++)
        if (ids[f] < 0 || ids[f] >= E) return ORACLE_ERR_BOUNDS;
    for (int e = 0; e <= E; e++) offsets[e] = 0;
    for (int64_t f = 0; f < n; f++) offsets[ids[f] + 1]++;
    for (int e = 0; e < E; e++) offsets[e + 1] += offsets[e];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; e++) fill[e] = offsets[e];
    for (int64_t f = 0; f < n; f++) {
        int32_t pos = fill[ids[f]]++;
        perm[pos] = (int32_t)f;
        inv_perm[f] = pos;
    }
    free(fill);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Experts                                                                  */
/* ------------------------------------------------------------------------ */

/* y[o] = sum_i dq(W[o][i]) * x[i] for a [rows][cols] matrix of logical codes
 * with scales [rows][cols/32]. */
static void dq_matvec(int bits, int rows, int cols, const uint8_t *codes, const uint16_t *scales,
                      const double *x, double *y)
{
    for (int o = 0; o < rows; o++) {
        double acc = 0.0;
        for (int i = 0; i < cols; i++)
            acc += oracle_dequant(bits, codes[(int64_t)o * cols + i],
                                  scales[(int64_t)o * (cols / 32) + i / 32]) * x[i];
        y[o] = acc;
    }
}

/*
 * One routed expert on one token.
 *   gate, up:  codes [I][H], scales [I][H/32];
 *   down:      codes [H][I], scales [H][I/32];
 *   g = dq(W_gate) x,  u = dq(W_up) x,  h = silu(g) * u,  y = dq(W_down) h.
 */
void oracle_expert_ffn(int bits, int H, int I, const uint8_t *gate_codes, const uint16_t *gate_scales,
                       const uint8_t *up_codes, const uint16_t *up_scales, const uint8_t *down_codes,
                       const uint16_t *down_scales, const double *x, double *y)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    dq_matvec(bits, I, H, gate_codes, gate_scales, x, g);
    dq_matvec(bits, I, H, up_codes, up_scales, x, u);
    for (int r = 0; r < I; r++) g[r] = silu(g[r]) * u[r];
    dq_matvec(bits, H, I, down_codes, down_scales, g, y);
    free(g);
    free(u);
}

/*
 * The FP8 variant of one routed expert on one token.  Every operand of the
 * three products is an e4m3 value after a power-of-two scaling; the products
 * are summed exactly (in double here) and the scaling undone afterwards:
 *   x:   one exponent ex for the token, x8_i = e4m3(x_i 2^ex);
 *   W:   one exponent kw_r per weight row, from the largest magnitude a code
 *        of the row can stand for (max|c - mid| times the row's largest |s|):
 *        W8_ri = e4m3(dq(W_ri) 2^kw_r);
 *   g_r = 2^-(kw_r + ex) sum_i Wg8_ri x8_i,  u_r likewise;
 *   h_r = fp16(silu(g_r) u_r)  (h is held in fp16 between the two products);
 *   eh from max_r |h_r|,  h8_r = e4m3(h_r 2^eh);
 *   y_o = 2^-(kw_o + eh) sum_r Wd8_or h8_r.
 * The exponents follow oracle_fp8_exponent.  Returns ORACLE_ERR_NONFINITE when
 * x, a scale or an h is not finite (h past fp16's range); y is then not set.
 */
static void fp8_weight_exponents(int bits, int rows, int cols, const uint16_t *scales, int *kw)
{
    double maxc = (bits == 3) ? 3.5 : 1.5;
    for (int o = 0; o < rows; o++) {
        double m = 0.0;
        for (int b = 0; b < cols / 32; b++) {
            double s = fabs(oracle_fp16_to_double(scales[(int64_t)o * (cols / 32) + b]));
            if (s > m) m = s;
        }
        kw[o] = oracle_fp8_exponent(maxc * m);
    }
}

/* y[o] = 2^-(kw_o + ex) sum_i e4m3(dq(W[o][i]) 2^kw_o) x8[i] for x8 already scaled by 2^ex. */
static void fp8_matvec(int bits, int rows, int cols, const uint8_t *codes, const uint16_t *scales,
                       const double *x8, int ex, double *y)
{
    int *kw = (int *)malloc(sizeof(int) * (size_t)rows);
    fp8_weight_exponents(bits, rows, cols, scales, kw);
    for (int o = 0; o < rows; o++) {
        double acc = 0.0;
        for (int i = 0; i < cols; i++) {
            double wq = oracle_e4m3_round(ldexp(oracle_dequant(bits, codes[(int64_t)o * cols + i],
                                                               scales[(int64_t)o * (cols / 32) + i / 32]),
                                                kw[o]));
            acc += wq * x8[i];
        }
        y[o] = ldexp(acc, -(kw[o] + ex));
    }
    free(kw);
}

/* Rounds a vector to e4m3 after its power-of-two scaling; returns the exponent. */
static int fp8_vector(int n, const double *v, double *v8)
{
    double amax = 0.0;
    for (int i = 0; i < n; i++)
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
    int e = oracle_fp8_exponent(amax);
    for (int i = 0; i < n; i++) v8[i] = oracle_e4m3_round(ldexp(v[i], e));
    return e;
}

int oracle_expert_ffn_fp8(int bits, int H, int I, const uint8_t *gate_codes, const uint16_t *gate_scales,
                          const uint8_t *up_codes, const uint16_t *up_scales, const uint8_t *down_codes,
                          const uint16_t *down_scales, const double *x, double *y)
{
    for (int i = 0; i < H; i++)
        if (!isfinite(x[i])) return ORACLE_ERR_NONFINITE;
    for (int64_t i = 0; i < (int64_t)I * (H / 32); i++)
        if (!isfinite(oracle_fp16_to_double(gate_scales[i])) || !isfinite(oracle_fp16_to_double(up_scales[i])))
            return ORACLE_ERR_NONFINITE;
    for (int64_t i = 0; i < (int64_t)H * (I / 32); i++)
        if (!isfinite(oracle_fp16_to_double(down_scales[i]))) return ORACLE_ERR_NONFINITE;
    double *x8 = (double *)malloc(sizeof(double) * (size_t)H);
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    int status = ORACLE_OK;
    int ex = fp8_vector(H, x, x8);
    fp8_matvec(bits, I, H, gate_codes, gate_scales, x8, ex, g);
    fp8_matvec(bits, I, H, up_codes, up_scales, x8, ex, u);
    for (int r = 0; r < I; r++) {
        g[r] = oracle_fp16_round(silu(g[r]) * u[r]);
        if (!isfinite(g[r])) status = ORACLE_ERR_NONFINITE;
    }
    if (status == ORACLE_OK) {
        int eh = fp8_vector(I, g, u);   /* u now holds h8 */
        fp8_matvec(bits, H, I, down_codes, down_scales, u, eh, y);
    }
    free(x8);
    free(g);
    free(u);
    return status;
}

/*
 * The always-on shared expert on one token, bf16 weights:
 *   wg, wu [I][H], wd [H][I];  y = wd (silu(wg x) * (wu x)).
 */
void oracle_shared_expert(int H, int I, const uint16_t *wg, const uint16_t *wu, const uint16_t *wd,
                          const double *x, double *y)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    for (int r = 0; r < I; r++) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < H; i++) {
            g += oracle_bf16_to_double(wg[(int64_t)r * H + i]) * x[i];
            u += oracle_bf16_to_double(wu[(int64_t)r * H + i]) * x[i];
        }
        h[r] = silu(g) * u;
    }
    for (int o = 0; o < H; o++) {
        double acc = 0.0;
        for (int r = 0; r < I; r++) acc += oracle_bf16_to_double(wd[(int64_t)o * I + r]) * h[r];
        y[o] = acc;
    }
    free(h);
}

/*
 * One MoE layer for T tokens, given the routing (ids, w) of every token.
 *   x:        bf16 [T][H]
 *   ids, w:   [T][k]; ids index the arena below
 *   arena:    gate codes [E][I][H], up codes [E][I][H], down codes [E][H][I]
 *             (one logical code per byte) with scales [E][I][H/32],
 *             [E][I][H/32], [E][H][I/32]
 *   shared:   bf16 wg [Is][H], wu [Is][H], wd [H][Is], or all NULL
 *   out[t][o] = shared(x_t)[o] + sum_j w[t][j] * y_{ids[t][j]}(x_t)[o],
 *   the routed sum taken in slot order j = 0..k-1.
 * An id outside [0, E) returns ORACLE_ERR_BOUNDS.
 */
static int moe_layer(int fp8, int bits, int T, int H, int I, int E, int k, const uint16_t *x_bf16,
                     const int32_t *ids, const double *w, const uint8_t *gate_codes,
                     const uint16_t *gate_scales, const uint8_t *up_codes, const uint16_t *up_scales,
                     const uint8_t *down_codes, const uint16_t *down_scales, int Is,
                     const uint16_t *swg, const uint16_t *swu, const uint16_t *swd, double *out)
{
    int status = ORACLE_OK;
    for (int64_t f = 0; f < (int64_t)T * k; f++)
        if (ids[f] < 0 || ids[f] >= E) return ORACLE_ERR_BOUNDS;
    double *x = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    int64_t gu_codes = (int64_t)I * H, gu_scales = (int64_t)I * (H / 32);
    int64_t d_codes = (int64_t)H * I, d_scales = (int64_t)H * (I / 32);
    for (int t = 0; t < T; t++) {
        for (int i = 0; i < H; i++) x[i] = oracle_bf16_to_double(x_bf16[(int64_t)t * H + i]);
        double *o = out + (int64_t)t * H;
        if (swg) oracle_shared_expert(H, Is, swg, swu, swd, x, o);
        else
            for (int i = 0; i < H; i++) o[i] = 0.0;
        double *routed = (double *)calloc((size_t)H, sizeof(double));
        for (int j = 0; j < k; j++) {
            int e = ids[(int64_t)t * k + j];
            if (fp8) {
                int st = oracle_expert_ffn_fp8(bits, H, I, gate_codes + e * gu_codes, gate_scales + e * gu_scales,
                                               up_codes + e * gu_codes, up_scales + e * gu_scales,
                                               down_codes + e * d_codes, down_scales + e * d_scales, x, y);
                if (st != ORACLE_OK) {
                    status = st;
                    continue;
                }
            } else {
                oracle_expert_ffn(bits, H, I, gate_codes + e * gu_codes, gate_scales + e * gu_scales,
                                  up_codes + e * gu_codes, up_scales + e * gu_scales,
                                  down_codes + e * d_codes, down_scales + e * d_scales, x, y);
            }
            for (int i = 0; i < H; i++) routed[i] += w[(int64_t)t * k + j] * y[i];
        }
        for (int i = 0; i < H; i++) o[i] += routed[i];
        free(routed);
    }
    free(x);
    free(y);
    return status;
}

int oracle_moe_layer(int bits, int T, int H, int I, int E, int k, const uint16_t *x_bf16,
                     const int32_t *ids, const double *w, const uint8_t *gate_codes,
                     const uint16_t *gate_scales, const uint8_t *up_codes, const uint16_t *up_scales,
                     const uint8_t *down_codes, const uint16_t *down_scales, int Is,
                     const uint16_t *swg, const uint16_t *swu, const uint16_t *swd, double *out)
{
    return moe_layer(0, bits, T, H, I, E, k, x_bf16, ids, w, gate_codes, gate_scales, up_codes, up_scales,
                     down_codes, down_scales, Is, swg, swu, swd, out);
}

/* The same layer with the routed experts in the FP8 variant (oracle_expert_ffn_fp8);
 * ORACLE_ERR_NONFINITE when one of them reports it. */
int oracle_moe_layer_fp8(int bits, int T, int H, int I, int E, int k, const uint16_t *x_bf16,
                         const int32_t *ids, const double *w, const uint8_t *gate_codes,
                         const uint16_t *gate_scales, const uint8_t *up_codes, const uint16_t *up_scales,
                         const uint8_t *down_codes, const uint16_t *down_scales, int Is,
                         const uint16_t *swg, const uint16_t *swu, const uint16_t *swd, double *out)
{
    return moe_layer(1, bits, T, H, I, E, k, x_bf16, ids, w, gate_codes, gate_scales, up_codes, up_scales,
                     down_codes, down_scales, Is, swg, swu, swd, out);
}

/* ------------------------------------------------------------------------ */
/* Residual stream                                                          */
/* ------------------------------------------------------------------------ */

/*
 * The input of each stacked layer: x / sqrt(mean(x^2) + eps) per token (a
 * root-mean-square normalisation without a learned gain), in double.
 *   x [T][H] fp32 residual stream;  y [T][H] double.
 * The pages' model feeds every MoE layer from a residual stream ("How Strata
 * runs a 125-billion-parameter model ...", Step 1 table: gated-residual
 * hyper-connections); the normalisation in front of the layer is the reading
 * taken for a stack of synthetic layers, whose plain residual sum diverges.
 */
void oracle_rms_norm(int T, int H, const float *x, double eps, double *y)
{
    for (int t = 0; t < T; t++) {
        double ss = 0.0;
        for (int i = 0; i < H; i++) ss += (double)x[(int64_t)t * H + i] * (double)x[(int64_t)t * H + i];
        double r = sqrt(ss / (double)H + eps);
        for (int i = 0; i < H; i++) y[(int64_t)t * H + i] = (double)x[(int64_t)t * H + i] / r;
    }
}
