/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) routed-expert MoE layer with
 * 2-bit / 3-bit block-quantised experts.
 *
 * The layer this library computes, per token x (bf16, hidden size H):
 *   logits = W_router x + b                      (fp32, E experts)
 *   ids, w = top-k of logits, ties to the lower id; w = the kept softmax
 *            probabilities renormalised to sum to 1
 *   out    = S(x) + sum_j w_j * FFN_{ids_j}(x)
 *   FFN_e(x) = Wd_e (silu(Wg_e x) * (Wu_e x)),  silu(g) = g / (1 + e^-g)
 *   S(x)   = the always-on shared expert, the same SwiGLU with bf16 weights.
 * The routed experts are stored in 32-weight blocks along each row's input
 * dimension with one fp16 scale s per block; a 2-bit code c stands for
 * (c - 1.5) s and a 3-bit code for (c - 3.5) s.
 *
 * Where this comes from.  "How Strata runs a 125-billion-parameter model on
 * a single 12 GB to 24 GB graphics card" (introduction and the Step 1
 * byte-census table) and "Strata Open-Source Runtime: Running a 125B-Parameter
 * Qwen3 Model on a 12GB GPU" (section "The Model Itself") describe a router
 * that keeps 10 of 512 experts per layer for every token, an always-on shared
 * expert, 48 layers, and 2-bit ("Q2_0") routed experts of which one token
 * reads 0.66 GB of 34.0 GB; "Strata serves a 125B MoE at 94 tokens/s from a
 * 12 GB card and 64 GB of RAM" (Table 1, "Where the weights live") repeats the
 * census.  The first page, Step 2, sums the finished expert vectors on the
 * GPU.  The pages give no bit layout, activation function, router
 * normalisation or shared-expert precision; the statements above are the
 * readings this library takes.
 *
 * Conventions for every call:
 *  - Status.  Every call returns a moe_status.  Argument errors are found on
 *    the host before anything is launched and leave all buffers untouched.
 *    A non-OK return also sets a thread-local message, moe_last_error(),
 *    that names the argument and, for sizes, the bytes or MiB involved.
 *  - Device-detected errors (bad ids, NaN logits, codes that do not fit,
 *    values outside the range of an fp16 tensor-core operand) are
 *    written into a caller-provided int32 status word in device memory
 *    (dev_status; the first error wins, 0 means OK; it may be NULL, in which
 *    case such errors are not reported).  Read it with moe_check_status().
 *    A kernel that detects such an error skips the offending element and
 *    still writes every output it owns.
 *  - Ownership.  The caller allocates every buffer and passes raw device
 *    pointers (unless a parameter says "host").  The library never allocates
 *    or frees memory and never synchronises a stream, except
 *    moe_check_status(), which synchronises the stream it is given.  Scratch
 *    memory comes from a caller-provided workspace whose size the matching
 *    *_workspace_size() call returns; a smaller workspace returns
 *    MOE_ERR_WORKSPACE with the bytes needed in the message.  One call is the
 *    exception: moe_permute_noalloc keeps its scratch in a fixed array inside
 *    the library (its own comment states the size, limit and sharing).
 *  - Asynchrony.  Work is enqueued on `stream` and returns at once.
 *  - Shapes.  H and I are multiples of 32; 1 <= E <= 1024;
 *    1 <= k <= min(E, 16); T >= 0 (T = 0 is a no-op that returns MOE_OK).
 *  - Types.  bf16 and fp16 values are passed as uint16_t bit patterns.
 *    Row-major everywhere.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same handle type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* a bad pointer, shape, code or scale           */
    MOE_ERR_UNSUPPORTED = 2, /* a valid request this library does not implement */
    MOE_ERR_WORKSPACE = 3,   /* workspace smaller than *_workspace_size()     */
    MOE_ERR_CUDA = 4,        /* a CUDA runtime call failed                    */
    MOE_ERR_TIMEOUT = 5,     /* a device-side wait ran out of its time limit  */
    MOE_ERR_NONFINITE = 6,   /* a NaN router logit                            */
    MOE_ERR_BOUNDS = 7,      /* an expert id outside [0, E)                   */
    MOE_ERR_RANGE = 8        /* a value outside the finite range of the fp16
                                or e4m3 operands the tensor cores take (see the
                                PREFILL and PREFILL_FP8 paths of
                                moe_expert_forward, moe_decode_forward) */
} moe_status;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum moe_path {
    MOE_PATH_AUTO = 0,        /* DECODE for T <= 8, PREFILL otherwise (never FP8) */
    MOE_PATH_DECODE = 1,      /* dequant-fused GEMVs on CUDA cores, fp32 maths  */
    MOE_PATH_PREFILL = 2,     /* grouped GEMM over the experts' token lists     */
    MOE_PATH_PREFILL_FP8 = 3  /* the same GEMMs on e4m3 operands: an opt-in
                                 approximation, see moe_expert_forward       */
} moe_path;

/* Message for the last non-OK status returned on this thread ("" if none). */
const char *moe_last_error(void);

/* Short name of a status code, e.g. "MOE_ERR_BOUNDS". */
const char *moe_status_name(moe_status s);

/*
 * Synchronise `stream`, read the int32 device status word and return it as a
 * moe_status (setting moe_last_error() when it is not MOE_OK).  If `reset` is
 * non-zero the word is set back to 0 afterwards.
 */
moe_status moe_check_status(int32_t *dev_status, int reset, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Packed block format                                                      */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of one packed [rows][cols] matrix.  cols is a multiple of 32.
 *   code plane:  rows * row_bytes, row_bytes = cols/4 (2-bit) or 3*cols/8
 *                (3-bit);
 *   scale plane: rows * (cols/32) fp16 values = rows * cols/16 bytes.
 * Layout of one packed row of codes:
 *   bytes [0, cols/4):     weight i's two low code bits at bits
 *                          2*(i%4) .. 2*(i%4)+1 of byte i/4;
 *   bytes [cols/4, 3cols/8) (3-bit only): one little-endian 32-bit word per
 *                          32-weight block b, at byte cols/4 + 4b, holding
 *                          the high bit of weight 32b+i at bit
 *                          (i&7) | ((i&8)<<1) | ((i&16)>>1).
 * The scale plane is [rows][cols/32] fp16, block b of row r covering weights
 * 32b .. 32b+31 of that row.  Sizes follow the byte census of the pages (a
 * 2-bit expert with H=2048, I=768 is 1,474,560 bytes; see the Step 1 table of
 * "How Strata runs a 125-billion-parameter model ...").
 */
moe_status moe_packed_size(int bits, int64_t rows, int64_t cols, size_t *code_bytes,
                           size_t *scale_bytes);

/*
 * Pack n_mats matrices of [rows][cols] logical codes (one code per byte,
 * device, 16-byte aligned) and their fp16 scales [rows][cols/32] (device) into
 * the layout of moe_packed_size.  packed_scales may equal scales (in place:
 * no copy).  A code >= 2^bits or a non-finite scale sets *dev_status to
 * MOE_ERR_INVALID_ARG; that block is still written, with the codes' low bits
 * and the scale as given.
 */
moe_status moe_pack_experts(int bits, int64_t n_mats, int64_t rows, int64_t cols,
                            const uint8_t *codes, const uint16_t *scales, uint8_t *packed_codes,
                            uint16_t *packed_scales, int32_t *dev_status, moe_stream_t stream);

/*
 * Inverse of moe_pack_experts for the code plane: packed -> one code per byte
 * (codes [n_mats][rows][cols], device).  The pages store the routed experts
 * at 2 bits per weight and count their bytes ("How Strata runs a
 * 125-billion-parameter model ...", introduction and the Step 1 byte-census
 * table); this call recovers the logical codes from that storage.
 */
moe_status moe_unpack_experts(int bits, int64_t n_mats, int64_t rows, int64_t cols,
                              const uint8_t *packed_codes, uint8_t *codes, moe_stream_t stream);

/*
 * The routed experts of one layer, resident in device memory (structure of
 * arrays; expert e's data starts at e times the per-expert size):
 *   gu_codes  [E][2I rows][row_bytes(H)]   rows 0..I-1 gate, I..2I-1 up
 *   gu_scales [E][2I][H/32] fp16
 *   d_codes   [E][H rows][row_bytes(I)]
 *   d_scales  [E][H][I/32] fp16
 * Every pointer must be 16-byte aligned.
 */
typedef struct moe_expert_arena {
    int32_t bits; /* 2 or 3 */
    int32_t H;
    int32_t I;
    int32_t E;
    const uint8_t *gu_codes;
    const uint16_t *gu_scales;
    const uint8_t *d_codes;
    const uint16_t *d_scales;
} moe_expert_arena;

/* ------------------------------------------------------------------------ */
/* Router                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * logits[t][e] = bias[e] + sum_i W[e][i] * x[t][i] in fp32; then the top-k
 * selection and weights of moe_topk_from_logits.
 *   x_bf16      [T][H] bf16
 *   w_router    [E][H] fp32 (16-byte aligned)
 *   bias        [E] fp32, or NULL for none
 *   logits_out  [T][E] fp32, or NULL (then the workspace holds them)
 *   topk_ids    [T][k] int32,  topk_w [T][k] fp32
 * T <= 8 runs an fp32 GEMV.  Larger T with H a multiple of 64 runs on the
 * tensor cores: W is split into three bf16 pieces (W1 + W2 + W3 carries
 * W's 24 significant bits), every product with the bf16 x is exact and
 * the sums are fp32; other shapes take an fp32 FFMA GEMM.
 * Workspace: moe_router_workspace_size (0 bytes when logits_out is given
 * and T <= 8; the split weights, E * 3H * 2 bytes, for the tensor cores).
 * A wait of the tensor-core kernel that runs out (about 2 s) sets
 * *dev_status = MOE_ERR_TIMEOUT.
 * The pages: the router keeps 10 of 512 experts per token per layer
 * ("Strata Open-Source Runtime ...", section "The Model Itself").
 */
moe_status moe_router_workspace_size(int T, int H, int E, int logits_given, size_t *bytes);
moe_status moe_router_topk(const uint16_t *x_bf16, int T, int H, const float *w_router,
                           const float *bias, int E, int k, float *logits_out, int32_t *topk_ids,
                           float *topk_w, void *ws, size_t ws_bytes, int32_t *dev_status,
                           moe_stream_t stream);

/*
 * Top-k of fp32 logits [T][E]:
 *   ids[t][j]: experts in the order (logit descending, id ascending), compared
 *              as IEEE floats (-0 == +0, so the lower id wins);
 *   w[t][j]  = softmax(logits[t])[ids[t][j]] / sum over the kept ones, which
 *              equals the softmax of the k kept logits; when the largest logit
 *              is infinite the weights are uniform over the kept experts that
 *              hold it (the softmax's limit).
 * A NaN logit sets *dev_status = MOE_ERR_NONFINITE; that token's ids are set
 * to 0..k-1 and its weights to 1/k.
 * The pages: the router keeps the 10 best of 512 experts for each token and
 * layer ("Strata Open-Source Runtime ...", section "The Model Itself"), and
 * ranks 0..9 carry decreasing router weights ("How Strata runs a
 * 125-billion-parameter model ...", Step 2, "Verify-window route tail
 * skip").  This call is the selection step alone, so that a test can feed
 * both this library and a reference the same fp32 logits.
 */
moe_status moe_topk_from_logits(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                                int32_t *dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Token -> expert permutation                                              */
/* ------------------------------------------------------------------------ */

/*
 * Stable counting sort of the T*k (token, slot) pairs by expert id:
 *   offsets [E+1]: offsets[e] = pairs with id < e, offsets[E] = T*k;
 *   perm    [T*k]: perm[p] = t*k + j of the p-th pair in (expert, t*k+j) order;
 *   inv_perm[T*k]: inv_perm[perm[p]] = p.
 * Bit-exact and deterministic.  An id of MOE_ID_NOT_LOCAL (-1) marks a pair
 * that another expert shard computes (see moe_shard_ids): it is left out
 * without an error.  Any other id outside [0, E) sets *dev_status to
 * MOE_ERR_BOUNDS and is left out the same way.  A left-out pair is not
 * counted in offsets, its inv_perm entry is -1 and perm entries past
 * offsets[E] are -1; moe_expert_forward skips such pairs (they add nothing
 * to their token's output).
 * The pages group the tokens of a verify window that share an expert
 * ("Strata serves a 125B MoE ...", section "Six billion active parameters
 * per token").
 */
moe_status moe_permute_workspace_size(int T, int k, int E, size_t *bytes);

/* The id of a (token, slot) pair whose expert lives on another shard. */
#define MOE_ID_NOT_LOCAL (-1)

/*
 * Expert parallelism: the ids of the shard that holds experts
 * [e0, e0 + e_count) of a layer.  local_ids[i] = ids[i] - e0 for ids in that
 * range, MOE_ID_NOT_LOCAL otherwise (n ids, device).  A shard then runs
 * moe_permute(local_ids, ..., E = e_count) and moe_expert_forward on an arena
 * of its e_count experts with the full routing weights: its output is the sum
 * of its own experts' terms, and the sum of all shards' outputs (plus the
 * shared expert once) is the layer.  The pages run the layer on one GPU;
 * sharding the 512 experts of a layer over several GPUs is this library's
 * extension for GPUs that serve the whole model from memory.
 */
moe_status moe_shard_ids(const int32_t *ids, int64_t n, int e0, int e_count, int32_t *local_ids,
                         moe_stream_t stream);
moe_status moe_permute(const int32_t *ids, int T, int k, int E, int32_t *offsets, int32_t *perm,
                       int32_t *inv_perm, void *ws, size_t ws_bytes, int32_t *dev_status,
                       moe_stream_t stream);

/*
 * moe_permute_noalloc -- the same stable counting sort as moe_permute, for
 * callers that cannot allocate device memory.  (This entry point has no
 * counterpart in the pages: it is a convenience of this library.)  Some
 * callers cannot call cudaMalloc or hand the library a workspace: a plugin
 * whose host framework owns every device allocation and offers no scratch
 * buffer, or a serving loop that must not allocate after start-up because an
 * allocation may synchronise the device or fail under memory pressure.  This
 * call allocates nothing and takes no workspace: its scratch is a fixed array
 * of 2 x 32,768 int32 (256 KiB) inside the library, which every GPU that
 * loads the library holds until the process exits.
 *   - Limit: ceil(T*k / 2048) * E <= 32,768 (e.g. T*k <= 65,536 pairs for
 *     E = 1024, <= 131,072 for E = 512); larger requests return
 *     MOE_ERR_INVALID_ARG with the sizes in the message.
 *   - Outputs, errors and ordering are those of moe_permute.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it together with the device's current
 *     context; a call under a new context (after cudaDeviceReset, say) looks
 *     it up again.  Make the first call on a device, and the first after a
 *     reset, before any stream capture.
 *   - Every call on a device shares the one array, and each call overwrites
 *     the cells it reads (nothing needs clearing between calls); calls whose
 *     kernels overlap on the GPU (other streams, other host threads) race on
 *     it, so serialise them.
 */
moe_status moe_permute_noalloc(const int32_t *ids, int T, int k, int E, int32_t *offsets,
                               int32_t *perm, int32_t *inv_perm, int32_t *dev_status,
                               moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Routed experts                                                           */
/* ------------------------------------------------------------------------ */

/*
 * out[t] = (accumulate ? out[t] : 0) + sum_{j<k} w[t][j] * FFN_{ids[t][j]}(x[t]),
 * the slot sum taken in slot order.  ids/w/offsets/perm/inv_perm come from
 * moe_router_topk (or the caller) and moe_permute.
 *   out: [T][H], fp32 (MOE_F32) or bf16 (MOE_BF16, round-to-nearest-even of
 *        the fp32 result).
 * DECODE: fp32 dequantisation and accumulation; a token's result does not
 *   depend on which other tokens share the call (bit-identical alone or in a
 *   group).
 * PREFILL: grouped GEMM over the experts' token lists.  With H and I
 *   multiples of 64 (2-bit) or 128 (3-bit) it runs on the tensor cores with
 *   fp16 operands: x converts to fp16 (exact for 2^-14 <= |x| <= 65504,
 *   fewer bits below, none below 2^-25), the weights (c - mid) s round once to
 *   fp16, h = silu(g) u rounds to fp16 between the two projections and each
 *   pair's y = Wd_e h is kept as fp16 until the combine (fp32 accumulation
 *   throughout; relative L2 error about 4e-4 on N(0,1) inputs).  The caller
 *   keeps every one of these inside fp16's finite range: |x|, |h| and |y|
 *   below 65504 and every block scale with |s| * max|c - mid| below 65520
 *   (max|c - mid| = 1.5 for 2 bits, 3.5 for 3 bits).  RMS-normalised inputs
 *   (|x| of order 1) and weight scales of order 0.02 stay far inside.  A value
 *   outside it sets *dev_status = MOE_ERR_RANGE and the affected outputs are
 *   not finite.  Other shapes take an fp32 FFMA form with no such limit.
 * PREFILL_FP8: the PREFILL GEMMs with e4m3 operands (kind::f8f6f4 tensor-core
 *   instructions), an opt-in approximation that AUTO never picks.  The pages
 *   run no 8-bit arithmetic; this scheme is the library's own.  2- and
 *   3-bit arenas with H and I multiples of 128 only; anything else returns
 *   MOE_ERR_UNSUPPORTED.  Every operand is an e4m3 value after a power-of-two
 *   scaling 2^e with e = 7 - floor(log2 m) (clamped to [-64, 64]), m the
 *   largest magnitude it covers: one e per weight row (m = max|c - mid|
 *   times the row's largest |s|), per pair for x, and per pair for h, which
 *   is first rounded to fp16 as in PREFILL; each weight is
 *   e4m3((c - mid) s 2^e), rounded once.  Products accumulate in fp32 and the scalings are undone on
 *   the accumulators; y is kept as fp16 until the combine.  The rounding of
 *   three operands to 3 mantissa bits costs a relative L2 error of about
 *   6e-2 on one expert's output and about 3e-2 on a layer whose bf16 shared
 *   expert is added (H=2048, I=768, N(0,1) inputs), not the 1e-3 of PREFILL.
 *   MOE_ERR_RANGE: a non-finite x or block scale, an |x| above 464 * 2^64, or
 *   an h or y outside fp16's range (as in PREFILL).
 * Workspace: moe_expert_forward_workspace_size for the same arguments.
 * The pages: each token's routed experts run on the GPU and their finished
 * output vectors are summed there, weighted by the router ("How Strata runs
 * a 125-billion-parameter model ...", Step 2, "Dynamic PCIe and CPU
 * co-execution"); long prompts are read in chunks of tokens ("Strata
 * Open-Source Runtime ...", section "Prefill and Long Context"), which the
 * PREFILL path serves as one grouped GEMM per chunk.
 */
moe_status moe_expert_forward_workspace_size(const moe_expert_arena *arena, int T, int k,
                                             moe_path path, size_t *bytes);
moe_status moe_expert_forward(const moe_expert_arena *arena, const uint16_t *x_bf16, int T,
                              const int32_t *ids, const float *w, int k, const int32_t *offsets,
                              const int32_t *perm, const int32_t *inv_perm, void *out,
                              moe_dtype out_dtype, int accumulate, moe_path path, void *ws,
                              size_t ws_bytes, int32_t *dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Shared expert                                                            */
/* ------------------------------------------------------------------------ */

/*
 * out[t] = (accumulate ? out[t] : 0) + Wd (silu(Wg x[t]) * (Wu x[t])),
 * bf16 weights wg [I][H], wu [I][H], wd [H][I] (I here is the shared
 * expert's width), fp32 accumulation.  T <= 8 runs fp32 GEMVs; larger T
 * with H and I multiples of 64 runs on the tensor cores with exact bf16
 * products, h carried as two bf16 halves (h_hi + h_lo, 16 significant
 * bits) into the down projection; other shapes take an fp32 FFMA GEMM.
 * A wait of the tensor-core kernels that runs out (about 2 s) sets
 * *dev_status = MOE_ERR_TIMEOUT (dev_status may be NULL: then it is not
 * reported).  The pages: one always-on shared expert per layer
 * ("Strata Open-Source Runtime ...", section "The Model Itself").
 * Workspace: moe_shared_expert_workspace_size.
 */
moe_status moe_shared_expert_workspace_size(int H, int I, int T, size_t *bytes);
moe_status moe_shared_expert(const uint16_t *wg, const uint16_t *wu, const uint16_t *wd, int H,
                             int I, const uint16_t *x_bf16, int T, void *out, moe_dtype out_dtype,
                             int accumulate, void *ws, size_t ws_bytes, int32_t *dev_status,
                             moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Fused decode over a stack of layers                                      */
/* ------------------------------------------------------------------------ */

/* The weights of one layer for moe_decode_forward (device pointers). */
typedef struct moe_layer_weights {
    moe_expert_arena experts;      /* routed experts (same shape in every layer) */
    const float *w_router;         /* [E][H] fp32 */
    const float *bias;             /* [E] fp32, or NULL */
    const uint16_t *shared_wg;     /* [shared_I][H] bf16 (ignored if shared_I == 0) */
    const uint16_t *shared_wu;     /* [shared_I][H] bf16 */
    const uint16_t *shared_wd;     /* [H][shared_I] bf16 */
    int32_t shared_I;              /* shared expert width, 0 for none */
} moe_layer_weights;

/*
 * Decode up to 4 tokens through n_layers (<= 64) MoE layers in one
 * persistent cooperative kernel, updating the fp32 residual stream in place:
 *   for each layer l:  u = bf16(x[t] / sqrt(mean(x[t]^2) + rms_eps))
 *                      x[t] += S_l(u) + sum_j w_tj FFN_{l,ids_tj}(u)
 * (rms_eps < 0: u = bf16(x[t]), no normalisation; see moe_rms_norm_bf16)
 * with the routing of moe_router_topk (fp32 logits, ties to the lower id,
 * renormalised softmax weights), exact dequantisation (centred codes c - mid
 * in fp16 on the tensor cores, the block scale applied in fp32) and fp32
 * accumulation.
 *   layers   host array of n_layers descriptors (copied into the launch)
 *   x        [T][H] fp32, device, 16-byte aligned, in/out
 *   ids_out, w_out  [n_layers][T][k] device outputs of the routing, or both NULL
 * A token's result does not depend on the other tokens of the call.  The
 * tensor-core operands are fp16: u must stay below 65520 in magnitude (always
 * so when normalised, |u| <= sqrt(H)) and so must h = silu(g) u; a value
 * outside sets *dev_status = MOE_ERR_RANGE.  Shapes:
 * H a multiple of 256 with at most 16 output rows per SM (H <= 2432 on 152
 * SMs), I a multiple of 128 up to 4096, shared_I a multiple of 64 up to 4096,
 * E <= 1024, k <= 16; MOE_ERR_UNSUPPORTED when the buffers do not fit in
 * shared memory.  The workspace (moe_decode_workspace_size) holds counters and
 * tagged exchange words that the call zeroes on the stream before its launch.
 * Every wait in the kernel gives up after about 2 s and reports
 * MOE_ERR_TIMEOUT through dev_status.  The pages: 48 layers of a
 * router, ten of 512 experts and a shared expert, verify windows of up to
 * four tokens ("Strata serves a 125B MoE ...", section "Six billion active
 * parameters per token").
 */
moe_status moe_decode_workspace_size(int T, int H, int I, int E, int k, int shared_I, size_t *bytes);
moe_status moe_decode_forward(const moe_layer_weights *layers, int n_layers, float *x, int T, int k,
                              float rms_eps, int32_t *ids_out, float *w_out, void *ws, size_t ws_bytes,
                              int32_t *dev_status, moe_stream_t stream);

/*
 * Options of moe_decode_forward_ex (all zero: the exact layer of
 * moe_decode_forward).
 *
 * route_tail_skip (an approximation, off at 0): from this rank on (0-based
 *   slot in the token's top-k order), a (token, slot) pair is left out of the
 *   layer -- its expert's weights are neither fetched nor multiplied -- when
 *   no token of the call keeps that expert at a lower rank and the expert is
 *   not marked hot.  The other pairs keep their weights (no renormalisation),
 *   so a token's output loses the left-out terms w_j FFN_j(u).  The pages
 *   skip, in a verify window of up to four tokens, the experts every token
 *   ranks 7, 8 or 9 of its top-10 (rank threshold 7) unless the expert is in
 *   the fast memory tier, trading a small shift of the output distribution
 *   for fewer expert reads ("How Strata runs a 125-billion-parameter model
 *   ...", Step 2, "Verify-window route tail skip").  Must be in [0, k].
 *   ids_out / w_out still report the router's full selection.
 * hot_experts (device, [n_layers][(E + 31) / 32] uint32 bit masks, bit e of
 *   layer l set for a hot expert, or NULL): the copies of a marked expert's
 *   weights carry an L2 evict-last hint and every other weight copy an
 *   evict-first hint, so that the marked experts stay in the 129 MB L2 from
 *   one decode step to the next -- the on-chip counterpart of the pages'
 *   adaptive expert cache ("How Strata runs ...", Step 1, "Tier 1: GPU VRAM
 *   ... adaptive expert cache"; "Strata serves a 125B MoE ...", "Where the
 *   weights live").  The results are the same bits with or without masks.
 *   The caller chooses the set (for instance from the routing the previous
 *   steps reported through ids_out) and may change it between calls.
 */
typedef struct moe_decode_options {
    int32_t route_tail_skip;
    const uint32_t *hot_experts;
} moe_decode_options;

/*
 * moe_decode_forward with options (opts may be NULL: moe_decode_forward).
 * Every other argument, the shapes, workspace and errors are those of
 * moe_decode_forward.
 */
moe_status moe_decode_forward_ex(const moe_layer_weights *layers, int n_layers, float *x, int T, int k,
                                 float rms_eps, const moe_decode_options *opts, int32_t *ids_out, float *w_out,
                                 void *ws, size_t ws_bytes, int32_t *dev_status, moe_stream_t stream);

/*
 * Self-test of the grid barrier's time limit used by moe_decode_forward: one
 * cooperative launch (one CTA per SM) runs a single barrier whose target is
 * `extra_arrivals` above the number of CTAs.  With extra_arrivals = 0 it
 * completes; otherwise every CTA gives up after timeout_ms, writes
 * MOE_ERR_TIMEOUT to *dev_status and returns, leaving the context usable.
 * ws: 8 bytes (int at ws+4 counts the CTAs that passed the barrier).
 */
moe_status moe_selftest_barrier(unsigned extra_arrivals, int timeout_ms, void *ws, size_t ws_bytes,
                                int32_t *dev_status, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Residual stream helper                                                   */
/* ------------------------------------------------------------------------ */

/* out_bf16[i] = round-to-nearest-even bf16 of in_f32[i], n elements. */
moe_status moe_f32_to_bf16(const float *in_f32, uint16_t *out_bf16, int64_t n, moe_stream_t stream);

/*
 * The input of a stacked layer: out[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps))
 * for x [T][H] fp32 (a root-mean-square normalisation without a gain).  The
 * pages' layers read a residual stream; a stack of synthetic layers without
 * this normalisation diverges, so the stacked workloads normalise in front
 * of every layer.
 */
moe_status moe_rms_norm_bf16(const float *x, uint16_t *out, int T, int H, float eps, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
