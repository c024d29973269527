/*
 * strata.h — C ABI of the block-quantized multi-token verify path for one GB300 (sm_103a).
 *
 * What it computes. A speculative VERIFY window runs T tokens (the last accepted token plus T-1
 * drafts) through dense block-quantized projections that are read from HBM once for all T tokens,
 * and every token's output column is bit for bit what the single-token launch (T = 1) produces
 * ("exact mode", multi-column MMVQ). The window ends in a vocabulary head whose per-token argmax
 * picks the next id, ties going to the lower id. A grouped MoE-expert variant of the same block
 * arithmetic covers prompt chunks.
 *   Sources: Strata commit "wire multi-token kernels into Verifier and MtpDrafter CUDA graphs",
 *   include/strata/core/verify.hpp, header comment (exact mode; one weight read for T tokens;
 *   `xq_` = "T columns of q8_1"; the pool's output layout (n_tok*k, n_embd));
 *   Strata pull request "sm_80 (GA100) tuning", commit message on the hoisted-load MMVQ-IL kernels
 *   (exact integer forms, fixed accumulation order and xor tree);
 *   dsv41-offload worker/tp2.py, module docstring "Collectives per draft step" and EmuComm.argmax
 *   (argmax ties go to the lower id).
 *
 * Conventions for every call.
 *   - All pointers except `const strata_expert*` host-side struct fields are DEVICE pointers unless
 *     stated. The library allocates and frees nothing; the caller owns every buffer.
 *   - Every call validates its arguments on the host first and returns a status code without
 *     launching anything when they are wrong. Otherwise it enqueues kernels on `stream` and
 *     returns at once (asynchronous); STRATA_ERR_CUDA reports a launch failure.
 *   - Kernels are launched with programmatic dependent launch, and every kernel lets the next one
 *     launch before it waits for its own predecessor. Activations, outputs and workspace are
 *     touched only after the preceding kernel on the stream has completed; WEIGHTS may be read
 *     (streamed, prefetched into L2) while earlier kernels of this library on the stream are still
 *     running, back to the nearest operation on the stream that is not a kernel of this library (a
 *     copy, an event wait, another kernel), which completes before anything after it starts. So
 *     weight buffers must be fully written before that operation completes (weights are static
 *     model data; a cudaMemcpy on the stream is a full dependency and is fine).
 *   - Floating point is IEEE fp32 with round-to-nearest; no fast-math.
 *
 * Block formats (32 weights per block along a row; cols % 32 == 0; nb = cols / 32).
 *   A weight matrix W[rows][cols] is ONE buffer holding two planes, the quant plane first:
 *     STRATA_Q4: quant plane rows*nb*16 bytes; block (r, b) at byte offset (r*nb + b)*16;
 *                byte j (0..15) holds element j in its low nibble and element j+16 in its high
 *                nibble, each an unsigned code q in 0..15; the weight is w = d * (q - 8).
 *     STRATA_Q8: quant plane rows*nb*32 bytes; block (r, b) at (r*nb + b)*32; byte j is element j
 *                as a signed code q in -127..127; the weight is w = d * q.
 *   followed by the scale plane: rows*nb IEEE binary16 scales d, little-endian, block (r, b) at
 *   index r*nb + b. Total bytes = rows*nb*18 (Q4) or rows*nb*34 (Q8), the same as interleaved
 *   {half d; codes} blocks, but both planes start on 16-byte boundaries so that every block's
 *   codes are one or two aligned 16-byte loads. W must be 16-byte aligned.
 *     STRATA_Q6 (the pages' 6-bit super-block type, 210 bytes per 256 weights; cols % 256 == 0):
 *                code plane rows*nb*24 bytes, block (r, b) at (r*nb + b)*24: bytes 0..15 hold the low
 *                4 bits of element j (low nibble) and of element j+16 (high nibble); byte 16+i
 *                (i < 8) holds the high 2 bits of elements i, i+8, i+16, i+24 in bits 0-1, 2-3, 4-5,
 *                6-7; the code q = low | high << 4 is in 0..63. Then rows*nb*2 bytes of int8
 *                sub-scales (s0, s1 of block (r, b) at 2*(r*nb + b): s0 for elements 0..15, s1 for
 *                16..31), then rows*(cols/256) fp16 super-block scales d (row r, super-block k at
 *                index r*(cols/256) + k). The weight is w = d * s * (q - 32); the integer dot is
 *                exact per 16 weights and each 16 contributes its own term d * s * d_x * isum16.
 *     STRATA_Q4K (the pages' 4-bit super-block type with minimums, 148 bytes per 256 weights;
 *                cols % 256 == 0): the Q4 code plane (16 bytes a block, codes q in 0..15 with no
 *                offset), then rows*nb byte pairs (sc, m) per block (6-bit scale and minimum, 0..63),
 *                then rows*(cols/256) pairs of fp16 (d, dmin) per super-block. The weight is
 *                w = d * sc * q - dmin * m; each block contributes d*sc*d_x*isum then
 *                -dmin*m*d_x*s, with isum = sum q*x exact and s the activation block sum.
 *     STRATA_Q5K (the pages' 5-bit super-block type, 180 bytes per 256 weights; cols % 256 == 0):
 *                Q4K with codes q in 0..31. Row r of the code plane (20*nb bytes at r*nb*20) holds
 *                the row's nb nibble blocks (16 bytes each, as Q4: low 4 bits of element j in the low
 *                nibble of byte j, of element j+16 in the high nibble), then nb 32-bit little-endian
 *                words of fifth bits: bit 8k + g of block b's word is the fifth bit of element 4g+k
 *                (g < 4) or 16+4(g-4)+k (g >= 4). The (sc, m) plane and the (d, dmin) plane follow
 *                as in Q4K; w = d * sc * q - dmin * m, with the same two terms per block.
 *   The block-dot hook (strata_block_dots) returns isum as defined per format: Q4 sum (q-8)x, Q8
 *   sum qx, Q6 s0*sum16 + s1*sum16, Q4K and Q5K sum qx.
 *
 * Quantized activations (q8_1-style, one scale and one sum per 32 values), for n rows of `cols`:
 *     xq int8  [n][cols]   codes q in -127..127
 *     xd fp32  [n][cols/32] scale d
 *     xs int32 [n][cols/32] exact block sum  s = sum of the 32 codes
 *   For each 32-block of x: amax = max|x_j| ; d = amax / 127 ; id = (d != 0) ? 1/d : 0 ;
 *   q_j = roundf(x_j * id) (round half away from zero) ; s = sum q_j. Each operation is one IEEE
 *   fp32 operation, so the codes are reproducible bit for bit on any IEEE machine.
 *
 * Block arithmetic shared by the GEMV family (one token t, one output row r):
 *     isum[t][r][b] = sum_j wq_j * xq[t][32b+j]   with wq_j = q_j - 8 (Q4) or q_j (Q8), exact int32
 *     y[t][r]       = sum_b (d_w[r][b] * xd[t][b]) * isum[t][r][b]      in fp32
 *   The fp32 summation order is fixed by (rows, cols, fmt) only, never by T, so column t of a
 *   T-token launch is bitwise equal to the T = 1 launch on that column's activations.
 */
#ifndef STRATA_H
#define STRATA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (every entry point returns one of these) ---- */
#define STRATA_OK              0   /* enqueued */
#define STRATA_ERR_NULL       -1   /* a required pointer is NULL */
#define STRATA_ERR_SHAPE      -2   /* cols % 32 != 0, a size <= 0 or above a stated maximum */
#define STRATA_ERR_T          -3   /* T outside [1, STRATA_MAX_T] */
#define STRATA_ERR_FMT        -4   /* unknown or unsupported block format */
#define STRATA_ERR_CUDA       -5   /* a CUDA launch or attribute call failed */
#define STRATA_ERR_EXPERT     -6   /* (device-side) an expert id was outside [0, n_expert) */
#define STRATA_ERR_ALIGN      -7   /* a pointer is not aligned as the call requires */
#define STRATA_ERR_WORKSPACE  -8   /* workspace NULL or smaller than the *_workspace() size */

#define STRATA_MAX_T 8             /* verify windows hold 1..8 tokens */

typedef enum { STRATA_Q4 = 0, STRATA_Q8 = 1, STRATA_Q6 = 2, STRATA_Q4K = 3, STRATA_Q5K = 4 } strata_fmt;

/* Static text for a status code (never NULL). */
const char* strata_error_string(int status);

/* Bytes of one weight matrix in `fmt` (0 if the shape is invalid). Host-only helper. */
size_t strata_weight_bytes(int64_t rows, int64_t cols, int fmt);

/*
 * strata_quantize_act — fp32 activations to int8 blocks of 32 with an fp32 scale and block sum.
 *   Source: verify.hpp header comment, member `xq_` ("T columns of q8_1") of the Strata commit
 *   "wire multi-token kernels into Verifier and MtpDrafter CUDA graphs"; the scale is fp32.
 *   x  : fp32 [n_rows][cols], row-major, 16-byte aligned.
 *   xq : int8 [n_rows][cols], 16-byte aligned.   xd : fp32 [n_rows][cols/32].
 *   xs : int32 [n_rows][cols/32].
 *   n_rows >= 1 (any count: T tokens, or a prompt chunk's tokens); cols % 32 == 0, cols >= 32.
 *   x must be finite. Errors: NULL, SHAPE, ALIGN, CUDA.
 */
int strata_quantize_act(const float* x, int64_t n_rows, int64_t cols,
                        int8_t* xq, float* xd, int32_t* xs, cudaStream_t stream);

/*
 * strata_mmvq_multi — y[t][r] for T <= 8 tokens, reading W once.
 *   Source: verify.hpp header comment (multi-column MMVQ in exact mode; dense weights read once
 *   for T tokens), and the pull request "sm_80 (GA100) tuning", commit message on the hoisted
 *   MMVQ-IL loads (integer dots exact, accumulation order and xor tree fixed).
 *   W  : weight matrix [rows][cols] in `fmt` (layout above), 16-byte aligned.
 *   xq, xd, xs : quantized activations of T rows of `cols` (xq 16-byte aligned).
 *   y  : fp32 [T][rows] (token-major, rows contiguous), 4-byte aligned.
 *   1 <= T <= 8, rows >= 1, cols % 32 == 0 (cols % 256 == 0 for STRATA_Q6, STRATA_Q4K and STRATA_Q5K),
 *   32 <= cols <= 65536, T*cols <= 131072, and the staged activations (T*cols*1.25 bytes, a little
 *   more for Q6) plus one four-row slot of W must fit in shared memory (for example Q8 with cols
 *   16384 at T = 8 does not): otherwise STRATA_ERR_SHAPE.
 *   Column t is bitwise identical for every T (see the block arithmetic above).
 *   Errors: NULL, SHAPE, T, FMT, ALIGN, CUDA.
 */
int strata_mmvq_multi(const void* W, int64_t rows, int64_t cols, int fmt,
                      const int8_t* xq, const float* xd, const int32_t* xs, int T,
                      float* y, cudaStream_t stream);

/*
 * strata_mmvq_grouped — many independent T-column GEMVs of one format in ONE launch.
 *   Each descriptor is one strata_mmvq_multi problem; all share `fmt` and T. Outputs are bitwise
 *   identical to separate strata_mmvq_multi calls (each row is summed in the same order). The
 *   launch streams all matrices back to back with every SM busy and no launch gaps, for the
 *   independent projections of a verify window (the q/k/v and gate/up products of a layer; the
 *   layers of a window whose inputs are all known up front).
 *   Source: verify.hpp header comment of the Strata commit "wire multi-token kernels into Verifier
 *   and MtpDrafter CUDA graphs" (the window's cost is the dense weights read once for T tokens),
 *   and the pull request "sm_80 (GA100) tuning", commit message on STRATA_PF_BATCH (several
 *   experts per launch, one persistent grid a layer).
 *   descs : HOST array of n descriptors, read during the call (1 <= n <= 192); each field as in
 *           strata_mmvq_multi. No y may overlap another y or any input of the launch.
 *   Errors: NULL, SHAPE, T, FMT, ALIGN, CUDA (the first bad descriptor decides).
 */
typedef struct {
    const void* W;
    int64_t rows;
    int64_t cols;
    const int8_t* xq;
    const float* xd;
    const int32_t* xs;
    float* y;
} strata_gemv_desc;
int strata_mmvq_grouped(const strata_gemv_desc* descs, int n, int fmt, int T, cudaStream_t stream);

/*
 * strata_device_error — the library's device error word, read synchronously (waits for the
 *   device). Bit 0: a bounded wait inside a kernel ran out (a bulk copy, a pipeline slot or a tensor
 *   core accumulator never completed, or the kernel's abort flag was raised); that kernel then
 *   skipped the rest of its work and left its outputs incomplete. Bits 1-4 name the wait: 1 the
 *   GEMV producer waiting for a free stage, 2 a GEMV consumer waiting for a stage's bytes, 3 the
 *   GEMV producer draining its last copies, 4 strata_wait_probe. Every kernel that can set it (GEMV,
 *   head, MoE, prompt GEMM, the probe) is covered. clear != 0 resets the word. Returns STRATA_OK or
 *   STRATA_ERR_CUDA. The error-word convention follows dsv41-offload worker/tp2.py (collectives set
 *   bits in an error word instead of trapping; the host reads and clears it).
 */
int strata_device_error(int* out, int clear);

/*
 * strata_wait_probe — test hook for the bounded device waits: one CTA waits on a pipeline barrier
 *   that nothing ever completes, so the wait can only end by its time limit (limit_ns, 1..1e9) or,
 *   when abort_after_ns >= 0 (at most 1e9), by a second warp raising the CTA's abort flag after that
 *   long. Either way the kernel returns and sets bits 0 and 4 of the device error word; nothing else
 *   is touched. Asynchronous on `stream`. Errors: SHAPE (limits out of range), CUDA.
 */
int strata_wait_probe(int64_t limit_ns, int64_t abort_after_ns, cudaStream_t stream);

/*
 * strata_head_argmax — vocabulary head GEMV fused with the per-token argmax.
 *   Source: verify.hpp, Verifier::run (argmax after each token) and `h_out_/m_out_`, `copy_logits`;
 *   tie rule from dsv41-offload worker/tp2.py, EmuComm.argmax and markov_local_argmax
 *   ("ties -> lowest"): among equal maximal logits the lowest vocabulary id wins.
 *   W : [vocab][cols] in `fmt` (Q8 in the verify configuration; Q4, Q6, Q4K and Q5K are accepted too).
 *   1 <= vocab < 2^27 (134,217,728): larger vocabularies are STRATA_ERR_SHAPE. The other shape rules
 *   are strata_mmvq_multi's.
 *   ids : int32 [T] device output.  logits : fp32 [T][vocab] or NULL (then not written).
 *   workspace : device scratch of strata_head_argmax_workspace(vocab, T) bytes, 16-byte aligned;
 *   its contents need no initialisation and are dead after the call.
 *   Logits are computed exactly as strata_mmvq_multi computes y for the same W and activations.
 *   Errors: NULL, SHAPE, T, FMT, ALIGN, WORKSPACE, CUDA.
 */
size_t strata_head_argmax_workspace(int64_t vocab, int T);
int strata_head_argmax(const void* W, int64_t vocab, int64_t cols, int fmt,
                       const int8_t* xq, const float* xd, const int32_t* xs, int T,
                       int32_t* ids, float* logits, void* workspace, size_t ws_bytes,
                       cudaStream_t stream);

/*
 * strata_head_argmax_margin — strata_head_argmax plus each token's top-2 margin.
 *   Source: dsv41-offload worker/tp2.py, EmuComm.margin: the merged pick keeps the tie rule, and
 *   the margin is the top value minus the larger of the remaining values (the two shards' best
 *   runner-up), i.e. top-1 minus top-2 over the whole vocabulary. A maximum that occurs at two or
 *   more ids gives margin 0; a one-row head gives +inf. It is the per-token confidence a batch of
 *   independent sequences (one token each, T = batch) reads beside its ids.
 *   margin : fp32 [T] device output, computed in fp32 as logits[ids[t]] - second[t] from the same
 *   fp32 logits this call computes (and writes when `logits` is given).
 *   Other arguments, workspace and errors as strata_head_argmax; margin NULL is STRATA_ERR_NULL.
 */
int strata_head_argmax_margin(const void* W, int64_t vocab, int64_t cols, int fmt,
                              const int8_t* xq, const float* xd, const int32_t* xs, int T,
                              int32_t* ids, float* margin, float* logits, void* workspace,
                              size_t ws_bytes, cudaStream_t stream);

/*
 * strata_head_argmax_noalloc — strata_head_argmax for callers that cannot allocate device memory.
 *   The pages have no counterpart: this entry point exists for callers such as plugins inside a
 *   host application that owns all device memory, or servers that fix their memory at start-up,
 *   which cannot provide the workspace strata_head_argmax asks for. Same arguments, layouts and
 *   results as strata_head_argmax minus the workspace; the per-CTA argmax candidates live in a
 *   64 KiB array inside the library, held on every device that loads it until the process exits.
 *   It allocates nothing and calls no allocating routine. Its first call on a device looks up the
 *   array's device address (make that first call before any stream capture). All calls share the
 *   array: calls that overlap on the GPU race on it. The address is looked up again in a new CUDA
 *   context (after a device reset), so that first-call rule holds per context. Returns
 *   STRATA_ERR_WORKSPACE when a launch would need more than the 64 KiB; otherwise the errors of
 *   strata_head_argmax, with the same shape rules (vocab < 2^27; a shape whose staged activations do
 *   not fit is STRATA_ERR_SHAPE). Formats: Q4 and Q8 only (others are STRATA_ERR_FMT).
 */
int strata_head_argmax_noalloc(const void* W, int64_t vocab, int64_t cols, int fmt,
                               const int8_t* xq, const float* xd, const int32_t* xs, int T,
                               int32_t* ids, float* logits, cudaStream_t stream);

/*
 * strata_gemm_q4 — dense prompt-chunk GEMM: n_tok quantized activation rows against one Q4 matrix on
 * the tensor cores (tcgen05, fp16 operands holding the exact codes, one TMEM accumulator per quant
 * block). The prompt path of the Strata pull request "sm_80 (GA100) tuning" multiplies whole prompt
 * chunks with the dense quantized weights (it dequantizes them every chunk); here the integer
 * block dots stay exact and the block arithmetic is the GEMV's:
 *     y[n][r] = sum_b (d_w[r][b] * xd[n][b]) * isum[n][r][b]        (fp32, block order)
 *   W : Q4 [rows][cols] (planar layout above).  xq int8 [n_tok][cols], xd fp32 [n_tok][cols/32]: from
 *   strata_quantize_act (the block sums are not needed).  y : fp32 [n_tok][rows], fully written.
 *   rows % 128 == 0, cols % 64 == 0, rows and cols <= 65536, 1 <= n_tok <= 2^24. W, xq, y 16-byte
 *   aligned, xd 4-byte aligned. Outputs are within the fp32 bound of the exact values; the summation
 *   order differs from strata_mmvq_multi's, so the two agree within the bound, not bit for bit.
 *   Errors: NULL, SHAPE, ALIGN, CUDA; a timed-out wait sets bit 0 of the device error word.
 */
int strata_gemm_q4(const void* W, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                   int64_t n_tok, float* y, cudaStream_t stream);

/*
 * strata_gemm_q4_dequant — the same dense prompt-chunk GEMM in the "wide dequant" arm of the Strata
 * pull request "sm_80 (GA100) tuning" (commit message on STRATA_DEQUANT_WIDE: the dense weights are
 * dequantized once per prompt chunk, then multiplied). A conversion pass writes the weight codes
 * q - 8 and the activation codes as fp16 (exact) into the workspace, in 128 x 32 tiles already in the
 * tensor cores' shared-memory order, with the matching d_w and d_x vectors; the GEMM then streams
 * them with bulk copies. Same arguments, rules and results as strata_gemm_q4, bit for bit (the same
 * block arithmetic in the same order), plus:
 *   workspace : strata_gemm_q4_dequant_workspace(rows, cols, n_tok) bytes, device, 256-byte aligned;
 *               contents need no initialisation and are dead after the call.
 *   Errors: NULL, SHAPE, ALIGN, WORKSPACE, CUDA; a timed-out wait sets bit 0 of the device error word.
 */
size_t strata_gemm_q4_dequant_workspace(int64_t rows, int64_t cols, int64_t n_tok);
int strata_gemm_q4_dequant(const void* W, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                           int64_t n_tok, float* y, void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * strata_moe_grouped — prompt-chunk MoE experts: per (token, slot) pair p = tok*k + slot routed to
 * expert e = ids[p]:
 *     g = W_gate[e] . xq(tok), u = W_up[e] . xq(tok)         (block arithmetic above, fp32)
 *     h = silu(g) * u,  silu(g) = g / (1 + exp(-g))          (fp32)
 *     (hq, hd, hs) = quantize_act(h)                          (same quantizer, blocks of 32)
 *     y[p][:] = W_down[e] . hq                                (fp32, unweighted row per pair)
 *   Source: verify.hpp, PoolMultiFn ("x_f (n_tok, n_embd), ids (n_tok, k) -> out (n_tok * k,
 *   n_embd)"), and the pull request "sm_80 (GA100) tuning", commit messages on the fused prompt
 *   MoE experts (one layer of 3,256 tokens; gate/up then down).
 *   experts : DEVICE array of n_expert strata_expert; each field a device pointer to a Q4 matrix:
 *             gate [inter][hidden], up [inter][hidden], down [hidden][inter].
 *   ids : int32 [n_tok][k], device.   x : fp32 [n_tok][hidden], device, 16-byte aligned.
 *   y   : fp32 [n_tok*k][hidden], device. Rows of pairs whose id is out of range are not written.
 *   workspace : strata_moe_grouped_workspace(...) bytes, 256-byte aligned, contents need no
 *               initialisation. err_word : device int32 or NULL; when non-NULL it is zeroed by the
 *               call and then gets bit 0 set if any id was outside [0, n_expert).
 *   hidden % 128 == 0, inter % 128 == 0, 1 <= k <= 16, n_expert >= 1.
 *   Pairs are grouped per expert in ascending (token, slot) order; each row of y is written once.
 *   Errors: NULL, SHAPE, ALIGN, WORKSPACE, CUDA (STRATA_ERR_EXPERT is reported in err_word).
 */
typedef struct { const void* gate; const void* up; const void* down; } strata_expert;

size_t strata_moe_grouped_workspace(int n_expert, int64_t n_tok, int k, int64_t hidden, int64_t inter);
int strata_moe_grouped(const strata_expert* experts, int n_expert, int64_t hidden, int64_t inter,
                       const int32_t* ids, int64_t n_tok, int k, const float* x, float* y,
                       void* workspace, size_t ws_bytes, int32_t* err_word, cudaStream_t stream);

/*
 * strata_moe_grouped_gu — test hook: strata_moe_grouped (same arguments, same kernels, same results)
 *   that also writes the fp32 gate and up outputs g, u of every pair with a valid id, exactly as the
 *   kernel holds them before SiLU: gu fp32 [n_tok*k][2][inter] (pair p = tok*k + slot; row p, plane 0
 *   is g, plane 1 is u), device, 16-byte aligned. Rows of pairs with an out-of-range id are not
 *   written. Errors: those of strata_moe_grouped; gu NULL is STRATA_ERR_NULL.
 */
int strata_moe_grouped_gu(const strata_expert* experts, int n_expert, int64_t hidden, int64_t inter,
                          const int32_t* ids, int64_t n_tok, int k, const float* x, float* y,
                          void* workspace, size_t ws_bytes, int32_t* err_word, float* gu, cudaStream_t stream);

/*
 * strata_moe_debug_views — byte offsets, inside a strata_moe_grouped workspace, of the grouping
 * and the re-quantized hidden activations a call leaves behind (test hook; no launch).
 *   counts int32 [n_expert], offsets int32 [n_expert+1], pairs int32 [n_tok*k] (pair p = tok*k+slot,
 *   grouped by expert, ascending within an expert), hq int8 [n_tok*k][inter] / hd fp32 /
 *   hs int32 [n_tok*k][inter/32] indexed by position in `pairs`. Offsets are written to the seven
 *   host size_t slots of `out` in that order. Errors: NULL, SHAPE.
 */
int strata_moe_debug_views(int n_expert, int64_t n_tok, int k, int64_t hidden, int64_t inter,
                           size_t* out);

/*
 * strata_block_dots — test hook: the exact integer block dots the GEMV kernels accumulate,
 *   isum[t][r][b] as int32 [T][rows][cols/32], computed by the same device block-dot code.
 *   Source: the pull request "sm_80 (GA100) tuning", hoisted-load MMVQ-IL commit (exact integer
 *   forms). Errors: NULL, SHAPE, T, FMT, ALIGN, CUDA.
 */
int strata_block_dots(const void* W, int64_t rows, int64_t cols, int fmt,
                      const int8_t* xq, const int32_t* xs, int T, int32_t* isum,
                      cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* STRATA_H */
