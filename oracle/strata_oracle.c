/*
 * strata_oracle.c — plain, slow CPU oracle of the block-quantized verify path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call this file; only the
 * tests, the package's smoke check and the benchmark's CPU-baseline leg use it. It shares no code,
 * header or table with the CUDA library: the fp16 decoder, the block layouts and the quantizer are
 * written out again here from their definitions.
 *
 * Sources (pages on the Strata engine):
 *   - commit "wire multi-token kernels into Verifier and MtpDrafter CUDA graphs", verify.hpp header
 *     comment: a T-token verify window whose per-token arithmetic equals the single-token
 *     kernel's (exact mode), the dense weights read once for T tokens, activations held as
 *     "T columns of q8_1" (member xq_), and the expert pool's output rows (n_tok * k, n_embd);
 *   - pull request "sm_80 (GA100) tuning", commit message of the hoisted-load MMVQ-IL kernels:
 *     integer block dots are exact and only their fp32 accumulation is ordered;
 *   - dsv41-offload worker/tp2.py, EmuComm.argmax / markov_local_argmax: argmax ties go to the
 *     lowest id.
 * Readings where the pages are silent (block formats, the quantizer, the MoE hidden activation):
 *   Q4 block = fp16 d + 32 unsigned 4-bit codes, w = d*(q-8); Q8 block = fp16 d + 32 int8 codes,
 *   w = d*q; Q6 (the pages' 6-bit super-block type, 210 bytes per 256 weights): per 256 weights an
 *   fp16 d, per 16 weights an int8 sub-scale s, 6-bit codes q, w = d*s*(q-32), with exact integer
 *   dots per 16 weights (one term per sub-scale); Q4K (the pages' 4-bit super-block type with
 *   minimums): per 32 weights a 6-bit scale sc and minimum m, per 256 weights fp16 d and dmin, 4-bit
 *   codes q, w = d*sc*q - dmin*m, two terms per 32 weights (d*sc*d_x*isum and -dmin*m*d_x*sum x);
 *   Q5K (the pages' 5-bit super-block type, whose dots take the same two exact forms as Q4K's):
 *   Q4K with 5-bit codes q in 0..31; a row's code plane holds its Q4-style nibble blocks, then one
 *   32-bit little-endian word per block whose bit 8k + w is the fifth bit of the k-th code of
 *   four-code group w (groups 0..3 = elements 0..15 in fours, 4..7 = elements 16..31);
 *   activations: per 32 values amax, d = amax/127 (fp32), q = roundf(x/d) via x*(1/d),
 *   s = sum q; MoE hidden h = silu(g)*u with silu(g) = g/(1+exp(-g)), re-quantized the same way.
 *
 * Arithmetic: integer dots in int64 (exact); block terms d_w * d_x * isum and all sums in fp64, in
 * block order; the activation quantizer in IEEE fp32 single operations, as defined. OpenMP only
 * splits independent output rows across threads; it never reorders any row's arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_Q4 0
#define OR_Q8 1
#define OR_Q6 2
#define OR_Q4K 3
#define OR_Q5K 4

/* ---- IEEE 754 binary16 -> double, from the format's definition ---------------------------- */
double or_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int mant = h & 0x3FF;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24);             /* subnormal: mant * 2^-24 */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + mant), expo - 25); /* (1 + mant/1024) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* ---- the planar weight layout ---------------------------------------------------------------- */
static int64_t qbytes(int fmt)
{
    if (fmt == OR_Q4 || fmt == OR_Q4K) return 16;
    if (fmt == OR_Q5K) return 20;  /* per block in the code plane: 16 nibble bytes + a 4-byte word */
    return fmt == OR_Q8 ? 32 : 24;
}

/* Q4/Q8: the fp16 scale of block (r, b). Q6: the fp16 d of the super-block holding block b, which
 * sits after the code plane (24 bytes a block) and the sub-scale plane (2 int8 a block). */
static double block_scale(const uint8_t* W, int64_t rows, int64_t nb, int fmt, int64_t r, int64_t b)
{
    const uint8_t* p;
    if (fmt == OR_Q6)
        p = W + rows * nb * 26 + 2 * (r * (nb / 8) + b / 8);
    else if (fmt == OR_Q4K || fmt == OR_Q5K)  /* d of the super-block (dmin follows it) */
        p = W + rows * nb * (qbytes(fmt) + 2) + 4 * (r * (nb / 8) + b / 8);
    else
        p = W + rows * nb * qbytes(fmt) + 2 * (r * nb + b);
    uint16_t bits = (uint16_t)(p[0] | (p[1] << 8));
    return or_half_to_double(bits);
}

/* Q4K / Q5K: the super-block's fp16 dmin, and block (r, b)'s 6-bit scale (k = 0) or minimum (k = 1);
 * both planes follow the code plane */
static double kq_dmin(const uint8_t* W, int64_t rows, int64_t nb, int fmt, int64_t r, int64_t b)
{
    const uint8_t* p = W + rows * nb * (qbytes(fmt) + 2) + 4 * (r * (nb / 8) + b / 8) + 2;
    return or_half_to_double((uint16_t)(p[0] | (p[1] << 8)));
}
static int kq_scale_min(const uint8_t* W, int64_t rows, int64_t nb, int fmt, int64_t r, int64_t b, int k)
{
    return (int)W[rows * nb * qbytes(fmt) + 2 * (r * nb + b) + k];
}

/* Q6: the int8 sub-scale of half h (elements 16h..16h+15) of block (r, b) */
static int q6_subscale(const uint8_t* W, int64_t rows, int64_t nb, int64_t r, int64_t b, int h)
{
    return (int)(int8_t)W[rows * nb * 24 + 2 * (r * nb + b) + h];
}

/* weight code of element j (0..31) of block (r, b), already offset: Q4 q-8, Q8 q */
/* Q5K code of element j (0..31) of block (r, b): the row's nibble blocks, then its fifth-bit words;
 * code = low nibble | fifth bit << 4 */
__attribute__((noinline)) static int q5k_code(const uint8_t* W, int64_t nb, int64_t r, int64_t b, int j)
{
    const uint8_t* row = W + r * nb * 20;
    int byte = row[16 * b + (j & 15)];
    int low = (j < 16) ? (byte & 0x0F) : (byte >> 4);
    const uint8_t* hw = row + 16 * nb + 4 * b;
    uint32_t bits = (uint32_t)hw[0] | ((uint32_t)hw[1] << 8) | ((uint32_t)hw[2] << 16) | ((uint32_t)hw[3] << 24);
    int group = (j < 16) ? j / 4 : 4 + (j - 16) / 4;
    int k = j % 4;
    int fifth = (int)((bits >> (8 * k + group)) & 1u);
    return low | (fifth << 4);
}

static int weight_code(const uint8_t* W, int64_t nb, int fmt, int64_t r, int64_t b, int j)
{
    if (fmt == OR_Q5K) return q5k_code(W, nb, r, b, j);
    const uint8_t* blk = W + (r * nb + b) * qbytes(fmt);
    if (fmt == OR_Q4 || fmt == OR_Q4K) {  /* Q4K codes carry no offset: its minimum does that */
        int byte = blk[j & 15];
        int q = (j < 16) ? (byte & 0x0F) : (byte >> 4);
        return fmt == OR_Q4 ? q - 8 : q;
    }
    if (fmt == OR_Q6) {
        /* bytes 0..15: low 4 bits of element j (low nibble) and of element j+16 (high nibble);
         * bytes 16..23: byte 16+i holds the high 2 bits of elements i, i+8, i+16, i+24 (bits 0-1, 2-3,
         * 4-5, 6-7); the code q = low | high << 4 in 0..63 stands for q - 32 */
        int byte = blk[j & 15];
        int low = (j < 16) ? (byte & 0x0F) : (byte >> 4);
        int high = (blk[16 + (j & 7)] >> (2 * (j >> 3))) & 3;
        return (low | (high << 4)) - 32;
    }
    return (int)(int8_t)blk[j];
}

/* ---- activation quantizer: fp32, one IEEE operation per step ------------------------------- */
void or_quantize_act(const float* x, int64_t n, int64_t cols, int8_t* q, float* d, int32_t* s)
{
    int64_t nb = cols / 32;
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* xb = x + i * cols + 32 * b;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                float a = fabsf(xb[j]);
                if (a > amax) amax = a;
            }
            float dd = amax / 127.0f;
            float id = (dd != 0.0f) ? 1.0f / dd : 0.0f;
            int32_t sum = 0;
            for (int j = 0; j < 32; ++j) {
                float prod = xb[j] * id;
                int qi = (int)roundf(prod);
                q[i * cols + 32 * b + j] = (int8_t)qi;
                sum += qi;
            }
            d[i * nb + b] = dd;
            s[i * nb + b] = sum;
        }
    }
}

/* ---- exact integer block dot ------------------------------------------------------------------ */
static int64_t half_isum(const uint8_t* W, int64_t nb, int fmt, int64_t r, int64_t b, const int8_t* xq_blk, int h)
{
    int64_t acc = 0;
    for (int j = 16 * h; j < 16 * h + 16; ++j)
        acc += (int64_t)weight_code(W, nb, fmt, r, b, j) * (int64_t)xq_blk[j];
    return acc;
}

/* the block's exact integer dot; Q6: sub-scale-weighted, s0 * (first 16) + s1 * (last 16) */
static int64_t block_isum(const uint8_t* W, int64_t rows, int64_t nb, int fmt, int64_t r, int64_t b,
                          const int8_t* xq_blk)
{
    if (fmt == OR_Q6)
        return q6_subscale(W, rows, nb, r, b, 0) * half_isum(W, nb, fmt, r, b, xq_blk, 0) +
               q6_subscale(W, rows, nb, r, b, 1) * half_isum(W, nb, fmt, r, b, xq_blk, 1);
    return half_isum(W, nb, fmt, r, b, xq_blk, 0) + half_isum(W, nb, fmt, r, b, xq_blk, 1);
}

/* isum[t][r][b] for every token, row and block (int64) */
void or_block_dots(const uint8_t* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq, int64_t T,
                   int64_t* isum)
{
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t b = 0; b < nb; ++b)
                isum[(t * rows + r) * nb + b] = block_isum(W, rows, nb, fmt, r, b, xq + t * cols + 32 * b);
}

/* one output: y = sum_b d_w * d_x * isum in fp64, block order; A = sum_b |term| */
static void row_dot(const uint8_t* W, int64_t rows, int64_t nb, int fmt, int64_t r,
                    const int8_t* xq_row, const float* xd_row, double* y, double* A)
{
    double acc = 0.0, aabs = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        if (fmt == OR_Q4K || fmt == OR_Q5K) {  /* d*sc*d_x*isum, then -dmin*m*d_x*(sum of the block's x codes) */
            int64_t isum = block_isum(W, rows, nb, fmt, r, b, xq_row + 32 * b), xsum = 0;
            for (int j = 0; j < 32; ++j) xsum += xq_row[32 * b + j];
            double t1 = block_scale(W, rows, nb, fmt, r, b) * (double)kq_scale_min(W, rows, nb, fmt, r, b, 0) *
                        (double)xd_row[b] * (double)isum;
            double t2 = -kq_dmin(W, rows, nb, fmt, r, b) * (double)kq_scale_min(W, rows, nb, fmt, r, b, 1) *
                        (double)xd_row[b] * (double)xsum;
            acc += t1;
            acc += t2;
            aabs += fabs(t1) + fabs(t2);
            continue;
        }
        if (fmt == OR_Q6) {  /* one term per 16 weights: d * s_h * d_x * isum_h */
            for (int h = 0; h < 2; ++h) {
                int64_t isum = half_isum(W, nb, fmt, r, b, xq_row + 32 * b, h);
                double term = block_scale(W, rows, nb, fmt, r, b) * (double)q6_subscale(W, rows, nb, r, b, h) *
                              (double)xd_row[b] * (double)isum;
                acc += term;
                aabs += fabs(term);
            }
            continue;
        }
        int64_t isum = block_isum(W, rows, nb, fmt, r, b, xq_row + 32 * b);
        double term = block_scale(W, rows, nb, fmt, r, b) * (double)xd_row[b] * (double)isum;
        acc += term;
        aabs += fabs(term);
    }
    *y = acc;
    *A = aabs;
}

/* y[t][r], A[t][r] for T token rows of quantized activations */
void or_mmvq(const uint8_t* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq, const float* xd,
             int64_t T, double* y, double* A)
{
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t t = 0; t < T; ++t)
            row_dot(W, rows, nb, fmt, r, xq + t * cols, xd + t * nb, &y[t * rows + r], &A[t * rows + r]);
}

/* same as or_mmvq restricted to the listed rows: y[t][i], A[t][i] for row sel[i] */
void or_mmvq_rows(const uint8_t* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq, const float* xd,
                  int64_t T, const int64_t* sel, int64_t n_sel, double* y, double* A)
{
    int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n_sel; ++i)
        for (int64_t t = 0; t < T; ++t)
            row_dot(W, rows, nb, fmt, sel[i], xq + t * cols, xd + t * nb, &y[t * n_sel + i], &A[t * n_sel + i]);
}

/* argmax over each of T rows of n values; ties go to the lowest index */
void or_argmax(const double* v, int64_t T, int64_t n, int32_t* ids)
{
    for (int64_t t = 0; t < T; ++t) {
        int64_t best = 0;
        for (int64_t i = 1; i < n; ++i)
            if (v[t * n + i] > v[t * n + best]) best = i;
        ids[t] = (int32_t)best;
    }
}

/* top-2 margin of each of T rows of n values (dsv41-offload worker/tp2.py, EmuComm.margin): the
 * largest value minus the largest of the values left once one occurrence of the largest is taken
 * out; a maximum that occurs twice gives 0; a single value gives +inf. */
void or_margin(const double* v, int64_t T, int64_t n, double* margin)
{
    for (int64_t t = 0; t < T; ++t) {
        const double* row = v + t * n;
        int64_t best = 0;
        for (int64_t i = 1; i < n; ++i)
            if (row[i] > row[best]) best = i;
        double second = -INFINITY;
        for (int64_t i = 0; i < n; ++i)
            if (i != best && row[i] > second) second = row[i];
        margin[t] = row[best] - second;
    }
}

/* ---- prompt-chunk MoE ---------------------------------------------------------------------------- */

/* group the (token, slot) pairs per expert, ascending pair index p = tok*k + slot within an expert.
 * counts[e], offsets[e] (exclusive prefix, offsets[n_expert] = valid pairs), pairs[...]; returns the
 * number of pairs whose id lies outside [0, n_expert) (those are left out). */
int64_t or_moe_bucket(const int32_t* ids, int64_t n_tok, int k, int n_expert,
                      int32_t* counts, int32_t* offsets, int32_t* pairs)
{
    int64_t bad = 0, n_pair = n_tok * k;
    for (int e = 0; e < n_expert; ++e) counts[e] = 0;
    for (int64_t p = 0; p < n_pair; ++p) {
        int32_t e = ids[p];
        if (e < 0 || e >= n_expert) { ++bad; continue; }
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < n_expert; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)calloc((size_t)n_expert, sizeof(int32_t));
    for (int64_t p = 0; p < n_pair; ++p) {
        int32_t e = ids[p];
        if (e < 0 || e >= n_expert) continue;
        pairs[offsets[e] + fill[e]] = (int32_t)p;
        fill[e] += 1;
    }
    free(fill);
    return bad;
}

/* The MoE output rows y[i][:] (fp64) and A[i][:] of the listed pairs sel[i] = tok*k + slot.
 * Optional (may be NULL): h[i][inter] fp64 hidden, hq/hd/hs its quantization; g[i][inter] and
 * u[i][inter] the fp64 gate and up outputs with their tolerance masses ag, au (sum of |block terms|).
 * If hq_in/hd_in are given, the down projection takes THOSE quantized hidden rows (indexed by i)
 * instead of quantizing the oracle's own h. Pairs with an out-of-range id get y = NaN. */
void or_moe_rows(const uint8_t* const* gate, const uint8_t* const* up, const uint8_t* const* down,
                 int n_expert, int64_t hidden, int64_t inter, const int32_t* ids, int64_t n_tok, int k,
                 const float* x, const int64_t* sel, int64_t n_sel, double* y, double* A,
                 double* h_out, int8_t* hq_out, float* hd_out, int32_t* hs_out,
                 const int8_t* hq_in, const float* hd_in,
                 double* g_out, double* u_out, double* ag_out, double* au_out)
{
    int64_t nbh = hidden / 32, nbi = inter / 32;
    (void)n_tok;
#pragma omp parallel
    {
        int8_t* xq = (int8_t*)malloc((size_t)hidden);
        float* xd = (float*)malloc(sizeof(float) * (size_t)nbh);
        int32_t* xs = (int32_t*)malloc(sizeof(int32_t) * (size_t)nbh);
        double* h = (double*)malloc(sizeof(double) * (size_t)inter);
        float* hf = (float*)malloc(sizeof(float) * (size_t)inter);
        int8_t* hq = (int8_t*)malloc((size_t)inter);
        float* hd = (float*)malloc(sizeof(float) * (size_t)nbi);
        int32_t* hs = (int32_t*)malloc(sizeof(int32_t) * (size_t)nbi);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_sel; ++i) {
            int64_t p = sel[i], tok = p / k;
            int32_t e = ids[p];
            if (e < 0 || e >= n_expert) {
                for (int64_t c = 0; c < hidden; ++c) { y[i * hidden + c] = NAN; A[i * hidden + c] = NAN; }
                continue;
            }
            or_quantize_act(x + tok * hidden, 1, hidden, xq, xd, xs);
            for (int64_t c = 0; c < inter; ++c) {
                double g, ag, u, au;
                row_dot(gate[e], inter, nbh, OR_Q4, c, xq, xd, &g, &ag);
                row_dot(up[e], inter, nbh, OR_Q4, c, xq, xd, &u, &au);
                if (g_out) { g_out[i * inter + c] = g; ag_out[i * inter + c] = ag; }
                if (u_out) { u_out[i * inter + c] = u; au_out[i * inter + c] = au; }
                h[c] = g / (1.0 + exp(-g)) * u;
                hf[c] = (float)h[c];
            }
            or_quantize_act(hf, 1, inter, hq, hd, hs);
            if (h_out) memcpy(h_out + i * inter, h, sizeof(double) * (size_t)inter);
            if (hq_out) memcpy(hq_out + i * inter, hq, (size_t)inter);
            if (hd_out) memcpy(hd_out + i * nbi, hd, sizeof(float) * (size_t)nbi);
            if (hs_out) memcpy(hs_out + i * nbi, hs, sizeof(int32_t) * (size_t)nbi);
            const int8_t* dq = hq_in ? hq_in + i * inter : hq;
            const float* dd = hd_in ? hd_in + i * nbi : hd;
            for (int64_t c = 0; c < hidden; ++c)
                row_dot(down[e], hidden, nbi, OR_Q4, c, dq, dd, &y[i * hidden + c], &A[i * hidden + c]);
        }
        free(xq); free(xd); free(xs); free(h); free(hf); free(hq); free(hd); free(hs);
    }
}

/* ---- threads ----------------------------------------------------------------------------------- */
void or_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int or_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
