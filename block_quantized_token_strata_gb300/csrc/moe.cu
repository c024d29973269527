// moe.cu — prompt-chunk MoE experts over block-quantized (Q4) expert matrices.
//
// Per (token, slot) pair p = tok*k + slot routed to expert e = ids[p]:
//   g = W_gate[e] . xq(tok), u = W_up[e] . xq(tok)      (exact int dots per 32-block, fp32 scale)
//   h = silu(g) * u, re-quantized per 32 values like the activations
//   y[p] = W_down[e] . hq                              (one unweighted output row per pair)
// The output layout (n_tok*k, n_embd) is the expert pool's (Strata commit "wire multi-token
// kernels into Verifier and MtpDrafter CUDA graphs", verify.hpp, PoolMultiFn); the grouped prompt
// path is the fused prompt MoE experts of the pull request "sm_80 (GA100) tuning" (one layer of
// 3,256 tokens).
//
// Steps: quantize x -> group pairs per expert (ascending pair order) -> gate/up + SiLU + requant
// -> down + scatter to rows p.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace strata {

struct ExpertPtrs {
    const uint8_t* gate;
    const uint8_t* up;
    const uint8_t* down;
};

static size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

MoeLayout moe_workspace_layout(int n_expert, int64_t n_tok, int k, int64_t hidden, int64_t inter)
{
    MoeLayout L = {};
    const size_t n_pair = size_t(n_tok) * size_t(k);
    size_t o = 0;
    L.xq = o;      o = al256(o + size_t(n_tok) * hidden);
    L.xd = o;      o = al256(o + size_t(n_tok) * (hidden / 32) * 4);
    L.xs = o;      o = al256(o + size_t(n_tok) * (hidden / 32) * 4);
    L.counts = o;  o = al256(o + size_t(n_expert) * 4);
    L.offsets = o; o = al256(o + size_t(n_expert + 1) * 4);
    L.pairs = o;   o = al256(o + n_pair * 4);
    L.hq = o;      o = al256(o + n_pair * inter);
    L.hd = o;      o = al256(o + n_pair * (inter / 32) * 4);
    L.hs = o;      o = al256(o + n_pair * (inter / 32) * 4);
    L.total = o;
    return L;
}

// ---- grouping -------------------------------------------------------------------------------------
// CTA e: offset = number of valid ids below e; then an ordered ballot compaction of the pairs
// routed to e, so that each expert's list is in ascending pair order without atomics.
__global__ void __launch_bounds__(256) moe_bucket_kernel(const int32_t* __restrict__ ids, int n_pair,
                                                         int n_expert, int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ pairs, int32_t* err_word)
{
    pdl_wait();
    pdl_launch();
    __shared__ int s_red[2][8];
    __shared__ int s_cnt[8];
    const int e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int below = 0, bad = 0;
    for (int i = threadIdx.x; i < n_pair; i += blockDim.x) {
        const int v = ids[i];
        below += (v >= 0 && v < e);
        bad += (v < 0 || v >= n_expert);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        below += __shfl_xor_sync(0xffffffffu, below, off);
        bad += __shfl_xor_sync(0xffffffffu, bad, off);
    }
    if (lane == 0) { s_red[0][warp] = below; s_red[1][warp] = bad; }
    __syncthreads();
    below = 0;
    bad = 0;
    for (int w = 0; w < 8; ++w) { below += s_red[0][w]; bad += s_red[1][w]; }

    const unsigned lt = (1u << lane) - 1u;
    int base = 0;
    for (int c0 = 0; c0 < n_pair; c0 += blockDim.x) {
        const int i = c0 + threadIdx.x;
        const bool m = i < n_pair && ids[i] == e;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (lane == 0) s_cnt[warp] = __popc(bal);
        __syncthreads();
        int wbase = 0, tot = 0;
        for (int w = 0; w < 8; ++w) {
            wbase += (w < warp) ? s_cnt[w] : 0;
            tot += s_cnt[w];
        }
        if (m) pairs[below + base + wbase + __popc(bal & lt)] = i;
        base += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        counts[e] = base;
        offsets[e] = below;
        if (e == n_expert - 1) offsets[n_expert] = below + base;
        if (e == 0 && err_word) *err_word = bad ? 1 : 0;
    }
}

// ---- gate/up + SiLU + requant (one warp = one pair position x 32 hidden columns) -------------------
__global__ void __launch_bounds__(256) moe_gateup_kernel(const ExpertPtrs* __restrict__ experts, int n_expert,
                                                         int hidden, int inter, const int32_t* __restrict__ ids,
                                                         int k, const int32_t* __restrict__ pairs,
                                                         const int32_t* __restrict__ offsets,
                                                         const int8_t* __restrict__ xq,
                                                         const float* __restrict__ xd,
                                                         const int32_t* __restrict__ xs, int8_t* __restrict__ hq,
                                                         float* __restrict__ hd, int32_t* __restrict__ hs)
{
    pdl_wait();
    pdl_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pos = blockIdx.x * 8 + warp;
    if (pos >= offsets[n_expert]) return;
    const int p = pairs[pos];
    const int tok = p / k;
    const ExpertPtrs ex = experts[ids[p]];
    const int nbh = hidden / 32;
    const int c = blockIdx.y * 32 + lane;
    const uint8_t* gq = ex.gate + size_t(c) * nbh * 16;
    const uint8_t* uq = ex.up + size_t(c) * nbh * 16;
    const unsigned short* gs = reinterpret_cast<const unsigned short*>(ex.gate + size_t(inter) * nbh * 16) + size_t(c) * nbh;
    const unsigned short* us = reinterpret_cast<const unsigned short*>(ex.up + size_t(inter) * nbh * 16) + size_t(c) * nbh;
    const uint4* xr = reinterpret_cast<const uint4*>(xq + size_t(tok) * hidden);
    const float* dr = xd + size_t(tok) * nbh;
    const int32_t* sr = xs + size_t(tok) * nbh;
    float g = 0.0f, u = 0.0f;
    for (int b = 0; b < nbh; ++b) {
        const uint4 xl = __ldg(xr + 2 * b), xh = __ldg(xr + 2 * b + 1);
        const int c0 = kMagicBits - 8 * __ldg(sr + b);
        const float dx = __ldg(dr + b);
        const uint4 wg = __ldg(reinterpret_cast<const uint4*>(gq) + b);
        const uint4 wu = __ldg(reinterpret_cast<const uint4*>(uq) + b);
        const float dg = __half2float(__ushort_as_half(__ldg(gs + b)));
        const float du = __half2float(__ushort_as_half(__ldg(us + b)));
        g = __fmaf_rn(__fmul_rn(dg, dx), magic_to_float(dot_q4(wg, xl, xh, c0)), g);
        u = __fmaf_rn(__fmul_rn(du, dx), magic_to_float(dot_q4(wu, xl, xh, c0)), u);
    }
    const float h = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
    float a = fabsf(h);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    const float d = __fdiv_rn(a, 127.0f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    const int q = int(roundf(__fmul_rn(h, id)));
    int s = q;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    hq[size_t(pos) * inter + c] = int8_t(q);
    if (lane == 0) {
        hd[size_t(pos) * (inter / 32) + blockIdx.y] = d;
        hs[size_t(pos) * (inter / 32) + blockIdx.y] = s;
    }
}

// ---- down + scatter (one warp = one pair position x 32 output columns) ------------------------------
__global__ void __launch_bounds__(256) moe_down_kernel(const ExpertPtrs* __restrict__ experts, int n_expert,
                                                       int hidden, int inter, const int32_t* __restrict__ ids,
                                                       const int32_t* __restrict__ pairs,
                                                       const int32_t* __restrict__ offsets,
                                                       const int8_t* __restrict__ hq, const float* __restrict__ hd,
                                                       const int32_t* __restrict__ hs, float* __restrict__ y)
{
    pdl_wait();
    pdl_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pos = blockIdx.x * 8 + warp;
    if (pos >= offsets[n_expert]) return;
    const int p = pairs[pos];
    const ExpertPtrs ex = experts[ids[p]];
    const int nbi = inter / 32;
    const int c = blockIdx.y * 32 + lane;
    const uint8_t* wq = ex.down + size_t(c) * nbi * 16;
    const unsigned short* ws = reinterpret_cast<const unsigned short*>(ex.down + size_t(hidden) * nbi * 16) + size_t(c) * nbi;
    const uint4* xr = reinterpret_cast<const uint4*>(hq + size_t(pos) * inter);
    float acc = 0.0f;
    for (int b = 0; b < nbi; ++b) {
        const uint4 xl = __ldg(xr + 2 * b), xh = __ldg(xr + 2 * b + 1);
        const int c0 = kMagicBits - 8 * __ldg(hs + size_t(pos) * nbi + b);
        const float dx = __ldg(hd + size_t(pos) * nbi + b);
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(wq) + b);
        const float dw = __half2float(__ushort_as_half(__ldg(ws + b)));
        acc = __fmaf_rn(__fmul_rn(dw, dx), magic_to_float(dot_q4(w, xl, xh, c0)), acc);
    }
    y[size_t(p) * hidden + c] = acc;
}

cudaError_t launch_moe_grouped(const void* experts, int n_expert, int64_t hidden, int64_t inter,
                               const int32_t* ids, int64_t n_tok, int k, const float* x, float* y,
                               uint8_t* ws, const MoeLayout& L, int32_t* err_word, cudaStream_t stream)
{
    const int n_pair = int(n_tok * k);
    int8_t* xq = reinterpret_cast<int8_t*>(ws + L.xq);
    float* xd = reinterpret_cast<float*>(ws + L.xd);
    int32_t* xs = reinterpret_cast<int32_t*>(ws + L.xs);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    int32_t* pairs = reinterpret_cast<int32_t*>(ws + L.pairs);
    int8_t* hq = reinterpret_cast<int8_t*>(ws + L.hq);
    float* hd = reinterpret_cast<float*>(ws + L.hd);
    int32_t* hs = reinterpret_cast<int32_t*>(ws + L.hs);
    const ExpertPtrs* ex = static_cast<const ExpertPtrs*>(experts);

    cudaError_t e = launch_quantize_act(x, n_tok, hidden, xq, xd, xs, stream);
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_bucket_kernel, dim3(n_expert), dim3(256), 0, stream, ids, n_pair, n_expert, counts,
                   offsets, pairs, err_word);
    if (e != cudaSuccess) return e;
    const unsigned gx = unsigned((n_pair + 7) / 8);
    e = launch_pdl(moe_gateup_kernel, dim3(gx, unsigned(inter / 32)), dim3(256), 0, stream, ex, n_expert,
                   int(hidden), int(inter), ids, k, (const int32_t*)pairs, (const int32_t*)offsets,
                   (const int8_t*)xq, (const float*)xd, (const int32_t*)xs, hq, hd, hs);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_down_kernel, dim3(gx, unsigned(hidden / 32)), dim3(256), 0, stream, ex, n_expert,
                      int(hidden), int(inter), ids, (const int32_t*)pairs, (const int32_t*)offsets,
                      (const int8_t*)hq, (const float*)hd, (const int32_t*)hs, y);
}

}  // namespace strata
