// mmvq.cu — multi-token block-quantized GEMV (T <= 8 columns, one weight read) and the fused
// vocabulary head + argmax.
//
// What it computes: y[t][r] = sum_b (d_w[r][b] * d_x[t][b]) * isum[t][r][b] with exact int32 block
// dots isum, for T tokens that share one read of W — the verify window's "multi-column MMVQ in
// exact mode" (Strata commit "wire multi-token kernels into Verifier and MtpDrafter CUDA graphs",
// verify.hpp header comment). As in the hoisted-load MMVQ-IL kernels of the pull request "sm_80
// (GA100) tuning", the integer dots are exact, the int->float conversion is the exact
// 1.5*2^23 magic form, and the fp32 accumulation order and the xor tree are fixed.
//
// Exactness across T (column t of a T-token launch == the T = 1 launch):
//   * lane l of the warp that owns row r takes blocks b = l, l+32, l+64, ... in ascending order and
//     folds each into acc = fma(d_w*d_x, float(isum), acc) with explicitly rounded intrinsics;
//   * the 32 lane partials are combined by the xor tree 16, 8, 4, 2, 1;
//   * neither the lane<->block map nor the tree depends on T, R (rows a warp holds at once), the
//     grid or the CTA size; T is only the trip count of an inner loop over independent columns.
//
// Data movement (GB300): W streams from HBM with 128-bit read-only loads that skip L1; before the
// kernel waits on its predecessor (programmatic dependent launch) each CTA issues bulk L2
// prefetches for the first rows of its contiguous row range, and every warp keeps prefetching a
// fixed distance ahead, so the HBM queue is full while the previous kernel drains. Activations
// (T x cols codes, scales, sums) are staged once per CTA in shared memory, split into the 16-byte
// halves each dp4a chain consumes so that lanes read consecutive 16-byte words (no conflicts).
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace strata {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int FMT> struct FmtInfo;
template <> struct FmtInfo<0> { static constexpr int kQB = 16; };  // Q4: 16 code bytes per block
template <> struct FmtInfo<1> { static constexpr int kQB = 32; };  // Q8: 32 code bytes per block

struct MmvqArgs {
    const uint8_t* W;
    int rows;
    int nb;
    const int8_t* xq;
    const float* xd;
    const int32_t* xs;
    float* y;          // [T][rows] or null
    float* cand_val;   // head: [T][gridDim.x] per-CTA maxima
    int* cand_idx;     // head: [T][gridDim.x] their row ids
    int rg_total;      // row groups of R rows
    int pf_rg;         // prefetch distance in row groups
};

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

template <int FMT, int T, int R, bool HEAD>
__global__ void __launch_bounds__(kThreads, 2) mmvq_kernel(const MmvqArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int QB = FmtInfo<FMT>::kQB;
    constexpr int QV = QB / 16;  // 16-byte code words per block
    const int nb = a.nb;
    const int rows = a.rows;
    uint4* sx = reinterpret_cast<uint4*>(smem);                               // [T][2][nb]
    int2* scd = reinterpret_cast<int2*>(smem + size_t(T) * 2 * nb * 16);     // [T][nb] (c0, d_x)
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int rg0 = int((int64_t(blockIdx.x) * a.rg_total) / gridDim.x);
    const int rg1 = int((int64_t(blockIdx.x + 1) * a.rg_total) / gridDim.x);
    const uint8_t* qplane = a.W;
    const unsigned short* splane =
        reinterpret_cast<const unsigned short*>(a.W + size_t(rows) * nb * QB);

    auto prefetch_groups = [&](int g0, int g1) {  // row groups [g0, g1) of this matrix
        const int r0 = g0 * R;
        const int r1 = min(g1 * R, rows);
        if (r0 >= r1) return;
        prefetch_l2(qplane + size_t(r0) * nb * QB, size_t(r1 - r0) * nb * QB);
        prefetch_l2(splane + size_t(r0) * nb, size_t(r1 - r0) * nb * 2);
    };

    // (1) weights are static data: start pulling this CTA's first rows toward L2 now
    if (threadIdx.x == 0) prefetch_groups(rg0, min(rg1, rg0 + a.pf_rg));

    // (2) activations may come from the previous kernel: wait, then let the next one start
    pdl_wait();
    pdl_launch();

    {
        const int nchunk = T * nb * 2;
        const uint4* src = reinterpret_cast<const uint4*>(a.xq);
        for (int i = threadIdx.x; i < nchunk; i += kThreads) {
            const int t = i / (2 * nb);
            const int c = i - t * 2 * nb;
            sx[(t * 2 + (c & 1)) * nb + (c >> 1)] = __ldg(src + i);
        }
        for (int i = threadIdx.x; i < T * nb; i += kThreads) {
            const int c0 = (FMT == 0) ? kMagicBits - 8 * __ldg(a.xs + i) : kMagicBits;
            scd[i] = make_int2(c0, __float_as_int(__ldg(a.xd + i)));
        }
    }
    __syncthreads();

    float best[HEAD ? T : 1];
    int bidx[HEAD ? T : 1];
    if constexpr (HEAD) {
#pragma unroll
        for (int t = 0; t < T; ++t) { best[t] = -FLT_MAX; bidx[t] = INT_MAX; }
    }

    for (int rg = rg0 + warp; rg < rg1; rg += kWarps) {
        if (lane == 0 && rg + a.pf_rg < rg1) prefetch_groups(rg + a.pf_rg, rg + a.pf_rg + 1);
        const int row0 = rg * R;
        const uint8_t* wr[R];
        const unsigned short* sr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int rr = min(row0 + r, rows - 1);
            wr[r] = qplane + size_t(rr) * nb * QB;
            sr[r] = splane + size_t(rr) * nb;
        }
        float acc[R][T];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < T; ++t) acc[r][t] = 0.0f;

        for (int kb0 = lane; kb0 < nb; kb0 += 64) {
            const int kb1 = kb0 + 32;
            const bool has1 = kb1 < nb;
            uint4 w[2][R][QV];
            float dw[2][R];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int kb = u ? (has1 ? kb1 : kb0) : kb0;
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int h = 0; h < QV; ++h) w[u][r][h] = ld_stream_v4(wr[r] + size_t(kb) * QB + h * 16);
                    dw[u][r] = __half2float(__ushort_as_half(ld_stream_u16(sr[r] + kb)));
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (u == 1 && !has1) break;
                const int kb = u ? kb1 : kb0;
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const uint4 xl = sx[(t * 2 + 0) * nb + kb];
                    const uint4 xh = sx[(t * 2 + 1) * nb + kb];
                    const int2 cd = scd[t * nb + kb];
                    const float dx = __int_as_float(cd.y);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        int c;
                        if constexpr (FMT == 0) c = dot_q4(w[u][r][0], xl, xh, cd.x);
                        else c = dot_q8(w[u][r][0], w[u][r][QV - 1], xl, xh, cd.x);
                        const float f = magic_to_float(c);
                        const float s = __fmul_rn(dw[u][r], dx);
                        acc[r][t] = __fmaf_rn(s, f, acc[r][t]);
                    }
                }
            }
        }

#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = row0 + r;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                float v = acc[r][t];
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 16));
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 8));
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
                if (row < rows) {
                    if (a.y != nullptr && lane == ((r * T + t) & 31)) a.y[size_t(t) * rows + row] = v;
                    if constexpr (HEAD) {
                        if (better(v, row, best[t], bidx[t])) { best[t] = v; bidx[t] = row; }
                    }
                }
            }
        }
    }

    if constexpr (HEAD) {
        float* rv = reinterpret_cast<float*>(scd + T * nb);   // [kWarps][T]
        int* ri = reinterpret_cast<int*>(rv + kWarps * T);
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < T; ++t) { rv[warp * T + t] = best[t]; ri[warp * T + t] = bidx[t]; }
        }
        __syncthreads();
        if (threadIdx.x < T) {
            const int t = threadIdx.x;
            float bv = rv[t];
            int bi = ri[t];
            for (int w2 = 1; w2 < kWarps; ++w2) {
                if (better(rv[w2 * T + t], ri[w2 * T + t], bv, bi)) { bv = rv[w2 * T + t]; bi = ri[w2 * T + t]; }
            }
            a.cand_val[size_t(t) * gridDim.x + blockIdx.x] = bv;
            a.cand_idx[size_t(t) * gridDim.x + blockIdx.x] = bi;
        }
    }
}

// one warp per token: reduce the per-CTA candidates with the tie rule (equal values -> lower id)
__global__ void __launch_bounds__(256) head_finalize_kernel(const float* __restrict__ cand_val,
                                                            const int* __restrict__ cand_idx, int ncand,
                                                            int T, int32_t* __restrict__ ids)
{
    pdl_wait();
    pdl_launch();
    const int t = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    float bv = -FLT_MAX;
    int bi = INT_MAX;
    for (int i = lane; i < ncand; i += 32) {
        const float v = cand_val[size_t(t) * ncand + i];
        const int j = cand_idx[size_t(t) * ncand + i];
        if (better(v, j, bv, bi)) { bv = v; bi = j; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) ids[t] = bi;
}

// test hook: isum[t][r][b] from the same dot_q4 / dot_q8 device code
template <int FMT>
__global__ void __launch_bounds__(256) block_dots_kernel(const uint8_t* __restrict__ W, int rows, int nb,
                                                         const int8_t* __restrict__ xq,
                                                         const int32_t* __restrict__ xs, int T,
                                                         int32_t* __restrict__ isum)
{
    pdl_wait();
    pdl_launch();
    constexpr int QB = FmtInfo<FMT>::kQB;
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= int64_t(rows) * nb) return;
    const int r = int(i / nb), b = int(i % nb);
    const uint4 w0 = ld_stream_v4(W + size_t(i) * QB);
    const uint4 w1 = (QB == 32) ? ld_stream_v4(W + size_t(i) * QB + 16) : w0;
    for (int t = 0; t < T; ++t) {
        const uint4* xp = reinterpret_cast<const uint4*>(xq + size_t(t) * nb * 32 + size_t(b) * 32);
        const uint4 xl = xp[0], xh = xp[1];
        const int c0 = (FMT == 0) ? kMagicBits - 8 * xs[size_t(t) * nb + b] : kMagicBits;
        const int c = (FMT == 0) ? dot_q4(w0, xl, xh, c0) : dot_q8(w0, w1, xl, xh, c0);
        isum[(size_t(t) * rows + r) * nb + b] = c - kMagicBits;
    }
}

// ---- host side -------------------------------------------------------------------------------------

int device_sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

static size_t staged_bytes(int T, int nb, bool head)
{
    return size_t(T) * nb * 40 + (head ? size_t(kWarps) * T * 8 : 0);
}

// rows a warp holds at once: only a throughput choice (it never changes any row's arithmetic)
static int choose_R(int64_t rows, int nsm)
{
    if (rows >= int64_t(4) * kWarps * 2 * nsm) return 4;
    if (rows >= int64_t(2) * kWarps * 2 * nsm) return 2;
    return 1;
}

template <int FMT, int T, int R, bool HEAD>
static cudaError_t launch_t(const MmvqArgs& base, int64_t rows, int nb, cudaStream_t stream, int* grid_out)
{
    MmvqArgs a = base;
    const int nsm = device_sm_count();
    a.rg_total = int((rows + R - 1) / R);
    const int want = (a.rg_total + kWarps - 1) / kWarps;
    const int grid = want < nsm * 4 ? want : nsm * 4;
    constexpr int QB = FmtInfo<FMT>::kQB;
    const size_t rg_bytes = size_t(R) * nb * (QB + 2);
    const size_t pf = (size_t(64) << 10) / (rg_bytes ? rg_bytes : 1);
    a.pf_rg = int(pf < 1 ? 1 : (pf > 4096 ? 4096 : pf));
    if (grid_out) *grid_out = grid;
    if (HEAD && a.cand_val == nullptr) return cudaSuccess;  // size query only
    const size_t smem = staged_bytes(T, nb, HEAD);
    auto kern = mmvq_kernel<FMT, T, R, HEAD>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, stream, a);
}

template <int FMT, int T, bool HEAD>
static cudaError_t launch_r(const MmvqArgs& a, int64_t rows, int nb, cudaStream_t stream, int* grid_out)
{
    if constexpr (HEAD) {
        return launch_t<FMT, T, 4, true>(a, rows, nb, stream, grid_out);
    } else {
        switch (choose_R(rows, device_sm_count())) {
            case 4: return launch_t<FMT, T, 4, false>(a, rows, nb, stream, grid_out);
            case 2: return launch_t<FMT, T, 2, false>(a, rows, nb, stream, grid_out);
            default: return launch_t<FMT, T, 1, false>(a, rows, nb, stream, grid_out);
        }
    }
}

template <int FMT, bool HEAD>
static cudaError_t launch_f(const MmvqArgs& a, int64_t rows, int nb, int T, cudaStream_t stream, int* grid_out)
{
    switch (T) {
        case 1: return launch_r<FMT, 1, HEAD>(a, rows, nb, stream, grid_out);
        case 2: return launch_r<FMT, 2, HEAD>(a, rows, nb, stream, grid_out);
        case 3: return launch_r<FMT, 3, HEAD>(a, rows, nb, stream, grid_out);
        case 4: return launch_r<FMT, 4, HEAD>(a, rows, nb, stream, grid_out);
        case 5: return launch_r<FMT, 5, HEAD>(a, rows, nb, stream, grid_out);
        case 6: return launch_r<FMT, 6, HEAD>(a, rows, nb, stream, grid_out);
        case 7: return launch_r<FMT, 7, HEAD>(a, rows, nb, stream, grid_out);
        case 8: return launch_r<FMT, 8, HEAD>(a, rows, nb, stream, grid_out);
        default: return cudaErrorInvalidValue;
    }
}

static cudaError_t dispatch(const MmvqArgs& a, int64_t rows, int nb, int fmt, int T, bool head,
                            cudaStream_t stream, int* grid_out)
{
    if (fmt == 0) return head ? launch_f<0, true>(a, rows, nb, T, stream, grid_out)
                              : launch_f<0, false>(a, rows, nb, T, stream, grid_out);
    return head ? launch_f<1, true>(a, rows, nb, T, stream, grid_out)
                : launch_f<1, false>(a, rows, nb, T, stream, grid_out);
}

cudaError_t launch_mmvq(const void* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq,
                        const float* xd, const int32_t* xs, int T, float* y, cudaStream_t stream)
{
    MmvqArgs a = {};
    a.W = static_cast<const uint8_t*>(W);
    a.rows = int(rows);
    a.nb = int(cols / kQK);
    a.xq = xq;
    a.xd = xd;
    a.xs = xs;
    a.y = y;
    return dispatch(a, rows, a.nb, fmt, T, false, stream, nullptr);
}

// the head grid is fixed by (vocab, device), so the workspace needs only a bound on it
static int head_grid_bound(int64_t vocab)
{
    const int64_t rg = (vocab + 3) / 4;
    const int64_t want = (rg + kWarps - 1) / kWarps;
    return int(want < 4096 ? want : 4096);
}

// scratch bytes one head launch uses on the current device (same grid formula as launch_t for R=4)
size_t head_launch_scratch_bytes(int64_t vocab, int T)
{
    const int64_t rg = (vocab + 3) / 4;
    const int64_t want = (rg + kWarps - 1) / kWarps;
    const int64_t cap = int64_t(device_sm_count()) * 4;
    return size_t(want < cap ? want : cap) * size_t(T) * 8;
}

size_t head_workspace_bytes(int64_t vocab, int T)
{
    return size_t(head_grid_bound(vocab)) * size_t(T) * 8 + 256;
}

cudaError_t launch_head_argmax(const void* W, int64_t vocab, int64_t cols, int fmt, const int8_t* xq,
                               const float* xd, const int32_t* xs, int T, int32_t* ids, float* logits,
                               void* workspace, cudaStream_t stream)
{
    MmvqArgs a = {};
    a.W = static_cast<const uint8_t*>(W);
    a.rows = int(vocab);
    a.nb = int(cols / kQK);
    a.xq = xq;
    a.xd = xd;
    a.xs = xs;
    a.y = logits;
    int grid = 0;
    cudaError_t e = dispatch(a, vocab, a.nb, fmt, T, true, stream, &grid);  // size query
    if (e != cudaSuccess) return e;
    if (grid > head_grid_bound(vocab)) return cudaErrorInvalidValue;
    a.cand_val = static_cast<float*>(workspace);
    a.cand_idx = reinterpret_cast<int*>(static_cast<char*>(workspace) + size_t(grid) * T * 4);
    e = dispatch(a, vocab, a.nb, fmt, T, true, stream, &grid);
    if (e != cudaSuccess) return e;
    return launch_pdl(head_finalize_kernel, dim3(1), dim3(32 * T), 0, stream,
                      (const float*)a.cand_val, (const int*)a.cand_idx, grid, T, ids);
}

cudaError_t launch_block_dots(const void* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq,
                              const int32_t* xs, int T, int32_t* isum, cudaStream_t stream)
{
    const int nb = int(cols / kQK);
    const int64_t n = rows * nb;
    const unsigned grid = unsigned((n + 255) / 256);
    const uint8_t* w = static_cast<const uint8_t*>(W);
    if (fmt == 0)
        return launch_pdl(block_dots_kernel<0>, dim3(grid), dim3(256), 0, stream, w, int(rows), nb, xq, xs, T, isum);
    return launch_pdl(block_dots_kernel<1>, dim3(grid), dim3(256), 0, stream, w, int(rows), nb, xq, xs, T, isum);
}

}  // namespace strata
