// gemm_dequant.cu — the dense prompt-chunk GEMM of a Q4 matrix in its "wide dequant" arm.
//
// The Strata pull request "sm_80 (GA100) tuning" (commit message on STRATA_DEQUANT_WIDE) runs the
// prompt path by dequantizing the dense quantized weights once per prompt chunk and then multiplying
// (857 -> 792 ms for a 3,259-token prompt there). This arm keeps that structure and the exactness of
// the no-dequant arm (strata_gemm_q4):
//   1. a conversion pass writes the weight codes q - 8 and the activation codes x as fp16 (exact) in
//      8 KB tiles of 128 rows x 32 values (one quant block), already in the K-major core-matrix order
//      the tensor cores read from shared memory, plus the matching 128-value vectors of d_w and d_x;
//   2. a persistent tcgen05 GEMM streams those tiles with bulk copies (one producer thread, no
//      per-thread gathers or conversions), runs two K = 16 kind::f16 MMAs per quant block into its own
//      TMEM accumulator, and the epilogue warps fold acc += (d_x * d_w) * isum in fp32, block by
//      block, exactly as the no-dequant arm does. The two arms give bitwise equal outputs.
// The price is the converted operands' traffic (fp16: 4x the Q4 weight bytes, 2x the int8
// activation bytes), written once per call and then read from L2 by every tile that needs them.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace strata {

namespace {

constexpr int kEpiWarps = 8;
constexpr int kProdWarp = kEpiWarps;      // one warp, lane 0 issues the bulk copies
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = (kEpiWarps + 2) * 32;
constexpr int kStages = 8;  // operand stages (A 8 KB + B 8 KB)
constexpr int kAcc = 4;     // TMEM accumulators, 128 fp32 columns each (all 512 columns)
constexpr int kScale = 8;   // scale slots (d_x 128 floats | d_w 128 floats)
constexpr int kTile = 8192; // bytes of one 128 x 32 fp16 operand tile
constexpr int kOffScale = kStages * 2 * kTile;
constexpr int kOffBars = kOffScale + kScale * 1024;
constexpr int kSmem = kOffBars + 512;
constexpr int kTmemCols = kAcc * 128 < 32 ? 32 : kAcc * 128;

// byte offset of element (r, k) of a 128-row x 32-value K-major fp16 tile: 8 x 8 core matrices of
// 128 contiguous bytes, adjacent along K at 128 bytes, along rows at 512 bytes
__device__ __forceinline__ int tile_elem_off(int r, int k) { return (r >> 3) * 512 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2; }

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// one thread per (weight row, quant block): the block's 32 codes q - 8 as fp16 into its tile, d_w
__global__ void __launch_bounds__(256) dequant_weights_kernel(const uint8_t* __restrict__ W, int rows, int kb,
                                                              uint8_t* __restrict__ tiles, float* __restrict__ dws)
{
    pdl_wait();
    pdl_launch();
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= int64_t(rows) * kb) return;
    const int r = int(i % rows), b = int(i / rows);  // consecutive threads: consecutive rows of a block
    const uint4 w = *reinterpret_cast<const uint4*>(W + (size_t(r) * kb + b) * 16);
    const unsigned short dbits = *reinterpret_cast<const unsigned short*>(W + size_t(rows) * kb * 16 + (size_t(r) * kb + b) * 2);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    uint8_t* tile = tiles + (size_t(r >> 7) * kb + b) * kTile;
    const int rt = r & 127;
    // elements 8c .. 8c+7: c < 2 low nibbles of bytes 8c.., c >= 2 high nibbles of bytes 8(c-2)..
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t lo = ww[(2 * c) & 3], hi = ww[(2 * c + 1) & 3];
        const int sh = c < 2 ? 0 : 4;
        float v[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[e] = float(int((lo >> (8 * e + sh)) & 15u) - 8);
            v[4 + e] = float(int((hi >> (8 * e + sh)) & 15u) - 8);
        }
        *reinterpret_cast<uint4*>(tile + tile_elem_off(rt, 8 * c)) =
            make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
    }
    dws[(size_t(r >> 7) * kb + b) * 128 + rt] = __half2float(__ushort_as_half(dbits));
}

// one thread per (activation row of the padded chunk, quant block): the 32 codes as fp16, d_x; rows
// past n_tok are zero
__global__ void __launch_bounds__(256) dequant_acts_kernel(const int8_t* __restrict__ xq, const float* __restrict__ xd,
                                                           int n_tok, int m_pad, int kb, uint8_t* __restrict__ tiles,
                                                           float* __restrict__ dxs)
{
    pdl_wait();
    pdl_launch();
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= int64_t(m_pad) * kb) return;
    const int r = int(i % m_pad), b = int(i / m_pad);
    const bool valid = r < n_tok;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    float d = 0.0f;
    if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(xq + size_t(r) * kb * 32 + size_t(b) * 32);
        lo = src[0];
        hi = src[1];
        d = xd[size_t(r) * kb + b];
    }
    const uint32_t xw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint8_t* tile = tiles + (size_t(r >> 7) * kb + b) * kTile;
    const int rt = r & 127;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = float(int(int8_t((xw[2 * c + (e >> 2)] >> (8 * (e & 3))) & 0xFFu)));
        *reinterpret_cast<uint4*>(tile + tile_elem_off(rt, 8 * c)) =
            make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
    }
    dxs[(size_t(r >> 7) * kb + b) * 128 + rt] = d;
}

struct PreArgs {
    const uint8_t* wt;   // weight tiles [NT][KB][8 KB]
    const float* dws;    // [NT][KB][128]
    const uint8_t* xt;   // activation tiles [MT][KB][8 KB]
    const float* dxs;    // [MT][KB][128]
    float* y;            // [n_tok][rows]
    int n_tok, rows, kb, mt, nt;
};

__global__ void __launch_bounds__(kThreads, 1) gemm_dequant_kernel(const PreArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ volatile int s_abort;
    __shared__ uint32_t s_tmem;

    pdl_wait();  // the converted operands come from the conversion kernels just ahead
    pdl_launch();
    const int total = a.mt * a.nt;
    if (int(blockIdx.x) >= total) return;
    const int KB = a.kb, NT = a.nt;

    uint8_t* stage = smem;                                        // [kStages][A 8 KB | B 8 KB]
    float* sscale = reinterpret_cast<float*>(smem + kOffScale);   // [kScale][d_x 128 | d_w 128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* full = bars;                 // [kStages] operands landed (bulk copies)
    uint64_t* empty = full + kStages;      // [kStages] MMAs done reading (commit)
    uint64_t* tfull = empty + kStages;     // [kAcc] block accumulator ready (commit)
    uint64_t* tempty = tfull + kAcc;       // [kAcc] accumulator read out (epilogue warps)
    uint64_t* sfull = tempty + kAcc;       // [kScale] scales landed (bulk copies)
    uint64_t* sempty = sfull + kScale;     // [kScale] scales read (epilogue warps)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(smem_u32(&tfull[i]), 1);
            mbar_init(smem_u32(&tempty[i]), kEpiWarps);
        }
        for (int i = 0; i < kScale; ++i) {
            mbar_init(smem_u32(&sfull[i]), 1);
            mbar_init(smem_u32(&sempty[i]), kEpiWarps);
        }
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s_tmem;

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ producer (one thread)
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int g = 0;
            bool run = true;
            for (int t = blockIdx.x; t < total && run; t += gridDim.x) {
                const int u = t / NT, nt = t - (t / NT) * NT;
                for (int b = 0; b < KB; ++b, ++g) {
                    const int s = g % kStages, ss = g % kScale;
                    if (g >= kStages && !mbar_wait(smem_u32(&empty[s]), ((g / kStages) - 1) & 1, &s_abort)) {
                        run = false;
                        break;
                    }
                    const uint32_t fs = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fs, 2 * kTile);
                    bulk_g2s(smem_u32(stage + s * 2 * kTile), a.xt + (size_t(u) * KB + b) * kTile, kTile, fs, pol);
                    bulk_g2s(smem_u32(stage + s * 2 * kTile + kTile), a.wt + (size_t(nt) * KB + b) * kTile, kTile, fs, pol);
                    if (g >= kScale && !mbar_wait(smem_u32(&sempty[ss]), ((g / kScale) - 1) & 1, &s_abort)) {
                        run = false;
                        break;
                    }
                    const uint32_t fsc = smem_u32(&sfull[ss]);
                    mbar_arrive_expect_tx(fsc, 1024);
                    bulk_g2s(smem_u32(sscale + ss * 256), a.dxs + (size_t(u) * KB + b) * 128, 512, fsc, pol);
                    bulk_g2s(smem_u32(sscale + ss * 256 + 128), a.dws + (size_t(nt) * KB + b) * 128, 512, fsc, pol);
                }
            }
            if (!run) {
                s_abort = 1;
                atomicOr(&g_strata_device_error, 1);
            }
            // no copy may still be landing when the CTA ends: wait (bounded) for the last stages and
            // scale slots issued, even after an abort
            const int no_abort = 0;
            for (int i = (g > kStages ? g - kStages : 0); i < g; ++i)
                mbar_wait(smem_u32(&full[i % kStages]), (i / kStages) & 1, &no_abort);
            for (int i = (g > kScale ? g - kScale : 0); i < g; ++i)
                mbar_wait(smem_u32(&sfull[i % kScale]), (i / kScale) & 1, &no_abort);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, 128);
            int g = 0;
            bool run = true;
            for (int t = blockIdx.x; t < total && run; t += gridDim.x) {
                for (int b = 0; b < KB; ++b) {
                    const int s = g % kStages, buf = g % kAcc;
                    if (!mbar_wait(smem_u32(&full[s]), (g / kStages) & 1, &s_abort) ||
                        (g >= kAcc && !mbar_wait(smem_u32(&tempty[buf]), ((g / kAcc) - 1) & 1, &s_abort))) {
                        run = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t As = smem_u32(stage + s * 2 * kTile), Bs = As + kTile;
                    const uint32_t d = tbase + buf * 128;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        tc_mma_f16(d, smem_desc_kmajor(As + kk * 256, 128, 512), smem_desc_kmajor(Bs + kk * 256, 128, 512),
                                   idesc, kk);
                    tc_commit(smem_u32(&empty[s]));
                    tc_commit(smem_u32(&tfull[buf]));
                    ++g;
                }
            }
            if (!run) {
                s_abort = 1;
                atomicOr(&g_strata_device_error, 1);
            }
            if (g > 0) {  // the accumulators must be idle before the TMEM is released
                const int gl = g - 1;
                const int no_abort = 0;
                mbar_wait(smem_u32(&tfull[gl % kAcc]), (gl / kAcc) & 1, &no_abort);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-7)
        const int sp = warp & 3, cg = warp >> 2;
        const int m = sp * 32 + lane;  // tile row of this thread; columns 64*cg .. 64*cg + 63
        const uint32_t tl = tbase + (uint32_t(sp * 32) << 16);
        bool ok = true;
        int g = 0;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const int u = t / NT, nt = t - (t / NT) * NT;
            f32x2 acc2[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) acc2[q] = 0ull;
            for (int b = 0; b < KB; ++b, ++g) {
                const int buf = g % kAcc, ss = g % kScale;
                ok = mbar_wait(smem_u32(&tfull[buf]), (g / kAcc) & 1, &s_abort) &&
                     mbar_wait(smem_u32(&sfull[ss]), (g / kScale) & 1, &s_abort);
                if (!ok) break;
                tc_fence_after();
                const float* sl = sscale + ss * 256;
                const float dx = sl[m];
                const f32x2 dx2 = pack_f2(dx, dx);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c0 = 64 * cg + 32 * half;
                    uint32_t v[2][16];
                    tmem_ld32(tl + buf * 128 + c0, v);
#pragma unroll
                    for (int q16 = 0; q16 < 2; ++q16) {
                        const float4* dw4 = reinterpret_cast<const float4*>(sl + 128 + c0 + 16 * q16);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 dw = dw4[q];
                            f32x2& a0 = acc2[16 * half + 8 * q16 + 2 * q];
                            f32x2& a1 = acc2[16 * half + 8 * q16 + 2 * q + 1];
                            // acc += (d_x * d_w) * isum, each half one IEEE op (the no-dequant arm's order)
                            a0 = fma_f2(mul_f2(dx2, pack_f2(dw.x, dw.y)),
                                        pack_f2(__uint_as_float(v[q16][4 * q]), __uint_as_float(v[q16][4 * q + 1])), a0);
                            a1 = fma_f2(mul_f2(dx2, pack_f2(dw.z, dw.w)),
                                        pack_f2(__uint_as_float(v[q16][4 * q + 2]), __uint_as_float(v[q16][4 * q + 3])), a1);
                        }
                    }
                }
                tc_fence_before();
                // The scale slot was read with generic loads and its next fill is an async-proxy bulk
                // copy: without a cross-proxy fence the release below orders only generic accesses,
                // and loads still in flight could see the next fill's d_w (the last columns a warp
                // reads went wrong that way).
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&tempty[buf]));
                    mbar_arrive(smem_u32(&sempty[ss]));
                }
            }
            if (!ok) break;
            const int row = u * 128 + m;
            if (row < a.n_tok) {
                float4* dst = reinterpret_cast<float4*>(a.y + size_t(row) * a.rows + nt * 128 + 64 * cg);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float x0, x1, x2, x3;
                    unpack_f2(acc2[2 * j], x0, x1);
                    unpack_f2(acc2[2 * j + 1], x2, x3);
                    dst[j] = make_float4(x0, x1, x2, x3);
                }
            }
        }
        if (!ok) {
            s_abort = 1;
            atomicOr(&g_strata_device_error, 1);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

cudaError_t read_device_error_gemm(int* out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_strata_device_error, sizeof(int));
    if (e != cudaSuccess || !clear) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_strata_device_error, &zero, sizeof(int));
}

// workspace: weight tiles + d_w vectors, activation tiles + d_x vectors (each section 256-byte aligned)
size_t gemm_dequant_workspace_bytes(int64_t rows, int64_t cols, int64_t n_tok)
{
    const size_t kb = size_t(cols / 32), nt = size_t(rows / 128), mt = size_t((n_tok + 127) / 128);
    return al256(nt * kb * kTile) + al256(nt * kb * 512) + al256(mt * kb * kTile) + al256(mt * kb * 512);
}

cudaError_t launch_gemm_dequant(const void* W, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                                int64_t n_tok, float* y, void* workspace, cudaStream_t stream)
{
    const int kb = int(cols / 32), nt = int(rows / 128), mt = int((n_tok + 127) / 128);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint8_t* wt = ws;
    float* dws = reinterpret_cast<float*>(ws + al256(size_t(nt) * kb * kTile));
    uint8_t* xt = reinterpret_cast<uint8_t*>(dws) + al256(size_t(nt) * kb * 512);
    float* dxs = reinterpret_cast<float*>(xt + al256(size_t(mt) * kb * kTile));
    const int64_t nw = rows * kb, na = int64_t(mt) * 128 * kb;
    cudaError_t e = launch_pdl(dequant_weights_kernel, dim3(unsigned((nw + 255) / 256)), dim3(256), 0, stream,
                               static_cast<const uint8_t*>(W), int(rows), kb, wt, dws);
    if (e != cudaSuccess) return e;
    e = launch_pdl(dequant_acts_kernel, dim3(unsigned((na + 255) / 256)), dim3(256), 0, stream, xq, xd, int(n_tok),
                   mt * 128, kb, xt, dxs);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_dequant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    PreArgs a;
    a.wt = wt;
    a.dws = dws;
    a.xt = xt;
    a.dxs = dxs;
    a.y = y;
    a.n_tok = int(n_tok);
    a.rows = int(rows);
    a.kb = kb;
    a.mt = mt;
    a.nt = nt;
    const int grid = int(std::min<int64_t>(int64_t(mt) * nt, device_sm_count()));
    return launch_pdl(gemm_dequant_kernel, dim3(unsigned(grid)), dim3(kThreads), size_t(kSmem), stream, a);
}

}  // namespace strata
