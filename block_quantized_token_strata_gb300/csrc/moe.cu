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
#include "tc.cuh"

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
    L.mcum = o;    o = al256(o + size_t(n_expert + 1) * 4);
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

// ---- grouped expert GEMMs on the tensor cores ------------------------------------------------------
//
// One CTA computes one tile: 128 pair positions of one expert (an M-tile of its grouped rows) against
// an N-tile of weight rows, over the whole K extent, one 32-wide quant block at a time:
//   gate/up phase: K = hidden, N-tile = 64 inter columns of W_gate and the same 64 of W_up;
//                  epilogue h = silu(g)*u, re-quantized per 32 columns, written by pair position;
//   down phase:    K = inter (A = the re-quantized h), N-tile = 128 rows of W_down;
//                  epilogue scatters row p = pairs[position] of y.
// Exactness: the codes (activation q in -127..127, weight q-8 in -8..7) are exact fp16 values,
// every product and every 32-term sum is an exact integer below 2^24, so one kind::f16 MMA pair
// (K = 16 + 16) with fp32 accumulation yields the exact integer block dot isum for all 128 x N
// outputs. Each quant block gets its own TMEM accumulator (two buffers, alternating), and the
// epilogue folds y += (d_x * d_w) * isum in fp32 — the block arithmetic of the GEMV.
// Roles: warps 0-7 epilogue (warp w reads TMEM lanes 32*(w%4).. = tile rows, column half w/4),
// warps 8-11 convert codes to fp16 in the K-major core-matrix layout the MMA reads (one tile row and
// one weight row per thread) and stage the block's scales, warp 12 owns TMEM and issues the MMAs.
// Every wait is bounded; a timeout sets bit 0 of the device error word and the CTA winds down.

constexpr int kTcEpiWarps = 8;
constexpr int kTcCvtWarps = 4;
constexpr int kTcMmaWarp = kTcEpiWarps + kTcCvtWarps;
constexpr int kTcThreads = (kTcEpiWarps + kTcCvtWarps + 1) * 32;
constexpr int kTcStages = 3;    // fp16 operand stages (A 8 KB + B 8 KB each)
constexpr int kTcScale = 4;     // scale slots (d_x per tile row, d_w per weight row)
constexpr int kTcTmemCols = 256;
constexpr int kTcSmem = kTcStages * 16384 + kTcScale * 1024 + 512;

extern __device__ int g_strata_device_error;

struct MoeTcArgs {
    const ExpertPtrs* experts;
    int n_expert, hidden, inter, k;
    const int32_t* pairs;
    const int32_t* offsets;
    const int32_t* counts;
    const int32_t* mcum;       // [n_expert+1] running count of 128-row M-tiles
    const int8_t* xq;          // gate/up: activations by token
    const float* xd;
    int8_t* hq;                // hidden rows by pair position (written by gate/up, read by down)
    float* hd;
    int32_t* hs;
    float* y;
};

// byte offset of row r, 8-element column group c in a 128-row x 32-element K-major fp16 tile
__device__ __forceinline__ int tile_off(int r, int c) { return (r >> 3) * 512 + c * 128 + (r & 7) * 16; }

template <int PHASE>
__global__ void __launch_bounds__(kTcThreads, 1) moe_tc_kernel(const MoeTcArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ volatile int s_abort;
    __shared__ uint32_t s_tmem;

    pdl_wait();  // the grouping, the tile counts and the activations come from the kernels ahead
    pdl_launch();
    const int NT = PHASE == 0 ? a.inter / 64 : a.hidden / 128;
    const int total = a.mcum[a.n_expert] * NT;
    const int t = blockIdx.x;
    if (t >= total) return;
    const int u = t / NT, nt = t - (t / NT) * NT;
    int e = 0;
    {
        int lo = 0, hi = a.n_expert;  // largest e with mcum[e] <= u
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (a.mcum[mid] <= u) lo = mid; else hi = mid;
        }
        e = lo;
    }
    const int mt = u - a.mcum[e];
    const int m0 = a.offsets[e] + mt * 128;
    const int mvalid = min(128, a.counts[e] - mt * 128);
    const int KB = PHASE == 0 ? a.hidden / 32 : a.inter / 32;

    uint8_t* stage = smem;                                              // [kTcStages][A 8K | B 8K]
    float* sscale = reinterpret_cast<float*>(smem + kTcStages * 16384); // [kTcScale][dx 128 | dw 128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTcStages * 16384 + kTcScale * 1024);
    uint64_t* full = bars;                    // [kTcStages] operands converted (4 converter warps)
    uint64_t* empty = bars + 3;               // [kTcStages] MMAs done reading (commit)
    uint64_t* tfull = bars + 6;               // [2] block accumulator ready (commit)
    uint64_t* tempty = bars + 8;              // [2] accumulator read out (8 epilogue warps)
    uint64_t* sfull = bars + 10;              // [kTcScale] scales staged (4 converter warps)
    uint64_t* sempty = bars + 14;             // [kTcScale] scales read (8 epilogue warps)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(smem_u32(&full[i]), kTcCvtWarps);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull[i]), 1);
            mbar_init(smem_u32(&tempty[i]), kTcEpiWarps);
        }
        for (int i = 0; i < kTcScale; ++i) {
            mbar_init(smem_u32(&sfull[i]), kTcCvtWarps);
            mbar_init(smem_u32(&sempty[i]), kTcEpiWarps);
        }
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == kTcMmaWarp) {
        tmem_alloc(smem_u32(&s_tmem), kTcTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s_tmem;
    const ExpertPtrs ex = a.experts[e];

    if (warp >= kTcEpiWarps && warp < kTcMmaWarp) {
        // ------------------------------------------------------------ converters
        const int r = threadIdx.x - kTcEpiWarps * 32;  // tile row and weight row of this thread
        const int P = m0 + r;
        const bool rvalid = r < mvalid;
        const int8_t* arow;
        const float* dxrow;
        int nbk;
        if (PHASE == 0) {
            const int tok = rvalid ? a.pairs[P] / a.k : 0;
            nbk = a.hidden / 32;
            arow = a.xq + size_t(tok) * a.hidden;
            dxrow = a.xd + size_t(tok) * nbk;
        } else {
            nbk = a.inter / 32;
            arow = a.hq + size_t(rvalid ? P : 0) * a.inter;
            dxrow = a.hd + size_t(rvalid ? P : 0) * nbk;
        }
        const uint8_t* W;
        int wrow, wrows;
        if (PHASE == 0) {
            W = r < 64 ? ex.gate : ex.up;
            wrow = nt * 64 + (r & 63);
            wrows = a.inter;
        } else {
            W = ex.down;
            wrow = nt * 128 + r;
            wrows = a.hidden;
        }
        const uint4* wq = reinterpret_cast<const uint4*>(W + size_t(wrow) * nbk * 16);
        const unsigned short* wd =
            reinterpret_cast<const unsigned short*>(W + size_t(wrows) * nbk * 16) + size_t(wrow) * nbk;
        const uint4* aq = reinterpret_cast<const uint4*>(arow);

        uint4 na0 = make_uint4(0, 0, 0, 0), na1 = na0, nw = na0;
        float ndx = 0.0f;
        unsigned short ndw = 0;
        auto fetch = [&](int b) {
            if (rvalid) { na0 = __ldg(aq + 2 * b); na1 = __ldg(aq + 2 * b + 1); ndx = __ldg(dxrow + b); }
            nw = __ldg(wq + b);
            ndw = __ldg(wd + b);
        };
        fetch(0);
        const uint32_t neg1152 = 0xE480E480u, neg1032 = 0xE408E408u;  // fp16 -1152, -1032
        for (int b = 0; b < KB; ++b) {
            const uint4 a0 = na0, a1 = na1, w = nw;
            const float dx = ndx;
            const unsigned short dwb = ndw;
            if (b + 1 < KB) fetch(b + 1);
            const int s = b % kTcStages, ss = b % kTcScale;
            if (b >= kTcStages && !mbar_wait(smem_u32(&empty[s]), ((b / kTcStages) - 1) & 1, &s_abort)) break;
            if (b >= kTcScale && !mbar_wait(smem_u32(&sempty[ss]), ((b / kTcScale) - 1) & 1, &s_abort)) break;
            uint8_t* As = stage + s * 16384;
            uint8_t* Bs = As + 8192;
            // activation codes x: fp16(1152 + x) - 1152 = x, exact
            const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t t0 = aw[2 * c] ^ 0x80808080u, t1 = aw[2 * c + 1] ^ 0x80808080u;
                uint4 o;
                o.x = h2_add(bytes_to_h2(t0, 0x5140), neg1152);
                o.y = h2_add(bytes_to_h2(t0, 0x5342), neg1152);
                o.z = h2_add(bytes_to_h2(t1, 0x5140), neg1152);
                o.w = h2_add(bytes_to_h2(t1, 0x5342), neg1152);
                *reinterpret_cast<uint4*>(As + tile_off(r, c)) = o;
            }
            // weight codes q (byte j: element j low nibble, element j+16 high): fp16(1024+q) - 1032 = q-8
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t x0 = ww[(2 * c) & 3], x1 = ww[(2 * c + 1) & 3];
                const uint32_t q0 = (c < 2 ? x0 : (x0 >> 4)) & 0x0F0F0F0Fu;
                const uint32_t q1 = (c < 2 ? x1 : (x1 >> 4)) & 0x0F0F0F0Fu;
                uint4 o;
                o.x = h2_add(bytes_to_h2(q0, 0x5140), neg1032);
                o.y = h2_add(bytes_to_h2(q0, 0x5342), neg1032);
                o.z = h2_add(bytes_to_h2(q1, 0x5140), neg1032);
                o.w = h2_add(bytes_to_h2(q1, 0x5342), neg1032);
                *reinterpret_cast<uint4*>(Bs + tile_off(r, c)) = o;
            }
            float* sl = sscale + ss * 256;
            sl[r] = rvalid ? dx : 0.0f;
            sl[128 + r] = __half2float(__ushort_as_half(dwb));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&full[s]));
                mbar_arrive(smem_u32(&sfull[ss]));
            }
        }
    } else if (warp == kTcMmaWarp) {
        // ------------------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            const uint32_t idesc = PHASE == 0 ? idesc_f16_f32(128, 64) : idesc_f16_f32(128, 128);
            int issued = 0;
            for (int b = 0; b < KB; ++b) {
                const int s = b % kTcStages, buf = b & 1;
                if (!mbar_wait(smem_u32(&full[s]), (b / kTcStages) & 1, &s_abort)) break;
                if (b >= 2 && !mbar_wait(smem_u32(&tempty[buf]), ((b >> 1) - 1) & 1, &s_abort)) break;
                tc_fence_after();
                const uint32_t As = smem_u32(stage + s * 16384), Bs = As + 8192;
                const uint32_t d = tbase + buf * 128;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint64_t ad = smem_desc_kmajor(As + kk * 256, 128, 512);
                    if (PHASE == 0) {
                        tc_mma_f16(d, ad, smem_desc_kmajor(Bs + kk * 256, 128, 512), idesc, kk);
                        tc_mma_f16(d + 64, ad, smem_desc_kmajor(Bs + 4096 + kk * 256, 128, 512), idesc, kk);
                    } else {
                        tc_mma_f16(d, ad, smem_desc_kmajor(Bs + kk * 256, 128, 512), idesc, kk);
                    }
                }
                tc_commit(smem_u32(&empty[s]));
                tc_commit(smem_u32(&tfull[buf]));
                issued = b + 1;
            }
            // the accumulators must be idle before the TMEM is released: wait for the last commit
            if (issued > 0) {
                const int b = issued - 1;
                mbar_wait(smem_u32(&tfull[b & 1]), (b >> 1) & 1, &s_abort);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-7)
        const int sp = warp & 3, cg = warp >> 2;
        const int m = sp * 32 + lane;               // tile row of this thread
        const uint32_t tl = tbase + (uint32_t(sp * 32) << 16);
        float acc[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
        bool ok = true;
        for (int b = 0; b < KB; ++b) {
            const int buf = b & 1, ss = b % kTcScale;
            ok = mbar_wait(smem_u32(&tfull[buf]), (b >> 1) & 1, &s_abort) &&
                 mbar_wait(smem_u32(&sfull[ss]), (b / kTcScale) & 1, &s_abort);
            if (!ok) break;
            tc_fence_after();
            const float* sl = sscale + ss * 256;
            const float dx = sl[m];
            // two halves of 32 columns: gate/up phase = the 32 gate then the 32 up columns of this
            // warp's inter range; down phase = 64 consecutive columns
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int c0 = PHASE == 0 ? 32 * cg + 64 * half : 64 * cg + 32 * half;  // tile column = weight row
                uint32_t v0[16], v1[16];
                tmem_ld16(tl + buf * 128 + c0, v0);
                tmem_ld16(tl + buf * 128 + c0 + 16, v1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    acc[32 * half + j] = __fmaf_rn(__fmul_rn(dx, sl[128 + c0 + j]), __uint_as_float(v0[j]),
                                                   acc[32 * half + j]);
                    acc[32 * half + 16 + j] = __fmaf_rn(__fmul_rn(dx, sl[128 + c0 + 16 + j]),
                                                        __uint_as_float(v1[j]), acc[32 * half + 16 + j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&tempty[buf]));
                mbar_arrive(smem_u32(&sempty[ss]));
            }
        }
        if (!ok) {
            s_abort = 1;
            atomicOr(&g_strata_device_error, 1);
        } else if (m < mvalid) {
            const int P = m0 + m;
            if (PHASE == 0) {
                // h = silu(g) * u for the 32 inter columns nt*64 + 32*cg + j, then one quant block
                float h[32];
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float g = acc[j], uu = acc[32 + j];
                    h[j] = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), uu);
                    amax = fmaxf(amax, fabsf(h[j]));
                }
                const float d = __fdiv_rn(amax, 127.0f);
                const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
                int sum = 0;
                uint32_t packed[8];
#pragma unroll
                for (int w4 = 0; w4 < 8; ++w4) {
                    uint32_t word = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int q = int(roundf(__fmul_rn(h[4 * w4 + i], id)));
                        sum += q;
                        word |= uint32_t(q & 0xFF) << (8 * i);
                    }
                    packed[w4] = word;
                }
                const int col0 = nt * 64 + 32 * cg;
                uint4* dst = reinterpret_cast<uint4*>(a.hq + size_t(P) * a.inter + col0);
                dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                a.hd[size_t(P) * (a.inter / 32) + col0 / 32] = d;
                a.hs[size_t(P) * (a.inter / 32) + col0 / 32] = sum;
            } else {
                const int prow = a.pairs[P];
                float4* dst = reinterpret_cast<float4*>(a.y + size_t(prow) * a.hidden + nt * 128 + 64 * cg);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    dst[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTcTmemCols);
    }
}

// running count of 128-row M-tiles per expert (one small CTA)
__global__ void moe_tiles_kernel(const int32_t* __restrict__ counts, int n_expert, int32_t* __restrict__ mcum)
{
    pdl_wait();
    pdl_launch();
    if (threadIdx.x == 0) {
        int acc = 0;
        mcum[0] = 0;
        for (int e = 0; e < n_expert; ++e) {
            acc += (counts[e] + 127) / 128;
            mcum[e + 1] = acc;
        }
    }
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
    int32_t* mcum = reinterpret_cast<int32_t*>(ws + L.mcum);
    const ExpertPtrs* ex = static_cast<const ExpertPtrs*>(experts);

    cudaError_t e = launch_quantize_act(x, n_tok, hidden, xq, xd, xs, stream);
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_bucket_kernel, dim3(n_expert), dim3(256), 0, stream, ids, n_pair, n_expert, counts,
                   offsets, pairs, err_word);
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_tiles_kernel, dim3(1), dim3(32), 0, stream, (const int32_t*)counts, n_expert, mcum);
    if (e != cudaSuccess) return e;

    MoeTcArgs a;
    a.experts = ex;
    a.n_expert = n_expert;
    a.hidden = int(hidden);
    a.inter = int(inter);
    a.k = k;
    a.pairs = pairs;
    a.offsets = offsets;
    a.counts = counts;
    a.mcum = mcum;
    a.xq = xq;
    a.xd = xd;
    a.hq = hq;
    a.hd = hd;
    a.hs = hs;
    a.y = y;
    // enough CTAs for any grouping: at most n_pair/128 + n_expert M-tiles
    const int max_mtiles = (n_pair + 127) / 128 + n_expert;
    e = cudaFuncSetAttribute(moe_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(moe_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_tc_kernel<0>, dim3(unsigned(max_mtiles * (inter / 64))), dim3(kTcThreads), kTcSmem,
                   stream, a);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_tc_kernel<1>, dim3(unsigned(max_mtiles * (hidden / 128))), dim3(kTcThreads), kTcSmem,
                      stream, a);
}

}  // namespace strata
