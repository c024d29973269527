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

#include <algorithm>

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
// A tile is 128 pair positions of one expert (an M-tile of its grouped rows) against an N-tile of
// weight rows, over the whole K extent, one 32-wide quant block at a time:
//   gate/up phase: K = hidden, N-tile = 64 inter columns of W_gate and the same 64 of W_up;
//                  epilogue h = silu(g)*u, re-quantized per 32 columns, written by pair position;
//   down phase:    K = inter (A = the re-quantized h), N-tile = 128 rows of W_down;
//                  epilogue scatters row p = pairs[position] of y.
// Exactness: the codes (activation q in -127..127, weight q-8 in -8..7) are exact fp16 values,
// every product and every 32-term sum is an exact integer below 2^24, so one kind::f16 MMA pair
// (K = 16 + 16) with fp32 accumulation yields the exact integer block dot isum for all 128 x N
// outputs. Each quant block gets its own TMEM accumulator (four 128-column buffers in turn), and
// the epilogue folds y += (d_x * d_w) * isum in fp32 — the block arithmetic of the GEMV.
// The kernel is persistent: CTA c takes tiles c, c + grid, ... and every role walks the same
// sequence of (tile, block) steps with one running step counter g, so the rings run on across
// tile boundaries (the MMAs of the next tile start while the epilogue finishes the last).
// Roles: warps 0-7 epilogue (warp w reads TMEM lanes 32*(w%4).. = tile rows, column half w/4);
// warps 8-11 convert (one tile row and one weight row per thread): each thread keeps its own
// raw codes kTcRaw steps ahead in shared memory with cp.async, then writes the fp16 operands in the
// K-major core-matrix layout the MMA reads and stages the block's scales; warp 12 owns TMEM and
// issues the MMAs. Every wait is bounded; a timeout sets bit 0 of the device error word and the
// CTA winds down.

constexpr int kTcEpiWarps = 8;
constexpr int kTcCvtWarps = 4;
constexpr int kTcMmaWarp = kTcEpiWarps + kTcCvtWarps;
constexpr int kTcThreads = (kTcEpiWarps + kTcCvtWarps + 1) * 32;
constexpr int kTcStages = 4;      // fp16 operand stages (A 8 KB + B 8 KB each)
constexpr int kTcAcc = 4;         // TMEM accumulators, 128 fp32 columns each
constexpr int kTcScale = 8;       // scale slots (d_x per tile row, d_w per weight row), 1 KB each
constexpr int kTcRaw = 8;         // raw-code ring depth per converter thread (steps loaded ahead)
// raw slot: activation bytes 0-15 | 16-31 | weight 16 bytes (each 128 rows x 16 B) | d_x | d_w word
constexpr int kTcRawA0 = 0, kTcRawA1 = 2048, kTcRawW = 4096, kTcRawDx = 6144, kTcRawDw = 6656;
constexpr int kTcRawSlot = 7168;
constexpr int kTcTmemCols = kTcAcc * 128;
constexpr int kTcOffScale = kTcStages * 16384;
constexpr int kTcOffRaw = kTcOffScale + kTcScale * 1024;
constexpr int kTcOffBars = kTcOffRaw + kTcRaw * kTcRawSlot;
constexpr int kTcSmem = kTcOffBars + 512;


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
    float* gu;                 // test hook (null in the product call): fp32 [n_pair][2][inter], g then u by pair
    // dense prompt GEMM (down-phase kernel only): the one Q4 matrix [hidden][inter] and the number of
    // activation rows; tiles then cover rows 0.. in order and row m of the output is y row m
    const uint8_t* dense_w;
    int dense_rows;
};

// byte offset of row r, 8-element column group c in a 128-row x 32-element K-major fp16 tile
__device__ __forceinline__ int tile_off(int r, int c) { return (r >> 3) * 512 + c * 128 + (r & 7) * 16; }

struct TcTile {
    int e;       // expert
    int m0;      // first pair position of the M-tile
    int mvalid;  // valid rows of the M-tile (1..128)
    int nt;      // N-tile
};

// tile t = u * NT + nt, u the running M-tile index over experts (mcum is its prefix count); the
// small tables it reads are shared by every thread of the CTA and stay in L1
__device__ __forceinline__ TcTile tc_tile(const MoeTcArgs& a, int t, int NT)
{
    TcTile tl;
    const int u = t / NT;
    tl.nt = t - u * NT;
    if (a.dense_w) {
        tl.e = 0;
        tl.m0 = u * 128;
        tl.mvalid = min(128, a.dense_rows - u * 128);
        return tl;
    }
    int lo = 0, hi = a.n_expert;  // largest e with mcum[e] <= u
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.mcum + mid) <= u) lo = mid; else hi = mid;
    }
    tl.e = lo;
    const int mt = u - __ldg(a.mcum + lo);
    tl.m0 = __ldg(a.offsets + lo) + mt * 128;
    tl.mvalid = min(128, __ldg(a.counts + lo) - mt * 128);
    return tl;
}

template <int PHASE>
__global__ void __launch_bounds__(kTcThreads, 1) moe_tc_kernel(const MoeTcArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ volatile int s_abort;
    __shared__ uint32_t s_tmem;

    pdl_wait();  // the grouping, the tile counts and the activations come from the kernels ahead
    pdl_launch();
    const int NT = PHASE == 0 ? a.inter / 64 : a.hidden / 128;
    const int total = (a.dense_w ? (a.dense_rows + 127) / 128 : a.mcum[a.n_expert]) * NT;
    if (int(blockIdx.x) >= total) return;
    const int KB = PHASE == 0 ? a.hidden / 32 : a.inter / 32;

    uint8_t* stage = smem;                                          // [kTcStages][A 8K | B 8K]
    float* sscale = reinterpret_cast<float*>(smem + kTcOffScale);   // [kTcScale][dx 128 | dw 128]
    uint8_t* raw = smem + kTcOffRaw;                                // [kTcRaw][kTcRawSlot]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTcOffBars);
    uint64_t* full = bars;                               // [kTcStages] operands converted (converter warps)
    uint64_t* empty = full + kTcStages;                  // [kTcStages] MMAs done reading (commit)
    uint64_t* tfull = empty + kTcStages;                 // [kTcAcc] block accumulator ready (commit)
    uint64_t* tempty = tfull + kTcAcc;                   // [kTcAcc] accumulator read out (epilogue warps)
    uint64_t* sfull = tempty + kTcAcc;                   // [kTcScale] scales staged (converter warps)
    uint64_t* sempty = sfull + kTcScale;                 // [kTcScale] scales read (epilogue warps)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(smem_u32(&full[i]), kTcCvtWarps);
            mbar_init(smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < kTcAcc; ++i) {
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

    if (warp >= kTcEpiWarps && warp < kTcMmaWarp) {
        // ------------------------------------------------------------ converters
        const int r = threadIdx.x - kTcEpiWarps * 32;  // tile row and weight row of this thread
        const int nbk = KB;                            // quant blocks per A row and per weight row
        // issue cursor: the (tile, block) step whose raw codes this thread loads next
        int it = blockIdx.x, ib = 0;
        const int8_t* i_arow = nullptr;
        const float* i_dxrow = nullptr;
        const uint8_t* i_wq = nullptr;
        const uint16_t* i_wd = nullptr;
        uint32_t i_abytes = 0;  // 16 for a valid tile row, 0 (zero fill) past the tile's rows
        // gate/up phase: the token of this thread's row in tile `it`, loaded one tile ahead so that
        // the gather address is ready when the issue cursor reaches the tile
        int tok_next = 0;
        auto row_pos = [&](int t) {
            const TcTile tl = tc_tile(a, t, NT);
            return tl.m0 + (r < tl.mvalid ? r : 0);
        };
        if (PHASE == 0 && it < total) tok_next = __ldg(a.pairs + row_pos(it)) / a.k;
        auto seek = [&]() {
            if (it >= total) return;
            const TcTile tl = tc_tile(a, it, NT);
            const ExpertPtrs ex = a.dense_w ? ExpertPtrs{nullptr, nullptr, a.dense_w} : a.experts[tl.e];
            const bool rvalid = r < tl.mvalid;
            const int P = tl.m0 + (rvalid ? r : 0);
            if (PHASE == 0) {
                const int tok = tok_next;
                if (it + int(gridDim.x) < total) tok_next = __ldg(a.pairs + row_pos(it + gridDim.x)) / a.k;
                i_arow = a.xq + size_t(tok) * a.hidden;
                i_dxrow = a.xd + size_t(tok) * nbk;
            } else {
                i_arow = a.hq + size_t(P) * a.inter;
                i_dxrow = a.hd + size_t(P) * nbk;
            }
            i_abytes = rvalid ? 16u : 0u;
            const uint8_t* W;
            int wrow, wrows;
            if (PHASE == 0) {
                W = r < 64 ? ex.gate : ex.up;
                wrow = tl.nt * 64 + (r & 63);
                wrows = a.inter;
            } else {
                W = ex.down;
                wrow = tl.nt * 128 + r;
                wrows = a.hidden;
            }
            i_wq = W + size_t(wrow) * nbk * 16;
            i_wd = reinterpret_cast<const uint16_t*>(W + size_t(wrows) * nbk * 16) + size_t(wrow) * nbk;
        };
        // one commit group per step (empty past the last tile, so that the group count stays uniform)
        auto issue = [&](int slot) {
            if (it < total) {
                const uint32_t rs = smem_u32(raw + slot * kTcRawSlot);
                cp_async16(rs + kTcRawA0 + r * 16, i_arow + ib * 32, i_abytes);
                cp_async16(rs + kTcRawA1 + r * 16, i_arow + ib * 32 + 16, i_abytes);
                cp_async16(rs + kTcRawW + r * 16, i_wq + ib * 16, 16u);
                cp_async4(rs + kTcRawDx + r * 4, i_dxrow + ib, i_abytes >> 2);
                // the aligned 32-bit word holding d_w of block ib (a row holds an even number of blocks)
                cp_async4(rs + kTcRawDw + r * 4, i_wd + (ib & ~1), 4u);
                if (++ib == KB) {
                    ib = 0;
                    it += gridDim.x;
                    seek();
                }
            }
            cp_async_commit();
        };
        seek();
#pragma unroll 1
        for (int i = 0; i < kTcRaw - 1; ++i) issue(i);

        const uint32_t neg1152 = 0xE480E480u, neg1032 = 0xE408E408u;  // fp16 -1152, -1032
        bool run = true;
        int g = 0;
        for (int t = blockIdx.x; t < total && run; t += gridDim.x) {
            for (int b = 0; b < KB; ++b, ++g) {
                issue((g + kTcRaw - 1) % kTcRaw);
                cp_async_wait<kTcRaw - 1>();  // step g's raw codes have landed (this thread's own copies)
                const uint8_t* rs = raw + (g % kTcRaw) * kTcRawSlot;
                const uint4 a0 = *reinterpret_cast<const uint4*>(rs + kTcRawA0 + r * 16);
                const uint4 a1 = *reinterpret_cast<const uint4*>(rs + kTcRawA1 + r * 16);
                const uint4 w = *reinterpret_cast<const uint4*>(rs + kTcRawW + r * 16);
                const float dx = *reinterpret_cast<const float*>(rs + kTcRawDx + r * 4);
                const uint32_t dww = *reinterpret_cast<const uint32_t*>(rs + kTcRawDw + r * 4);
                const unsigned short dwb = (unsigned short)((b & 1) ? (dww >> 16) : (dww & 0xFFFFu));

                const int s = g % kTcStages, ss = g % kTcScale;
                if (g >= kTcStages && !mbar_wait(smem_u32(&empty[s]), ((g / kTcStages) - 1) & 1, &s_abort)) {
                    run = false;
                    break;
                }
                if (g >= kTcScale && !mbar_wait(smem_u32(&sempty[ss]), ((g / kTcScale) - 1) & 1, &s_abort)) {
                    run = false;
                    break;
                }
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
                sl[r] = dx;  // zero past the tile's rows (zero-filled copy)
                sl[128 + r] = __half2float(__ushort_as_half(dwb));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&full[s]));
                    mbar_arrive(smem_u32(&sfull[ss]));
                }
            }
        }
        cp_async_wait<0>();  // no copy of this thread is left in flight when the CTA ends
    } else if (warp == kTcMmaWarp) {
        // ------------------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            const uint32_t idesc = PHASE == 0 ? idesc_f16_f32(128, 64) : idesc_f16_f32(128, 128);
            int g = 0;
            bool run = true;
            for (int t = blockIdx.x; t < total && run; t += gridDim.x) {
                for (int b = 0; b < KB; ++b) {
                    const int s = g % kTcStages, buf = g % kTcAcc;
                    if (!mbar_wait(smem_u32(&full[s]), (g / kTcStages) & 1, &s_abort) ||
                        (g >= kTcAcc && !mbar_wait(smem_u32(&tempty[buf]), ((g / kTcAcc) - 1) & 1, &s_abort))) {
                        run = false;
                        break;
                    }
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
                    ++g;
                }
            }
            // the accumulators must be idle before the TMEM is released: wait for the last commit
            // (its phase is the newest of that barrier, so the parity cannot alias; bounded in time)
            if (g > 0) {
                const int gl = g - 1;
                const int no_abort = 0;
                mbar_wait(smem_u32(&tfull[gl % kTcAcc]), (gl / kTcAcc) & 1, &no_abort);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-7)
        const int sp = warp & 3, cg = warp >> 2;
        const int m = sp * 32 + lane;               // tile row of this thread
        const uint32_t tl = tbase + (uint32_t(sp * 32) << 16);
        bool ok = true;
        int g = 0;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TcTile tile = tc_tile(a, t, NT);
            // down phase: the output row of this thread's pair, loaded now, used after the K loop
            const int prow = (PHASE == 1 && m < tile.mvalid)
                                 ? (a.dense_w ? tile.m0 + m : __ldg(a.pairs + tile.m0 + m)) : 0;
            f32x2 acc2[32];  // acc2[q] = columns (2q, 2q+1) of this thread's 64
#pragma unroll
            for (int q = 0; q < 32; ++q) acc2[q] = 0ull;
            for (int b = 0; b < KB; ++b, ++g) {
                const int buf = g % kTcAcc, ss = g % kTcScale;
                ok = mbar_wait(smem_u32(&tfull[buf]), (g / kTcAcc) & 1, &s_abort) &&
                     mbar_wait(smem_u32(&sfull[ss]), (g / kTcScale) & 1, &s_abort);
                if (!ok) break;
                tc_fence_after();
                const float* sl = sscale + ss * 256;
                const float dx = sl[m];
                const f32x2 dx2 = pack_f2(dx, dx);
                // two halves of 32 columns: gate/up phase = the 32 gate then the 32 up columns of
                // this warp's inter range; down phase = 64 consecutive columns
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c0 = PHASE == 0 ? 32 * cg + 64 * half : 64 * cg + 32 * half;  // tile column
                    uint32_t v[2][16];  // both 16-column loads of the half in flight, one wait
                    tmem_ld32(tl + buf * 128 + c0, v);
#pragma unroll
                    for (int q16 = 0; q16 < 2; ++q16) {
                        const float4* dw4 = reinterpret_cast<const float4*>(sl + 128 + c0 + 16 * q16);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 dw = dw4[q];  // d_w of columns c0 + 16 q16 + 4q .. + 3
                            f32x2& a0 = acc2[16 * half + 8 * q16 + 2 * q];
                            f32x2& a1 = acc2[16 * half + 8 * q16 + 2 * q + 1];
                            // acc += (d_x * d_w) * isum, each half one IEEE op
                            a0 = fma_f2(mul_f2(dx2, pack_f2(dw.x, dw.y)),
                                        pack_f2(__uint_as_float(v[q16][4 * q]), __uint_as_float(v[q16][4 * q + 1])), a0);
                            a1 = fma_f2(mul_f2(dx2, pack_f2(dw.z, dw.w)),
                                        pack_f2(__uint_as_float(v[q16][4 * q + 2]), __uint_as_float(v[q16][4 * q + 3])), a1);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&tempty[buf]));
                    mbar_arrive(smem_u32(&sempty[ss]));
                }
            }
            if (!ok) break;
            if (m < tile.mvalid) {
                float acc[64];
#pragma unroll
                for (int q = 0; q < 32; ++q) unpack_f2(acc2[q], acc[2 * q], acc[2 * q + 1]);
                const int P = tile.m0 + m;
                if (PHASE == 0) {
                    if (a.gu != nullptr) {  // the fp32 gate and up outputs of this pair, as computed
                        float* gd = a.gu + size_t(__ldg(a.pairs + P)) * 2 * a.inter + tile.nt * 64 + 32 * cg;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            reinterpret_cast<float4*>(gd)[j] =
                                make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
                            reinterpret_cast<float4*>(gd + a.inter)[j] =
                                make_float4(acc[32 + 4 * j], acc[33 + 4 * j], acc[34 + 4 * j], acc[35 + 4 * j]);
                        }
                    }
                    // h = silu(g) * u for the 32 inter columns nt*64 + 32*cg + j, then one quant block
                    float h[32];
                    float amax = 0.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float gg = acc[j], uu = acc[32 + j];
                        h[j] = __fmul_rn(__fdiv_rn(gg, __fadd_rn(1.0f, expf(-gg))), uu);
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
                    const int col0 = tile.nt * 64 + 32 * cg;
                    uint4* dst = reinterpret_cast<uint4*>(a.hq + size_t(P) * a.inter + col0);
                    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    a.hd[size_t(P) * (a.inter / 32) + col0 / 32] = d;
                    a.hs[size_t(P) * (a.inter / 32) + col0 / 32] = sum;
                } else {
                    float4* dst = reinterpret_cast<float4*>(a.y + size_t(prow) * a.hidden + tile.nt * 128 + 64 * cg);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        dst[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
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
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTcTmemCols);
    }
}

cudaError_t read_device_error_moe(int* out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_strata_device_error, sizeof(int));
    if (e != cudaSuccess || !clear) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_strata_device_error, &zero, sizeof(int));
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
                               uint8_t* ws, const MoeLayout& L, int32_t* err_word, float* gu,
                               cudaStream_t stream)
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

    MoeTcArgs a = {};  // dense_w null: the grouped MoE
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
    a.gu = gu;
    // persistent: one CTA per SM, or fewer when even the largest grouping has fewer tiles
    // (at most n_pair/128 + n_expert M-tiles)
    const int max_mtiles = (n_pair + 127) / 128 + n_expert;
    const int sms = device_sm_count();
    e = cudaFuncSetAttribute(moe_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(moe_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    const int grid0 = int(std::min<int64_t>(int64_t(max_mtiles) * (inter / 64), sms));
    const int grid1 = int(std::min<int64_t>(int64_t(max_mtiles) * (hidden / 128), sms));
    e = launch_pdl(moe_tc_kernel<0>, dim3(unsigned(grid0)), dim3(kTcThreads), kTcSmem, stream, a);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_tc_kernel<1>, dim3(unsigned(grid1)), dim3(kTcThreads), kTcSmem, stream, a);
}

// Dense prompt GEMM y[n][r] = sum_b (d_w[r][b] * xd[n][b]) * isum[n][r][b] on the tensor cores: the
// down-phase kernel with one matrix and the activation rows in order (no grouping).
cudaError_t launch_prompt_gemm(const void* W, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                               int64_t n_tok, float* y, cudaStream_t stream)
{
    MoeTcArgs a = {};
    a.n_expert = 1;
    a.hidden = int(rows);
    a.inter = int(cols);
    a.k = 1;
    a.hq = const_cast<int8_t*>(xq);
    a.hd = const_cast<float*>(xd);
    a.y = y;
    a.dense_w = static_cast<const uint8_t*>(W);
    a.dense_rows = int(n_tok);
    cudaError_t e = cudaFuncSetAttribute(moe_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((n_tok + 127) / 128) * (rows / 128);
    const int grid = int(std::min<int64_t>(tiles, device_sm_count()));
    return launch_pdl(moe_tc_kernel<1>, dim3(unsigned(grid)), dim3(kTcThreads), kTcSmem, stream, a);
}

}  // namespace strata
