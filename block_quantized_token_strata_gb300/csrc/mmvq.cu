// mmvq.cu — multi-token block-quantized GEMV (T <= 8 columns, one weight read), its grouped form
// (many independent matrices in one persistent launch) and the fused vocabulary head + argmax.
//
// What it computes: y[t][r] = sum_b (d_w[r][b] * d_x[t][b]) * isum[t][r][b] with exact int32 block
// dots isum, for T tokens that share one read of W — the verify window's "multi-column MMVQ in
// exact mode" (Strata commit "wire multi-token kernels into Verifier and MtpDrafter CUDA graphs",
// verify.hpp header comment). As in the hoisted-load MMVQ-IL kernels of the pull request "sm_80
// (GA100) tuning", the integer dots are exact, the int->float conversion is the exact 1.5*2^23
// magic form, and the fp32 accumulation order and the xor tree are fixed.
//
// Exactness across T (column t of a T-token launch == the T = 1 launch), by construction:
//   * a row is owned by a group of G lanes: half a warp (G = 16), a warp, or KS = G/32 warps; G is
//     a function of (cols, fmt) only;
//   * lane g (0 <= g < G) folds blocks b = g, g+G, g+2G, ... in ascending order into
//     acc = fma(d_w*d_x, float(isum), acc) with explicitly rounded intrinsics;
//   * each half-warp or warp combines its partials in the xor order (16,) 8, 4, 2, 1 (done as a
//     butterfly reduce-scatter, which performs exactly the same pairwise additions for every value),
//     then the KS warp sums are added in warp order;
//   * T only sets the trip count of loops over independent columns. Nothing else depends on it.
//
// Data movement (GB300): a producer warp streams each CTA's contiguous rows with bulk (TMA) copies
// into a ring of shared-memory stages (several row groups of four rows each, up to STRATA_STAGE_KB),
// completion tracked by mbarriers; it starts before the kernel waits on its predecessor
// (programmatic dependent launch), so weight bytes are in flight while the previous kernel
// finishes. 12 or 15 consumer warps (by T) read codes and scales from the stages (consecutive
// lanes, consecutive 16-byte words) and the T activation columns from a shared-memory copy made
// once per matrix, laid out as the 16-byte halves each dp4a chain consumes. Every wait is bounded;
// a timeout sets the device error word.
#include <float.h>
#include <limits.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace strata {

// Launch-plan tunables, fixed at compile time (the defaults are the values measured best on GB300):
// stage size cap, ring budget, L2 prefetch distance, and the lanes-per-row rule (LPR_MIN lanes,
// doubled up to LPR_MAX while every lane keeps at least the format's kMinBlocksPerLane blocks).
#ifndef STRATA_STAGE_KB
#define STRATA_STAGE_KB 60
#endif
#ifndef STRATA_RING_KB
#define STRATA_RING_KB 200
#endif
#ifndef STRATA_PF_STAGES
#define STRATA_PF_STAGES 2
#endif
#ifndef STRATA_LPR_MIN
#define STRATA_LPR_MIN 16
#endif
#ifndef STRATA_LPR_MAX
#define STRATA_LPR_MAX 128
#endif
#ifndef STRATA_CW
#define STRATA_CW 12
#endif
#ifndef STRATA_SG_POW2
#define STRATA_SG_POW2 0
#endif
#ifndef STRATA_NST_POW2
#define STRATA_NST_POW2 0
#endif
#ifndef STRATA_MAXNREG
#define STRATA_MAXNREG 128
#endif

// Consumer warps (+1 producer; at most 15: 16 warps x 128 registers fill the SM), by T: 15 at
// T = 2..4, where more warps hide more of the dp4a latency, else 12 (measured best on GB300). The
// count only schedules work: each row's arithmetic does not depend on it.
#ifndef STRATA_CW_MID
#define STRATA_CW_MID 15
#endif
#ifndef STRATA_CW_HEAD
#define STRATA_CW_HEAD 12
#endif
// the vocabulary head (a single Q8 matrix with the argmax epilogue) keeps its own count
constexpr int cw_for(int T, bool head = false) {
    return head ? STRATA_CW_HEAD : ((T >= 2 && T <= 4) ? STRATA_CW_MID : STRATA_CW);
}
constexpr int kCWMax = STRATA_CW > STRATA_CW_MID ? STRATA_CW : STRATA_CW_MID;
static_assert(kCWMax <= 15 && STRATA_CW_HEAD <= 15, "at most 15 consumer warps");
constexpr int kR = 4;                     // rows per row group (= per ring slot)
constexpr int kMaxGroup = 192;            // matrices per grouped launch
constexpr int kMaxGrid = 1024;
constexpr int kCtasPerSm = 1;             // resident CTAs per SM the launch plans for

// Device error word bits set here: bit 0 a bounded wait ran out; bit 1 the producer waiting for a
// free stage; bit 2 a consumer waiting for a stage's bytes; bit 3 the producer draining its last copies.

template <int FMT> struct FmtInfo;
template <> struct FmtInfo<0> { static constexpr int kQB = 16; };  // Q4: 16 code bytes per block
template <> struct FmtInfo<1> { static constexpr int kQB = 32; };  // Q8: 32 code bytes per block
// Q6: 24 code bytes per block (16 of low 4-bit parts, 8 of high 2-bit parts); its "scale plane" holds
// the two int8 sub-scales of each block, and a third plane one fp16 d per 8 blocks (256 weights)
template <> struct FmtInfo<2> { static constexpr int kQB = 24; };
// Q4K: Q4's 16 code bytes (codes 0..15, no offset); its "scale plane" holds each block's 6-bit scale
// and minimum, the third plane fp16 d and dmin per 8 blocks
template <> struct FmtInfo<3> { static constexpr int kQB = 16; };
// Q5K: Q4K with 5-bit codes; a row's code plane is its nibble blocks (16 bytes each) followed by one
// 32-bit word of fifth bits per block, so kQB counts 20 bytes a block
template <> struct FmtInfo<4> { static constexpr int kQB = 20; };
// bytes per super-block (256 weights) in the third plane
template <int FMT> struct SuperInfo { static constexpr int kDB = FMT == 2 ? 2 : ((FMT == 3 || FMT == 4) ? 4 : 0); };

struct GemvMat {
    const uint8_t* W;
    const int8_t* xq;
    const float* xd;
    const int32_t* xs;
    float* y;
    int rows, nb, lpr;  // lpr: lanes that share a row group (16, 32, 64 or 128)
    int sg;      // chunks (row groups) per ring stage
    int chunk0;  // first chunk of this matrix in the launch's chunk sequence
};

template <int MAXM>
struct GemvParams {
    int n_mat;
    int n_chunk;     // row groups over all matrices
    int cstage;      // bytes per stage in the code ring (multiple of 128)
    int sstage;      // bytes per stage in the scale ring (multiple of 128, 32 bytes of slack)
    int dstage;      // Q6: bytes per stage in the super-block scale ring (multiple of 128, 32 of slack)
    int nst;         // stages in the ring (1..32)
    int nb_max;      // widest matrix, for the activation copy
    int pf;          // stages the producer prefetches into L2 ahead of its bulk copies
    float* cand_val; // head: [T][gridDim.x] per-CTA maxima
    int* cand_idx;   // head: [T][gridDim.x] their row ids
    float* cand_sec; // head: [T][gridDim.x] per-CTA second-largest values (-inf if the CTA saw one row)
    int plan[MAXM > 1 ? kMaxGrid + 1 : 1];  // grouped: first chunk of each CTA (and the end)
    GemvMat m[MAXM];
};

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}
// Merge a candidate (best v at row i, its own second s) into a running (best bv at row bi, second bs):
// the best by the tie rule, and the largest of the values left over (a repeated maximum counts twice,
// so equal top values give second == best). bi == INT_MAX marks an empty side.
__device__ __forceinline__ void top2_merge(float v, int i, float s, float& bv, int& bi, float& bs) {
    if (i == INT_MAX) return;
    if (better(v, i, bv, bi)) {
        if (bi != INT_MAX) bs = fmaxf(bs, bv);
        bs = fmaxf(bs, s);
        bv = v;
        bi = i;
    } else {
        bs = fmaxf(bs, v);  // v >= s, so the candidate's own second is covered
    }
}

// V values per lane over a group of 2^LV lanes (LV = 5: the warp; LV = 4: a half-warp) -> after the
// LV xor levels (2^(LV-1), ..., 2, 1) lane l holds the full group sums of values vidx(l) ..
// vidx(l) + R - 1 in v[0 .. R-1], R = max(1, V >> LV). Every value meets the same pairwise additions
// whatever V is: a reduce-scatter, not a different tree. `mask` names the group's lanes only: the
// other half of a warp may have no rows in this stage and not take part.
template <int V, int LV>
__device__ __forceinline__ void butterfly(float (&v)[V], int lane, int& vidx, unsigned mask) {
    vidx = 0;
#pragma unroll
    for (int lvl = 0; lvl < LV; ++lvl) {
        const int o = (1 << (LV - 1)) >> lvl;
        const int c = (V >> lvl) > 1 ? (V >> lvl) : 1;  // values still held before this level
        if (c > 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int q = 0; q < c / 2; ++q) {
                const float send = up ? v[q] : v[q + c / 2];
                const float keep = up ? v[q + c / 2] : v[q];
                v[q] = __fadd_rn(keep, __shfl_xor_sync(mask, send, o));
            }
            vidx += up ? c / 2 : 0;
        } else {
            v[0] = __fadd_rn(v[0], __shfl_xor_sync(mask, v[0], o));
        }
    }
}

template <int N> struct Pow2Ceil { static constexpr int v = N <= 1 ? 1 : 2 * Pow2Ceil<(N + 1) / 2>::v; };

// Activations in shared memory, one record per block b: the T tokens' 32 codes (16-byte low half,
// then high half, token after token), then T scales and T dp4a seeds (each padded to TPP). The
// record size is 16 mod 32 bytes, so lanes reading consecutive blocks hit distinct bank groups, and
// every token's operand sits at an immediate offset from one per-block address.
// Q6 records hold two seeds a token (one per 16-code half) after the scales. The size is a multiple
// of 16 (every record starts on a 16-byte boundary for the 16-byte code loads and stores).
template <int T, int FMT>
struct XRec {
    static constexpr int tpp = T <= 2 ? 2 : (T <= 4 ? 4 : 8);
    static constexpr int raw = (T * 32 + tpp * (FMT == 2 ? 12 : 8) + 15) / 16 * 16;
    static constexpr int bytes = (raw % 32 == 0) ? raw + 16 : raw;
    static_assert(bytes % 16 == 0 && bytes % 32 == 16, "activation records: 16 mod 32 bytes");
};
static int xrec_bytes(int T, int fmt)
{
    const int tpp = T <= 2 ? 2 : (T <= 4 ? 4 : 8);
    const int raw = (T * 32 + tpp * (fmt == 2 ? 12 : 8) + 15) / 16 * 16;
    return (raw % 32 == 0) ? raw + 16 : raw;
}
template <> struct Pow2Ceil<1> { static constexpr int v = 1; };

// The matrices a CTA touches, as segments: chunks [gs, ge) of matrix mi within [g0, g1).
template <int MAXM>
struct SegIter {
    const GemvParams<MAXM>* p;
    int g1, mi, gs, ge;
    __device__ void init(const GemvParams<MAXM>& prm, int g0, int gend) {
        p = &prm;
        g1 = gend;
        mi = 0;
        if constexpr (MAXM > 1) {
            while (mi + 1 < prm.n_mat && prm.m[mi + 1].chunk0 <= g0) ++mi;
        }
        gs = g0;
        settle();
    }
    __device__ void settle() {
        const int mend = (MAXM > 1 && mi + 1 < p->n_mat) ? p->m[mi + 1].chunk0 : p->n_chunk;
        ge = min(g1, mend);
    }
    __device__ bool valid() const { return gs < g1; }
    __device__ void next() { gs = ge; ++mi; if (gs < g1) settle(); }
};

// Walks a CTA's chunks as ring stages: runs of m.sg row groups of one matrix (up to STRATA_STAGE_KB).
template <int MAXM>
struct StageIter {
    SegIter<MAXM> seg;
    int sg, se;  // stage chunks [sg, se)
    __device__ void init(const GemvParams<MAXM>& prm, int g0, int gend) {
        seg.init(prm, g0, gend);
        sg = seg.gs;
        settle();
    }
    __device__ void settle() { se = min(sg + seg.p->m[seg.mi].sg, seg.ge); }
    __device__ bool valid() const { return sg < seg.g1; }
    __device__ void next() {
        sg = se;
        if (sg >= seg.ge) {
            seg.next();
            if (!seg.valid()) return;
            sg = seg.gs;
        }
        settle();
    }
};

template <int FMT, int T, int MAXM, bool HEAD>
// registers: 128 a thread. The register file is split between the SM's four schedulers (16K each) and
// a CTA of 13 to 16 warps puts four warps on one of them, so 128 is the most either launch size
// (13 or 16 warps) can start with.
__global__ void __maxnreg__(STRATA_MAXNREG) gemv_kernel(const __grid_constant__ GemvParams<MAXM> p)
{
    constexpr int QB = FmtInfo<FMT>::kQB;
    constexpr int QV = QB / 16;
    constexpr int V = Pow2Ceil<kR * T>::v;
    constexpr int TPP = T <= 2 ? 2 : (T <= 4 ? 4 : 8);  // tokens padded for the scale vectors
    constexpr int NP = (T + 1) / 2;                      // token pairs
    constexpr int RX = XRec<T, FMT>::bytes;              // activation record per block
    constexpr int kCW = cw_for(T, HEAD);                 // consumer warps of this launch
    // sums a lane owns after a half-warp group's reduction (2 when the group's 4T values outnumber its
    // 16 lanes), and the head's candidate slots per lane (one per owned sum)
    constexpr int RM = V > 16 ? 2 : 1;
    constexpr int HS = HEAD ? RM : 1;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ volatile int s_abort;

    const int NST = p.nst;  // ring stages
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);                 // full[NST], empty[NST]
    uint8_t* xsm = smem + 2 * 8 * 32;                                    // activations
    float* red = reinterpret_cast<float*>(xsm + p.nb_max * RX);          // [2][kCW][32]
    float* hv = red + 2 * kCW * 32;                                      // head: [HS][kCW*32] values
    int* hi = reinterpret_cast<int*>(hv + HS * kCW * 32);                // head: [HS][kCW*32] ids
    float* hs = reinterpret_cast<float*>(hi + HS * kCW * 32);            // head: [HS][kCW*32] second values
    // codes [NST][cstage]: an offset from `smem` (not an integer round trip), so that the compiler keeps
    // the ring in the shared address space and its reads stay shared-memory loads
    uint8_t* cring = smem + ((reinterpret_cast<uint8_t*>(hs + HS * kCW * 32) - smem + 127) & ~ptrdiff_t(127));
    uint8_t* sring = cring + NST * p.cstage;                                      // scales [NST][sstage]
    uint8_t* dring = sring + NST * p.sstage;                                      // Q6 d [NST][dstage]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int g0, g1;  // this CTA's chunks
    if constexpr (MAXM > 1) {
        g0 = p.plan[blockIdx.x];
        g1 = p.plan[blockIdx.x + 1];
    } else {
        g0 = int((int64_t(blockIdx.x) * p.n_chunk) / gridDim.x);
        g1 = int((int64_t(blockIdx.x + 1) * p.n_chunk) / gridDim.x);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);           // full: the producer's expect_tx arrival
            mbar_init(smem_u32(&bars[NST + s]), kCW);   // empty: one arrival per consumer warp
        }
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    // ------------------------------------------------------------------ producer warp
    if (warp == kCW) {
        pdl_launch();  // every thread of the CTA triggers its dependents before it waits (see below)
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            StageIter<MAXM> it, pf;
            it.init(p, g0, g1);
            pf.init(p, g0, g1);
            // L2 prefetch runs p.pf stages ahead of the bulk copies, so that they find their bytes in
            // L2 rather than waiting out HBM latency under load.
            auto prefetch_next = [&]() {
                if (!pf.valid()) return;
                const GemvMat& m = p.m[pf.seg.mi];
                const int r0 = (pf.sg - m.chunk0) * kR;
                const int nr = min((pf.se - pf.sg) * kR, m.rows - r0);
                bulk_prefetch_l2(m.W + size_t(r0) * m.nb * QB, uint32_t(nr) * m.nb * QB);
                const uintptr_t sa = reinterpret_cast<uintptr_t>(m.W + size_t(m.rows) * m.nb * QB + size_t(r0) * m.nb * 2);
                const uintptr_t lo = (sa + 15) & ~uintptr_t(15), hi2 = (sa + uint32_t(nr) * m.nb * 2) & ~uintptr_t(15);
                if (hi2 > lo) bulk_prefetch_l2(reinterpret_cast<const void*>(lo), uint32_t(hi2 - lo));
                if constexpr (SuperInfo<FMT>::kDB > 0) {
                    constexpr int DB = SuperInfo<FMT>::kDB;
                    const uintptr_t da = reinterpret_cast<uintptr_t>(m.W + size_t(m.rows) * m.nb * (QB + 2) +
                                                                     size_t(r0) * (m.nb / 8) * DB);
                    const uintptr_t dlo = (da + 15) & ~uintptr_t(15), dhi = (da + uint32_t(nr) * (m.nb / 8) * DB) & ~uintptr_t(15);
                    if (dhi > dlo) bulk_prefetch_l2(reinterpret_cast<const void*>(dlo), uint32_t(dhi - dlo));
                }
                pf.next();
            };
            for (int q = 0; q < p.pf; ++q) prefetch_next();
            bool waited = false;
            int k = 0, s = 0, lap = 0;  // stage count, its slot and ring lap (k = lap * NST + s)
            for (; it.valid(); it.next(), ++k, s = (s + 1 == NST) ? 0 : s + 1, lap += (s == 0)) {
                if (k == NST) {  // the ring is full: from here on, order after the predecessor
                    pdl_wait();
                    waited = true;
                }
                if (k >= NST) {
                    if (!mbar_wait(smem_u32(&bars[NST + s]), (lap - 1) & 1, &s_abort)) {
                        s_abort = 1;
                        atomicOr(&g_strata_device_error, 1 | 2);
                        break;
                    }
                }
                prefetch_next();
                const GemvMat& m = p.m[it.seg.mi];
                const int r0 = (it.sg - m.chunk0) * kR;
                const int nr = min((it.se - it.sg) * kR, m.rows - r0);
                const uint8_t* qsrc = m.W + size_t(r0) * m.nb * QB;
                const uint32_t qbytes = uint32_t(nr) * m.nb * QB;
                const uint8_t* ssrc = m.W + size_t(m.rows) * m.nb * QB + size_t(r0) * m.nb * 2;
                const uint32_t sbytes = uint32_t(nr) * m.nb * 2;
                const uint32_t mis = uint32_t(reinterpret_cast<uintptr_t>(ssrc) & 15);
                uint8_t* sdst = sring + s * p.sstage + mis;   // same alignment mod 16 as ssrc
                const uint32_t head = min(sbytes, (16u - mis) & 15u);
                const uint32_t mid = (sbytes - head) & ~15u;
                const uint32_t tail = sbytes - head - mid;
                for (uint32_t b = 0; b < head; ++b) sdst[b] = __ldg(ssrc + b);
                for (uint32_t b = sbytes - tail; b < sbytes; ++b) sdst[b] = __ldg(ssrc + b);
                // Q6: the super-block scales of the same rows, placed like the scales (same alignment
                // mod 16 as the source; the unaligned ends by plain loads)
                const uint8_t* dsrc = nullptr;
                uint8_t* ddst = nullptr;
                uint32_t dhead = 0, dmid = 0;
                if constexpr (SuperInfo<FMT>::kDB > 0) {
                    constexpr int DB = SuperInfo<FMT>::kDB;
                    const int ns = m.nb / 8;
                    dsrc = m.W + size_t(m.rows) * m.nb * (QB + 2) + size_t(r0) * ns * DB;
                    const uint32_t dbytes = uint32_t(nr) * ns * DB;
                    const uint32_t dmis = uint32_t(reinterpret_cast<uintptr_t>(dsrc) & 15);
                    ddst = dring + s * p.dstage + dmis;
                    dhead = min(dbytes, (16u - dmis) & 15u);
                    dmid = (dbytes - dhead) & ~15u;
                    const uint32_t dtail = dbytes - dhead - dmid;
                    for (uint32_t b = 0; b < dhead; ++b) ddst[b] = __ldg(dsrc + b);
                    for (uint32_t b = dbytes - dtail; b < dbytes; ++b) ddst[b] = __ldg(dsrc + b);
                    if (dhead | dtail) fence_proxy_async_smem();
                }
                if (head | tail) fence_proxy_async_smem();
                const uint32_t fb = smem_u32(&bars[s]);
                mbar_arrive_expect_tx(fb, qbytes + mid + dmid);
                bulk_g2s(smem_u32(cring + s * p.cstage), qsrc, qbytes, fb, pol);
                if (mid) bulk_g2s(smem_u32(sdst + head), ssrc + head, mid, fb, pol);
                if (dmid) bulk_g2s(smem_u32(ddst + dhead), dsrc + dhead, dmid, fb, pol);
            }
            if (!waited) pdl_wait();
            // no copy may still be landing in shared memory when the CTA leaves: the issued copies are
            // waited for (bounded) even after an abort
            const int no_abort = 0;
            for (int i = (k > NST ? k - NST : 0); i < k; ++i)
                if (!mbar_wait(smem_u32(&bars[i % NST]), (i / NST) & 1, &no_abort)) {
                    atomicOr(&g_strata_device_error, 1 | 8);
                    break;
                }
        } else {
            pdl_wait();
        }
        return;
    }

    // ------------------------------------------------------------------ consumer warps
    // Dependents may launch now (they wait for this grid's completion before they read what it
    // writes, and can stream their weights meanwhile); this grid's own inputs come after the wait.
    pdl_launch();
    pdl_wait();

    // head, per slot j < HS: the best value this lane saw, its row, the largest value after it (a
    // multiset's second) and the token of the sums it holds in that slot
    float best[HS], second[HS];
    int bidx[HS], tval[HS];
#pragma unroll
    for (int j = 0; j < HS; ++j) {
        best[j] = -FLT_MAX;
        second[j] = -INFINITY;
        bidx[j] = INT_MAX;
        tval[j] = 0;
    }

    SegIter<MAXM> sgi;
    sgi.init(p, g0, g1);
    int k0 = 0;  // ring stage of the segment's first chunk, in step with the producer
    for (; sgi.valid(); sgi.next()) {
        const GemvMat& m = p.m[sgi.mi];
        const int nb = m.nb;
        const int rows = m.rows;
        const int gs = sgi.gs;
        const int nseg = sgi.ge - gs;

        // activations of this matrix -> shared memory, one record per block (see XRec)
        {
            const uint4* src = reinterpret_cast<const uint4*>(m.xq);
            for (int i = threadIdx.x; i < T * nb * 2; i += kCW * 32) {
                const int t = i / (2 * nb);
                const int c = i - t * 2 * nb;
                *reinterpret_cast<uint4*>(xsm + (c >> 1) * RX + t * 32 + (c & 1) * 16) = __ldg(src + i);
            }
            for (int i = threadIdx.x; i < nb * TPP; i += kCW * 32) {
                const int b = i / TPP, t = i - (i / TPP) * TPP;
                float d = 0.0f;
                int c0 = (FMT == 3 || FMT == 4) ? 0 : kMagicBits, c1 = kMagicBits;  // Q4K/Q5K: the block sum as a float
                if (t < T) {
                    d = __ldg(m.xd + t * nb + b);
                    if (FMT == 0) c0 = kMagicBits - 8 * __ldg(m.xs + t * nb + b);
                    if (FMT == 3 || FMT == 4) c0 = __float_as_int(float(__ldg(m.xs + t * nb + b)));  // exact: |s| <= 4064
                    if (FMT == 2) {
                        // Q6 codes stand for q - 32 and carry one sub-scale per 16: seed each half's chain
                        // with -32 times that half's activation sum
                        const uint4* xb = src + size_t(t) * nb * 2 + size_t(b) * 2;
                        const uint4 lo = __ldg(xb), hi = __ldg(xb + 1);
                        int sl = 0, sh = 0;
                        sl = __dp4a(int(lo.x), 0x01010101, sl); sl = __dp4a(int(lo.y), 0x01010101, sl);
                        sl = __dp4a(int(lo.z), 0x01010101, sl); sl = __dp4a(int(lo.w), 0x01010101, sl);
                        sh = __dp4a(int(hi.x), 0x01010101, sh); sh = __dp4a(int(hi.y), 0x01010101, sh);
                        sh = __dp4a(int(hi.z), 0x01010101, sh); sh = __dp4a(int(hi.w), 0x01010101, sh);
                        c0 = kMagicBits - 32 * sl;
                        c1 = kMagicBits - 32 * sh;
                    }
                }
                *reinterpret_cast<float*>(xsm + b * RX + T * 32 + t * 4) = d;
                *reinterpret_cast<int*>(xsm + b * RX + T * 32 + TPP * 4 + t * 4) = c0;
                if (FMT == 2) *reinterpret_cast<int*>(xsm + b * RX + T * 32 + TPP * 8 + t * 4) = c1;
            }
        }
        named_bar_sync(1, kCW * 32);

        // A row group is owned by L = m.lpr lanes: a half-warp (L = 16, two groups per warp), a warp,
        // or KS = L / 32 warps that add their warp sums through shared memory.
        const int L = m.lpr;
        const bool half = L < 32;
        const int KS = half ? 1 : L >> 5;
        const int NG = half ? 2 * kCW : kCW / KS;
        const int grp = half ? 2 * warp + (lane >> 4) : warp / KS;
        const int wig = half ? 0 : warp - grp * KS;
        const int G = L;
        const int gl = half ? (lane & 15) : wig * 32 + lane;
        const int rsw = nb * QB;  // row stride of the codes in a stage

        // Every consumer warp waits on, and then releases, every stage in order — also the stages in
        // which its group has no rows. A stage is therefore never refilled before each warp has seen
        // its current phase, so no warp can fall a ring lap behind and take a later phase for an
        // earlier one (a parity wait cannot tell them apart). Slot, phase parity and this group's
        // place in the stage advance incrementally.
        const int SG = m.sg;
        int s = k0 % NST, par = (k0 / NST) & 1;
        int base = 0;  // group of the stage's first chunk
        for (int c0 = 0, jj = 0; c0 < nseg; c0 += SG) {
            int pos = grp - base;
            if (pos < 0) pos += NG;
            const bool active = grp < NG && pos < min(SG, nseg - c0);  // warps past NG*KS idle
            const int r0s = (gs + c0 - m.chunk0) * kR;           // first row of the stage
            const int row0 = r0s + pos * kR;
            const int nr = min(kR, rows - row0);
            const bool ok = !s_abort && mbar_wait(smem_u32(&bars[s]), par, &s_abort);
            if (!ok) {
                s_abort = 1;
                atomicOr(&g_strata_device_error, 1 | 4);
            }
            if (active) {
                float v[V];
#pragma unroll
                for (int q = 0; q < V; ++q) v[q] = 0.0f;
                if (ok) {
                    const uint8_t* cb = cring + s * p.cstage + pos * kR * rsw;
                    const uintptr_t ssrc = reinterpret_cast<uintptr_t>(m.W + size_t(rows) * nb * QB + size_t(r0s) * nb * 2);
                    const unsigned short* sc = reinterpret_cast<const unsigned short*>(
                        sring + s * p.sstage + int(ssrc & 15) + pos * (kR * 2) * nb);
                    const f32x2 negm = pack_f2(-kMagic, -kMagic);
                    f32x2 acc[kR][NP];
#pragma unroll
                    for (int r = 0; r < kR; ++r)
#pragma unroll
                        for (int q = 0; q < NP; ++q) acc[r][q] = 0ull;
                    if constexpr (FMT == 2) {
                        // Q6: per block 24 code bytes, two int8 sub-scales, the super-block's fp16 d
                        const uintptr_t dsrc = reinterpret_cast<uintptr_t>(m.W + size_t(rows) * nb * (QB + 2) +
                                                                           size_t(r0s) * (nb / 8) * 2);
                        const unsigned short* dpl = reinterpret_cast<const unsigned short*>(
                            dring + s * p.dstage + int(dsrc & 15) + pos * (kR * 2) * (nb / 8));
                        const int ns = nb / 8;
                        for (int kb = gl; kb < nb; kb += G) {
                            const uint8_t* wp = cb + kb * QB;
                            const unsigned short* sp = sc + kb;
                            const uint8_t* xr = xsm + kb * RX;
                            uint2 wl0[kR], wl1[kR], wh[kR];
                            f32x2 sdl2[kR], sdh2[kR];
#pragma unroll
                            for (int r = 0; r < kR; ++r) {
                                wl0[r] = *reinterpret_cast<const uint2*>(wp + r * rsw);
                                wl1[r] = *reinterpret_cast<const uint2*>(wp + r * rsw + 8);
                                wh[r] = *reinterpret_cast<const uint2*>(wp + r * rsw + 16);
                                const unsigned short su = sp[r * nb];
                                const float dd = __half2float(__ushort_as_half(dpl[r * ns + (kb >> 3)]));
                                // d * s is exact in fp32 (11 + 7 significant bits)
                                const float s0 = __fmul_rn(dd, float(int(int8_t(su & 0xFF))));
                                const float s1 = __fmul_rn(dd, float(int(int8_t(su >> 8))));
                                sdl2[r] = pack_f2(s0, s0);
                                sdh2[r] = pack_f2(s1, s1);
                            }
                            float dxv[TPP];
                            int c0v[TPP], c1v[TPP];
#pragma unroll
                            for (int q = 0; q < TPP; q += 2) {
                                const float2 dd = *reinterpret_cast<const float2*>(xr + T * 32 + q * 4);
                                const int2 cc = *reinterpret_cast<const int2*>(xr + T * 32 + TPP * 4 + q * 4);
                                const int2 ch = *reinterpret_cast<const int2*>(xr + T * 32 + TPP * 8 + q * 4);
                                dxv[q] = dd.x; dxv[q + 1] = dd.y;
                                c0v[q] = cc.x; c0v[q + 1] = cc.y;
                                c1v[q] = ch.x; c1v[q + 1] = ch.y;
                            }
#pragma unroll
                            for (int q = 0; q < NP; ++q) {
                                const int ta = 2 * q, tb = 2 * q + 1;
                                const uint4 xla = *reinterpret_cast<const uint4*>(xr + ta * 32);
                                const uint4 xha = *reinterpret_cast<const uint4*>(xr + ta * 32 + 16);
                                uint4 xlb = xla, xhb = xha;
                                if (tb < T) {
                                    xlb = *reinterpret_cast<const uint4*>(xr + tb * 32);
                                    xhb = *reinterpret_cast<const uint4*>(xr + tb * 32 + 16);
                                }
                                const f32x2 dx2 = pack_f2(dxv[ta], dxv[tb]);
#pragma unroll
                                for (int r = 0; r < kR; ++r) {
                                    uint32_t qw[8];
                                    unpack_q6(wl0[r], wl1[r], wh[r], qw);
                                    const int la = dot16(qw, xla, c0v[ta]), ha = dot16(qw + 4, xha, c1v[ta]);
                                    const int lb = (tb < T) ? dot16(qw, xlb, c0v[tb]) : kMagicBits;
                                    const int hb = (tb < T) ? dot16(qw + 4, xhb, c1v[tb]) : kMagicBits;
                                    // one term per sub-scale, the low half first: acc += (d*s*d_x) * isum_half
                                    const f32x2 fl = add_f2(pack_f2(__int_as_float(la), __int_as_float(lb)), negm);
                                    const f32x2 fh = add_f2(pack_f2(__int_as_float(ha), __int_as_float(hb)), negm);
                                    acc[r][q] = fma_f2(mul_f2(sdl2[r], dx2), fl, acc[r][q]);
                                    acc[r][q] = fma_f2(mul_f2(sdh2[r], dx2), fh, acc[r][q]);
                                }
                            }
                        }
                    } else if constexpr (FMT == 3 || FMT == 4) {
                        // Q4K: per block 16 code bytes (codes 0..15), a 6-bit scale and minimum; per 8
                        // blocks fp16 d and dmin. Terms: (d*sc*d_x)*isum, then (-dmin*m*d_x)*sum(x).
                        // Q5K: the same with each block's fifth-bit word after the row's nibble blocks
                        const uintptr_t dsrc = reinterpret_cast<uintptr_t>(m.W + size_t(rows) * nb * (QB + 2) +
                                                                           size_t(r0s) * (nb / 8) * 4);
                        const unsigned short* dpl = reinterpret_cast<const unsigned short*>(
                            dring + s * p.dstage + int(dsrc & 15) + pos * (kR * 4) * (nb / 8));
                        const int ns = nb / 8;
                        for (int kb = gl; kb < nb; kb += G) {
                            const uint8_t* wp = cb + kb * 16;
                            const uint8_t* hp = cb + 16 * nb + kb * 4;  // Q5K: the block's fifth-bit word
                            const unsigned short* sp = sc + kb;
                            const uint8_t* xr = xsm + kb * RX;
                            uint4 w[kR];
                            uint32_t hbw[kR];
                            f32x2 sc2[kR], mn2[kR];
#pragma unroll
                            for (int r = 0; r < kR; ++r) {
                                w[r] = *reinterpret_cast<const uint4*>(wp + r * rsw);
                                hbw[r] = (FMT == 4) ? *reinterpret_cast<const uint32_t*>(hp + r * rsw) : 0u;
                                const unsigned short su = sp[r * nb];
                                const int di = 2 * (r * ns + (kb >> 3));
                                const float dd = __half2float(__ushort_as_half(dpl[di]));
                                const float dm = __half2float(__ushort_as_half(dpl[di + 1]));
                                // d * sc and dmin * m are exact in fp32 (11 + 6 significant bits)
                                const float sv = __fmul_rn(dd, float(su & 0xFF));
                                const float mv = __fmul_rn(dm, float(su >> 8));
                                sc2[r] = pack_f2(sv, sv);
                                mn2[r] = pack_f2(-mv, -mv);
                            }
                            float dxv[TPP], xsv[TPP];
#pragma unroll
                            for (int q = 0; q < TPP; q += 2) {
                                const float2 dd = *reinterpret_cast<const float2*>(xr + T * 32 + q * 4);
                                const float2 ss = *reinterpret_cast<const float2*>(xr + T * 32 + TPP * 4 + q * 4);
                                dxv[q] = dd.x; dxv[q + 1] = dd.y;
                                xsv[q] = ss.x; xsv[q + 1] = ss.y;
                            }
#pragma unroll
                            for (int q = 0; q < NP; ++q) {
                                const int ta = 2 * q, tb = 2 * q + 1;
                                const uint4 xla = *reinterpret_cast<const uint4*>(xr + ta * 32);
                                const uint4 xha = *reinterpret_cast<const uint4*>(xr + ta * 32 + 16);
                                uint4 xlb = xla, xhb = xha;
                                if (tb < T) {
                                    xlb = *reinterpret_cast<const uint4*>(xr + tb * 32);
                                    xhb = *reinterpret_cast<const uint4*>(xr + tb * 32 + 16);
                                }
                                const f32x2 dx2 = pack_f2(dxv[ta], dxv[tb]);
                                const f32x2 xs2 = pack_f2(xsv[ta], xsv[tb]);
#pragma unroll
                                for (int r = 0; r < kR; ++r) {
                                    int ca, cbv;
                                    if constexpr (FMT == 4) {
                                        ca = dot_q5(w[r], hbw[r], xla, xha, kMagicBits);
                                        cbv = (tb < T) ? dot_q5(w[r], hbw[r], xlb, xhb, kMagicBits) : kMagicBits;
                                    } else {
                                        ca = dot_q4(w[r], xla, xha, kMagicBits);
                                        cbv = (tb < T) ? dot_q4(w[r], xlb, xhb, kMagicBits) : kMagicBits;
                                    }
                                    const f32x2 f2 = add_f2(pack_f2(__int_as_float(ca), __int_as_float(cbv)), negm);
                                    acc[r][q] = fma_f2(mul_f2(sc2[r], dx2), f2, acc[r][q]);
                                    acc[r][q] = fma_f2(mul_f2(mn2[r], dx2), xs2, acc[r][q]);
                                }
                            }
                        }
                    } else {
                    for (int kb = gl; kb < nb; kb += G) {
                        const uint8_t* wp = cb + kb * QB;
                        const unsigned short* sp = sc + kb;
                        const uint8_t* xr = xsm + kb * RX;
                        uint4 w[kR][QV];
                        f32x2 dw2[kR];
#pragma unroll
                        for (int r = 0; r < kR; ++r) {
#pragma unroll
                            for (int h = 0; h < QV; ++h)
                                w[r][h] = *reinterpret_cast<const uint4*>(wp + r * rsw + h * 16);
                            const float d = __half2float(__ushort_as_half(sp[r * nb]));
                            dw2[r] = pack_f2(d, d);
                        }
                        float dxv[TPP];
                        int c0v[TPP];
#pragma unroll
                        for (int q = 0; q < TPP; q += 2) {
                            const float2 dd = *reinterpret_cast<const float2*>(xr + T * 32 + q * 4);
                            const int2 cc = *reinterpret_cast<const int2*>(xr + T * 32 + TPP * 4 + q * 4);
                            dxv[q] = dd.x; dxv[q + 1] = dd.y;
                            c0v[q] = cc.x; c0v[q + 1] = cc.y;
                        }
#pragma unroll
                        for (int q = 0; q < NP; ++q) {
                            const int ta = 2 * q, tb = 2 * q + 1;
                            const uint4 xla = *reinterpret_cast<const uint4*>(xr + ta * 32);
                            const uint4 xha = *reinterpret_cast<const uint4*>(xr + ta * 32 + 16);
                            uint4 xlb = xla, xhb = xha;
                            if (tb < T) {
                                xlb = *reinterpret_cast<const uint4*>(xr + tb * 32);
                                xhb = *reinterpret_cast<const uint4*>(xr + tb * 32 + 16);
                            }
                            const f32x2 dx2 = pack_f2(dxv[ta], dxv[tb]);
#pragma unroll
                            for (int r = 0; r < kR; ++r) {
                                int ca, cbv;
                                if constexpr (FMT == 0) {
                                    ca = dot_q4(w[r][0], xla, xha, c0v[ta]);
                                    cbv = (tb < T) ? dot_q4(w[r][0], xlb, xhb, c0v[tb]) : kMagicBits;
                                } else {
                                    ca = dot_q8(w[r][0], w[r][QV - 1], xla, xha, c0v[ta]);
                                    cbv = (tb < T) ? dot_q8(w[r][0], w[r][QV - 1], xlb, xhb, c0v[tb]) : kMagicBits;
                                }
                                // (F - 1.5*2^23) is exact; then acc += (d_w*d_x)*isum, each half one IEEE op
                                const f32x2 f2 = add_f2(pack_f2(__int_as_float(ca), __int_as_float(cbv)), negm);
                                acc[r][q] = fma_f2(mul_f2(dw2[r], dx2), f2, acc[r][q]);
                            }
                        }
                    }
                    }  // Q4 / Q8
#pragma unroll
                    for (int r = 0; r < kR; ++r)
#pragma unroll
                        for (int q = 0; q < NP; ++q) {
                            float lo, hi2;
                            unpack_f2(acc[r][q], lo, hi2);
                            if (2 * q < T) v[r * T + 2 * q] = lo;
                            if (2 * q + 1 < T) v[r * T + 2 * q + 1] = hi2;
                        }
                }
                int vidx;
                // group sums: lane l owns R consecutive values from vidx; with fewer values than
                // lanes, each sum sits in 2^k lanes and the lowest of them owns it
                int R = 1;
                bool owner;
                // this group's lanes: the whole warp, or its own half (shuffles and the warp barrier
                // below name no lane of the other half, which may be idle in this stage)
                const unsigned gmask = half ? (lane < 16 ? 0x0000ffffu : 0xffff0000u) : 0xffffffffu;
                if (half) {
                    butterfly<V, 4>(v, lane, vidx, gmask);
                    R = V > 16 ? V / 16 : 1;
                    owner = V >= 16 || (lane & (16 / V - 1)) == 0;
                } else {
                    butterfly<V, 5>(v, lane, vidx, gmask);
                    owner = V >= 32 || (lane & (32 / V - 1)) == 0;
                }
                bool final_lane = (KS == 1);
                if (KS > 1) {  // (R == 1 here: a warp holds at most 32 values)
                    float* rb = red + ((jj & 1) * kCW + warp) * 32;
                    if (owner && vidx < kR * T) rb[vidx] = v[0];
                    named_bar_sync(2 + grp, G);
                    if (wig == 0) {
                        final_lane = true;
                        if (owner && vidx < kR * T) {
                            const float* base2 = red + ((jj & 1) * kCW + grp * KS) * 32;
                            float tot = base2[vidx];
                            for (int w2 = 1; w2 < KS; ++w2) tot = __fadd_rn(tot, base2[w2 * 32 + vidx]);
                            v[0] = tot;
                        }
                    }
                } else {
                    __syncwarp(gmask);
                }
                if (final_lane && owner && ok) {
#pragma unroll
                    for (int j = 0; j < RM; ++j) {
                        const int idx = vidx + j;
                        if (j >= R || idx >= kR * T) continue;
                        const int r = idx / T, t = idx - (idx / T) * T;
                        if (r >= nr) continue;
                        const float tot = v[j];
                        const int row = row0 + r;
                        if (m.y != nullptr) m.y[size_t(t) * rows + row] = tot;
                        if constexpr (HEAD) {
                            // slot j always holds the same token in this launch (vidx depends on the
                            // lane only), so one token per slot
                            const int js = HS > 1 ? j : 0;
                            tval[js] = t;
                            if (better(tot, row, best[js], bidx[js])) {
                                if (bidx[js] != INT_MAX) second[js] = fmaxf(second[js], best[js]);
                                best[js] = tot;
                                bidx[js] = row;
                            } else {
                                second[js] = fmaxf(second[js], tot);
                            }
                        }
                    }
                }
                ++jj;
            }
            // this warp is done with the stage (the sums above read registers and `red` only)
            if (lane == 0 && ok) mbar_arrive(smem_u32(&bars[NST + s]));
            if (++s == NST) { s = 0; par ^= 1; }
            base += SG;
            if (base >= NG) base -= NG;
        }
        k0 += (nseg + SG - 1) / SG;
        named_bar_sync(1, kCW * 32);  // everyone is done with this matrix's activations
    }

    if constexpr (HEAD) {
#pragma unroll
        for (int j = 0; j < HS; ++j) {
            hv[j * kCW * 32 + threadIdx.x] = best[j];
            hi[j * kCW * 32 + threadIdx.x] = (bidx[j] == INT_MAX) ? INT_MAX : (bidx[j] | (tval[j] << 27));  // token in the top bits
            hs[j * kCW * 32 + threadIdx.x] = second[j];
        }
        named_bar_sync(1, kCW * 32);
        if (threadIdx.x < T) {
            const int t = threadIdx.x;
            float bv = -FLT_MAX, bs = -INFINITY;
            int bi = INT_MAX;
            for (int q = 0; q < HS * kCW * 32; ++q) {
                const int code = hi[q];
                if (code == INT_MAX || (code >> 27) != t) continue;
                const int id = code & ((1 << 27) - 1);
                top2_merge(hv[q], id, hs[q], bv, bi, bs);
            }
            p.cand_val[size_t(t) * gridDim.x + blockIdx.x] = bv;
            p.cand_idx[size_t(t) * gridDim.x + blockIdx.x] = bi;
            if (p.cand_sec) p.cand_sec[size_t(t) * gridDim.x + blockIdx.x] = bs;
        }
    }
}

// one warp per token: reduce the per-CTA candidates with the tie rule (equal values -> lower id);
// with `margin`, also the largest of the other values: margin = top-1 value - top-2 value
// (0 when the maximum occurs twice, +inf for a one-row head)
__global__ void __launch_bounds__(256) head_finalize_kernel(const float* __restrict__ cand_val,
                                                            const int* __restrict__ cand_idx,
                                                            const float* __restrict__ cand_sec, int ncand,
                                                            int T, int32_t* __restrict__ ids,
                                                            float* __restrict__ margin)
{
    pdl_launch();
    pdl_wait();
    const int t = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    float bv = -FLT_MAX, bs = -INFINITY;
    int bi = INT_MAX;
    for (int i = lane; i < ncand; i += 32) {
        const float v = cand_val[size_t(t) * ncand + i];
        const int j = cand_idx[size_t(t) * ncand + i];
        const float s = cand_sec ? cand_sec[size_t(t) * ncand + i] : -INFINITY;
        top2_merge(v, j, s, bv, bi, bs);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        const float os = __shfl_xor_sync(0xffffffffu, bs, off);
        top2_merge(ov, oi, os, bv, bi, bs);
    }
    if (lane == 0) {
        ids[t] = bi;
        if (margin) margin[t] = __fsub_rn(bv, bs);
    }
}

// test hook: isum[t][r][b] from the same dot_q4 / dot_q8 device code
template <int FMT>
__global__ void __launch_bounds__(256) block_dots_kernel(const uint8_t* __restrict__ W, int rows, int nb,
                                                         const int8_t* __restrict__ xq,
                                                         const int32_t* __restrict__ xs, int T,
                                                         int32_t* __restrict__ isum)
{
    pdl_launch();
    pdl_wait();
    constexpr int QB = FmtInfo<FMT>::kQB;
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= int64_t(rows) * nb) return;
    const int r = int(i / nb), b = int(i % nb);
    if constexpr (FMT == 2) {
        // Q6: s0 * sum over the first 16 of (q-32)*x + s1 * the same over the last 16 (exact int)
        const uint8_t* blk = W + size_t(i) * 24;
        const uint2 lo0 = *reinterpret_cast<const uint2*>(blk), lo1 = *reinterpret_cast<const uint2*>(blk + 8);
        const uint2 hi = *reinterpret_cast<const uint2*>(blk + 16);
        const unsigned short su = *reinterpret_cast<const unsigned short*>(W + size_t(rows) * nb * 24 + size_t(i) * 2);
        uint32_t qw[8];
        unpack_q6(lo0, lo1, hi, qw);
        for (int t = 0; t < T; ++t) {
            const uint4* xp = reinterpret_cast<const uint4*>(xq + size_t(t) * nb * 32 + size_t(b) * 32);
            const uint4 xl = xp[0], xh = xp[1];
            int sl = 0, sh = 0;
            sl = __dp4a(int(xl.x), 0x01010101, sl); sl = __dp4a(int(xl.y), 0x01010101, sl);
            sl = __dp4a(int(xl.z), 0x01010101, sl); sl = __dp4a(int(xl.w), 0x01010101, sl);
            sh = __dp4a(int(xh.x), 0x01010101, sh); sh = __dp4a(int(xh.y), 0x01010101, sh);
            sh = __dp4a(int(xh.z), 0x01010101, sh); sh = __dp4a(int(xh.w), 0x01010101, sh);
            const int l = dot16(qw, xl, -32 * sl), h = dot16(qw + 4, xh, -32 * sh);
            isum[(size_t(t) * rows + r) * nb + b] = int(int8_t(su & 0xFF)) * l + int(int8_t(su >> 8)) * h;
        }
        return;
    }
    if constexpr (FMT == 4) {
        // Q5K: codes 0..31, the row's nibble blocks then its fifth-bit words; no offset
        const uint8_t* row = W + size_t(r) * nb * 20;
        const uint4 w = ld_stream_v4(row + size_t(b) * 16);
        const uint32_t hb = *reinterpret_cast<const uint32_t*>(row + size_t(nb) * 16 + size_t(b) * 4);
        for (int t = 0; t < T; ++t) {
            const uint4* xp = reinterpret_cast<const uint4*>(xq + size_t(t) * nb * 32 + size_t(b) * 32);
            isum[(size_t(t) * rows + r) * nb + b] = dot_q5(w, hb, xp[0], xp[1], kMagicBits) - kMagicBits;
        }
        return;
    }
    const uint4 w0 = ld_stream_v4(W + size_t(i) * QB);
    const uint4 w1 = (QB == 32) ? ld_stream_v4(W + size_t(i) * QB + 16) : w0;
    for (int t = 0; t < T; ++t) {
        const uint4* xp = reinterpret_cast<const uint4*>(xq + size_t(t) * nb * 32 + size_t(b) * 32);
        const uint4 xl = xp[0], xh = xp[1];
        const int c0 = (FMT == 0) ? kMagicBits - 8 * xs[size_t(t) * nb + b] : kMagicBits;
        const int c = (FMT == 0 || FMT == 3) ? dot_q4(w0, xl, xh, c0) : dot_q8(w0, w1, xl, xh, c0);
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

static int qbytes_of(int fmt) { return (fmt == 0 || fmt == 3) ? 16 : (fmt == 1 ? 32 : (fmt == 4 ? 20 : 24)); }
// weight bytes per row group beyond the codes and the per-block 2-byte plane: Q6's super-block d
static int64_t dbytes_per_row(int64_t cols, int fmt) { return fmt == 2 ? (cols / 256) * 2 : ((fmt == 3 || fmt == 4) ? (cols / 256) * 4 : 0); }

// Lanes per row group: a function of (cols, fmt) only, so every launch of a shape (any T, single or
// grouped) sums each row in the same order. As few lanes as keep at least the format's
// kMinBlocksPerLane blocks per lane (fewer lanes per row = a shorter tree per row and more blocks
// folded between reductions): for Q4, 16 lanes for rows of 2,048 values, 32 for 4,096 and 6,144, 64
// for 8,192.
// The blocks each lane keeps at least, per format (Q4, Q8, Q6, Q4K, Q5K): the GB300 sweep's winners
// over 2, 3 and 4 on the verify window's 48 layers at T = 2 and 4 (Q8: the vocabulary head).
constexpr int kMinBlocksPerLane[5] = {4, 2, 2, 4, 3};

int gemv_lanes_per_row(int64_t cols, int fmt)
{
    const int64_t nb = cols / kQK;
    const int minb = kMinBlocksPerLane[(fmt >= 0 && fmt < 5) ? fmt : 0];
    int lpr = STRATA_LPR_MIN;
    while (lpr < STRATA_LPR_MAX && nb >= int64_t(minb) * lpr * 2) lpr *= 2;
    return lpr;
}

// Chunks per ring stage: at most the group count (every group gets at most one row group of a
// stage), about STRATA_STAGE_KB of codes and scales; a power of two when STRATA_SG_POW2 is set.
#ifndef STRATA_STAGE_KB_HEAD
#define STRATA_STAGE_KB_HEAD 36
#endif
#ifndef STRATA_STAGE_KB_HI_T
#define STRATA_STAGE_KB_HI_T 48
#endif
// stage size cap (it only schedules work): the head (one long Q8 matrix) prefers smaller stages up
// to T = 4; from T = 5 the wider activation records leave less room, and 48 KB stages beat 60 KB
// (the T = 8 window: 541 -> 512 us)
static int stage_kb(int T, bool head)
{
    if (head) return T <= 4 ? STRATA_STAGE_KB_HEAD : STRATA_STAGE_KB;
    return T >= 5 ? STRATA_STAGE_KB_HI_T : STRATA_STAGE_KB;
}

static int stage_chunks(int64_t cols, int fmt, int lpr, int kCW, int stage_kb_cap)
{
    const int64_t chunk = int64_t(kR) * ((cols / kQK) * (qbytes_of(fmt) + 2) + dbytes_per_row(cols, fmt));
    const int ng = lpr < 32 ? 2 * kCW : kCW / (lpr / 32);  // row groups a CTA works on at once
    if (STRATA_SG_POW2) {
        int l = 0;
        while ((2 << l) <= ng && chunk * (2 << l) <= (int64_t(stage_kb_cap) << 10)) ++l;
        return 1 << l;
    }
    int sg = int(std::min<int64_t>(ng, (int64_t(stage_kb_cap) << 10) / chunk));
    // half-warp groups: an even count, so that a stage's groups start on an even group and fill both
    // halves of each warp they use (an odd start leaves one half of a warp idle for that stage)
    if (lpr < 32 && sg >= 2) sg &= ~1;
    return std::max(sg, 1);
}

struct Plan {
    int cstage, sstage, dstage, ns, nb_max;
    size_t smem;
};

constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kRingBudget = size_t(STRATA_RING_KB) << 10;
constexpr int kPrefetchStages = STRATA_PF_STAGES;

// Shared-memory plan: activation copy + fixed scratch + a ring of stages (sizes: the largest over
// the launch's matrices), as many stages as fit in kRingBudget and shared memory (at least one).
static Plan plan_for(int T, const GemvMat* ms, int n, int fmt, bool head = false)
{
    Plan pl;
    size_t cmax = 0, smax = 0, dmax = 0;
    int nb_max = 0;
    for (int i = 0; i < n; ++i) {
        const size_t rows = size_t(ms[i].sg) * kR;
        cmax = std::max(cmax, rows * ms[i].nb * qbytes_of(fmt));
        smax = std::max(smax, rows * ms[i].nb * 2);
        dmax = std::max(dmax, rows * size_t(dbytes_per_row(int64_t(ms[i].nb) * kQK, fmt)));
        nb_max = std::max(nb_max, ms[i].nb);
    }
    pl.nb_max = nb_max;
    pl.cstage = int((cmax + 127) & ~size_t(127));
    pl.sstage = int((smax + 32 + 127) & ~size_t(127));
    pl.dstage = (fmt == 2 || fmt == 3 || fmt == 4) ? int((dmax + 32 + 127) & ~size_t(127)) : 0;
    const int cw = cw_for(T, head);
    // barriers, activation records, the cross-warp sums, the head's candidate slots (two per lane when
    // a half-warp group holds more sums than lanes, T > 4)
    const size_t fixed = 2 * 8 * 32 + size_t(nb_max) * xrec_bytes(T, fmt) + size_t(2 * cw * 32) * 4 +
                         size_t(cw * 32) * 12 * ((head && T > 4) ? 2 : 1);
    const size_t base = ((fixed + 127) & ~size_t(127)) + 128;
    const size_t per = size_t(pl.cstage) + pl.sstage + pl.dstage;
    const size_t room = base < kSmemLimit ? kSmemLimit - base : 0;
    int ns = int(std::min(kRingBudget, room) / per);
    ns = std::min(ns, 32);
    int pw = 1;
    while (pw * 2 <= ns) pw *= 2;
    pl.ns = ns >= 1 ? (STRATA_NST_POW2 ? pw : ns) : 0;
    pl.smem = base + size_t(std::max(pl.ns, 0)) * per;
    return pl;
}

static bool shape_fits_as(int64_t cols, int fmt, int T, bool head)
{
    GemvMat m = {};
    m.nb = int(cols / kQK);
    m.lpr = gemv_lanes_per_row(cols, fmt);
    m.sg = stage_chunks(cols, fmt, m.lpr, cw_for(T, head), stage_kb(T, head));
    const Plan pl = plan_for(T, &m, 1, fmt, head);
    return pl.ns >= 1 && pl.smem <= kSmemLimit;
}

// the shape can be launched both as a GEMV and as a head
bool gemv_shape_fits(int64_t cols, int fmt, int T)
{
    return shape_fits_as(cols, fmt, T, false) && shape_fits_as(cols, fmt, T, true);
}

template <int FMT, int T, int MAXM, bool HEAD>
static cudaError_t launch_gemv(GemvParams<MAXM>& prm, const Plan& pl, int grid, cudaStream_t stream)
{
    prm.cstage = pl.cstage;
    prm.sstage = pl.sstage;
    prm.dstage = pl.dstage;
    prm.nst = pl.ns;
    prm.nb_max = pl.nb_max;
    prm.pf = kPrefetchStages;
    auto kern = gemv_kernel<FMT, T, MAXM, HEAD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3((cw_for(T, HEAD) + 1) * 32), pl.smem, stream, prm);
}

static GemvMat make_mat(const void* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq, const float* xd,
                        const int32_t* xs, float* y, int chunk0, int T)
{
    GemvMat m;
    m.W = static_cast<const uint8_t*>(W);
    m.xq = xq;
    m.xd = xd;
    m.xs = xs;
    m.y = y;
    m.rows = int(rows);
    m.nb = int(cols / kQK);
    m.lpr = gemv_lanes_per_row(cols, fmt);
    m.sg = stage_chunks(cols, fmt, m.lpr, cw_for(T), stage_kb(T, false));
    m.chunk0 = chunk0;
    return m;
}

template <int FMT, int T, bool HEAD>
static cudaError_t single_t(const GemvMat& m, float* cv, int* ci, cudaStream_t stream, int* grid_out)
{
    GemvParams<1> prm = {};
    prm.n_mat = 1;
    prm.n_chunk = (m.rows + kR - 1) / kR;
    GemvMat mm = m;
    if (HEAD) mm.sg = stage_chunks(int64_t(m.nb) * kQK, FMT, m.lpr, cw_for(T, true), stage_kb(T, true));
    const int grid = std::min(prm.n_chunk, kCtasPerSm * device_sm_count());
    prm.m[0] = mm;
    prm.cand_val = cv;
    prm.cand_idx = ci;
    prm.cand_sec = (HEAD && ci) ? reinterpret_cast<float*>(ci + size_t(grid) * T) : nullptr;  // [T][grid] after ids
    if (grid_out) *grid_out = grid;
    if (HEAD && cv == nullptr) return cudaSuccess;  // size query
    const Plan pl = plan_for(T, &mm, 1, FMT, HEAD);
    if (pl.ns < 1) return cudaErrorInvalidValue;
    return launch_gemv<FMT, T, 1, HEAD>(prm, pl, grid, stream);
}

template <int FMT, bool HEAD>
static cudaError_t single_f(const GemvMat& m, int T, float* cv, int* ci, cudaStream_t s, int* g)
{
    switch (T) {
        case 1: return single_t<FMT, 1, HEAD>(m, cv, ci, s, g);
        case 2: return single_t<FMT, 2, HEAD>(m, cv, ci, s, g);
        case 3: return single_t<FMT, 3, HEAD>(m, cv, ci, s, g);
        case 4: return single_t<FMT, 4, HEAD>(m, cv, ci, s, g);
        case 5: return single_t<FMT, 5, HEAD>(m, cv, ci, s, g);
        case 6: return single_t<FMT, 6, HEAD>(m, cv, ci, s, g);
        case 7: return single_t<FMT, 7, HEAD>(m, cv, ci, s, g);
        case 8: return single_t<FMT, 8, HEAD>(m, cv, ci, s, g);
        default: return cudaErrorInvalidValue;
    }
}

static cudaError_t single(const GemvMat& m, int fmt, int T, bool head, float* cv, int* ci, cudaStream_t s, int* g)
{
    if (fmt == 0) return head ? single_f<0, true>(m, T, cv, ci, s, g) : single_f<0, false>(m, T, cv, ci, s, g);
    if (fmt == 2) return head ? single_f<2, true>(m, T, cv, ci, s, g) : single_f<2, false>(m, T, cv, ci, s, g);
    if (fmt == 3) return head ? single_f<3, true>(m, T, cv, ci, s, g) : single_f<3, false>(m, T, cv, ci, s, g);
    if (fmt == 4) return head ? single_f<4, true>(m, T, cv, ci, s, g) : single_f<4, false>(m, T, cv, ci, s, g);
    return head ? single_f<1, true>(m, T, cv, ci, s, g) : single_f<1, false>(m, T, cv, ci, s, g);
}

cudaError_t launch_mmvq(const void* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq,
                        const float* xd, const int32_t* xs, int T, float* y, cudaStream_t stream)
{
    const GemvMat m = make_mat(W, rows, cols, fmt, xq, xd, xs, y, 0, T);
    return single(m, fmt, T, false, nullptr, nullptr, stream, nullptr);
}

// ---- grouped launch ---------------------------------------------------------------------------------
template <int FMT, int T>
static cudaError_t grouped_t(const strata_gemv_desc* d, int n, cudaStream_t stream)
{
    GemvParams<kMaxGroup> prm;
    prm.n_mat = n;
    prm.cand_val = nullptr;
    prm.cand_idx = nullptr;
    prm.cand_sec = nullptr;
    int chunks = 0;
    std::vector<double> cum(1, 0.0);
    for (int i = 0; i < n; ++i) {
        prm.m[i] = make_mat(d[i].W, d[i].rows, d[i].cols, FMT, d[i].xq, d[i].xd, d[i].xs, d[i].y, chunks, T);
        const int nc = int((d[i].rows + kR - 1) / kR);
        const double cb = double(kR) * ((d[i].cols / kQK) * (qbytes_of(FMT) + 2) + dbytes_per_row(d[i].cols, FMT));
        for (int c = 0; c < nc; ++c) cum.push_back(cum.back() + cb);
        chunks += nc;
    }
    prm.n_chunk = chunks;
    const int grid = std::min(std::min(chunks, kCtasPerSm * device_sm_count()), kMaxGrid);
    // split the chunk sequence into `grid` runs of about equal bytes
    int c = 0;
    for (int b = 0; b <= grid; ++b) {
        const double target = cum.back() * b / grid;
        while (c < chunks && cum[c] < target) ++c;
        prm.plan[b] = (b == grid) ? chunks : c;
    }
    const Plan pl = plan_for(T, prm.m, n, FMT);
    if (pl.ns < 1) return cudaErrorInvalidValue;
    return launch_gemv<FMT, T, kMaxGroup, false>(prm, pl, grid, stream);
}

template <int FMT>
static cudaError_t grouped_f(const strata_gemv_desc* d, int n, int T, cudaStream_t s)
{
    switch (T) {
        case 1: return grouped_t<FMT, 1>(d, n, s);
        case 2: return grouped_t<FMT, 2>(d, n, s);
        case 3: return grouped_t<FMT, 3>(d, n, s);
        case 4: return grouped_t<FMT, 4>(d, n, s);
        case 5: return grouped_t<FMT, 5>(d, n, s);
        case 6: return grouped_t<FMT, 6>(d, n, s);
        case 7: return grouped_t<FMT, 7>(d, n, s);
        case 8: return grouped_t<FMT, 8>(d, n, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mmvq_grouped(const strata_gemv_desc* d, int n, int fmt, int T, cudaStream_t stream)
{
    if (fmt == 2) return grouped_f<2>(d, n, T, stream);
    if (fmt == 3) return grouped_f<3>(d, n, T, stream);
    if (fmt == 4) return grouped_f<4>(d, n, T, stream);
    return fmt == 0 ? grouped_f<0>(d, n, T, stream) : grouped_f<1>(d, n, T, stream);
}

// ---- head ---------------------------------------------------------------------------------------------
static int head_grid(int64_t vocab)
{
    const int64_t chunks = (vocab + kR - 1) / kR;
    return int(std::min<int64_t>(chunks, int64_t(kCtasPerSm) * device_sm_count()));
}

// per-CTA candidates: values, row ids and second values, each [T][grid]
size_t head_launch_scratch_bytes(int64_t vocab, int T)
{
    return size_t(head_grid(vocab)) * size_t(T) * 12;
}

// the head grid is at most one CTA per SM; bound it without a device for the workspace query
static int head_grid_bound(int64_t vocab)
{
    const int64_t chunks = (vocab + kR - 1) / kR;
    return int(std::min<int64_t>(chunks, kMaxGrid));
}

size_t head_workspace_bytes(int64_t vocab, int T)
{
    return size_t(head_grid_bound(vocab)) * size_t(T) * 12 + 256;
}

cudaError_t launch_head_argmax(const void* W, int64_t vocab, int64_t cols, int fmt, const int8_t* xq,
                               const float* xd, const int32_t* xs, int T, int32_t* ids, float* margin,
                               float* logits, void* workspace, cudaStream_t stream)
{
    const GemvMat m = make_mat(W, vocab, cols, fmt, xq, xd, xs, logits, 0, T);
    const int grid = head_grid(vocab);
    if (grid > head_grid_bound(vocab)) return cudaErrorInvalidValue;
    float* cv = static_cast<float*>(workspace);
    int* ci = reinterpret_cast<int*>(static_cast<char*>(workspace) + size_t(grid) * T * 4);
    int g2 = 0;
    cudaError_t e = single(m, fmt, T, true, cv, ci, stream, &g2);
    if (e != cudaSuccess) return e;
    const float* cs = reinterpret_cast<const float*>(ci + size_t(grid) * T);
    return launch_pdl(head_finalize_kernel, dim3(1), dim3(32 * T), 0, stream, (const float*)cv, (const int*)ci,
                      cs, grid, T, ids, margin);
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
    if (fmt == 3)
        return launch_pdl(block_dots_kernel<3>, dim3(grid), dim3(256), 0, stream, w, int(rows), nb, xq, xs, T, isum);
    if (fmt == 2)
        return launch_pdl(block_dots_kernel<2>, dim3(grid), dim3(256), 0, stream, w, int(rows), nb, xq, xs, T, isum);
    if (fmt == 4)
        return launch_pdl(block_dots_kernel<4>, dim3(grid), dim3(256), 0, stream, w, int(rows), nb, xq, xs, T, isum);
    return launch_pdl(block_dots_kernel<1>, dim3(grid), dim3(256), 0, stream, w, int(rows), nb, xq, xs, T, isum);
}

cudaError_t read_device_error_gemv(int* out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_strata_device_error, sizeof(int));
    if (e != cudaSuccess || !clear) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_strata_device_error, &zero, sizeof(int));
}

}  // namespace strata
