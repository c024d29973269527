// quantize.cu — fp32 activations to int8 blocks of 32 with an fp32 scale and an exact block sum.
//
// Per 32-block: amax = max|x_j|, d = amax/127, id = (d != 0) ? 1/d : 0, q_j = roundf(x_j*id),
// s = sum q_j — the activation format of the verify window's multi-column MMVQ ("T columns of
// q8_1", member xq_ of verify.hpp in the Strata commit "wire multi-token kernels into Verifier and
// MtpDrafter CUDA graphs"), with an fp32 scale. Every step is one correctly rounded IEEE fp32
// operation (__fdiv_rn, __frcp_rn, __fmul_rn, roundf), so the codes are reproducible exactly.
//
// Layout: eight lanes own one block (one float4 each); the block maximum and sum are combined
// with three xor shuffles inside the eight-lane group. Loads are 128-bit and coalesced.
#include "common.cuh"
#include "internal.h"

namespace strata {

__global__ void __launch_bounds__(256)
quantize_act_kernel(const float4* __restrict__ x, int64_t nblk, int* __restrict__ xq,
                    float* __restrict__ xd, int32_t* __restrict__ xs)
{
    pdl_launch();   // the next kernel may launch and stream its weights meanwhile
    pdl_wait();     // x may be the output of the kernel ahead of this one
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t blk = gid >> 3;
    const int sub = threadIdx.x & 7;
    const bool valid = blk < nblk;
    const float4 v = valid ? x[blk * 8 + sub] : make_float4(0.f, 0.f, 0.f, 0.f);

    float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));

    const float d = __fdiv_rn(a, 127.0f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    const int q0 = int(roundf(__fmul_rn(v.x, id)));
    const int q1 = int(roundf(__fmul_rn(v.y, id)));
    const int q2 = int(roundf(__fmul_rn(v.z, id)));
    const int q3 = int(roundf(__fmul_rn(v.w, id)));

    int s = q0 + q1 + q2 + q3;
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);

    if (valid) {
        xq[blk * 8 + sub] = (q0 & 0xFF) | ((q1 & 0xFF) << 8) | ((q2 & 0xFF) << 16) | (int(unsigned(q3) << 24));
        if (sub == 0) {
            xd[blk] = d;
            xs[blk] = s;
        }
    }
}

cudaError_t launch_quantize_act(const float* x, int64_t n_rows, int64_t cols, int8_t* xq, float* xd,
                                int32_t* xs, cudaStream_t stream)
{
    const int64_t nblk = n_rows * (cols / kQK);
    const int64_t threads = nblk * 8;
    const unsigned grid = unsigned((threads + 255) / 256);
    return launch_pdl(quantize_act_kernel, dim3(grid), dim3(256), 0, stream,
                      reinterpret_cast<const float4*>(x), nblk, reinterpret_cast<int*>(xq), xd, xs);
}

}  // namespace strata
