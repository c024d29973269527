// internal.h — launchers shared between the kernel translation units and the C-ABI layer.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <utility>

#include "strata.h"

namespace strata {

// Launch with programmatic stream serialization: the kernel may start while the previous kernel on
// the stream is finishing; it orders itself with griddepcontrol.wait before touching activations,
// outputs or workspace.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int device_sm_count();  // SMs of the current device (cached per device)

cudaError_t launch_quantize_act(const float* x, int64_t n_rows, int64_t cols, int8_t* xq, float* xd,
                                int32_t* xs, cudaStream_t stream);

// y may be null only when head candidates are requested (cand_val != null).
cudaError_t launch_mmvq(const void* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq,
                        const float* xd, const int32_t* xs, int T, float* y, cudaStream_t stream);

size_t head_workspace_bytes(int64_t vocab, int T);
size_t head_launch_scratch_bytes(int64_t vocab, int T);  // bytes one launch uses on the current device
cudaError_t launch_head_argmax(const void* W, int64_t vocab, int64_t cols, int fmt, const int8_t* xq,
                               const float* xd, const int32_t* xs, int T, int32_t* ids, float* margin,
                               float* logits, void* workspace, cudaStream_t stream);

// many independent matrices of one format in one persistent launch
cudaError_t launch_mmvq_grouped(const strata_gemv_desc* d, int n, int fmt, int T, cudaStream_t stream);
constexpr int kMaxGroupedMatrices = 192;
// warps per row of the GEMV for a shape (fixes the fp32 summation order; independent of T)
int gemv_lanes_per_row(int64_t cols, int fmt);
// whether the shared-memory plan of a shape fits at T
bool gemv_shape_fits(int64_t cols, int fmt, int T);
// device error word: bit 0 = a bounded wait in a kernel ran out (the OR of every unit's copy)
cudaError_t read_device_error(int* out, bool clear);
cudaError_t read_device_error_gemv(int* out, bool clear);
cudaError_t read_device_error_moe(int* out, bool clear);
cudaError_t read_device_error_probe(int* out, bool clear);
cudaError_t read_device_error_gemm(int* out, bool clear);
// test hook: one CTA waits, bounded by limit_ns, on an mbarrier nobody arrives at (abort_after_ns
// >= 0: a second warp raises the CTA's abort flag after that long instead)
cudaError_t launch_wait_probe(int64_t limit_ns, int64_t abort_after_ns, cudaStream_t stream);

cudaError_t launch_block_dots(const void* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq,
                              const int32_t* xs, int T, int32_t* isum, cudaStream_t stream);

// largest T * cols the GEMV kernels stage in shared memory
constexpr int64_t kMaxStagedTCols = 131072;
// the head's per-lane candidates carry the token in bits 27-29 of the row id, so vocab < 2^27
constexpr int64_t kHeadMaxVocab = int64_t(1) << 27;

// ---- prompt-chunk MoE ----------------------------------------------------------------------------
// Byte offsets of the sections of a strata_moe_grouped workspace (each 256-byte aligned).
struct MoeLayout {
    size_t xq, xd, xs;              // quantized x: int8 [n_tok][hidden], fp32/int32 [n_tok][hidden/32]
    size_t counts, offsets, pairs;  // int32 [n_expert], [n_expert+1], [n_tok*k]
    size_t hq, hd, hs;              // re-quantized hidden rows by pair position: [n_pair][inter], [n_pair][inter/32]
    size_t mcum;                    // int32 [n_expert+1]: running count of 128-row M-tiles
    size_t total;
};
MoeLayout moe_workspace_layout(int n_expert, int64_t n_tok, int k, int64_t hidden, int64_t inter);

struct ExpertPtrs;  // device-side view of strata_expert (three const void*)
// gu (may be null): fp32 [n_tok*k][2][inter], the gate then the up outputs of every valid pair
cudaError_t launch_moe_grouped(const void* experts, int n_expert, int64_t hidden, int64_t inter,
                               const int32_t* ids, int64_t n_tok, int k, const float* x, float* y,
                               uint8_t* ws, const MoeLayout& L, int32_t* err_word, float* gu,
                               cudaStream_t stream);
cudaError_t launch_prompt_gemm(const void* W, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                               int64_t n_tok, float* y, cudaStream_t stream);
// the prompt GEMM's wide-dequant arm (gemm_dequant.cu)
size_t gemm_dequant_workspace_bytes(int64_t rows, int64_t cols, int64_t n_tok);
cudaError_t launch_gemm_dequant(const void* W, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                                int64_t n_tok, float* y, void* workspace, cudaStream_t stream);

}  // namespace strata
