// abi.cu — the extern "C" entry points of libstrata: argument checks on the host, then launches.
// Every check runs before any CUDA call, so a rejected call touches neither the device nor the
// stream. Declarations and the contract of each call are in include/strata.h.
#include <limits.h>

#include "strata.h"
#include "internal.h"

using namespace strata;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? STRATA_OK : STRATA_ERR_CUDA; }

}  // namespace

namespace strata {
// the device error word as the C ABI reports it: the copies of every translation unit whose kernels
// set it, ORed
cudaError_t read_device_error(int* out, bool clear)
{
    int a = 0, b = 0, c = 0, d = 0;
    cudaError_t e = read_device_error_gemv(&a, clear);
    if (e == cudaSuccess) e = read_device_error_moe(&b, clear);
    if (e == cudaSuccess) e = read_device_error_probe(&c, clear);
    if (e == cudaSuccess) e = read_device_error_gemm(&d, clear);
    *out = a | b | c | d;
    return e;
}
}  // namespace strata

namespace {

int check_matrix(int64_t rows, int64_t cols, int fmt)
{
    if (fmt != STRATA_Q4 && fmt != STRATA_Q8 && fmt != STRATA_Q6 && fmt != STRATA_Q4K && fmt != STRATA_Q5K)
        return STRATA_ERR_FMT;
    if (rows <= 0 || cols < 32 || cols % 32 != 0) return STRATA_ERR_SHAPE;
    if ((fmt == STRATA_Q6 || fmt == STRATA_Q4K || fmt == STRATA_Q5K) && cols % 256 != 0) return STRATA_ERR_SHAPE;
    if (rows > INT_MAX / 2 || cols > 65536) return STRATA_ERR_SHAPE;
    return STRATA_OK;
}

int check_acts(const int8_t* xq, const float* xd, const int32_t* xs)
{
    if (!xq || !xd || !xs) return STRATA_ERR_NULL;
    if (!aligned(xq, 16) || !aligned(xd, 4) || !aligned(xs, 4)) return STRATA_ERR_ALIGN;
    return STRATA_OK;
}

}  // namespace

extern "C" {

const char* strata_error_string(int status)
{
    switch (status) {
        case STRATA_OK: return "ok";
        case STRATA_ERR_NULL: return "a required pointer is NULL";
        case STRATA_ERR_SHAPE: return "bad shape (cols % 32 != 0, a size <= 0, or above a stated maximum)";
        case STRATA_ERR_T: return "T outside [1, 8]";
        case STRATA_ERR_FMT: return "unknown or unsupported block format";
        case STRATA_ERR_CUDA: return "CUDA launch or attribute call failed";
        case STRATA_ERR_EXPERT: return "expert id outside [0, n_expert)";
        case STRATA_ERR_ALIGN: return "pointer not aligned as required";
        case STRATA_ERR_WORKSPACE: return "workspace NULL or too small";
        default: return "unknown status";
    }
}

size_t strata_weight_bytes(int64_t rows, int64_t cols, int fmt)
{
    if (check_matrix(rows, cols, fmt) != STRATA_OK) return 0;
    if (fmt == STRATA_Q6) return size_t(rows) * size_t(cols / 256) * 210u;
    if (fmt == STRATA_Q4K) return size_t(rows) * size_t(cols / 256) * 148u;
    if (fmt == STRATA_Q5K) return size_t(rows) * size_t(cols / 256) * 180u;
    return size_t(rows) * size_t(cols / 32) * (fmt == STRATA_Q4 ? 18u : 34u);
}

int strata_quantize_act(const float* x, int64_t n_rows, int64_t cols, int8_t* xq, float* xd, int32_t* xs,
                        cudaStream_t stream)
{
    if (!x || !xq || !xd || !xs) return STRATA_ERR_NULL;
    if (n_rows <= 0 || cols < 32 || cols % 32 != 0) return STRATA_ERR_SHAPE;
    if (n_rows > (int64_t(1) << 40) / cols) return STRATA_ERR_SHAPE;
    if (!aligned(x, 16) || !aligned(xq, 16) || !aligned(xd, 4) || !aligned(xs, 4)) return STRATA_ERR_ALIGN;
    return cuda_status(launch_quantize_act(x, n_rows, cols, xq, xd, xs, stream));
}

int strata_mmvq_multi(const void* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq, const float* xd,
                      const int32_t* xs, int T, float* y, cudaStream_t stream)
{
    if (!W || !y) return STRATA_ERR_NULL;
    int st = check_acts(xq, xd, xs);
    if (st != STRATA_OK) return st;
    st = check_matrix(rows, cols, fmt);
    if (st != STRATA_OK) return st;
    if (T < 1 || T > STRATA_MAX_T) return STRATA_ERR_T;
    if (int64_t(T) * cols > kMaxStagedTCols || !gemv_shape_fits(cols, fmt, T)) return STRATA_ERR_SHAPE;
    if (!aligned(W, 16) || !aligned(y, 4)) return STRATA_ERR_ALIGN;
    return cuda_status(launch_mmvq(W, rows, cols, fmt, xq, xd, xs, T, y, stream));
}

int strata_mmvq_grouped(const strata_gemv_desc* descs, int n, int fmt, int T, cudaStream_t stream)
{
    if (!descs) return STRATA_ERR_NULL;
    if (n < 1 || n > kMaxGroupedMatrices) return STRATA_ERR_SHAPE;
    if (fmt != STRATA_Q4 && fmt != STRATA_Q8 && fmt != STRATA_Q6 && fmt != STRATA_Q4K && fmt != STRATA_Q5K)
        return STRATA_ERR_FMT;
    if (T < 1 || T > STRATA_MAX_T) return STRATA_ERR_T;
    int64_t cols_max = 0, total_rows = 0;
    for (int i = 0; i < n; ++i) {
        const strata_gemv_desc& d = descs[i];
        if (!d.W || !d.y) return STRATA_ERR_NULL;
        int st = check_acts(d.xq, d.xd, d.xs);
        if (st != STRATA_OK) return st;
        st = check_matrix(d.rows, d.cols, fmt);
        if (st != STRATA_OK) return st;
        if (int64_t(T) * d.cols > kMaxStagedTCols || !gemv_shape_fits(d.cols, fmt, T)) return STRATA_ERR_SHAPE;
        if (!aligned(d.W, 16) || !aligned(d.y, 4)) return STRATA_ERR_ALIGN;
        cols_max = d.cols > cols_max ? d.cols : cols_max;
        total_rows += d.rows;
    }
    if (!gemv_shape_fits(cols_max, fmt, T) || total_rows > (int64_t(1) << 30)) return STRATA_ERR_SHAPE;
    return cuda_status(launch_mmvq_grouped(descs, n, fmt, T, stream));
}

int strata_device_error(int* out, int clear)
{
    if (!out) return STRATA_ERR_NULL;
    return cuda_status(read_device_error(out, clear != 0));
}

size_t strata_head_argmax_workspace(int64_t vocab, int T)
{
    if (vocab <= 0 || T < 1 || T > STRATA_MAX_T) return 0;
    return head_workspace_bytes(vocab, T);
}

static int head_call(const void* W, int64_t vocab, int64_t cols, int fmt, const int8_t* xq, const float* xd,
                     const int32_t* xs, int T, int32_t* ids, float* margin, float* logits, void* workspace,
                     size_t ws_bytes, cudaStream_t stream)
{
    if (!W || !ids) return STRATA_ERR_NULL;
    int st = check_acts(xq, xd, xs);
    if (st != STRATA_OK) return st;
    st = check_matrix(vocab, cols, fmt);
    if (st != STRATA_OK) return st;
    if (vocab >= kHeadMaxVocab) return STRATA_ERR_SHAPE;
    if (T < 1 || T > STRATA_MAX_T) return STRATA_ERR_T;
    if (int64_t(T) * cols > kMaxStagedTCols || !gemv_shape_fits(cols, fmt, T)) return STRATA_ERR_SHAPE;
    if (!aligned(W, 16) || !aligned(ids, 4) || (logits && !aligned(logits, 4)) || (margin && !aligned(margin, 4)))
        return STRATA_ERR_ALIGN;
    if (!workspace || ws_bytes < head_workspace_bytes(vocab, T)) return STRATA_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return STRATA_ERR_ALIGN;
    return cuda_status(launch_head_argmax(W, vocab, cols, fmt, xq, xd, xs, T, ids, margin, logits, workspace, stream));
}

int strata_head_argmax(const void* W, int64_t vocab, int64_t cols, int fmt, const int8_t* xq, const float* xd,
                       const int32_t* xs, int T, int32_t* ids, float* logits, void* workspace, size_t ws_bytes,
                       cudaStream_t stream)
{
    return head_call(W, vocab, cols, fmt, xq, xd, xs, T, ids, nullptr, logits, workspace, ws_bytes, stream);
}

int strata_head_argmax_margin(const void* W, int64_t vocab, int64_t cols, int fmt, const int8_t* xq,
                              const float* xd, const int32_t* xs, int T, int32_t* ids, float* margin,
                              float* logits, void* workspace, size_t ws_bytes, cudaStream_t stream)
{
    if (!margin) return STRATA_ERR_NULL;
    return head_call(W, vocab, cols, fmt, xq, xd, xs, T, ids, margin, logits, workspace, ws_bytes, stream);
}

int strata_gemm_q4(const void* W, int64_t rows, int64_t cols, const int8_t* xq, const float* xd, int64_t n_tok,
                   float* y, cudaStream_t stream)
{
    if (!W || !xq || !xd || !y) return STRATA_ERR_NULL;
    if (rows < 128 || rows % 128 != 0 || cols < 64 || cols % 64 != 0 || n_tok < 1) return STRATA_ERR_SHAPE;
    if (rows > 65536 || cols > 65536 || n_tok > (int64_t(1) << 24)) return STRATA_ERR_SHAPE;
    if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(xd, 4) || !aligned(y, 16)) return STRATA_ERR_ALIGN;
    return cuda_status(launch_prompt_gemm(W, rows, cols, xq, xd, n_tok, y, stream));
}

size_t strata_gemm_q4_dequant_workspace(int64_t rows, int64_t cols, int64_t n_tok)
{
    if (rows < 128 || rows % 128 != 0 || cols < 64 || cols % 64 != 0 || n_tok < 1) return 0;
    if (rows > 65536 || cols > 65536 || n_tok > (int64_t(1) << 24)) return 0;
    return gemm_dequant_workspace_bytes(rows, cols, n_tok);
}

int strata_gemm_q4_dequant(const void* W, int64_t rows, int64_t cols, const int8_t* xq, const float* xd,
                           int64_t n_tok, float* y, void* workspace, size_t ws_bytes, cudaStream_t stream)
{
    if (!W || !xq || !xd || !y) return STRATA_ERR_NULL;
    if (rows < 128 || rows % 128 != 0 || cols < 64 || cols % 64 != 0 || n_tok < 1) return STRATA_ERR_SHAPE;
    if (rows > 65536 || cols > 65536 || n_tok > (int64_t(1) << 24)) return STRATA_ERR_SHAPE;
    if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(xd, 4) || !aligned(y, 16)) return STRATA_ERR_ALIGN;
    if (!workspace || ws_bytes < gemm_dequant_workspace_bytes(rows, cols, n_tok)) return STRATA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return STRATA_ERR_ALIGN;
    return cuda_status(launch_gemm_dequant(W, rows, cols, xq, xd, n_tok, y, workspace, stream));
}

int strata_block_dots(const void* W, int64_t rows, int64_t cols, int fmt, const int8_t* xq, const int32_t* xs,
                      int T, int32_t* isum, cudaStream_t stream)
{
    if (!W || !xq || !xs || !isum) return STRATA_ERR_NULL;
    int st = check_matrix(rows, cols, fmt);
    if (st != STRATA_OK) return st;
    if (T < 1 || T > STRATA_MAX_T) return STRATA_ERR_T;
    if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(xs, 4) || !aligned(isum, 4)) return STRATA_ERR_ALIGN;
    return cuda_status(launch_block_dots(W, rows, cols, fmt, xq, xs, T, isum, stream));
}

size_t strata_moe_grouped_workspace(int n_expert, int64_t n_tok, int k, int64_t hidden, int64_t inter)
{
    if (n_expert < 1 || n_tok < 1 || k < 1 || k > 16 || hidden <= 0 || inter <= 0) return 0;
    if (hidden % 128 != 0 || inter % 128 != 0) return 0;
    return moe_workspace_layout(n_expert, n_tok, k, hidden, inter).total;
}

int strata_moe_debug_views(int n_expert, int64_t n_tok, int k, int64_t hidden, int64_t inter, size_t* out)
{
    if (!out) return STRATA_ERR_NULL;
    if (strata_moe_grouped_workspace(n_expert, n_tok, k, hidden, inter) == 0) return STRATA_ERR_SHAPE;
    const MoeLayout L = moe_workspace_layout(n_expert, n_tok, k, hidden, inter);
    out[0] = L.counts;
    out[1] = L.offsets;
    out[2] = L.pairs;
    out[3] = L.hq;
    out[4] = L.hd;
    out[5] = L.hs;
    out[6] = L.total;
    return STRATA_OK;
}

static int moe_call(const strata_expert* experts, int n_expert, int64_t hidden, int64_t inter,
                    const int32_t* ids, int64_t n_tok, int k, const float* x, float* y, void* workspace,
                    size_t ws_bytes, int32_t* err_word, float* gu, cudaStream_t stream)
{
    if (!experts || !ids || !x || !y) return STRATA_ERR_NULL;
    if (n_expert < 1 || n_tok < 1 || k < 1 || k > 16) return STRATA_ERR_SHAPE;
    if (hidden < 128 || inter < 128 || hidden % 128 != 0 || inter % 128 != 0) return STRATA_ERR_SHAPE;
    if (hidden > 16384 || inter > 16384 || n_tok * k > (int64_t(1) << 30)) return STRATA_ERR_SHAPE;
    if (!aligned(experts, 8) || !aligned(ids, 4) || !aligned(x, 16) || !aligned(y, 16)) return STRATA_ERR_ALIGN;
    if (err_word && !aligned(err_word, 4)) return STRATA_ERR_ALIGN;
    if (gu && !aligned(gu, 16)) return STRATA_ERR_ALIGN;
    const MoeLayout L = moe_workspace_layout(n_expert, n_tok, k, hidden, inter);
    if (!workspace || ws_bytes < L.total) return STRATA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return STRATA_ERR_ALIGN;
    return cuda_status(launch_moe_grouped(experts, n_expert, hidden, inter, ids, n_tok, k, x, y,
                                          static_cast<uint8_t*>(workspace), L, err_word, gu, stream));
}

int strata_moe_grouped(const strata_expert* experts, int n_expert, int64_t hidden, int64_t inter,
                       const int32_t* ids, int64_t n_tok, int k, const float* x, float* y, void* workspace,
                       size_t ws_bytes, int32_t* err_word, cudaStream_t stream)
{
    return moe_call(experts, n_expert, hidden, inter, ids, n_tok, k, x, y, workspace, ws_bytes, err_word,
                    nullptr, stream);
}

int strata_moe_grouped_gu(const strata_expert* experts, int n_expert, int64_t hidden, int64_t inter,
                          const int32_t* ids, int64_t n_tok, int k, const float* x, float* y, void* workspace,
                          size_t ws_bytes, int32_t* err_word, float* gu, cudaStream_t stream)
{
    if (!gu) return STRATA_ERR_NULL;
    return moe_call(experts, n_expert, hidden, inter, ids, n_tok, k, x, y, workspace, ws_bytes, err_word, gu,
                    stream);
}

int strata_wait_probe(int64_t limit_ns, int64_t abort_after_ns, cudaStream_t stream)
{
    if (limit_ns < 1 || limit_ns > 1000000000 || abort_after_ns > 1000000000) return STRATA_ERR_SHAPE;
    return cuda_status(launch_wait_probe(limit_ns, abort_after_ns < 0 ? -1 : abort_after_ns, stream));
}

}  // extern "C"
