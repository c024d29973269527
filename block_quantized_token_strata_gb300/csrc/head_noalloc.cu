// head_noalloc.cu — strata_head_argmax_noalloc: the vocabulary head + argmax for callers that
// cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not available or not allowed — a plugin inside a
// host application that owns all device memory and hands out no allocator, a serving process that
// reserves its memory budget at start-up and forbids any later allocation, or a caller that only
// ever enqueues work into an existing stream and cannot create or size a scratch buffer. Such a
// caller still passes its inputs and outputs; the per-CTA candidates the argmax needs live in a
// fixed array inside this library instead of a caller-provided workspace.
//
// The scratch is one file-scope __device__ array of kNoallocScratchBytes (64 KiB). Every device
// that loads the library holds it until the process exits. Its device address is looked up with the
// device current on the first call made in each CUDA context (normally once per device: the
// runtime's primary context); make that first call before any stream capture. A device reset
// (cudaDeviceReset) ends the context, and the next call then looks the address up again in the new
// one. All calls share the array, and it keeps whatever the last call wrote: every candidate slot a
// call reads is written by the same call first, so nothing needs clearing, but two calls whose
// kernels overlap on the GPU (different streams, no ordering between them) race on it and may
// return wrong ids.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "strata.h"
#include "internal.h"

using namespace strata;

namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 10;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_head_scratch[kNoallocScratchBytes];

struct ScratchSlot {
    unsigned long long ctx_id;  // the CUDA context the address belongs to
    void* addr;
};
std::mutex g_mu;
ScratchSlot g_slot[kMaxDevices] = {};

// The id of the calling thread's current CUDA context. The two driver calls are looked up through
// the runtime on first use, so that the library does not link the driver library itself (it loads
// and answers host-side argument checks on machines without a GPU driver).
bool current_context_id(unsigned long long* id)
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    if (get_current == nullptr || get_id == nullptr) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
            return false;
        get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
        get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
    }
    CUcontext ctx = nullptr;
    return get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr && get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_head_scratch in the current device's current context. The name is only a
// host-side stand-in for the array, so the address must come from the runtime; it is cached per
// device together with the id of the context it was taken in.
int scratch_address(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return STRATA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long id = 0;
    if (current_context_id(&id) && g_slot[dev].addr != nullptr && g_slot[dev].ctx_id == id) {
        *out = g_slot[dev].addr;
        return STRATA_OK;
    }
    void* p = nullptr;  // the lookup makes the runtime's context current if none was yet
    if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess || p == nullptr) return STRATA_ERR_CUDA;
    if (!current_context_id(&id)) return STRATA_ERR_CUDA;
    g_slot[dev].ctx_id = id;
    g_slot[dev].addr = p;
    *out = p;
    return STRATA_OK;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int strata_head_argmax_noalloc(const void* W, int64_t vocab, int64_t cols, int fmt, const int8_t* xq,
                                          const float* xd, const int32_t* xs, int T, int32_t* ids, float* logits,
                                          cudaStream_t stream)
{
    if (!W || !ids || !xq || !xd || !xs) return STRATA_ERR_NULL;
    if (fmt != STRATA_Q4 && fmt != STRATA_Q8) return STRATA_ERR_FMT;
    if (vocab <= 0 || cols < 32 || cols % 32 != 0 || vocab >= kHeadMaxVocab || cols > 65536) return STRATA_ERR_SHAPE;
    if (T < 1 || T > STRATA_MAX_T) return STRATA_ERR_T;
    if (int64_t(T) * cols > kMaxStagedTCols || !gemv_shape_fits(cols, fmt, T)) return STRATA_ERR_SHAPE;
    if (!is_aligned(W, 16) || !is_aligned(xq, 16) || !is_aligned(xd, 4) || !is_aligned(xs, 4) ||
        !is_aligned(ids, 4) || (logits && !is_aligned(logits, 4)))
        return STRATA_ERR_ALIGN;
    if (head_launch_scratch_bytes(vocab, T) > kNoallocScratchBytes) return STRATA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != STRATA_OK) return st;
    const cudaError_t e = launch_head_argmax(W, vocab, cols, fmt, xq, xd, xs, T, ids, nullptr, logits, scratch, stream);
    return e == cudaSuccess ? STRATA_OK : STRATA_ERR_CUDA;
}
