// noalloc.cu -- attn_fp8_fwd_noalloc: the FP8 forward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run attention: a host that hands out all device memory itself and
// forbids extra allocations, a plugin running inside another runtime's
// stream-ordered region, or a latency-critical path where an allocation could
// synchronise the device. The regular attn_fp8_fwd needs a caller-provided
// workspace for its document table, work list and V reference scales. This
// entry point instead keeps that scratch in one file-scope device array of
// fixed size that every GPU loading the library holds until the process exits.
//
// Set-up: the first call on each device (with that device current) looks up
// the array's device address with cudaGetSymbolAddress, and looks it up again
// if the device's context has changed since; make that first call before any
// stream capture. Every call shares the one array and leaves its
// contents behind; calls whose work overlaps on the GPU (different streams,
// no ordering between them) race on it.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "params.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mu;

// The array's device address is a property of the module as loaded into one
// context: cache it per device together with the context it was looked up in,
// and look it up again when the device's current context is another one (after
// a cudaDeviceReset, for instance, the module is loaded afresh).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    return fn;
}

struct ScratchSlot {
    CUcontext ctx;
    void* ptr;
};
ScratchSlot g_slot[kMaxDevices] = {};

// device address of the scratch array on the current device
attn_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    CUcontext ctx = nullptr;   // null until the runtime has made the device's context current
    CtxGetCurrentFn get = ctx_get_current();
    if (!get || get(&ctx) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_slot[dev].ptr || g_slot[dev].ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS) return ATTN_ERR_CUDA;   // the lookup made the context current if it was not
        g_slot[dev].ctx = ctx;
        g_slot[dev].ptr = p;
    }
    *out = g_slot[dev].ptr;
    return ATTN_OK;
}

}  // namespace

namespace pa {
attn_status fp8_fwd_check(const attn_qtensor* q, const attn_qtensor* k, const attn_qtensor* v,
                          const attn_shape* shape, int causal, int causal_exact, float softmax_scale, const void* o,
                          const float* lse, bool check_workspace, void* workspace, size_t workspace_bytes,
                          int* mode);
}

extern "C" attn_status attn_fp8_fwd_noalloc(const attn_qtensor* q, const attn_qtensor* k, const attn_qtensor* v,
                                            const attn_shape* shape, int32_t causal, int32_t causal_exact,
                                            float softmax_scale, void* o, float* lse, uint32_t* status,
                                            void* stream) {
    // every argument check first: a refused call touches neither the array nor `status`
    int mode = 0;
    attn_status st =
        pa::fp8_fwd_check(q, k, v, shape, causal, causal_exact, softmax_scale, o, lse, false, nullptr, 0, &mode);
    if (st != ATTN_OK) return st;
    size_t need = 0;
    if ((st = attn_workspace_size(shape, &need)) != ATTN_OK) return st;
    if (need > kNoallocScratchBytes) return ATTN_ERR_UNSUPPORTED;   // shape needs more scratch than the array holds
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != ATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word must start at zero so that it reports this call only;
    // the document table, work list and V references are rewritten every call
    if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s) != cudaSuccess) return ATTN_ERR_CUDA;
    st = attn_fp8_fwd(q, k, v, shape, causal, causal_exact, softmax_scale, o, lse, scratch, kNoallocScratchBytes,
                      stream);
    if (st != ATTN_OK) return st;
    if (status && cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}
