// macaq_linear without a caller-provided workspace.
//
// The quantised activations that macaq_linear keeps between its two kernels
// normally live in a workspace the caller allocates.  Some callers have no
// way to allocate device memory at the point of the call: a plugin whose
// host framework owns every device allocation, or a runtime that fixes its
// device memory at start-up and forbids cudaMalloc afterwards.  For them the
// library keeps one scratch array of fixed size in its own module image, so
// the call needs nothing beyond the caller's inputs and outputs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "macaq.h"

namespace macaq {
namespace {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) uint8_t g_linear_scratch[MACAQ_LINEAR_STATIC_SCRATCH_BYTES];

// Device address of g_linear_scratch, looked up once per device with that
// device current.  The array's name in host code is only a host-side handle;
// its device address belongs to the CUDA context that loaded the module, so
// the entry also records that context: when a different context is current on
// the device (after cudaDeviceReset, or under a caller's own driver-API
// context) the address is looked up again instead of reusing a stale one.
struct ScratchEntry {
    CUcontext ctx = nullptr;
    void *addr = nullptr;
};
ScratchEntry g_scratch[64];
std::mutex g_scratch_mu;

// cuCtxGetCurrent through the runtime's driver entry-point query (the library
// does not link the driver library itself).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn ctx_get_current_fn()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    return fn;
}

cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (get_ctx == nullptr) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchEntry &e = g_scratch[dev];
    if (e.addr == nullptr || ctx == nullptr || e.ctx != ctx) {
        // with no context current yet, the lookup itself makes the device's
        // primary context current; the entry records whichever is current
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_linear_scratch);
        if (err != cudaSuccess) return err;
        if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
        e.ctx = ctx;
        e.addr = p;
    }
    *out = e.addr;
    return cudaSuccess;
}

}  // namespace
}  // namespace macaq

extern "C" macaq_status macaq_linear_no_alloc(const void *X, int64_t ldx, const float *inv_s,
                                              const uint8_t *w_codes, const uint8_t *w_scales,
                                              int64_t M, int64_t N, int64_t K, void *Y,
                                              int64_t ldy, macaq_stream_t stream)
{
    if (K <= 0 || K % 32 != 0 || M < 0 || N < 0) return MACAQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return MACAQ_OK;
    const size_t need = macaq_linear_workspace_bytes(M, K);
    if (need == 0 || need > MACAQ_LINEAR_STATIC_SCRATCH_BYTES) return MACAQ_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (macaq::scratch_address(&scratch) != cudaSuccess) return MACAQ_ERR_CUDA;
    // macaq_linear checks every other argument; its quantisation kernel
    // writes every scratch byte the GEMM then reads (up to 6 token rows the
    // layer is one kernel that uses no scratch), so the contents left by an
    // earlier call need no clearing.
    return macaq_linear(X, ldx, inv_s, w_codes, w_scales, M, N, K, Y, ldy, scratch,
                        MACAQ_LINEAR_STATIC_SCRATCH_BYTES, stream);
}
