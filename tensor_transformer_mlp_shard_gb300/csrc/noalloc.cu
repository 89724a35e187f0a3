// tp_linear_row_bwd_noalloc: the row-layer backward for callers that cannot
// allocate device memory.
//
// tp_linear_row_bwd takes a caller workspace: the token-chunk partial column
// sums of dY for the bias gradient and, for narrow layers, the split-K
// partial sums of the weight gradient and the tail-split scratch.  Some
// callers have no way to provide one: a plugin inside another framework is
// handed only the op's own tensors and has no allocator to ask; a process
// whose device memory is already fully reserved by another (caching)
// allocator can see cudaMalloc fail; and a latency-critical loop cannot
// afford cudaMalloc's implicit device synchronisation.  For them this entry
// point takes its scratch from a fixed array compiled into the library.
//
// The array is file-scope device memory of kScratchBytes.  Every GPU that
// loads the library holds it until the process exits.  Host code cannot use
// the array's name as a device address (in host code it is only a stand-in
// for the symbol), so the device address is looked up with
// cudaGetSymbolAddress while the device is current, once per device and CUDA
// context: a device reset gives the device a new context (and the module a
// new load), and the next call looks the address up again.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB

}  // namespace

static __device__ __align__(256) unsigned char tp_noalloc_scratch[kScratchBytes];

namespace {

struct ScratchAddr {
    unsigned long long ctx_id = 0;  // 0: not looked up yet
    void *ptr = nullptr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch[64];

// Unique ID of the calling thread's current CUDA context (never reused in a
// process), through the driver entry points the runtime exposes.
tp_status current_context_id(unsigned long long *id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return tpmlp::set_error(TP_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId unavailable");
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return tpmlp::set_error(TP_ERR_CUDA, "cuCtxGetCurrent failed");
    if (!ctx) {
        // no context yet on this thread: make the device's primary context
        // current (cudaSetDevice initialises it and allocates no memory)
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaSetDevice(dev);
        if (e != cudaSuccess) return tpmlp::cuda_check(e, "cudaSetDevice");
        if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return tpmlp::set_error(TP_ERR_CUDA, "no current CUDA context");
    }
    if (get_id(ctx, id) != CUDA_SUCCESS) return tpmlp::set_error(TP_ERR_CUDA, "cuCtxGetId failed");
    return TP_OK;
}

// Device address of the scratch array on the current device: set-up on the
// first call per device and context.
tp_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tpmlp::cuda_check(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return tpmlp::set_error(TP_ERR_UNSUPPORTED, "device ordinal %d above 63", dev);
    unsigned long long ctx = 0;
    tp_status s = current_context_id(&ctx);
    if (s != TP_OK) return s;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr &a = g_scratch[dev];
    if (a.ctx_id != ctx || !a.ptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, tp_noalloc_scratch);
        if (e != cudaSuccess) return tpmlp::cuda_check(e, "cudaGetSymbolAddress(tp_noalloc_scratch)");
        a.ptr = p;
        a.ctx_id = ctx;
    }
    *out = a.ptr;
    return TP_OK;
}

}  // namespace

extern "C" {

tp_status tp_linear_row_bwd_noalloc(const tp_mlp_desc *desc, const void *const *dY, const void *const *X,
                                    const void *const *W, void *const *dX, void *const *dW, void *db,
                                    void *stream) {
    // FP8 reads the quantised forward operands from the forward's workspace
    if (desc && desc->dtype == TP_DT_FP8)
        return tpmlp::set_error(TP_ERR_UNSUPPORTED,
                                "the FP8 backward reads the forward's codes from its workspace (tp_linear_row_bwd)");
    // the row layer's own bias partials (0 without a bias, or for an invalid
    // descriptor: the row backward then reports the error)
    const size_t need = tpmlp::linear_row_bias_bytes(desc);
    if (need > kScratchBytes)
        return tpmlp::set_error(TP_ERR_UNSUPPORTED,
                                "bias gradient needs %zu bytes of scratch; the built-in scratch holds %zu "
                                "(use tp_linear_row_bwd with a caller workspace)",
                                need, kScratchBytes);
    // When the whole single-layer workspace fits, the array serves as one:
    // the same plan as tp_linear_row_bwd (split-K and tail split included).
    // Otherwise the weight gradient runs without either split and the array
    // holds only the bias partials.
    const size_t full = tp_linear_workspace_bytes(desc);
    const bool split = full <= kScratchBytes;
    void *ws = nullptr;
    if (split ? full : need) {
        tp_status s = scratch_address(&ws);
        if (s != TP_OK) return s;
    }
    // Every partial sum is written in full before it is read, and the tail
    // split's counters are zeroed on the call's stream (cudaMemsetAsync)
    // before the GEMM that counts with them, so nothing in the array has to
    // start at zero and a previous call's contents are never observed.
    return tpmlp::linear_row_bwd_impl(desc, dY, X, W, dX, dW, db, ws, ws ? kScratchBytes : 0, stream, split);
}

}  // extern "C"
