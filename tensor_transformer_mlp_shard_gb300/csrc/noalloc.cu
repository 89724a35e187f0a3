// tp_linear_row_bwd_noalloc: the row-layer backward for callers that cannot
// allocate device memory.
//
// tp_linear_row_bwd needs a small device workspace for the bias gradient: the
// token-chunk partial column sums of dY that the second pass adds up.  Some
// callers have no way to provide one: a plugin inside another framework is
// handed only the op's own tensors and has no allocator to ask; a process whose
// device memory is already fully reserved by another (caching) allocator can
// see cudaMalloc fail; and a latency-critical loop cannot afford cudaMalloc's
// implicit device synchronisation.  For them this entry point takes its
// scratch from a fixed array compiled into the library instead.
//
// The array is file-scope device memory of kScratchBytes.  Every GPU that
// loads the library holds it until the process exits.  Host code cannot use
// the array's name as a device address (in host code it is only a stand-in
// for the symbol), so the device address is looked up with
// cudaGetSymbolAddress once per device, on the first call made while that
// device is current, and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB

}  // namespace

static __device__ __align__(256) unsigned char tp_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_scratch_mu;
void *g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
tp_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tpmlp::cuda_check(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return tpmlp::set_error(TP_ERR_UNSUPPORTED, "device ordinal %d above 63", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, tp_noalloc_scratch);
        if (e != cudaSuccess) return tpmlp::cuda_check(e, "cudaGetSymbolAddress(tp_noalloc_scratch)");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return TP_OK;
}

}  // namespace

extern "C" {

tp_status tp_linear_row_bwd_noalloc(const tp_mlp_desc *desc, const void *const *dY, const void *const *X,
                                    const void *const *W, void *const *dX, void *const *dW, void *db,
                                    void *stream) {
    // 0 for an invalid descriptor too: the row backward then reports the error.
    const size_t need = tpmlp::linear_bias_workspace_bytes(desc);
    if (need > kScratchBytes)
        return tpmlp::set_error(TP_ERR_UNSUPPORTED,
                                "bias gradient needs %zu bytes of scratch; the built-in scratch holds %zu "
                                "(use tp_linear_row_bwd with a caller workspace)",
                                need, kScratchBytes);
    // split-K partials of the weight gradient only when they fit as well
    const size_t full = tp_linear_workspace_bytes(desc);
    const bool split = full <= kScratchBytes;
    void *ws = nullptr;
    if (split ? full : need) {
        tp_status s = scratch_address(&ws);
        if (s != TP_OK) return s;
    }
    // The partial sums are written in full before they are read, so nothing
    // in the array has to start at zero and stale contents of a previous call
    // are never observed.
    return tpmlp::linear_row_bwd_impl(desc, dY, X, W, dX, dW, db, ws, ws ? kScratchBytes : 0, stream, split);
}

}  // extern "C"
