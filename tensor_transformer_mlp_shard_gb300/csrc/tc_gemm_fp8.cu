// FP8 (E4M3 / E5M2 operands, tcgen05 kind::f8f6f4) instantiations of the GEMM
// kernels, compiled as a unit of their own.
#include "device_common.cuh"
#include "internal.h"
#include "tc_gemm_kernels.cuh"

namespace tpmlp {
namespace tc {

typedef void (*KernelFn)(Params);

KernelFn fp8_kernel_at(int i, bool pair) {
    switch (i) {
        case 0: return pair ? tc_gemm_pair_kernel<EPI_COL, false, false, true> : tc_gemm_kernel<EPI_COL, false, false, true>;
        case 1: return pair ? tc_gemm_pair_kernel<EPI_PLAIN, false, false, true> : tc_gemm_kernel<EPI_PLAIN, false, false, true>;
        case 2: return pair ? tc_gemm_pair_kernel<EPI_PLAIN, false, true, true> : tc_gemm_kernel<EPI_PLAIN, false, true, true>;
        case 3: return pair ? tc_gemm_pair_kernel<EPI_DACT, false, true, true> : tc_gemm_kernel<EPI_DACT, false, true, true>;
        case 4: return pair ? tc_gemm_pair_kernel<EPI_F32, true, true, true> : tc_gemm_kernel<EPI_F32, true, true, true>;
        case 5: return pair ? tc_gemm_pair_kernel<EPI_F32, true, true, true, true> : tc_gemm_kernel<EPI_F32, true, true, true>;
    }
    return nullptr;
}

}  // namespace tc
}  // namespace tpmlp
