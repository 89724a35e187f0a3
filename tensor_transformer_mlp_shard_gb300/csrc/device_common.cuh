// Device helpers shared by the kernels: activation math, bounded waits and
// the status protocol.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/tp_mlp.h"

namespace tpmlp {

// GeLU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
constexpr float kGeluK0 = 0.7978845608028654f;  // sqrt(2/pi)
constexpr float kGeluK1 = 0.044715f;

__device__ __forceinline__ float gelu_tanh_f(float x) {
    float u = kGeluK0 * fmaf(kGeluK1 * x * x, x, x);
    return 0.5f * x * (1.0f + tanhf(u));
}

// d/dx gelu_tanh = 0.5(1+t) + 0.5 x (1-t^2) sqrt(2/pi) (1 + 3*0.044715 x^2)
__device__ __forceinline__ float gelu_tanh_grad_f(float x) {
    float t = tanhf(kGeluK0 * fmaf(kGeluK1 * x * x, x, x));
    return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * kGeluK0 * fmaf(3.0f * kGeluK1, x * x, 1.0f);
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// FP8 per-tensor scale: fmax / amax in fp32 (IEEE division), 1 when amax is
// 0 or not finite.  The quantiser and the GEMM epilogues share it.
__device__ __forceinline__ float fp8_scale(float amax, float fmax) {
    return (amax > 0.0f && amax <= 3.0e38f) ? fmax / amax : 1.0f;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Record an error in the device status word (first error wins) and mark the
// launch `launch_id` as aborted so that its other threads stop waiting.
__device__ __forceinline__ void raise_device_error(int *status, unsigned *abort_word, unsigned launch_id,
                                                   int code) {
    atomicCAS(status, 0, code);
    atomicExch(abort_word, launch_id);
    __threadfence();
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace tpmlp
