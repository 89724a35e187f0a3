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

// Philox4x32-10 (Salmon, Moraes, Dror & Shaw, SC 2011): 10 rounds of
// (c0..c3) <- (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)),
// the key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Dropout draws: element e of a [rows, ld] tensor uses word e mod 4 of
// Philox4x32-10 at counter (e div 4) with key (seed lo, seed hi); it is kept
// when the word's top 24 bits reach `threshold` = floor(p * 2^24).
struct DropoutParams {
    int on;
    uint32_t threshold;
    float scale;  // 1 / (1 - p)
    uint32_t seed_lo, seed_hi;
    long long ld;  // columns of the whole tensor (element index = row * ld + col)
    // keep-mask output (or null): bit c % 32 of word row * mask_ld + c / 32 is
    // the keep flag of element (row, c)
    uint32_t *mask;
    long long mask_ld;
};

// keep flags of the 4 elements starting at e (e % 4 == 0), applied to v[0..3]
__device__ __forceinline__ void dropout4(const DropoutParams &d, long long e, float *v) {
    const unsigned long long q = static_cast<unsigned long long>(e) >> 2;
    const uint4 r = philox4x32_10(make_uint4(static_cast<uint32_t>(q), static_cast<uint32_t>(q >> 32), 0u, 0u),
                                  d.seed_lo, d.seed_hi);
    v[0] = (r.x >> 8) >= d.threshold ? v[0] * d.scale : 0.0f;
    v[1] = (r.y >> 8) >= d.threshold ? v[1] * d.scale : 0.0f;
    v[2] = (r.z >> 8) >= d.threshold ? v[2] * d.scale : 0.0f;
    v[3] = (r.w >> 8) >= d.threshold ? v[3] * d.scale : 0.0f;
}

// dropout4 that also returns the 4 keep flags (bit k: element e + k kept)
__device__ __forceinline__ uint32_t dropout4_bits(const DropoutParams &d, long long e, float *v) {
    const unsigned long long q = static_cast<unsigned long long>(e) >> 2;
    const uint4 r = philox4x32_10(make_uint4(static_cast<uint32_t>(q), static_cast<uint32_t>(q >> 32), 0u, 0u),
                                  d.seed_lo, d.seed_hi);
    const uint32_t k0 = (r.x >> 8) >= d.threshold, k1 = (r.y >> 8) >= d.threshold;
    const uint32_t k2 = (r.z >> 8) >= d.threshold, k3 = (r.w >> 8) >= d.threshold;
    v[0] = k0 ? v[0] * d.scale : 0.0f;
    v[1] = k1 ? v[1] * d.scale : 0.0f;
    v[2] = k2 ? v[2] * d.scale : 0.0f;
    v[3] = k3 ? v[3] * d.scale : 0.0f;
    return k0 | (k1 << 1) | (k2 << 2) | (k3 << 3);
}

// dropout of 32 consecutive elements of one row from column col0 (a multiple
// of 32), storing their keep word when the mask is requested and the row exists
__device__ __forceinline__ void dropout32(const DropoutParams &d, int row, int col0, bool row_ok, float *v) {
    const long long e0 = static_cast<long long>(row) * d.ld + col0;
    if (!d.mask) {
#pragma unroll
        for (int k = 0; k < 8; ++k) dropout4(d, e0 + 4 * k, v + 4 * k);
        return;
    }
    uint32_t bits = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) bits |= dropout4_bits(d, e0 + 4 * k, v + 4 * k) << (4 * k);
    if (row_ok) d.mask[static_cast<long long>(row) * d.mask_ld + col0 / 32] = bits;
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
