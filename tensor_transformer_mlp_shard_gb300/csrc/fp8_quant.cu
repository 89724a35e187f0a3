// Per-tensor FP8 quantisation of bf16 tensors ("Megatron-LM 源码精读", s8.2:
// per-tensor scaling from the amax; E4M3 forward, E5M2 backward).
//
// A logical tensor may be split over several buffers (its shards); its amax is
// the maximum over all of them -- the cross-shard amax all-reduce done as a
// device-wide max.  Pass 1 (amax_kernel) reduces |x| into one fp32 slot per
// tensor with an integer atomicMax on the bit pattern (valid for non-negative
// floats).  Pass 2 (quant_kernel) computes scale = fmax / amax and writes
// fp8(x * scale) with round-to-nearest-even, saturating to +-fmax.  Both passes
// are HBM bound: 16-byte loads of 8 bf16, 8-byte stores of 8 fp8 codes.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace tpmlp {

// Work split: every segment is cut into chunks of kChunkVec 16-byte vectors
// and every block takes one chunk (block_start[k] = first block of segment
// k), so the big segments (X, dY) and the small ones (weight shards) load
// the GPU evenly; a thread keeps kUnroll loads in flight.
constexpr int kQuantThreads = 256;
constexpr int kUnroll = 8;
constexpr long long kChunkVec = static_cast<long long>(kQuantThreads) * kUnroll * 4;  // 8192 vectors, 128 KB

struct QuantParams {
    QuantSeg seg[kMaxQuantSegs];
    int block_start[kMaxQuantSegs + 1];
    int nseg;
    float *amax;
    const float *scale_amax;  // cast: the amax the scale derives from (null: amax[slot])
    int accumulate;           // cast: also reduce |x| into amax[slot] (one pass)
};

// segment of block b and the block's index within it
__device__ __forceinline__ int seg_of_block(const QuantParams &p, int b, int *lb) {
    int k = 0;
    while (k + 1 < p.nseg && b >= p.block_start[k + 1]) ++k;
    *lb = b - p.block_start[k];
    return k;
}

__device__ __forceinline__ float absmax8(const uint4 &w) {
    const float a = fmaxf(fmaxf(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x))), fmaxf(fabsf(bf16_lo(w.y)), fabsf(bf16_hi(w.y))));
    const float b = fmaxf(fmaxf(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z))), fmaxf(fabsf(bf16_lo(w.w)), fabsf(bf16_hi(w.w))));
    return fmaxf(a, b);
}

__global__ void __launch_bounds__(kQuantThreads) amax_kernel(const __grid_constant__ QuantParams p) {
    int lb;
    const QuantSeg &sg = p.seg[seg_of_block(p, blockIdx.x, &lb)];
    const uint4 *in = static_cast<const uint4 *>(sg.in);
    const long long nv = sg.n / 8;
    const long long v0 = lb * kChunkVec, v1 = min(nv, v0 + kChunkVec);
    float m = 0.0f;
    for (long long base = v0 + threadIdx.x; base < v1; base += static_cast<long long>(kQuantThreads) * kUnroll) {
        uint4 w[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = base + static_cast<long long>(u) * kQuantThreads;
            w[u] = i < v1 ? in[i] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) m = fmaxf(m, absmax8(w[u]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float red[kQuantThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kQuantThreads / 32; ++w) m = fmaxf(m, red[w]);
        atomicMax(reinterpret_cast<unsigned *>(p.amax + sg.slot), __float_as_uint(m));
    }
}

__device__ __forceinline__ uint16_t to_fp8x2(float a, float b, int fmt) {
    const float2 v = make_float2(a, b);
    return fmt == FP8_E5M2 ? __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E5M2)
                           : __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint2 quant8(const uint4 &w, float s, int fmt) {
    // x * scale is rounded to fp32 first, then to FP8
    const float x0 = bf16_lo(w.x) * s, x1 = bf16_hi(w.x) * s, x2 = bf16_lo(w.y) * s, x3 = bf16_hi(w.y) * s;
    const float x4 = bf16_lo(w.z) * s, x5 = bf16_hi(w.z) * s, x6 = bf16_lo(w.w) * s, x7 = bf16_hi(w.w) * s;
    uint2 o;
    o.x = uint32_t(to_fp8x2(x0, x1, fmt)) | (uint32_t(to_fp8x2(x2, x3, fmt)) << 16);
    o.y = uint32_t(to_fp8x2(x4, x5, fmt)) | (uint32_t(to_fp8x2(x6, x7, fmt)) << 16);
    return o;
}

__global__ void __launch_bounds__(kQuantThreads) quant_kernel(const __grid_constant__ QuantParams p) {
    int lb;
    const QuantSeg &sg = p.seg[seg_of_block(p, blockIdx.x, &lb)];
    const float s = fp8_scale(p.scale_amax ? p.scale_amax[sg.slot] : p.amax[sg.slot],
                              sg.fmt == FP8_E5M2 ? 57344.0f : 448.0f);
    const uint4 *in = static_cast<const uint4 *>(sg.in);
    uint2 *out = static_cast<uint2 *>(sg.out);
    const long long nv = sg.n / 8;
    const long long v0 = lb * kChunkVec, v1 = min(nv, v0 + kChunkVec);
    float m = 0.0f;
    for (long long base = v0 + threadIdx.x; base < v1; base += static_cast<long long>(kQuantThreads) * kUnroll) {
        uint4 w[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = base + static_cast<long long>(u) * kQuantThreads;
            w[u] = i < v1 ? in[i] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = base + static_cast<long long>(u) * kQuantThreads;
            if (i < v1) out[i] = quant8(w[u], s, sg.fmt);
            if (p.accumulate) m = fmaxf(m, absmax8(w[u]));
        }
    }
    if (p.accumulate) {  // block-uniform
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        __shared__ float red[kQuantThreads / 32];
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < kQuantThreads / 32; ++w) m = fmaxf(m, red[w]);
            atomicMax(reinterpret_cast<unsigned *>(p.amax + sg.slot), __float_as_uint(m));
        }
    }
}

// Amax history of delayed scaling, one thread per tensor slot: prepare
// (scale_amax[s] = max of the first `fill` entries of row s of the history,
// or amax[s] when fill is 0) or push (row s, column pos = amax[s]).
struct HistParams {
    float *hist;
    float *scale_amax;
    const float *amax;
    int slots[8];
    int nslots, fill, pos, push, ld;
};

__global__ void fp8_history_kernel(const __grid_constant__ HistParams p) {
    const int k = threadIdx.x;
    if (k >= p.nslots) return;
    const int s = p.slots[k];
    if (p.push) {
        p.hist[s * p.ld + p.pos] = p.amax[s];
        return;
    }
    float m = p.fill ? 0.0f : p.amax[s];
    for (int i = 0; i < p.fill; ++i) m = fmaxf(m, p.hist[s * p.ld + i]);
    p.scale_amax[s] = m;
}

tp_status launch_fp8_history(float *hist, int ld, float *scale_amax, const float *amax, const int *slots, int nslots,
                             int fill, int pos, bool push, cudaStream_t st) {
    if (nslots < 1 || nslots > 8 || fill < 0 || fill > ld || pos < 0 || pos >= ld)
        return set_error(TP_ERR_ARG, "bad amax-history request");
    HistParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.hist = hist;
    prm.scale_amax = scale_amax;
    prm.amax = amax;
    for (int i = 0; i < nslots; ++i) prm.slots[i] = slots[i];
    prm.nslots = nslots;
    prm.fill = fill;
    prm.pos = pos;
    prm.push = push ? 1 : 0;
    prm.ld = ld;
    const char *name = push ? "fp8_history_push" : "fp8_history_scale";
    launch_begin(name, st);
    fp8_history_kernel<<<1, 32, 0, st>>>(prm);
    cudaError_t e = cudaGetLastError();
    launch_end(name, st);
    return cuda_check(e, name);
}

static tp_status launch_pass(bool amax_pass, const QuantSeg *segs, int nseg, float *amax, cudaStream_t st,
                             const float *scale_amax = nullptr, bool accumulate = false) {
    if (nseg <= 0) return TP_OK;
    if (nseg > kMaxQuantSegs) return set_error(TP_ERR_UNSUPPORTED, "too many quantisation segments (%d)", nseg);
    QuantParams prm;
    memset(&prm, 0, sizeof(prm));
    long long blocks = 0;
    for (int i = 0; i < nseg; ++i) {
        if (segs[i].n % 8) return set_error(TP_ERR_SHAPE, "quantised buffer length %lld not a multiple of 8", segs[i].n);
        prm.seg[i] = segs[i];
        prm.block_start[i] = static_cast<int>(blocks);
        blocks += (segs[i].n / 8 + kChunkVec - 1) / kChunkVec;
    }
    prm.block_start[nseg] = static_cast<int>(blocks);
    prm.nseg = nseg;
    prm.amax = amax;
    prm.scale_amax = scale_amax;
    prm.accumulate = accumulate ? 1 : 0;
    if (blocks == 0) return TP_OK;
    if (blocks > (1ll << 31) - 1) return set_error(TP_ERR_SHAPE, "quantised tensor too large");
    const char *name = amax_pass ? "fp8_amax" : "fp8_quant";
    launch_begin(name, st);
    if (amax_pass)
        amax_kernel<<<static_cast<unsigned>(blocks), kQuantThreads, 0, st>>>(prm);
    else
        quant_kernel<<<static_cast<unsigned>(blocks), kQuantThreads, 0, st>>>(prm);
    cudaError_t e = cudaGetLastError();
    launch_end(name, st);
    return cuda_check(e, name);
}

tp_status launch_fp8_cast(const QuantSeg *segs, int nseg, float *amax, const float *scale_amax, bool accumulate,
                          cudaStream_t st) {
    return launch_pass(false, segs, nseg, amax, st, scale_amax, accumulate);
}

tp_status launch_fp8_quantize(const QuantSeg *segs, int nseg, float *amax, bool zero_slots, cudaStream_t st,
                              bool amax_known) {
    if (amax_known) return launch_pass(false, segs, nseg, amax, st);  // amax already reduced by the producer
    if (zero_slots) {  // one memset per distinct slot (the buffers of a tensor share one)
        uint64_t done = 0;
        for (int i = 0; i < nseg; ++i) {
            const int sl = segs[i].slot;
            if (sl >= 0 && sl < 64 && (done >> sl) & 1u) continue;
            if (sl >= 0 && sl < 64) done |= uint64_t(1) << sl;
            cudaError_t e = cudaMemsetAsync(amax + sl, 0, sizeof(float), st);
            if (e != cudaSuccess) return cuda_check(e, "cudaMemsetAsync(amax)");
        }
    }
    tp_status s = launch_pass(true, segs, nseg, amax, st);
    if (s != TP_OK) return s;
    return launch_pass(false, segs, nseg, amax, st);
}

}  // namespace tpmlp
