// Kernels of the TransformerLayer MLP sub-block (the gitcode.csdn.net Megatron
// Core walk-through, s03: LayerNorm -> MLP -> bias/dropout/residual add):
// LayerNorm forward and backward and the dropout backward.  All three are HBM
// bound: one pass over their [M, H] operands with 16-byte vector accesses,
// one token row per block (the forward) or kLnBwdRows rows per block (the
// backward, which also emits one row of dgamma/dbeta partial sums).
// Sequence-parallel tensors (X, dY, dX) are addressed through the token shard
// holding the row.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace tpmlp {

constexpr int kLnThreads = 256;
constexpr int kLnMaxVpt = 4;    // 16-byte vectors per thread and row: H <= 8192 (bf16), 4096 (fp32)
constexpr int kLnBwdRows = 16;  // rows per backward block

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16 *p, float *v) {
        const uint4 w = *reinterpret_cast<const uint4 *>(p);
        v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
        v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
    }
    __device__ static void store(__nv_bfloat16 *p, const float *v) {
        uint4 w;
        w.x = pack_bf16x2(v[0], v[1]); w.y = pack_bf16x2(v[2], v[3]);
        w.z = pack_bf16x2(v[4], v[5]); w.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4 *>(p) = w;
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const float *p, float *v) {
        const float4 w = *reinterpret_cast<const float4 *>(p);
        v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    }
    __device__ static void store(float *p, const float *v) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

// element offset of token `row` in its shard, and the shard
__device__ __forceinline__ long long shard_offset(int rows_split, int row, int H, int *shard) {
    int j = 0, lr = row;
    if (rows_split) {
        j = row / rows_split;
        lr = row - j * rows_split;
    }
    *shard = j;
    return static_cast<long long>(lr) * H;
}

// sums over the block (every thread receives them)
__device__ __forceinline__ float2 block_sum2(float a, float b) {
    __shared__ float2 red[kLnThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    __syncthreads();  // the previous call's readers are done with red
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float2(a, b);
    __syncthreads();
    float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int w = 0; w < kLnThreads / 32; ++w) {
        s.x += red[w].x;
        s.y += red[w].y;
    }
    return s;
}

// ---------------------------------------------------------------------------
// LayerNorm forward, one block per token row: mean and population variance in
// fp32 from two passes over the row held in registers, rstd = 1/sqrt(var+eps),
// Xn = (x - mean) * rstd * gamma + beta.
// ---------------------------------------------------------------------------
template <typename T, int VPT>
__global__ void __launch_bounds__(kLnThreads) ln_fwd_kernel(const __grid_constant__ LnPlan p) {
    using V = Vec<T>;
    const int row = blockIdx.x;
    int j0;
    const long long off = shard_offset(p.rows_split, row, p.H, &j0);
    const T *x = static_cast<const T *>(p.x[j0]) + off;
    T *y = static_cast<T *>(p.xn) + static_cast<long long>(row) * p.H;
    const int nv = p.H / V::N;
    float xv[VPT][V::N];
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
        if (i < nv) {
            V::load(x + i * V::N, xv[k]);
#pragma unroll
            for (int j = 0; j < V::N; ++j) s += xv[k][j];
        }
    }
    const float mean = block_sum2(s, 0.0f).x / p.H;
    float q = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
        if (i < nv) {
#pragma unroll
            for (int j = 0; j < V::N; ++j) {
                const float d = xv[k][j] - mean;
                q += d * d;
            }
        }
    }
    const float rstd = 1.0f / sqrtf(block_sum2(q, 0.0f).x / p.H + p.eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
        if (i < nv) {
            float g[V::N], b[V::N], o[V::N];
            V::load(static_cast<const T *>(p.gamma) + i * V::N, g);
            V::load(static_cast<const T *>(p.beta) + i * V::N, b);
#pragma unroll
            for (int j = 0; j < V::N; ++j) o[j] = (xv[k][j] - mean) * rstd * g[j] + b[j];
            V::store(y + i * V::N, o);
        }
    }
    if (threadIdx.x == 0) {
        p.mean[row] = mean;
        p.rstd[row] = rstd;
    }
}

// ---------------------------------------------------------------------------
// LayerNorm backward over kLnBwdRows token rows per block.  With
// g = dXn * gamma and xhat = (x - mean) * rstd:
//   dX = dY + rstd * (g - mean_h(g) - xhat * mean_h(g * xhat))
// (dY: the residual branch of the sub-block), and the block's partial column
// sums of dXn * xhat (dgamma) and dXn (dbeta) into
// partials[0][blockIdx.x][:] and partials[1][blockIdx.x][:].
// ---------------------------------------------------------------------------
template <typename T, int VPT>
__global__ void __launch_bounds__(kLnThreads) ln_bwd_kernel(const __grid_constant__ LnPlan p) {
    using V = Vec<T>;
    const int nv = p.H / V::N;
    float gm[VPT][V::N], pg[VPT][V::N], pb[VPT][V::N];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
#pragma unroll
        for (int j = 0; j < V::N; ++j) pg[k][j] = pb[k][j] = gm[k][j] = 0.0f;
        if (i < nv) V::load(static_cast<const T *>(p.gamma) + i * V::N, gm[k]);
    }
    const int r0 = blockIdx.x * kLnBwdRows;
    const int r1 = min(p.M, r0 + kLnBwdRows);
#pragma unroll 1
    for (int row = r0; row < r1; ++row) {
        int js;
        const long long off = shard_offset(p.rows_split, row, p.H, &js);
        const T *x = static_cast<const T *>(p.x[js]) + off;
        const T *dy = static_cast<const T *>(p.dy[js]) + off;
        T *dx = static_cast<T *>(p.dx[js]) + off;
        const T *dxn = static_cast<const T *>(p.dxn) + static_cast<long long>(row) * p.H;
        const float mean = p.mean[row], rstd = p.rstd[row];
        float xh[VPT][V::N], g[VPT][V::N];
        float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int i = threadIdx.x + k * kLnThreads;
            if (i < nv) {
                float xv[V::N], d[V::N];
                V::load(x + i * V::N, xv);
                V::load(dxn + i * V::N, d);
#pragma unroll
                for (int j = 0; j < V::N; ++j) {
                    xh[k][j] = (xv[j] - mean) * rstd;
                    g[k][j] = d[j] * gm[k][j];
                    s1 += g[k][j];
                    s2 += g[k][j] * xh[k][j];
                    pg[k][j] += d[j] * xh[k][j];
                    pb[k][j] += d[j];
                }
            }
        }
        const float2 s = block_sum2(s1, s2);
        const float mg = s.x / p.H, mgx = s.y / p.H;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int i = threadIdx.x + k * kLnThreads;
            if (i < nv) {
                float r[V::N], o[V::N];
                V::load(dy + i * V::N, r);
#pragma unroll
                for (int j = 0; j < V::N; ++j) o[j] = r[j] + rstd * (g[k][j] - mg - xh[k][j] * mgx);
                V::store(dx + i * V::N, o);
            }
        }
    }
    const long long chunks = gridDim.x;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
        if (i < nv) {
            float *og = p.partials + static_cast<long long>(blockIdx.x) * p.H + i * V::N;
            float *ob = p.partials + (chunks + blockIdx.x) * p.H + i * V::N;
#pragma unroll
            for (int j = 0; j < V::N; j += 4) {
                *reinterpret_cast<float4 *>(og + j) = make_float4(pg[k][j], pg[k][j + 1], pg[k][j + 2], pg[k][j + 3]);
                *reinterpret_cast<float4 *>(ob + j) = make_float4(pb[k][j], pb[k][j + 1], pb[k][j + 2], pb[k][j + 3]);
            }
        }
    }
}

// Dropout backward: dZ = dY * keep / (1 - p), the keep flags redrawn from the
// forward's Philox stream (element m*H + h); dY token-sharded, dZ contiguous.
template <typename T>
__global__ void __launch_bounds__(256) dropout_bwd_kernel(const __grid_constant__ LnPlan p) {
    using V = Vec<T>;
    DropoutParams d;
    d.on = 1;
    d.threshold = p.drop_threshold;
    d.scale = p.drop_scale;
    d.seed_lo = static_cast<uint32_t>(p.drop_seed);
    d.seed_hi = static_cast<uint32_t>(p.drop_seed >> 32);
    d.ld = p.H;
    const int vpr = p.H / V::N;  // vectors per row
    const long long nv = static_cast<long long>(p.M) * vpr;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nv;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int row = static_cast<int>(i / vpr);
        const int col = static_cast<int>(i - static_cast<long long>(row) * vpr) * V::N;
        int js;
        const long long off = shard_offset(p.rows_split, row, p.H, &js);
        float v[V::N];
        V::load(static_cast<const T *>(p.dy[js]) + off + col, v);
        const long long e = static_cast<long long>(row) * p.H + col;
#pragma unroll
        for (int j = 0; j < V::N; j += 4) dropout4(d, e + j, v + j);
        V::store(static_cast<T *>(p.dz) + e, v);
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
int ln_bwd_chunks(int M) { return M <= 0 ? 1 : (M + kLnBwdRows - 1) / kLnBwdRows; }

static int ln_vpt(int H, int dtype) {
    const int nv = H / (dtype == TP_DT_F32 ? 4 : 8);
    for (int v = 1; v <= kLnMaxVpt; v *= 2)
        if (nv <= v * kLnThreads) return v;
    return 0;
}

bool ln_supported(int H, int dtype) { return H % (dtype == TP_DT_F32 ? 4 : 8) == 0 && ln_vpt(H, dtype) > 0; }

template <typename T>
static void ln_fwd_dispatch(const LnPlan &p, int vpt, cudaStream_t st) {
    if (vpt == 1)
        ln_fwd_kernel<T, 1><<<p.M, kLnThreads, 0, st>>>(p);
    else if (vpt == 2)
        ln_fwd_kernel<T, 2><<<p.M, kLnThreads, 0, st>>>(p);
    else
        ln_fwd_kernel<T, 4><<<p.M, kLnThreads, 0, st>>>(p);
}

template <typename T>
static void ln_bwd_dispatch(const LnPlan &p, int vpt, int chunks, cudaStream_t st) {
    if (vpt == 1)
        ln_bwd_kernel<T, 1><<<chunks, kLnThreads, 0, st>>>(p);
    else if (vpt == 2)
        ln_bwd_kernel<T, 2><<<chunks, kLnThreads, 0, st>>>(p);
    else
        ln_bwd_kernel<T, 4><<<chunks, kLnThreads, 0, st>>>(p);
}

tp_status launch_ln_fwd(const LnPlan &p, int dtype, cudaStream_t st) {
    if (p.M == 0) return TP_OK;
    const int vpt = ln_vpt(p.H, dtype);
    if (!vpt) return set_error(TP_ERR_UNSUPPORTED, "LayerNorm width H=%d above the kernel's row capacity", p.H);
    launch_begin("layernorm_fwd", st);
    if (dtype == TP_DT_F32)
        ln_fwd_dispatch<float>(p, vpt, st);
    else
        ln_fwd_dispatch<__nv_bfloat16>(p, vpt, st);
    cudaError_t e = cudaGetLastError();
    launch_end("layernorm_fwd", st);
    return cuda_check(e, "layernorm_fwd");
}

tp_status launch_ln_bwd(const LnPlan &p, int dtype, cudaStream_t st) {
    const int vpt = ln_vpt(p.H, dtype);
    if (!vpt) return set_error(TP_ERR_UNSUPPORTED, "LayerNorm width H=%d above the kernel's row capacity", p.H);
    if (p.M == 0) {
        cudaError_t e = cudaMemsetAsync(p.dgamma, 0, sizeof(float) * p.H, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(p.dbeta, 0, sizeof(float) * p.H, st);
        return cuda_check(e, "cudaMemsetAsync(dgamma, dbeta)");
    }
    const int chunks = ln_bwd_chunks(p.M);
    launch_begin("layernorm_bwd", st);
    if (dtype == TP_DT_F32)
        ln_bwd_dispatch<float>(p, vpt, chunks, st);
    else
        ln_bwd_dispatch<__nv_bfloat16>(p, vpt, chunks, st);
    cudaError_t e = cudaGetLastError();
    launch_end("layernorm_bwd", st);
    if (e != cudaSuccess) return cuda_check(e, "layernorm_bwd");
    // dgamma, dbeta = sums of the per-block partial rows
    ColsumPlan c;
    c.name = "ln_param_grads";
    c.P = 2;
    c.M = p.M;
    c.N = p.H;
    c.out[0] = p.dgamma;
    c.out[1] = p.dbeta;
    c.partials = p.partials;
    return launch_colsum_finalize(c, chunks, st);
}

tp_status launch_dropout_bwd(const LnPlan &p, int dtype, cudaStream_t st) {
    if (p.M == 0) return TP_OK;
    const long long nv = static_cast<long long>(p.M) * p.H / (dtype == TP_DT_F32 ? 4 : 8);
    const long long want = (nv + 255) / 256, cap = 8ll * num_sms();
    const int grid = static_cast<int>(want < cap ? want : cap);
    launch_begin("dropout_bwd", st);
    if (dtype == TP_DT_F32)
        dropout_bwd_kernel<float><<<grid, 256, 0, st>>>(p);
    else
        dropout_bwd_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    launch_end("dropout_bwd", st);
    return cuda_check(e, "dropout_bwd");
}

}  // namespace tpmlp
