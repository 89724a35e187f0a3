// Kernels of the TransformerLayer MLP sub-block (the gitcode.csdn.net Megatron
// Core walk-through, s03: LayerNorm -> MLP -> bias/dropout/residual add):
// LayerNorm forward and backward and the dropout backward.  All three are HBM
// bound: one pass over their [M, H] operands with 16-byte vector accesses,
// one token row per block (the forward), a run of rows per block (the
// backward, which also emits one row of dgamma/dbeta partial sums) or a
// kDropRows-row column strip per block (the dropout backward, which emits
// one row of db2 partial sums).
// Sequence-parallel tensors (X, dY, dX) are addressed through the token shard
// holding the row.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace tpmlp {

constexpr int kLnThreads = 256;
constexpr int kLnMaxVpt = 4;    // 16-byte vectors per thread and row: H <= 8192 (bf16), 4096 (fp32)
constexpr int kLnBwdMinRows = 8;  // fewest rows per backward block (bounds the partials)

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    using Raw = uint4;
    __device__ static Raw load_raw(const __nv_bfloat16 *p) { return *reinterpret_cast<const uint4 *>(p); }
    __device__ static void unpack(const Raw &w, float *v) {
        v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
        v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
    }
    __device__ static Raw pack(const float *v) {
        Raw w;
        w.x = pack_bf16x2(v[0], v[1]); w.y = pack_bf16x2(v[2], v[3]);
        w.z = pack_bf16x2(v[4], v[5]); w.w = pack_bf16x2(v[6], v[7]);
        return w;
    }
    __device__ static float first(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
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
    using Raw = float4;
    __device__ static Raw load_raw(const float *p) { return *reinterpret_cast<const float4 *>(p); }
    __device__ static void unpack(const Raw &w, float *v) { v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w; }
    __device__ static Raw pack(const float *v) { return make_float4(v[0], v[1], v[2], v[3]); }
    __device__ static float first(const float *p) { return *p; }
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
// LayerNorm forward, one block per token row.  The row, gamma and beta are
// loaded up front; the statistics come from one block reduction of the
// shifted sums S1 = sum(x - k), S2 = sum((x - k)^2) with k = x[0] (so that a
// large row mean does not cancel digits): mean = k + S1/H,
// var = S2/H - (S1/H)^2 (population variance), rstd = 1/sqrt(var + eps),
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
    typename V::Raw rx[VPT], rg[VPT], rb[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
        if (i < nv) {
            rx[k] = V::load_raw(x + i * V::N);
            rg[k] = V::load_raw(static_cast<const T *>(p.gamma) + i * V::N);
            rb[k] = V::load_raw(static_cast<const T *>(p.beta) + i * V::N);
        }
    }
    const float shift = V::first(x);
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
        if (i < nv) {
            float v[V::N];
            V::unpack(rx[k], v);
#pragma unroll
            for (int j = 0; j < V::N; ++j) {
                const float d = v[j] - shift;
                s1 += d;
                s2 = fmaf(d, d, s2);
            }
        }
    }
    const float2 s = block_sum2(s1, s2);
    const float m1 = s.x / p.H;
    const float mean = shift + m1;
    const float var = fmaxf(s.y / p.H - m1 * m1, 0.0f);
    const float rstd = 1.0f / sqrtf(var + p.eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
        if (i < nv) {
            float v[V::N], g[V::N], b[V::N];
            V::unpack(rx[k], v);
            V::unpack(rg[k], g);
            V::unpack(rb[k], b);
#pragma unroll
            for (int j = 0; j < V::N; ++j) v[j] = (v[j] - mean) * rstd * g[j] + b[j];
            V::store(y + i * V::N, v);
        }
    }
    if (threadIdx.x == 0) {
        p.mean[row] = mean;
        p.rstd[row] = rstd;
    }
}

// The same LayerNorm forward with one warp per token row (rows of up to
// 32 * VPW vectors): no block barrier, and a block keeps 8 rows in flight.
template <typename T, int VPW>
__global__ void __launch_bounds__(kLnThreads) ln_fwd_warp_kernel(const __grid_constant__ LnPlan p) {
    using V = Vec<T>;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (kLnThreads / 32) + (threadIdx.x >> 5);
    if (row >= p.M) return;  // whole warps leave; no block barrier follows
    int j0;
    const long long off = shard_offset(p.rows_split, row, p.H, &j0);
    const T *x = static_cast<const T *>(p.x[j0]) + off;
    T *y = static_cast<T *>(p.xn) + static_cast<long long>(row) * p.H;
    const int nv = p.H / V::N;
    typename V::Raw rx[VPW];
#pragma unroll
    for (int k = 0; k < VPW; ++k) {
        const int i = lane + 32 * k;
        if (i < nv) rx[k] = V::load_raw(x + i * V::N);
    }
    const float shift = V::first(x);
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int k = 0; k < VPW; ++k) {
        const int i = lane + 32 * k;
        if (i < nv) {
            float v[V::N];
            V::unpack(rx[k], v);
#pragma unroll
            for (int j = 0; j < V::N; ++j) {
                const float d = v[j] - shift;
                s1 += d;
                s2 = fmaf(d, d, s2);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    const float m1 = s1 / p.H;
    const float mean = shift + m1;
    const float var = fmaxf(s2 / p.H - m1 * m1, 0.0f);
    const float rstd = 1.0f / sqrtf(var + p.eps);
#pragma unroll
    for (int k = 0; k < VPW; ++k) {
        const int i = lane + 32 * k;
        if (i < nv) {
            float v[V::N], g[V::N], b[V::N];
            V::unpack(rx[k], v);
            V::unpack(V::load_raw(static_cast<const T *>(p.gamma) + i * V::N), g);
            V::unpack(V::load_raw(static_cast<const T *>(p.beta) + i * V::N), b);
#pragma unroll
            for (int j = 0; j < V::N; ++j) v[j] = (v[j] - mean) * rstd * g[j] + b[j];
            V::store(y + i * V::N, v);
        }
    }
    if (lane == 0) {
        p.mean[row] = mean;
        p.rstd[row] = rstd;
    }
}

// ---------------------------------------------------------------------------
// LayerNorm backward over `rows` token rows per block (chosen so that the
// grid is one wave of resident blocks).  With
// g = dXn * gamma and xhat = (x - mean) * rstd:
//   dX = dY + rstd * (g - mean_h(g) - xhat * mean_h(g * xhat))
// (dY: the residual branch of the sub-block), and the block's partial column
// sums of dXn * xhat (dgamma) and dXn (dbeta) into
// partials[0][blockIdx.x][:] and partials[1][blockIdx.x][:].  The loads of
// row r + 1 (x, dXn, dY, kept as raw 16-byte vectors) are issued before row
// r is reduced, so that every thread has two rows of loads in flight.
// ---------------------------------------------------------------------------
template <typename T, int VPT>
struct LnRowRaw {
    typename Vec<T>::Raw x[VPT], d[VPT], r[VPT];
    float mean, rstd;
};

template <typename T, int VPT>
__device__ __forceinline__ void ln_bwd_load(const LnPlan &p, int row, int nv, LnRowRaw<T, VPT> &o) {
    using V = Vec<T>;
    int js;
    const long long off = shard_offset(p.rows_split, row, p.H, &js);
    const T *x = static_cast<const T *>(p.x[js]) + off;
    const T *dy = static_cast<const T *>(p.dy[js]) + off;
    const T *dxn = static_cast<const T *>(p.dxn) + static_cast<long long>(row) * p.H;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
        if (i < nv) {
            o.x[k] = V::load_raw(x + i * V::N);
            o.d[k] = V::load_raw(dxn + i * V::N);
            o.r[k] = V::load_raw(dy + i * V::N);
        }
    }
    o.mean = p.mean[row];
    o.rstd = p.rstd[row];
}

template <typename T, int VPT>
__global__ void __launch_bounds__(kLnThreads) ln_bwd_kernel(const __grid_constant__ LnPlan p, int rows) {
    using V = Vec<T>;
    const int nv = p.H / V::N;
    typename V::Raw rgm[VPT];
    float pg[VPT][V::N], pb[VPT][V::N];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * kLnThreads;
#pragma unroll
        for (int j = 0; j < V::N; ++j) pg[k][j] = pb[k][j] = 0.0f;
        if (i < nv) rgm[k] = V::load_raw(static_cast<const T *>(p.gamma) + i * V::N);
    }
    const int r0 = blockIdx.x * rows;
    const int r1 = min(p.M, r0 + rows);
    LnRowRaw<T, VPT> cur, nxt;
    ln_bwd_load<T, VPT>(p, r0, nv, cur);
#pragma unroll 1
    for (int row = r0; row < r1; ++row) {
        if (row + 1 < r1) ln_bwd_load<T, VPT>(p, row + 1, nv, nxt);
        const float mean = cur.mean, rstd = cur.rstd;
        float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int i = threadIdx.x + k * kLnThreads;
            if (i < nv) {
                float xv[V::N], d[V::N], gm[V::N];
                V::unpack(cur.x[k], xv);
                V::unpack(cur.d[k], d);
                V::unpack(rgm[k], gm);
#pragma unroll
                for (int j = 0; j < V::N; ++j) {
                    const float xh = (xv[j] - mean) * rstd;
                    const float g = d[j] * gm[j];
                    s1 += g;
                    s2 = fmaf(g, xh, s2);
                    pg[k][j] = fmaf(d[j], xh, pg[k][j]);
                    pb[k][j] += d[j];
                }
            }
        }
        const float2 s = block_sum2(s1, s2);
        const float mg = s.x / p.H, mgx = s.y / p.H;
        int js;
        const long long off = shard_offset(p.rows_split, row, p.H, &js);
        T *dx = static_cast<T *>(p.dx[js]) + off;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int i = threadIdx.x + k * kLnThreads;
            if (i < nv) {
                float xv[V::N], d[V::N], gm[V::N], o[V::N];
                V::unpack(cur.x[k], xv);
                V::unpack(cur.d[k], d);
                V::unpack(rgm[k], gm);
                V::unpack(cur.r[k], o);
#pragma unroll
                for (int j = 0; j < V::N; ++j) {
                    const float xh = (xv[j] - mean) * rstd;
                    o[j] += rstd * (d[j] * gm[j] - mg - xh * mgx);
                }
                V::store(dx + i * V::N, o);
            }
        }
        cur = nxt;
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

// ---------------------------------------------------------------------------
// Dropout backward fused with the column sums of its output:
//   dZ = dY * keep / (1 - p)   (keep flags read from the forward's keep-mask,
//                               or redrawn from its Philox stream, element
//                               m*H + h, when there is none),
//   partials[blockIdx.y][c] = sum over the block's kDropRows rows of dZ[:, c]
// (db2 = the sum of the partial rows).  A block covers kDropRows token rows
// and 8 * kDropThreads (bf16) or 4 * kDropThreads (fp32) columns; each thread
// walks its column vector down the rows with kDropUnroll loads in flight.
// dY is token-sharded, dZ contiguous.
// ---------------------------------------------------------------------------
constexpr int kDropThreads = 128;
constexpr int kDropRows = 32;
constexpr int kDropUnroll = 8;

template <typename T>
__global__ void __launch_bounds__(kDropThreads) dropout_bwd_kernel(const __grid_constant__ LnPlan p) {
    using V = Vec<T>;
    DropoutParams d;
    d.on = 1;
    d.threshold = p.drop_threshold;
    d.scale = p.drop_scale;
    d.seed_lo = static_cast<uint32_t>(p.drop_seed);
    d.seed_hi = static_cast<uint32_t>(p.drop_seed >> 32);
    d.ld = p.H;
    d.mask = nullptr;
    d.mask_ld = 0;
    const int col = (blockIdx.x * kDropThreads + threadIdx.x) * V::N;
    const bool active = col < p.H;
    const int r0 = blockIdx.y * kDropRows;
    const int r1 = min(p.M, r0 + kDropRows);
    // With the forward's keep-mask: V::N bits of one word per row, no Philox.
    // The block first checks the mask's bits of its first row against the
    // Philox stream and redraws every flag itself if any differs (a mask the
    // workspace no longer holds is caught here, whatever the host believed).
    const long long mask_ld = (p.H + 31) / 32;
    const uint32_t *mask = p.drop_mask;
    if (mask) {
        bool bad = false;
        if (active && r0 < r1) {
            float probe[V::N];
#pragma unroll
            for (int j = 0; j < V::N; ++j) probe[j] = 1.0f;
            const long long e = static_cast<long long>(r0) * p.H + col;
            uint32_t bits = 0;
#pragma unroll
            for (int j = 0; j < V::N; j += 4) bits |= dropout4_bits(d, e + j, probe + j) << j;
            const uint32_t want = (mask[r0 * mask_ld + col / 32] >> (col % 32)) & ((1u << V::N) - 1u);
            bad = bits != want;
        }
        if (__syncthreads_or(bad)) mask = nullptr;
    }
    if (!active) return;
    float acc[V::N];
#pragma unroll
    for (int j = 0; j < V::N; ++j) acc[j] = 0.0f;
#pragma unroll 1
    for (int rb = r0; rb < r1; rb += kDropUnroll) {
        typename V::Raw raw[kDropUnroll];
        uint32_t keep[kDropUnroll];
#pragma unroll
        for (int u = 0; u < kDropUnroll; ++u) {
            const int row = rb + u;
            if (row < r1) {
                int js;
                const long long off = shard_offset(p.rows_split, row, p.H, &js);
                raw[u] = V::load_raw(static_cast<const T *>(p.dy[js]) + off + col);
                if (mask) keep[u] = __ldg(mask + row * mask_ld + col / 32) >> (col % 32);
            }
        }
#pragma unroll
        for (int u = 0; u < kDropUnroll; ++u) {
            const int row = rb + u;
            if (row < r1) {
                float v[V::N];
                V::unpack(raw[u], v);
                const long long e = static_cast<long long>(row) * p.H + col;
                if (mask) {
#pragma unroll
                    for (int j = 0; j < V::N; ++j) v[j] = (keep[u] >> j) & 1u ? v[j] * d.scale : 0.0f;
                } else {
#pragma unroll
                    for (int j = 0; j < V::N; j += 4) dropout4(d, e + j, v + j);
                }
                V::store(static_cast<T *>(p.dz) + e, v);
                // the column sums take the stored (rounded) values: db2 = sum_m dZ as the MLP sees it
                V::unpack(V::pack(v), v);
#pragma unroll
                for (int j = 0; j < V::N; ++j) acc[j] += v[j];
            }
        }
    }
    float *out = p.partials + static_cast<long long>(blockIdx.y) * p.H + col;
#pragma unroll
    for (int j = 0; j < V::N; j += 4) *reinterpret_cast<float4 *>(out + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
int ln_bwd_chunks(int M) { return M <= 0 ? 1 : (M + kLnBwdMinRows - 1) / kLnBwdMinRows; }

static int ln_vpt(int H, int dtype) {
    const int nv = H / (dtype == TP_DT_F32 ? 4 : 8);
    for (int v = 1; v <= kLnMaxVpt; v *= 2)
        if (nv <= v * kLnThreads) return v;
    return 0;
}

bool ln_supported(int H, int dtype) { return H % (dtype == TP_DT_F32 ? 4 : 8) == 0 && ln_vpt(H, dtype) > 0; }

// Rows of up to 128 vectors (1024 bf16 / 512 fp32) take one warp each; wider
// rows one block each (a 256-thread block per row keeps more rows' loads in
// flight per SM at widths like 4096 than a 98-register warp per row does:
// 26 us against 30 us for 8192 x 4096 bf16 under ncu).
constexpr int kLnWarpMaxVpw = 4;

template <typename T>
static void ln_fwd_dispatch(const LnPlan &p, int vpt, cudaStream_t st) {
    const int nv = p.H / Vec<T>::N;
    if (nv <= 32 * kLnWarpMaxVpw) {
        const int grid = (p.M + kLnThreads / 32 - 1) / (kLnThreads / 32);
        if (nv <= 32)
            ln_fwd_warp_kernel<T, 1><<<grid, kLnThreads, 0, st>>>(p);
        else if (nv <= 64)
            ln_fwd_warp_kernel<T, 2><<<grid, kLnThreads, 0, st>>>(p);
        else
            ln_fwd_warp_kernel<T, 4><<<grid, kLnThreads, 0, st>>>(p);
        return;
    }
    if (vpt == 1)
        ln_fwd_kernel<T, 1><<<p.M, kLnThreads, 0, st>>>(p);
    else if (vpt == 2)
        ln_fwd_kernel<T, 2><<<p.M, kLnThreads, 0, st>>>(p);
    else
        ln_fwd_kernel<T, 4><<<p.M, kLnThreads, 0, st>>>(p);
}

template <typename T, int VPT>
static void ln_bwd_launch(const LnPlan &p, int *chunks_out, cudaStream_t st) {
    // one wave: rows per block = M / (resident blocks), at least kLnBwdMinRows
    static const int per_sm = [] {  // same value on every device of one architecture
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ln_bwd_kernel<T, VPT>, kLnThreads, 0) != cudaSuccess ||
            n < 1)
            n = 1;
        return n;
    }();
    const long long slots = static_cast<long long>(per_sm) * num_sms();
    int rows = static_cast<int>((p.M + slots - 1) / slots);
    if (rows < kLnBwdMinRows) rows = kLnBwdMinRows;
    const int chunks = (p.M + rows - 1) / rows;
    *chunks_out = chunks;
    ln_bwd_kernel<T, VPT><<<chunks, kLnThreads, 0, st>>>(p, rows);
}

template <typename T>
static void ln_bwd_dispatch(const LnPlan &p, int vpt, int *chunks, cudaStream_t st) {
    if (vpt == 1)
        ln_bwd_launch<T, 1>(p, chunks, st);
    else if (vpt == 2)
        ln_bwd_launch<T, 2>(p, chunks, st);
    else
        ln_bwd_launch<T, 4>(p, chunks, st);
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
    int chunks = 1;
    launch_begin("layernorm_bwd", st);
    if (dtype == TP_DT_F32)
        ln_bwd_dispatch<float>(p, vpt, &chunks, st);
    else
        ln_bwd_dispatch<__nv_bfloat16>(p, vpt, &chunks, st);
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

int dropout_bwd_chunks(int M) { return M <= 0 ? 1 : (M + kDropRows - 1) / kDropRows; }

tp_status launch_dropout_bwd(const LnPlan &p, int dtype, cudaStream_t st) {
    if (p.M == 0) return TP_OK;
    const int vec = dtype == TP_DT_F32 ? 4 : 8;
    const int chunks = dropout_bwd_chunks(p.M);
    const dim3 grid((p.H / vec + kDropThreads - 1) / kDropThreads, chunks);
    launch_begin("dropout_bwd", st);
    if (dtype == TP_DT_F32)
        dropout_bwd_kernel<float><<<grid, kDropThreads, 0, st>>>(p);
    else
        dropout_bwd_kernel<__nv_bfloat16><<<grid, kDropThreads, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    launch_end("dropout_bwd", st);
    if (e != cudaSuccess) return cuda_check(e, "dropout_bwd");
    if (!p.db2) return TP_OK;  // no bias gradient wanted
    ColsumPlan c;
    c.name = "bias_grad_row";
    c.P = 1;
    c.M = p.M;
    c.N = p.H;
    c.out[0] = p.db2;
    c.partials = p.partials;
    return launch_colsum_finalize(c, chunks, st);
}

}  // namespace tpmlp
