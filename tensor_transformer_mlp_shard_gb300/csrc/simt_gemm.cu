// fp32 GEMM engine (CUDA cores, FFMA) for the fp32 problems: the same plans
// and epilogues as the tcgen05 engine, computed in fp32 end to end so that
// results stay within ~1e-6 relative of an fp64 evaluation (tensor-core tf32
// would not).  Tile 64 x 64 per block, 16 x 16 threads, 4 x 4 outputs per
// thread, K staged through shared memory 16 at a time.
#include <cuda_runtime.h>

#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace tpmlp {
namespace simt {

constexpr int TM = 64, TN = 64, TK = 16;

struct Op {
    const float *ptr[kMaxShards];
    int p_stride, s_stride, rows_split, ld, mn_major;
};
struct Out {
    float *ptr[kMaxShards];
    int p_stride, rows_split;
    long long ld;
};
struct Params {
    Op A, B;
    Out out, out2, aux;
    const float *bias[kMaxShards];
    int bias_p_stride, has_bias, has_out2, has_aux;
    int M, N, P, S, Kseg, kind, act, b_dual_off, accumulate;
    DropoutParams drop;
};

// element (mn, k) of an operand for problem pi and K segment s; zero outside
__device__ __forceinline__ float op_get(const Op &o, int pi, int s, int mn, int k) {
    int row = o.mn_major ? k : mn;
    const int col = o.mn_major ? mn : k;
    int idx = pi * o.p_stride + s * o.s_stride;
    if (o.rows_split) {
        idx += row / o.rows_split;
        row %= o.rows_split;
    }
    return o.ptr[idx][static_cast<long long>(row) * o.ld + col];
}

__device__ __forceinline__ float *out_at(const Out &o, int pi, int row) {
    int idx = pi * o.p_stride;
    if (o.rows_split) {
        idx += row / o.rows_split;
        row %= o.rows_split;
    }
    return o.ptr[idx] + static_cast<long long>(row) * o.ld;
}

// Base pointer of an operand for problem pi and K segment s when it is not
// token-sharded (then every element comes from one buffer), else null.
__device__ __forceinline__ const float *op_base(const Op &o, int pi, int s) {
    return o.rows_split ? nullptr : o.ptr[pi * o.p_stride + s * o.s_stride];
}

__device__ __forceinline__ float op_at(const Op &o, const float *base, int pi, int s, int mn, int k) {
    if (base) return base[static_cast<long long>(o.mn_major ? k : mn) * o.ld + (o.mn_major ? mn : k)];
    return op_get(o, pi, s, mn, k);
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const __grid_constant__ Params p) {
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs[TK][TN + 4];
    __shared__ float Bs2[TK][TN + 4];
    const int pi = blockIdx.z;
    const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const bool dual = p.b_dual_off != 0;
    float acc[4][4] = {}, acc2[4][4] = {};
    for (int s = 0; s < p.S; ++s) {
        const float *abase = op_base(p.A, pi, s), *bbase = op_base(p.B, pi, s);
        for (int k0 = 0; k0 < p.Kseg; k0 += TK) {
            for (int e = threadIdx.x; e < TK * TM; e += blockDim.x) {
                // consecutive threads walk the operand's contiguous dimension
                int kk, mm;
                if (p.A.mn_major) { mm = e % TM; kk = e / TM; } else { kk = e % TK; mm = e / TK; }
                const int m = m0 + mm, k = k0 + kk;
                As[kk][mm] = (m < p.M && k < p.Kseg) ? op_at(p.A, abase, pi, s, m, k) : 0.0f;
            }
            for (int e = threadIdx.x; e < TK * TN; e += blockDim.x) {
                int kk, nn;
                if (p.B.mn_major) { nn = e % TN; kk = e / TN; } else { kk = e % TK; nn = e / TK; }
                const int n = n0 + nn, k = k0 + kk;
                const bool ok = n < p.N && k < p.Kseg;
                Bs[kk][nn] = ok ? op_at(p.B, bbase, pi, s, n, k) : 0.0f;
                if (dual) Bs2[kk][nn] = ok ? op_at(p.B, bbase, pi, s, n + p.b_dual_off, k) : 0.0f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < TK; ++kk) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                if (dual) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) b[j] = Bs2[kk][tx * 4 + j];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc2[i][j] = fmaf(a[i], b[j], acc2[i][j]);
                }
            }
            __syncthreads();
        }
    }
    const float *bias = p.has_bias ? p.bias[pi * p.bias_p_stride] : nullptr;
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= p.M) continue;
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= p.N) continue;
            float v = acc[i][j];
            if (p.kind == EPI_COL) {
                if (p.act == TP_ACT_SWIGLU) {
                    float G = v, U = acc2[i][j];
                    if (bias) {
                        G += bias[n];
                        U += bias[p.N + n];
                    }
                    if (p.has_out2) {
                        float *pre = out_at(p.out2, pi, m);
                        pre[n] = G;
                        pre[p.N + n] = U;
                    }
                    out_at(p.out, pi, m)[n] = G * sigmoid_f(G) * U;
                } else {
                    if (bias) v += bias[n];
                    if (p.has_out2) out_at(p.out2, pi, m)[n] = v;
                    out_at(p.out, pi, m)[n] = p.act == TP_ACT_GELU_TANH ? gelu_tanh_f(v) : v;
                }
            } else if (p.kind == EPI_PLAIN) {
                if (bias) v += bias[n];
                if (p.drop.on) {
                    // draw of element (m, n): word (e mod 4) of the Philox block e div 4
                    const long long e = static_cast<long long>(m) * p.drop.ld + n;
                    float w4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    w4[e & 3] = v;
                    dropout4(p.drop, e & ~3ll, w4);
                    v = w4[e & 3];
                }
                if (p.has_aux) v += out_at(p.aux, pi, m)[n];
                out_at(p.out, pi, m)[n] = v;
            } else if (p.kind == EPI_DACT) {
                const float *pre = out_at(p.aux, pi, m);
                float *o = out_at(p.out, pi, m);
                if (p.act == TP_ACT_GELU_TANH) {
                    o[n] = v * gelu_tanh_grad_f(pre[n]);
                } else if (p.act == TP_ACT_SWIGLU) {
                    const float G = pre[n], U = pre[p.N + n], sg = sigmoid_f(G);
                    o[n] = v * U * sg * (1.0f + G * (1.0f - sg));
                    o[p.N + n] = v * G * sg;
                } else {
                    o[n] = v;
                }
            } else {  // EPI_F32
                float *o = out_at(p.out, pi, m);
                o[n] = p.accumulate ? o[n] + v : v;
            }
        }
    }
}

static void copy_op(Op &o, const OperandPlan &src) {
    for (int i = 0; i < kMaxShards; ++i) o.ptr[i] = i < src.n ? static_cast<const float *>(src.ptr[i]) : nullptr;
    o.p_stride = src.p_stride;
    o.s_stride = src.s_stride;
    o.rows_split = src.rows_split;
    o.ld = src.cols;
    o.mn_major = src.mn_major ? 1 : 0;
}

static void copy_out(Out &o, const OutPlan &src) {
    for (int i = 0; i < kMaxShards; ++i) o.ptr[i] = i < src.n ? static_cast<float *>(src.ptr[i]) : nullptr;
    o.p_stride = src.p_stride;
    o.rows_split = src.rows_split;
    o.ld = src.ld;
}

}  // namespace simt

tp_status launch_simt_gemm(const GemmPlan &g, cudaStream_t st) {
    using namespace simt;
    Params prm;
    memset(&prm, 0, sizeof(prm));
    copy_op(prm.A, g.A);
    copy_op(prm.B, g.B);
    copy_out(prm.out, g.out);
    copy_out(prm.out2, g.out2);
    copy_out(prm.aux, g.aux);
    for (int i = 0; i < kMaxShards; ++i) prm.bias[i] = g.has_bias ? static_cast<const float *>(g.bias[i]) : nullptr;
    prm.bias_p_stride = g.bias_p_stride;
    prm.has_bias = g.has_bias;
    prm.has_out2 = g.out2.n > 0;
    prm.has_aux = g.aux.n > 0;
    prm.M = g.M;
    prm.N = g.N;
    prm.P = g.P;
    prm.S = g.S;
    prm.Kseg = g.Kseg;
    prm.kind = g.kind;
    prm.act = g.act;
    prm.b_dual_off = g.b_dual_off;
    prm.accumulate = g.accumulate;
    prm.drop.on = g.dropout ? 1 : 0;
    prm.drop.threshold = g.drop_threshold;
    prm.drop.scale = g.drop_scale;
    prm.drop.seed_lo = static_cast<uint32_t>(g.drop_seed);
    prm.drop.seed_hi = static_cast<uint32_t>(g.drop_seed >> 32);
    prm.drop.ld = g.N;
    prm.drop.mask = nullptr;  // the fp32 engine recomputes keep flags in the backward
    prm.drop.mask_ld = 0;
    if (g.dropout && g.drop_mask)
        return set_error(TP_ERR_UNSUPPORTED, "the fp32 engine does not write a dropout keep-mask");
    if (g.M == 0 || g.N == 0 || g.P == 0) return TP_OK;
    dim3 grid((g.N + TN - 1) / TN, (g.M + TM - 1) / TM, g.P);
    launch_begin(g.name, st);
    simt_gemm_kernel<<<grid, 256, 0, st>>>(prm);
    cudaError_t e = cudaGetLastError();
    launch_end(g.name, st);
    return cuda_check(e, g.name);
}

}  // namespace tpmlp
