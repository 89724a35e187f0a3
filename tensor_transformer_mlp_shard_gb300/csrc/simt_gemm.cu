// fp32 GEMM engine (CUDA cores, FFMA) for the fp32 problems: the same plans
// and epilogues as the tcgen05 engine, computed in fp32 end to end so that
// results stay within ~1e-6 relative of an fp64 evaluation (tensor-core tf32
// would not).  Tile 64 x 64 per block, 16 x 16 threads, 4 x 4 outputs per
// thread, K staged through shared memory 16 at a time, the next 16 loaded
// into registers while the current ones are multiplied.  The fp32 problems
// are small (few output tiles, long K), so the K range of a tile is split
// over the KS blocks of a thread-block cluster: each adds its part into its
// own shared memory, and after a cluster barrier each block sums one KS-th
// of the tile's rows over the KS parts, in rank order, through distributed
// shared memory and runs the epilogue on them (no workspace, deterministic).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace tpmlp {
namespace simt {

constexpr int TM = 64, TN = 64, TK = 16;
constexpr int KS_MAX = 8;  // K splits per tile: the portable cluster size

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
    int ks;  // K splits per tile (the cluster size along x), a power of two <= KS_MAX
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

// Epilogue of output (m, n) of problem pi: v the accumulator, v2 the up
// half's (SwiGLU column forward)
__device__ __forceinline__ void epilogue_elem(const Params &p, const float *bias, int pi, int m, int n, float v,
                                              float v2) {
    if (p.kind == EPI_COL) {
        if (p.act == TP_ACT_SWIGLU) {
            float G = v, U = v2;
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

// element e (0 .. TK * T - 1) of a K tile: its (k, mn) within the tile, with
// consecutive threads walking the operand's contiguous dimension
__device__ __forceinline__ void tile_pos(bool mn_major, int T, int e, int &kk, int &mm) {
    if (mn_major) {
        mm = e % T;
        kk = e / T;
    } else {
        kk = e % TK;
        mm = e / TK;
    }
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const __grid_constant__ Params p) {
    namespace cg = cooperative_groups;
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs[TK][TN + 4];
    __shared__ float Bs2[TK][TN + 4];
    __shared__ float red[TM][TN + 1];   // this block's part of the tile
    __shared__ float red2[TM][TN + 1];  // ... of the up half (SwiGLU)
    cg::cluster_group cl = cg::this_cluster();
    const int ks = static_cast<int>(cl.block_rank());  // K split of this block (cluster dims {KS, 1, 1})
    const int pi = blockIdx.z;
    const int m0 = blockIdx.y * TM, n0 = (blockIdx.x / p.ks) * TN;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const bool dual = p.b_dual_off != 0;
    // this block's K tiles: [t0, t1) of the S * tps tiles of the K loop over
    // (segment, 16-wide K tile)
    const int tps = (p.Kseg + TK - 1) / TK;
    const int kt = p.S * tps;
    const int t0 = static_cast<int>(static_cast<long long>(ks) * kt / p.ks);
    const int t1 = static_cast<int>(static_cast<long long>(ks + 1) * kt / p.ks);
    float acc[4][4] = {}, acc2[4][4] = {};
    float ra[4], rb[4], rb2[4];  // the next K tile, four elements of each operand per thread
    auto load = [&](int t) {
        const int s = t / tps, k0 = (t - s * tps) * TK;
        const float *abase = op_base(p.A, pi, s), *bbase = op_base(p.B, pi, s);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = threadIdx.x + 256 * i;
            int kk, mm;
            tile_pos(p.A.mn_major, TM, e, kk, mm);
            ra[i] = (m0 + mm < p.M && k0 + kk < p.Kseg) ? op_at(p.A, abase, pi, s, m0 + mm, k0 + kk) : 0.0f;
            tile_pos(p.B.mn_major, TN, e, kk, mm);
            const bool ok = n0 + mm < p.N && k0 + kk < p.Kseg;
            rb[i] = ok ? op_at(p.B, bbase, pi, s, n0 + mm, k0 + kk) : 0.0f;
            rb2[i] = dual && ok ? op_at(p.B, bbase, pi, s, n0 + mm + p.b_dual_off, k0 + kk) : 0.0f;
        }
    };
    if (t0 < t1) load(t0);
    for (int t = t0; t < t1; ++t) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = threadIdx.x + 256 * i;
            int kk, mm;
            tile_pos(p.A.mn_major, TM, e, kk, mm);
            As[kk][mm] = ra[i];
            tile_pos(p.B.mn_major, TN, e, kk, mm);
            Bs[kk][mm] = rb[i];
            if (dual) Bs2[kk][mm] = rb2[i];
        }
        __syncthreads();
        if (t + 1 < t1) load(t + 1);  // in flight while this tile is multiplied
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
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            red[ty * 4 + i][tx * 4 + j] = acc[i][j];
            if (dual) red2[ty * 4 + i][tx * 4 + j] = acc2[i][j];
        }
    cl.sync();  // every part of the tile is in its block's shared memory
    // rows [r0, r0 + TM / KS) of the tile: the KS parts added in rank order
    const int rows = TM / p.ks, r0 = ks * rows;
    const float *bias = p.has_bias ? p.bias[pi * p.bias_p_stride] : nullptr;
    for (int e = threadIdx.x; e < rows * TN; e += blockDim.x) {
        const int r = r0 + e / TN, c = e % TN;
        const int m = m0 + r, n = n0 + c;
        float v = 0.0f, v2 = 0.0f;
        for (int q = 0; q < p.ks; ++q) {
            v += cl.map_shared_rank(&red[0][0], q)[r * (TN + 1) + c];
            if (dual) v2 += cl.map_shared_rank(&red2[0][0], q)[r * (TN + 1) + c];
        }
        if (m < p.M && n < p.N) epilogue_elem(p, bias, pi, m, n, v, v2);
    }
    cl.sync();  // no block exits while another may still read its part
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
    // K splits: double them while the grid stays within two blocks per SM
    // and every split keeps at least four 16-wide K tiles
    const long long tiles = static_cast<long long>((g.N + TN - 1) / TN) * ((g.M + TM - 1) / TM) * g.P;
    const long long kt = static_cast<long long>(g.S) * ((g.Kseg + TK - 1) / TK);
    int ks = 1;
    while (ks * 2 <= KS_MAX && tiles * ks * 2 <= 2ll * num_sms() && kt / (ks * 2) >= 4) ks *= 2;
    prm.ks = ks;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(((g.N + TN - 1) / TN) * ks, (g.M + TM - 1) / TM, g.P);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    launch_begin(g.name, st);
    cudaError_t e = cudaLaunchKernelEx(&cfg, simt_gemm_kernel, prm);
    launch_end(g.name, st);
    return cuda_check(e, g.name);
}

}  // namespace tpmlp
