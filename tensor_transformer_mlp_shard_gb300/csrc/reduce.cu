// Token-dimension column sums (the bias gradients db = sum_m dOut[m, :]),
// the device status words and the bounded-wait self-test kernel.
//
// The column sum is HBM-bound: one pass over the input with 16-byte
// coalesced loads.  Pass 1 sums fixed chunks of token rows per column strip
// into fp32 partials (workspace); pass 2 adds the partials of each column in
// chunk order.  Both passes use a fixed order, so results are run-to-run
// deterministic (no atomics).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace tpmlp {

// ---------------------------------------------------------------------------
// status words
// ---------------------------------------------------------------------------
// One status word and one abort word per slot.  Slot 0 belongs to the calls
// without a handle (the single-layer entry points, the FP8 quantiser and the
// wait self-test); every MLP or sub-block handle owns a slot of its own for
// its lifetime, so that a timeout is reported to, and cleared by, the handle
// whose launch raised it.
__device__ int g_tp_status[kStatusSlots];  // first device-side error per slot
__device__ unsigned g_tp_abort[kStatusSlots];
__device__ unsigned g_tp_never_set = 0;
// SM cycles and wall-clock nanoseconds summed over the CTAs of the GEMM
// launches made while the per-kernel timer is on (clock64 and %globaltimer
// read by one thread at the start and end of each CTA), one pair per kernel
// name: their ratio is the SM clock those kernels actually ran at.
__device__ unsigned long long g_tp_clk[2 * kClockSlots];

static std::mutex g_slot_mu;
static bool g_slot_used[kStatusSlots] = {true};  // slot 0 is never handed out
static thread_local int g_cur_slot = 0;

int alloc_status_slot() {
    std::lock_guard<std::mutex> lock(g_slot_mu);
    for (int i = 1; i < kStatusSlots; ++i)
        if (!g_slot_used[i]) {
            g_slot_used[i] = true;
            return i;
        }
    return -1;
}

void free_status_slot(int slot) {
    if (slot <= 0 || slot >= kStatusSlots) return;
    std::lock_guard<std::mutex> lock(g_slot_mu);
    g_slot_used[slot] = false;
}

StatusScope::StatusScope(int slot) : prev_(g_cur_slot) { g_cur_slot = slot; }
StatusScope::~StatusScope() { g_cur_slot = prev_; }

tp_status device_words(DeviceWords *w, const char *kernel) {
    static int *st_base[64] = {};
    static unsigned *ab_base[64] = {};
    static unsigned long long *clk_base[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return set_error(TP_ERR_UNSUPPORTED, "device ordinal %d above 63", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!st_base[dev]) {
        void *ps = nullptr, *pa = nullptr, *pc = nullptr;
        e = cudaGetSymbolAddress(&ps, g_tp_status);
        if (e != cudaSuccess) return cuda_check(e, "cudaGetSymbolAddress(status)");
        e = cudaGetSymbolAddress(&pa, g_tp_abort);
        if (e != cudaSuccess) return cuda_check(e, "cudaGetSymbolAddress(abort)");
        e = cudaGetSymbolAddress(&pc, g_tp_clk);
        if (e != cudaSuccess) return cuda_check(e, "cudaGetSymbolAddress(clock)");
        st_base[dev] = static_cast<int *>(ps);
        ab_base[dev] = static_cast<unsigned *>(pa);
        clk_base[dev] = static_cast<unsigned long long *>(pc);
    }
    w->status = st_base[dev] + g_cur_slot;
    w->abort_word = ab_base[dev] + g_cur_slot;
    const int slot = kernel ? prof_clock_slot(kernel) : -1;
    w->clk = slot >= 0 ? clk_base[dev] + 2 * slot : nullptr;
    return TP_OK;
}

tp_status read_and_clear_status(cudaStream_t st, int slot, int *out) {
    if (slot < 0 || slot >= kStatusSlots) return set_error(TP_ERR_ARG, "bad status slot %d", slot);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_check(e, "cudaStreamSynchronize");
    const size_t off = sizeof(int) * static_cast<size_t>(slot);
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_tp_status, sizeof(int), off);
    if (e != cudaSuccess) return cuda_check(e, "cudaMemcpyFromSymbol(status)");
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_tp_status, &zero, sizeof(int), off);
    if (e != cudaSuccess) return cuda_check(e, "cudaMemcpyToSymbol(status)");
    *out = v;
    return TP_OK;
}

tp_status read_and_clear_clocks(unsigned long long *v) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_check(e, "cudaDeviceSynchronize");
    e = cudaMemcpyFromSymbol(v, g_tp_clk, sizeof(unsigned long long) * 2 * kClockSlots);
    if (e != cudaSuccess) return cuda_check(e, "cudaMemcpyFromSymbol(clock)");
    static const unsigned long long zero[2 * kClockSlots] = {};
    e = cudaMemcpyToSymbol(g_tp_clk, zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_check(e, "cudaMemcpyToSymbol(clock)");
    return TP_OK;
}

// Waits for a flag that nothing sets; the wall-clock bound ends the wait and
// the kernel records TP_ERR_TIMEOUT, like any of the GEMM kernels' waits.
__global__ void wait_timeout_kernel(unsigned long long limit_ns, int *status) {
    const uint64_t t0 = global_timer_ns();
    while (*reinterpret_cast<volatile unsigned *>(&g_tp_never_set) == 0) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicCAS(status, 0, TP_ERR_TIMEOUT);
            return;
        }
        __nanosleep(1000);
    }
}

tp_status launch_wait_timeout(unsigned long long limit_ns, cudaStream_t st) {
    DeviceWords w;
    tp_status s = device_words(&w);
    if (s != TP_OK) return s;
    launch_begin("wait_timeout", st);
    wait_timeout_kernel<<<1, 1, 0, st>>>(limit_ns, w.status);
    cudaError_t e = cudaGetLastError();
    launch_end("wait_timeout", st);
    return cuda_check(e, "wait_timeout_kernel");
}

// ---------------------------------------------------------------------------
// column sums
// ---------------------------------------------------------------------------
constexpr int kChunkRows = 256;
constexpr int kWarps = 8;

int colsum_chunks(int M) { return M <= 0 ? 1 : (M + kChunkRows - 1) / kChunkRows; }

struct ColsumParams {
    const void *ptr[kMaxShards];
    int p_stride, rows_split;
    long long ld;
    int M, N, chunks;
    float *partials;
    float *out[kMaxShards];
};

template <typename T>
__device__ __forceinline__ void load_vec(const T *src, float *dst);

template <>
__device__ __forceinline__ void load_vec<__nv_bfloat16>(const __nv_bfloat16 *src, float *dst) {
    const uint4 w = *reinterpret_cast<const uint4 *>(src);
    dst[0] = bf16_lo(w.x); dst[1] = bf16_hi(w.x);
    dst[2] = bf16_lo(w.y); dst[3] = bf16_hi(w.y);
    dst[4] = bf16_lo(w.z); dst[5] = bf16_hi(w.z);
    dst[6] = bf16_lo(w.w); dst[7] = bf16_hi(w.w);
}

template <>
__device__ __forceinline__ void load_vec<float>(const float *src, float *dst) {
    const float4 w = *reinterpret_cast<const float4 *>(src);
    dst[0] = w.x; dst[1] = w.y; dst[2] = w.z; dst[3] = w.w;
}

// grid: x = column strips of 32*VEC columns, y = row chunks, z = problems
template <typename T, int VEC>
__global__ void __launch_bounds__(32 * kWarps) colsum_partial_kernel(const __grid_constant__ ColsumParams p) {
    __shared__ float red[kWarps][32 * VEC];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int z = blockIdx.z;
    const int col = blockIdx.x * 32 * VEC + lane * VEC;
    const int r0 = blockIdx.y * kChunkRows;
    const int r1 = min(p.M, r0 + kChunkRows);
    float acc[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.0f;
    if (col < p.N) {
        for (int r = r0 + warp; r < r1; r += kWarps) {
            int idx = z * p.p_stride, lr = r;
            if (p.rows_split) {
                idx += r / p.rows_split;
                lr = r % p.rows_split;
            }
            const T *src = static_cast<const T *>(p.ptr[idx]) + static_cast<long long>(lr) * p.ld + col;
            float v[VEC];
            load_vec<T>(src, v);
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc[j] += v[j];
        }
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) red[warp][lane * VEC + j] = acc[j];
    __syncthreads();
    for (int c = threadIdx.x; c < 32 * VEC; c += blockDim.x) {
        const int gc = blockIdx.x * 32 * VEC + c;
        if (gc >= p.N) continue;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[w][c];
        p.partials[(static_cast<long long>(z) * p.chunks + blockIdx.y) * p.N + gc] = s;
    }
}

// Second pass: out_z[c] = sum_k partials[z][k][c].  A cluster of S blocks owns
// 32 columns and block s of it the partial rows of slice [s K / S, (s + 1) K / S):
// its warp w of 16 adds the rows lo + w, lo + w + 16, ... in increasing order
// (four interleaved accumulators for memory-level parallelism, combined in a
// fixed order) and warp 0 adds the warps' sums in warp order; after a cluster
// barrier block 0 adds the S slice sums in rank order through distributed
// shared memory.  Deterministic for a given S, which the host derives from the
// shape alone (S > 1 spreads tall, narrow sums such as a 65536-token bias
// gradient over more SMs).
constexpr int kFinWarps = 16;
__global__ void __launch_bounds__(32 * kFinWarps) colsum_finalize_kernel(const __grid_constant__ ColsumParams p) {
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    __shared__ float red[kFinWarps][32];
    __shared__ float slice[32];
    const unsigned S = cl.num_blocks(), rank = cl.block_rank();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int z = blockIdx.y;
    const int c = static_cast<int>(blockIdx.x / S) * 32 + lane;
    const int lo = static_cast<int>(static_cast<long long>(p.chunks) * rank / S);
    const int hi = static_cast<int>(static_cast<long long>(p.chunks) * (rank + 1) / S);
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    if (c < p.N) {
        const float *src = p.partials + static_cast<long long>(z) * p.chunks * p.N + c;
        const long long step = static_cast<long long>(kFinWarps) * p.N;
        int k = lo + warp;
        for (; k + 3 * kFinWarps < hi; k += 4 * kFinWarps) {
            const float *q = src + static_cast<long long>(k) * p.N;
            a0 += q[0];
            a1 += q[step];
            a2 += q[2 * step];
            a3 += q[3 * step];
        }
        for (; k < hi; k += kFinWarps) a0 += src[static_cast<long long>(k) * p.N];
    }
    red[warp][lane] = (a0 + a1) + (a2 + a3);
    __syncthreads();
    if (warp == 0) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < kFinWarps; ++w) t += red[w][lane];
        slice[lane] = t;
    }
    cl.sync();
    if (rank == 0 && warp == 0 && c < p.N) {
        float t = slice[lane];
        for (unsigned r = 1; r < S; ++r) t += cl.map_shared_rank(slice, r)[lane];
        p.out[z][c] = t;
    }
    cl.sync();  // the other blocks' slice sums stay until block 0 has read them
}

// The finalize over P problems of N columns and K partial rows: S (the
// cluster size) doubles up to 8 while the grid stays within two blocks per SM
// and every slice keeps 64 rows.
static tp_status launch_finalize(const ColsumParams &prm, int P, cudaStream_t st) {
    const int ncb = (prm.N + 31) / 32;
    int S = 1;
    while (S < 8 && static_cast<long long>(ncb) * P * (2 * S) <= 2ll * num_sms() && prm.chunks / (2 * S) >= 64)
        S *= 2;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(ncb * S, P, 1);
    cfg.blockDim = dim3(32 * kFinWarps, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    launch_begin("colsum_finalize", st);
    cudaError_t e = cudaLaunchKernelEx(&cfg, colsum_finalize_kernel, prm);
    launch_end("colsum_finalize", st);
    return cuda_check(e, "colsum_finalize");
}

tp_status launch_colsum_finalize(const ColsumPlan &c, int chunks, cudaStream_t st) {
    ColsumParams prm;
    memset(&prm, 0, sizeof(prm));
    for (int i = 0; i < kMaxShards; ++i) prm.out[i] = i < c.P ? c.out[i] : nullptr;
    prm.M = c.M;
    prm.N = c.N;
    prm.chunks = chunks;
    prm.partials = c.partials;
    if (c.N == 0 || c.P == 0) return TP_OK;
    return launch_finalize(prm, c.P, st);
}

// ---------------------------------------------------------------------------
// split-K reduction of the weight gradients: four fp32 per thread, splits
// added in index order (deterministic)
// ---------------------------------------------------------------------------
struct SplitkParams {
    const float *part;
    float *out[kMaxShards];
    int ksplit, P, M, split_rows, N, accumulate;
};

__global__ void __launch_bounds__(256) splitk_reduce_kernel(const __grid_constant__ SplitkParams p) {
    const int z = blockIdx.y;
    const long long nq = static_cast<long long>(p.M) * p.N / 4;  // float4 groups of one problem
    const long long plane = static_cast<long long>(p.split_rows) * p.N;
    for (long long q = blockIdx.x * 256ll + threadIdx.x; q < nq; q += static_cast<long long>(gridDim.x) * 256) {
        const long long e = q * 4;
        const float *src = p.part + static_cast<long long>(z) * plane + e;
        float4 s = *reinterpret_cast<const float4 *>(src);
        // eight splits' loads in flight at a time, added in split order
        for (int k0 = 1; k0 < p.ksplit; k0 += 8) {
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (k0 + j < p.ksplit)
                    v[j] = *reinterpret_cast<const float4 *>(src + static_cast<long long>(k0 + j) * p.P * plane);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (k0 + j < p.ksplit) {
                    s.x += v[j].x;
                    s.y += v[j].y;
                    s.z += v[j].z;
                    s.w += v[j].w;
                }
            }
        }
        float4 *dst = reinterpret_cast<float4 *>(p.out[z] + e);
        if (p.accumulate) {
            const float4 o = *dst;
            s.x += o.x;
            s.y += o.y;
            s.z += o.z;
            s.w += o.w;
        }
        *dst = s;
    }
}

tp_status launch_splitk_reduce(const float *part, int ksplit, int P, int M, int split_rows, int N,
                               float *const *out, bool accumulate, cudaStream_t st) {
    if (N % 4) return set_error(TP_ERR_SHAPE, "split-K reduction needs N %% 4 == 0 (N=%d)", N);
    SplitkParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.part = part;
    for (int i = 0; i < kMaxShards; ++i) prm.out[i] = i < P ? out[i] : nullptr;
    prm.ksplit = ksplit;
    prm.P = P;
    prm.M = M;
    prm.split_rows = split_rows;
    prm.N = N;
    prm.accumulate = accumulate ? 1 : 0;
    const long long nq = static_cast<long long>(M) * N / 4;
    if (nq == 0 || P == 0) return TP_OK;
    long long blocks = (nq + 255) / 256;
    const long long cap = 4ll * num_sms();
    if (blocks > cap) blocks = cap;
    launch_begin("splitk_reduce", st);
    splitk_reduce_kernel<<<dim3(static_cast<unsigned>(blocks), P), 256, 0, st>>>(prm);
    cudaError_t e = cudaGetLastError();
    launch_end("splitk_reduce", st);
    return cuda_check(e, "splitk_reduce");
}

tp_status launch_colsum(const ColsumPlan &c, int dtype, cudaStream_t st) {
    ColsumParams prm;
    memset(&prm, 0, sizeof(prm));
    for (int i = 0; i < kMaxShards; ++i) {
        prm.ptr[i] = i < c.in.n ? c.in.ptr[i] : nullptr;
        prm.out[i] = i < c.P ? c.out[i] : nullptr;
    }
    prm.p_stride = c.in.p_stride;
    prm.rows_split = c.in.rows_split;
    prm.ld = c.in.ld;
    prm.M = c.M;
    prm.N = c.N;
    prm.chunks = colsum_chunks(c.M);
    prm.partials = c.partials;
    if (c.N == 0 || c.P == 0) return TP_OK;
    if (c.M == 0) {
        for (int z = 0; z < c.P; ++z) {
            cudaError_t e = cudaMemsetAsync(c.out[z], 0, sizeof(float) * c.N, st);
            if (e != cudaSuccess) return cuda_check(e, "cudaMemsetAsync(colsum)");
        }
        return TP_OK;
    }
    const int vec = dtype == TP_DT_BF16 ? 8 : 4;
    dim3 g1((c.N + 32 * vec - 1) / (32 * vec), prm.chunks, c.P);
    launch_begin(c.name, st);
    if (dtype == TP_DT_BF16)
        colsum_partial_kernel<__nv_bfloat16, 8><<<g1, 32 * kWarps, 0, st>>>(prm);
    else
        colsum_partial_kernel<float, 4><<<g1, 32 * kWarps, 0, st>>>(prm);
    cudaError_t e = cudaGetLastError();
    launch_end(c.name, st);
    if (e != cudaSuccess) return cuda_check(e, c.name);
    return launch_finalize(prm, c.P, st);
}

}  // namespace tpmlp
