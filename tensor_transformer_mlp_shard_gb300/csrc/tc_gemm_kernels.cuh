// GEMM engine for sm_103a (kernels): TMA -> shared-memory ring -> tcgen05.mma
// -> TMEM accumulators -> fused epilogue, in one persistent, warp-specialised
// kernel.  Operands are bf16 (kind::f16) or, for the FP8 variant, E4M3/E5M2
// (kind::f8f6f4) with a per-GEMM dequantisation factor in the epilogue.  Every product of the tensor-parallel MLP runs on it:
//   column forward   pre_p = X W1_p^T (+b1_p), A_p = act(pre_p)      EPI_COL
//   row forward      Y = sum_s A_s W2_s^T (+b2) (+X)                EPI_PLAIN, S = T
//   row dgrad        dPre_p = (dY W2_p) * act'(pre_p)               EPI_DACT
//   column dgrad     dX = sum_s dPre_s W1_s (+dY)                   EPI_PLAIN, S = T
//   weight grads     dW = G^T Act (fp32, both operands MN-major)     EPI_F32
// The cross-shard sums (the forward and backward all-reduces of the
// multi-GPU layer) are the K loop over segments s: every shard's K range is
// accumulated into the same fp32 TMEM accumulator in shard order.
//
// Tile: 128 x 256 (tcgen05 M=128, N=256, cta_group::1); a stage holds one
// 128-byte swizzle row of K per operand row: 64 bf16 or 128 fp8 elements
// (4 MMAs of K=16 bf16 or K=32 fp8).  Warp 0 issues TMA, warp 1 issues
// MMAs, warps 2-9 run the epilogue out of one of two TMEM accumulators while
// the next tile accumulates into the other.
#pragma once
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace tpmlp {
namespace tc {

constexpr int BM = 128, BN = 256, STAGES = 4;
constexpr int ROW_BYTES = 128;           // one swizzle row of K per operand row and stage
constexpr int A_BYTES = BM * ROW_BYTES;  // 16 KB
constexpr int B_BYTES = BN * ROW_BYTES;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter, each owning half the columns
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int TMEM_COLS = 2 * BN;  // two fp32 accumulators of 128 lanes x 256 columns

// Element-type dependent shapes: K elements per stage (one 128-byte row),
// MN elements per MN-major box (one 128-byte row), bytes of one MN-major box,
// and the shared-memory advance of one MMA's K step in an MN-major tile.
template <bool F8>
struct Elem {
    static constexpr int BKE = F8 ? 128 : 64;
    static constexpr int MNB = F8 ? 128 : 64;
    static constexpr uint32_t MNB_BYTES = ROW_BYTES * BKE;      // 16 KB fp8, 8 KB bf16
    static constexpr uint32_t KADV_MN = ROW_BYTES * (F8 ? 32 : 16);
};
// Epilogue staging: each epilogue warp owns two 2 KB buffers of 32 rows x
// 64 bytes (64-byte swizzle) that feed bulk tensor stores.
constexpr int EPI_STAGE_BYTES = 4096;
constexpr int EPI_SMEM = EPI_WARPS * EPI_STAGE_BYTES;  // 32 KB
constexpr int BAR_BYTES = 1024;                          // barriers + TMEM slot
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES + EPI_SMEM;

struct Sel {
    int p_stride, s_stride, rows_split, nsplit;  // nsplit: token shards (when rows_split > 0)
};
struct Out {
    void *ptr[kMaxShards];
    int p_stride, rows_split, nsplit;
    long long ld;
};

struct Params {
    CUtensorMap mapA[kMaxShards];
    CUtensorMap mapB[kMaxShards];
    CUtensorMap mapO[kMaxShards];    // bulk-store maps of `out` (when out_tma)
    CUtensorMap mapO2[kMaxShards];   // ... and of `out2`
    int out_tma;                     // epilogue writes through shared memory + bulk tensor stores
    Sel selA, selB;
    Out out, out2, aux;
    const void *bias[kMaxShards];
    int bias_p_stride, has_bias, has_out2, has_aux;
    int M, N, P, S, Kseg, num_kb;
    int m_tiles, n_tiles, total_tiles, group_m;
    // split-K (weight gradients): tile t covers K blocks [ks * kb_split, ...) of
    // split ks = t / tiles_per_split and writes fp32 partial sums at row
    // (ks * P + p) * split_rows of the single partial buffer (split_rows = 0:
    // no split, the plain output addressing)
    int tiles_per_split, kb_split, split_rows;
    // Tail split (CTA-pair kernel): when the tiles leave the last round of the
    // persistent grid part-filled, each tile from tail_first on is cut along
    // its flattened (segment, K block) range into tail_s units, so that the
    // last round's work spreads over more pairs.  The work items are the
    // tiles below tail_first, then the units; total_work counts them.  A unit
    // writes its raw fp32 accumulator to tail_ws; the warp that completes a
    // 32-row x 128-column slice (counted in tail_cnt, zeroed before the
    // launch) sums the units' slices in unit order and runs the epilogue.
    int total_work, tail_first, tail_s;
    // CTA-pair kernel, bf16: an MN-major operand whose MN extent is a multiple
    // of 64 is loaded as one 3D box {64 elements, 64 K rows, 2 groups of 64}
    // (its map views [K, MN] as {64, K, MN / 64} with strides {row pitch, 128
    // bytes}), landing as the two 8 KB swizzle atoms of the 128-wide tile that
    // two 2D boxes would write
    int a3d, b3d;
    // CTA-pair kernel: the producer walks the K loop of a whole tile
    // backwards in every other round of the persistent loop.  Consecutive
    // rounds share operand panels (the same band of row tiles, a column
    // tile), and a round that starts where the previous one ended re-reads
    // from L2 the K blocks that round loaded last instead of from HBM.
    int k_reverse;
    float *tail_ws;                  // [tail tile][tail_s][256 rows][BN] fp32
    unsigned *tail_cnt;              // [tail tile][16 warp slices]
    int act, b_dual_off, accumulate;
    uint32_t idesc;                  // tcgen05 instruction descriptor (formats, majors, M, N)
    DropoutParams drop;              // EPI_PLAIN: out = residual + dropout(acc + bias)
    // FP8 codes of the bf16 output (A of the column forward, dPre of the act'
    // dgrad) written by the epilogue when the scale is known in advance (FP8
    // delayed scaling): codes = fp8(bf16(out) * fmax / *q_scale_amax)
    CUtensorMap mapQ[kMaxShards];    // [rows, cols] bytes, boxes of 32 rows x 32 bytes
    int q_out, q_fmt, q_only;        // q_only (EPI_DACT): store the codes, not the bf16 out
    const float *q_scale_amax;
    float *amax_out;                 // bulk-store epilogue: atomic max |bf16 output| (A / dPre), or null
    float *col_partials;             // DACT bulk-store epilogue: per-32-row-block column sums, or null
    int partial_ld;                  //   [P][ceil(M/32)][partial_ld] floats
    const float *amax_a, *amax_b;    // FP8: per-tensor amax of the two operands, else null
    float fmax_a, fmax_b;            // FP8: largest finite value of each operand's format
    int *status;
    unsigned *abort_word;
    unsigned launch_id;
    unsigned long long wait_limit_ns;
    // when non-null: thread 0 of every CTA adds the SM cycles (clock64) and
    // nanoseconds (%globaltimer) between the CTA's start and end to clk[0]
    // and clk[1] -- the SM clock the kernel ran at, for the per-kernel timer
    unsigned long long *clk;
};

// Start and end of a CTA's clock record (see Params::clk).
struct ClockMark {
    unsigned long long c0 = 0, t0 = 0;
    __device__ __forceinline__ void start(const unsigned long long *clk) {
        if (clk && threadIdx.x == 0) {
            c0 = clock64();
            t0 = global_timer_ns();
        }
    }
    __device__ __forceinline__ void stop(unsigned long long *clk) const {
        if (clk && threadIdx.x == 0) {
            atomicAdd(clk, static_cast<unsigned long long>(clock64()) - c0);
            atomicAdd(clk + 1, global_timer_ns() - t0);
        }
    }
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with parity `parity` to complete.  Gives up when
// another thread of this launch aborted, or after the wall-clock limit (then
// it records TP_ERR_TIMEOUT and aborts the launch).  The first 17 tries do not
// read the clock: most waits of the MMA and TMA threads end within them, and
// a %globaltimer read between two tries delays the reaction to the barrier
// (GPT step 0.5% fewer cycles).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Params &p) {
    if (mbar_try_wait(bar, parity)) return true;
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0) {
            if (*reinterpret_cast<volatile unsigned *>(p.abort_word) == p.launch_id) return false;
            if (global_timer_ns() - t0 > p.wait_limit_ns) {
                raise_device_error(p.status, p.abort_word, p.launch_id, TP_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Wait used only while draining on the way out: bounded, ignores the abort word.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return;
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <bool F8>
__device__ __forceinline__ void umma_op(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if (F8)
        umma_f8(d, a, b, idesc, acc);
    else
        umma_bf16(d, a, b, idesc, acc);
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1 at bit 46 and the
// 128-byte swizzle layout (value 2 at bits 61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Dequantisation factor 1 / (scale_a * scale_b) of a product of two FP8
// operands (fp8_scale in device_common.cuh); 1 for bf16.
__device__ __forceinline__ float dequant_factor(const Params &p) {
    if (!p.amax_a) return 1.0f;
    return 1.0f / (fp8_scale(*p.amax_a, p.fmax_a) * fp8_scale(*p.amax_b, p.fmax_b));
}

// ---------------------------------------------------------------------------
// tile schedule: tiles are grouped in bands of `group_m` row tiles; within a
// band the row tile varies fastest.  Column tiles of all problems are laid
// side by side (problem p owns column tiles [p*n_tiles, (p+1)*n_tiles)).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tile_coords(const Params &p, int t, int &pi, int &mt, int &nt) {
    t %= p.tiles_per_split;
    const int n_tot = p.P * p.n_tiles;
    const int per_group = p.group_m * n_tot;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(p.m_tiles - first_m, p.group_m);
    const int r = t - g * per_group;
    mt = first_m + r % gm;
    const int n = r / gm;
    pi = n / p.n_tiles;
    nt = n - pi * p.n_tiles;
}

// K blocks [kb0, kb1) of tile t (its split-K range)
__device__ __forceinline__ void tile_kblocks(const Params &p, int t, int &kb0, int &kb1) {
    kb0 = (t / p.tiles_per_split) * p.kb_split;
    kb1 = min(p.num_kb, kb0 + p.kb_split);
}

// Work item w of the CTA-pair kernel: tile t, its steps [f0, f1) of the
// flattened K loop (step f = segment f / num_kb, K block f % num_kb), and
// for a tail unit its index j within the tile (-1 for a whole tile).
struct Work {
    int t, f0, f1, j;
};
__device__ __forceinline__ Work work_item(const Params &p, int w) {
    Work r;
    if (w < p.tail_first) {
        int kb0, kb1;
        tile_kblocks(p, w, kb0, kb1);  // split-K tiles have S == 1
        r.t = w;
        r.f0 = kb0;
        r.f1 = (p.S - 1) * p.num_kb + kb1;
        r.j = -1;
    } else {
        const int u = w - p.tail_first;
        const int nk = p.S * p.num_kb;
        r.t = p.tail_first + u / p.tail_s;
        r.j = u % p.tail_s;
        r.f0 = static_cast<int>(static_cast<long long>(r.j) * nk / p.tail_s);
        r.f1 = static_cast<int>(static_cast<long long>(r.j + 1) * nk / p.tail_s);
    }
    return r;
}

// Tensor map and local row for buffer row `row`.  A row past the last token
// shard (the second half of a CTA-pair tile beyond M) stays on the last shard's
// map at a row past its end, where the TMA load reads zero fill.
__device__ __forceinline__ void select(const Sel &s, int pi, int seg, int row, int &idx, int &lrow) {
    idx = pi * s.p_stride + seg * s.s_stride;
    lrow = row;
    if (s.rows_split) {
        const int j = min(row / s.rows_split, s.nsplit - 1);
        idx += j;
        lrow = row - j * s.rows_split;
    }
}

// select() carried along a K loop for an MN-major operand split into token
// shards: the map and local row of the current K block, advanced without a
// division per step (shards are multiples of the K block, so a step never
// straddles two of them).
struct SelCursor {
    int idx, lrow, j;
    __device__ __forceinline__ void init(const Sel &s, int pi, int seg, int row) {
        idx = pi * s.p_stride + seg * s.s_stride;
        lrow = row;
        j = 0;
        if (s.rows_split) {
            j = min(row / s.rows_split, s.nsplit - 1);
            idx += j;
            lrow = row - j * s.rows_split;
        }
    }
    __device__ __forceinline__ void advance(const Sel &s, int step) {
        lrow += step;
        if (s.rows_split && lrow >= s.rows_split && j < s.nsplit - 1) {
            lrow -= s.rows_split;
            ++j;
            ++idx;
        }
    }
    // the K block before the current one (a K loop walked backwards)
    __device__ __forceinline__ void retreat(const Sel &s, int step) {
        lrow -= step;
        if (s.rows_split && lrow < 0 && j > 0) {
            lrow += s.rows_split;
            --j;
            --idx;
        }
    }
};

template <typename T>
__device__ __forceinline__ T *row_ptr(const Out &o, int pi, int row) {
    int idx = pi * o.p_stride;
    int lrow = row;
    if (o.rows_split) {
        idx += row / o.rows_split;
        lrow = row % o.rows_split;
    }
    return reinterpret_cast<T *>(o.ptr[idx]) + static_cast<long long>(lrow) * o.ld;
}

__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16 *src, float *dst) {
    const uint4 w = *reinterpret_cast<const uint4 *>(src);
    dst[0] = bf16_lo(w.x); dst[1] = bf16_hi(w.x);
    dst[2] = bf16_lo(w.y); dst[3] = bf16_hi(w.y);
    dst[4] = bf16_lo(w.z); dst[5] = bf16_hi(w.z);
    dst[6] = bf16_lo(w.w); dst[7] = bf16_hi(w.w);
}

__device__ __forceinline__ void store_bf16x8(__nv_bfloat16 *dst, const float *v) {
    uint4 w;
    w.x = pack_bf16x2(v[0], v[1]);
    w.y = pack_bf16x2(v[2], v[3]);
    w.z = pack_bf16x2(v[4], v[5]);
    w.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4 *>(dst) = w;
}

// ---------------------------------------------------------------------------
// epilogues: thread (warp q, lane l) owns output row m0 + 32q + l and walks
// its half of the accumulator (`half` selects 128 of the 256 columns; for
// SwiGLU 64 gate + the matching 64 up columns) in 32-column chunks.  Columns
// come in groups of 8 that are either all inside N or all outside (N % 8 == 0).
// ---------------------------------------------------------------------------
// Activations of the bf16 epilogues use the SFU's tanh.approx.f32 (maximum
// relative error about 2^-11, far below the 2^-8 resolution of the bf16
// results they produce).  sigmoid(x) = (1 + tanh(x/2)) / 2.
//
// The elementwise arithmetic runs on fp32 pairs (FFMA2 / FMUL2 / FADD2,
// sm_100 and later): each component rounds like the scalar operation, and a
// pair issues as one instruction.  The epilogue warps share the SM's issue
// slots with the TMA and MMA warps: on the GPT-size act' dgrad (K = 4096, so
// one epilogue per 64 K steps) halving the activation's instruction count
// took 5% (bf16) and 10% (FP8) off the kernel's time.
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 tanh_fast2(float2 x) { return make_float2(tanh_fast(x.x), tanh_fast(x.y)); }
__device__ __forceinline__ float2 ld2(const float *x) { return make_float2(x[0], x[1]); }
__device__ __forceinline__ void st2(float *x, float2 v) {
    x[0] = v.x;
    x[1] = v.y;
}
// u = sqrt(2/pi) (x + 0.044715 x^3) = x (k0 + k0 k1 x^2);  t = tanh(u)
__device__ __forceinline__ float2 gelu_u2(float2 x, float2 x2) {
    return __fmul2_rn(__ffma2_rn(x2, f2(kGeluK0 * kGeluK1), f2(kGeluK0)), x);
}
// gelu(x) = x/2 (1 + t) = fma(x/2, t, x/2)
__device__ __forceinline__ float2 gelu_tanh2(float2 x) {
    const float2 t = tanh_fast2(gelu_u2(x, __fmul2_rn(x, x)));
    const float2 hx = __fmul2_rn(x, f2(0.5f));
    return __ffma2_rn(hx, t, hx);
}
// gelu'(x) = (1 + t)/2 + x/2 (1 - t^2) u'(x),  u' = k0 (1 + 3 k1 x^2);
// with 1 - t^2 = (1 + t)(1 - t):  gelu' = (1 + t)/2 * (1 + (1 - t) x u')
__device__ __forceinline__ float2 gelu_tanh_grad2(float2 x) {
    const float2 x2 = __fmul2_rn(x, x);
    const float2 t = tanh_fast2(gelu_u2(x, x2));
    const float2 xdu = __fmul2_rn(__ffma2_rn(x2, f2(3.0f * kGeluK0 * kGeluK1), f2(kGeluK0)), x);
    const float2 r = __ffma2_rn(__ffma2_rn(t, f2(-1.0f), f2(1.0f)), xdu, f2(1.0f));
    return __fmul2_rn(__ffma2_rn(t, f2(0.5f), f2(0.5f)), r);
}
__device__ __forceinline__ float2 sigmoid2(float2 x) {
    return __ffma2_rn(tanh_fast2(__fmul2_rn(x, f2(0.5f))), f2(0.5f), f2(0.5f));
}

// the same over N (even) consecutive values
template <int N>
__device__ __forceinline__ void scale_n(float *x, float s) {
#pragma unroll
    for (int j = 0; j < N; j += 2) st2(x + j, __fmul2_rn(ld2(x + j), f2(s)));
}
// v = accumulator * dq (dq = 1 for bf16 operands: no multiply)
template <int N>
__device__ __forceinline__ void acc_to_f32(const uint32_t *r, float dq, float *v) {
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] = __uint_as_float(r[j]);
    if (dq != 1.0f) scale_n<N>(v, dq);
}
template <int N>
__device__ __forceinline__ void add_n(float *x, const float *y) {
#pragma unroll
    for (int j = 0; j < N; j += 2) st2(x + j, __fadd2_rn(ld2(x + j), ld2(y + j)));
}
template <int N>
__device__ __forceinline__ void gelu_tanh_n(float *x) {
#pragma unroll
    for (int j = 0; j < N; j += 2) st2(x + j, gelu_tanh2(ld2(x + j)));
}
// d *= gelu'(x)
template <int N>
__device__ __forceinline__ void mul_gelu_tanh_grad_n(float *d, const float *x) {
#pragma unroll
    for (int j = 0; j < N; j += 2) st2(d + j, __fmul2_rn(ld2(d + j), gelu_tanh_grad2(ld2(x + j))));
}
// G <- silu(G) * U
template <int N>
__device__ __forceinline__ void swiglu_n(float *G, const float *U) {
#pragma unroll
    for (int j = 0; j < N; j += 2) {
        const float2 g = ld2(G + j);
        st2(G + j, __fmul2_rn(__fmul2_rn(g, sigmoid2(g)), ld2(U + j)));
    }
}
// d (the gradient of silu(G) U) <- dG = d U s (1 + G (1 - s)),  dU = d G s
template <int N>
__device__ __forceinline__ void swiglu_grad_n(float *d, float *dU, const float *G, const float *U) {
#pragma unroll
    for (int j = 0; j < N; j += 2) {
        const float2 g = ld2(G + j);
        const float2 sg = sigmoid2(g);
        const float2 ds = __fmul2_rn(ld2(d + j), sg);
        const float2 q = __ffma2_rn(g, __ffma2_rn(sg, f2(-1.0f), f2(1.0f)), f2(1.0f));
        st2(dU + j, __fmul2_rn(ds, g));
        st2(d + j, __fmul2_rn(__fmul2_rn(ds, ld2(U + j)), q));
    }
}

// ---------------------------------------------------------------------------
// epilogue through shared memory: every epilogue warp stages a 32-row x
// 64-byte block (lane = row, 4 x 16 bytes, 64-byte swizzle) in one of its two
// buffers and writes it with one bulk tensor store, which clips rows and
// columns outside the output.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
// element-wise add of the staged block into the tensor (the L2 performs the adds)
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t a, const uint4 &v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

struct Stager {
    uint32_t base;    // this warp's 4 KB
    uint32_t toggle;  // which 2 KB half is next
};

__device__ __forceinline__ void stage_store(Stager &st, const CUtensorMap *map, int x, int y, const uint4 (&w)[4],
                                            int lane, bool add = false) {
    const uint32_t buf = st.base + st.toggle * 2048u;
    st.toggle ^= 1u;
    if (lane == 0) bulk_wait_read<1>();  // the store that last used this half has read it
    __syncwarp();
    const uint32_t rowa = buf + static_cast<uint32_t>(lane) * 64u;
    const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
    for (int j = 0; j < 4; ++j) st_shared_v4(rowa + ((static_cast<uint32_t>(j) ^ sw) << 4), w[j]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (add)
            tma_reduce_add_2d(map, buf, x, y);
        else
            tma_store_2d(map, buf, x, y);
        bulk_commit();
    }
}

// 32 FP8 codes of one row (32 bytes) staged as a 32-row x 32-byte block in
// one of the warp's two 2 KB halves and written with one bulk tensor store
__device__ __forceinline__ void stage_store_q(Stager &st, const CUtensorMap *map, int x, int y,
                                              const uint4 (&wq)[2], int lane) {
    const uint32_t buf = st.base + st.toggle * 2048u;
    st.toggle ^= 1u;
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    const uint32_t rowa = buf + static_cast<uint32_t>(lane) * 32u;
    st_shared_v4(rowa, wq[0]);
    st_shared_v4(rowa + 16u, wq[1]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(map, buf, x, y);
        bulk_commit();
    }
}

// FP8 codes of 32 bf16 values (packed in w) at scale s: fp32 product, then
// round-to-nearest-even with saturation, as the quantiser does
__device__ __forceinline__ void fp8_codes32(const uint4 (&w)[4], float s, int fmt, uint4 (&wq)[2]) {
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t ws[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 a = __fmul2_rn(make_float2(bf16_lo(ws[k]), bf16_hi(ws[k])), f2(s));
            const uint32_t v = fmt == FP8_E5M2 ? __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E5M2)
                                               : __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
            lo |= v << (16 * k);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 a = __fmul2_rn(make_float2(bf16_lo(ws[2 + k]), bf16_hi(ws[2 + k])), f2(s));
            const uint32_t v = fmt == FP8_E5M2 ? __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E5M2)
                                               : __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
            hi |= v << (16 * k);
        }
        c[2 * j] = lo;
        c[2 * j + 1] = hi;
    }
    wq[0] = make_uint4(c[0], c[1], c[2], c[3]);
    wq[1] = make_uint4(c[4], c[5], c[6], c[7]);
}

__device__ __forceinline__ void pack_bf16x32(const float *v, uint4 (&w)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        w[j].x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
        w[j].y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
        w[j].z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
        w[j].w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
    }
}

__device__ __forceinline__ void pack_f32x16(const float *v, uint4 (&w)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w[j] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                          __float_as_uint(v[4 * j + 3]));
}

// output map index and local row of the 32-row block starting at row0
__device__ __forceinline__ void out_index(const Out &o, int pi, int row0, int &idx, int &lrow) {
    idx = pi * o.p_stride;
    lrow = row0;
    if (o.rows_split) {
        const int j = min(row0 / o.rows_split, o.nsplit - 1);
        idx += j;
        lrow = row0 - j * o.rows_split;
    }
}

// 8 bf16 from global, or zeros when the group lies outside [0, limit)
__device__ __forceinline__ void load_bf16x8_guarded(const __nv_bfloat16 *src, bool ok, float *dst) {
    if (ok) {
        load_bf16x8(src, dst);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = 0.0f;
    }
}

// Column sums of a 32 x 32 block held one row per lane (v[j] = column j of
// this lane's row): a recursive-halving exchange leaves the sum of column
// `lane` in v[0] after 31 shuffles.
__device__ __forceinline__ float warp_column_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int o = 16; o >= 2; o >>= 1) {  // adds on fp32 pairs
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < o; j += 2) {
            const float2 lo = ld2(v + j), hi = ld2(v + j + o);
            const float2 send = upper ? lo : hi;
            const float2 keep = upper ? hi : lo;
            const float2 got = make_float2(__shfl_xor_sync(0xffffffffu, send.x, o),
                                           __shfl_xor_sync(0xffffffffu, send.y, o));
            st2(v + j, __fadd2_rn(keep, got));
        }
    }
    const bool upper = (lane & 1) != 0;
    const float send = upper ? v[0] : v[1];
    const float keep = upper ? v[1] : v[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Column sums (bias-gradient partials) of one 32-column block of fp32 values,
// one row per lane: rows past M and columns past N contribute nothing.
__device__ __forceinline__ void col_partial_sums(const Params &p, int pi, int row0, int col0, const float *vals,
                                                 bool row_ok, int lane, int part_off = 0) {
    if (!p.col_partials) return;
    float v[32];
    if (row_ok && col0 + 32 <= p.N) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = vals[j];
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (row_ok && col0 + j < p.N) ? vals[j] : 0.0f;
    }
    const float sum = warp_column_sum32(v, lane);
    if (col0 + lane < p.N)
        p.col_partials[(static_cast<long long>(pi) * ((p.M + 31) / 32) + row0 / 32) * p.partial_ld + part_off + col0 +
                       lane] = sum;
}

// Running max |x| over the bf16 outputs (the FP8 scale of A or dPre), taken on
// the packed pairs the epilogue stores: max.xorsign.abs keeps max(|a|, |b|) in
// each half (its sign bits are ignored).  Max |bf16(v)| is the same as the
// rounded max |v| (rounding is monotone).  Rows past M and column pairs past N
// contribute nothing (N % 8 == 0, so a pair is inside or outside).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ void amax_bf16x32(const Params &p, const uint4 (&w)[4], bool row_ok, int col0,
                                             uint32_t &amx) {
    if (!p.amax_out || !row_ok) return;
    const bool full = col0 + 32 <= p.N;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t q[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (full || col0 + 8 * k + 2 * i < p.N) amx = absmax_bf16x2(amx, q[i]);
    }
}

__device__ __forceinline__ void flush_amax(const Params &p, uint32_t amx2) {
    if (!p.amax_out) return;
    float amx = fmaxf(fabsf(bf16_lo(amx2)), fabsf(bf16_hi(amx2)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amx = fmaxf(amx, __shfl_xor_sync(0xffffffffu, amx, o));
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned *>(p.amax_out), __float_as_uint(amx));
}

// Tail-split slices: one unit's raw fp32 accumulator (256 x BN) is stored as
// 16 warp slices of 32 rows x 128 columns (16 KB each, slice = CTA rank * 8 +
// lane quarter * 2 + column half).  Inside a slice, float4 k (0..7) of chunk
// c (0..3) of lane l sits at float4 index (c * 8 + k) * 32 + l, so that every
// warp-wide access covers 512 contiguous bytes.  Accesses go through L2.
constexpr size_t TAIL_SLICE_FLOATS = 32 * 128;
constexpr size_t TAIL_UNIT_FLOATS = 16 * TAIL_SLICE_FLOATS;

__device__ __forceinline__ void tail_store32(float *slice, int c, int lane, const uint32_t (&r)[32]) {
    float4 *d4 = reinterpret_cast<float4 *>(slice) + c * 256 + lane;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        __stcg(d4 + 32 * k, make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                        __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3])));
}

// chunk c of the tile's accumulator as the sum of its units' slices, added
// in unit order
__device__ __forceinline__ void tail_sum32(const float *slice, int c, int lane, int units, uint32_t (&r)[32]) {
    float acc[32];
    const float *src = slice + (c * 256 + lane) * 4;
    {
        const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 x = __ldcg(s4 + 32 * k);
            acc[4 * k] = x.x;
            acc[4 * k + 1] = x.y;
            acc[4 * k + 2] = x.z;
            acc[4 * k + 3] = x.w;
        }
    }
    for (int i = 1; i < units; ++i) {
        const float4 *s4 = reinterpret_cast<const float4 *>(src + i * TAIL_UNIT_FLOATS);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 x = __ldcg(s4 + 32 * k);
            acc[4 * k] += x.x;
            acc[4 * k + 1] += x.y;
            acc[4 * k + 2] += x.z;
            acc[4 * k + 3] += x.w;
        }
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(acc[k]);
}

// Bulk-store epilogue of one warp's 32 rows x 128 columns.  The accumulator
// comes from TMEM at taddr, or, for a tail-split tile (ws_slice non-null),
// from the sum of the ws_units slices from ws_slice (this warp's in unit 0).
template <int EPI>
__device__ __forceinline__ void run_epilogue_tma(const Params &p, int pi, int row, int nt, uint32_t taddr, int half,
                                                 float dq, Stager &stg, int lane, int t,
                                                 const float *ws_slice = nullptr, int ws_units = 0) {
    const int row0 = row - lane;             // first row of this warp's block
    const bool block_ok = row0 < p.M;        // warp-uniform
    const bool row_ok = row < p.M;
    int oi, oy, oi2 = 0, oy2 = 0;
    out_index(p.out, pi, row0, oi, oy);
    if (EPI == EPI_F32 && p.split_rows) {  // split-K partial of split t / tiles_per_split
        oi = 0;
        oy = ((t / p.tiles_per_split) * p.P + pi) * p.split_rows + row0;
    }
    if (p.has_out2) out_index(p.out2, pi, row0, oi2, oy2);
    const __nv_bfloat16 *bias =
        p.has_bias ? reinterpret_cast<const __nv_bfloat16 *>(p.bias[pi * p.bias_p_stride]) : nullptr;
    uint32_t amx = 0;  // max |bf16 output| of this thread, as a bf16 pair (FP8 scale of A / dPre)
    uint4 w[4];
    if (EPI == EPI_COL && p.act == TP_ACT_SWIGLU) {
        // accumulator columns [0,128) = gate units, [128,256) = up units (N % 32 == 0 here)
        const int ubase = nt * (BN / 2);
#pragma unroll 1
        for (int c = 2 * half; c < 2 * half + 2; ++c) {
            uint32_t rg[32], ru[32];
            __syncwarp();
            tmem_ld32(taddr + c * 32, rg);
            tmem_ld32(taddr + BN / 2 + c * 32, ru);
            tmem_ld_wait();
            const int u0 = ubase + c * 32;
            if (!block_ok || u0 >= p.N) continue;
            float G[32], U[32];
            acc_to_f32<32>(rg, dq, G);
            acc_to_f32<32>(ru, dq, U);
            if (bias) {
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    float bg[8], bu[8];
                    load_bf16x8(bias + u0 + 8 * g8, bg);
                    load_bf16x8(bias + p.N + u0 + 8 * g8, bu);
                    add_n<8>(G + 8 * g8, bg);
                    add_n<8>(U + 8 * g8, bu);
                }
            }
            if (p.has_out2) {
                pack_bf16x32(G, w);
                stage_store(stg, &p.mapO2[oi2], u0, oy2, w, lane);
                pack_bf16x32(U, w);
                stage_store(stg, &p.mapO2[oi2], p.N + u0, oy2, w, lane);
            }
            swiglu_n<32>(G, U);
            pack_bf16x32(G, w);
            amax_bf16x32(p, w, row_ok, u0, amx);
            stage_store(stg, &p.mapO[oi], u0, oy, w, lane);
        }
        flush_amax(p, amx);
        return;
    }
    const int n0 = nt * BN;
#pragma unroll 1
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
        uint32_t r[32];
        __syncwarp();
        const int col0 = n0 + c * 32;
        if (ws_slice) {
            if (!block_ok || col0 >= p.N) continue;
            tail_sum32(ws_slice, c - 4 * half, lane, ws_units, r);
        } else {
            tmem_ld32(taddr + c * 32, r);
            tmem_ld_wait();
            if (!block_ok || col0 >= p.N) continue;
        }
        float v[32];
        acc_to_f32<32>(r, dq, v);
        if (EPI == EPI_F32) {  // with accumulate: dW += through bulk reduce-add stores
            const bool add = p.accumulate != 0;
            pack_f32x16(v, w);
            stage_store(stg, &p.mapO[oi], col0, oy, w, lane, add);
            if (col0 + 16 < p.N) {
                pack_f32x16(v + 16, w);
                stage_store(stg, &p.mapO[oi], col0 + 16, oy, w, lane, add);
            }
            continue;
        }
        if (EPI == EPI_COL || EPI == EPI_PLAIN) {
            if (bias) {
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    float b[8];
                    load_bf16x8_guarded(bias + col0 + 8 * g8, col0 + 8 * g8 < p.N, b);
                    add_n<8>(v + 8 * g8, b);
                }
            }
        }
        if (EPI == EPI_COL) {
            if (p.has_out2) {
                pack_bf16x32(v, w);
                stage_store(stg, &p.mapO2[oi2], col0, oy2, w, lane);
            }
            if (p.act == TP_ACT_GELU_TANH) gelu_tanh_n<32>(v);
            pack_bf16x32(v, w);
            amax_bf16x32(p, w, row_ok, col0, amx);
            stage_store(stg, &p.mapO[oi], col0, oy, w, lane);
            if (p.q_out) {
                uint4 wq[2];
                fp8_codes32(w, fp8_scale(*p.q_scale_amax, p.q_fmt == FP8_E5M2 ? 57344.0f : 448.0f), p.q_fmt, wq);
                stage_store_q(stg, &p.mapQ[oi], col0, oy, wq, lane);
            }
        } else if (EPI == EPI_PLAIN) {
            if (p.drop.on) dropout32(p.drop, row, col0, row_ok, v);
            if (p.has_aux) {
                const __nv_bfloat16 *res = row_ptr<const __nv_bfloat16>(p.aux, pi, row_ok ? row : row0);
                float r32[32];
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    load_bf16x8_guarded(res + col0 + 8 * g8, row_ok && col0 + 8 * g8 < p.N, r32 + 8 * g8);
                    add_n<8>(v + 8 * g8, r32 + 8 * g8);
                }
                // column sums of the residual per 32-row block (the row layer's
                // bias gradient, sum_m dY, when the residual is dY)
                col_partial_sums(p, pi, row0, col0, r32, row_ok, lane);
            }
            pack_bf16x32(v, w);
            stage_store(stg, &p.mapO[oi], col0, oy, w, lane);
        } else if (EPI == EPI_DACT) {
            const __nv_bfloat16 *pre = row_ptr<const __nv_bfloat16>(p.aux, pi, row_ok ? row : row0);
            if (p.act == TP_ACT_SWIGLU) {
                float dU[32];
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    float G[8], U[8];
                    const bool ok = row_ok && col0 + 8 * g8 < p.N;
                    load_bf16x8_guarded(pre + col0 + 8 * g8, ok, G);
                    load_bf16x8_guarded(pre + p.N + col0 + 8 * g8, ok, U);
                    swiglu_grad_n<8>(v + 8 * g8, dU + 8 * g8, G, U);
                }
                // dG feeds db1 columns [0, N), dU columns [N, 2N)
                col_partial_sums(p, pi, row0, col0, v, row_ok, lane);
                col_partial_sums(p, pi, row0, col0, dU, row_ok, lane, p.N);
                pack_bf16x32(v, w);
                amax_bf16x32(p, w, row_ok, col0, amx);
                stage_store(stg, &p.mapO[oi], col0, oy, w, lane);
                pack_bf16x32(dU, w);
                amax_bf16x32(p, w, row_ok, col0, amx);
                stage_store(stg, &p.mapO[oi], p.N + col0, oy, w, lane);
            } else {
                if (p.act == TP_ACT_GELU_TANH) {
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8) {
                        float x[8];
                        load_bf16x8_guarded(pre + col0 + 8 * g8, row_ok && col0 + 8 * g8 < p.N, x);
                        mul_gelu_tanh_grad_n<8>(v + 8 * g8, x);
                    }
                }
                col_partial_sums(p, pi, row0, col0, v, row_ok, lane);
                pack_bf16x32(v, w);
                amax_bf16x32(p, w, row_ok, col0, amx);
                if (!p.q_only) stage_store(stg, &p.mapO[oi], col0, oy, w, lane);
                if (p.q_out) {
                    uint4 wq[2];
                    fp8_codes32(w, fp8_scale(*p.q_scale_amax, p.q_fmt == FP8_E5M2 ? 57344.0f : 448.0f), p.q_fmt,
                                wq);
                    stage_store_q(stg, &p.mapQ[oi], col0, oy, wq, lane);
                }
            }
        }
    }
    flush_amax(p, amx);
}

template <int EPI>
__device__ __forceinline__ void run_epilogue(const Params &p, int pi, int row, int nt, uint32_t taddr, int half,
                                             float dq) {
    const bool row_ok = row < p.M;
    if (EPI == EPI_COL && p.act == TP_ACT_SWIGLU) {
        // accumulator columns [0,128) = gate units, [128,256) = up units
        const int ubase = nt * (BN / 2);
        const __nv_bfloat16 *bias =
            p.has_bias ? reinterpret_cast<const __nv_bfloat16 *>(p.bias[pi * p.bias_p_stride]) : nullptr;
#pragma unroll 1
        for (int c = 2 * half; c < 2 * half + 2; ++c) {
            uint32_t rg[32], ru[32];
            __syncwarp();
            tmem_ld32(taddr + c * 32, rg);
            tmem_ld32(taddr + BN / 2 + c * 32, ru);
            tmem_ld_wait();
            const int u0 = ubase + c * 32;
            if (!row_ok) continue;
            __nv_bfloat16 *pre = p.has_out2 ? row_ptr<__nv_bfloat16>(p.out2, pi, row) : nullptr;
            __nv_bfloat16 *act = row_ptr<__nv_bfloat16>(p.out, pi, row);
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int u = u0 + g8 * 8;
                if (u >= p.N) break;
                float G[8], U[8];
                acc_to_f32<8>(rg + g8 * 8, dq, G);
                acc_to_f32<8>(ru + g8 * 8, dq, U);
                if (bias) {
                    float bg[8], bu[8];
                    load_bf16x8(bias + u, bg);
                    load_bf16x8(bias + p.N + u, bu);
                    add_n<8>(G, bg);
                    add_n<8>(U, bu);
                }
                if (pre) {
                    store_bf16x8(pre + u, G);
                    store_bf16x8(pre + p.N + u, U);
                }
                swiglu_n<8>(G, U);
                store_bf16x8(act + u, G);
            }
        }
        return;
    }
    const int n0 = nt * BN;
#pragma unroll 1
    for (int c = 4 * half; c < 4 * half + 4; ++c) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + c * 32, r);
        tmem_ld_wait();
        const int col0 = n0 + c * 32;
        if (!row_ok || col0 >= p.N) continue;
        float v[32];
        acc_to_f32<32>(r, dq, v);
        if (EPI == EPI_F32) {
            float *o = row_ptr<float>(p.out, pi, row) + col0;
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
                if (col0 + g4 * 4 >= p.N) break;
                float4 w = make_float4(v[g4 * 4], v[g4 * 4 + 1], v[g4 * 4 + 2], v[g4 * 4 + 3]);
                if (p.accumulate) {
                    const float4 old = *reinterpret_cast<const float4 *>(o + g4 * 4);
                    w.x += old.x; w.y += old.y; w.z += old.z; w.w += old.w;
                }
                *reinterpret_cast<float4 *>(o + g4 * 4) = w;
            }
            continue;
        }
        if (EPI == EPI_COL) {
            const __nv_bfloat16 *bias =
                p.has_bias ? reinterpret_cast<const __nv_bfloat16 *>(p.bias[pi * p.bias_p_stride]) : nullptr;
            __nv_bfloat16 *pre = p.has_out2 ? row_ptr<__nv_bfloat16>(p.out2, pi, row) : nullptr;
            __nv_bfloat16 *act = row_ptr<__nv_bfloat16>(p.out, pi, row);
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int col = col0 + g8 * 8;
                if (col >= p.N) break;
                float *x = v + g8 * 8;
                if (bias) {
                    float b[8];
                    load_bf16x8(bias + col, b);
                    add_n<8>(x, b);
                }
                if (pre) store_bf16x8(pre + col, x);
                if (p.act == TP_ACT_GELU_TANH) gelu_tanh_n<8>(x);
                store_bf16x8(act + col, x);
            }
        } else if (EPI == EPI_PLAIN) {
            const __nv_bfloat16 *bias =
                p.has_bias ? reinterpret_cast<const __nv_bfloat16 *>(p.bias[pi * p.bias_p_stride]) : nullptr;
            const __nv_bfloat16 *res = p.has_aux ? row_ptr<const __nv_bfloat16>(p.aux, pi, row) : nullptr;
            __nv_bfloat16 *o = row_ptr<__nv_bfloat16>(p.out, pi, row);
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int col = col0 + g8 * 8;
                if (col >= p.N) break;
                float *x = v + g8 * 8;
                if (bias) {
                    float b[8];
                    load_bf16x8(bias + col, b);
                    add_n<8>(x, b);
                }
                if (p.drop.on) {
                    const long long e0 = static_cast<long long>(row) * p.drop.ld + col;
                    dropout4(p.drop, e0, x);
                    dropout4(p.drop, e0 + 4, x + 4);
                }
                if (res) {
                    float rr[8];
                    load_bf16x8(res + col, rr);
                    add_n<8>(x, rr);
                }
                store_bf16x8(o + col, x);
            }
        } else if (EPI == EPI_DACT) {
            const __nv_bfloat16 *pre = row_ptr<const __nv_bfloat16>(p.aux, pi, row);
            __nv_bfloat16 *o = row_ptr<__nv_bfloat16>(p.out, pi, row);
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const int u = col0 + g8 * 8;
                if (u >= p.N) break;
                float *d = v + g8 * 8;
                if (p.act == TP_ACT_GELU_TANH) {
                    float x[8];
                    load_bf16x8(pre + u, x);
                    mul_gelu_tanh_grad_n<8>(d, x);
                    store_bf16x8(o + u, d);
                } else if (p.act == TP_ACT_SWIGLU) {
                    float G[8], U[8], dU[8];
                    load_bf16x8(pre + u, G);
                    load_bf16x8(pre + p.N + u, U);
                    swiglu_grad_n<8>(d, dU, G, U);
                    store_bf16x8(o + u, d);
                    store_bf16x8(o + p.N + u, dU);
                } else {
                    store_bf16x8(o + u, d);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int EPI, bool A_MN, bool B_MN, bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_kernel(const __grid_constant__ Params p) {
    ClockMark clk_mark;
    clk_mark.start(p.clk);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * STAGES;
    const uint32_t tfull0 = empty0 + 8 * STAGES;
    const uint32_t tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    const uint32_t smem_base = smem_u32(smem);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    using E = Elem<F8>;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull0 + 8 * i, 1);
            mbar_init(tempty0 + 8 * i, 32 * EPI_WARPS);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_par = 0;  // per stage: armed phase not yet known consumed
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
                int pi, mt, nt;
                tile_coords(p, t, pi, mt, nt);
                const int m0 = mt * BM;
                const int n0 = p.b_dual_off ? nt * (BN / 2) : nt * BN;
                int kb0, kb1;
                tile_kblocks(p, t, kb0, kb1);
                for (int s = 0; ok && s < p.S; ++s) {
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = full0 + 8 * stage;
                        mbar_arrive_expect_tx(fb, STAGE_BYTES);
                        armed |= 1u << stage;
                        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                        const uint32_t sa = smem_base + stage * STAGE_BYTES;
                        const uint32_t sb = sa + A_BYTES;
                        const int k0 = kb * E::BKE;
                        int idx, lrow;
                        if (!A_MN) {
                            select(p.selA, pi, s, m0, idx, lrow);
                            tma_load_2d(sa, &p.mapA[idx], fb, k0, lrow);
                        } else {
                            select(p.selA, pi, s, k0, idx, lrow);
#pragma unroll
                            for (int j = 0; j < BM / E::MNB; ++j)
                                tma_load_2d(sa + j * E::MNB_BYTES, &p.mapA[idx], fb, m0 + j * E::MNB, lrow);
                        }
                        if (!B_MN) {
                            select(p.selB, pi, s, n0, idx, lrow);
                            if (p.b_dual_off) {
                                tma_load_2d(sb, &p.mapB[idx], fb, k0, lrow);
                                tma_load_2d(sb + B_BYTES / 2, &p.mapB[idx], fb, k0, lrow + p.b_dual_off);
                            } else {
                                tma_load_2d(sb, &p.mapB[idx], fb, k0, lrow);
                            }
                        } else {
                            select(p.selB, pi, s, k0, idx, lrow);
#pragma unroll
                            for (int j = 0; j < BN / E::MNB; ++j)
                                tma_load_2d(sb + j * E::MNB_BYTES, &p.mapB[idx], fb, n0 + j * E::MNB, lrow);
                        }
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // Make sure no bulk copy is still landing in shared memory when the
            // CTA exits (only matters on the abort path).
            for (int i = 0; i < STAGES; ++i)
                if (armed & (1u << i)) mbar_wait_drain(full0 + 8 * i, (armed_par >> i) & 1u, p.wait_limit_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            const uint32_t idesc = p.idesc;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                if (!mbar_wait(tempty0 + 8 * acc, acc_par ^ 1u, p)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                uint32_t accumulate = 0;
                int kb0, kb1;
                tile_kblocks(p, t, kb0, kb1);
                for (int s = 0; ok && s < p.S; ++s) {
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(full0 + 8 * stage, phase, p)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_base + stage * STAGE_BYTES;
                        const uint32_t sb = sa + A_BYTES;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // K-major: advance one MMA's K (32 B) inside the swizzle row.
                            // MN-major: advance one MMA's K rows (2 or 4 swizzle atoms of 1 KB).
                            const uint64_t ad = A_MN ? smem_desc(sa + kk * E::KADV_MN, E::MNB_BYTES, 1024)
                                                     : smem_desc(sa + kk * 32, 16, 1024);
                            const uint64_t bd = B_MN ? smem_desc(sb + kk * E::KADV_MN, E::MNB_BYTES, 1024)
                                                     : smem_desc(sb + kk * 32, 16, 1024);
                            umma_op<F8>(d, ad, bd, idesc, accumulate);
                            accumulate = 1;
                        }
                        umma_commit(empty0 + 8 * stage);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                umma_commit(tfull0 + 8 * acc);
            }
            // all issued MMAs complete before TMEM is released
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..9) ----------------
        const int q = warp & 3;             // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;   // which 128 accumulator columns it drains
        const float dq = dequant_factor(p);
        Stager stg{smem_base + STAGES * STAGE_BYTES + BAR_BYTES + (warp - 2) * EPI_STAGE_BYTES, 0u};
        int it = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            const bool ok = mbar_wait(tfull0 + 8 * acc, acc_par, p);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            int pi, mt, nt;
            tile_coords(p, t, pi, mt, nt);
            const int row = mt * BM + q * 32 + lane;
            const uint32_t taddr = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
            if (p.out_tma)
                run_epilogue_tma<EPI>(p, pi, row, nt, taddr, half, dq, stg, lane, t);
            else
                run_epilogue<EPI>(p, pi, row, nt, taddr, half, dq);
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * acc);
        }
        if (lane == 0) bulk_wait<0>();  // bulk stores done before the CTA leaves
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
    clk_mark.stop(p.clk);
}

// ---------------------------------------------------------------------------
// CTA-pair variant: a cluster of two CTAs on two SMs computes one 256 x 256
// tile with tcgen05.mma.cta_group::2 (M = 256).  CTA r of the pair loads rows
// [128r, 128r + 128) of the A tile and rows [128r, 128r + 128) of the B tile
// (for SwiGLU: CTA 0 the gate rows, CTA 1 the up rows) into its own shared
// memory; the MMA, issued by CTA 0, reads both CTAs' halves and leaves rows
// [128r, 128r + 128) of the accumulator in CTA r's TMEM.  Each SM thus reads
// half of the B tile it would read alone, and a stage is 32 KB, so the ring
// is 6 stages deep (5 for the act' dgrad, below).
//
// Barriers: every load of both CTAs completes on CTA 0's full[s] (CTA 0 arms
// it for both); the MMA commit multicasts to empty[s] and tfull[a] of both
// CTAs; both CTAs' epilogue threads arrive on CTA 0's tempty[a].
// ---------------------------------------------------------------------------
constexpr int P_STAGES = 6;
constexpr int P_A_BYTES = 128 * ROW_BYTES;  // 16 KB: this CTA's 128 rows of A
constexpr int P_B_BYTES = 128 * ROW_BYTES;  // 16 KB: this CTA's 128 rows of B
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
// Ring depth, in 32 KB units: six everywhere (three stages of two K blocks in
// bf16) except the FP8 act' dgrad, which reads pre through L1 (the shared
// memory a block does not claim) and runs five stages of one K block (L1
// about 60 KB instead of 28 KB: 5% fewer SM cycles, 1% in time under the
// power cap).  The bf16 act' dgrad gained the same way with one K block per
// stage, but with two it is 3% faster still at six units, level with the
// column forward; two stages of two K blocks (more L1) made it 27% slower.
template <int EPI, bool F8>
constexpr int pair_stages() {
    return (EPI == EPI_DACT && F8) ? 5 : P_STAGES;
}
// K blocks per stage (see tc_gemm_pair_kernel): two for bf16
template <int EPI, bool F8>
constexpr int pair_kb2() {
    return F8 ? 1 : 2;
}
constexpr int pair_smem_bytes(int stages) { return stages * P_STAGE_BYTES + 1024 + BAR_BYTES + EPI_SMEM; }
// dynamic shared memory of a pair-kernel instance: the ring as the kernel
// lays it out (whole stages of KB2 K blocks) and the rest
template <int EPI, bool F8>
constexpr int pair_smem_total() {
    return pair_smem_bytes(pair_stages<EPI, F8>() / pair_kb2<EPI, F8>() * pair_kb2<EPI, F8>());
}
constexpr int P_SMEM_BYTES = pair_smem_bytes(P_STAGES);
constexpr int P_TILE_M = 256;
static_assert(TAIL_UNIT_FLOATS == static_cast<size_t>(P_TILE_M) * BN, "tail slices hold one pair tile");
static_assert(EPI_WARPS == 8, "16 tail slices: 2 CTAs x 4 lane quarters x 2 column halves");

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t map_to_cta(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream is still
// running; griddepcontrol.wait returns once that kernel has completed and its
// writes are visible (at once for a launch without the attribute), so
// nothing before it may touch global memory.  launch_dependents lets the
// next such kernel start its CTAs on the SMs this grid leaves free.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster, int c0,
                                                 int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster, int c0,
                                                 int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <bool F8>
__device__ __forceinline__ void umma_op_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if (F8)
        umma_f8_pair(d, a, b, idesc, acc);
    else
        umma_bf16_pair(d, a, b, idesc, acc);
}

// arrive on the barrier at this shared-memory offset in both CTAs of the pair
// once all previously issued MMAs of this thread have completed
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// TS: the MN-major operands are split into token shards (the weight
// gradients under sequence parallelism); their maps follow a SelCursor.
template <int EPI, bool A_MN, bool B_MN, bool F8, bool TS = false>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_pair_kernel(const __grid_constant__ Params p) {
    ClockMark clk_mark;
    clk_mark.start(p.clk);
    using E = Elem<F8>;
    // K blocks per stage: two for bf16, in half as many stages of twice the
    // size (the same shared memory).  An MN-major operand comes as
    // one 3D box of {64, 128 K rows, 2 atoms}, a K-major one as one 3D box
    // {64, 128 rows, 2 K blocks} (or two 2D boxes when its K extent is not a
    // multiple of 64): half the loads and barrier operations per K for the
    // producer thread, and eight MMAs per full barrier instead of four.
    constexpr int KB2 = pair_kb2<EPI, F8>();
    constexpr int NST = pair_stages<EPI, F8>() / KB2;
    constexpr int STG = P_STAGE_BYTES * KB2;  // bytes of one stage in this CTA
    constexpr int BKS = E::BKE * KB2;         // K elements of one stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NST * STG);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * NST + 5);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * NST;
    const uint32_t tfull0 = empty0 + 8 * NST;
    const uint32_t tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    const uint32_t smem_base = smem_u32(smem);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();  // 0 = leader (issues the MMAs), 1 = peer
    const int pair_id = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull0 + 8 * i, 1);
            mbar_init(tempty0 + 8 * i, 2 * 32 * EPI_WARPS);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // set-up above overlaps the previous kernel; operands and outputs below
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            // One thread issues both operands' loads of every stage.  In the
            // weight gradients (both operands MN-major) its instruction path
            // per K step is what the MMAs wait on, so everything that does not
            // change within a K segment is computed once per segment.
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_par = 0;
            bool ok = true;
            int it = 0;
            const uint32_t full0_c = map_to_cta(full0, 0);  // CTA 0's full barriers, cluster window
            for (int w = pair_id; ok && w < p.total_work; w += npairs, ++it) {
                const Work wk = work_item(p, w);
                int pi, mt, nt;
                tile_coords(p, wk.t, pi, mt, nt);
                const int m0 = mt * P_TILE_M + 128 * rank;
                // B rows of this CTA: its half of the 256 tile columns, or for
                // SwiGLU the gate (rank 0) / up (rank 1) rows of 128 units
                const int n0 = p.b_dual_off ? nt * (BN / 2) + (rank ? p.b_dual_off : 0) : nt * BN + 128 * rank;
                // odd rounds walk a whole tile's K steps from the last one down
                const bool rev = p.k_reverse && wk.j < 0 && (it & 1);
                const int dkb = rev ? -1 : 1;
                const int f_first = rev ? wk.f1 - 1 : wk.f0;
                int s = f_first / p.num_kb, kb = f_first - s * p.num_kb;
                // Maps and rows for the current K segment.  K-major operands
                // select by the tile row (under sequence parallelism a division
                // per K step cost the SP GEMMs 6-9%).  MN-major operands outside
                // the token-sharded instance are never split into token shards:
                // their map depends on the problem and the segment only and
                // their row is the K offset; in that instance a cursor follows
                // the token shards along the K loop.
                const CUtensorMap *ma = nullptr, *mb = nullptr;
                int ra = 0, rb = 0;
                auto segment_maps = [&]() {
                    int idx = 0;
                    if (!A_MN) {
                        select(p.selA, pi, s, m0, idx, ra);
                        ma = &p.mapA[idx];
                    } else if (!TS) {
                        ma = &p.mapA[pi * p.selA.p_stride + s * p.selA.s_stride];
                    }
                    if (!B_MN) {
                        select(p.selB, pi, s, n0, idx, rb);
                        mb = &p.mapB[idx];
                    } else if (!TS) {
                        mb = &p.mapB[pi * p.selB.p_stride + s * p.selB.s_stride];
                    }
                };
                segment_maps();
                SelCursor ca, cb;
                if constexpr (TS) {
                    if (A_MN) ca.init(p.selA, pi, s, kb * BKS);
                    if (B_MN) cb.init(p.selB, pi, s, kb * BKS);
                }
                const int a_grp = m0 / 64, b_grp = n0 / 64;  // 3D boxes: 64-wide group of the MN origin
                for (int f = wk.f0; f < wk.f1; ++f) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0_c + 8 * stage;
                    if (rank == 0) {
                        mbar_arrive_expect_tx(full0 + 8 * stage, 2 * STG);
                        armed |= 1u << stage;
                        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    }
                    const uint32_t sa = smem_base + stage * STG;
                    const uint32_t sb = sa + P_A_BYTES * KB2;
                    const int k0 = kb * BKS;
                    if (!A_MN) {
                        if (KB2 == 1) {
                            tma_load_2d_pair(sa, ma, fb, k0, ra);
                        } else if (p.a3d) {
                            tma_load_3d_pair(sa, ma, fb, 0, ra, k0 / E::BKE);
                        } else {
                            tma_load_2d_pair(sa, ma, fb, k0, ra);
                            tma_load_2d_pair(sa + P_A_BYTES, ma, fb, k0 + E::BKE, ra);
                        }
                    } else {
                        const CUtensorMap *m = ma;
                        int lrow = k0;
                        if constexpr (TS) {
                            m = &p.mapA[ca.idx];
                            lrow = ca.lrow;
                        }
                        if (!F8 && p.a3d) {
                            tma_load_3d_pair(sa, m, fb, 0, lrow, a_grp);
                        } else {
#pragma unroll
                            for (int j = 0; j < 128 / E::MNB; ++j)
                                tma_load_2d_pair(sa + j * E::MNB_BYTES * KB2, m, fb, m0 + j * E::MNB, lrow);
                        }
                    }
                    if (!B_MN) {
                        if (KB2 == 1) {
                            tma_load_2d_pair(sb, mb, fb, k0, rb);
                        } else if (p.b3d) {
                            tma_load_3d_pair(sb, mb, fb, 0, rb, k0 / E::BKE);
                        } else {
                            tma_load_2d_pair(sb, mb, fb, k0, rb);
                            tma_load_2d_pair(sb + P_B_BYTES, mb, fb, k0 + E::BKE, rb);
                        }
                    } else {
                        const CUtensorMap *m = mb;
                        int lrow = k0;
                        if constexpr (TS) {
                            m = &p.mapB[cb.idx];
                            lrow = cb.lrow;
                        }
                        if (!F8 && p.b3d) {
                            tma_load_3d_pair(sb, m, fb, 0, lrow, b_grp);
                        } else {
#pragma unroll
                            for (int j = 0; j < 128 / E::MNB; ++j)
                                tma_load_2d_pair(sb + j * E::MNB_BYTES * KB2, m, fb, n0 + j * E::MNB, lrow);
                        }
                    }
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    kb += dkb;
                    if (kb == p.num_kb || kb < 0) {  // next (or, walking backwards, previous) K segment
                        s += dkb;
                        kb = rev ? p.num_kb - 1 : 0;
                        if (s >= 0 && s < p.S) {
                            segment_maps();
                            if constexpr (TS) {
                                if (A_MN) ca.init(p.selA, pi, s, kb * BKS);
                                if (B_MN) cb.init(p.selB, pi, s, kb * BKS);
                            }
                        }
                    } else if constexpr (TS) {
                        if (rev) {
                            if (A_MN) ca.retreat(p.selA, BKS);
                            if (B_MN) cb.retreat(p.selB, BKS);
                        } else {
                            if (A_MN) ca.advance(p.selA, BKS);
                            if (B_MN) cb.advance(p.selB, BKS);
                        }
                    }
                }
            }
            // CTA 0's full barriers count both CTAs' bytes: wait until every
            // copy it armed has landed before the pair can exit.
            for (int i = 0; i < NST; ++i)
                if (armed & (1u << i)) mbar_wait_drain(full0 + 8 * i, (armed_par >> i) & 1u, p.wait_limit_ns);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (CTA 0 only) ----------------
            const uint32_t idesc = p.idesc;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int w = pair_id; ok && w < p.total_work; w += npairs, ++it) {
                const int acc = it & 1;
                const uint32_t acc_par = (it >> 1) & 1;
                if (!mbar_wait(tempty0 + 8 * acc, acc_par ^ 1u, p)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * BN;
                uint32_t accumulate = 0;
                const Work wk = work_item(p, w);
                {
                    for (int f = wk.f0; f < wk.f1; ++f) {
                        if (!mbar_wait(full0 + 8 * stage, phase, p)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_base + stage * STG;
                        const uint32_t sb = sa + P_A_BYTES * KB2;
#pragma unroll
                        for (int kk = 0; kk < 4 * KB2; ++kk) {
                            // K-major: K block kk / 4 is its own 16 KB slab
                            const uint64_t ad =
                                A_MN ? smem_desc(sa + kk * E::KADV_MN, E::MNB_BYTES * KB2, 1024)
                                     : smem_desc(sa + (kk >> 2) * P_A_BYTES + (kk & 3) * 32, 16, 1024);
                            const uint64_t bd =
                                B_MN ? smem_desc(sb + kk * E::KADV_MN, E::MNB_BYTES * KB2, 1024)
                                     : smem_desc(sb + (kk >> 2) * P_B_BYTES + (kk & 3) * 32, 16, 1024);
                            umma_op_pair<F8>(d, ad, bd, idesc, accumulate);
                            accumulate = 1;
                        }
                        umma_commit_pair_mc(empty0 + 8 * stage);
                        if (++stage == NST) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(tfull0 + 8 * acc);
            }
            umma_commit_pair(drain);
            mbar_wait_drain(drain, 0, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..9 of both CTAs) ----------------
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const float dq = dequant_factor(p);
        Stager stg{smem_base + NST * STG + BAR_BYTES + (warp - 2) * EPI_STAGE_BYTES, 0u};
        const uint32_t tempty_leader = map_to_cta(tempty0, 0);
        int it = 0;
        for (int w = pair_id; w < p.total_work; w += npairs, ++it) {
            const int acc = it & 1;
            const uint32_t acc_par = (it >> 1) & 1;
            const bool ok = mbar_wait(tfull0 + 8 * acc, acc_par, p);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const Work wk = work_item(p, w);
            int pi, mt, nt;
            tile_coords(p, wk.t, pi, mt, nt);
            const int row = mt * P_TILE_M + 128 * rank + q * 32 + lane;
            const uint32_t taddr = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
            if (EPI == EPI_COL || EPI == EPI_DACT || wk.j < 0) {  // the split is planned for PLAIN / F32 only
                if (p.out_tma)
                    run_epilogue_tma<EPI>(p, pi, row, nt, taddr, half, dq, stg, lane, wk.t);
                else
                    run_epilogue<EPI>(p, pi, row, nt, taddr, half, dq);
                tc_fence_before();
                mbar_arrive_cluster(tempty_leader + 8 * acc);
            } else if constexpr (EPI == EPI_PLAIN || EPI == EPI_F32) {
                // tail unit: park this warp's raw accumulator slice, free the
                // accumulator, and finish the slice if it is the last to arrive
                const int tt = wk.t - p.tail_first;
                const int slot = static_cast<int>(rank) * 8 + q * 2 + half;
                float *ws_slice = p.tail_ws + (static_cast<size_t>(tt) * p.tail_s * 16 + slot) * TAIL_SLICE_FLOATS;
                float *mine = ws_slice + static_cast<size_t>(wk.j) * TAIL_UNIT_FLOATS;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld32(taddr + (4 * half + c) * 32, r);
                    tmem_ld_wait();
                    tail_store32(mine, c, lane, r);
                }
                tc_fence_before();
                mbar_arrive_cluster(tempty_leader + 8 * acc);
                __threadfence();  // this thread's slice is visible before the warp's arrival counts
                __syncwarp();
                unsigned prev = 0;
                if (lane == 0) prev = atomicAdd(p.tail_cnt + tt * 16 + slot, 1u);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev == static_cast<unsigned>(p.tail_s - 1)) {
                    __threadfence();  // and the other units' slices are visible to this warp
                    run_epilogue_tma<EPI>(p, pi, row, nt, taddr, half, dq, stg, lane, wk.t, ws_slice, p.tail_s);
                }
            }
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    clk_mark.stop(p.clk);
}

}  // namespace tc
}  // namespace tpmlp
