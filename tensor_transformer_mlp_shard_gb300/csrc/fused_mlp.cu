// Fused MLP forward for narrow layers (Megatron's FlashFusedMLP,
// "Megatron-LM 源码精读" s7, the fusions/ entry): one persistent
// kernel per 128-token tile runs
//   for every shard i and every 128-unit chunk c of shard i:
//     acc1  = X_tile W1_i[c]^T                    (tcgen05, TMEM, N = 128)
//     pre   = acc1 + b1_i[c]  -> HBM (kept for the backward)
//     A     = act(pre)        -> HBM (kept for the backward)
//                             -> shared memory, two 128-byte swizzled K-major atoms
//     Y    += A W2_i[:, c]^T                      (tcgen05, TMEM, K = 128)
//   Y = (X +) dropout(Y + b2) -> HBM   (dropout only in the TransformerLayer)
// so A never makes the round trip HBM -> row GEMM, and the cross-shard sum of
// the row layer (the forward all-reduce) is the Y accumulation over (i, c).
// Under SwiGLU (the kernel's second instance) a chunk is 64 units of A: the
// column GEMM's 128 columns are 64 gate and the 64 matching up units, and
// A = silu(gate) * up.
// The output tile [128 x H] lives in TMEM next to two 128-column
// accumulators of the column GEMM, so H <= 256: at wider layers the output
// row does not fit on chip and the two-kernel path (tc_gemm) runs instead.
// Token tiles go to the CTAs whole, or, when they spill over whole rounds of
// the SMs by a little, as an even split of (tile, chunk) units (below).
//
// Warp roles (320 threads): warp 0 issues TMA (the X tile once per token
// tile, then W1 and W2 boxes of 16 KB in consumption order through a 6-slot
// ring), warp 1 issues the MMAs (column GEMM of chunk c, then row GEMM of
// chunk c - 2, so that the tensor core works while two epilogue groups turn
// chunks c - 1 and c - 2 into A), warps 2-9 run the epilogues in two groups
// that take alternate chunks.  A group writes A into its shared-memory
// operand buffer, from which one bulk tensor store per 64 units copies it to
// HBM; the group's output columns of Y are staged in the same buffer at the
// end of a tile and stored the same way, 32 rows per warp; pre goes out with
// direct 32-byte stores (staging it too measured slower).  Every wait is
// bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "tc_gemm_kernels.cuh"

namespace tpmlp {
namespace tc {
tp_status encode_map_ex(CUtensorMap *m, const void *ptr, int rows, int cols, long long ld, int box_inner,
                        int box_rows, CUtensorMapDataType type, int esize, CUtensorMapSwizzle swz);
tp_status encode_map(CUtensorMap *m, const void *ptr, int rows, int cols, int box_inner, int box_rows, bool fp8);
}  // namespace tc

namespace fm {
using namespace tc;

constexpr int kRows = 128;      // token rows per tile (tcgen05 M)
constexpr int kChunk = 128;     // hidden units per chunk: column GEMM N, row GEMM K
constexpr int kMaxH = 256;      // output tile [128 x H] + 2 x 128 accumulator columns <= 512 TMEM columns
constexpr int kBox = 128 * 128; // one [128 rows x 64] bf16 box (128-byte rows): 16 KB
constexpr int kSlots = 6;
constexpr int kNB = 2;          // column-GEMM accumulators and A buffers
constexpr int kLag = 2;         // the row GEMM of chunk c is issued after the column GEMM of chunk c + 2
constexpr int kXBytes = kMaxH / 64 * (kRows * 128);  // X tile: H/64 boxes of [128 x 64]
constexpr int kAtom = kRows * 128;                   // [128 rows x 64] bf16, one 128-byte swizzle atom
constexpr int kABytes = kChunk / 64 * kAtom;         // A chunk [128 x 128] bf16: two K-major atoms
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kOffX = kSlots * kBox;
constexpr int kOffA = kOffX + kXBytes;
constexpr int kOffBar = kOffA + kNB * kABytes;
constexpr int kSmemBytes = kOffBar + 1024 + 1024;  // + barriers, + alignment slack
constexpr int kTmemCols = 512;
constexpr int kAccCol = 256;  // column-GEMM accumulators at TMEM columns 256 and 384
constexpr int kPartF4 = 4 * 8 * 32;  // one warp's parked sums: 32 rows x 128 columns fp32, in float4
static_assert(2 * kSlots + 5 + 5 * kNB <= 64, "barriers overlap the TMEM address slot");
static_assert(kAccCol + kNB * kChunk <= kTmemCols, "column accumulators beyond TMEM");
static_assert(kLag <= kNB, "the row GEMM must not lag the column GEMM by more than a buffer cycle");
static_assert(kSmemBytes <= 232448, "shared memory above the 227 KB a block may use");

struct FusedParams {
    CUtensorMap mapX[kMaxShards];    // X token shards, boxes [128 rows x 64], 128-byte swizzle
    CUtensorMap mapW1[kMaxShards];   // W1_i [Fs, H], boxes [128 units x 64]
    CUtensorMap mapW2[kMaxShards];   // W2_i [H, Fs], boxes [128 rows of H x 64 units]
    CUtensorMap mapA[kMaxShards];    // A_i [M, Fs], boxes [128 tokens x 64 units] stored from shared memory
    __nv_bfloat16 *pre[kMaxShards];  // pre_i [M, Fs] (or null)
    CUtensorMap mapY[kMaxShards];    // Y token shards [rows_split or M, H], boxes [32 tokens x 64], stored
    const __nv_bfloat16 *b1[kMaxShards];
    const __nv_bfloat16 *b2;
    const __nv_bfloat16 *res[kMaxShards];
    DropoutParams drop;        // Y = R + dropout(sum + b2) (TransformerLayer bias-dropout-add)
    int rows_split, n_tok;
    int M, H, Fs, T, act, has_bias, has_res, has_pre;
    int pre_v8;  // every pre_i 32-byte aligned: 32-byte stores
    int swiglu;  // SwiGLU: a chunk is 64 gate and the 64 matching up units
    int uc;      // units of A per chunk: 128, or 64 under SwiGLU
    int pre_ld;  // row stride of pre_i: Fs, or 2 Fs (gate | up) under SwiGLU
    int m_tiles, cps, nc, kb;  // chunks per shard, chunks per tile (T * cps), H / 64
    int nh;                    // 128-column halves of the output (H / 128 rounded up)
    // Even split: CTA b takes the (tile, chunk position) units
    // [b W / G, (b + 1) W / G) of the W = m_tiles * nc in tile-major order
    // (0: CTA b takes whole tiles b, b + G, ...).  A tile cut at a range
    // boundary is finished by whichever of its two CTAs gets there second.
    int split;
    long long work;
    float *part;         // [G][8 warps][4096] fp32 output slices of the cut tiles
    unsigned *part_cnt;  // [G][8] arrivals per cut tile and warp, then [G][8] ready flags (zeroed)
    uint32_t idesc;            // bf16 x bf16 -> fp32, both K-major, M = 128, N = 128
    int *status;
    unsigned *abort_word;
    unsigned launch_id;
    unsigned long long wait_limit_ns;
};

__device__ __forceinline__ bool fwait(uint32_t bar, uint32_t parity, const FusedParams &p) {
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

// Chunk at position c of token tile t.  Every tile walks all nc chunks, but
// starting at chunk t mod nc, so that the CTAs (which start together) stream
// different weight chunks at any moment instead of all asking the same L2
// lines for the same boxes.  The order changes only the fp32 order of the
// additions into the output tile.
__device__ __forceinline__ int chunk_at(const FusedParams &p, int t, int c) {
    const int ch = c + t % p.nc;
    return ch < p.nc ? ch : ch - p.nc;
}

// The k-th run of this CTA's work: chunk positions [c0, c1) of token tile t.
// With the even split a CTA's range holds at least nc units (the host takes
// it only with more tiles than CTAs), so a tile is cut at most once: the
// first run of CTA b may start inside a tile (c0 > 0) and the last run of
// CTA b - 1 then ends at the same position (c1 < nc).
__device__ __forceinline__ bool segment(const FusedParams &p, int k, int &t, int &c0, int &c1) {
    if (!p.split) {
        t = blockIdx.x + k * gridDim.x;
        c0 = 0;
        c1 = p.nc;
        return t < p.m_tiles;
    }
    const long long s = p.work * blockIdx.x / gridDim.x, e = p.work * (blockIdx.x + 1) / gridDim.x;
    const long long u = k == 0 ? s : (s / p.nc + k) * p.nc;
    if (u >= e) return false;
    t = static_cast<int>(u / p.nc);
    const long long base = static_cast<long long>(t) * p.nc;
    c0 = static_cast<int>(u - base);
    c1 = static_cast<int>(e - base < p.nc ? e - base : p.nc);
    return true;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *a) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned *a, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// bounded wait for a flag another CTA of this launch sets
__device__ __forceinline__ bool flag_wait(const unsigned *f, const FusedParams &p) {
    if (ld_acquire_u32(f) != 0u) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (ld_acquire_u32(f) != 0u) return true;
        if ((n & 63u) == 0) {
            if (*reinterpret_cast<volatile unsigned *>(p.abort_word) == p.launch_id) return false;
            if (global_timer_ns() - t0 > p.wait_limit_ns) {
                raise_device_error(p.status, p.abort_word, p.launch_id, TP_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// token shard and local row of global row `row0`
__device__ __forceinline__ void tok_index(const FusedParams &p, int row0, int &j, int &lrow) {
    j = 0;
    lrow = row0;
    if (p.rows_split) {
        j = min(row0 / p.rows_split, p.n_tok - 1);
        lrow = row0 - j * p.rows_split;
    }
}

// v[0..8) += the 8 bf16 of w, two lanes of fp32 at a time
__device__ __forceinline__ void add_bf16x8(float *v, const uint4 &w) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) st2(v + 2 * k, __fadd2_rn(ld2(v + 2 * k), make_float2(bf16_lo(u[k]), bf16_hi(u[k]))));
}

// 32 bf16 of one row: four 16-byte stores (the row's 64 bytes are contiguous)
// the same as two 32-byte stores (dst 32-byte aligned): half the store
// instructions for a warp whose lanes each write a different row
__device__ __forceinline__ void store_row32_v8(__nv_bfloat16 *dst, const uint4 (&w)[4]) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * j),
                     "r"(w[2 * j].x), "r"(w[2 * j].y), "r"(w[2 * j].z), "r"(w[2 * j].w), "r"(w[2 * j + 1].x),
                     "r"(w[2 * j + 1].y), "r"(w[2 * j + 1].z), "r"(w[2 * j + 1].w)
                     : "memory");
}
__device__ __forceinline__ void store_row32(__nv_bfloat16 *dst, const uint4 (&w)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) reinterpret_cast<uint4 *>(dst)[j] = w[j];
}

// A SwiGLU chunk's epilogue (one thread = one token row): the accumulator
// holds the 64 gate units u0.. in columns [0, 64) and the matching up units in
// [64, 128); pre gets both (gate | up halves of its row), A = silu(gate) * up
// goes into atom 0 of the group's buffer, in two 32-unit pieces.  The same
// arithmetic as the two-kernel path's column epilogue.
template <typename Release>
__device__ __forceinline__ bool swiglu_chunk(const FusedParams &p, int i, int u0, int b, uint32_t use, int row,
                                             bool row_ok, uint32_t r_tile, uint32_t lane_off, uint32_t tmem_base,
                                             uint32_t buf, uint32_t accf0, uint32_t acce0, uint32_t ae0,
                                             Release &release) {
    auto fetch = [&](int jp, uint4 (&bg)[4], uint4 (&bu)[4]) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            bg[k] = p.has_bias ? *reinterpret_cast<const uint4 *>(p.b1[i] + u0 + 32 * jp + 8 * k) : make_uint4(0, 0, 0, 0);
            bu[k] = p.has_bias ? *reinterpret_cast<const uint4 *>(p.b1[i] + p.Fs + u0 + 32 * jp + 8 * k)
                               : make_uint4(0, 0, 0, 0);
        }
    };
    uint4 bg[4], bu[4];
    fetch(0, bg, bu);
    bool good = fwait(accf0 + 8 * b, use & 1u, p);
    if (!__all_sync(0xffffffffu, good)) return false;
    tc_fence_after();
    const uint32_t acc = tmem_base + kAccCol + kChunk * b + lane_off;
#pragma unroll
    for (int jp = 0; jp < 2; ++jp) {
        uint32_t rg[32], ru[32];
        tmem_ld32(acc + 32 * jp, rg);
        tmem_ld32(acc + 64 + 32 * jp, ru);
        tmem_ld_wait();
        if (jp == 1) {
            tc_fence_before();
            mbar_arrive(acce0 + 8 * b);  // the column GEMM may reuse the accumulator
        }
        float G[32], U[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            G[j] = __uint_as_float(rg[j]);
            U[j] = __uint_as_float(ru[j]);
        }
        if (p.has_bias) {
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                add_bf16x8(G + 8 * g8, bg[g8]);
                add_bf16x8(U + 8 * g8, bu[g8]);
            }
        }
        if (jp == 0) fetch(1, bg, bu);
        uint4 wa[4];
        if (p.has_pre && row_ok) {
            __nv_bfloat16 *dst = p.pre[i] + static_cast<long long>(row) * p.pre_ld + u0 + 32 * jp;
            pack_bf16x32(G, wa);
            if (p.pre_v8)
                store_row32_v8(dst, wa);
            else
                store_row32(dst, wa);
            pack_bf16x32(U, wa);
            if (p.pre_v8)
                store_row32_v8(dst + p.Fs, wa);
            else
                store_row32(dst + p.Fs, wa);
        }
        swiglu_n<32>(G, U);
        pack_bf16x32(G, wa);
        if (jp == 0) {
            // the A buffer is free once the bulk stores from it have read it and the
            // row GEMM of chunk cg - kNB is done
            good = release() && fwait(ae0 + 8 * b, (use & 1u) ^ 1u, p);
            if (!__all_sync(0xffffffffu, good)) return false;
        }
        // atom 0, row r_tile, 16-byte chunks 4 jp .. + 3, 128-byte swizzle
        const uint32_t rowa = buf + r_tile * 128u;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint32_t c16 = 4u * static_cast<uint32_t>(jp) + static_cast<uint32_t>(jj);
            st_shared_v4(rowa + ((c16 ^ (r_tile & 7u)) << 4), wa[jj]);
        }
    }
    return true;
}

template <bool SWIGLU>  // the SwiGLU chunk layout (p.swiglu), compiled apart from the GeLU one
__global__ void __launch_bounds__(kThreads, 1) fused_mlp_fwd_kernel(const __grid_constant__ FusedParams p) {
    constexpr int UC = SWIGLU ? 64 : kChunk;  // units of A per chunk (p.uc)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 64);  // after the 2 * kSlots + 5 + 5 * kNB barriers
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * kSlots;
    const uint32_t xfull = empty0 + 8 * kSlots, xempty = xfull + 8;
    const uint32_t accf0 = xempty + 8, acce0 = accf0 + 8 * kNB;  // column-GEMM accumulator full / drained
    const uint32_t af0 = acce0 + 8 * kNB, ae0 = af0 + 8 * kNB;    // A buffer written / consumed
    const uint32_t yfull = ae0 + 8 * kNB, yempty = yfull + 8, drain = yempty + 8;
    const uint32_t bufr0 = drain + 8;  // per epilogue group: the bulk stores from its buffer have read it
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr uint32_t kEpiThreads = 32 * kEpiWarps;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        mbar_init(xfull, 1);
        mbar_init(xempty, 1);
        for (int b = 0; b < kNB; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, kEpiThreads / 2);  // one epilogue group per buffer
            mbar_init(af0 + 8 * b, kEpiThreads / 2);
            mbar_init(ae0 + 8 * b, 1);
        }
        mbar_init(yfull, 1);
        mbar_init(yempty, kEpiThreads);
        mbar_init(drain, 1);
        for (int g = 0; g < kNB; ++g) mbar_init(bufr0 + 8 * g, kEpiThreads / 2);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // launched with programmatic dependent launch: the set-up above overlaps the
    // previous kernel, and nothing in global memory is touched before it is done
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int slot = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool x_armed = false, ok = true;
            uint32_t x_par = 0;
            // one 16 KB box [128 rows x 64], or (c1b >= 0) two [64 rows x 64]
            // boxes stacked in the slot: the gate and up rows of a SwiGLU chunk
            auto load_box = [&](const CUtensorMap *map, int c0, int c1, int c1b = -1) -> bool {
                if (!fwait(empty0 + 8 * slot, phase ^ 1u, p)) return false;
                const uint32_t fb = full0 + 8 * slot;
                mbar_arrive_expect_tx(fb, kBox);
                armed |= 1u << slot;
                armed_par = (armed_par & ~(1u << slot)) | (phase << slot);
                tma_load_2d(sbase + slot * kBox, map, fb, c0, c1);
                if (c1b >= 0) tma_load_2d(sbase + slot * kBox + kBox / 2, map, fb, c0, c1b);
                if (++slot == kSlots) {
                    slot = 0;
                    phase ^= 1u;
                }
                return true;
            };
            int t, c0, c1;
            for (int it = 0; ok && segment(p, it, t, c0, c1); ++it) {
                int tj, tl;
                tok_index(p, t * kRows, tj, tl);
                if (!fwait(xempty, (it & 1) ^ 1u, p)) break;
                mbar_arrive_expect_tx(xfull, p.kb * kRows * 128);
                x_armed = true;
                x_par = it & 1;
                for (int kb = 0; kb < p.kb; ++kb)
                    tma_load_2d(sbase + kOffX + kb * kRows * 128, &p.mapX[tj], xfull, kb * 64, tl);
                // boxes in the order the MMA warp consumes them; position c of
                // tile t holds chunk (c + t) mod nc
                for (int c = c0; ok && c < c1 + kLag; ++c) {
                    if (c < c1) {
                        const int ch = chunk_at(p, t, c), i = ch / p.cps, u0 = (ch % p.cps) * UC;
                        for (int kb = 0; ok && kb < p.kb; ++kb)
                            ok = load_box(&p.mapW1[i], kb * 64, u0, SWIGLU ? p.Fs + u0 : -1);
                    }
                    if (ok && c - kLag >= c0) {
                        const int ch = chunk_at(p, t, c - kLag), i = ch / p.cps, u0 = (ch % p.cps) * UC;
                        for (int h = 0; ok && h < p.nh; ++h)
                            for (int k2 = 0; ok && k2 < UC / 64; ++k2)
                                ok = load_box(&p.mapW2[i], u0 + 64 * k2, h * 128);
                    }
                }
            }
            // no bulk copy may still be landing in shared memory when the CTA exits
            for (int i = 0; i < kSlots; ++i)
                if (armed & (1u << i)) mbar_wait_drain(full0 + 8 * i, (armed_par >> i) & 1u, p.wait_limit_ns);
            if (x_armed) mbar_wait_drain(xfull, x_par, p.wait_limit_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int slot = 0;
            uint32_t phase = 0;
            bool ok = true;
            int cgb = 0, t, c0, c1;  // cgb: chunks of earlier runs (accumulator and A buffer turns)
            for (int it = 0; ok && segment(p, it, t, c0, c1); ++it, cgb += c1 - c0) {
                for (int c = c0; ok && c < c1 + kLag; ++c) {
                    if (c < c1) {
                        // column GEMM of chunk c: acc1[b] = X_tile W1 chunk^T (K = H)
                        const int cg = cgb + c - c0, b = cg % kNB;
                        const uint32_t use = static_cast<uint32_t>(cg) / kNB;
                        if (!fwait(acce0 + 8 * b, (use & 1u) ^ 1u, p)) {
                            ok = false;
                            break;
                        }
                        if (c == c0 && !fwait(xfull, it & 1, p)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem_base + kAccCol + kChunk * b;
                        for (int kb = 0; kb < p.kb; ++kb) {
                            if (!fwait(full0 + 8 * slot, phase, p)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t sx = sbase + kOffX + kb * kRows * 128, sw = sbase + slot * kBox;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                umma_bf16(d, smem_desc(sx + kk * 32, 16, 1024), smem_desc(sw + kk * 32, 16, 1024),
                                          p.idesc, (kb | kk) ? 1u : 0u);
                            umma_commit(empty0 + 8 * slot);
                            if (++slot == kSlots) {
                                slot = 0;
                                phase ^= 1u;
                            }
                        }
                        if (!ok) break;
                        umma_commit(accf0 + 8 * b);
                        if (c == c1 - 1) umma_commit(xempty);  // the run's last read of X
                    }
                    if (c - kLag >= c0) {
                        // row GEMM of chunk c - kLag: Y[:, 128h..] += A W2 chunk^T (K = 128)
                        const int cg = cgb + c - kLag - c0, b = cg % kNB;
                        const uint32_t use = static_cast<uint32_t>(cg) / kNB;
                        if (!fwait(af0 + 8 * b, use & 1u, p)) {
                            ok = false;
                            break;
                        }
                        if (c == c0 + kLag && !fwait(yempty, (it & 1) ^ 1u, p)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = sbase + kOffA + b * kABytes;
                        for (int h = 0; ok && h < p.nh; ++h) {
                            for (int k2 = 0; k2 < UC / 64; ++k2) {
                                if (!fwait(full0 + 8 * slot, phase, p)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                const uint32_t sw = sbase + slot * kBox;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    umma_bf16(tmem_base + 128 * h, smem_desc(sa + k2 * kAtom + kk * 32, 16, 1024),
                                              smem_desc(sw + kk * 32, 16, 1024), p.idesc,
                                              (c > c0 + kLag || k2 > 0 || kk > 0) ? 1u : 0u);
                                umma_commit(empty0 + 8 * slot);
                                if (++slot == kSlots) {
                                    slot = 0;
                                    phase ^= 1u;
                                }
                            }
                        }
                        if (!ok) break;
                        umma_commit(ae0 + 8 * b);
                    }
                }
                if (!ok) break;
                umma_commit(yfull);
            }
            // all issued MMAs complete before TMEM is released
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ---------------- epilogues (warps 2..9) ----------------
        // Two groups of four warps take alternate chunks (group g: the chunks
        // whose accumulator / A buffer is g), so one group turns a chunk into A
        // while the other waits for the next accumulator; within a group warp
        // w owns TMEM lane quarter w & 3 (32 token rows) and all 64 columns.
        const int q = warp & 3;            // TMEM lane quarter: rows q*32 .. q*32+31 of the tile
        const int h = (warp - 2) >> 2;     // group: chunks with buffer h; output columns 128h..
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t r_tile = static_cast<uint32_t>(q * 32 + lane);  // row within the tile
        const bool elect = lane == 0 && ((warp - 2) & 3) == 0;          // issues the group's bulk stores
        const uint32_t buf = sbase + kOffA + h * kABytes;  // the group's A buffer (= buffer h), Y staging too
        uint32_t nrel = 0;
        // Before the group writes its buffer: the bulk stores issued from it have
        // read it.  A warp's lane 0 waits for its own (each warp stages and stores
        // its 32 rows of Y; the elected thread also the whole buffer's A), then
        // the group's 128 threads meet on its barrier.
        auto release = [&]() -> bool {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            mbar_arrive(bufr0 + 8 * h);
            return fwait(bufr0 + 8 * h, nrel++ & 1u, p);
        };
        int cgb = 0, t, c0, c1;
        bool ok = true;
        for (int it = 0; ok && segment(p, it, t, c0, c1); ++it, cgb += c1 - c0) {
            const int row0 = t * kRows + q * 32;
            const int row = row0 + lane;
            const bool block_ok = row0 < p.M;  // warp-uniform
            const bool row_ok = row < p.M;
            for (int c = c0 + ((cgb & 1) == h ? 0 : 1); c < c1; c += 2) {
                const int cg = cgb + c - c0, b = cg % kNB;
                const uint32_t use = static_cast<uint32_t>(cg) / kNB;
                const int ch = chunk_at(p, t, c), i = ch / p.cps, u0 = (ch % p.cps) * UC;
                if constexpr (SWIGLU) {
                    ok = swiglu_chunk(p, i, u0, b, use, row, row_ok, r_tile, lane_off, tmem_base, buf, accf0, acce0,
                                      ae0, release);
                    if (!ok) break;
                } else {
                // b1 of one 32-unit piece: the first piece's while the accumulator
                // fills, each next piece's while the current one is computed
                auto fetch_b1 = [&](int hh, uint4 (&bw)[4]) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        bw[k] = p.has_bias ? *reinterpret_cast<const uint4 *>(p.b1[i] + u0 + 32 * hh + 8 * k)
                                           : make_uint4(0, 0, 0, 0);
                };
                uint4 bcur[4], bnext[4];
                fetch_b1(0, bcur);
                ok = fwait(accf0 + 8 * b, use & 1u, p);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t rowa = buf + r_tile * 128u;
#pragma unroll
                for (int hh = 0; hh < kChunk / 32; ++hh) {  // 32 units at a time
                    const int u = u0 + 32 * hh;
                    uint32_t r[32];
                    tmem_ld32(tmem_base + kAccCol + kChunk * b + 32 * hh + lane_off, r);
                    tmem_ld_wait();
                    if (hh + 1 < kChunk / 32) fetch_b1(hh + 1, bnext);
                    if (hh == kChunk / 32 - 1) {
                        tc_fence_before();
                        mbar_arrive(acce0 + 8 * b);  // the column GEMM may reuse the accumulator
                    }
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if (p.has_bias) {
#pragma unroll
                        for (int g8 = 0; g8 < 4; ++g8) add_bf16x8(v + 8 * g8, bcur[g8]);
                    }
                    uint4 wa[4];
                    if (p.has_pre) {
                        pack_bf16x32(v, wa);
                        if (row_ok) {
                            __nv_bfloat16 *dst = p.pre[i] + static_cast<long long>(row) * p.pre_ld + u;
                            if (p.pre_v8)
                                store_row32_v8(dst, wa);
                            else
                                store_row32(dst, wa);
                        }
                    }
                    if (p.act == TP_ACT_GELU_TANH) gelu_tanh_n<32>(v);
                    pack_bf16x32(v, wa);
                    if (hh == 0) {
                        // the A buffer is free once the bulk stores from it have read it and
                        // the row GEMM of chunk cg - kNB is done (waited for only now, so
                        // that the first piece is computed meanwhile)
                        ok = release() && fwait(ae0 + 8 * b, (use & 1u) ^ 1u, p);
                        if (!__all_sync(0xffffffffu, ok)) {
                            ok = false;
                            break;
                        }
                    }
                    // A into the row GEMM's operand buffer (which a bulk store then copies
                    // to A_i, clipping rows past M): K-major atom hh / 2, row
                    // r_tile, 16-byte chunks 4 (hh % 2) .. + 3 of its 128-byte line,
                    // 128-byte swizzle (chunk ^ (row & 7))
                    const uint32_t atom = rowa + static_cast<uint32_t>(hh >> 1) * kAtom;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint32_t c16 = 4u * static_cast<uint32_t>(hh & 1) + static_cast<uint32_t>(jj);
                        st_shared_v4(atom + ((c16 ^ (r_tile & 7u)) << 4), wa[jj]);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) bcur[k] = bnext[k];
                }
                if (!ok) break;
                }
                fence_async_smem();
                mbar_arrive(af0 + 8 * b);
                if (elect) {  // once the group's 128 rows are in, A goes to HBM in two boxes
                    ok = fwait(af0 + 8 * b, use & 1u, p);
                    if (ok) {
                        for (int k2 = 0; k2 < UC / 64; ++k2) tma_store_2d(&p.mapA[i], buf + k2 * kAtom, u0 + 64 * k2, t * kRows);
                        bulk_commit();
                    }
                }
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            int tj, tl;
            tok_index(p, row0, tj, tl);
            const __nv_bfloat16 *res_row =
                p.has_res ? p.res[tj] + static_cast<long long>(row_ok ? tl + lane : tl) * p.H : nullptr;
            // b2 and the residual of 32 output columns (the first piece's while Y accumulates,
            // each later piece's while the one before it is computed)
            auto fetch = [&](int cb, uint4 (&bb)[4], uint4 (&rr)[4]) {
                const int col = h * 128 + cb * 32;
                const bool in = col < p.H;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    bb[k] = p.has_bias && in ? *reinterpret_cast<const uint4 *>(p.b2 + col + 8 * k) : make_uint4(0, 0, 0, 0);
                    rr[k] = res_row && in && row_ok ? *reinterpret_cast<const uint4 *>(res_row + col + 8 * k)
                                                    : make_uint4(0, 0, 0, 0);
                }
            };
            uint4 bb[4], rr[4];
            fetch(0, bb, rr);  // while the last row GEMMs run
            ok = fwait(yfull, it & 1, p);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            // The group's output columns are staged in its buffer, free once the last
            // row GEMM is done (which yfull says) and the bulk stores from it have
            // read it; every warp of the group takes part, whatever it does next.
            const int ycols = min(128, p.H - h * 128);
            if (ycols > 0) {
                ok = release();
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            // A tile cut between two CTAs: the first of them to get here parks
            // its raw sums (this warp's 32 rows x 128 columns) and moves on; the
            // second adds them to its own and runs the epilogue.  The sum of the
            // two parts is the same whichever arrives first.
            int other = -1;  // the parked slot to add, if this warp arrived second
            if (p.split && (c0 > 0 || c1 < p.nc)) {
                const int slot = (c0 > 0 ? blockIdx.x : blockIdx.x + 1) * kEpiWarps + (warp - 2);
                float4 *mine = reinterpret_cast<float4 *>(p.part) + static_cast<size_t>(slot) * kPartF4;
                unsigned *ready = p.part_cnt + gridDim.x * kEpiWarps + slot;
                unsigned prev = 0;
                if (lane == 0) prev = atomicAdd(p.part_cnt + slot, 1u);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev == 0) {
#pragma unroll 1
                    for (int cb = 0; cb < 4; ++cb) {
                        if (h * 128 + cb * 32 >= p.H) break;
                        uint32_t r[32];
                        tmem_ld32(tmem_base + h * 128 + cb * 32 + lane_off, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mine[(cb * 8 + k) * 32 + lane] =
                                make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                            __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
                    }
                    tc_fence_before();
                    mbar_arrive(yempty);
                    __threadfence();  // every lane's slice is visible before the flag
                    __syncwarp();
                    if (lane == 0) st_release_u32(ready, 1u);
                    continue;
                }
                // the first CTA claimed its arrival before this one, so it is
                // running and its flag comes without waiting on anything else
                ok = flag_wait(ready, p);
                if (!__all_sync(0xffffffffu, ok)) break;
                other = slot;
            }
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                const int col = h * 128 + cb * 32;
                if (col >= p.H) break;
                uint32_t r[32];
                tmem_ld32(tmem_base + col + lane_off, r);
                tmem_ld_wait();
                uint4 bn[4], rn[4];  // the next piece's b2 and residual, in flight while this one is computed
                if (cb + 1 < 4) fetch(cb + 1, bn, rn);
                if (block_ok) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if (other >= 0) {  // the other CTA's part: plain loads, ordered after the flag's acquire
                        const float4 *src = reinterpret_cast<const float4 *>(p.part) +
                                            static_cast<size_t>(other) * kPartF4 + cb * 8 * 32 + lane;
#pragma unroll
                        for (int k4 = 0; k4 < 8; k4 += 4) {
                            float4 o[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) o[k] = src[(k4 + k) * 32];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                v[4 * (k4 + k) + 0] += o[k].x; v[4 * (k4 + k) + 1] += o[k].y;
                                v[4 * (k4 + k) + 2] += o[k].z; v[4 * (k4 + k) + 3] += o[k].w;
                            }
                        }
                    }
                    if (p.has_bias) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) add_bf16x8(v + 8 * k, bb[k]);
                    }
                    if (p.drop.on) dropout32(p.drop, row, col, row_ok, v);
                    if (res_row) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) add_bf16x8(v + 8 * k, rr[k]);
                    }
                    uint4 w[4];
                    pack_bf16x32(v, w);
                    const uint32_t atom = buf + r_tile * 128u + static_cast<uint32_t>(cb >> 1) * kAtom;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint32_t c16 = 4u * static_cast<uint32_t>(cb & 1) + static_cast<uint32_t>(jj);
                        st_shared_v4(atom + ((c16 ^ (r_tile & 7u)) << 4), w[jj]);
                    }
                }
                if (cb + 1 < 4) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        bb[k] = bn[k];
                        rr[k] = rn[k];
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(yempty);
            if (ycols > 0 && block_ok) {  // this warp's 32 rows, staged: one bulk store per 64 columns
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    for (int k2 = 0; k2 < ycols / 64; ++k2)
                        tma_store_2d(&p.mapY[tj], buf + static_cast<uint32_t>(q * 32 * 128 + k2 * kAtom),
                                     h * 128 + 64 * k2, tl);
                    bulk_commit();
                }
            }
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait<0>();  // the epilogue warps' bulk stores are done
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace fm

static std::atomic<int> g_fused_mode{TP_FUSED_AUTO};
void set_fused_fwd_mode(int mode) { g_fused_mode.store(mode); }
int fused_fwd_mode() { return g_fused_mode.load(); }

bool fused_fwd_supported(int H, int Fs, int act, int dtype) {
    const int uc = act == TP_ACT_SWIGLU ? 64 : fm::kChunk;  // units of A per chunk
    return dtype == TP_DT_BF16 && H >= 64 && H <= fm::kMaxH && H % 64 == 0 && Fs >= uc && Fs % uc == 0;
}

// Bytes of scratch the even split of an M-token forward takes: the parked
// sums of one cut tile per CTA and two words per cut tile and warp.  0 (whole
// tiles per CTA) unless the tiles spill over whole rounds of the SMs by at
// most a quarter of a round: measured on GB300, the split won there (54
// against 68 us at 1.09 rounds) and lost to whole tiles from about a third of
// a round on (142 against 133 us at 3.37 rounds), because the even split
// gives most CTAs one more run of chunks to start and drain.
size_t fused_fwd_scratch_bytes(long long M) {
    using namespace fm;
    const long long tiles = (M + kRows - 1) / kRows, g = num_sms();
    if (tiles <= g || tiles % g == 0 || tiles % g > g / 4) return 0;
    return static_cast<size_t>(g) * kEpiWarps * (kPartF4 * sizeof(float4) + 2 * sizeof(unsigned));
}

tp_status launch_fused_mlp_fwd(const FusedPlan &f, cudaStream_t st) {
    using namespace fm;
    if (f.M == 0) return TP_OK;
    if (f.T < 1 || f.T > kMaxShards || f.n_tok < 1 || f.n_tok > kMaxShards)
        return set_error(TP_ERR_ARG, "fused forward: bad shard counts");
    if (!fused_fwd_supported(f.H, f.Fs, f.act, TP_DT_BF16))
        return set_error(TP_ERR_UNSUPPORTED, "fused forward: H=%d, F/T=%d, act=%d outside its shapes", f.H, f.Fs,
                         f.act);
    FusedParams prm;
    memset(&prm, 0, sizeof(prm));
    const int tok_rows = f.rows_split ? f.rows_split : f.M;
    for (int j = 0; j < f.n_tok; ++j) {
        tp_status s = tc::encode_map(&prm.mapX[j], f.X[j], tok_rows, f.H, 64, kRows, false);
        if (s == TP_OK) s = tc::encode_map(&prm.mapY[j], f.Y[j], tok_rows, f.H, 64, 32, false);
        if (s != TP_OK) return s;
        prm.res[j] = f.has_res ? static_cast<const __nv_bfloat16 *>(f.R[j]) : nullptr;
    }
    for (int i = 0; i < f.T; ++i) {
        // W1_i [g Fs, H]; a SwiGLU chunk loads its gate and up rows as two 64-row boxes
        tp_status s = f.act == TP_ACT_SWIGLU ? tc::encode_map(&prm.mapW1[i], f.W1[i], 2 * f.Fs, f.H, 64, 64, false)
                                             : tc::encode_map(&prm.mapW1[i], f.W1[i], f.Fs, f.H, 64, kChunk, false);
        if (s == TP_OK) s = tc::encode_map(&prm.mapW2[i], f.W2[i], f.H, f.Fs, 64, 128, false);
        if (s == TP_OK) s = tc::encode_map(&prm.mapA[i], f.A[i], f.M, f.Fs, 64, kRows, false);
        if (s != TP_OK) return s;
        prm.pre[i] = f.has_pre ? static_cast<__nv_bfloat16 *>(f.pre[i]) : nullptr;
        prm.b1[i] = f.has_bias ? static_cast<const __nv_bfloat16 *>(f.b1[i]) : nullptr;
    }
    prm.b2 = f.has_bias ? static_cast<const __nv_bfloat16 *>(f.b2) : nullptr;
    prm.drop.on = f.dropout ? 1 : 0;
    prm.drop.threshold = f.drop_threshold;
    prm.drop.scale = f.drop_scale;
    prm.drop.seed_lo = static_cast<uint32_t>(f.drop_seed);
    prm.drop.seed_hi = static_cast<uint32_t>(f.drop_seed >> 32);
    prm.drop.ld = f.H;
    prm.drop.mask = f.dropout ? f.drop_mask : nullptr;
    prm.drop.mask_ld = (f.H + 31) / 32;
    prm.rows_split = f.rows_split;
    prm.n_tok = f.n_tok;
    prm.M = f.M;
    prm.H = f.H;
    prm.Fs = f.Fs;
    prm.T = f.T;
    prm.act = f.act;
    prm.has_bias = f.has_bias ? 1 : 0;
    prm.has_res = f.has_res ? 1 : 0;
    prm.has_pre = f.has_pre ? 1 : 0;
    prm.pre_v8 = 1;
    for (int i = 0; i < f.T; ++i)
        if (f.has_pre && (reinterpret_cast<uintptr_t>(f.pre[i]) & 31u)) prm.pre_v8 = 0;
    prm.m_tiles = (f.M + kRows - 1) / kRows;
    prm.swiglu = f.act == TP_ACT_SWIGLU ? 1 : 0;
    prm.uc = prm.swiglu ? 64 : kChunk;
    prm.pre_ld = prm.swiglu ? 2 * f.Fs : f.Fs;
    prm.cps = f.Fs / prm.uc;
    prm.nc = f.T * prm.cps;
    prm.kb = f.H / 64;
    prm.nh = (f.H + 127) / 128;
    // fp32 accumulator (bit 4), bf16 A and B (bits 7-9, 10-12), both K-major,
    // N/8 at bit 17, M/16 at bit 24
    prm.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kChunk >> 3) << 17) | (uint32_t(kRows >> 4) << 24);
    DeviceWords w;
    tp_status s = device_words(&w);
    if (s != TP_OK) return s;
    prm.status = w.status;
    prm.abort_word = w.abort_word;
    prm.launch_id = next_launch_id();
    prm.wait_limit_ns = wait_limit_ns();

    // opt in to > 48 KB of dynamic shared memory, once per device
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev % 64]) {
            cudaError_t e = cudaFuncSetAttribute(fused_mlp_fwd_kernel<false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(fused_mlp_fwd_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
            if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(fused_mlp_fwd)");
            attr_set[dev % 64] = true;
        }
    }
    const int grid = prm.m_tiles < num_sms() ? prm.m_tiles : num_sms();
    const size_t need = fused_fwd_scratch_bytes(f.M);
    if (need > 0 && f.scratch && f.scratch_bytes >= need && (reinterpret_cast<uintptr_t>(f.scratch) & 15u) == 0) {
        prm.split = 1;
        prm.work = static_cast<long long>(prm.m_tiles) * prm.nc;
        prm.part = static_cast<float *>(f.scratch);
        prm.part_cnt = reinterpret_cast<unsigned *>(static_cast<char *>(f.scratch) +
                                                    static_cast<size_t>(grid) * kEpiWarps * kPartF4 * sizeof(float4));
        s = cuda_check(cudaMemsetAsync(prm.part_cnt, 0, static_cast<size_t>(grid) * kEpiWarps * 2 * sizeof(unsigned), st),
                       "cudaMemsetAsync(fused split flags)");
        if (s != TP_OK) return s;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_on() ? 1 : 0;
    launch_begin("fused_mlp_fwd", st);
    cudaError_t e = prm.swiglu ? cudaLaunchKernelEx(&cfg, fused_mlp_fwd_kernel<true>, prm)
                               : cudaLaunchKernelEx(&cfg, fused_mlp_fwd_kernel<false>, prm);
    launch_end("fused_mlp_fwd", st);
    return cuda_check(e, "fused_mlp_fwd");
}

}  // namespace tpmlp
