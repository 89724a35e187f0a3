// GEMM engine for sm_103a, host side: tensor maps, tiling choice, launch.
// The kernels live in tc_gemm_kernels.cuh; this unit instantiates the bf16
// ones and tc_gemm_fp8.cu the FP8 ones.  Every product of the tensor-parallel
// MLP runs on them:
//   column forward   pre_p = X W1_p^T (+b1_p), A_p = act(pre_p)      EPI_COL
//   row forward      Y = sum_s A_s W2_s^T (+b2) (+X)                EPI_PLAIN, S = T
//   row dgrad        dPre_p = (dY W2_p) * act'(pre_p)               EPI_DACT
//   column dgrad     dX = sum_s dPre_s W1_s (+dY)                   EPI_PLAIN, S = T
//   weight grads     dW = G^T Act (fp32, both operands MN-major)     EPI_F32
// The cross-shard sums (the forward and backward all-reduces of the
// multi-GPU layer) are the K loop over segments s: every shard's K range is
// accumulated into the same fp32 TMEM accumulator in shard order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "tc_gemm_kernels.cuh"

namespace tpmlp {
namespace tc {

typedef void (*KernelFn)(Params);
constexpr int kNumKernels = 6;
KernelFn fp8_kernel_at(int i, bool pair);  // tc_gemm_fp8.cu

// The five (epilogue, A major, B major) combinations the MLP uses, the
// weight gradient twice: plain, and with token-sharded operands (sequence
// parallelism), whose K loop crosses shards.
static int kernel_index(const GemmPlan &g) {
    const int kind = g.kind;
    const bool amn = g.A.mn_major, bmn = g.B.mn_major;
    if (kind == EPI_COL && !amn && !bmn) return 0;
    if (kind == EPI_PLAIN && !amn && !bmn) return 1;
    if (kind == EPI_PLAIN && !amn && bmn) return 2;
    if (kind == EPI_DACT && !amn && bmn) return 3;
    if (kind == EPI_F32 && amn && bmn) return g.A.rows_split || g.B.rows_split ? 5 : 4;
    return -1;
}

static KernelFn kernel_at(int i, bool pair, bool fp8) {
    if (fp8) return fp8_kernel_at(i, pair);
    switch (i) {
        case 0: return pair ? tc_gemm_pair_kernel<EPI_COL, false, false, false> : tc_gemm_kernel<EPI_COL, false, false, false>;
        case 1: return pair ? tc_gemm_pair_kernel<EPI_PLAIN, false, false, false> : tc_gemm_kernel<EPI_PLAIN, false, false, false>;
        case 2: return pair ? tc_gemm_pair_kernel<EPI_PLAIN, false, true, false> : tc_gemm_kernel<EPI_PLAIN, false, true, false>;
        case 3: return pair ? tc_gemm_pair_kernel<EPI_DACT, false, true, false> : tc_gemm_kernel<EPI_DACT, false, true, false>;
        case 4: return pair ? tc_gemm_pair_kernel<EPI_F32, true, true, false> : tc_gemm_kernel<EPI_F32, true, true, false>;
        case 5: return pair ? tc_gemm_pair_kernel<EPI_F32, true, true, false, true> : tc_gemm_kernel<EPI_F32, true, true, false>;
    }
    return nullptr;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2D tensor map of a row-major [rows, cols] buffer with leading dimension
// `ld` elements.
tp_status encode_map_ex(CUtensorMap *m, const void *ptr, int rows, int cols, long long ld, int box_inner,
                        int box_rows, CUtensorMapDataType type, int esize, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return set_error(TP_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, type, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%d x %d] box [%d x %d]", int(r),
                         rows, cols, box_rows, box_inner);
    return TP_OK;
}

// operand map: 1-byte (FP8) or 2-byte (bf16) elements, 128-byte swizzle
tp_status encode_map(CUtensorMap *m, const void *ptr, int rows, int cols, int box_inner, int box_rows, bool fp8) {
    return encode_map_ex(m, ptr, rows, cols, cols, box_inner, box_rows,
                         fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, fp8 ? 1 : 2,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

// bf16 operand [rows x cols], cols % 64 == 0, as the 3D tensor {64
// elements, rows, cols / 64 groups} with strides {row pitch, 128 bytes}: a
// box {64, box_rows, 2} lands as two [box_rows x 128 bytes] swizzle atoms,
// one after the other (the CTA-pair kernel's a3d/b3d).  MN-major [K x MN]:
// the two 64-wide MN atoms of a 128-wide tile, box_rows = the K elements of
// one stage; K-major [rows x K]: two consecutive K blocks of 128 rows.
static tp_status encode_map_mn3d(CUtensorMap *m, const void *ptr, int rows, int cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return set_error(TP_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for the 3D view of [%d x %d]", int(r),
                         rows, cols);
    return TP_OK;
}

// bulk-store map of an epilogue output: boxes of 32 rows x 64 bytes
// (32 bf16 or 16 fp32), 64-byte swizzle, matching the staging layout
static tp_status encode_out_maps(CUtensorMap *maps, const OutPlan &o, int rows, int cols, bool f32) {
    for (int i = 0; i < o.n; ++i) {
        tp_status s = encode_map_ex(&maps[i], o.ptr[i], rows, cols, o.ld, f32 ? 16 : 32, 32,
                                    f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                    f32 ? 4 : 2, CU_TENSOR_MAP_SWIZZLE_64B);
        if (s != TP_OK) return s;
    }
    return TP_OK;
}

static void copy_out(Out &o, const OutPlan &src) {
    for (int i = 0; i < kMaxShards; ++i) o.ptr[i] = i < src.n ? src.ptr[i] : nullptr;
    o.p_stride = src.p_stride;
    o.rows_split = src.rows_split;
    o.nsplit = src.n;
    o.ld = src.ld;
}

static std::atomic<int> g_tile_mode{0};
static std::atomic<bool> g_tail_split{true};
static std::atomic<bool> g_k_reverse{true};
static std::atomic<int> g_band_rows{0};
static std::atomic<int> g_max_pairs{0};
static std::atomic<bool> g_pdl{true};
static std::atomic<uint64_t> g_tail_launches{0};

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Persistent round structure: `total` tiles over `pairs` CTA pairs leave
// rem = total % pairs tiles for a last, part-filled round.  When rem is at
// most half the pairs, each of those tiles is cut along K into
// s = min(pairs / rem, 4) units (each at least 4 of the nk K blocks of
// 128-byte rows; a stage may hold two), which
// all run in one round of 1/s of a tile's time.  Measured on GB300: with a
// single round of units the split pays (the GPT-size weight gradients, 36
// tiles over 76 pairs, 1.3% faster); spreading a fuller last round over
// several rounds of units does not (56 tiles as 3 rounds of quarter tiles:
// 1.3% slower, the units of a round sharing fewer operand panels in L2 than
// whole tiles do).  Only grids with at least one full round split (smaller
// problems keep their results bit for bit with the whole-tile path).
struct TailPlan {
    int s = 0, rem = 0;
    size_t slices = 0, bytes = 0;
};
static TailPlan tail_plan(int total, int pairs, int nk) {
    TailPlan r;
    if (!g_tail_split.load() || pairs <= 0 || total <= pairs) return r;
    const int rem = total % pairs;
    if (rem == 0) return r;
    const int s = std::min(std::min(pairs / rem, 4), nk / 4);
    if (s < 2) return r;
    r.s = s;
    r.rem = rem;
    r.slices = sizeof(float) * static_cast<size_t>(rem) * s * P_TILE_M * BN;
    r.bytes = r.slices + align256(sizeof(unsigned) * 16 * static_cast<size_t>(rem));
    return r;
}

static int pair_limit(int fit) {
    const int lim = g_max_pairs.load();
    return lim > 0 && lim < fit ? lim : fit;
}

}  // namespace tc

void set_tile_mode(int mode) { tc::g_tile_mode.store(mode); }
void set_tail_split(bool on) { tc::g_tail_split.store(on); }
void set_k_reverse(bool on) { tc::g_k_reverse.store(on); }
void set_band_rows(int g) { tc::g_band_rows.store(g > 0 ? g : 0); }
void set_max_gemm_pairs(int n) { tc::g_max_pairs.store(n > 0 ? n : 0); }
void set_pdl(bool on) { tc::g_pdl.store(on); }
bool pdl_on() { return tc::g_pdl.load(); }
uint64_t tail_split_launches() { return tc::g_tail_launches.load(); }

size_t tc_tail_bytes(int M, int N, int P, int S, int Kseg, bool fp8) {
    using namespace tc;
    const int mode = g_tile_mode.load();
    if (M <= BM || mode == TP_TILE_SINGLE || M <= 0 || N <= 0 || P <= 0 || S <= 0 || Kseg <= 0) return 0;
    const int bke = fp8 ? Elem<true>::BKE : Elem<false>::BKE;
    const long long total = static_cast<long long>((M + P_TILE_M - 1) / P_TILE_M) * ((N + BN - 1) / BN) * P;
    if (total > (1LL << 30)) return 0;
    const int nk = S * ((Kseg + bke - 1) / bke);
    return tail_plan(static_cast<int>(total), pair_limit(num_sms() / 2), nk).bytes;
}

bool tc_fused_epilogue(const GemmPlan &g) { return !g.accumulate && !(g.act == TP_ACT_SWIGLU && g.N % 32); }

// FP8 codes from the epilogue: the column forward and the GeLU dgrad on the
// bulk-store path (not SwiGLU, whose epilogues produce two halves per tile)
bool tc_writes_fp8(const GemmPlan &g) {
    return tc_fused_epilogue(g) && g.act != TP_ACT_SWIGLU &&
           (g.kind == EPI_COL || (g.kind == EPI_DACT && g.act == TP_ACT_GELU_TANH));
}

tp_status launch_tc_gemm(const GemmPlan &g, cudaStream_t st) {
    using namespace tc;
    const int ki = kernel_index(g);
    if (ki < 0)
        return set_error(TP_ERR_UNSUPPORTED, "no tcgen05 kernel for epilogue %d / majors %d%d", g.kind,
                         int(g.A.mn_major), int(g.B.mn_major));
    // CTA pairs (256-row tiles) unless single-CTA tiles are requested or the
    // problem has a single 128-row tile.
    const int mode = g_tile_mode.load();
    const bool use_pair = mode == TP_TILE_PAIR || (mode == TP_TILE_AUTO && g.M > BM);
    const bool fp8 = g.fp8;
    // the pair kernels take an MN-major operand's K rows as the row itself
    // except in the token-sharded instance (index 5)
    if (use_pair && ki != 5 && ((g.A.mn_major && g.A.rows_split) || (g.B.mn_major && g.B.rows_split)))
        return set_error(TP_ERR_UNSUPPORTED, "token-sharded MN-major operand outside the token-sharded GEMM instance");
    KernelFn fn = kernel_at(ki, use_pair, fp8);
    // K elements per stage: one 128-byte row of each operand, two for the
    // pair kernel's bf16 GEMMs (tc_gemm_pair_kernel's KB2)
    static_assert(pair_kb2<EPI_COL, false>() == 2 && pair_kb2<EPI_PLAIN, false>() == 2 &&
                      pair_kb2<EPI_DACT, false>() == 2 && pair_kb2<EPI_F32, false>() == 2 &&
                      pair_kb2<EPI_COL, true>() == 1 && pair_kb2<EPI_PLAIN, true>() == 1 &&
                      pair_kb2<EPI_DACT, true>() == 1 && pair_kb2<EPI_F32, true>() == 1,
                  "the host's K blocks per stage match the kernels'");
    const int kb2 = use_pair && !fp8 ? 2 : 1;
    const int bke1 = fp8 ? Elem<true>::BKE : Elem<false>::BKE;  // K elements of one 128-byte row
    const int bke = bke1 * kb2;
    const int mnb = fp8 ? Elem<true>::MNB : Elem<false>::MNB;  // MN elements per MN-major box
    const int tile_m = use_pair ? P_TILE_M : BM;
    // rows of the B tile that one CTA loads per box
    const int b_box_rows = (use_pair || g.b_dual_off) ? BN / 2 : BN;
    Params prm;
    memset(&prm, 0, sizeof(prm));
    // one 3D box instead of two 2D boxes per operand and stage (pair kernel,
    // bf16): an MN-major operand's two 64-wide atoms (the weight gradients
    // run 11% faster, GB300, GPT sizes), or a K-major operand's two K blocks
    // when a stage holds two (both need the extent along the box groups to
    // be a multiple of 64)
    prm.a3d = use_pair && !fp8 && g.A.cols % 64 == 0 && (g.A.mn_major || kb2 == 2);
    prm.b3d = use_pair && !fp8 && g.B.cols % 64 == 0 && (g.B.mn_major ? !g.b_dual_off : kb2 == 2);
    for (int i = 0; i < g.A.n; ++i) {
        tp_status s = prm.a3d ? encode_map_mn3d(&prm.mapA[i], g.A.ptr[i], g.A.rows, g.A.cols, g.A.mn_major ? bke : BM)
                      : g.A.mn_major ? encode_map(&prm.mapA[i], g.A.ptr[i], g.A.rows, g.A.cols, mnb, bke, fp8)
                                     : encode_map(&prm.mapA[i], g.A.ptr[i], g.A.rows, g.A.cols, bke1, BM, fp8);
        if (s != TP_OK) return s;
    }
    for (int i = 0; i < g.B.n; ++i) {
        tp_status s =
            prm.b3d ? encode_map_mn3d(&prm.mapB[i], g.B.ptr[i], g.B.rows, g.B.cols, g.B.mn_major ? bke : b_box_rows)
            : g.B.mn_major ? encode_map(&prm.mapB[i], g.B.ptr[i], g.B.rows, g.B.cols, mnb, bke, fp8)
                           : encode_map(&prm.mapB[i], g.B.ptr[i], g.B.rows, g.B.cols, bke1, b_box_rows, fp8);
        if (s != TP_OK) return s;
    }
    prm.selA = {g.A.p_stride, g.A.s_stride, g.A.rows_split, g.A.n};
    prm.selB = {g.B.p_stride, g.B.s_stride, g.B.rows_split, g.B.n};
    copy_out(prm.out, g.out);
    copy_out(prm.out2, g.out2);
    copy_out(prm.aux, g.aux);
    for (int i = 0; i < kMaxShards; ++i) prm.bias[i] = g.has_bias ? g.bias[i] : nullptr;
    prm.bias_p_stride = g.bias_p_stride;
    prm.has_bias = g.has_bias ? 1 : 0;
    prm.has_out2 = g.out2.n > 0;
    prm.has_aux = g.aux.n > 0;
    prm.M = g.M;
    prm.N = g.N;
    prm.P = g.P;
    prm.S = g.S;
    prm.Kseg = g.Kseg;
    prm.num_kb = (g.Kseg + bke - 1) / bke;
    prm.m_tiles = (g.M + tile_m - 1) / tile_m;
    const int n_per_tile = g.b_dual_off ? BN / 2 : BN;
    prm.n_tiles = (g.N + n_per_tile - 1) / n_per_tile;
    prm.tiles_per_split = prm.m_tiles * prm.n_tiles * g.P;
    // split-K: every split gets at least one K block
    const bool split = g.kind == EPI_F32 && g.S == 1 && g.ksplit > 1 && g.split_ws && prm.num_kb > 1;
    prm.kb_split = split ? (prm.num_kb + g.ksplit - 1) / g.ksplit : prm.num_kb;
    const int ksplit = split ? (prm.num_kb + prm.kb_split - 1) / prm.kb_split : 1;
    prm.split_rows = split ? prm.m_tiles * tile_m : 0;
    prm.total_tiles = prm.tiles_per_split * ksplit;
    prm.total_work = prm.total_tiles;
    prm.tail_first = prm.total_tiles;
    // bands of 16 pair-tile rows: measured on GB300 against 2, 4, 8, 32 and
    // 64 (GPT, SwiGLU and sequence-parallel workloads), the fastest or
    // within 0.5% of it for every GEMM, with the least DRAM traffic overall
    prm.group_m = use_pair ? (g_band_rows.load() > 0 ? g_band_rows.load() : 16) : 16;
    // alternate-round K order for the GEMMs whose operands are re-read most
    // (row forward, column dgrad, weight gradients); the column forward and
    // the act' dgrad keep one order (their results are compared bit for bit
    // with the fused forward kernel and across calls of different shapes)
    prm.k_reverse = use_pair && g_k_reverse.load() && (g.kind == EPI_PLAIN || g.kind == EPI_F32) ? 1 : 0;
    prm.act = g.act;
    prm.b_dual_off = g.b_dual_off;
    prm.accumulate = (g.accumulate && !split) ? 1 : 0;  // split-K: the reduction accumulates
    // instruction descriptor: fp32 accumulator (bit 4), A/B formats (bits 7-9,
    // 10-12: bf16 = 1 for kind::f16; E4M3 = 0, E5M2 = 1 for kind::f8f6f4),
    // A/B MN-major (bits 15, 16), N/8 at bit 17, M/16 at bit 24
    const uint32_t fa = fp8 ? uint32_t(g.fmt_a) : 1u, fb = fp8 ? uint32_t(g.fmt_b) : 1u;
    prm.idesc = (1u << 4) | (fa << 7) | (fb << 10) | (uint32_t(g.A.mn_major) << 15) |
                (uint32_t(g.B.mn_major) << 16) | (uint32_t(BN >> 3) << 17) | (uint32_t(tile_m >> 4) << 24);
    // Epilogue outputs go through shared memory and bulk tensor stores (for
    // dW accumulation, bulk reduce-add stores), except for SwiGLU with a unit
    // count that is not a multiple of 32 (a 32-column gate block would reach
    // into the up half of pre / dPre, which a store clipped at the buffer's
    // width cannot prevent).
    prm.out_tma = (tc_fused_epilogue(g) || split || (g.kind == EPI_F32 && g.accumulate)) ? 1 : 0;
    if (split) {
        // partial sums [ksplit][P][split_rows][N] fp32 in the caller's workspace
        Out &o = prm.out;
        memset(&o, 0, sizeof(o));
        o.ptr[0] = g.split_ws;
        o.nsplit = 1;
        o.ld = g.N;
        tp_status s = encode_map_ex(&prm.mapO[0], g.split_ws, ksplit * g.P * prm.split_rows, g.N, g.N, 16, 32,
                                    CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_64B);
        if (s != TP_OK) return s;
    } else if (prm.out_tma) {
        const bool f32 = g.kind == EPI_F32;
        // columns of a whole output row: pre / dPre hold both SwiGLU halves
        const int ocols = static_cast<int>(g.out.ld);
        const int orows = g.out.rows_split ? g.out.rows_split : g.M;
        tp_status s = encode_out_maps(prm.mapO, g.out, orows, ocols, f32);
        if (s != TP_OK) return s;
        if (g.out2.n) {
            s = encode_out_maps(prm.mapO2, g.out2, g.out2.rows_split ? g.out2.rows_split : g.M,
                                static_cast<int>(g.out2.ld), false);
            if (s != TP_OK) return s;
        }
        if (g.q && tc_writes_fp8(g)) {
            for (int i = 0; i < g.out.n; ++i) {
                s = encode_map_ex(&prm.mapQ[i], g.q_out[i], orows, ocols, g.out.ld, 32, 32,
                                  CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
                if (s != TP_OK) return s;
            }
            prm.q_out = 1;
            prm.q_fmt = g.q_fmt;
            prm.q_scale_amax = g.q_scale_amax;
            prm.q_only = g.q_only && g.kind == EPI_DACT ? 1 : 0;
        }
    }
    prm.drop.on = g.dropout ? 1 : 0;
    prm.drop.threshold = g.drop_threshold;
    prm.drop.scale = g.drop_scale;
    prm.drop.seed_lo = static_cast<uint32_t>(g.drop_seed);
    prm.drop.seed_hi = static_cast<uint32_t>(g.drop_seed >> 32);
    prm.drop.ld = g.N;
    prm.drop.mask = g.dropout ? g.drop_mask : nullptr;
    prm.drop.mask_ld = (g.N + 31) / 32;
    if (prm.drop.mask && !prm.out_tma)
        return set_error(TP_ERR_UNSUPPORTED, "dropout keep-mask output needs the bulk-store epilogue");
    prm.amax_out = prm.out_tma ? g.amax_out : nullptr;
    prm.col_partials =
        prm.out_tma && (g.kind == EPI_DACT || (g.kind == EPI_PLAIN && g.aux.n > 0)) ? g.col_partials : nullptr;
    prm.partial_ld = static_cast<int>(g.out.ld);
    prm.amax_a = fp8 ? g.amax_a : nullptr;
    prm.amax_b = fp8 ? g.amax_b : nullptr;
    prm.fmax_a = g.fmt_a == FP8_E5M2 ? 57344.0f : 448.0f;
    prm.fmax_b = g.fmt_b == FP8_E5M2 ? 57344.0f : 448.0f;
    DeviceWords w;
    tp_status s = device_words(&w, g.name);
    if (s != TP_OK) return s;
    prm.status = w.status;
    prm.abort_word = w.abort_word;
    prm.clk = w.clk;
    prm.launch_id = next_launch_id();
    prm.wait_limit_ns = wait_limit_ns();
    if (prm.total_tiles == 0 || prm.num_kb == 0) return TP_OK;

    // opt in to > 48 KB of dynamic shared memory and size the persistent
    // grid, once per kernel and device
    static std::mutex mu;
    static bool attr_set[64][2][2][kNumKernels] = {};
    static int max_pairs[64][2][kNumKernels] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const int smem_bytes = !use_pair              ? SMEM_BYTES
                           : g.kind != EPI_DACT ? (fp8 ? pair_smem_total<EPI_PLAIN, true>() : pair_smem_total<EPI_PLAIN, false>())
                           : fp8                ? pair_smem_total<EPI_DACT, true>()
                                                : pair_smem_total<EPI_DACT, false>();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev % 64][fp8][use_pair][ki]) {
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
            if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute");
            if (use_pair) {
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
                (void)e;
                cudaLaunchConfig_t cfg = {};
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 2;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
                cfg.blockDim = dim3(NUM_THREADS, 1, 1);
                cfg.dynamicSmemBytes = smem_bytes;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int n = 0;
                e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
                if (e != cudaSuccess || n <= 0) {
                    cudaGetLastError();
                    n = num_sms() / 2;
                }
                max_pairs[dev % 64][fp8][ki] = n;
            }
            attr_set[dev % 64][fp8][use_pair][ki] = true;
        }
    }
    cudaError_t e;
    const int pairs = std::min(prm.total_tiles, pair_limit(max_pairs[dev % 64][fp8][ki]));
    if (use_pair && prm.out_tma && !split && (g.kind == EPI_PLAIN || g.kind == EPI_F32) && g.tail_ws) {
        const TailPlan tp = tail_plan(prm.total_tiles, pairs, g.S * prm.num_kb * kb2);
        if (tp.s > 1 && tp.bytes <= g.tail_bytes && (reinterpret_cast<uintptr_t>(g.tail_ws) & 255u) == 0) {
            prm.tail_s = tp.s;
            prm.tail_first = prm.total_tiles - tp.rem;
            prm.total_work = prm.tail_first + tp.rem * tp.s;
            prm.tail_ws = static_cast<float *>(g.tail_ws);
            prm.tail_cnt = reinterpret_cast<unsigned *>(static_cast<char *>(g.tail_ws) + tp.slices);
            e = cudaMemsetAsync(prm.tail_cnt, 0, sizeof(unsigned) * 16 * static_cast<size_t>(tp.rem), st);
            if (e != cudaSuccess) return cuda_check(e, "cudaMemsetAsync(tail counters)");
            g_tail_launches.fetch_add(1);
        }
    }
    launch_begin(g.name, st);
    if (use_pair) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        // programmatic dependent launch: the pairs' set-up (barriers, TMEM)
        // overlaps the previous kernel, and the kernel waits for it in
        // griddepcontrol.wait before it touches global memory
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(2 * pairs, 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = g_pdl.load() ? 2 : 1;
        e = cudaLaunchKernelEx(&cfg, fn, prm);
    } else {
        const int grid = prm.total_tiles < num_sms() ? prm.total_tiles : num_sms();
        fn<<<grid, NUM_THREADS, smem_bytes, st>>>(prm);
        e = cudaGetLastError();
    }
    launch_end(g.name, st);
    if (e != cudaSuccess || !split) return cuda_check(e, g.name);
    float *outs[kMaxShards];
    for (int i = 0; i < kMaxShards; ++i) outs[i] = i < g.P ? static_cast<float *>(g.out.ptr[i * g.out.p_stride]) : nullptr;
    return launch_splitk_reduce(g.split_ws, ksplit, g.P, g.M, prm.split_rows, g.N, outs, g.accumulate, st);
}

}  // namespace tpmlp
