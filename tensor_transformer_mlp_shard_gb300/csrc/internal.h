// Host-side internal interfaces of libtpmlp: the GEMM plan that the C-ABI
// layer builds for every product in the tensor-parallel MLP, and the launchers
// that execute a plan on the tcgen05 (bf16) or SIMT (fp32) kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/tp_mlp.h"

namespace tpmlp {

constexpr int kMaxShards = TP_MAX_SHARDS;

enum Fp8Format : int { FP8_E4M3 = 0, FP8_E5M2 = 1 };

// Epilogue kinds shared by both GEMM engines.
enum EpiKind : int {
    EPI_COL = 0,    // + bias, store pre, store act(pre)          (column forward)
    EPI_PLAIN = 1,  // + bias, + residual, store                   (row forward, dgrads)
    EPI_DACT = 2,   // * act'(pre) (SwiGLU: writes dG and dU)      (row-layer dgrad)
    EPI_F32 = 3     // store or accumulate fp32                    (weight gradients)
};

// One GEMM operand: a set of row-major buffers [rows, cols] with leading
// dimension `cols`.  K-major operands have the output's M (or N) dimension as
// rows and K as cols; MN-major operands have K as rows.  For problem p, K
// segment s and buffer row r the buffer used is
//   p * p_stride + s * s_stride + (rows_split ? r / rows_split : 0)
// at local row r % rows_split (token shards under sequence parallelism).
struct OperandPlan {
    const void *ptr[kMaxShards];
    int n = 0;
    int rows = 0, cols = 0;
    bool mn_major = false;
    int p_stride = 0, s_stride = 0, rows_split = 0;
};

// An output (or auxiliary input) addressed by problem and token row.
struct OutPlan {
    void *ptr[kMaxShards];
    int n = 0;
    int p_stride = 0, rows_split = 0;
    long long ld = 0;  // elements
};

// D_p[M, N] = sum_{s < S} A_{p,s}[M, Kseg] * B_{p,s}[N, Kseg]^T for p < P, then
// the epilogue.  For SwiGLU (act == TP_ACT_SWIGLU) N counts hidden units and
// the gate/up halves sit `N` columns apart in pre / dPre / bias.
struct GemmPlan {
    const char *name = "";
    int kind = EPI_PLAIN;
    int act = TP_ACT_NONE;
    int M = 0, N = 0, P = 1, S = 1, Kseg = 0;
    OperandPlan A, B;
    int b_dual_off = 0;   // column forward with SwiGLU: up rows start here in W1_i
    OutPlan out;          // main output
    OutPlan out2;         // pre (EPI_COL); n == 0 -> not stored
    OutPlan aux;          // residual (EPI_PLAIN) or pre (EPI_DACT); n == 0 -> none
    const void *bias[kMaxShards];
    int bias_p_stride = 0;
    bool has_bias = false;
    bool accumulate = false;  // EPI_F32
    // FP8 operands (1-byte elements): formats and per-tensor amax of A and B;
    // the epilogue scales the sum by 1 / (scale_a * scale_b)
    bool fp8 = false;
    int fmt_a = 0, fmt_b = 0;  // FP8_E4M3 / FP8_E5M2
    const float *amax_a = nullptr, *amax_b = nullptr;
    // Reductions fused into the bulk-store epilogue (tc_fused_epilogue(g)):
    // atomic max of |out| as bf16 (the FP8 amax of A / dPre; zero it first) and,
    // for EPI_DACT, column sums of out per 32-row block into
    // col_partials[P][ceil(M/32)][out.ld] (the db1 partials); for EPI_PLAIN
    // with aux, the same column sums of the residual (db2 from dY).
    float *amax_out = nullptr;
    float *col_partials = nullptr;
    // FP8 codes of the output written by the epilogue (tc_writes_fp8(g)):
    // q_out[p] [M, out.ld] bytes, scale fmax(q_fmt) / *q_scale_amax
    bool q = false;
    void *q_out[kMaxShards];
    int q_fmt = 0;
    const float *q_scale_amax = nullptr;
    // with q on an EPI_DACT plan: the codes are all that is kept, the bf16 out
    // is not stored (out's maps are still encoded and must be valid)
    bool q_only = false;
    // EPI_F32 split-K (S == 1): the token (K) range is split `ksplit` ways,
    // every split writes fp32 partial tiles into split_ws
    // ([ksplit][P][roundup(M, 256)][N]) and a reduction adds them in split
    // order into out (= or += with accumulate); ksplit = 1 or no split_ws: none
    int ksplit = 1;
    float *split_ws = nullptr;
    // Tail split of the CTA-pair kernel (EPI_PLAIN / EPI_F32 on the bulk-store
    // path, no split-K): scratch of tail_bytes at tail_ws (null: no split);
    // tc_tail_bytes gives what a shape may use
    void *tail_ws = nullptr;
    size_t tail_bytes = 0;
    // EPI_PLAIN: out = residual + dropout(acc + bias) (TransformerLayer bias-dropout-add);
    // drop_mask (or null): the keep flags, bit c % 32 of word row * ceil(N/32) + c / 32
    bool dropout = false;
    uint32_t drop_threshold = 0;
    float drop_scale = 1.0f;
    uint64_t drop_seed = 0;
    uint32_t *drop_mask = nullptr;
};

// out_p[m][n] (=, or += with accumulate) sum_{k < ksplit} part[k][p][m][n],
// part rows padded to split_rows per (k, p); fixed k order
tp_status launch_splitk_reduce(const float *part, int ksplit, int P, int M, int split_rows, int N,
                               float *const *out, bool accumulate, cudaStream_t st);

// Column sums over token rows: out_p[c] = sum_m in_p[m, c] for c < N, fp32.
struct ColsumPlan {
    const char *name = "";
    OutPlan in;      // P problems, token rows (may be token-sharded)
    int P = 1, M = 0, N = 0;
    float *out[kMaxShards];
    float *partials = nullptr;  // workspace: P * chunks * N floats
};

int colsum_chunks(int M);

// One buffer of a tensor to quantise to FP8: n bf16 elements (n % 8 == 0) at
// `in`, n codes written at `out`; `slot` indexes the tensor's amax in the
// amax array (all buffers of one tensor share a slot and hence a scale).
struct QuantSeg {
    const void *in = nullptr;
    void *out = nullptr;
    long long n = 0;
    int slot = 0;
    int fmt = 0;  // FP8_E4M3 / FP8_E5M2
};
constexpr int kMaxQuantSegs = 40;

// amax pass (slots optionally zeroed first) then quantise pass.
tp_status launch_fp8_quantize(const QuantSeg *segs, int nseg, float *amax, bool zero_slots, cudaStream_t st,
                              bool amax_known = false);

// One pass: out = fp8(in * scale), the scale from scale_amax[slot] (delayed
// scaling) or amax[slot]; with accumulate, |in| is also reduced into
// amax[slot] (zero it first).
tp_status launch_fp8_cast(const QuantSeg *segs, int nseg, float *amax, const float *scale_amax, bool accumulate,
                          cudaStream_t st);
// Amax history [slot][ld] of delayed scaling: prepare scale_amax for the
// slots (max of the first `fill` history entries, amax itself when fill is 0)
// or push amax into column pos.
tp_status launch_fp8_history(float *hist, int ld, float *scale_amax, const float *amax, const int *slots, int nslots,
                             int fill, int pos, bool push, cudaStream_t st);

// Launchers (return a tp_status).  They only enqueue work on `st`.
tp_status launch_tc_gemm(const GemmPlan &g, cudaStream_t st);
bool tc_fused_epilogue(const GemmPlan &g);  // true when amax_out / col_partials are honoured
bool tc_writes_fp8(const GemmPlan &g);      // true when q / q_out are honoured
void set_tile_mode(int mode);  // TP_TILE_*
// Tail split of the pair GEMMs on (default) or off, and an upper bound on the
// CTA pairs of their persistent grid (0: as many as fit)
void set_tail_split(bool on);
// K order of the pair GEMMs' whole tiles: every other persistent round walks
// K backwards (default) or every round forwards
void set_k_reverse(bool on);
// rows of pair tiles per raster band of the pair GEMMs' tile order (0: default)
void set_band_rows(int g);
void set_pdl(bool on);
bool pdl_on();  // kernels that take it are launched with programmatic dependent launch
void set_max_gemm_pairs(int n);
uint64_t tail_split_launches();  // pair GEMM launches that split their tail
// Scratch bytes a pair GEMM of this shape (out M x N per problem, P problems,
// K = S segments of Kseg) may use for its tail split at the current settings;
// 0 when it would not split
size_t tc_tail_bytes(int M, int N, int P, int S, int Kseg, bool fp8);
tp_status launch_simt_gemm(const GemmPlan &g, cudaStream_t st);
tp_status launch_colsum(const ColsumPlan &c, int dtype, cudaStream_t st);
// second pass only: out_p[c] = sum_{k < chunks} partials[p][k][c]
tp_status launch_colsum_finalize(const ColsumPlan &c, int chunks, cudaStream_t st);

// Fused MLP forward (one kernel for the column GEMM, the activation and the
// row GEMM; A passes through shared memory on its way to the row GEMM).
// Pointer arrays as in the MLP entry points: X, R, Y have n_tok token shards
// of rows_split rows (n_tok = 1, rows_split = 0 without sequence
// parallelism); W1, b1, W2, pre, A have T entries.
struct FusedPlan {
    const void *X[kMaxShards];
    const void *R[kMaxShards];  // residual (null entries: none)
    void *Y[kMaxShards];
    const void *W1[kMaxShards], *b1[kMaxShards], *W2[kMaxShards];
    const void *b2 = nullptr;
    void *pre[kMaxShards];      // null entries: not stored (act = none)
    void *A[kMaxShards];
    int n_tok = 1, rows_split = 0;
    int M = 0, H = 0, Fs = 0, T = 1, act = TP_ACT_NONE;
    bool has_bias = false, has_res = false, has_pre = false;
    bool dropout = false;  // as GemmPlan's dropout of the row forward
    uint32_t drop_threshold = 0;
    float drop_scale = 1.0f;
    uint64_t drop_seed = 0;
    uint32_t *drop_mask = nullptr;  // as GemmPlan's drop_mask (ceil(H/32) words per row)
    void *scratch = nullptr;        // the workspace's scratch: the even split of the work over the SMs
    size_t scratch_bytes = 0;       // runs only when it holds fused_fwd_scratch_bytes(M)
};
size_t fused_fwd_scratch_bytes(long long M);
void set_fused_fwd_mode(int mode);  // TP_FUSED_*
int fused_fwd_mode();
bool fused_fwd_supported(int H, int Fs, int act, int dtype);  // shapes the fused kernel takes
tp_status launch_fused_mlp_fwd(const FusedPlan &f, cudaStream_t st);

// LayerNorm and dropout-backward operands of the TransformerLayer MLP
// sub-block.  X, dY and dX are token-row tensors in `rows_split`-row shards
// (0: one buffer); Xn, dXn and dZ are single contiguous [M, H] buffers.
struct LnPlan {
    int M = 0, H = 0, rows_split = 0;
    float eps = 1e-5f;
    const void *x[kMaxShards];   // X (forward and backward)
    const void *dy[kMaxShards];  // dY (LayerNorm backward residual term, dropout backward input)
    void *dx[kMaxShards];        // LayerNorm backward output dX
    void *xn = nullptr;          // forward output Xn
    const void *dxn = nullptr;   // backward input: gradient of Xn
    void *dz = nullptr;          // dropout backward output
    const void *gamma = nullptr, *beta = nullptr;  // [H], activation dtype
    float *mean = nullptr, *rstd = nullptr;        // [M]
    float *partials = nullptr;   // LayerNorm backward: 2 * ln_bwd_chunks(M) * H floats (at most);
                                 // dropout backward: dropout_bwd_chunks(M) * H floats
    float *dgamma = nullptr, *dbeta = nullptr;     // [H] fp32
    float *db2 = nullptr;        // dropout backward: sum_m dZ ([H] fp32), or null
    uint32_t drop_threshold = 0;
    float drop_scale = 1.0f;
    uint64_t drop_seed = 0;
    // dropout backward: the forward's keep-mask (ceil(H/32) words per row), or
    // null to recompute the keep flags from the seed
    const uint32_t *drop_mask = nullptr;
};

int ln_bwd_chunks(int M);  // upper bound on the LayerNorm backward's blocks
int dropout_bwd_chunks(int M);
bool ln_supported(int H, int dtype);  // H within the LayerNorm kernels' row capacity
tp_status launch_ln_fwd(const LnPlan &p, int dtype, cudaStream_t st);
tp_status launch_ln_bwd(const LnPlan &p, int dtype, cudaStream_t st);
tp_status launch_dropout_bwd(const LnPlan &p, int dtype, cudaStream_t st);

// tp_linear_row_bwd with split-K optional (the allocation-free entry point
// runs it on a fixed scratch array that may not hold split partials), and the
// workspace it needs without splitting: the row layer's bias partials,
// 4 * ceil(M/256) * H bytes rounded up to 256 (0 without a bias or for an
// invalid descriptor).
tp_status linear_row_bwd_impl(const tp_mlp_desc *desc, const void *const *dY, const void *const *X,
                              const void *const *W, void *const *dX, void *const *dW, void *db, void *workspace,
                              size_t workspace_bytes, void *stream, bool allow_split);
size_t linear_row_bias_bytes(const tp_mlp_desc *desc);

// Device status words, the wait limit and the launch counter.  Status and
// abort words come in slots: slot 0 for the calls without a handle, one slot
// per live MLP / sub-block handle.  The entry points of a handle run under a
// StatusScope naming its slot, and every launch made on that thread in the
// meantime reports to that slot.
constexpr int kStatusSlots = 1024;
constexpr int kClockSlots = 32;  // kernel names with clock counters of their own
struct DeviceWords {
    int *status = nullptr;
    unsigned *abort_word = nullptr;
    unsigned long long *clk = nullptr;  // the kernel's clock counters (per-kernel timer on), or null
};
// words of the calling thread's current slot, and, with the per-kernel timer
// on and a kernel name given, that kernel's clock counters
tp_status device_words(DeviceWords *w, const char *kernel = nullptr);
int alloc_status_slot();                  // 1..kStatusSlots-1, or -1 when all are taken
void free_status_slot(int slot);
class StatusScope {
   public:
    explicit StatusScope(int slot);
    ~StatusScope();
    StatusScope(const StatusScope &) = delete;
    StatusScope &operator=(const StatusScope &) = delete;

   private:
    int prev_;
};
tp_status read_and_clear_status(cudaStream_t st, int slot, int *out);
// all kernels' clock counters (2 * kClockSlots values: cycles, ns per slot), then zeroed
tp_status read_and_clear_clocks(unsigned long long *v);
int prof_clock_slot(const char *kernel);  // clock slot of a kernel name, -1 with the timer off
tp_status launch_wait_timeout(unsigned long long limit_ns, cudaStream_t st);
bool prof_enabled();
uint64_t wait_limit_ns();
unsigned next_launch_id();
int num_sms();

// Profiling + launch accounting around every kernel launch.
void launch_begin(const char *name, cudaStream_t st);
void launch_end(const char *name, cudaStream_t st);

// Error message of the calling thread.
tp_status set_error(tp_status s, const char *fmt, ...);
tp_status cuda_check(cudaError_t e, const char *what);

}  // namespace tpmlp
