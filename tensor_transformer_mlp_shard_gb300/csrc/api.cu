// C-ABI of libtpmlp: argument validation, the GEMM plans of every
// tensor-parallel product, dispatch to the bf16 (tcgen05) or fp32 (SIMT)
// engine, device status, launch accounting and per-kernel timing.
//
// Mapping from the multi-GPU layers to single-GPU plans ("Megatron-LM 源码精读"
// s3.1-s3.5):
//   ColumnParallelLinear forward: T independent problems (no communication);
//   RowParallelLinear forward:    one problem whose K loop runs over the T
//                                 shards (the all-reduce as an fp32 sum);
//   ColumnParallelLinear dgrad:   the same K loop over shards (the backward
//                                 all-reduce);
//   RowParallelLinear dgrad:      T independent problems;
//   sequence parallelism:         token-sharded buffers selected per row
//                                 (all-gather / reduce-scatter as addressing).
#include <cuda_runtime.h>

#include <atomic>
#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

struct tp_mlp {
    tp_mlp_desc d;
    int status_slot = 0;  // this handle's device status word (see StatusScope)
    int fp8_history = 0;  // 0: current scaling; n: delayed scaling over the last n amaxes
    long long fp8_fwd_steps = 0, fp8_bwd_steps = 0;  // quantisations since the history was set
};

struct tp_layer {
    tp_layer_desc d;
    int status_slot = 0;  // as tp_mlp
    tp_mlp_desc inner;  // the MLP inside the sub-block: d.mlp with the residual handled by the block
    uint32_t drop_threshold;
    float drop_scale;
    int fp8_history = 0;  // as tp_mlp
    long long fp8_fwd_steps = 0, fp8_bwd_steps = 0;
    // workspaces whose keep-mask region a forward of this handle filled, with
    // the seed it used (the mask is a function of the seed, p and the shape)
    std::map<const void *, uint64_t> masks;
};

namespace tpmlp {

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
static thread_local char g_err[512] = "";

tp_status set_error(tp_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

tp_status cuda_check(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return TP_OK;
    return set_error(TP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------
// runtime state
// ---------------------------------------------------------------------------
static std::atomic<uint64_t> g_launches{0};
static std::atomic<unsigned> g_launch_id{0};
static std::atomic<uint64_t> g_wait_limit{4000000000ull};

uint64_t wait_limit_ns() { return g_wait_limit.load(); }

unsigned next_launch_id() {
    unsigned id = ++g_launch_id;
    if (id == 0) id = ++g_launch_id;  // 0 never names a launch
    return id;
}

int num_sms() {
    static int cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    int &c = cache[dev % 64];
    if (c == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        c = n;
    }
    return c;
}

// per-kernel timing
struct ProfRec {
    std::string name;
    cudaEvent_t a, b;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::string g_prof_only;  // non-empty: only launches of this kernel get events
static std::vector<ProfRec> g_prof_recs;
static std::vector<cudaEvent_t> g_event_pool;
static thread_local cudaEvent_t g_pending = nullptr;

bool prof_enabled() {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    return g_prof_on;
}

// clock counter slot per kernel name (the last slot is shared by any names
// beyond the first kClockSlots - 1)
static std::vector<std::string> g_clock_names;

int prof_clock_slot(const char *kernel) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (!g_prof_on) return -1;
    for (size_t i = 0; i < g_clock_names.size(); ++i)
        if (g_clock_names[i] == kernel) return static_cast<int>(i);
    if (static_cast<int>(g_clock_names.size()) < kClockSlots - 1) {
        g_clock_names.push_back(kernel);
        return static_cast<int>(g_clock_names.size()) - 1;
    }
    return kClockSlots - 1;
}

static cudaEvent_t get_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void launch_begin(const char *name, cudaStream_t st) {
    g_launches.fetch_add(1);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_pending = nullptr;
    if (!g_prof_on || (!g_prof_only.empty() && g_prof_only != name)) return;
    cudaEvent_t e = get_event();
    if (e && cudaEventRecord(e, st) == cudaSuccess) g_pending = e;
}

void launch_end(const char *name, cudaStream_t st) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (!g_prof_on || !g_pending) return;
    cudaEvent_t e = get_event();
    if (e && cudaEventRecord(e, st) == cudaSuccess) g_prof_recs.push_back({name, g_pending, e});
    g_pending = nullptr;
}

// ---------------------------------------------------------------------------
// validation helpers
// ---------------------------------------------------------------------------
static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static tp_status check_array(const void *const *arr, int n, const char *name) {
    if (!arr) return set_error(TP_ERR_ARG, "%s: pointer array is NULL", name);
    for (int i = 0; i < n; ++i) {
        if (!arr[i]) return set_error(TP_ERR_ARG, "%s[%d] is NULL", name, i);
        if (!aligned16(arr[i])) return set_error(TP_ERR_ARG, "%s[%d] is not 16-byte aligned", name, i);
    }
    return TP_OK;
}

static tp_status check_one(const void *p, const char *name) {
    if (!p) return set_error(TP_ERR_ARG, "%s is NULL", name);
    if (!aligned16(p)) return set_error(TP_ERR_ARG, "%s is not 16-byte aligned", name);
    return TP_OK;
}

#define TRY(x)                        \
    do {                              \
        tp_status _s = (x);           \
        if (_s != TP_OK) return _s;   \
    } while (0)

static tp_status validate_desc(const tp_mlp_desc *d) {
    if (!d) return set_error(TP_ERR_ARG, "descriptor is NULL");
    if (d->act < TP_ACT_NONE || d->act > TP_ACT_SWIGLU) return set_error(TP_ERR_ARG, "bad act %d", d->act);
    if (d->dtype != TP_DT_F32 && d->dtype != TP_DT_BF16 && d->dtype != TP_DT_FP8)
        return set_error(TP_ERR_ARG, "bad dtype %d", d->dtype);
    const int flags[4] = {d->has_bias, d->residual, d->seq_parallel, d->wgrad_accumulate};
    for (int f : flags)
        if (f != 0 && f != 1) return set_error(TP_ERR_ARG, "boolean flags must be 0 or 1");
    if (d->T < 1 || d->T > TP_MAX_SHARDS)
        return set_error(TP_ERR_SHAPE, "T=%d outside 1..%d", d->T, TP_MAX_SHARDS);
    if (d->S < 0 || d->B < 0) return set_error(TP_ERR_SHAPE, "negative S or B");
    const long long M = static_cast<long long>(d->S) * d->B;
    if (M > (1ll << 24)) return set_error(TP_ERR_SHAPE, "M = S*B = %lld exceeds 2^24 tokens", M);
    if (d->H < 8 || d->H % 8) return set_error(TP_ERR_SHAPE, "H=%d must be a positive multiple of 8", d->H);
    if (d->F < 1 || d->F % d->T)
        return set_error(TP_ERR_SHAPE, "F=%d is not divisible by T=%d (divide(output_size, world_size))", d->F,
                         d->T);
    const int Fs = d->F / d->T;
    if (Fs % 8) return set_error(TP_ERR_SHAPE, "F/T=%d must be a multiple of 8", Fs);
    if (d->H > (1 << 20) || Fs > (1 << 20)) return set_error(TP_ERR_SHAPE, "width above 2^20");
    if (d->dtype == TP_DT_FP8 && (d->H % 16 || Fs % 16))
        return set_error(TP_ERR_SHAPE, "FP8 needs H and F/T to be multiples of 16 (H=%d, F/T=%d)", d->H, Fs);
    if (d->seq_parallel) {
        if (d->S % d->T) return set_error(TP_ERR_SHAPE, "sequence parallel needs S %% T == 0 (S=%d, T=%d)", d->S, d->T);
        if (d->dtype == TP_DT_BF16 && M > 0 && (M / d->T) % 128)
            return set_error(TP_ERR_SHAPE, "bf16 sequence parallel needs M/T %% 128 == 0 (M/T=%lld)", M / d->T);
    }
    return TP_OK;
}

struct Dims {
    int M, H, Fs, T, g, nx, rs;
    size_t es;
};

static Dims dims_of(const tp_mlp_desc *d) {
    Dims x;
    x.M = d->S * d->B;
    x.H = d->H;
    x.T = d->T;
    x.Fs = d->F / d->T;
    x.g = d->act == TP_ACT_SWIGLU ? 2 : 1;
    x.nx = d->seq_parallel ? d->T : 1;
    x.rs = d->seq_parallel ? x.M / d->T : 0;
    x.es = d->dtype == TP_DT_F32 ? 4 : 2;  // FP8 keeps bf16 buffers at the interface
    return x;
}

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Scratch of a GEMM's tail split (null: the GEMM does not split its tail)
struct Scratch {
    void *p = nullptr;
    size_t n = 0;
};
static void set_tail(GemmPlan &g, Scratch t) {
    g.tail_ws = t.p;
    g.tail_bytes = t.p ? t.n : 0;
}

static tp_status run_gemm(const GemmPlan &g, int dtype, cudaStream_t st) {
    return dtype == TP_DT_F32 ? launch_simt_gemm(g, st) : launch_tc_gemm(g, st);
}

// plan helpers --------------------------------------------------------------
static void set_operand(OperandPlan &o, const void *const *ptrs, int n, int rows, int cols, bool mn, int p_stride,
                        int s_stride, int rows_split) {
    for (int i = 0; i < kMaxShards; ++i) o.ptr[i] = i < n ? ptrs[i] : nullptr;
    o.n = n;
    o.rows = rows;
    o.cols = cols;
    o.mn_major = mn;
    o.p_stride = p_stride;
    o.s_stride = s_stride;
    o.rows_split = rows_split;
}

static void set_out(OutPlan &o, const void *const *ptrs, int n, int p_stride, int rows_split, long long ld) {
    for (int i = 0; i < kMaxShards; ++i) o.ptr[i] = i < n ? const_cast<void *>(ptrs[i]) : nullptr;
    o.n = n;
    o.p_stride = p_stride;
    o.rows_split = rows_split;
    o.ld = ld;
}

static void set_bias(GemmPlan &g, const void *const *b, int n, int p_stride) {
    g.has_bias = b != nullptr;
    for (int i = 0; i < kMaxShards; ++i) g.bias[i] = (b && i < n) ? b[i] : nullptr;
    g.bias_p_stride = p_stride;
}

// Column forward: out_i = act(X W_i^T + b_i), i < T (no reduction).
static tp_status column_fwd(const tp_mlp_desc *d, const void *const *X, const void *const *W,
                            const void *const *b, void *const *out, void *const *pre, cudaStream_t st) {
    const Dims x = dims_of(d);
    GemmPlan g;
    g.name = "col_fwd";
    g.kind = EPI_COL;
    g.act = d->act;
    g.M = x.M;
    g.N = x.Fs;
    g.P = x.T;
    g.S = 1;
    g.Kseg = x.H;
    set_operand(g.A, X, x.nx, x.rs ? x.rs : x.M, x.H, false, 0, 0, x.rs);
    set_operand(g.B, W, x.T, x.g * x.Fs, x.H, false, 1, 0, 0);
    g.b_dual_off = d->act == TP_ACT_SWIGLU ? x.Fs : 0;
    set_out(g.out, reinterpret_cast<const void *const *>(out), x.T, 1, 0, x.Fs);
    if (pre) set_out(g.out2, reinterpret_cast<const void *const *>(pre), x.T, 1, 0, (long long)x.g * x.Fs);
    set_bias(g, d->has_bias ? b : nullptr, x.T, 1);
    return run_gemm(g, d->dtype, st);
}

// Dropout of the row forward's output (TransformerLayer bias-dropout-add):
// Y = R + dropout(sum + b), element m*H + h drawn from Philox4x32-10 under `seed`.
struct DropCfg {
    bool on = false;
    uint32_t threshold = 0;  // floor(p * 2^24)
    float scale = 1.0f;      // 1 / (1 - p)
    uint64_t seed = 0;
    uint32_t *mask = nullptr;  // keep-mask output (ceil(H/32) words per token row), or null
};

static void set_drop(GemmPlan &g, const DropCfg *dc) {
    if (!dc || !dc->on) return;
    g.dropout = true;
    g.drop_threshold = dc->threshold;
    g.drop_scale = dc->scale;
    g.drop_seed = dc->seed;
    g.drop_mask = dc->mask;
}

// Row forward: Y = sum_i X_i W_i^T + b (+R); the K loop runs over shards.
static tp_status row_fwd(const tp_mlp_desc *d, const void *const *Xs, const void *const *W, const void *b,
                         const void *const *R, void *const *Y, cudaStream_t st, const DropCfg *drop = nullptr,
                         Scratch tail = {}) {
    const Dims x = dims_of(d);
    GemmPlan g;
    g.name = "row_fwd";
    g.kind = EPI_PLAIN;
    g.M = x.M;
    g.N = x.H;
    g.P = 1;
    g.S = x.T;
    g.Kseg = x.Fs;
    set_operand(g.A, Xs, x.T, x.M, x.Fs, false, 0, 1, 0);
    set_operand(g.B, W, x.T, x.H, x.Fs, false, 0, 1, 0);
    set_out(g.out, reinterpret_cast<const void *const *>(Y), x.nx, 0, x.rs, x.H);
    if (R) set_out(g.aux, R, x.nx, 0, x.rs, x.H);
    const void *bb[1] = {b};
    set_bias(g, (d->has_bias && b) ? bb : nullptr, 1, 0);
    set_drop(g, drop);
    set_tail(g, tail);
    return run_gemm(g, d->dtype, st);
}

// Row-layer dgrad: dOut_i = (dY W_i) [* act'(pre_i)], i < T (no reduction).
static tp_status row_dgrad(const tp_mlp_desc *d, int act, const void *const *dY, const void *const *W,
                           const void *const *pre, void *const *dOut, long long ld_out, cudaStream_t st,
                           float *col_partials = nullptr, bool *fused = nullptr, Scratch tail = {}) {
    const Dims x = dims_of(d);
    GemmPlan g;
    g.name = act == TP_ACT_NONE ? "row_dgrad" : "row_dgrad_act";
    g.kind = act == TP_ACT_NONE ? EPI_PLAIN : EPI_DACT;
    g.act = act;
    g.M = x.M;
    g.N = x.Fs;
    g.P = x.T;
    g.S = 1;
    g.Kseg = x.H;
    set_operand(g.A, dY, x.nx, x.rs ? x.rs : x.M, x.H, false, 0, 0, x.rs);
    set_operand(g.B, W, x.T, x.H, x.Fs, true, 1, 0, 0);
    set_out(g.out, reinterpret_cast<const void *const *>(dOut), x.T, 1, 0, ld_out);
    if (act != TP_ACT_NONE) set_out(g.aux, pre, x.T, 1, 0, ld_out);
    // db1 column sums fused into the bf16 epilogue when it can take them
    const bool fuse = col_partials && act != TP_ACT_NONE && d->dtype != TP_DT_F32 && tc_fused_epilogue(g);
    if (fuse) g.col_partials = col_partials;
    if (fused) *fused = fuse;
    set_tail(g, tail);
    return run_gemm(g, d->dtype, st);
}

// Split-K of a weight gradient (P outputs [Mo x No], K = M tokens): when its
// 256 x 256 output tiles would occupy fewer than half of about 74 CTA pairs,
// split the tokens so that the tiles fill them (at most 16 ways, at least 8
// K blocks of 64 tokens per split).  A fixed pair count keeps the workspace
// size a function of the shapes alone.
constexpr int kSplitTargetPairs = 74;

static int wgrad_ksplit(int Mo, int No, int P, int K) {
    const long long tiles = static_cast<long long>((Mo + 255) / 256) * ((No + 255) / 256) * P;
    if (tiles == 0 || tiles * 2 > kSplitTargetPairs) return 1;
    int ks = static_cast<int>(kSplitTargetPairs / tiles);
    ks = std::min(ks, std::min(16, ((K + 63) / 64) / 8));
    return std::max(ks, 1);
}

static size_t split_bytes(const tp_mlp_desc *d, int Mo, int No) {
    const Dims x = dims_of(d);
    if (d->dtype == TP_DT_F32) return 0;  // the fp32 engine does not split
    const int ks = wgrad_ksplit(Mo, No, x.T, x.M);
    if (ks <= 1) return 0;
    return align256(sizeof(float) * ks * x.T * static_cast<size_t>((Mo + 255) / 256 * 256) * No);
}

// Weight gradient dW_i = G_i^T Act_i over all tokens (fp32).  G has width
// gw (the output side of the layer), Act width aw; either may be token-sharded
// (1 buffer or nx buffers) or per shard (T buffers).  split_ws (or null):
// workspace for split-K partial sums, split_bytes(d, gw, aw) bytes.
static tp_status wgrad(const tp_mlp_desc *d, const char *name, const void *const *G, int g_per_shard, int gw,
                       const void *const *Act, int a_per_shard, int aw, void *const *dW, cudaStream_t st,
                       float *split_ws, Scratch tail = {}) {
    const Dims x = dims_of(d);
    GemmPlan g;
    g.name = name;
    g.kind = EPI_F32;
    g.M = gw;
    g.N = aw;
    g.P = x.T;
    g.S = 1;
    g.Kseg = x.M;
    if (g_per_shard)
        set_operand(g.A, G, x.T, x.M, gw, true, 1, 0, 0);
    else
        set_operand(g.A, G, x.nx, x.rs ? x.rs : x.M, gw, true, 0, 0, x.rs);
    if (a_per_shard)
        set_operand(g.B, Act, x.T, x.M, aw, true, 1, 0, 0);
    else
        set_operand(g.B, Act, x.nx, x.rs ? x.rs : x.M, aw, true, 0, 0, x.rs);
    set_out(g.out, reinterpret_cast<const void *const *>(dW), x.T, 1, 0, aw);
    g.accumulate = d->wgrad_accumulate != 0;
    if (split_ws && split_bytes(d, gw, aw)) {
        g.ksplit = wgrad_ksplit(gw, aw, x.T, x.M);
        g.split_ws = split_ws;
    }
    set_tail(g, tail);
    return run_gemm(g, d->dtype, st);
}

// Column-layer dgrad: dX = sum_i dOut_i W_i (+R); the K loop runs over shards.
static tp_status column_dgrad(const tp_mlp_desc *d, const void *const *dOut, int kw, const void *const *W,
                              const void *const *R, void *const *dX, cudaStream_t st, Scratch tail = {},
                              float *res_partials = nullptr) {
    const Dims x = dims_of(d);
    GemmPlan g;
    g.name = "col_dgrad";
    g.kind = EPI_PLAIN;
    g.M = x.M;
    g.N = x.H;
    g.P = 1;
    g.S = x.T;
    g.Kseg = kw;
    set_operand(g.A, dOut, x.T, x.M, kw, false, 0, 1, 0);
    set_operand(g.B, W, x.T, kw, x.H, true, 0, 1, 0);
    set_out(g.out, reinterpret_cast<const void *const *>(dX), x.nx, 0, x.rs, x.H);
    if (R) set_out(g.aux, R, x.nx, 0, x.rs, x.H);
    // the residual's per-32-row column sums (db2 partials), tcgen05 engine only
    if (R && d->dtype != TP_DT_F32) g.col_partials = res_partials;
    set_bias(g, nullptr, 0, 0);
    set_tail(g, tail);
    return run_gemm(g, d->dtype, st);
}

static tp_status colsum(const tp_mlp_desc *d, const char *name, const void *const *in, int n_in, int p_stride,
                        int rows_split, int P, int N, void *const *out, float *partials, cudaStream_t st) {
    const Dims x = dims_of(d);
    ColsumPlan c;
    c.name = name;
    set_out(c.in, in, n_in, p_stride, rows_split, N);
    c.P = P;
    c.M = x.M;
    c.N = N;
    for (int i = 0; i < kMaxShards; ++i) c.out[i] = i < P ? static_cast<float *>(out[i]) : nullptr;
    c.partials = partials;
    return launch_colsum(c, d->dtype == TP_DT_F32 ? TP_DT_F32 : TP_DT_BF16, st);
}

// db1 from the fused epilogue's per-32-row-block column sums
static tp_status db1_finalize(const tp_mlp_desc *d, int gw, void *const *db1, float *partials, cudaStream_t st) {
    const Dims x = dims_of(d);
    ColsumPlan c;
    c.name = "bias_grad_col";
    c.P = x.T;
    c.M = x.M;
    c.N = gw;
    for (int i = 0; i < kMaxShards; ++i) c.out[i] = i < x.T ? static_cast<float *>(db1[i]) : nullptr;
    c.partials = partials;
    return launch_colsum_finalize(c, (x.M + 31) / 32, st);
}

// db2 from the column dgrad epilogue's per-32-row-block sums of its residual dY
static tp_status db2_finalize(const tp_mlp_desc *d, void *db2, float *partials, cudaStream_t st) {
    const Dims x = dims_of(d);
    ColsumPlan c;
    c.name = "bias_grad_row";
    c.P = 1;
    c.M = x.M;
    c.N = x.H;
    for (int i = 0; i < kMaxShards; ++i) c.out[i] = i == 0 ? static_cast<float *>(db2) : nullptr;
    c.partials = partials;
    return launch_colsum_finalize(c, (x.M + 31) / 32, st);
}

static size_t partials_bytes(const tp_mlp_desc *d, int P, int N) {
    const Dims x = dims_of(d);
    return align256(sizeof(float) * static_cast<size_t>(P) * colsum_chunks(x.M) * N);
}

// Workspace of the backward: dPre_i (bf16/fp32), the bias partials, then
// the split-K partials of the weight gradients.
static size_t bias_part_bytes(const tp_mlp_desc *d) {
    const Dims x = dims_of(d);
    if (!d->has_bias) return 0;
    // db1: colsum partials, or the fused epilogue's per-32-row-block sums
    const size_t a = partials_bytes(d, x.T, x.g * x.Fs), b = partials_bytes(d, 1, x.H);
    const size_t c = align256(sizeof(float) * size_t(x.T) * ((x.M + 31) / 32) * x.g * x.Fs);
    const size_t e = align256(sizeof(float) * size_t((x.M + 31) / 32) * x.H);  // db2 from the column dgrad
    return std::max(std::max(a, e), std::max(b, c));
}

static size_t bwd_ws_bytes(const tp_mlp_desc *d, size_t *dpre_shard_bytes, size_t *split_off = nullptr) {
    const Dims x = dims_of(d);
    const size_t shard = align256(static_cast<size_t>(x.M) * x.g * x.Fs * x.es);
    if (dpre_shard_bytes) *dpre_shard_bytes = shard;
    const size_t off = shard * x.T + bias_part_bytes(d);
    if (split_off) *split_off = off;
    return off + std::max(split_bytes(d, x.H, x.Fs), split_bytes(d, x.g * x.Fs, x.H));
}

// FP8 region (after the backward region): amax slots, then the quantised
// operands.  The forward fills Xq, W1q, W2q, Aq and their amax slots; the
// backward reads them and fills dYq, dPq.
enum { AMAX_X = 0, AMAX_W1, AMAX_W2, AMAX_A, AMAX_DY, AMAX_DP, AMAX_SLOTS = 8 };
constexpr int kMaxFp8History = 64;
// amax region: this step's amax per slot at +0, the amax each scale derives
// from at +128 (delayed scaling; equal to the first under current scaling)
constexpr size_t kScaleAmaxOff = 128;
struct Fp8Layout {
    size_t amax, hist, xq, w1q, w1q_shard, w2q, w2q_shard, aq, aq_shard, dyq, dpq, dpq_shard, end;
};

// Delayed scaling of one call: history length n (0: current scaling), the
// valid history entries and the column this call's amaxes go to.
struct Fp8Recipe {
    int n = 0, fill = 0, pos = 0;
};

static Fp8Layout fp8_layout(const tp_mlp_desc *d) {
    const Dims x = dims_of(d);
    Fp8Layout L;
    size_t o = align256(bwd_ws_bytes(d, nullptr));
    L.amax = o;
    o += 256;
    L.hist = o;  // [AMAX_SLOTS][kMaxFp8History] floats, kept between calls under delayed scaling
    o += align256(sizeof(float) * AMAX_SLOTS * kMaxFp8History);
    L.xq = o;
    o += align256(size_t(x.M) * x.H);
    L.w1q_shard = align256(size_t(x.g) * x.Fs * x.H);
    L.w1q = o;
    o += L.w1q_shard * x.T;
    L.w2q_shard = align256(size_t(x.H) * x.Fs);
    L.w2q = o;
    o += L.w2q_shard * x.T;
    L.aq_shard = align256(size_t(x.M) * x.Fs);
    L.aq = o;
    o += L.aq_shard * x.T;
    L.dyq = o;
    o += align256(size_t(x.M) * x.H);
    L.dpq_shard = align256(size_t(x.M) * x.g * x.Fs);
    L.dpq = o;
    o += L.dpq_shard * x.T;
    L.end = o;
    return L;
}

// Tail-split scratch of the MLP's pair GEMMs (row forward, column dgrad,
// both weight gradients) and of the fused forward's even split: the largest
// any of them may use.  It depends on the GEMM settings and the device, so it
// comes after everything else in a workspace: validation asks only for the
// part before it, and a kernel uses it only when the scratch a caller's
// workspace leaves is large enough.
static size_t tail_scratch_bytes(const tp_mlp_desc *d) {
    if (d->dtype == TP_DT_F32) return 0;  // the fp32 engine does not split
    const Dims x = dims_of(d);
    const bool f8 = d->dtype == TP_DT_FP8;
    const int gw = x.g * x.Fs;
    size_t r = tc_tail_bytes(x.M, x.H, 1, x.T, x.Fs, f8);
    r = std::max(r, tc_tail_bytes(x.M, x.H, 1, x.T, gw, f8));
    r = std::max(r, tc_tail_bytes(x.H, x.Fs, x.T, 1, x.M, f8));
    r = std::max(r, tc_tail_bytes(gw, x.H, x.T, 1, x.M, f8));
    if (fused_fwd_supported(x.H, x.Fs, d->act, d->dtype)) r = std::max(r, fused_fwd_scratch_bytes(x.M));
    return align256(r);
}

// the MLP workspace without its tail-split scratch (what a call requires)
static size_t mlp_ws_layout(const tp_mlp_desc *d, size_t *dpre_shard_bytes) {
    const size_t b = bwd_ws_bytes(d, dpre_shard_bytes);
    return align256(d->dtype == TP_DT_FP8 ? fp8_layout(d).end : b);
}

// the scratch a workspace of `bytes` leaves after its first `used` bytes
static Scratch scratch_after(void *workspace, size_t bytes, size_t used) {
    Scratch t;
    if (workspace && bytes > used) {
        t.p = static_cast<char *>(workspace) + used;
        t.n = bytes - used;
    }
    return t;
}

static tp_status zero_grads(const tp_mlp_desc *d, void *const *dW, int nW, size_t wbytes, void *const *db, int ndb,
                            size_t dbbytes, cudaStream_t st) {
    if (!d->wgrad_accumulate)
        for (int i = 0; i < nW; ++i) TRY(cuda_check(cudaMemsetAsync(dW[i], 0, wbytes, st), "cudaMemsetAsync(dW)"));
    if (db)
        for (int i = 0; i < ndb; ++i) TRY(cuda_check(cudaMemsetAsync(db[i], 0, dbbytes, st), "cudaMemsetAsync(db)"));
    return TP_OK;
}

// ---------------------------------------------------------------------------
// FP8 variant ("Megatron-LM 源码精读" s8.2): every GEMM operand is quantised
// per tensor -- E4M3 for X, W1, W2 and A in the forward, E5M2 for dY and
// dPre in the backward -- with one scale per tensor over all its shards; the
// GEMMs run on tcgen05 kind::f8f6f4 and dequantise in the epilogue.  pre, A,
// dPre, Y and dX stay bf16; bias gradients sum the unquantised bf16 tensors.
// ---------------------------------------------------------------------------
static void set_fp8(GemmPlan &g, int fa, int fb, const float *amax, int slot_a, int slot_b) {
    g.fp8 = true;
    g.fmt_a = fa;
    g.fmt_b = fb;
    g.amax_a = amax + slot_a;
    g.amax_b = amax + slot_b;
}

static tp_status fp8_fwd(const tp_mlp_desc *d, const void *const *X, const void *const *W1, const void *const *b1,
                         const void *const *W2, const void *b2, const void *const *R, void *const *Y,
                         void *const *pre, void *const *A, void *ws, cudaStream_t st, const DropCfg *drop,
                         const Fp8Recipe &rc, Scratch tail) {
    const Dims x = dims_of(d);
    const int gw = x.g * x.Fs;
    const Fp8Layout L = fp8_layout(d);
    char *base = static_cast<char *>(ws);
    float *amax = reinterpret_cast<float *>(base + L.amax);
    void *xq = base + L.xq;
    void *w1q[kMaxShards], *w2q[kMaxShards], *aq[kMaxShards];
    for (int i = 0; i < x.T; ++i) {
        w1q[i] = base + L.w1q + i * L.w1q_shard;
        w2q[i] = base + L.w2q + i * L.w2q_shard;
        aq[i] = base + L.aq + i * L.aq_shard;
    }
    // scales: under delayed scaling every GEMM dequantises with the amax its
    // operand's scale came from (samax); under current scaling that is the
    // tensor's own amax
    const bool delayed = rc.n > 0;
    float *samax = reinterpret_cast<float *>(base + L.amax + kScaleAmaxOff);
    float *hist = reinterpret_cast<float *>(base + L.hist);
    const float *sa = delayed ? samax : amax;
    // quantise X (E4M3; sequence shards are gathered into one buffer), W1, W2
    QuantSeg segs[kMaxQuantSegs];
    int n = 0;
    const size_t rows = x.rs ? x.rs : x.M;
    for (int j = 0; j < x.nx; ++j)
        segs[n++] = {X[j], static_cast<char *>(xq) + j * rows * x.H, (long long)(rows * x.H), AMAX_X, FP8_E4M3};
    for (int i = 0; i < x.T; ++i) segs[n++] = {W1[i], w1q[i], (long long)gw * x.H, AMAX_W1, FP8_E4M3};
    for (int i = 0; i < x.T; ++i) segs[n++] = {W2[i], w2q[i], (long long)x.H * x.Fs, AMAX_W2, FP8_E4M3};
    const int xw_slots[3] = {AMAX_X, AMAX_W1, AMAX_W2};
    if (!delayed || rc.fill == 0) {
        TRY(launch_fp8_quantize(segs, n, amax, true, st));  // amax pass, then the cast
        if (delayed) TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, xw_slots, 3, 0, 0, false, st));
    } else {
        // one pass: scale from the history, this step's amax reduced on the way
        TRY(cuda_check(cudaMemsetAsync(amax + AMAX_X, 0, 3 * sizeof(float), st), "cudaMemsetAsync(amax)"));
        TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, xw_slots, 3, rc.fill, 0, false, st));
        TRY(launch_fp8_cast(segs, n, amax, samax, true, st));
    }
    // column GEMM: pre_i = Xq W1q_i^T / (s_x s_w1) + b1_i, A_i = act(pre_i)
    bool a_fused = false, a_direct = false;
    {
        GemmPlan g;
        g.name = "col_fwd";
        g.kind = EPI_COL;
        g.act = d->act;
        g.M = x.M;
        g.N = x.Fs;
        g.P = x.T;
        g.S = 1;
        g.Kseg = x.H;
        const void *xa[1] = {xq};
        set_operand(g.A, xa, 1, x.M, x.H, false, 0, 0, 0);
        set_operand(g.B, w1q, x.T, gw, x.H, false, 1, 0, 0);
        g.b_dual_off = d->act == TP_ACT_SWIGLU ? x.Fs : 0;
        set_out(g.out, reinterpret_cast<const void *const *>(A), x.T, 1, 0, x.Fs);
        if (pre) set_out(g.out2, reinterpret_cast<const void *const *>(pre), x.T, 1, 0, gw);
        set_bias(g, d->has_bias ? b1 : nullptr, x.T, 1);
        set_fp8(g, FP8_E4M3, FP8_E4M3, sa, AMAX_X, AMAX_W1);
        a_fused = tc_fused_epilogue(g);
        if (a_fused) {  // the epilogue reduces amax(A) as it stores A
            TRY(cuda_check(cudaMemsetAsync(amax + AMAX_A, 0, sizeof(float), st), "cudaMemsetAsync(amax)"));
            g.amax_out = amax + AMAX_A;
        }
        if (delayed && rc.fill > 0 && a_fused && tc_writes_fp8(g)) {
            // A's scale is known before A exists: the epilogue writes its codes too
            const int a_slot[1] = {AMAX_A};
            TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, a_slot, 1, rc.fill, 0, false, st));
            g.q = true;
            for (int i = 0; i < x.T; ++i) g.q_out[i] = aq[i];
            g.q_fmt = FP8_E4M3;
            g.q_scale_amax = samax + AMAX_A;
            a_direct = true;
        }
        TRY(launch_tc_gemm(g, st));
    }
    // quantise A (E4M3, one scale over all shards)
    n = 0;
    for (int i = 0; i < x.T; ++i) segs[n++] = {A[i], aq[i], (long long)x.M * x.Fs, AMAX_A, FP8_E4M3};
    const int a_slot[1] = {AMAX_A};
    if (a_direct) {
        // codes written by the column GEMM
    } else if (!delayed) {
        TRY(launch_fp8_quantize(segs, n, amax, true, st, a_fused));
    } else if (rc.fill == 0) {
        if (!a_fused) TRY(launch_fp8_quantize(segs, n, amax, true, st));  // amax, then a cast from it
        TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, a_slot, 1, 0, 0, false, st));
        if (a_fused) TRY(launch_fp8_cast(segs, n, amax, samax, false, st));
    } else {
        if (!a_fused) TRY(cuda_check(cudaMemsetAsync(amax + AMAX_A, 0, sizeof(float), st), "cudaMemsetAsync(amax)"));
        TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, a_slot, 1, rc.fill, 0, false, st));
        TRY(launch_fp8_cast(segs, n, amax, samax, !a_fused, st));
    }
    // row GEMM: Y = sum_i Aq_i W2q_i^T / (s_a s_w2) + b2 (+ R), optionally through dropout
    GemmPlan g;
    g.name = "row_fwd";
    g.kind = EPI_PLAIN;
    g.M = x.M;
    g.N = x.H;
    g.P = 1;
    g.S = x.T;
    g.Kseg = x.Fs;
    set_operand(g.A, aq, x.T, x.M, x.Fs, false, 0, 1, 0);
    set_operand(g.B, w2q, x.T, x.H, x.Fs, false, 0, 1, 0);
    set_out(g.out, reinterpret_cast<const void *const *>(Y), x.nx, 0, x.rs, x.H);
    if (R) set_out(g.aux, R, x.nx, 0, x.rs, x.H);
    const void *bb[1] = {b2};
    set_bias(g, d->has_bias ? bb : nullptr, 1, 0);
    set_fp8(g, FP8_E4M3, FP8_E4M3, sa, AMAX_A, AMAX_W2);
    set_drop(g, drop);
    set_tail(g, tail);
    TRY(launch_tc_gemm(g, st));
    if (delayed) {  // this step's amaxes join the history
        const int fwd_slots[4] = {AMAX_X, AMAX_W1, AMAX_W2, AMAX_A};
        TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, fwd_slots, 4, 0, rc.pos, true, st));
    }
    return TP_OK;
}

static tp_status fp8_bwd(const tp_mlp_desc *d, const void *const *dY, const void *const *pre, void *const *dX,
                         void *const *dW1, void *const *db1, void *const *dW2, void *db2, void *ws, cudaStream_t st,
                         const Fp8Recipe &rc, Scratch tail) {
    const Dims x = dims_of(d);
    const int gw = x.g * x.Fs;
    const Fp8Layout L = fp8_layout(d);
    size_t shard_bytes = 0, split_off = 0;
    bwd_ws_bytes(d, &shard_bytes, &split_off);
    char *base = static_cast<char *>(ws);
    float *amax = reinterpret_cast<float *>(base + L.amax);
    float *partials = reinterpret_cast<float *>(base + x.T * shard_bytes);
    float *split = reinterpret_cast<float *>(base + split_off);
    void *xq = base + L.xq, *dyq = base + L.dyq;
    void *w1q[kMaxShards], *w2q[kMaxShards], *aq[kMaxShards], *dpq[kMaxShards], *dpre[kMaxShards];
    for (int i = 0; i < x.T; ++i) {
        w1q[i] = base + L.w1q + i * L.w1q_shard;
        w2q[i] = base + L.w2q + i * L.w2q_shard;
        aq[i] = base + L.aq + i * L.aq_shard;
        dpq[i] = base + L.dpq + i * L.dpq_shard;
        dpre[i] = base + i * shard_bytes;
    }
    const bool delayed = rc.n > 0;
    float *samax = reinterpret_cast<float *>(base + L.amax + kScaleAmaxOff);
    float *hist = reinterpret_cast<float *>(base + L.hist);
    const float *sa = delayed ? samax : amax;  // the forward left samax for X, W1, W2, A
    // quantise dY (E5M2; sequence shards gathered)
    QuantSeg segs[kMaxQuantSegs];
    int n = 0;
    const size_t rows = x.rs ? x.rs : x.M;
    for (int j = 0; j < x.nx; ++j)
        segs[n++] = {dY[j], static_cast<char *>(dyq) + j * rows * x.H, (long long)(rows * x.H), AMAX_DY, FP8_E5M2};
    const int dy_slot[1] = {AMAX_DY}, dp_slot[1] = {AMAX_DP};
    if (!delayed || rc.fill == 0) {
        TRY(launch_fp8_quantize(segs, n, amax, true, st));
        if (delayed) TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, dy_slot, 1, 0, 0, false, st));
    } else {
        TRY(cuda_check(cudaMemsetAsync(amax + AMAX_DY, 0, sizeof(float), st), "cudaMemsetAsync(amax)"));
        TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, dy_slot, 1, rc.fill, 0, false, st));
        TRY(launch_fp8_cast(segs, n, amax, samax, true, st));
    }
    const void *dya[1] = {dyq};
    const void *xa[1] = {xq};
    // row layer dgrad: dPre_i = (dYq W2q_i) / (s_dy s_w2) * act'(pre_i)
    bool dp_fused = false, dp_direct = false;
    {
        GemmPlan g;
        g.name = d->act == TP_ACT_NONE ? "row_dgrad" : "row_dgrad_act";
        g.kind = d->act == TP_ACT_NONE ? EPI_PLAIN : EPI_DACT;
        g.act = d->act;
        g.M = x.M;
        g.N = x.Fs;
        g.P = x.T;
        g.S = 1;
        g.Kseg = x.H;
        set_operand(g.A, dya, 1, x.M, x.H, false, 0, 0, 0);
        set_operand(g.B, w2q, x.T, x.H, x.Fs, true, 1, 0, 0);
        set_out(g.out, dpre, x.T, 1, 0, gw);
        if (d->act != TP_ACT_NONE) set_out(g.aux, pre, x.T, 1, 0, gw);
        set_fp8(g, FP8_E5M2, FP8_E4M3, sa, AMAX_DY, AMAX_W2);
        dp_fused = d->act != TP_ACT_NONE && tc_fused_epilogue(g);
        if (dp_fused) {  // the epilogue reduces amax(dPre) and the db1 partials
            TRY(cuda_check(cudaMemsetAsync(amax + AMAX_DP, 0, sizeof(float), st), "cudaMemsetAsync(amax)"));
            g.amax_out = amax + AMAX_DP;
            if (d->has_bias) g.col_partials = partials;
        }
        if (delayed && rc.fill > 0 && dp_fused && tc_writes_fp8(g)) {
            // dPre's scale is known before dPre exists: the epilogue writes its codes too
            TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, dp_slot, 1, rc.fill, 0, false, st));
            g.q = true;
            for (int i = 0; i < x.T; ++i) g.q_out[i] = dpq[i];
            g.q_fmt = FP8_E5M2;
            g.q_scale_amax = samax + AMAX_DP;
            g.q_only = true;  // nothing reads the bf16 dPre: db1 comes from the fused partials
            dp_direct = true;
        }
        TRY(launch_tc_gemm(g, st));
    }
    // quantise dPre (E5M2, one scale over all shards)
    n = 0;
    for (int i = 0; i < x.T; ++i) segs[n++] = {dpre[i], dpq[i], (long long)x.M * gw, AMAX_DP, FP8_E5M2};
    if (dp_direct) {
        // codes written by the row-layer dgrad
    } else if (!delayed) {
        TRY(launch_fp8_quantize(segs, n, amax, true, st, dp_fused));
    } else if (rc.fill == 0) {
        if (!dp_fused) TRY(launch_fp8_quantize(segs, n, amax, true, st));
        TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, dp_slot, 1, 0, 0, false, st));
        if (dp_fused) TRY(launch_fp8_cast(segs, n, amax, samax, false, st));
    } else {
        if (!dp_fused) TRY(cuda_check(cudaMemsetAsync(amax + AMAX_DP, 0, sizeof(float), st), "cudaMemsetAsync(amax)"));
        TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, dp_slot, 1, rc.fill, 0, false, st));
        TRY(launch_fp8_cast(segs, n, amax, samax, !dp_fused, st));
    }
    if (delayed) {  // this step's amaxes join the history
        const int bwd_slots[2] = {AMAX_DY, AMAX_DP};
        TRY(launch_fp8_history(hist, kMaxFp8History, samax, amax, bwd_slots, 2, 0, rc.pos, true, st));
    }
    // weight gradients (both operands MN-major over the tokens)
    {
        GemmPlan g;
        g.name = "wgrad_row";
        g.kind = EPI_F32;
        g.M = x.H;
        g.N = x.Fs;
        g.P = x.T;
        g.S = 1;
        g.Kseg = x.M;
        set_operand(g.A, dya, 1, x.M, x.H, true, 0, 0, 0);
        set_operand(g.B, aq, x.T, x.M, x.Fs, true, 1, 0, 0);
        set_out(g.out, reinterpret_cast<const void *const *>(dW2), x.T, 1, 0, x.Fs);
        g.accumulate = d->wgrad_accumulate != 0;
        if (split_bytes(d, x.H, x.Fs)) {
            g.ksplit = wgrad_ksplit(x.H, x.Fs, x.T, x.M);
            g.split_ws = split;
        }
        set_fp8(g, FP8_E5M2, FP8_E4M3, sa, AMAX_DY, AMAX_A);
        set_tail(g, tail);
        TRY(launch_tc_gemm(g, st));
    }
    {
        GemmPlan g;
        g.name = "wgrad_col";
        g.kind = EPI_F32;
        g.M = gw;
        g.N = x.H;
        g.P = x.T;
        g.S = 1;
        g.Kseg = x.M;
        set_operand(g.A, dpq, x.T, x.M, gw, true, 1, 0, 0);
        set_operand(g.B, xa, 1, x.M, x.H, true, 0, 0, 0);
        set_out(g.out, reinterpret_cast<const void *const *>(dW1), x.T, 1, 0, x.H);
        g.accumulate = d->wgrad_accumulate != 0;
        if (split_bytes(d, gw, x.H)) {
            g.ksplit = wgrad_ksplit(gw, x.H, x.T, x.M);
            g.split_ws = split;
        }
        set_fp8(g, FP8_E5M2, FP8_E4M3, sa, AMAX_DP, AMAX_X);
        set_tail(g, tail);
        TRY(launch_tc_gemm(g, st));
    }
    if (d->has_bias) {  // db1 now: the partials region then takes the db2 partials
        if (dp_fused)
            TRY(db1_finalize(d, gw, db1, partials, st));
        else
            TRY(colsum(d, "bias_grad_col", dpre, x.T, 1, 0, x.T, gw, db1, partials, st));
    }
    // column layer dgrad: dX = sum_i dPq_i W1q_i / (s_dp s_w1) (+ dY); with the
    // residual its epilogue also sums dY per 32-row block (db2 = sum_m dY)
    const bool db2_fused = db2 && d->residual;
    {
        GemmPlan g;
        g.name = "col_dgrad";
        g.kind = EPI_PLAIN;
        g.M = x.M;
        g.N = x.H;
        g.P = 1;
        g.S = x.T;
        g.Kseg = gw;
        set_operand(g.A, dpq, x.T, x.M, gw, false, 0, 1, 0);
        set_operand(g.B, w1q, x.T, gw, x.H, true, 0, 1, 0);
        set_out(g.out, reinterpret_cast<const void *const *>(dX), x.nx, 0, x.rs, x.H);
        if (d->residual) set_out(g.aux, dY, x.nx, 0, x.rs, x.H);
        if (db2_fused) g.col_partials = partials;
        set_bias(g, nullptr, 0, 0);
        set_fp8(g, FP8_E5M2, FP8_E4M3, sa, AMAX_DP, AMAX_W1);
        set_tail(g, tail);
        TRY(launch_tc_gemm(g, st));
    }
    if (db2) {
        void *const *db2a = reinterpret_cast<void *const *>(&db2);
        if (db2_fused)
            TRY(db2_finalize(d, db2, partials, st));
        else
            TRY(colsum(d, "bias_grad_row", dY, x.nx, 0, x.rs, 1, x.H, db2a, partials, st));
    }
    return TP_OK;
}

}  // namespace tpmlp

using namespace tpmlp;

// ---------------------------------------------------------------------------
// exported C ABI
// ---------------------------------------------------------------------------
extern "C" {

int tp_abi_version(void) { return TP_MLP_ABI_VERSION; }

const char *tp_status_str(tp_status s) {
    switch (s) {
        case TP_OK: return "TP_OK";
        case TP_ERR_ARG: return "TP_ERR_ARG";
        case TP_ERR_SHAPE: return "TP_ERR_SHAPE";
        case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
        case TP_ERR_CUDA: return "TP_ERR_CUDA";
        case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT";
    }
    return "TP_ERR_UNKNOWN";
}

const char *tp_last_error(void) { return g_err; }

tp_status tp_mlp_create(const tp_mlp_desc *desc, tp_mlp **out) {
    if (!out) return set_error(TP_ERR_ARG, "out is NULL");
    *out = nullptr;
    TRY(validate_desc(desc));
    tp_mlp *h = new (std::nothrow) tp_mlp;
    if (!h) return set_error(TP_ERR_ARG, "out of host memory");
    h->d = *desc;
    h->status_slot = alloc_status_slot();
    if (h->status_slot < 0) {
        delete h;
        return set_error(TP_ERR_UNSUPPORTED, "more than %d live handles (each owns a device status word)",
                         kStatusSlots - 1);
    }
    *out = h;
    return TP_OK;
}

void tp_mlp_destroy(tp_mlp *h) {
    if (!h) return;
    free_status_slot(h->status_slot);
    delete h;
}

size_t tp_mlp_workspace_bytes(const tp_mlp *h) {
    return h ? mlp_ws_layout(&h->d, nullptr) + tail_scratch_bytes(&h->d) : 0;
}

// MLP forward on validated arguments: Y = R + dropout(MLP(X)) with R and the
// dropout optional (the plain MLP passes R = X iff residual, no dropout).
static tp_status mlp_fwd_core(const tp_mlp_desc *d, const void *const *X, const void *const *W1,
                              const void *const *b1, const void *const *W2, const void *b2, const void *const *R,
                              void *const *Y, void *const *pre, void *const *A, void *workspace, const DropCfg *drop,
                              cudaStream_t st, const Fp8Recipe &rc = Fp8Recipe(), Scratch tail = {}) {
    if (d->dtype == TP_DT_FP8)
        return fp8_fwd(d, X, W1, d->has_bias ? b1 : nullptr, W2, b2, R, Y, pre, A, workspace, st, drop, rc, tail);
    const Dims x = dims_of(d);
    // The fused kernel wherever it takes the shape, unless switched off: it
    // measured faster than the two GEMMs from 16 to 2048 token tiles on 152
    // SMs (1.03-1.5x).
    if (fused_fwd_mode() != TP_FUSED_OFF && fused_fwd_supported(x.H, x.Fs, d->act, d->dtype)) {
        FusedPlan f;
        for (int j = 0; j < kMaxShards; ++j) {
            f.X[j] = j < x.nx ? X[j] : nullptr;
            f.R[j] = (R && j < x.nx) ? R[j] : nullptr;
            f.Y[j] = j < x.nx ? Y[j] : nullptr;
            f.W1[j] = j < x.T ? W1[j] : nullptr;
            f.b1[j] = (d->has_bias && j < x.T) ? b1[j] : nullptr;
            f.W2[j] = j < x.T ? W2[j] : nullptr;
            f.pre[j] = (pre && j < x.T) ? pre[j] : nullptr;
            f.A[j] = j < x.T ? A[j] : nullptr;
        }
        f.b2 = d->has_bias ? b2 : nullptr;
        f.n_tok = x.nx;
        f.rows_split = x.rs;
        f.M = x.M;
        f.H = x.H;
        f.Fs = x.Fs;
        f.T = x.T;
        f.act = d->act;
        f.has_bias = d->has_bias != 0;
        f.has_res = R != nullptr;
        f.has_pre = pre != nullptr;
        if (drop && drop->on) {
            f.dropout = true;
            f.drop_threshold = drop->threshold;
            f.drop_scale = drop->scale;
            f.drop_seed = drop->seed;
            f.drop_mask = drop->mask;
        }
        f.scratch = tail.p;
        f.scratch_bytes = tail.n;
        return launch_fused_mlp_fwd(f, st);
    }
    TRY(column_fwd(d, X, W1, d->has_bias ? b1 : nullptr, A, pre, st));
    return row_fwd(d, reinterpret_cast<const void *const *>(A), W2, d->has_bias ? b2 : nullptr, R, Y, st, drop,
                   tail);
}

// MLP backward on validated arguments (workspace checked by the caller).
// db2_done: the caller has produced db2 already (the sub-block's dropout
// backward sums dZ as it writes it).
static tp_status mlp_bwd_core(const tp_mlp_desc *d, const void *const *dY, const void *const *X,
                              const void *const *W1, const void *const *W2, const void *const *pre,
                              const void *const *A, void *const *dX, void *const *dW1, void *const *db1,
                              void *const *dW2, void *db2, void *workspace, cudaStream_t st,
                              bool db2_done = false, const Fp8Recipe &rc = Fp8Recipe(), Scratch tail = {}) {
    const Dims x = dims_of(d);
    const int gw = x.g * x.Fs;
    size_t shard_bytes = 0;
    mlp_ws_layout(d, &shard_bytes);
    void *const *db2a = reinterpret_cast<void *const *>(&db2);
    if (x.M == 0) {
        TRY(zero_grads(d, dW1, x.T, sizeof(float) * gw * x.H, d->has_bias ? db1 : nullptr, x.T, sizeof(float) * gw, st));
        return zero_grads(d, dW2, x.T, sizeof(float) * x.H * x.Fs, d->has_bias ? db2a : nullptr, 1,
                          sizeof(float) * x.H, st);
    }
    if (d->dtype == TP_DT_FP8)
        return fp8_bwd(d, dY, pre, dX, dW1, d->has_bias ? db1 : nullptr, dW2,
                       (d->has_bias && !db2_done) ? db2 : nullptr, workspace, st, rc, tail);
    void *dpre[kMaxShards];
    for (int i = 0; i < x.T; ++i) dpre[i] = static_cast<char *>(workspace) + i * shard_bytes;
    float *partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + x.T * shard_bytes);
    size_t split_off = 0;
    bwd_ws_bytes(d, nullptr, &split_off);
    float *split = reinterpret_cast<float *>(static_cast<char *>(workspace) + split_off);
    // row layer: dPre_i = (dY W2_i) * act'(pre_i), dW2_i = dY^T A_i
    bool db1_fused = false;
    TRY(row_dgrad(d, d->act, dY, W2, pre, dpre, gw, st, d->has_bias ? partials : nullptr, &db1_fused));
    if (d->has_bias) {  // db1 now: the partials region then takes the db2 partials
        if (db1_fused)
            TRY(db1_finalize(d, gw, db1, partials, st));
        else
            TRY(colsum(d, "bias_grad_col", dpre, x.T, 1, 0, x.T, gw, db1, partials, st));
    }
    TRY(wgrad(d, "wgrad_row", dY, 0, x.H, A, 1, x.Fs, dW2, st, split, tail));
    // column layer: dW1_i = dPre_i^T X, dX = sum_i dPre_i W1_i (+ dY); with the
    // residual its epilogue also sums dY per 32-row block (db2 = sum_m dY)
    TRY(wgrad(d, "wgrad_col", dpre, 1, gw, X, 0, x.H, dW1, st, split, tail));
    const bool db2_fused = d->has_bias && !db2_done && d->residual && d->dtype != TP_DT_F32;
    TRY(column_dgrad(d, dpre, gw, W1, d->residual ? dY : nullptr, dX, st, tail, db2_fused ? partials : nullptr));
    if (d->has_bias && !db2_done) {
        if (db2_fused)
            TRY(db2_finalize(d, db2, partials, st));
        else
            TRY(colsum(d, "bias_grad_row", dY, x.nx, 0, x.rs, 1, x.H, db2a, partials, st));
    }
    return TP_OK;
}

// delayed-scaling state of a handle's next call (steps: its quantisations so far)
static Fp8Recipe fp8_recipe(int dtype, int history, long long steps) {
    Fp8Recipe rc;
    if (dtype != TP_DT_FP8 || history <= 0) return rc;
    rc.n = history;
    rc.fill = static_cast<int>(steps < rc.n ? steps : rc.n);
    rc.pos = static_cast<int>(steps % rc.n);
    return rc;
}

static tp_status mlp_fwd_impl(tp_mlp *h, const void *const *X, const void *const *W1, const void *const *b1,
                              const void *const *W2, const void *b2, void *const *Y, void *const *pre,
                              void *const *A, void *workspace, size_t workspace_bytes, bool has_ws, void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    const StatusScope scope(h->status_slot);
    const tp_mlp_desc *d = &h->d;
    const Dims x = dims_of(d);
    TRY(check_array(W1, x.T, "W1"));
    TRY(check_array(W2, x.T, "W2"));
    if (d->has_bias) {
        TRY(check_array(b1, x.T, "b1"));
        TRY(check_one(b2, "b2"));
    }
    if (d->dtype == TP_DT_FP8) {
        if (!has_ws) return set_error(TP_ERR_ARG, "the FP8 forward needs a workspace: call tp_mlp_fwd_ws");
        const size_t need = mlp_ws_layout(d, nullptr);
        if (workspace_bytes < need)
            return set_error(TP_ERR_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return set_error(TP_ERR_ARG, "workspace must be non-NULL and 256-byte aligned");
    } else if (!has_ws || !workspace || workspace_bytes < mlp_ws_layout(d, nullptr) ||
               (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
        workspace = nullptr;  // optional for bf16 / fp32: used only when it is large enough
        workspace_bytes = 0;
    }
    if (x.M == 0) return TP_OK;  // no tokens: activation buffers may be empty (NULL)
    TRY(check_array(X, x.nx, "X"));
    TRY(check_array(reinterpret_cast<const void *const *>(Y), x.nx, "Y"));
    TRY(check_array(reinterpret_cast<const void *const *>(A), x.T, "A"));
    if (d->act != TP_ACT_NONE || pre) TRY(check_array(reinterpret_cast<const void *const *>(pre), x.T, "pre"));
    const Fp8Recipe rc = fp8_recipe(d->dtype, h->fp8_history, h->fp8_fwd_steps);
    TRY(mlp_fwd_core(d, X, W1, b1, W2, b2, d->residual ? X : nullptr, Y, pre, A, workspace, nullptr,
                     static_cast<cudaStream_t>(stream), rc,
                     scratch_after(workspace, workspace_bytes, mlp_ws_layout(d, nullptr))));
    if (d->dtype == TP_DT_FP8 && rc.n) ++h->fp8_fwd_steps;
    return TP_OK;
}

tp_status tp_mlp_fwd(tp_mlp *h, const void *const *X, const void *const *W1, const void *const *b1,
                     const void *const *W2, const void *b2, void *const *Y, void *const *pre, void *const *A,
                     void *stream) {
    return mlp_fwd_impl(h, X, W1, b1, W2, b2, Y, pre, A, nullptr, 0, false, stream);
}

tp_status tp_mlp_fwd_ws(tp_mlp *h, const void *const *X, const void *const *W1, const void *const *b1,
                        const void *const *W2, const void *b2, void *const *Y, void *const *pre, void *const *A,
                        void *workspace, size_t workspace_bytes, void *stream) {
    return mlp_fwd_impl(h, X, W1, b1, W2, b2, Y, pre, A, workspace, workspace_bytes, true, stream);
}

tp_status tp_mlp_bwd(tp_mlp *h, const void *const *dY, const void *const *X, const void *const *W1,
                     const void *const *W2, const void *const *pre, const void *const *A, void *const *dX,
                     void *const *dW1, void *const *db1, void *const *dW2, void *db2, void *workspace,
                     size_t workspace_bytes, void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    const StatusScope scope(h->status_slot);
    const tp_mlp_desc *d = &h->d;
    const Dims x = dims_of(d);
    TRY(check_array(W1, x.T, "W1"));
    TRY(check_array(W2, x.T, "W2"));
    if (x.M > 0) {  // no tokens: activation buffers may be empty (NULL)
        TRY(check_array(dY, x.nx, "dY"));
        TRY(check_array(X, x.nx, "X"));
        if (d->act != TP_ACT_NONE) TRY(check_array(pre, x.T, "pre"));
        TRY(check_array(A, x.T, "A"));
        TRY(check_array(reinterpret_cast<const void *const *>(dX), x.nx, "dX"));
    }
    TRY(check_array(reinterpret_cast<const void *const *>(dW1), x.T, "dW1"));
    TRY(check_array(reinterpret_cast<const void *const *>(dW2), x.T, "dW2"));
    if (d->has_bias) {
        TRY(check_array(reinterpret_cast<const void *const *>(db1), x.T, "db1"));
        TRY(check_one(db2, "db2"));
    }
    const size_t need = mlp_ws_layout(d, nullptr);
    if (workspace_bytes < need)
        return set_error(TP_ERR_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if (need && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return set_error(TP_ERR_ARG, "workspace must be non-NULL and 256-byte aligned");
    const Fp8Recipe rc = fp8_recipe(d->dtype, h->fp8_history, h->fp8_bwd_steps);
    TRY(mlp_bwd_core(d, dY, X, W1, W2, pre, A, dX, dW1, db1, dW2, db2, workspace, static_cast<cudaStream_t>(stream),
                     false, rc, scratch_after(workspace, workspace_bytes, need)));
    if (d->dtype == TP_DT_FP8 && rc.n && x.M > 0) ++h->fp8_bwd_steps;
    return TP_OK;
}

// single-layer workspace: [bias partials | split-K partials of the weight
// gradient | (FP8) amax slots and operand codes | tail-split scratch]
static size_t linear_part_bytes(const tp_mlp_desc *desc) {
    if (!desc->has_bias) return 0;
    const Dims x = dims_of(desc);
    size_t a = partials_bytes(desc, x.T, x.g * x.Fs), b = partials_bytes(desc, 1, x.H);
    return a > b ? a : b;
}

static size_t linear_split_bytes(const tp_mlp_desc *desc) {
    const Dims x = dims_of(desc);
    return std::max(split_bytes(desc, x.Fs, x.H), split_bytes(desc, x.H, x.Fs));
}

// FP8 region of a single-layer workspace ("Megatron-LM 源码精读" s8.2 applied
// to one layer): the amax of the layer's input activation (X), its weight (W)
// and its upstream gradient (G), then their codes.  The forward fills X and W
// (E4M3), the backward reads them and fills G (E5M2).  A column layer's X is
// one [M, H] buffer (token shards gathered), its W shards [g*Fs, H] and its G
// shards [M, Fs]; a row layer's X shards are [M, Fs], its W shards [H, Fs]
// and its G one [M, H] buffer.
enum { LAMAX_X = 0, LAMAX_W = 1, LAMAX_G = 2 };
struct LinFp8Layout {
    size_t amax, xq, xq_shard, wq, wq_shard, gq, gq_shard, end;
};

static LinFp8Layout linear_fp8_layout(const tp_mlp_desc *d) {
    const Dims x = dims_of(d);
    LinFp8Layout L;
    size_t o = align256(linear_part_bytes(d) + linear_split_bytes(d));
    L.amax = o;
    o += 256;
    const size_t full = align256(size_t(x.M) * x.H);
    L.xq_shard = align256(size_t(x.M) * x.Fs);
    L.xq = o;
    o += std::max(full, L.xq_shard * x.T);
    L.wq_shard = align256(size_t(x.g) * x.Fs * x.H);
    L.wq = o;
    o += L.wq_shard * x.T;
    L.gq_shard = align256(size_t(x.M) * x.Fs);
    L.gq = o;
    o += std::max(full, L.gq_shard * x.T);
    L.end = o;
    return L;
}

// what a single-layer call requires (the part before the tail-split scratch)
static size_t linear_need(const tp_mlp_desc *desc) {
    if (desc->dtype == TP_DT_FP8) return linear_fp8_layout(desc).end;
    return linear_part_bytes(desc) + linear_split_bytes(desc);
}

// ... then the tail-split scratch of its pair GEMMs (column layer: dgrad and
// weight gradient; row layer: forward, dgrad and weight gradient), at the end
static size_t linear_tail_off(const tp_mlp_desc *desc) { return align256(linear_need(desc)); }

static size_t linear_tail_bytes(const tp_mlp_desc *desc) {
    if (desc->dtype == TP_DT_F32) return 0;  // the fp32 engine does not split
    const Dims x = dims_of(desc);
    const bool f8 = desc->dtype == TP_DT_FP8;
    size_t r = tc_tail_bytes(x.M, x.H, 1, x.T, x.Fs, f8);
    r = std::max(r, tc_tail_bytes(x.Fs, x.H, x.T, 1, x.M, f8));
    r = std::max(r, tc_tail_bytes(x.M, x.Fs, x.T, 1, x.H, f8));
    r = std::max(r, tc_tail_bytes(x.H, x.Fs, x.T, 1, x.M, f8));
    return align256(r);
}

static tp_status check_ws(const tp_mlp_desc *d, void *ws, size_t bytes) {
    const size_t need = linear_need(d);
    if (bytes < need) return set_error(TP_ERR_ARG, "workspace too small: %zu < %zu bytes", bytes, need);
    if (need && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)))
        return set_error(TP_ERR_ARG, "workspace must be non-NULL and 256-byte aligned");
    return TP_OK;
}

// FP8 single layers: the codes and amax slots inside a checked workspace
struct LinFp8 {
    float *amax;
    char *xq, *wq, *gq;
    size_t xs, ws, gs;  // shard strides
    void *x_at(int i) const { return xq + i * xs; }
    void *w_at(int i) const { return wq + i * ws; }
    void *g_at(int i) const { return gq + i * gs; }
};

static LinFp8 lin_fp8(const tp_mlp_desc *d, void *workspace) {
    const LinFp8Layout L = linear_fp8_layout(d);
    char *b = static_cast<char *>(workspace);
    return {reinterpret_cast<float *>(b + L.amax), b + L.xq, b + L.wq, b + L.gq, L.xq_shard, L.wq_shard, L.gq_shard};
}

// one tensor of `nbuf` buffers of `elems` elements each, quantised into
// consecutive slots `dst_stride` bytes apart, all with the tensor's one scale
static void add_segs(QuantSeg *segs, int &n, const void *const *src, int nbuf, long long elems, char *dst,
                     size_t dst_stride, int slot, int fmt) {
    for (int j = 0; j < nbuf; ++j) segs[n++] = {src[j], dst + j * dst_stride, elems, slot, fmt};
}

// column layer forward: out_i = act(Xq Wq_i^T / (s_x s_w) + b_i)
static tp_status fp8_linear_col_fwd(const tp_mlp_desc *d, const void *const *X, const void *const *W,
                                    const void *const *b, void *const *out, void *const *pre, void *workspace,
                                    cudaStream_t st) {
    const Dims x = dims_of(d);
    const int gw = x.g * x.Fs;
    const LinFp8 q = lin_fp8(d, workspace);
    QuantSeg segs[kMaxQuantSegs];
    int n = 0;
    const size_t rows = x.rs ? x.rs : x.M;
    add_segs(segs, n, X, x.nx, (long long)(rows * x.H), q.xq, rows * x.H, LAMAX_X, FP8_E4M3);
    add_segs(segs, n, W, x.T, (long long)gw * x.H, q.wq, q.ws, LAMAX_W, FP8_E4M3);
    TRY(launch_fp8_quantize(segs, n, q.amax, true, st));
    GemmPlan g;
    g.name = "col_fwd";
    g.kind = EPI_COL;
    g.act = d->act;
    g.M = x.M;
    g.N = x.Fs;
    g.P = x.T;
    g.S = 1;
    g.Kseg = x.H;
    const void *xa[1] = {q.xq};
    const void *wq[kMaxShards];
    for (int i = 0; i < x.T; ++i) wq[i] = q.w_at(i);
    set_operand(g.A, xa, 1, x.M, x.H, false, 0, 0, 0);
    set_operand(g.B, wq, x.T, gw, x.H, false, 1, 0, 0);
    g.b_dual_off = d->act == TP_ACT_SWIGLU ? x.Fs : 0;
    set_out(g.out, reinterpret_cast<const void *const *>(out), x.T, 1, 0, x.Fs);
    if (pre) set_out(g.out2, reinterpret_cast<const void *const *>(pre), x.T, 1, 0, gw);
    set_bias(g, b, x.T, 1);
    set_fp8(g, FP8_E4M3, FP8_E4M3, q.amax, LAMAX_X, LAMAX_W);
    return launch_tc_gemm(g, st);
}

// row layer forward: Y = sum_i Xq_i Wq_i^T / (s_x s_w) + b (+R)
static tp_status fp8_linear_row_fwd(const tp_mlp_desc *d, const void *const *X, const void *const *W, const void *b,
                                    const void *const *R, void *const *Y, void *workspace, cudaStream_t st,
                                    Scratch tail) {
    const Dims x = dims_of(d);
    const LinFp8 q = lin_fp8(d, workspace);
    QuantSeg segs[kMaxQuantSegs];
    int n = 0;
    add_segs(segs, n, X, x.T, (long long)x.M * x.Fs, q.xq, q.xs, LAMAX_X, FP8_E4M3);
    add_segs(segs, n, W, x.T, (long long)x.H * x.Fs, q.wq, q.ws, LAMAX_W, FP8_E4M3);
    TRY(launch_fp8_quantize(segs, n, q.amax, true, st));
    GemmPlan g;
    g.name = "row_fwd";
    g.kind = EPI_PLAIN;
    g.M = x.M;
    g.N = x.H;
    g.P = 1;
    g.S = x.T;
    g.Kseg = x.Fs;
    const void *xq[kMaxShards], *wq[kMaxShards];
    for (int i = 0; i < x.T; ++i) {
        xq[i] = q.x_at(i);
        wq[i] = q.w_at(i);
    }
    set_operand(g.A, xq, x.T, x.M, x.Fs, false, 0, 1, 0);
    set_operand(g.B, wq, x.T, x.H, x.Fs, false, 0, 1, 0);
    set_out(g.out, reinterpret_cast<const void *const *>(Y), x.nx, 0, x.rs, x.H);
    if (R) set_out(g.aux, R, x.nx, 0, x.rs, x.H);
    const void *bb[1] = {b};
    set_bias(g, b ? bb : nullptr, 1, 0);
    set_fp8(g, FP8_E4M3, FP8_E4M3, q.amax, LAMAX_X, LAMAX_W);
    set_tail(g, tail);
    return launch_tc_gemm(g, st);
}

// column layer backward (no activation): dX = sum_i dOq_i Wq_i / (s_g s_w),
// dW_i = dOq_i^T Xq / (s_g s_x), db_i = sum_m dOut_i
static tp_status fp8_linear_col_bwd(const tp_mlp_desc *d, const void *const *dOut, void *const *dX,
                                    void *const *dW, void *const *db, void *workspace, cudaStream_t st,
                                    Scratch tail) {
    const Dims x = dims_of(d);
    const LinFp8 q = lin_fp8(d, workspace);
    QuantSeg segs[kMaxQuantSegs];
    int n = 0;
    add_segs(segs, n, dOut, x.T, (long long)x.M * x.Fs, q.gq, q.gs, LAMAX_G, FP8_E5M2);
    TRY(launch_fp8_quantize(segs, n, q.amax, true, st));
    const void *gq[kMaxShards], *wq[kMaxShards];
    for (int i = 0; i < x.T; ++i) {
        gq[i] = q.g_at(i);
        wq[i] = q.w_at(i);
    }
    {
        GemmPlan g;
        g.name = "col_dgrad";
        g.kind = EPI_PLAIN;
        g.M = x.M;
        g.N = x.H;
        g.P = 1;
        g.S = x.T;
        g.Kseg = x.Fs;
        set_operand(g.A, gq, x.T, x.M, x.Fs, false, 0, 1, 0);
        set_operand(g.B, wq, x.T, x.Fs, x.H, true, 0, 1, 0);
        set_out(g.out, reinterpret_cast<const void *const *>(dX), x.nx, 0, x.rs, x.H);
        set_bias(g, nullptr, 0, 0);
        set_fp8(g, FP8_E5M2, FP8_E4M3, q.amax, LAMAX_G, LAMAX_W);
        set_tail(g, tail);
        TRY(launch_tc_gemm(g, st));
    }
    {
        GemmPlan g;
        g.name = "wgrad_col";
        g.kind = EPI_F32;
        g.M = x.Fs;
        g.N = x.H;
        g.P = x.T;
        g.S = 1;
        g.Kseg = x.M;
        const void *xa[1] = {q.xq};
        set_operand(g.A, gq, x.T, x.M, x.Fs, true, 1, 0, 0);
        set_operand(g.B, xa, 1, x.M, x.H, true, 0, 0, 0);
        set_out(g.out, reinterpret_cast<const void *const *>(dW), x.T, 1, 0, x.H);
        g.accumulate = d->wgrad_accumulate != 0;
        if (split_bytes(d, x.Fs, x.H)) {
            g.ksplit = wgrad_ksplit(x.Fs, x.H, x.T, x.M);
            g.split_ws = reinterpret_cast<float *>(static_cast<char *>(workspace) + linear_part_bytes(d));
        }
        set_fp8(g, FP8_E5M2, FP8_E4M3, q.amax, LAMAX_G, LAMAX_X);
        set_tail(g, tail);
        TRY(launch_tc_gemm(g, st));
    }
    if (db) TRY(colsum(d, "bias_grad_col", dOut, x.T, 1, 0, x.T, x.Fs, db, static_cast<float *>(workspace), st));
    return TP_OK;
}

// row layer backward: dX_i = dYq Wq_i / (s_g s_w), dW_i = dYq^T Xq_i /
// (s_g s_x), db = sum_m dY
static tp_status fp8_linear_row_bwd(const tp_mlp_desc *d, const void *const *dY, void *const *dX, void *const *dW,
                                    void *db, void *workspace, cudaStream_t st, Scratch tail) {
    const Dims x = dims_of(d);
    const LinFp8 q = lin_fp8(d, workspace);
    QuantSeg segs[kMaxQuantSegs];
    int n = 0;
    const size_t rows = x.rs ? x.rs : x.M;
    add_segs(segs, n, dY, x.nx, (long long)(rows * x.H), q.gq, rows * x.H, LAMAX_G, FP8_E5M2);
    TRY(launch_fp8_quantize(segs, n, q.amax, true, st));
    const void *ga[1] = {q.gq};
    const void *xq[kMaxShards], *wq[kMaxShards];
    for (int i = 0; i < x.T; ++i) {
        xq[i] = q.x_at(i);
        wq[i] = q.w_at(i);
    }
    {
        GemmPlan g;
        g.name = "row_dgrad";
        g.kind = EPI_PLAIN;
        g.M = x.M;
        g.N = x.Fs;
        g.P = x.T;
        g.S = 1;
        g.Kseg = x.H;
        set_operand(g.A, ga, 1, x.M, x.H, false, 0, 0, 0);
        set_operand(g.B, wq, x.T, x.H, x.Fs, true, 1, 0, 0);
        set_out(g.out, reinterpret_cast<const void *const *>(dX), x.T, 1, 0, x.Fs);
        set_bias(g, nullptr, 0, 0);
        set_fp8(g, FP8_E5M2, FP8_E4M3, q.amax, LAMAX_G, LAMAX_W);
        set_tail(g, tail);
        TRY(launch_tc_gemm(g, st));
    }
    {
        GemmPlan g;
        g.name = "wgrad_row";
        g.kind = EPI_F32;
        g.M = x.H;
        g.N = x.Fs;
        g.P = x.T;
        g.S = 1;
        g.Kseg = x.M;
        set_operand(g.A, ga, 1, x.M, x.H, true, 0, 0, 0);
        set_operand(g.B, xq, x.T, x.M, x.Fs, true, 1, 0, 0);
        set_out(g.out, reinterpret_cast<const void *const *>(dW), x.T, 1, 0, x.Fs);
        g.accumulate = d->wgrad_accumulate != 0;
        if (split_bytes(d, x.H, x.Fs)) {
            g.ksplit = wgrad_ksplit(x.H, x.Fs, x.T, x.M);
            g.split_ws = reinterpret_cast<float *>(static_cast<char *>(workspace) + linear_part_bytes(d));
        }
        set_fp8(g, FP8_E5M2, FP8_E4M3, q.amax, LAMAX_G, LAMAX_X);
        set_tail(g, tail);
        TRY(launch_tc_gemm(g, st));
    }
    if (db) {
        void *const *dba = reinterpret_cast<void *const *>(&db);
        TRY(colsum(d, "bias_grad_row", dY, x.nx, 0, x.rs, 1, x.H, dba, static_cast<float *>(workspace), st));
    }
    return TP_OK;
}

// workspace of a single-layer forward: required (checked) for FP8, optional
// otherwise (then used only for the row forward's tail split, and only when
// it holds at least what a backward call requires)
static tp_status linear_fwd_ws(const tp_mlp_desc *d, bool has_ws, void *&workspace, size_t &workspace_bytes) {
    if (d->dtype == TP_DT_FP8) {
        if (!has_ws)
            return set_error(TP_ERR_ARG, "the FP8 single-layer forward needs a workspace: call the _ws variant");
        return check_ws(d, workspace, workspace_bytes);
    }
    if (!has_ws || !workspace || workspace_bytes < linear_need(d) || (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
        workspace = nullptr;
        workspace_bytes = 0;
    }
    return TP_OK;
}

static tp_status linear_col_impl(const tp_mlp_desc *desc, const void *const *X, const void *const *W,
                                 const void *const *b, void *const *out, void *const *pre, void *workspace,
                                 size_t workspace_bytes, bool has_ws, void *stream) {
    TRY(validate_desc(desc));
    const Dims x = dims_of(desc);
    TRY(check_array(W, x.T, "W"));
    if (desc->has_bias) TRY(check_array(b, x.T, "b"));
    TRY(linear_fwd_ws(desc, has_ws, workspace, workspace_bytes));
    if (x.M == 0) return TP_OK;
    TRY(check_array(X, x.nx, "X"));
    TRY(check_array(reinterpret_cast<const void *const *>(out), x.T, "out"));
    if (pre) TRY(check_array(reinterpret_cast<const void *const *>(pre), x.T, "pre"));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (desc->dtype == TP_DT_FP8)
        return fp8_linear_col_fwd(desc, X, W, desc->has_bias ? b : nullptr, out, pre, workspace, st);
    return column_fwd(desc, X, W, desc->has_bias ? b : nullptr, out, pre, st);
}

static tp_status linear_row_impl(const tp_mlp_desc *desc, const void *const *X, const void *const *W, const void *b,
                                 const void *const *R, void *const *Y, void *workspace, size_t workspace_bytes,
                                 bool has_ws, void *stream) {
    TRY(validate_desc(desc));
    const Dims x = dims_of(desc);
    TRY(check_array(W, x.T, "W"));
    if (desc->has_bias) TRY(check_one(b, "b"));
    if (!desc->residual && R) return set_error(TP_ERR_ARG, "R given but desc->residual is 0");
    TRY(linear_fwd_ws(desc, has_ws, workspace, workspace_bytes));
    if (x.M == 0) return TP_OK;
    TRY(check_array(X, x.T, "X"));
    TRY(check_array(reinterpret_cast<const void *const *>(Y), x.nx, "Y"));
    if (desc->residual) TRY(check_array(R, x.nx, "R"));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Scratch tail = scratch_after(workspace, workspace_bytes, linear_tail_off(desc));
    if (desc->dtype == TP_DT_FP8)
        return fp8_linear_row_fwd(desc, X, W, desc->has_bias ? b : nullptr, desc->residual ? R : nullptr, Y,
                                  workspace, st, tail);
    return row_fwd(desc, X, W, desc->has_bias ? b : nullptr, desc->residual ? R : nullptr, Y, st, nullptr, tail);
}

tp_status tp_linear_col(const tp_mlp_desc *desc, const void *const *X, const void *const *W, const void *const *b,
                        void *const *out, void *const *pre, void *stream) {
    return linear_col_impl(desc, X, W, b, out, pre, nullptr, 0, false, stream);
}

tp_status tp_linear_col_ws(const tp_mlp_desc *desc, const void *const *X, const void *const *W,
                           const void *const *b, void *const *out, void *const *pre, void *workspace,
                           size_t workspace_bytes, void *stream) {
    return linear_col_impl(desc, X, W, b, out, pre, workspace, workspace_bytes, true, stream);
}

tp_status tp_linear_row(const tp_mlp_desc *desc, const void *const *X, const void *const *W, const void *b,
                        const void *const *R, void *const *Y, void *stream) {
    return linear_row_impl(desc, X, W, b, R, Y, nullptr, 0, false, stream);
}

tp_status tp_linear_row_ws(const tp_mlp_desc *desc, const void *const *X, const void *const *W, const void *b,
                           const void *const *R, void *const *Y, void *workspace, size_t workspace_bytes,
                           void *stream) {
    return linear_row_impl(desc, X, W, b, R, Y, workspace, workspace_bytes, true, stream);
}

size_t tp_linear_workspace_bytes(const tp_mlp_desc *desc) {
    if (validate_desc(desc) != TP_OK) return 0;
    const size_t t = linear_tail_bytes(desc);
    return t ? linear_tail_off(desc) + t : linear_need(desc);
}

tp_status tp_linear_col_bwd(const tp_mlp_desc *desc, const void *const *dOut, const void *const *X,
                            const void *const *W, void *const *dX, void *const *dW, void *const *db, void *workspace,
                            size_t workspace_bytes, void *stream) {
    TRY(validate_desc(desc));
    if (desc->act != TP_ACT_NONE)
        return set_error(TP_ERR_UNSUPPORTED, "tp_linear_col_bwd takes act = TP_ACT_NONE (use tp_mlp_bwd)");
    const Dims x = dims_of(desc);
    if (x.M > 0) {
        TRY(check_array(dOut, x.T, "dOut"));
        TRY(check_array(X, x.nx, "X"));
        TRY(check_array(reinterpret_cast<const void *const *>(dX), x.nx, "dX"));
    }
    TRY(check_array(W, x.T, "W"));
    TRY(check_array(reinterpret_cast<const void *const *>(dW), x.T, "dW"));
    if (desc->has_bias) TRY(check_array(reinterpret_cast<const void *const *>(db), x.T, "db"));
    TRY(check_ws(desc, workspace, workspace_bytes));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (x.M == 0)
        return zero_grads(desc, dW, x.T, sizeof(float) * x.Fs * x.H, desc->has_bias ? db : nullptr, x.T,
                          sizeof(float) * x.Fs, st);
    const Scratch tail = scratch_after(workspace, workspace_bytes, linear_tail_off(desc));
    if (desc->dtype == TP_DT_FP8)
        return fp8_linear_col_bwd(desc, dOut, dX, dW, desc->has_bias ? db : nullptr, workspace, st, tail);
    TRY(column_dgrad(desc, dOut, x.Fs, W, nullptr, dX, st, tail));
    TRY(wgrad(desc, "wgrad_col", dOut, 1, x.Fs, X, 0, x.H, dW, st,
              reinterpret_cast<float *>(static_cast<char *>(workspace) + linear_part_bytes(desc)), tail));
    if (desc->has_bias)
        TRY(colsum(desc, "bias_grad_col", dOut, x.T, 1, 0, x.T, x.Fs, db, static_cast<float *>(workspace), st));
    return TP_OK;
}

tp_status tp_linear_row_bwd(const tp_mlp_desc *desc, const void *const *dY, const void *const *X,
                            const void *const *W, void *const *dX, void *const *dW, void *db, void *workspace,
                            size_t workspace_bytes, void *stream) {
    return linear_row_bwd_impl(desc, dY, X, W, dX, dW, db, workspace, workspace_bytes, stream, true);
}

}  // extern "C"

namespace tpmlp {

size_t linear_row_bias_bytes(const tp_mlp_desc *desc) {
    if (validate_desc(desc) != TP_OK || !desc->has_bias) return 0;
    return partials_bytes(desc, 1, desc->H);
}

// tp_linear_row_bwd; without allow_split the weight gradient is never split
// over tokens and the workspace need only hold the bias partials.
tp_status linear_row_bwd_impl(const tp_mlp_desc *desc, const void *const *dY, const void *const *X,
                              const void *const *W, void *const *dX, void *const *dW, void *db, void *workspace,
                              size_t workspace_bytes, void *stream, bool allow_split) {
    TRY(validate_desc(desc));
    if (desc->dtype == TP_DT_FP8 && !allow_split)
        return set_error(TP_ERR_UNSUPPORTED, "FP8 needs the workspace of the forward (tp_linear_row_bwd)");
    const Dims x = dims_of(desc);
    if (x.M > 0) {
        TRY(check_array(dY, x.nx, "dY"));
        TRY(check_array(X, x.T, "X"));
        TRY(check_array(reinterpret_cast<const void *const *>(dX), x.T, "dX"));
    }
    TRY(check_array(W, x.T, "W"));
    TRY(check_array(reinterpret_cast<const void *const *>(dW), x.T, "dW"));
    if (desc->has_bias) TRY(check_one(db, "db"));
    if (allow_split) {
        TRY(check_ws(desc, workspace, workspace_bytes));
    } else {
        const size_t need = linear_row_bias_bytes(desc);
        if (workspace_bytes < need)
            return set_error(TP_ERR_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
        if (need && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
            return set_error(TP_ERR_ARG, "workspace must be non-NULL and 256-byte aligned");
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *const *dba = reinterpret_cast<void *const *>(&db);
    if (x.M == 0)
        return zero_grads(desc, dW, x.T, sizeof(float) * x.H * x.Fs, desc->has_bias ? dba : nullptr, 1,
                          sizeof(float) * x.H, st);
    const Scratch tail = allow_split ? scratch_after(workspace, workspace_bytes, linear_tail_off(desc)) : Scratch();
    if (desc->dtype == TP_DT_FP8)
        return fp8_linear_row_bwd(desc, dY, dX, dW, desc->has_bias ? db : nullptr, workspace, st, tail);
    TRY(row_dgrad(desc, TP_ACT_NONE, dY, W, nullptr, dX, x.Fs, st, nullptr, nullptr, tail));
    float *split = allow_split ? reinterpret_cast<float *>(static_cast<char *>(workspace) + linear_part_bytes(desc))
                               : nullptr;
    TRY(wgrad(desc, "wgrad_row", dY, 0, x.H, X, 1, x.Fs, dW, st, split, tail));
    if (desc->has_bias)
        TRY(colsum(desc, "bias_grad_row", dY, x.nx, 0, x.rs, 1, x.H, dba, static_cast<float *>(workspace), st));
    return TP_OK;
}

}  // namespace tpmlp

extern "C" {

// ---------------------------------------------------------------------------
// TransformerLayer MLP sub-block: Y = X + dropout(MLP(LayerNorm(X)))
// ---------------------------------------------------------------------------
tp_status tp_layer_create(const tp_layer_desc *desc, tp_layer **out) {
    if (!out) return set_error(TP_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (!desc) return set_error(TP_ERR_ARG, "descriptor is NULL");
    TRY(validate_desc(&desc->mlp));
    if (desc->mlp.residual)
        return set_error(TP_ERR_ARG, "mlp.residual must be 0: the sub-block adds X after the dropout");
    const double p = desc->dropout_p;
    if (!(p >= 0.0 && p < 1.0)) return set_error(TP_ERR_ARG, "dropout_p=%g outside [0, 1)", p);
    if (!(desc->ln_eps > 0.0f && desc->ln_eps < 1.0e30f)) return set_error(TP_ERR_ARG, "ln_eps must be positive");
    const int ln_dtype = desc->mlp.dtype == TP_DT_F32 ? TP_DT_F32 : TP_DT_BF16;
    if (!ln_supported(desc->mlp.H, ln_dtype))
        return set_error(TP_ERR_UNSUPPORTED, "LayerNorm width H=%d above %d", desc->mlp.H,
                         ln_dtype == TP_DT_F32 ? 4096 : 8192);
    tp_layer *h = new (std::nothrow) tp_layer;
    if (!h) return set_error(TP_ERR_ARG, "out of host memory");
    h->d = *desc;
    h->inner = desc->mlp;
    h->status_slot = alloc_status_slot();
    if (h->status_slot < 0) {
        delete h;
        return set_error(TP_ERR_UNSUPPORTED, "more than %d live handles (each owns a device status word)",
                         kStatusSlots - 1);
    }
    // keep iff the draw's top 24 bits >= floor(p * 2^24); kept values scaled by 1/(1-p)
    h->drop_threshold = static_cast<uint32_t>(p * 16777216.0);
    h->drop_scale = static_cast<float>(1.0 / (1.0 - p));
    *out = h;
    return TP_OK;
}

void tp_layer_destroy(tp_layer *h) {
    if (!h) return;
    free_status_slot(h->status_slot);
    delete h;
}

// Workspace: [MLP workspace | dZ, later the LayerNorm partials | dXn, before
// that the db2 partials of the dropout backward | the dropout keep-mask the
// forward stores for the backward (bf16 / FP8 with dropout)]
struct LayerWs {
    size_t mlp, dz, dxn, mask, end;
};

static LayerWs layer_ws(const tp_layer *h) {
    const Dims x = dims_of(&h->inner);
    const size_t act = align256(static_cast<size_t>(x.M) * x.H * x.es);
    const size_t ln_part = align256(sizeof(float) * 2 * static_cast<size_t>(ln_bwd_chunks(x.M)) * x.H);
    const size_t drop_part = align256(sizeof(float) * static_cast<size_t>(dropout_bwd_chunks(x.M)) * x.H);
    LayerWs L;
    L.mlp = 0;
    L.dz = align256(mlp_ws_layout(&h->inner, nullptr));
    L.dxn = L.dz + std::max(act, ln_part);
    L.mask = L.dxn + std::max(act, drop_part);
    const bool mask = h->d.dropout_p > 0.0f && h->inner.dtype != TP_DT_F32;
    L.end = L.mask + (mask ? align256(sizeof(uint32_t) * static_cast<size_t>(x.M) * ((x.H + 31) / 32)) : 0);
    return L;
}

// ... and after them the MLP's tail-split scratch
size_t tp_layer_workspace_bytes(const tp_layer *h) {
    return h ? align256(layer_ws(h).end) + tail_scratch_bytes(&h->inner) : 0;
}

static Scratch layer_tail(const tp_layer *h, void *ws, size_t bytes) {
    return scratch_after(ws, bytes, align256(layer_ws(h).end));
}

static tp_status check_layer_ws(const tp_layer *h, void *ws, size_t bytes) {
    const size_t need = layer_ws(h).end;
    if (bytes < need) return set_error(TP_ERR_ARG, "workspace too small: %zu < %zu bytes", bytes, need);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return set_error(TP_ERR_ARG, "workspace must be non-NULL and 256-byte aligned");
    return TP_OK;
}

// shard pointers into a contiguous [M, H] buffer (1 entry without sequence parallelism)
static void split_rows(void *base, const Dims &x, void **out) {
    const size_t shard = static_cast<size_t>(x.rs) * x.H * x.es;
    for (int j = 0; j < x.nx; ++j) out[j] = static_cast<char *>(base) + j * shard;
}

static LnPlan ln_plan(const tp_layer *h) {
    const Dims x = dims_of(&h->inner);
    LnPlan lp;
    memset(lp.x, 0, sizeof(lp.x));
    memset(lp.dy, 0, sizeof(lp.dy));
    memset(lp.dx, 0, sizeof(lp.dx));
    lp.M = x.M;
    lp.H = x.H;
    lp.rows_split = x.rs;
    lp.eps = h->d.ln_eps;
    lp.drop_threshold = h->drop_threshold;
    lp.drop_scale = h->drop_scale;
    return lp;
}

tp_status tp_layer_fwd(tp_layer *h, const void *const *X, const void *gamma, const void *beta,
                       const void *const *W1, const void *const *b1, const void *const *W2, const void *b2,
                       uint64_t seed, void *const *Y, void *Xn, float *mean, float *rstd, void *const *pre,
                       void *const *A, void *workspace, size_t workspace_bytes, void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    const StatusScope scope(h->status_slot);
    const tp_mlp_desc *d = &h->inner;
    const Dims x = dims_of(d);
    TRY(check_one(gamma, "gamma"));
    TRY(check_one(beta, "beta"));
    TRY(check_array(W1, x.T, "W1"));
    TRY(check_array(W2, x.T, "W2"));
    if (d->has_bias) {
        TRY(check_array(b1, x.T, "b1"));
        TRY(check_one(b2, "b2"));
    }
    if (d->dtype == TP_DT_FP8)
        TRY(check_layer_ws(h, workspace, workspace_bytes));
    else if (!workspace || workspace_bytes < layer_ws(h).end || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        workspace = nullptr;  // optional for bf16 / fp32: used only when it is a full one
    if (x.M == 0) return TP_OK;
    TRY(check_array(X, x.nx, "X"));
    TRY(check_array(reinterpret_cast<const void *const *>(Y), x.nx, "Y"));
    TRY(check_one(Xn, "Xn"));
    TRY(check_one(mean, "mean"));
    TRY(check_one(rstd, "rstd"));
    TRY(check_array(reinterpret_cast<const void *const *>(A), x.T, "A"));
    if (d->act != TP_ACT_NONE || pre) TRY(check_array(reinterpret_cast<const void *const *>(pre), x.T, "pre"));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int ln_dtype = d->dtype == TP_DT_F32 ? TP_DT_F32 : TP_DT_BF16;
    LnPlan lp = ln_plan(h);
    for (int j = 0; j < x.nx; ++j) lp.x[j] = X[j];
    lp.xn = Xn;
    lp.gamma = gamma;
    lp.beta = beta;
    lp.mean = mean;
    lp.rstd = rstd;
    TRY(launch_ln_fwd(lp, ln_dtype, st));
    void *xn[kMaxShards];
    split_rows(Xn, x, xn);
    DropCfg dc;
    dc.on = h->d.dropout_p > 0.0f;
    dc.threshold = h->drop_threshold;
    dc.scale = h->drop_scale;
    dc.seed = seed;
    const LayerWs L = layer_ws(h);
    const bool store_mask = dc.on && workspace && L.end > L.mask;  // a full workspace: keep the flags
    if (store_mask) dc.mask = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + L.mask);
    const Fp8Recipe rc = fp8_recipe(d->dtype, h->fp8_history, h->fp8_fwd_steps);
    if (workspace) h->masks.erase(workspace);  // rewritten below, or no longer a pure function of its seed
    TRY(mlp_fwd_core(d, xn, W1, b1, W2, b2, X, Y, pre, A, workspace, &dc, st, rc,
                     layer_tail(h, workspace, workspace ? workspace_bytes : 0)));
    if (store_mask) h->masks[workspace] = seed;
    if (rc.n) ++h->fp8_fwd_steps;
    return TP_OK;
}

tp_status tp_layer_bwd(tp_layer *h, const void *const *dY, const void *const *X, const void *gamma, const void *Xn,
                       const float *mean, const float *rstd, const void *const *W1, const void *const *W2,
                       const void *const *pre, const void *const *A, uint64_t seed, void *const *dX, float *dgamma,
                       float *dbeta, void *const *dW1, void *const *db1, void *const *dW2, void *db2,
                       void *workspace, size_t workspace_bytes, void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    const StatusScope scope(h->status_slot);
    const tp_mlp_desc *d = &h->inner;
    const Dims x = dims_of(d);
    TRY(check_one(gamma, "gamma"));
    TRY(check_one(dgamma, "dgamma"));
    TRY(check_one(dbeta, "dbeta"));
    TRY(check_array(W1, x.T, "W1"));
    TRY(check_array(W2, x.T, "W2"));
    if (x.M > 0) {
        TRY(check_array(dY, x.nx, "dY"));
        TRY(check_array(X, x.nx, "X"));
        TRY(check_one(Xn, "Xn"));
        TRY(check_one(mean, "mean"));
        TRY(check_one(rstd, "rstd"));
        if (d->act != TP_ACT_NONE) TRY(check_array(pre, x.T, "pre"));
        TRY(check_array(A, x.T, "A"));
        TRY(check_array(reinterpret_cast<const void *const *>(dX), x.nx, "dX"));
    }
    TRY(check_array(reinterpret_cast<const void *const *>(dW1), x.T, "dW1"));
    TRY(check_array(reinterpret_cast<const void *const *>(dW2), x.T, "dW2"));
    if (d->has_bias) {
        TRY(check_array(reinterpret_cast<const void *const *>(db1), x.T, "db1"));
        TRY(check_one(db2, "db2"));
    }
    TRY(check_layer_ws(h, workspace, workspace_bytes));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int ln_dtype = d->dtype == TP_DT_F32 ? TP_DT_F32 : TP_DT_BF16;
    const LayerWs L = layer_ws(h);
    char *base = static_cast<char *>(workspace);
    LnPlan lp = ln_plan(h);
    lp.gamma = gamma;
    lp.dgamma = dgamma;
    lp.dbeta = dbeta;
    if (x.M == 0) {
        TRY(mlp_bwd_core(d, dY, X, W1, W2, pre, A, dX, dW1, db1, dW2, db2, base + L.mlp, st));
        return launch_ln_bwd(lp, ln_dtype, st);
    }
    for (int j = 0; j < x.nx; ++j) {
        lp.x[j] = X[j];
        lp.dy[j] = dY[j];
        lp.dx[j] = dX[j];
    }
    // dZ = dY * keep / (1 - p) and db2 = sum_m dZ (without dropout the MLP takes dY itself)
    void *dzs[kMaxShards];
    const void *dz[kMaxShards];
    const bool dropout = h->d.dropout_p > 0.0f;
    if (dropout) {
        LnPlan dp = lp;
        dp.dz = base + L.dz;
        dp.drop_seed = seed;
        dp.partials = reinterpret_cast<float *>(base + L.dxn);  // free until the MLP writes dXn
        dp.db2 = d->has_bias ? static_cast<float *>(db2) : nullptr;
        // the keep flags from the mask this handle's forward stored in this
        // workspace with this seed; otherwise redrawn from the seed
        const auto it = h->masks.find(workspace);
        if (L.end > L.mask && it != h->masks.end() && it->second == seed)
            dp.drop_mask = reinterpret_cast<const uint32_t *>(base + L.mask);
        TRY(launch_dropout_bwd(dp, ln_dtype, st));
        split_rows(dp.dz, x, dzs);
        for (int j = 0; j < x.nx; ++j) dz[j] = dzs[j];
    } else {
        for (int j = 0; j < x.nx; ++j) dz[j] = dY[j];
    }
    // MLP backward on (dZ, Xn) into dXn
    void *xn[kMaxShards], *dxn[kMaxShards];
    split_rows(const_cast<void *>(Xn), x, xn);
    split_rows(base + L.dxn, x, dxn);
    const Fp8Recipe rc = fp8_recipe(d->dtype, h->fp8_history, h->fp8_bwd_steps);
    TRY(mlp_bwd_core(d, dz, xn, W1, W2, pre, A, dxn, dW1, db1, dW2, db2, base + L.mlp, st, dropout, rc,
                     layer_tail(h, workspace, workspace_bytes)));
    if (rc.n) ++h->fp8_bwd_steps;
    // LayerNorm backward plus the residual branch: dX = dY + LN'(dXn); partials reuse the dZ region
    lp.dxn = base + L.dxn;
    lp.mean = const_cast<float *>(mean);
    lp.rstd = const_cast<float *>(rstd);
    lp.partials = reinterpret_cast<float *>(base + L.dz);
    return launch_ln_bwd(lp, ln_dtype, st);
}

tp_status tp_fp8_quantize(const void *const *in, void *const *out, const int64_t *n, int nbuf, int fmt, float *amax,
                          void *stream) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return set_error(TP_ERR_ARG, "bad FP8 format %d", fmt);
    if (nbuf < 1 || nbuf > kMaxQuantSegs) return set_error(TP_ERR_ARG, "nbuf=%d outside 1..%d", nbuf, kMaxQuantSegs);
    if (!n || !amax) return set_error(TP_ERR_ARG, "n or amax is NULL");
    TRY(check_array(in, nbuf, "in"));
    TRY(check_array(reinterpret_cast<const void *const *>(out), nbuf, "out"));
    QuantSeg segs[kMaxQuantSegs];
    for (int i = 0; i < nbuf; ++i) {
        if (n[i] < 0 || n[i] % 8) return set_error(TP_ERR_SHAPE, "n[%d]=%lld is not a non-negative multiple of 8", i, (long long)n[i]);
        segs[i] = {in[i], out[i], (long long)n[i], 0, fmt};
    }
    return launch_fp8_quantize(segs, nbuf, amax, true, static_cast<cudaStream_t>(stream));
}

static tp_status sync_slot(int slot, void *stream) {
    int v = 0;
    TRY(read_and_clear_status(static_cast<cudaStream_t>(stream), slot, &v));
    if (v == TP_OK) return TP_OK;
    return set_error(static_cast<tp_status>(v), "device reported %s", tp_status_str(static_cast<tp_status>(v)));
}

tp_status tp_sync_status(void *stream) { return sync_slot(0, stream); }

tp_status tp_mlp_sync_status(tp_mlp *h, void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    return sync_slot(h->status_slot, stream);
}

tp_status tp_layer_sync_status(tp_layer *h, void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    return sync_slot(h->status_slot, stream);
}

tp_status tp_mlp_debug_wait_timeout(tp_mlp *h, uint64_t limit_ns, void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    const StatusScope scope(h->status_slot);
    return launch_wait_timeout(limit_ns, static_cast<cudaStream_t>(stream));
}


void tp_set_wait_limit_ns(uint64_t ns) { g_wait_limit.store(ns ? ns : 1); }

tp_status tp_debug_wait_timeout(uint64_t limit_ns, void *stream) {
    const StatusScope scope(0);
    return launch_wait_timeout(limit_ns, static_cast<cudaStream_t>(stream));
}

uint64_t tp_launch_count(void) { return g_launches.load(); }

uint64_t tp_tail_split_count(void) { return tail_split_launches(); }

tp_status tp_mlp_set_fp8_history(tp_mlp *h, int n) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    if (n < 0 || n > kMaxFp8History) return set_error(TP_ERR_ARG, "history length %d outside 0..%d", n, kMaxFp8History);
    h->fp8_history = n;
    h->fp8_fwd_steps = h->fp8_bwd_steps = 0;
    return TP_OK;
}

// the amax slots of an FP8 MLP workspace (the MLP's part of a sub-block's
// workspace starts at offset 0)
static tp_status fp8_amax_copy(const tp_mlp_desc *d, const void *workspace, size_t workspace_bytes, float *out,
                               void *stream) {
    if (!out) return set_error(TP_ERR_ARG, "out is NULL");
    if (d->dtype != TP_DT_FP8) return set_error(TP_ERR_ARG, "the handle is not TP_DT_FP8");
    const Fp8Layout L = fp8_layout(d);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.end)
        return set_error(TP_ERR_ARG, "workspace must be the handle's (non-NULL, 256-byte aligned, %zu bytes)", L.end);
    const char *src = static_cast<const char *>(workspace) + L.amax;
    return cuda_check(cudaMemcpyAsync(out, src, sizeof(float) * TP_FP8_AMAX_COUNT, cudaMemcpyDefault,
                                      static_cast<cudaStream_t>(stream)),
                      "cudaMemcpyAsync(amax)");
}

tp_status tp_mlp_fp8_amax(const tp_mlp *h, const void *workspace, size_t workspace_bytes, float *out, void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    return fp8_amax_copy(&h->d, workspace, workspace_bytes, out, stream);
}

tp_status tp_layer_fp8_amax(const tp_layer *h, const void *workspace, size_t workspace_bytes, float *out,
                            void *stream) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    return fp8_amax_copy(&h->inner, workspace, workspace_bytes, out, stream);
}

tp_status tp_layer_set_fp8_history(tp_layer *h, int n) {
    if (!h) return set_error(TP_ERR_ARG, "handle is NULL");
    if (n < 0 || n > kMaxFp8History) return set_error(TP_ERR_ARG, "history length %d outside 0..%d", n, kMaxFp8History);
    h->fp8_history = n;
    h->fp8_fwd_steps = h->fp8_bwd_steps = 0;
    return TP_OK;
}

tp_status tp_set_fused_fwd(int mode) {
    if (mode != TP_FUSED_AUTO && mode != TP_FUSED_OFF && mode != TP_FUSED_ON)
        return set_error(TP_ERR_ARG, "unknown fused-forward mode %d", mode);
    set_fused_fwd_mode(mode);
    return TP_OK;
}

tp_status tp_set_tile_mode(int mode) {
    if (mode != TP_TILE_AUTO && mode != TP_TILE_SINGLE && mode != TP_TILE_PAIR)
        return set_error(TP_ERR_ARG, "unknown tile mode %d", mode);
    set_tile_mode(mode);
    return TP_OK;
}

tp_status tp_set_tail_split(int on) {
    if (on != 0 && on != 1) return set_error(TP_ERR_ARG, "tail split flag must be 0 or 1, got %d", on);
    set_tail_split(on != 0);
    return TP_OK;
}

tp_status tp_set_band_rows(int rows) {
    if (rows < 0 || rows > 4096) return set_error(TP_ERR_ARG, "band rows %d outside 0..4096", rows);
    set_band_rows(rows);
    return TP_OK;
}

tp_status tp_set_k_order(int alternate) {
    if (alternate != 0 && alternate != 1)
        return set_error(TP_ERR_ARG, "K-order flag must be 0 or 1, got %d", alternate);
    set_k_reverse(alternate != 0);
    return TP_OK;
}

tp_status tp_set_launch_overlap(int on) {
    if (on != 0 && on != 1) return set_error(TP_ERR_ARG, "launch-overlap flag must be 0 or 1, got %d", on);
    set_pdl(on != 0);
    return TP_OK;
}

tp_status tp_set_max_gemm_pairs(int n) {
    if (n < 0) return set_error(TP_ERR_ARG, "pair limit must be >= 0, got %d", n);
    set_max_gemm_pairs(n);
    return TP_OK;
}

void tp_prof_enable(int on) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_on = on != 0;
}

void tp_prof_select(const char *kernel) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_only = kernel ? kernel : "";
}

int tp_prof_collect(tp_prof_entry *entries, int max_entries) {
    std::vector<ProfRec> recs;
    std::vector<std::string> clock_names;
    {
        std::lock_guard<std::mutex> lock(g_prof_mu);
        recs.swap(g_prof_recs);
        clock_names = g_clock_names;
    }
    std::map<std::string, std::pair<int, double>> agg;
    std::vector<std::string> order;
    int rc = 0;
    for (auto &r : recs) {
        float ms = 0.0f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) rc = -1;
        if (!agg.count(r.name)) order.push_back(r.name);
        auto &e = agg[r.name];
        e.first += 1;
        e.second += ms;
    }
    {
        std::lock_guard<std::mutex> lock(g_prof_mu);
        for (auto &r : recs) {
            g_event_pool.push_back(r.a);
            g_event_pool.push_back(r.b);
        }
    }
    if (rc) {
        set_error(TP_ERR_CUDA, "event timing failed");
        return -1;
    }
    // the kernels' clock counters (only kernels launched with the timer on
    // have a slot; reading them also clears them)
    unsigned long long clk[2 * kClockSlots] = {};
    if (!clock_names.empty() && read_and_clear_clocks(clk) != TP_OK) return -1;
    // kernels counted by the clock counters but not timed by events (a
    // selection is in force) are listed after the timed ones, launches 0
    for (size_t s = 0; s < clock_names.size(); ++s)
        if (!agg.count(clock_names[s]) && (clk[2 * s] || clk[2 * s + 1])) {
            order.push_back(clock_names[s]);
            agg[clock_names[s]] = {0, 0.0};
        }
    int n = 0;
    for (auto &name : order) {
        if (!entries || n >= max_entries) break;
        tp_prof_entry &e = entries[n++];
        memset(&e, 0, sizeof(e));
        snprintf(e.name, sizeof(e.name), "%s", name.c_str());
        e.launches = agg[name].first;
        e.total_ms = agg[name].second;
        for (size_t s = 0; s < clock_names.size(); ++s)
            if (clock_names[s] == name) {
                e.sm_cycles = clk[2 * s];
                e.sm_ns = clk[2 * s + 1];
            }
    }
    return n;
}

}  // extern "C"
