/*
 * tp_mlp.h -- C ABI of the single-GPU tensor-parallel MLP library (libtpmlp.so).
 *
 * What it computes.  The Megatron tensor-parallel MLP: a ColumnParallelLinear,
 * an activation, then a RowParallelLinear ("Megatron-LM 源码精读", s3.1-s3.3
 * and the s3.3 figure; the gitcode.csdn.net walk-through, s02).  All T shards
 * live in one GPU's memory, each shard in its own buffer.  The two all-reduces
 * of the multi-GPU layer become fp32 sums over shards inside one kernel:
 *   forward  (row layer):    Y  = sum_i A_i W2_i^T + b2 [+ X]
 *   backward (column layer): dX = sum_i dPre_i W1_i     [+ dY]
 * The sequence-parallel variant ("Megatron-LM 源码精读" s3.5; walk-through s06)
 * stores X, Y, dY and dX as T token shards of [S/T, B, H]; the all-gather and
 * reduce-scatter become shard-indexed loads and stores.
 *
 * Conventions used by every entry point.
 *   Tokens.  M = S*B tokens; activations are row-major [S, B, width], i.e. a
 *     [M, width] matrix with token m = s*B + b.
 *   Weights.  PyTorch [out, in] layout; a linear layer computes X W^T
 *     ("Megatron-LM 源码精读" s3.1: weight shape [out_per_part, in]).
 *   Shards.  g = 2 for SwiGLU, else 1; Fs = F/T.
 *     W1_i : [g*Fs, H]   column shard i (SwiGLU: Fs gate rows, then Fs up rows)
 *     b1_i : [g*Fs]      sharded with W1 (same stacking)
 *     W2_i : [H, Fs]     row shard i = columns [i*Fs, (i+1)*Fs) of W2
 *     b2   : [H]         replicated, added once after the shard sum
 *     pre_i: [M, g*Fs]   pre-activation of shard i (kept for the backward)
 *     A_i  : [M, Fs]     activation of shard i (input of row shard i)
 *   Pointer arrays.  Arguments typed `const void* const*` are host arrays of
 *     device pointers, one per shard (T entries) or, for activations under
 *     sequence parallelism, one per token shard (T entries of [M/T, width]);
 *     without sequence parallelism activations take a 1-entry array.
 *   Element types.  dtype TP_DT_BF16: every activation, weight, bias and
 *     activation gradient is bf16; weight and bias gradients (dW*, db*) are
 *     fp32.  dtype TP_DT_F32: everything is fp32.  TP_DT_FP8: the buffers of
 *     TP_DT_BF16, FP8 products inside (see tp_dtype).  Products accumulate in
 *     fp32.
 *   Alignment.  Every device pointer is 16-byte aligned; H, F/T and (for the
 *     row layer input) the shard width are multiples of 8.
 *   Ownership.  The caller owns every device buffer, including the workspace.
 *     The library keeps host state only (the handle); it allocates no device
 *     memory in any entry point below.
 *   Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).
 *     Every compute entry point only enqueues work: no host synchronisation.
 *   Errors.  Argument and shape errors return before anything is enqueued.
 *     Launch failures return TP_ERR_CUDA.  A kernel whose internal wait
 *     exceeds the wait limit records TP_ERR_TIMEOUT in a device status word
 *     and returns early.  Every MLP and sub-block handle owns a status word
 *     of its own, which tp_mlp_sync_status() / tp_layer_sync_status() report
 *     (and clear); the calls without a handle (single layers, FP8 quantiser)
 *     share one word, which tp_sync_status() reports (and clears).
 *     tp_last_error() gives a message for the last failing call of the
 *     calling thread.
 */
#ifndef TP_MLP_H
#define TP_MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

#define TP_MLP_ABI_VERSION 1
#define TP_MAX_SHARDS 16

typedef enum {
    TP_OK = 0,
    TP_ERR_ARG = 1,          /* null/misaligned pointer, bad enum, bad workspace */
    TP_ERR_SHAPE = 2,        /* F % T, S % T under SP, width % 8, T range, ... */
    TP_ERR_UNSUPPORTED = 3,  /* valid request this library does not implement */
    TP_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    TP_ERR_TIMEOUT = 5       /* a kernel's bounded wait ran out (device status) */
} tp_status;

typedef enum { TP_ACT_NONE = 0, TP_ACT_GELU_TANH = 1, TP_ACT_SWIGLU = 2 } tp_act;
/* TP_DT_FP8: bf16 buffers at the interface (exactly as TP_DT_BF16), FP8 GEMMs
 * inside ("Megatron-LM 源码精读" s8.2): every GEMM operand is quantised per
 * tensor with scale = fmax / amax, the amax taken over all shards of the
 * tensor -- E4M3 (fmax 448) for X, W1, W2 and the activation A in the forward,
 * E5M2 (fmax 57344) for dY and dPre in the backward -- the products run on
 * tcgen05 kind::f8f6f4 in fp32 and are dequantised by 1/(scale_a*scale_b)
 * before the epilogue.  pre, A, Y, dX stay bf16 (and dPre, except under
 * delayed scaling, where the act' dgrad stores only its codes); bias
 * gradients sum dPre and dY before quantisation.  Needs H and F/T multiples
 * of 16, the forward through tp_mlp_fwd_ws, and the same workspace for the
 * following backward (it carries the quantised forward operands).  The single
 * layers take the same recipe per layer (current scaling): the forward
 * (tp_linear_col_ws / tp_linear_row_ws) quantises the layer's input
 * activation and weight E4M3 into the workspace, and the backward given that
 * workspace, unchanged, quantises the upstream gradient E5M2 and reuses the
 * forward's codes. */
typedef enum { TP_DT_F32 = 0, TP_DT_BF16 = 1, TP_DT_FP8 = 2 } tp_dtype;

/* Problem description shared by the MLP and the single-layer entry points.
 * For the single layers, H is the replicated width (column input, row output)
 * and F the split width (column output, row input) before sharding. */
typedef struct {
    int S, B;              /* sequence length and micro-batch: M = S*B tokens */
    int H;                 /* hidden (replicated) width */
    int F;                 /* FFN (split) width, divisible by T */
    int T;                 /* tensor-parallel size, 1..TP_MAX_SHARDS */
    int act;               /* tp_act (column layer) */
    int dtype;             /* tp_dtype */
    int has_bias;          /* b1/b2 present (column/row bias) */
    int residual;          /* row output adds a residual: MLP Y = X + MLP(X) */
    int seq_parallel;      /* activations stored as T token shards */
    int wgrad_accumulate;  /* dW += instead of dW = (gradient-accumulation fusion) */
} tp_mlp_desc;

typedef struct tp_mlp tp_mlp; /* opaque handle: validated descriptor */

/* ---- handle ------------------------------------------------------------ */

/* Validate `desc` and create a handle.  Host only: no CUDA call.  The handle
 * takes one of 1023 device status words (the walk-through s02's layer object
 * is one unit of state; here its state includes where its kernels report a
 * timeout), released by tp_mlp_destroy.
 * Returns TP_ERR_SHAPE for F % T != 0, T outside 1..TP_MAX_SHARDS, widths not
 * multiples of 8, S % T != 0 under sequence parallelism (bf16 additionally
 * needs M/T % 128 == 0 under sequence parallelism); TP_ERR_ARG for bad
 * enums, flags other than 0/1 or a null pointer; TP_ERR_UNSUPPORTED when
 * 1023 MLP and sub-block handles are already live. */
TP_API tp_status tp_mlp_create(const tp_mlp_desc *desc, tp_mlp **out);
TP_API void tp_mlp_destroy(tp_mlp *h);

/* Bytes of device workspace tp_mlp_bwd (and, for TP_DT_FP8, tp_mlp_fwd_ws)
 * needs (256-byte aligned start).  It holds dPre_i (M x g*Fs per shard, bf16
 * or fp32), fp32 partial column sums for the bias gradients, fp32 split-K
 * partial sums of the weight gradients when their outputs have few tiles and
 * many tokens (bf16 and FP8: up to 16 token splits, added in split order by a
 * reduction kernel) and, for FP8, the per-tensor amax values and the
 * quantised operands; those parts are a function of the descriptor alone and
 * are what the calls require.  After them comes the scratch of the GEMMs'
 * tail split (tp_set_tail_split), sized for the GEMM settings and the current
 * device's SM count at the time of the query: a workspace without it is
 * accepted and the split skipped. */
TP_API size_t tp_mlp_workspace_bytes(const tp_mlp *h);

/* ---- MLP forward ("Megatron-LM 源码精读" s3.3 figure) ------------------------
 * X   : 1 pointer [M, H], or T token shards [M/T, H] under seq_parallel
 * W1  : T pointers [g*Fs, H];  b1: T pointers [g*Fs] or NULL (has_bias = 0)
 * W2  : T pointers [H, Fs];    b2: [H] or NULL
 * Y   : 1 pointer [M, H], or T token shards [M/T, H] under seq_parallel
 * pre : T pointers [M, g*Fs]; may be NULL when act = TP_ACT_NONE
 * A   : T pointers [M, Fs]
 * Computes pre_i = X W1_i^T + b1_i, A_i = act(pre_i) (no reduction), then
 * Y = sum_{i=0}^{T-1} A_i W2_i^T + b2 (+ X if residual) with the sum in fp32
 * inside one kernel, in shard order. */
TP_API tp_status tp_mlp_fwd(tp_mlp *h, const void *const *X, const void *const *W1,
                     const void *const *b1, const void *const *W2, const void *b2,
                     void *const *Y, void *const *pre, void *const *A, void *stream);

/* tp_mlp_fwd with a workspace (>= tp_mlp_workspace_bytes, 256-byte aligned).
 * Required for TP_DT_FP8, where the forward quantises X, W1, W2 and A into the
 * workspace and tp_mlp_bwd must then be given the same workspace, unchanged in
 * between; for bf16 it is optional and only the row GEMM's tail-split scratch
 * is used (a NULL, unaligned or too small workspace is ignored).  TP_DT_FP8
 * through tp_mlp_fwd returns TP_ERR_ARG. */
TP_API tp_status tp_mlp_fwd_ws(tp_mlp *h, const void *const *X, const void *const *W1,
                               const void *const *b1, const void *const *W2, const void *b2,
                               void *const *Y, void *const *pre, void *const *A, void *workspace,
                               size_t workspace_bytes, void *stream);

/* FP8 scaling recipe of a TP_DT_FP8 handle ("Megatron-LM 源码精读" s2, the
 * fp8_utils.py entry: per-tensor scaling with an amax history).  n = 0
 * (default): current scaling -- every tensor is scaled from its own amax, one
 * extra read pass per tensor.  n = 1..64: delayed scaling -- each of X, W1,
 * W2, A, dY, dPre is scaled from the maximum amax its last n quantisations
 * recorded (n = 1: the previous call's), so the cast needs no amax pass (the
 * cast reduces the amax it records as it goes); the first call after this one
 * has no history and scales each tensor from its own amax.  Values beyond the
 * range a stale scale covers saturate to +-fmax.  The history lives in the
 * workspace: under delayed scaling every tp_mlp_fwd_ws / tp_mlp_bwd call of
 * the handle must get the same workspace, untouched in between.  Calling this
 * again clears the history.  Host only.  TP_ERR_ARG for n outside 0..64. */
TP_API tp_status tp_mlp_set_fp8_history(tp_mlp *h, int n);

/* The per-tensor amaxes (max |x| over all shards, fp32: the cross-shard amax
 * reduction of "Megatron-LM 源码精读" s8.2, the values the amax history of s2,
 * the fp8_utils.py entry, records) the last calls of a
 * TP_DT_FP8 handle recorded in `workspace` (the one passed to them), in the
 * order X, W1, W2, A (set by tp_mlp_fwd_ws), dY, dPre (set by tp_mlp_bwd):
 * the values that enter the scales of the next call (delayed scaling) or
 * gave this call's (current scaling).  A's and dPre's come from the GEMM
 * epilogues that produce them when their scale is known beforehand, and are
 * the max over the bf16 values they round to.  out: TP_FP8_AMAX_COUNT floats
 * in device or host memory (copied with cudaMemcpyDefault on `stream`;
 * pageable host memory makes the copy synchronous).  TP_ERR_ARG for a NULL
 * handle or out, a handle that is not TP_DT_FP8, or a workspace that is
 * NULL, unaligned or smaller than the FP8 region. */
#define TP_FP8_AMAX_COUNT 6
TP_API tp_status tp_mlp_fp8_amax(const tp_mlp *h, const void *workspace, size_t workspace_bytes, float *out,
                                 void *stream);

/* ---- MLP backward ------------------------------------------------------------
 * dY  : like Y;  X, W1, W2, pre, A: as passed to / produced by tp_mlp_fwd
 * dX  : like X (bf16/f32 per dtype)
 * dW1 : T pointers [g*Fs, H] fp32;  db1: T pointers [g*Fs] fp32 or NULL
 * dW2 : T pointers [H, Fs] fp32;    db2: [H] fp32 or NULL
 * workspace: >= tp_mlp_workspace_bytes(h) bytes of device memory, 256-byte
 *   aligned; contents on entry are ignored and on return are undefined.
 * Computes dA_i = dY W2_i and dPre_i = dA_i (.) act'(pre_i) (no reduction:
 * the row layer's backward has no communication, s3.2), dW2_i = dY^T A_i,
 * db2 = sum_m dY, dW1_i = dPre_i^T X, db1_i = sum_m dPre_i and
 * dX = sum_i dPre_i W1_i (+ dY if residual) in fp32 inside one kernel.
 * With wgrad_accumulate the weight gradients are added to dW1/dW2 (one fp32
 * add per element and call, done by bulk reduce-add stores; bias
 * gradients are always overwritten). */
TP_API tp_status tp_mlp_bwd(tp_mlp *h, const void *const *dY, const void *const *X,
                     const void *const *W1, const void *const *W2,
                     const void *const *pre, const void *const *A,
                     void *const *dX, void *const *dW1, void *const *db1,
                     void *const *dW2, void *db2, void *workspace,
                     size_t workspace_bytes, void *stream);

/* ---- single layers ("Megatron-LM 源码精读" s3.1, s3.2; walk-through s02) ------
 * tp_linear_col: out_i = act(X W_i^T + b_i) for every shard, no reduction.
 *   X: like tp_mlp_fwd's X; W: T x [g*Fs, H]; b: T x [g*Fs] or NULL;
 *   out: T x [M, Fs]; pre: T x [M, g*Fs] or NULL (not stored).
 *   TP_DT_FP8 needs tp_linear_col_ws (TP_ERR_ARG here). */
TP_API tp_status tp_linear_col(const tp_mlp_desc *desc, const void *const *X,
                        const void *const *W, const void *const *b,
                        void *const *out, void *const *pre, void *stream);

/* tp_linear_col with a workspace (>= tp_linear_workspace_bytes, 256-byte
 *   aligned).  Required for TP_DT_FP8 ("Megatron-LM 源码精读" s8.2): X and the
 *   W shards are quantised E4M3, each with one scale over all its shards,
 *   into the workspace, and out_i = act(Xq Wq_i^T / (s_x s_w) + b_i) with pre
 *   and out stored bf16; tp_linear_col_bwd must then get the same workspace,
 *   unchanged.  For bf16 / fp32 the workspace is not used. */
TP_API tp_status tp_linear_col_ws(const tp_mlp_desc *desc, const void *const *X,
                                  const void *const *W, const void *const *b,
                                  void *const *out, void *const *pre, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* tp_linear_row: Y = sum_i X_i W_i^T + b (+ R), the sum over shards in fp32
 *   inside one kernel.  X: T x [M, Fs]; W: T x [H, Fs]; b: [H] or NULL;
 *   R: like Y, or NULL (required iff desc->residual); Y: 1 x [M, H] or T token
 *   shards under seq_parallel.  desc->act is ignored.  TP_DT_FP8 needs
 *   tp_linear_row_ws (TP_ERR_ARG here). */
TP_API tp_status tp_linear_row(const tp_mlp_desc *desc, const void *const *X,
                        const void *const *W, const void *b,
                        const void *const *R, void *const *Y, void *stream);

/* tp_linear_row with a workspace (>= tp_linear_workspace_bytes, 256-byte
 *   aligned).  Required for TP_DT_FP8: the X and W shards are quantised E4M3
 *   (one scale per tensor over its shards) into the workspace and
 *   Y = sum_i Xq_i Wq_i^T / (s_x s_w) + b (+ R); tp_linear_row_bwd must then
 *   get the same workspace, unchanged.  For bf16 the workspace's tail-split
 *   scratch lets the row GEMM split its last round (tp_set_tail_split); a
 *   workspace smaller than what tp_linear_row_bwd requires is ignored. */
TP_API tp_status tp_linear_row_ws(const tp_mlp_desc *desc, const void *const *X,
                                  const void *const *W, const void *b,
                                  const void *const *R, void *const *Y, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Workspace bytes for the single layers: bias partials, then split-K partials
 * of the weight gradient (as for tp_mlp_bwd), then for TP_DT_FP8 the amax
 * slots and the codes of the layer's input activation, weight and upstream
 * gradient, then the tail-split scratch of the bf16 / FP8 pair GEMMs
 * (optional, as for tp_mlp_workspace_bytes).  One size serves a column and a
 * row layer of the descriptor. */
TP_API size_t tp_linear_workspace_bytes(const tp_mlp_desc *desc);

/* tp_linear_col_bwd: gradients of tp_linear_col with act = TP_ACT_NONE
 *   (TP_ERR_UNSUPPORTED otherwise; the fused activation backward belongs to
 *   tp_mlp_bwd).  dOut: T x [M, Fs]; X, W as in the forward;
 *   dX = sum_i dOut_i W_i (fp32 sum over shards in one kernel), stored like X;
 *   dW_i = dOut_i^T X (fp32, T x [Fs, H]); db_i = sum_m dOut_i (fp32) or NULL.
 *   TP_DT_FP8: the workspace of the tp_linear_col_ws call, unchanged; dOut is
 *   quantised E5M2 (one scale over its shards) and the products use the
 *   forward's codes of X and W; db sums the unquantised dOut. */
TP_API tp_status tp_linear_col_bwd(const tp_mlp_desc *desc, const void *const *dOut,
                            const void *const *X, const void *const *W,
                            void *const *dX, void *const *dW, void *const *db,
                            void *workspace, size_t workspace_bytes, void *stream);

/* tp_linear_row_bwd: gradients of tp_linear_row (no reduction over shards).
 *   dY: like Y; X, W as in the forward; dX_i = dY W_i (T x [M, Fs]);
 *   dW_i = dY^T X_i (fp32, T x [H, Fs]); db = sum_m dY (fp32 [H]) or NULL.
 *   The residual's gradient is dY itself and is not materialised.
 *   TP_DT_FP8: the workspace of the tp_linear_row_ws call, unchanged; dY is
 *   quantised E5M2 and the products use the forward's codes of X and W; db
 *   sums the unquantised dY. */
TP_API tp_status tp_linear_row_bwd(const tp_mlp_desc *desc, const void *const *dY,
                            const void *const *X, const void *const *W,
                            void *const *dX, void *const *dW, void *db,
                            void *workspace, size_t workspace_bytes, void *stream);

/* tp_linear_row_bwd_noalloc: tp_linear_row_bwd without a caller workspace.
 *   The pages have no counterpart: this entry point exists for callers that
 *   cannot allocate device memory when they call -- a plugin that is handed
 *   only the op's tensors and has no allocator of its own, a process whose
 *   device memory is fully reserved by another (caching) allocator, or a
 *   latency-critical loop that cannot take cudaMalloc's implicit device
 *   synchronisation.  It allocates nothing: its scratch is a 4 MiB array
 *   compiled into the library (held on every GPU that loads the library until
 *   the process exits).  Arguments are those of tp_linear_row_bwd minus the
 *   workspace.  Two regimes:
 *   - tp_linear_workspace_bytes(desc) <= 4 MiB: the array serves as that
 *     workspace, and the call runs exactly the plan of tp_linear_row_bwd
 *     (split-K and tail split of the weight gradient included), with the
 *     same results bit for bit;
 *   - otherwise the weight gradient runs without token splitting and without
 *     the tail split, and the array holds only the bias-gradient partials
 *     (results differ from tp_linear_row_bwd by fp32 summation order where
 *     that call splits).
 *   A problem whose bias partials exceed 4 MiB (4 * ceil(M/256) * H bytes,
 *   rounded up to 256, when has_bias) returns TP_ERR_UNSUPPORTED, and so does
 *   TP_DT_FP8 (its backward needs the forward's workspace).
 *   The device address of the array is looked up on the first call per
 *   device and CUDA context (with that device current); make that first call
 *   before any stream capture.  All calls share the one array and each call
 *   overwrites the part it reads (nothing needs to start at zero), so calls
 *   that overlap on the GPU -- on different streams, or from several host
 *   threads -- race. */
TP_API tp_status tp_linear_row_bwd_noalloc(const tp_mlp_desc *desc, const void *const *dY,
                                           const void *const *X, const void *const *W,
                                           void *const *dX, void *const *dW, void *db,
                                           void *stream);

/* ---- TransformerLayer MLP sub-block (walk-through s03; "Megatron-LM 源码精读"
 * s3.5) ---------------------------------------------------------------------
 * The MLP half of a transformer layer, on the tensor-parallel MLP above:
 *   Xn = LayerNorm(X; gamma, beta)  per token over H: (x - mean) * rstd *
 *                                   gamma + beta, population variance,
 *                                   rstd = 1 / sqrt(var + ln_eps)
 *   Z  = MLP(Xn)                    as tp_mlp_fwd (b2 included), no residual
 *   Y  = X + dropout_p(Z)           bias-dropout-add; the residual is X
 * Dropout: element (m, h) of Z, m the global token index (sequence sharding
 * does not change it), uses word e mod 4 of Philox4x32-10 (Salmon et al.,
 * SC 2011) with counter (q mod 2^32, q div 2^32, 0, 0), q = e div 4,
 * e = m*H + h, and key (seed mod 2^32, seed div 2^32); it is kept iff the
 * word's top 24 bits are >= floor(p * 2^24) and kept values are scaled by
 * 1/(1-p).  The backward redraws the flags from the same seed.  p = 0 skips
 * the dropout.  Under sequence parallelism X, Y, dY and dX are T token shards
 * as in the MLP; Xn is one contiguous [M, H] buffer (the gathered LayerNorm
 * output the column layer reads). */
typedef struct {
    tp_mlp_desc mlp;  /* the MLP; mlp.residual must be 0 (the block adds X) */
    float dropout_p;  /* in [0, 1) */
    float ln_eps;     /* > 0 (1e-5 in Megatron) */
} tp_layer_desc;

typedef struct tp_layer tp_layer;

/* Validate and create (host only; takes a status word like tp_mlp_create).
 * Besides tp_mlp_create's checks: TP_ERR_ARG
 * for mlp.residual != 0, p outside [0, 1) or ln_eps <= 0; TP_ERR_UNSUPPORTED
 * for H above 8192 (bf16, FP8) or 4096 (fp32), the LayerNorm kernels' row
 * capacity. */
TP_API tp_status tp_layer_create(const tp_layer_desc *desc, tp_layer **out);
TP_API void tp_layer_destroy(tp_layer *h);

/* Bytes of device workspace for tp_layer_bwd (and, for TP_DT_FP8,
 * tp_layer_fwd, whose quantised operands the backward reads from it): the
 * MLP's workspace, dZ and dXn ([M, H] each), the dropout keep-mask (bf16 and
 * FP8 with dropout: one bit per element, ceil(H/32) 32-bit words per row),
 * then the MLP GEMMs' tail-split scratch (optional, as for
 * tp_mlp_workspace_bytes). */
TP_API size_t tp_layer_workspace_bytes(const tp_layer *h);

/* FP8 scaling recipe of a TP_DT_FP8 sub-block: as tp_mlp_set_fp8_history
 * (the history lives in the sub-block's workspace, which every
 * tp_layer_fwd / tp_layer_bwd call must then get, untouched in between). */
TP_API tp_status tp_layer_set_fp8_history(tp_layer *h, int n);

/* The per-tensor amaxes a TP_DT_FP8 sub-block's last calls recorded in
 * `workspace`, as tp_mlp_fp8_amax returns them for the MLP inside: X is the
 * LayerNorm output that enters the MLP and dY the gradient at the MLP's
 * output (after the dropout backward).  Same arguments and errors as
 * tp_mlp_fp8_amax. */
TP_API tp_status tp_layer_fp8_amax(const tp_layer *h, const void *workspace, size_t workspace_bytes, float *out,
                                   void *stream);

/* Forward.  X, Y: like tp_mlp_fwd's X and Y; gamma, beta: [H] (bf16, fp32 for
 * TP_DT_F32); W1, b1, W2, b2, pre, A: as in tp_mlp_fwd; seed: dropout key.
 * Outputs kept for the backward: Xn [M, H] (activation dtype), mean and rstd
 * [M] fp32, pre, A.  workspace: required (>= tp_layer_workspace_bytes,
 * 256-byte aligned) for TP_DT_FP8 and then passed unchanged to tp_layer_bwd;
 * optional otherwise (may be NULL).  With dropout (bf16, FP8) the forward
 * stores its keep flags in the workspace, and a tp_layer_bwd of the same
 * handle given the same workspace and the same seed reads them instead of
 * redrawing them from the Philox stream (the same flags either way; the
 * backward of the dropout becomes a pure HBM pass).  The backward checks
 * each block's first row of the mask against the Philox stream and redraws
 * the flags where it does not match, so a workspace changed in between costs
 * time, not correctness. */
TP_API tp_status tp_layer_fwd(tp_layer *h, const void *const *X, const void *gamma, const void *beta,
                              const void *const *W1, const void *const *b1, const void *const *W2,
                              const void *b2, uint64_t seed, void *const *Y, void *Xn, float *mean,
                              float *rstd, void *const *pre, void *const *A, void *workspace,
                              size_t workspace_bytes, void *stream);

/* Backward.  dY, dX: like Y and X; X, gamma, Xn, mean, rstd, W1, W2, pre, A
 * and seed: as given to / produced by tp_layer_fwd.  Computes
 *   dZ  = dY * keep / (1 - p),
 *   the MLP backward on (dZ, Xn): dW1, db1, dW2, db2 exactly as tp_mlp_bwd
 *     (fp32, wgrad_accumulate honoured) and dXn,
 *   dX  = dY + rstd * (g - mean_h(g) - xhat * mean_h(g * xhat)) with
 *         g = dXn * gamma, xhat = (X - mean) * rstd,
 *   dgamma = sum_m dXn * xhat, dbeta = sum_m dXn ([H] fp32, overwritten).
 * workspace: >= tp_layer_workspace_bytes, 256-byte aligned. */
TP_API tp_status tp_layer_bwd(tp_layer *h, const void *const *dY, const void *const *X, const void *gamma,
                              const void *Xn, const float *mean, const float *rstd,
                              const void *const *W1, const void *const *W2, const void *const *pre,
                              const void *const *A, uint64_t seed, void *const *dX, float *dgamma,
                              float *dbeta, void *const *dW1, void *const *db1, void *const *dW2,
                              void *db2, void *workspace, size_t workspace_bytes, void *stream);

/* Per-tensor FP8 quantisation of one logical tensor split over `nbuf` bf16
 * buffers (its shards): amax = max |x| over all buffers (the cross-shard amax
 * reduction), scale = fmax / amax in fp32 (1 if amax is 0), then
 * out_k = fp8(in_k * scale) with round-to-nearest-even, saturating to +-fmax
 * ("Megatron-LM 源码精读" s8.2).  fmt: 0 = E4M3 (fmax 448), 1 = E5M2 (57344).
 * in/out: nbuf (<= 40) pointers, buffer k holding n[k] elements (n[k] % 8 == 0;
 * out one byte per element).  amax: one device float, overwritten.  This is
 * the quantiser the TP_DT_FP8 path uses for every operand. */
TP_API tp_status tp_fp8_quantize(const void *const *in, void *const *out, const int64_t *n, int nbuf,
                                 int fmt, float *amax, void *stream);

/* ---- status, limits, diagnostics ---------------------------------------- */

/* Synchronise `stream`, then read and clear the status word shared by the
 * calls without a handle (tp_linear_*, tp_fp8_quantize,
 * tp_debug_wait_timeout).  Returns TP_OK, TP_ERR_TIMEOUT (a bounded wait ran
 * out) or TP_ERR_CUDA. */
TP_API tp_status tp_sync_status(void *stream);

/* Synchronise `stream`, then read and clear the status word of handle h:
 * TP_ERR_TIMEOUT iff a kernel launched by one of h's calls (tp_mlp_fwd,
 * tp_mlp_fwd_ws, tp_mlp_bwd; tp_layer_fwd, tp_layer_bwd) ran out of its wait
 * limit since the last read.  Launches of other handles, on this or other
 * streams, neither set nor clear it.  TP_ERR_ARG for a NULL handle,
 * TP_ERR_CUDA when the synchronisation or the read fails. */
TP_API tp_status tp_mlp_sync_status(tp_mlp *h, void *stream);
TP_API tp_status tp_layer_sync_status(tp_layer *h, void *stream);

/* Wall-clock bound of every in-kernel wait, in nanoseconds (default 4e9).
 * Applies to launches made after the call. */
TP_API void tp_set_wait_limit_ns(uint64_t ns);

/* Launch a kernel that waits for a device flag nothing ever sets, bounded by
 * limit_ns; it records TP_ERR_TIMEOUT in the status word and returns.  Used
 * to test the failure path without faulting or hanging the GPU. */
TP_API tp_status tp_debug_wait_timeout(uint64_t limit_ns, void *stream);

/* As tp_debug_wait_timeout, reporting to the status word of handle h (read
 * with tp_mlp_sync_status): tests that a timeout reaches only its handle. */
TP_API tp_status tp_mlp_debug_wait_timeout(tp_mlp *h, uint64_t limit_ns, void *stream);

/* GEMM tiling of the bf16 engine, for all launches made after the call:
 * TP_TILE_AUTO (default) uses 256-row tiles computed by a pair of CTAs on two
 * SMs (tcgen05 cta_group::2) whenever M > 128, else 128-row single-CTA tiles;
 * TP_TILE_SINGLE / TP_TILE_PAIR force one or the other.  Both accumulate every
 * output element over K in the same order.  Returns TP_ERR_ARG for an unknown
 * mode. */
typedef enum { TP_TILE_AUTO = 0, TP_TILE_SINGLE = 1, TP_TILE_PAIR = 2 } tp_tile_mode;
TP_API tp_status tp_set_tile_mode(int mode);

/* Tail split of the pair-tile GEMMs, for all launches made after the call
 * (on = 1, the default; 0 turns it off).  The pair kernels are persistent:
 * P CTA pairs take the tiles round-robin, so when the tile count is not a
 * multiple of P the last round runs part-filled (GPT-size weight gradients:
 * 1024 tiles on 76 pairs, 13.5 rounds in the time of 14).  When that round
 * holds rem <= P/2 tiles, the split cuts each of them along K into
 * s = min(P / rem, 4) units that run side by side in one round; every unit
 * parks its fp32 partial sum in the workspace and the last unit of each
 * 32 x 128 slice to finish adds the slices in unit order and runs the tile's
 * epilogue.  No unit waits for another.  Only whole-tile output GEMMs that
 * run after at least one full round split (row forward, column dgrad, weight
 * gradients, single-layer dgrads), and only when the call has the scratch:
 * tp_mlp_workspace_bytes,
 * tp_linear_workspace_bytes and tp_layer_workspace_bytes include it at the
 * end of the workspace, sized for the settings and device current at the
 * query; a workspace without it (or the plain tp_mlp_fwd) skips the split.
 * Split tiles sum K in another grouping, so they differ from unsplit ones by
 * fp32 rounding; a given configuration is run-to-run deterministic.
 * TP_ERR_ARG unless on is 0 or 1. */
TP_API tp_status tp_set_tail_split(int on);

/* K order of the pair-tile GEMMs' whole tiles, for all launches made after
 * the call.  The persistent CTA pairs take their tiles round by round, and
 * consecutive rounds share operand panels (the same band of row tiles and a
 * column tile).  With alternate = 1 (the default) the row forward, the
 * column dgrads and the weight gradients walk the K loop of every other
 * round from its last block down, so that a round starts on the K blocks
 * the previous round loaded last, which are still in L2, instead of on the
 * ones L2 has already evicted: fewer operand re-reads from HBM.  Such tiles
 * add the same products over K in the reverse order (fp32 rounding differs;
 * a given configuration is run-to-run deterministic).  alternate = 0 walks
 * every tile forwards.  TP_ERR_ARG unless alternate is 0 or 1. */
TP_API tp_status tp_set_k_order(int alternate);

/* Tile order of the pair-tile GEMMs, for all launches made after the call:
 * output tiles are taken in bands of `rows` rows of 256-row tiles, the row
 * fastest within a band and the columns of all problems side by side.  A
 * band's operand panels are what a round of the persistent grid shares in
 * L2, so the band height trades re-reads of the A panels (one per band)
 * against re-reads of the B panels (once per band).  0 (the default) picks
 * the library's choice.  TP_ERR_ARG for rows outside 0..4096. */
TP_API tp_status tp_set_band_rows(int rows);

/* Programmatic dependent launch of the pair-tile GEMMs, for all launches
 * made after the call.  With on = 1 (the default) each pair-tile GEMM is
 * launched with programmatic stream serialization: its CTAs may start on
 * SMs the previous kernel in the stream has left, set up their barriers and
 * tensor memory there, and wait in griddepcontrol.wait until that kernel
 * has completed and its writes are visible before they read an operand or
 * write an output, so stream order and results are unchanged.  on = 0
 * launches them in plain stream order.  TP_ERR_ARG unless on is 0 or 1. */
TP_API tp_status tp_set_launch_overlap(int on);

/* Upper bound on the CTA pairs of the persistent pair-tile GEMMs, for all
 * launches made after the call (0, the default: as many as fit on the
 * device).  Leaves SMs free for concurrent work and sets the round structure
 * the tail split sees.  TP_ERR_ARG for n < 0. */
TP_API tp_status tp_set_max_gemm_pairs(int n);

/* Forward of the MLP (and of the sub-block) as one fused kernel, for all
 * calls made after this one.  The fused kernel keeps a 128-token tile's
 * output [128 x H] in tensor memory and streams the F dimension through it
 * in 128-unit chunks: per chunk the column GEMM, bias and activation (pre and
 * A are still stored for the backward), then A goes from shared memory
 * straight into the row GEMM, so A is never read back from HBM.  It takes
 * bf16 with H a multiple of 64 up to 256 and act = none or GeLU-tanh with F/T
 * a multiple of 128, or SwiGLU with F/T a multiple of 64 (a chunk is then 64
 * gate and the 64 matching up units); other problems always use the
 * two-kernel path.  With a
 * workspace (tp_mlp_fwd_ws, tp_layer_fwd) of the size the handle reports,
 * the work is split evenly over the SMs when the token tiles spill over a
 * whole number of rounds of the SMs by at most a quarter of a round.
 * TP_FUSED_AUTO (default) and TP_FUSED_ON run the fused kernel for every
 * problem it takes (on GB300 it measured faster than the two GEMMs from 16 to
 * 2048 128-token tiles: 124 us against 155 us for 65536 tokens at H = 256,
 * F = 1024, T = 2), TP_FUSED_OFF never.  pre and A are bit-identical
 * between the paths; Y accumulates the same fp32 products in another order.
 * The pre buffers take 32-byte stores when they are 32-byte aligned (16-byte
 * ones otherwise).  Returns TP_ERR_ARG for an unknown mode. */
typedef enum { TP_FUSED_AUTO = 0, TP_FUSED_OFF = 1, TP_FUSED_ON = 2 } tp_fused_mode;
TP_API tp_status tp_set_fused_fwd(int mode);

/* Number of kernels this library has launched since load. */
TP_API uint64_t tp_launch_count(void);

/* Number of pair-tile GEMM launches since load that split their last round's
 * tiles (tp_set_tail_split). */
TP_API uint64_t tp_tail_split_count(void);

/* Per-kernel timing ("timers"): when enabled, every launch is bracketed by
 * CUDA events recorded on its own stream, and the GEMM kernels count their
 * CTAs' SM cycles and nanoseconds.  tp_prof_collect synchronises the
 * recorded events (and, when there are clock counts, the device) and
 * returns, per kernel name, launches, total device milliseconds and the
 * clock counts; it then clears the records.  Returns the number of entries
 * written (<= max_entries) or -1 on error. */
typedef struct {
    char name[48];
    int launches;
    double total_ms;
    /* GEMM kernels: SM cycles (clock64) and nanoseconds (%globaltimer)
     * between the start and the end of every CTA, summed over the CTAs of
     * the recorded launches: sm_cycles / sm_ns * 1000 is the SM clock in
     * MHz they ran at; 0 for kernels without the counter. */
    uint64_t sm_cycles;
    uint64_t sm_ns;
} tp_prof_entry;
TP_API void tp_prof_enable(int on);
TP_API int tp_prof_collect(tp_prof_entry *entries, int max_entries);
/* Restrict the timers' events to the launches of one kernel (its name as
 * tp_prof_collect reports it); NULL or "" times every launch again.  The
 * other launches then carry no events in their stream (each event pair
 * costs the stream a few microseconds between kernels), while the GEMMs'
 * clock counters keep counting: tp_prof_collect lists such kernels after the
 * timed ones with launches = 0 and total_ms = 0.  The string is copied. */
TP_API void tp_prof_select(const char *kernel);

TP_API const char *tp_status_str(tp_status s);
TP_API const char *tp_last_error(void);
TP_API int tp_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TP_MLP_H */
