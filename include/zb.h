/*
 * zb.h - C ABI of libzb: the split backward (B / W) of one Zero-Bubble
 * pipeline stage, on one GB300 (sm_103a).
 *
 * Sources (page title, section):
 *  [G1] "Zero-Bubble Pipeline Parallelism Guide for LLMs", section
 *       "Core Innovation 1: Mathematical Decomposition of the Backward Pass":
 *       for Y = X W the backward splits into B, the input gradient
 *       dX = dY W^T (critical path: the previous stage waits for it), and W,
 *       the weight gradient dW = X^T dY (local; only the optimizer step
 *       needs it, so it can be deferred).
 *  [G2] same page, section "Step-by-Step Implementation": weights are stored
 *       [out, in] and y = x W^T; the forward keeps x, B keeps dY and returns
 *       dY W, W pops x and dY and adds dY^T x into the weight gradient.
 *  [G3] same page, section "Memory Management & Activation Rollback": an
 *       activation is freed only after its W; a hard ceiling bounds the
 *       microbatches whose activations are held; weight gradients are
 *       accumulated in place in fixed buffers.
 *  [G4] same page, section "Core Innovation 2: The Zero-Bubble Scheduling
 *       Family" (ZB-1F1B: 1F1B memory, F and B first, W fills idle slots,
 *       steady F -> B -> W, W drained at the end) and the bubble formulas of
 *       section "Mathematical Modeling: Bubble Fractions, Memory Bounds, and
 *       Speedups".
 *
 * Conventions for every call:
 *  - bf16 tensors are passed as `void*` / `const void*` to 16-bit storage;
 *    float tensors as `float*`.  All matrices are row-major and dense (the row
 *    stride equals the row length).  "[T, n]" means T rows of n elements;
 *    T is the number of tokens of one microbatch.
 *  - Tensor pointers are DEVICE pointers on the current CUDA device, 16-byte
 *    aligned.  The caller owns every buffer; the library never allocates
 *    device memory on these paths.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call only enqueues work on `stream` and returns; results are valid once
 *    the stream reaches that point.
 *  - Arguments are checked on the host before anything is enqueued.  A call
 *    that returns an error has enqueued nothing and changed no state.
 *  - Feature sizes (hidden, ffn, in/out features, head_dim * heads) must be
 *    positive multiples of 64; tokens may be any value >= 0 (0 enqueues
 *    nothing).  Other sizes return ZB_ERR_SHAPE.
 *  - Kernels never wait without a limit.  A wait that runs out sets a device
 *    status word, the kernel returns early, and the next zb_device_status()
 *    or zb_stage_sync() reports ZB_ERR_DEVICE_TIMEOUT.
 *  - Not thread-safe: calls on one zb_stage_t must come from one host thread
 *    and one stream (or be ordered by the caller).
 *  - The library keeps, per device, the addresses of its own device variables
 *    (the status word, the array of the _noalloc call).  cudaDeviceReset() on
 *    a device invalidates them: do not use the library on that device again in
 *    the same process afterwards.
 */
#ifndef ZB_H_
#define ZB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZB_OK = 0,
    ZB_ERR_ARG = -1,            /* null pointer, bad enum, negative size */
    ZB_ERR_SHAPE = -2,          /* a size is not supported (see conventions) */
    ZB_ERR_ORDER = -3,          /* F -> B -> W order of one microbatch broken */
    ZB_ERR_STASH_FULL = -4,     /* F while max_inflight microbatches are held */
    ZB_ERR_NO_MB = -5,          /* microbatch id unknown to the stage */
    ZB_ERR_CUDA = -6,           /* a CUDA runtime call failed */
    ZB_ERR_DEVICE_TIMEOUT = -7, /* a kernel wait ran out (device status word) */
    ZB_ERR_CAPACITY = -8,       /* output array of zb_schedule too small */
    ZB_ERR_DEVICE = -9,         /* current device is not sm_103 */
    ZB_ERR_WORKSPACE = -10      /* workspace or scratch too small / misaligned */
} zb_status;

/* Readable name of a status code (static string). */
const char* zb_status_string(zb_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t zb_version(void);

/* ========================================================================
 * F/B/W order of one pipeline stage (CPU only, no device calls)
 * ====================================================================== */

typedef enum {
    ZB_SCHED_1F1B = 0,  /* [G4] and the guide's section "2. The 1F1B ...":
                           stage s runs p-s forwards, then alternates B and F;
                           each W right after its B */
    ZB_SCHED_ZBH1 = 1,  /* [G4] ZB-1F1B: 1F1B order of F and B, W deferred into
                           slots that would idle, at most p microbatches held */
    ZB_SCHED_GPIPE = 2, /* the guide's section "1. The GPipe Bubble": all F,
                           then each B followed by its W */
    ZB_SCHED_ZB2P = 3   /* [G4] ZB-2p: the ZB-H1 policy with 2(p-s)-1 warm-up
                           forwards and at most 2p microbatches held; no idle
                           inside any stage's own window when m >= 2p - 1 */
} zb_sched_kind;

typedef struct {
    uint8_t kind;   /* 'F', 'B' or 'W' */
    uint8_t pad[3];
    int32_t mb;     /* microbatch id, 0 .. m-1 */
} zb_op;

/* Order of the 3m ops that stage `stage` (0 = first) of a p-stage pipeline
 * runs for m microbatches.  Writes min(cap, 3m) ops to `out` and 3m to
 * `*n_out`.  Errors: ZB_ERR_ARG (p < 1, m < 1, stage outside [0, p),
 * null n_out, out null with cap > 0); ZB_ERR_CAPACITY when cap < 3m (then
 * *n_out = 3m and nothing is written).  For ZB-H1 with m >= p the order is
 * emitted in closed form; with m < p, and for ZB-2p, it comes from a
 * unit-time run of the policy.  All give every W after its B after its F. */
zb_status zb_schedule(zb_sched_kind kind, int32_t stage, int32_t p, int32_t m,
                      zb_op* out, int32_t cap, int32_t* n_out);

/* Unit-time model of the whole pipeline (every op one unit, free
 * communication; without the B/W split a stage sends its input gradient
 * only after B and W), following section "Mathematical Modeling".  Returns
 * the makespan in units and the bubble as idle / compute summed over the p
 * stages (e.g. 1F1B at p=8, m=16: 7/16).  Any output pointer may be NULL. */
zb_status zb_schedule_bubble(zb_sched_kind kind, int32_t p, int32_t m,
                             int32_t* makespan, double* idle_over_compute,
                             double* idle_over_wall);

/* Same model, idle counted inside each stage's own window (from its first op's
 * start to its last op's end) instead of over the common makespan: the sense
 * in which the guide's section "Core Innovation 2" says ZB-2p leaves every GPU
 * busy.  Returns the summed idle units and idle / compute.  Any output
 * pointer may be NULL. */
zb_status zb_schedule_window_idle(zb_sched_kind kind, int32_t p, int32_t m,
                                  int64_t* idle_units, double* idle_over_compute);

/* Memory-limited ZB order with measured op times.  "Zero Bubble Pipeline
 * Parallelism" (the abstract: an algorithm finds the best schedule for a
 * given configuration and memory limit) and the guide's section "Core
 * Innovation 2" (ZB-H1 holds p microbatches, ZB-2p 2p).  Reading: for each
 * ceiling L in [p, min(2p, mem_limit)], the ZB-H1 policy holding at most L
 * microbatches, with min(L - s, 2(p - s) - 1) forwards before the first B of
 * stage s (ZB-H1 at L = p, ZB-2p at L = 2p), run on all p stages with F, B and
 * W taking t_f, t_b and t_w (positive integers in any one unit; communication
 * free).  The L whose run ends first wins (the smallest on ties); `out` gets
 * stage `stage`'s order under it.  *chosen_limit and *makespan (in the unit of
 * the durations) are written when not NULL.
 * Errors: ZB_ERR_ARG (mem_limit < p, a duration < 1, p m > 2^20, bad stage),
 * ZB_ERR_CAPACITY (cap < 3m; *n_out = 3m). */
zb_status zb_schedule_search(int32_t stage, int32_t p, int32_t m, int32_t mem_limit, int32_t t_f,
                             int32_t t_b, int32_t t_w, zb_op* out, int32_t cap, int32_t* n_out,
                             int32_t* chosen_limit, int64_t* makespan);

/* ========================================================================
 * Per-step operations (stateless).  One call per step of the hot path; the
 * stage calls below are built from exactly these launches.
 * ====================================================================== */

/* F, one linear [G2]: y[T,out] = x[T,in] w[out,in]^T, plus residual[T,out]
 * when `residual` is not NULL (y may alias residual).  bf16 in and out,
 * float32 accumulation in tensor memory. */
zb_status zb_op_linear_forward(const void* x, const void* w, const void* residual,
                               void* y, int32_t tokens, int32_t in_features,
                               int32_t out_features, void* stream);

/* B, one linear [G1][G2]: dx[T,in] = dy[T,out] w[out,in].  bf16. */
zb_status zb_op_backward_input(const void* dy, const void* w, void* dx,
                               int32_t tokens, int32_t in_features,
                               int32_t out_features, void* stream);

/* B of the SwiGLU down projection with the SwiGLU backward in the GEMM
 * epilogue: ds = dy[T,H] w_down[H,F]; with g = gu[:, :F], u = gu[:, F:],
 *   dgu[:, :F] = ds * u * sig(g) * (1 + g (1 - sig(g))),  dgu[:, F:] = ds * silu(g).
 * `dgu` may equal `gu` (in place).  bf16 in and out, float32 epilogue. */
zb_status zb_op_backward_input_swiglu(const void* dy, const void* w_down,
                                      const void* gu, void* dgu, int32_t tokens,
                                      int32_t hidden, int32_t ffn, void* stream);

/* B of a linear that reads an RMSNorm output, then the RMSNorm backward:
 *   dn[T,H] = dy[T,out] w[out,H]
 *   dx[T,H] = dres[T,H] + r * (gamma * dn - xh * mean_j(gamma_j dn_j xh_j)),
 *   xh = x * r, r = rstd[T] (float32), gamma[H] float32.
 * dn is written (bf16) because W needs it for the gamma gradient. */
zb_status zb_op_backward_input_rmsnorm(const void* dy, const void* w, const void* x,
                                       const float* rstd, const float* gamma,
                                       const void* dres, void* dn, void* dx,
                                       int32_t tokens, int32_t hidden, int32_t out_features,
                                       void* stream);

/* B of the attention output projection followed by the backward of the
 * weight-free attention stand-in (a_h = q_h + k_j + v_j, j = h / (nh/nkv)):
 *   da = dh[T,H] w_o[H,H];  dqkv[:, q] = da;  dqkv[:, k_j] = dqkv[:, v_j] = sum_{h in j} da_h.
 * dqkv is [T, (nh + 2 nkv) hd], bf16. */
zb_status zb_op_backward_input_attention(const void* dh, const void* w_o, void* dqkv,
                                         int32_t tokens, int32_t n_heads,
                                         int32_t n_kv_heads, int32_t head_dim,
                                         void* stream);

/* W, one linear [G1][G2][G3]: dw[out,in] (float32) += dy[T,out]^T x[T,in].
 * The contraction runs over the T tokens; each element of dw receives one
 * float32 add per call, so results are bitwise reproducible. */
zb_status zb_op_backward_weight(const void* dy, const void* x, float* dw,
                                int32_t tokens, int32_t in_features,
                                int32_t out_features, void* stream);

/* W of n (1..16) linears over the same tokens in one launch, [G1]: for each i,
 * dw[i][out_i, in_i] (float32) += dy[i][T, out_i]^T x[i][T, in_i].  The arrays
 * are host arrays of device pointers and sizes.  The products are independent
 * (outputs must not overlap), so one stream of output tiles serves them all and
 * the last wave of each fills with tiles of the others.  Each dw element gets
 * one float32 add per call, in the same order as from zb_op_backward_weight, so
 * the results are the same bits as n separate calls. */
zb_status zb_op_backward_weight_group(int32_t n, const void* const* dy, const void* const* x,
                                      float* const* dw, int32_t tokens, const int32_t* in_features,
                                      const int32_t* out_features, void* stream);

/* W of an RMSNorm weight: dgamma[H] (float32) += sum_t dn[t,:] * x[t,:] * rstd[t].
 * Two passes in a fixed order (per-block partial sums in `scratch`, then one
 * ordered sum), so results are bitwise reproducible.  `scratch` is device
 * memory of at least zb_op_rmsnorm_backward_gamma_scratch_bytes(T, H) bytes,
 * owned by the caller, contents ignored on entry. */
size_t zb_op_rmsnorm_backward_gamma_scratch_bytes(int32_t tokens, int32_t hidden);
zb_status zb_op_rmsnorm_backward_gamma(const void* dn, const void* x, const float* rstd,
                                       float* dgamma, int32_t tokens, int32_t hidden,
                                       void* scratch, size_t scratch_bytes, void* stream);

/* The same gamma-gradient reduction for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a convenience of this
 * library.  Some callers get only their input and output tensors from a host
 * framework, for example a plugin or custom-op interface that offers no
 * workspace.  Others run where all device memory belongs to another allocator,
 * so a cudaMalloc of their own would fail or synchronise the device.  These
 * callers cannot provide `scratch`, so this variant keeps the partial sums in
 * a fixed 512 KiB float32 array inside the library.
 *  - Every GPU that loads the library holds that array until the process exits.
 *  - Size limit: zb_op_rmsnorm_backward_gamma_scratch_bytes(tokens, hidden)
 *    must not exceed 4 * zb_op_rmsnorm_backward_gamma_noalloc_max_floats()
 *    bytes (512 KiB).  The reduction's partition takes at most 131072 / hidden
 *    partial rows, so every token count fits for hidden <= 131072 (multiples
 *    of 64); wider rows return ZB_ERR_SHAPE and enqueue nothing.
 *  - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *    routine.
 *  - The first call on a device looks up the array's device address (with that
 *    device current).  Make that first call before any stream capture.
 *  - All calls share the one array, and it keeps the last call's contents.
 *    Every partial sum a call reads is first written by that same call, so
 *    nothing needs clearing.
 *  - Calls that overlap on the GPU (other streams, other host threads) race on
 *    the array and give wrong results: order them.
 * Arguments, layout and result are as for zb_op_rmsnorm_backward_gamma. */
size_t zb_op_rmsnorm_backward_gamma_noalloc_max_floats(void);
zb_status zb_op_rmsnorm_backward_gamma_noalloc(const void* dn, const void* x, const float* rstd,
                                               float* dgamma, int32_t tokens, int32_t hidden,
                                               void* stream);

/* F pieces.  RMSNorm: rstd[t] = (mean_j x[t,j]^2 + eps)^(-1/2) (float32),
 * n = gamma * x * rstd (bf16).  SwiGLU: s[T,F] = silu(gu[:, :F]) * gu[:, F:].
 * Attention stand-in: a[T, nh hd] from qkv[T, (nh + 2 nkv) hd] as above. */
zb_status zb_op_rmsnorm_forward(const void* x, const float* gamma, float eps, void* n,
                                float* rstd, int32_t tokens, int32_t hidden, void* stream);
zb_status zb_op_swiglu_forward(const void* gu, void* s, int32_t tokens, int32_t ffn,
                               void* stream);
zb_status zb_op_attention_forward(const void* qkv, void* a, int32_t tokens,
                                  int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                  void* stream);

/* Causal softmax attention with grouped K/V heads: the attention core in
 * its full form.  The pages name the qkv and output projections around it but
 * not the core itself; this is the usual one, without position encoding.
 * For head h, with j = h / (nh / nkv):
 *   a_h = softmax(q_h k_j^T / sqrt(hd), keys <= query) v_j
 * over independent sequences of seq_len consecutive tokens (0: the `tokens`
 * rows are one sequence; the last sequence may be shorter than seq_len).
 *  - qkv [T, (nh + 2 nkv) hd] bf16 (q heads, then k heads, then v heads);
 *    a and da [T, nh hd] bf16; dqkv like qkv.
 *  - lse float32 [nh][zb_op_attention_stat_stride(T)]: per head and query
 *    row, log2 of the softmax denominator in units of the scaled score.  The
 *    forward writes it; the backward reads it.  dvec is caller-owned float32
 *    scratch of the same shape (contents ignored).
 *  - hd is 64 or 128; seq_len is 0 or a multiple of 128.  Other shapes
 *    return ZB_ERR_SHAPE.
 *  - The backward writes every column of dqkv.  Each output element is
 *    written by one thread after a fixed-order sum, so results are bitwise
 *    reproducible.
 *  - Streams: the backward runs its dK/dV kernel on `stream` and its dQ
 *    kernel on a library-owned stream of the current device, forked from
 *    `stream` after the work already queued there and joined back before the
 *    call returns; work queued on `stream` afterwards sees all of dqkv.  The
 *    library creates that stream, two events and a 4-byte device counter
 *    (the dQ kernel's tile counter, zeroed on that stream before each
 *    launch) at the first causal backward on a device, or at a causal
 *    stage's first forward; they live until the process ends. */
int32_t zb_op_attention_stat_stride(int32_t tokens);
zb_status zb_op_attention_causal_forward(const void* qkv, void* a, float* lse, int32_t tokens,
                                         int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                         int32_t seq_len, void* stream);
zb_status zb_op_attention_causal_backward(const void* qkv, const void* a, const void* da,
                                          const float* lse, float* dvec, void* dqkv,
                                          int32_t tokens, int32_t n_heads, int32_t n_kv_heads,
                                          int32_t head_dim, int32_t seq_len, void* stream);

/* Device status word shared by all kernels of the library on the current
 * device: 0 = fine, else the code of the first wait that ran out:
 *   1  GEMM TMA producer waiting for a free shared-memory stage
 *   2  GEMM MMA issuer waiting for a loaded stage
 *   3  GEMM MMA issuer waiting for the epilogue to free an accumulator
 *   4  GEMM epilogue waiting for a finished accumulator
 *   5  teardown waiting for copies or MMAs in flight
 *   6  the two CTAs of a GEMM pair got different tensor-memory columns
 *   7  K-split epilogue waiting for the other half's partial tile
 *   8  attention kernels (any of their pipeline waits)
 *   9  zb_selftest_wait_timeout
 *   10 GEMM epilogue waiting for SwiGLU side inputs loaded by TMA
 * Reading synchronises `stream`; `reset` != 0 clears the word afterwards.
 * Returns ZB_ERR_DEVICE_TIMEOUT when the word was set, ZB_OK otherwise. */
zb_status zb_device_status(void* stream, int32_t reset, int32_t* code);

/* Runs one bounded wait on an mbarrier that nothing arrives on, with a limit
 * of `limit_us` microseconds, so that callers can see the timeout path work
 * without faulting anything.  Sets the device status word. */
zb_status zb_selftest_wait_timeout(int32_t limit_us, void* stream);

/* ========================================================================
 * One pipeline stage: activation stash, float32 accumulators, F -> B -> W
 * ====================================================================== */

typedef enum {
    ZB_LAYER_LINEAR = 0,      /* y = x W^T, W [ffn (out), hidden (in)]; n_layers must be 1 */
    ZB_LAYER_MLP = 1,         /* h = x; n2 = RMSNorm(h; g2); [g|u] = n2 W_gu^T;
                                 y = h + (silu(g) * u) W_down^T */
    ZB_LAYER_TRANSFORMER = 2  /* n1 = RMSNorm(x; g1); a = A(n1 W_qkv^T);
                                 h = x + a W_o^T; then the MLP part */
} zb_layer_kind;

/* The attention core A of a TRANSFORMER layer. */
typedef enum {
    ZB_ATTN_STANDIN = 0,  /* weight-free stand-in a_h = q_h + k_j + v_j (per token) */
    ZB_ATTN_CAUSAL = 1    /* causal softmax attention, as zb_op_attention_causal_forward;
                             the stash also keeps qkv and the row log-sum-exp */
} zb_attention_kind;

typedef struct {
    int32_t kind;          /* zb_layer_kind */
    int32_t n_layers;
    int32_t hidden;        /* H (LINEAR: in_features) */
    int32_t ffn;           /* F (LINEAR: out_features) */
    int32_t n_heads;       /* TRANSFORMER only: n_heads * head_dim == hidden */
    int32_t n_kv_heads;    /* divides n_heads */
    int32_t head_dim;
    float eps;             /* RMSNorm epsilon */
    int32_t max_tokens;    /* largest T of any microbatch */
    int32_t max_inflight;  /* stash slots: microbatches between F and W [G3] */
    int32_t attention;     /* TRANSFORMER: zb_attention_kind */
    int32_t seq_len;       /* ZB_ATTN_CAUSAL: tokens per sequence, 0 or a multiple of 128
                              (0: each microbatch is one sequence) */
} zb_stage_config;

/* Per-layer device pointers.  Weights bf16 [out, in]; gamma float32 [H];
 * accumulators float32, same shapes, zeroed by the caller, then only added
 * to [G3].  W_gu = [W_gate; W_up] (gate rows first), [2F, H]; W_qkv rows are
 * q heads, then k heads, then v heads.  Unused fields may be NULL. */
typedef struct {
    const void* w_qkv;  float* dw_qkv;    /* [(nh + 2 nkv) hd, H] */
    const void* w_o;    float* dw_o;      /* [H, H] */
    const void* w_gu;   float* dw_gu;     /* [2F, H] */
    const void* w_down; float* dw_down;   /* [H, F] */
    const float* gamma1; float* dgamma1;  /* [H], TRANSFORMER */
    const float* gamma2; float* dgamma2;  /* [H], MLP and TRANSFORMER */
    const void* w;      float* dw;        /* LINEAR: [F, H] */
} zb_layer_params;

typedef struct zb_stage* zb_stage_t;

/* Bytes of device workspace a stage needs (stash slots for max_inflight
 * microbatches of max_tokens tokens, forward temporaries, reduction
 * scratch).  0 when the config is invalid. */
size_t zb_stage_workspace_bytes(const zb_stage_config* cfg);

/* Creates a stage.  `layers` has n_layers entries (copied).  `workspace` is
 * caller-owned device memory of at least zb_stage_workspace_bytes(cfg)
 * bytes, 256-byte aligned, that must outlive the stage; weights and
 * accumulators must outlive it too, and a weight must not change between
 * the F and the W of a microbatch (the optimizer runs after the flush). */
zb_status zb_stage_create(const zb_stage_config* cfg, const zb_layer_params* layers,
                          void* workspace, size_t workspace_bytes, zb_stage_t* out);
zb_status zb_stage_destroy(zb_stage_t st);

/* F of microbatch `mb` [G2]: claims a stash slot, keeps what B and W need,
 * writes y[T, out] (out = ffn for LINEAR, else hidden).  x is copied, so the
 * caller may reuse it once the stream passes this call.
 * Errors: ZB_ERR_ORDER (mb already in flight), ZB_ERR_STASH_FULL,
 * ZB_ERR_SHAPE (tokens > max_tokens or < 0), ZB_ERR_ARG. */
zb_status zb_stage_forward(zb_stage_t st, int32_t mb, const void* x, int32_t tokens,
                           void* y, void* stream);

/* B of microbatch `mb` [G1][G2]: from dy[T, out] computes dx[T, hidden]
 * through every layer, top first, and keeps each linear's dY for the
 * deferred W.  Only dX-side products run here.
 * Errors: ZB_ERR_NO_MB (no F for mb), ZB_ERR_ORDER (B already ran). */
zb_status zb_backward_input(zb_stage_t st, int32_t mb, const void* dy, void* dx,
                            void* stream);

/* W of microbatch `mb` [G1][G3]: dW += dY^T X for every linear and
 * dgamma += sum_t dn * xh for every RMSNorm, into the float32 accumulators;
 * then releases the stash slot.
 * Errors: ZB_ERR_NO_MB, ZB_ERR_ORDER (B not run yet). */
zb_status zb_backward_weight(zb_stage_t st, int32_t mb, void* stream);

/* Runs W for every microbatch whose B ran and whose W did not, then
 * releases their stash slots.  The accumulators hold the sum over all
 * microbatches once `stream` gets there.  Microbatches of max_tokens tokens
 * in consecutive stash slots are done as one W over their concatenated
 * tokens: one GEMM per weight with k * max_tokens contraction length and one
 * float32 add into each accumulator element, instead of k.  That is exact
 * arithmetic (every op but the weight contractions acts per token), and it
 * rounds differently from k separate W calls.  The batches run in ascending
 * slot order, so a given sequence of calls always gives the same bits. */
zb_status zb_wgrad_flush(zb_stage_t st, void* stream);

/* Synchronises `stream` and reads the device status word (see
 * zb_device_status); ZB_ERR_DEVICE_TIMEOUT if a kernel wait ran out. */
zb_status zb_stage_sync(zb_stage_t st, void* stream);

/* Microbatches held now, the most ever held, and the stash bytes in use now. */
zb_status zb_stage_stats(zb_stage_t st, int32_t* inflight, int32_t* peak_inflight,
                         size_t* stash_bytes);

/* ------------------------------------------------------------------------
 * Read-only view of the activation stash, for tests and diagnostics.  An
 * oracle that takes a layer's inputs from here consumes exactly the bf16
 * values the kernels consumed, so each step of every layer can be checked
 * against the plain definition on its own (the guide's section "2.
 * Convergence and Numerical Stability": B and W are the plain backward's
 * arithmetic, split), apart from the roundings of the steps before it.
 * ---------------------------------------------------------------------- */
typedef enum {
    ZB_STASH_X = 0,    /* layer input x [T, H] (LINEAR: [T, hidden]); MLP: also h */
    ZB_STASH_RSTD1,    /* float32 [T], TRANSFORMER */
    ZB_STASH_N1,       /* RMSNorm(x; gamma1) [T, H], TRANSFORMER */
    ZB_STASH_A,        /* attention output [T, H], TRANSFORMER */
    ZB_STASH_H,        /* x + a W_o^T [T, H] (MLP: the same region as x) */
    ZB_STASH_RSTD2,    /* float32 [T] */
    ZB_STASH_N2,       /* RMSNorm(h; gamma2) [T, H] */
    ZB_STASH_GU,       /* [T, 2F]: [g | u] after F; [dg | du] once B ran (written in place) */
    ZB_STASH_S,        /* silu(g) * u [T, F] */
    ZB_STASH_DY,       /* the layer's output gradient [T, H] (LINEAR: [T, ffn]); written by B */
    ZB_STASH_DN2,      /* dgu W_gu [T, H]; written by B */
    ZB_STASH_DH,       /* gradient of h [T, H], TRANSFORMER; written by B */
    ZB_STASH_DQKV,     /* [T, (nh + 2 nkv) hd], TRANSFORMER; written by B */
    ZB_STASH_DN1,      /* dqkv W_qkv [T, H], TRANSFORMER; written by B */
    ZB_STASH_QKV,      /* attention input [T, (nh + 2 nkv) hd], ZB_ATTN_CAUSAL only */
    ZB_STASH_LSE,      /* float32 [nh, zb_op_attention_stat_stride(max_tokens)], ZB_ATTN_CAUSAL only */
    ZB_STASH_COUNT
} zb_stash_tensor;

/* Device address, shape and element size (2: bf16, 4: float32) of one stashed
 * tensor of layer `layer` of microbatch `mb` (rows are the microbatch's T
 * tokens, or the heads for ZB_STASH_LSE; rows are dense, `cols` elements
 * apart).  The address points into the caller's workspace and holds the
 * tensor from the call that writes it (F, or B for the gradients) until the
 * microbatch's W; read it only after `stream` has passed that call.  Nothing
 * is enqueued.  Errors: ZB_ERR_NO_MB (mb not between F and W), ZB_ERR_ARG
 * (layer outside [0, n_layers), a tensor this layer kind does not stash, a
 * NULL output pointer). */
zb_status zb_stage_stash_view(zb_stage_t st, int32_t mb, int32_t layer, int32_t tensor, const void** ptr,
                              int64_t* rows, int64_t* cols, int32_t* elem_bytes);

/* ------------------------------------------------------------------------
 * Per-launch tracing (the guide's section "Operational Checklist" asks for
 * per-stage telemetry; this is its per-kernel form).  When enabled, the stage
 * records a CUDA event pair on the call's stream around every launch and
 * books it under a kernel class with the launch's algorithmic work:
 *   FLOPs = 2 M N K per GEMM; bytes = every operand read once and every
 *   result written once (float32 accumulators read and written).
 * ---------------------------------------------------------------------- */
typedef enum {
    ZB_KCLASS_GEMM_FORWARD = 0,      /* F GEMMs */
    ZB_KCLASS_GEMM_BACKWARD_INPUT,   /* B GEMMs, incl. the fused SwiGLU backward and the causal
                                        attention's D in the output projection's dgrad */
    ZB_KCLASS_GEMM_BACKWARD_WEIGHT,  /* W GEMMs (float32 accumulation) */
    ZB_KCLASS_ROW_BACKWARD_INPUT,    /* B row kernels: RMSNorm backward, stand-in backward */
    ZB_KCLASS_ROW_BACKWARD_WEIGHT,   /* W row kernels: gamma-gradient reduction */
    ZB_KCLASS_ROW_FORWARD,           /* F row kernels */
    ZB_KCLASS_ATTN_FORWARD,          /* F causal attention */
    ZB_KCLASS_ATTN_BACKWARD,         /* B causal attention (dK/dV and dQ kernels, and the rowsum kernel
                                        when the output projection's dgrad does not form D) */
    ZB_KCLASS_STASH_COPY,            /* the stash copies of the caller's x (F) and dy (B):
                                        device-to-device cudaMemcpyAsync, not a kernel of the
                                        library (time and bytes count, launches do not) */
    ZB_KCLASS_COUNT
} zb_kernel_class;

typedef struct {
    int32_t launches;  /* kernels of the library launched (stash copies count time and bytes, not launches) */
    int32_t pad;
    double ms;         /* summed event time */
    double flops;      /* algorithmic FLOPs */
    double bytes;      /* algorithmic bytes */
} zb_kernel_stats;

/* Turns tracing on (enable != 0) or off.  Events come from a pool that grows
 * on first use, so run one traced warm-up before a timed region. */
zb_status zb_stage_set_tracing(zb_stage_t st, int32_t enable);

/* Waits for the recorded events, writes ZB_KCLASS_COUNT entries to `out`,
 * and clears the records when `reset` != 0. */
zb_status zb_stage_read_tracing(zb_stage_t st, zb_kernel_stats* out, int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* ZB_H_ */
