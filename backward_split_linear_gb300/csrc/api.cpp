// C ABI of libzb: argument checks, the per-step operations and the stage
// runtime (activation stash, F -> B -> W order per microbatch, flush).
//
// The stage follows "Zero-Bubble Pipeline Parallelism Guide for LLMs":
// section "Step-by-Step Implementation" (forward keeps x, B keeps dY and
// returns dY W, W pops both and adds into the weight gradient) and section
// "Memory Management & Activation Rollback" (activations live from F until
// their W; at most max_inflight microbatches are held; weight gradients are
// accumulated in place in fixed buffers).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/zb.h"
#include "launch.h"

using zbk::Epilogue;
using zbk::GemmArgs;
using zbk::GemmKind;

namespace {

constexpr int32_t kMaxFeature = 1 << 20;
constexpr int32_t kMaxTokens = 1 << 24;

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A tensor with `tokens` rows: may be NULL when there are no rows.
inline bool rows_ok(const void* p, int32_t tokens) { return tokens == 0 ? (p == nullptr || aligned16(p)) : (p && aligned16(p)); }

// A tensor whose size does not depend on the tokens.
inline bool fixed_ok(const void* p) { return p && aligned16(p); }

inline bool feature_ok(int32_t f) { return f > 0 && f <= kMaxFeature && f % 64 == 0; }

inline bool tokens_ok(int32_t t) { return t >= 0 && t <= kMaxTokens; }

zb_status device_ok() {
    const int arch = zbk::device_arch();
    if (arch < 0) return ZB_ERR_CUDA;
    return arch == 103 ? ZB_OK : ZB_ERR_DEVICE;
}

inline zb_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ZB_OK : ZB_ERR_CUDA; }

#define ZB_TRY(expr)                        \
    do {                                    \
        const zb_status zb_s_ = (expr);     \
        if (zb_s_ != ZB_OK) return zb_s_;   \
    } while (0)

// ------------------------------------------------------------ op bodies (checked by callers)

// K-split scratch of a stage (see GemmArgs); the per-step ops run without it.
struct SplitWs {
    uint32_t* flags;
    float* partial;
    int tiles;
};

void set_split(GemmArgs& g, const SplitWs* ws) {
    if (!ws) return;
    g.split_flags = ws->flags;
    g.split_partial = ws->partial;
    g.split_tiles = ws->tiles;
}

zb_status run_linear_forward(const void* x, const void* w, const void* residual, void* y, int t,
                             int in, int out, cudaStream_t s, const SplitWs* ws = nullptr) {
    GemmArgs g{};
    g.kind = GemmKind::Forward;
    g.epi = residual ? Epilogue::AddResidual : Epilogue::StoreBf16;
    g.a = x;
    g.lda = in;
    g.b = w;
    g.ldb = in;
    g.m = t;
    g.n = out;
    g.k = in;
    g.out = y;
    g.ldo = out;
    g.aux = residual;
    g.ld_aux = out;
    set_split(g, ws);
    return cuda_status(zbk::launch_gemm(g, s));
}

// F of the gate|up linear with the SwiGLU forward in its epilogue: gu = x w_gu^T
// ([g | u], bf16) and s = silu(g) u from the bf16 g and u.  The CTA-pair GEMM
// only (t >= 256, ffn a multiple of 128); see swiglu_forward_fused below.
zb_status run_linear_forward_swiglu(const void* x, const void* w_gu, void* gu, void* s_out, int t, int hidden,
                                    int ffn, cudaStream_t s, const SplitWs* ws = nullptr) {
    GemmArgs g{};
    g.kind = GemmKind::Forward;
    g.epi = Epilogue::SwigluFwd;
    g.a = x;
    g.lda = hidden;
    g.b = w_gu;
    g.ldb = hidden;
    g.m = t;
    g.n = 2 * ffn;
    g.k = hidden;
    g.out = gu;
    g.ldo = 2 * static_cast<int64_t>(ffn);
    g.out2 = s_out;
    g.ldo2 = ffn;
    g.ffn = ffn;
    set_split(g, ws);
    return cuda_status(zbk::launch_gemm(g, s));
}

// Whether the gate|up F runs fused with the SwiGLU forward (the CTA-pair GEMM
// takes outputs of at least 256 rows; a tile holds 128 features of g and u).
bool swiglu_forward_fused(int t, int ffn) { return t >= 256 && ffn % 128 == 0; }

zb_status run_backward_input(const void* dy, const void* w, void* dx, int t, int in, int out,
                             int64_t ldo, cudaStream_t s, const SplitWs* ws = nullptr) {
    GemmArgs g{};
    g.kind = GemmKind::BackwardInput;
    g.epi = Epilogue::StoreBf16;
    g.a = dy;
    g.lda = out;
    g.b = w;
    g.ldb = in;
    g.m = t;
    g.n = in;
    g.k = out;
    g.out = dx;
    g.ldo = ldo;
    set_split(g, ws);
    return cuda_status(zbk::launch_gemm(g, s));
}

// dx = dy w, and per row and head the attention backward's D = rowsum(dx * a)
// from the stored bf16 dx (CTA-pair GEMMs only: gemm_takes_pair(t, in)).
zb_status run_backward_input_rowdot(const void* dy, const void* w, void* dx, const void* a, float* dvec,
                                    int64_t ld_stat, int head_dim, int t, int in, int out, cudaStream_t s,
                                    const SplitWs* ws) {
    GemmArgs g{};
    g.kind = GemmKind::BackwardInput;
    g.epi = Epilogue::StoreBf16RowDot;
    g.a = dy;
    g.lda = out;
    g.b = w;
    g.ldb = in;
    g.m = t;
    g.n = in;
    g.k = out;
    g.out = dx;
    g.ldo = in;
    g.aux = a;
    g.ld_aux = in;
    g.dot = dvec;
    g.ld_dot = ld_stat;
    g.dot_cols = head_dim;
    set_split(g, ws);
    return cuda_status(zbk::launch_gemm(g, s));
}

zb_status run_backward_input_swiglu(const void* dy, const void* w_down, const void* gu, void* dgu,
                                    int t, int hidden, int ffn, cudaStream_t s, const SplitWs* ws = nullptr) {
    GemmArgs g{};
    g.kind = GemmKind::BackwardInput;
    g.epi = Epilogue::SwigluBwd;
    g.a = dy;
    g.lda = hidden;
    g.b = w_down;
    g.ldb = ffn;
    g.m = t;
    g.n = ffn;
    g.k = hidden;
    g.out = dgu;
    g.ldo = 2 * static_cast<int64_t>(ffn);
    g.aux = gu;
    g.ld_aux = 2 * static_cast<int64_t>(ffn);
    g.ffn = ffn;
    set_split(g, ws);
    return cuda_status(zbk::launch_gemm(g, s));
}

zb_status run_backward_input_rmsnorm(const void* dy, const void* w, const void* x, const float* rstd,
                                     const float* gamma, const void* dres, void* dn, void* dx, int t,
                                     int hidden, int out, cudaStream_t s) {
    ZB_TRY(run_backward_input(dy, w, dn, t, hidden, out, hidden, s));
    return cuda_status(zbk::launch_rmsnorm_backward_input(dn, x, rstd, gamma, dres, dx, t, hidden, s));
}

zb_status run_backward_input_attention(const void* dh, const void* w_o, void* dqkv, int t, int nh,
                                       int nkv, int hd, cudaStream_t s) {
    const int width = nh * hd;
    const int64_t qkv_w = static_cast<int64_t>(nh + 2 * nkv) * hd;
    ZB_TRY(run_backward_input(dh, w_o, dqkv, t, width, width, qkv_w, s));
    return cuda_status(zbk::launch_attention_backward_kv(dqkv, t, nh, nkv, hd, s));
}

GemmArgs wgrad_args(const void* dy, const void* x, float* dw, int t, int in, int out) {
    GemmArgs g{};
    g.kind = GemmKind::BackwardWeight;
    g.epi = Epilogue::AccumF32;
    g.a = dy;
    g.lda = out;
    g.b = x;
    g.ldb = in;
    g.m = out;
    g.n = in;
    g.k = t;
    g.out = dw;
    g.ldo = in;
    return g;
}

zb_status run_backward_weight(const void* dy, const void* x, float* dw, int t, int in, int out,
                              cudaStream_t s, const SplitWs* ws = nullptr) {
    GemmArgs g{};
    g.kind = GemmKind::BackwardWeight;
    g.epi = Epilogue::AccumF32;
    g.a = dy;
    g.lda = out;
    g.b = x;
    g.ldb = in;
    g.m = out;
    g.n = in;
    g.k = t;
    g.out = dw;
    g.ldo = in;
    set_split(g, ws);
    return cuda_status(zbk::launch_gemm(g, s));
}

bool heads_ok(int32_t nh, int32_t nkv, int32_t hd) {
    if (nh <= 0 || nkv <= 0 || hd <= 0 || hd % 8 != 0 || nh % nkv != 0) return false;
    if (!feature_ok(nh * hd) || !feature_ok((nh + 2 * nkv) * hd)) return false;
    return true;
}

// Causal attention: head_dim 64 or 128, sequences of a multiple of 128 tokens (or one sequence).
bool causal_ok(int32_t nh, int32_t nkv, int32_t hd, int32_t seq_len) {
    return heads_ok(nh, nkv, hd) && (hd == 64 || hd == 128) && seq_len >= 0 && seq_len % 128 == 0;
}

// Floats per head row of the attention statistics (lse, rowsum): whole 128-row blocks.
int32_t stat_stride(int32_t tokens) { return std::max<int32_t>(128, (tokens + 127) / 128 * 128); }

zbk::AttnShape attn_shape(int t, int nh, int nkv, int hd, int seq_len, int ld_stat) {
    zbk::AttnShape a;
    a.tokens = t;
    a.n_heads = nh;
    a.n_kv_heads = nkv;
    a.head_dim = hd;
    a.seq_len = seq_len;
    a.ld_stat = ld_stat;
    return a;
}

// Query-key pairs a causal mask leaves visible over the sequences of t tokens.
double causal_pairs(int t, int seq_len) {
    const int step = seq_len > 0 ? seq_len : std::max(t, 1);
    double n = 0.0;
    for (int s0 = 0; s0 < t; s0 += step) {
        const double len = std::min(t, s0 + step) - s0;
        n += len * (len + 1.0) / 2.0;
    }
    return n;
}

}  // namespace

// ======================================================================== misc

extern "C" const char* zb_status_string(zb_status s) {
    switch (s) {
        case ZB_OK: return "ok";
        case ZB_ERR_ARG: return "invalid argument";
        case ZB_ERR_SHAPE: return "unsupported shape";
        case ZB_ERR_ORDER: return "F -> B -> W order of a microbatch broken";
        case ZB_ERR_STASH_FULL: return "activation stash full (max_inflight microbatches held)";
        case ZB_ERR_NO_MB: return "unknown microbatch";
        case ZB_ERR_CUDA: return "CUDA runtime error";
        case ZB_ERR_DEVICE_TIMEOUT: return "a kernel wait ran out of time";
        case ZB_ERR_CAPACITY: return "output array too small";
        case ZB_ERR_DEVICE: return "current device is not sm_103";
        case ZB_ERR_WORKSPACE: return "workspace or scratch too small or misaligned";
    }
    return "unknown status";
}

extern "C" int32_t zb_version(void) { return 100; }

extern "C" zb_status zb_device_status(void* stream, int32_t reset, int32_t* code) {
    ZB_TRY(device_ok());
    int* w = zbk::status_word();
    if (!w) return ZB_ERR_CUDA;
    int v = 0;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(&v, w, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return ZB_ERR_CUDA;
    if (reset && cudaMemsetAsync(w, 0, sizeof(int), s) != cudaSuccess) return ZB_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ZB_ERR_CUDA;
    if (code) *code = v;
    return v ? ZB_ERR_DEVICE_TIMEOUT : ZB_OK;
}

extern "C" zb_status zb_selftest_wait_timeout(int32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return cuda_status(zbk::launch_selftest_wait(limit_us, as_stream(stream)));
}

// ======================================================================== ops

extern "C" zb_status zb_op_linear_forward(const void* x, const void* w, const void* residual, void* y,
                                          int32_t tokens, int32_t in_features, int32_t out_features,
                                          void* stream) {
    if (!tokens_ok(tokens) || !feature_ok(in_features) || !feature_ok(out_features)) return ZB_ERR_SHAPE;
    if (!rows_ok(x, tokens) || !fixed_ok(w) || !rows_ok(y, tokens) || (residual && !aligned16(residual)))
        return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return run_linear_forward(x, w, residual, y, tokens, in_features, out_features, as_stream(stream));
}

extern "C" zb_status zb_op_backward_input(const void* dy, const void* w, void* dx, int32_t tokens,
                                          int32_t in_features, int32_t out_features, void* stream) {
    if (!tokens_ok(tokens) || !feature_ok(in_features) || !feature_ok(out_features)) return ZB_ERR_SHAPE;
    if (!rows_ok(dy, tokens) || !fixed_ok(w) || !rows_ok(dx, tokens)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return run_backward_input(dy, w, dx, tokens, in_features, out_features, in_features,
                              as_stream(stream));
}

extern "C" zb_status zb_op_backward_input_swiglu(const void* dy, const void* w_down, const void* gu,
                                                 void* dgu, int32_t tokens, int32_t hidden, int32_t ffn,
                                                 void* stream) {
    if (!tokens_ok(tokens) || !feature_ok(hidden) || !feature_ok(ffn)) return ZB_ERR_SHAPE;
    if (!rows_ok(dy, tokens) || !fixed_ok(w_down) || !rows_ok(gu, tokens) || !rows_ok(dgu, tokens))
        return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return run_backward_input_swiglu(dy, w_down, gu, dgu, tokens, hidden, ffn, as_stream(stream));
}

extern "C" zb_status zb_op_backward_input_rmsnorm(const void* dy, const void* w, const void* x,
                                                  const float* rstd, const float* gamma, const void* dres,
                                                  void* dn, void* dx, int32_t tokens, int32_t hidden,
                                                  int32_t out_features, void* stream) {
    if (!tokens_ok(tokens) || !feature_ok(hidden) || !feature_ok(out_features)) return ZB_ERR_SHAPE;
    const void* rows[] = {dy, x, rstd, dres, dn, dx};
    for (const void* p : rows)
        if (!rows_ok(p, tokens)) return ZB_ERR_ARG;
    if (!fixed_ok(w) || !fixed_ok(gamma)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return run_backward_input_rmsnorm(dy, w, x, rstd, gamma, dres, dn, dx, tokens, hidden, out_features,
                                      as_stream(stream));
}

extern "C" zb_status zb_op_backward_input_attention(const void* dh, const void* w_o, void* dqkv,
                                                    int32_t tokens, int32_t n_heads, int32_t n_kv_heads,
                                                    int32_t head_dim, void* stream) {
    if (!tokens_ok(tokens) || !heads_ok(n_heads, n_kv_heads, head_dim)) return ZB_ERR_SHAPE;
    if (!rows_ok(dh, tokens) || !fixed_ok(w_o) || !rows_ok(dqkv, tokens)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return run_backward_input_attention(dh, w_o, dqkv, tokens, n_heads, n_kv_heads, head_dim,
                                        as_stream(stream));
}

extern "C" zb_status zb_op_backward_weight(const void* dy, const void* x, float* dw, int32_t tokens,
                                           int32_t in_features, int32_t out_features, void* stream) {
    if (!tokens_ok(tokens) || !feature_ok(in_features) || !feature_ok(out_features)) return ZB_ERR_SHAPE;
    if (!rows_ok(dy, tokens) || !rows_ok(x, tokens) || !fixed_ok(dw)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return run_backward_weight(dy, x, dw, tokens, in_features, out_features, as_stream(stream));
}

extern "C" zb_status zb_op_backward_weight_group(int32_t n, const void* const* dy, const void* const* x,
                                                 float* const* dw, int32_t tokens, const int32_t* in_features,
                                                 const int32_t* out_features, void* stream) {
    if (n < 1 || n > 16 || !dy || !x || !dw || !in_features || !out_features) return ZB_ERR_ARG;
    if (!tokens_ok(tokens)) return ZB_ERR_SHAPE;
    std::vector<GemmArgs> gs;
    for (int i = 0; i < n; ++i) {
        if (!feature_ok(in_features[i]) || !feature_ok(out_features[i])) return ZB_ERR_SHAPE;
        if (!rows_ok(dy[i], tokens) || !rows_ok(x[i], tokens) || !fixed_ok(dw[i])) return ZB_ERR_ARG;
        gs.push_back(wgrad_args(dy[i], x[i], dw[i], tokens, in_features[i], out_features[i]));
    }
    ZB_TRY(device_ok());
    if (tokens == 0) return ZB_OK;
    return cuda_status(zbk::launch_gemm_group(gs.data(), n, as_stream(stream)));
}

extern "C" size_t zb_op_rmsnorm_backward_gamma_scratch_bytes(int32_t tokens, int32_t hidden) {
    if (!tokens_ok(tokens) || !feature_ok(hidden)) return 0;
    return zbk::rmsnorm_gamma_scratch_bytes(tokens, hidden);
}

extern "C" zb_status zb_op_rmsnorm_backward_gamma(const void* dn, const void* x, const float* rstd,
                                                  float* dgamma, int32_t tokens, int32_t hidden,
                                                  void* scratch, size_t scratch_bytes, void* stream) {
    if (!tokens_ok(tokens) || !feature_ok(hidden)) return ZB_ERR_SHAPE;
    if (!rows_ok(dn, tokens) || !rows_ok(x, tokens) || !rows_ok(rstd, tokens) || !fixed_ok(dgamma))
        return ZB_ERR_ARG;
    const size_t need = zbk::rmsnorm_gamma_scratch_bytes(tokens, hidden);
    if (need > 0 && (!scratch || !aligned16(scratch) || scratch_bytes < need)) return ZB_ERR_WORKSPACE;
    ZB_TRY(device_ok());
    return cuda_status(zbk::launch_rmsnorm_backward_gamma(dn, x, rstd, dgamma, tokens, hidden,
                                                          static_cast<float*>(scratch), as_stream(stream)));
}

extern "C" zb_status zb_op_rmsnorm_forward(const void* x, const float* gamma, float eps, void* n,
                                           float* rstd, int32_t tokens, int32_t hidden, void* stream) {
    if (!tokens_ok(tokens) || !feature_ok(hidden)) return ZB_ERR_SHAPE;
    if (!rows_ok(x, tokens) || !fixed_ok(gamma) || !rows_ok(n, tokens) || !rows_ok(rstd, tokens) || !(eps >= 0.f))
        return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return cuda_status(zbk::launch_rmsnorm_forward(x, gamma, eps, n, rstd, tokens, hidden, as_stream(stream)));
}

extern "C" zb_status zb_op_swiglu_forward(const void* gu, void* s, int32_t tokens, int32_t ffn,
                                          void* stream) {
    if (!tokens_ok(tokens) || !feature_ok(ffn)) return ZB_ERR_SHAPE;
    if (!rows_ok(gu, tokens) || !rows_ok(s, tokens)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return cuda_status(zbk::launch_swiglu_forward(gu, s, tokens, ffn, as_stream(stream)));
}

extern "C" int32_t zb_op_attention_stat_stride(int32_t tokens) { return tokens_ok(tokens) ? stat_stride(tokens) : 0; }

extern "C" zb_status zb_op_attention_causal_forward(const void* qkv, void* a, float* lse, int32_t tokens,
                                                    int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                                    int32_t seq_len, void* stream) {
    if (!tokens_ok(tokens) || !causal_ok(n_heads, n_kv_heads, head_dim, seq_len)) return ZB_ERR_SHAPE;
    if (!rows_ok(qkv, tokens) || !rows_ok(a, tokens) || !rows_ok(lse, tokens)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return cuda_status(zbk::launch_attention_causal_forward(
        attn_shape(tokens, n_heads, n_kv_heads, head_dim, seq_len, stat_stride(tokens)), qkv, a, lse,
        as_stream(stream)));
}

extern "C" zb_status zb_op_attention_causal_backward(const void* qkv, const void* a, const void* da,
                                                     const float* lse, float* dvec, void* dqkv, int32_t tokens,
                                                     int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                                     int32_t seq_len, void* stream) {
    if (!tokens_ok(tokens) || !causal_ok(n_heads, n_kv_heads, head_dim, seq_len)) return ZB_ERR_SHAPE;
    const void* rows[] = {qkv, a, da, lse, dvec, dqkv};
    for (const void* p : rows)
        if (!rows_ok(p, tokens)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return cuda_status(zbk::launch_attention_causal_backward(
        attn_shape(tokens, n_heads, n_kv_heads, head_dim, seq_len, stat_stride(tokens)), qkv, a, da, lse, dvec,
        dqkv, as_stream(stream)));
}

extern "C" zb_status zb_op_attention_forward(const void* qkv, void* a, int32_t tokens, int32_t n_heads,
                                             int32_t n_kv_heads, int32_t head_dim, void* stream) {
    if (!tokens_ok(tokens) || !heads_ok(n_heads, n_kv_heads, head_dim)) return ZB_ERR_SHAPE;
    if (!rows_ok(qkv, tokens) || !rows_ok(a, tokens)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    return cuda_status(zbk::launch_attention_forward(qkv, a, tokens, n_heads, n_kv_heads, head_dim,
                                                     as_stream(stream)));
}

// ======================================================================== stage

namespace {

constexpr size_t kNone = ~static_cast<size_t>(0);
constexpr size_t kAlign = 256;

inline size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// A stashed tensor: one region of the workspace holding it for every slot,
// slot after slot with no padding ([slot][max_tokens][width]), so the stashes
// of consecutive slots form one larger matrix.
struct Region {
    size_t off = kNone;  // byte offset of slot 0
    size_t stride = 0;   // bytes per slot
};

// What one layer keeps for B and W.
struct LayerSlot {
    Region x, r1, n1, a, h, r2, n2, gu, s, dy, dn2, dh, dqkv, dn1;
    Region qkv, lse;  // causal attention only: its input and row statistics, for B
};

enum class MbState { Forwarded, BackwardInputDone };

struct MbEntry {
    MbState state;
    int slot;
    int tokens;
};

struct Layout {
    std::vector<LayerSlot> layers;
    size_t slot_bytes = 0;  // stash bytes of one microbatch
    size_t qkv_tmp = kNone;      // forward temporary, offset from the workspace start
    size_t da_tmp = kNone;       // causal attention: gradient of a, B temporary
    size_t dvec = kNone;         // causal attention: rowsum(dO * O), B temporary
    int32_t ld_stat = 0;         // causal attention: floats per head row of lse / dvec
    size_t gamma_scratch = kNone;
    size_t gamma_scratch_bytes = 0;
    size_t split_flags = kNone;  // K-split scratch of the GEMMs (flags, then partial tiles)
    size_t split_partial = kNone;
    int split_tiles = 0;
    size_t total = 0;
};

int qkv_width(const zb_stage_config& c) { return (c.n_heads + 2 * c.n_kv_heads) * c.head_dim; }

zb_status check_config(const zb_stage_config* c) {
    if (!c) return ZB_ERR_ARG;
    if (c->n_layers < 1 || c->n_layers > 4096 || c->max_inflight < 1 || c->max_inflight > 4096 ||
        !(c->eps >= 0.f) || c->max_tokens < 1 || c->max_tokens > kMaxTokens)
        return ZB_ERR_ARG;
    if (c->attention != ZB_ATTN_STANDIN && c->attention != ZB_ATTN_CAUSAL) return ZB_ERR_ARG;
    if (c->attention == ZB_ATTN_STANDIN && c->seq_len != 0) return ZB_ERR_ARG;
    if (c->attention == ZB_ATTN_CAUSAL && c->kind != ZB_LAYER_TRANSFORMER) return ZB_ERR_ARG;
    switch (c->kind) {
        case ZB_LAYER_LINEAR:
            if (c->n_layers != 1) return ZB_ERR_ARG;
            if (!feature_ok(c->hidden) || !feature_ok(c->ffn)) return ZB_ERR_SHAPE;
            return ZB_OK;
        case ZB_LAYER_MLP:
            if (!feature_ok(c->hidden) || !feature_ok(c->ffn)) return ZB_ERR_SHAPE;
            return ZB_OK;
        case ZB_LAYER_TRANSFORMER:
            if (!feature_ok(c->hidden) || !feature_ok(c->ffn)) return ZB_ERR_SHAPE;
            if (!heads_ok(c->n_heads, c->n_kv_heads, c->head_dim) || c->n_heads * c->head_dim != c->hidden)
                return ZB_ERR_SHAPE;
            if (c->attention == ZB_ATTN_CAUSAL && !causal_ok(c->n_heads, c->n_kv_heads, c->head_dim, c->seq_len))
                return ZB_ERR_SHAPE;
            return ZB_OK;
    }
    return ZB_ERR_ARG;
}

Layout make_layout(const zb_stage_config& c) {
    Layout L;
    const size_t T = static_cast<size_t>(c.max_tokens);
    const size_t H = static_cast<size_t>(c.hidden), F = static_cast<size_t>(c.ffn);
    const size_t slots = static_cast<size_t>(c.max_inflight);
    size_t off = 0;
    auto take = [&](size_t per_slot) {
        Region r;
        r.off = off;
        r.stride = per_slot;
        off += round_up(per_slot * slots);
        L.slot_bytes += per_slot;
        return r;
    };
    for (int l = 0; l < c.n_layers; ++l) {
        LayerSlot s;
        if (c.kind == ZB_LAYER_LINEAR) {
            s.x = take(T * H * 2);
            s.dy = take(T * F * 2);
        } else {
            s.x = take(T * H * 2);
            if (c.kind == ZB_LAYER_TRANSFORMER) {
                s.r1 = take(T * 4);
                s.n1 = take(T * H * 2);
                s.a = take(T * H * 2);
                s.h = take(T * H * 2);
                s.dh = take(T * H * 2);
                s.dqkv = take(T * static_cast<size_t>(qkv_width(c)) * 2);
                s.dn1 = take(T * H * 2);
                if (c.attention == ZB_ATTN_CAUSAL) {
                    s.qkv = take(T * static_cast<size_t>(qkv_width(c)) * 2);
                    s.lse = take(static_cast<size_t>(c.n_heads) * stat_stride(c.max_tokens) * 4);
                }
            } else {
                s.h = s.x;  // MLP layer: h = x
            }
            s.r2 = take(T * 4);
            s.n2 = take(T * H * 2);
            s.gu = take(T * 2 * F * 2);  // [g | u] from F, overwritten in place by [dg | du] in B
            s.s = take(T * F * 2);
            s.dy = take(T * H * 2);
            s.dn2 = take(T * H * 2);
        }
        L.layers.push_back(s);
    }
    size_t total = off;
    if (c.kind == ZB_LAYER_TRANSFORMER && c.attention == ZB_ATTN_CAUSAL) {
        L.ld_stat = stat_stride(c.max_tokens);
        L.da_tmp = total;
        total += round_up(T * H * 2);
        L.dvec = total;
        total += round_up(static_cast<size_t>(c.n_heads) * L.ld_stat * 4);
    } else if (c.kind == ZB_LAYER_TRANSFORMER) {
        L.qkv_tmp = total;
        total += round_up(T * static_cast<size_t>(qkv_width(c)) * 2);
    }
    if (c.kind != ZB_LAYER_LINEAR) {
        // one launch reduces up to kMaxGammaProblems gammas of a W call; a flush
        // covers up to max_inflight microbatches at once
        const int per_layer = c.kind == ZB_LAYER_TRANSFORMER ? 2 : 1;
        const size_t batch = static_cast<size_t>(std::min(zbk::kMaxGammaProblems, per_layer * c.n_layers));
        L.gamma_scratch_bytes = batch * zbk::rmsnorm_gamma_scratch_bytes(
            static_cast<int>(std::min<size_t>(T * slots, static_cast<size_t>(kMaxTokens))), c.hidden);
        L.gamma_scratch = total;
        total += round_up(L.gamma_scratch_bytes);
    }
    // K-split scratch for the split tiles of one launch: no more than the
    // tiles of the stage's largest GEMM output, nor than kSplitMaxTiles.
    {
        const int64_t Tt = static_cast<int64_t>(c.max_tokens);
        auto tiles = [](int64_t m, int64_t n) { return ((m + 255) / 256) * ((n + 255) / 256); };
        int64_t most = 0;
        const int64_t Hh = c.hidden, Ff = c.ffn;
        if (c.kind == ZB_LAYER_LINEAR) {
            most = std::max({tiles(Tt, Ff), tiles(Tt, Hh), tiles(Ff, Hh)});
        } else {
            most = std::max({tiles(Tt, 2 * Ff), tiles(Tt, Hh), tiles(2 * Ff, Hh), tiles(Hh, Ff)});
            if (c.kind == ZB_LAYER_TRANSFORMER) most = std::max(most, tiles(qkv_width(c), Hh));
        }
        L.split_tiles = static_cast<int>(std::min<int64_t>(most, zbk::kSplitMaxTiles));
        L.split_flags = total;
        total += round_up(static_cast<size_t>(L.split_tiles) * zbk::kSplitTileFlagBytes);
        L.split_partial = total;
        total += round_up(static_cast<size_t>(L.split_tiles) * zbk::kSplitTilePartialBytes);
    }
    L.total = total;
    return L;
}

}  // namespace

// Event pairs around launches, booked per kernel class (zb_stage_set_tracing).
struct Tracer {
    struct Rec {
        int cls;
        int launches;
        double flops, bytes;
        cudaEvent_t a, b;
    };
    bool on = false;
    std::vector<cudaEvent_t> pool;
    size_t used = 0;
    std::vector<Rec> recs;

    cudaEvent_t next() {
        if (used == pool.size()) {
            cudaEvent_t e = nullptr;
            if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
            pool.push_back(e);
        }
        return pool[used++];
    }
    ~Tracer() {
        for (cudaEvent_t e : pool) cudaEventDestroy(e);
    }
};

struct zb_stage {
    zb_stage_config cfg;
    Tracer tr;
    std::vector<zb_layer_params> prm;
    uint8_t* ws = nullptr;
    Layout lay;
    std::vector<char> slot_used;
    std::map<int32_t, MbEntry> mbs;
    int32_t inflight = 0;
    int32_t peak = 0;
    bool split_zeroed = false;  // K-split flags cleared on the device

    template <typename T = void>
    T* at(int slot, const Region& r) const {
        return reinterpret_cast<T*>(ws + r.off + r.stride * static_cast<size_t>(slot));
    }
};

namespace {

// Runs `fn` (which enqueues on `s`); with tracing on, brackets it with events
// and books `launches` kernels doing `flops` / `bytes` of algorithmic work.
template <typename Fn>
zb_status traced(zb_stage* st, zb_kernel_class cls, int launches, double flops, double bytes,
                 cudaStream_t s, Fn&& fn) {
    if (!st->tr.on) return fn();
    cudaEvent_t a = st->tr.next(), b = st->tr.next();
    if (!a || !b || cudaEventRecord(a, s) != cudaSuccess) return ZB_ERR_CUDA;
    const zb_status r = fn();
    if (cudaEventRecord(b, s) != cudaSuccess) return ZB_ERR_CUDA;
    st->tr.recs.push_back(Tracer::Rec{cls, launches, flops, bytes, a, b});
    return r;
}

// The stage's K-split scratch; its flags are cleared on `s` before first use.
zb_status stage_split_ws(zb_stage* st, cudaStream_t s, SplitWs* out) {
    const Layout& L = st->lay;
    if (!st->split_zeroed) {
        if (cudaMemsetAsync(st->ws + L.split_flags, 0, static_cast<size_t>(L.split_tiles) * zbk::kSplitTileFlagBytes,
                            s) != cudaSuccess)
            return ZB_ERR_CUDA;
        st->split_zeroed = true;
    }
    out->flags = reinterpret_cast<uint32_t*>(st->ws + L.split_flags);
    out->partial = reinterpret_cast<float*>(st->ws + L.split_partial);
    out->tiles = L.split_tiles;
    return ZB_OK;
}

// Algorithmic work of one GEMM launch (every operand read once, every result
// written once; float32 accumulators read and written).
double gemm_flops(double m, double n, double k) { return 2.0 * m * n * k; }
double fwd_bytes(double m, double n, double k, bool resid) { return 2.0 * (m * k + n * k + m * n) + (resid ? 2.0 * m * n : 0.0); }
double dgrad_bytes(double m, double n, double k) { return 2.0 * (m * k + k * n + m * n); }
double dgrad_swiglu_bytes(double m, double n, double k) { return 2.0 * (m * k + k * n) + 8.0 * m * n; }
double wgrad_bytes(double m, double n, double k) { return 2.0 * (k * m + k * n) + 8.0 * m * n; }
double rms_bwd_bytes(double t, double h) { return 8.0 * t * h + 4.0 * t + 4.0 * h; }
double dgamma_bytes(double t, double h) { return 4.0 * t * h + 4.0 * t + 8.0 * h; }

zb_status check_layer_params(const zb_stage_config& c, const zb_layer_params& p) {
    auto ok = [](const void* q) { return q && aligned16(q); };
    switch (c.kind) {
        case ZB_LAYER_LINEAR:
            return ok(p.w) && ok(p.dw) ? ZB_OK : ZB_ERR_ARG;
        case ZB_LAYER_TRANSFORMER:
            if (!ok(p.w_qkv) || !ok(p.dw_qkv) || !ok(p.w_o) || !ok(p.dw_o) || !ok(p.gamma1) ||
                !ok(p.dgamma1))
                return ZB_ERR_ARG;
            [[fallthrough]];
        case ZB_LAYER_MLP:
            if (!ok(p.w_gu) || !ok(p.dw_gu) || !ok(p.w_down) || !ok(p.dw_down) || !ok(p.gamma2) ||
                !ok(p.dgamma2))
                return ZB_ERR_ARG;
            return ZB_OK;
    }
    return ZB_ERR_ARG;
}

// Stash copy of a caller tensor (x at F, dy at B), booked in its own class: its
// time and bytes count, but not as a launch (it is a copy, not one of the
// library's kernels).
zb_status stash_copy(zb_stage* st, void* dst, const void* src, size_t bytes, cudaStream_t s) {
    if (!bytes) return ZB_OK;
    return traced(st, ZB_KCLASS_STASH_COPY, 0, 0.0, 2.0 * bytes, s, [&] {
        return cuda_status(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s));
    });
}

// F of one microbatch already holding `slot`.
zb_status stage_forward_body(zb_stage* st, int slot, const void* x, int t, void* y, cudaStream_t s) {
    const zb_stage_config& c = st->cfg;
    const int H = c.hidden, F = c.ffn, Q = qkv_width(c);
    const double T = t;
    ZB_TRY(stash_copy(st, st->at(slot, st->lay.layers[0].x), x, static_cast<size_t>(t) * H * 2, s));
    if (t == 0) return ZB_OK;
    SplitWs ws;
    ZB_TRY(stage_split_ws(st, s, &ws));
    if (c.kind == ZB_LAYER_LINEAR) {
        const zb_layer_params& p = st->prm[0];
        return traced(st, ZB_KCLASS_GEMM_FORWARD, 1, gemm_flops(T, F, H), fwd_bytes(T, F, H, false), s, [&] {
            return run_linear_forward(st->at(slot, st->lay.layers[0].x), p.w, nullptr, y, t, H, F, s, &ws);
        });
    }
    for (int l = 0; l < c.n_layers; ++l) {
        const zb_layer_params& p = st->prm[l];
        const LayerSlot& L = st->lay.layers[l];
        void* xin = st->at(slot, L.x);
        void* yout = l + 1 < c.n_layers ? st->at(slot, st->lay.layers[l + 1].x) : y;
        if (c.kind == ZB_LAYER_TRANSFORMER) {
            const bool causal = c.attention == ZB_ATTN_CAUSAL;
            void* qkv = causal ? st->at(slot, L.qkv) : st->ws + st->lay.qkv_tmp;
            ZB_TRY(traced(st, ZB_KCLASS_ROW_FORWARD, 1, 0.0, 4.0 * T * H + 4.0 * T, s, [&] {
                return cuda_status(zbk::launch_rmsnorm_forward(xin, p.gamma1, c.eps, st->at(slot, L.n1),
                                                               st->at<float>(slot, L.r1), t, H, s));
            }));
            ZB_TRY(traced(st, ZB_KCLASS_GEMM_FORWARD, 1, gemm_flops(T, Q, H), fwd_bytes(T, Q, H, false), s, [&] {
                return run_linear_forward(st->at(slot, L.n1), p.w_qkv, nullptr, qkv, t, H, Q, s, &ws);
            }));
            if (causal) {
                const double pairs = causal_pairs(t, c.seq_len) * c.n_heads;
                ZB_TRY(traced(st, ZB_KCLASS_ATTN_FORWARD, 1, 4.0 * c.head_dim * pairs, 2.0 * T * (Q + H) + 4.0 * T * c.n_heads, s,
                              [&] {
                                  return cuda_status(zbk::launch_attention_causal_forward(
                                      attn_shape(t, c.n_heads, c.n_kv_heads, c.head_dim, c.seq_len, st->lay.ld_stat), qkv,
                                      st->at(slot, L.a), st->at<float>(slot, L.lse), s));
                              }));
            } else {
                ZB_TRY(traced(st, ZB_KCLASS_ROW_FORWARD, 1, 0.0, 2.0 * T * (Q + H), s, [&] {
                    return cuda_status(zbk::launch_attention_forward(qkv, st->at(slot, L.a), t, c.n_heads,
                                                                     c.n_kv_heads, c.head_dim, s));
                }));
            }
            ZB_TRY(traced(st, ZB_KCLASS_GEMM_FORWARD, 1, gemm_flops(T, H, H), fwd_bytes(T, H, H, true), s, [&] {
                return run_linear_forward(st->at(slot, L.a), p.w_o, xin, st->at(slot, L.h), t, H, H, s, &ws);
            }));
        }
        void* h = st->at(slot, L.h);
        ZB_TRY(traced(st, ZB_KCLASS_ROW_FORWARD, 1, 0.0, 4.0 * T * H + 4.0 * T, s, [&] {
            return cuda_status(zbk::launch_rmsnorm_forward(h, p.gamma2, c.eps, st->at(slot, L.n2),
                                                           st->at<float>(slot, L.r2), t, H, s));
        }));
        if (swiglu_forward_fused(t, F)) {
            // one launch: the epilogue also writes s (2 T F bytes more than the plain GEMM)
            ZB_TRY(traced(st, ZB_KCLASS_GEMM_FORWARD, 1, gemm_flops(T, 2.0 * F, H),
                          fwd_bytes(T, 2.0 * F, H, false) + 2.0 * T * F, s, [&] {
                              return run_linear_forward_swiglu(st->at(slot, L.n2), p.w_gu, st->at(slot, L.gu),
                                                               st->at(slot, L.s), t, H, F, s, &ws);
                          }));
        } else {
            ZB_TRY(traced(st, ZB_KCLASS_GEMM_FORWARD, 1, gemm_flops(T, 2.0 * F, H), fwd_bytes(T, 2.0 * F, H, false),
                          s, [&] {
                              return run_linear_forward(st->at(slot, L.n2), p.w_gu, nullptr, st->at(slot, L.gu), t, H,
                                                        2 * F, s, &ws);
                          }));
            ZB_TRY(traced(st, ZB_KCLASS_ROW_FORWARD, 1, 0.0, 6.0 * T * F, s, [&] {
                return cuda_status(zbk::launch_swiglu_forward(st->at(slot, L.gu), st->at(slot, L.s), t, F, s));
            }));
        }
        ZB_TRY(traced(st, ZB_KCLASS_GEMM_FORWARD, 1, gemm_flops(T, H, F), fwd_bytes(T, H, F, true), s, [&] {
            return run_linear_forward(st->at(slot, L.s), p.w_down, h, yout, t, F, H, s, &ws);
        }));
    }
    return ZB_OK;
}

// B of one microbatch: every layer top first, only products with weights.
zb_status stage_backward_input_body(zb_stage* st, int slot, const void* dy, void* dx, int t,
                                    cudaStream_t s) {
    const zb_stage_config& c = st->cfg;
    const int H = c.hidden, F = c.ffn, Q = qkv_width(c);
    const double T = t;
    const int top = c.n_layers - 1;
    const int out_dim = c.kind == ZB_LAYER_LINEAR ? F : H;
    ZB_TRY(stash_copy(st, st->at(slot, st->lay.layers[top].dy), dy, static_cast<size_t>(t) * out_dim * 2, s));
    if (t == 0) return ZB_OK;
    SplitWs ws;
    ZB_TRY(stage_split_ws(st, s, &ws));
    if (c.kind == ZB_LAYER_LINEAR)
        return traced(st, ZB_KCLASS_GEMM_BACKWARD_INPUT, 1, gemm_flops(T, H, F), dgrad_bytes(T, H, F), s, [&] {
            return run_backward_input(st->at(slot, st->lay.layers[0].dy), st->prm[0].w, dx, t, H, F, H, s, &ws);
        });
    for (int l = top; l >= 0; --l) {
        const zb_layer_params& p = st->prm[l];
        const LayerSlot& L = st->lay.layers[l];
        void* dyl = st->at(slot, L.dy);
        void* dx_out = l > 0 ? st->at(slot, st->lay.layers[l - 1].dy) : dx;
        void* gu = st->at(slot, L.gu);
        void* dn2 = st->at(slot, L.dn2);
        // a1: down projection B with the SwiGLU backward fused; [g|u] becomes [dg|du]
        ZB_TRY(traced(st, ZB_KCLASS_GEMM_BACKWARD_INPUT, 1, gemm_flops(T, F, H), dgrad_swiglu_bytes(T, F, H), s,
                      [&] { return run_backward_input_swiglu(dyl, p.w_down, gu, gu, t, H, F, s, &ws); }));
        // a2: gate|up B, then RMSNorm backward onto the residual gradient
        void* dh = c.kind == ZB_LAYER_TRANSFORMER ? st->at(slot, L.dh) : dx_out;
        ZB_TRY(traced(st, ZB_KCLASS_GEMM_BACKWARD_INPUT, 1, gemm_flops(T, H, 2.0 * F), dgrad_bytes(T, H, 2.0 * F), s,
                      [&] { return run_backward_input(gu, p.w_gu, dn2, t, H, 2 * F, H, s, &ws); }));
        ZB_TRY(traced(st, ZB_KCLASS_ROW_BACKWARD_INPUT, 1, 0.0, rms_bwd_bytes(T, H), s, [&] {
            return cuda_status(zbk::launch_rmsnorm_backward_input(dn2, st->at(slot, L.h), st->at<float>(slot, L.r2),
                                                                  p.gamma2, dyl, dh, t, H, s));
        }));
        if (c.kind == ZB_LAYER_TRANSFORMER) {
            void* dqkv = st->at(slot, L.dqkv);
            void* dn1 = st->at(slot, L.dn1);
            const double kv = static_cast<double>(c.n_kv_heads) * c.head_dim;
            if (c.attention == ZB_ATTN_CAUSAL) {
                // a3: output projection B into a temporary, then the attention backward
                // (dK/dV, dQ) writes every column of dqkv.  D = rowsum(da * a) per
                // head comes from the GEMM's epilogue when the CTA-pair kernel
                // takes it, else from a row kernel before dK/dV and dQ.
                void* da = st->ws + st->lay.da_tmp;
                float* dvec = reinterpret_cast<float*>(st->ws + st->lay.dvec);
                const bool d_in_gemm = zbk::gemm_takes_pair(t, H);
                ZB_TRY(traced(st, ZB_KCLASS_GEMM_BACKWARD_INPUT, 1, gemm_flops(T, H, H),
                              dgrad_bytes(T, H, H) + (d_in_gemm ? 2.0 * T * H + 4.0 * T * c.n_heads : 0.0), s, [&] {
                                  return d_in_gemm ? run_backward_input_rowdot(dh, p.w_o, da, st->at(slot, L.a), dvec,
                                                                               st->lay.ld_stat, c.head_dim, t, H, H,
                                                                               s, &ws)
                                                   : run_backward_input(dh, p.w_o, da, t, H, H, H, s, &ws);
                              }));
                const double pairs = causal_pairs(t, c.seq_len) * c.n_heads;
                ZB_TRY(traced(st, ZB_KCLASS_ATTN_BACKWARD, d_in_gemm ? 2 : 3, 10.0 * c.head_dim * pairs,
                              2.0 * T * (2.0 * Q + (d_in_gemm ? 1.0 : 2.0) * H) + 8.0 * T * c.n_heads, s, [&] {
                                  return cuda_status(zbk::launch_attention_causal_backward(
                                      attn_shape(t, c.n_heads, c.n_kv_heads, c.head_dim, c.seq_len, st->lay.ld_stat),
                                      st->at(slot, L.qkv), st->at(slot, L.a), da, st->at<float>(slot, L.lse), dvec,
                                      dqkv, s, d_in_gemm));
                              }));
            } else {
                // a3: output projection B (into the q columns of dqkv) and the stand-in backward
                ZB_TRY(traced(st, ZB_KCLASS_GEMM_BACKWARD_INPUT, 1, gemm_flops(T, H, H), dgrad_bytes(T, H, H), s,
                              [&] { return run_backward_input(dh, p.w_o, dqkv, t, H, H, Q, s, &ws); }));
                ZB_TRY(traced(st, ZB_KCLASS_ROW_BACKWARD_INPUT, 1, 0.0, 2.0 * T * H + 4.0 * T * kv, s, [&] {
                    return cuda_status(zbk::launch_attention_backward_kv(dqkv, t, c.n_heads, c.n_kv_heads, c.head_dim, s));
                }));
            }
            // a4: qkv B, then RMSNorm backward onto dh
            ZB_TRY(traced(st, ZB_KCLASS_GEMM_BACKWARD_INPUT, 1, gemm_flops(T, H, Q), dgrad_bytes(T, H, Q), s,
                          [&] { return run_backward_input(dqkv, p.w_qkv, dn1, t, H, Q, H, s, &ws); }));
            ZB_TRY(traced(st, ZB_KCLASS_ROW_BACKWARD_INPUT, 1, 0.0, rms_bwd_bytes(T, H), s, [&] {
                return cuda_status(zbk::launch_rmsnorm_backward_input(dn1, st->at(slot, L.x), st->at<float>(slot, L.r1),
                                                                      p.gamma1, dh, dx_out, t, H, s));
            }));
        }
    }
    return ZB_OK;
}

// W of one microbatch: dW += dY^T X for every linear, dgamma reductions.
zb_status stage_backward_weight_body(zb_stage* st, int slot, int t, cudaStream_t s) {
    if (t == 0) return ZB_OK;
    const zb_stage_config& c = st->cfg;
    const int H = c.hidden, F = c.ffn, Q = qkv_width(c);
    const double T = t;
    SplitWs ws;
    ZB_TRY(stage_split_ws(st, s, &ws));
    if (c.kind == ZB_LAYER_LINEAR) {
        const LayerSlot& L = st->lay.layers[0];
        return traced(st, ZB_KCLASS_GEMM_BACKWARD_WEIGHT, 1, gemm_flops(F, H, T), wgrad_bytes(F, H, T), s, [&] {
            return run_backward_weight(st->at(slot, L.dy), st->at(slot, L.x), st->prm[0].dw, t, H, F, s, &ws);
        });
    }
    // Every weight gradient of the call, run as grouped launches: the GEMMs are
    // independent, and one stream of tiles fills the last waves of the small
    // ones with tiles of the others.
    std::vector<GemmArgs> wg;
    auto wgrad = [&](const void* dyv, const void* xv, float* dw, int in, int out) {
        wg.push_back(wgrad_args(dyv, xv, dw, t, in, out));
        return ZB_OK;
    };
    float* scratch = reinterpret_cast<float*>(st->ws + st->lay.gamma_scratch);
    // Every RMSNorm gamma reduction of the call runs in one launch pair.
    std::vector<zbk::GammaProblem> gammas;
    for (int l = 0; l < c.n_layers; ++l) {
        const zb_layer_params& p = st->prm[l];
        const LayerSlot& L = st->lay.layers[l];
        ZB_TRY(wgrad(st->at(slot, L.dy), st->at(slot, L.s), p.dw_down, F, H));
        ZB_TRY(wgrad(st->at(slot, L.gu), st->at(slot, L.n2), p.dw_gu, H, 2 * F));
        gammas.push_back({st->at(slot, L.dn2), st->at(slot, L.h), st->at<float>(slot, L.r2), p.dgamma2});
        if (c.kind == ZB_LAYER_TRANSFORMER) {
            ZB_TRY(wgrad(st->at(slot, L.dh), st->at(slot, L.a), p.dw_o, H, H));
            ZB_TRY(wgrad(st->at(slot, L.dqkv), st->at(slot, L.n1), p.dw_qkv, H, Q));
            gammas.push_back({st->at(slot, L.dn1), st->at(slot, L.x), st->at<float>(slot, L.r1), p.dgamma1});
        }
    }
    for (size_t g0 = 0; g0 < wg.size(); g0 += zbk::kMaxGroup) {
        const int n = static_cast<int>(std::min<size_t>(zbk::kMaxGroup, wg.size() - g0));
        double fl = 0.0, by = 0.0;
        for (int i = 0; i < n; ++i) {
            const GemmArgs& g = wg[g0 + i];
            fl += gemm_flops(g.m, g.n, g.k);
            by += wgrad_bytes(g.m, g.n, g.k);
        }
        ZB_TRY(traced(st, ZB_KCLASS_GEMM_BACKWARD_WEIGHT, 1, fl, by, s,
                      [&] { return cuda_status(zbk::launch_gemm_group(wg.data() + g0, n, s)); }));
    }
    for (size_t g0 = 0; g0 < gammas.size(); g0 += zbk::kMaxGammaProblems) {
        const int n = static_cast<int>(std::min<size_t>(zbk::kMaxGammaProblems, gammas.size() - g0));
        ZB_TRY(traced(st, ZB_KCLASS_ROW_BACKWARD_WEIGHT, 2, 0.0, n * dgamma_bytes(T, H), s, [&] {
            return cuda_status(zbk::launch_rmsnorm_backward_gamma_batch(gammas.data() + g0, n, t, H, scratch, s));
        }));
    }
    return ZB_OK;
}

}  // namespace

extern "C" size_t zb_stage_workspace_bytes(const zb_stage_config* cfg) {
    if (check_config(cfg) != ZB_OK) return 0;
    return make_layout(*cfg).total;
}

extern "C" zb_status zb_stage_create(const zb_stage_config* cfg, const zb_layer_params* layers,
                                     void* workspace, size_t workspace_bytes, zb_stage_t* out) {
    if (!out) return ZB_ERR_ARG;
    *out = nullptr;
    ZB_TRY(check_config(cfg));
    if (!layers) return ZB_ERR_ARG;
    for (int l = 0; l < cfg->n_layers; ++l) ZB_TRY(check_layer_params(*cfg, layers[l]));
    const Layout lay = make_layout(*cfg);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 || workspace_bytes < lay.total)
        return ZB_ERR_WORKSPACE;
    zb_stage* st = new (std::nothrow) zb_stage();
    if (!st) return ZB_ERR_ARG;
    st->cfg = *cfg;
    st->prm.assign(layers, layers + cfg->n_layers);
    st->ws = static_cast<uint8_t*>(workspace);
    st->lay = lay;
    st->slot_used.assign(cfg->max_inflight, 0);
    *out = st;
    return ZB_OK;
}

extern "C" zb_status zb_stage_destroy(zb_stage_t st) {
    delete st;
    return ZB_OK;
}

extern "C" zb_status zb_stage_forward(zb_stage_t st, int32_t mb, const void* x, int32_t tokens, void* y,
                                      void* stream) {
    if (!st || mb < 0) return ZB_ERR_ARG;
    if (tokens < 0 || tokens > st->cfg.max_tokens) return ZB_ERR_SHAPE;
    if (!rows_ok(x, tokens) || !rows_ok(y, tokens)) return ZB_ERR_ARG;
    if (st->mbs.count(mb)) return ZB_ERR_ORDER;
    int slot = -1;
    for (int i = 0; i < st->cfg.max_inflight; ++i)
        if (!st->slot_used[i]) {
            slot = i;
            break;
        }
    if (slot < 0) return ZB_ERR_STASH_FULL;
    ZB_TRY(device_ok());
    if (st->cfg.attention == ZB_ATTN_CAUSAL && zbk::attention_prepare() != cudaSuccess) return ZB_ERR_CUDA;
    ZB_TRY(stage_forward_body(st, slot, x, tokens, y, as_stream(stream)));
    st->slot_used[slot] = 1;
    st->mbs[mb] = MbEntry{MbState::Forwarded, slot, tokens};
    st->inflight += 1;
    st->peak = std::max(st->peak, st->inflight);
    return ZB_OK;
}

extern "C" zb_status zb_backward_input(zb_stage_t st, int32_t mb, const void* dy, void* dx, void* stream) {
    if (!st || mb < 0) return ZB_ERR_ARG;
    auto it = st->mbs.find(mb);
    if (it == st->mbs.end()) return ZB_ERR_NO_MB;
    if (it->second.state != MbState::Forwarded) return ZB_ERR_ORDER;
    if (!rows_ok(dy, it->second.tokens) || !rows_ok(dx, it->second.tokens)) return ZB_ERR_ARG;
    ZB_TRY(device_ok());
    ZB_TRY(stage_backward_input_body(st, it->second.slot, dy, dx, it->second.tokens, as_stream(stream)));
    it->second.state = MbState::BackwardInputDone;
    return ZB_OK;
}

extern "C" zb_status zb_backward_weight(zb_stage_t st, int32_t mb, void* stream) {
    if (!st || mb < 0) return ZB_ERR_ARG;
    auto it = st->mbs.find(mb);
    if (it == st->mbs.end()) return ZB_ERR_NO_MB;
    if (it->second.state != MbState::BackwardInputDone) return ZB_ERR_ORDER;
    ZB_TRY(device_ok());
    ZB_TRY(stage_backward_weight_body(st, it->second.slot, it->second.tokens, as_stream(stream)));
    st->slot_used[it->second.slot] = 0;
    st->mbs.erase(it);
    st->inflight -= 1;
    return ZB_OK;
}

extern "C" zb_status zb_wgrad_flush(zb_stage_t st, void* stream) {
    if (!st) return ZB_ERR_ARG;
    // Pending microbatches (B done, W not), by stash slot.
    std::vector<std::pair<int, int32_t>> pending;  // (slot, mb)
    for (const auto& kv : st->mbs)
        if (kv.second.state == MbState::BackwardInputDone) pending.emplace_back(kv.second.slot, kv.first);
    if (pending.empty()) return ZB_OK;
    ZB_TRY(device_ok());
    std::sort(pending.begin(), pending.end());
    const int full = st->cfg.max_tokens;
    cudaStream_t s = as_stream(stream);
    size_t i = 0;
    while (i < pending.size()) {
        // A run: consecutive slots whose microbatches all have max_tokens tokens.
        // Their stashes are one [k * max_tokens, width] matrix per tensor, so one W
        // over the concatenated tokens gives the sum of the k microbatches' W
        // (every op but the weight contractions is per token).
        size_t j = i + 1;
        const bool first_full = st->mbs[pending[i].second].tokens == full;
        while (first_full && j < pending.size() && pending[j].first == pending[j - 1].first + 1 &&
               st->mbs[pending[j].second].tokens == full &&
               static_cast<int64_t>(j + 1 - i) * full <= kMaxTokens)
            ++j;
        const int slot0 = pending[i].first;
        const int tokens = first_full ? static_cast<int>(j - i) * full : st->mbs[pending[i].second].tokens;
        ZB_TRY(stage_backward_weight_body(st, slot0, tokens, s));
        for (size_t q = i; q < j; ++q) {
            st->slot_used[pending[q].first] = 0;
            st->mbs.erase(pending[q].second);
            st->inflight -= 1;
        }
        i = j;
    }
    return ZB_OK;
}

extern "C" zb_status zb_stage_sync(zb_stage_t st, void* stream) {
    if (!st) return ZB_ERR_ARG;
    return zb_device_status(stream, 0, nullptr);
}

extern "C" zb_status zb_stage_stats(zb_stage_t st, int32_t* inflight, int32_t* peak_inflight,
                                    size_t* stash_bytes) {
    if (!st) return ZB_ERR_ARG;
    if (inflight) *inflight = st->inflight;
    if (peak_inflight) *peak_inflight = st->peak;
    if (stash_bytes) *stash_bytes = st->lay.slot_bytes * static_cast<size_t>(st->inflight);
    return ZB_OK;
}

extern "C" zb_status zb_stage_stash_view(zb_stage_t st, int32_t mb, int32_t layer, int32_t tensor,
                                        const void** ptr, int64_t* rows, int64_t* cols, int32_t* elem_bytes) {
    if (!st || !ptr || !rows || !cols || !elem_bytes || mb < 0) return ZB_ERR_ARG;
    const zb_stage_config& c = st->cfg;
    if (layer < 0 || layer >= c.n_layers || tensor < 0 || tensor >= ZB_STASH_COUNT) return ZB_ERR_ARG;
    auto it = st->mbs.find(mb);
    if (it == st->mbs.end()) return ZB_ERR_NO_MB;
    const LayerSlot& L = st->lay.layers[layer];
    const int64_t t = it->second.tokens;
    const int64_t H = c.hidden, F = c.ffn, Q = c.kind == ZB_LAYER_TRANSFORMER ? qkv_width(c) : 0;
    const Region* r = nullptr;
    int64_t nr = t, nc = H;
    int32_t eb = 2;
    switch (tensor) {
        case ZB_STASH_X: r = &L.x; break;
        case ZB_STASH_RSTD1: r = &L.r1; nc = 1; eb = 4; break;
        case ZB_STASH_N1: r = &L.n1; break;
        case ZB_STASH_A: r = &L.a; break;
        case ZB_STASH_H: r = &L.h; break;
        case ZB_STASH_RSTD2: r = &L.r2; nc = 1; eb = 4; break;
        case ZB_STASH_N2: r = &L.n2; break;
        case ZB_STASH_GU: r = &L.gu; nc = 2 * F; break;
        case ZB_STASH_S: r = &L.s; nc = F; break;
        case ZB_STASH_DY: r = &L.dy; nc = c.kind == ZB_LAYER_LINEAR ? F : H; break;
        case ZB_STASH_DN2: r = &L.dn2; break;
        case ZB_STASH_DH: r = &L.dh; break;
        case ZB_STASH_DQKV: r = &L.dqkv; nc = Q; break;
        case ZB_STASH_DN1: r = &L.dn1; break;
        case ZB_STASH_QKV: r = &L.qkv; nc = Q; break;
        case ZB_STASH_LSE: r = &L.lse; nr = c.n_heads; nc = st->lay.ld_stat; eb = 4; break;
        default: return ZB_ERR_ARG;
    }
    if (!r || r->off == kNone) return ZB_ERR_ARG;  // not stashed for this layer kind
    *ptr = st->ws + r->off + r->stride * static_cast<size_t>(it->second.slot);
    *rows = nr;
    *cols = nc;
    *elem_bytes = eb;
    return ZB_OK;
}

extern "C" zb_status zb_stage_set_tracing(zb_stage_t st, int32_t enable) {
    if (!st) return ZB_ERR_ARG;
    st->tr.on = enable != 0;
    return ZB_OK;
}

extern "C" zb_status zb_stage_read_tracing(zb_stage_t st, zb_kernel_stats* out, int32_t reset) {
    if (!st || !out) return ZB_ERR_ARG;
    for (int i = 0; i < ZB_KCLASS_COUNT; ++i) out[i] = zb_kernel_stats{0, 0, 0.0, 0.0, 0.0};
    for (const Tracer::Rec& r : st->tr.recs) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return ZB_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return ZB_ERR_CUDA;
        zb_kernel_stats& o = out[r.cls];
        o.launches += r.launches;
        o.ms += ms;
        o.flops += r.flops;
        o.bytes += r.bytes;
    }
    if (reset) {
        st->tr.recs.clear();
        st->tr.used = 0;
    }
    return ZB_OK;
}
