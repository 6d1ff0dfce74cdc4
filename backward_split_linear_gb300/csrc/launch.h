// Host-side launchers of the sm_103a kernels (internal to libzb).
// Every launcher enqueues on `stream` and returns a cudaError_t from the
// launch; argument checking happens in the C-ABI layer above.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace zbk {

// Which operand layouts a GEMM sees (see gemm.cu):
//   Forward:       C[M,N] = A[M,K] B[N,K]^T   (x w^T: both K-major)
//   BackwardInput: C[M,N] = A[M,K] B[K,N]     (dy w: B is MN-major)
//   BackwardWeight C[M,N] += A[K,M]^T B[K,N]  (dy^T x: both MN-major)
enum class GemmKind : int { Forward = 0, BackwardInput = 1, BackwardWeight = 2 };

enum class Epilogue : int {
    StoreBf16 = 0,     // out bf16 = acc
    AddResidual = 1,   // out bf16 = acc + aux (bf16, row stride ld_aux)
    SwigluBwd = 2,     // acc = ds; aux holds [g | u] (row stride ld_aux), out = [dg | du]
    AccumF32 = 3,      // out f32 += acc
    SwigluFwd = 4,     // b = [W_gate; W_up] (2 ffn rows): out = [g | u] (bf16, row stride ldo) and
                       // out2 = silu(g) u from the bf16 g and u (row stride ldo2); n = 2 ffn
    StoreBf16RowDot = 5,  // out bf16 = acc, and for every row m and every group j of dot_cols output
                          // columns dot[j ld_dot + m] = sum over the group of bf16(acc) aux (bf16, row
                          // stride ld_aux): the attention backward's D = rowsum(dO * O) per head when
                          // out is dO and aux is O.  CTA-pair kernel, BackwardInput only
};

struct GemmArgs {
    GemmKind kind;
    Epilogue epi;
    const void* a;     // bf16
    int64_t lda;       // row stride of a in elements
    const void* b;     // bf16
    int64_t ldb;
    int m, n, k;
    void* out;         // bf16 or f32 (AccumF32)
    int64_t ldo;
    const void* aux;   // residual or [g | u]
    int64_t ld_aux;
    int ffn;           // SwigluBwd, SwigluFwd: column offset of u (and du) in aux and out
    void* out2;        // SwigluFwd: s [m, ffn] bf16
    int64_t ldo2;
    // Optional K-split scratch.  A CTA-pair launch whose last wave of tiles
    // would leave at least half of the CTA pairs idle cuts the K of that
    // wave's tiles in two halves computed by different CTA pairs; the half
    // that finishes second adds the other's float32 partial tile.
    // `split_flags` holds kSplitTileFlagBytes per split tile and must be
    // zeroed once before its first use (it is never reset: each launch tags
    // its flags with a new epoch); `split_partial` holds
    // kSplitTilePartialBytes per split tile.  Launches whose last wave has
    // more tiles than `split_tiles` do not split.  Launches sharing the
    // scratch must not overlap.
    uint32_t* split_flags;
    float* split_partial;
    int split_tiles;
    // StoreBf16RowDot: float32 sums, one row of m per column group (dot_cols is
    // 32, 64 or 128 and divides n; aux 16-byte aligned, ld_aux a multiple of 8).
    float* dot;
    int64_t ld_dot;
    int dot_cols;
};

constexpr size_t kSplitTileFlagBytes = 8 * 4;            // one word per 32 rows of a 256 x 256 tile
constexpr size_t kSplitTilePartialBytes = 256 * 256 * 4;  // one float32 tile
// At most this many tiles split in one launch (16 MiB of partials): a last
// wave that splits holds at most half as many tiles as there are CTA pairs.
constexpr int kSplitMaxTiles = 64;

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream);
// Whether an m x n output takes the CTA-pair kernel (the one that has the
// StoreBf16RowDot epilogue).
bool gemm_takes_pair(int m, int n);

// Up to kMaxGroup independent GEMMs in one launch when they all take the
// CTA-pair kernel with the same layouts and epilogue (else one launch each).
// Their outputs must not overlap.  Grouped GEMMs never split K.
constexpr int kMaxGroup = 16;
cudaError_t launch_gemm_group(const GemmArgs* gs, int n, cudaStream_t stream);

cudaError_t launch_rmsnorm_forward(const void* x, const float* gamma, float eps, void* n,
                                   float* rstd, int tokens, int hidden, cudaStream_t stream);
cudaError_t launch_rmsnorm_backward_input(const void* dn, const void* x, const float* rstd,
                                          const float* gamma, const void* dres, void* dx,
                                          int tokens, int hidden, cudaStream_t stream);
// One gamma-gradient reduction: dgamma[j] += sum_t dn[t, j] x[t, j] rstd[t].
struct GammaProblem {
    const void* dn;
    const void* x;
    const float* rstd;
    float* dgamma;
};
constexpr int kMaxGammaProblems = 16;

// Scratch bytes of one reduction; a batch of n needs n times as much.  For
// hidden <= kGammaMaxPartialFloats it is at most 4 * kGammaMaxPartialFloats
// bytes, whatever the token count.
constexpr int kGammaMaxPartialFloats = 1 << 17;
size_t rmsnorm_gamma_scratch_bytes(int tokens, int hidden);
// Up to kMaxGammaProblems reductions of the same [tokens, hidden] shape in one
// launch pair; each problem's result is the same bits as when run alone.
cudaError_t launch_rmsnorm_backward_gamma_batch(const GammaProblem* probs, int n, int tokens, int hidden,
                                                float* scratch, cudaStream_t stream);
cudaError_t launch_rmsnorm_backward_gamma(const void* dn, const void* x, const float* rstd,
                                          float* dgamma, int tokens, int hidden, float* scratch,
                                          cudaStream_t stream);
cudaError_t launch_swiglu_forward(const void* gu, void* s, int tokens, int ffn,
                                  cudaStream_t stream);
cudaError_t launch_attention_forward(const void* qkv, void* a, int tokens, int n_heads,
                                     int n_kv_heads, int head_dim, cudaStream_t stream);
// dqkv holds da in its q columns on entry; fills the k and v columns.
cudaError_t launch_attention_backward_kv(void* dqkv, int tokens, int n_heads, int n_kv_heads,
                                         int head_dim, cudaStream_t stream);
cudaError_t launch_selftest_wait(int limit_us, cudaStream_t stream);

// Causal softmax attention with grouped K/V heads (attention.cu).  qkv is
// [tokens, (n_heads + 2 n_kv_heads) head_dim] bf16 (q heads, then k, then v),
// a and da are [tokens, n_heads head_dim] bf16, lse and dvec are float32
// [n_heads][ld_stat] with ld_stat a multiple of 128 and >= tokens rounded up
// to 128.  head_dim is 64 or 128; seq_len is 0 or a multiple of 128.
struct AttnShape {
    int tokens, n_heads, n_kv_heads, head_dim, seq_len, ld_stat;
};
cudaError_t launch_attention_causal_forward(const AttnShape& s, const void* qkv, void* a, float* lse,
                                            cudaStream_t stream);
// Writes all of dqkv (dq, dk, dv); dvec is scratch of the lse's shape.  Runs the
// dK/dV kernel on `stream` and the dQ kernel on a per-device side stream forked
// from it and joined back.  With dvec_ready, dvec already holds D = rowsum(da * a)
// per head (from the epilogue of the GEMM that wrote da) and the row kernel that
// forms it is skipped.
cudaError_t launch_attention_causal_backward(const AttnShape& s, const void* qkv, const void* a, const void* da,
                                             const float* lse, float* dvec, void* dqkv, cudaStream_t stream,
                                             bool dvec_ready = false);
// Creates the current device's side stream, events and dQ tile counter ahead
// of the first backward (a stage calls it at its first forward, so that nothing
// is created or allocated while the caller's stream may be capturing a graph).
cudaError_t attention_prepare();

// Device status word of the current device (see zb_device_status).
int* status_word();
int sm_count();
int device_arch();  // major * 10 + minor of the current device, or -1

}  // namespace zbk
