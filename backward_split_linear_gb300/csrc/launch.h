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
    int ffn;           // SwigluBwd: column offset of u in aux and of du in out
};

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream);

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

// Scratch bytes of one reduction; a batch of n needs n times as much.
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

// Device status word of the current device (see zb_device_status).
int* status_word();
int sm_count();
int device_arch();  // major * 10 + minor of the current device, or -1

}  // namespace zbk
