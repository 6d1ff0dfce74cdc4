// Memory-bound kernels of the stage: RMSNorm forward / input backward, the
// RMSNorm gamma-gradient reduction, SwiGLU forward and the attention stand-in.
// All of them stream bf16 rows with 16-byte vector accesses (8 elements per
// access); per-row reductions use warp shuffles and one shared-memory step.
#include <algorithm>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace zbk {

namespace {

__device__ int g_status_word;  // see zb_device_status

constexpr int kRowThreads = 256;

struct V8 {
    float v[8];
};

__device__ __forceinline__ V8 load8(const uint16_t* p) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    V8 r;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        r.v[2 * e] = bf16_lo(w[e]);
        r.v[2 * e + 1] = bf16_hi(w[e]);
    }
    return r;
}

__device__ __forceinline__ void store8(uint16_t* p, const float (&v)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                              pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x < 32) {
        s = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) red[0] = s;
    }
    __syncthreads();
    s = red[0];
    __syncthreads();
    return s;
}

// ---------------------------------------------------------------- RMSNorm forward
// One block per row; thread t owns 8-element chunks t, t + 256, ... (VPT of them).
template <int VPT>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_fwd_kernel(const uint16_t* __restrict__ x,
                                                                  const float* __restrict__ gamma,
                                                                  float eps, uint16_t* __restrict__ n,
                                                                  float* __restrict__ rstd, int hidden) {
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int chunks = hidden >> 3;
    const uint16_t* xr = x + row * hidden;
    V8 xv[VPT];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * kRowThreads;
        if (c < chunks) {
            xv[i] = load8(xr + 8 * c);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss += xv[i].v[e] * xv[i].v[e];
        }
    }
    const float r = rsqrtf(block_sum(ss, red) / static_cast<float>(hidden) + eps);
    if (threadIdx.x == 0) rstd[row] = r;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * kRowThreads;
        if (c < chunks) {
            const float4 g0 = *reinterpret_cast<const float4*>(gamma + 8 * c);
            const float4 g1 = *reinterpret_cast<const float4*>(gamma + 8 * c + 4);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = g[e] * (xv[i].v[e] * r);
            store8(n + row * hidden + 8 * c, o);
        }
    }
}

// ---------------------------------------------------------------- RMSNorm input backward
// dx = dres + r (gamma dn - xh * mean(gamma dn xh)), xh = x r.
// Every load of the row (dn, x, dres) is issued before the row reduction, so
// a block keeps all of its row's bytes in flight at once.
template <int VPT>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_bwd_kernel(
    const uint16_t* __restrict__ dn, const uint16_t* __restrict__ x, const float* __restrict__ rstd,
    const float* __restrict__ gamma, const uint16_t* dres, uint16_t* dx, int hidden) {
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int chunks = hidden >> 3;
    const float r = rstd[row];
    uint4 dv[VPT], xv[VPT], rv[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * kRowThreads;
        if (c < chunks) {
            dv[i] = *reinterpret_cast<const uint4*>(dn + row * hidden + 8 * c);
            xv[i] = *reinterpret_cast<const uint4*>(x + row * hidden + 8 * c);
            rv[i] = *reinterpret_cast<const uint4*>(dres + row * hidden + 8 * c);
        }
    }
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * kRowThreads;
        if (c < chunks) {
            const float4 g0 = *reinterpret_cast<const float4*>(gamma + 8 * c);
            const float4 g1 = *reinterpret_cast<const float4*>(gamma + 8 * c + 4);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const uint32_t dw[4] = {dv[i].x, dv[i].y, dv[i].z, dv[i].w};
            const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float d = (e & 1) ? bf16_hi(dw[e >> 1]) : bf16_lo(dw[e >> 1]);
                const float xx = (e & 1) ? bf16_hi(xw[e >> 1]) : bf16_lo(xw[e >> 1]);
                dot += g[e] * d * (xx * r);
            }
        }
    }
    const float mean = block_sum(dot, red) / static_cast<float>(hidden);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int c = threadIdx.x + i * kRowThreads;
        if (c < chunks) {
            const float4 g0 = *reinterpret_cast<const float4*>(gamma + 8 * c);
            const float4 g1 = *reinterpret_cast<const float4*>(gamma + 8 * c + 4);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const uint32_t dw[4] = {dv[i].x, dv[i].y, dv[i].z, dv[i].w};
            const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
            const uint32_t rw[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float d = (e & 1) ? bf16_hi(dw[e >> 1]) : bf16_lo(dw[e >> 1]);
                const float xx = (e & 1) ? bf16_hi(xw[e >> 1]) : bf16_lo(xw[e >> 1]);
                const float res = (e & 1) ? bf16_hi(rw[e >> 1]) : bf16_lo(rw[e >> 1]);
                o[e] = res + r * (g[e] * d - (xx * r) * mean);
            }
            store8(dx + row * hidden + 8 * c, o);
        }
    }
}

// ---------------------------------------------------------------- RMSNorm gamma gradient
// Pass 1: block (cx, cy) covers columns [256 cx, 256 cx + 256) and the cy-th
// of `parts` equal token ranges.  Thread (g, c) (g = 0..7 row group, c = 0..31
// chunk of 8 columns) streams tokens t0 + g, t0 + g + 8, ... of that range,
// four tokens of loads in flight; the 8 row groups are then added in order
// g = 0..7 in shared memory and the block writes part[cy][256 columns].
// `parts` depends only on T and H (about 512 blocks in all), never on the
// device, so the partition and hence the float32 sums are reproducible.
// Pass 2: dgamma[j] += part[0][j] + part[1][j] + ... in order.
constexpr int kGammaCols = 256;                           // columns per block
constexpr int kGammaChunks = kGammaCols / 8;              // 32 threads across the columns
constexpr int kGammaGroups = kRowThreads / kGammaChunks;  // 8 row groups
constexpr int kGammaTargetBlocks = 512;
constexpr int kGammaUnroll = 4;

// parts = min(ceil(512 / column blocks), ceil(T / 8), 2^17 / H), at least 1.
// The last bound keeps the partial sums (parts * H floats) within 2^17 floats
// for every H <= 2^17, whatever T: a fixed 512 KiB buffer then serves every
// token count of those widths.  Up to H = 16384 it is never below the first
// bound, so it does not change the partition of the stage's widths.
int gamma_parts(int tokens, int hidden) {
    const int col_blocks = (hidden + kGammaCols - 1) / kGammaCols;
    const int want = (kGammaTargetBlocks + col_blocks - 1) / col_blocks;
    const int most = (tokens + kGammaGroups - 1) / kGammaGroups;  // at least 8 tokens per part
    const int fit = kGammaMaxPartialFloats / hidden;
    return std::max(1, std::min({want, most, fit}));
}

// Several reductions of the same shape in one launch: problem blockIdx.z.
struct GammaBatch {
    GammaProblem prob[kMaxGammaProblems];
    int tokens, hidden, parts;
};

__global__ void __launch_bounds__(kRowThreads) dgamma_partial_kernel(const __grid_constant__ GammaBatch b,
                                                                     float* __restrict__ part_all) {
    __shared__ float acc_s[kGammaGroups][kGammaCols];
    const uint16_t* __restrict__ dn = static_cast<const uint16_t*>(b.prob[blockIdx.z].dn);
    const uint16_t* __restrict__ x = static_cast<const uint16_t*>(b.prob[blockIdx.z].x);
    const float* __restrict__ rstd = b.prob[blockIdx.z].rstd;
    const int tokens = b.tokens, hidden = b.hidden, parts = b.parts;
    float* __restrict__ part = part_all + static_cast<int64_t>(blockIdx.z) * parts * hidden;
    const int cl = threadIdx.x % kGammaChunks;
    const int grp = threadIdx.x / kGammaChunks;
    const int col = blockIdx.x * kGammaCols + 8 * cl;
    const int per = (tokens + parts - 1) / parts;
    const int t0 = blockIdx.y * per;
    const int t1 = min(tokens, t0 + per);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (col < hidden) {
        for (int tb = t0 + grp; tb < t1; tb += kGammaGroups * kGammaUnroll) {
            uint4 dv[kGammaUnroll], xv[kGammaUnroll];
            float rr[kGammaUnroll];
#pragma unroll
            for (int i = 0; i < kGammaUnroll; ++i) {
                const int t = tb + i * kGammaGroups;
                if (t < t1) {
                    dv[i] = *reinterpret_cast<const uint4*>(dn + static_cast<int64_t>(t) * hidden + col);
                    xv[i] = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * hidden + col);
                    rr[i] = rstd[t];
                }
            }
#pragma unroll
            for (int i = 0; i < kGammaUnroll; ++i) {
                if (tb + i * kGammaGroups < t1) {
                    const uint32_t dw[4] = {dv[i].x, dv[i].y, dv[i].z, dv[i].w};
                    const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float d = (e & 1) ? bf16_hi(dw[e >> 1]) : bf16_lo(dw[e >> 1]);
                        const float xx = (e & 1) ? bf16_hi(xw[e >> 1]) : bf16_lo(xw[e >> 1]);
                        acc[e] += d * (xx * rr[i]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) acc_s[grp][8 * cl + e] = acc[e];
    __syncthreads();
    // thread j of the block finishes column j of the block's 256
    const int j = threadIdx.x;
    if (blockIdx.x * kGammaCols + j < hidden) {
        float s = 0.f;
#pragma unroll
        for (int g = 0; g < kGammaGroups; ++g) s += acc_s[g][j];
        part[static_cast<int64_t>(blockIdx.y) * hidden + blockIdx.x * kGammaCols + j] = s;
    }
}

// Pass 2: block covers 32 columns; thread (c, g) adds the partials q = g,
// g + 8, g + 16, ... of column c in order (loads issued first), then thread
// (c, 0) adds the 8 sums in order g = 0..7 and accumulates into dgamma.
constexpr int kFinalCols = 32;
constexpr int kFinalGroups = 8;
constexpr int kFinalMaxPerThread = 8;  // parts <= 64 loads issued together; more loop

__global__ void __launch_bounds__(kFinalCols * kFinalGroups) dgamma_final_kernel(const __grid_constant__ GammaBatch b,
                                                                                 const float* __restrict__ part_all) {
    __shared__ float sums[kFinalGroups][kFinalCols];
    const int parts = b.parts, hidden = b.hidden;
    const float* __restrict__ part = part_all + static_cast<int64_t>(blockIdx.y) * parts * hidden;
    float* dgamma = b.prob[blockIdx.y].dgamma;
    const int c = threadIdx.x % kFinalCols;
    const int g = threadIdx.x / kFinalCols;
    const int j = blockIdx.x * kFinalCols + c;
    float s = 0.f;
    if (j < hidden) {
        for (int q0 = g; q0 < parts; q0 += kFinalGroups * kFinalMaxPerThread) {
            float v[kFinalMaxPerThread];
#pragma unroll
            for (int i = 0; i < kFinalMaxPerThread; ++i) {
                const int q = q0 + i * kFinalGroups;
                v[i] = q < parts ? part[static_cast<int64_t>(q) * hidden + j] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kFinalMaxPerThread; ++i) s += v[i];
        }
    }
    sums[g][c] = s;
    __syncthreads();
    if (g == 0 && j < hidden) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < kFinalGroups; ++k) t += sums[k][c];
        dgamma[j] += t;
    }
}

// ---------------------------------------------------------------- SwiGLU forward
__global__ void swiglu_fwd_kernel(const uint16_t* __restrict__ gu, uint16_t* __restrict__ s,
                                  int tokens, int ffn) {
    const int cpr = ffn >> 3;
    const int64_t total = static_cast<int64_t>(tokens) * cpr;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / cpr;
        const int c = static_cast<int>(i - t * cpr);
        const uint16_t* row = gu + t * 2 * ffn;
        const V8 g = load8(row + 8 * c);
        const V8 u = load8(row + ffn + 8 * c);
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = swiglu_value(g.v[e], u.v[e]);
        store8(s + t * ffn + 8 * c, o);
    }
}

// ---------------------------------------------------------------- attention stand-in
// a[:, h] = q_h + k_j + v_j with j = h / (nh / nkv); qkv row = [q heads | k heads | v heads].
__global__ void attn_fwd_kernel(const uint16_t* __restrict__ qkv, uint16_t* __restrict__ a,
                                int tokens, int nh, int nkv, int hd) {
    const int width = nh * hd;
    const int qkv_w = (nh + 2 * nkv) * hd;
    const int group = nh / nkv;
    const int cpr = width >> 3;
    const int64_t total = static_cast<int64_t>(tokens) * cpr;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / cpr;
        const int col = 8 * static_cast<int>(i - t * cpr);
        const int h = col / hd, off = col - h * hd;
        const int j = h / group;
        const uint16_t* row = qkv + t * qkv_w;
        const V8 q = load8(row + col);
        const V8 k = load8(row + width + j * hd + off);
        const V8 v = load8(row + width + nkv * hd + j * hd + off);
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = q.v[e] + k.v[e] + v.v[e];
        store8(a + t * width + col, o);
    }
}

// dqkv holds da in its q columns; writes dk_j = dv_j = sum over the heads of group j.
__global__ void attn_bwd_kv_kernel(uint16_t* dqkv, int tokens, int nh, int nkv, int hd) {
    const int width = nh * hd;
    const int qkv_w = (nh + 2 * nkv) * hd;
    const int group = nh / nkv;
    const int cpr = (nkv * hd) >> 3;
    const int64_t total = static_cast<int64_t>(tokens) * cpr;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / cpr;
        const int col = 8 * static_cast<int>(i - t * cpr);  // inside the k block
        const int j = col / hd, off = col - j * hd;
        uint16_t* row = dqkv + t * qkv_w;
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int h = j * group; h < (j + 1) * group; ++h) {
            const V8 d = load8(row + h * hd + off);
#pragma unroll
            for (int e = 0; e < 8; ++e) s[e] += d.v[e];
        }
        store8(row + width + col, s);
        store8(row + width + nkv * hd + col, s);
    }
}

// ---------------------------------------------------------------- self test
__global__ void selftest_wait_kernel(int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    mbar_fence_init();
    // Nothing ever arrives: the bounded wait must give up and record the site.
    mbar_wait(b, 0, status, kSiteSelftest, limit_ns);
}

int grid_for(int64_t items, int threads) {
    const int64_t blocks = (items + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

int* status_word() {
    static int* ptrs[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

int sm_count() {
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (!counts[dev]) {
        int c = 0;
        cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
        counts[dev] = c > 0 ? c : 1;
    }
    return counts[dev];
}

int device_arch() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return -1;
    return major * 10 + minor;
}

#define ZB_ROW_DISPATCH(KERNEL, VPT_NEEDED, ...)                                          \
    do {                                                                                  \
        if ((VPT_NEEDED) <= 1) KERNEL<1><<<grid, kRowThreads, 0, stream>>>(__VA_ARGS__);  \
        else if ((VPT_NEEDED) <= 2) KERNEL<2><<<grid, kRowThreads, 0, stream>>>(__VA_ARGS__); \
        else if ((VPT_NEEDED) <= 4) KERNEL<4><<<grid, kRowThreads, 0, stream>>>(__VA_ARGS__); \
        else KERNEL<8><<<grid, kRowThreads, 0, stream>>>(__VA_ARGS__);                    \
    } while (0)

cudaError_t launch_rmsnorm_forward(const void* x, const float* gamma, float eps, void* n,
                                   float* rstd, int tokens, int hidden, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    const int vpt = (hidden / 8 + kRowThreads - 1) / kRowThreads;
    const int grid = tokens;
    ZB_ROW_DISPATCH(rmsnorm_fwd_kernel, vpt, static_cast<const uint16_t*>(x), gamma, eps,
                    static_cast<uint16_t*>(n), rstd, hidden);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_backward_input(const void* dn, const void* x, const float* rstd,
                                          const float* gamma, const void* dres, void* dx,
                                          int tokens, int hidden, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    const int vpt = (hidden / 8 + kRowThreads - 1) / kRowThreads;
    const int grid = tokens;
    ZB_ROW_DISPATCH(rmsnorm_bwd_kernel, vpt, static_cast<const uint16_t*>(dn),
                    static_cast<const uint16_t*>(x), rstd, gamma, static_cast<const uint16_t*>(dres),
                    static_cast<uint16_t*>(dx), hidden);
    return cudaGetLastError();
}

size_t rmsnorm_gamma_scratch_bytes(int tokens, int hidden) {
    if (tokens <= 0 || hidden <= 0) return 0;
    return static_cast<size_t>(gamma_parts(tokens, hidden)) * static_cast<size_t>(hidden) * sizeof(float);
}

cudaError_t launch_rmsnorm_backward_gamma_batch(const GammaProblem* probs, int n, int tokens, int hidden,
                                                float* scratch, cudaStream_t stream) {
    if (tokens <= 0 || n <= 0) return cudaSuccess;
    if (n > kMaxGammaProblems) return cudaErrorInvalidValue;
    GammaBatch b{};
    for (int i = 0; i < n; ++i) b.prob[i] = probs[i];
    b.tokens = tokens;
    b.hidden = hidden;
    b.parts = gamma_parts(tokens, hidden);
    const dim3 grid1((hidden + kGammaCols - 1) / kGammaCols, b.parts, n);
    dgamma_partial_kernel<<<grid1, kRowThreads, 0, stream>>>(b, scratch);
    const dim3 grid2((hidden + kFinalCols - 1) / kFinalCols, n);
    dgamma_final_kernel<<<grid2, kFinalCols * kFinalGroups, 0, stream>>>(b, scratch);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_backward_gamma(const void* dn, const void* x, const float* rstd,
                                          float* dgamma, int tokens, int hidden, float* scratch,
                                          cudaStream_t stream) {
    const GammaProblem p{dn, x, rstd, dgamma};
    return launch_rmsnorm_backward_gamma_batch(&p, 1, tokens, hidden, scratch, stream);
}

cudaError_t launch_swiglu_forward(const void* gu, void* s, int tokens, int ffn, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    const int64_t items = static_cast<int64_t>(tokens) * (ffn / 8);
    swiglu_fwd_kernel<<<grid_for(items, 256), 256, 0, stream>>>(static_cast<const uint16_t*>(gu),
                                                                static_cast<uint16_t*>(s), tokens, ffn);
    return cudaGetLastError();
}

cudaError_t launch_attention_forward(const void* qkv, void* a, int tokens, int n_heads,
                                     int n_kv_heads, int head_dim, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    const int64_t items = static_cast<int64_t>(tokens) * (n_heads * head_dim / 8);
    attn_fwd_kernel<<<grid_for(items, 256), 256, 0, stream>>>(
        static_cast<const uint16_t*>(qkv), static_cast<uint16_t*>(a), tokens, n_heads, n_kv_heads,
        head_dim);
    return cudaGetLastError();
}

cudaError_t launch_attention_backward_kv(void* dqkv, int tokens, int n_heads, int n_kv_heads,
                                         int head_dim, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    const int64_t items = static_cast<int64_t>(tokens) * (n_kv_heads * head_dim / 8);
    attn_bwd_kv_kernel<<<grid_for(items, 256), 256, 0, stream>>>(static_cast<uint16_t*>(dqkv), tokens,
                                                                 n_heads, n_kv_heads, head_dim);
    return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int limit_us, cudaStream_t stream) {
    int* st = status_word();
    if (!st) return cudaErrorInvalidDevice;
    selftest_wait_kernel<<<1, 1, 0, stream>>>(st, static_cast<uint64_t>(limit_us) * 1000ull);
    return cudaGetLastError();
}

}  // namespace zbk
