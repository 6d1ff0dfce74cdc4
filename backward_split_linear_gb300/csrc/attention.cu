// Causal softmax attention with grouped K/V heads on tcgen05 (sm_103a).
//
// The attention core between the qkv and output projections of a layer:
//   a_h = softmax(q_h k_j^T / sqrt(d), keys <= query) v_j,  j = h / (n_heads / n_kv_heads),
// over independent sequences of seq_len consecutive tokens (0: one sequence).
// The linears around it are the ones whose backward Zero-Bubble splits
// ("Zero-Bubble Pipeline Parallelism Guide for LLMs", "Core Innovation 1");
// the core has no weights, so all of its backward belongs to B.
//
// Three kernels on 128-row tiles (the forward one CTA per tile, or per two
// tiles of one kv group; dK/dV one CTA per tile; dQ persistent with one CTA
// per SM):
//   warp 0     one thread issues TMA loads
//   warp 1     allocates tensor memory; the whole warp runs the MMA issue loop
//              and its elected lane carries each tcgen05.mma and commit
//   warps 2-5  one row each: softmax / gradient arithmetic, epilogue
//   warps 6-9  (backward kernels) a second group of row warps, on the other
//              64 columns of every 128-wide step; (two-tile forward) the
//              softmax warps of the second tile
//   warp 10    (dK/dV) the statistics warp: lse and D of each step's queries
//              into the B operand of the score products' extra K step;
//              (dQ) a second MMA warp, for the dQ products
//
//   attn_causal_fwd_kernel   (head h, query block):  S = Q K^T -> online softmax ->
//                     O += P V over the key blocks up to the diagonal; writes
//                     a and the row log-sum-exp (base 2) for the backward.
//   attn_causal_fwd_pair_kernel  the same for two heads of one kv group and
//                     one query block, when the group has an even number of
//                     heads: the two tiles share every K / V load.
//   attn_causal_dkdv_kernel  (kv head j, key block): for every query head of group j
//                     and every query block from the diagonal on:
//                     S^T = K Q^T, dP^T = V dO^T, P^T = exp2(S^T c - lse),
//                     dS^T = P^T (dP^T - D); dV += P^T dO, dK += dS^T Q.
//   attn_causal_dq_kernel    tiles (head h, query block), taken from a counter:
//                     S = Q K^T, dP = dO V^T, dS as above, dQ += dS K over
//                     the key blocks up to the diagonal.
// dQ has its own kernel (it recomputes S and dP) so that no two CTAs add into
// the same output: results are the same bits on every run.  D = rowsum(dO * O)
// comes from a small row kernel first, or, inside a stage, from the epilogue of
// the output projection's dgrad that writes dO; then dK/dV (on the caller's
// stream) and dQ (on a side stream forked from it and joined back) run side by
// side.
//
// Tiles are 128 rows x d columns of bf16 in 128-byte-swizzled layout: d / 64
// blocks of 128 rows x 128 bytes (16 KiB each), as TMA writes them.  A tile
// serves as a K-major operand (contraction over d) or, through another
// descriptor, as an MN-major one (contraction over its 128 rows).  P and dS
// stay in tensor memory: each row thread packs them to bf16 over the score
// columns it has read, and the next product takes them as its A operand.
// A later score product then overwrites those columns with no wait for the
// reading product to complete. That relies on the tensor cores executing a
// CTA's MMAs in the order they were issued. The PTX ISA promises this only
// for MMAs of the same accumulator and shape, so it is an assumption about
// the hardware. The full-size parity tests cover every such reuse.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace zbk {

namespace {

constexpr int kAttnThreads = 192;
// The backward kernels run two groups of four row warps (warps 2-5 and 6-9),
// each on every other sub-block.
constexpr int kAttnBwdThreads = 320;
// The dQ kernel adds a warp that issues the dQ products (warp 10).
constexpr int kAttnDqThreads = kAttnBwdThreads + 32;
constexpr int kDqWarp = kAttnBwdThreads / 32;
constexpr int kRows = 128;             // query and key block
// Every attention CTA allocates all 512 tensor-memory columns; asking for at
// least this much shared memory keeps two CTAs off one SM (the second would
// wait in its allocation until the first ends).
constexpr size_t kMinSmem = 120 * 1024;

struct AttnParams {
    int tokens;
    int n_heads, n_kv_heads;
    int seq_len;    // 0: the whole microbatch is one sequence
    int n_blocks;   // ceil(tokens / 128)
    int ld_stat;    // floats per head row of lse / dvec
    void* out;      // forward: a [T, n_heads d]; backward: dqkv [T, (n_heads + 2 n_kv_heads) d]
    int64_t ld_out;
    float* lse;        // [n_heads][ld_stat]: log2 of the softmax denominator, in units of the scaled score
    const float* dvec;  // [n_heads][ld_stat]: rowsum(dO * O)
    float scale_log2;   // log2(e) / sqrt(d)
    float scale;        // 1 / sqrt(d)
    int* status;
};

__device__ __forceinline__ void seq_bounds(const AttnParams& p, int t0, int& s0, int& s1) {
    if (p.seq_len > 0) {
        s0 = (t0 / p.seq_len) * p.seq_len;
        s1 = min(p.tokens, s0 + p.seq_len);
    } else {
        s0 = 0;
        s1 = p.tokens;
    }
}

// K-major operand from a tile whose rows are the M (or N) index and whose
// columns are the contraction: step kk covers columns 16 kk .. 16 kk + 15.
// The descriptor of step kk is the tile's descriptor plus the step's byte
// offset / 16 in its start-address field, so callers build the base once.
__device__ __forceinline__ uint64_t kdesc_base(uint32_t tile) { return smem_desc_sw128(tile, 16, 1024); }
__device__ __forceinline__ uint64_t kdesc_at(uint64_t base, int kk) {
    return base + static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
}

// MN-major operand from the same kind of tile: the contraction runs over its
// 128 rows (step kk = rows 16 kk .. +15), the MN index over its columns.
__device__ __forceinline__ uint64_t mndesc_base(uint32_t tile) { return smem_desc_sw128(tile, 16384, 1024); }
__device__ __forceinline__ uint64_t mndesc_at(uint64_t base, int kk) {
    return base + static_cast<uint64_t>((kk * 2048) >> 4);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// v where `visible`, else +0.0: a bit mask, not a branch.  A select written as a
// short-circuit condition per element compiled to a branch per element, and
// branch resolution then dominated the elementwise passes.
__device__ __forceinline__ float keep_if(float v, bool visible) {
    return __uint_as_float(__float_as_uint(v) & (0u - static_cast<uint32_t>(visible)));
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A wait taken by every lane of a warp, with one verdict for the warp (the
// tensor-memory loads that follow are warp-wide).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* status) {
    const bool ok = mbar_wait_fast(bar, parity, status, kSiteAttn);
    return __all_sync(0xffffffffu, ok);
}

// One arrival for the whole warp, after every lane's prior work: each lane has
// waited for its tensor-memory stores and fenced them before this call.  One
// arrival per warp instead of one per thread keeps 256 shared-memory atomics
// on one barrier off the path between the row warps and the MMA thread.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// Loads one 128-row tile (d / 64 boxes) of columns col .. col + d - 1 at row r0.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar, int col, int r0) {
#pragma unroll
    for (int b = 0; b < D / 64; ++b) tma_load_2d(dst + b * 16384u, map, bar, col + 64 * b, r0);
}
// The same boxes into L2 only.
template <int D>
__device__ __forceinline__ void prefetch_tile(const CUtensorMap* map, int col, int r0) {
#pragma unroll
    for (int b = 0; b < D / 64; ++b) tma_prefetch_l2_2d(map, col + 64 * b, r0);
}

// ------------------------------------------------------------------------ forward

// P is written, as packed bf16 pairs, over the tensor-memory columns of the
// scores it came from, and O += P V takes it from there as its A operand; the
// shared memory this frees holds a third K / V stage.
template <int D>
struct FwdSmem {
    static constexpr int kStages = 3;
    static constexpr uint32_t kTile = D * 256;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kKV = kTile;  // stage s: K at kKV + 2 s kTile, V after it
    static constexpr uint32_t kBars = kKV + 2 * kStages * kTile;
    static constexpr size_t kBytes = 1024 + kBars + 16 * 8 > kMinSmem ? 1024 + kBars + 16 * 8 : kMinSmem;
};

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_causal_fwd_kernel(const __grid_constant__ CUtensorMap map_qkv, const AttnParams p) {
    using L = FwdSmem<D>;
    constexpr int NS = L::kStages;
    constexpr uint32_t kTile = L::kTile;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t s_q = base + L::kQ, s_kv = base + L::kKV;
    const uint32_t bars = base + L::kBars;
    const uint32_t q_full = bars;
    auto kv_full = [&](int s) { return bars + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return bars + 8u * (1 + NS + s); };
    auto s_full = [&](int s) { return bars + 8u * (1 + 2 * NS + s); };
    const uint32_t p_full = bars + 8u * (3 + 2 * NS), p_free = bars + 8u * (4 + 2 * NS),
                   drain = bars + 8u * (5 + 2 * NS);
    const uint32_t tmem_slot = bars + 8u * (6 + 2 * NS);
    volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_slot - raw));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qb = p.n_blocks - 1 - static_cast<int>(blockIdx.x) / p.n_heads;  // longest rows first
    const int h = static_cast<int>(blockIdx.x) % p.n_heads;
    const int g = h / (p.n_heads / p.n_kv_heads);
    const int q0 = qb * kRows;
    int s0, s1;
    seq_bounds(p, q0, s0, s1);
    const int kb0 = s0 / kRows;
    const int nk = qb - kb0 + 1;
    const int qcol = h * D, kcol = (p.n_heads + g) * D, vcol = (p.n_heads + p.n_kv_heads + g) * D;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int s = 0; s < 2; ++s) mbar_init(s_full(s), 1);
        mbar_init(p_full, 4);
        mbar_init(p_free, 1);
        mbar_init(drain, 1);
        mbar_fence_init();
        tma_prefetch_map(&map_qkv);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot_ptr;
    // columns 0-255: two score buffers (P packed into the first 64 columns of
    // its buffer once read); 256..: O
    const uint32_t t_o = tmem_base + 256;

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, kTile);
            load_tile<D>(s_q, &map_qkv, q_full, qcol, q0);
            uint32_t n_fills = 0;
            for (int j = 0; j < nk; ++j) {
                const int st = j % NS;
                if (!mbar_wait_fast(kv_empty(st), ((j / NS) & 1) ^ 1u, p.status, kSiteAttn)) break;
                mbar_arrive_expect_tx(kv_full(st), 2 * kTile);
                const int k0 = (kb0 + j) * kRows;
                load_tile<D>(s_kv + 2 * st * kTile, &map_qkv, kv_full(st), kcol, k0);
                load_tile<D>(s_kv + (2 * st + 1) * kTile, &map_qkv, kv_full(st), vcol, k0);
                ++n_fills;
            }
            mbar_wait_fast(q_full, 0, p.status, kSiteDrain);
            for (int s = 0; s < NS; ++s) {
                const uint32_t u = ring_uses(n_fills, NS, s);
                if (u > 0) mbar_wait_fast(kv_full(s), (u - 1) & 1, p.status, kSiteDrain);
            }
        }
    } else if (warp == 1) {
        // the whole warp runs the issue loop; its elected lane carries each instruction
        const uint32_t leader = elect_one_sync();
        constexpr uint32_t idesc_s = mma_idesc_bf16(128, 128, false, false);
        constexpr uint32_t idesc_o = mma_idesc_bf16(128, D, false, true);
        bool ok = warp_wait(q_full, 0, p.status);
        for (int j = 0; ok && j <= nk; ++j) {
            if (j < nk) {
                // S_j reuses the buffer of S_{j-2}, whose P feeds O += P V of
                // step j - 2: that product was issued before and runs first
                const int st = j % NS;
                if (!warp_wait(kv_full(st), (j / NS) & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t a_desc = kdesc_base(s_q), b_desc = kdesc_base(s_kv + 2 * st * kTile);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_bf16_elected(leader, tmem_base + (j & 1) * 128, kdesc_at(a_desc, kk), kdesc_at(b_desc, kk),
                                      idesc_s, kk > 0);
                umma_commit_elected(leader, s_full(j & 1));
            }
            if (j > 0) {
                const int jj = j - 1, st = jj % NS;
                if (!warp_wait(p_full, jj & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t v_desc = mndesc_base(s_kv + (2 * st + 1) * kTile);
                const uint32_t t_p = tmem_base + (jj & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk)
                    umma_bf16_ts_elected(leader, t_o, t_p + 8 * kk, mndesc_at(v_desc, kk), idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                umma_commit_elected(leader, kv_empty(st));
                umma_commit_elected(leader, p_free);
            }
        }
        umma_commit_elected(leader, drain);
        mbar_wait_fast(drain, 0, p.status, kSiteDrain);
    } else {
        // ---------------- softmax rows
        const int qw = warp & 3;
        const int row = qw * 32 + lane;
        const int q = q0 + row;
        const uint32_t t_row = static_cast<uint32_t>(qw * 32) << 16;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nk && ok; ++j) {
            const int sb = j & 1;
            if (!warp_wait(s_full(sb), (j >> 1) & 1, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[128];
            {
                uint32_t r[128];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tmem_load_32(tmem_base + t_row + sb * 128 + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
                tmem_wait_load();
#pragma unroll
                for (int e = 0; e < 128; ++e) s[e] = __uint_as_float(r[e]);
            }
            const int k0 = (kb0 + j) * kRows;
            const int lim = min(q - k0, s1 - 1 - k0);  // last visible key column of this row
            // eight running maxima and sums, not one chain of 128 dependent operations
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
            // the maximum of the raw scores (the scale is positive), the scale
            // folded into the exponent's FMA below
            if (__all_sync(0xffffffffu, lim >= 127)) {  // below the diagonal: no mask
#pragma unroll
                for (int c = 0; c < 128; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    // -inf where masked, by bit operations (no branch per element)
                    const uint32_t mk = 0u - static_cast<uint32_t>(c <= lim);
                    s[c] = __uint_as_float((__float_as_uint(s[c]) & mk) | (0xff800000u & ~mk));
                    mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * p.scale_log2;
            if (j > 0 && !warp_wait(p_free, (j - 1) & 1, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (j == 0) {
                m = mx;
            } else if (__any_sync(0xffffffffu, mx > m + 8.f)) {
                // A row's maximum rose far above its reference: the warp rescales
                // O and l of all its rows to their new maxima (the tensor-memory
                // loads and stores are warp-wide, so the decision is the warp's;
                // rescaling to any larger reference is exact).
                const float m_new = fmaxf(m, mx);
                const float alpha = ex2(m - m_new);
                l *= alpha;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_load_32(t_o + t_row + 32 * c, r);
                    tmem_wait_load();
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                    tmem_store_32(t_o + t_row + 32 * c, r);
                }
                m = m_new;
            }
            float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float a = ex2(fmaf(s[32 * c + 2 * e], p.scale_log2, -m));
                    const float b = ex2(fmaf(s[32 * c + 2 * e + 1], p.scale_log2, -m));
                    sum8[e & 7] += a + b;
                    w[e] = pack_bf16x2(a, b);
                }
                tmem_store_16(tmem_base + t_row + sb * 128 + 16 * c, w);
            }
            l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
            tmem_wait_store();
            tc_fence_before();
            warp_arrive(p_full, lane);
        }
        if (ok && warp_wait(p_free, (nk - 1) & 1, p.status)) {
            tc_fence_after();
            const float inv = 1.f / l;
            const bool valid = q < s1;
            uint16_t* dst = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(q) * p.ld_out + h * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_load_32(t_o + t_row + 32 * c, r);
                tmem_wait_load();
                if (valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        d4[k] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * k]) * inv, __uint_as_float(r[8 * k + 1]) * inv),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv));
                }
            }
            if (valid) p.lse[static_cast<int64_t>(h) * p.ld_stat + q] = m + lg2(l);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------------ backward: common

// Tensor-memory column of the packed bf16 operand of K step kk (16 rows of the
// contraction) when the two groups of row warps each pack their 64 columns of
// a 128-column buffer into its first 32: group kk / 4 at 64 (kk / 4), then 8
// columns per K step.
__device__ __forceinline__ uint32_t packed_col(int kk) { return static_cast<uint32_t>(64 * (kk >> 2) + 8 * (kk & 3)); }

// Two query heads of one kv group per CTA: the same query block and the same
// keys, tile A head h0 and tile B head h0 + 1.  Each tile has one score buffer
// and one O accumulator (the four 128-column regions of tensor memory) and a
// group of four softmax warps of its own.  The MMA order per key block j is
// PV_A[j], S_A[j+1], PV_B[j], S_B[j+1]: one group's softmax over block j runs
// while the other tile's products run.  (With one tile per CTA the four
// softmax warps held the kernel: the tensor pipe was 46 % active.)  S_X[j+1]
// reuses the columns P_X[j] was packed into, after PV_X[j] in issue order, and
// when S_X[j] completes PV_X[j-1] has too, so the softmax rescales O_X without
// a further wait.  Used when the group has an even number of heads.
template <int D>
struct FwdPairSmem {
    static constexpr int kStages = 2;
    static constexpr uint32_t kTile = D * 256;
    static constexpr uint32_t kQ = 0;           // Q of tile A, then Q of tile B
    static constexpr uint32_t kKV = 2 * kTile;  // stage s: K at kKV + 2 s kTile, V after it
    static constexpr uint32_t kBars = kKV + 2 * kStages * kTile;
    static constexpr size_t kUsed = 1024 + kBars + 16 * 8;
    static constexpr size_t kBytes = kUsed > kMinSmem ? kUsed : kMinSmem;
};

template <int D>
__global__ void __launch_bounds__(kAttnBwdThreads, 1)
    attn_causal_fwd_pair_kernel(const __grid_constant__ CUtensorMap map_qkv, const AttnParams p) {
    using L = FwdPairSmem<D>;
    constexpr int NS = L::kStages;
    constexpr uint32_t kTile = L::kTile;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t s_q = base + L::kQ, s_kv = base + L::kKV;
    const uint32_t bars = base + L::kBars;
    const uint32_t q_full = bars;
    auto kv_full = [&](int s) { return bars + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return bars + 8u * (1 + NS + s); };
    auto s_full = [&](int x) { return bars + 8u * (1 + 2 * NS + x); };
    auto p_full = [&](int x) { return bars + 8u * (3 + 2 * NS + x); };
    const uint32_t done = bars + 8u * (5 + 2 * NS), drain = bars + 8u * (6 + 2 * NS);
    const uint32_t tmem_slot = bars + 8u * (7 + 2 * NS);
    volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_slot - raw));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pairs = p.n_heads / 2;
    const int qb = p.n_blocks - 1 - static_cast<int>(blockIdx.x) / pairs;  // longest rows first
    const int h0 = 2 * (static_cast<int>(blockIdx.x) % pairs);
    const int g = h0 / (p.n_heads / p.n_kv_heads);
    const int q0 = qb * kRows;
    int s0, s1;
    seq_bounds(p, q0, s0, s1);
    const int kb0 = s0 / kRows;
    const int nk = qb - kb0 + 1;
    const int kcol = (p.n_heads + g) * D, vcol = (p.n_heads + p.n_kv_heads + g) * D;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(p_full(x), 4);
        }
        mbar_init(done, 1);
        mbar_init(drain, 1);
        mbar_fence_init();
        tma_prefetch_map(&map_qkv);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot_ptr;
    // columns: S_A 0-127, S_B 128-255 (P packed into the first 64 columns of its
    // buffer once read), O_A 256.., O_B 384..
    auto t_s = [&](int x) { return tmem_base + 128u * static_cast<uint32_t>(x); };
    auto t_o = [&](int x) { return tmem_base + 256u + 128u * static_cast<uint32_t>(x); };

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2 * kTile);
            load_tile<D>(s_q, &map_qkv, q_full, h0 * D, q0);
            load_tile<D>(s_q + kTile, &map_qkv, q_full, (h0 + 1) * D, q0);
            uint32_t n_fills = 0;
            for (int j = 0; j < nk; ++j) {
                const int st = j % NS;
                if (!mbar_wait_fast(kv_empty(st), ((j / NS) & 1) ^ 1u, p.status, kSiteAttn)) break;
                mbar_arrive_expect_tx(kv_full(st), 2 * kTile);
                const int k0 = (kb0 + j) * kRows;
                load_tile<D>(s_kv + 2 * st * kTile, &map_qkv, kv_full(st), kcol, k0);
                load_tile<D>(s_kv + (2 * st + 1) * kTile, &map_qkv, kv_full(st), vcol, k0);
                ++n_fills;
            }
            mbar_wait_fast(q_full, 0, p.status, kSiteDrain);
            for (int s = 0; s < NS; ++s) {
                const uint32_t u = ring_uses(n_fills, NS, s);
                if (u > 0) mbar_wait_fast(kv_full(s), (u - 1) & 1, p.status, kSiteDrain);
            }
        }
    } else if (warp == 1) {
        // the whole warp runs the issue loop; its elected lane carries each instruction
        const uint32_t leader = elect_one_sync();
        constexpr uint32_t idesc_s = mma_idesc_bf16(128, 128, false, false);
        constexpr uint32_t idesc_o = mma_idesc_bf16(128, D, false, true);
        auto issue_s = [&](int x, int j) {
            const int st = j % NS;
            const uint64_t a_desc = kdesc_base(s_q + static_cast<uint32_t>(x) * kTile),
                           b_desc = kdesc_base(s_kv + 2 * st * kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_bf16_elected(leader, t_s(x), kdesc_at(a_desc, kk), kdesc_at(b_desc, kk), idesc_s, kk > 0);
            umma_commit_elected(leader, s_full(x));
        };
        auto issue_pv = [&](int x, int j) {
            if (!warp_wait(p_full(x), j & 1, p.status)) return false;
            tc_fence_after();
            const uint64_t v_desc = mndesc_base(s_kv + (2 * (j % NS) + 1) * kTile);
#pragma unroll
            for (int kk = 0; kk < kRows / 16; ++kk)
                umma_bf16_ts_elected(leader, t_o(x), t_s(x) + 8 * kk, mndesc_at(v_desc, kk), idesc_o,
                                     (j > 0 || kk > 0) ? 1u : 0u);
            return true;
        };
        auto kv_ready = [&](int j) {
            if (!warp_wait(kv_full(j % NS), (j / NS) & 1, p.status)) return false;
            tc_fence_after();
            return true;
        };
        bool ok = warp_wait(q_full, 0, p.status) && kv_ready(0);
        if (ok) {
            issue_s(0, 0);
            issue_s(1, 0);
        }
        for (int j = 0; ok && j < nk; ++j) {
            const bool more = j + 1 < nk;
            if (!issue_pv(0, j) || (more && !kv_ready(j + 1))) break;
            if (more) issue_s(0, j + 1);
            if (!issue_pv(1, j)) break;
            umma_commit_elected(leader, kv_empty(j % NS));
            if (more) issue_s(1, j + 1);
        }
        umma_commit_elected(leader, done);
        umma_commit_elected(leader, drain);
        mbar_wait_fast(drain, 0, p.status, kSiteDrain);
    } else {
        // ---------------- softmax rows: warps 2-5 tile A, warps 6-9 tile B
        const int x = (warp - 2) >> 2;
        const int h = h0 + x;
        const int qw = warp & 3;
        const int row = qw * 32 + lane;
        const int q = q0 + row;
        const uint32_t t_row = static_cast<uint32_t>(qw * 32) << 16;
        const uint32_t ts = t_s(x), to = t_o(x);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nk && ok; ++j) {
            if (!warp_wait(s_full(x), j & 1, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[128];
            {
                uint32_t r[128];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tmem_load_32(ts + t_row + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
                tmem_wait_load();
#pragma unroll
                for (int e = 0; e < 128; ++e) s[e] = __uint_as_float(r[e]);
            }
            const int k0 = (kb0 + j) * kRows;
            const int lim = min(q - k0, s1 - 1 - k0);  // last visible key column of this row
            // eight running maxima and sums, not one chain of 128 dependent operations
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
            // the maximum of the raw scores (the scale is positive), the scale
            // folded into the exponent's FMA below
            if (__all_sync(0xffffffffu, lim >= 127)) {  // below the diagonal: no mask
#pragma unroll
                for (int c = 0; c < 128; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    // -inf where masked, by bit operations (no branch per element)
                    const uint32_t mk = 0u - static_cast<uint32_t>(c <= lim);
                    s[c] = __uint_as_float((__float_as_uint(s[c]) & mk) | (0xff800000u & ~mk));
                    mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * p.scale_log2;
            if (j == 0) {
                m = mx;
            } else if (__any_sync(0xffffffffu, mx > m + 8.f)) {
                // A row's maximum rose far above its reference: the warp rescales
                // O and l of all its rows to their new maxima (warp-wide
                // tensor-memory loads and stores; rescaling to any larger
                // reference is exact).  PV_X[j-1] completed before S_X[j].
                const float m_new = fmaxf(m, mx);
                const float alpha = ex2(m - m_new);
                l *= alpha;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_load_32(to + t_row + 32 * c, r);
                    tmem_wait_load();
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                    tmem_store_32(to + t_row + 32 * c, r);
                }
                m = m_new;
            }
            float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float a = ex2(fmaf(s[32 * c + 2 * e], p.scale_log2, -m));
                    const float b = ex2(fmaf(s[32 * c + 2 * e + 1], p.scale_log2, -m));
                    sum8[e & 7] += a + b;
                    w[e] = pack_bf16x2(a, b);
                }
                tmem_store_16(ts + t_row + 16 * c, w);
            }
            l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
            tmem_wait_store();
            tc_fence_before();
            warp_arrive(p_full(x), lane);
        }
        if (ok && warp_wait(done, 0, p.status)) {
            tc_fence_after();
            const float inv = 1.f / l;
            const bool valid = q < s1;
            uint16_t* dst = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(q) * p.ld_out + h * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_load_32(to + t_row + 32 * c, r);
                tmem_wait_load();
                if (valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        d4[k] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * k]) * inv, __uint_as_float(r[8 * k + 1]) * inv),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv),
                                           pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv));
                }
            }
            if (valid) p.lse[static_cast<int64_t>(h) * p.ld_stat + q] = m + lg2(l);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------------ backward: dq

// A persistent kernel, one CTA per SM.  Each CTA takes (query head, query
// block) tiles from a counter in global memory, longest rows first, and walks
// a tile's key blocks up to the diagonal, 128 keys a step.  Per step the
// tensor cores run S = Q K^T, dP = dO V^T (both 128 x 128, K-major operands)
// and dQ += dS K (A = dS from tensor memory, B = K as an MN-major operand).
// S has two tensor-memory buffers, dP one: the MMA order is S[j+1], dP[j+1],
// dQ[j], so the row warps' pass over step j (P = exp2(S c - lse) into
// registers as soon as S lands, then dS = P (dP - D), packed over the S
// columns just read) overlaps the products of its neighbours.  Two groups of
// four row warps take 64 key columns each.  K streams through three stages,
// V through two, on one barrier per step.
//
// Two warps issue the MMAs: warp 1 the S and dP products, warp 10 the dQ
// products.  With one issuing warp, the waits and commits between batches of
// 128 x 128 products left the tensor pipe idle for about a quarter of each
// step (a timed copy that observed every batch's completion); with two, one
// warp's waits run while the other's products execute.  The warps order their
// products through two barriers: S[j+2] reuses the buffer that dQ[j] reads,
// so warp 1 issues it after warp 10 has issued dQ[j]; and warp 10 issues
// dQ[j] after warp 1 has issued dP[j+1], which the row warps wait for.
//
// The steps of a CTA's tiles form one sequence: the rings, the S buffers and
// the barriers' phases run on from one tile to the next.  The next tile's Q
// and dO load as soon as the last S and dP products of the current one are
// done, and its first products run while the row warps store the finished
// tile's dQ.  (With one CTA per tile, an SM sat idle for about 4.6 us between
// one CTA's exit and the next one's start, and again while Q and dO loaded:
// with about 7 tiles per SM, a fifth of the kernel.)  A tile goes to whichever
// CTA asks next, so CTAs that start late, on SMs held by the dK/dV kernel's
// longest CTAs, take fewer; a CTA asks when it issues its current tile's last
// K / V load, and pulls the new tile's Q and dO into L2 at once.  Each tile is
// computed by one CTA in one order: the results do not depend on which CTA
// took it.
template <int D>
struct DqSmem {
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr uint32_t kTile = D * 256;
    static constexpr uint32_t kQ = 0, kDO = kTile, kK = 2 * kTile;
    static constexpr uint32_t kV = kK + kKStages * kTile;
    static constexpr uint32_t kBars = kV + kVStages * kTile;
    // q full / empty, the K ring (full, empty), the V ring (empty), S (2), dP,
    // dS (2), done, drain, the two tile slots (full, empty), dQ issued (2)
    static constexpr int kNumBars = 2 + 2 * kKStages + kVStages + 2 + 5 + 4 + 4;
    static constexpr uint32_t kTmemSlot = kBars + 8 * kNumBars;
    static constexpr uint32_t kTileSlot = kTmemSlot + 8;  // the tile number held by each slot (two ints)
    static constexpr size_t kUsed = kTileSlot + 8 + 16;
    static constexpr size_t kBytes = kUsed > kMinSmem ? kUsed : kMinSmem;
};

// Tile t of the dQ kernel: query block n_blocks - 1 - t / n_heads (the
// longest rows first), head t % n_heads; its key blocks run from the first
// of the query block's sequence up to the diagonal.
struct DqTile {
    int h, q0, s1, kb0, nk;
};
__device__ __forceinline__ DqTile dq_tile(const AttnParams& p, int t) {
    DqTile d;
    const int qb = p.n_blocks - 1 - t / p.n_heads;
    d.h = t % p.n_heads;
    d.q0 = qb * kRows;
    int s0;
    seq_bounds(p, d.q0, s0, d.s1);
    d.kb0 = s0 / kRows;
    d.nk = qb - d.kb0 + 1;
    return d;
}

template <int D>
__global__ void __launch_bounds__(kAttnDqThreads, 1)
    attn_causal_dq_kernel(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_do,
                          const AttnParams p, int* tile_counter) {
    using L = DqSmem<D>;
    constexpr int NK = L::kKStages, NV = L::kVStages;
    constexpr uint32_t kTile = L::kTile;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_addr(smem_raw);
    if (base & 1023u) {  // the tiles' 128-byte swizzle needs a 1 KiB-aligned start
        if (threadIdx.x == 0) atomicCAS(p.status, 0, kSiteAttn);
        return;
    }
    const uint32_t s_q = base + L::kQ, s_do = base + L::kDO, s_k = base + L::kK, s_v = base + L::kV;
    const uint32_t bars = base + L::kBars;
    const uint32_t q_full = bars, q_empty = bars + 8u;
    auto k_full = [&](uint32_t s) { return bars + 8u * (2 + s); };
    auto k_empty = [&](uint32_t s) { return bars + 8u * (2 + NK + s); };
    auto v_empty = [&](uint32_t s) { return bars + 8u * (2 + 2 * NK + s); };
    constexpr int kB = 2 + 2 * NK + NV;
    auto s_full = [&](uint32_t b) { return bars + 8u * (kB + b); };
    const uint32_t dp_full = bars + 8u * (kB + 2), done = bars + 8u * (kB + 3), drain = bars + 8u * (kB + 4);
    auto ds_full = [&](uint32_t g) { return bars + 8u * (kB + 5 + (g & 1u)); };
    auto tile_full = [&](uint32_t s) { return bars + 8u * (kB + 7 + s); };
    auto tile_empty = [&](uint32_t s) { return bars + 8u * (kB + 9 + s); };
    auto dq_issued = [&](uint32_t g) { return bars + 8u * (kB + 11 + (g & 1u)); };
    auto dp_issued = [&](uint32_t g) { return bars + 8u * (kB + 13 + (g & 1u)); };
    const uint32_t tmem_slot = base + L::kTmemSlot;
    volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(smem_raw + L::kTmemSlot);
    volatile int* tile_slot = reinterpret_cast<volatile int*>(smem_raw + L::kTileSlot);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = p.n_blocks * p.n_heads;
    const int group = p.n_heads / p.n_kv_heads;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < NK; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < NV; ++s) mbar_init(v_empty(s), 1);
        mbar_init(s_full(0), 1);
        mbar_init(s_full(1), 1);
        mbar_init(dp_full, 1);
        mbar_init(done, 1);
        mbar_init(drain, 2);  // both MMA warps
        for (int s = 0; s < 2; ++s) {
            mbar_init(ds_full(s), 8);
            mbar_init(tile_full(s), 1);
            mbar_init(tile_empty(s), 10);  // the two MMA warps and the eight row warps
            mbar_init(dq_issued(s), 1);
            mbar_init(dp_issued(s), 1);
        }
        mbar_fence_init();
        tma_prefetch_map(&map_qkv);
        tma_prefetch_map(&map_do);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot_ptr;
    // columns: S buffers 0-127 and 128-255 (dS packed into columns 0-31 and
    // 64-95 of a buffer once read), dP 256-383, dQ 384..
    const uint32_t t_dp = tmem_base + 256, t_dq = tmem_base + 384;
    auto t_s = [&](uint32_t g) { return tmem_base + 128u * (g & 1u); };
    // A consumer warp's view of tile slot n & 1: the tile number (-1: none left),
    // after which the warp releases the slot.
    auto take_tile = [&](uint32_t n, int& t) {
        if (!warp_wait(tile_full(n & 1u), (n >> 1) & 1u, p.status)) return false;
        t = tile_slot[n & 1u];
        __syncwarp();
        if (lane == 0) mbar_arrive(tile_empty(n & 1u));
        return true;
    };

    if (warp == 0) {
        if (lane == 0) {
            // Fills slot n & 1 with the number of this CTA's tile n once every
            // consumer has read the slot's previous tile; -1 when none is left,
            // -2 when the wait failed.
            auto fetch = [&](uint32_t n) {
                if (!mbar_wait_fast(tile_empty(n & 1u), ((n >> 1) & 1u) ^ 1u, p.status, kSiteAttn)) return -2;
                int t = atomicAdd(tile_counter, 1);
                if (t >= n_tiles) t = -1;
                tile_slot[n & 1u] = t;
                mbar_arrive(tile_full(n & 1u));
                return t;
            };
            uint32_t nq = 0, nkf = 0;  // Q / dO loads and K / V steps issued
            int t = fetch(0);
            for (uint32_t n = 0; t >= 0; ++n) {
                const DqTile tl = dq_tile(p, t);
                // Q and dO once the previous tile's S and dP products are done
                if (!mbar_wait_fast(q_empty, (n & 1u) ^ 1u, p.status, kSiteAttn)) break;
                mbar_arrive_expect_tx(q_full, 2 * kTile);
                load_tile<D>(s_q, &map_qkv, q_full, tl.h * D, tl.q0);
                load_tile<D>(s_do, &map_do, q_full, tl.h * D, tl.q0);
                ++nq;
                const int g = tl.h / group;
                const int kcol = (p.n_heads + g) * D, vcol = (p.n_heads + p.n_kv_heads + g) * D;
                int t_next = -2;
                for (int j = 0; j < tl.nk; ++j) {
                    const uint32_t u = nkf;
                    // K[j] and V[j] land on one barrier: one wait per step for the MMA warp
                    if (!mbar_wait_fast(k_empty(u % NK), ((u / NK) & 1u) ^ 1u, p.status, kSiteAttn)) break;
                    if (!mbar_wait_fast(v_empty(u % NV), ((u / NV) & 1u) ^ 1u, p.status, kSiteAttn)) break;
                    mbar_arrive_expect_tx(k_full(u % NK), 2 * kTile);
                    load_tile<D>(s_k + (u % NK) * kTile, &map_qkv, k_full(u % NK), kcol, (tl.kb0 + j) * kRows);
                    load_tile<D>(s_v + (u % NV) * kTile, &map_qkv, k_full(u % NK), vcol, (tl.kb0 + j) * kRows);
                    ++nkf;
                    // The next tile's number at this tile's last load, two or three steps
                    // before its end (taken earlier, the CTAs that start first took more
                    // than their share of the long tiles), and its Q and dO into L2.
                    if (j == tl.nk - 1) {
                        t_next = fetch(n + 1);
                        if (t_next >= 0) {
                            const DqTile nx = dq_tile(p, t_next);
                            prefetch_tile<D>(&map_qkv, nx.h * D, nx.q0);
                            prefetch_tile<D>(&map_do, nx.h * D, nx.q0);
                        }
                    }
                }
                t = t_next;  // -2 after a failed wait ends the loop
            }
            // no copy may land after the CTA has gone
            if (nq > 0) mbar_wait_fast(q_full, (nq - 1) & 1u, p.status, kSiteDrain);
            for (int s = 0; s < NK; ++s) {
                const uint32_t u = ring_uses(nkf, NK, s);
                if (u > 0) mbar_wait_fast(k_full(s), (u - 1) & 1u, p.status, kSiteDrain);
            }
        }
    } else if (warp == 1) {
        // ---------------- S and dP products.  The whole warp runs the issue loop;
        // its elected lane carries each instruction.
        const uint32_t leader = elect_one_sync();
        constexpr uint32_t idesc_s = mma_idesc_bf16(128, 128, false, false);
        const uint64_t q_desc = kdesc_base(s_q), do_desc = kdesc_base(s_do);
        auto issue_s = [&](uint32_t g) {
            const uint32_t st = g % NK;
            if (!warp_wait(k_full(st), (g / NK) & 1u, p.status)) return false;
            tc_fence_after();
            const uint64_t k_desc = kdesc_base(s_k + st * kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_bf16_elected(leader, t_s(g), kdesc_at(q_desc, kk), kdesc_at(k_desc, kk), idesc_s, kk > 0);
            umma_commit_elected(leader, s_full(g & 1u));
            return true;
        };
        auto issue_dp = [&](uint32_t g) {
            const uint32_t st = g % NV;  // V[g] landed with K[g] (issue_s(g) waited for both)
            const uint64_t v_desc = kdesc_base(s_v + st * kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_bf16_elected(leader, t_dp, kdesc_at(do_desc, kk), kdesc_at(v_desc, kk), idesc_s, kk > 0);
            umma_commit_elected(leader, dp_full);
            umma_commit_elected(leader, v_empty(st));
        };
        // S[g] overwrites the S buffer of step g - 2 once the dQ warp has issued
        // dQ[g - 2], which reads dS[g - 2] from it; dP[g] overwrites dP[g - 1]
        // once the row warps are done with it.
        auto may_issue_s = [&](uint32_t g) {
            if (g < 2) return true;
            if (!warp_wait(dq_issued(g - 2), ((g - 2) >> 1) & 1u, p.status)) return false;
            tc_fence_after();
            return true;
        };
        auto may_issue_dp = [&](uint32_t g) {
            if (g < 1) return true;
            if (!warp_wait(ds_full(g - 1), ((g - 1) >> 1) & 1u, p.status)) return false;
            tc_fence_after();
            return true;
        };
        uint32_t g = 0;  // steps of this CTA so far, over all its tiles
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
            int t;
            if (!take_tile(n, t) || t < 0) break;
            const int nk = dq_tile(p, t).nk;
            if (!warp_wait(q_full, n & 1u, p.status)) break;
            tc_fence_after();
            // the MMA order per step is S[g+1], dP[g+1] (here) beside dQ[g] (the dQ warp)
            for (int j = 0; j < nk; ++j, ++g) {
                if (!may_issue_s(g) || !issue_s(g) || !may_issue_dp(g)) {
                    ok = false;
                    break;
                }
                issue_dp(g);
                tc_fence_before();
                if (leader) mbar_arrive(dp_issued(g));
                // Q and dO are free for the next tile once its last S and dP are done
                if (j + 1 == nk) umma_commit_elected(leader, q_empty);
            }
        }
        umma_commit_elected(leader, drain);
        mbar_wait_fast(drain, 0, p.status, kSiteDrain);
    } else if (warp == kDqWarp) {
        // ---------------- dQ products: dQ[g] += dS[g] K[g] as soon as the row warps
        // have packed dS[g]; then the K stage goes back to the producer and the S
        // warp may overwrite the buffer.
        const uint32_t leader = elect_one_sync();
        constexpr uint32_t idesc_q = mma_idesc_bf16(128, D, false, true);
        uint32_t g = 0;
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
            int t;
            if (!take_tile(n, t) || t < 0) break;
            const int nk = dq_tile(p, t).nk;
            for (int j = 0; j < nk; ++j, ++g) {
                if (!warp_wait(ds_full(g), (g >> 1) & 1u, p.status) ||
                    (j + 1 < nk && !warp_wait(dp_issued(g + 1), ((g + 1) >> 1) & 1u, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t k_mn = mndesc_base(s_k + (g % NK) * kTile);
#pragma unroll
                for (int kk = 0; kk < kRows / 16; ++kk)
                    umma_bf16_ts_elected(leader, t_dq, t_s(g) + packed_col(kk), mndesc_at(k_mn, kk), idesc_q,
                                         (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit_elected(leader, k_empty(g % NK));
                tc_fence_before();
                if (leader) mbar_arrive(dq_issued(g));
            }
            if (ok) umma_commit_elected(leader, done);
        }
        umma_commit_elected(leader, drain);
        mbar_wait_fast(drain, 0, p.status, kSiteDrain);
    } else {
        // ---------------- two groups of four warps, one query row per thread in each:
        // group gi takes key columns 64 gi .. 64 gi + 63 of every step
        const int gi = (warp - 2) >> 2;
        const int qw = warp & 3;
        const int row = qw * 32 + lane;
        const uint32_t t_row = (static_cast<uint32_t>(qw * 32) << 16) + 64u * gi;
        uint32_t g = 0;
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
            int t;
            if (!take_tile(n, t) || t < 0) break;
            const DqTile tl = dq_tile(p, t);
            const int q = tl.q0 + row;
            const bool valid = q < tl.s1;
            const float lse = valid ? p.lse[static_cast<int64_t>(tl.h) * p.ld_stat + q] : 0.f;
            const float dv = valid ? p.dvec[static_cast<int64_t>(tl.h) * p.ld_stat + q] : 0.f;
            for (int j = 0; j < tl.nk; ++j, ++g) {
                const int c0 = (tl.kb0 + j) * kRows + 64 * gi;
                const int lim = valid ? min(q - c0, tl.s1 - 1 - c0) : -1;  // last visible key column of this row
                if (!warp_wait(s_full(g & 1u), (g >> 1) & 1u, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float pr[64];
                uint32_t rs[64];
                tmem_load_32(t_s(g) + t_row, *reinterpret_cast<uint32_t(*)[32]>(rs));
                tmem_load_32(t_s(g) + t_row + 32, *reinterpret_cast<uint32_t(*)[32]>(rs + 32));
                tmem_wait_load();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (__all_sync(0xffffffffu, lim >= 32 * c + 31)) {  // every column visible: no mask
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pr[32 * c + i] = ex2(fmaf(__uint_as_float(rs[32 * c + i]), p.scale_log2, -lse));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pr[32 * c + i] =
                                keep_if(ex2(fmaf(__uint_as_float(rs[32 * c + i]), p.scale_log2, -lse)), 32 * c + i <= lim);
                    }
                }
                if (!warp_wait(dp_full, g & 1u, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t rp[64];
                tmem_load_32(t_dp + t_row, *reinterpret_cast<uint32_t(*)[32]>(rp));
                tmem_load_32(t_dp + t_row + 32, *reinterpret_cast<uint32_t(*)[32]>(rp + 32));
                tmem_wait_load();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack_bf16x2(pr[32 * c + 2 * e] * (__uint_as_float(rp[32 * c + 2 * e]) - dv),
                                           pr[32 * c + 2 * e + 1] * (__uint_as_float(rp[32 * c + 2 * e + 1]) - dv));
                    // packed columns 16 c .. 16 c + 15 of the group's S columns, all read above
                    tmem_store_16(t_s(g) + t_row + 16 * c, w);
                }
                tmem_wait_store();
                tc_fence_before();
                warp_arrive(ds_full(g), lane);
            }
            if (!ok || !warp_wait(done, n & 1u, p.status)) break;
            // group gi stores dQ columns [D/2 gi, D/2 (gi + 1)); the tile's next
            // dQ product waits for this group's next dS arrival, after these loads
            tc_fence_after();
            uint16_t* dst = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(q) * p.ld_out + tl.h * D;
            const uint32_t t_q = t_dq + (static_cast<uint32_t>(qw * 32) << 16) + 32u * (gi * (D / 64));
            constexpr int kChunks = D / 64;  // 32-column chunks of this group's half
            uint32_t r[kChunks][32];
#pragma unroll
            for (int c = 0; c < kChunks; ++c) tmem_load_32(t_q + 32 * c, r[c]);
            tmem_wait_load();
            tc_fence_before();
            if (valid) {
                const float sc = p.scale;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * (gi * kChunks + c));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        d4[k] = make_uint4(
                            pack_bf16x2(__uint_as_float(r[c][8 * k]) * sc, __uint_as_float(r[c][8 * k + 1]) * sc),
                            pack_bf16x2(__uint_as_float(r[c][8 * k + 2]) * sc, __uint_as_float(r[c][8 * k + 3]) * sc),
                            pack_bf16x2(__uint_as_float(r[c][8 * k + 4]) * sc, __uint_as_float(r[c][8 * k + 5]) * sc),
                            pack_bf16x2(__uint_as_float(r[c][8 * k + 6]) * sc, __uint_as_float(r[c][8 * k + 7]) * sc));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------------ backward: dk, dv

// One CTA per (kv head, key block) walks every query head of the group and
// every query block from the diagonal on, 128 queries a step.  Per step the
// tensor cores run S^T = K Q^T and dP^T = V dO^T (128 x 128, K-major
// operands), then dV += P^T dO and dK += dS^T Q (A = P^T / dS^T from tensor
// memory, B = dO / Q as MN-major operands).  The MMA order is dV[i],
// S^T[i+1], dK[i], dP^T[i+1]: the row warps turn S^T[i] into P^T while
// dK[i-1] and dP^T[i] run, and dP^T[i] into dS^T while dV[i] and S^T[i+1]
// run, so single S^T and dP^T buffers keep the tensor pipe fed and leave room
// for the dV and dK accumulators in the 512 tensor-memory columns.  Two groups
// of four row warps take 64 query columns each; P stays in registers between
// the two passes.
//
// The per-query statistics enter through the tensor cores, not the row warps:
// each score product gets one more K step whose A operand holds ones and
// whose B operand holds, per query, -lse / c (for S^T) or -D (for dP^T) as
// the sum of three bf16 parts, so the accumulators come out as S^T - lse / c
// and dP^T - D.  Every row thread would otherwise read all 64 statistics of
// its columns from shared memory each pass, and those broadcast reads took
// about a quarter of the shared-memory bandwidth that the score products'
// operands need.  A statistics warp turns each step's lse and D (landed by
// TMA) into that B operand.  The three-part split leaves an error of about
// 2^-27 of lse / c, far below the bf16 rounding of P.
template <int D>
struct DkvSmem {
    static constexpr int kQStages = 2, kDoStages = 2, kStatStages = 2, kAugStages = 2;
    static constexpr uint32_t kTile = D * 256;
    static constexpr uint32_t kAugTile = 128 * 16 * 2;  // 128 rows x one K step of 16 bf16, no swizzle
    static constexpr uint32_t kK = 0, kV = kTile, kQ = 2 * kTile;
    static constexpr uint32_t kDO = kQ + kQStages * kTile;
    static constexpr uint32_t kOnes = kDO + kDoStages * kTile;  // two constant A operands: lse, D selectors
    static constexpr uint32_t kAug = kOnes + 2 * kAugTile;      // stage s: the B operand of step s
    static constexpr uint32_t kStat = kAug + kAugStages * kAugTile;  // stage s: lse (512 bytes) then D (512 bytes)
    static constexpr uint32_t kBars = kStat + 1024 * kStatStages;
    // kv full; Q (with dO and statistics) full / empty; statistics full / empty;
    // statistics operand empty; S^T, dP^T, P^T and dS^T chunks, done, drain
    static constexpr int kNumBars = 1 + 2 * (kQStages + kStatStages) + kAugStages + 8;
    static constexpr size_t kBytes = kBars + 8 * kNumBars + 16;
};
constexpr int kAttnDkvThreads = kAttnBwdThreads + 32;  // + the statistics warp
constexpr int kStatWarp = kAttnBwdThreads / 32;

// Byte offset of row r, K chunk kc (8 bf16) of a no-swizzle K-major operand of
// one K step: 8-row groups 256 bytes apart (the stride-dimension offset), the
// two 8-column chunks of a row group 128 bytes apart (the leading-dimension
// offset), rows of a chunk 16 bytes apart.
__device__ __forceinline__ uint32_t aug_offset(int r, int kc) {
    return static_cast<uint32_t>((r >> 3) * 256 + kc * 128 + (r & 7) * 16);
}
__device__ __forceinline__ uint64_t aug_desc(uint32_t tile) {
    return static_cast<uint64_t>((tile & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(256 >> 4) << 32) | (1ull << 46);  // swizzle mode 0: none
}

// v as hi + mid + lo, each bf16 (round to nearest), as the low 48 bits of a
// 64-bit word (bf16 columns 0, 1, 2; column 3 zero).
__device__ __forceinline__ uint2 split3_bf16(float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    return make_uint2(static_cast<uint32_t>(__bfloat16_as_ushort(hi)) | (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16),
                      static_cast<uint32_t>(__bfloat16_as_ushort(lo)));
}

template <int D>
__global__ void __launch_bounds__(kAttnDkvThreads, 1)
    attn_causal_dkdv_kernel(const __grid_constant__ CUtensorMap map_qkv, const __grid_constant__ CUtensorMap map_do,
                            const AttnParams p) {
    using L = DkvSmem<D>;
    constexpr int NQ = L::kQStages, ND = L::kDoStages, NT = L::kStatStages, NA = L::kAugStages;
    constexpr uint32_t kTile = L::kTile;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_addr(smem_raw);
    if (base & 1023u) {  // the tiles' 128-byte swizzle needs a 1 KiB-aligned start
        if (threadIdx.x == 0) atomicCAS(p.status, 0, kSiteAttn);
        return;
    }
    const uint32_t s_k = base + L::kK, s_v = base + L::kV, s_q = base + L::kQ, s_do = base + L::kDO,
                   s_ones = base + L::kOnes, s_aug = base + L::kAug, s_stat = base + L::kStat;
    const uint32_t bars = base + L::kBars;
    const uint32_t kv_full = bars;
    auto q_full = [&](int s) { return bars + 8u * (1 + s); };
    // q_empty(s) releases Q, dO (same ring position, ND == NQ) and nothing else
    auto q_empty = [&](int s) { return bars + 8u * (1 + NQ + s); };
    auto st_full = [&](int s) { return bars + 8u * (1 + 2 * NQ + s); };
    auto st_empty = [&](int s) { return bars + 8u * (1 + 2 * NQ + NT + s); };
    auto aug_empty = [&](int s) { return bars + 8u * (1 + 2 * NQ + 2 * NT + s); };
    constexpr int kB = 1 + 2 * (NQ + NT) + NA;
    static_assert(NQ == ND, "Q and dO share their ring position and release");
    // p_full(c) / ds_full(c): chunk c (32 query columns of each group) of P^T / dS^T is packed
    auto p_full = [&](int c) { return bars + 8u * (kB + 2 + c); };
    auto ds_full = [&](int c) { return bars + 8u * (kB + 4 + c); };
    const uint32_t s_full = bars + 8u * kB, dp_full = bars + 8u * (kB + 1), done = bars + 8u * (kB + 6),
                   drain = bars + 8u * (kB + 7);
    const uint32_t tmem_slot = bars + 8u * L::kNumBars;
    volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_slot - base));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = p.n_heads / p.n_kv_heads;
    const int kb = static_cast<int>(blockIdx.x) / p.n_kv_heads;  // earliest keys (most work) first
    const int g = static_cast<int>(blockIdx.x) % p.n_kv_heads;
    const int k0 = kb * kRows;
    int s0, s1;
    seq_bounds(p, k0, s0, s1);
    const int qb_last = (s1 - 1) / kRows;
    const int n_steps = group * (qb_last - kb + 1);  // (query block, head of the group) pairs
    const int kcol = (p.n_heads + g) * D, vcol = (p.n_heads + p.n_kv_heads + g) * D;

    // The constant A operands of the statistics step (ones in bf16 columns 0-2
    // for lse, 8-10 for D) and zeros in the B operands' unused columns; the
    // statistics warp rewrites only columns 0-2 and 8-10 of a B operand.
    {
        uint4* z = reinterpret_cast<uint4*>(smem_raw + L::kOnes);
        constexpr int n16 = (2 + NA) * L::kAugTile / 16;
        for (int e = threadIdx.x; e < n16; e += kAttnDkvThreads) {
            const int tile = e / (L::kAugTile / 16);
            const int kc = (e >> 3) & 1;  // 16-byte rows: 8 rows per chunk, chunks alternate every 128 bytes
            const bool ones = tile < 2 && kc == tile;
            z[e] = ones ? make_uint4(0x3F803F80u, 0x3F80u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < NQ; ++s) {
            mbar_init(q_full(s), 2);  // the Q and dO tiles' TMA and the statistics warp's B operand
            mbar_init(q_empty(s), 1);
        }
        for (int s = 0; s < NT; ++s) {
            mbar_init(st_full(s), 1);
            mbar_init(st_empty(s), 1);
        }
        for (int s = 0; s < NA; ++s) mbar_init(aug_empty(s), 1);
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        for (int c = 0; c < 2; ++c) {
            mbar_init(p_full(c), 8);
            mbar_init(ds_full(c), 8);
        }
        mbar_init(done, 1);
        mbar_init(drain, 1);
        mbar_fence_init();
        tma_prefetch_map(&map_qkv);
        tma_prefetch_map(&map_do);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot_ptr;
    // columns: S^T 0-127 (P^T packed into 0-31 and 64-95 once read), dP^T
    // 128-255 (dS^T likewise), dV 256.., dK 256 + D..
    const uint32_t t_s = tmem_base, t_dp = tmem_base + 128, t_dv = tmem_base + 256, t_dk = tmem_base + 256 + D;

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(kv_full, 2 * kTile);
            load_tile<D>(s_k, &map_qkv, kv_full, kcol, k0);
            load_tile<D>(s_v, &map_qkv, kv_full, vcol, k0);
            uint32_t nq = 0, nt = 0;
            for (int i = 0; i < n_steps; ++i) {
                const int qb = kb + i / group;
                const int h = g * group + i % group;
                const int r0 = qb * kRows;
                if (!mbar_wait_fast(st_empty(i % NT), ((i / NT) & 1) ^ 1u, p.status, kSiteAttn)) break;
                const uint32_t stat = s_stat + 1024u * (i % NT);
                mbar_arrive_expect_tx(st_full(i % NT), 1024);
                bulk_load_1d(stat, p.lse + static_cast<int64_t>(h) * p.ld_stat + r0, 512, st_full(i % NT));
                bulk_load_1d(stat + 512, p.dvec + static_cast<int64_t>(h) * p.ld_stat + r0, 512, st_full(i % NT));
                ++nt;
                // Q[i] and dO[i] land on one barrier (with the statistics operand):
                // one wait per step for the MMA warp
                // one release covers the Q and dO stages (dK[i - 2], after dV[i - 2], read the last of them)
                if (!mbar_wait_fast(q_empty(i % NQ), ((i / NQ) & 1) ^ 1u, p.status, kSiteAttn)) break;
                mbar_arrive_expect_tx(q_full(i % NQ), 2 * kTile);
                load_tile<D>(s_q + (i % NQ) * kTile, &map_qkv, q_full(i % NQ), h * D, r0);
                load_tile<D>(s_do + (i % ND) * kTile, &map_do, q_full(i % NQ), h * D, r0);
                ++nq;
            }
            mbar_wait_fast(kv_full, 0, p.status, kSiteDrain);
            for (int s = 0; s < NQ; ++s) {
                const uint32_t u = ring_uses(nq, NQ, s);
                if (u > 0) mbar_wait_fast(q_full(s), (u - 1) & 1, p.status, kSiteDrain);
            }
            for (int s = 0; s < NT; ++s) {
                const uint32_t u = ring_uses(nt, NT, s);
                if (u > 0) mbar_wait_fast(st_full(s), (u - 1) & 1, p.status, kSiteDrain);
            }
        }
    } else if (warp == 1) {
        // the whole warp runs the issue loop; its elected lane carries each instruction
        const uint32_t leader = elect_one_sync();
        constexpr uint32_t idesc_s = mma_idesc_bf16(128, 128, false, false);
        constexpr uint32_t idesc_g = mma_idesc_bf16(128, D, false, true);
        const uint64_t k_desc = kdesc_base(s_k), v_desc = kdesc_base(s_v);
        const uint64_t ones_lse = aug_desc(s_ones), ones_d = aug_desc(s_ones + L::kAugTile);
        auto issue_s = [&](int i) {
            const int st = i % NQ;
            // Q tile i and statistics operand i % NA (NA = NQ) complete one phase together
            if (!warp_wait(q_full(st), (i / NQ) & 1, p.status)) return false;
            tc_fence_after();
            const uint64_t q_desc = kdesc_base(s_q + st * kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_bf16_elected(leader, t_s, kdesc_at(k_desc, kk), kdesc_at(q_desc, kk), idesc_s, kk > 0);
            umma_bf16_elected(leader, t_s, ones_lse, aug_desc(s_aug + (i % NA) * L::kAugTile), idesc_s, 1u);
            umma_commit_elected(leader, s_full);
            return true;
        };
        auto issue_dp = [&](int i) {  // after issue_s(i), which waited for dO[i] and the statistics too
            const int st = i % ND;
            const uint64_t do_desc = kdesc_base(s_do + st * kTile);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma_bf16_elected(leader, t_dp, kdesc_at(v_desc, kk), kdesc_at(do_desc, kk), idesc_s, kk > 0);
            umma_bf16_elected(leader, t_dp, ones_d, aug_desc(s_aug + (i % NA) * L::kAugTile), idesc_s, 1u);
            umma_commit_elected(leader, dp_full);
            umma_commit_elected(leader, aug_empty(i % NA));
            return true;
        };
        bool ok = warp_wait(kv_full, 0, p.status) && issue_s(0) && issue_dp(0);
        // K steps of dV / dK in the order their P^T / dS^T chunks are packed:
        // chunk c of group g holds the K steps 4 g + 2 c and 4 g + 2 c + 1
        constexpr int kOrder[8] = {0, 1, 4, 5, 2, 3, 6, 7};
        for (int i = 0; ok && i < n_steps; ++i) {
            const uint64_t do_mn = mndesc_base(s_do + (i % ND) * kTile);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!warp_wait(p_full(c), i & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kk = kOrder[4 * c + e];
                    umma_bf16_ts_elected(leader, t_dv, t_s + packed_col(kk), mndesc_at(do_mn, kk), idesc_g,
                                         (i > 0 || kk > 0) ? 1u : 0u);
                }
            }
            if (!ok) break;
            // S^T[i+1] overwrites the S^T buffer after dV[i] has read P^T[i] from it
            if (i + 1 < n_steps && !issue_s(i + 1)) break;
            const uint64_t q_mn = mndesc_base(s_q + (i % NQ) * kTile);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!warp_wait(ds_full(c), i & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kk = kOrder[4 * c + e];
                    umma_bf16_ts_elected(leader, t_dk, t_dp + packed_col(kk), mndesc_at(q_mn, kk), idesc_g,
                                         (i > 0 || kk > 0) ? 1u : 0u);
                }
            }
            if (!ok) break;
            // Q[i] and dO[i]: dK[i] is the last product that reads either
            umma_commit_elected(leader, q_empty(i % NQ));
            if (i + 1 < n_steps && !issue_dp(i + 1)) break;
        }
        umma_commit_elected(leader, done);
        umma_commit_elected(leader, drain);
        mbar_wait_fast(drain, 0, p.status, kSiteDrain);
    } else if (warp == kStatWarp) {
        // ---------------- statistics warp: step i's lse and D into B operand i % NA
        const float inv_c = 1.f / p.scale_log2;
        for (int i = 0; i < n_steps; ++i) {
            if (!warp_wait(st_full(i % NT), (i / NT) & 1, p.status) ||
                !warp_wait(aug_empty(i % NA), ((i / NA) & 1) ^ 1u, p.status))
                break;
            const float* stat = reinterpret_cast<const float*>(smem_raw + L::kStat + 1024u * (i % NT));
            uint8_t* aug = smem_raw + L::kAug + (i % NA) * L::kAugTile;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = lane + 32 * u;
                // statistics past the sequence end are never written: whatever they
                // hold only reaches masked columns
                *reinterpret_cast<uint2*>(aug + aug_offset(r, 0)) = split3_bf16(-stat[r] * inv_c);
                *reinterpret_cast<uint2*>(aug + aug_offset(r, 1)) = split3_bf16(-stat[128 + r]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(q_full(i % NQ));
                mbar_arrive(st_empty(i % NT));
            }
        }
    } else {
        // ---------------- two groups of four warps, one key row per thread in each:
        // group gi takes query columns 64 gi .. 64 gi + 63 of every step
        const int gi = (warp - 2) >> 2;
        const int qw = warp & 3;
        const int row = qw * 32 + lane;
        const int k = k0 + row;
        const uint32_t t_row = (static_cast<uint32_t>(qw * 32) << 16) + 64u * gi;
        bool ok = true;
        for (int i = 0; i < n_steps; ++i) {
            const int qc0 = (kb + i / group) * kRows + 64 * gi;  // query of this group's first column
            // query column c is visible to this key when first <= c <= last
            const int first = k - qc0;
            const int last = s1 - 1 - qc0;
            if (!warp_wait(s_full, i & 1, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float pr[64];
            uint32_t rs[64];
            tmem_load_32(t_s + t_row, *reinterpret_cast<uint32_t(*)[32]>(rs));
            tmem_load_32(t_s + t_row + 32, *reinterpret_cast<uint32_t(*)[32]>(rs + 32));
            tmem_wait_load();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                // below the diagonal and inside the sequence every column is visible;
                // masked elements (which may carry statistics past the sequence end)
                // are selected away, never used
                const bool all_vis = __all_sync(0xffffffffu, first <= 32 * c && last >= 32 * c + 31);
#pragma unroll
                for (int j = 0; j < 32; ++j) pr[32 * c + j] = ex2(__uint_as_float(rs[32 * c + j]) * p.scale_log2);
                if (!all_vis) {  // one warp-uniform branch per chunk, bit masks inside
#pragma unroll
                    for (int j = 0; j < 32; ++j) pr[32 * c + j] = keep_if(pr[32 * c + j], (32 * c + j >= first) & (32 * c + j <= last));
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(pr[32 * c + 2 * e], pr[32 * c + 2 * e + 1]);
                // packed columns 16 c .. 16 c + 15 of the group's columns, all read above
                tmem_store_16(t_s + t_row + 16 * c, w);
                tmem_wait_store();
                tc_fence_before();
                warp_arrive(p_full(c), lane);
            }
            if (!warp_wait(dp_full, i & 1, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t rp[64];
            tmem_load_32(t_dp + t_row, *reinterpret_cast<uint32_t(*)[32]>(rp));
            tmem_load_32(t_dp + t_row + 32, *reinterpret_cast<uint32_t(*)[32]>(rp + 32));
            tmem_wait_load();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const bool all_vis = __all_sync(0xffffffffu, first <= 32 * c && last >= 32 * c + 31);
                float ds[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) ds[j] = pr[32 * c + j] * __uint_as_float(rp[32 * c + j]);
                if (!all_vis) {  // masked columns may hold statistics past the sequence end
#pragma unroll
                    for (int j = 0; j < 32; ++j) ds[j] = keep_if(ds[j], (32 * c + j >= first) & (32 * c + j <= last));
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(ds[2 * e], ds[2 * e + 1]);
                tmem_store_16(t_dp + t_row + 16 * c, w);
                tmem_wait_store();
                tc_fence_before();
                warp_arrive(ds_full(c), lane);
            }
        }
        // group 0 stores dK, group 1 dV
        if (ok && warp_wait(done, 0, p.status)) {
            tc_fence_after();
            const bool valid = k < s1;
            const uint32_t t_acc = (gi == 0 ? t_dk : t_dv) + (static_cast<uint32_t>(qw * 32) << 16);
            uint16_t* dst = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(k) * p.ld_out + (gi == 0 ? kcol : vcol);
            const float sc = gi == 0 ? p.scale : 1.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_load_32(t_acc + 32 * c, r);
                tmem_wait_load();
                if (valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        d4[q] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * q]) * sc, __uint_as_float(r[8 * q + 1]) * sc),
                                           pack_bf16x2(__uint_as_float(r[8 * q + 2]) * sc, __uint_as_float(r[8 * q + 3]) * sc),
                                           pack_bf16x2(__uint_as_float(r[8 * q + 4]) * sc, __uint_as_float(r[8 * q + 5]) * sc),
                                           pack_bf16x2(__uint_as_float(r[8 * q + 6]) * sc, __uint_as_float(r[8 * q + 7]) * sc));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------------ D = rowsum(dO * O)

// dvec[h][t] = sum_c da[t, h d + c] * a[t, h d + c].  Row r = t n_heads + h of
// da and a starts at element r d (rows are contiguous); d / 8 lanes read one
// row in 16-byte pieces (pointers and d keep them 16-byte aligned), so every
// load instruction covers 512 contiguous bytes of each tensor, and a warp
// takes 8 consecutive rows.  All of a warp's loads are issued before the first
// sum: with a reduction between one pair of rows and the next, the kernel ran
// at about 0.6 of the HBM bandwidth.
template <int D>
__global__ void attn_causal_rowsum_kernel(const uint16_t* __restrict__ da, const uint16_t* __restrict__ a, float* dvec,
                                          int tokens, int n_heads, int ld_stat) {
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRowsPerPass = 32 / kLanesPerRow;
    constexpr int kRowsPerWarp = 8;
    constexpr int kPasses = kRowsPerWarp / kRowsPerPass;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31, sub = lane / kLanesPerRow, pl = lane % kLanesPerRow;
    const int64_t n_rows = static_cast<int64_t>(tokens) * n_heads;
    uint4 u[kPasses], v[kPasses];
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
        const int64_t r = warp_id * kRowsPerWarp + i * kRowsPerPass + sub;
        u[i] = make_uint4(0u, 0u, 0u, 0u);
        v[i] = u[i];
        if (r < n_rows) {
            u[i] = *reinterpret_cast<const uint4*>(da + r * D + 8 * pl);
            v[i] = *reinterpret_cast<const uint4*>(a + r * D + 8 * pl);
        }
    }
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
        float acc = bf16_lo(u[i].x) * bf16_lo(v[i].x) + bf16_hi(u[i].x) * bf16_hi(v[i].x) +
                    bf16_lo(u[i].y) * bf16_lo(v[i].y) + bf16_hi(u[i].y) * bf16_hi(v[i].y) +
                    bf16_lo(u[i].z) * bf16_lo(v[i].z) + bf16_hi(u[i].z) * bf16_hi(v[i].z) +
                    bf16_lo(u[i].w) * bf16_lo(v[i].w) + bf16_hi(u[i].w) * bf16_hi(v[i].w);
#pragma unroll
        for (int o = kLanesPerRow / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);  // within a row's lanes
        const int64_t r = warp_id * kRowsPerWarp + i * kRowsPerPass + sub;
        if (pl == 0 && r < n_rows) {
            const int t = static_cast<int>(r / n_heads), h = static_cast<int>(r % n_heads);
            dvec[static_cast<int64_t>(h) * ld_stat + t] = acc;
        }
    }
}

// ------------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [rows, cols] bf16, row stride ld elements; boxes of 64 columns x 128 rows, 128B swizzle.
bool attn_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld) {
    auto fn = attn_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

AttnParams make_params(const AttnShape& s) {
    AttnParams p{};
    p.tokens = s.tokens;
    p.n_heads = s.n_heads;
    p.n_kv_heads = s.n_kv_heads;
    p.seq_len = s.seq_len;
    p.n_blocks = (s.tokens + kRows - 1) / kRows;
    p.ld_stat = s.ld_stat;
    p.scale = 1.0f / sqrtf(static_cast<float>(s.head_dim));
    p.scale_log2 = 1.4426950408889634f * p.scale;
    p.status = status_word();
    return p;
}

template <int D>
cudaError_t fwd_launch(const AttnShape& s, const void* qkv, void* a, float* lse, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = set_smem(attn_causal_fwd_kernel<D>, FwdSmem<D>::kBytes);
        if (err == cudaSuccess) err = set_smem(attn_causal_fwd_pair_kernel<D>, FwdPairSmem<D>::kBytes);
    });
    if (err != cudaSuccess) return err;
    const int qkv_w = (s.n_heads + 2 * s.n_kv_heads) * D;
    CUtensorMap m;
    if (!attn_map(&m, qkv, s.tokens, qkv_w, qkv_w)) return cudaErrorInvalidValue;
    AttnParams p = make_params(s);
    if (!p.status) return cudaErrorInvalidDevice;
    p.out = a;
    p.ld_out = static_cast<int64_t>(s.n_heads) * D;
    p.lse = lse;
    if ((s.n_heads / s.n_kv_heads) % 2 == 0)  // two heads of a group per CTA
        attn_causal_fwd_pair_kernel<D><<<p.n_blocks * (s.n_heads / 2), kAttnBwdThreads, FwdPairSmem<D>::kBytes,
                                          stream>>>(m, p);
    else
        attn_causal_fwd_kernel<D><<<p.n_blocks * s.n_heads, kAttnThreads, FwdSmem<D>::kBytes, stream>>>(m, p);
    return cudaGetLastError();
}

// A second stream per device for the dQ kernel.  dQ and dK/dV read the same
// inputs and write disjoint columns of dqkv, so they run side by side: the dK/dV
// kernel's CTAs carry up to 32 times different work (the first key block of
// each kv head sees every query block), and on one stream the SMs that finish
// early sat idle until its longest CTAs were done.  The caller's stream forks
// to the side stream after the row kernel and joins it after both launches; a
// mutex keeps concurrent callers from interleaving the fork and join events.
// The stream also owns the dQ kernel's tile counter (one int of device memory,
// zeroed on the side stream before each launch) and the device's SM count
// (the persistent kernel's grid).
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    int* tiles = nullptr;
    int sms = 0;
    std::mutex mu;
};

SideStream* side_stream() {
    static SideStream sides[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    SideStream& s = sides[dev];
    if (!s.stream) {
        cudaStream_t st = nullptr;
        cudaEvent_t f = nullptr, j = nullptr;
        int* tiles = nullptr;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return nullptr;
        if (cudaMalloc(&tiles, sizeof(int)) != cudaSuccess) return nullptr;
        if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
            cudaFree(tiles);
            return nullptr;
        }
        if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
            if (f) cudaEventDestroy(f);
            cudaStreamDestroy(st);
            cudaFree(tiles);
            return nullptr;
        }
        s.stream = st;
        s.fork = f;
        s.join = j;
        s.tiles = tiles;
        s.sms = sms;
    }
    return &s;
}

template <int D>
cudaError_t bwd_launch(const AttnShape& s, const void* qkv, const void* a, const void* da, const float* lse,
                       float* dvec, void* dqkv, cudaStream_t stream, bool dvec_ready) {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = set_smem(attn_causal_dq_kernel<D>, DqSmem<D>::kBytes);
        if (err == cudaSuccess) err = set_smem(attn_causal_dkdv_kernel<D>, DkvSmem<D>::kBytes);
    });
    if (err != cudaSuccess) return err;
    const int qkv_w = (s.n_heads + 2 * s.n_kv_heads) * D;
    const int hw = s.n_heads * D;
    CUtensorMap mq, md;
    if (!attn_map(&mq, qkv, s.tokens, qkv_w, qkv_w) || !attn_map(&md, da, s.tokens, hw, hw))
        return cudaErrorInvalidValue;
    AttnParams p = make_params(s);
    if (!p.status) return cudaErrorInvalidDevice;
    p.out = dqkv;
    p.ld_out = qkv_w;
    p.lse = const_cast<float*>(lse);
    p.dvec = dvec;
    cudaError_t e = cudaSuccess;
    if (!dvec_ready) {
        const int64_t warps = (static_cast<int64_t>(s.tokens) * s.n_heads + 7) / 8;  // 8 rows per warp
        attn_causal_rowsum_kernel<D><<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(
            static_cast<const uint16_t*>(da), static_cast<const uint16_t*>(a), dvec, s.tokens, s.n_heads, s.ld_stat);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    SideStream* side = side_stream();
    if (!side) return cudaErrorInitializationError;
    std::lock_guard<std::mutex> lock(side->mu);
    if ((e = cudaEventRecord(side->fork, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(side->stream, side->fork, 0)) != cudaSuccess) return e;
    attn_causal_dkdv_kernel<D><<<p.n_blocks * s.n_kv_heads, kAttnDkvThreads, DkvSmem<D>::kBytes, stream>>>(mq, md, p);
    const cudaError_t e_kv = cudaGetLastError();
    const int n_tiles = p.n_blocks * s.n_heads;
    cudaError_t e_q = cudaMemsetAsync(side->tiles, 0, sizeof(int), side->stream);
    if (e_q == cudaSuccess) {
        attn_causal_dq_kernel<D><<<static_cast<unsigned>(std::min(n_tiles, side->sms)), kAttnDqThreads,
                                   DqSmem<D>::kBytes, side->stream>>>(mq, md, p, side->tiles);
        e_q = cudaGetLastError();
    }
    // the join is recorded whatever happened above, so the caller's stream never
    // runs ahead of work already queued on the side stream
    if ((e = cudaEventRecord(side->join, side->stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(stream, side->join, 0)) != cudaSuccess) return e;
    return e_kv != cudaSuccess ? e_kv : e_q;
}

}  // namespace

cudaError_t launch_attention_causal_forward(const AttnShape& s, const void* qkv, void* a, float* lse,
                                            cudaStream_t stream) {
    if (s.tokens <= 0) return cudaSuccess;
    if (s.head_dim == 128) return fwd_launch<128>(s, qkv, a, lse, stream);
    if (s.head_dim == 64) return fwd_launch<64>(s, qkv, a, lse, stream);
    return cudaErrorInvalidValue;
}

cudaError_t attention_prepare() { return side_stream() ? cudaSuccess : cudaErrorInitializationError; }

cudaError_t launch_attention_causal_backward(const AttnShape& s, const void* qkv, const void* a, const void* da,
                                             const float* lse, float* dvec, void* dqkv, cudaStream_t stream,
                                             bool dvec_ready) {
    if (s.tokens <= 0) return cudaSuccess;
    if (s.head_dim == 128) return bwd_launch<128>(s, qkv, a, da, lse, dvec, dqkv, stream, dvec_ready);
    if (s.head_dim == 64) return bwd_launch<64>(s, qkv, a, da, lse, dvec, dqkv, stream, dvec_ready);
    return cudaErrorInvalidValue;
}

}  // namespace zbk
