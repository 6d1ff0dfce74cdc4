// Persistent tcgen05 GEMM for sm_103a with fused epilogues.
//
// One CTA per SM walks output tiles of BM x BN = 128 x 256.  Warp roles:
//   warp 0   one thread issues TMA tile loads into a 4-stage ring of 48 KiB
//   warp 1   allocates tensor memory; one thread issues tcgen05.mma (bf16 in,
//            f32 accumulate) into one of two 128 x BN f32 accumulators
//   warps 2-5 epilogue: tcgen05.ld the accumulator (one row per thread), apply
//            the fused op, store to global memory
// Two accumulators (512 tensor-memory columns) let the epilogue of one tile run
// while the MMAs of the next tile fill the other.
//
// Operand layouts (the three GEMMs of a split backward, "Zero-Bubble Pipeline
// Parallelism Guide for LLMs", "Core Innovation 1"; weights [out, in] as in
// its "Step-by-Step Implementation"):
//   Forward        y  = x w^T    A = x  [M=T, K=in]  K-major, B = w [N=out, K=in] K-major
//   BackwardInput  dx = dy w     A = dy [M=T, K=out] K-major, B = w [K=out, N=in] MN-major
//   BackwardWeight dw += dy^T x  A = dy [K=T, M=out] MN-major, B = x [K=T, N=in] MN-major
// All tiles use 128-byte swizzling.  A K-major tile is rows of 64 bf16 (128 B);
// an MN-major tile is BK rows of 64 MN-elements per 64-wide block, one TMA box
// per block.  Out-of-range rows and columns of a box read as zero, so ragged
// M, N and K need no special mainloop; the epilogue masks rows >= M, cols >= N.
//
// Tile order: tiles are walked in groups of G rows (or columns) of tiles so that
// the tiles in flight at once share operand panels in L2.  The host picks G
// per launch with a small model of the DRAM bytes each wave of tiles fetches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "device_common.cuh"
#include "launch.h"

namespace zbk {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
constexpr uint32_t kAStageBytes = BM * BK * 2;   // 16 KiB
constexpr uint32_t kMnBlockBytes = 64 * BK * 2;  // one 64-wide MN block of an MN-major tile

// A 128 x 128 tile was tried for launches whose 128 x 256 tiling leaves a
// poor last wave: on GB300 it ran at about two thirds of the wide tile's rate
// per FLOP (twice the A-operand shared-memory traffic per MMA FLOP), so every
// launch of the one-CTA kernel uses the wide tile.  The CTA-pair kernel cuts
// only its short last wave: into K halves when K is long enough to pay for
// exchanging float32 partials, else into 256 x 128 column halves.
constexpr int kBN = 256;

template <int BN>
struct Cfg {
    static constexpr int STAGES = 4;
    static constexpr uint32_t kBStageBytes = BN * BK * 2;
    static constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
    static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr size_t kSmemBytes = 1024 + STAGES * kStageBytes + kNumBars * 8 + 16;
};
static_assert(Cfg<kBN>::kSmemBytes <= 232448, "shared memory");

struct KParams {
    int m, n, k;
    int tiles_m, tiles_n, num_tiles, k_blocks;
    int group;      // tiles per group along the grouped dimension
    int group_m;    // 1: groups of `group` tile rows (m fastest inside); 0: groups of tile columns
    void* out;
    int64_t ldo;
    const void* aux;
    int64_t ld_aux;
    int ffn;
    int* status;
    // MN-major 128B-swizzled operands: the leading-dimension offset steps between
    // 64-element MN blocks, the stride-dimension offset between 8-row K groups.
    uint32_t mn_lbo;
    uint32_t mn_sbo;
    // K split of the last wave (CTA-pair kernel only): tiles from split_from on
    // are two work units each, unit split_from + 2 (t - split_from) + h
    // covering k-blocks [0, kb_split) for h = 0 and [kb_split, k_blocks) for
    // h = 1; earlier tiles are one unit each.  split == 1: no tile splits
    // (split_from == num_tiles).
    int split;
    int split_from;
    int kb_split;
    // Narrow last wave (CTA-pair kernel, no K split): tiles from narrow_from on
    // are two work units each, unit narrow_from + 2 (t - narrow_from) + h
    // covering output columns 128 h .. 128 h + 127 of the tile over the whole
    // K; narrow_from == num_tiles: none.
    int narrow_from;
    int num_units;
    uint32_t* flags;   // one word per 32 rows of a split tile: 2 epoch (claimed), 2 epoch + 1 (partial written)
    float* partial;    // one float32 256 x 256 tile per split tile
    uint32_t epoch;
    float* dot;        // row-dot epilogue: [n / dot_cols][ld_dot] float32 sums
    int64_t ld_dot;
    int dot_cols;
};

struct Unit {
    int tile, half, kb0, kb1;
    int nh;       // the column half of a narrow unit
    bool split;   // one of the two K halves of a split tile
    bool narrow;  // one of the two 128-column halves of a tile
};

template <bool SPLIT>
__device__ __forceinline__ Unit unit_of(const KParams& p, int u) {
    Unit w;
    w.nh = 0;
    w.narrow = false;
    if (SPLIT && u >= p.split_from) {
        const int v = u - p.split_from;
        w.tile = p.split_from + (v >> 1);
        w.half = v & 1;
        w.kb0 = w.half ? p.kb_split : 0;
        w.kb1 = w.half ? p.k_blocks : p.kb_split;
        w.split = true;
    } else if (!SPLIT && u >= p.narrow_from) {
        const int v = u - p.narrow_from;
        w.tile = p.narrow_from + (v >> 1);
        w.nh = v & 1;
        w.narrow = true;
        w.half = 0;
        w.kb0 = 0;
        w.kb1 = p.k_blocks;
        w.split = false;
    } else {
        w.tile = u;
        w.half = 0;
        w.kb0 = 0;
        w.kb1 = p.k_blocks;
        w.split = false;
    }
    return w;
}

// A CTA-pair launch: up to kMaxGroup independent GEMMs of the same operand
// layouts and epilogue, run as one stream of work units (problem after
// problem), so that the last wave of one fills with the first tiles of the
// next.  A single GEMM is a group of one.
struct PairGroup {
    CUtensorMap map[2 * kMaxGroup];   // A and B of each problem
    CUtensorMap omap[kMaxGroup];      // output of each problem (all epilogues but the SwiGLU backward)
    CUtensorMap xmap[4];              // SwiGLU backward (never grouped): g, u, dg, du
    KParams kp[kMaxGroup];
    int unit_begin[kMaxGroup + 1];   // first work unit of each problem; the last entry is the total
    int n_probs;
};

__device__ __forceinline__ int problem_of(const PairGroup& G, int u) {
    int pi = 0;
    while (pi + 1 < G.n_probs && u >= G.unit_begin[pi + 1]) ++pi;
    return pi;
}

// Tile index -> (tile row, tile column) under the grouped raster.
__device__ __forceinline__ void tile_coords(const KParams& p, int tile, int& tm, int& tn) {
    if (p.group_m) {
        const int per = p.group * p.tiles_n;
        const int g = tile / per;
        const int in = tile - g * per;
        const int rows = min(p.group, p.tiles_m - g * p.group);
        tm = g * p.group + in % rows;
        tn = in / rows;
    } else {
        const int per = p.group * p.tiles_m;
        const int g = tile / per;
        const int in = tile - g * per;
        const int cols = min(p.group, p.tiles_n - g * p.group);
        tn = g * p.group + in % cols;
        tm = in / cols;
    }
}

// bf16 results of one 32-column chunk of a row: o0 holds the stored values
// (dg for the SwiGLU backward), o1 holds du (SwiGLU backward only).
template <int EPI>
__device__ __forceinline__ void epilogue_pack(const uint32_t (&r)[32], const uint4 (&x0)[4], const uint4 (&x1)[4],
                                              uint4 (&o0)[4], uint4 (&o1)[4]) {
    if constexpr (EPI == static_cast<int>(Epilogue::SwigluBwd)) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t gw[4] = {x0[j].x, x0[j].y, x0[j].z, x0[j].w};
            const uint32_t uw[4] = {x1[j].x, x1[j].y, x1[j].z, x1[j].w};
            uint32_t dgw[4], duw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float dg2[2], du2[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float ds = __uint_as_float(r[8 * j + 2 * e + h]);
                    const float g = h ? bf16_hi(gw[e]) : bf16_lo(gw[e]);
                    const float u = h ? bf16_hi(uw[e]) : bf16_lo(uw[e]);
                    const float sg = __fdividef(1.0f, 1.0f + __expf(-g));
                    dg2[h] = ds * u * sg * (1.0f + g * (1.0f - sg));
                    du2[h] = ds * g * sg;
                }
                dgw[e] = pack_bf16x2(dg2[0], dg2[1]);
                duw[e] = pack_bf16x2(du2[0], du2[1]);
            }
            o0[j] = make_uint4(dgw[0], dgw[1], dgw[2], dgw[3]);
            o1[j] = make_uint4(duw[0], duw[1], duw[2], duw[3]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[8 * j + e]);
            if constexpr (EPI == static_cast<int>(Epilogue::AddResidual)) {
                const uint32_t rw[4] = {x0[j].x, x0[j].y, x0[j].z, x0[j].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[2 * e] += bf16_lo(rw[e]);
                    v[2 * e + 1] += bf16_hi(rw[e]);
                }
            }
            o0[j] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                               pack_bf16x2(v[6], v[7]));
        }
    }
}

// Row-dot epilogue: the sum over one 32-column chunk of a row of the stored
// (bf16-rounded) results times aux, in four interleaved float32 chains.
__device__ __forceinline__ float row_dot_bf16(const uint32_t (&r)[32], const uint4 (&x0)[4]) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t xw[4] = {x0[j].x, x0[j].y, x0[j].z, x0[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t v = pack_bf16x2(__uint_as_float(r[8 * j + 2 * e]), __uint_as_float(r[8 * j + 2 * e + 1]));
            acc[e] = fmaf(bf16_lo(v), bf16_lo(xw[e]), acc[e]);
            acc[e] = fmaf(bf16_hi(v), bf16_hi(xw[e]), acc[e]);
        }
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Epilogue of one 32-column chunk of row m, written straight to global memory.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const KParams& p, int m, int n, const uint32_t (&r)[32],
                                               const uint4 (&x0)[4], const uint4 (&x1)[4]) {
    if constexpr (EPI == static_cast<int>(Epilogue::AccumF32)) {
        float* dst = static_cast<float*>(p.out) + static_cast<int64_t>(m) * p.ldo + n;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * j),
                         "f"(__uint_as_float(r[4 * j])), "f"(__uint_as_float(r[4 * j + 1])),
                         "f"(__uint_as_float(r[4 * j + 2])), "f"(__uint_as_float(r[4 * j + 3]))
                         : "memory");
        }
    } else {
        uint4 o0[4], o1[4];
        epilogue_pack<EPI>(r, x0, x1, o0, o1);
        uint16_t* base = static_cast<uint16_t*>(p.out) + static_cast<int64_t>(m) * p.ldo;
        uint4* dst = reinterpret_cast<uint4*>(base + n);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = o0[j];
        if constexpr (EPI == static_cast<int>(Epilogue::SwigluBwd)) {
            uint4* du_dst = reinterpret_cast<uint4*>(base + p.ffn + n);
#pragma unroll
            for (int j = 0; j < 4; ++j) du_dst[j] = o1[j];
        }
    }
}

// Output staging of the CTA-pair kernel: each epilogue warp writes a chunk of
// its 32 rows x 32 columns into a shared-memory box and one lane hands the box
// to a TMA bulk-tensor store (bf16) or reduce-add (float32).  A bf16 row is 64
// bytes and takes the 64-byte TMA swizzle (16-byte word j of row r at word
// j ^ ((r >> 1) & 3)); a float32 row is 128 bytes and takes the 128-byte
// swizzle (word j of row r at word j ^ (r & 7)).  Either way eight
// consecutive rows cover all banks.
constexpr uint32_t kBf16BoxBytes = 32 * 64;  // 32 rows x 32 bf16 columns

template <int EPI>
__host__ __device__ constexpr uint32_t out_box_bytes() {
    return EPI == static_cast<int>(Epilogue::AccumF32) ? 32 * 128 : kBf16BoxBytes;
}

// SwiGLU backward of one 32-column chunk in place in a side-input ring slot:
// the g box (64-byte swizzle, as TMA loaded it) becomes dg and the u box du,
// ready for the TMA stores.
__device__ __forceinline__ void swiglu_chunk_in_smem(uint32_t slot, int lane, const uint32_t (&r)[32]) {
    const uint32_t l = static_cast<uint32_t>(lane);
    const uint32_t sw = (l >> 1) & 3u;
    const uint32_t grow = slot + l * 64u, urow = slot + kBf16BoxBytes + l * 64u;
    uint4 x0[4], x1[4], o0[4], o1[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t off = (static_cast<uint32_t>(j) ^ sw) << 4;
        x0[j] = ld_shared_v4(grow + off);
        x1[j] = ld_shared_v4(urow + off);
    }
    epilogue_pack<static_cast<int>(Epilogue::SwigluBwd)>(r, x0, x1, o0, o1);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t off = (static_cast<uint32_t>(j) ^ sw) << 4;
        st_shared_v4(grow + off, o0[j]);
        st_shared_v4(urow + off, o1[j]);
    }
}

template <int EPI>
__device__ __forceinline__ void epilogue_chunk_to_smem(uint32_t box, int lane, const uint32_t (&r)[32],
                                                       const uint4 (&x0)[4]) {
    const uint32_t l = static_cast<uint32_t>(lane);
    if constexpr (EPI == static_cast<int>(Epilogue::AccumF32)) {
        const uint32_t row = box + l * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(row + ((static_cast<uint32_t>(j) ^ (l & 7u)) << 4),
                         make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]));
    } else {
        uint4 o0[4], unused[4];
        epilogue_pack<EPI>(r, x0, x0, o0, unused);
        const uint32_t row = box + l * 64u;
        const uint32_t sw = (l >> 1) & 3u;
#pragma unroll
        for (int j = 0; j < 4; ++j) st_shared_v4(row + ((static_cast<uint32_t>(j) ^ sw) << 4), o0[j]);
    }
}

template <int BN, bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const KParams p) {
    constexpr int STAGES = Cfg<BN>::STAGES;
    constexpr uint32_t kBStageBytes = Cfg<BN>::kBStageBytes;
    constexpr uint32_t kStageBytes = Cfg<BN>::kStageBytes;
    constexpr uint32_t kTmemCols = Cfg<BN>::kTmemCols;
    constexpr int kNumBars = Cfg<BN>::kNumBars;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t s_a = base;
    const uint32_t s_b = base + STAGES * kAStageBytes;
    const uint32_t bars = s_b + STAGES * kBStageBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * STAGES + 4);
    const uint32_t tmem_slot = bars + 8u * kNumBars;
    volatile uint32_t* tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_slot - raw));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128);
        }
        mbar_init(drain_bar, 1);
        mbar_fence_init();
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot_ptr;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            uint32_t n_fills = 0;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                int tm, tn;
                tile_coords(p, tile, tm, tn);
                const int m0 = tm * BM;
                const int n0 = tn * BN;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.status, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(stage);
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    const int k0 = kb * BK;
                    const uint32_t a_dst = s_a + stage * kAStageBytes;
                    const uint32_t b_dst = s_b + stage * kBStageBytes;
                    if constexpr (A_MN) {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d(a_dst + j * kMnBlockBytes, &map_a, fb, m0 + 64 * j, k0);
                    } else {
                        tma_load_2d(a_dst, &map_a, fb, k0, m0);
                    }
                    if constexpr (B_MN) {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_2d(b_dst + j * kMnBlockBytes, &map_b, fb, n0 + 64 * j, k0);
                    } else {
                        tma_load_2d(b_dst, &map_b, fb, k0, n0);
                    }
                    ++n_fills;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every load issued must land before the CTA's shared memory goes away.
            for (int s = 0; s < STAGES; ++s) {
                const uint32_t u = ring_uses(n_fills, STAGES, s);
                if (u > 0) mbar_wait(full_bar(s), (u - 1u) & 1u, p.status, kSiteDrain, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: the whole warp, its elected lane carries each instruction
        const uint32_t issuer = elect_one_sync();
        constexpr uint32_t idesc = mma_idesc_bf16(BM, BN, A_MN, B_MN);
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t aph = (static_cast<uint32_t>(it) >> 1) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait_fast(tempty_bar(acc), aph ^ 1u, p.status, kSiteMmaTmemEmpty))) break;
            tc_fence_after();
            const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait_fast(full_bar(stage), phase, p.status, kSiteMmaFull))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = s_a + stage * kAStageBytes;
                const uint32_t b0 = s_b + stage * kBStageBytes;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    // K-major: the 16-element K step is 32 bytes inside the
                    // 128-byte swizzled row; MN-major: it is 16 rows of 128 B.
                    const uint64_t ad = A_MN ? smem_desc_sw128(a0 + k * 2048, p.mn_lbo, p.mn_sbo)
                                             : smem_desc_sw128(a0 + k * 32, 16, 1024);
                    const uint64_t bd = B_MN ? smem_desc_sw128(b0 + k * 2048, p.mn_lbo, p.mn_sbo)
                                             : smem_desc_sw128(b0 + k * 32, 16, 1024);
                    umma_bf16_elected(issuer, d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                }
                umma_commit_elected(issuer, empty_bar(stage));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit_elected(issuer, tfull_bar(acc));
        }
        // No MMA may still run when tensor memory is freed.
        umma_commit_elected(issuer, drain_bar);
        mbar_wait(drain_bar, 0, p.status, kSiteDrain, kWaitLimitNs);
    } else {
        // ---------------- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t aph = (static_cast<uint32_t>(it) >> 1) & 1u;
            // one verdict per warp: the tensor-memory loads below are warp-wide
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), aph, p.status, kSiteEpiTmemFull))) break;
            tc_fence_after();
            int tm, tn;
            tile_coords(p, tile, tm, tn);
            const int m = tm * BM + row;
            const int n_base = tn * BN;
            const bool row_ok = m < p.m;
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int n = n_base + c * 32;
                const bool ok = row_ok && n < p.n;
                uint4 x0[4], x1[4];
                if constexpr (EPI == static_cast<int>(Epilogue::AddResidual) ||
                              EPI == static_cast<int>(Epilogue::SwigluBwd)) {
                    if (ok) {
                        const uint16_t* rowp =
                            static_cast<const uint16_t*>(p.aux) + static_cast<int64_t>(m) * p.ld_aux;
                        const uint4* s0 = reinterpret_cast<const uint4*>(rowp + n);
#pragma unroll
                        for (int j = 0; j < 4; ++j) x0[j] = s0[j];
                        if constexpr (EPI == static_cast<int>(Epilogue::SwigluBwd)) {
                            const uint4* s1 = reinterpret_cast<const uint4*>(rowp + p.ffn + n);
#pragma unroll
                            for (int j = 0; j < 4; ++j) x1[j] = s1[j];
                        }
                    }
                }
                uint32_t r[32];
                tmem_load_32(tbase + static_cast<uint32_t>(c * 32), r);
                tmem_wait_load();
                if (c == BN / 32 - 1) {
                    tc_fence_before();
                    mbar_arrive(tempty_bar(acc));
                }
                if (ok) epilogue_chunk<EPI>(p, m, n, r, x0, x1);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- CTA-pair kernel
//
// The two CTAs of a cluster compute one 256 x 256 output tile with
// tcgen05.mma.cta_group::2.  CTA r (cluster rank r) keeps rows 128 r .. +127
// of the A tile and columns 128 r .. +127 of the B tile in its own shared
// memory; the MMA, issued by one thread of rank 0, reads both halves, and
// each CTA's tensor memory receives its 128 rows of D.  Per SM this moves a
// third less operand data through shared memory than the one-CTA 128 x 256
// tile, and a stage is 32 KiB, so the ring is 6 stages deep.
//
// Synchronisation across the pair:
//   full[s]    lives in rank 0; rank 0 expects both CTAs' bytes, each CTA's
//              TMA completes its share there (cta_group::2 loads);
//   empty[s]   in each CTA; the MMA commit multicasts to both;
//   tfull[a]   in each CTA; the MMA commit multicasts to both;
//   tempty[a]  lives in rank 0; all 256 epilogue threads of the pair arrive.
constexpr int kPairM = 256;
constexpr int kPairN = 256;
constexpr int kHalf = 128;
constexpr uint32_t kPairAStage = kHalf * BK * 2;  // 16 KiB
constexpr uint32_t kPairBStage = kHalf * BK * 2;  // 16 KiB
constexpr uint32_t kPairStage = kPairAStage + kPairBStage;
// Side-input ring of the SwiGLU backward: per epilogue warp two slots, each
// the g and u boxes of one 32-column chunk, so that the operand ring keeps all
// six stages (four slots and five stages: the SwiGLU dgrad took 306.7 us
// against 295.5 us, same bits; three slots and five stages: 310.3 us).
constexpr int kSideSlots = 2;
constexpr uint32_t kSideSlotBytes = 2 * kBf16BoxBytes;
template <int EPI>
__host__ __device__ constexpr int pair_stages() {
    return 6;
}
template <int EPI>
__host__ __device__ constexpr int pair_num_bars() {
    return 2 * pair_stages<EPI>() + 5 + (EPI == static_cast<int>(Epilogue::SwigluBwd) ? 4 * kSideSlots : 0);
}
// bf16 outputs of the plain and residual epilogues leave through staging boxes
// and TMA stores (4.2 % faster for a 4096 x 14336 dgrad, 4.9 % for a
// 4096 x 28672 forward on GB300), and the float32 weight-gradient sums through
// TMA reduce-adds, where the L2 does the read-modify-write.  The SwiGLU
// backward has its side inputs g and u brought in by TMA as well, into a ring
// that runs one chunk ahead, computes dg and du in place there and stores
// them by TMA: its epilogue warps touch no global memory with per-row accesses.
template <int EPI>
__host__ __device__ constexpr bool tma_out() {
    return EPI != static_cast<int>(Epilogue::SwigluBwd);
}
// Output staging or the side-input ring.  Staging: two boxes per epilogue
// warp, used in turn; the SwiGLU forward has one set of three (its g, u and s
// boxes), so that the operand ring keeps all six stages (with two sets and five
// stages its GEMM ran 2 % slower).
template <int EPI>
__host__ __device__ constexpr uint32_t pair_boxes_per_set() {
    return EPI == static_cast<int>(Epilogue::SwigluFwd) ? 3 : 1;
}
template <int EPI>
__host__ __device__ constexpr uint32_t pair_out_sets() {
    return EPI == static_cast<int>(Epilogue::SwigluFwd) ? 1 : 2;
}
template <int EPI>
__host__ __device__ constexpr uint32_t pair_out_bytes() {
    return tma_out<EPI>() ? 4 * pair_out_sets<EPI>() * pair_boxes_per_set<EPI>() * out_box_bytes<EPI>()
                          : 4 * kSideSlots * kSideSlotBytes;
}
template <int EPI>
__host__ __device__ constexpr size_t pair_smem_bytes() {
    return 1024 + pair_stages<EPI>() * kPairStage + pair_out_bytes<EPI>() + pair_num_bars<EPI>() * 8 + 16;
}
static_assert(pair_smem_bytes<static_cast<int>(Epilogue::AccumF32)>() <= 232448, "shared memory");
static_assert(pair_smem_bytes<static_cast<int>(Epilogue::SwigluBwd)>() <= 232448, "shared memory");
static_assert(pair_smem_bytes<static_cast<int>(Epilogue::SwigluFwd)>() <= 232448, "shared memory");

// SwiGLU forward of one 32-column chunk pair: g (rg) and u (ru) rounded to bf16
// into their boxes, and s = silu(g) u from the rounded values into the third
// (64-byte swizzle, as for every bf16 box).
__device__ __forceinline__ void swiglu_fwd_chunk_to_smem(uint32_t set, int lane, const uint32_t (&rg)[32],
                                                         const uint32_t (&ru)[32]) {
    const uint32_t l = static_cast<uint32_t>(lane);
    const uint32_t sw = (l >> 1) & 3u;
    const uint32_t grow = set + l * 64u, urow = grow + kBf16BoxBytes, srow = grow + 2 * kBf16BoxBytes;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t gw[4], uw[4], sv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            gw[e] = pack_bf16x2(__uint_as_float(rg[8 * j + 2 * e]), __uint_as_float(rg[8 * j + 2 * e + 1]));
            uw[e] = pack_bf16x2(__uint_as_float(ru[8 * j + 2 * e]), __uint_as_float(ru[8 * j + 2 * e + 1]));
            sv[e] = pack_bf16x2(swiglu_value(bf16_lo(gw[e]), bf16_lo(uw[e])), swiglu_value(bf16_hi(gw[e]), bf16_hi(uw[e])));
        }
        const uint32_t off = (static_cast<uint32_t>(j) ^ sw) << 4;
        st_shared_v4(grow + off, make_uint4(gw[0], gw[1], gw[2], gw[3]));
        st_shared_v4(urow + off, make_uint4(uw[0], uw[1], uw[2], uw[3]));
        st_shared_v4(srow + off, make_uint4(sv[0], sv[1], sv[2], sv[3]));
    }
}

template <bool A_MN, bool B_MN, int EPI, int NACC, bool SPLIT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ PairGroup G) {
    int* const status = G.kp[0].status;
    const uint32_t mn_lbo = G.kp[0].mn_lbo, mn_sbo = G.kp[0].mn_sbo;
    const int num_units = G.unit_begin[G.n_probs];
    constexpr uint32_t kTmemCols = NACC * kPairN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t s_a = base;
    constexpr int kStages = pair_stages<EPI>();
    constexpr int kNumBars = pair_num_bars<EPI>();
    const uint32_t s_b = base + kStages * kPairAStage;
    constexpr bool kTmaOut = tma_out<EPI>();
    const uint32_t s_out = s_b + kStages * kPairBStage;  // 2 KiB-aligned boxes
    constexpr uint32_t kBoxBytes = out_box_bytes<EPI>();
    const uint32_t bars = s_out + pair_out_bytes<EPI>();
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * kStages + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * kStages + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * kStages + 4);
    const uint32_t side_bars = bars + 8u * (2 * kStages + 5);  // SwiGLU backward: 4 warps x kSideSlots
    const uint32_t tmem_slot = bars + 8u * kNumBars;
    volatile uint32_t* tmem_slot_ptr = reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_slot - raw));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        if constexpr (!kTmaOut)
            for (int s = 0; s < 4 * kSideSlots; ++s) mbar_init(side_bars + 8u * s, 1);
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * 128);
        }
        mbar_init(drain_bar, 1);
        mbar_fence_init();
        for (int i = 0; i < 2 * G.n_probs; ++i) tma_prefetch_map(&G.map[i]);
        if constexpr (kTmaOut)
            for (int i = 0; i < G.n_probs; ++i) tma_prefetch_map(&G.omap[i]);
        else
            for (int i = 0; i < 4; ++i) tma_prefetch_map(&G.xmap[i]);
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised, tensor memory allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot_ptr;
    // Both CTAs must hold the accumulator at the same columns.
    const uint32_t peer_base = ld_shared_cluster_u32(map_to_cta(tmem_slot, rank ^ 1u));
    const bool usable = peer_base == tmem_base;
    if (!usable && threadIdx.x == 0) atomicCAS(status, 0, kSitePairTmem);

    if (usable && warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs)
            uint32_t n_fills = 0;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = pair; ok && u < num_units; u += npairs) {
                const int pi = problem_of(G, u);
                const KParams& p = G.kp[pi];
                const Unit w = unit_of<SPLIT>(p, u - G.unit_begin[pi]);
                int tm, tn;
                tile_coords(p, w.tile, tm, tn);
                const int m0 = tm * kPairM + static_cast<int>(rank) * kHalf;
                // SwiGLU forward: rank 0 takes 128 gate rows, rank 1 the same 128 up
                // rows (ffn further on), so each CTA's accumulator holds g and u of
                // the same features side by side
                // A narrow unit's 128 columns split 64 / 64 between the CTAs; the
                // loads keep their full boxes (the 64 columns past them are
                // loaded and not read, or zero-filled past N)
                const int n0 = EPI == static_cast<int>(Epilogue::SwigluFwd)
                                   ? tn * kHalf + (rank != 0 ? p.ffn : 0)
                                   : (w.narrow ? tn * kPairN + w.nh * kHalf + static_cast<int>(rank) * (kHalf / 2)
                                               : tn * kPairN + static_cast<int>(rank) * kHalf);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, status, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = full_bar(stage);
                    if (leader) mbar_arrive_expect_tx(fb_local, 2 * kPairStage);
                    const uint32_t fb = map_to_cta(fb_local, 0);
                    const int k0 = kb * BK;
                    const uint32_t a_dst = s_a + stage * kPairAStage;
                    const uint32_t b_dst = s_b + stage * kPairBStage;
                    if constexpr (A_MN) {
#pragma unroll
                        for (int j = 0; j < kHalf / 64; ++j)
                            tma_load_2d_pair(a_dst + j * kMnBlockBytes, &G.map[2 * pi], fb, m0 + 64 * j, k0);
                    } else {
                        tma_load_2d_pair(a_dst, &G.map[2 * pi], fb, k0, m0);
                    }
                    if constexpr (B_MN) {
#pragma unroll
                        for (int j = 0; j < kHalf / 64; ++j)
                            tma_load_2d_pair(b_dst + j * kMnBlockBytes, &G.map[2 * pi + 1], fb, n0 + 64 * j, k0);
                    } else {
                        tma_load_2d_pair(b_dst, &G.map[2 * pi + 1], fb, k0, n0);
                    }
                    ++n_fills;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Loads must land before shared memory goes away: rank 0 sees its
            // full barriers complete; rank 1 sees the MMA release each stage.
            for (int s = 0; s < kStages; ++s) {
                const uint32_t u = ring_uses(n_fills, kStages, s);
                if (u > 0) {
                    if (leader)
                        mbar_wait_cluster(full_bar(s), (u - 1u) & 1u, status, kSiteDrain, kWaitLimitNs);
                    else
                        mbar_wait_cluster(empty_bar(s), (u - 1u) & 1u, status, kSiteDrain, kWaitLimitNs);
                }
            }
        }
    } else if (usable && warp == 1) {
        if (leader) {
            // ---------------- MMA issuer (rank 0 only): the whole warp, its elected
            // lane carries each instruction
            const uint32_t issuer = elect_one_sync();
            constexpr uint32_t idesc_wide = mma_idesc_bf16(kPairM, kPairN, A_MN, B_MN);
            constexpr uint32_t idesc_narrow = mma_idesc_bf16(kPairM, kHalf, A_MN, B_MN);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = pair; ok && u < num_units; u += npairs, ++it) {
                const int pi = problem_of(G, u);
                const KParams& p = G.kp[pi];
                const Unit w = unit_of<SPLIT>(p, u - G.unit_begin[pi]);
                const int acc = it % NACC;
                const uint32_t aph = static_cast<uint32_t>(it / NACC) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait_cluster_fast(tempty_bar(acc), aph ^ 1u, status, kSiteMmaTmemEmpty)))
                    break;
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kPairN);
                const uint32_t idesc = w.narrow ? idesc_narrow : idesc_wide;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!__all_sync(0xffffffffu, mbar_wait_cluster_fast(full_bar(stage), phase, status, kSiteMmaFull))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = s_a + stage * kPairAStage;
                    const uint32_t b0 = s_b + stage * kPairBStage;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = A_MN ? smem_desc_sw128(a0 + k * 2048, mn_lbo, mn_sbo)
                                                 : smem_desc_sw128(a0 + k * 32, 16, 1024);
                        const uint64_t bd = B_MN ? smem_desc_sw128(b0 + k * 2048, mn_lbo, mn_sbo)
                                                 : smem_desc_sw128(b0 + k * 32, 16, 1024);
                        umma_bf16_pair_elected(issuer, d, ad, bd, idesc, (kb != w.kb0 || k != 0) ? 1u : 0u);
                    }
                    umma_commit_pair_elected(issuer, empty_bar(stage), 0x3);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_elected(issuer, tfull_bar(acc), 0x3);
            }
            umma_commit_pair_elected(issuer, drain_bar, 0x1);
            mbar_wait(drain_bar, 0, status, kSiteDrain, kWaitLimitNs);
        }
    } else if (usable && warp >= 2) {
        // ---------------- epilogue (both CTAs): warp w reads lanes 32 (w % 4) .. +31
        constexpr bool kSide = !kTmaOut;  // SwiGLU backward: side inputs by TMA into a ring
        constexpr int kChunks = kPairN / 32;
        const int q = warp & 3;
        const int row = q * 32 + lane;
        constexpr uint32_t kSetBytes = pair_boxes_per_set<EPI>() * kBoxBytes;
        const uint32_t out_stage = s_out + static_cast<uint32_t>(q) * pair_out_sets<EPI>() * kSetBytes;
        uint32_t n_stored = 0;  // staged chunks this warp has handed to TMA stores
        // Side-input ring (SwiGLU backward): chunk k of this warp is column
        // chunk k % 8 of its (k / 8)-th work unit; lane 0 requests the g and u
        // boxes of its 32 rows into slot k % kSideSlots, kSideSlots - 1 chunks
        // ahead (across units: side inputs do not depend on the accumulator).
        const uint32_t ring = s_out + static_cast<uint32_t>(q) * (kSideSlots * kSideSlotBytes);
        auto side_bar = [&](int slot) { return side_bars + 8u * static_cast<uint32_t>(q * kSideSlots + slot); };
        const int my_units = pair < num_units ? (num_units - 1 - pair) / npairs + 1 : 0;
        const int n_chunks = kSide ? my_units * kChunks : 0;
        auto issue_side = [&](int k) {
            const int u = pair + (k / kChunks) * npairs;
            const int pi = problem_of(G, u);
            const KParams& p = G.kp[pi];
            const Unit w = unit_of<SPLIT>(p, u - G.unit_begin[pi]);
            int tm, tn;
            tile_coords(p, w.tile, tm, tn);
            const int n = tn * kPairN + (k % kChunks) * 32;
            const int row0 = tm * kPairM + static_cast<int>(rank) * kHalf + q * 32;
            const uint32_t slot = ring + static_cast<uint32_t>(k % kSideSlots) * kSideSlotBytes;
            const uint32_t bar = side_bar(k % kSideSlots);
            mbar_arrive_expect_tx(bar, kSideSlotBytes);
            tma_load_2d(slot, &G.xmap[0], bar, n, row0);
            tma_load_2d(slot + kBf16BoxBytes, &G.xmap[1], bar, n, row0);
        };
        int issued = 0;  // chunks whose side inputs lane 0 has requested
        int k = 0;       // chunks this warp has consumed
        if (kSide && lane == 0)
            for (; issued < kSideSlots - 1 && issued < n_chunks; ++issued) issue_side(issued);
        bool alive = true;
        int it = 0;
        for (int u = pair; alive && u < num_units; u += npairs, ++it) {
            const int pi = problem_of(G, u);
            const KParams& p = G.kp[pi];
            const Unit w = unit_of<SPLIT>(p, u - G.unit_begin[pi]);
            const int acc = it % NACC;
            const uint32_t aph = static_cast<uint32_t>(it / NACC) & 1u;
            // one verdict per warp: the tensor-memory loads below are warp-wide
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(tfull_bar(acc), aph, status, kSiteEpiTmemFull)))
                break;
            tc_fence_after();
            int tm, tn;
            tile_coords(p, w.tile, tm, tn);
            const int trow = static_cast<int>(rank) * kHalf + row;  // row inside the 256-row tile
            const int m = tm * kPairM + trow;
            const int row0 = m - lane;  // first row of this warp's 32
            // a narrow unit's accumulator is its first 128 columns
            const int n_base = tn * kPairN + (w.narrow ? w.nh * kHalf : 0);
            const int unit_chunks = w.narrow ? kChunks / 2 : kChunks;
            const bool row_ok = m < p.m;
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kPairN);
            // K split: per warp (32 rows of the tile), the half whose
            // accumulator is ready first stores it as float32 partial rows and
            // marks them written; the other half adds them to its own and runs
            // the epilogue.  Which half is first does not change the result
            // (p0 + p1 == p1 + p0).  The decision is taken once per warp, by
            // lane 0, because the tensor-memory loads below are warp-wide; the
            // second half waits only on a warp that is already past its MMAs
            // and has no waits left before it marks the rows.
            bool store_partial = false;
            bool give_up = false;
            uint32_t* flag = nullptr;
            const size_t split_slot = SPLIT && w.split ? static_cast<size_t>(w.tile - p.split_from) : 0;
            const float* prow =
                SPLIT && w.split ? p.partial + (split_slot * kPairM + static_cast<size_t>(trow)) * kPairN : nullptr;
            if (SPLIT && w.split) {
                flag = p.flags + split_slot * 8 + rank * 4 + static_cast<uint32_t>(q);
                const uint32_t claimed = 2u * p.epoch;
                uint32_t old = 0;
                if (lane == 0) old = atom_exch_acq_rel(flag, claimed);
                old = __shfl_sync(0xffffffffu, old, 0);
                store_partial = old != claimed && old != claimed + 1u;
                if (old == claimed) {
                    int ready = 1;
                    if (lane == 0) ready = wait_value(flag, claimed + 1u, status, kSiteSplitFlag) ? 1 : 0;
                    give_up = __shfl_sync(0xffffffffu, ready, 0) == 0;
                }
                __syncwarp();  // the partial rows read below come after lane 0's acquire
            }
            const bool run_epi = row_ok && !store_partial && !give_up;
            if constexpr (EPI == static_cast<int>(Epilogue::SwigluFwd)) {
                // columns 0-127 of the accumulator are g, 128-255 u, of features
                // tn * 128 ...: four rounds of one 32-column g chunk and its u chunk
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t rg[32], ru[32];
                    tmem_load_32(tbase + static_cast<uint32_t>(c * 32), rg);
                    tmem_load_32(tbase + static_cast<uint32_t>(kHalf + c * 32), ru);
                    tmem_wait_load();
                    if (c == 3) {
                        tc_fence_before();
                        if (leader)
                            mbar_arrive(tempty_bar(acc));
                        else
                            mbar_arrive_cluster(map_to_cta(tempty_bar(acc), 0));
                    }
                    if (SPLIT && store_partial) {
                        float4* dg = reinterpret_cast<float4*>(const_cast<float*>(prow) + c * 32);
                        float4* du = reinterpret_cast<float4*>(const_cast<float*>(prow) + kHalf + c * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            dg[j] = make_float4(__uint_as_float(rg[4 * j]), __uint_as_float(rg[4 * j + 1]),
                                                __uint_as_float(rg[4 * j + 2]), __uint_as_float(rg[4 * j + 3]));
                            du[j] = make_float4(__uint_as_float(ru[4 * j]), __uint_as_float(ru[4 * j + 1]),
                                                __uint_as_float(ru[4 * j + 2]), __uint_as_float(ru[4 * j + 3]));
                        }
                        continue;
                    }
                    if (SPLIT && w.split && run_epi) {
                        const float4* sg = reinterpret_cast<const float4*>(prow + c * 32);
                        const float4* su = reinterpret_cast<const float4*>(prow + kHalf + c * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 vg = sg[j], vu = su[j];
                            rg[4 * j] = __float_as_uint(__uint_as_float(rg[4 * j]) + vg.x);
                            rg[4 * j + 1] = __float_as_uint(__uint_as_float(rg[4 * j + 1]) + vg.y);
                            rg[4 * j + 2] = __float_as_uint(__uint_as_float(rg[4 * j + 2]) + vg.z);
                            rg[4 * j + 3] = __float_as_uint(__uint_as_float(rg[4 * j + 3]) + vg.w);
                            ru[4 * j] = __float_as_uint(__uint_as_float(ru[4 * j]) + vu.x);
                            ru[4 * j + 1] = __float_as_uint(__uint_as_float(ru[4 * j + 1]) + vu.y);
                            ru[4 * j + 2] = __float_as_uint(__uint_as_float(ru[4 * j + 2]) + vu.z);
                            ru[4 * j + 3] = __float_as_uint(__uint_as_float(ru[4 * j + 3]) + vu.w);
                        }
                    }
                    // the TMA drops rows >= M; every column is a feature below ffn
                    if (!give_up && row0 < p.m) {
                        // the set is rewritten only after the previous round's
                        // stores have finished reading it
                        const uint32_t set = out_stage;
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
                        if (run_epi) swiglu_fwd_chunk_to_smem(set, lane, rg, ru);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const int col = tn * kHalf + c * 32;
                            tma_store_2d(&G.omap[pi], set, col, row0);
                            tma_store_2d(&G.omap[pi], set + kBf16BoxBytes, p.ffn + col, row0);
                            tma_store_2d(&G.xmap[0], set + 2 * kBf16BoxBytes, col, row0);
                            bulk_commit_group();
                        }
                        ++n_stored;
                    }
                }
            } else {
                float row_dot = 0.f;  // row-dot epilogue: this row's sum over the current column group
    #pragma unroll 1
                for (int c = 0; c < unit_chunks; ++c) {
                    const int n = n_base + c * 32;
                    const bool ok = run_epi && n < p.n;
                    uint4 x0[4];
                    if constexpr (EPI == static_cast<int>(Epilogue::AddResidual) ||
                                  EPI == static_cast<int>(Epilogue::StoreBf16RowDot)) {
                        if (ok) {
                            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.aux) +
                                                                              static_cast<int64_t>(m) * p.ld_aux + n);
    #pragma unroll
                            for (int j = 0; j < 4; ++j) x0[j] = src[j];
                        }
                    }
                    if constexpr (kSide) {
                        const uint32_t sb = side_bar(k % kSideSlots);
                        const uint32_t sph = static_cast<uint32_t>(k / kSideSlots) & 1u;
                        if (!__all_sync(0xffffffffu, mbar_wait(sb, sph, status, kSiteEpiSideInput))) {
                            alive = false;
                            break;
                        }
                    }
                    uint32_t r[32];
                    tmem_load_32(tbase + static_cast<uint32_t>(c * 32), r);
                    tmem_wait_load();
                    if (c == unit_chunks - 1) {
                        tc_fence_before();
                        if (leader)
                            mbar_arrive(tempty_bar(acc));
                        else
                            mbar_arrive_cluster(map_to_cta(tempty_bar(acc), 0));
                    }
                    bool stored = false;
                    if (SPLIT && store_partial) {
                        float4* dst = reinterpret_cast<float4*>(const_cast<float*>(prow) + c * 32);
    #pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    } else {
                        if (SPLIT && w.split && ok) {
                            const float4* src = reinterpret_cast<const float4*>(prow + c * 32);
    #pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 v = src[j];
                                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + v.x);
                                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + v.y);
                                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + v.z);
                                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + v.w);
                            }
                        }
                        if constexpr (EPI == static_cast<int>(Epilogue::StoreBf16RowDot)) {
                            // a column group never crosses a unit (128 divides
                            // n_base and is a multiple of dot_cols), so its
                            // chunks are all this thread's, in order
                            if (ok) row_dot += row_dot_bf16(r, x0);
                            if ((n + 32) % p.dot_cols == 0) {
                                if (ok) p.dot[static_cast<int64_t>(n / p.dot_cols) * p.ld_dot + m] = row_dot;
                                row_dot = 0.f;
                            }
                        }
                        // The box is stored when any of the warp's rows lies inside
                        // M (the TMA drops rows >= M and columns >= N); the
                        // decision is warp-uniform.
                        stored = !give_up && row0 < p.m && n < p.n;
                        if (stored) {
                            if constexpr (kSide) {
                                const uint32_t slot = ring + static_cast<uint32_t>(k % kSideSlots) * kSideSlotBytes;
                                if (ok) swiglu_chunk_in_smem(slot, lane, r);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_2d(&G.xmap[2], slot, n, row0);
                                    tma_store_2d(&G.xmap[3], slot + kBf16BoxBytes, n, row0);
                                    bulk_commit_group();
                                }
                            } else {
                                // a box is rewritten only after the store that read
                                // it, two chunks back, has finished reading
                                const uint32_t box = out_stage + (n_stored & 1u) * kBoxBytes;
                                if (lane == 0) bulk_wait_group_read<1>();
                                __syncwarp();
                                if (ok) epilogue_chunk_to_smem<EPI>(box, lane, r, x0);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    if constexpr (EPI == static_cast<int>(Epilogue::AccumF32))
                                        tma_reduce_add_2d(&G.omap[pi], box, n, row0);
                                    else
                                        tma_store_2d(&G.omap[pi], box, n, row0);
                                    bulk_commit_group();
                                }
                                ++n_stored;
                            }
                        }
                    }
                    if constexpr (kSide) {
                        // Refill the slot chunk k - 1 used, once the stores that
                        // read it are done (all but this chunk's own group).
                        if (lane == 0 && issued < n_chunks) {
                            if (stored)
                                bulk_wait_group_read<1>();
                            else
                                bulk_wait_group_read<0>();
                            issue_side(issued);
                            ++issued;
                        }
                        ++k;
                    }
                }
            }
            if (SPLIT && store_partial && alive) {
                __syncwarp();  // every lane's partial rows before lane 0's release
                if (lane == 0) {
                    __threadfence();
                    st_release(flag, 2u * p.epoch + 1u);
                }
            }
        }
        // The staging boxes and the ring must stay until the last stores have
        // read them, and side inputs still in flight (after a wait gave up)
        // must land before the CTA leaves.
        if (lane == 0) {
            bulk_wait_group_all();
            for (; k < issued; ++k)
                mbar_drain(side_bar(k % kSideSlots), static_cast<uint32_t>(k / kSideSlots) & 1u, kWaitLimitNs);
        }
    }

    tc_fence_before();
    cluster_sync_all();  // neither CTA leaves while the other may still signal it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Row-major bf16 matrix of `rows` x `cols` with row stride `ld` elements,
// boxes of box_cols x box_rows, zero fill out of range (loads) and no writes
// out of range (stores).  Operand boxes take the 128-byte swizzle of the MMA
// descriptors; output boxes (32 x 32) the 64-byte swizzle of the staging boxes.
// Loads promote to 256-byte L2 fills, except the SwiGLU side inputs (64-byte
// box rows): 128-byte fills made that dgrad 3 % faster on GB300 (325.4 ->
// 315.6 us) for the same DRAM bytes.
bool encode_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld,
                uint32_t box_cols, uint32_t box_rows,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t esize = dtype == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool A_MN, bool B_MN, int EPI>
cudaError_t launch_variant(const CUtensorMap& ma, const CUtensorMap& mb, const KParams& p,
                           cudaStream_t stream) {
    auto kern = gemm_kernel<BN, A_MN, B_MN, EPI>;
    constexpr size_t smem = Cfg<BN>::kSmemBytes;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int grid = p.num_tiles < sm_count() ? p.num_tiles : sm_count();
    kern<<<grid, kThreads, smem, stream>>>(ma, mb, p);
    return cudaGetLastError();
}

// Accumulators per CTA pair: two 256-column f32 accumulators (all 512 tensor-
// memory columns) let the epilogue of one tile overlap the MMAs of the next.
// The pair allocation is collective: both CTAs receive the same columns (the
// kernel checks this and reports kSitePairTmem otherwise).
constexpr int kPairAccums = 2;

static_assert(sizeof(PairGroup) <= 32000, "kernel parameter space");

template <bool A_MN, bool B_MN, int EPI, bool SPLIT>
cudaError_t launch_pair_split_variant(const PairGroup& G, cudaStream_t stream) {
    auto kern = gemm_pair_kernel<A_MN, B_MN, EPI, kPairAccums, SPLIT>;
    constexpr size_t kSmem = pair_smem_bytes<EPI>();
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int max_clusters = 0;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmem));
        if (attr_err != cudaSuccess) return;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(sm_count()));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
    });
    if (attr_err != cudaSuccess) return attr_err;
    if (max_clusters < 1) return cudaErrorInvalidConfiguration;
    const int units = G.unit_begin[G.n_probs];
    const int pairs = units < max_clusters ? units : max_clusters;
    kern<<<2 * pairs, kThreads, kSmem, stream>>>(G);
    return cudaGetLastError();
}

template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_pair_variant(const PairGroup& G, cudaStream_t stream) {
    return G.kp[0].split == 2 ? launch_pair_split_variant<A_MN, B_MN, EPI, true>(G, stream)
                              : launch_pair_split_variant<A_MN, B_MN, EPI, false>(G, stream);
}

// DRAM bytes a raster fetches, modelled wave by wave: a wave reads the A
// panels (one tile row over all of K) and B panels (one tile column) of its
// tiles; panels of the previous wave are still in L2 if that wave's panels fit.
double raster_cost(int tiles_m, int tiles_n, double panel_a, double panel_b, int grid, int group, bool group_m,
                   double l2_bytes) {
    KParams q{};
    q.tiles_m = tiles_m;
    q.tiles_n = tiles_n;
    q.group = group;
    q.group_m = group_m ? 1 : 0;
    const int total = tiles_m * tiles_n;
    std::vector<char> pm(tiles_m, 0), pn(tiles_n, 0), cm(tiles_m), cn(tiles_n);
    double prev_bytes = 0.0, cost = 0.0;
    for (int w0 = 0; w0 < total; w0 += grid) {
        std::fill(cm.begin(), cm.end(), 0);
        std::fill(cn.begin(), cn.end(), 0);
        for (int t = w0; t < std::min(total, w0 + grid); ++t) {
            int tm, tn;
            if (q.group_m) {
                const int per = group * tiles_n, g = t / per, in = t - g * per;
                const int rows = std::min(group, tiles_m - g * group);
                tm = g * group + in % rows;
                tn = in / rows;
            } else {
                const int per = group * tiles_m, g = t / per, in = t - g * per;
                const int cols = std::min(group, tiles_n - g * group);
                tn = g * group + in % cols;
                tm = in / cols;
            }
            cm[tm] = 1;
            cn[tn] = 1;
        }
        const bool kept = prev_bytes <= l2_bytes;
        double bytes = 0.0;
        for (int i = 0; i < tiles_m; ++i)
            if (cm[i]) {
                bytes += panel_a;
                if (!kept || !pm[i]) cost += panel_a;
            }
        for (int j = 0; j < tiles_n; ++j)
            if (cn[j]) {
                bytes += panel_b;
                if (!kept || !pn[j]) cost += panel_b;
            }
        pm.swap(cm);
        pn.swap(cn);
        prev_bytes = bytes;
    }
    return cost;
}

struct Raster {
    int group;
    bool group_m;
};

Raster choose_raster(int tiles_m, int tiles_n, int bm, int bn, int k, int grid) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, int>, Raster> cache;
    const auto key = std::make_tuple(tiles_m, tiles_n, bm, bn, k, grid);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const double pa = 2.0 * bm * k, pb = 2.0 * bn * k;
    const double l2 = 64.0 * 1024 * 1024;  // about half of the 129 MB L2
    Raster best{tiles_m, true};             // plain m-fastest order
    double best_cost = raster_cost(tiles_m, tiles_n, pa, pb, grid, tiles_m, true, l2);
    for (int g = 1; g < 256; g *= 2) {
        if (g < tiles_m) {
            const double c = raster_cost(tiles_m, tiles_n, pa, pb, grid, g, true, l2);
            if (c < best_cost * 0.98) best = {g, true}, best_cost = c;
        }
        if (g < tiles_n) {
            const double c = raster_cost(tiles_m, tiles_n, pa, pb, grid, g, false, l2);
            if (c < best_cost * 0.98) best = {g, false}, best_cost = c;
        }
    }
    cache.emplace(key, best);
    return best;
}

template <int BN>
cudaError_t dispatch(const GemmArgs& g, const CUtensorMap& ma, const CUtensorMap& mb, KParams& p,
                     cudaStream_t stream) {
    constexpr int kStore = static_cast<int>(Epilogue::StoreBf16);
    constexpr int kResid = static_cast<int>(Epilogue::AddResidual);
    constexpr int kSwiglu = static_cast<int>(Epilogue::SwigluBwd);
    constexpr int kAccum = static_cast<int>(Epilogue::AccumF32);
    switch (g.kind) {
        case GemmKind::Forward:
            if (g.epi == Epilogue::StoreBf16) return launch_variant<BN, false, false, kStore>(ma, mb, p, stream);
            if (g.epi == Epilogue::AddResidual) return launch_variant<BN, false, false, kResid>(ma, mb, p, stream);
            break;
        case GemmKind::BackwardInput:
            if (g.epi == Epilogue::StoreBf16) return launch_variant<BN, false, true, kStore>(ma, mb, p, stream);
            if (g.epi == Epilogue::SwigluBwd) return launch_variant<BN, false, true, kSwiglu>(ma, mb, p, stream);
            break;
        case GemmKind::BackwardWeight:
            if (g.epi == Epilogue::AccumF32) return launch_variant<BN, true, true, kAccum>(ma, mb, p, stream);
            break;
    }
    return cudaErrorInvalidValue;
}

cudaError_t dispatch_pair(const GemmArgs& g, const PairGroup& G, cudaStream_t stream) {
    constexpr int kStore = static_cast<int>(Epilogue::StoreBf16);
    constexpr int kResid = static_cast<int>(Epilogue::AddResidual);
    constexpr int kSwiglu = static_cast<int>(Epilogue::SwigluBwd);
    constexpr int kAccum = static_cast<int>(Epilogue::AccumF32);
    constexpr int kSwigluFwd = static_cast<int>(Epilogue::SwigluFwd);
    constexpr int kRowDot = static_cast<int>(Epilogue::StoreBf16RowDot);
    switch (g.kind) {
        case GemmKind::Forward:
            if (g.epi == Epilogue::StoreBf16) return launch_pair_variant<false, false, kStore>(G, stream);
            if (g.epi == Epilogue::AddResidual) return launch_pair_variant<false, false, kResid>(G, stream);
            if (g.epi == Epilogue::SwigluFwd) return launch_pair_variant<false, false, kSwigluFwd>(G, stream);
            break;
        case GemmKind::BackwardInput:
            if (g.epi == Epilogue::StoreBf16) return launch_pair_variant<false, true, kStore>(G, stream);
            if (g.epi == Epilogue::SwigluBwd) return launch_pair_variant<false, true, kSwiglu>(G, stream);
            if (g.epi == Epilogue::StoreBf16RowDot) return launch_pair_variant<false, true, kRowDot>(G, stream);
            break;
        case GemmKind::BackwardWeight:
            if (g.epi == Epilogue::AccumF32) return launch_pair_variant<true, true, kAccum>(G, stream);
            break;
    }
    return cudaErrorInvalidValue;
}

// Clusters of the CTA-pair kernel that fit on the current device at once (the
// same for every variant: same threads and cluster shape, and every variant's
// shared memory allows one CTA per SM).
int pair_max_clusters() {
    static int counts[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!counts[dev]) {
        constexpr int kStore = static_cast<int>(Epilogue::StoreBf16);
        auto kern = gemm_pair_kernel<false, true, kStore, kPairAccums, false>;
        constexpr size_t kSmem = pair_smem_bytes<kStore>();
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem)) !=
            cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(sm_count()));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

// Each K-split launch tags the flags it writes with a new epoch, so the flags
// never need clearing between launches.
std::atomic<uint32_t> g_split_epoch{0};

// Shortest K half (in 64-element blocks) of a split tile.
constexpr int kMinHalfKBlocks = 48;

}  // namespace

namespace {

// Tensor maps and kernel parameters of one GEMM; `pair` says which kernel
// takes it.  A K split is considered only when `allow_split`.
cudaError_t prepare(const GemmArgs& g, bool allow_split, CUtensorMap& ma, CUtensorMap& mb, CUtensorMap& mo,
                    CUtensorMap* mx, KParams& p, bool& pair) {
    const int sms = sm_count();
    // A CTA pair takes 256 x 256 tiles; small outputs keep the one-CTA kernel.
    pair = gemm_takes_pair(g.m, g.n);
    const int tile_m = pair ? kPairM : BM;
    const int tile_n = pair ? kPairN : kBN;
    const uint32_t b_rows = pair ? kHalf : kBN;  // rows of a K-major B box
    bool ok = true;
    switch (g.kind) {
        case GemmKind::Forward:
            ok = encode_map(&ma, g.a, g.m, g.k, g.lda, 64, BM) && encode_map(&mb, g.b, g.n, g.k, g.ldb, 64, b_rows);
            break;
        case GemmKind::BackwardInput:
            ok = encode_map(&ma, g.a, g.m, g.k, g.lda, 64, BM) && encode_map(&mb, g.b, g.k, g.n, g.ldb, 64, BK);
            break;
        case GemmKind::BackwardWeight:
            ok = encode_map(&ma, g.a, g.k, g.m, g.lda, 64, BK) && encode_map(&mb, g.b, g.k, g.n, g.ldb, 64, BK);
            break;
    }
    // Output of the CTA-pair kernel's TMA stores (bf16) and reduce-adds (float32).
    if (ok && pair &&
        (g.epi == Epilogue::StoreBf16 || g.epi == Epilogue::AddResidual || g.epi == Epilogue::StoreBf16RowDot))
        ok = encode_map(&mo, g.out, g.m, g.n, g.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    // Row dots: every column group lies inside one 128-column half of a tile
    // (so inside one work unit, wide or narrow), and the per-row reads of aux
    // are 16-byte loads.
    if (g.epi == Epilogue::StoreBf16RowDot &&
        (!pair || g.kind != GemmKind::BackwardInput || !g.aux || !g.dot || g.ld_dot < g.m ||
         (g.dot_cols != 32 && g.dot_cols != 64 && g.dot_cols != 128) || g.n % g.dot_cols != 0 || g.ld_aux < g.n ||
         g.ld_aux % 8 != 0 || reinterpret_cast<uintptr_t>(g.aux) % 16 != 0))
        return cudaErrorInvalidValue;
    if (ok && pair && g.epi == Epilogue::AccumF32)
        ok = encode_map(&mo, g.out, g.m, g.n, g.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
    // SwiGLU backward of the CTA-pair kernel: g and u (loaded) and dg and du
    // (stored), each [M, ffn] inside a row of 2 ffn, 32 x 32 boxes.
    if (ok && pair && g.epi == Epilogue::SwigluBwd) {
        if (!mx) return cudaErrorInvalidValue;
        const uint16_t* aux = static_cast<const uint16_t*>(g.aux);
        uint16_t* out = static_cast<uint16_t*>(g.out);
        constexpr auto kBf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        constexpr auto kFill128 = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
        ok = encode_map(&mx[0], aux, g.m, g.n, g.ld_aux, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, kBf16, kFill128) &&
             encode_map(&mx[1], aux + g.ffn, g.m, g.n, g.ld_aux, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, kBf16,
                        kFill128) &&
             encode_map(&mx[2], out, g.m, g.n, g.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_map(&mx[3], out + g.ffn, g.m, g.n, g.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    }
    // SwiGLU forward (CTA-pair kernel only): [g | u] out through the output map,
    // s through the first extra map, 32 x 32 boxes each; each 256-column tile
    // holds 128 features of g and the same 128 of u.
    if (g.epi == Epilogue::SwigluFwd) {
        if (!pair || !mx || g.kind != GemmKind::Forward || g.ffn <= 0 || g.ffn % kHalf != 0 || g.n != 2 * g.ffn ||
            !g.out2)
            return cudaErrorInvalidValue;
        ok = ok && encode_map(&mo, g.out, g.m, g.n, g.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_map(&mx[0], g.out2, g.m, g.ffn, g.ldo2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    }
    if (!ok) return cudaErrorInvalidValue;
    p = KParams{};
    p.m = g.m;
    p.n = g.n;
    p.k = g.k;
    p.tiles_m = (g.m + tile_m - 1) / tile_m;
    p.tiles_n = (g.n + tile_n - 1) / tile_n;
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.k_blocks = (g.k + BK - 1) / BK;
    p.split = 1;
    p.split_from = p.num_tiles;
    p.kb_split = p.k_blocks;
    p.narrow_from = p.num_tiles;
    p.num_units = p.num_tiles;
    // K split of the last wave: when the tiles left over after the full waves
    // of CTA pairs would keep at most half of the pairs busy, each of those
    // tiles becomes two half-K units, so the last round costs half a tile
    // instead of a whole one (a 4096 x 4096 output is 256 tiles: on 76 pairs
    // three full waves and 28 split tiles, 3.5 tile times instead of 4).  Only
    // the split tiles exchange float32 partials.  Halves keep at least 48 k-blocks: on GB300 (ncu) the split
    // gained 3 % at K = 6144 (146 -> 141 us), 8 % at K = 14336 (320 -> 294 us)
    // and 6 % at K = 28672 against splitting every tile (610 -> 575 us), while
    // at K = 4096 the exchange of partials cost what the half tile saved.
    // Only with caller scratch.
    if (allow_split && pair && g.split_flags && g.split_partial && p.k_blocks >= 2 * kMinHalfKBlocks) {
        const int pairs = pair_max_clusters();
        const int rem = pairs > 0 ? p.num_tiles % pairs : 0;
        if (rem > 0 && 2 * rem <= pairs && rem <= g.split_tiles && rem <= kSplitMaxTiles) {
            p.split = 2;
            p.split_from = p.num_tiles - rem;
            p.kb_split = p.k_blocks / 2;
            p.num_units = p.split_from + 2 * rem;
            p.flags = g.split_flags;
            p.partial = g.split_partial;
            p.epoch = ++g_split_epoch;
        }
    }
    // Otherwise the same short last wave is split along N: each leftover tile
    // becomes two 256 x 128 units over the whole K (no partials to exchange;
    // each output element takes the same K steps in the same order, so the
    // results are the wide tile's bits).  Plain stores and float32 reduce-adds
    // only (the SwiGLU epilogues pair columns across a full tile).  On GB300,
    // at 4096 tokens: B of the O projection (K 4096) 98.3 -> 93.1 us, F of the
    // QKV projection 141.0 -> 134.4 us, F of the O projection with its
    // residual 105.1 -> 96.6 us.
    if (allow_split && pair && p.split == 1 &&
        (g.epi == Epilogue::StoreBf16 || g.epi == Epilogue::AddResidual || g.epi == Epilogue::AccumF32 ||
         g.epi == Epilogue::StoreBf16RowDot)) {
        const int pairs = pair_max_clusters();
        const int rem = pairs > 0 ? p.num_tiles % pairs : 0;
        if (rem > 0 && 2 * rem <= pairs) {
            p.narrow_from = p.num_tiles - rem;
            p.num_units = p.narrow_from + 2 * rem;
        }
    }
    const int waves_of = pair ? sms / 2 : sms;
    const Raster r = choose_raster(p.tiles_m, p.tiles_n, tile_m, tile_n, g.k, std::min(p.num_tiles, waves_of));
    p.group = r.group;
    p.group_m = r.group_m ? 1 : 0;
    p.out = g.out;
    p.ldo = g.ldo;
    p.aux = g.aux;
    p.ld_aux = g.ld_aux;
    p.ffn = g.ffn;
    p.dot = g.dot;
    p.ld_dot = g.ld_dot;
    p.dot_cols = g.dot_cols;
    p.status = status_word();
    p.mn_lbo = kMnBlockBytes;
    p.mn_sbo = 1024;
    if (!p.status) return cudaErrorInvalidDevice;
    return cudaSuccess;
}

}  // namespace

bool gemm_takes_pair(int m, int n) { return m >= kPairM && n >= kPairN; }

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream) {
    if (g.m <= 0 || g.n <= 0 || g.k <= 0) return cudaSuccess;
    CUtensorMap ma, mb, mo = {}, mx[4] = {};
    KParams p;
    bool pair = false;
    const cudaError_t e = prepare(g, true, ma, mb, mo, mx, p, pair);
    if (e != cudaSuccess) return e;
    if (!pair) return dispatch<kBN>(g, ma, mb, p, stream);
    PairGroup G;
    G.map[0] = ma;
    G.map[1] = mb;
    G.omap[0] = mo;
    for (int i = 0; i < 4; ++i) G.xmap[i] = mx[i];
    G.kp[0] = p;
    G.unit_begin[0] = 0;
    G.unit_begin[1] = p.num_units;
    G.n_probs = 1;
    return dispatch_pair(g, G, stream);
}

cudaError_t launch_gemm_group(const GemmArgs* gs, int n, cudaStream_t stream) {
    // One grouped launch when every GEMM takes the CTA-pair kernel with the
    // same layouts and epilogue; otherwise one launch each.  The SwiGLU
    // backward (side-input maps for one problem per launch) is never grouped.
    bool grouped = n > 1 && n <= kMaxGroup;
    for (int i = 0; grouped && i < n; ++i)
        grouped = gs[i].m >= kPairM && gs[i].n >= kPairN && gs[i].k > 0 && gs[i].kind == gs[0].kind &&
                  gs[i].epi == gs[0].epi && gs[i].epi != Epilogue::SwigluBwd && gs[i].epi != Epilogue::SwigluFwd;
    if (!grouped) {
        for (int i = 0; i < n; ++i) {
            const cudaError_t e = launch_gemm(gs[i], stream);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    PairGroup G;
    G.unit_begin[0] = 0;
    for (int i = 0; i < n; ++i) {
        bool pair = false;
        const cudaError_t e = prepare(gs[i], false, G.map[2 * i], G.map[2 * i + 1], G.omap[i], nullptr, G.kp[i], pair);
        if (e != cudaSuccess) return e;
        G.unit_begin[i + 1] = G.unit_begin[i] + G.kp[i].num_units;
    }
    G.n_probs = n;
    return dispatch_pair(gs[0], G, stream);
}

}  // namespace zbk
