// exact_select.cu -- exact block attention mass (pass 2 of the block-oracle selector).
//
// "Can sparse attention close the quality gap in diffusion transformers", section
// "质量差距有三个可分离来源": the oracles compared there keep, at the same density,
// the KV blocks that retain the most attention mass under the exact dense attention
// probabilities. With the dense row logsumexp LSE_r of pass 1 (bsa_forward over a
// full index), the mass of the block pair (i, j) is
//   mass_ij = sum over rows r of Q block i and keys c of KV block j of
//             exp(scale * q_r . k_c - LSE_r),
// and the selector keeps the top-k KV blocks of every Q block by mass (ties to the
// lower index, as the mean-pooled selector).
//
// This pass is a dense QK^T: per 128-row query tile, S = Q K_j^T for every KV block j
// on tcgen05 (fp32 accumulators in TMEM); one thread per row sums
// p = 2^(s * scale * log2 e - LSE_r * log2 e) over the block's columns, the warp sums
// its 32 rows, and lane 0 writes one partial per (warp, KV block). The selection
// kernel adds a Q block's partials in a fixed order. Warp roles: 4 mass warps, a TMA
// producer warp and a QK^T issuer warp (converged, one elected issuing lane); every
// wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"
#include "sync.cuh"

namespace bsa {
namespace {

constexpr int kMTile = 128;
constexpr int kMassWarps = 4, kMassProducer = 4, kMassIssuer = 5, kMassThreads = 6 * 32;

struct MassParams {
    int N, nKB, tiles_per_bh, n_tiles;
    int last_rows;     // keys in the last KV block (fewer than BS for a ragged sequence)
    float scale_log2;
    const float *LSE;  // [B*H*N] dense logsumexp, natural log
    float *part;       // [n_tiles][4][nKB] partial masses (one per mass warp and KV block)
    uint32_t *err;
    unsigned long long wait_limit_ns;
};

template <int D, int BS, int NK, int NSB>
struct MassCfg {
    static constexpr int kQBytes = kMTile * D * 2;
    static constexpr int kKBytes = BS * D * 2;
    static constexpr int kQChunk = kMTile * 128;  // one 64-column swizzled slab of Q
    static constexpr int kKChunk = BS * 128;      // one 64-column swizzled slab of a K block
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + kQBytes;
    static constexpr int BAR_OFF = K_OFF + NK * kKBytes;
    static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + NK;
    static constexpr int B_SFULL = B_KEMPTY + NK, B_SEMPTY = B_SFULL + NSB, B_DRAIN = B_SEMPTY + NSB;
    static constexpr int NBAR = B_DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int SMEM = MISC_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;  // manual 1024-byte alignment
    static constexpr int TCOLS = NSB * BS <= 128 ? 128 : (NSB * BS <= 256 ? 256 : 512);
    static constexpr uint32_t IDESC = idesc_bf16_f32(kMTile, BS, 0, 0);
};

template <int D, int BS, int NK, int NSB>
__global__ void __launch_bounds__(kMassThreads, 2)
    mass_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK, const MassParams p)
{
    using C = MassCfg<D, BS, NK, NSB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int idx) -> uint32_t { return sbase + C::BAR_OFF + 8u * idx; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);  // [0] TMEM base, [1] abort flag
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_QEMPTY), 1);
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
        }
        for (int b = 0; b < NSB; ++b) {
            mbar_init(bar(C::B_SFULL + b), 1);
            mbar_init(bar(C::B_SEMPTY + b), kMassWarps);
        }
        mbar_init(bar(C::B_DRAIN), 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == kMassIssuer) {
        tmem_alloc(smem_u32(misc), C::TCOLS);
        tmem_relinquish();
    }
    if (warp == kMassProducer && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const Ctl ctl{reinterpret_cast<volatile uint32_t *>(misc + 1), p.err, p.wait_limit_ns};

    if (warp == kMassProducer) {
        // ------------------------------------------------------------ TMA producer
        int G = 0, e = 0, last_k = -1, q_issued = -1;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.n_tiles; tile += gridDim.x, ++e) {
            const int64_t bh = tile / p.tiles_per_bh;
            const int qt = tile % p.tiles_per_bh;
            // the single Q slot was last read by the previous tile's QK^T
            if (e >= 1 && !warp_wait_all(bar(C::B_QEMPTY), (e - 1) & 1, ctl)) break;
            __syncwarp();
            if (elect_one()) {
                mbar_arrive_expect_tx(bar(C::B_QFULL), C::kQBytes);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sbase + C::Q_OFF + c * C::kQChunk, &tmQ, c * 64, qt * kMTile, static_cast<int>(bh),
                                bar(C::B_QFULL));
            }
            __syncwarp();
            q_issued = e;
            for (int j = 0; j < p.nKB; ++j, ++G) {
                const int s = G % NK;
                // K slot s was last read by the QK^T of step G - NK
                if (G >= NK && !warp_wait_all(bar(C::B_KEMPTY + s), ((G / NK) - 1) & 1, ctl)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                if (elect_one()) {
                    mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::kKBytes);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_3d(sbase + C::K_OFF + s * C::kKBytes + c * C::kKChunk, &tmK, c * 64, j * BS,
                                    static_cast<int>(bh), bar(C::B_KFULL + s));
                }
                __syncwarp();
                last_k = G;
            }
        }
        if (lane == 0 && *ctl.abort_flag) {
            // never leave while our copies may still land in shared memory
            for (int g = last_k - NK + 1; g <= last_k; ++g)
                if (g >= 0) wait_bar_drain(bar(C::B_KFULL + g % NK), (g / NK) & 1, p.wait_limit_ns);
            if (q_issued >= 0) wait_bar_drain(bar(C::B_QFULL), q_issued & 1, p.wait_limit_ns);
        }
        __syncwarp();
    } else if (warp == kMassIssuer) {
        // ------------------------------------------------------------ QK^T issuer
        const uint64_t qdesc = sdesc_sw128(sbase + C::Q_OFF, 16, 1024);
        const uint64_t kdesc0 = sdesc_sw128(sbase + C::K_OFF, 16, 1024);
        int G = 0, e = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.n_tiles; tile += gridDim.x, ++e) {
            if (!warp_wait_all(bar(C::B_QFULL), e & 1, ctl)) break;
            tc_fence_after();
            for (int j = 0; j < p.nKB; ++j, ++G) {
                const int s = G % NK, b = G % NSB;
                if (!warp_wait_all(bar(C::B_KFULL + s), (G / NK) & 1, ctl)) {
                    ok = false;
                    break;
                }
                // S buffer b was last read by the mass warps at step G - NSB
                if (G >= NSB && !warp_wait_all(bar(C::B_SEMPTY + b), ((G / NSB) - 1) & 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t kdesc = kdesc0 + static_cast<uint64_t>(s * (C::kKBytes >> 4));
                __syncwarp();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off_q = static_cast<uint64_t>(((kk >> 2) * C::kQChunk + (kk & 3) * 32) >> 4);
                        const uint64_t off_k = static_cast<uint64_t>(((kk >> 2) * C::kKChunk + (kk & 3) * 32) >> 4);
                        mma_ss(tmem + b * BS, qdesc + off_q, kdesc + off_k, C::IDESC, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(C::B_SFULL + b));
                    tc_commit(bar(C::B_KEMPTY + s));
                }
                __syncwarp();
            }
            if (!ok) break;
            // the tile's last QK^T: the Q slot is free once these MMAs complete
            if (elect_one()) tc_commit(bar(C::B_QEMPTY));
            __syncwarp();
        }
        // all MMAs issued by the elected lane have completed before TMEM is freed
        __syncwarp();
        if (elect_one()) {
            tc_commit(bar(C::B_DRAIN));
            wait_bar_drain(bar(C::B_DRAIN), 0, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ mass warps (thread = row = TMEM lane)
        const uint32_t tS = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float log2e = 1.4426950408889634f;
        int G = 0;
        bool alive = true;
        for (int tile = blockIdx.x; alive && tile < p.n_tiles; tile += gridDim.x) {
            const int64_t bh = tile / p.tiles_per_bh;
            const int qt = tile % p.tiles_per_bh;
            const int row = qt * kMTile + warp * 32 + lane;
            const bool valid = row < p.N;
            // rows past the sequence (a ragged last tile) contribute nothing
            const float lse2 = valid ? p.LSE[bh * p.N + row] * log2e : CUDART_INF_F;
            float *part = p.part + (static_cast<size_t>(tile) * kMassWarps + warp) * p.nKB;
            for (int j = 0; j < p.nKB; ++j, ++G) {
                const int b = G % NSB;
                if (!warp_wait_all(bar(C::B_SFULL + b), (G / NSB) & 1, ctl)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[BS / 32][32];
#pragma unroll
                for (int c = 0; c < BS / 32; ++c) tmem_ld32(tS + b * BS + c * 32, sv[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < BS / 32; ++c) reg_fence32(sv[c]);
                // S is in registers: the buffer is free for the next QK^T
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_SEMPTY + b));
                if (j == p.nKB - 1 && p.last_rows < BS) {
                    // keys past the sequence end (read as zeros) hold no mass
#pragma unroll
                    for (int c = 0; c < BS / 32; ++c)
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (c * 32 + t >= p.last_rows) sv[c][t] = 0xFF800000u;
                }
                float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
                for (int c = 0; c < BS / 32; ++c)
#pragma unroll
                    for (int t = 0; t < 32; t += 4) {
                        a0 += ex2_approx(fmaf(__uint_as_float(sv[c][t]), p.scale_log2, -lse2));
                        a1 += ex2_approx(fmaf(__uint_as_float(sv[c][t + 1]), p.scale_log2, -lse2));
                        a2 += ex2_approx(fmaf(__uint_as_float(sv[c][t + 2]), p.scale_log2, -lse2));
                        a3 += ex2_approx(fmaf(__uint_as_float(sv[c][t + 3]), p.scale_log2, -lse2));
                    }
                float sum = valid ? (a0 + a1) + (a2 + a3) : 0.0f;
                // the warp's 32 rows, summed in a fixed butterfly order
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                if (lane == 0) part[j] = sum;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMassIssuer) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TCOLS);
    }
}

template <int D, int BS, int NK, int NSB>
bsa_status launch_mass(const ExactArgs &a, cudaStream_t st)
{
    using C = MassCfg<D, BS, NK, NSB>;
    static_assert(2 * (C::SMEM_ALLOC + 1024) <= 233472, "shared memory for two CTAs per SM");
    static_assert(2 * C::TCOLS <= 512, "TMEM for two CTAs per SM");
    auto kern = mass_kernel<D, BS, NK, NSB>;
    static int grid_cap = 0;
    if (grid_cap == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) != cudaSuccess)
            return BSA_ERR_CUDA;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return BSA_ERR_CUDA;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BSA_ERR_CUDA;
        grid_cap = 2 * sms;
    }
    const int64_t BH = static_cast<int64_t>(a.B) * a.H;
    CUtensorMap mq, mk;
    if (!make_tma_map_bf16(&mq, a.Q, BH, a.N, D, kMTile) || !make_tma_map_bf16(&mk, a.K, BH, a.N, D, BS))
        return BSA_ERR_CUDA;
    MassParams p{};
    p.N = a.N;
    p.nKB = a.nKB;
    p.last_rows = a.N - (a.nKB - 1) * BS;
    p.tiles_per_bh = (a.N + kMTile - 1) / kMTile;
    p.n_tiles = static_cast<int>(BH * p.tiles_per_bh);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.LSE = a.LSE;
    p.part = reinterpret_cast<float *>(a.ws + kWsHeader);
    p.err = reinterpret_cast<uint32_t *>(a.ws);
    p.wait_limit_ns = a.wait_limit_ns;
    const int grid = p.n_tiles < grid_cap ? p.n_tiles : grid_cap;
    kern<<<grid, kMassThreads, C::SMEM_ALLOC, st>>>(mq, mk, p);
    if (cudaGetLastError() != cudaSuccess) return BSA_ERR_CUDA;
    return launch_mass_select(p.part, a, p.tiles_per_bh, st);
}

// ---------------------------------------------------------------- token masses
//
// The token oracle of "Can sparse attention close the quality gap in diffusion
// transformers" (section "质量差距有三个可分离来源"), with the tile-aligned query groups
// of section "token 级选择需要瓦片对齐的查询分组": per group g of 128 queries and key t,
//   mass[g][t] = sum over rows r of g of exp(scale * q_r . k_t - LSE_r).
// On tcgen05 as S^T = K_chunk Q_g^T: the MMA's M = 128 rows are 128 consecutive keys
// (a TMA tile of K) and its N = 128 columns are the group's queries (gathered through
// the permutation once per group), so one thread holds one key's 128 scores and sums its
// mass alone, in column order: no reduction across threads. Warp roles as mass_kernel.

struct TokMassParams {
    int N, groups, n_tiles;  // groups per head (N / 128); tiles = B*H*groups
    float scale_log2;
    const float *LSE;        // [B*H*N] dense logsumexp, natural log
    const int32_t *perm;     // [B*H][N]
    float *mass;             // [tiles][N]
    uint32_t *err;
    unsigned long long wait_limit_ns;
};

template <int D, int NK>
struct TokMassCfg {
    static constexpr int kQBytes = kMTile * D * 2;  // the group's queries: the MMA's B operand
    static constexpr int kKBytes = kMTile * D * 2;  // 128 keys: the A operand
    static constexpr int kChunk = kMTile * 128;     // one 64-column swizzled slab (128 rows)
    static constexpr int NSB = 2;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + kQBytes;
    static constexpr int BAR_OFF = K_OFF + NK * kKBytes;
    static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + NK;
    static constexpr int B_SFULL = B_KEMPTY + NK, B_SEMPTY = B_SFULL + NSB, B_DRAIN = B_SEMPTY + NSB;
    static constexpr int NBAR = B_DRAIN + 1;
    // per mass warp, the group's LSE * log2 e [128] (16-byte aligned: read as float4)
    static constexpr int LSE_OFF = (BAR_OFF + NBAR * 8 + 15) / 16 * 16;
    static constexpr int MISC_OFF = LSE_OFF + kMassWarps * kMTile * 4;
    static constexpr int SMEM = MISC_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;  // manual 1024-byte alignment
    static constexpr int TCOLS = NSB * kMTile;       // 256: two CTAs per SM
    static constexpr uint32_t IDESC = idesc_bf16_f32(kMTile, kMTile, 0, 0);
};

template <int D, int NK>
__global__ void __launch_bounds__(kMassThreads, 2)
    token_mass_kernel(const __grid_constant__ CUtensorMap tmQrows, const __grid_constant__ CUtensorMap tmK,
                      const TokMassParams p)
{
    using C = TokMassCfg<D, NK>;
    constexpr int NSB = C::NSB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int idx) -> uint32_t { return sbase + C::BAR_OFF + 8u * idx; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);  // [0] TMEM base, [1] abort flag
    float *lse_s = reinterpret_cast<float *>(smem + C::LSE_OFF);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = p.N / kMTile;  // key chunks per group

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_QEMPTY), 1);
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
        }
        for (int b = 0; b < NSB; ++b) {
            mbar_init(bar(C::B_SFULL + b), 1);
            mbar_init(bar(C::B_SEMPTY + b), kMassWarps);
        }
        mbar_init(bar(C::B_DRAIN), 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == kMassIssuer) {
        tmem_alloc(smem_u32(misc), C::TCOLS);
        tmem_relinquish();
    }
    if (warp == kMassProducer && lane == 0) {
        tma_prefetch_map(&tmQrows);
        tma_prefetch_map(&tmK);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const Ctl ctl{reinterpret_cast<volatile uint32_t *>(misc + 1), p.err, p.wait_limit_ns};

    if (warp == kMassProducer) {
        // ------------------------------------------------------------ producer: Q rows by gather, K by tile
        int G = 0, e = 0, last_k = -1, q_issued = -1;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.n_tiles; tile += gridDim.x, ++e) {
            const int64_t bh = tile / p.groups;
            // the Q slot was last read by the previous tile's MMAs
            if (e >= 1 && !warp_wait_all(bar(C::B_QEMPTY), (e - 1) & 1, ctl)) break;
            int rows[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int r = __ldg(p.perm + static_cast<int64_t>(tile) * kMTile + 4 * lane + i);
                if (r < 0 || r >= p.N) r = 0;  // reported by the mass warps, which give it no mass
                rows[i] = static_cast<int>(bh * p.N + r);
            }
            if (lane == 0) mbar_arrive_expect_tx(bar(C::B_QFULL), C::kQBytes);
            __syncwarp();
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tma_gather4(sbase + C::Q_OFF + c * C::kChunk + lane * 512, &tmQrows, c * 64, rows[0], rows[1], rows[2],
                            rows[3], bar(C::B_QFULL));
            __syncwarp();
            q_issued = e;
            for (int j = 0; j < nch; ++j, ++G) {
                const int s = G % NK;
                if (G >= NK && !warp_wait_all(bar(C::B_KEMPTY + s), ((G / NK) - 1) & 1, ctl)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                if (elect_one()) {
                    mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::kKBytes);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_3d(sbase + C::K_OFF + s * C::kKBytes + c * C::kChunk, &tmK, c * 64, j * kMTile,
                                    static_cast<int>(bh), bar(C::B_KFULL + s));
                }
                __syncwarp();
                last_k = G;
            }
        }
        if (lane == 0 && *ctl.abort_flag) {
            // never leave while our copies may still land in shared memory
            for (int g = last_k - NK + 1; g <= last_k; ++g)
                if (g >= 0) wait_bar_drain(bar(C::B_KFULL + g % NK), (g / NK) & 1, p.wait_limit_ns);
            if (q_issued >= 0) wait_bar_drain(bar(C::B_QFULL), q_issued & 1, p.wait_limit_ns);
        }
        __syncwarp();
    } else if (warp == kMassIssuer) {
        // ------------------------------------------------------------ S^T = K_chunk Q_g^T issuer
        const uint64_t qdesc = sdesc_sw128(sbase + C::Q_OFF, 16, 1024);
        const uint64_t kdesc0 = sdesc_sw128(sbase + C::K_OFF, 16, 1024);
        int G = 0, e = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.n_tiles; tile += gridDim.x, ++e) {
            if (!warp_wait_all(bar(C::B_QFULL), e & 1, ctl)) break;
            tc_fence_after();
            for (int j = 0; j < nch; ++j, ++G) {
                const int s = G % NK, b = G % NSB;
                if (!warp_wait_all(bar(C::B_KFULL + s), (G / NK) & 1, ctl)) {
                    ok = false;
                    break;
                }
                if (G >= NSB && !warp_wait_all(bar(C::B_SEMPTY + b), ((G / NSB) - 1) & 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t kdesc = kdesc0 + static_cast<uint64_t>(s * (C::kKBytes >> 4));
                __syncwarp();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kChunk + (kk & 3) * 32) >> 4);
                        mma_ss(tmem + b * kMTile, kdesc + off, qdesc + off, C::IDESC, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(C::B_SFULL + b));
                    tc_commit(bar(C::B_KEMPTY + s));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) tc_commit(bar(C::B_QEMPTY));
            __syncwarp();
        }
        __syncwarp();
        if (elect_one()) {
            tc_commit(bar(C::B_DRAIN));
            wait_bar_drain(bar(C::B_DRAIN), 0, p.wait_limit_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ mass warps (thread = key = TMEM lane)
        const uint32_t tS = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float log2e = 1.4426950408889634f;
        int G = 0;
        bool alive = true, nan_seen = false;
        float *lse_w = lse_s + warp * kMTile;  // this warp's copy: no barrier across the mass warps
        for (int tile = blockIdx.x; alive && tile < p.n_tiles; tile += gridDim.x) {
            const int64_t bh = tile / p.groups;
            // the group's LSE (log2 units); a row outside [0, N) is reported and holds no mass
            __syncwarp();  // the previous tile's values are no longer read
#pragma unroll
            for (int i = 0; i < kMTile / 32; ++i) {
                const int c = 32 * i + lane;
                const int r = __ldg(p.perm + static_cast<int64_t>(tile) * kMTile + c);
                const bool valid = r >= 0 && r < p.N;
                if (!valid && warp == 0) raise_error(p.err, BSA_ERR_INVALID_ARG);
                lse_w[c] = valid ? __ldg(p.LSE + bh * p.N + r) * log2e : CUDART_INF_F;
            }
            __syncwarp();
            float *out = p.mass + static_cast<int64_t>(tile) * p.N + warp * 32 + lane;
            for (int j = 0; j < nch; ++j, ++G) {
                const int b = G % NSB;
                if (!warp_wait_all(bar(C::B_SFULL + b), (G / NSB) & 1, ctl)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[kMTile / 32][32];
#pragma unroll
                for (int c = 0; c < kMTile / 32; ++c) tmem_ld32(tS + b * kMTile + c * 32, sv[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < kMTile / 32; ++c) reg_fence32(sv[c]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_SEMPTY + b));
                float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
                for (int c = 0; c < kMTile / 32; ++c)
#pragma unroll
                    for (int t = 0; t < 32; t += 4) {
                        const float4 l4 = *reinterpret_cast<const float4 *>(lse_w + c * 32 + t);
                        a0 += ex2_approx(fmaf(__uint_as_float(sv[c][t]), p.scale_log2, -l4.x));
                        a1 += ex2_approx(fmaf(__uint_as_float(sv[c][t + 1]), p.scale_log2, -l4.y));
                        a2 += ex2_approx(fmaf(__uint_as_float(sv[c][t + 2]), p.scale_log2, -l4.z));
                        a3 += ex2_approx(fmaf(__uint_as_float(sv[c][t + 3]), p.scale_log2, -l4.w));
                    }
                const float m = (a0 + a1) + (a2 + a3);
                nan_seen |= isnan(m);
                out[static_cast<int64_t>(j) * kMTile] = m;
            }
        }
        if (__any_sync(0xffffffffu, nan_seen) && lane == 0) raise_error(p.err, BSA_ERR_NONFINITE);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMassIssuer) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TCOLS);
    }
}

template <int D, int NK>
bsa_status launch_token_mass(const TokenSelectArgs &a, float *mass, cudaStream_t st)
{
    using C = TokMassCfg<D, NK>;
    static_assert(2 * (C::SMEM_ALLOC + 1024) <= 233472, "shared memory for two CTAs per SM");
    static_assert(2 * C::TCOLS <= 512, "TMEM for two CTAs per SM");
    auto kern = token_mass_kernel<D, NK>;
    static int grid_cap = 0;
    if (grid_cap == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) != cudaSuccess)
            return BSA_ERR_CUDA;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return BSA_ERR_CUDA;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BSA_ERR_CUDA;
        grid_cap = 2 * sms;
    }
    const int64_t BH = static_cast<int64_t>(a.B) * a.H;
    CUtensorMap mq, mk;
    if (!make_tma_map_bf16_rows(&mq, a.Q, static_cast<uint64_t>(BH) * a.N, D) ||
        !make_tma_map_bf16(&mk, a.K, BH, a.N, D, kMTile))
        return BSA_ERR_CUDA;
    TokMassParams p{};
    p.N = a.N;
    p.groups = a.N / kMTile;
    p.n_tiles = static_cast<int>(BH * p.groups);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.LSE = a.LSE;
    p.perm = a.perm;
    p.mass = mass;
    p.err = reinterpret_cast<uint32_t *>(a.ws);
    p.wait_limit_ns = a.wait_limit_ns;
    const int grid = p.n_tiles < grid_cap ? p.n_tiles : grid_cap;
    kern<<<grid, kMassThreads, C::SMEM_ALLOC, st>>>(mq, mk, p);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace

bsa_status launch_token_mass_tc(const TokenSelectArgs &a, float *mass, cudaStream_t st)
{
    // <D, K stages>: two CTAs per SM
    if (a.d == 64) return launch_token_mass<64, 4>(a, mass, st);
    if (a.d == 128) return launch_token_mass<128, 2>(a, mass, st);
    return BSA_ERR_SHAPE;
}

size_t exact_workspace_bytes(int B, int H, int N, int d, int block)
{
    (void)d;
    const size_t tiles = static_cast<size_t>(B) * H * ((N + kMTile - 1) / kMTile);
    const size_t nKB = static_cast<size_t>((N + block - 1) / block);
    return kWsHeader + align_up(tiles * kMassWarps * nKB * sizeof(float), 256);
}

bsa_status launch_build_mask_exact(const ExactArgs &a, cudaStream_t st)
{
    // <D, BS, K stages, S buffers>: two CTAs per SM (shared memory and TMEM checked above)
    if (a.d == 64 && a.block == 64) return launch_mass<64, 64, 6, 4>(a, st);
    if (a.d == 128 && a.block == 64) return launch_mass<128, 64, 4, 4>(a, st);
    if (a.d == 64 && a.block == 128) return launch_mass<64, 128, 4, 2>(a, st);
    if (a.d == 128 && a.block == 128) return launch_mass<128, 128, 2, 2>(a, st);
    return BSA_ERR_SHAPE;
}

}  // namespace bsa
