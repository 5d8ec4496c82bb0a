// query_groups.cu -- tile-aligned query groups for token-level selection.
//
// "Can sparse attention close the quality gap in diffusion transformers", section
// "token 级选择需要瓦片对齐的查询分组": the queries of a head are split recursively at the
// median of their projection on the group's principal direction until every group holds
// exactly C = 128 queries. A group of m*C rows keeps its first ceil(m/2)*C rows, ordered
// by (projection, row index), as the first half; groups come out in depth-first order,
// rows ascending inside a group (the layout bsa_select_tokens and bsa_forward_tokens take).
//
// The split tree depends on N only, so the splits run level by level, every segment of
// every head at once, in place in the working permutation of each head. Each segment of a
// level is cut into P slices of at most kSliceRows rows in whole 64-row chunks (P the same
// for the whole level), and a level is five launches:
//   slice_sum_kernel      per slice: the sum of its rows (fp32; each warp adds its rows in
//                         order, then the warps in order);
//   slice_gram_tc_kernel  (bf16, d = 128) per slice on tcgen05: sum x x^T over the slice's
//                         rows, uncentred (bf16 products are exact, the sums fp32); or
//   slice_scatter_kernel  (otherwise) per slice on CUDA cores: the segment's mean (the slice
//                         sums in slice order, over the length), then sum (x - mu)(x - mu)^T
//                         over the slice's rows (a thread owns a block and adds the rows in
//                         order); either way only the blocks on or above the diagonal;
//   direction_kernel      per segment: S = the slices' blocks added in slice order (less the
//                         rank-one mean term after the tensor-core pass), and the principal
//                         direction by kPowerIters steps of power iteration on S from a fixed
//                         start (sign: its largest-magnitude entry positive);
//   slice_keys_kernel     per slice: 64-bit keys (projection as an order-preserving key, row
//                         index);
//   cut_kernel            per segment: the cut-th smallest key by an exact radix select
//                         (8-bit digits), and a stable partition (first half: keys up to the
//                         cut) through a scratch copy.
// Every sum runs in a fixed order, so the groups do not change from run to run. A final
// launch sorts each group's rows ascending. fp32 and an iterative eigenvector: near the
// median a row may fall on the other side than in an exact eigendecomposition, so results
// are judged by the partition they form, and bit for bit where no row lies within the
// rounding bound of a cut.
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "sync.cuh"

namespace bsa {
namespace {

constexpr int kGrpThreads = 256;
constexpr int kGrpWarps = kGrpThreads / 32;
constexpr int kPowerIters = 32;
constexpr int kStageRows = 32;                 // rows staged per step of the scatter pass
constexpr int kSliceRows = 4 * kTokenGroup;    // rows per slice at most
constexpr int kTriBlocks = 136;                // blocks of a 16 x 16 grid on or above the diagonal
constexpr int kScatThreads = 160;              // kTriBlocks computing threads, 5 warps staging rows
constexpr int kGramRows = 64;                  // rows per tcgen05 chunk of the bf16 scatter pass
constexpr int kGramStages = 4;                 // gather ring stages of that pass

__device__ __forceinline__ uint32_t order_key_asc(float s)
{
    uint32_t u = __float_as_uint(s);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Segment `seg` of level `level` (path of `level` bits, the most significant first: 0 the
// first half, 1 the second) of a head of N rows; false when the path ends in a final group
// before that depth (nothing to split there).
__device__ __forceinline__ bool segment_of(int N, int level, int seg, int &s, int &len)
{
    constexpr int C = kTokenGroup;
    s = 0;
    len = N;
    for (int l = level - 1; l >= 0; --l) {
        if (len <= C) return false;
        const int cut = ((len / C + 1) / 2) * C;
        if ((seg >> l) & 1) {
            s += cut;
            len -= cut;
        } else {
            len = cut;
        }
    }
    return len > C;
}

// Slices: a segment of `len` rows at a level with P slices per segment is cut into P runs
// of ceil(len / P) rows rounded up to whole 64-row chunks (len is a multiple of 128, so
// every run is whole chunks; the last may be shorter or empty). False when the segment
// is final.
__device__ __forceinline__ bool slice_of(int N, int level, int P, int slot, int &seg, int &s, int &len, int &r0,
                                         int &r1)
{
    seg = slot / P;
    const int p = slot - seg * P;
    if (!segment_of(N, level, seg, s, len)) return false;
    const int chunk = ((len + P - 1) / P + kGramRows - 1) / kGramRows * kGramRows;
    r0 = min(len, p * chunk);
    r1 = min(len, r0 + chunk);
    return true;
}

// VEC consecutive elements of a row as fp32 (8- or 16-byte loads).
template <int VEC>
__device__ __forceinline__ void ldvec(const float *p, float (&o)[VEC])
{
    static_assert(VEC == 2 || VEC == 4, "8- or 16-byte loads");
    if constexpr (VEC == 4) {
        const float4 f = *reinterpret_cast<const float4 *>(p);
        o[0] = f.x, o[1] = f.y, o[2] = f.z, o[3] = f.w;
    } else {
        const float2 f = *reinterpret_cast<const float2 *>(p);
        o[0] = f.x, o[1] = f.y;
    }
}
template <int VEC>
__device__ __forceinline__ void ldvec(const __nv_bfloat16 *p, float (&o)[VEC])
{
    static_assert(VEC == 2 || VEC == 4 || VEC == 8, "4-, 8- or 16-byte loads");
    if constexpr (VEC == 8) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) o[2 * k] = __uint_as_float(w[k] << 16), o[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    } else if constexpr (VEC == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        o[0] = __uint_as_float(u.x << 16), o[1] = __uint_as_float(u.x & 0xFFFF0000u);
        o[2] = __uint_as_float(u.y << 16), o[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        o[0] = __uint_as_float(u << 16), o[1] = __uint_as_float(u & 0xFFFF0000u);
    }
}

// Row passes with 16-byte loads: a lane holds E elements of a row, LPR lanes one row,
// a warp RPI rows per load and kInFlight loads in flight.
template <typename T, int D>
struct RowPass {
    static constexpr int E = 16 / static_cast<int>(sizeof(T));
    static constexpr int LPR = D / E;
    static constexpr int RPI = 32 / LPR;
    static constexpr int ROWS = RPI * 4;  // rows per warp per step
};

// Block (bi, bj), bi <= bj, of the 16 x 16 grid of the scatter matrix owned by thread t of
// kTriBlocks: row blocks p and 15 - p share 17 consecutive threads (16 - p + p + 1 blocks).
__device__ __forceinline__ void tri_block(int t, int &bi, int &bj)
{
    const int pr = t / 17, k = t - 17 * (t / 17);
    if (k < 16 - pr) {
        bi = pr;
        bj = pr + k;
    } else {
        bi = 15 - pr;
        bj = bi + k - (16 - pr);
    }
}

// Column c of a staged row in the scatter pass (4 padding floats after every 32).
__device__ __forceinline__ int pad(int c) { return c + 4 * (c >> 5); }

// The segment's mean: its slices' sums added in slice order, over len.
template <int D>
__device__ __forceinline__ void segment_mean(const float *__restrict__ psum, int64_t slot0, int P, int len, float *mu)
{
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float m = 0.0f;
        for (int q = 0; q < P; ++q) m += psum[(slot0 + q) * D + c];
        mu[c] = m / static_cast<float>(len);
    }
}

// Per slice: the sum of its rows. grid (2^level * P, B*H).
template <typename T, int D>
__global__ void __launch_bounds__(kGrpThreads) slice_sum_kernel(const T *__restrict__ X, int N, int level, int P,
                                                                int G, const int32_t *__restrict__ work,
                                                                float *__restrict__ psum)
{
    using RP = RowPass<T, D>;
    constexpr int E = RP::E;
    __shared__ float part[kGrpWarps][D];
    grid_dependency_wait();
    int seg, s, len, r0, r1;
    if (!slice_of(N, level, P, blockIdx.x, seg, s, len, r0, r1)) return;  // block-uniform
    const int64_t bh = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rs = lane / RP::LPR, cp = lane % RP::LPR;  // row of the load, columns cp*E ..
    const T *x = X + bh * static_cast<int64_t>(N) * D + cp * E;
    const int32_t *idx = work + bh * N + s;
    float acc[E];
#pragma unroll
    for (int t = 0; t < E; ++t) acc[t] = 0.0f;
    // each lane adds the rows of its load slot in order
    for (int i0 = r0 + warp * RP::ROWS; i0 < r1; i0 += kGrpWarps * RP::ROWS) {
        float vals[4][E];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * RP::RPI + rs;
            if (i < r1) {
                ldvec<E>(x + static_cast<int64_t>(idx[i]) * D, vals[u]);
            } else {
#pragma unroll
                for (int t = 0; t < E; ++t) vals[u][t] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int t = 0; t < E; ++t) acc[t] += vals[u][t];
    }
    // the warp's load slots (xor butterfly: every lane of a column part ends with one sum)
#pragma unroll
    for (int o = RP::LPR; o < 32; o <<= 1)
#pragma unroll
        for (int t = 0; t < E; ++t) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    if (rs == 0) {
#pragma unroll
        for (int t = 0; t < E; ++t) part[warp][cp * E + t] = acc[t];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kGrpThreads) {
        float m = 0.0f;
        for (int w = 0; w < kGrpWarps; ++w) m += part[w][c];
        psum[(bh * G + blockIdx.x) * D + c] = m;
    }
}

// Per slice: sum over its rows of (x - mu)(x - mu)^T, the blocks on or above the diagonal.
// Thread t < kTriBlocks owns one BLK x BLK block and adds the rows in order; entry e of
// block t goes to pS[slot][e][t]. grid (2^level * P, B*H).
template <typename T, int D>
__global__ void __launch_bounds__(kScatThreads, 3)
    slice_scatter_kernel(const T *__restrict__ X, int N, int level, int P, int G, const int32_t *__restrict__ work,
                         const float *__restrict__ psum, float *__restrict__ pS)
{
    constexpr int VEC = D / 32;
    constexpr int BLK = D / 16;
    constexpr int NW = kScatThreads / 32;
    constexpr int RPW = (kStageRows + NW - 1) / NW;  // staged rows per warp
    constexpr int XW = D + D / 8;  // staged row: 4 padding floats after every 32 (float4 reads of 8-float blocks hit distinct banks)
    __shared__ __align__(16) float xs[kStageRows][XW];
    __shared__ float mu[D];
    grid_dependency_wait();
    int seg, s, len, r0, r1;
    if (!slice_of(N, level, P, blockIdx.x, seg, s, len, r0, r1)) return;  // block-uniform
    const int64_t bh = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const T *x = X + bh * static_cast<int64_t>(N) * D;
    const int32_t *idx = work + bh * N + s;
    segment_mean<D>(psum, bh * G + static_cast<int64_t>(seg) * P, P, len, mu);
    const bool comp = threadIdx.x < kTriBlocks;
    int bi = 0, bj = 0;
    tri_block(comp ? threadIdx.x : 0, bi, bj);
    float acc[BLK][BLK];
#pragma unroll
    for (int a = 0; a < BLK; ++a)
#pragma unroll
        for (int b = 0; b < BLK; ++b) acc[a][b] = 0.0f;
    // the next stage of rows is loaded into registers while this one is used
    float nxt[RPW][VEC];
    auto fetch = [&](int a0) {
#pragma unroll
        for (int u = 0; u < RPW; ++u) {
            const int r = warp + NW * u;
            if (r < kStageRows && a0 + r < r1) {
                ldvec<VEC>(x + static_cast<int64_t>(idx[a0 + r]) * D + lane * VEC, nxt[u]);
            } else {
#pragma unroll
                for (int t = 0; t < VEC; ++t) nxt[u][t] = 0.0f;
            }
        }
    };
    fetch(r0);
    __syncthreads();  // mu
    for (int a0 = r0; a0 < r1; a0 += kStageRows) {
        if (a0 != r0) __syncthreads();
#pragma unroll
        for (int u = 0; u < RPW; ++u) {
            const int r = warp + NW * u;
            if (r < kStageRows) {
#pragma unroll
                for (int t = 0; t < VEC; ++t)
                    xs[r][pad(lane * VEC + t)] = a0 + r < r1 ? nxt[u][t] - mu[lane * VEC + t] : 0.0f;
            }
        }
        __syncthreads();
        if (a0 + kStageRows < r1) fetch(a0 + kStageRows);
        const int nr = min(kStageRows, r1 - a0);
        if (comp) {
            for (int r = 0; r < nr; ++r) {
                float a_[BLK], b_[BLK];
#pragma unroll
                for (int q = 0; q < BLK / 4; ++q) {
                    const float4 fa = *reinterpret_cast<const float4 *>(&xs[r][pad(BLK * bi + 4 * q)]);
                    const float4 fb = *reinterpret_cast<const float4 *>(&xs[r][pad(BLK * bj + 4 * q)]);
                    a_[4 * q] = fa.x, a_[4 * q + 1] = fa.y, a_[4 * q + 2] = fa.z, a_[4 * q + 3] = fa.w;
                    b_[4 * q] = fb.x, b_[4 * q + 1] = fb.y, b_[4 * q + 2] = fb.z, b_[4 * q + 3] = fb.w;
                }
#pragma unroll
                for (int a = 0; a < BLK; ++a)
#pragma unroll
                    for (int b = 0; b < BLK; ++b) acc[a][b] = fmaf(a_[a], b_[b], acc[a][b]);
            }
        }
    }
    if (comp) {
        float *out = pS + (bh * G + blockIdx.x) * static_cast<int64_t>(BLK * BLK * kTriBlocks) + threadIdx.x;
#pragma unroll
        for (int a = 0; a < BLK; ++a)
#pragma unroll
            for (int b = 0; b < BLK; ++b) out[(a * BLK + b) * kTriBlocks] = acc[a][b];
    }
}

// Index within the kTriBlocks blocks of block (bi, bj), bi <= bj (the inverse of tri_block).
__device__ __forceinline__ int tri_index(int bi, int bj) { return bi <= 7 ? 17 * bi + (bj - bi) : 17 * (15 - bi) + 1 + bj; }

// bf16, d = 128: per slice, G = sum over its rows of x x^T (raw, not centred) on tcgen05;
// the segment's rank-one mean term comes off in direction_kernel. The rows arrive through
// the permutation by TMA tile::gather4 (64 rows per chunk, both 64-column slabs, into a
// 128-byte-swizzled ring) and one chunk is both MMA operands: A = X^T and B = X, both
// MN-major (the tile is [rows][d] with d contiguous), M = N = 128, K = 16 rows per MMA,
// accumulated in TMEM in fp32 (bf16 products are exact). Warp 0 gathers, warp 1 issues
// (and owns TMEM), then all four warps write the blocks on or above the diagonal in the
// same [slot][entry][block] layout as slice_scatter_kernel. grid (2^level * P, B*H).
struct GramCfg {
    static constexpr int kSlab = kGramRows * 128;     // one 64-column slab of a chunk, 8 KB
    static constexpr int kStage = 2 * kSlab;          // d = 128: two slabs
    static constexpr int BAR_OFF = kGramStages * kStage;
    static constexpr int B_FULL = 0, B_EMPTY = kGramStages, B_DONE = 2 * kGramStages, B_DRAIN = B_DONE + 1;
    static constexpr int NBAR = B_DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;  // [0] TMEM base, [1] abort flag
    static constexpr int SMEM = MISC_OFF + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;       // manual 1024-byte alignment
    static constexpr int TCOLS = 128;
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, 128, 1, 1);
};

__global__ void __launch_bounds__(128) slice_gram_tc_kernel(const __grid_constant__ CUtensorMap tmX, int N, int level,
                                                            int P, int G, const int32_t *__restrict__ work,
                                                            float *__restrict__ pS, uint32_t *err,
                                                            unsigned long long wait_limit_ns)
{
    using C = GramCfg;
    constexpr int D = 128, BLK = D / 16, PER = BLK * BLK * kTriBlocks;
    extern __shared__ uint8_t gram_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gram_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int idx) -> uint32_t { return sbase + C::BAR_OFF + 8u * idx; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    grid_dependency_wait();
    int seg, s, len, r0, r1;
    if (!slice_of(N, level, P, blockIdx.x, seg, s, len, r0, r1)) return;  // block-uniform
    const int64_t bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = (r1 - r0) / kGramRows;  // whole chunks (slice_of)
    float *out = pS + (bh * G + blockIdx.x) * static_cast<int64_t>(PER);
    if (nch == 0) {  // an empty slice adds nothing
        for (int e = threadIdx.x; e < PER; e += blockDim.x) out[e] = 0.0f;
        return;
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < kGramStages; ++st) {
            mbar_init(bar(C::B_FULL + st), 1);
            mbar_init(bar(C::B_EMPTY + st), 1);
        }
        mbar_init(bar(C::B_DONE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), C::TCOLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) tma_prefetch_map(&tmX);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const Ctl ctl{reinterpret_cast<volatile uint32_t *>(misc + 1), err, wait_limit_ns};
    const int32_t *idx = work + bh * N + s;

    if (warp == 0) {
        // ------------------------------------------------------------ gather producer
        // lane l gathers rows 4(l % 16) .. +3 of each chunk into slab l / 16; the slice's row
        // indices (at most kMaxChunks chunks) are all loaded first, so no gather waits on one
        constexpr int kMaxChunks = kSliceRows / kGramRows;
        const int slab = lane >> 4, q0 = 4 * (lane & 15);
        int y[kMaxChunks][4];
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                y[c][q] = c < nch ? static_cast<int>(bh * N + idx[r0 + c * kGramRows + q0 + q]) : 0;
        int last = -1;
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
            if (c >= nch) break;
            const int st = c % kGramStages;
            if (c >= kGramStages && !warp_wait_all(bar(C::B_EMPTY + st), ((c / kGramStages) - 1) & 1, ctl)) break;
            if (lane == 0) mbar_arrive_expect_tx(bar(C::B_FULL + st), C::kStage);
            __syncwarp();
            tma_gather4(sbase + st * C::kStage + slab * C::kSlab + q0 * 128, &tmX, slab * 64, y[c][0], y[c][1],
                        y[c][2], y[c][3], bar(C::B_FULL + st));
            __syncwarp();
            last = c;
        }
        if (lane == 0 && *ctl.abort_flag) {
            // never leave while our copies may still land in shared memory
            for (int c = last - kGramStages + 1; c <= last; ++c)
                if (c >= 0) wait_bar_drain(bar(C::B_FULL + c % kGramStages), (c / kGramStages) & 1, wait_limit_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint64_t desc0 = sdesc_sw128(sbase, C::kSlab, 1024);
        for (int c = 0; c < nch; ++c) {
            const int st = c % kGramStages;
            if (!warp_wait_all(bar(C::B_FULL + st), (c / kGramStages) & 1, ctl)) break;
            tc_fence_after();
            const uint64_t desc = desc0 + static_cast<uint64_t>(st * (C::kStage >> 4));
            __syncwarp();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kGramRows / 16; ++kk) {
                    const uint64_t d = desc + static_cast<uint64_t>(kk * (16 * 128 >> 4));
                    mma_ss(tmem, d, d, C::IDESC, (c > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(C::B_EMPTY + st));
                if (c == nch - 1) tc_commit(bar(C::B_DONE));
            }
            __syncwarp();
        }
        __syncwarp();
        if (elect_one()) {
            tc_commit(bar(C::B_DRAIN));
            wait_bar_drain(bar(C::B_DRAIN), 0, wait_limit_ns);
        }
        __syncwarp();
    }
    // ------------------------------------------------------------ epilogue: thread = row i of G
    if (warp_wait_all(bar(C::B_DONE), 0, ctl)) {
        tc_fence_after();
        const int i = warp * 32 + lane, bi = i / BLK, a = i % BLK;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 32, v);
            tmem_wait_ld();
            reg_fence32(v);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int j = c * 32 + q, bj = j / BLK;
                if (bj >= bi) out[(a * BLK + j % BLK) * kTriBlocks + tri_index(bi, bj)] = __uint_as_float(v[q]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TCOLS);
    }
}

// Per segment: S = its slices' scatter blocks added in slice order (mirrored below the
// diagonal), then the principal direction by kPowerIters steps of power iteration from a
// fixed start; writes dir[seg] = (mu, v). grid (2^level, B*H).
template <int D, bool RAW>
__global__ void __launch_bounds__(kGrpThreads) direction_kernel(int N, int level, int P, int G,
                                                                const float *__restrict__ psum,
                                                                const float *__restrict__ pS,
                                                                float *__restrict__ dir)
{
    constexpr int BLK = D / 16;
    constexpr int PER = BLK * BLK * kTriBlocks;
    constexpr int SW = D + 8;  // row stride of S: 16-byte rows, 8 rows x 2 halves on distinct banks
    constexpr int EB = 4;      // entries per thread per batch
    constexpr int QB = 4;      // slices per batch
    static_assert(2 * D <= kGrpThreads, "two threads per row of S");
    extern __shared__ float4 grp_dyn[];
    float *S = reinterpret_cast<float *>(grp_dyn);
    __shared__ __align__(16) float v[D];
    __shared__ float mu[D], red[kGrpWarps];
    grid_dependency_wait();
    int s, len;
    if (!segment_of(N, level, blockIdx.x, s, len)) return;  // block-uniform
    const int64_t bh = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t slot0 = bh * G + static_cast<int64_t>(blockIdx.x) * P;
    segment_mean<D>(psum, slot0, P, len, mu);
    __syncthreads();  // mu
    const float rlen = sqrtf(static_cast<float>(len));
    // each entry: its slices added in order; EB entries x QB slices of loads in flight
    // (RAW: uncentred sums, less len * mu_i * mu_j taken as (sqrt(len) mu_i)(sqrt(len) mu_j),
    // the same value for (i, j) and (j, i))
    const float *src = pS + slot0 * PER;
    for (int e0 = threadIdx.x; e0 < PER; e0 += EB * kGrpThreads) {
        float m[EB];
#pragma unroll
        for (int k = 0; k < EB; ++k) m[k] = 0.0f;
        for (int q0 = 0; q0 < P; q0 += QB) {
            float val[QB][EB];
#pragma unroll
            for (int q = 0; q < QB; ++q)
#pragma unroll
                for (int k = 0; k < EB; ++k) {
                    const int e = e0 + k * kGrpThreads;
                    val[q][k] = q0 + q < P && e < PER ? src[static_cast<int64_t>(q0 + q) * PER + e] : 0.0f;
                }
#pragma unroll
            for (int q = 0; q < QB; ++q)
#pragma unroll
                for (int k = 0; k < EB; ++k)
                    if (q0 + q < P) m[k] += val[q][k];
        }
#pragma unroll
        for (int k = 0; k < EB; ++k) {
            const int e = e0 + k * kGrpThreads;
            if (e < PER) {
                const int t = e % kTriBlocks, ent = e / kTriBlocks;
                int bi, bj;
                tri_block(t, bi, bj);
                const int a = ent / BLK, b = ent % BLK;
                const int i = BLK * bi + a, j = BLK * bj + b;
                if (bi == bj && a > b) continue;  // a diagonal block: its upper half, mirrored
                float v = m[k];
                if (RAW) v = fmaf(-(rlen * mu[i]), rlen * mu[j], v);
                S[i * SW + j] = v;
                S[j * SW + i] = v;
            }
        }
    }
    if (threadIdx.x < D) v[threadIdx.x] = (1.0f + 0.01f * threadIdx.x) * rsqrtf(static_cast<float>(D));
    __syncthreads();
    // w = S v: two threads per row, each over alternate 4-column chunks of the row (held in
    // registers) with 4 accumulators
    const bool act = threadIdx.x < 2 * D;
    const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
    float sreg[D / 2];
#pragma unroll
    for (int m = 0; m < D / 8; ++m) {
        float4 sv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (act) sv = *reinterpret_cast<const float4 *>(S + row * SW + 8 * m + 4 * half);
        sreg[4 * m] = sv.x, sreg[4 * m + 1] = sv.y, sreg[4 * m + 2] = sv.z, sreg[4 * m + 3] = sv.w;
    }
    for (int it = 0; it < kPowerIters; ++it) {
        float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int m = 0; m < D / 8; ++m) {
            const float4 vv = *reinterpret_cast<const float4 *>(v + 8 * m + 4 * half);
            a4[0] = fmaf(sreg[4 * m], vv.x, a4[0]);
            a4[1] = fmaf(sreg[4 * m + 1], vv.y, a4[1]);
            a4[2] = fmaf(sreg[4 * m + 2], vv.z, a4[2]);
            a4[3] = fmaf(sreg[4 * m + 3], vv.w, a4[3]);
        }
        float w = (a4[0] + a4[1]) + (a4[2] + a4[3]);
        w += __shfl_xor_sync(0xffffffffu, w, 1);  // both threads of a row hold the same sum
        float sq = act && half == 0 ? w * w : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (lane == 0) red[warp] = sq;
        __syncthreads();
        float nrm2 = 0.0f;
#pragma unroll
        for (int ww = 0; ww < kGrpWarps; ++ww) nrm2 += red[ww];
        if (act && half == 0 && nrm2 > 0.0f) v[row] = w * rsqrtf(nrm2);
        __syncthreads();
    }
    // sign: the entry of largest magnitude (lowest index on ties) is positive
    if (warp == 0) {
        float best = -1.0f;
        int bj = 0;
        for (int j = lane; j < D; j += 32) {
            const float a = fabsf(v[j]);
            if (a > best) {
                best = a;
                bj = j;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
            if (ob > best || (ob == best && oj < bj)) {
                best = ob;
                bj = oj;
            }
        }
        const float sgn = v[bj] < 0.0f ? -1.0f : 1.0f;
        float *o = dir + (bh * G + blockIdx.x) * 2 * D;
        for (int j = lane; j < D; j += 32) {
            o[j] = mu[j];
            o[D + j] = v[j] * sgn;
        }
    }
}

// Per slice: the keys (projection on the segment's direction as an ascending key, row
// index) of its rows. grid (2^level * P, B*H).
template <typename T, int D>
__global__ void __launch_bounds__(kGrpThreads) slice_keys_kernel(const T *__restrict__ X, int N, int level, int P,
                                                                 int G, const int32_t *__restrict__ work,
                                                                 const float *__restrict__ dir,
                                                                 unsigned long long *__restrict__ keys)
{
    using RP = RowPass<T, D>;
    constexpr int E = RP::E;
    __shared__ float mu[D], v[D];
    grid_dependency_wait();
    int seg, s, len, r0, r1;
    if (!slice_of(N, level, P, blockIdx.x, seg, s, len, r0, r1)) return;  // block-uniform
    const int64_t bh = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rs = lane / RP::LPR, cp = lane % RP::LPR;
    const T *x = X + bh * static_cast<int64_t>(N) * D + cp * E;
    const int32_t *idx = work + bh * N + s;
    unsigned long long *key = keys + bh * N + s;
    const float *dv = dir + (bh * G + seg) * 2 * D;
    for (int c = threadIdx.x; c < D; c += kGrpThreads) {
        mu[c] = dv[c];
        v[c] = dv[D + c];
    }
    __syncthreads();
    float mu_[E], v_[E];
#pragma unroll
    for (int t = 0; t < E; ++t) {
        mu_[t] = mu[cp * E + t];
        v_[t] = v[cp * E + t];
    }
    for (int i0 = r0 + warp * RP::ROWS; i0 < r1; i0 += kGrpWarps * RP::ROWS) {
        float vals[4][E];
        int rr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * RP::RPI + rs;
            rr[u] = idx[i < r1 ? i : r0];
            ldvec<E>(x + static_cast<int64_t>(rr[u]) * D, vals[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float dot = 0.0f;
#pragma unroll
            for (int t = 0; t < E; ++t) dot = fmaf(vals[u][t] - mu_[t], v_[t], dot);
            // over the row's LPR lanes (xor butterfly: every lane of the row ends with one sum)
#pragma unroll
            for (int o = RP::LPR / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            const int i = i0 + u * RP::RPI + rs;
            if (cp == 0 && i < r1)
                key[i] = (static_cast<unsigned long long>(order_key_asc(dot)) << 32) | static_cast<uint32_t>(rr[u]);
        }
    }
}

// Per segment: the cut-th smallest key (keys are unique: the row index breaks ties) by an
// exact radix select, 8-bit digits, then a stable partition (first half: the keys up to it)
// through the scratch copy. grid (2^level, B*H).
__global__ void __launch_bounds__(kGrpThreads) cut_kernel(int N, int level, int32_t *__restrict__ work,
                                                          const unsigned long long *__restrict__ keys,
                                                          int32_t *__restrict__ scratch)
{
    constexpr int C = kTokenGroup;
    __shared__ int hist[256];
    __shared__ int redi[kGrpWarps];
    __shared__ int s_digit, s_krem;
    __shared__ bool s_one;
    grid_dependency_wait();
    int s, len;
    if (!segment_of(N, level, blockIdx.x, s, len)) return;  // block-uniform
    const int64_t bh = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t *idx = work + bh * N + s;
    const unsigned long long *key = keys + bh * N + s;
    int32_t *tmp = scratch + bh * N + s;
    const int cut = ((len / C + 1) / 2) * C;
    unsigned long long prefix = 0ull, pmask = 0ull;
    int krem = cut;
    for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        for (int b = threadIdx.x; b < 256; b += kGrpThreads) hist[b] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < len; i += kGrpThreads) {
            const unsigned long long k = key[i];
            if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255ull], 1);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l covers digits 8l .. 8l + 7 (ascending): counts below each lane by a scan
            int cnt[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                cnt[q] = hist[8 * lane + q];
                sum += cnt[q];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - sum;
            const unsigned who = __ballot_sync(0xffffffffu, excl < krem && krem <= incl);
            if (lane == __ffs(who) - 1) {
                int below = excl;
                for (int q = 0; q < 8; ++q) {
                    if (below + cnt[q] >= krem) {
                        s_digit = 8 * lane + q;
                        s_krem = krem - below;
                        s_one = cnt[q] == 1;
                        break;
                    }
                    below += cnt[q];
                }
            }
        }
        __syncthreads();
        prefix |= static_cast<unsigned long long>(s_digit) << shift;
        pmask |= 0xFFull << shift;
        krem = s_krem;
        const bool one = s_one;
        __syncthreads();
        // a lone key under this prefix is the cut-th smallest: no other key shares the prefix
        if (one) {
            prefix |= ~pmask;
            break;
        }
    }
    const unsigned long long Tk = prefix;  // the cut-th smallest key, or a bound no other key reaches: keys <= Tk form the first half
    // stable partition through the scratch copy: warp w takes the w-th run of whole 32-row
    // chunks; ballots give each row its place
    const int nch = (len + 31) / 32;
    const int c0 = warp * nch / kGrpWarps, c1 = (warp + 1) * nch / kGrpWarps;
    const unsigned below = (1u << lane) - 1u;
    int mine = 0;
    for (int c = c0; c < c1; ++c) {
        const int i = 32 * c + lane;
        mine += __popc(__ballot_sync(0xffffffffu, i < len && key[i] <= Tk));
    }
    if (lane == 0) redi[warp] = mine;
    __syncthreads();
    int first = 0;
    for (int w = 0; w < warp; ++w) first += redi[w];
    int second = cut + 32 * c0 - first;  // rows before this run that go second
    for (int c = c0; c < c1; ++c) {
        const int i = 32 * c + lane;
        const bool valid = i < len;
        const bool f = valid && key[i] <= Tk;
        const unsigned bf = __ballot_sync(0xffffffffu, f), bs = __ballot_sync(0xffffffffu, valid && !f);
        if (valid) tmp[f ? first + __popc(bf & below) : second + __popc(bs & below)] = idx[i];
        first += __popc(bf);
        second += __popc(bs);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < len; i += kGrpThreads) idx[i] = tmp[i];
}

// Each group of C rows in ascending row order. grid (N / C, B*H), C threads.
__global__ void __launch_bounds__(kTokenGroup) sort_groups_kernel(const int32_t *__restrict__ work, int N,
                                                                  int32_t *__restrict__ perm)
{
    __shared__ int32_t g[kTokenGroup];
    const int64_t base = static_cast<int64_t>(blockIdx.y) * N + static_cast<int64_t>(blockIdx.x) * kTokenGroup;
    const int r = work[base + threadIdx.x];
    g[threadIdx.x] = r;
    __syncthreads();
    int rank = 0;
    for (int j = 0; j < kTokenGroup; ++j) rank += g[j] < r ? 1 : 0;
    perm[base + rank] = r;
}

__global__ void init_work_kernel(int32_t *__restrict__ work, int N, int64_t total)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < total) work[i] = static_cast<int32_t>(i % N);
}

// Largest segment at `level`, in rows: repeated ceil/floor halving of G groups leaves
// ceil(G / 2^level) groups at most.
int max_segment_rows(int G, int level) { return ((G + (1 << level) - 1) >> level) * kTokenGroup; }

template <typename T, int D>
bsa_status launch(const GroupArgs &a, cudaStream_t st)
{
    const QueryGroupWs l = query_groups_ws_layout(a.B, a.H, a.N, a.d);
    int32_t *work = reinterpret_cast<int32_t *>(a.ws + l.work);
    auto *keys = reinterpret_cast<unsigned long long *>(a.ws + l.keys);
    int32_t *scratch = reinterpret_cast<int32_t *>(a.ws + l.scratch);
    float *psum = reinterpret_cast<float *>(a.ws + l.psum);
    float *pS = reinterpret_cast<float *>(a.ws + l.pscatter);
    float *dir = reinterpret_cast<float *>(a.ws + l.dir);
    const int BH = a.B * a.H;
    const int64_t total = static_cast<int64_t>(BH) * a.N;
    init_work_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(work, a.N, total);
    const int G = a.N / kTokenGroup;
    int depth = 0;
    while ((1 << depth) < G) ++depth;  // levels until every segment is one group
    // bf16 at d = 128: the scatter blocks on tcgen05 (raw sums; the mean term comes off per
    // segment); otherwise on CUDA cores, centred per slice
    constexpr bool kTc = std::is_same<T, __nv_bfloat16>::value && D == 128;
    const size_t smem = sizeof(float) * D * (D + 8);
    if (cudaFuncSetAttribute(direction_kernel<D, kTc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return BSA_ERR_CUDA;
    CUtensorMap mx;
    if (kTc) {
        if (!make_tma_map_bf16_rows(&mx, a.Q, static_cast<uint64_t>(BH) * a.N, D)) return BSA_ERR_CUDA;
        if (cudaFuncSetAttribute(slice_gram_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GramCfg::SMEM_ALLOC) != cudaSuccess)
            return BSA_ERR_CUDA;
    }
    uint32_t *err = reinterpret_cast<uint32_t *>(a.ws);
    const T *X = static_cast<const T *>(a.Q);
    for (int level = 0; level < depth; ++level) {
        const int P = (max_segment_rows(G, level) + kSliceRows - 1) / kSliceRows;
        const int slots = (1 << level) * P;  // <= G with slices of 4 groups: the workspace holds G per head
        if (slots > G) return BSA_ERR_INVALID_ARG;
        const dim3 sl(static_cast<unsigned>(slots), static_cast<unsigned>(BH));
        const dim3 sg(1u << level, static_cast<unsigned>(BH));
        // programmatic dependent launches (no early trigger: CTAs waiting at
        // griddepcontrol.wait slow the kernel they wait for): a launch is set up while the
        // previous kernel runs and its CTAs start as that kernel's complete
        bool ok = pdl_launch(slice_sum_kernel<T, D>, sl, kGrpThreads, 0, st, X, a.N, level, P, G,
                             static_cast<const int32_t *>(work), psum);
        if (kTc)
            ok = ok && pdl_launch(slice_gram_tc_kernel, sl, 128, static_cast<size_t>(GramCfg::SMEM_ALLOC), st, mx,
                                  a.N, level, P, G, static_cast<const int32_t *>(work), pS, err, a.wait_limit_ns);
        else
            ok = ok && pdl_launch(slice_scatter_kernel<T, D>, sl, kScatThreads, 0, st, X, a.N, level, P, G,
                                  static_cast<const int32_t *>(work), static_cast<const float *>(psum), pS);
        ok = ok && pdl_launch(direction_kernel<D, kTc>, sg, kGrpThreads, smem, st, a.N, level, P, G,
                              static_cast<const float *>(psum), static_cast<const float *>(pS), dir);
        ok = ok && pdl_launch(slice_keys_kernel<T, D>, sl, kGrpThreads, 0, st, X, a.N, level, P, G,
                              static_cast<const int32_t *>(work), static_cast<const float *>(dir), keys);
        ok = ok && pdl_launch(cut_kernel, sg, kGrpThreads, 0, st, a.N, level, work,
                              static_cast<const unsigned long long *>(keys), scratch);
        if (!ok) return BSA_ERR_CUDA;
    }
    sort_groups_kernel<<<dim3(static_cast<unsigned>(G), static_cast<unsigned>(BH)), kTokenGroup, 0, st>>>(
        work, a.N, a.perm);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace

QueryGroupWs query_groups_ws_layout(int B, int H, int N, int d)
{
    const size_t n = static_cast<size_t>(B) * H * N;
    const size_t slots = static_cast<size_t>(B) * H * (N / kTokenGroup);  // one per group of each head
    QueryGroupWs l{};
    l.work = kWsHeader;
    l.keys = l.work + align_up(n * sizeof(int32_t), 256);
    l.scratch = l.keys + align_up(n * sizeof(unsigned long long), 256);
    l.psum = l.scratch + align_up(n * sizeof(int32_t), 256);
    l.pscatter = l.psum + align_up(slots * d * sizeof(float), 256);
    l.dir = l.pscatter + align_up(slots * (static_cast<size_t>(d) * d / 256 * kTriBlocks) * sizeof(float), 256);
    l.total = l.dir + align_up(slots * 2 * d * sizeof(float), 256);
    return l;
}

bsa_status launch_query_groups(const GroupArgs &a, cudaStream_t st)
{
    if (a.dt == BSA_BF16) {
        if (a.d == 64) return launch<__nv_bfloat16, 64>(a, st);
        if (a.d == 128) return launch<__nv_bfloat16, 128>(a, st);
    } else {
        if (a.d == 64) return launch<float, 64>(a, st);
        if (a.d == 128) return launch<float, 128>(a, st);
    }
    return BSA_ERR_SHAPE;
}

}  // namespace bsa
