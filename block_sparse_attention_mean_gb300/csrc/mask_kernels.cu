// mask_kernels.cu -- block-mask builder for sm_103a.
//
// Dynamic mode is the naive block-sparse selector of "Can sparse attention close
// the quality gap in diffusion transformers" (mean-pooled block scoring):
//   pool_kernel        Q, K [BH][N][d] -> Qbar, Kbar fp32 [BH][nB][d]   (HBM-bound)
//   score_kernel       every (Q block, KV block) score (fmaf chains, outer-product
//                      tiling, cp.async-staged chunks) as an order-preserving key in
//                      the workspace
//   select_kernel      per Q block: exact top-k by a bitwise radix select on the
//                      keys held in registers (over the few keys above a lane-maximum
//                      bound where k <= 32), emits the bitmap row and the CSR row
//                      (row_ptr = r * k, no scan).
// Static mode evaluates the block predicates of "多模态DiT中的块稀疏注意力" §3.1-§3.2
// (text dense + image band + anchors, or video cuboids + faces + text) or copies
// an explicit bitmap:
//   pattern_kernel + emit_pattern_kernel (one pattern for every head: band, cuboid,
//   broadcast bitmap): build it once, copy it into every head; per-head bitmaps use
//   static_rows_kernel -> counts, scan_kernel -> row_ptr, emit_kernel -> col_idx
//   ascending (§4.1 index forms).
// Arithmetic of the selector is fixed so results are reproducible bit for bit:
// pooled sums in token order with round-to-nearest adds, divided by the block's
// token count (round to nearest; a full block's 1/bs scaling is exact);
// scores as an fmaf chain over channels from +0; order by value with -0 == +0,
// ties to the lower block index.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>


#include "internal.h"
#include "ptx.cuh"

namespace bsa {
namespace {

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

constexpr int kPoolThreads = 128;

// ------------------------------------------------------------------ pooling

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&x)[8])
{
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void load8(const float *p, float (&x)[8])
{
    float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// One thread = 8 channels of one (bh, block); blockIdx.y picks Q (0) or K (1).
template <typename T>
__global__ void __launch_bounds__(kPoolThreads) pool_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                            float *__restrict__ qbar, float *__restrict__ kbar,
                                                            int64_t n_groups, int N, int d, int bs, int nB)
{
    const int64_t g = static_cast<int64_t>(blockIdx.x) * kPoolThreads + threadIdx.x;
    if (g >= n_groups) return;
    const T *X = blockIdx.y == 0 ? Q : K;
    float *out = blockIdx.y == 0 ? qbar : kbar;
    const int groups_per_row = d / 8;
    const int cg = static_cast<int>(g % groups_per_row);
    const int64_t rest = g / groups_per_row;
    const int i = static_cast<int>(rest % nB);
    const int64_t bh = rest / nB;
    const T *src = X + (bh * N + static_cast<int64_t>(i) * bs) * d + cg * 8;
    const int cnt = min(bs, N - i * bs);  // a ragged last block holds fewer tokens
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll 8
    for (int t = 0; t < cnt; ++t) {
        float x[8];
        load8(src + static_cast<int64_t>(t) * d, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
    }
    const float n = static_cast<float>(cnt);
    float *dst = out + (bh * nB + i) * static_cast<int64_t>(d) + cg * 8;
    float4 lo = make_float4(__fdiv_rn(acc[0], n), __fdiv_rn(acc[1], n), __fdiv_rn(acc[2], n), __fdiv_rn(acc[3], n));
    float4 hi = make_float4(__fdiv_rn(acc[4], n), __fdiv_rn(acc[5], n), __fdiv_rn(acc[6], n), __fdiv_rn(acc[7], n));
    reinterpret_cast<float4 *>(dst)[0] = lo;
    reinterpret_cast<float4 *>(dst)[1] = hi;
}

// ------------------------------------------------------------ score + top-k

// Order-preserving unsigned key of a float: larger float -> larger key,
// -0 and +0 map to the same key.
__device__ __forceinline__ uint32_t order_key(float s)
{
    uint32_t u = __float_as_uint(s);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exact top-k of one row of order keys held in shared memory (one warp): the k
// largest (key, -index) pairs, written as a bitmap row and an ascending CSR row.
// The k-th largest key of row[lo..hi) by a bitwise radix select (T), and how many
// keys equal to T to keep (the lowest indices first). k = 0 keeps nothing.
__device__ void kth_key(const uint32_t *row, int lo, int hi, int k, int lane, uint32_t &T, int &need)
{
    if (k <= 0 || lo >= hi) {
        T = 0xffffffffu;
        need = 0;
        return;
    }
    // Largest T with #{key >= T} >= k: the k-th largest key value.
    T = 0;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = T | (1u << bit);
        int cnt = 0;
        for (int j = lo + lane; j < hi; j += 32) cnt += row[j] >= cand;
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        if (cnt >= k) T = cand;
    }
    int gt = 0;
    for (int j = lo + lane; j < hi; j += 32) gt += row[j] > T;
    gt = __reduce_add_sync(0xffffffffu, gt);
    need = k - gt;
}

// Top kA keys among the text columns [0, n_text) and top kB among the image
// columns [n_text, nKB) of one row (ties: lower index first within each group);
// writes the row's bitmap words and, in ascending order from out_base, its
// col_idx entries. With n_text = 0 this is the plain top-kB of the row.
__device__ void select_row(const uint32_t *row, int nKB, int n_text, int kA, int kB, int W, int64_t r_global,
                           int64_t out_base, int32_t *__restrict__ col_idx, uint32_t *__restrict__ bitmap, int lane)
{
    uint32_t TA, TB;
    int needA, needB;
    kth_key(row, 0, n_text, kA, lane, TA, needA);
    kth_key(row, n_text, nKB, kB, lane, TB, needB);
    int taken = 0, tiesA = 0, tiesB = 0;
    for (int w = 0; w < W; ++w) {
        const int j = w * 32 + lane;
        const uint32_t key = j < nKB ? row[j] : 0u;
        const bool inA = j < n_text;
        const uint32_t T = inA ? TA : TB;
        const bool is_gt = j < nKB && key > T;
        const bool is_eq = j < nKB && key == T;
        const uint32_t eqA = __ballot_sync(0xffffffffu, is_eq && inA);
        const uint32_t eqB = __ballot_sync(0xffffffffu, is_eq && !inA);
        const int eq_rank = inA ? tiesA + __popc(eqA & lanemask_lt()) : tiesB + __popc(eqB & lanemask_lt());
        const bool sel = is_gt || (is_eq && eq_rank < (inA ? needA : needB));
        const uint32_t sel_mask = __ballot_sync(0xffffffffu, sel);
        if (lane == 0) bitmap[r_global * W + w] = sel_mask;
        if (sel) col_idx[out_base + taken + __popc(sel_mask & lanemask_lt())] = j;
        taken += __popc(sel_mask);
        tiesA += __popc(eqA);
        tiesB += __popc(eqB);
    }
}

// First col_idx slot of row i of head bh when text rows keep Kt blocks and image
// rows Ki (rows ordered (b, h, i); the first n_text rows of a head are text).
__device__ __forceinline__ int64_t row_base(int64_t bh, int i, int nQB, int n_text, int Kt, int Ki)
{
    const int64_t per_head = static_cast<int64_t>(n_text) * Kt + static_cast<int64_t>(nQB - n_text) * Ki;
    const int64_t within = i < n_text ? static_cast<int64_t>(i) * Kt
                                      : static_cast<int64_t>(n_text) * Kt + static_cast<int64_t>(i - n_text) * Ki;
    return bh * per_head + within;
}

// Scores of every (Q block, KV block) pair of a head, then top-k per Q block, in two
// launches:
//   score_kernel   an outer-product tiling over channels (the SGEMM pattern): a CTA
//                  stages 32-channel chunks of a 64-row Qbar tile and a 64-row Kbar
//                  tile in shared memory and each thread accumulates a 4 x 8 block of
//                  scores, so every staged value feeds 8 or 4 FMAs and a head's Kbar is
//                  read nQB/64 times, not once per Q block. Each score is still one fmaf
//                  chain over channels 0..d-1 in order from +0. The scores go to the
//                  workspace as order-preserving keys [BH][nQB][nKB].
//   select_kernel  one warp per Q block: the row's keys in registers (key j in lane
//                  j%32, slot j/32), an exact bitwise radix select of the k-th largest
//                  key, and the bitmap and ascending CSR row.
constexpr int kScoreTile = 64;     // Q blocks and KV blocks of a score tile
constexpr int kScoreThreads = 128;
constexpr int kScoreChunk = 32;    // channels per staged chunk
constexpr int kSelectWarps = 8;
constexpr int kSelectCand = 128;   // candidate keys the prefiltered search holds (4 per lane)

// Per-modality counts ("多模态DiT中的块稀疏注意力" §3.3): k[a][b] blocks kept among the
// key blocks of modality b (0 text, 1 image) by a query block of modality a; the
// plain selector is n_text = 0 with k[1][1] = k.
struct RegionK {
    int n_text;
    int k[2][2];
};

// Keys of a row outside columns [lo, hi) replaced by 0, which is below every radix
// candidate (a valid key is never 0: that would be the NaN 0xffffffff).
template <int R, int KPL>
__device__ __forceinline__ void keys_in_range(const uint32_t (&kv)[R][KPL], int lo, int hi, int lane,
                                              uint32_t (&x)[R][KPL])
{
#pragma unroll
    for (int q = 0; q < R; ++q)
#pragma unroll
        for (int m = 0; m < KPL; ++m) {
            const int j = 32 * m + lane;
            x[q][m] = j >= lo && j < hi ? kv[q][m] : 0u;
        }
}

// The k-th largest key of one row (slots outside the group hold 0) by a bitwise
// radix search, narrowed as it goes: it keeps the bounds T (at least k keys are
// >= T) and U (fewer than k keys are >= U); once at most 32 keys lie in [T, U) they
// are gathered into one register per lane (through buf, 32 words of this warp's
// shared memory) and the remaining bits test that register only. Returns T and how
// many keys equal to it to keep (the lowest columns first). k <= 0 keeps nothing.
template <int KPL>
__device__ __forceinline__ void kth_narrowing(const uint32_t (&x)[KPL], int k, int lane, uint32_t *buf,
                                              uint32_t &T, int &need)
{
    if (k <= 0) {
        T = 0xffffffffu;
        need = 0;
        return;
    }
    T = 0;
    uint64_t U = 1ull << 32;  // exclusive upper bound
    int cT = 32 * KPL, cU = 0;  // keys >= T (all slots, zeros included), keys >= U
    int bit = 31;
    for (; bit >= 0; --bit) {
        if (cT - cU <= 32) break;
        const uint32_t c = T | (1u << bit);
        int n = 0;
#pragma unroll
        for (int m = 0; m < KPL; ++m) n += x[m] >= c ? 1 : 0;
        n = static_cast<int>(__reduce_add_sync(0xffffffffu, n));
        if (n >= k) {
            T = c;
            cT = n;
        } else {
            U = c;
            cU = n;
        }
    }
    if (bit < 0) {  // every bit decided on the full row
        int g = 0;
#pragma unroll
        for (int m = 0; m < KPL; ++m) g += x[m] > T ? 1 : 0;
        need = k - static_cast<int>(__reduce_add_sync(0xffffffffu, g));
        return;
    }
    // gather the keys of [T, U) (at most 32) into buf, one per lane
    int off = 0;
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        const bool in = x[m] >= T && static_cast<uint64_t>(x[m]) < U;
        const uint32_t b = __ballot_sync(0xffffffffu, in);
        if (in) buf[off + __popc(b & lanemask_lt())] = x[m];
        off += __popc(b);
    }
    __syncwarp();
    const uint32_t y = lane < off ? buf[lane] : 0u;  // 0 is below every remaining candidate
    __syncwarp();
    for (; bit >= 0; --bit) {
        const uint32_t c = T | (1u << bit);
        // keys >= c: the cU keys at or above U plus the gathered ones
        const int n = cU + static_cast<int>(__reduce_add_sync(0xffffffffu, y >= c ? 1u : 0u));
        if (n >= k) T = c;
    }
    need = k - cU - static_cast<int>(__reduce_add_sync(0xffffffffu, y > T ? 1u : 0u));
}

// The k-th largest key among candidate keys gathered in buf[0, C) (NR words per lane,
// slots past C read as 0, below every candidate), all of them in [L, M] with M the largest:
// the bits above the highest bit in which L and M differ are M's, and the search decides
// the rest. Also returns how many keys equal to it to keep, and how many candidates equal it.
template <int NR>
__device__ __forceinline__ void kth_of_candidates(const uint32_t *buf, int C, int k, uint32_t L, uint32_t M,
                                                  int lane, uint32_t &T, int &need, int &n_eq)
{
    uint32_t y[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) y[r] = 32 * r + lane < C ? buf[32 * r + lane] : 0u;
    const uint32_t D = L ^ M;
    const int hb = D ? 31 - __clz(D) : -1;
    T = D ? M & ~((2u << hb) - 1u) : M;
    for (int bit = hb; bit >= 0; --bit) {
        const uint32_t c = T | (1u << bit);
        int n = 0;
#pragma unroll
        for (int r = 0; r < NR; ++r) n += __popc(__ballot_sync(0xffffffffu, y[r] >= c));
        if (n >= k) T = c;
    }
    int g = 0, e = 0;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        g += __popc(__ballot_sync(0xffffffffu, y[r] > T));
        e += __popc(__ballot_sync(0xffffffffu, y[r] == T));
    }
    need = k - g;
    n_eq = e;
}

// The k-th largest key of one row for 1 <= k <= 32 (slots outside the row hold 0). The k
// lanes with the largest maxima each hold a key >= the k-th largest lane maximum, so that
// maximum, and anything below it, is a lower bound on the k-th largest key; L is the k-th
// largest lane maximum with its low 16 bits cleared (found on the top 16 bits only, which
// is cheaper and still a lower bound). The k largest keys are all >= L; those keys (a few
// dozen on typical rows) are gathered into buf (kSelectCand words of this warp's shared
// memory) and searched bit by bit. Returns false, deciding nothing, when more than
// kSelectCand keys are >= L.
template <int KPL>
__device__ __forceinline__ bool kth_prefiltered(const uint32_t (&x)[KPL], int k, int lane, uint32_t *buf,
                                                uint32_t &T, int &need, int &n_eq)
{
    uint32_t mx = x[0];
#pragma unroll
    for (int m = 1; m < KPL; ++m) mx = max(mx, x[m]);
    const uint32_t M = __reduce_max_sync(0xffffffffu, mx);
    const uint32_t mn = __reduce_min_sync(0xffffffffu, mx);
    // the k-th largest lane maximum lies in [mn, M]: search below their common top bits
    const uint32_t D = (mn ^ M) & 0xFFFF0000u;
    uint32_t L = M & 0xFFFF0000u;
    if (D) {
        const int hb = 31 - __clz(D);
        L = M & ~((2u << hb) - 1u);
        for (int bit = hb; bit >= 16; --bit) {
            const uint32_t c = L | (1u << bit);
            if (__popc(__ballot_sync(0xffffffffu, mx >= c)) >= k) L = c;
        }
    }
    int C = 0;
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        const bool in = x[m] >= L;
        const uint32_t b = __ballot_sync(0xffffffffu, in);
        const int at = C + __popc(b & lanemask_lt());
        if (in && at < kSelectCand) buf[at] = x[m];
        C += __popc(b);
    }
    __syncwarp();
    if (C > kSelectCand) return false;
    if (C <= 32)
        kth_of_candidates<1>(buf, C, k, L, M, lane, T, need, n_eq);
    else if (C <= 64)
        kth_of_candidates<2>(buf, C, k, L, M, lane, T, need, n_eq);
    else
        kth_of_candidates<kSelectCand / 32>(buf, C, k, L, M, lane, T, need, n_eq);
    return true;
}

// Bitmap words and ascending col_idx of one row of the plain selector: keys above T plus
// the first `need` keys equal to T (ties: lower column first; all_ties: need is the number
// of keys equal to T, so every key >= T is kept). Lane l stores the bitmap
// words 32c + l.
template <int KPL>
__device__ __forceinline__ void emit_row_plain(const uint32_t (&kv)[KPL], int nKB, uint32_t T, int need,
                                               bool all_ties, int W,
                                               int64_t r_global, int64_t out_base, int32_t *__restrict__ col_idx,
                                               uint32_t *__restrict__ bitmap, int lane)
{
    int taken = 0, ties = 0;
    uint32_t word = 0;
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        if (m >= W) break;
        const int j = 32 * m + lane;
        const bool valid = j < nKB;
        bool sel;
        if (all_ties) {  // every key equal to T is kept
            sel = valid && kv[m] >= T;
        } else {
            const bool is_eq = valid && kv[m] == T;
            const uint32_t eq = __ballot_sync(0xffffffffu, is_eq);
            sel = (valid && kv[m] > T) || (is_eq && ties + __popc(eq & lanemask_lt()) < need);
            ties += __popc(eq);
        }
        const uint32_t sel_mask = __ballot_sync(0xffffffffu, sel);
        if (lane == (m & 31)) word = sel_mask;
        if (sel) col_idx[out_base + taken + __popc(sel_mask & lanemask_lt())] = j;
        taken += __popc(sel_mask);
        if ((m & 31) == 31 || m == W - 1) {  // words m & ~31 .. m are complete
            if ((m & ~31) + lane <= m) bitmap[r_global * W + (m & ~31) + lane] = word;
        }
    }
}

// Bitmap words and ascending col_idx of one row from its thresholds: text columns
// [0, n_text) keep keys above TA plus the first needA equal to it, image columns keep
// keys above TB plus the first needB equal to it (ties: lower column first).
template <int KPL>
__device__ __forceinline__ void emit_row_regs(const uint32_t (&kv)[KPL], int nKB, int n_text, uint32_t TA, int needA,
                                              uint32_t TB, int needB, int W, int64_t r_global, int64_t out_base,
                                              int32_t *__restrict__ col_idx, uint32_t *__restrict__ bitmap, int lane)
{
    int taken = 0, tiesA = 0, tiesB = 0;
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        if (m >= W) break;
        const int j = 32 * m + lane;
        const bool valid = j < nKB;
        const bool inA = j < n_text;
        const uint32_t T = inA ? TA : TB;
        const bool is_gt = valid && kv[m] > T;
        const bool is_eq = valid && kv[m] == T;
        const uint32_t eqA = __ballot_sync(0xffffffffu, is_eq && inA);
        const uint32_t eqB = __ballot_sync(0xffffffffu, is_eq && !inA);
        const int eq_rank = inA ? tiesA + __popc(eqA & lanemask_lt()) : tiesB + __popc(eqB & lanemask_lt());
        const bool sel = is_gt || (is_eq && eq_rank < (inA ? needA : needB));
        const uint32_t sel_mask = __ballot_sync(0xffffffffu, sel);
        if (lane == 0) bitmap[r_global * W + m] = sel_mask;
        if (sel) col_idx[out_base + taken + __popc(sel_mask & lanemask_lt())] = j;
        taken += __popc(sel_mask);
        tiesA += __popc(eqA);
        tiesB += __popc(eqB);
    }
}

// Shared memory of score_kernel: two stages, each a 32-channel chunk of 64 Qbar rows and of
// 64 Kbar rows, row-major with rows padded to 36 floats: the four consecutive Q rows and the
// eight consecutive K rows a warp reads per channel quad start 16 bytes apart in the bank
// space, so neither read conflicts, and every read is at a constant offset from the
// thread's row base. 36 KB: six CTAs share an SM.
constexpr int kScorePitch = kScoreChunk + 4;
constexpr int kScoreStageFloats = 2 * kScoreTile * kScorePitch;
size_t score_smem(int) { return sizeof(float) * 2 * static_cast<size_t>(kScoreStageFloats); }

// Starts the copy of channels [c0, c0 + 32) of rows [row0, row0 + 64) of one head's
// pooled blocks into dst (rows at or past n are zero-filled). Eight consecutive threads
// copy one row's 128 bytes.
__device__ __forceinline__ void stage_rows(const float *__restrict__ src, int row0, int n, int d, int c0,
                                           uint32_t dst)
{
#pragma unroll
    for (int u = 0; u < kScoreTile * 8 / kScoreThreads; ++u) {
        const int e = u * kScoreThreads + static_cast<int>(threadIdx.x);
        const int r = e >> 3, q4 = e & 7;
        const bool ok = row0 + r < n;
        cp_async16(dst + 4u * static_cast<uint32_t>(r * kScorePitch + 4 * q4),
                   ok ? src + static_cast<int64_t>(row0 + r) * d + c0 + 4 * q4 : src, ok ? 16u : 0u);
    }
}

// grid (BH, nQB tiles, nKB tiles), 64 x 64 scores per CTA. Thread (warp w, lane l): rows
// rg + 16a (rg = 4w + l%4, a < 4) and columns cg + 8n (cg = l/4, n < 8) of the tile. Per
// 4-channel quad a thread loads 4 Q and 8 K quads (16 bytes each) for 128 FMAs. The chunk
// after the current one is copied (cp.async) while the current one is consumed; the
// accumulators carry each score's fmaf chain on from quad to quad and chunk to chunk, so
// every score is one chain over channels 0..d-1 in order.
__global__ void __launch_bounds__(kScoreThreads, 6) score_kernel(const float *__restrict__ qbar,
                                                             const float *__restrict__ kbar, int nQB, int nKB,
                                                             int d, uint32_t *__restrict__ keys, uint32_t *err)
{
    extern __shared__ float4 sm4[];
    float *sm = reinterpret_cast<float *>(sm4);
    const int64_t bh = blockIdx.x;
    const int i0 = blockIdx.y * kScoreTile, j0 = blockIdx.z * kScoreTile;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = 4 * warp + (lane & 3);
    const int cg = lane >> 2;
    const float *qsrc = qbar + bh * nQB * static_cast<int64_t>(d);
    const float *ksrc = kbar + bh * nKB * static_cast<int64_t>(d);
    float acc[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int n = 0; n < 8; ++n) acc[a][n] = 0.0f;
    grid_dependency_wait();  // the pooled blocks come from the previous launch
    const int nch = d / kScoreChunk;
    const uint32_t sm_u = smem_u32(sm);
    stage_rows(qsrc, i0, nQB, d, 0, sm_u);
    stage_rows(ksrc, j0, nKB, d, 0, sm_u + 4u * kScoreTile * kScorePitch);
    cp_async_commit();
    for (int ch = 0; ch < nch; ++ch) {
        cp_async_wait_group<0>();
        __syncthreads();  // chunk ch is visible to every thread; the other stage is consumed
        if (ch + 1 < nch) {
            const uint32_t nx = sm_u + 4u * ((ch + 1) & 1) * kScoreStageFloats;
            stage_rows(qsrc, i0, nQB, d, (ch + 1) * kScoreChunk, nx);
            stage_rows(ksrc, j0, nKB, d, (ch + 1) * kScoreChunk, nx + 4u * kScoreTile * kScorePitch);
        }
        cp_async_commit();
        const float *qs = sm + (ch & 1) * kScoreStageFloats + rg * kScorePitch;
        const float *ks = sm + (ch & 1) * kScoreStageFloats + (kScoreTile + cg) * kScorePitch;
#pragma unroll 4
        for (int q4 = 0; q4 < kScoreChunk / 4; ++q4) {
            float4 qv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
                qv[a] = *reinterpret_cast<const float4 *>(qs + 16 * a * kScorePitch + 4 * q4);
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const float4 kv = *reinterpret_cast<const float4 *>(ks + 8 * n * kScorePitch + 4 * q4);
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    acc[a][n] = __fmaf_rn(qv[a].x, kv.x, acc[a][n]);
                    acc[a][n] = __fmaf_rn(qv[a].y, kv.y, acc[a][n]);
                    acc[a][n] = __fmaf_rn(qv[a].z, kv.z, acc[a][n]);
                    acc[a][n] = __fmaf_rn(qv[a].w, kv.w, acc[a][n]);
                }
            }
        }
    }
    bool nan_seen = false;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = i0 + rg + 16 * a;
        if (i >= nQB) continue;
        uint32_t *row = keys + (bh * nQB + i) * static_cast<int64_t>(nKB);
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int j = j0 + cg + 8 * n;
            if (j < nKB) {
                nan_seen |= isnan(acc[a][n]);
                row[j] = order_key(acc[a][n]);
            }
        }
    }
    if (nan_seen) raise_error(err, BSA_ERR_NONFINITE);
}

// One warp per Q block row r (of BH * nQB): top-k of the row's keys, bitmap and CSR.
template <int KPL>
__global__ void __launch_bounds__(32 * kSelectWarps, KPL <= 16 ? 4 : 1)
    select_kernel(const uint32_t *__restrict__ keys, int64_t R, int nQB, int nKB, RegionK rk, int W,
                  int32_t *__restrict__ row_ptr, int32_t *__restrict__ col_idx, uint32_t *__restrict__ bitmap)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kSelectWarps + (threadIdx.x >> 5);
    if (r >= R) return;
    const int64_t bh = r / nQB;
    const int i = static_cast<int>(r % nQB);
    const uint32_t *row = keys + r * nKB;
    grid_dependency_wait();  // the keys come from the previous launch
    uint32_t kv[1][KPL];
#pragma unroll
    for (int m = 0; m < KPL; ++m) {
        const int j = 32 * m + lane;
        kv[0][m] = j < nKB ? __ldg(row + j) : 0u;
    }
    __shared__ uint32_t gather[kSelectWarps][kSelectCand];
    uint32_t *buf = gather[threadIdx.x >> 5];
    const int qm = i < rk.n_text ? 0 : 1;
    uint32_t TA = 0xffffffffu, TB;
    int nA = 0, nB;
    if (rk.n_text == 0) {  // the plain selector: every column is in the image group
        const int k = rk.k[qm][1];
        const int Ki = rk.k[1][0] + rk.k[1][1];
        const int64_t base = static_cast<int64_t>(r) * Ki;
        int n_eq = -1;
        if (k < 1 || k > 32 || !kth_prefiltered<KPL>(kv[0], k, lane, buf, TB, nB, n_eq))
            kth_narrowing<KPL>(kv[0], k, lane, buf, TB, nB);
        emit_row_plain<KPL>(kv[0], nKB, TB, nB, n_eq == nB, W, r, base, col_idx, bitmap, lane);
        if (lane == 0) {
            row_ptr[r] = static_cast<int32_t>(base);
            if (r == R - 1) row_ptr[R] = static_cast<int32_t>(base + Ki);
        }
        return;
    } else {
        uint32_t x[1][KPL];
        keys_in_range<1, KPL>(kv, 0, rk.n_text, lane, x);
        kth_narrowing<KPL>(x[0], rk.k[qm][0], lane, buf, TA, nA);
        keys_in_range<1, KPL>(kv, rk.n_text, nKB, lane, x);
        kth_narrowing<KPL>(x[0], rk.k[qm][1], lane, buf, TB, nB);
    }
    const int Kt = rk.k[0][0] + rk.k[0][1], Ki = rk.k[1][0] + rk.k[1][1];
    const int64_t base = row_base(bh, i, nQB, rk.n_text, Kt, Ki);
    emit_row_regs<KPL>(kv[0], nKB, rk.n_text, TA, nA, TB, nB, W, r, base, col_idx, bitmap, lane);
    if (lane == 0) {
        row_ptr[r] = static_cast<int32_t>(base);
        if (r == R - 1) row_ptr[R] = static_cast<int32_t>(row_base(bh + 1, 0, nQB, rk.n_text, Kt, Ki));
    }
}

template <int KPL>
bsa_status launch_select(const uint32_t *keys, const MaskArgs &a, const RegionK &rk, int64_t R, cudaStream_t st)
{
    const dim3 g(static_cast<unsigned>((R + kSelectWarps - 1) / kSelectWarps));
    return pdl_launch(select_kernel<KPL>, g, 32 * kSelectWarps, 0, st, keys, R, a.nQB, a.nKB, rk, a.W, a.row_ptr,
                      a.col_idx, a.bitmap)
               ? BSA_OK
               : BSA_ERR_CUDA;
}

// ------------------------------------------------------------ static masks

struct StaticPred {
    int kind, n_text, band, n_anchors, gt, gh, gw, broadcast;
    int anchors[BSA_MAX_ANCHORS];
};

__device__ __forceinline__ bool static_active(const StaticPred &p, int i, int j)
{
    if (i < p.n_text || j < p.n_text) return true;
    const int r = i - p.n_text, c = j - p.n_text;
    if (p.kind == BSA_STATIC_MODALITY_BAND) {
        if (abs(r - c) <= p.band) return true;
        for (int a = 0; a < p.n_anchors; ++a)
            if (r == p.anchors[a] || c == p.anchors[a]) return true;
        return false;
    }
    // cuboid: t-major raster over (gt, gh, gw); same cuboid or a shared face
    const int hw = p.gh * p.gw;
    const int rt = r / hw, rh = (r / p.gw) % p.gh, rw = r % p.gw;
    const int ct = c / hw, ch = (c / p.gw) % p.gh, cw = c % p.gw;
    return abs(rt - ct) + abs(rh - ch) + abs(rw - cw) <= 1;
}

// One warp per index row r = bh * nQB + i.
__global__ void __launch_bounds__(256) static_rows_kernel(StaticPred p, int64_t R, int nQB, int nKB, int W,
                                                          const uint32_t *__restrict__ src,
                                                          uint32_t *__restrict__ bitmap,
                                                          int32_t *__restrict__ counts)
{
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= R) return;
    const int i = static_cast<int>(r % nQB);
    int count = 0;
    for (int w = 0; w < W; ++w) {
        uint32_t word;
        if (p.kind == BSA_STATIC_EXPLICIT) {
            const int64_t srow = p.broadcast ? i : r;
            word = src[srow * W + w];
            const int valid = nKB - w * 32;
            if (valid < 32) word &= (1u << valid) - 1u;
        } else {
            const int j = w * 32 + lane;
            word = __ballot_sync(0xffffffffu, j < nKB && static_active(p, i, j));
        }
        if (lane == 0) bitmap[r * W + w] = word;
        count += __popc(word);
    }
    if (lane == 0) counts[r] = count;
}

// Masks shared by every (b, h) (band, cuboid, broadcast bitmap). The pattern of
// one head is built once by pattern_kernel (bitmap words and per-row counts,
// scanned by the CTA that finishes last), then emit_pattern_kernel writes every
// head's bitmap, row_ptr and col_idx from it, head bh offset by bh * nnz_per_head.
__device__ __forceinline__ uint32_t static_word(const StaticPred &p, const uint32_t *src, int i, int w, int nKB,
                                                int lane)
{
    if (p.kind == BSA_STATIC_EXPLICIT) {
        uint32_t word = src[static_cast<int64_t>(i) * ((nKB + 31) / 32) + w];
        const int valid = nKB - w * 32;
        if (valid < 32) word &= (1u << valid) - 1u;
        return word;
    }
    const int j = w * 32 + lane;
    return __ballot_sync(0xffffffffu, j < nKB && static_active(p, i, j));
}

// pat_rp: [nQB + 1] row offsets within a head; pat_bm: [nQB][W].
// One warp per pattern row (bitmap words + count); the CTA that finishes last
// scans the counts.
__global__ void __launch_bounds__(256) pattern_kernel(StaticPred p, int nQB, int nKB, int W,
                                                      const uint32_t *__restrict__ src, int32_t *__restrict__ pat_rp,
                                                      uint32_t *__restrict__ pat_bm, uint32_t *done)
{
    __shared__ int32_t wsum[8];
    __shared__ bool is_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + warp;
    if (i < nQB) {
        int c = 0;
        for (int w = 0; w < W; ++w) {
            const uint32_t word = static_word(p, src, i, w, nKB, lane);
            if (lane == 0) pat_bm[static_cast<int64_t>(i) * W + w] = word;
            c += __popc(word);
        }
        if (lane == 0) pat_rp[i + 1] = c;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // inclusive scan of pat_rp[1..nQB] (each thread scans a contiguous chunk)
    const int chunk = (nQB + blockDim.x - 1) / blockDim.x;
    const int b = threadIdx.x * chunk, e = min(nQB, b + chunk);
    int local = 0;
    for (int r = b; r < e; ++r) local += __ldcg(pat_rp + r + 1);
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int v = lane < 8 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (lane < 8) wsum[lane] = v;
    }
    __syncthreads();
    int run = x - local + (warp > 0 ? wsum[warp - 1] : 0);
    for (int r = b; r < e; ++r) {
        const int c = __ldcg(pat_rp + r + 1);
        pat_rp[r + 1] = run + c;
        run += c;
    }
    if (threadIdx.x == 0) {
        pat_rp[0] = 0;
        *done = 0u;
    }
}

// One warp per index row r = bh * nQB + i: copies pattern row i into head bh
// (bitmap words, row_ptr = bh * nnz_per_head + pattern offset, col_idx).
__global__ void __launch_bounds__(256) emit_pattern_kernel(int64_t R, int nQB, int W, const int32_t *__restrict__ pat_rp,
                                                           const uint32_t *__restrict__ pat_bm,
                                                           uint32_t *__restrict__ bitmap, int32_t *__restrict__ row_ptr,
                                                           int32_t *__restrict__ col_idx, int64_t capacity, uint32_t *err)
{
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= R) return;
    const int i = static_cast<int>(r % nQB);
    const int64_t bh = r / nQB;
    const int64_t nnz_head = pat_rp[nQB];
    int64_t pos = bh * nnz_head + pat_rp[i];
    if (lane == 0) {
        row_ptr[r] = static_cast<int32_t>(pos);
        if (r == R - 1) row_ptr[R] = static_cast<int32_t>((bh + 1) * nnz_head);
    }
    bool overflow = false;
    for (int w = 0; w < W; ++w) {
        const uint32_t word = pat_bm[static_cast<int64_t>(i) * W + w];
        if (lane == 0) bitmap[r * W + w] = word;
        if ((word >> lane) & 1u) {
            const int64_t q = pos + __popc(word & lanemask_lt());
            if (q < capacity) col_idx[q] = w * 32 + lane;
            else overflow = true;
        }
        pos += __popc(word);
    }
    if (overflow) raise_error(err, BSA_ERR_CAPACITY);
}

// Exclusive scan of R counts into row_ptr[0..R] (one CTA of 1024 threads).
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t *__restrict__ counts, int64_t R,
                                                    int32_t *__restrict__ row_ptr)
{
    __shared__ int64_t warp_sums[32];
    const int t = threadIdx.x;
    const int64_t chunk = (R + 1023) / 1024;
    const int64_t b = t * chunk, e = min(R, b + chunk);
    int64_t local = 0;
    for (int64_t r = b; r < e; ++r) local += counts[r];
    // inclusive scan of `local` across the CTA
    int64_t x = local;
    const int lane = t & 31, warp = t >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    int64_t run = x - local + (warp > 0 ? warp_sums[warp - 1] : 0);
    for (int64_t r = b; r < e; ++r) {
        row_ptr[r] = static_cast<int32_t>(run);
        run += counts[r];
    }
    if (t == 1023) row_ptr[R] = static_cast<int32_t>(warp_sums[31]);
}

// One warp per row: col_idx from the bitmap in ascending order.
__global__ void __launch_bounds__(256) emit_kernel(const uint32_t *__restrict__ bitmap,
                                                   const int32_t *__restrict__ row_ptr, int64_t R, int W,
                                                   int32_t *__restrict__ col_idx, int64_t capacity,
                                                   uint32_t *err)
{
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= R) return;
    int64_t pos = row_ptr[r];
    bool overflow = false;
    for (int w = 0; w < W; ++w) {
        const uint32_t word = bitmap[r * W + w];
        if ((word >> lane) & 1u) {
            const int64_t p = pos + __popc(word & lanemask_lt());
            if (p < capacity) col_idx[p] = w * 32 + lane;
            else overflow = true;
        }
        pos += __popc(word);
    }
    if (overflow) raise_error(err, BSA_ERR_CAPACITY);
}

// One warp per row: structural checks of a CSR + bitmap index.
__global__ void __launch_bounds__(256) validate_kernel(const int32_t *__restrict__ row_ptr,
                                                       const int32_t *__restrict__ col_idx,
                                                       const uint32_t *__restrict__ bitmap, int64_t R,
                                                       int nKB, int W, uint32_t *err)
{
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= R) return;
    const int32_t b = row_ptr[r], e = row_ptr[r + 1];
    bool bad = (r == 0 && b != 0) || e < b;
    if (!bad) {
        for (int32_t p = b + lane; p < e; p += 32) {
            const int32_t c = col_idx[p];
            if (c < 0 || c >= nKB) bad = true;
            else if (p > b && col_idx[p - 1] >= c) bad = true;
            else if (bitmap && !((bitmap[r * W + c / 32] >> (c % 32)) & 1u)) bad = true;
        }
        if (bitmap) {
            int pc = 0;
            for (int w = lane; w < W; w += 32) {
                uint32_t word = bitmap[r * W + w];
                const int valid = nKB - w * 32;
                if (valid < 32 && (word >> valid) != 0u) bad = true;
                pc += __popc(word);
            }
            pc = __reduce_add_sync(0xffffffffu, pc);
            if (pc != e - b) bad = true;
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(err, BSA_ERR_INVALID_ARG);
}

}  // namespace

// Workspace after the header: the dynamic path uses Qbar and Kbar; the static
// path uses per-row counts (per-head bitmaps) and one head's pattern
// (row offsets, bitmap words).
struct MaskWs {
    size_t qbar, kbar, keys;                    // dynamic
    size_t counts, pat_rp, pat_bm;              // static
    size_t dyn_end, static_end;                 // bytes a dynamic / static build touches
    size_t total;
};

MaskWs mask_ws_layout(int B, int H, int N, int d, int block)
{
    const size_t BH = static_cast<size_t>(B) * H;
    const size_t nB = static_cast<size_t>((N + block - 1) / block);
    const size_t W = (nB + 31) / 32;
    MaskWs l{};
    l.qbar = kWsHeader;
    l.kbar = l.qbar + align_up(BH * nB * d * sizeof(float), 256);
    l.keys = l.kbar + align_up(BH * nB * d * sizeof(float), 256);
    const size_t dyn_end = l.keys + align_up(BH * nB * nB * sizeof(uint32_t), 256);
    l.counts = kWsHeader;
    l.pat_rp = l.counts + align_up(BH * nB * sizeof(int32_t), 256);
    l.pat_bm = l.pat_rp + align_up((nB + 1) * sizeof(int32_t), 256);
    const size_t static_end = l.pat_bm + align_up(nB * W * sizeof(uint32_t), 256);
    l.total = dyn_end > static_end ? dyn_end : static_end;
    l.dyn_end = dyn_end;
    l.static_end = static_end;
    return l;
}

size_t mask_workspace_bytes(int B, int H, int N, int d, int block)
{
    return mask_ws_layout(B, H, N, d, block).total;
}

size_t mask_workspace_need(int B, int H, int N, int d, int block, bool dynamic)
{
    const MaskWs l = mask_ws_layout(B, H, N, d, block);
    return dynamic ? l.dyn_end : l.static_end;
}

bsa_status launch_build_mask(const MaskArgs &a, cudaStream_t st)
{
    const int64_t BH = static_cast<int64_t>(a.B) * a.H;
    const int64_t R = BH * a.nQB;
    uint32_t *err = reinterpret_cast<uint32_t *>(a.ws);
    const MaskWs l = mask_ws_layout(a.B, a.H, a.N, a.d, a.block);
    float *qbar = reinterpret_cast<float *>(a.ws + l.qbar);
    float *kbar = reinterpret_cast<float *>(a.ws + l.kbar);
    int32_t *counts = reinterpret_cast<int32_t *>(a.ws + l.counts);

    if (a.spec == nullptr) {
        RegionK rk{};
        rk.n_text = a.n_text;
        for (int x = 0; x < 2; ++x)
            for (int y = 0; y < 2; ++y) rk.k[x][y] = a.kq[x][y];
        uint32_t *keys = reinterpret_cast<uint32_t *>(a.ws + l.keys);
        const size_t smem = score_smem(a.d);
        if (cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
                cudaSuccess ||
            cudaFuncSetAttribute(score_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return BSA_ERR_CUDA;
        const int64_t groups = BH * a.nQB * (a.d / 8);
        const dim3 pg(static_cast<unsigned>((groups + kPoolThreads - 1) / kPoolThreads), 2);
        if (a.dt == BSA_BF16)
            pool_kernel<__nv_bfloat16><<<pg, kPoolThreads, 0, st>>>(
                static_cast<const __nv_bfloat16 *>(a.Q), static_cast<const __nv_bfloat16 *>(a.K), qbar, kbar,
                groups, a.N, a.d, a.block, a.nQB);
        else
            pool_kernel<float><<<pg, kPoolThreads, 0, st>>>(static_cast<const float *>(a.Q),
                                                            static_cast<const float *>(a.K), qbar, kbar, groups,
                                                            a.N, a.d, a.block, a.nQB);
        // the scoring and the selection wait for their inputs with griddepcontrol.wait, so each
        // is set up while the launch before it drains
        const dim3 sg(static_cast<unsigned>(BH), (a.nQB + kScoreTile - 1) / kScoreTile,
                      (a.nKB + kScoreTile - 1) / kScoreTile);
        if (!pdl_launch(score_kernel, sg, kScoreThreads, smem, st, static_cast<const float *>(qbar),
                        static_cast<const float *>(kbar), a.nQB, a.nKB, a.d, keys, err))
            return BSA_ERR_CUDA;
        // keys per lane of the register-held rows: nKB <= 32 * KPL
        const bsa_status s = a.nKB <= 128   ? launch_select<4>(keys, a, rk, R, st)
                             : a.nKB <= 512 ? launch_select<16>(keys, a, rk, R, st)
                                            : launch_select<64>(keys, a, rk, R, st);
        if (s != BSA_OK) return s;
    } else {
        StaticPred pr{};
        pr.kind = a.spec->kind;
        pr.n_text = a.spec->n_text_blocks;
        pr.band = a.spec->band;
        pr.n_anchors = a.spec->n_anchors;
        for (int t = 0; t < BSA_MAX_ANCHORS; ++t) pr.anchors[t] = a.spec->anchors[t];
        pr.gt = a.spec->grid_t;
        pr.gh = a.spec->grid_h;
        pr.gw = a.spec->grid_w;
        pr.broadcast = a.spec->broadcast_bh;
        if (pr.kind != BSA_STATIC_EXPLICIT || pr.broadcast) {
            // one pattern for every (b, h): build it once, then copy it into every head
            int32_t *pat_rp = reinterpret_cast<int32_t *>(a.ws + l.pat_rp);     // [nQB + 1]
            uint32_t *pat_bm = reinterpret_cast<uint32_t *>(a.ws + l.pat_bm);   // [nQB][W]
            WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
            pattern_kernel<<<(a.nQB + 7) / 8, 256, 0, st>>>(pr, a.nQB, a.nKB, a.W, a.spec->bitmap, pat_rp, pat_bm,
                                                            &hdr->order_done);
            emit_pattern_kernel<<<static_cast<unsigned>((R + 7) / 8), 256, 0, st>>>(
                R, a.nQB, a.W, pat_rp, pat_bm, a.bitmap, a.row_ptr, a.col_idx, a.col_capacity, err);
        } else {
            const unsigned g = static_cast<unsigned>((R + 7) / 8);
            static_rows_kernel<<<g, 256, 0, st>>>(pr, R, a.nQB, a.nKB, a.W, a.spec->bitmap, a.bitmap, counts);
            scan_kernel<<<1, 1024, 0, st>>>(counts, R, a.row_ptr);
            emit_kernel<<<g, 256, 0, st>>>(a.bitmap, a.row_ptr, R, a.W, a.col_idx, a.col_capacity, err);
        }
    }
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

// ------------------------------------------------------------ exact block-mass selection
//
// One warp per row (b, h, i): the block masses of the row are the sum of its Q block's
// partials in a fixed order (warps 2h, 2h + 1 of the tile at block size 64, warps
// 0..3 at 128), then the same exact top-k as the mean-pooled selector.
constexpr int kSelWarps = 8;

__global__ void __launch_bounds__(kSelWarps * 32) mass_select_kernel(const float *__restrict__ part, int64_t R,
                                                                     int nQB, int nKB, int BS, int tiles_per_bh, int k,
                                                                     int W, int32_t *__restrict__ row_ptr,
                                                                     int32_t *__restrict__ col_idx,
                                                                     uint32_t *__restrict__ bitmap, uint32_t *err)
{
    extern __shared__ uint32_t sel_keys[];  // [kSelWarps][nKB]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kSelWarps + warp;
    if (r >= R) return;
    uint32_t *keys = sel_keys + warp * nKB;
    const int64_t bh = r / nQB;
    const int i = static_cast<int>(r % nQB);
    const int qt = BS == 128 ? i : i / 2;
    const float *base = part + (bh * tiles_per_bh + qt) * 4 * static_cast<int64_t>(nKB);
    bool nan_seen = false;
    for (int j = lane; j < nKB; j += 32) {
        float m;
        if (BS == 128) {
            m = ((base[j] + base[nKB + j]) + base[2 * nKB + j]) + base[3 * nKB + j];
        } else {
            const int h = i % 2;
            m = base[(2 * h) * nKB + j] + base[(2 * h + 1) * nKB + j];
        }
        nan_seen |= isnan(m);
        keys[j] = order_key(m);
    }
    if (__any_sync(0xffffffffu, nan_seen) && lane == 0) raise_error(err, BSA_ERR_NONFINITE);
    __syncwarp();
    select_row(keys, nKB, 0, 0, k, W, r, r * k, col_idx, bitmap, lane);
    if (lane == 0) {
        row_ptr[r] = static_cast<int32_t>(r * k);
        if (r == R - 1) row_ptr[R] = static_cast<int32_t>(R * k);
    }
}

bsa_status launch_mass_select(const float *part, const ExactArgs &a, int tiles_per_bh, cudaStream_t st)
{
    const int64_t R = static_cast<int64_t>(a.B) * a.H * a.nQB;
    const size_t smem = sizeof(uint32_t) * kSelWarps * a.nKB;
    if (cudaFuncSetAttribute(mass_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return BSA_ERR_CUDA;
    const unsigned g = static_cast<unsigned>((R + kSelWarps - 1) / kSelWarps);
    mass_select_kernel<<<g, kSelWarps * 32, smem, st>>>(part, R, a.nQB, a.nKB, a.block, tiles_per_bh, a.k, a.W,
                                                        a.row_ptr, a.col_idx, a.bitmap,
                                                        reinterpret_cast<uint32_t *>(a.ws));
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

// ------------------------------------------------------------ token selection
//
// "Can sparse attention close the quality gap in diffusion transformers", sections
// "质量差距有三个可分离来源" (the token oracle) and "token 级选择需要瓦片对齐的查询分组": per group
// g of 128 queries (rows perm[g*128 ..] of a head) and key token t,
//   mass[g][t] = sum over rows r of g of exp(scale * q_r . k_t - LSE_r),
// with the dense row logsumexp, then the n_keep tokens of largest mass (ties to the lower
// index) in ascending order: the same exact top-k as the block selectors, on a row of N keys.
//
// One CTA per (b, h, group), on CUDA cores (first path): the group's rows are gathered
// into shared memory; per chunk of 32 tokens, lane l of warp w sums exp over the warp's 16
// rows for token l, the 8 warp sums are added in warp order, and the mass goes to the
// workspace and, as an order key, to a shared-memory row that warp 0 then selects from.
template <typename T, int D>
__global__ void __launch_bounds__(256) token_select_kernel(const T *__restrict__ Q, const T *__restrict__ K, int N,
                                                           const int32_t *__restrict__ perm,
                                                           const float *__restrict__ LSE, float scale, int n_keep,
                                                           float *__restrict__ mass, uint32_t *__restrict__ bitmap,
                                                           int32_t *__restrict__ tokens, uint32_t *err)
{
    constexpr int C = kTokenGroup, RPW = C / 8;
    extern __shared__ float tsm[];
    float *qs = tsm;                                                // [C][D]
    float *ks = qs + C * D;                                         // [32][D + 1]
    uint32_t *keys = reinterpret_cast<uint32_t *>(ks + 32 * (D + 1));  // [N]
    __shared__ int32_t rows[C];
    __shared__ float lse[C];
    __shared__ float colsum[8][32];
    const int g = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int G = N / C;
    const int64_t rg = bh * G + g;  // selection row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = threadIdx.x; r < C; r += blockDim.x) {
        int row = perm[bh * N + static_cast<int64_t>(g) * C + r];
        if (row < 0 || row >= N) {
            raise_error(err, BSA_ERR_INVALID_ARG);
            row = -1;
        }
        rows[r] = row;
        lse[r] = row >= 0 ? LSE[bh * N + row] : CUDART_INF_F;  // a skipped row adds nothing
    }
    __syncthreads();
    for (int e = threadIdx.x; e < C * D; e += blockDim.x) {
        const int r = e / D, c = e % D;
        qs[e] = rows[r] >= 0 ? static_cast<float>(Q[(bh * N + rows[r]) * D + c]) : 0.0f;
    }
    bool nan_seen = false;
    for (int c0 = 0; c0 < N; c0 += 32) {
        __syncthreads();
        for (int e = threadIdx.x; e < 32 * D; e += blockDim.x) {
            const int kk = e / D, c = e % D;
            ks[kk * (D + 1) + c] = static_cast<float>(K[(bh * N + c0 + kk) * D + c]);
        }
        __syncthreads();
        const float *k = ks + lane * (D + 1);
        float acc = 0.0f;
        for (int r = 0; r < RPW; ++r) {
            const int rr = warp * RPW + r;
            const float *q = qs + rr * D;
            float s = 0.0f;
#pragma unroll 16
            for (int c = 0; c < D; ++c) s = fmaf(q[c], k[c], s);
            acc += expf(s * scale - lse[rr]);
        }
        colsum[warp][lane] = acc;
        __syncthreads();
        if (warp == 0) {
            float m = colsum[0][lane];
#pragma unroll
            for (int w = 1; w < 8; ++w) m += colsum[w][lane];
            nan_seen |= isnan(m);
            mass[rg * N + c0 + lane] = m;
            keys[c0 + lane] = order_key(m);
        }
    }
    __syncthreads();
    if (warp == 0) {
        if (__any_sync(0xffffffffu, nan_seen) && lane == 0) raise_error(err, BSA_ERR_NONFINITE);
        select_row(keys, N, 0, 0, n_keep, N / 32, rg, rg * n_keep, tokens, bitmap, lane);
    }
}

template <typename T, int D>
static bsa_status launch_token_select(const TokenSelectArgs &a, cudaStream_t st)
{
    const TokenSelectWs l = token_select_ws_layout(a.B, a.H, a.N);
    const size_t smem = sizeof(float) * (kTokenGroup * D + 32 * (D + 1)) + sizeof(uint32_t) * a.N;
    if (cudaFuncSetAttribute(token_select_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return BSA_ERR_CUDA;
    dim3 grid(a.N / kTokenGroup, a.B * a.H);
    token_select_kernel<T, D><<<grid, 256, smem, st>>>(
        static_cast<const T *>(a.Q), static_cast<const T *>(a.K), a.N, a.perm, a.LSE, a.scale, a.n_keep,
        reinterpret_cast<float *>(a.ws + l.mass), reinterpret_cast<uint32_t *>(a.ws + l.bitmap), a.tokens,
        reinterpret_cast<uint32_t *>(a.ws));
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

// The n_keep tokens of largest mass of one selection row (one group of one head), from
// the masses in global memory, for any N: an exact radix select with 8-bit digits (four
// passes, each a shared-memory histogram of the keys that match the digits found so far),
// then the bitmap words and the ascending token list (keys above the threshold, and the
// lowest-indexed keys equal to it). Ties go to the lower index, as in select_row.
constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;

__global__ void __launch_bounds__(kTopkThreads) token_topk_kernel(const float *__restrict__ mass, int N, int n_keep,
                                                                  uint32_t *__restrict__ bitmap,
                                                                  int32_t *__restrict__ tokens, uint32_t *err)
{
    __shared__ int hist[kTopkWarps][256];
    __shared__ int total[256];
    __shared__ int s_digit, s_krem;
    __shared__ int w_gt[kTopkWarps], w_eq[kTopkWarps];
    const int64_t rg = blockIdx.x;
    const float *row = mass + rg * N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t prefix = 0u, pmask = 0u;
    int krem = n_keep;
    bool nan_seen = false;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < kTopkWarps * 256; i += kTopkThreads) (&hist[0][0])[i] = 0;
        __syncthreads();
        for (int t = threadIdx.x; t < N; t += kTopkThreads) {
            const float m = __ldg(row + t);
            if (pass == 0) nan_seen |= isnan(m);
            const uint32_t key = order_key(m);
            if ((key & pmask) == prefix) atomicAdd(&hist[warp][(key >> shift) & 255u], 1);
        }
        __syncthreads();
        for (int dg = threadIdx.x; dg < 256; dg += kTopkThreads) {
            int c = 0;
#pragma unroll
            for (int w = 0; w < kTopkWarps; ++w) c += hist[w][dg];
            total[dg] = c;
        }
        __syncthreads();
        if (warp == 0) {
            // lane l covers digits 255 - 8l down to 248 - 8l: counts above each lane by a scan
            int cnt[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                cnt[i] = total[255 - 8 * lane - i];
                sum += cnt[i];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - sum;  // matching keys with a larger digit than this lane's
            const unsigned who = __ballot_sync(0xffffffffu, excl < krem && krem <= incl);
            if (lane == __ffs(who) - 1) {
                int above = excl;
                for (int i = 0; i < 8; ++i) {
                    if (above + cnt[i] >= krem) {
                        s_digit = 255 - 8 * lane - i;
                        s_krem = krem - above;
                        break;
                    }
                    above += cnt[i];
                }
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(s_digit) << shift;
        pmask |= 0xFFu << shift;
        krem = s_krem;
        __syncthreads();  // every thread has read s_digit / s_krem
    }
    if (__syncthreads_or(nan_seen) && threadIdx.x == 0) raise_error(err, BSA_ERR_NONFINITE);
    // keys above T = prefix, plus the first `krem` keys equal to it; each warp takes a
    // contiguous range of 32-key words, counted first so that its output offset is known
    const uint32_t T = prefix;
    const int need = krem, W = N / 32;
    const int per = (W + kTopkWarps - 1) / kTopkWarps;
    const int w0 = warp * per, w1 = min(W, w0 + per);
    int cgt = 0, ceq = 0;
    for (int w = w0; w < w1; ++w) {
        const uint32_t key = order_key(__ldg(row + 32 * w + lane));
        cgt += __popc(__ballot_sync(0xffffffffu, key > T));
        ceq += __popc(__ballot_sync(0xffffffffu, key == T));
    }
    if (lane == 0) {
        w_gt[warp] = cgt;
        w_eq[warp] = ceq;
    }
    __syncthreads();
    int eq_before = 0, out = 0;
    for (int w = 0; w < warp; ++w) {
        out += w_gt[w] + max(0, min(w_eq[w], need - eq_before));
        eq_before += w_eq[w];
    }
    const int64_t base = rg * n_keep;
    for (int w = w0; w < w1; ++w) {
        const int j = 32 * w + lane;
        const uint32_t key = order_key(__ldg(row + j));
        const uint32_t eq = __ballot_sync(0xffffffffu, key == T);
        const bool sel = key > T || (key == T && eq_before + __popc(eq & lanemask_lt()) < need);
        const uint32_t sm = __ballot_sync(0xffffffffu, sel);
        if (lane == 0) bitmap[rg * W + w] = sm;
        if (sel) tokens[base + out + __popc(sm & lanemask_lt())] = j;
        out += __popc(sm);
        eq_before += __popc(eq);
    }
}

TokenSelectWs token_select_ws_layout(int B, int H, int N)
{
    const size_t rows = static_cast<size_t>(B) * H * (N / kTokenGroup);
    TokenSelectWs l{};
    l.mass = kWsHeader;
    l.bitmap = l.mass + align_up(rows * N * sizeof(float), 256);
    l.total = l.bitmap + align_up(rows * (N / 32) * sizeof(uint32_t), 256);
    return l;
}

bsa_status launch_select_tokens(const TokenSelectArgs &a, cudaStream_t st)
{
    if (a.dt == BSA_BF16) {
        // masses on tcgen05 into the workspace, then the radix top-k of every group's row
        const TokenSelectWs l = token_select_ws_layout(a.B, a.H, a.N);
        float *mass = reinterpret_cast<float *>(a.ws + l.mass);
        const bsa_status s = launch_token_mass_tc(a, mass, st);
        if (s != BSA_OK) return s;
        const int64_t rows = static_cast<int64_t>(a.B) * a.H * (a.N / kTokenGroup);
        token_topk_kernel<<<static_cast<unsigned>(rows), kTopkThreads, 0, st>>>(
            mass, a.N, a.n_keep, reinterpret_cast<uint32_t *>(a.ws + l.bitmap), a.tokens,
            reinterpret_cast<uint32_t *>(a.ws));
        return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
    } else {
        if (a.d == 64) return launch_token_select<float, 64>(a, st);
        if (a.d == 128) return launch_token_select<float, 128>(a, st);
    }
    return BSA_ERR_SHAPE;
}

bsa_status launch_validate_index(int R, int nKB, const int32_t *row_ptr, const int32_t *col_idx,
                                 const uint32_t *bitmap, char *ws, cudaStream_t st)
{
    const int W = (nKB + 31) / 32;
    const unsigned g = static_cast<unsigned>((static_cast<int64_t>(R) + 7) / 8);
    validate_kernel<<<g, 256, 0, st>>>(row_ptr, col_idx, bitmap, R, nKB, W, reinterpret_cast<uint32_t *>(ws));
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace bsa
