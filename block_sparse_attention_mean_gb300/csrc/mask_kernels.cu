// mask_kernels.cu -- block-mask builder for sm_103a.
//
// Dynamic mode is the naive block-sparse selector of "Can sparse attention close
// the quality gap in diffusion transformers" (mean-pooled block scoring):
//   pool_kernel        Q, K [BH][N][d] -> Qbar, Kbar fp32 [BH][nB][d]   (HBM-bound)
//   score_topk_kernel  per Q block: nKB scores (fmaf chains), exact top-k by a
//                      bitwise radix select on order-preserving keys, emits the
//                      bitmap row and the CSR row (row_ptr = r * k, no scan).
// Static mode evaluates the block predicates of "多模态DiT中的块稀疏注意力" §3.1-§3.2
// (text dense + image band + anchors, or video cuboids + faces + text) or copies
// an explicit bitmap:
//   static_rows_kernel -> bitmap + per-row counts; scan_kernel -> row_ptr;
//   emit_kernel -> col_idx ascending (§4.1 index forms).
// Arithmetic of the selector is fixed so results are reproducible bit for bit:
// pooled sums in token order with round-to-nearest adds, scaled by 1/bs (exact);
// scores as an fmaf chain over channels from +0; order by value with -0 == +0,
// ties to the lower block index.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace bsa {
namespace {

constexpr int kPoolThreads = 128;
constexpr int kRowsPerCta = 8;   // Q blocks per score/top-k CTA (one warp each)
constexpr int kKvTile = 32;      // KV blocks staged per step

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

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
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll 8
    for (int t = 0; t < bs; ++t) {
        float x[8];
        load8(src + static_cast<int64_t>(t) * d, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
    }
    const float inv = 1.0f / static_cast<float>(bs);  // power of two: exact
    float *dst = out + (bh * nB + i) * static_cast<int64_t>(d) + cg * 8;
    float4 lo = make_float4(__fmul_rn(acc[0], inv), __fmul_rn(acc[1], inv), __fmul_rn(acc[2], inv),
                            __fmul_rn(acc[3], inv));
    float4 hi = make_float4(__fmul_rn(acc[4], inv), __fmul_rn(acc[5], inv), __fmul_rn(acc[6], inv),
                            __fmul_rn(acc[7], inv));
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

__global__ void __launch_bounds__(256) score_topk_kernel(const float *__restrict__ qbar,
                                                         const float *__restrict__ kbar, int nQB,
                                                         int nKB, int d, int k, int W,
                                                         int32_t *__restrict__ row_ptr,
                                                         int32_t *__restrict__ col_idx,
                                                         uint32_t *__restrict__ bitmap, uint32_t *err)
{
    extern __shared__ float sm[];
    float *qs = sm;                                  // [8][d]
    float *ks = qs + kRowsPerCta * d;                // [32][d + 1]
    uint32_t *keys = reinterpret_cast<uint32_t *>(ks + kKvTile * (d + 1));  // [8][nKB]
    const int bh = blockIdx.y;
    const int i0 = blockIdx.x * kRowsPerCta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int e = threadIdx.x; e < kRowsPerCta * d; e += blockDim.x) {
        const int r = e / d, c = e % d;
        qs[e] = (i0 + r < nQB) ? qbar[(static_cast<int64_t>(bh) * nQB + i0 + r) * d + c] : 0.0f;
    }
    bool nan_seen = false;
    for (int j0 = 0; j0 < nKB; j0 += kKvTile) {
        __syncthreads();
        for (int e = threadIdx.x; e < kKvTile * d; e += blockDim.x) {
            const int jj = e / d, c = e % d;
            ks[jj * (d + 1) + c] =
                (j0 + jj < nKB) ? kbar[(static_cast<int64_t>(bh) * nKB + j0 + jj) * d + c] : 0.0f;
        }
        __syncthreads();
        const int r = warp, j = j0 + lane;
        if (i0 + r < nQB && j < nKB) {
            const float *a = qs + r * d;
            const float *b = ks + lane * (d + 1);
            float acc = 0.0f;
            for (int c = 0; c < d; ++c) acc = __fmaf_rn(a[c], b[c], acc);
            nan_seen |= isnan(acc);
            keys[r * nKB + j] = order_key(acc);
        }
    }
    if (nan_seen) raise_error(err, BSA_ERR_NONFINITE);
    __syncthreads();

    const int i = i0 + warp;
    if (i >= nQB) return;
    const uint32_t *row = keys + warp * nKB;
    // Largest T with #{key >= T} >= k: the k-th largest key value.
    uint32_t T = 0;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = T | (1u << bit);
        int cnt = 0;
        for (int j = lane; j < nKB; j += 32) cnt += row[j] >= cand;
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        if (cnt >= k) T = cand;
    }
    int gt = 0;
    for (int j = lane; j < nKB; j += 32) gt += row[j] > T;
    gt = __reduce_add_sync(0xffffffffu, gt);
    const int need = k - gt;  // how many of the keys equal to T, lowest index first
    const int64_t r_global = static_cast<int64_t>(bh) * nQB + i;
    const int64_t out_base = r_global * k;
    int taken = 0, ties = 0;
    for (int w = 0; w < W; ++w) {
        const int j = w * 32 + lane;
        const uint32_t key = j < nKB ? row[j] : 0u;
        const bool is_gt = j < nKB && key > T;
        const bool is_eq = j < nKB && key == T;
        const uint32_t eq_mask = __ballot_sync(0xffffffffu, is_eq);
        const int eq_rank = ties + __popc(eq_mask & lanemask_lt());
        const bool sel = is_gt || (is_eq && eq_rank < need);
        const uint32_t sel_mask = __ballot_sync(0xffffffffu, sel);
        if (lane == 0) bitmap[r_global * W + w] = sel_mask;
        if (sel) col_idx[out_base + taken + __popc(sel_mask & lanemask_lt())] = j;
        taken += __popc(sel_mask);
        ties += __popc(eq_mask);
    }
    if (lane == 0) {
        row_ptr[r_global] = static_cast<int32_t>(out_base);
        if (r_global == static_cast<int64_t>(gridDim.y) * nQB - 1)
            row_ptr[r_global + 1] = static_cast<int32_t>(out_base + k);
    }
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

size_t mask_workspace_bytes(int B, int H, int N, int d, int block)
{
    const size_t BH = static_cast<size_t>(B) * H;
    const size_t nB = static_cast<size_t>(N / block);
    size_t bytes = kWsHeader;
    bytes += align_up(BH * nB * d * sizeof(float), 256) * 2;  // Qbar, Kbar
    bytes += align_up(BH * nB * sizeof(int32_t), 256);        // static row counts
    return bytes;
}

bsa_status launch_build_mask(const MaskArgs &a, cudaStream_t st)
{
    const int64_t BH = static_cast<int64_t>(a.B) * a.H;
    const int64_t R = BH * a.nQB;
    uint32_t *err = reinterpret_cast<uint32_t *>(a.ws);
    char *p = a.ws + kWsHeader;
    float *qbar = reinterpret_cast<float *>(p);
    p += align_up(static_cast<size_t>(BH) * a.nQB * a.d * sizeof(float), 256);
    float *kbar = reinterpret_cast<float *>(p);
    p += align_up(static_cast<size_t>(BH) * a.nKB * a.d * sizeof(float), 256);
    int32_t *counts = reinterpret_cast<int32_t *>(p);

    if (a.spec == nullptr) {
        const int64_t groups = BH * a.nQB * (a.d / 8);
        dim3 pg(static_cast<unsigned>((groups + kPoolThreads - 1) / kPoolThreads), 2);
        if (a.dt == BSA_BF16)
            pool_kernel<__nv_bfloat16><<<pg, kPoolThreads, 0, st>>>(
                static_cast<const __nv_bfloat16 *>(a.Q), static_cast<const __nv_bfloat16 *>(a.K), qbar,
                kbar, groups, a.N, a.d, a.block, a.nQB);
        else
            pool_kernel<float><<<pg, kPoolThreads, 0, st>>>(static_cast<const float *>(a.Q),
                                                            static_cast<const float *>(a.K), qbar, kbar,
                                                            groups, a.N, a.d, a.block, a.nQB);
        const size_t smem = sizeof(float) * (kRowsPerCta * a.d + kKvTile * (a.d + 1)) +
                            sizeof(uint32_t) * kRowsPerCta * a.nKB;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(score_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return BSA_ERR_CUDA;
        }
        dim3 sg((a.nQB + kRowsPerCta - 1) / kRowsPerCta, static_cast<unsigned>(BH));
        score_topk_kernel<<<sg, 256, smem, st>>>(qbar, kbar, a.nQB, a.nKB, a.d, a.k, a.W, a.row_ptr,
                                                 a.col_idx, a.bitmap, err);
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
        const unsigned g = static_cast<unsigned>((R + 7) / 8);
        static_rows_kernel<<<g, 256, 0, st>>>(pr, R, a.nQB, a.nKB, a.W, a.spec->bitmap, a.bitmap, counts);
        scan_kernel<<<1, 1024, 0, st>>>(counts, R, a.row_ptr);
        emit_kernel<<<g, 256, 0, st>>>(a.bitmap, a.row_ptr, R, a.W, a.col_idx, a.col_capacity, err);
    }
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
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
