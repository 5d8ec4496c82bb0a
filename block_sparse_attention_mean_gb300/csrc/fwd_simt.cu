// fwd_simt.cu -- fp32 block-sparse attention forward on CUDA cores.
//
// The fp32 input path: a bf16 tensor-core path would round the inputs and miss
// the LSE tolerance, so fp32 inputs run this exact-fp32 tile loop instead
// ("多模态DiT中的块稀疏注意力" §4.1 loop over active_kv_blocks[i]; §4.3 online softmax
// over active blocks only, normalised by the true active-only sum at the end).
//
// One CTA per (b, h, Q block); 8 warps, each owning bs/8 query rows. K/V are
// staged 32 keys at a time in shared memory; lane l scores key l of the chunk,
// then every lane accumulates its d/32 output channels.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "walk.cuh"

namespace bsa {
namespace {

constexpr int kWarps = 8;
constexpr int kChunk = 32;

template <int D, int BS>
__global__ void __launch_bounds__(kWarps * 32) fwd_simt_kernel(const float *__restrict__ Q, const float *__restrict__ K,
                                                              const float *__restrict__ V, int N, int nQB, int nKB,
                                                              int W, const int32_t *__restrict__ row_ptr,
                                                              const int32_t *__restrict__ col_idx,
                                                              const uint32_t *__restrict__ bitmap, int index_mode,
                                                              float scale, float *__restrict__ O,
                                                              float *__restrict__ LSE, const float *__restrict__ R)
{
    constexpr int RPW = BS / kWarps;  // query rows per warp
    constexpr int DPL = D / 32;       // channels per lane
    extern __shared__ float sm[];
    float *qs = sm;                    // [BS][D]
    float *ks = qs + BS * D;           // [kChunk][D + 1]
    float *vs = ks + kChunk * (D + 1); // [kChunk][D]

    const int i = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = bh * N + static_cast<int64_t>(i) * BS;

    // rows of a ragged last block past the sequence end are zeros (and never written)
    const int rows = min(BS, N - i * BS);
    for (int e = threadIdx.x; e < BS * D; e += blockDim.x) qs[e] = e / D < rows ? Q[row0 * D + e] : 0.0f;

    float m[RPW], l[RPW], o[RPW][DPL];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        m[r] = -CUDART_INF_F;
        l[r] = 0.0f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) o[r][t] = 0.0f;
    }

    TileWalk walk;
    walk.init(index_mode, row_ptr, col_idx, bitmap, W, bh * nQB + i, -1, 1u);
    int j;
    uint32_t mbits;
    while (walk.next(j, mbits)) {
        if (j < 0 || j >= nKB) continue;  // never read outside the head
        const int keys = min(BS, N - j * BS);  // a ragged last KV block holds fewer keys
        for (int c0 = 0; c0 < keys; c0 += kChunk) {
            __syncthreads();
            const int64_t krow = bh * N + static_cast<int64_t>(j) * BS + c0;
            for (int e = threadIdx.x; e < kChunk * D; e += blockDim.x) {
                const int kk = e / D, c = e % D;
                const bool in = c0 + kk < keys;
                ks[kk * (D + 1) + c] = in ? K[(krow + kk) * D + c] : 0.0f;
                if (V) vs[e] = in ? V[(krow + kk) * D + c] : 0.0f;  // no V: the LSE only
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const float *q = qs + (warp * RPW + r) * D;
                const float *k = ks + lane * (D + 1);
                float s = 0.0f;
#pragma unroll 16
                for (int c = 0; c < D; ++c) s = fmaf(q[c], k[c], s);
                s = c0 + lane < keys ? s * scale : -CUDART_INF_F;  // keys past the end do not count
                float cm = s;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
                const float mn = fmaxf(m[r], cm);
                const float alpha = expf(m[r] - mn);  // m = -inf -> 0
                const float p = expf(s - mn);
                float ps = p;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
                l[r] = l[r] * alpha + ps;
                m[r] = mn;
#pragma unroll
                for (int t = 0; t < DPL; ++t) o[r][t] *= alpha;
                if (!V) continue;
                for (int kk = 0; kk < kChunk; ++kk) {
                    const float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
                    for (int t = 0; t < DPL; ++t) o[r][t] = fmaf(pk, vs[kk * D + lane + 32 * t], o[r][t]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        if (warp * RPW + r >= rows) break;
        const int64_t row = row0 + warp * RPW + r;
        const float inv = l[r] > 0.0f ? 1.0f / l[r] : 0.0f;
        if (O) {
#pragma unroll
            for (int t = 0; t < DPL; ++t)
                O[row * D + lane + 32 * t] = o[r][t] * inv + (R ? R[row * D + lane + 32 * t] : 0.0f);
        }
        if (lane == 0) LSE[row] = l[r] > 0.0f ? m[r] + logf(l[r]) : -CUDART_INF_F;
    }
}

template <int D, int BS>
bsa_status launch(const FwdArgs &a, cudaStream_t st)
{
    const size_t smem = sizeof(float) * (BS * D + kChunk * (D + 1) + kChunk * D);
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(fwd_simt_kernel<D, BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return BSA_ERR_CUDA;
        attr_set = true;
    }
    dim3 grid(a.nQB, a.B * a.H);
    fwd_simt_kernel<D, BS><<<grid, kWarps * 32, smem, st>>>(
        static_cast<const float *>(a.Q), static_cast<const float *>(a.K), static_cast<const float *>(a.V), a.N,
        a.nQB, a.nKB, a.W, a.row_ptr, a.col_idx, a.bitmap, a.index_mode, a.scale, static_cast<float *>(a.O),
        a.LSE, a.R);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace

bsa_status launch_forward_simt(const FwdArgs &a, cudaStream_t st)
{
    if (a.d == 64 && a.block == 64) return launch<64, 64>(a, st);
    if (a.d == 64 && a.block == 128) return launch<64, 128>(a, st);
    if (a.d == 128 && a.block == 64) return launch<128, 64>(a, st);
    if (a.d == 128 && a.block == 128) return launch<128, 128>(a, st);
    return BSA_ERR_SHAPE;
}

}  // namespace bsa
