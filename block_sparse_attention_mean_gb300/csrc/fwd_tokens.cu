// fwd_tokens.cu -- token-sparse attention over tile-aligned query groups (CUDA cores).
//
// "Can sparse attention close the quality gap in diffusion transformers", section
// "token 级选择需要瓦片对齐的查询分组": C similar queries of a head form a group that shares
// one set of individually selected KV tokens, gathered by index rather than repacked
// into blocks. Row r of group g gets
//   O_r = sum_t softmax_t(scale * q_r . k_t) v_t,  LSE_r = ln sum_t exp(scale * q_r . k_t),
// t over the group's tokens.
//
// One CTA per (b, h, group): the group's C = 128 query rows are gathered through the row
// permutation into shared memory (fp32), the tokens' K and V rows are gathered 32 at a
// time, lane l scores token l of the chunk for each of its warp's 16 rows, and every lane
// accumulates d/32 output channels with an online softmax in fp32. An index outside
// [0, N) raises BSA_ERR_INVALID_ARG in the workspace and is skipped.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"

namespace bsa {
namespace {

constexpr int kTokWarps = 8;
constexpr int kTokChunk = 32;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T, int D>
__global__ void __launch_bounds__(kTokWarps * 32) fwd_tokens_kernel(const T *__restrict__ Q, const T *__restrict__ K,
                                                                   const T *__restrict__ V, int N,
                                                                   const int32_t *__restrict__ perm,
                                                                   const int32_t *__restrict__ tokens, int n_tokens,
                                                                   float scale, T *__restrict__ O,
                                                                   float *__restrict__ LSE, uint32_t *err)
{
    constexpr int C = kTokenGroup;
    constexpr int RPW = C / kTokWarps;  // query rows per warp
    constexpr int DPL = D / 32;         // output channels per lane
    extern __shared__ float sm[];
    float *qs = sm;                         // [C][D]
    float *ks = qs + C * D;                 // [kTokChunk][D + 1]
    float *vs = ks + kTokChunk * (D + 1);   // [kTokChunk][D]
    __shared__ int32_t rows[C];
    __shared__ int32_t toks[kTokChunk];

    const int g = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_groups = N / C;

    for (int r = threadIdx.x; r < C; r += blockDim.x) {
        int row = perm[bh * N + static_cast<int64_t>(g) * C + r];
        if (row < 0 || row >= N) {
            raise_error(err, BSA_ERR_INVALID_ARG);
            row = -1;
        }
        rows[r] = row;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < C * D; e += blockDim.x) {
        const int r = e / D, c = e % D;
        qs[e] = rows[r] >= 0 ? to_f32(Q[(bh * N + rows[r]) * D + c]) : 0.0f;
    }

    float m[RPW], l[RPW], o[RPW][DPL];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        m[r] = -CUDART_INF_F;
        l[r] = 0.0f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) o[r][t] = 0.0f;
    }

    const int32_t *tk = tokens + (bh * n_groups + g) * static_cast<int64_t>(n_tokens);
    for (int c0 = 0; c0 < n_tokens; c0 += kTokChunk) {
        __syncthreads();
        if (threadIdx.x < kTokChunk) {
            int t = -1;
            if (c0 + threadIdx.x < n_tokens) {
                t = tk[c0 + threadIdx.x];
                if (t < 0 || t >= N) {
                    raise_error(err, BSA_ERR_INVALID_ARG);
                    t = -1;
                }
            }
            toks[threadIdx.x] = t;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kTokChunk * D; e += blockDim.x) {
            const int kk = e / D, c = e % D;
            const int t = toks[kk];
            ks[kk * (D + 1) + c] = t >= 0 ? to_f32(K[(bh * N + t) * D + c]) : 0.0f;
            vs[e] = t >= 0 ? to_f32(V[(bh * N + t) * D + c]) : 0.0f;
        }
        __syncthreads();
        const bool live = toks[lane] >= 0;  // lane's token of this chunk exists
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float *q = qs + (warp * RPW + r) * D;
            const float *k = ks + lane * (D + 1);
            float s = 0.0f;
#pragma unroll 16
            for (int c = 0; c < D; ++c) s = fmaf(q[c], k[c], s);
            s = live ? s * scale : -CUDART_INF_F;
            float cm = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
            if (cm == -CUDART_INF_F) continue;  // no token in this chunk (warp-uniform)
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
            for (int kk = 0; kk < kTokChunk; ++kk) {
                const float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
                for (int t = 0; t < DPL; ++t) o[r][t] = fmaf(pk, vs[kk * D + lane + 32 * t], o[r][t]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int row = rows[warp * RPW + r];
        if (row < 0) continue;
        const int64_t gr = bh * N + row;
        const float inv = l[r] > 0.0f ? 1.0f / l[r] : 0.0f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) store_out(O + gr * D + lane + 32 * t, o[r][t] * inv);
        if (lane == 0) LSE[gr] = l[r] > 0.0f ? m[r] + logf(l[r]) : -CUDART_INF_F;
    }
}

template <typename T, int D>
bsa_status launch(const TokenArgs &a, cudaStream_t st)
{
    const size_t smem = sizeof(float) * (kTokenGroup * D + kTokChunk * (D + 1) + kTokChunk * D);
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(fwd_tokens_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return BSA_ERR_CUDA;
        attr_set = true;
    }
    dim3 grid(a.N / kTokenGroup, a.B * a.H);
    fwd_tokens_kernel<T, D><<<grid, kTokWarps * 32, smem, st>>>(
        static_cast<const T *>(a.Q), static_cast<const T *>(a.K), static_cast<const T *>(a.V), a.N, a.perm,
        a.tokens, a.n_tokens, a.scale, static_cast<T *>(a.O), a.LSE, reinterpret_cast<uint32_t *>(a.ws));
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace

bsa_status launch_forward_tokens(const TokenArgs &a, cudaStream_t st)
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
