// query_groups.cu -- tile-aligned query groups for token-level selection (CUDA cores).
//
// "Can sparse attention close the quality gap in diffusion transformers", section
// "token 级选择需要瓦片对齐的查询分组": the queries of a head are split recursively at the
// median of their projection on the group's principal direction until every group holds
// exactly C = 128 queries. A group of m*C rows keeps its first ceil(m/2)*C rows, ordered
// by (projection, row index), as the first half; groups come out in depth-first order,
// rows ascending inside a group (the layout bsa_select_tokens and bsa_forward_tokens take).
//
// One CTA of 1024 threads per (b, h); the splits of a level run one after another on the
// whole CTA, in place in a working permutation:
//   mean of the segment's rows (fp32, warps over rows, a fixed-order reduction),
//   principal direction by kPowerIters steps of power iteration on the centred rows from a
//   fixed start vector (sign: its largest-magnitude entry positive),
//   projections as order-preserving keys, the cut by a bitwise radix select with ties to
//   the lower row index, and a stable two-way partition through a scratch copy.
// fp32 and an iterative eigenvector: near the median a row may fall on the other side than
// in an exact eigendecomposition, so results are judged by the partition they form.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace bsa {
namespace {

constexpr int kGrpThreads = 1024;
constexpr int kGrpWarps = kGrpThreads / 32;
constexpr int kPowerIters = 32;
constexpr int kMaxSegments = kMaxQueryGroups;

__device__ __forceinline__ float ld(const float *p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ uint32_t order_key_asc(float s)
{
    uint32_t u = __float_as_uint(s);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sum over the CTA of one value per thread (fixed order: warp butterflies, then warps in order).
__device__ __forceinline__ float block_sum(float v, float *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.0f;
    for (int w = 0; w < kGrpWarps; ++w) t += red[w];
    return t;
}

__device__ __forceinline__ int block_count(int v, int *redi)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_add_sync(0xffffffffu, v);
    __syncthreads();
    if (lane == 0) redi[warp] = v;
    __syncthreads();
    int t = 0;
    for (int w = 0; w < kGrpWarps; ++w) t += redi[w];
    return t;
}

template <typename T, int D>
__global__ void __launch_bounds__(kGrpThreads) query_groups_kernel(const T *__restrict__ X, int N,
                                                                   int32_t *__restrict__ work,
                                                                   uint32_t *__restrict__ keys,
                                                                   int32_t *__restrict__ scratch,
                                                                   int32_t *__restrict__ perm)
{
    constexpr int C = kTokenGroup;
    constexpr int DPL = D / 32;  // dimensions per lane
    __shared__ float red[kGrpWarps];
    __shared__ int redi[kGrpWarps];
    __shared__ float part[kGrpWarps][D];
    __shared__ float mu[D], v[D];
    __shared__ int seg_s[kMaxSegments], seg_n[kMaxSegments], nxt_s[kMaxSegments], nxt_n[kMaxSegments];
    __shared__ int n_seg;
    const int64_t bh = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const T *x = X + bh * static_cast<int64_t>(N) * D;
    int32_t *idx = work + bh * N;
    uint32_t *key = keys + bh * N;
    int32_t *tmp = scratch + bh * N;
    for (int i = threadIdx.x; i < N; i += kGrpThreads) idx[i] = i;
    if (threadIdx.x == 0) {
        seg_s[0] = 0;
        seg_n[0] = N;
        n_seg = 1;
    }
    __syncthreads();
    for (;;) {
        const int count = n_seg;  // segments of this level
        bool split_any = false;
        for (int sgi = 0; sgi < count; ++sgi) {
            const int s = seg_s[sgi], len = seg_n[sgi];
            if (len <= C) continue;
            split_any = true;
            // mean
            float acc[DPL];
#pragma unroll
            for (int t = 0; t < DPL; ++t) acc[t] = 0.0f;
            for (int i = warp; i < len; i += kGrpWarps) {
                const T *row = x + static_cast<int64_t>(idx[s + i]) * D;
#pragma unroll
                for (int t = 0; t < DPL; ++t) acc[t] += ld(row + lane + 32 * t);
            }
#pragma unroll
            for (int t = 0; t < DPL; ++t) part[warp][lane + 32 * t] = acc[t];
            __syncthreads();
            if (threadIdx.x < D) {
                float m = 0.0f;
                for (int w = 0; w < kGrpWarps; ++w) m += part[w][threadIdx.x];
                mu[threadIdx.x] = m / static_cast<float>(len);
                v[threadIdx.x] = (1.0f + 0.01f * threadIdx.x) * rsqrtf(static_cast<float>(D));
            }
            __syncthreads();
            // power iteration on the centred rows
            for (int it = 0; it < kPowerIters; ++it) {
#pragma unroll
                for (int t = 0; t < DPL; ++t) acc[t] = 0.0f;
                for (int i = warp; i < len; i += kGrpWarps) {
                    const T *row = x + static_cast<int64_t>(idx[s + i]) * D;
                    float xc[DPL], dot = 0.0f;
#pragma unroll
                    for (int t = 0; t < DPL; ++t) {
                        xc[t] = ld(row + lane + 32 * t) - mu[lane + 32 * t];
                        dot = fmaf(xc[t], v[lane + 32 * t], dot);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
#pragma unroll
                    for (int t = 0; t < DPL; ++t) acc[t] = fmaf(dot, xc[t], acc[t]);
                }
#pragma unroll
                for (int t = 0; t < DPL; ++t) part[warp][lane + 32 * t] = acc[t];
                __syncthreads();
                float wj = 0.0f;
                if (threadIdx.x < D)
                    for (int w = 0; w < kGrpWarps; ++w) wj += part[w][threadIdx.x];
                const float nrm2 = block_sum(threadIdx.x < D ? wj * wj : 0.0f, red);
                if (threadIdx.x < D && nrm2 > 0.0f) v[threadIdx.x] = wj * rsqrtf(nrm2);
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
                __syncwarp();
                for (int j = lane; j < D; j += 32) v[j] *= sgn;
            }
            __syncthreads();
            // projections as ascending keys
            for (int i = warp; i < len; i += kGrpWarps) {
                const T *row = x + static_cast<int64_t>(idx[s + i]) * D;
                float dot = 0.0f;
#pragma unroll
                for (int t = 0; t < DPL; ++t) dot = fmaf(ld(row + lane + 32 * t) - mu[lane + 32 * t], v[lane + 32 * t], dot);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                if (lane == 0) key[s + i] = order_key_asc(dot);
            }
            __syncthreads();
            // the cut: the cut-th smallest key T, and how many keys equal to T go first
            const int m = len / C;
            const int cut = ((m + 1) / 2) * C;
            uint32_t Tk = 0u;
            for (int bit = 31; bit >= 0; --bit) {
                // smallest T with #{key <= T} >= cut: keep bit 0 where the count already suffices
                const uint32_t cand = Tk | ((1u << bit) - 1u);
                int c = 0;
                for (int i = threadIdx.x; i < len; i += kGrpThreads) c += key[s + i] <= cand ? 1 : 0;
                if (block_count(c, redi) < cut) Tk |= 1u << bit;
            }
            int lt = 0;
            for (int i = threadIdx.x; i < len; i += kGrpThreads) lt += key[s + i] < Tk ? 1 : 0;
            const int need = cut - block_count(lt, redi);  // keys equal to T that go first
            // stable partition through the scratch copy: first half, then second half
            const int per = (len + kGrpThreads - 1) / kGrpThreads;
            const int b0 = threadIdx.x * per, b1 = min(len, b0 + per);
            int mine = 0;
            for (int i = b0; i < b1; ++i) {
                const uint32_t k = key[s + i];
                bool first = k < Tk;
                if (k == Tk) {  // rank among the equal keys by row index
                    int r = 0;
                    for (int j = 0; j < len; ++j) r += (key[s + j] == Tk && idx[s + j] < idx[s + i]) ? 1 : 0;
                    first = r < need;
                }
                mine += first ? 1 : 0;
            }
            // exclusive scan of the first-half counts over threads (contiguous chunks)
            int xs = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, xs, o);
                if (lane >= o) xs += y;
            }
            __syncthreads();
            if (lane == 31) redi[warp] = xs;
            __syncthreads();
            int wbase = 0;
            for (int w = 0; w < warp; ++w) wbase += redi[w];
            int pos_first = wbase + xs - mine;
            int pos_second = cut + (b0 - pos_first);  // elements before this chunk not in the first half
            for (int i = b0; i < b1; ++i) {
                const uint32_t k = key[s + i];
                bool first = k < Tk;
                if (k == Tk) {
                    int r = 0;
                    for (int j = 0; j < len; ++j) r += (key[s + j] == Tk && idx[s + j] < idx[s + i]) ? 1 : 0;
                    first = r < need;
                }
                if (first) tmp[s + pos_first++] = idx[s + i];
                else tmp[s + pos_second++] = idx[s + i];
            }
            __syncthreads();
            for (int i = threadIdx.x; i < len; i += kGrpThreads) idx[s + i] = tmp[s + i];
            __syncthreads();
        }
        if (!split_any) break;
        // next level: every segment of this level becomes its two halves (or stays, if final)
        __syncthreads();
        if (threadIdx.x == 0) {
            int n = 0;
            for (int sgi = 0; sgi < count; ++sgi) {
                const int s = seg_s[sgi], len = seg_n[sgi];
                if (len <= C) {
                    nxt_s[n] = s;
                    nxt_n[n++] = len;
                } else {
                    const int cut = ((len / C + 1) / 2) * C;
                    nxt_s[n] = s;
                    nxt_n[n++] = cut;
                    nxt_s[n] = s + cut;
                    nxt_n[n++] = len - cut;
                }
            }
            for (int k2 = 0; k2 < n; ++k2) {
                seg_s[k2] = nxt_s[k2];
                seg_n[k2] = nxt_n[k2];
            }
            n_seg = n;
        }
        __syncthreads();
    }
    // every group of C rows in ascending row order
    for (int i = threadIdx.x; i < N; i += kGrpThreads) {
        const int g0 = (i / C) * C;
        const int r = idx[i];
        int rank = 0;
        for (int j = g0; j < g0 + C; ++j) rank += idx[j] < r ? 1 : 0;
        perm[bh * N + g0 + rank] = r;
    }
}

template <typename T, int D>
bsa_status launch(const GroupArgs &a, cudaStream_t st)
{
    const QueryGroupWs l = query_groups_ws_layout(a.B, a.H, a.N);
    query_groups_kernel<T, D><<<a.B * a.H, kGrpThreads, 0, st>>>(
        static_cast<const T *>(a.Q), a.N, reinterpret_cast<int32_t *>(a.ws + l.work),
        reinterpret_cast<uint32_t *>(a.ws + l.keys), reinterpret_cast<int32_t *>(a.ws + l.scratch), a.perm);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace

QueryGroupWs query_groups_ws_layout(int B, int H, int N)
{
    const size_t n = static_cast<size_t>(B) * H * N;
    QueryGroupWs l{};
    l.work = kWsHeader;
    l.keys = l.work + align_up(n * sizeof(int32_t), 256);
    l.scratch = l.keys + align_up(n * sizeof(uint32_t), 256);
    l.total = l.scratch + align_up(n * sizeof(int32_t), 256);
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
