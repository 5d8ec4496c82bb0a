// query_groups.cu -- tile-aligned query groups for token-level selection (CUDA cores).
//
// "Can sparse attention close the quality gap in diffusion transformers", section
// "token 级选择需要瓦片对齐的查询分组": the queries of a head are split recursively at the
// median of their projection on the group's principal direction until every group holds
// exactly C = 128 queries. A group of m*C rows keeps its first ceil(m/2)*C rows, ordered
// by (projection, row index), as the first half; groups come out in depth-first order,
// rows ascending inside a group (the layout bsa_select_tokens and bsa_forward_tokens take).
//
// The split tree depends on N only, so the splits run level by level: one launch per
// level, one CTA per (b, h, segment of that level), every segment of every head at once.
// A CTA, in place in the working permutation of its head:
//   mean of the segment's rows (fp32; warps over rows, then the warps in order),
//   the centred scatter matrix S = sum (x - mu)(x - mu)^T in one pass (each thread owns a
//   block of entries and adds the rows in order),
//   the principal direction by kPowerIters steps of power iteration on S from a fixed start
//   (sign: its largest-magnitude entry positive),
//   64-bit keys (projection as an order-preserving key, row index) in the workspace,
//   the cut: the cut-th smallest key by an exact radix select (8-bit digits), and a
//   stable partition (first half: keys up to the cut) through a scratch copy.
// A final launch sorts each group's rows ascending. fp32 and an iterative eigenvector:
// near the median a row may fall on the other side than in an exact eigendecomposition,
// so results are judged by the partition they form, and bit for bit where no row lies
// within the rounding bound of a cut.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace bsa {
namespace {

constexpr int kGrpThreads = 256;
constexpr int kGrpWarps = kGrpThreads / 32;
constexpr int kPowerIters = 32;
constexpr int kStageRows = 32;  // rows staged per step of the scatter-matrix pass

__device__ __forceinline__ float ld(const float *p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

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

// Sum over the CTA, the warps in order (fixed order).
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

// One split of every segment of one level. grid (2^level, B*H).
template <typename T, int D>
__global__ void __launch_bounds__(kGrpThreads) split_level_kernel(const T *__restrict__ X, int N, int level,
                                                                  int32_t *__restrict__ work,
                                                                  unsigned long long *__restrict__ keys,
                                                                  int32_t *__restrict__ scratch)
{
    constexpr int C = kTokenGroup;
    constexpr int DPL = D / 32;             // dimensions per lane (row-wise passes)
    constexpr int BLK = D / 16;             // scatter-matrix block per thread: BLK x BLK entries
    __shared__ float red[kGrpWarps];
    __shared__ int redi[kGrpWarps];
    __shared__ float part[kGrpWarps][D];
    __shared__ __align__(16) float mu[D];
    __shared__ float v[D], w[D];
    __shared__ int hist[256];
    // dynamic: the scatter matrix S [D][D + 1] (padded rows) and the staged centred rows [32][D]
    extern __shared__ float4 grp_dyn[];
    float (*S)[D + 1] = reinterpret_cast<float (*)[D + 1]>(grp_dyn);
    float (*xs)[D] = reinterpret_cast<float (*)[D]>(reinterpret_cast<float *>(grp_dyn) + D * (D + 1));
    __shared__ int s_digit, s_krem;
    int s, len;
    if (!segment_of(N, level, blockIdx.x, s, len)) return;  // block-uniform
    const int64_t bh = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const T *x = X + bh * static_cast<int64_t>(N) * D;
    int32_t *idx = work + bh * N + s;
    unsigned long long *key = keys + bh * N + s;
    int32_t *tmp = scratch + bh * N + s;

    // mean
    {
        float acc[DPL];
#pragma unroll
        for (int t = 0; t < DPL; ++t) acc[t] = 0.0f;
        // four rows per warp in flight; each warp still adds its rows in order
        for (int i0 = warp * 4; i0 < len; i0 += kGrpWarps * 4) {
            float vals[4][DPL];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                const T *row = x + static_cast<int64_t>(i < len ? idx[i] : idx[0]) * D;
#pragma unroll
                for (int t = 0; t < DPL; ++t) vals[u][t] = i < len ? ld(row + lane + 32 * t) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int t = 0; t < DPL; ++t) acc[t] += vals[u][t];
        }
#pragma unroll
        for (int t = 0; t < DPL; ++t) part[warp][lane + 32 * t] = acc[t];
        __syncthreads();
        if (threadIdx.x < D) {
            float m = 0.0f;
            for (int ww = 0; ww < kGrpWarps; ++ww) m += part[ww][threadIdx.x];
            mu[threadIdx.x] = m / static_cast<float>(len);
        }
        __syncthreads();
    }
    // centred scatter matrix: thread (ti, tj) owns rows BLK*ti.. and columns BLK*tj..
    {
        const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
        float acc[BLK][BLK];
#pragma unroll
        for (int a = 0; a < BLK; ++a)
#pragma unroll
            for (int b = 0; b < BLK; ++b) acc[a][b] = 0.0f;
        // the next batch of rows is loaded into registers while this one is used
        constexpr int PER = kStageRows * D / kGrpThreads;
        float nxt[PER];
        auto fetch = [&](int r0) {
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int e = q * kGrpThreads + threadIdx.x;
                const int r = e / D, c = e % D;
                nxt[q] = r0 + r < len ? ld(x + static_cast<int64_t>(idx[r0 + r]) * D + c) : 0.0f;
            }
        };
        fetch(0);
        for (int r0 = 0; r0 < len; r0 += kStageRows) {
            __syncthreads();
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                const int e = q * kGrpThreads + threadIdx.x;
                const int r = e / D, c = e % D;
                xs[r][c] = r0 + r < len ? nxt[q] - mu[c] : 0.0f;
            }
            __syncthreads();
            if (r0 + kStageRows < len) fetch(r0 + kStageRows);
            for (int r = 0; r < kStageRows; ++r) {
                float a_[BLK], b_[BLK];
#pragma unroll
                for (int a = 0; a < BLK; ++a) {
                    a_[a] = xs[r][BLK * ti + a];
                    b_[a] = xs[r][BLK * tj + a];
                }
#pragma unroll
                for (int a = 0; a < BLK; ++a)
#pragma unroll
                    for (int b = 0; b < BLK; ++b) acc[a][b] = fmaf(a_[a], b_[b], acc[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < BLK; ++a)
#pragma unroll
            for (int b = 0; b < BLK; ++b) S[BLK * ti + a][BLK * tj + b] = acc[a][b];
        if (threadIdx.x < D) v[threadIdx.x] = (1.0f + 0.01f * threadIdx.x) * rsqrtf(static_cast<float>(D));
        __syncthreads();
    }
    // power iteration on S
    for (int it = 0; it < kPowerIters; ++it) {
        float wi = 0.0f;
        if (threadIdx.x < D) {
            for (int j = 0; j < D; ++j) wi = fmaf(S[threadIdx.x][j], v[j], wi);
            w[threadIdx.x] = wi;
        }
        const float nrm2 = block_sum(threadIdx.x < D ? wi * wi : 0.0f, red);
        if (threadIdx.x < D && nrm2 > 0.0f) v[threadIdx.x] = wi * rsqrtf(nrm2);
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
    // keys: (projection as an ascending key, row index)
    for (int i0 = warp * 4; i0 < len; i0 += kGrpWarps * 4) {
        float vals[4][DPL];
        int rr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // four rows per warp in flight
            const int i = i0 + u;
            rr[u] = i < len ? idx[i] : idx[0];
            const T *row = x + static_cast<int64_t>(rr[u]) * D;
#pragma unroll
            for (int t = 0; t < DPL; ++t) vals[u][t] = ld(row + lane + 32 * t);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float dot = 0.0f;
#pragma unroll
            for (int t = 0; t < DPL; ++t) dot = fmaf(vals[u][t] - mu[lane + 32 * t], v[lane + 32 * t], dot);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            if (lane == 0 && i0 + u < len)
                key[i0 + u] = (static_cast<unsigned long long>(order_key_asc(dot)) << 32) | static_cast<uint32_t>(rr[u]);
        }
    }
    __syncthreads();
    // the cut-th smallest key (keys are unique: the row index breaks ties), digit by digit
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
        __syncthreads();
    }
    const unsigned long long Tk = prefix;  // the cut-th smallest: keys <= Tk form the first half
    // stable partition through the scratch copy (contiguous chunks per thread)
    const int per = (len + kGrpThreads - 1) / kGrpThreads;
    const int b0 = min(len, threadIdx.x * per), b1 = min(len, b0 + per);
    int mine = 0;
    for (int i = b0; i < b1; ++i) mine += key[i] <= Tk ? 1 : 0;
    int xsum = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xsum, o);
        if (lane >= o) xsum += y;
    }
    __syncthreads();
    if (lane == 31) redi[warp] = xsum;
    __syncthreads();
    int wbase = 0;
    for (int ww = 0; ww < warp; ++ww) wbase += redi[ww];
    int pos_first = wbase + xsum - mine;
    int pos_second = cut + (b0 - pos_first);  // elements before this chunk that go second
    for (int i = b0; i < b1; ++i) {
        if (key[i] <= Tk) tmp[pos_first++] = idx[i];
        else tmp[pos_second++] = idx[i];
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

template <typename T, int D>
bsa_status launch(const GroupArgs &a, cudaStream_t st)
{
    const QueryGroupWs l = query_groups_ws_layout(a.B, a.H, a.N);
    int32_t *work = reinterpret_cast<int32_t *>(a.ws + l.work);
    auto *keys = reinterpret_cast<unsigned long long *>(a.ws + l.keys);
    int32_t *scratch = reinterpret_cast<int32_t *>(a.ws + l.scratch);
    const int BH = a.B * a.H;
    const int64_t total = static_cast<int64_t>(BH) * a.N;
    init_work_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(work, a.N, total);
    const int G = a.N / kTokenGroup;
    int depth = 0;
    while ((1 << depth) < G) ++depth;  // levels until every segment is one group
    const size_t smem = sizeof(float) * (D * (D + 1) + kStageRows * D);
    if (cudaFuncSetAttribute(split_level_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return BSA_ERR_CUDA;
    for (int level = 0; level < depth; ++level)
        split_level_kernel<T, D><<<dim3(1u << level, static_cast<unsigned>(BH)), kGrpThreads, smem, st>>>(
            static_cast<const T *>(a.Q), a.N, level, work, keys, scratch);
    sort_groups_kernel<<<dim3(static_cast<unsigned>(G), static_cast<unsigned>(BH)), kTokenGroup, 0, st>>>(
        work, a.N, a.perm);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace

QueryGroupWs query_groups_ws_layout(int B, int H, int N)
{
    const size_t n = static_cast<size_t>(B) * H * N;
    QueryGroupWs l{};
    l.work = kWsHeader;
    l.keys = l.work + align_up(n * sizeof(int32_t), 256);
    l.scratch = l.keys + align_up(n * sizeof(unsigned long long), 256);
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
