// fwd_tc.cu -- bf16 block-sparse FlashAttention forward on sm_103a tensor cores.
//
// Method: "多模态DiT中的块稀疏注意力：从原理到工程落地" §4.1 (FlashAttention tile loop
// whose inner loop walks only active_kv_blocks[i], read from a CSR or bitmap
// index in device memory) and §4.3 (skipped blocks count as -inf: they are never
// visited, and the output is divided by the true sum over the active blocks).
//
// Design (GB300-first, not the pages' Triton/xFormers recipes):
//   * Persistent CTAs pull work items from a list with an atomic counter: items of
//     at least an eighth of the per-CTA share of steps longest first (rows with very
//     different active counts, §5.3), the rest in tile order (a head's tiles together,
//     its K and V in L2). An item is a
//     128-row query tile, or one KV-range chunk of a tile that is far longer than
//     the per-CTA share of steps; the last chunk to finish merges the chunks'
//     partial (O, max, sums).
//   * Warp roles: 4 or 8 softmax + epilogue warps, a scheduler + Q/K producer
//     warp, a V producer warp, a QK^T issuer warp and a PV issuer warp. The two
//     producers walk the index on their own, so a V slot still held by a
//     lagging PV never holds back a K load. The role warps run converged and issue
//     TMA copies, tcgen05.mma and tcgen05.commit from one elect.sync lane; every
//     warp waits on mbarriers with all lanes and a vote (a lone lane waiting or
//     issuing while the others park costs several times more on this GPU).
//   * With 4 softmax warps a thread owns one query row (32x32b TMEM accesses);
//     with 8, a thread owns two rows and a quarter of their columns (16x256b /
//     16x128b accesses) and a row's max and sums are combined over 4 lanes.
//   * Q tile and K/V blocks arrive by TMA (128-byte swizzle), K/V fetched by
//     block index into separate K and V shared-memory rings (a K slot frees when
//     its QK^T completes, a V slot when its PV completes).
//   * S = Q K^T and O += P V run on tcgen05 with fp32 accumulators in TMEM. The
//     K producer walks with one step of lookahead and leaves a step descriptor
//     (blocks, members, last) beside each K slot; the QK^T issuer, which reads no
//     index, runs up to NSB steps ahead and passes the descriptor on beside each
//     S buffer. P (bf16) overwrites S in TMEM and feeds the PV MMA directly.
//   * Online softmax in the log2 domain with one FFMA + one ex2 per score;
//     the running max is only raised (and O rescaled in TMEM) when it grows by
//     more than 2^8, which keeps the result exact while skipping most rescales.
//   * At block size 64 a tile holds Q blocks 2t and 2t+1 and walks the union of
//     their lists; rows of a Q block that does not have the current KV block
//     get P = 0 and leave their running max and sum untouched.
//   * Every wait is bounded (BSA_ERR_TIMEOUT in the workspace, clean exit).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"
#include "sync.cuh"
#include "walk.cuh"

namespace bsa {
namespace {

// Warp roles: 4 * SPLIT softmax warps, then the TMA producer, the QK^T issuer
// and the PV issuer (one thread each; TMEM is allocated by the PV issuer's warp).
template <int SPLIT>
struct Roles {
    static constexpr int kSoftmaxWarps = 4 * SPLIT;
    static constexpr int kProducerWarp = kSoftmaxWarps, kQkWarp = kSoftmaxWarps + 1, kMmaWarp = kSoftmaxWarps + 2;
    static constexpr int kVProducerWarp = kSoftmaxWarps + 3;
    static constexpr int kThreads = (kSoftmaxWarps + 4) * 32;
};
constexpr int kTileM = 128;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleSum = 256.0f;  // 2^kRescaleLog2
constexpr uint32_t kDbgStall = 1u;     // skip loads and MMAs (the softmax's first wait runs out)
constexpr uint32_t kDbgNoSplit = 2u;   // never split a query tile
constexpr uint32_t kDbgSplitAll = 4u;  // split every tile with two or more steps (as the budget allows)

// Work items (load balance, "多模态DiT中的块稀疏注意力" §5.3: rows with very different
// active counts throttle a uniform launch). A query tile whose KV step count is
// above the per-CTA share of all steps is split by KV block range into up to
// kMaxChunks chunks; each chunk is one item and writes an unnormalised partial
// O with its row max and sums, which the chunk that finishes last merges.
constexpr int kMaxChunks = 8;
constexpr int kMinChunkSteps = 4;
constexpr int kMaxPartials = 640;    // partial-result slots per launch
constexpr int kItemTileBits = 24;    // item = tile | chunk << 24 | (chunks - 1) << 27
constexpr int kMergeWarps = 8;       // merge counters per split tile (one per softmax warp)

struct TcParams {
    int N, nQB, nKB, W, tiles_per_bh, n_tiles;
    int ragged_kb;             // index of the last KV block when it holds fewer than BS keys, else -1
    int last_rows;             // keys (and query rows) in the last block
    const int32_t *row_ptr;
    const int32_t *col_idx;
    const uint32_t *bitmap;
    int index_mode;
    float scale_log2;
    __nv_bfloat16 *O;
    float *LSE;
    const int32_t *tile_list;  // work items: long ones longest first, the rest in tile order
    const uint32_t *n_items;
    uint32_t *tile_counter;
    uint32_t *err;
    unsigned long long wait_limit_ns;
    uint32_t dbg;
    int split_ok;              // items carry chunk fields (fewer than 2^24 tiles)
    const int32_t *split_base; // per tile: first partial slot of a split tile, else -1
    uint32_t *merge_cnt;       // per split tile and softmax warp: chunks finished
    float *part_o;             // [slot][128][D] unnormalised partial O
    const float *R;            // residual added to O before rounding ([B][H][N][D] fp32), or nullptr
    float4 *part_stats;        // [slot][128] (row max in log2 units, fp32 sum, sum of bf16-rounded P, 0)
    // token mode (tile = (b, h, query group); steps are 128-token chunks of the group's keys)
    const int32_t *perm;       // [B*H][N]: group g of a head is rows perm[g*128 .. g*128+127]
    const int32_t *tokens;     // [B*H][N/128][n_tok]: each group's keys
    int n_tok;                 // keys per group
    int groups;                // query groups per head (N / 128)
    const __nv_bfloat16 *Kg, *Vg; // K and V rows [B*H*N][D], copied by cp.async in token mode
};

struct Item {
    int tile, chunk, nchunk;
};

__device__ __forceinline__ Item decode_item(const TcParams &p, int v)
{
    Item it;
    if (p.split_ok) {
        it.tile = v & ((1 << kItemTileBits) - 1);
        it.chunk = (v >> kItemTileBits) & 7;
        it.nchunk = ((v >> (kItemTileBits + 3)) & 7) + 1;
    } else {
        it.tile = v;
        it.chunk = 0;
        it.nchunk = 1;
    }
    return it;
}

// KV blocks [j_lo, j_hi) of an item (the whole row for an unsplit tile)
__device__ __forceinline__ void chunk_range(const TcParams &p, const Item &it, int &j_lo, int &j_hi)
{
    if (it.nchunk == 1) {
        j_lo = 0;
        j_hi = 0x7fffffff;
        return;
    }
    j_lo = static_cast<int>(static_cast<long long>(it.chunk) * p.nKB / it.nchunk);
    j_hi = static_cast<int>(static_cast<long long>(it.chunk + 1) * p.nKB / it.nchunk);
}

// One KV step = PAIR consecutive KV blocks of the walk (PAIR = 2 at block 64:
// QK^T then runs as N = 128 MMAs). A K or V ring stage holds one step: per
// 64-column slab, PAIR * BS rows of 128 bytes, block p of the step at row p * BS.
template <int D, int BS, int NK, int NV, int NSB, int QS, int PAIR>
struct Cfg {
    static constexpr int kStep = PAIR * BS;       // KV rows (S columns) per step
    static constexpr int kQBytes = kTileM * D * 2;
    static constexpr int kKVBytes = kStep * D * 2;
    static constexpr int kQChunk = kTileM * 128;  // bytes of one 64-column swizzled slab
    static constexpr int kKVChunk = kStep * 128;
    static constexpr int Q_OFF = 0;  // QS Q slots: tile e uses slot e % QS
    static constexpr int K_OFF = Q_OFF + QS * kQBytes;   // NK-stage K ring
    static constexpr int V_OFF = K_OFF + NK * kKVBytes;  // NV-stage V ring
    static constexpr int BAR_OFF = V_OFF + NV * kKVBytes;
    // barrier indices
    static constexpr int B_QFULL = 0, B_QEMPTY = 2;  // two each
    static constexpr int B_KFULL = 4, B_KEMPTY = B_KFULL + NK, B_VFULL = B_KEMPTY + NK, B_VEMPTY = B_VFULL + NV;
    static constexpr int B_SFULL = B_VEMPTY + NV, B_PFULL = B_SFULL + NSB, B_PVDONE = B_SFULL + 2 * NSB;
    static constexpr int B_OEMPTY = B_SFULL + 3 * NSB, B_TFULL = B_OEMPTY + 1, B_TEMPTY = B_TFULL + 2;
    static constexpr int B_DRAIN = B_TEMPTY + 2;  // two: one per MMA-issuing thread
    static constexpr int NBAR = B_DRAIN + 2;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    // TMEM base, abort flag, 2 tile ids, NSB step descriptors of the S/P buffers, NK of the K ring
    static constexpr int MISC_WORDS = 4 + NSB + NK;
    static constexpr int SMEM = MISC_OFF + 4 * ((MISC_WORDS + 7) & ~7);
    static constexpr int SMEM_ALLOC = SMEM + 1024;  // manual 1024-byte alignment
    static constexpr int TCOLS_USED = NSB * kStep + D;
    static constexpr int TCOLS = TCOLS_USED <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC_QK = idesc_bf16_f32(kTileM, kStep, 0, 0);
    static constexpr uint32_t IDESC_QK_HALF = idesc_bf16_f32(kTileM, BS, 0, 0);  // a step with one block
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(kTileM, D, 0, 1);
};

// The producer marks a tile whose walk is empty in the scheduler ring, so the
// other roles need not walk the index to find out.
constexpr int32_t kEmptyTile = 1 << 30;

// Step descriptor (written by the K producer, copied beside S/P buffer b by the
// QK^T issuer): bits 0-1 blocks in the step, bits 2-3 and 4-5 which of the tile's
// Q blocks have block 0 and block 1 of the step, bit 6 set on the tile's last
// step, bits 7 and 8 set when block 0 / block 1 of the step is a ragged last KV
// block (keys past the sequence end must not count). The S-full barrier publishes
// it to the softmax warps and the P-full barrier carries it on to the PV issuer.
__device__ __forceinline__ uint32_t step_desc(int cnt, const uint32_t (&ms)[2], bool last, uint32_t ragged)
{
    return static_cast<uint32_t>(cnt) | (ms[0] << 2) | (ms[1] << 4) | (last ? 64u : 0u) | (ragged << 7);
}
__device__ __forceinline__ uint32_t desc_ragged(uint32_t d) { return (d >> 7) & 3u; }
// bit q set when block q of the step is the ragged last KV block
__device__ __forceinline__ uint32_t ragged_bits(const TcParams &p, const int (&js)[2], int cnt)
{
    return (cnt > 0 && js[0] == p.ragged_kb ? 1u : 0u) | (cnt > 1 && js[1] == p.ragged_kb ? 2u : 0u);
}
__device__ __forceinline__ int desc_count(uint32_t d) { return static_cast<int>(d & 3u); }
__device__ __forceinline__ uint32_t desc_members(uint32_t d, int q) { return (d >> (2 + 2 * q)) & 3u; }
__device__ __forceinline__ bool desc_last(uint32_t d) { return (d & 64u) != 0u; }

// warp_wait_all for S buffer `b`, then the step descriptor written before it.
// Returns 0xFFFFFFFF when the wait failed.
__device__ __forceinline__ uint32_t warp_wait_step(uint32_t bar, uint32_t parity, const Ctl &c,
                                                   const volatile uint32_t *desc)
{
    return warp_wait_all(bar, parity, c) ? *desc : 0xFFFFFFFFu;
}

__device__ __forceinline__ void tile_coords(const TcParams &p, int tile, int64_t &bh, int &qt)
{
    bh = tile / p.tiles_per_bh;
    qt = tile % p.tiles_per_bh;
}

// Global output row (b*H + h)*N + row of tile row `trow`, and whether it exists: the
// tile's rows in order, or in token mode the group's rows as the permutation lists them
// (an index outside [0, N) was reported by the Q producer and is not written).
template <bool TOK>
__device__ __forceinline__ int64_t out_row(const TcParams &p, int tile, int trow, bool &valid)
{
    if constexpr (TOK) {
        const int64_t bh = tile / p.groups;
        const int r = __ldg(p.perm + static_cast<int64_t>(tile) * kTileM + trow);
        valid = r >= 0 && r < p.N;
        return bh * p.N + (valid ? r : 0);
    } else {
        int64_t bh;
        int qt;
        tile_coords(p, tile, bh, qt);
        const int row = qt * kTileM + trow;
        valid = row < p.N;
        return bh * p.N + row;
    }
}

// Token mode: the global row ((b*H + h)*N + token) of each of this lane's four rows
// (4*lane .. 4*lane + 3) of a 128-row gather, from idx[0 .. n) (rows past n repeat
// idx[n - 1]: a valid key whose score the softmax masks). An index outside [0, N) is
// reported and replaced by 0.
__device__ __forceinline__ void gather_idx(const int32_t *idx, int n, int lane, int (&v)[4])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = 4 * lane + i;
        v[i] = __ldg(idx + (k < n ? k : n - 1));
    }
}
__device__ __forceinline__ void gather_rows_of(const TcParams &p, const int (&v)[4], int64_t bh, int (&rows)[4])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int x = v[i];
        if (x < 0 || x >= p.N) {
            raise_error(p.err, BSA_ERR_INVALID_ARG);
            x = 0;
        }
        rows[i] = static_cast<int>(bh * p.N + x);
    }
}
__device__ __forceinline__ void gather_rows(const TcParams &p, const int32_t *idx, int n, int64_t bh, int lane,
                                            int (&rows)[4])
{
    int v[4];
    gather_idx(idx, n, lane, v);
    gather_rows_of(p, v, bh, rows);
}

// Token mode: the 128 rows of a step (lane l holds the global rows of 4l .. 4l + 3, as
// gather_rows_of gives them) copied into a K or V stage by 16-byte cp.async, in the
// layout the TMA loads write: D/64 slabs of 128-byte rows, 16-byte chunk c of slab row r
// at c ^ (r & 7) (the 128-byte swizzle; slabs are 1024-byte aligned). A warp instruction
// covers 256 / D whole rows, so each copies whole 128-byte lines.
template <int D>
__device__ __forceinline__ void copy_rows_async(uint32_t dst, uint32_t slab_bytes, const __nv_bfloat16 *src, const int (&rows)[4], int lane)
{
    constexpr int CPR = D / 8, RPI = 32 / CPR;
    const int rr = lane / CPR, cj = lane % CPR, sc = cj >> 3, ch = cj & 7;
    const uint32_t slab = dst + sc * slab_bytes;
#pragma unroll 4
    for (int m = 0; m < 32; ++m) {
        int r4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) r4[i] = __shfl_sync(0xffffffffu, rows[i], m);
#pragma unroll
        for (int h = 0; h < 4 / RPI; ++h) {
            const int k = RPI * h + rr;
            const int grow = k == 0 ? r4[0] : k == 1 ? r4[1] : k == 2 ? r4[2] : r4[3];
            const int r = 4 * m + k;
            cp_async16(slab + r * 128 + ((ch ^ (r & 7)) << 4), src + static_cast<int64_t>(grow) * D + sc * 64 + ch * 8);
        }
    }
}

template <int BS>
__device__ __forceinline__ void walk_init(TileWalk &w, const TcParams &p, int64_t bh, int qt, int j_lo = 0,
                                          int j_hi = 0x7fffffff)
{
    if (BS == 128) {
        w.init(p.index_mode, p.row_ptr, p.col_idx, p.bitmap, p.W, bh * p.nQB + qt, -1, 3u, j_lo, j_hi);
    } else {
        const int i0 = 2 * qt, i1 = 2 * qt + 1;
        w.init(p.index_mode, p.row_ptr, p.col_idx, p.bitmap, p.W, bh * p.nQB + i0,
               i1 < p.nQB ? bh * p.nQB + i1 : -1, 0u, j_lo, j_hi);
    }
}

// ---------------------------------------------------------------- softmax roles
//
// Both variants process, per visited KV block, the S tile of their rows:
// row max (skipped blocks are never visited, so they contribute nothing),
// lazy running-max update, p = 2^(s * scale * log2 e - m) (one packed FFMA and
// one ex2 per score), P packed to bf16 and stored over S in TMEM for the PV MMA,
// and two running sums: the fp32 one for LSE and the bf16 one that normalises O
// (P's rounding then cancels between numerator and denominator).

template <class C>
__device__ __forceinline__ uint32_t barrier_addr(uint32_t sbase, int idx)
{
    return sbase + C::BAR_OFF + 8u * idx;
}

// Fetch the next tile id from the scheduler ring (lane 0 waits, all lanes get it).
template <class C>
__device__ __forceinline__ bool fetch_tile(uint32_t sbase, volatile int32_t *tile_ids, const Ctl &ctl, int lane,
                                           int &tcount, int &tile)
{
    const int slot = tcount & 1;
    if (!warp_wait_all(barrier_addr<C>(sbase, C::B_TFULL + slot), (tcount >> 1) & 1, ctl)) return false;
    tile = tile_ids[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(barrier_addr<C>(sbase, C::B_TEMPTY + slot));
    ++tcount;
    return true;
}

// ---------------------------------------------------------------- split tiles
//
// The chunks of a split tile hold, per row, an unnormalised partial O_k (P V summed
// over the chunk's KV blocks, P relative to the chunk's row max m_k) with the sums
// l_k (fp32 P) and lp_k (bf16-rounded P). The merged row is
//   O = sum_k w_k O_k / sum_k w_k lp_k,  LSE = ln2 (M + log2 sum_k w_k l_k),
//   w_k = 2^(m_k - M), M = max_k m_k (m in log2 units),
// the same quantities the unsplit loop forms, summed in another order. The chunk
// that finishes last (per softmax warp, by an atomic count) merges; its loads
// bypass L1 because other SMs wrote the partials.

// Per-chunk weights of one row; returns M, L and LP.
__device__ __forceinline__ void merge_weights(const TcParams &p, int base, int nchunk, int row, float (&w)[kMaxChunks],
                                              float &M, float &L, float &LP)
{
    M = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k)
        if (k < nchunk) M = fmaxf(M, __ldcg(&p.part_stats[static_cast<size_t>(base + k) * kTileM + row]).x);
    L = 0.0f;
    LP = 0.0f;
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
        w[k] = 0.0f;
        if (k < nchunk) {
            const float4 st = __ldcg(&p.part_stats[static_cast<size_t>(base + k) * kTileM + row]);
            if (st.x != -CUDART_INF_F) {
                w[k] = ex2_approx(st.x - M);
                L += w[k] * st.y;
                LP += w[k] * st.z;
            }
        }
    }
}

// One thread merges its whole row (one-thread-per-row softmax). Out of line: it
// runs once per split tile and warp, and inlined it would crowd the main loop's
// registers.
template <int D>
__device__ __noinline__ void merge_row(const TcParams &p, int base, int nchunk, int trow, __nv_bfloat16 *orow,
                                          float *lse, const float *rrow)
{
    float w[kMaxChunks], M, L, LP;
    merge_weights(p, base, nchunk, trow, w, M, L, LP);
    const float inv = LP > 0.0f ? 1.0f / LP : 0.0f;
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
        float a[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) a[q] = 0.0f;
#pragma unroll
        for (int k = 0; k < kMaxChunks; ++k) {
            if (k >= nchunk || w[k] == 0.0f) continue;
            const float4 *src =
                reinterpret_cast<const float4 *>(p.part_o + (static_cast<size_t>(base + k) * kTileM + trow) * D + c * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = __ldcg(src + q);
                a[4 * q] += w[k] * v.x;
                a[4 * q + 1] += w[k] * v.y;
                a[4 * q + 2] += w[k] * v.z;
                a[4 * q + 3] += w[k] * v.w;
            }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) a[q] *= inv;
        if (rrow) {  // residual compensation: O_sparse + R
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 r = __ldg(reinterpret_cast<const float4 *>(rrow + c * 16) + q);
                a[4 * q] += r.x;
                a[4 * q + 1] += r.y;
                a[4 * q + 2] += r.z;
                a[4 * q + 3] += r.w;
            }
        }
        uint32_t pk[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) pk[q] = pack_bf16x2(a[2 * q], a[2 * q + 1]);
        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 16);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
    *lse = L > 0.0f ? (M + log2f(L)) * 0.69314718055994530942f : -CUDART_INF_F;
}

// A thread of the 4-lanes-per-row layout merges rows r and r + 8 at its column
// pairs 8g + cpair (g < D / 8).
template <int D>
__device__ __noinline__ void merge_quad(const TcParams &p, int base, int nchunk, int r, int cpair, int lane,
                                           bool lo_valid, bool hi_valid, uint32_t *o_lo, uint32_t *o_hi, float *lse_lo,
                                           float *lse_hi, const float *r_lo, const float *r_hi)
{
    float wl[kMaxChunks], wh[kMaxChunks], Ml, Ll, LPl, Mh, Lh, LPh;
    merge_weights(p, base, nchunk, r, wl, Ml, Ll, LPl);
    merge_weights(p, base, nchunk, r + 8, wh, Mh, Lh, LPh);
    const float il = LPl > 0.0f ? 1.0f / LPl : 0.0f, ih = LPh > 0.0f ? 1.0f / LPh : 0.0f;
#pragma unroll 1
    for (int g = 0; g < D / 8; ++g) {
        float2 al = make_float2(0.0f, 0.0f), ah = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < kMaxChunks; ++k) {
            if (k >= nchunk) continue;
            const float *bk = p.part_o + static_cast<size_t>(base + k) * kTileM * D + 8 * g + cpair;
            if (wl[k] != 0.0f) {
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(bk + static_cast<size_t>(r) * D));
                al.x += wl[k] * v.x;
                al.y += wl[k] * v.y;
            }
            if (wh[k] != 0.0f) {
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(bk + static_cast<size_t>(r + 8) * D));
                ah.x += wh[k] * v.x;
                ah.y += wh[k] * v.y;
            }
        }
        float2 rl = make_float2(0.0f, 0.0f), rh = make_float2(0.0f, 0.0f);
        if (r_lo) {  // residual compensation: O_sparse + R
            if (lo_valid) rl = __ldg(reinterpret_cast<const float2 *>(r_lo + 8 * g));
            if (hi_valid) rh = __ldg(reinterpret_cast<const float2 *>(r_hi + 8 * g));
        }
        if (lo_valid) o_lo[4 * g] = pack_bf16x2(fmaf(al.x, il, rl.x), fmaf(al.y, il, rl.y));
        if (hi_valid) o_hi[4 * g] = pack_bf16x2(fmaf(ah.x, ih, rh.x), fmaf(ah.y, ih, rh.y));
    }
    if ((lane & 3) == 0) {
        if (lo_valid) *lse_lo = Ll > 0.0f ? (Ml + log2f(Ll)) * 0.69314718055994530942f : -CUDART_INF_F;
        if (hi_valid) *lse_hi = Lh > 0.0f ? (Mh + log2f(Lh)) * 0.69314718055994530942f : -CUDART_INF_F;
    }
}

// Counts this warp's chunk as finished; true for the warp that finished last.
__device__ __forceinline__ bool last_chunk(const TcParams &p, int base, int nchunk, int warp, int lane)
{
    __threadfence();
    __syncwarp();
    uint32_t done = 0u;
    if (lane == 0) done = atomicAdd(p.merge_cnt + static_cast<size_t>(base) * kMergeWarps + warp, 1u);
    done = __shfl_sync(0xffffffffu, done, 0);
    const bool last = done == static_cast<uint32_t>(nchunk - 1);
    if (last) __threadfence();
    return last;
}

// SPLIT == 1: warp w (0-3) owns TMEM lanes 32w..32w+31; thread = one query row,
// all kStep columns of S (32x32b TMEM accesses). A step holds PAIR KV blocks;
// block q of the step occupies S columns [q * BS, (q + 1) * BS) and is skipped
// (P = 0, no effect on the max or the sums) when the step has no block q or the
// row's Q block does not have it.
template <int D, int BS, int NSB, int PAIR, class C, bool TOK, bool LSE>
__device__ __forceinline__ void softmax_rows(const TcParams &p, uint32_t sbase, uint32_t tmem,
                                             volatile int32_t *tile_ids, const volatile uint32_t *desc,
                                             const Ctl &ctl, int warp, int lane)
{
    auto bar = [&](int idx) -> uint32_t { return barrier_addr<C>(sbase, idx); };
    static_assert(D % 64 == 0, "the epilogue reads O in pairs of 32-column chunks");
    constexpr int kStep = C::kStep;
    constexpr int NC = kStep / 32;  // 32-column chunks of a step
    constexpr int CPB = BS / 32;    // chunks per block
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base;
    const uint32_t tO = tmem + lane_base + NSB * kStep;
    const uint32_t qblk = BS == 128 ? 0u : static_cast<uint32_t>(warp >> 1);
    const int trow = warp * 32 + lane;
    int G = 0, tcount = 0;
    for (;;) {
        int tile;
        if (!fetch_tile<C>(sbase, tile_ids, ctl, lane, tcount, tile) || tile < 0) return;
        const bool empty = (tile & kEmptyTile) != 0;
        bool row_valid;
        const int64_t grow = out_row<TOK>(p, decode_item(p, tile & ~kEmptyTile).tile, trow, row_valid);
        __nv_bfloat16 *orow = p.O + grow * D;
        if (p.R && row_valid) {  // the epilogue reads this row of the residual: start it towards L2 now
#pragma unroll
            for (int c = 0; c < D / 32; ++c) prefetch_l2(p.R + grow * D + c * 32);
        }
        if (empty && decode_item(p, tile & ~kEmptyTile).nchunk == 1) {
            if (row_valid) {
                if constexpr (!LSE) {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4 *>(orow)[c] = z;
                }
                p.LSE[grow] = -CUDART_INF_F;
            }
            continue;
        }
        // running max; the row sums stay split over partial accumulators (packed fp32
        // pairs for the fp32 sum, eight floats for the sum of bf16-rounded P) until
        // the epilogue, and a rescale scales them all
        float m_run = -CUDART_INF_F;
        uint64_t acc[2] = {0ull, 0ull};
        float accp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        bool last = empty;  // an empty chunk of a split tile has no step
        while (!last) {
            const int b = G % NSB;
            const uint32_t sd = warp_wait_step(bar(C::B_SFULL + b), (G / NSB) & 1, ctl, desc + b);
            if (sd == 0xFFFFFFFFu) return;
            tc_fence_after();
            last = desc_last(sd);
            bool act[PAIR];
            bool any = false;
#pragma unroll
            for (int q = 0; q < PAIR; ++q) {
                act[q] = q < desc_count(sd) && ((desc_members(sd, q) >> qblk) & 1u) != 0u;
                any |= act[q];
            }
            bool resc = false;
            float alpha = 1.0f;
            if (any) {
                uint32_t sv[NC][32];
#pragma unroll
                for (int c = 0; c < NC; ++c)
                    if (act[c / CPB]) tmem_ld32(tS + b * kStep + c * 32, sv[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < NC; ++c) reg_fence32(sv[c]);
                if (desc_ragged(sd) != 0u) {
                    // keys past the sequence end in a ragged last block score -inf (p = 0)
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        if (((desc_ragged(sd) >> (c / CPB)) & 1u) == 0u) continue;
                        const int key0 = (c % CPB) * 32;  // first key of chunk c within its block
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (key0 + t >= p.last_rows) sv[c][t] = 0xFF800000u;
                    }
                }
                // row max of the step's active scores, log2 units
                auto step_max = [&]() -> float {
                    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F, mx2 = -CUDART_INF_F, mx3 = -CUDART_INF_F;
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        if (!act[c / CPB]) continue;
#pragma unroll
                        for (int t = 0; t < 32; t += 8) {
                            mx0 = fmax3(mx0, __uint_as_float(sv[c][t]), __uint_as_float(sv[c][t + 1]));
                            mx1 = fmax3(mx1, __uint_as_float(sv[c][t + 2]), __uint_as_float(sv[c][t + 3]));
                            mx2 = fmax3(mx2, __uint_as_float(sv[c][t + 4]), __uint_as_float(sv[c][t + 5]));
                            mx3 = fmax3(mx3, __uint_as_float(sv[c][t + 6]), __uint_as_float(sv[c][t + 7]));
                        }
                    }
                    return fmax3(fmaxf(mx0, mx1), mx2, mx3) * p.scale_log2;
                };
                // p = 2^(s * scale * log2 e - m), P to bf16 and stored over S, and the step's two sums
                const uint64_t c2x = f2_pack(p.scale_log2, p.scale_log2);
                uint64_t sacc[2];
                float sap[4];
                auto exps = [&](float m) {
                    const uint64_t nm2 = f2_pack(-m, -m);
                    sacc[0] = sacc[1] = 0ull;
#pragma unroll
                    for (int k = 0; k < 4; ++k) sap[k] = 0.0f;
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            if (!act[c / CPB]) {
                                pk[q] = 0u;
                                continue;
                            }
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c][2 * q]), __uint_as_float(sv[c][2 * q + 1])),
                                             c2x, nm2),
                                      x0, x1);
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            sacc[q & 1] = f2_add(sacc[q & 1], f2_pack(p0, p1));
                            if constexpr (!LSE) {  // P for the PV MMA and its bf16-rounded sum
                                pk[q] = pack_bf16x2(p0, p1);
                                add_bf16x2_to_f32(sap[2 * (q & 1)], sap[2 * (q & 1) + 1], pk[q]);
                            }
                        }
                        if constexpr (!LSE) tmem_st16(tS + b * kStep + c * 16, pk);
                    }
                };
                if (m_run == -CUDART_INF_F) m_run = step_max();  // a tile's first step
                exps(m_run);
                // Lazy rescale without a max pass: a step sum of at most 2^8 bounds every p by 2^8,
                // the same condition as "no score more than 8 above the running max"; a larger sum
                // (or inf) raises the running max to the step's and redoes the step.
                // The decision is per row (register work only); the redo stores P to TMEM, so the
                // whole warp redoes the step when any row raised its max (tcgen05 accesses are
                // warp-collective), the other rows recomputing the same values.
                float s0, s1;
                f2_unpack(f2_add(sacc[0], sacc[1]), s0, s1);
                if (!(s0 + s1 <= kRescaleSum)) {
                    const float m_tile = step_max();
                    alpha = ex2_approx(m_run - m_tile);
                    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                    for (int k = 0; k < 2; ++k) acc[k] = f2_fma(acc[k], a2, 0ull);
#pragma unroll
                    for (int k = 0; k < 4; ++k) accp[k] *= alpha;
                    m_run = m_tile;
                    resc = true;
                }
                if (__any_sync(0xffffffffu, resc)) {
                    tmem_wait_st();  // the first pass's P stores land before they are overwritten
                    exps(m_run);
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) acc[k] = f2_add(acc[k], sacc[k]);
#pragma unroll
                for (int k = 0; k < 4; ++k) accp[k] += sap[k];
            } else if constexpr (!LSE) {
                uint32_t z[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) z[q] = 0u;
#pragma unroll
                for (int c = 0; c < NC; ++c) tmem_st16(tS + b * kStep + c * 16, z);
            }
            if (!LSE && __any_sync(0xffffffffu, resc)) {
                // O holds the previous steps' sum: rescale it once the last PV landed
                const int t = G - 1;
                if (!warp_wait_all(bar(C::B_PVDONE + t % NSB), (t / NSB) & 1, ctl)) return;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tO + c * 32, ov);
                    tmem_wait_ld();
                    reg_fence32(ov);
#pragma unroll
                    for (int q = 0; q < 32; ++q) ov[q] = __float_as_uint(__uint_as_float(ov[q]) * alpha);
                    tmem_st32(tO + c * 32, ov);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_PFULL + b));
            ++G;
        }
        float e0, e1;
        f2_unpack(f2_add(acc[0], acc[1]), e0, e1);
        const float l_run = e0 + e1;
        const float lp_run = (accp[0] + accp[1]) + (accp[2] + accp[3]);
        const Item it = decode_item(p, tile & ~kEmptyTile);  // decoded again: not live across the loop
        if constexpr (LSE) {  // no O: the row's LSE only (tiles are never split in this mode)
            if (row_valid) p.LSE[grow] = l_run > 0.0f ? (m_run + log2f(l_run)) * 0.69314718055994530942f : -CUDART_INF_F;
            continue;
        }
        if (it.nchunk > 1) {
            // chunk of a split tile: unnormalised partial O and the row's (m, l, lp)
            const int base = p.split_base[it.tile];
            const size_t prow = static_cast<size_t>(base + it.chunk) * kTileM + trow;
            float4 *po = reinterpret_cast<float4 *>(p.part_o + prow * D);
            if (!empty) {
                const int t = G - 1;
                if (!warp_wait_all(bar(C::B_PVDONE + t % NSB), (t / NSB) & 1, ctl)) return;
                tc_fence_after();
                // O in pairs of 32-column chunks (one load wait per pair); O is released to the
                // next tile's PV as soon as the last pair is in registers
#pragma unroll
                for (int c0 = 0; c0 < D / 32; c0 += 2) {
                    uint32_t ov[2][32];
                    tmem_ld32(tO + c0 * 32, ov[0]);
                    tmem_ld32(tO + (c0 + 1) * 32, ov[1]);
                    tmem_wait_ld();
                    reg_fence32(ov[0]);
                    reg_fence32(ov[1]);
                    if (c0 + 2 == D / 32) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(C::B_OEMPTY));
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            po[(c0 + h) * 8 + q] =
                                make_float4(__uint_as_float(ov[h][4 * q]), __uint_as_float(ov[h][4 * q + 1]),
                                            __uint_as_float(ov[h][4 * q + 2]), __uint_as_float(ov[h][4 * q + 3]));
                }
            } else {
#pragma unroll
                for (int q = 0; q < D / 4; ++q) po[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            p.part_stats[prow] = make_float4(m_run, l_run, lp_run, 0.0f);
            if (last_chunk(p, base, it.nchunk, warp, lane) && row_valid)
                merge_row<D>(p, base, it.nchunk, trow, orow, p.LSE + grow, p.R ? p.R + grow * D : nullptr);
            continue;
        }
        // epilogue: O / l, LSE = ln2 * (m + log2 l)
        const int t = G - 1;
        if (!warp_wait_all(bar(C::B_PVDONE + t % NSB), (t / NSB) & 1, ctl)) return;
        tc_fence_after();
        const float inv_l = lp_run > 0.0f ? 1.0f / lp_run : 0.0f;
        // O in pairs of 32-column chunks (one load wait per pair); O is released to the next
        // tile's PV as soon as the last pair is in registers
#pragma unroll
        for (int c0 = 0; c0 < D / 32; c0 += 2) {
            uint32_t ov[2][32];
            tmem_ld32(tO + c0 * 32, ov[0]);
            tmem_ld32(tO + (c0 + 1) * 32, ov[1]);
            tmem_wait_ld();
            reg_fence32(ov[0]);
            reg_fence32(ov[1]);
            if (c0 + 2 == D / 32) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_OEMPTY));
            }
            if (row_valid) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = c0 + h;
                    uint32_t pk[16];
                    if (p.R) {  // residual compensation: O_sparse + R
                        const float4 *rs = reinterpret_cast<const float4 *>(p.R + grow * D + c * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 r = __ldg(rs + q);
                            pk[2 * q] = pack_bf16x2(fmaf(__uint_as_float(ov[h][4 * q]), inv_l, r.x),
                                                    fmaf(__uint_as_float(ov[h][4 * q + 1]), inv_l, r.y));
                            pk[2 * q + 1] = pack_bf16x2(fmaf(__uint_as_float(ov[h][4 * q + 2]), inv_l, r.z),
                                                        fmaf(__uint_as_float(ov[h][4 * q + 3]), inv_l, r.w));
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            pk[q] = pack_bf16x2(__uint_as_float(ov[h][2 * q]) * inv_l,
                                                __uint_as_float(ov[h][2 * q + 1]) * inv_l);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
        }
        if (row_valid) p.LSE[grow] = l_run > 0.0f ? (m_run + log2f(l_run)) * 0.69314718055994530942f : -CUDART_INF_F;
    }
}

// SPLIT == 2: eight warps; warp w owns the 16 TMEM lanes 32*(w%4) + 16*(w/4)..
// (16x256b / 16x128b accesses). Thread t holds rows t/4 and t/4 + 8 of that
// group and, in every 8-column group of S and O, columns 2(t%4) and +1; a row's
// max and sums are reduced over its 4 lanes with two shuffles. A step holds PAIR
// KV blocks: 8-column group g of the step belongs to block g / (BS / 8).
template <int D, int BS, int NSB, int PAIR, class C, bool TOK, bool LSE>
__device__ __forceinline__ void softmax_quads(const TcParams &p, uint32_t sbase, uint32_t tmem,
                                              volatile int32_t *tile_ids, const volatile uint32_t *desc,
                                              const Ctl &ctl, int warp, int lane)
{
    auto bar = [&](int idx) -> uint32_t { return barrier_addr<C>(sbase, idx); };
    constexpr int RS = C::kStep / 8;  // 8-column groups of a step's S
    constexpr int GPB = BS / 8;       // groups per block
    constexpr int RO = D / 8;   // 8-column groups of O
    const int quarter = warp & 3;
    const int lane0 = 32 * quarter + 16 * (warp >> 2);  // first tile row of this warp
    const uint32_t tbase = tmem + (static_cast<uint32_t>(lane0) << 16);
    const uint32_t tO = tbase + NSB * C::kStep;
    const int r_lo = lane0 + (lane >> 2);  // this thread's rows r_lo and r_lo + 8
    const int cpair = 2 * (lane & 3);
    const uint32_t qblk = BS == 128 ? 0u : static_cast<uint32_t>(quarter >> 1);
    int G = 0, tcount = 0;
    for (;;) {
        int tile;
        if (!fetch_tile<C>(sbase, tile_ids, ctl, lane, tcount, tile) || tile < 0) return;
        const bool empty = (tile & kEmptyTile) != 0;
        const Item it = decode_item(p, tile & ~kEmptyTile);
        bool lo_valid, hi_valid;
        const int64_t g_lo = out_row<TOK>(p, it.tile, r_lo, lo_valid);
        const int64_t g_hi = out_row<TOK>(p, it.tile, r_lo + 8, hi_valid);
        uint32_t *o_lo = reinterpret_cast<uint32_t *>(p.O + g_lo * D + cpair);
        uint32_t *o_hi = reinterpret_cast<uint32_t *>(p.O + g_hi * D + cpair);
        if (p.R && (lane & 3) < D / 32) {  // the epilogue reads these residual rows: start them towards L2 now
            if (lo_valid) prefetch_l2(p.R + g_lo * D + 32 * (lane & 3));
            if (hi_valid) prefetch_l2(p.R + g_hi * D + 32 * (lane & 3));
        }
        if (empty && it.nchunk == 1) {
            if constexpr (!LSE) {
#pragma unroll
                for (int g = 0; g < RO; ++g) {
                    if (lo_valid) o_lo[4 * g] = 0u;
                    if (hi_valid) o_hi[4 * g] = 0u;
                }
            }
            if ((lane & 3) == 0) {
                if (lo_valid) p.LSE[g_lo] = -CUDART_INF_F;
                if (hi_valid) p.LSE[g_hi] = -CUDART_INF_F;
            }
            continue;
        }
        // running maxima; the sums of this thread's columns stay in partial
        // accumulators (packed fp32 pairs; floats for the bf16-rounded P) until the
        // epilogue, and a rescale scales them
        float m_lo = -CUDART_INF_F, m_hi = -CUDART_INF_F;
        uint64_t acc_lo[2] = {0ull, 0ull}, acc_hi[2] = {0ull, 0ull};
        float ap_lo[4] = {0.0f, 0.0f, 0.0f, 0.0f}, ap_hi[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        bool last = empty;  // an empty chunk of a split tile has no step
        while (!last) {
            const int b = G % NSB;
            const uint32_t sd = warp_wait_step(bar(C::B_SFULL + b), (G / NSB) & 1, ctl, desc + b);
            if (sd == 0xFFFFFFFFu) return;
            tc_fence_after();
            last = desc_last(sd);
            bool resc = false;
            float a_lo = 1.0f, a_hi = 1.0f;
            bool act[PAIR];
            bool any = false;
#pragma unroll
            for (int q = 0; q < PAIR; ++q) {
                act[q] = q < desc_count(sd) && ((desc_members(sd, q) >> qblk) & 1u) != 0u;
                any |= act[q];
            }
            if (any) {
                uint32_t sv[4 * RS];
                tmem_ld_16x256b<RS>(tbase + b * C::kStep, sv);
                tmem_wait_ld();
                reg_fence(sv);
                if (desc_ragged(sd) != 0u) {
                    // keys past the sequence end in a ragged last block score -inf (p = 0)
#pragma unroll
                    for (int g = 0; g < RS; ++g) {
                        if (((desc_ragged(sd) >> (g / GPB)) & 1u) == 0u) continue;
                        const int key = (g % GPB) * 8 + cpair;  // this thread's first key of group g
                        if (key >= p.last_rows) sv[4 * g] = sv[4 * g + 2] = 0xFF800000u;
                        if (key + 1 >= p.last_rows) sv[4 * g + 1] = sv[4 * g + 3] = 0xFF800000u;
                    }
                }
                float x0 = -CUDART_INF_F, x1 = -CUDART_INF_F, y0 = -CUDART_INF_F, y1 = -CUDART_INF_F;
#pragma unroll
                for (int g = 0; g < RS; g += 2) {
                    if (!act[g / GPB]) continue;
                    x0 = fmax3(x0, __uint_as_float(sv[4 * g]), __uint_as_float(sv[4 * g + 1]));
                    y0 = fmax3(y0, __uint_as_float(sv[4 * g + 2]), __uint_as_float(sv[4 * g + 3]));
                    x1 = fmax3(x1, __uint_as_float(sv[4 * g + 4]), __uint_as_float(sv[4 * g + 5]));
                    y1 = fmax3(y1, __uint_as_float(sv[4 * g + 6]), __uint_as_float(sv[4 * g + 7]));
                }
                float mx_lo = fmaxf(x0, x1), mx_hi = fmaxf(y0, y1);
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
                const float t_lo = mx_lo * p.scale_log2, t_hi = mx_hi * p.scale_log2;
                if (m_lo == -CUDART_INF_F) {
                    m_lo = t_lo;
                } else if (t_lo > m_lo + kRescaleLog2) {
                    a_lo = ex2_approx(m_lo - t_lo);
                    const uint64_t a2 = f2_pack(a_lo, a_lo);
                    acc_lo[0] = f2_fma(acc_lo[0], a2, 0ull);
                    acc_lo[1] = f2_fma(acc_lo[1], a2, 0ull);
#pragma unroll
                    for (int k = 0; k < 4; ++k) ap_lo[k] *= a_lo;
                    m_lo = t_lo;
                    resc = true;
                }
                if (m_hi == -CUDART_INF_F) {
                    m_hi = t_hi;
                } else if (t_hi > m_hi + kRescaleLog2) {
                    a_hi = ex2_approx(m_hi - t_hi);
                    const uint64_t a2 = f2_pack(a_hi, a_hi);
                    acc_hi[0] = f2_fma(acc_hi[0], a2, 0ull);
                    acc_hi[1] = f2_fma(acc_hi[1], a2, 0ull);
#pragma unroll
                    for (int k = 0; k < 4; ++k) ap_hi[k] *= a_hi;
                    m_hi = t_hi;
                    resc = true;
                }
                const uint64_t c2x = f2_pack(p.scale_log2, p.scale_log2);
                const uint64_t nm_lo = f2_pack(-m_lo, -m_lo), nm_hi = f2_pack(-m_hi, -m_hi);
                uint32_t pk[2 * RS];
#pragma unroll
                for (int g = 0; g < RS; ++g) {
                    if (!act[g / GPB]) {
                        pk[2 * g] = pk[2 * g + 1] = 0u;
                        continue;
                    }
                    float x, y;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[4 * g]), __uint_as_float(sv[4 * g + 1])), c2x, nm_lo),
                              x, y);
                    const float p0 = ex2_approx(x), p1 = ex2_approx(y);
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[4 * g + 2]), __uint_as_float(sv[4 * g + 3])), c2x,
                                     nm_hi),
                              x, y);
                    const float p2 = ex2_approx(x), p3 = ex2_approx(y);
                    acc_lo[g & 1] = f2_add(acc_lo[g & 1], f2_pack(p0, p1));
                    acc_hi[g & 1] = f2_add(acc_hi[g & 1], f2_pack(p2, p3));
                    if constexpr (!LSE) {  // P for the PV MMA and its bf16-rounded sums
                        pk[2 * g] = pack_bf16x2(p0, p1);      // row r_lo, packed column 4g + t%4
                        pk[2 * g + 1] = pack_bf16x2(p2, p3);  // row r_lo + 8
                        add_bf16x2_to_f32(ap_lo[2 * (g & 1)], ap_lo[2 * (g & 1) + 1], pk[2 * g]);
                        add_bf16x2_to_f32(ap_hi[2 * (g & 1)], ap_hi[2 * (g & 1) + 1], pk[2 * g + 1]);
                    }
                }
                if constexpr (!LSE) tmem_st_16x128b<RS>(tbase + b * C::kStep, pk);
            } else if constexpr (!LSE) {
                uint32_t z[2 * RS];
#pragma unroll
                for (int q = 0; q < 2 * RS; ++q) z[q] = 0u;
                tmem_st_16x128b<RS>(tbase + b * C::kStep, z);
            }
            if (!LSE && __any_sync(0xffffffffu, resc)) {
                const int t = G - 1;
                if (!warp_wait_all(bar(C::B_PVDONE + t % NSB), (t / NSB) & 1, ctl)) return;
                tc_fence_after();
                uint32_t ov[4 * RO];
                tmem_ld_16x256b<RO>(tO, ov);
                tmem_wait_ld();
                reg_fence(ov);
#pragma unroll
                for (int g = 0; g < RO; ++g) {
                    ov[4 * g] = __float_as_uint(__uint_as_float(ov[4 * g]) * a_lo);
                    ov[4 * g + 1] = __float_as_uint(__uint_as_float(ov[4 * g + 1]) * a_lo);
                    ov[4 * g + 2] = __float_as_uint(__uint_as_float(ov[4 * g + 2]) * a_hi);
                    ov[4 * g + 3] = __float_as_uint(__uint_as_float(ov[4 * g + 3]) * a_hi);
                }
                tmem_st_16x256b<RO>(tO, ov);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_PFULL + b));
            ++G;
        }
        // epilogue: whole-row sums over the 4 lanes of each row, then O / l and LSE
        float l_lo, l_hi;
        {
            float u0, u1, w0, w1;
            f2_unpack(f2_add(acc_lo[0], acc_lo[1]), u0, u1);
            f2_unpack(f2_add(acc_hi[0], acc_hi[1]), w0, w1);
            l_lo = u0 + u1;
            l_hi = w0 + w1;
        }
        float lp_lo = (ap_lo[0] + ap_lo[1]) + (ap_lo[2] + ap_lo[3]);
        float lp_hi = (ap_hi[0] + ap_hi[1]) + (ap_hi[2] + ap_hi[3]);
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, o);
            l_hi += __shfl_xor_sync(0xffffffffu, l_hi, o);
            lp_lo += __shfl_xor_sync(0xffffffffu, lp_lo, o);
            lp_hi += __shfl_xor_sync(0xffffffffu, lp_hi, o);
        }
        if constexpr (LSE) {  // no O: the rows' LSE only (tiles are never split in this mode)
            if ((lane & 3) == 0) {
                if (lo_valid) p.LSE[g_lo] = l_lo > 0.0f ? (m_lo + log2f(l_lo)) * 0.69314718055994530942f : -CUDART_INF_F;
                if (hi_valid) p.LSE[g_hi] = l_hi > 0.0f ? (m_hi + log2f(l_hi)) * 0.69314718055994530942f : -CUDART_INF_F;
            }
            continue;
        }
        if (it.nchunk > 1) {
            // chunk of a split tile: unnormalised partial O and the rows' (m, l, lp)
            const int base = p.split_base[it.tile];
            const size_t srow = static_cast<size_t>(base + it.chunk) * kTileM;
            float *po_lo = p.part_o + (srow + r_lo) * D + cpair;
            float *po_hi = p.part_o + (srow + r_lo + 8) * D + cpair;
            if (!empty) {
                const int t = G - 1;
                if (!warp_wait_all(bar(C::B_PVDONE + t % NSB), (t / NSB) & 1, ctl)) return;
                tc_fence_after();
                uint32_t ov[4 * RO];
                tmem_ld_16x256b<RO>(tO, ov);
                tmem_wait_ld();
                reg_fence(ov);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_OEMPTY));
#pragma unroll
                for (int g = 0; g < RO; ++g) {
                    *reinterpret_cast<float2 *>(po_lo + 8 * g) =
                        make_float2(__uint_as_float(ov[4 * g]), __uint_as_float(ov[4 * g + 1]));
                    *reinterpret_cast<float2 *>(po_hi + 8 * g) =
                        make_float2(__uint_as_float(ov[4 * g + 2]), __uint_as_float(ov[4 * g + 3]));
                }
            } else {
#pragma unroll
                for (int g = 0; g < RO; ++g) {
                    *reinterpret_cast<float2 *>(po_lo + 8 * g) = make_float2(0.0f, 0.0f);
                    *reinterpret_cast<float2 *>(po_hi + 8 * g) = make_float2(0.0f, 0.0f);
                }
            }
            if ((lane & 3) == 0) {
                p.part_stats[srow + r_lo] = make_float4(m_lo, l_lo, lp_lo, 0.0f);
                p.part_stats[srow + r_lo + 8] = make_float4(m_hi, l_hi, lp_hi, 0.0f);
            }
            if (last_chunk(p, base, it.nchunk, warp, lane))
                merge_quad<D>(p, base, it.nchunk, r_lo, cpair, lane, lo_valid, hi_valid, o_lo, o_hi, p.LSE + g_lo,
                              p.LSE + g_hi, p.R ? p.R + g_lo * D + cpair : nullptr,
                              p.R ? p.R + g_hi * D + cpair : nullptr);
            continue;
        }
        const int t = G - 1;
        if (!warp_wait_all(bar(C::B_PVDONE + t % NSB), (t / NSB) & 1, ctl)) return;
        tc_fence_after();
        uint32_t ov[4 * RO];
        tmem_ld_16x256b<RO>(tO, ov);
        tmem_wait_ld();
        reg_fence(ov);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_OEMPTY));
        const float i_lo = lp_lo > 0.0f ? 1.0f / lp_lo : 0.0f, i_hi = lp_hi > 0.0f ? 1.0f / lp_hi : 0.0f;
#pragma unroll
        for (int g = 0; g < RO; ++g) {
            float2 rl = make_float2(0.0f, 0.0f), rh = make_float2(0.0f, 0.0f);
            if (p.R) {  // residual compensation: O_sparse + R
                if (lo_valid) rl = __ldg(reinterpret_cast<const float2 *>(p.R + g_lo * D + cpair + 8 * g));
                if (hi_valid) rh = __ldg(reinterpret_cast<const float2 *>(p.R + g_hi * D + cpair + 8 * g));
            }
            if (lo_valid)
                o_lo[4 * g] = pack_bf16x2(fmaf(__uint_as_float(ov[4 * g]), i_lo, rl.x),
                                          fmaf(__uint_as_float(ov[4 * g + 1]), i_lo, rl.y));
            if (hi_valid)
                o_hi[4 * g] = pack_bf16x2(fmaf(__uint_as_float(ov[4 * g + 2]), i_hi, rh.x),
                                          fmaf(__uint_as_float(ov[4 * g + 3]), i_hi, rh.y));
        }
        if ((lane & 3) == 0) {
            if (lo_valid) p.LSE[g_lo] = l_lo > 0.0f ? (m_lo + log2f(l_lo)) * 0.69314718055994530942f : -CUDART_INF_F;
            if (hi_valid) p.LSE[g_hi] = l_hi > 0.0f ? (m_hi + log2f(l_hi)) * 0.69314718055994530942f : -CUDART_INF_F;
        }
    }
}

template <int D, int BS, int NK, int NV, int NSB, int QS, int SPLIT, int PAIR, int MINB, bool TOK = false,
          bool LSE = false>
__global__ void __launch_bounds__((4 * SPLIT + 4) * 32, MINB)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const TcParams p)
{
    static_assert(!TOK || (BS == kTileM && PAIR == 1), "token mode: 128-key steps");
    static_assert(!(TOK && LSE), "the LSE-only mode runs over a block index");
    using C = Cfg<D, BS, NK, NV, NSB, QS, PAIR>;
    using R = Roles<SPLIT>;
    constexpr int kProducerWarp = R::kProducerWarp, kQkWarp = R::kQkWarp, kMmaWarp = R::kMmaWarp;
    constexpr int kVProducerWarp = R::kVProducerWarp;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int idx) -> uint32_t { return sbase + C::BAR_OFF + 8u * idx; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    // misc[0]: TMEM base, misc[1]: abort flag, misc[2..3]: tile ids of the scheduler ring,
    // misc[4..4+NSB): step descriptors of the S/P buffers, misc[4+NSB..4+NSB+NK): those of the K ring
    volatile int32_t *tile_ids = reinterpret_cast<volatile int32_t *>(misc + 2);
    volatile uint32_t *desc = reinterpret_cast<volatile uint32_t *>(misc + 4);
    volatile uint32_t *kdesc = desc + NSB;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int q = 0; q < QS; ++q) {
            mbar_init(bar(C::B_QFULL + q), 1);
            mbar_init(bar(C::B_QEMPTY + q), 1);
        }
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_VEMPTY + s), 1);
        }
        for (int b = 0; b < NSB; ++b) {
            mbar_init(bar(C::B_SFULL + b), 2);  // the issuer's arrive (descriptor) + the QK^T commit
            mbar_init(bar(C::B_PFULL + b), R::kSoftmaxWarps);
            mbar_init(bar(C::B_PVDONE + b), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::B_TFULL + b), 1);
            mbar_init(bar(C::B_TEMPTY + b), R::kSoftmaxWarps + 3);  // softmax, QK^T, PV, V producer
        }
        mbar_init(bar(C::B_OEMPTY), R::kSoftmaxWarps);
        mbar_init(bar(C::B_DRAIN), 1);
        mbar_init(bar(C::B_DRAIN + 1), 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(misc), C::TCOLS);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the prologue above may overlap the work-list launch; its results are read from here on
    grid_dependency_wait();
    const uint32_t tmem = misc[0];
    const Ctl ctl{reinterpret_cast<volatile uint32_t *>(misc + 1), p.err, p.wait_limit_ns};
    const bool stall = (p.dbg & kDbgStall) != 0u;

    if (TOK && warp == kProducerWarp) {
        // ------------------------------------------------------------ token mode: tiles, Q and K
        // Every tile (one query group) has the same steps, so CTA b takes tiles b, b + grid,
        // ... in order. Q rows come through the permutation by TMA gathers (four rows per
        // gather, every lane issuing its own rows). K rows come through the group's token
        // list by cp.async: the TMA engine's gathers of scattered rows ran at about 3 TB/s
        // and set the pace of a step, the load/store path moves them faster. A step is
        // published one step late: once its copies have landed (wait_group 1 while the next
        // step's are in flight) and been fenced for the tensor-core reads, one lane arrives on
        // its K-full barrier with the step descriptor; a tile's last step is published before
        // the next tile's Q slot is awaited.
        if constexpr (TOK) {
            const int steps = (p.n_tok + kTileM - 1) / kTileM;
            const bool ragged = p.n_tok % kTileM != 0;
            int G = 0, e = 0, tcount = 0, kpend = -1;  // kpend: the step copied but not yet published
            int q_issued = -1;
            bool ok = true;
            while (ok) {
                const int slot = tcount & 1;
                if (tcount >= 2 && !warp_wait_all(bar(C::B_TEMPTY + slot), ((tcount >> 1) - 1) & 1, ctl)) break;
                const int id = blockIdx.x + tcount * static_cast<int>(gridDim.x);
                const int item = id < p.n_tiles ? id : -1;
                if (lane == 0) {
                    tile_ids[slot] = item;
                    mbar_arrive(bar(C::B_TFULL + slot));
                }
                ++tcount;
                if (item < 0) break;
                if (stall) continue;
                const int64_t bh = item / p.groups;
                const int qs = e % QS;
                if (e >= QS && !warp_wait_all(bar(C::B_QEMPTY + qs), ((e / QS) - 1) & 1, ctl)) break;
                const int32_t *toks = p.tokens + static_cast<int64_t>(item) * p.n_tok;
                // the first K step's indices load with the Q rows'; later ones one step ahead
                int nxt[4];
                gather_idx(toks, min(kTileM, p.n_tok), lane, nxt);
                int rows[4];
                gather_rows(p, p.perm + static_cast<int64_t>(item) * kTileM, kTileM, bh, lane, rows);
                if (lane == 0) mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::kQBytes);
                __syncwarp();
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_gather4(sbase + C::Q_OFF + qs * C::kQBytes + c * C::kQChunk + lane * 512, &tmQ, c * 64,
                                rows[0], rows[1], rows[2], rows[3], bar(C::B_QFULL + qs));
                __syncwarp();
                q_issued = e;
                for (int st = 0; st < steps; ++st) {
                    const int ks = G % NK;
                    gather_rows_of(p, nxt, bh, rows);
                    if (st + 1 < steps)
                        gather_idx(toks + (st + 1) * kTileM, min(kTileM, p.n_tok - (st + 1) * kTileM), lane, nxt);
                    if (G >= NK && !warp_wait_all(bar(C::B_KEMPTY + ks), ((G / NK) - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        const uint32_t ms[2] = {3u, 0u};
                        kdesc[ks] = step_desc(1, ms, st == steps - 1, ragged && st == steps - 1 ? 1u : 0u);
                    }
                    copy_rows_async<D>(sbase + C::K_OFF + ks * C::kKVBytes, C::kKVChunk, p.Kg, rows, lane);
                    cp_async_commit();
                    if (kpend >= 0) {
                        cp_async_wait_group<1>();
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(C::B_KFULL + kpend % NK));
                    }
                    kpend = G;
                    ++G;
                }
                if (kpend >= 0) {
                    cp_async_wait_group<0>();
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_KFULL + kpend % NK));
                    kpend = -1;
                }
                ++e;
            }
            // never leave while our copies or gathers may still land in shared memory
            cp_async_wait_group<0>();
            if (lane == 0 && *ctl.abort_flag) {
                for (int e2 = q_issued - (QS - 1) < 0 ? 0 : q_issued - (QS - 1); e2 <= q_issued; ++e2)
                    wait_bar_drain(bar(C::B_QFULL + e2 % QS), (e2 / QS) & 1, p.wait_limit_ns);
            }
            __syncwarp();
        }
    } else if (TOK && warp == kVProducerWarp) {
        // ------------------------------------------------------------ token mode: V by cp.async
        // Like K: the step's rows copied by cp.async, published one step late on V-full.
        if constexpr (TOK) {
            if (!stall) {
                const int steps = (p.n_tok + kTileM - 1) / kTileM;
                int G = 0, tcount = 0, vpend = -1;  // vpend: the step copied but not yet published
                bool ok = true;
                while (ok) {
                    int tile;
                    if (!fetch_tile<C>(sbase, tile_ids, ctl, lane, tcount, tile)) break;
                    if (tile < 0) break;
                    const int64_t bh = tile / p.groups;
                    const int32_t *toks = p.tokens + static_cast<int64_t>(tile) * p.n_tok;
                    int nxt[4];  // the next step's indices, loaded one step ahead
                    gather_idx(toks, min(kTileM, p.n_tok), lane, nxt);
                    for (int st = 0; st < steps; ++st) {
                        const int vs = G % NV;
                        int rows[4];
                        gather_rows_of(p, nxt, bh, rows);
                        if (st + 1 < steps)
                            gather_idx(toks + (st + 1) * kTileM, min(kTileM, p.n_tok - (st + 1) * kTileM), lane, nxt);
                        if (G >= NV && !warp_wait_all(bar(C::B_VEMPTY + vs), ((G / NV) - 1) & 1, ctl)) {
                            ok = false;
                            break;
                        }
                        copy_rows_async<D>(sbase + C::V_OFF + vs * C::kKVBytes, C::kKVChunk, p.Vg, rows, lane);
                        cp_async_commit();
                        if (vpend >= 0) {
                            cp_async_wait_group<1>();
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar(C::B_VFULL + vpend % NV));
                        }
                        vpend = G;
                        ++G;
                    }
                    if (vpend >= 0) {
                        cp_async_wait_group<0>();
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(C::B_VFULL + vpend % NV));
                        vpend = -1;
                    }
                }
                cp_async_wait_group<0>();  // never leave while copies may still land in shared memory
                __syncwarp();
            }
        }
    } else if (warp == kProducerWarp) {
        // ------------------------------------------------------------ tile scheduler, Q and K producer
        // Whole-warp loop (uniform waits and walk); one elected lane issues the copies.
        // This warp is the walker of the K side: with one step of lookahead it leaves
        // each step's descriptor (blocks, members, last) beside its K slot, released by
        // the K-full barrier, so the QK^T issuer has no index reads on its path.
        {
            int G = 0, e = 0, tcount = 0;
            int last_issue = -1;  // last step whose K loads were issued
            int q_issued = -1;
            bool ok = true;
            // written by the tile-order launch before this one (or the plan gate of a planned call)
            const uint32_t n_items = *p.n_items;
            while (ok) {
                const int slot = tcount & 1;
                if (tcount >= 2 && !warp_wait_all(bar(C::B_TEMPTY + slot), ((tcount >> 1) - 1) & 1, ctl)) break;
                int item = -1;
                if (lane == 0) {
                    const uint32_t id = atomicAdd(p.tile_counter, 1u);
                    item = id < n_items ? p.tile_list[id] : -1;
                }
                item = __shfl_sync(0xffffffffu, item, 0);
                int64_t bh = 0;
                int qt = 0;
                TileWalk walk;
                int js[2], jn[2];
                uint32_t ms[2], mn[2];
                int cnt = 0;
                if (item >= 0) {
                    const Item it = decode_item(p, item);
                    int j_lo, j_hi;
                    chunk_range(p, it, j_lo, j_hi);
                    tile_coords(p, it.tile, bh, qt);
                    walk_init<BS>(walk, p, bh, qt, j_lo, j_hi);
                    cnt = walk.next_step<PAIR>(js, ms);
                }
                if (lane == 0) {
                    tile_ids[slot] = item >= 0 && cnt == 0 ? (item | kEmptyTile) : item;
                    mbar_arrive(bar(C::B_TFULL + slot));
                }
                ++tcount;
                if (item < 0) break;
                if (stall || cnt == 0) continue;  // empty tile: nothing to load
                const int qs = e % QS;  // Q slot; it was last used by tile e - QS
                if (e >= QS && !warp_wait_all(bar(C::B_QEMPTY + qs), ((e / QS) - 1) & 1, ctl)) break;
                __syncwarp();
                if (elect_one()) {
                    mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::kQBytes);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_3d(sbase + C::Q_OFF + qs * C::kQBytes + c * C::kQChunk, &tmQ, c * 64, qt * kTileM,
                                    static_cast<int>(bh), bar(C::B_QFULL + qs));
                }
                __syncwarp();
                q_issued = e;
                int cnt_n = walk.next_step<PAIR>(jn, mn);
                do {
                    // K slot: freed when the QK^T that read it completes
                    const int ks = G % NK;
                    if (G >= NK && !warp_wait_all(bar(C::B_KEMPTY + ks), ((G / NK) - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        // released by the arrive below
                        kdesc[ks] = step_desc(cnt, ms, cnt_n == 0, ragged_bits(p, js, cnt));
                        mbar_arrive_expect_tx(bar(C::B_KFULL + ks), static_cast<uint32_t>(cnt * BS * D * 2));
                        for (int q = 0; q < cnt; ++q) {
#pragma unroll
                            for (int c = 0; c < D / 64; ++c)
                                tma_load_3d(sbase + C::K_OFF + ks * C::kKVBytes + c * C::kKVChunk + q * BS * 128,
                                            &tmK, c * 64, js[q] * BS, static_cast<int>(bh), bar(C::B_KFULL + ks));
                        }
                    }
                    __syncwarp();
                    last_issue = G;
                    ++G;
                    cnt = cnt_n;
                    js[0] = jn[0];
                    js[1] = jn[1];
                    ms[0] = mn[0];
                    ms[1] = mn[1];
                    if (cnt != 0) cnt_n = walk.next_step<PAIR>(jn, mn);
                } while (cnt != 0);
                ++e;
            }
            if (lane == 0 && *ctl.abort_flag) {
                // never leave while our copies may still land in shared memory
                for (int g = last_issue - NK + 1; g <= last_issue; ++g)
                    if (g >= 0) wait_bar_drain(bar(C::B_KFULL + g % NK), (g / NK) & 1, p.wait_limit_ns);
                for (int e2 = q_issued - (QS - 1) < 0 ? 0 : q_issued - (QS - 1); e2 <= q_issued; ++e2)
                    wait_bar_drain(bar(C::B_QFULL + e2 % QS), (e2 / QS) & 1, p.wait_limit_ns);
            }
            __syncwarp();
        }
    } else if (LSE && warp == kVProducerWarp) {
        // ------------------------------------------------------------ LSE only: no V to load
        int tcount = 0;
        for (;;) {
            int tile;
            if (!fetch_tile<C>(sbase, tile_ids, ctl, lane, tcount, tile) || tile < 0) break;
        }
    } else if (warp == kVProducerWarp) {
        // ------------------------------------------------------------ V producer
        // Walks each tile on its own, so a V slot still held by a lagging PV never
        // delays the K loads that QK^T waits for.
        if (!stall) {
            int G = 0, tcount = 0;
            int last_issue = -1;  // last step whose V loads were issued
            bool ok = true;
            while (ok) {
                int tile;
                if (!fetch_tile<C>(sbase, tile_ids, ctl, lane, tcount, tile)) break;
                if (tile < 0) break;
                if (tile & kEmptyTile) continue;
                const Item it = decode_item(p, tile);
                int j_lo, j_hi;
                chunk_range(p, it, j_lo, j_hi);
                int64_t bh;
                int qt;
                tile_coords(p, it.tile, bh, qt);
                TileWalk walk;
                walk_init<BS>(walk, p, bh, qt, j_lo, j_hi);
                int js[2];
                uint32_t ms[2];
                int cnt;
                while ((cnt = walk.next_step<PAIR>(js, ms)) != 0) {
                    // V slot: freed when the PV that read it completes
                    const int vs = G % NV;
                    if (G >= NV && !warp_wait_all(bar(C::B_VEMPTY + vs), ((G / NV) - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        mbar_arrive_expect_tx(bar(C::B_VFULL + vs), static_cast<uint32_t>(cnt * BS * D * 2));
                        for (int q = 0; q < cnt; ++q) {
#pragma unroll
                            for (int c = 0; c < D / 64; ++c)
                                tma_load_3d(sbase + C::V_OFF + vs * C::kKVBytes + c * C::kKVChunk + q * BS * 128,
                                            &tmV, c * 64, js[q] * BS, static_cast<int>(bh), bar(C::B_VFULL + vs));
                        }
                    }
                    __syncwarp();
                    last_issue = G;
                    ++G;
                }
            }
            if (lane == 0 && *ctl.abort_flag) {
                for (int g = last_issue - NV + 1; g <= last_issue; ++g)
                    if (g >= 0) wait_bar_drain(bar(C::B_VFULL + g % NV), (g / NV) & 1, p.wait_limit_ns);
            }
            __syncwarp();
        }
    } else if (warp == kQkWarp) {
        // ------------------------------------------------------------ QK^T issuer
        // Runs ahead of the softmax: QK^T of step G needs only K(G) and S/P buffer
        // G % NSB, which is free once PV(G - NSB) completed. The whole warp runs the
        // loop (waits are warp-uniform) and one elected lane issues: tcgen05
        // issue from converged code is several times cheaper than from a lone lane.
        if (!stall) {
            const uint32_t tS = tmem;  // NSB S/P buffers of kStep columns
            // shared-memory descriptor of K slot 0 (slots and steps are added as offsets:
            // the address field holds addr >> 4 and never carries for these sizes)
            const uint64_t kdesc0 = sdesc_sw128(sbase + C::K_OFF, 16, 1024);
            int G = 0, e = 0, tcount = 0;
            bool ok = true;
            while (ok) {
                const int slot = tcount & 1;
                if (!warp_wait_all(bar(C::B_TFULL + slot), (tcount >> 1) & 1, ctl)) break;
                const int tile = tile_ids[slot];
                if (lane == 0) mbar_arrive(bar(C::B_TEMPTY + slot));
                ++tcount;
                if (tile < 0) break;
                if (tile & kEmptyTile) continue;
                const int qs = e % QS;
                if (!warp_wait_all(bar(C::B_QFULL + qs), (e / QS) & 1, ctl)) break;
                tc_fence_after();
                const uint64_t qdesc = sdesc_sw128(sbase + C::Q_OFF + qs * C::kQBytes, 16, 1024);
                bool last;
                do {
                    const int s = G % NK, b = G % NSB;
                    // the step's descriptor comes with its K slot (left there by the K producer)
                    const uint32_t sd = warp_wait_step(bar(C::B_KFULL + s), (G / NK) & 1, ctl, kdesc + s);
                    if (sd == 0xFFFFFFFFu) { ok = false; break; }
                    // S/P buffer b (and its descriptor) was last read by PV(G - NSB)
                    if (G >= NSB && !warp_wait_all(bar(C::B_PVDONE + b), ((G / NSB) - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        desc[b] = sd;
                        mbar_arrive(bar(C::B_SFULL + b));  // release: the descriptor is visible with the phase
                    }
                    tc_fence_after();
                    last = desc_last(sd);
                    // K-major, 128-byte swizzle: step kk is 32 bytes into 64-column slab kk / 4
                    const uint64_t kdesc_s = kdesc0 + static_cast<uint64_t>(s * (C::kKVBytes >> 4));
                    const uint32_t idesc = desc_count(sd) == PAIR ? C::IDESC_QK : C::IDESC_QK_HALF;
                    __syncwarp();
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t off_q = static_cast<uint64_t>(((kk >> 2) * C::kQChunk + (kk & 3) * 32) >> 4);
                            const uint64_t off_k = static_cast<uint64_t>(((kk >> 2) * C::kKVChunk + (kk & 3) * 32) >> 4);
                            mma_ss(tS + b * C::kStep, qdesc + off_q, kdesc_s + off_k, idesc, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(bar(C::B_SFULL + b));
                        tc_commit(bar(C::B_KEMPTY + s));
                    }
                    __syncwarp();
                    ++G;
                } while (!last);
                if (!ok) break;
                // the tile's last QK^T: its Q slot is free once these MMAs complete
                if (elect_one()) tc_commit(bar(C::B_QEMPTY + qs));
                __syncwarp();
                ++e;
            }
            // all MMAs issued by the elected lane have completed before TMEM is freed
            __syncwarp();
            if (elect_one()) {
                tc_commit(bar(C::B_DRAIN + 1));
                wait_bar_drain(bar(C::B_DRAIN + 1), 0, p.wait_limit_ns);
            }
            __syncwarp();
        }
    } else if (LSE && warp == kMmaWarp) {
        // ------------------------------------------------------------ LSE only: no PV
        // A buffer is free again as soon as every softmax warp has loaded its S.
        if (!stall) {
            int G = 0, tcount = 0;
            bool ok = true;
            while (ok) {
                const int slot = tcount & 1;
                if (!warp_wait_all(bar(C::B_TFULL + slot), (tcount >> 1) & 1, ctl)) break;
                const int tile = tile_ids[slot];
                if (lane == 0) mbar_arrive(bar(C::B_TEMPTY + slot));
                ++tcount;
                if (tile < 0) break;
                if (tile & kEmptyTile) continue;
                bool last;
                do {
                    const int b = G % NSB;
                    if (!warp_wait_all(bar(C::B_PFULL + b), (G / NSB) & 1, ctl)) { ok = false; break; }
                    last = desc_last(desc[b]);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_PVDONE + b));
                    ++G;
                } while (!last);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ PV issuer
        // Whole-warp loop with one elected issuing lane, like the QK^T issuer.
        if (!stall) {
            const uint32_t tS = tmem;                   // NSB S/P buffers of kStep columns
            const uint32_t tO = tmem + NSB * C::kStep;  // O accumulator, D columns
            const uint64_t vdesc0 = sdesc_sw128(sbase + C::V_OFF, C::kKVChunk, 1024);
            int G = 0, e = 0, tcount = 0;
            bool ok = true;
            while (ok) {
                const int slot = tcount & 1;
                if (!warp_wait_all(bar(C::B_TFULL + slot), (tcount >> 1) & 1, ctl)) break;
                const int tile = tile_ids[slot];
                if (lane == 0) mbar_arrive(bar(C::B_TEMPTY + slot));
                ++tcount;
                if (tile < 0) break;
                if (tile & kEmptyTile) continue;
                bool first = true, last;
                do {
                    const int b = G % NSB, s = G % NV;
                    // V(G) normally landed long ago: test it first so that only the P wait
                    // sits between the softmax's arrival and the MMAs
                    if (!warp_wait_all(bar(C::B_VFULL + s), (G / NV) & 1, ctl)) { ok = false; break; }
                    // the descriptor was written by the QK^T issuer before S(G); P-full orders it after that write
                    if (!warp_wait_all(bar(C::B_PFULL + b), (G / NSB) & 1, ctl)) { ok = false; break; }
                    const uint32_t sd = desc[b];
                    const int cnt = desc_count(sd);
                    last = desc_last(sd);
                    // the first PV of a tile overwrites O: the previous tile's epilogue must have read it
                    if (first && e >= 1 && !warp_wait_all(bar(C::B_OEMPTY), (e - 1) & 1, ctl)) { ok = false; break; }
                    tc_fence_after();
                    // V slot s: descriptor of its first 16-row step; step kk adds kk * 2048 bytes
                    const uint64_t vdesc = vdesc0 + static_cast<uint64_t>(s * (C::kKVBytes >> 4));
                    const uint32_t pa = tS + b * C::kStep;
                    const int nk = cnt * (BS / 16);  // 16-row K steps of the blocks this step holds
                    __syncwarp();
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < C::kStep / 16; ++kk)
                            if (kk < nk)
                                mma_ts(tO, pa + kk * 8, vdesc + static_cast<uint64_t>(kk * (16 * 128 >> 4)),
                                       C::IDESC_PV, (first && kk == 0) ? 0u : 1u);
                        tc_commit(bar(C::B_PVDONE + b));
                        tc_commit(bar(C::B_VEMPTY + s));
                    }
                    __syncwarp();
                    first = false;
                    ++G;
                } while (!last);
                if (!ok) break;
                ++e;
            }
            // all MMAs issued by the elected lane have completed before TMEM is freed
            __syncwarp();
            if (elect_one()) {
                tc_commit(bar(C::B_DRAIN));
                wait_bar_drain(bar(C::B_DRAIN), 0, p.wait_limit_ns);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        if constexpr (SPLIT == 1)
            softmax_rows<D, BS, NSB, PAIR, C, TOK, LSE>(p, sbase, tmem, tile_ids, desc, ctl, warp, lane);
        else
            softmax_quads<D, BS, NSB, PAIR, C, TOK, LSE>(p, sbase, tmem, tile_ids, desc, ctl, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TCOLS);
    }
}

// ---------------------------------------------------------------- tile order

constexpr int kBuckets = 1024;

// Length of a tile for ordering and splitting: the sum of its Q blocks' row
// lengths (an upper bound of the union's step count at block size 64).
__device__ __forceinline__ int tile_length(const TcParams &p, int tile, int BS)
{
    const int64_t bh = tile / p.tiles_per_bh;
    const int qt = tile % p.tiles_per_bh;
    const int nrows = BS == 128 ? 1 : 2;
    int len = 0;
    for (int h = 0; h < nrows; ++h) {
        const int i = BS == 128 ? qt : 2 * qt + h;
        if (i >= p.nQB) break;
        const int64_t r = bh * p.nQB + i;
        if (p.index_mode == 0) {
            len += p.row_ptr[r + 1] - p.row_ptr[r];
        } else {
#pragma unroll 4
            for (int w = 0; w < p.W; ++w) len += __popc(__ldg(p.bitmap + r * p.W + w));
        }
    }
    return len;
}

// Exclusive prefix of v over the 1024 threads of the block, and the block total.
__device__ __forceinline__ int block_scan_excl(int v, int &total, int *wsum)
{
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s2 = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s2, o);
            if (lane >= o) s2 += y;
        }
        wsum[lane] = s2;
    }
    __syncthreads();
    total = wsum[31];
    const int excl = x - v + (warp > 0 ? wsum[warp - 1] : 0);
    __syncthreads();  // wsum is reused by the next call
    return excl;
}

// Chunks of a tile of `len` steps: a tile is split only when it is well above the
// per-CTA share (a chunk costs a Q load, a partial write and a merge).
__device__ __forceinline__ bool splits(int len, int share) { return len > share + share / 2; }

__device__ __forceinline__ int n_chunks(int len, int share, uint32_t dbg)
{
    if (dbg & kDbgSplitAll) return len >= 2 ? (len < kMaxChunks ? len : kMaxChunks) : 1;
    if (!splits(len, share)) return 1;
    const int n = (len + share - 1) / share;
    return n < kMaxChunks ? n : kMaxChunks;
}

// Counting-sort bucket of an item of `len` steps: items of at least long_min steps longest first,
// the rest after them in one bucket, so that (the sort being stable) they keep tile order and
// each head's tiles run together while its K and V stay in L2. long_min = share / 8: items that
// matter for the balance of the launch's last round go first.
__device__ __forceinline__ int length_bucket(int len, int long_min)
{
    if (len < long_min) return kBuckets - 1;
    return kBuckets - 2 - (len < kBuckets - 2 ? len : kBuckets - 2);
}
__device__ __forceinline__ int long_item_min(int share) { return share / 8 > 1 ? share / 8 : 1; }

// Reserves n consecutive slots of bucket bk (n = 0: none), returning the first.
// Lanes of a warp whose tile is whole (n == 1) and shares the bucket take their
// slots with one atomic (top-k masks give every tile the same length: per-lane
// atomics on one shared address would serialise). Called by all 32 lanes.
__device__ __forceinline__ int reserve_slots(int *hist, int bk, int n)
{
    const int lane = threadIdx.x & 31;
    const unsigned key = n == 1 ? static_cast<unsigned>(bk) : (n == 0 ? 0xfffffffeu : (0x80000000u | lane));
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    const int leader = __ffs(grp) - 1;
    int base = 0;
    if (lane == leader && n > 0) base = atomicAdd(&hist[bk], n == 1 ? __popc(grp) : n);
    base = __shfl_sync(0xffffffffu, base, leader);
    return base + (n == 1 ? __popc(grp & ((1u << lane) - 1u)) : 0);
}

// Stable placement of one 1024-tile chunk (one tile per thread, in tile order):
// a tile's n items go to bucket bk after every item of the same bucket from
// earlier chunks and from lower threads of this chunk, so items of equal length
// keep tile order. Persistent CTAs then take neighbouring tiles of one head
// together and its K and V stay in L2 (an order that interleaves heads re-reads
// them from DRAM). hist[bk] holds the bucket's next free position and is advanced.
// cnt is a [kBuckets][32] table of per-warp item counts in dynamic shared memory,
// zero on entry and on return (each entry is written and cleared by the one lane
// that leads its warp's group of the bucket). Called by all threads of the block; n = 0 places
// nothing.
constexpr size_t kOrderTableBytes = sizeof(uint16_t) * kBuckets * 32;

__device__ __forceinline__ int place_ordered(int *hist, int bk, int n, uint16_t *cnt)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int key = n > 0 ? bk : -1;
    // lanes with the same bucket (one group when the warp agrees: no match needed)
    const unsigned grp = __all_sync(0xffffffffu, key == __shfl_sync(0xffffffffu, key, 0))
                             ? 0xffffffffu
                             : __match_any_sync(0xffffffffu, key);
    const unsigned lower = (1u << lane) - 1u;
    // rank among earlier lanes of the same bucket, weighted by items, and the group total
    int rank, total;
    if (!__any_sync(0xffffffffu, n > 1)) {
        rank = __popc(grp & lower);
        total = __popc(grp);
    } else {  // a split tile in this warp: items per lane differ
        rank = total = 0;
#pragma unroll 8
        for (int l = 0; l < 32; ++l) {
            const int nl = __shfl_sync(0xffffffffu, n, l);
            if ((grp >> l) & 1u) {
                total += nl;
                if (l < lane) rank += nl;
            }
        }
    }
    const bool leader = key >= 0 && lane == __ffs(grp) - 1;
    if (leader) cnt[bk * 32 + warp] = static_cast<uint16_t>(total);
    __syncthreads();
    int pos = 0;
    if (key >= 0) {
        // items of this bucket from lower warps of the chunk: the row's first `warp` counts
        const uint4 *row = reinterpret_cast<const uint4 *>(cnt + bk * 32);
        int pref = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = row[q];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int w0 = 8 * q + 2 * h;  // warps of the two halves of this word
                if (w0 < warp) pref += static_cast<int>(w4[h] & 0xffffu);
                if (w0 + 1 < warp) pref += static_cast<int>(w4[h] >> 16);
            }
        }
        pos = hist[bk] + pref + rank;
    }
    __syncthreads();  // every thread has read hist and the table
    // each (warp, bucket) leader advances its bucket and clears its own entry, which
    // leaves the table zero for the next chunk
    if (leader) {
        atomicAdd(&hist[bk], total);
        cnt[bk * 32 + warp] = 0;
    }
    __syncthreads();
    return pos;
}

// zero the count table once per launch
__device__ __forceinline__ void clear_order_table(uint16_t *cnt)
{
    uint4 *p = reinterpret_cast<uint4 *>(cnt);
    for (int i = threadIdx.x; i < static_cast<int>(kOrderTableBytes / 16); i += blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

constexpr int kOrderPerThread = 8;  // 1024-tile chunks handled per batch (tiles per thread)

struct OrderArgs {
    int BS, grid, budget;
    int32_t *items, *lens, *split_base;
    uint32_t *merge_cnt;
    WsHeader *hdr;
    uint32_t plan_sig;      // signature of the configuration (stamped into the header)
};

// Work list for one forward launch, in one launch: every CTA computes the step
// counts of its 1024 tiles; the CTA that finishes last splits the tiles well above
// the per-CTA share (partial slots in tile order, within the budget; skipped when
// even the longest tile is not), then sorts the items (counting sort on item length,
// clamped: items of at least share / 8 steps longest first, the rest in tile order)
// and resets the scheduler counter.
__global__ void __launch_bounds__(1024) tile_order_kernel(TcParams p, OrderArgs o)
{
    grid_launch_dependents();  // the forward's prologue may start now (it waits for this grid's results)
    __shared__ int hist[kBuckets];
    extern __shared__ uint4 order_dyn[];
    uint16_t *ocnt = reinterpret_cast<uint16_t *>(order_dyn);
    __shared__ int wsum[32];
    __shared__ bool is_last;
    const int t = threadIdx.x;
    const int tile0 = blockIdx.x * 1024 + t;
    int len = 0;
    if (p.index_mode == 0) {
        if (tile0 < p.n_tiles) len = tile_length(p, tile0, o.BS);
    } else {
        // Bitmap lengths, coalesced: the index rows of consecutive tiles are consecutive,
        // so a warp reads the words of its 32 tiles as one contiguous run (lane-strided)
        // and adds each word's popcount to its tile's count in shared memory. (One tile
        // per thread would read words 4*W bytes apart: 32 sectors per load instruction.)
        int *tl = hist;  // the bucket histogram is not in use yet
        tl[t] = 0;
        __syncthreads();
        const int lane = t & 31;
        const int first = blockIdx.x * 1024 + (t & ~31);  // this warp's first tile
        const int last = min(first + 32, p.n_tiles);      // one past its last tile
        if (first < last) {
            const int per = o.BS == 128 ? 1 : 2;  // Q blocks per tile
            // rows of the warp's tiles, relative to the first tile's head: tile index
            // arithmetic stays in 32 bits (64-bit divisions are emulated and slow)
            const int bh0 = first / p.tiles_per_bh;
            const int qt0 = first - bh0 * p.tiles_per_bh;
            const int64_t row0 = static_cast<int64_t>(bh0) * p.nQB + qt0 * per;  // first row of `first`
            const int bhl = (last - 1) / p.tiles_per_bh;
            const int qtl = (last - 1) - bhl * p.tiles_per_bh;
            const int rows = static_cast<int>(static_cast<int64_t>(bhl) * p.nQB + min(qtl * per + per, p.nQB) - row0);
            const uint32_t *words = p.bitmap + row0 * p.W;
            const int n_words = rows * p.W;
            for (int e0 = lane; e0 < n_words; e0 += 32 * 8) {
                uint32_t v[8];  // eight loads in flight before any is used
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = e0 + 32 * u < n_words ? __ldg(words + e0 + 32 * u) : 0u;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = e0 + 32 * u;
                    if (e >= n_words) break;
                    const int lr = qt0 * per + e / p.W;  // row within head bh0 (may run into later heads)
                    const int dh = lr / p.nQB;
                    const int tile = first - qt0 + dh * p.tiles_per_bh + (lr - dh * p.nQB) / per;
                    atomicAdd(&tl[tile - blockIdx.x * 1024], __popc(v[u]));
                }
            }
        }
        __syncthreads();
        len = tile0 < p.n_tiles ? tl[t] : 0;
        __syncthreads();
    }
    if (tile0 < p.n_tiles) o.lens[tile0] = len;
    // block sum, max and min of the lengths, then one atomic each
    {
        const unsigned wsum_l = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(len));
        const unsigned wmax_l = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(len));
        const unsigned wmin_c = __reduce_max_sync(0xffffffffu, tile0 < p.n_tiles ? ~static_cast<unsigned>(len) : 0u);
        if ((t & 31) == 0) {
            wsum[t >> 5] = static_cast<int>(wsum_l);
            hist[t >> 5] = static_cast<int>(wmax_l);
            hist[32 + (t >> 5)] = static_cast<int>(wmin_c);
        }
        __syncthreads();
        if (t < 32) {
            const unsigned bs = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(wsum[t]));
            const unsigned bm = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(hist[t]));
            const unsigned bmc = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(hist[32 + t]));
            if (t == 0) {
                atomicAdd(&o.hdr->total_steps, static_cast<unsigned long long>(bs));
                atomicMax(&o.hdr->max_len, bm);
                atomicMax(&o.hdr->min_len_c, bmc);
            }
        }
    }
    __threadfence();
    __syncthreads();
    if (t == 0) is_last = atomicAdd(&o.hdr->order_done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // every CTA's atomics precede its count, so plain L2 loads see the final values
    const unsigned long long total = __ldcg(&o.hdr->total_steps);
    unsigned long long share = (total + o.grid - 1) / o.grid;
    if (share < kMinChunkSteps) share = kMinChunkSteps;
    if (share > 0x7fffffffull) share = 0x7fffffffull;
    const int T = static_cast<int>(share);
    const int max_len = static_cast<int>(__ldcg(&o.hdr->max_len));
    const int min_len = static_cast<int>(~__ldcg(&o.hdr->min_len_c));
    const bool can_split = p.split_ok && o.budget > 0 && !(p.dbg & kDbgNoSplit) &&
                           ((p.dbg & kDbgSplitAll) || splits(max_len, T));
    int n_items;
    if (!can_split && min_len == max_len) {
        // every tile has the same length (any top-k mask): the stable longest-first
        // order is tile order
        for (int i = t; i < p.n_tiles; i += 1024) o.items[i] = i;
        n_items = p.n_tiles;
    } else {
    // The passes below walk the tiles in batches of kOrderPerThread 1024-tile chunks
    // whose lengths (and split slots) are loaded together: one round trip per batch.
    constexpr int KB = kOrderPerThread;
    // split decisions: partial slots are handed out in tile order while the budget lasts
    int carry = 0;
    for (int s0 = 0; can_split && s0 < p.n_tiles; s0 += 1024 * KB) {
        int Lb[KB];
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const int tile = s0 + k * 1024 + t;
            Lb[k] = tile < p.n_tiles ? __ldcg(o.lens + tile) : 0;
        }
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            if (s0 + k * 1024 >= p.n_tiles) break;  // block-uniform
            const int tile = s0 + k * 1024 + t;
            const int n0 = tile < p.n_tiles ? n_chunks(Lb[k], T, p.dbg) : 1;
            const int want = n0 > 1 ? n0 : 0;
            int step_total;
            const int excl = carry + block_scan_excl(want, step_total, wsum);
            if (tile < p.n_tiles) {
                const bool fits = want > 0 && excl + want <= o.budget;
                o.split_base[tile] = fits ? excl : -1;
                if (fits)
                    for (int w = 0; w < kMergeWarps; ++w)
                        o.merge_cnt[static_cast<size_t>(excl) * kMergeWarps + w] = 0u;
            }
            carry += step_total;
        }
    }
    __syncthreads();
    // items and length bucket of the tiles of one batch
    auto batch = [&](int s0, int (&nb)[KB], int (&bkb)[KB]) {
        int Lb[KB], sb[KB];
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const int tile = s0 + k * 1024 + t;
            const bool valid = tile < p.n_tiles;
            Lb[k] = valid ? __ldcg(o.lens + tile) : 0;
            sb[k] = valid && can_split ? o.split_base[tile] : -1;
        }
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const bool valid = s0 + k * 1024 + t < p.n_tiles;
            nb[k] = !valid ? 0 : (sb[k] >= 0 ? n_chunks(Lb[k], T, p.dbg) : 1);
            bkb[k] = length_bucket(nb[k] > 0 ? (Lb[k] + nb[k] - 1) / nb[k] : 0, long_item_min(T));
        }
    };
    // histogram of item lengths, longest first
    for (int bk = t; bk < kBuckets; bk += 1024) hist[bk] = 0;
    __syncthreads();
    for (int s0 = 0; s0 < p.n_tiles; s0 += 1024 * KB) {
        int nb[KB], bkb[KB];
        batch(s0, nb, bkb);
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            if (s0 + k * 1024 + (t & ~31) >= p.n_tiles) continue;  // no tile in this warp (warp-uniform)
            (void)reserve_slots(hist, bkb[k], nb[k]);
        }
    }
    clear_order_table(ocnt);
    __syncthreads();
    const int excl = block_scan_excl(hist[t], n_items, wsum);
    hist[t] = excl;
    __syncthreads();
    for (int s0 = 0; s0 < p.n_tiles; s0 += 1024 * KB) {
        int nb[KB], bkb[KB];
        batch(s0, nb, bkb);
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            if (s0 + k * 1024 >= p.n_tiles) break;  // block-uniform
            const int tile = s0 + k * 1024 + t;
            const int n = nb[k];
            const int pos = place_ordered(hist, bkb[k], n, ocnt);
            for (int c = 0; c < n; ++c)
                o.items[pos + c] = tile | (c << kItemTileBits) | ((n - 1) << (kItemTileBits + 3));
        }
    }
    }  // lengths differ or tiles split
    if (t == 0) {
        o.hdr->n_items = static_cast<uint32_t>(n_items);
        o.hdr->chunk_steps = static_cast<uint32_t>(T);
        o.hdr->total_steps = 0ull;
        o.hdr->max_len = 0u;
        o.hdr->min_len_c = 0u;
        *p.tile_counter = 0u;
        o.hdr->run_items = static_cast<uint32_t>(n_items);
        o.hdr->plan_sig = o.plan_sig;
        o.hdr->order_done = 0u;
    }
}

// The same work list from one CTA for a CSR index whose tiles fit its registers
// (up to kOrderPerThread per thread): no length array, no election between CTAs.
// A tile's Q blocks are consecutive index rows, so its length is one difference
// of row_ptr; all the loads are issued before any is used. (Bitmap lengths are
// popcounts of rows strided across the threads: one SM would pull them too
// slowly, so bitmap indexes take the multi-CTA launch.)
__global__ void __launch_bounds__(1024) tile_order_small_kernel(TcParams p, OrderArgs o)
{
    grid_launch_dependents();  // the forward's prologue may start now (it waits for this grid's results)
    __shared__ int hist[kBuckets];
    extern __shared__ uint4 order_dyn[];
    uint16_t *ocnt = reinterpret_cast<uint16_t *>(order_dyn);
    __shared__ int wsum[32];
    __shared__ unsigned red[96];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int L[kOrderPerThread];
    // first index row of each of this thread's tiles and how many rows it holds
    int64_t r0[kOrderPerThread];
    int nr[kOrderPerThread];
#pragma unroll
    for (int k = 0; k < kOrderPerThread; ++k) {
        const int tile = k * 1024 + t;
        r0[k] = 0;
        nr[k] = 0;
        if (tile < p.n_tiles) {
            const int64_t bh = tile / p.tiles_per_bh;
            const int qt = tile % p.tiles_per_bh;
            const int i0 = o.BS == 128 ? qt : 2 * qt;
            r0[k] = bh * p.nQB + i0;
            nr[k] = o.BS == 128 || i0 + 1 >= p.nQB ? 1 : 2;
        }
    }
    {
        // a tile's Q blocks are consecutive index rows: its length is one row_ptr difference
        int lo[kOrderPerThread], hi[kOrderPerThread];
#pragma unroll
        for (int k = 0; k < kOrderPerThread; ++k) {
            lo[k] = nr[k] ? __ldg(p.row_ptr + r0[k]) : 0;
            hi[k] = nr[k] ? __ldg(p.row_ptr + r0[k] + nr[k]) : 0;
        }
#pragma unroll
        for (int k = 0; k < kOrderPerThread; ++k) L[k] = hi[k] - lo[k];
    }
    unsigned sum = 0u, mx = 0u, mnc = 0u;  // mnc: ~(shortest length)
#pragma unroll
    for (int k = 0; k < kOrderPerThread; ++k) {
        sum += static_cast<unsigned>(L[k]);
        mx = max(mx, static_cast<unsigned>(L[k]));
        if (nr[k]) mnc = max(mnc, ~static_cast<unsigned>(L[k]));
    }
    sum = __reduce_add_sync(0xffffffffu, sum);
    mx = __reduce_max_sync(0xffffffffu, mx);
    mnc = __reduce_max_sync(0xffffffffu, mnc);
    if (lane == 0) {
        red[warp] = sum;
        red[32 + warp] = mx;
        red[64 + warp] = mnc;
    }
    for (int b = t; b < kBuckets; b += 1024) hist[b] = 0;
    __syncthreads();
    const unsigned total = __reduce_add_sync(0xffffffffu, red[lane]);
    const unsigned max_len = __reduce_max_sync(0xffffffffu, red[32 + lane]);
    const unsigned min_len = ~__reduce_max_sync(0xffffffffu, red[64 + lane]);
    unsigned share = (total + o.grid - 1) / o.grid;
    if (share < kMinChunkSteps) share = kMinChunkSteps;
    const int T = static_cast<int>(share < 0x7fffffffu ? share : 0x7fffffffu);
    const bool can_split = p.split_ok && o.budget > 0 && !(p.dbg & kDbgNoSplit) &&
                           ((p.dbg & kDbgSplitAll) || splits(static_cast<int>(max_len), T));
    int n_items;
    if (!can_split && min_len == max_len) {
        // every tile has the same length (any top-k mask): the stable longest-first
        // order is tile order
        for (int i = t; i < p.n_tiles; i += 1024) o.items[i] = i;
        n_items = p.n_tiles;
    } else {
    int n[kOrderPerThread];
#pragma unroll
    for (int k = 0; k < kOrderPerThread; ++k) n[k] = 1;
    if (can_split) {
        int carry = 0;
#pragma unroll
        for (int k = 0; k < kOrderPerThread; ++k) {
            const int tile = k * 1024 + t;
            const int n0 = tile < p.n_tiles ? n_chunks(L[k], T, p.dbg) : 1;
            const int want = n0 > 1 ? n0 : 0;
            int step_total;
            const int excl = carry + block_scan_excl(want, step_total, wsum);
            if (tile < p.n_tiles) {
                const bool fits = want > 0 && excl + want <= o.budget;
                o.split_base[tile] = fits ? excl : -1;
                if (fits) {
                    n[k] = n0;
                    for (int w = 0; w < kMergeWarps; ++w) o.merge_cnt[static_cast<size_t>(excl) * kMergeWarps + w] = 0u;
                }
            }
            carry += step_total;
        }
    }
#pragma unroll
    for (int k = 0; k < kOrderPerThread; ++k) {
        if (k * 1024 + (t & ~31) >= p.n_tiles) continue;  // no tile in this warp (warp-uniform)
        const bool valid = k * 1024 + t < p.n_tiles;
        (void)reserve_slots(hist, length_bucket((L[k] + n[k] - 1) / n[k], long_item_min(T)), valid ? n[k] : 0);
    }
    clear_order_table(ocnt);
    __syncthreads();
    const int excl = block_scan_excl(hist[t], n_items, wsum);
    hist[t] = excl;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kOrderPerThread; ++k) {
        if (k * 1024 >= p.n_tiles) break;  // no tile in this chunk (block-uniform)
        const int tile = k * 1024 + t;
        const bool valid = tile < p.n_tiles;
        const int pos =
            place_ordered(hist, length_bucket((L[k] + n[k] - 1) / n[k], long_item_min(T)), valid ? n[k] : 0, ocnt);
        if (valid)
            for (int c = 0; c < n[k]; ++c)
                o.items[pos + c] = tile | (c << kItemTileBits) | ((n[k] - 1) << (kItemTileBits + 3));
    }
    }  // lengths differ or tiles split
    if (t == 0) {
        o.hdr->n_items = static_cast<uint32_t>(n_items);
        o.hdr->chunk_steps = static_cast<uint32_t>(T);
        *p.tile_counter = 0u;
        o.hdr->run_items = static_cast<uint32_t>(n_items);
        o.hdr->plan_sig = o.plan_sig;
    }
}

// Before a forward on a work list made by an earlier launch: the list runs only if it was
// made for this configuration (else BSA_ERR_INVALID_ARG and nothing runs), and the
// scheduler and merge counters start from zero again.
__global__ void __launch_bounds__(256) plan_gate_kernel(WsHeader *hdr, uint32_t sig, uint32_t *merge_cnt, int n_merge)
{
    grid_launch_dependents();  // the forward's prologue may start now (it waits for this grid's results)
    for (int i = threadIdx.x; i < n_merge; i += blockDim.x) merge_cnt[i] = 0u;
    if (threadIdx.x == 0) {
        const bool ok = hdr->plan_sig == sig;
        hdr->run_items = ok ? hdr->n_items : 0u;
        hdr->tile_counter = 0u;
        if (!ok) raise_error(&hdr->err, BSA_ERR_INVALID_ARG);
    }
}

// ---------------------------------------------------------------- host side

// Forward workspace: header, item list, per-tile lengths and partial slots, merge
// counters, then the partial results of split tiles (all 256-byte aligned).
struct FwdLayout {
    size_t tiles, budget, items, lens, split_base, merge_cnt, part_stats, part_o, bytes;
};

FwdLayout fwd_layout(int B, int H, int N, int d)
{
    FwdLayout l{};
    l.tiles = static_cast<size_t>(B) * H * ((N + kTileM - 1) / kTileM);
    // split tiles need item ids with chunk fields; partial slots: at most 8 per tile
    l.budget = l.tiles < (size_t(1) << kItemTileBits)
                   ? (l.tiles * kMaxChunks < size_t(kMaxPartials) ? l.tiles * kMaxChunks : size_t(kMaxPartials))
                   : 0;
    size_t off = kWsHeader;
    l.items = off;
    off += align_up((l.tiles + l.budget) * sizeof(int32_t), 256);
    l.lens = off;
    off += align_up(l.tiles * sizeof(int32_t), 256);
    l.split_base = off;
    off += align_up(l.tiles * sizeof(int32_t), 256);
    l.merge_cnt = off;
    off += align_up(l.budget * kMergeWarps * sizeof(uint32_t), 256);
    l.part_stats = off;
    off += align_up(l.budget * kTileM * sizeof(float4), 256);
    l.part_o = off;
    off += align_up(l.budget * kTileM * static_cast<size_t>(d) * sizeof(float), 256);
    l.bytes = off;
    return l;
}

// Resident CTAs of a forward instance over the whole GPU (set-up once per instance:
// shared-memory attributes, then registers, shared memory and TMEM per SM).
template <int D, int BS, int NK, int NV, int NSB, int QS, int SPLIT, int PAIR, int MINB, bool TOK, bool LSE = false>
bsa_status forward_grid_cap(int &cap)
{
    using C = Cfg<D, BS, NK, NV, NSB, QS, PAIR>;
    constexpr int kThreads = Roles<SPLIT>::kThreads;
    static_assert(MINB * (C::SMEM_ALLOC + 1024) <= 233472, "shared memory for MINB CTAs per SM");
    static_assert(C::SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(C::TCOLS_USED <= C::TCOLS, "TMEM budget");
    auto kern = fwd_tc_kernel<D, BS, NK, NV, NSB, QS, SPLIT, PAIR, MINB, TOK, LSE>;
    static int grid_cap = 0;
    if (grid_cap == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) != cudaSuccess)
            return BSA_ERR_CUDA;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return BSA_ERR_CUDA;
        int dev = 0, sms = 0, smem_sm = 0, occ = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BSA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
            return BSA_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, C::SMEM_ALLOC) != cudaSuccess)
            return BSA_ERR_CUDA;
        // resident CTAs per SM: registers are sized for MINB by the launch bounds,
        // shared memory (+1 KB reserved per CTA) and TMEM columns bound the rest
        const int by_smem = smem_sm / (C::SMEM_ALLOC + 1024);
        const int by_tmem = 512 / C::TCOLS;
        int per_sm = MINB < by_smem ? MINB : by_smem;
        if (occ > per_sm) per_sm = occ;
        if (per_sm > by_tmem) per_sm = by_tmem;
        if (per_sm < 1) return BSA_ERR_UNSUPPORTED;
        grid_cap = sms * per_sm;
    }
    cap = grid_cap;
    return BSA_OK;
}

// Signature of the configuration a work list is made for: the launch shape and every input
// of the ordering except the index contents (never 0, so a zeroed header matches nothing).
uint32_t plan_signature(int n_tiles, int grid, int index_mode, int D, int BS, int budget, uint32_t dbg, int N, int BH)
{
    uint32_t h = 0x811C9DC5u;
    const uint32_t v[8] = {static_cast<uint32_t>(n_tiles), static_cast<uint32_t>(grid),
                           static_cast<uint32_t>(index_mode), static_cast<uint32_t>(D | (BS << 8)),
                           static_cast<uint32_t>(budget), dbg & (kDbgNoSplit | kDbgSplitAll),
                           static_cast<uint32_t>(N), static_cast<uint32_t>(BH)};
    for (uint32_t x : v)
        for (int b = 0; b < 4; ++b) h = (h ^ ((x >> (8 * b)) & 0xFFu)) * 0x01000193u;
    return h | 1u;
}

// mode: kRunOrderAndForward, kRunForward (a plan is in the workspace), kRunOrder (make the plan)
enum { kRunOrderAndForward = 0, kRunForward = 1, kRunOrder = 2 };

// LSE: the LSE-only kernel (no V, no O; tiles never split)
template <int D, int BS, int NK, int NV, int NSB, int QS, int SPLIT, int PAIR, int MINB, bool LSE = false>
bsa_status launch_tc(const FwdArgs &a, cudaStream_t st, int mode)
{
    using C = Cfg<D, BS, NK, NV, NSB, QS, PAIR>;
    constexpr int kThreads = Roles<SPLIT>::kThreads;
    auto kern = fwd_tc_kernel<D, BS, NK, NV, NSB, QS, SPLIT, PAIR, MINB, false, LSE>;
    int grid_cap = 0;
    {
        const bsa_status s = forward_grid_cap<D, BS, NK, NV, NSB, QS, SPLIT, PAIR, MINB, false, LSE>(grid_cap);
        if (s != BSA_OK) return s;
    }
    const int64_t BH = static_cast<int64_t>(a.B) * a.H;
    CUtensorMap mq, mk, mv;
    if (!make_tma_map_bf16(&mq, a.Q, BH, a.N, D, kTileM) || !make_tma_map_bf16(&mk, a.K, BH, a.N, D, BS) ||
        !make_tma_map_bf16(&mv, LSE ? a.K : a.V, BH, a.N, D, BS))  // the LSE-only kernel reads no V
        return BSA_ERR_CUDA;
    WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
    TcParams p{};
    p.N = a.N;
    p.nQB = a.nQB;
    p.nKB = a.nKB;
    p.last_rows = a.N - (a.nKB - 1) * BS;
    p.ragged_kb = p.last_rows < BS ? a.nKB - 1 : -1;
    p.W = a.W;
    p.tiles_per_bh = (a.N + kTileM - 1) / kTileM;
    p.n_tiles = static_cast<int>(BH * p.tiles_per_bh);
    p.row_ptr = a.row_ptr;
    p.col_idx = a.col_idx;
    p.bitmap = a.bitmap;
    p.index_mode = a.index_mode;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.O = static_cast<__nv_bfloat16 *>(a.O);
    p.LSE = a.LSE;
    const FwdLayout lay = fwd_layout(a.B, a.H, a.N, a.d);
    OrderArgs o{};
    o.BS = BS;
    o.budget = static_cast<int>(lay.budget);
    o.items = reinterpret_cast<int32_t *>(a.ws + lay.items);
    o.lens = reinterpret_cast<int32_t *>(a.ws + lay.lens);
    o.split_base = reinterpret_cast<int32_t *>(a.ws + lay.split_base);
    o.merge_cnt = reinterpret_cast<uint32_t *>(a.ws + lay.merge_cnt);
    o.hdr = hdr;
    p.tile_list = o.items;
    p.n_items = &hdr->run_items;  // the items this launch runs (the order kernel or the plan gate sets it)
    p.split_ok = lay.budget > 0 ? 1 : 0;
    p.split_base = o.split_base;
    p.merge_cnt = o.merge_cnt;
    p.part_stats = reinterpret_cast<float4 *>(a.ws + lay.part_stats);
    p.part_o = reinterpret_cast<float *>(a.ws + lay.part_o);
    p.R = a.R;
    p.tile_counter = &hdr->tile_counter;
    p.err = &hdr->err;
    p.wait_limit_ns = a.wait_limit_ns;
    p.dbg = a.dbg_flags;
    if (LSE) p.dbg = (p.dbg & ~kDbgSplitAll) | kDbgNoSplit;  // a chunk's partial O has nowhere to go
    // persistent CTAs; with splitting on, the item count is only known on the device
    const int64_t max_items = static_cast<int64_t>(p.n_tiles) + static_cast<int64_t>(lay.budget);
    const int grid = static_cast<int>(max_items < grid_cap ? max_items : grid_cap);
    o.grid = grid;
    o.plan_sig = plan_signature(p.n_tiles, grid, p.index_mode, D, BS, static_cast<int>(lay.budget), p.dbg, a.N,
                                static_cast<int>(BH));
    static bool order_smem_set = false;
    if (!order_smem_set) {
        if (cudaFuncSetAttribute(tile_order_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kOrderTableBytes)) != cudaSuccess ||
            cudaFuncSetAttribute(tile_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kOrderTableBytes)) != cudaSuccess)
            return BSA_ERR_CUDA;
        order_smem_set = true;
    }
    if (mode != kRunForward) {
        if (p.index_mode == 0 && p.n_tiles <= 1024 * kOrderPerThread)
            tile_order_small_kernel<<<1, 1024, kOrderTableBytes, st>>>(p, o);
        else
            tile_order_kernel<<<(p.n_tiles + 1023) / 1024, 1024, kOrderTableBytes, st>>>(p, o);
    } else {
        plan_gate_kernel<<<1, 256, 0, st>>>(hdr, o.plan_sig, o.merge_cnt,
                                            static_cast<int>(lay.budget) * kMergeWarps);
    }
    if (mode == kRunOrder) return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
    // programmatic dependent launch: the forward's CTAs set up barriers and TMEM while the
    // work-list launch runs, and wait for its results in-kernel
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, p) != cudaSuccess) return BSA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

// Token-sparse forward ("Can sparse attention close the quality gap in diffusion
// transformers", section "token 级选择需要瓦片对齐的查询分组"): the block-128 kernel in
// token mode. A tile is one query group of 128 rows gathered through the permutation;
// its steps are 128-key chunks of the group's token list, gathered by index (the last
// chunk's missing keys are masked); outputs go back to the rows the permutation names.
template <int D, int NK, int NV, int NSB, int QS, int SPLIT, int MINB>
bsa_status launch_tc_tokens(const TokenArgs &a, cudaStream_t st)
{
    using C = Cfg<D, kTileM, NK, NV, NSB, QS, 1>;
    constexpr int kThreads = Roles<SPLIT>::kThreads;
    auto kern = fwd_tc_kernel<D, kTileM, NK, NV, NSB, QS, SPLIT, 1, MINB, true>;
    int grid_cap = 0;
    {
        const bsa_status s = forward_grid_cap<D, kTileM, NK, NV, NSB, QS, SPLIT, 1, MINB, true>(grid_cap);
        if (s != BSA_OK) return s;
    }
    const int64_t BH = static_cast<int64_t>(a.B) * a.H;
    const uint64_t rows = static_cast<uint64_t>(BH) * a.N;
    CUtensorMap mq, mk, mv;
    if (!make_tma_map_bf16_rows(&mq, a.Q, rows, D) || !make_tma_map_bf16_rows(&mk, a.K, rows, D) ||
        !make_tma_map_bf16_rows(&mv, a.V, rows, D))
        return BSA_ERR_CUDA;
    TcParams p{};
    p.N = a.N;
    p.groups = a.N / kTileM;
    p.n_tiles = static_cast<int>(BH * p.groups);
    p.n_tok = a.n_tokens;
    p.last_rows = a.n_tokens - (a.n_tokens - 1) / kTileM * kTileM;  // keys in the last 128-key step
    p.ragged_kb = -1;
    p.perm = a.perm;
    p.tokens = a.tokens;
    p.Kg = static_cast<const __nv_bfloat16 *>(a.K);
    p.Vg = static_cast<const __nv_bfloat16 *>(a.V);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.O = static_cast<__nv_bfloat16 *>(a.O);
    p.LSE = a.LSE;
    p.split_ok = 0;
    p.err = &reinterpret_cast<WsHeader *>(a.ws)->err;
    p.wait_limit_ns = a.wait_limit_ns;
    const int grid = p.n_tiles < grid_cap ? p.n_tiles : grid_cap;
    kern<<<grid, kThreads, C::SMEM_ALLOC, st>>>(mq, mk, mv, p);
    return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

}  // namespace

bsa_status launch_forward_tokens_tc(const TokenArgs &a, cudaStream_t st)
{
    // the block-128 instances' stages and layouts: <D, K stages, V stages, S/P buffers, Q slots, threads per row, CTAs per SM>
    if (a.d == 64) return launch_tc_tokens<64, 5, 6, 3, 2, 2, 1>(a, st);
    if (a.d == 128) return launch_tc_tokens<128, 3, 3, 3, 1, 2, 1>(a, st);  // 3 + 3 stages: measured best
    return BSA_ERR_SHAPE;
}

size_t fwd_workspace_bytes(int B, int H, int N, int d, int block)
{
    (void)block;
    return fwd_layout(B, H, N, d).bytes;
}

static bsa_status launch_forward_mode(const FwdArgs &a, cudaStream_t st, int mode)
{
    // <D, BS, K stages, V stages, S/P buffers, Q slots, threads per row, blocks per step, CTAs per SM>
    if (a.d == 64 && a.block == 64) return launch_tc<64, 64, 4, 5, 3, 2, 1, 1, 2>(a, st, mode);
    if (a.d == 128 && a.block == 64) return launch_tc<128, 64, 2, 2, 2, 1, 1, 1, 2>(a, st, mode);
    if (a.d == 64 && a.block == 128) return launch_tc<64, 128, 5, 6, 3, 2, 2, 1, 1>(a, st, mode);
    if (a.d == 128 && a.block == 128) return launch_tc<128, 128, 2, 4, 3, 1, 2, 1, 1>(a, st, mode);
    return BSA_ERR_SHAPE;
}

bsa_status launch_forward_tc(const FwdArgs &a, cudaStream_t st)
{
    return launch_forward_mode(a, st, a.planned ? kRunForward : kRunOrderAndForward);
}

bsa_status launch_forward_plan_tc(const FwdArgs &a, cudaStream_t st)
{
    return launch_forward_mode(a, st, kRunOrder);
}

bsa_status launch_forward_lse_tc(const FwdArgs &a, cudaStream_t st)
{
    // the forward's instances, LSE only
    if (a.d == 64 && a.block == 64) return launch_tc<64, 64, 4, 5, 3, 2, 1, 1, 2, true>(a, st, kRunOrderAndForward);
    if (a.d == 128 && a.block == 64) return launch_tc<128, 64, 2, 2, 2, 1, 1, 1, 2, true>(a, st, kRunOrderAndForward);
    if (a.d == 64 && a.block == 128) return launch_tc<64, 128, 5, 6, 3, 2, 2, 1, 1, true>(a, st, kRunOrderAndForward);
    if (a.d == 128 && a.block == 128) return launch_tc<128, 128, 2, 4, 3, 1, 2, 1, 1, true>(a, st, kRunOrderAndForward);
    return BSA_ERR_SHAPE;
}

// ---------------------------------------------------------------- TMA descriptors

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 2-D view [rows][d] of a bf16 tensor with 64-column x 1-row boxes and 128-byte swizzle:
// the map of tile::gather4 loads (four rows by index per copy).
bool make_tma_map_bf16_rows(CUtensorMap *m, const void *base, uint64_t rows, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[2] = {64u, 1u};
    const cuuint32_t es[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view [heads][n][d] of a bf16 tensor, 64-column x box_rows boxes, 128-byte swizzle.
bool make_tma_map_bf16(CUtensorMap *m, const void *base, uint64_t heads, uint64_t n, int d, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    // {column, row, head}: a box never crosses into the next head; rows >= n read as zeros
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(heads)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 2 * n};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
    const cuuint32_t es[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace bsa
