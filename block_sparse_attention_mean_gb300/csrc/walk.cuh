// walk.cuh -- ascending walk over the active KV blocks of a query tile.
//
// "多模态DiT中的块稀疏注意力" §4.1 keeps active_kv_blocks[i] per Q block in device
// memory either as CSR or as a bitmap tested with popcount; the kernels read one
// of the two. A 128-row query tile covers one Q block at block size 128 and two
// consecutive Q blocks (2t, 2t+1) at block size 64; the walk then visits the
// ascending union of both lists and reports, per KV block, which of the tile's
// Q blocks has it active (bit 0: first, bit 1: second). A walk can be limited to
// the KV blocks [j_lo, j_hi) (one chunk of a query tile whose list is split over
// several CTAs): CSR rows are cut by binary search, bitmap words are masked.
#pragma once

#include <cstdint>

namespace bsa {

// First element >= v of the ascending range [b, e).
__device__ __forceinline__ const int32_t *lower_bound_i32(const int32_t *b, const int32_t *e, int v)
{
    while (b < e) {
        const int32_t *m = b + (e - b) / 2;
        if (*m < v) b = m + 1;
        else e = m;
    }
    return b;
}

struct TileWalk {
    // CSR cursors
    const int32_t *c0, *e0, *c1, *e1;
    // bitmap state: words [w_lo, w_end) are visited, the first and last masked
    const uint32_t *w0, *w1;
    int W, w, w_lo, w_end;
    uint32_t m_lo, m_hi;
    uint32_t b0, b1, pend;
    int mode;   // 0: CSR, 1: bitmap
    uint32_t full;  // mask reported for every block when the tile is one Q block (block 128)

    // rows: index rows of the tile's Q blocks (r1 < 0 when there is no second block);
    // [j_lo, j_hi): the KV blocks to visit (0, nKB for the whole row)
    __device__ __forceinline__ void init(int index_mode, const int32_t *row_ptr, const int32_t *col_idx,
                                         const uint32_t *bitmap, int nW, int64_t r0, int64_t r1,
                                         uint32_t single_mask, int j_lo = 0, int j_hi = 0x7fffffff)
    {
        mode = index_mode;
        full = single_mask;
        if (mode == 0) {
            c0 = col_idx + row_ptr[r0];
            e0 = col_idx + row_ptr[r0 + 1];
            if (r1 >= 0) {
                c1 = col_idx + row_ptr[r1];
                e1 = col_idx + row_ptr[r1 + 1];
            } else {
                c1 = e1 = nullptr;
            }
            if (j_lo > 0) {
                c0 = lower_bound_i32(c0, e0, j_lo);
                if (c1) c1 = lower_bound_i32(c1, e1, j_lo);
            }
            if (j_hi < 0x7fffffff) {
                e0 = lower_bound_i32(c0, e0, j_hi);
                if (c1) e1 = lower_bound_i32(c1, e1, j_hi);
            }
        } else {
            W = nW;
            w_lo = j_lo >> 5;
            const int we = j_hi == 0x7fffffff ? nW : (j_hi + 31) >> 5;
            w_end = we < nW ? we : nW;
            w = w_lo - 1;
            m_lo = ~0u << (j_lo & 31);
            m_hi = (j_hi == 0x7fffffff || (j_hi & 31) == 0) ? ~0u : ((1u << (j_hi & 31)) - 1u);
            w0 = bitmap + r0 * nW;
            w1 = r1 >= 0 ? bitmap + r1 * nW : nullptr;
            b0 = b1 = pend = 0u;
        }
    }

    __device__ __forceinline__ bool next(int &j, uint32_t &m)
    {
        if (mode == 0) {
            const bool h0 = c0 < e0, h1 = c1 < e1;
            if (h0 && h1) {
                const int j0 = *c0, j1 = *c1;
                if (j0 < j1) { j = j0; m = 1u; ++c0; }
                else if (j1 < j0) { j = j1; m = 2u; ++c1; }
                else { j = j0; m = 3u; ++c0; ++c1; }
            } else if (h0) {
                j = *c0++;
                m = 1u;
            } else if (h1) {
                j = *c1++;
                m = 2u;
            } else {
                return false;
            }
            if (full) m = full;
            return true;
        }
        while (pend == 0u) {
            if (++w >= w_end) return false;
            const uint32_t msk = (w == w_lo ? m_lo : ~0u) & (w == w_end - 1 ? m_hi : ~0u);
            b0 = w0[w] & msk;
            b1 = w1 ? (w1[w] & msk) : 0u;
            pend = b0 | b1;
        }
        const int bit = __ffs(pend) - 1;
        pend &= pend - 1u;
        j = w * 32 + bit;
        m = full ? full : (((b0 >> bit) & 1u) | (((b1 >> bit) & 1u) << 1));
        return true;
    }

    // Up to P consecutive items of the walk (one KV step); returns how many (0 = done).
    template <int P>
    __device__ __forceinline__ int next_step(int (&js)[2], uint32_t (&ms)[2])
    {
        if (!next(js[0], ms[0])) return 0;
        if (P == 2 && next(js[1], ms[1])) return 2;
        ms[1] = 0u;
        return 1;
    }
};

}  // namespace bsa
