// walk.cuh -- ascending walk over the active KV blocks of a query tile.
//
// "多模态DiT中的块稀疏注意力" §4.1 keeps active_kv_blocks[i] per Q block in device
// memory either as CSR or as a bitmap tested with popcount; the kernels read one
// of the two. A 128-row query tile covers one Q block at block size 128 and two
// consecutive Q blocks (2t, 2t+1) at block size 64; the walk then visits the
// ascending union of both lists and reports, per KV block, which of the tile's
// Q blocks has it active (bit 0: first, bit 1: second).
#pragma once

#include <cstdint>

namespace bsa {

struct TileWalk {
    // CSR cursors
    const int32_t *c0, *e0, *c1, *e1;
    // bitmap state
    const uint32_t *w0, *w1;
    int W, w;
    uint32_t b0, b1, pend;
    int mode;   // 0: CSR, 1: bitmap
    uint32_t full;  // mask reported for every block when the tile is one Q block (block 128)

    // rows: index rows of the tile's Q blocks (r1 < 0 when there is no second block)
    __device__ __forceinline__ void init(int index_mode, const int32_t *row_ptr, const int32_t *col_idx,
                                         const uint32_t *bitmap, int nW, int64_t r0, int64_t r1,
                                         uint32_t single_mask)
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
        } else {
            W = nW;
            w = -1;
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
            if (++w >= W) return false;
            b0 = w0[w];
            b1 = w1 ? w1[w] : 0u;
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
