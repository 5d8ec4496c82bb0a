// internal.h -- declarations shared by the host API (api.cu) and the kernel
// translation units. Not part of the public C ABI.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include <cuda.h>

#include "../../include/bsa.h"

namespace bsa {

// Launch with programmatic stream serialisation: the grid may be scheduled while the
// previous kernel on the stream drains; it waits for that kernel's results with
// griddepcontrol.wait before reading them.
template <typename... KArgs, typename... Args>
inline bool pdl_launch(void (*kern)(KArgs...), dim3 grid, int threads, size_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess;
}

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
    uint32_t err;          // first device-raised bsa_status (0 = none)
    uint32_t tile_counter; // forward: dynamic tile scheduler counter
    uint32_t order_done;   // CTAs of a last-CTA-finishes launch that are done (tile order, static pattern)
    uint32_t n_items;      // forward: work items (query tiles or chunks of them) in the item list
    unsigned long long total_steps;  // forward: sum of the tiles' KV steps (tile order, then cleared)
    uint32_t chunk_steps;  // forward: the per-CTA share of steps (chunk length of split tiles)
    uint32_t max_len;      // forward: longest tile (tile order, then cleared)
    uint32_t min_len_c;    // forward: ~(shortest tile) (tile order, then cleared)
    uint32_t plan_sig;     // forward: signature of the configuration the work list was made for
    uint32_t run_items;    // forward: items the next forward launch runs (n_items, or 0 for a bad plan)
    uint32_t pad[53];
};
static_assert(sizeof(WsHeader) == 256, "workspace header size");
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kWsHeader = 256;
constexpr int kMaxKvBlocks = 2048;     // nKB limit of the selector (16 score rows in smem)
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // bounded device waits: 2 s

// Records `code` as the workspace's device error unless one is already set.
__device__ __forceinline__ void raise_error(uint32_t *err, uint32_t code)
{
    atomicCAS(err, 0u, code);
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------ mask builder
struct MaskArgs {
    const void *Q, *K;
    int dt, B, H, N, d, block;
    int nQB, nKB, W;       // blocks per row/column, bitmap words per row
    int k;                 // dynamic: blocks kept per row (plain selector)
    int n_text;            // dynamic: leading text blocks (0 for the plain selector)
    int kq[2][2];          // dynamic: blocks kept by a query block of modality a among key modality b
    const bsa_static_spec *spec;  // host copy (NULL -> dynamic)
    int32_t *row_ptr, *col_idx;
    int64_t col_capacity;
    uint32_t *bitmap;
    char *ws;              // workspace base (device)
    int sm_count;          // streaming multiprocessors of the current device
};

size_t mask_workspace_bytes(int B, int H, int N, int d, int block);
// bytes of the workspace that one build reads or writes: the dynamic (pooled
// blocks) or the static (counts, one head's pattern) part of the layout
size_t mask_workspace_need(int B, int H, int N, int d, int block, bool dynamic);
// Every host-side check of bsa_build_mask except the workspace's: fills `a`
// (all but `ws`) and touches no device state, so a failing call enqueues nothing.
bsa_status prepare_build_mask(const void *Q, const void *K, int dt, int B, int H, int N, int d, int block,
                              float density, const bsa_static_spec *spec, int32_t *row_ptr, int32_t *col_idx,
                              int64_t col_capacity, uint32_t *bitmap, MaskArgs *a);
// streaming multiprocessors of the current device (a host query; enqueues nothing)
bsa_status current_sm_count(int *sm_count);
bsa_status launch_build_mask(const MaskArgs &a, cudaStream_t st);
bsa_status launch_validate_index(int R, int nKB, const int32_t *row_ptr, const int32_t *col_idx,
                                 const uint32_t *bitmap, char *ws, cudaStream_t st);

// ------------------------------------------------------------ exact block-mass selector
struct ExactArgs {
    const void *Q, *K;
    int B, H, N, d, block;
    int nQB, nKB, W;
    int k;                 // blocks kept per Q block
    float scale;           // > 0
    const float *LSE;      // dense logsumexp per query row (natural log)
    int32_t *row_ptr, *col_idx;
    uint32_t *bitmap;
    char *ws;
    uint64_t wait_limit_ns;
};

size_t exact_workspace_bytes(int B, int H, int N, int d, int block);
bsa_status launch_build_mask_exact(const ExactArgs &a, cudaStream_t st);
// top-k of the block masses whose partials (4 per 128-row tile, warp order) are at `part`
bsa_status launch_mass_select(const float *part, const ExactArgs &a, int tiles_per_bh, cudaStream_t st);

// ------------------------------------------------------------ forward
struct FwdArgs {
    const void *Q, *K, *V;
    int dt, B, H, N, d, block;
    int nQB, nKB, W;
    const int32_t *row_ptr, *col_idx;
    const uint32_t *bitmap;
    int index_mode;
    float scale;           // > 0
    void *O;
    float *LSE;
    const float *R;        // residual added to O before rounding (nullptr: none)
    char *ws;
    uint32_t dbg_flags;
    uint64_t wait_limit_ns;
    int planned;           // the work list is already in the workspace (bsa_forward_plan)
};

size_t fwd_workspace_bytes(int B, int H, int N, int d, int block);
// 3-D TMA view [heads][n][d] of a bf16 tensor with 64-column x box_rows boxes and 128-byte swizzle;
// rows at or past n (a ragged last block) read as zeros
bool make_tma_map_bf16(CUtensorMap *m, const void *base, uint64_t heads, uint64_t n, int d, int box_rows);
bsa_status launch_forward_tc(const FwdArgs &a, cudaStream_t st);    // bf16, tcgen05
bsa_status launch_forward_plan_tc(const FwdArgs &a, cudaStream_t st);  // bf16: the work list only
bsa_status launch_forward_lse_tc(const FwdArgs &a, cudaStream_t st);   // bf16: LSE only (no V, no O)
bsa_status launch_forward_simt(const FwdArgs &a, cudaStream_t st);  // fp32, CUDA cores
bsa_status launch_residual_capture(const void *dense, const void *sparse, int dt, int64_t count, float *R,
                                   cudaStream_t st);

// ------------------------------------------------------------ token-sparse forward
constexpr int kTokenGroup = 128;  // queries per group (the query tile)

struct TokenArgs {
    const void *Q, *K, *V;
    int dt, B, H, N, d;
    const int32_t *perm;    // [B*H][N]: group g of a head is rows perm[g*128 .. g*128+127]
    const int32_t *tokens;  // [B*H][N/128][n_tokens]: the keys of each group
    int n_tokens;
    float scale;            // > 0
    void *O;
    float *LSE;
    char *ws;               // error word in the first bytes
    uint64_t wait_limit_ns; // bounded device waits (tensor-core path)
};
bsa_status launch_forward_tokens(const TokenArgs &a, cudaStream_t st);     // CUDA cores (fp32 and bf16)
bsa_status launch_forward_tokens_tc(const TokenArgs &a, cudaStream_t st);  // bf16, tcgen05 with row gathers
bool make_tma_map_bf16_rows(CUtensorMap *m, const void *base, uint64_t rows, int d);

// token selection: per group of 128 queries, the n_keep tokens of largest exact mass
struct TokenSelectArgs {
    const void *Q, *K;
    int dt, B, H, N, d;
    const int32_t *perm;   // [B*H][N] query groups
    const float *LSE;      // [B*H][N] dense logsumexp (natural log)
    float scale;           // > 0
    int n_keep;            // tokens per group
    int32_t *tokens;       // [B*H][N/128][n_keep] (written, ascending per group)
    char *ws;
    uint64_t wait_limit_ns;  // bounded device waits (tensor-core path)
};
// workspace: header, masses fp32 [B*H*N/128][N], bitmap words [B*H*N/128][N/32]
struct TokenSelectWs {
    size_t mass, bitmap, total;
};
TokenSelectWs token_select_ws_layout(int B, int H, int N);
bsa_status launch_select_tokens(const TokenSelectArgs &a, cudaStream_t st);
// bf16: the masses of every (group, key) on tcgen05 into mass [B*H*N/128][N]
bsa_status launch_token_mass_tc(const TokenSelectArgs &a, float *mass, cudaStream_t st);

// query groups: per head, the median-split principal-direction partition into groups of 128
constexpr int kMaxQueryGroups = 512;  // groups per head (N <= 65536)
struct GroupArgs {
    const void *Q;
    int dt, B, H, N, d;
    int32_t *perm;  // [B*H][N] (written)
    char *ws;
    uint64_t wait_limit_ns;  // bounded device waits (the tcgen05 scatter pass)
};
// workspace: header; working permutation, projection keys and a scratch copy, [B*H][N]
// each; per head N/128 slots of a slice's row sum [d], a slice's scatter blocks
// [d*d/256 * 136] and a segment's (mean, direction) [2][d]
struct QueryGroupWs {
    size_t work, keys, scratch, psum, pscatter, dir, total;
};
QueryGroupWs query_groups_ws_layout(int B, int H, int N, int d);
bsa_status launch_query_groups(const GroupArgs &a, cudaStream_t st);

}  // namespace bsa
