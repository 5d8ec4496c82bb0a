// api.cu -- the C ABI of libbsa.so: argument validation, workspace layout and
// dispatch to the kernels. Every check runs on the host before any launch.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>

#include "internal.h"

namespace {

uint32_t g_dbg_flags = 0;
uint64_t g_wait_limit_ns = bsa::kDefaultWaitNs;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// index_mode 0 reads the CSR arrays, 1 the bitmap
bool index_args_ok(const int32_t *row_ptr, const int32_t *col_idx, const uint32_t *bitmap, int index_mode)
{
    if (index_mode == 0) return row_ptr && col_idx;
    if (index_mode == 1) return bitmap != nullptr;
    return false;
}

// Blocks per row or column; a sequence that is not a multiple of the block size ends in a
// ragged block ("多模态DiT中的块稀疏注意力" §4.1: the tile loop masks the padding).
int n_blocks(int N, int block) { return (N + block - 1) / block; }

bsa_status check_shape(int B, int H, int N, int d, int block)
{
    if (B <= 0 || H <= 0 || N <= 0) return BSA_ERR_SHAPE;
    if (d != 64 && d != 128) return BSA_ERR_SHAPE;
    if (block != 64 && block != 128) return BSA_ERR_SHAPE;
    const int64_t rows = static_cast<int64_t>(B) * H * N;
    if (rows > INT32_MAX) return BSA_ERR_SHAPE;  // TMA row coordinates are int32
    return BSA_OK;
}

// Blocks kept per Q block: max(1, floor(density * nKB)), density as given (fp32).
int topk_keep(float density, int nKB)
{
    int k = static_cast<int>(std::floor(static_cast<double>(density) * static_cast<double>(nKB)));
    if (k < 1) k = 1;
    if (k > nKB) k = nKB;
    return k;
}

bool valid_density(float density) { return std::isfinite(density) && density > 0.0f && density <= 1.0f; }

// Per-modality counts ("多模态DiT中的块稀疏注意力" §3.3): a group of n key blocks with
// density rho keeps max(1, floor(rho * n)) of them (at most n); rho = 0 switches the
// group off. density = {text->text, text->image, image->text, image->image}.
int region_keep(float density, int n)
{
    if (n <= 0 || density <= 0.0f) return 0;
    return topk_keep(density, n);
}

bool valid_modal(int nB, int n_text, const float *density)
{
    if (!density || n_text < 0 || n_text > nB) return false;
    for (int g = 0; g < 4; ++g)
        if (!std::isfinite(density[g]) || density[g] < 0.0f || density[g] > 1.0f) return false;
    return true;
}

// kq[a][b] and the per-(b, h) count for the modality groups
int64_t modal_counts(int nB, int n_text, const float *density, int kq[2][2])
{
    const int n_img = nB - n_text;
    kq[0][0] = region_keep(density[0], n_text);
    kq[0][1] = region_keep(density[1], n_img);
    kq[1][0] = region_keep(density[2], n_text);
    kq[1][1] = region_keep(density[3], n_img);
    return static_cast<int64_t>(n_text) * (kq[0][0] + kq[0][1]) + static_cast<int64_t>(n_img) * (kq[1][0] + kq[1][1]);
}

// Static spec: structural checks; `count` gets the per-(b, h) active block count
// (band and cuboid only).
bsa_status check_spec(const bsa_static_spec *s, int nB, int64_t *count)
{
    *count = -1;
    if (s->kind == BSA_STATIC_EXPLICIT) {
        if (!s->bitmap || !aligned(s->bitmap, 4)) return BSA_ERR_INVALID_ARG;
        return BSA_OK;
    }
    if (s->n_text_blocks < 0 || s->n_text_blocks > nB) return BSA_ERR_INVALID_ARG;
    const int nt = s->n_text_blocks;
    int64_t c = 0;
    if (s->kind == BSA_STATIC_MODALITY_BAND) {
        if (s->band < 0 || s->n_anchors < 0 || s->n_anchors > BSA_MAX_ANCHORS) return BSA_ERR_INVALID_ARG;
        for (int a = 0; a < s->n_anchors; ++a)
            if (s->anchors[a] < 0 || s->anchors[a] >= nB - nt) return BSA_ERR_INVALID_ARG;
        for (int i = 0; i < nB; ++i)
            for (int j = 0; j < nB; ++j) {
                bool on = i < nt || j < nt;
                if (!on) {
                    const int r = i - nt, cc = j - nt;
                    on = std::abs(r - cc) <= s->band;
                    for (int a = 0; a < s->n_anchors && !on; ++a) on = r == s->anchors[a] || cc == s->anchors[a];
                }
                c += on;
            }
    } else if (s->kind == BSA_STATIC_CUBOID) {
        if (s->grid_t <= 0 || s->grid_h <= 0 || s->grid_w <= 0) return BSA_ERR_INVALID_ARG;
        const int64_t cells = static_cast<int64_t>(s->grid_t) * s->grid_h * s->grid_w;
        if (nt + cells != nB) return BSA_ERR_SHAPE;
        // text rows and columns, then each cuboid's own cell plus its in-grid faces
        c = static_cast<int64_t>(nt) * nB + cells * nt;
        for (int t = 0; t < s->grid_t; ++t)
            for (int h = 0; h < s->grid_h; ++h)
                for (int w = 0; w < s->grid_w; ++w)
                    c += 1 + (t > 0) + (t + 1 < s->grid_t) + (h > 0) + (h + 1 < s->grid_h) + (w > 0) +
                         (w + 1 < s->grid_w);
    } else {
        return BSA_ERR_INVALID_ARG;
    }
    *count = c;
    return BSA_OK;
}

}  // namespace

namespace bsa {

bsa_status current_sm_count(int *sm_count)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BSA_ERR_CUDA;
    return BSA_OK;
}

bsa_status prepare_build_mask(const void *Q, const void *K, int dt, int B, int H, int N, int d, int block,
                              float density, const bsa_static_spec *spec, int32_t *row_ptr, int32_t *col_idx,
                              int64_t col_capacity, uint32_t *bitmap, MaskArgs *out)
{
    bsa_status s = check_shape(B, H, N, d, block);
    if (s != BSA_OK) return s;
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    if (!row_ptr || !col_idx || !bitmap || col_capacity < 0) return BSA_ERR_INVALID_ARG;
    if (!aligned(row_ptr, 4) || !aligned(col_idx, 4) || !aligned(bitmap, 4)) return BSA_ERR_INVALID_ARG;
    const int nB = n_blocks(N, block);
    const int64_t R = static_cast<int64_t>(B) * H * nB;
    MaskArgs a{};
    a.Q = Q;
    a.K = K;
    a.dt = dt;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.block = block;
    a.nQB = nB;
    a.nKB = nB;
    a.W = (nB + 31) / 32;
    a.spec = spec;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.col_capacity = col_capacity;
    a.bitmap = bitmap;
    int64_t nnz;
    if (!spec) {
        if (!Q || !K || !aligned(Q, 16) || !aligned(K, 16)) return BSA_ERR_INVALID_ARG;
        if (!valid_density(density)) return BSA_ERR_INVALID_ARG;
        if (nB > kMaxKvBlocks) return BSA_ERR_UNSUPPORTED;
        a.k = topk_keep(density, nB);
        a.n_text = 0;
        a.kq[1][1] = a.k;
        nnz = R * a.k;
    } else {
        int64_t c = 0;
        s = check_spec(spec, nB, &c);
        if (s != BSA_OK) return s;
        nnz = spec->kind == BSA_STATIC_EXPLICIT ? -1 : R / nB * c;
    }
    if (nnz > col_capacity) return BSA_ERR_CAPACITY;
    if (R * nB > INT32_MAX && (nnz < 0 || nnz > INT32_MAX)) return BSA_ERR_UNSUPPORTED;  // row_ptr is int32
    *out = a;
    return BSA_OK;
}

}  // namespace bsa

extern "C" {

const char *bsa_status_string(int status)
{
    switch (status) {
    case BSA_OK: return "ok";
    case BSA_ERR_INVALID_ARG: return "invalid argument";
    case BSA_ERR_SHAPE: return "unsupported shape";
    case BSA_ERR_DTYPE: return "unsupported dtype";
    case BSA_ERR_CAPACITY: return "col_idx capacity too small";
    case BSA_ERR_NONFINITE: return "non-finite block score";
    case BSA_ERR_TIMEOUT: return "device wait timed out";
    case BSA_ERR_CUDA: return "CUDA runtime error";
    case BSA_ERR_UNSUPPORTED: return "unsupported request";
    case BSA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

bsa_status bsa_mask_nnz_modal(int B, int H, int N, int block, int n_text_blocks, const float *density,
                              int64_t *nnz)
{
    if (!nnz) return BSA_ERR_INVALID_ARG;
    const bsa_status s = check_shape(B, H, N, 64, block);
    if (s != BSA_OK) return s;
    const int nB = n_blocks(N, block);
    if (!valid_modal(nB, n_text_blocks, density)) return BSA_ERR_INVALID_ARG;
    int kq[2][2];
    *nnz = static_cast<int64_t>(B) * H * modal_counts(nB, n_text_blocks, density, kq);
    return BSA_OK;
}

bsa_status bsa_build_mask_modal(const void *Q, const void *K, int dt, int B, int H, int N, int d, int block,
                                int n_text_blocks, const float *density, int32_t *row_ptr, int32_t *col_idx,
                                int64_t col_capacity, uint32_t *bitmap, void *workspace, size_t workspace_bytes,
                                void *stream)
{
    bsa_status s = check_shape(B, H, N, d, block);
    if (s != BSA_OK) return s;
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    if (!Q || !K || !aligned(Q, 16) || !aligned(K, 16)) return BSA_ERR_INVALID_ARG;
    if (!row_ptr || !col_idx || !bitmap || col_capacity < 0) return BSA_ERR_INVALID_ARG;
    if (!aligned(row_ptr, 4) || !aligned(col_idx, 4) || !aligned(bitmap, 4)) return BSA_ERR_INVALID_ARG;
    const int nB = n_blocks(N, block);
    if (!valid_modal(nB, n_text_blocks, density)) return BSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::mask_workspace_bytes(B, H, N, d, block))
        return BSA_ERR_WORKSPACE;
    if (nB > bsa::kMaxKvBlocks) return BSA_ERR_UNSUPPORTED;
    bsa::MaskArgs a{};
    a.Q = Q;
    a.K = K;
    a.dt = dt;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.block = block;
    a.nQB = nB;
    a.nKB = nB;
    a.W = (nB + 31) / 32;
    a.spec = nullptr;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.col_capacity = col_capacity;
    a.bitmap = bitmap;
    a.ws = static_cast<char *>(workspace);
    a.n_text = n_text_blocks;
    const int64_t nnz = static_cast<int64_t>(B) * H * modal_counts(nB, n_text_blocks, density, a.kq);
    a.k = 0;
    if (nnz > col_capacity) return BSA_ERR_CAPACITY;
    if (nnz > INT32_MAX) return BSA_ERR_UNSUPPORTED;  // row_ptr is int32
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&a.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BSA_ERR_CUDA;
    return bsa::launch_build_mask(a, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_build_mask_exact(const void *Q, const void *K, int dt, int B, int H, int N, int d, int block,
                                float density, float scale, const float *LSE, int32_t *row_ptr, int32_t *col_idx,
                                int64_t col_capacity, uint32_t *bitmap, void *workspace, size_t workspace_bytes,
                                void *stream)
{
    bsa_status s = check_shape(B, H, N, d, block);
    if (s != BSA_OK) return s;
    if (dt == BSA_FP32) return BSA_ERR_UNSUPPORTED;  // the mass pass runs on bf16 tensor cores
    if (dt != BSA_BF16) return BSA_ERR_DTYPE;
    if (!Q || !K || !LSE || !aligned(Q, 16) || !aligned(K, 16) || !aligned(LSE, 4)) return BSA_ERR_INVALID_ARG;
    if (!row_ptr || !col_idx || !bitmap || col_capacity < 0) return BSA_ERR_INVALID_ARG;
    if (!aligned(row_ptr, 4) || !aligned(col_idx, 4) || !aligned(bitmap, 4)) return BSA_ERR_INVALID_ARG;
    if (!valid_density(density)) return BSA_ERR_INVALID_ARG;
    if (std::isnan(scale) || std::isinf(scale)) return BSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::exact_workspace_bytes(B, H, N, d, block))
        return BSA_ERR_WORKSPACE;
    const int nB = n_blocks(N, block);
    if (nB > bsa::kMaxKvBlocks) return BSA_ERR_UNSUPPORTED;
    const int64_t R = static_cast<int64_t>(B) * H * nB;
    bsa::ExactArgs a{};
    a.Q = Q;
    a.K = K;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.block = block;
    a.nQB = nB;
    a.nKB = nB;
    a.W = (nB + 31) / 32;
    a.k = topk_keep(density, nB);
    a.scale = scale > 0.0f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    a.LSE = LSE;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.bitmap = bitmap;
    a.ws = static_cast<char *>(workspace);
    a.wait_limit_ns = g_wait_limit_ns;
    const int64_t nnz = R * a.k;
    if (nnz > col_capacity) return BSA_ERR_CAPACITY;
    if (nnz > INT32_MAX) return BSA_ERR_UNSUPPORTED;  // row_ptr is int32
    return bsa::launch_build_mask_exact(a, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_workspace_size(int which, int B, int H, int N, int d, int block, size_t *bytes)
{
    if (!bytes) return BSA_ERR_INVALID_ARG;
    const bsa_status s = check_shape(B, H, N, d, block);
    if (s != BSA_OK) return s;
    if (which == 0) *bytes = bsa::mask_workspace_bytes(B, H, N, d, block);
    else if (which == 1) *bytes = bsa::fwd_workspace_bytes(B, H, N, d, block);
    else if (which == 2) *bytes = bsa::exact_workspace_bytes(B, H, N, d, block);
    else if (which == 3) {
        if (N % bsa::kTokenGroup != 0) return BSA_ERR_SHAPE;
        *bytes = bsa::token_select_ws_layout(B, H, N).total;
    } else if (which == 4) {
        if (N % bsa::kTokenGroup != 0) return BSA_ERR_SHAPE;
        *bytes = bsa::query_groups_ws_layout(B, H, N, d).total;
    } else return BSA_ERR_INVALID_ARG;
    return BSA_OK;
}

bsa_status bsa_mask_nnz(int B, int H, int N, int block, float density, const bsa_static_spec *spec, int64_t *nnz)
{
    if (!nnz) return BSA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || N <= 0 || (block != 64 && block != 128)) return BSA_ERR_SHAPE;
    const int nB = n_blocks(N, block);
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (!spec) {
        if (!valid_density(density)) return BSA_ERR_INVALID_ARG;
        *nnz = BH * nB * topk_keep(density, nB);
        return BSA_OK;
    }
    int64_t c = 0;
    const bsa_status s = check_spec(spec, nB, &c);
    if (s != BSA_OK) return s;
    *nnz = spec->kind == BSA_STATIC_EXPLICIT ? BH * nB * nB : BH * c;
    return BSA_OK;
}

bsa_status bsa_build_mask(const void *Q, const void *K, int dt, int B, int H, int N, int d, int block, float density,
                          const bsa_static_spec *spec, int32_t *row_ptr, int32_t *col_idx, int64_t col_capacity,
                          uint32_t *bitmap, void *workspace, size_t workspace_bytes, void *stream)
{
    bsa::MaskArgs a{};
    bsa_status s = bsa::prepare_build_mask(Q, K, dt, B, H, N, d, block, density, spec, row_ptr, col_idx,
                                           col_capacity, bitmap, &a);
    if (s != BSA_OK) return s;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::mask_workspace_bytes(B, H, N, d, block))
        return BSA_ERR_WORKSPACE;
    a.ws = static_cast<char *>(workspace);
    // all argument checks passed: only now touch the device
    s = bsa::current_sm_count(&a.sm_count);
    if (s != BSA_OK) return s;
    return bsa::launch_build_mask(a, static_cast<cudaStream_t>(stream));
}

static bsa_status forward_impl(const void *Q, const void *K, const void *V, int dt, int B, int H, int N, int d,
                               int block, const int32_t *row_ptr, const int32_t *col_idx, const uint32_t *bitmap,
                               int index_mode, float scale, const float *R, void *O, float *LSE, void *workspace,
                               size_t workspace_bytes, void *stream)
{
    bsa_status s = check_shape(B, H, N, d, block);
    if (s != BSA_OK) return s;
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    if (!Q || !K || !V || !O || !LSE) return BSA_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(LSE, 4))
        return BSA_ERR_INVALID_ARG;
    const bool planned = (index_mode & BSA_INDEX_PLANNED) != 0;
    index_mode &= ~BSA_INDEX_PLANNED;
    if (!index_args_ok(row_ptr, col_idx, bitmap, index_mode)) return BSA_ERR_INVALID_ARG;
    if (std::isnan(scale) || std::isinf(scale)) return BSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::fwd_workspace_bytes(B, H, N, d, block))
        return BSA_ERR_WORKSPACE;
    bsa::FwdArgs a{};
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.dt = dt;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.block = block;
    a.nQB = n_blocks(N, block);
    a.nKB = n_blocks(N, block);
    a.W = (a.nKB + 31) / 32;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.bitmap = bitmap;
    a.index_mode = index_mode;
    a.scale = scale > 0.0f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    a.O = O;
    a.LSE = LSE;
    a.R = R;
    a.ws = static_cast<char *>(workspace);
    a.dbg_flags = g_dbg_flags;
    a.wait_limit_ns = g_wait_limit_ns;
    a.planned = planned ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return dt == BSA_BF16 ? bsa::launch_forward_tc(a, st) : bsa::launch_forward_simt(a, st);
}

bsa_status bsa_forward_lse(const void *Q, const void *K, int dt, int B, int H, int N, int d, int block,
                           const int32_t *row_ptr, const int32_t *col_idx, const uint32_t *bitmap, int index_mode,
                           float scale, float *LSE, void *workspace, size_t workspace_bytes, void *stream)
{
    bsa_status s = check_shape(B, H, N, d, block);
    if (s != BSA_OK) return s;
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    if (!Q || !K || !LSE || !aligned(Q, 16) || !aligned(K, 16) || !aligned(LSE, 4)) return BSA_ERR_INVALID_ARG;
    if (!index_args_ok(row_ptr, col_idx, bitmap, index_mode)) return BSA_ERR_INVALID_ARG;
    if (std::isnan(scale) || std::isinf(scale)) return BSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::fwd_workspace_bytes(B, H, N, d, block))
        return BSA_ERR_WORKSPACE;
    bsa::FwdArgs a{};
    a.Q = Q;
    a.K = K;
    a.dt = dt;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.block = block;
    a.nQB = n_blocks(N, block);
    a.nKB = n_blocks(N, block);
    a.W = (a.nKB + 31) / 32;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.bitmap = bitmap;
    a.index_mode = index_mode;
    a.scale = scale > 0.0f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    a.LSE = LSE;
    a.ws = static_cast<char *>(workspace);
    a.dbg_flags = g_dbg_flags;
    a.wait_limit_ns = g_wait_limit_ns;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // V and O stay null: the kernels read no V and write no O
    return dt == BSA_BF16 ? bsa::launch_forward_lse_tc(a, st) : bsa::launch_forward_simt(a, st);
}

bsa_status bsa_forward_plan(int dt, int B, int H, int N, int d, int block, const int32_t *row_ptr,
                            const int32_t *col_idx, const uint32_t *bitmap, int index_mode, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    bsa_status s = check_shape(B, H, N, d, block);
    if (s != BSA_OK) return s;
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    if (!index_args_ok(row_ptr, col_idx, bitmap, index_mode)) return BSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::fwd_workspace_bytes(B, H, N, d, block))
        return BSA_ERR_WORKSPACE;
    if (dt == BSA_FP32) return BSA_OK;  // the CUDA-core forward keeps no work list
    bsa::FwdArgs a{};
    a.dt = dt;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.block = block;
    a.nQB = n_blocks(N, block);
    a.nKB = n_blocks(N, block);
    a.W = (a.nKB + 31) / 32;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.bitmap = bitmap;
    a.index_mode = index_mode;
    a.ws = static_cast<char *>(workspace);
    a.dbg_flags = g_dbg_flags;
    a.wait_limit_ns = g_wait_limit_ns;
    return bsa::launch_forward_plan_tc(a, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_forward(const void *Q, const void *K, const void *V, int dt, int B, int H, int N, int d, int block,
                       const int32_t *row_ptr, const int32_t *col_idx, const uint32_t *bitmap, int index_mode,
                       float scale, void *O, float *LSE, void *workspace, size_t workspace_bytes, void *stream)
{
    return forward_impl(Q, K, V, dt, B, H, N, d, block, row_ptr, col_idx, bitmap, index_mode, scale, nullptr, O, LSE,
                        workspace, workspace_bytes, stream);
}

bsa_status bsa_forward_residual(const void *Q, const void *K, const void *V, int dt, int B, int H, int N, int d,
                                int block, const int32_t *row_ptr, const int32_t *col_idx, const uint32_t *bitmap,
                                int index_mode, float scale, const float *R, void *O, float *LSE, void *workspace,
                                size_t workspace_bytes, void *stream)
{
    if (!R || !aligned(R, 16)) return BSA_ERR_INVALID_ARG;
    return forward_impl(Q, K, V, dt, B, H, N, d, block, row_ptr, col_idx, bitmap, index_mode, scale, R, O, LSE,
                        workspace, workspace_bytes, stream);
}

bsa_status bsa_forward_tokens(const void *Q, const void *K, const void *V, int dt, int B, int H, int N, int d,
                              const int32_t *perm, const int32_t *tokens, int n_tokens, float scale, void *O,
                              float *LSE, void *workspace, size_t workspace_bytes, void *stream)
{
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || N % bsa::kTokenGroup != 0) return BSA_ERR_SHAPE;
    if (static_cast<int64_t>(B) * H * N > INT32_MAX || static_cast<int64_t>(B) * H > 65535) return BSA_ERR_SHAPE;
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    if (!Q || !K || !V || !O || !LSE || !perm || !tokens) return BSA_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(LSE, 4) ||
        !aligned(perm, 4) || !aligned(tokens, 4))
        return BSA_ERR_INVALID_ARG;
    if (n_tokens < 1 || n_tokens > N) return BSA_ERR_INVALID_ARG;
    if (std::isnan(scale) || std::isinf(scale)) return BSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::kWsHeader) return BSA_ERR_WORKSPACE;
    bsa::TokenArgs a{};
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.dt = dt;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.perm = perm;
    a.tokens = tokens;
    a.n_tokens = n_tokens;
    a.scale = scale > 0.0f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    a.O = O;
    a.LSE = LSE;
    a.ws = static_cast<char *>(workspace);
    a.wait_limit_ns = g_wait_limit_ns;
    // bf16 on the tensor cores (rows gathered by index); fp32 on CUDA cores
    return dt == BSA_BF16 ? bsa::launch_forward_tokens_tc(a, static_cast<cudaStream_t>(stream))
                          : bsa::launch_forward_tokens(a, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_query_groups(const void *Q, int dt, int B, int H, int N, int d, int32_t *perm, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || N % bsa::kTokenGroup != 0) return BSA_ERR_SHAPE;
    if (N / bsa::kTokenGroup > bsa::kMaxQueryGroups || static_cast<int64_t>(B) * H * N > INT32_MAX ||
        static_cast<int64_t>(B) * H > 65535)
        return BSA_ERR_SHAPE;
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    if (!Q || !perm || !aligned(Q, 16) || !aligned(perm, 4)) return BSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::query_groups_ws_layout(B, H, N, d).total)
        return BSA_ERR_WORKSPACE;
    bsa::GroupArgs a{};
    a.Q = Q;
    a.dt = dt;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.perm = perm;
    a.ws = static_cast<char *>(workspace);
    a.wait_limit_ns = g_wait_limit_ns;
    return bsa::launch_query_groups(a, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_select_tokens(const void *Q, const void *K, int dt, int B, int H, int N, int d, const int32_t *perm,
                             const float *LSE, float density, float scale, int32_t *tokens, int64_t tokens_capacity,
                             void *workspace, size_t workspace_bytes, void *stream)
{
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || N % bsa::kTokenGroup != 0) return BSA_ERR_SHAPE;
    if (static_cast<int64_t>(B) * H * N > INT32_MAX || static_cast<int64_t>(B) * H > 65535) return BSA_ERR_SHAPE;
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    // fp32 runs on CUDA cores with a shared-memory row of N keys per group
    if (dt == BSA_FP32 &&
        sizeof(float) * (bsa::kTokenGroup * d + 32 * (d + 1)) + sizeof(uint32_t) * static_cast<size_t>(N) > 232448)
        return BSA_ERR_SHAPE;
    if (!Q || !K || !perm || !LSE || !tokens) return BSA_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(perm, 4) || !aligned(LSE, 4) || !aligned(tokens, 4))
        return BSA_ERR_INVALID_ARG;
    if (!valid_density(density) || std::isnan(scale) || std::isinf(scale)) return BSA_ERR_INVALID_ARG;
    const int n_keep = topk_keep(density, N);
    if (tokens_capacity < static_cast<int64_t>(B) * H * (N / bsa::kTokenGroup) * n_keep) return BSA_ERR_CAPACITY;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::token_select_ws_layout(B, H, N).total)
        return BSA_ERR_WORKSPACE;
    bsa::TokenSelectArgs a{};
    a.Q = Q;
    a.K = K;
    a.dt = dt;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.perm = perm;
    a.LSE = LSE;
    a.scale = scale > 0.0f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    a.n_keep = n_keep;
    a.tokens = tokens;
    a.ws = static_cast<char *>(workspace);
    a.wait_limit_ns = g_wait_limit_ns;
    return bsa::launch_select_tokens(a, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_tokens_per_group(int N, float density, int *n_tokens)
{
    if (!n_tokens) return BSA_ERR_INVALID_ARG;
    if (N <= 0) return BSA_ERR_SHAPE;
    if (!valid_density(density)) return BSA_ERR_INVALID_ARG;
    *n_tokens = topk_keep(density, N);
    return BSA_OK;
}

bsa_status bsa_residual_capture(const void *O_dense, const void *O_sparse, int dt, int64_t count, float *R,
                                void *stream)
{
    if (dt != BSA_BF16 && dt != BSA_FP32) return BSA_ERR_DTYPE;
    if (count < 0) return BSA_ERR_INVALID_ARG;
    if (count == 0) return BSA_OK;
    if (!O_dense || !O_sparse || !R) return BSA_ERR_INVALID_ARG;
    if (!aligned(O_dense, 16) || !aligned(O_sparse, 16) || !aligned(R, 16)) return BSA_ERR_INVALID_ARG;
    return bsa::launch_residual_capture(O_dense, O_sparse, dt, count, R, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_check_device_error(void *workspace, void *stream)
{
    if (!workspace) return BSA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t err = 0;
    if (cudaMemcpyAsync(&err, workspace, sizeof(err), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return BSA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return BSA_ERR_CUDA;
    if (err != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof(err), st) != cudaSuccess) return BSA_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return BSA_ERR_CUDA;
    }
    return static_cast<bsa_status>(err);
}

bsa_status bsa_validate_index(int B, int H, int N, int block, const int32_t *row_ptr, const int32_t *col_idx,
                              const uint32_t *bitmap, void *workspace, size_t workspace_bytes, void *stream)
{
    if (B <= 0 || H <= 0 || N <= 0 || (block != 64 && block != 128)) return BSA_ERR_SHAPE;
    if (!row_ptr || !col_idx) return BSA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < bsa::kWsHeader) return BSA_ERR_WORKSPACE;
    const int64_t R = static_cast<int64_t>(B) * H * n_blocks(N, block);
    if (R > INT32_MAX) return BSA_ERR_SHAPE;
    return bsa::launch_validate_index(static_cast<int>(R), n_blocks(N, block), row_ptr, col_idx, bitmap,
                                      static_cast<char *>(workspace), static_cast<cudaStream_t>(stream));
}

bsa_status bsa_debug_config(uint32_t flags, uint64_t wait_limit_ns)
{
    g_dbg_flags = flags;
    g_wait_limit_ns = wait_limit_ns ? wait_limit_ns : bsa::kDefaultWaitNs;
    return BSA_OK;
}

}  // extern "C"
