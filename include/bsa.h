/*
 * bsa.h -- C ABI of the GB300 block-sparse attention forward library (libbsa.so).
 *
 * The library computes, on one GPU (sm_103a), the hot path described in
 *   [P1] "多模态DiT中的块稀疏注意力：从原理到工程落地"
 *   [P3] "Can sparse attention close the quality gap in diffusion transformers"
 * in two calls:
 *   bsa_build_mask  -- block mask -> per-Q-block active KV block lists (CSR) + bitmap
 *   bsa_forward     -- block-sparse FlashAttention forward over those lists -> O, LSE
 *
 * Conventions shared by every call
 *   - Q, K, V, O are row-major [B][H][N][d], contiguous, in device memory.
 *     dtype BSA_BF16 (bf16 inputs, bf16 O) or BSA_FP32 (fp32 inputs, fp32 O).
 *     LSE is fp32 [B][H][N], natural logarithm.
 *   - block (bs) in {64, 128}; d in {64, 128}; N >= 1; nQB = nKB = ceil(N / block).
 *     When N is not a multiple of block the last block is ragged: it holds the tokens
 *     up to N ("多模态DiT中的块稀疏注意力" §4.1, the tile loop's padding mask); keys past N
 *     do not count, rows past N do not exist, and mean pooling averages the tokens the
 *     block holds.
 *   - Index: rows r = (b*H + h)*nQB + i.
 *       row_ptr  int32 [B*H*nQB + 1], exclusive prefix sums of row lengths;
 *       col_idx  int32 [nnz], the active KV block ids of each row, strictly ascending;
 *       bitmap   uint32 [B*H*nQB][W], W = ceil(nKB / 32); bit (j % 32) of word j / 32
 *                is set iff KV block j is active for the row.
 *   - Ownership: the caller allocates and owns every buffer (device memory for
 *     tensors, index and workspace). No call allocates, frees or synchronises
 *     except bsa_check_device_error, which synchronises `stream`.
 *   - Streams: device work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and runs asynchronously.
 *   - Errors: argument checks run on the host before any launch; a failed check
 *     returns its status and enqueues nothing. Conditions only the device can see
 *     (a NaN block score, a capacity overflow of an explicit bitmap, a bounded wait
 *     that gave up) are recorded in the first bytes of the call's workspace and are
 *     returned by bsa_check_device_error on that workspace.
 *   - Workspaces are caller-provided device buffers of at least the size
 *     bsa_workspace_size reports; they must be 256-byte aligned. A new workspace
 *     must be zero-filled once before its first call (e.g. cudaMemset): its first
 *     bytes hold the device status word and the counters of the launches whose
 *     last CTA finishes the work (the forward's work list, a static pattern), and
 *     every call leaves them ready for the next one.
 *   - Calls that share a workspace, or write the same outputs, must not overlap
 *     on the GPU (put them on one stream or order them with events).
 */
#ifndef BSA_H_
#define BSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BSA_OK = 0,
    BSA_ERR_INVALID_ARG = 1, /* null pointer, bad enum, density out of (0, 1], misaligned buffer */
    BSA_ERR_SHAPE = 2,       /* unsupported B, H, N, d or block */
    BSA_ERR_DTYPE = 3,       /* dtype not supported for this call */
    BSA_ERR_CAPACITY = 4,    /* col_capacity smaller than the mask's nnz */
    BSA_ERR_NONFINITE = 5,   /* a block score was NaN (device-raised) */
    BSA_ERR_TIMEOUT = 6,     /* a bounded device wait gave up (device-raised) */
    BSA_ERR_CUDA = 7,        /* a CUDA runtime call failed */
    BSA_ERR_UNSUPPORTED = 8, /* valid request this build does not implement */
    BSA_ERR_WORKSPACE = 9    /* workspace null or smaller than bsa_workspace_size */
} bsa_status;

typedef enum { BSA_BF16 = 0, BSA_FP32 = 1 } bsa_dtype;

typedef enum {
    BSA_STATIC_EXPLICIT = 0,      /* a caller-given block bitmap */
    BSA_STATIC_MODALITY_BAND = 1, /* [P1] §3.1-§3.2: text dense + image band + anchors */
    BSA_STATIC_CUBOID = 2         /* [P1] §3.2: video cuboids + face neighbours + text */
} bsa_static_kind;

#define BSA_MAX_ANCHORS 8

/* A static block mask ([P1] §2.3: fixed before the run, from the task's structure).
 * Leading `n_text_blocks` blocks are text: their rows and columns are dense
 * ([P1] §3.1: text-text dense, text is a global condition for every image block). */
typedef struct {
    int kind;                     /* bsa_static_kind */
    const uint32_t *bitmap;       /* EXPLICIT: device bitmap, layout as the index bitmap:
                                     [B*H*nQB][W], or [nQB][W] when broadcast_bh != 0 */
    int broadcast_bh;             /* EXPLICIT: 1 = one nQB x nKB mask for every (b, h) */
    int n_text_blocks;            /* MODALITY_BAND, CUBOID: leading text blocks */
    int band;                     /* MODALITY_BAND: image block rows r, cols c active iff |r-c| <= band */
    int n_anchors;                /* MODALITY_BAND: number of anchor image blocks (<= 8) */
    int anchors[BSA_MAX_ANCHORS]; /* MODALITY_BAND: image-block ids dense in both directions */
    int grid_t, grid_h, grid_w;   /* CUBOID: cuboid grid; image blocks are cuboids in t-major
                                     raster order, active iff equal or sharing a face */
} bsa_static_spec;

/*
 * bsa_build_mask -- build the block mask and emit both index forms.
 *
 * Dynamic (spec == NULL): the naive block-sparse selector of [P3] (section on
 * mean-pooled block scoring): each Q and K block is mean-pooled, every
 * (Q block i, KV block j) pair is scored by the dot product of the pooled
 * vectors, and each Q block keeps its k = max(1, floor(density * nKB)) best KV
 * blocks ([P1] §5.3: a per-Q-block target count). Exact arithmetic, so results
 * are reproducible bit for bit: pooled sums run over the block's tokens in order
 * in fp32 round-to-nearest, divided by the block's token count (round to nearest;
 * a ragged last block holds fewer than `block` tokens); scores are an fmaf chain over
 * channels 0..d-1 starting at +0; ranking is by value descending with -0 == +0 and
 * ties going to the lower block index. A NaN score raises BSA_ERR_NONFINITE on
 * the device (the emitted index is then unspecified).
 *
 * Static (spec != NULL): evaluates the spec's block predicate ([P1] §2.3, §3.1,
 * §3.2, pre-generated on the GPU as §5.3 recommends) for every (b, h).
 *
 *   Q, K            device [B][H][N][d], dtype dt; read only in dynamic mode (may be
 *                   NULL in static mode)
 *   density         dynamic mode: in (0, 1]; ignored in static mode
 *   row_ptr         device int32 [B*H*nQB + 1] (written)
 *   col_idx         device int32 [col_capacity] (first nnz entries written)
 *   col_capacity    entries available in col_idx; must be >= nnz. For dynamic,
 *                   band and cuboid masks nnz is known on the host
 *                   (bsa_mask_nnz) and a short capacity returns BSA_ERR_CAPACITY
 *                   without launching; for EXPLICIT masks the device checks and
 *                   raises BSA_ERR_CAPACITY (writes stay within capacity).
 *   bitmap          device uint32 [B*H*nQB][W] (written)
 *   workspace       device, >= bsa_workspace_size(0, ...) bytes, 256-byte aligned
 */
bsa_status bsa_build_mask(const void *Q, const void *K, int dt, int B, int H, int N, int d,
                          int block, float density, const bsa_static_spec *spec,
                          int32_t *row_ptr, int32_t *col_idx, int64_t col_capacity,
                          uint32_t *bitmap, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * bsa_build_mask_modal -- the dynamic selector of bsa_build_mask with a density per
 * modality pair ([P1] §3.3: text tokens are few and image patches many, so one
 * global sparsity starves the text blocks; set the density per group of the
 * attention matrix instead, and shift it between groups across denoising steps).
 * Blocks [0, n_text_blocks) are text, the rest image (the static specs' order).
 *   density[4]  {text->text, text->image, image->text, image->image}, each in [0, 1]:
 *               a query block of modality a keeps, among the key blocks of modality
 *               b (n_b of them), the top max(1, floor(density * n_b)) by the pooled
 *               score (at most n_b; density 0 keeps none), ties to the lower index,
 *               the same arithmetic as bsa_build_mask. A row keeps the union of
 *               its two groups.
 * Rows of the same modality have equal lengths, so row_ptr is exact and
 * bsa_mask_nnz_modal gives nnz. Other arguments, outputs, workspace and errors as
 * bsa_build_mask (dynamic); an invalid density or n_text_blocks outside [0, nB]
 * is BSA_ERR_INVALID_ARG. With n_text_blocks = 0 and density[3] = rho this is
 * bsa_build_mask(density = rho) bit for bit.
 */
bsa_status bsa_build_mask_modal(const void *Q, const void *K, int dt, int B, int H, int N, int d,
                                int block, int n_text_blocks, const float *density,
                                int32_t *row_ptr, int32_t *col_idx, int64_t col_capacity,
                                uint32_t *bitmap, void *workspace, size_t workspace_bytes,
                                void *stream);

/* Host-only: exact nnz of bsa_build_mask_modal. */
bsa_status bsa_mask_nnz_modal(int B, int H, int N, int block, int n_text_blocks,
                              const float *density, int64_t *nnz);

/*
 * bsa_build_mask_exact -- the block-oracle selector of [P3] (section "质量差距有三个可
 * 分离来源": at the same density, keep the blocks that retain the most attention mass
 * under the exact dense attention). Pass 1 is the caller's: LSE of the dense
 * attention (bsa_forward with every block active). This call is pass 2 and the
 * selection: mass_ij = sum over rows r of Q block i and keys c of KV block j of
 * exp(scale * q_r . k_c - LSE_r) (a dense QK^T on tensor cores, fp32 sums), then the
 * top k = max(1, floor(density * nKB)) blocks per Q block by mass, ties to the lower
 * index; CSR and bitmap as bsa_build_mask. Work: 2 * N^2 * d FLOPs per head.
 *   Q, K        device [B][H][N][d] bf16 (BSA_FP32 is BSA_ERR_UNSUPPORTED), 16-byte aligned
 *   scale       the attention's softmax scale; <= 0 selects 1/sqrt(d)
 *   LSE         device fp32 [B][H][N], the dense logsumexp (natural log) of pass 1
 *   workspace   device, >= bsa_workspace_size(2, ...) bytes, 256-byte aligned
 * nnz = B*H*nQB*k. Errors as bsa_build_mask; a NaN mass is BSA_ERR_NONFINITE.
 */
bsa_status bsa_build_mask_exact(const void *Q, const void *K, int dt, int B, int H, int N, int d,
                                int block, float density, float scale, const float *LSE,
                                int32_t *row_ptr, int32_t *col_idx, int64_t col_capacity,
                                uint32_t *bitmap, void *workspace, size_t workspace_bytes,
                                void *stream);

/* index_mode flag of bsa_forward / bsa_forward_residual: reuse the work list already in
 * the workspace (bsa_forward_plan) instead of building it in the call. */
#define BSA_INDEX_PLANNED 0x100

/*
 * bsa_forward -- block-sparse FlashAttention forward ([P1] §4.1 tile loop with the
 * inner KV loop replaced by the active list, §4.3 skipped blocks count as -inf and
 * the output is normalised by the true sum over active blocks only).
 *
 * For each (b, h) and query row r of Q block i, with A(i) the active KV blocks:
 *   s_rc = scale * q_r . k_c for keys c in blocks of A(i);
 *   O_r  = sum_c exp(s_rc) v_c / sum_c exp(s_rc);   LSE_r = ln sum_c exp(s_rc).
 * A row with no active block gets O_r = 0 and LSE_r = -inf.
 *
 *   Q, K, V     device [B][H][N][d], dtype dt
 *   row_ptr, col_idx   CSR index (read when index_mode == 0)
 *   bitmap      bitmap index (read when index_mode == 1); unused pointers may be NULL
 *   index_mode  0: CSR, 1: bitmap + popcount ([P1] §4.1); either may carry
 *               BSA_INDEX_PLANNED (see bsa_forward_plan)
 *   scale       softmax scale; <= 0 selects 1/sqrt(d)
 *   O           device [B][H][N][d], dtype dt (written)
 *   LSE         device fp32 [B][H][N] (written)
 *   workspace   device, >= bsa_workspace_size(1, ...) bytes, 256-byte aligned
 * The index must be well formed (row_ptr non-decreasing from 0, col_idx strictly
 * ascending in [0, nKB)); bsa_validate_index checks one on the device.
 * bf16 runs as two launches on `stream`: the work list (long tiles split by KV range,
 * [P1] §5.3; items of at least an eighth of the per-CTA share longest first, the rest
 * in tile order so that a head's tiles run together) into the workspace, then the
 * tcgen05 kernel. With BSA_INDEX_PLANNED the first is replaced by a one-CTA launch that checks
 * the work list an earlier bsa_forward_plan (or bsa_forward) left in the workspace
 * against this call and resets the scheduler's counters.
 */
bsa_status bsa_forward(const void *Q, const void *K, const void *V, int dt, int B, int H, int N,
                       int d, int block, const int32_t *row_ptr, const int32_t *col_idx,
                       const uint32_t *bitmap, int index_mode, float scale, void *O, float *LSE,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * bsa_forward_lse -- the LSE alone of bsa_forward over the same index: LSE_r = ln sum over
 * the keys c of the row's active blocks of exp(scale * q_r . k_c), -inf for a row with no
 * active block. With every block active it is pass 1 (the dense logsumexp) of the exact
 * selectors ("Can sparse attention close the quality gap in diffusion transformers",
 * section "质量差距有三个可分离来源": bsa_build_mask_exact and bsa_select_tokens take it).
 * No V is read and no O is written: QK^T and the softmax sums only, so about half the
 * forward's MMA work and no PV chain. The values are those bsa_forward writes for LSE, bit
 * for bit, as long as bsa_forward splits no tile (this call never splits one).
 *   Q, K        device [B][H][N][d], dtype dt
 *   row_ptr, col_idx, bitmap, index_mode   as bsa_forward (index_mode 0 or 1, not planned)
 *   scale       softmax scale; <= 0 selects 1/sqrt(d)
 *   LSE         device fp32 [B][H][N] (written)
 *   workspace   device, >= bsa_workspace_size(1, ...) bytes, 256-byte aligned
 * Errors: as bsa_forward.
 */
bsa_status bsa_forward_lse(const void *Q, const void *K, int dt, int B, int H, int N, int d, int block,
                           const int32_t *row_ptr, const int32_t *col_idx, const uint32_t *bitmap,
                           int index_mode, float scale, float *LSE, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * bsa_forward_plan -- the forward's work list for one index, made once into the forward
 * workspace, for a mask used by many calls ([P1] §5.3: static masks are pre-generated
 * once). The list depends on the index's row lengths and the launch shape, not on Q, K,
 * V: it stays valid for bsa_forward / bsa_forward_residual calls with index_mode |
 * BSA_INDEX_PLANNED, the same dt, B, H, N, d, block, index_mode and workspace, while
 * every query tile's row lengths are those of the planned index (a static mask rebuilt
 * into the same buffers, or any plain top-k mask of the same shape and density). A
 * planned call whose workspace holds no plan for its shape raises BSA_ERR_INVALID_ARG
 * on the device and writes nothing. Each planned call resets the counters it uses, so
 * one plan serves any number of calls in stream order.
 *   row_ptr, col_idx, bitmap, index_mode   as bsa_forward (index_mode 0 or 1)
 *   workspace   device, >= bsa_workspace_size(1, ...) bytes, 256-byte aligned
 * One launch (none for BSA_FP32, whose CUDA-core forward keeps no work list).
 * Errors: BSA_ERR_SHAPE, BSA_ERR_DTYPE, BSA_ERR_INVALID_ARG, BSA_ERR_WORKSPACE.
 */
bsa_status bsa_forward_plan(int dt, int B, int H, int N, int d, int block, const int32_t *row_ptr,
                            const int32_t *col_idx, const uint32_t *bitmap, int index_mode,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Residual compensation ([P3] section "残差补偿找回被丢弃的尾部"; reuse across steps:
 * section "复用精确选择优于重算均值池化"). The blocks a sparse mask drops carry small
 * but nonzero attention mass; the dense-minus-sparse residual changes across
 * denoising steps less than the attention output itself. At an anchor step the
 * caller runs bsa_forward with a full index (every block active) and with the
 * sparse index, and captures R = O_dense - O_sparse; later steps call
 * bsa_forward_residual, which returns O_sparse + R (LSE stays the sparse one).
 *
 * bsa_residual_capture: R[i] = float(O_dense[i]) - float(O_sparse[i]) for
 *   i < count, computed in fp32 (exact widening of bf16, one rounding).
 *   O_dense, O_sparse  device, dtype dt, >= count elements, 16-byte aligned
 *   R                  device fp32, >= count elements, 16-byte aligned (written)
 *   count == 0 enqueues nothing. Errors: BSA_ERR_DTYPE, BSA_ERR_INVALID_ARG (null
 *   or misaligned pointers, negative count), BSA_ERR_CUDA.
 */
bsa_status bsa_residual_capture(const void *O_dense, const void *O_sparse, int dt, int64_t count, float *R,
                                void *stream);

/*
 * bsa_forward_residual: bsa_forward whose output is O_sparse + R, with R added in
 * fp32 before the output is rounded to dt. R: device fp32 [B][H][N][d], 16-byte
 * aligned, read only. Every other argument, the LSE and the error behaviour are
 * those of bsa_forward; a null or misaligned R is BSA_ERR_INVALID_ARG.
 */
bsa_status bsa_forward_residual(const void *Q, const void *K, const void *V, int dt, int B, int H, int N,
                                int d, int block, const int32_t *row_ptr, const int32_t *col_idx,
                                const uint32_t *bitmap, int index_mode, float scale, const float *R,
                                void *O, float *LSE, void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * bsa_query_groups -- tile-aligned query groups for token-level selection ("Can sparse
 * attention close the quality gap in diffusion transformers", section "token 级选择需要瓦片
 * 对齐的查询分组"): the queries of each head are split recursively at the median of their
 * projection on the group's principal direction until every group holds 128 queries. A
 * group of m*128 rows keeps its first ceil(m/2)*128 rows in (projection, row index) order
 * as its first half. perm receives per head the groups in depth-first order, each group's
 * rows ascending: group g = perm[(b*H+h)*N + g*128 .. +127] (the layout of
 * bsa_select_tokens and bsa_forward_tokens).
 *
 *   Q           device [B][H][N][d], dtype dt; N a multiple of 128, N/128 <= 512, B*H <= 65535
 *   perm        device int32 [B*H][N] (written)
 *   workspace   device, >= bsa_workspace_size(4, ...) bytes (it depends on d), 256-byte aligned
 * The principal direction comes from fp32 power iteration (32 steps from a fixed start) on
 * the segment's centred scatter matrix, so a row lying within rounding of a median may land
 * on the other side than an exact eigendecomposition would put it. Every sum runs in a
 * fixed order: the same Q gives the same groups. Errors: BSA_ERR_SHAPE, BSA_ERR_DTYPE,
 * BSA_ERR_INVALID_ARG, BSA_ERR_WORKSPACE; device-raised BSA_ERR_TIMEOUT (a bounded wait of the
 * tensor-core pass gave up). The split tree runs level by level: the row sums, scatter
 * matrices and projections over slices of at most 512 rows of each segment, the power
 * iteration and the cut over one CTA per segment. The scatter matrices of bf16 queries at
 * d = 128 run on tcgen05 as uncentred sums (the mean term taken off per segment, which loses
 * accuracy when a segment's mean is large against its spread); fp32 and d = 64 run centred
 * on CUDA cores.
 */
bsa_status bsa_query_groups(const void *Q, int dt, int B, int H, int N, int d, int32_t *perm, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * bsa_select_tokens -- the token oracle's selection for token-sparse attention ("Can
 * sparse attention close the quality gap in diffusion transformers", sections
 * "质量差距有三个可分离来源" and "token 级选择需要瓦片对齐的查询分组").
 *
 * For each (b, h) and group g = rows perm[g*128 .. g*128+127]:
 *   mass[g][t] = sum over rows r of g of exp(scale * q_r . k_t - LSE_r),  t = 0..N-1,
 * and the group keeps the K = max(1, floor(density * N)) tokens of largest mass (ties to
 * the lower index), written ascending to tokens[(b*H+h)*(N/128) + g][0..K-1].
 *
 *   Q, K        device [B][H][N][d], dtype dt; N a multiple of 128
 *   perm        device int32 [B*H][N]: per head a permutation of 0..N-1 (the groups)
 *   LSE         device fp32 [B][H][N]: the dense logsumexp (natural log), e.g. bsa_forward
 *               over a full index
 *   density     in (0, 1]; scale <= 0 selects 1/sqrt(d)
 *   tokens      device int32, capacity >= B*H*(N/128)*K entries
 *   workspace   device, >= bsa_workspace_size(3, ...) bytes, 256-byte aligned; after the call
 *               it holds the masses fp32 [B*H*N/128][N] at byte offset 256
 * Errors: BSA_ERR_SHAPE (N not a multiple of 128, d, B*H > 65535; for fp32 also N too
 * large for its shared-memory row of N keys), BSA_ERR_DTYPE, BSA_ERR_INVALID_ARG,
 * BSA_ERR_CAPACITY, BSA_ERR_WORKSPACE; device-raised: BSA_ERR_INVALID_ARG (perm index
 * outside [0, N), skipped), BSA_ERR_NONFINITE (a NaN mass).
 * bf16: the masses run on tcgen05 as K_chunk Q_g^T (one thread per key sums its mass over
 * the group's 128 queries), then an exact 8-bit radix top-K per group reads them from the
 * workspace (any N). fp32: CUDA cores.
 */
bsa_status bsa_select_tokens(const void *Q, const void *K, int dt, int B, int H, int N, int d, const int32_t *perm,
                             const float *LSE, float density, float scale, int32_t *tokens, int64_t tokens_capacity,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Host-only: the tokens each query group keeps in bsa_select_tokens ("Can sparse attention
 * close the quality gap in diffusion transformers", section "质量差距有三个可分离来源": the
 * token oracle keeps a fixed share of the keys), K = max(1, floor(density * N)) with density
 * as given (fp32) and the product in double, at most N. Sizes the tokens buffer
 * (B*H*(N/128)*K entries). Errors: BSA_ERR_INVALID_ARG (null out, density outside (0, 1]),
 * BSA_ERR_SHAPE (N <= 0). */
bsa_status bsa_tokens_per_group(int N, float density, int *n_tokens);

/*
 * bsa_forward_tokens -- token-sparse attention over tile-aligned query groups
 * ("Can sparse attention close the quality gap in diffusion transformers", section
 * "token 级选择需要瓦片对齐的查询分组": groups of 128 similar queries share one set of
 * individually selected KV tokens, gathered by index).
 *
 * For each (b, h), group g = rows perm[g*128 .. g*128+127] of the head, and every row r
 * of the group:
 *   O_r = sum_t softmax_t(scale * q_r . k_t) v_t,  LSE_r = ln sum_t exp(scale * q_r . k_t),
 *   t over tokens[g][0 .. n_tokens-1].
 *
 *   Q, K, V     device [B][H][N][d], dtype dt; N a multiple of 128
 *   perm        device int32 [B*H][N]: per head a permutation of 0..N-1 (the groups)
 *   tokens      device int32 [B*H][N/128][n_tokens]: each group's key tokens in [0, N)
 *   n_tokens    keys per group, 1..N
 *   scale       softmax scale; <= 0 selects 1/sqrt(d)
 *   O, LSE      as bsa_forward (written for every row that perm names)
 *   workspace   device, >= 256 bytes, 256-byte aligned (its first bytes hold the
 *               device error word, read by bsa_check_device_error)
 * Errors: BSA_ERR_SHAPE (N not a multiple of 128, d, B*H > 65535), BSA_ERR_DTYPE, BSA_ERR_INVALID_ARG
 * (null or misaligned pointers, n_tokens out of range, non-finite scale),
 * BSA_ERR_WORKSPACE. An index outside [0, N) in perm or tokens raises BSA_ERR_INVALID_ARG in
 * the workspace (the row or key is then not computed as asked: the results are undefined).
 * bf16 runs on tcgen05: a 128-query group is one tile (its query rows gathered by TMA
 * tile::gather4), its keys arrive 128 per step with the K and V rows copied by index
 * (cp.async), the last step masked. fp32 runs on CUDA cores.
 */
bsa_status bsa_forward_tokens(const void *Q, const void *K, const void *V, int dt, int B, int H, int N, int d,
                              const int32_t *perm, const int32_t *tokens, int n_tokens, float scale, void *O,
                              float *LSE, void *workspace, size_t workspace_bytes, void *stream);

/*
 * bsa_build_mask_noalloc -- bsa_build_mask without a caller workspace (the pages
 * have no counterpart: this is a convenience of this library).
 *
 * For callers that cannot allocate device memory: code under a framework that
 * owns all device memory from start-up on, or a process whose device-memory
 * budget is frozen once it serves. The scratch comes from a fixed array of
 * BSA_NOALLOC_SCRATCH_BYTES in the library's device memory; every GPU that loads
 * the library holds it until the process exits. Arguments and results are those
 * of bsa_build_mask, minus the workspace; the call allocates and frees nothing.
 *
 *   device_status  optional device uint32 (NULL = not wanted): receives, in stream
 *                  order at the end of the call, the device-raised status of this
 *                  build (BSA_OK, BSA_ERR_NONFINITE or BSA_ERR_CAPACITY).
 *
 * Every argument check of bsa_build_mask runs before anything is enqueued: a
 * call that returns an error has enqueued no work. Returns BSA_ERR_WORKSPACE,
 * before any launch, when the problem needs more scratch than the array holds:
 * a dynamic build needs the pooled blocks (about 2 * B*H*nB*d*4 bytes), a static
 * one only per-row counts and one head's pattern (about B*H*nB*4 + nB*(nB/8)
 * bytes). The first call on a device looks up the array's
 * device address (once per device, with that device current): make that first
 * call before any stream capture. All calls share the one array: calls whose
 * work overlaps on the GPU (different streams without ordering, or different
 * host threads) race on it and must be serialised by the caller.
 */
#define BSA_NOALLOC_SCRATCH_BYTES (16u << 20)
bsa_status bsa_build_mask_noalloc(const void *Q, const void *K, int dt, int B, int H, int N, int d,
                                  int block, float density, const bsa_static_spec *spec,
                                  int32_t *row_ptr, int32_t *col_idx, int64_t col_capacity,
                                  uint32_t *bitmap, uint32_t *device_status, void *stream);

/* Host-only: number of active blocks the builder will emit for these arguments.
 * Dynamic: B*H*nQB*k. MODALITY_BAND / CUBOID: exact count times B*H.
 * EXPLICIT: the bitmap lives on the device, so the upper bound B*H*nQB*nKB. */
bsa_status bsa_mask_nnz(int B, int H, int N, int block, float density,
                        const bsa_static_spec *spec, int64_t *nnz);

/* Host-only: workspace bytes for which = 0 (bsa_build_mask, bsa_build_mask_modal),
 * 1 (bsa_forward, bsa_forward_residual), 2 (bsa_build_mask_exact), 3 (bsa_select_tokens) or
 * 4 (bsa_query_groups); for 3 and 4 N is a multiple of 128 and block any valid value. */
bsa_status bsa_workspace_size(int which, int B, int H, int N, int d, int block, size_t *bytes);

/* Synchronises `stream`, returns the device-raised status recorded in `workspace`
 * by earlier calls (BSA_OK if none), and clears it. */
bsa_status bsa_check_device_error(void *workspace, void *stream);

/* Checks an index on the device: row_ptr[0] == 0 and non-decreasing, col_idx
 * strictly ascending within each row and < nKB, and (when bitmap != NULL) each
 * row's bitmap popcount equals its CSR length with the same bits. A violation is
 * recorded as BSA_ERR_INVALID_ARG in `workspace` (read it with
 * bsa_check_device_error). */
bsa_status bsa_validate_index(int B, int H, int N, int block, const int32_t *row_ptr,
                              const int32_t *col_idx, const uint32_t *bitmap, void *workspace,
                              size_t workspace_bytes, void *stream);

/* Diagnostics for tests: `flags` bit 0 makes the next bsa_forward launches skip
 * their loads and MMAs so the softmax warps' first wait runs out (nothing is in
 * flight); bit 1 keeps every query tile whole and bit 2 splits every tile with two
 * or more KV steps over several CTAs (as far as the workspace's partial slots
 * allow), overriding the load-balance rule that splits only tiles above the
 * per-CTA share of steps; `wait_limit_ns` bounds every device wait (0 restores
 * the default of 2 s). Host-global; not thread safe. */
bsa_status bsa_debug_config(uint32_t flags, uint64_t wait_limit_ns);

/* Static string for a status code. */
const char *bsa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H_ */
