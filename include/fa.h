/*
 * fa.h -- C ABI of block_sparse_masked_fa_gb300: exact softmax attention whose
 * mask is summarised at tile level, for one NVIDIA GB300 (sm_103a).
 *
 * The method (speedrun notes "FlexAttention", Context paragraph and the
 * tile-summary paragraph after the mask_mod code block; tutorial "FlexAttention
 * in PyTorch: Custom and Sparse Attention Without Writing Kernels", section
 * "The two hooks: score_mod and mask_mod"): a boolean mask_mod decides which
 * (query, key) pairs are visible; a builder summarises it over BLOCK x BLOCK
 * tiles into, per query-tile row, the count and column indices of the tiles
 * that are not fully masked; the attention kernels loop over those lists only,
 * skip the mask on fully visible tiles, apply it element by element on partial
 * ones, and let an optional score_mod edit every surviving logit.
 *
 * Conventions for every call:
 *  - Tensors are device pointers into caller-owned memory; the library never
 *    allocates, frees or keeps a pointer after a call returns (the block mask
 *    descriptor keeps pointers into the caller's block-mask buffer).
 *  - q, out, dq, dO are bf16 [B, H, q_len, D]; k, v, dk, dv are bf16
 *    [B, H, kv_len, D]; lse is fp32 [B, H, q_len]; all contiguous, row-major,
 *    16-byte aligned.
 *  - Every call is asynchronous on `stream` (no host synchronisation) except
 *    fa_get_status and fa_block_mask_summary, which synchronise the stream.
 *  - Errors that the host can see (null pointers, bad shapes, unsupported
 *    head dims, misalignment, buffers too small) are returned before any GPU
 *    work is queued.  Errors that only the device sees (a bounded wait that
 *    gave up) set bits in the block mask's device status word; read them with
 *    fa_get_status.  Nothing traps.  No C++ exception crosses this boundary.
 */
#ifndef BLOCK_SPARSE_MASKED_FA_GB300_FA_H
#define BLOCK_SPARSE_MASKED_FA_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, unknown enum value, malformed mask program */
  FA_ERR_UNSUPPORTED = 2,  /* well-formed but not implemented (head dim, block size)   */
  FA_ERR_SHAPE = 3,        /* sizes out of range or inconsistent with the block mask    */
  FA_ERR_ALIGNMENT = 4,    /* a pointer is not 16-byte aligned                          */
  FA_ERR_CUDA = 5,         /* a CUDA runtime or driver call failed                      */
  FA_ERR_TIMEOUT = 6,      /* device: a bounded wait inside a kernel gave up            */
  FA_ERR_DEVICE_CHECK = 7, /* device: a range check inside a kernel failed              */
  FA_ERR_WORKSPACE = 8     /* a caller-provided buffer is smaller than required         */
} fa_status;

/* ------------------------------------------------------------------------
 * Mask programs (mask_mod as a fixed, parameterised set).
 *
 * A program is up to FA_MAX_MASK_NODES nodes in postfix order; atoms push one
 * predicate of (b, q_idx, kv_idx), FA_M_AND / FA_M_OR pop two and push one
 * (tutorial, Pattern 3: compose with and_masks / or_masks).  The stack never
 * holds more than FA_MAX_MASK_STACK values.  Parameters live in DEVICE memory
 * so that they can change between calls without rebuilding anything (speedrun
 * notes, Record #13: the window is read from a tensor):
 *
 *   FA_M_TRUE      every pair visible                       param: NULL
 *   FA_M_CAUSAL    q_idx >= kv_idx                          param: NULL
 *                  (speedrun notes, mask_mod code; tutorial, "The two hooks")
 *   FA_M_SAME_DOC  doc[b][q_idx] == doc[b][kv_idx]          param: int32 doc ids
 *                  [Bm][doc_len], e.g. the inclusive cumsum of end-of-text flags
 *                  (speedrun notes, mask_mod code; tutorial, Pattern 1).  Every
 *                  SAME_DOC node of one program must use the same array.
 *   FA_M_WINDOW    q_idx - kv_idx < W                       param: int32 W (1 value)
 *                  (speedrun notes, mask_mod code; tutorial, Pattern 2).  No
 *                  lower bound: combine with FA_M_CAUSAL for a causal window.
 *   FA_M_SINK      kv_idx < n_sink                          param: int32 n_sink (1 value)
 *                  (tutorial, Pattern 2)
 *   FA_M_PREFIX    kv_idx < prefix_len[b]                   param: int32 [Bm]
 *                  (prefix-LM, named in the tutorial's introduction; the usual
 *                  form is FA_M_CAUSAL OR FA_M_PREFIX)
 * ---------------------------------------------------------------------- */
#define FA_MAX_MASK_NODES 16
#define FA_MAX_MASK_STACK 8

typedef enum {
  FA_M_TRUE = 0,
  FA_M_CAUSAL = 1,
  FA_M_SAME_DOC = 2,
  FA_M_WINDOW = 3,
  FA_M_SINK = 4,
  FA_M_PREFIX = 5,
  FA_M_AND = 6,
  FA_M_OR = 7
} fa_mask_op;

typedef struct {
  int32_t op;           /* fa_mask_op                      */
  const int32_t* param; /* device pointer, see the table   */
} fa_mask_node;

typedef struct {
  int32_t n;         /* number of nodes, 1..FA_MAX_MASK_NODES                    */
  int64_t doc_len;   /* row length (elements) of the SAME_DOC array; must be
                        >= max(q_len, kv_len) when SAME_DOC is used, else 0     */
  fa_mask_node node[FA_MAX_MASK_NODES];
  /* Position of query row 0 in the sequence the program describes: query row i
   * is position i + q_offset for CAUSAL, WINDOW and SAME_DOC (and for ALiBi's
   * i - j), key j is position j.  0 for training shapes; kv_len - q_len when
   * the queries are the newest tokens of a cache (tutorial "Decoding and paged
   * KV caches": a mask built for training shapes is wrong during generation).
   * Must lie in [0, max(q_len, kv_len) - q_len] (FA_ERR_INVALID_ARG). */
  int64_t q_offset;
} fa_mask_spec;

/* ------------------------------------------------------------------------
 * Score mods (score_mod as a fixed set; tutorial, Pattern 3).  The score that
 * a score_mod sees is the scaled logit x = scale * (q . k).
 *   FA_S_NONE     s = x                                 param: NULL
 *   FA_S_SOFTCAP  s = c * tanh(x / c)                   param: device fp32 c (1 value), c > 0
 *   FA_S_ALIBI    s = x - slope[h] * (q_idx - kv_idx)   param: device fp32 slopes [H]
 *   FA_S_RELBIAS  s = x + bias[h][t],                   param: device fp32 table [H][bias_len]
 *                 t = clamp(q_idx - kv_idx - bias_d0, 0, bias_len - 1)
 * FA_S_RELBIAS is a learned relative-position bias (Pattern 3: "a learned
 * relative-position bias trains"): one entry per query-minus-key distance from
 * bias_d0 to bias_d0 + bias_len - 1, distances outside that range taking the
 * nearest end entry.  q_idx is the query's position (row + the mask program's
 * q_offset), as for ALiBi and the mask atoms.
 * ---------------------------------------------------------------------- */
typedef enum { FA_S_NONE = 0, FA_S_SOFTCAP = 1, FA_S_ALIBI = 2, FA_S_RELBIAS = 3 } fa_score_op;

typedef struct {
  int32_t op;          /* fa_score_op */
  const float* param;  /* device pointer, see the table */
  /* fa_backward / fa_backward_noalloc only (fa_forward ignores it): the
   * gradient of L = sum(out * dO) with respect to the score mod's learned
   * parameter (tutorial Pattern 3: a learned relative-position bias trains
   * through the fused backward), overwritten, not accumulated -- device fp32
   * [H] receiving dL/dslope[h] for FA_S_ALIBI, or [H][bias_len] receiving
   * dL/dbias[h][t] for FA_S_RELBIAS; or NULL for no parameter gradient.
   * Non-NULL with another op: FA_ERR_UNSUPPORTED (the soft-cap constant is not
   * a learned parameter on the pages). */
  float* param_grad;
  /* FA_S_RELBIAS only: the table's length per head, in [1, 2^24]
   * (FA_ERR_INVALID_ARG otherwise), and the distance of its entry 0, in
   * [-2^30, 2^30]. */
  int32_t bias_len;
  int32_t bias_d0;
} fa_score_spec;

/* ------------------------------------------------------------------------
 * Block mask (the tile summary of a mask program).
 *
 * Tile (I, J) covers query rows [I*block, (I+1)*block) and key rows
 * [J*block, (J+1)*block), cut at q_len / kv_len.  Its class is EMPTY when no
 * in-range pair is visible, FULL when every one is, PARTIAL otherwise
 * (tutorial, "The two hooks": empty / partially masked / full blocks).
 *
 *   kv_num_blocks      int32 [Bm][Hm][nq]        PARTIAL tiles of each query-tile row
 *   kv_indices         int32 [Bm][Hm][nq][nkv]   their J, ascending, zero padded
 *   full_kv_num_blocks int32 [Bm][Hm][nq]        FULL tiles of each row
 *   full_kv_indices    int32 [Bm][Hm][nq][nkv]   their J, ascending, zero padded
 *   q_num_blocks, q_indices, full_q_num_blocks, full_q_indices:
 *                      the same per key-tile column ([..][nkv], [..][nkv][nq]),
 *                      used by the backward.
 *   row_order, col_order: rows / columns sorted by descending tile count (the
 *                      order the attention kernels take their work in).
 *   tile_class         uint8 [Bm][Hm][nq][nkv]: 0 EMPTY, 1 PARTIAL, 2 FULL.
 *   doc_runs           int32 [Bm][max(q_len, kv_len)][2] then int32 [Bm]: for
 *                      every position the run [lo, hi) of neighbouring positions
 *                      with the same document id, and per batch row a flag set
 *                      when the ids never decrease (then doc[i] == doc[j] iff j
 *                      lies in i's run, which the kernels use on PARTIAL tiles).
 *                      Filled only when the program has SAME_DOC.
 *   row_segs           int32 [Bm][2][max(q_len, kv_len)][4]: for every query
 *                      row i ([bm][0][i]) the key columns it sees, and for
 *                      every key column j ([bm][1][j]) the query rows that see
 *                      it, as two intervals [lo0, hi0) and [lo1, hi1) (empty
 *                      when lo == hi) -- or lo0 = -1 where that does not
 *                      describe the row (more pieces, or document ids that
 *                      decrease somewhere).  The attention kernels build their
 *                      PARTIAL tiles' mask words from it, and evaluate the
 *                      program per element where lo0 = -1.
 *   status             device status word (bit 0: a wait timed out; bit 1: a
 *                      device check failed, e.g. invalid caller tile lists).
 *
 * With block < 128 (tutorial, sharp edge 4: a smaller BLOCK_SIZE captures more
 * of a fine-grained mask's sparsity) the attention kernels still multiply
 * 128-row query tiles; the builder also derives, from tile_class, the coarser
 * tiles they walk (a coarse tile is EMPTY when all of its block tiles are, FULL
 * when all are, PARTIAL otherwise -- exact):
 *   fwd_*              the forward's: per query tile of 128 rows (fwd_nq rows)
 *                      the key tiles of fwd_kv_block = 64 columns (fwd_nkv)
 *                      that are not EMPTY -- counts [Bm][Hm][fwd_nq], indices
 *                      [Bm][Hm][fwd_nq][fwd_nkv], PARTIAL and FULL as above --
 *                      with fwd_row_order and the classes fwd_tile_class;
 *   bwd_*              the backward's: per key tile of 128 columns (bwd_nkv)
 *                      the query tiles of 128 rows (bwd_nq), [Bm][Hm][bwd_nkv]
 *                      and [Bm][Hm][bwd_nkv][bwd_nq], with bwd_col_order and
 *                      bwd_tile_class.
 * At block == 128 these pointers are NULL and the kernels walk the lists above.
 * from_blocks is 1 for a block mask of caller-chosen tiles
 * (fa_block_mask_from_kv_blocks); the attention kernels take those at block
 * 128 only.
 *
 * The union kv_num_blocks + full_kv_num_blocks is the count of "tiles that are
 * not fully masked" of the speedrun notes' tile-summary paragraph.  Bm is 1 or
 * B and Hm is 1 or H: a size of 1 is broadcast over that dimension (tutorial,
 * B=None / H=None).  All pointers point into one caller-owned device buffer of
 * fa_block_mask_bytes() bytes; `spec` is a copy of the mask program, which the
 * attention kernels evaluate on PARTIAL tiles.  Rebuild the block mask when
 * any mask parameter changes; the kernels need no rebuild.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t Bm, Hm, block, nq, nkv;
  int64_t q_len, kv_len;
  int32_t* kv_num_blocks;
  int32_t* kv_indices;
  int32_t* full_kv_num_blocks;
  int32_t* full_kv_indices;
  int32_t* q_num_blocks;
  int32_t* q_indices;
  int32_t* full_q_num_blocks;
  int32_t* full_q_indices;
  int32_t* row_order;
  int32_t* col_order;
  uint8_t* tile_class;
  int32_t* tile_summary;
  int32_t* doc_runs;
  int32_t* row_segs;
  uint32_t* status;
  fa_mask_spec spec;
  int32_t from_blocks;
  int32_t fwd_kv_block, fwd_nq, fwd_nkv, bwd_nq, bwd_nkv;
  int32_t* fwd_kv_num_blocks;
  int32_t* fwd_kv_indices;
  int32_t* fwd_full_kv_num_blocks;
  int32_t* fwd_full_kv_indices;
  int32_t* fwd_row_order;
  uint8_t* fwd_tile_class;
  int32_t* bwd_q_num_blocks;
  int32_t* bwd_q_indices;
  int32_t* bwd_full_q_num_blocks;
  int32_t* bwd_full_q_indices;
  int32_t* bwd_col_order;
  uint8_t* bwd_tile_class;
} fa_block_mask;

/* Bytes of device memory a block mask of this shape needs.
 * block: a power of two in [16, 128].  Returns FA_ERR_SHAPE for non-positive
 * sizes or more than 2^31 tiles. */
fa_status fa_block_mask_bytes(int32_t Bm, int32_t Hm, int64_t q_len, int64_t kv_len, int32_t block,
                              size_t* bytes);

/* Builds the block mask of `spec` (speedrun notes, tile-summary paragraph:
 * create_block_mask evaluates mask_mod over the index grid and stores per
 * query-tile row the count and the column indices of the non-empty tiles).
 * buffer: device memory of at least fa_block_mask_bytes() bytes, 256-byte
 * aligned, owned by the caller and used until the block mask is dropped.
 * bm: host struct, filled with pointers into `buffer` and a copy of `spec`.
 * Queues 4-6 kernels on `stream` (4 more with block < 128, for the attention
 * kernels' coarser tiles); clears the status word. */
fa_status fa_create_block_mask(const fa_mask_spec* spec, int32_t Bm, int32_t Hm, int64_t q_len, int64_t kv_len,
                               int32_t block, void* buffer, size_t buffer_bytes, fa_block_mask* bm,
                               cudaStream_t stream);

/* Builds a block mask from caller-chosen tiles instead of a program's tile
 * classes (tutorial "FlexAttention in PyTorch": sparse patterns that attend
 * only to a selected subset of blocks; "Decoding and paged KV caches":
 * BlockMask.from_kv_blocks).  The visible pairs are every in-range pair of a
 * tile listed as FULL, and the pairs of a tile listed as PARTIAL where `spec`
 * holds; nothing else.
 *   kv_num_blocks       device int32 [Bm][Hm][nq]              PARTIAL tiles per query-tile row
 *   kv_indices          device int32 [Bm][Hm][nq][idx_stride]  their J, in any order
 *   full_kv_num_blocks, full_kv_indices: the same for FULL tiles; both NULL for none
 *   idx_stride          row length of the index arrays, >= 1 (nkv for the lists
 *                       of another fa_block_mask); entries past a row's count
 *                       are not read
 *   spec                mask program applied on PARTIAL tiles, or NULL: every
 *                       pair of a PARTIAL tile is visible (one FA_M_TRUE node)
 * The caller's lists are only read, by the first kernel; they may be freed or
 * reused once it has run (stream order).  The block mask's own lists are
 * rebuilt from them: ascending, zero padded, with the per-column lists and
 * work orders of fa_create_block_mask.  The lists are checked on the device:
 * a count outside [0, min(nkv, idx_stride)] (clamped), an index outside
 * [0, nkv) (dropped) or a tile listed twice (a tile in both lists stays FULL)
 * sets the status word's check bit, which fa_get_status reports as
 * FA_ERR_DEVICE_CHECK.  Other arguments and errors as fa_create_block_mask;
 * the pointers must be 4-byte aligned (FA_ERR_ALIGNMENT). */
fa_status fa_block_mask_from_kv_blocks(const int32_t* kv_num_blocks, const int32_t* kv_indices,
                                       const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                                       int32_t idx_stride, const fa_mask_spec* spec, int32_t Bm, int32_t Hm,
                                       int64_t q_len, int64_t kv_len, int32_t block, void* buffer,
                                       size_t buffer_bytes, fa_block_mask* bm, cudaStream_t stream);

/* Forward: out and LSE (speedrun notes, Context: the two matmuls and the
 * softmax fused in one tiled kernel that never writes the score matrix; the
 * kernel visits only the listed tiles).
 *   out_i = sum_{j visible} softmax_j(s_i) v_j,  LSE_i = ln sum_{j visible} exp(s_ij)
 * with s_ij = score_mod(scale * q_i . k_j).  A row with no visible key gets
 * out = 0 and LSE = -inf.  scale: > 0, or 0 for 1/sqrt(D).
 * D: 64 or 128.  bm: built for this q_len / kv_len with any block (below 128
 * the kernel walks 128 x 64 tiles, see fa_block_mask; caller-chosen tiles only
 * at block 128, else FA_ERR_UNSUPPORTED), Bm in {1, B}, Hm in {1, H}. */
fa_status fa_forward(const void* q, const void* k, const void* v, int32_t B, int32_t H, int64_t q_len,
                     int64_t kv_len, int32_t D, const fa_block_mask* bm, const fa_score_spec* score, float scale,
                     void* out, float* lse, cudaStream_t stream);

/* Forward over a paged key / value cache (tutorial "FlexAttention in
 * PyTorch", "Decoding and paged KV caches": the logical tile indices go
 * through a page table to physical blocks, so any mask works on a paged cache
 * without a kernel per variant).  Computes exactly what fa_forward computes on
 * the logical keys and values
 *   k[b][h][j] = k_pool[h][128 * page_table[b][j / 128] + j % 128]   (v alike).
 *   k_pool, v_pool  bf16 [H][n_pages * 128][D], 16-byte aligned; a page holds
 *                   128 rows of every head
 *   page_table      device int32 [B][bm->nkv]: page of each logical key tile,
 *                   4-byte aligned; a page may serve several tiles or batch rows
 *   n_pages         pages in the pools, 1 .. (2^31 - 1) / 128
 * The block mask is built on logical positions (q_len, kv_len).  Rows of the
 * last key tile's page past kv_len are read and masked out; they must hold
 * finite values (their weight is 0, but 0 * NaN is NaN).  A page index outside
 * [0, n_pages) sets the status word's check bit (FA_ERR_DEVICE_CHECK from
 * fa_get_status) and page 0 is read in its place.  Other arguments, results
 * and errors as fa_forward; there is no paged backward. */
fa_status fa_forward_paged(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                           int32_t n_pages, int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                           const fa_block_mask* bm, const fa_score_spec* score, float scale, void* out, float* lse,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Short-query forward (tutorial "FlexAttention in PyTorch", "Decoding and
 * paged KV caches": a dedicated decoding path optimised for short queries).
 * Computes what fa_forward or fa_forward_paged computes, for q_len up to
 * FA_DECODE_MAX_Q, with the listed key tiles of every (b, h) split over
 * several CTAs and the shares merged by their LSE.
 * ---------------------------------------------------------------------- */
#define FA_DECODE_MAX_Q 16

/* Workspace fa_forward_decode needs on the current device (fp32 partial
 * results of every share: splits * B * H * q_len * (D + 1) floats).
 * q_len in [1, FA_DECODE_MAX_Q], D 64 or 128 and B * H <= 65535 (else
 * FA_ERR_UNSUPPORTED). */
fa_status fa_forward_decode_workspace_bytes(int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                                            size_t* bytes);

/* The short-query forward: out and LSE exactly as fa_forward (page_table =
 * NULL) or fa_forward_paged (page_table != NULL, k / v pools
 * [H][n_pages * 128][D]) define them, for q_len <= FA_DECODE_MAX_Q (bm built
 * for this q_len, so nq = 1), over the keys [0, kv_len).  Keys past kv_len are
 * never read.
 * Bucketed caches (tutorial "Decoding and paged KV caches": keep the cache
 * length bucketed, e.g. to multiples of 1024, and reuse the block mask): bm
 * may be built for a longer key length C = bm->kv_len >= kv_len, once per
 * bucket; key tiles it lists past kv_len are skipped, and the visible set is
 * the mask's restricted to j < kv_len.  Without a page table k / v are
 * [B][H][C][D] (rows past kv_len unused); with one, page_table is [B][bm->nkv]
 * and only the entries of tiles below kv_len are read.
 * workspace: device memory of fa_forward_decode_workspace_bytes() bytes,
 * 16-byte aligned, caller-owned (FA_ERR_WORKSPACE when smaller).  Queues two
 * kernels on `stream`; errors as fa_forward / fa_forward_paged. */
fa_status fa_forward_decode(const void* q, const void* k, const void* v, const int32_t* page_table, int32_t n_pages,
                            int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D, const fa_block_mask* bm,
                            const fa_score_spec* score, float scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/* Device workspace fa_backward needs: an fp32 dq accumulator
 * (B*H*q_len*D floats), per 128-row query tile the rows' LSE and
 * sum(dO * out) (B*H*ceil(q_len/128)*256 floats), and a work counter (one
 * uint32), each 256-byte aligned. */
fa_status fa_backward_workspace_bytes(int32_t B, int32_t H, int64_t q_len, int32_t D, size_t* bytes);

/* Backward: dq, dk, dv of L = sum(out * dO) (tutorial, Pattern 3: the
 * score mods are differentiable and the backward is fused).  out and lse are
 * the forward's results for the same inputs.  dk and dv are written once per
 * key tile (no atomics); dq is accumulated in fp32 in `workspace` and then
 * converted.  Same shape rules as fa_forward. */
fa_status fa_backward(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                      const fa_block_mask* bm, const fa_score_spec* score, float scale, void* dq, void* dk,
                      void* dv, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * A forward that prepares the backward's workspace, and the backward that
 * takes it prepared.  fa_forward_prepare_backward computes exactly what
 * fa_forward computes; while it runs, its producer warps also set the
 * workspace's fp32 dq accumulator (its first B*H*q_len*D*4 bytes) to zero, in
 * bulk copies beside the K / V loads -- work the backward's preprocessing
 * kernel otherwise does, at half of its memory traffic.  fa_backward_prepared
 * is fa_backward for such a workspace: it takes the accumulator as zero.  The
 * pair must see the same B, H, q_len and D, and nothing else may use the
 * workspace between them (a second fa_backward_prepared on it would add into a
 * spent accumulator: call fa_backward, which clears it, instead).
 * workspace: device, 16-byte aligned, >= fa_backward_workspace_bytes(B, H,
 * q_len, D) (FA_ERR_WORKSPACE); other arguments and errors as fa_forward /
 * fa_backward.  Asynchronous on the stream.
 * ---------------------------------------------------------------------- */
fa_status fa_forward_prepare_backward(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                                      int64_t q_len, int64_t kv_len, int32_t D, const fa_block_mask* bm,
                                      const fa_score_spec* score, float scale, void* out, float* lse,
                                      void* workspace, size_t workspace_bytes, cudaStream_t stream);
fa_status fa_backward_prepared(const void* q, const void* k, const void* v, const void* out, const float* lse,
                               const void* dout, int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                               const fa_block_mask* bm, const fa_score_spec* score, float scale, void* dq, void* dk,
                               void* dv, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Backward without a caller-provided workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory when they call the backward -- for example code running
 * inside a framework that reserves the GPU's memory for its own pool at start
 * up and allows no further cudaMalloc, or a latency-critical path that cannot
 * afford the implicit device synchronisation of an allocation.
 *
 * It computes exactly what fa_backward computes, with the same arguments
 * except the workspace: the fp32 dq accumulator and the per-row
 * sum(dO * out) live in a static device array of FA_NOALLOC_SCRATCH_BYTES
 * owned by the library.  Every GPU that loads the library holds that array
 * until the process exits.  The caller still passes (and owns) every input
 * and output.  The call allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.
 *  - Size limit: returns FA_ERR_WORKSPACE, before any GPU work, when
 *    fa_backward_workspace_bytes(B, H, q_len, D) exceeds
 *    FA_NOALLOC_SCRATCH_BYTES (16 MiB: e.g. B*H*q_len up to about 32,000
 *    rows at D = 128 or 63,000 rows at D = 64).
 *  - Set-up: the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make that
 *    first call before any stream capture.  The cached address belongs to the
 *    device's context: after cudaDeviceReset (or any loss of the primary
 *    context) it is stale, so a device that was reset must not be used with
 *    this entry point again in the same process.
 *  - Sharing: all calls on a device use the same array, which keeps the last
 *    call's contents; each call re-initialises the part it uses.  Calls whose
 *    GPU work overlaps (different streams, no ordering between them) race on
 *    the array and give wrong gradients: order them on one stream or with
 *    events. */
#define FA_NOALLOC_SCRATCH_BYTES (16u << 20)
fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* out, const float* lse,
                              const void* dout, int32_t B, int32_t H, int64_t q_len, int64_t kv_len, int32_t D,
                              const fa_block_mask* bm, const fa_score_spec* score, float scale, void* dq,
                              void* dk, void* dv, cudaStream_t stream);

/* Synchronises `stream`, reads the block mask's device status word and
 * returns FA_OK, FA_ERR_TIMEOUT or FA_ERR_DEVICE_CHECK.  clear != 0 resets the
 * word to 0. */
fa_status fa_get_status(const fa_block_mask* bm, int32_t clear, cudaStream_t stream);

/* Synchronises `stream` and counts EMPTY, PARTIAL and FULL tiles over the
 * whole [Bm][Hm][nq][nkv] grid into counts[0..2] (host memory) -- the numbers
 * behind the tutorial's sparsity map (sharp edge 6). */
fa_status fa_block_mask_summary(const fa_block_mask* bm, int64_t counts[3], cudaStream_t stream);

/* Static description of a status code. */
const char* fa_status_string(fa_status status);

/* Library ABI version (major * 100 + minor). */
int32_t fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BLOCK_SPARSE_MASKED_FA_GB300_FA_H */
