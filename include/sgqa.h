/*
 * sgqa.h -- C ABI of the GB300 (sm_103a) block-wise Sparse GQA prefill library.
 *
 * The method is the Sparse GQA layer of "Inside Step 5 Preview: Architecture
 * and Training for Agentic Work" (StepFun blog), section "Sparse GQA":
 *   - "Reducing indexer's cost": the index keys of B adjacent historical
 *     positions are compressed into one block representation (B = 8), which
 *     cuts indexer and top-k cost by B;
 *   - "Efficient implementation of sparse attention": the top-k results of
 *     adjacent tokens are unioned so that their overlapping work is batched;
 *   - "Trade-off between top-k and block size": k = 4096 tokens, i.e.
 *     k / B = 512 selected historical blocks;
 *   - Figure 3 caption: each KV group selects history independently, and the
 *     main path reads the selected historical blocks plus the causally
 *     visible positions of the current block.
 *
 * Readings fixed by this library where the pages are silent: the block
 * representation is the mean of the block's keys (fp32, summed as a fixed
 * pairwise tree); the indexer score of query t against block j of KV group g
 * is the dot product of the group's mean query with the block mean (no
 * scale); only complete blocks strictly before the query's own block are
 * candidates; ties go to the lower block index; query head h belongs to KV
 * group h / G with G = n_q_heads / n_kv_heads.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, allocated and owned by the
 *     caller.  The library never allocates, frees or synchronises (except
 *     sgqa_read_status, which synchronises the given stream by design); all
 *     work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *   - `status` is a caller-owned device buffer of 4 int32 (16 bytes) that the
 *     caller zeroes (sgqa_reset_status).  Kernels record the first
 *     device-side error there (SGQA_ERR_CAPACITY, SGQA_ERR_TIMEOUT,
 *     SGQA_ERR_BOUNDS) with a detail word; outputs are undefined after one.
 *     Word 0 = code, word 1 = detail (the place that reported it), word 2 =
 *     count of errors, word 3 = debug request (0 in normal use; see
 *     SGQA_DEBUG_STALL).
 *   - The return value reports host-side validation (SGQA_ERR_INVALID_ARG,
 *     SGQA_ERR_UNSUPPORTED, SGQA_ERR_ALIGNMENT, SGQA_ERR_WORKSPACE) and
 *     launch failures (SGQA_ERR_CUDA); nothing is enqueued when it is not
 *     SGQA_OK.
 *   - Positions: query t (0 <= t < seq_q) sits at position pos(t) =
 *     q_offset + t and seq_kv >= q_offset + seq_q.  nblk = seq_kv / B
 *     complete blocks; query t may select among its nh(t) = pos(t) / B
 *     historical blocks and keeps Ks(t) = min(topk_tokens / B, nh(t)).
 *   - Layouts (row-major, innermost last): Q and O [seq_q][n_q_heads][head_dim];
 *     contiguous K and V [seq_kv][n_kv_heads][head_dim]; paged K and V
 *     [n_pages][n_kv_heads][page_size][head_dim] with page_table[ceil(seq_kv /
 *     page_size)] mapping logical page i to its physical page (the last page
 *     may be partly filled: positions from seq_kv on are never read); block keys
 *     Kbar [n_kv_heads][nblk][head_dim] fp32; scores
 *     [n_kv_heads][q_end - q_begin][nblk] fp32; lse [n_q_heads][seq_q] fp32
 *     (natural log).
 *   - Union tiles are tau = [tau * tile_q, min(tau * tile_q + tile_q, seq_q)),
 *     aligned to query 0 of the call; ntiles = ceil(seq_q / tile_q).
 *   - Batches: with batch = N > 1 the call covers N independent sequences of
 *     the same lengths and every per-sequence tensor gains an outer dimension
 *     of N: Q and O [N][seq_q][n_q_heads][head_dim]; contiguous K and V
 *     [N][seq_kv][n_kv_heads][head_dim]; Kbar [N][n_kv_heads][nblk][head_dim];
 *     scores [N][n_kv_heads][q_end - q_begin][nblk]; topk_idx
 *     [N][n_kv_heads][q_end - q_begin][k / B]; lse [N][n_q_heads][seq_q];
 *     union_off and union_len [N][n_kv_heads][ntiles]; union_blk and
 *     union_mask [N][sgqa_union_capacity(p) / N], each sequence's offsets
 *     relative to its own part.  A paged cache keeps one page pool shared by all sequences
 *     (K and V [n_pages][n_kv_heads][page_size][head_dim]) and page_table
 *     [N][ceil(seq_kv / page_size)].  The sequences are enqueued one after
 *     another on the stream and share the workspace and the status word, so
 *     sgqa_workspace_bytes is that of one sequence, while
 *     sgqa_union_capacity and sgqa_prefill_plan's launch count cover all N.
 */
#ifndef SGQA_H
#define SGQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SGQA_API __attribute__((visibility("default")))
#else
#define SGQA_API
#endif

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st* sgqa_stream_t;

enum sgqa_status_code {
  SGQA_OK = 0,
  SGQA_ERR_INVALID_ARG = 1, /* bad shape, range, null pointer or parameter */
  SGQA_ERR_UNSUPPORTED = 2, /* a valid combination this build does not implement */
  SGQA_ERR_ALIGNMENT = 3,   /* a pointer that TMA needs 16-byte aligned is not */
  SGQA_ERR_WORKSPACE = 4,   /* ws_bytes below sgqa_workspace_bytes(), or ws NULL */
  SGQA_ERR_CUDA = 5,        /* a CUDA runtime/driver call or launch failed */
  SGQA_ERR_CAPACITY = 6,    /* device: a union list exceeded its slot capacity */
  SGQA_ERR_TIMEOUT = 7,     /* device: a pipeline wait gave up (the kernel returned) */
  SGQA_ERR_BOUNDS = 8       /* device: an index check failed */
};

enum sgqa_dtype { SGQA_BF16 = 0, SGQA_FP32 = 1 };

/* Debug request, written by the caller into word 3 of a status buffer.  With
 * SGQA_DEBUG_STALL there, the first work item of the next attention launch
 * (sgqa_sparse_attn_fwd, or the attention inside sgqa_prefill) waits on a
 * barrier that nothing arrives on; after 1 ms it gives up the way any stalled
 * pipeline wait does: every role of the work item stops, the copies it has in
 * flight land, its tensor memory is released and the kernel returns, leaving
 * SGQA_ERR_TIMEOUT with detail 220 in the status buffer (outputs of that call
 * are undefined; the stream and context stay usable).  It exists to test the
 * give-up path without a fault.  sgqa_reset_status clears the word. */
#define SGQA_DEBUG_STALL 0x5354414c

/* Union semantics ("Efficient implementation of sparse attention").
 * MASKED (default): the union only batches work; query t attends to its own
 * selected blocks plus its current block, so results do not depend on tile_q.
 * FULL: every query of a tile attends to all of the tile's union blocks that
 * lie strictly before its own block, plus its current block. */
enum sgqa_union_mode { SGQA_UNION_MASKED = 0, SGQA_UNION_FULL = 1 };

/* Precision of the indexer scores.
 * SPLIT (default): fp32 scores from a two-term bf16 split of both operands
 * (about 1e-5 of |qt| |Kbar|), so selections follow the exact scores.
 * BF16: the lower-precision indexer: one bf16 product (both operands rounded
 * to bf16 from their fp32 values, fp32 accumulation) with each score then
 * rounded to bf16 (nearest even; stored in the fp32 score layout).  A third
 * of the tensor work; selections are exact on these scores (ties to the
 * lower block index) and differ from the SPLIT selection near the k-th score
 * (its recall against SPLIT is what to measure). */
enum sgqa_index_mode { SGQA_INDEX_SPLIT = 0, SGQA_INDEX_BF16 = 1 };

typedef struct sgqa_params {
  int32_t seq_q;        /* T >= 1 */
  int32_t seq_kv;       /* Tkv >= q_offset + seq_q */
  int32_t q_offset;     /* position of query 0 */
  int32_t n_q_heads;    /* H, a multiple of n_kv_heads */
  int32_t n_kv_heads;   /* Hkv >= 1 */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t block_size;   /* B: 1, 2, 4, 8 or 16 */
  int32_t topk_tokens;  /* k: a multiple of B; k / B blocks are selected */
  int32_t tile_q;       /* W: 1..64 queries per union tile */
  int32_t page_size;    /* 0 = contiguous K/V; else a multiple of B and of 8 */
  int32_t dtype;        /* enum sgqa_dtype of Q, K, V and O */
  int32_t union_mode;   /* enum sgqa_union_mode */
  float softmax_scale;  /* 0 -> 1 / sqrt(head_dim) */
  int32_t batch;        /* sequences of these lengths in one call; 0 or 1 = one */
  int32_t index_mode;   /* enum sgqa_index_mode */
} sgqa_params;

/* Workspace queries: `which` names the entry point. */
enum sgqa_ws_kind {
  SGQA_WS_INDEX_SCORES = 1,
  SGQA_WS_TOPK_UNION = 2,
  SGQA_WS_SPARSE_ATTN = 3,
  SGQA_WS_PREFILL = 4,
  SGQA_WS_ATTN_BWD = 5,
  SGQA_WS_DECODE = 6
};

/* Bytes of device workspace the entry point `which` needs for these params
 * (and, for SGQA_WS_INDEX_SCORES / SGQA_WS_TOPK_UNION, a query range of up to
 * seq_q queries).  0 on invalid params. */
SGQA_API size_t sgqa_workspace_bytes(const sgqa_params* p, int which);

/* Total union slots for the whole call: the sum over KV groups and tiles of
 * min(|tile| * k / B, nh(last query of the tile)).  Size union_blk and
 * union_mask with it.  -1 on invalid params. */
SGQA_API int64_t sgqa_union_capacity(const sgqa_params* p);

/* Step 1, block merge ("Reducing indexer's cost").
 * Kbar[g][j][:] = (1/B) * sum_{i<B} K[j*B + i][g][:] for j in [blk_begin, blk_end),
 * summed in fp32 as adjacent pairs level by level (((k0+k1)+(k2+k3))+((k4+k5)+(k6+k7))
 * for B = 8) and then multiplied by 1/B.  K is contiguous or paged (page_table
 * non-NULL iff p->page_size > 0).  Other blocks of Kbar are left untouched, so a
 * chunked prefill can extend a cached Kbar.  0 <= blk_begin <= blk_end <= nblk;
 * Kbar may be NULL for an empty range. */
SGQA_API int sgqa_block_merge(const sgqa_params* p, const void* K, const int32_t* page_table,
                              int32_t blk_begin, int32_t blk_end, float* Kbar, int32_t* status,
                              sgqa_stream_t stream);

/* Steps 2-3, indexer scores (Figure 3: each KV group scores every causal block).
 * scores[g][t - q_begin][j] = qt[g][t] . Kbar[g][j] for j < nh(t) and -inf for
 * j >= nh(t), for t in [q_begin, q_end), where qt[g][t] = (1/G) sum of the G
 * query heads of group g.  Computed on tcgen05 tensor cores from a two-term
 * bf16 split of both operands (hi*hi + hi*lo + lo*hi, fp32 accumulation), so
 * the error against an fp64 evaluation is about 1e-5 of |qt| |Kbar|.
 * Workspace: sgqa_workspace_bytes(p, SGQA_WS_INDEX_SCORES).  With no complete
 * block (seq_kv < block_size) there is nothing to score and Kbar and scores
 * may be NULL. */
SGQA_API int sgqa_index_scores(const sgqa_params* p, const void* Q, const float* Kbar,
                               int32_t q_begin, int32_t q_end, float* scores, void* ws,
                               size_t ws_bytes, int32_t* status, sgqa_stream_t stream);

/* Steps 4-5, top-k selection and tile union ("Trade-off between top-k and
 * block size"; "Efficient implementation of sparse attention").
 * Input: scores of queries [q_begin, q_end) laid out as sgqa_index_scores
 * writes them; q_begin must be a multiple of tile_q and q_end a multiple of
 * tile_q or seq_q.  Only entries j < nh(t) are read.
 * topk_idx (nullable) [Hkv][q_end - q_begin][k / B]: the selected blocks of each
 * query in ascending order, -1 padded; selection keeps the Ks(t) largest
 * scores, comparing fp32 bit patterns through the order-preserving map, with
 * ties going to the lower block index.
 * Union outputs, indexed by KV group and tile of the whole call
 * ([Hkv][ntiles]): union_off[g][tau] = first slot of the tile's list (a fixed,
 * capacity-based layout), union_len[g][tau] = its length; union_blk[slot] =
 * block ids in ascending order; union_mask[slot] bit i set iff query
 * tau * tile_q + i selected that block.  union_cap = length of union_blk and
 * union_mask, at least sgqa_union_capacity(p) (when that is 0, no query has a
 * historical block, and union_blk / union_mask may be NULL here and in the
 * attention calls).
 * Workspace: sgqa_workspace_bytes(p, SGQA_WS_TOPK_UNION). */
SGQA_API int sgqa_topk_union(const sgqa_params* p, const float* scores, int32_t q_begin,
                             int32_t q_end, int32_t* topk_idx, int64_t* union_off,
                             int32_t* union_len, int32_t* union_blk, uint64_t* union_mask,
                             int64_t union_cap, void* ws, size_t ws_bytes, int32_t* status,
                             sgqa_stream_t stream);

/* Step 6, main-path sparse attention (Figure 3 caption).  For query t, head h
 * of group g: softmax over the allowed positions of scale * Q[t][h] . K[p][g],
 * times V[p][g], where the allowed positions are, in SGQA_UNION_MASKED mode,
 * the positions of the blocks whose union_mask bit for t is set plus the
 * positions of t's own block up to pos(t) (SGQA_UNION_FULL: every union block
 * of t's tile that lies before t's own block, plus the same current part).
 * O in the dtype of Q; lse[h][t] = log of the softmax denominator, with the
 * maximum added back.  Runs on tcgen05 tensor cores (bf16 operands, fp32
 * accumulation and fp32 online softmax).  The workspace receives the staged
 * operands: fp32 inputs rounded to bf16 (K and V, when gathered key by key,
 * into a contiguous copy read through the page table), and for B >= 8, when
 * the call selects at least as many blocks as the cache holds (seq_q * k / B
 * >= nblk) or the inputs are fp32, a block-packed copy of K and V (each block
 * contiguous, in the tensor cores' shared-memory layout) that the kernel
 * gathers with one bulk copy per block.  Otherwise (B < 8, or a few queries
 * over a long cache) keys are gathered four rows at a time straight from K
 * and V; bf16 inputs then need no workspace.  Union arrays as written by
 * sgqa_topk_union for all tiles of the call.  Workspace:
 * sgqa_workspace_bytes(p, SGQA_WS_SPARSE_ATTN). */
SGQA_API int sgqa_sparse_attn_fwd(const sgqa_params* p, const void* Q, const void* K,
                                  const void* V, const int32_t* page_table,
                                  const int64_t* union_off, const int32_t* union_len,
                                  const int32_t* union_blk, const uint64_t* union_mask, void* O,
                                  float* lse, void* ws, size_t ws_bytes, int32_t* status,
                                  sgqa_stream_t stream);

/* Backward of step 6: the gradients of the main-path attention, for training
 * (the Step 5 pages use the layer in training as well as inference).  With
 * the softmax weights P of each (query, head) row over the same allowed
 * positions as sgqa_sparse_attn_fwd (same params, union_mode and union
 * arrays), O and lse the forward's outputs and dO the gradient of O:
 *   D = rowsum(dO * O),  dS = P * (dO V^T - D),
 *   dQ = scale * dS K,   dK = scale * dS^T Q,   dV = P^T dO,
 * dK and dV summed over every row (all heads of the group) that attends the
 * key.  P is recomputed from lse.  Outputs are fp32: dQ [seq_q][n_q_heads]
 * [head_dim], dK and dV [seq_kv][n_kv_heads][head_dim] at logical positions
 * (also for a paged K/V), every element written (0 for keys nothing attends).
 * Deterministic: each output element is accumulated in one place in a fixed
 * order.  Supported: bf16 inputs, block_size 8 or 16, n_q_heads / n_kv_heads
 * a power of two (SGQA_ERR_UNSUPPORTED otherwise).  Workspace:
 * sgqa_workspace_bytes(p, SGQA_WS_ATTN_BWD) (block-packed K and V, D, and the
 * key stages each union tile attends). */
SGQA_API int sgqa_sparse_attn_bwd(const sgqa_params* p, const void* Q, const void* K,
                                  const void* V, const int32_t* page_table,
                                  const int64_t* union_off, const int32_t* union_len,
                                  const int32_t* union_blk, const uint64_t* union_mask,
                                  const void* O, const float* lse, const void* dO, float* dQ,
                                  float* dK, float* dV, void* ws, size_t ws_bytes,
                                  int32_t* status, sgqa_stream_t stream);

/* Top-k and tile union without a workspace, for callers that cannot
 * allocate device memory (code running inside another framework's memory
 * pool, serving loops whose device memory is carved once up front, runtimes
 * with a fixed memory plan).  The pages have no counterpart: this is an
 * interface variant of sgqa_topk_union, with the same inputs, outputs and
 * results, whose per-query selection lists live in a library-owned static
 * device array of 2^21 int32 entries (8 MiB, held by every GPU that loads the
 * library until exit).  topk_idx is not produced.
 *   - Rejects n_kv_heads * (q_end - q_begin) * (k / B) > 2^21 with
 *     SGQA_ERR_WORKSPACE (call it on smaller query ranges).
 *   - Allocates nothing.  The first call on a device looks up the array's
 *     device address (cudaGetSymbolAddress) with that device current; make
 *     that first call before any stream capture.  The address is kept for
 *     the life of the process: after cudaDeviceReset (or anything else that
 *     destroys the device's primary context) it is stale, so do not call
 *     this entry point on that device again after such a reset.
 *   - All calls share the one array, so calls whose kernels overlap on the GPU
 *     (different streams, or different host threads) race; serialise them.
 *     Nothing in the array needs to start at zero. */
SGQA_API int sgqa_topk_union_noalloc(const sgqa_params* p, const float* scores, int32_t q_begin,
                                     int32_t q_end, int64_t* union_off, int32_t* union_len,
                                     int32_t* union_blk, uint64_t* union_mask, int64_t union_cap,
                                     int32_t* status, sgqa_stream_t stream);

/* Steps 1-6 fused into one enqueue: merge -> index scores -> top-k -> union ->
 * attention, chunked over queries so that intermediates stay within the
 * workspace.  Kbar is a caller-owned block-key cache [Hkv][nblk] fp32 (NULL
 * allowed when seq_kv < block_size, i.e. nblk = 0): blocks
 * [0, kbar_valid_blocks) are taken as already merged (earlier chunks of a
 * chunked prefill) and the rest are merged here.  Same outputs and numerics
 * as the step-by-step entry points.  Workspace: sgqa_workspace_bytes(p,
 * SGQA_WS_PREFILL); chunks are sized so that a chunk's fp32 score rows take
 * up to 8 GiB (4 GiB when rows exceed 16384 blocks), which with the
 * candidate lists and operand copies comes to about 12 GiB for 131072 queries
 * over 8 KV groups of 16384 blocks. */
SGQA_API int sgqa_prefill(const sgqa_params* p, const void* Q, const void* K, const void* V,
                          const int32_t* page_table, float* Kbar, int32_t kbar_valid_blocks,
                          void* O, float* lse, void* ws, size_t ws_bytes, int32_t* status,
                          sgqa_stream_t stream);

/* Separate index inputs for sgqa_prefill_ex (the index keys the Figure 3
 * caption speaks of, and the query side of a separate index projection).
 * Either pointer may be NULL.
 *   Qidx: [seq_q][n_kv_heads][head_dim] (batch: an outer dimension), in the
 *         dtype of Q: the index query of each KV group, used as is in place
 *         of the mean of the group's query heads.
 *   Kidx: the index keys, in K's layout and dtype (contiguous, or paged
 *         through the same page table): the block merge reads them in place
 *         of K, so Kbar holds their block means.  The attention still reads
 *         K and V.
 * Both must be 16-byte aligned. */
typedef struct sgqa_index_inputs {
  const void* Qidx;
  const void* Kidx;
} sgqa_index_inputs;

/* sgqa_prefill with separate index inputs (idx may be NULL, or have NULL
 * members, which then default as in sgqa_prefill).  With both NULL the
 * results equal sgqa_prefill's bit for bit.  Same workspace. */
SGQA_API int sgqa_prefill_ex(const sgqa_params* p, const void* Q, const void* K, const void* V,
                             const sgqa_index_inputs* idx, const int32_t* page_table,
                             float* Kbar, int32_t kbar_valid_blocks, void* O, float* lse,
                             void* ws, size_t ws_bytes, int32_t* status, sgqa_stream_t stream);

/* A caller-owned block-key cache that persists across decode steps, with a
 * fixed number of block rows per KV group so that the context can grow:
 *   Kbar:   [n_kv_heads][cap_blocks][head_dim] fp32 block keys (batch: an
 *           outer dimension), as sgqa_block_merge computes them;
 *   Ksplit: [2][n_kv_heads][cap_blocks][head_dim] bf16, the hi and lo halves
 *           of Kbar that the indexer reads (batch: an outer dimension of the
 *           pair), kept in step with Kbar by sgqa_decode;
 *   cap_blocks: rows per group, at least seq_kv / block_size of every call
 *           (cap_blocks * head_dim * 2 a multiple of 16);
 *   valid_blocks: blocks [0, valid_blocks) of both are up to date (0 for a
 *           fresh cache); each call merges and splits only the blocks past it
 *           and sets it to seq_kv / block_size. */
typedef struct sgqa_block_key_cache {
  float* Kbar;
  void* Ksplit;
  int32_t cap_blocks;
  int32_t valid_blocks;
} sgqa_block_key_cache;

/* Decode steps (the inference side of the layer: a few queries, typically
 * one, at the end of a long cached context): the same result as sgqa_prefill
 * on these params, computed with a persistent block-key cache and with each
 * attention work item split over ranges of its selected blocks when the call
 * has few work items (the ranges' partial outputs merged in a fixed order, so
 * results do not depend on scheduling; they may differ from sgqa_prefill's in
 * the last bits).  The call merges and splits only the blocks that completed
 * since the previous step.  Workspace: sgqa_workspace_bytes(p,
 * SGQA_WS_DECODE). */
SGQA_API int sgqa_decode(const sgqa_params* p, const void* Q, const void* K, const void* V,
                         const int32_t* page_table, sgqa_block_key_cache* cache, void* O,
                         float* lse, void* ws, size_t ws_bytes, int32_t* status,
                         sgqa_stream_t stream);

/* Plan of one sgqa_prefill call: queries per chunk (*chunk_queries) and the
 * number of kernel launches it enqueues (*launches).  Either pointer may be
 * NULL.  Returns an sgqa_status_code. */
SGQA_API int sgqa_prefill_plan(const sgqa_params* p, int64_t* chunk_queries, int32_t* launches);

/* Kernel classes named in the launch log. */
enum sgqa_kernel_kind {
  SGQA_K_MERGE = 1,        /* block merge */
  SGQA_K_SPLIT = 2,        /* bf16 hi/lo split of cached block keys; sampled-key gather */
  SGQA_K_INDEX_QUERY = 3,  /* group index query (mean of heads, hi/lo split) */
  SGQA_K_INDEX_SCORES = 4, /* tensor-core indexer GEMM */
  SGQA_K_TOPK_UNION = 5,   /* top-k selection (per query row) */
  SGQA_K_ATTN = 6,         /* sparse attention */
  SGQA_K_STAGE = 7,        /* attention operand staging: bf16 rounding, K/V block packing */
  SGQA_K_TILE_UNION = 8,   /* tile union and member masks */
  SGQA_K_SAMPLE_SCORES = 9, /* indexer GEMM over the sampled blocks (fused prefill) */
  SGQA_K_ROW_TAU = 10,      /* candidate thresholds from the sampled scores */
  SGQA_K_ATTN_BWD = 11      /* attention backward (dQ; dK and dV) */
};

/* Optional launch log for measurement.  While a log is installed, every
 * kernel launch of the library records caller-created CUDA events (cudaEvent_t
 * handles in start[i] / stop[i]) on the launch stream immediately before and
 * after the launch, stores its kind in kind[i] (host memory) and increments
 * count, until count reaches capacity (later launches are not logged).  The
 * library only records the events; it creates and destroys nothing.  The log
 * is process-wide and not thread-safe; NULL uninstalls it. */
typedef struct sgqa_launch_log {
  int32_t capacity;
  int32_t count;
  void** start;
  void** stop;
  int32_t* kind;
} sgqa_launch_log;
SGQA_API int sgqa_set_launch_log(sgqa_launch_log* log);

/* Zero a status buffer (enqueued on stream). */
SGQA_API int sgqa_reset_status(int32_t* status, sgqa_stream_t stream);

/* Synchronise `stream`, copy the status buffer to the host and return its
 * first word (an sgqa_status_code); *detail (nullable) receives the second. */
SGQA_API int sgqa_read_status(const int32_t* status, int32_t* detail, sgqa_stream_t stream);

/* Static description of a status code. */
SGQA_API const char* sgqa_status_string(int code);

/* Library version: major * 10000 + minor * 100 + patch. */
SGQA_API int sgqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGQA_H */
