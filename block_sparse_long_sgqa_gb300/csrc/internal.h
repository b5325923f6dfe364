// Host-side definitions shared by the translation units of libsgqa.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "sgqa.h"

namespace sgqa {

// Parameters of one call, validated and derived once on the host.
struct Dims {
  int64_t T, Tkv, off;       // queries, keys, position of query 0
  int H, Hkv, G, d;          // heads, KV groups, heads per group, head dim
  int B, Ks, W;              // block size, blocks selected per query, union tile
  int64_t nblk, ntiles;      // complete blocks, union tiles of the call
  int ps;                    // page size (0 = contiguous)
  int dtype, mode;           // enum sgqa_dtype, enum sgqa_union_mode
  float scale;               // softmax scale
  int elem;                  // bytes per Q/K/V element
  int batch;                 // sequences in the call (processed one after another)
  int index_bf16;            // SGQA_INDEX_BF16: one bf16 product, scores rounded to bf16
};

// Validate `p` and fill `dm`; returns SGQA_OK or an error code.
int derive(const sgqa_params* p, Dims* dm);

// nh of query t (absolute index within the call): historical complete blocks.
inline int64_t nh_of(const Dims& dm, int64_t t) {
  int64_t nh = (dm.off + t) / dm.B;
  return nh < dm.nblk ? nh : dm.nblk;
}

// Union slot capacity of tile tau of one group, and of one whole group.
int64_t tile_cap(const Dims& dm, int64_t tau);
int64_t group_cap(const Dims& dm);

// cuTensorMapEncodeTiled, fetched once through the runtime's driver entry
// point (so the library does not link the driver); nullptr if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn();

// Encode a tiled TMA descriptor (2-D, 128-byte swizzle, bf16) through the
// driver entry point; returns false on failure.
bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// Launch-log hooks (see sgqa_set_launch_log): called immediately around every
// kernel launch of the library.
void log_begin(int kind, cudaStream_t st);
void log_end(cudaStream_t st);

// ---- launchers (all asynchronous on `st`; return cudaSuccess or the launch error)
cudaError_t launch_block_merge(const Dims& dm, const void* K, const int32_t* page_table,
                               int64_t blk_begin, int64_t blk_end, float* Kbar,
                               __nv_bfloat16* khi, __nv_bfloat16* klo, cudaStream_t st);
cudaError_t launch_split_kbar(const Dims& dm, const float* Kbar, __nv_bfloat16* khi,
                              __nv_bfloat16* klo, cudaStream_t st);
cudaError_t launch_index_query(const Dims& dm, const void* Q, int64_t q_begin, int64_t q_end,
                               __nv_bfloat16* qhi, __nv_bfloat16* qlo, cudaStream_t st);
cudaError_t launch_to_bf16(const float* in, __nv_bfloat16* out, int64_t n, cudaStream_t st);
// fp32 K or V (contiguous or paged) -> bf16 contiguous [Tkv][Hkv][d].
cudaError_t launch_kv_to_bf16(const Dims& dm, const float* in, const int32_t* page_table,
                              __nv_bfloat16* out, cudaStream_t st);

// Block-packed, pre-swizzled copy of K or V for the attention gathers (B >= 8):
// [Hkv][ceil(Tkv/B) + 1][B * d] bf16, the last block of each head all zeros.
cudaError_t launch_kv_pack(const Dims& dm, const void* X, const int32_t* page_table,
                           __nv_bfloat16* out, cudaStream_t st);
inline int64_t kv_pack_elems(const Dims& dm) {
  return (int64_t)dm.Hkv * ((dm.Tkv + dm.B - 1) / dm.B + 1) * dm.B * dm.d;
}

// ---- threshold candidates of the fused prefill
// A row (query, group) selects from candidates when it has 2048 .. 16384
// historical blocks and keeps at most 768 of them: its threshold comes from
// the scores of the sampled blocks (8 adjacent blocks of every 64; the row's
// complete 64-block groups give (nh / 64) * 8 samples), the indexer keeps
// every score at or above it, and the row is selected from those candidates
// unless they miss the selection or overflow (then from its full scores).
constexpr int64_t kFiltMinNh = 2048, kFiltMaxNh = 16384;
constexpr int64_t kFiltMaxNeed = 768;
constexpr int kCandHalf = 1024;  // candidates per half-row list
__host__ __device__ inline bool filter_row(int64_t nh, int64_t need) {
  return nh >= kFiltMinNh && nh <= kFiltMaxNh && need <= kFiltMaxNeed && need < nh;
}
// Sampled key rows per group.
inline int64_t sampled_cols(const Dims& dm) { return (dm.nblk >> 6) << 3; }

// Gather the sampled blocks' hi keys (and lo keys when slo is not null):
// [Hkv][sampled_cols][d] each.
// krows: block-key rows per group of khi/klo (0: dm.nblk).
cudaError_t launch_sample_keys(const Dims& dm, const __nv_bfloat16* khi, const __nv_bfloat16* klo,
                               __nv_bfloat16* shi, __nv_bfloat16* slo, cudaStream_t st,
                               int64_t krows = 0);

// Optional modes of the indexer GEMM (all zero: plain scores).  In filter
// mode the full score rows are stored only for rows whose threshold is NaN.
struct IndexMode {
  int sample;        // khi holds the sampled keys (klo unread): scores [Hkv][nq][sampled_cols]
                     // of the single product hi * hi
  const float* tau;  // filter mode: [Hkv][nq] thresholds (NaN: no candidates)
  uint2* cand;       // [Hkv][nq][2][caph] (score bits, block index)
  int32_t* ccnt;     // [Hkv][nq][2][2] front / back counts per half
  int caph;
  // refill mode: full score rows of the listed (group, row tile) pairs only,
  // entries (g << 20) | (local row / 128), *nflist of them (set on the device)
  const int32_t* flist;
  const int32_t* nflist;
  // block-key rows per group in khi/klo (0: the call's nblk, or the sampled
  // columns in sampled mode); a persistent block-key cache has a fixed one
  int64_t krows;
};

// scores [Hkv][q_end-q_begin][nblk]; qhi/qlo are [Hkv][q_end-q_begin][d].
// Every score of a causal block is written, and -inf for the other blocks of
// each row's last 128-block tile; fill_tail also writes -inf for all blocks
// past that tile (the public contract), which the fused prefill skips.
int launch_index_scores(const Dims& dm, const __nv_bfloat16* qhi, const __nv_bfloat16* qlo,
                        const __nv_bfloat16* khi, const __nv_bfloat16* klo, int64_t q_begin,
                        int64_t q_end, float* scores, bool fill_tail, int32_t* status,
                        cudaStream_t st, const IndexMode* mode = nullptr);

// Candidate select of every row of [q_begin, q_end) (lists into sel
// [Hkv][nq][Ks]); rows it leaves go to rest (counters[0] of them), and the
// row tiles of those that had candidates to flist (counters[1]; tflag
// [Hkv][ceil(nq / 128)] marks them).  Zeroes counters and tflag first.
int launch_cand_rows(const Dims& dm, int64_t q_begin, int64_t q_end, int32_t* sel,
                     const uint2* cand, const int32_t* ccnt, int caph, int32_t* rest,
                     int32_t* counters, int32_t* tflag, int32_t* flist, int32_t* status,
                     cudaStream_t st);

// Candidate thresholds [Hkv][nq] of the call's queries [q_begin, q_end) from
// their sampled scores [Hkv][nq][sampled_cols] (NaN for rows that do not
// select from candidates).
int launch_row_tau(const Dims& dm, const float* sample_scores, int64_t q_begin, int64_t q_end,
                   float* tau, cudaStream_t st);

// Rows of more than kFiltMaxNh blocks (that do not take every block) are
// selected one CTA per row: local rows [long_rows_first(..), q_end - q_begin)
// of each group, by launch_select_long (scores and sel laid out as for
// launch_topk_union).
int64_t long_rows_first(const Dims& dm, int64_t q_begin, int64_t q_end);
int launch_select_long(const Dims& dm, const float* scores, int64_t q_begin, int64_t q_end,
                       int64_t r_first, int32_t* sel, int32_t* status, cudaStream_t st);

size_t topk_union_ws_bytes(const Dims& dm, int64_t nq);
// Kernel launches of one top-k/union call over [q_begin, q_end) (without the
// candidate path).
int topk_union_launches(const Dims& dm, int64_t q_begin, int64_t q_end);
int launch_topk_union(const Dims& dm, const float* scores, int64_t q_begin, int64_t q_end,
                      int32_t* sel, int64_t* union_off, int32_t* union_len, int32_t* union_blk,
                      uint64_t* union_mask, int64_t union_cap, int32_t* status, cudaStream_t st);

// Attention over the tiles [tau_begin, tau_end) of the call.  Q/K/V are bf16;
// Kp/Vp are their block-packed copies (launch_kv_pack, B >= 8) or null, in
// which case keys are gathered from K/V (contiguous, or paged through
// page_table).
int launch_sparse_attn(const Dims& dm, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                       const __nv_bfloat16* V, const __nv_bfloat16* Kp, const __nv_bfloat16* Vp,
                       const int32_t* page_table, const int64_t* union_off,
                       const int32_t* union_len, const int32_t* union_blk,
                       const uint64_t* union_mask, void* O, float* lse, int64_t tau_begin,
                       int64_t tau_end, int32_t* status, cudaStream_t st);

// Attention backward over the union lists of the whole call (B >= 8, bf16):
// K/V from their block-packed copies; ws holds D, the per-stage tile bitmaps
// and first slots, laid out by attn_bwd_ws_bytes (offsets returned).
size_t attn_bwd_ws_bytes(const Dims& dm, size_t* off_D, size_t* off_bits, size_t* off_first);
int launch_attn_bwd(const Dims& dm, const __nv_bfloat16* Q, const __nv_bfloat16* Kp,
                    const __nv_bfloat16* Vp, const int64_t* union_off, const int32_t* union_len,
                    const int32_t* union_blk, const uint64_t* union_mask, const void* O,
                    const float* lse, const void* dO, float* dQ, float* dK, float* dV, void* ws,
                    int32_t* status, cudaStream_t st);

}  // namespace sgqa
