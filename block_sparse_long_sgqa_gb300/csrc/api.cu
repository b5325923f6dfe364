// C ABI of libsgqa.so: validation, workspace layout and orchestration.
// Every entry point is declared and documented in include/sgqa.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace sgqa {

// launchers with an explicit slot layout (defined next to their kernels)
int launch_topk_union_layout(const Dims& dm, const float* scores, int64_t q_begin, int64_t q_end,
                             int32_t* sel, int64_t* union_off, int32_t* union_len,
                             int32_t* union_blk, uint64_t* union_mask, int64_t union_cap,
                             int64_t lay_tau0, int64_t lay_ntiles, int64_t capG,
                             int32_t* status, cudaStream_t st, int32_t* rest,
                             int32_t* nrest);
int launch_sparse_attn_layout(const Dims& dm, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                              const __nv_bfloat16* V, const __nv_bfloat16* Kp,
                              const __nv_bfloat16* Vp, const int32_t* page_table,
                              const int64_t* union_off, const int32_t* union_len,
                              const int32_t* union_blk, const uint64_t* union_mask, void* O,
                              float* lse, int64_t tau_begin, int64_t tau_end, int64_t lay_tau0,
                              int64_t lay_ntiles, int32_t* status, cudaStream_t st, int nsplit,
                              float* opart, float* lpart);

// ---------------------------------------------------------------- launch log
static sgqa_launch_log* g_log = nullptr;

void log_begin(int kind, cudaStream_t st) {
  sgqa_launch_log* l = g_log;
  if (l == nullptr || l->count >= l->capacity) return;
  cudaEventRecord(static_cast<cudaEvent_t>(l->start[l->count]), st);
  l->kind[l->count] = kind;
}

void log_end(cudaStream_t st) {
  sgqa_launch_log* l = g_log;
  if (l == nullptr || l->count >= l->capacity) return;
  cudaEventRecord(static_cast<cudaEvent_t>(l->stop[l->count]), st);
  ++l->count;
}

int derive(const sgqa_params* p, Dims* dm) {
  if (p == nullptr || dm == nullptr) return SGQA_ERR_INVALID_ARG;
  if (p->seq_q < 1 || p->q_offset < 0 || p->seq_kv < 1 ||
      (int64_t)p->q_offset + p->seq_q > p->seq_kv)
    return SGQA_ERR_INVALID_ARG;
  if (p->n_kv_heads < 1 || p->n_q_heads < 1 || p->n_q_heads % p->n_kv_heads)
    return SGQA_ERR_INVALID_ARG;
  if (p->block_size < 1 || p->topk_tokens < 0 || p->topk_tokens % p->block_size)
    return SGQA_ERR_INVALID_ARG;
  if (p->tile_q < 1 || p->dtype < 0 || p->dtype > 1 || p->union_mode < 0 || p->union_mode > 1)
    return SGQA_ERR_INVALID_ARG;
  if (!(p->softmax_scale >= 0.0f) || !std::isfinite(p->softmax_scale))
    return SGQA_ERR_INVALID_ARG;
  if (p->page_size < 0 || p->batch < 0 || p->index_mode < 0 || p->index_mode > 1)
    return SGQA_ERR_INVALID_ARG;
  const int B = p->block_size;
  if (B != 1 && B != 2 && B != 4 && B != 8 && B != 16) return SGQA_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128) return SGQA_ERR_UNSUPPORTED;
  if (p->tile_q > 64) return SGQA_ERR_UNSUPPORTED;
  if (p->n_q_heads / p->n_kv_heads > 128) return SGQA_ERR_UNSUPPORTED;
  if (p->page_size > 0 && (p->page_size % B || p->page_size % 8)) return SGQA_ERR_UNSUPPORTED;
  dm->T = p->seq_q;
  dm->Tkv = p->seq_kv;
  dm->off = p->q_offset;
  dm->H = p->n_q_heads;
  dm->Hkv = p->n_kv_heads;
  dm->G = p->n_q_heads / p->n_kv_heads;
  dm->d = p->head_dim;
  dm->B = B;
  dm->Ks = p->topk_tokens / B;
  dm->W = p->tile_q;
  dm->nblk = p->seq_kv / B;
  dm->ntiles = (p->seq_q + p->tile_q - 1) / p->tile_q;
  dm->ps = p->page_size;
  dm->dtype = p->dtype;
  dm->mode = p->union_mode;
  dm->scale = p->softmax_scale > 0.0f ? p->softmax_scale : 1.0f / std::sqrt((float)p->head_dim);
  dm->elem = p->dtype == SGQA_BF16 ? 2 : 4;
  dm->batch = p->batch > 1 ? p->batch : 1;
  dm->index_bf16 = p->index_mode == SGQA_INDEX_BF16 ? 1 : 0;
  return SGQA_OK;
}

int64_t tile_cap(const Dims& dm, int64_t tau) {
  const int64_t first = tau * dm.W;
  const int64_t len = std::min<int64_t>(dm.W, dm.T - first);
  const int64_t nh = std::min<int64_t>((dm.off + first + len - 1) / dm.B, dm.nblk);
  return std::min<int64_t>(len * dm.Ks, nh);
}

static int64_t caps_between(const Dims& dm, int64_t tau0, int64_t tau1) {
  int64_t s = 0;
  for (int64_t t = tau0; t < tau1; ++t) s += tile_cap(dm, t);
  return s;
}

int64_t group_cap(const Dims& dm) { return caps_between(dm, 0, dm.ntiles); }

// ------------------------------------------------------------------ TMA encode
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = tmap_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// ------------------------------------------------------------ workspace plans
namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Carve {  // bump allocator over a caller-owned workspace
  uint8_t* p;
  size_t used = 0;
  explicit Carve(void* base) : p(static_cast<uint8_t*>(base)) {}
  template <typename T>
  T* take(size_t n) {
    T* r = p ? reinterpret_cast<T*>(p + used) : nullptr;
    used += up(n * sizeof(T));
    return r;
  }
};

// Queries handled per prefill chunk, a multiple of lcm(tile_q, 128): bounded
// so the chunk's fp32 score rows (kept only for rows off the candidate path
// and for refilled row tiles) stay near 8 GiB when every row fits the
// candidate path, near 4 GiB otherwise (rows of more than kFiltMaxNh blocks
// are scored in full).  Larger chunks mean fewer, fuller launches: on the
// 128K workload 16384-query chunks take 46.1 ms per prefill against 49.2 for
// 4096; on the 1M chunked one (rows of 131072 blocks) 1024-query chunks take
// 31.9 ms against 34.2 for 512 and 32.5 for 2048.
int64_t prefill_chunk(const Dims& dm) {
  int64_t a = dm.W, b = 128;
  while (b) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  const int64_t L = dm.W / a * 128;
  const int64_t per_q = std::max<int64_t>(1, (int64_t)dm.Hkv * dm.nblk * 4);
  const int64_t bound = dm.nblk > kFiltMaxNh ? (int64_t(1) << 32) : (int64_t(1) << 33);
  int64_t c = bound / per_q / L * L;
  if (c < L) c = L;
  const int64_t tl = (dm.T + L - 1) / L * L;
  return std::min(c, tl);
}

struct IndexWs {
  __nv_bfloat16 *khi, *klo, *qhi, *qlo;
};
IndexWs carve_index(Carve& c, const Dims& dm, int64_t nq, bool key_split = true) {
  IndexWs w{nullptr, nullptr, nullptr, nullptr};
  const size_t nk = (size_t)dm.Hkv * dm.nblk * dm.d, nqe = (size_t)dm.Hkv * nq * dm.d;
  if (key_split) {
    w.khi = c.take<__nv_bfloat16>(nk);
    w.klo = c.take<__nv_bfloat16>(nk);
  }
  w.qhi = c.take<__nv_bfloat16>(nqe);
  w.qlo = c.take<__nv_bfloat16>(nqe);
  return w;
}

// Whether the attention reads K/V from block-packed copies made by the call
// (B >= 8): worth it when the call gathers at least as many blocks as the
// cache holds, and always for fp32 inputs (the copy converts them on the
// way).  Otherwise (a few queries over a long cache, as in a decode step) the
// keys are gathered from the cache itself.
bool use_pack(const Dims& dm) {
  return dm.B >= 8 && (dm.dtype == SGQA_FP32 || dm.T * dm.Ks >= dm.nblk);
}

struct AttnWs {
  __nv_bfloat16 *Q, *K, *V;  // bf16 copies of fp32 inputs (null when not needed)
  __nv_bfloat16 *Kp, *Vp;    // block-packed K/V (use_pack)
};
AttnWs carve_attn(Carve& c, const Dims& dm) {
  AttnWs w{nullptr, nullptr, nullptr, nullptr, nullptr};
  if (dm.dtype == SGQA_FP32) w.Q = c.take<__nv_bfloat16>((size_t)dm.T * dm.H * dm.d);
  if (use_pack(dm)) {  // packed copies (converted to bf16 on the way)
    w.Kp = c.take<__nv_bfloat16>((size_t)kv_pack_elems(dm));
    w.Vp = c.take<__nv_bfloat16>((size_t)kv_pack_elems(dm));
  } else if (dm.dtype == SGQA_FP32) {
    w.K = c.take<__nv_bfloat16>((size_t)dm.Tkv * dm.Hkv * dm.d);
    w.V = c.take<__nv_bfloat16>((size_t)dm.Tkv * dm.Hkv * dm.d);
  }
  return w;
}

// Whether some query of [q0, q1) selects from threshold candidates (nh grows
// with the query, so the range's ends bound it).
bool chunk_filtered(const Dims& dm, int64_t q0, int64_t q1) {
  if (q1 <= q0 || dm.Ks > kFiltMaxNeed || sampled_cols(dm) == 0) return false;
  const int64_t lo = nh_of(dm, q0), hi = nh_of(dm, q1 - 1);
  return hi >= kFiltMinNh && lo <= kFiltMaxNh;
}

struct PrefillWs {
  IndexWs ix;
  AttnWs at;
  bool filt;              // some chunk selects from threshold candidates
  __nv_bfloat16* shi;     // sampled block keys (hi halves) [Hkv][sampled_cols][d]
  float* ssc;             // sampled scores [Hkv][chunk][sampled_cols]
  float* tau;             // thresholds [Hkv][chunk]
  uint2* cand;            // candidates [Hkv][chunk][2][kCandHalf]
  int32_t* ccnt;          // counts [Hkv][chunk][2][2]
  int32_t* rest;          // rows left for the full-row select [Hkv][chunk]
  int32_t* counters;      // [0]: rows in rest, [1]: row tiles in flist
  int32_t *tflag, *flist;  // row tiles to score in full [Hkv][ceil(chunk / 128)]
  float* scores;
  int32_t* sel;
  int64_t* uoff;
  int32_t* ulen;
  int32_t* ublk;
  uint64_t* umask;
  int64_t ucap, chunk, chunk_tiles, capG;
};
PrefillWs carve_prefill(Carve& c, const Dims& dm, bool key_split = true) {
  PrefillWs w;
  w.chunk = prefill_chunk(dm);
  w.chunk_tiles = w.chunk / dm.W;
  w.ix = carve_index(c, dm, w.chunk, key_split);
  w.at = carve_attn(c, dm);
  w.filt = dm.nblk > 0 && chunk_filtered(dm, 0, dm.T);
  w.shi = nullptr;
  w.ssc = w.tau = nullptr;
  w.cand = nullptr;
  w.ccnt = nullptr;
  w.rest = w.counters = w.tflag = w.flist = nullptr;
  if (w.filt) {
    const int64_t ns = sampled_cols(dm), rows = (int64_t)dm.Hkv * w.chunk;
    w.shi = c.take<__nv_bfloat16>((size_t)dm.Hkv * ns * dm.d);
    w.ssc = c.take<float>((size_t)rows * ns);
    w.tau = c.take<float>((size_t)rows);
    w.cand = c.take<uint2>((size_t)rows * 2 * kCandHalf);
    w.ccnt = c.take<int32_t>((size_t)rows * 4);
    w.rest = c.take<int32_t>((size_t)rows);
    w.counters = c.take<int32_t>(2);
    const size_t nrt = (size_t)dm.Hkv * ((w.chunk + 127) / 128);
    w.tflag = c.take<int32_t>(nrt);
    w.flist = c.take<int32_t>(nrt);
  }
  w.scores = c.take<float>((size_t)dm.Hkv * w.chunk * std::max<int64_t>(dm.nblk, 1));
  w.sel = c.take<int32_t>((size_t)dm.Hkv * w.chunk * std::max(dm.Ks, 1));
  // slot layout of one chunk: the largest chunk's caps
  int64_t capG = 0;
  for (int64_t t0 = 0; t0 < dm.ntiles; t0 += w.chunk_tiles)
    capG = std::max(capG, caps_between(dm, t0, std::min(dm.ntiles, t0 + w.chunk_tiles)));
  w.capG = capG;
  w.ucap = capG * dm.Hkv;
  w.uoff = c.take<int64_t>((size_t)dm.Hkv * w.chunk_tiles);
  w.ulen = c.take<int32_t>((size_t)dm.Hkv * w.chunk_tiles);
  w.ublk = c.take<int32_t>((size_t)std::max<int64_t>(w.ucap, 1));
  w.umask = c.take<uint64_t>((size_t)std::max<int64_t>(w.ucap, 1));
  return w;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA; }

struct AttnSplitWs {
  int n;
  float* opart;
  float* lpart;
};

// Attention splits of a decode call: enough work items to cover every SM
// about twice, up to 16 per item, and only when the call is one chunk.
constexpr int kMaxSplit = 16;
int decode_splits(const Dims& dm) {
  if (prefill_chunk(dm) < dm.T) return 1;
  const int64_t QS = 128 / dm.G < dm.W ? 128 / dm.G : dm.W;
  const int64_t items = dm.ntiles * dm.Hkv * ((std::min<int64_t>(dm.T, dm.W) + QS - 1) / QS);
  const int64_t want = (2 * 152 + items - 1) / items;
  return (int)std::max<int64_t>(1, std::min<int64_t>(kMaxSplit, want));
}
void carve_decode(Carve& c, const Dims& dm, PrefillWs* pw, AttnSplitWs* sw) {
  PrefillWs w = carve_prefill(c, dm, false);
  if (pw) *pw = w;
  AttnSplitWs a;
  a.n = decode_splits(dm);
  a.opart = a.n > 1 ? c.take<float>((size_t)a.n * dm.T * dm.H * dm.d) : nullptr;
  a.lpart = a.n > 1 ? c.take<float>((size_t)a.n * dm.H * dm.T) : nullptr;
  if (sw) *sw = a;
}

// Element strides between consecutive sequences of a batched call (the
// batch layout of include/sgqa.h).  A paged cache shares its page pool, so
// only the page table moves.
struct SeqStride {
  int64_t q_bytes;    // Q and O
  int64_t kv_bytes;   // contiguous K and V (0 when paged)
  int64_t pt;         // page-table entries
  int64_t kbar;       // Kbar floats
  int64_t lse;        // lse floats
  int64_t tiles;      // union_off / union_len entries
};
SeqStride seq_stride(const Dims& dm) {
  SeqStride s;
  s.q_bytes = dm.T * dm.H * dm.d * dm.elem;
  s.kv_bytes = dm.ps > 0 ? 0 : dm.Tkv * dm.Hkv * dm.d * dm.elem;
  s.pt = dm.ps > 0 ? (dm.Tkv + dm.ps - 1) / dm.ps : 0;
  s.kbar = (int64_t)dm.Hkv * dm.nblk * dm.d;
  s.lse = (int64_t)dm.H * dm.T;
  s.tiles = (int64_t)dm.Hkv * dm.ntiles;
  return s;
}
template <typename T>
inline T* at_b(T* p, int64_t b, int64_t stride) {
  return p == nullptr ? nullptr : p + b * stride;
}
inline const void* at_bytes(const void* p, int64_t b, int64_t stride) {
  return p == nullptr ? nullptr : static_cast<const uint8_t*>(p) + b * stride;
}
inline void* at_bytes(void* p, int64_t b, int64_t stride) {
  return p == nullptr ? nullptr : static_cast<uint8_t*>(p) + b * stride;
}

// Attention operands: fp32 inputs rounded to bf16, and with use_pack the
// block-packed K/V.  Sets q/k/v to the buffers the attention kernel reads and
// `ad` to the dims it reads them with: fp32 K/V that are gathered key by key
// are converted into a contiguous bf16 copy (page_size 0 in `ad`).
cudaError_t stage_attn(const Dims& dm, const void* Q, const void* K, const void* V,
                       const int32_t* page_table, const AttnWs& w, const __nv_bfloat16** q,
                       const __nv_bfloat16** k, const __nv_bfloat16** v, Dims* ad,
                       cudaStream_t st) {
  *q = static_cast<const __nv_bfloat16*>(Q);
  *k = static_cast<const __nv_bfloat16*>(K);
  *v = static_cast<const __nv_bfloat16*>(V);
  *ad = dm;
  cudaError_t e = cudaSuccess;
  const bool pack = use_pack(dm);
  if (dm.dtype == SGQA_FP32) {
    e = launch_to_bf16(static_cast<const float*>(Q), w.Q, dm.T * dm.H * dm.d, st);
    *q = w.Q;
    if (!pack) {
      if (e == cudaSuccess) e = launch_kv_to_bf16(dm, static_cast<const float*>(K), page_table, w.K, st);
      if (e == cudaSuccess) e = launch_kv_to_bf16(dm, static_cast<const float*>(V), page_table, w.V, st);
      *k = w.K;
      *v = w.V;
      ad->ps = 0;
    }
  }
  if (pack) {
    if (e == cudaSuccess) e = launch_kv_pack(dm, K, page_table, w.Kp, st);
    if (e == cudaSuccess) e = launch_kv_pack(dm, V, page_table, w.Vp, st);
  }
  return e;
}

}  // namespace
}  // namespace sgqa

using namespace sgqa;

extern "C" {

SGQA_API int sgqa_version(void) { return 100; }

SGQA_API const char* sgqa_status_string(int code) {
  switch (code) {
    case SGQA_OK: return "ok";
    case SGQA_ERR_INVALID_ARG: return "invalid argument";
    case SGQA_ERR_UNSUPPORTED: return "unsupported configuration";
    case SGQA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case SGQA_ERR_WORKSPACE: return "workspace missing or too small";
    case SGQA_ERR_CUDA: return "CUDA call or launch failed";
    case SGQA_ERR_CAPACITY: return "union list exceeded its capacity";
    case SGQA_ERR_TIMEOUT: return "pipeline wait timed out";
    case SGQA_ERR_BOUNDS: return "index check failed";
    default: return "unknown status";
  }
}

SGQA_API size_t sgqa_workspace_bytes(const sgqa_params* p, int which) {
  Dims dm;
  if (derive(p, &dm) != SGQA_OK) return 0;
  Carve c(nullptr);
  switch (which) {
    case SGQA_WS_INDEX_SCORES: carve_index(c, dm, dm.T); break;
    case SGQA_WS_TOPK_UNION: c.take<int32_t>(topk_union_ws_bytes(dm, dm.T) / 4); break;
    case SGQA_WS_SPARSE_ATTN: carve_attn(c, dm); break;
    case SGQA_WS_PREFILL: carve_prefill(c, dm); break;
    case SGQA_WS_DECODE: carve_decode(c, dm, nullptr, nullptr); break;
    case SGQA_WS_ATTN_BWD: {
      c.take<__nv_bfloat16>((size_t)kv_pack_elems(dm));
      c.take<__nv_bfloat16>((size_t)kv_pack_elems(dm));
      size_t a, b, f;
      c.take<uint8_t>(attn_bwd_ws_bytes(dm, &a, &b, &f));
      break;
    }
    default: return 0;
  }
  return c.used + kAlign;  // slack to align the caller's base
}

SGQA_API int64_t sgqa_union_capacity(const sgqa_params* p) {
  Dims dm;
  if (derive(p, &dm) != SGQA_OK) return -1;
  return group_cap(dm) * dm.Hkv * dm.batch;
}

static void* align_ws(void* ws) {
  return reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + kAlign - 1) &
                                 ~static_cast<uintptr_t>(kAlign - 1));
}

SGQA_API int sgqa_block_merge(const sgqa_params* p, const void* K, const int32_t* page_table,
                              int32_t blk_begin, int32_t blk_end, float* Kbar, int32_t* status,
                              sgqa_stream_t stream) {
  Dims dm;
  int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  if (K == nullptr || (Kbar == nullptr && blk_end > blk_begin) || blk_begin < 0 ||
      blk_end < blk_begin || blk_end > dm.nblk || ((dm.ps > 0) != (page_table != nullptr)))
    return SGQA_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(Kbar)) return SGQA_ERR_ALIGNMENT;
  (void)status;
  const SeqStride ss = seq_stride(dm);
  for (int64_t b = 0; b < dm.batch; ++b) {
    const cudaError_t e = launch_block_merge(dm, at_bytes(K, b, ss.kv_bytes),
                                             at_b(page_table, b, ss.pt), blk_begin, blk_end,
                                             at_b(Kbar, b, ss.kbar), nullptr, nullptr,
                                             reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return SGQA_ERR_CUDA;
  }
  return SGQA_OK;
}

SGQA_API int sgqa_index_scores(const sgqa_params* p, const void* Q, const float* Kbar,
                               int32_t q_begin, int32_t q_end, float* scores, void* ws,
                               size_t ws_bytes, int32_t* status, sgqa_stream_t stream) {
  Dims dm;
  int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  if (Q == nullptr || ((Kbar == nullptr || scores == nullptr) && dm.nblk > 0) || q_begin < 0 ||
      q_end < q_begin || q_end > dm.T)
    return SGQA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(Kbar) || !aligned16(scores)) return SGQA_ERR_ALIGNMENT;
  if (ws == nullptr || ws_bytes < sgqa_workspace_bytes(p, SGQA_WS_INDEX_SCORES))
    return SGQA_ERR_WORKSPACE;
  if (q_end == q_begin || dm.nblk == 0) return SGQA_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carve c(align_ws(ws));
  IndexWs w = carve_index(c, dm, q_end - q_begin);
  const SeqStride ss = seq_stride(dm);
  const int64_t sc_stride = (int64_t)dm.Hkv * (q_end - q_begin) * dm.nblk;
  for (int64_t b = 0; b < dm.batch; ++b) {
    cudaError_t e = launch_split_kbar(dm, at_b(Kbar, b, ss.kbar), w.khi, w.klo, st);
    if (e == cudaSuccess)
      e = launch_index_query(dm, at_bytes(Q, b, ss.q_bytes), q_begin, q_end, w.qhi, w.qlo, st);
    if (e != cudaSuccess) return SGQA_ERR_CUDA;
    rc = launch_index_scores(dm, w.qhi, w.qlo, w.khi, w.klo, q_begin, q_end,
                             at_b(scores, b, sc_stride), true, status, st);
    if (rc != SGQA_OK) return rc;
  }
  return SGQA_OK;
}

SGQA_API int sgqa_topk_union(const sgqa_params* p, const float* scores, int32_t q_begin,
                             int32_t q_end, int32_t* topk_idx, int64_t* union_off,
                             int32_t* union_len, int32_t* union_blk, uint64_t* union_mask,
                             int64_t union_cap, void* ws, size_t ws_bytes, int32_t* status,
                             sgqa_stream_t stream) {
  Dims dm;
  int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  if (q_begin < 0 || q_end < q_begin || q_end > dm.T || q_begin % dm.W ||
      (q_end % dm.W && q_end != dm.T))
    return SGQA_ERR_INVALID_ARG;
  if ((dm.nblk > 0 && scores == nullptr) || union_off == nullptr || union_len == nullptr ||
      ((union_blk == nullptr || union_mask == nullptr) && group_cap(dm) > 0))
    return SGQA_ERR_INVALID_ARG;
  if (scores && !aligned16(scores)) return SGQA_ERR_ALIGNMENT;
  if (union_cap < sgqa_union_capacity(p)) return SGQA_ERR_WORKSPACE;
  if (topk_idx == nullptr &&
      (ws == nullptr || ws_bytes < sgqa_workspace_bytes(p, SGQA_WS_TOPK_UNION)))
    return SGQA_ERR_WORKSPACE;
  const SeqStride ss = seq_stride(dm);
  const int64_t nq = q_end - q_begin;
  const int64_t sc_stride = (int64_t)dm.Hkv * nq * dm.nblk;
  const int64_t sel_stride = (int64_t)dm.Hkv * nq * dm.Ks;
  // the union slots of one sequence (sgqa_union_capacity / batch)
  const int64_t ucap_b = group_cap(dm) * dm.Hkv;
  for (int64_t b = 0; b < dm.batch; ++b) {
    int32_t* sel = topk_idx ? topk_idx + b * sel_stride : static_cast<int32_t*>(align_ws(ws));
    rc = launch_topk_union(dm, at_b(scores, b, sc_stride), q_begin, q_end, sel,
                           union_off + b * ss.tiles, union_len + b * ss.tiles,
                           union_blk + b * ucap_b, union_mask + b * ucap_b, ucap_b, status,
                           reinterpret_cast<cudaStream_t>(stream));
    if (rc != SGQA_OK) return rc;
  }
  return SGQA_OK;
}

SGQA_API int sgqa_sparse_attn_fwd(const sgqa_params* p, const void* Q, const void* K,
                                  const void* V, const int32_t* page_table,
                                  const int64_t* union_off, const int32_t* union_len,
                                  const int32_t* union_blk, const uint64_t* union_mask, void* O,
                                  float* lse, void* ws, size_t ws_bytes, int32_t* status,
                                  sgqa_stream_t stream) {
  Dims dm;
  int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr || lse == nullptr ||
      union_off == nullptr || union_len == nullptr ||
      ((union_blk == nullptr || union_mask == nullptr) && group_cap(dm) > 0) ||
      ((dm.ps > 0) != (page_table != nullptr)))
    return SGQA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
    return SGQA_ERR_ALIGNMENT;
  const size_t need = sgqa_workspace_bytes(p, SGQA_WS_SPARSE_ATTN);
  if ((dm.dtype == SGQA_FP32 || use_pack(dm)) && (ws == nullptr || ws_bytes < need))
    return SGQA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carve c(align_ws(ws));
  AttnWs w = carve_attn(c, dm);
  const SeqStride ss = seq_stride(dm);
  // the union slots of one sequence: its groups' capacity (sgqa_union_capacity / batch)
  const int64_t ucap_b = group_cap(dm) * dm.Hkv;
  for (int64_t b = 0; b < dm.batch; ++b) {
    const __nv_bfloat16 *q, *k, *v;
    Dims ad;
    const int32_t* pt = at_b(page_table, b, ss.pt);
    if (stage_attn(dm, at_bytes(Q, b, ss.q_bytes), at_bytes(K, b, ss.kv_bytes),
                   at_bytes(V, b, ss.kv_bytes), pt, w, &q, &k, &v, &ad, st) != cudaSuccess)
      return SGQA_ERR_CUDA;
    rc = launch_sparse_attn(ad, q, k, v, w.Kp, w.Vp, ad.ps > 0 ? pt : nullptr,
                            union_off + b * ss.tiles, union_len + b * ss.tiles,
                            union_blk + b * ucap_b, union_mask + b * ucap_b,
                            at_bytes(O, b, ss.q_bytes), lse + b * ss.lse, 0, dm.ntiles, status,
                            st);
    if (rc != SGQA_OK) return rc;
  }
  return SGQA_OK;
}

SGQA_API int sgqa_sparse_attn_bwd(const sgqa_params* p, const void* Q, const void* K,
                                  const void* V, const int32_t* page_table,
                                  const int64_t* union_off, const int32_t* union_len,
                                  const int32_t* union_blk, const uint64_t* union_mask,
                                  const void* O, const float* lse, const void* dO, float* dQ,
                                  float* dK, float* dV, void* ws, size_t ws_bytes,
                                  int32_t* status, sgqa_stream_t stream) {
  Dims dm;
  int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr || lse == nullptr ||
      dO == nullptr || dQ == nullptr || dK == nullptr || dV == nullptr || union_off == nullptr ||
      union_len == nullptr ||
      ((union_blk == nullptr || union_mask == nullptr) && group_cap(dm) > 0) ||
      ((dm.ps > 0) != (page_table != nullptr)))
    return SGQA_ERR_INVALID_ARG;
  if (dm.dtype != SGQA_BF16 || dm.B < 8 || (dm.G & (dm.G - 1)) != 0 ||
      group_cap(dm) * dm.Hkv >= (int64_t(1) << 31))
    return SGQA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) ||
      !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
    return SGQA_ERR_ALIGNMENT;
  if (ws == nullptr || ws_bytes < sgqa_workspace_bytes(p, SGQA_WS_ATTN_BWD))
    return SGQA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carve c(align_ws(ws));
  __nv_bfloat16* Kp = c.take<__nv_bfloat16>((size_t)kv_pack_elems(dm));
  __nv_bfloat16* Vp = c.take<__nv_bfloat16>((size_t)kv_pack_elems(dm));
  size_t a0, b0, f0;
  uint8_t* rest = c.take<uint8_t>(attn_bwd_ws_bytes(dm, &a0, &b0, &f0));
  const SeqStride ss = seq_stride(dm);
  const int64_t ucap_b = group_cap(dm) * dm.Hkv;
  const int64_t kv_elems = dm.Tkv * dm.Hkv * dm.d;
  for (int64_t b = 0; b < dm.batch; ++b) {
    const int32_t* pt = at_b(page_table, b, ss.pt);
    cudaError_t e = launch_kv_pack(dm, at_bytes(K, b, ss.kv_bytes), pt, Kp, st);
    if (e == cudaSuccess) e = launch_kv_pack(dm, at_bytes(V, b, ss.kv_bytes), pt, Vp, st);
    if (e != cudaSuccess) return SGQA_ERR_CUDA;
    rc = launch_attn_bwd(dm, static_cast<const __nv_bfloat16*>(at_bytes(Q, b, ss.q_bytes)), Kp, Vp,
                         union_off + b * ss.tiles, union_len + b * ss.tiles,
                         union_blk + b * ucap_b, union_mask + b * ucap_b,
                         at_bytes(O, b, ss.q_bytes), lse + b * ss.lse,
                         at_bytes(dO, b, ss.q_bytes), dQ + b * (dm.T * dm.H * dm.d),
                         dK + b * kv_elems, dV + b * kv_elems, rest, status, st);
    if (rc != SGQA_OK) return rc;
  }
  return SGQA_OK;
}

namespace {

// A caller-owned block-key cache with a fixed row stride (sgqa_decode):
// Kbar and its bf16 hi/lo halves, blocks [0, valid) already merged and split.
struct KeyCache {
  __nv_bfloat16* khi = nullptr;
  __nv_bfloat16* klo = nullptr;
  int64_t rows = 0;  // block rows per group (0: no cache; Kbar rows are nblk)
};

// Attention split over its union entries (sgqa_decode): partial outputs.
struct AttnSplit {
  int n = 1;
  float* opart = nullptr;
  float* lpart = nullptr;
};

// One sequence of sgqa_prefill (arguments validated by the caller).  Qidx
// (nullable) replaces the mean of each group's query heads as the index
// query, Kidx (nullable) replaces K as the merge's input.  With a key cache,
// Kbar has kc.rows rows per group, only blocks [kbar_valid_blocks, nblk) are
// merged (and split into the cache), and the indexer reads the cache.
int prefill_one(const Dims& dm, const void* Q, const void* K, const void* V, const void* Qidx,
                const void* Kidx, const int32_t* page_table, float* Kbar,
                int32_t kbar_valid_blocks, void* O, float* lse, void* ws, int32_t* status,
                cudaStream_t st, const KeyCache& kc = KeyCache(),
                const AttnSplit& sp = AttnSplit()) {
  int rc = SGQA_OK;
  Carve c(align_ws(ws));
  PrefillWs w = carve_prefill(c, dm, kc.rows == 0);
  if (kc.rows > 0) {  // the indexer's key operand is the persistent cache
    w.ix.khi = kc.khi;
    w.ix.klo = kc.klo;
  }
  // the index query's source: Q with G heads per group, or Qidx with one
  Dims qd = dm;
  const void* qsrc = Q;
  if (Qidx != nullptr) {
    qd.H = dm.Hkv;
    qd.G = 1;
    qsrc = Qidx;
  }

  // step 1: merge the blocks not yet in the cache (and split all of them for the indexer)
  Dims md = dm;  // the merge writes rows of the cache's stride
  if (kc.rows > 0) md.nblk = kc.rows;
  cudaError_t e = launch_block_merge(md, Kidx != nullptr ? Kidx : K, page_table,
                                     kbar_valid_blocks, dm.nblk, Kbar, w.ix.khi, w.ix.klo, st);
  if (e == cudaSuccess && kbar_valid_blocks > 0 && kc.rows == 0) {
    Dims part = dm;  // split the cached prefix: per group, blocks [0, kbar_valid_blocks)
    for (int g = 0; g < dm.Hkv && e == cudaSuccess; ++g) {
      part.Hkv = 1;
      part.nblk = kbar_valid_blocks;
      const size_t o = (size_t)g * dm.nblk * dm.d;
      e = launch_split_kbar(part, Kbar + o, w.ix.khi + o, w.ix.klo + o, st);
    }
  }
  if (e == cudaSuccess && w.filt)
    e = launch_sample_keys(dm, w.ix.khi, w.ix.klo, w.shi, nullptr, st, kc.rows);
  const __nv_bfloat16 *q, *k, *v;
  Dims ad;  // the dims the attention reads its K/V with
  if (e == cudaSuccess) e = stage_attn(dm, Q, K, V, page_table, w.at, &q, &k, &v, &ad, st);
  if (e != cudaSuccess) return SGQA_ERR_CUDA;

  for (int64_t q0 = 0; q0 < dm.T; q0 += w.chunk) {
    const int64_t q1 = std::min<int64_t>(dm.T, q0 + w.chunk);
    const int64_t tau0 = q0 / dm.W, tau1 = (q1 + dm.W - 1) / dm.W;
    const bool filt = w.filt && chunk_filtered(dm, q0, q1);
    if (dm.nblk > 0) {
      e = launch_index_query(qd, qsrc, q0, q1, w.ix.qhi, w.ix.qlo, st);
      if (e != cudaSuccess) return SGQA_ERR_CUDA;
      IndexMode mode{};
      mode.krows = kc.rows;
      if (filt) {  // thresholds from the sampled blocks' scores, then candidates
        IndexMode ms{};
        ms.sample = 1;
        rc = launch_index_scores(dm, w.ix.qhi, w.ix.qlo, w.shi, w.shi, q0, q1, w.ssc, false,
                                 status, st, &ms);
        if (rc == SGQA_OK) rc = launch_row_tau(dm, w.ssc, q0, q1, w.tau, st);
        if (rc != SGQA_OK) return rc;
        mode.tau = w.tau;
        mode.cand = w.cand;
        mode.ccnt = w.ccnt;
        mode.caph = kCandHalf;
      }
      rc = launch_index_scores(dm, w.ix.qhi, w.ix.qlo, w.ix.khi, w.ix.klo, q0, q1, w.scores,
                               false, status, st, &mode);
      if (rc != SGQA_OK) return rc;
      if (filt) {  // candidate select; row tiles it could not decide get full score rows
        rc = launch_cand_rows(dm, q0, q1, w.sel, w.cand, w.ccnt, kCandHalf, w.rest, w.counters,
                              w.tflag, w.flist, status, st);
        if (rc != SGQA_OK) return rc;
        IndexMode mr{};
        mr.flist = w.flist;
        mr.nflist = w.counters + 1;
        mr.krows = kc.rows;
        rc = launch_index_scores(dm, w.ix.qhi, w.ix.qlo, w.ix.khi, w.ix.klo, q0, q1, w.scores,
                                 false, status, st, &mr);
        if (rc != SGQA_OK) return rc;
      }
    }
    // full-row select (in a filtered chunk: of the rows the candidates left) and union
    rc = launch_topk_union_layout(dm, w.scores, q0, q1, w.sel, w.uoff, w.ulen, w.ublk, w.umask,
                                  w.ucap, tau0, w.chunk_tiles, w.capG, status, st,
                                  filt ? w.rest : nullptr, filt ? w.counters : nullptr);
    if (rc != SGQA_OK) return rc;
    rc = launch_sparse_attn_layout(ad, q, k, v, w.at.Kp, w.at.Vp,
                                   ad.ps > 0 ? page_table : nullptr, w.uoff, w.ulen,
                                   w.ublk, w.umask, O, lse, tau0, tau1, tau0, w.chunk_tiles,
                                   status, st, sp.n, sp.opart, sp.lpart);
    if (rc != SGQA_OK) return rc;
  }
  return SGQA_OK;
}

}  // namespace

SGQA_API int sgqa_prefill_ex(const sgqa_params* p, const void* Q, const void* K, const void* V,
                             const sgqa_index_inputs* idx, const int32_t* page_table,
                             float* Kbar, int32_t kbar_valid_blocks, void* O, float* lse,
                             void* ws, size_t ws_bytes, int32_t* status, sgqa_stream_t stream) {
  Dims dm;
  int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr || lse == nullptr ||
      (Kbar == nullptr && dm.nblk > 0) || kbar_valid_blocks < 0 ||
      kbar_valid_blocks > dm.nblk || ((dm.ps > 0) != (page_table != nullptr)))
    return SGQA_ERR_INVALID_ARG;
  const void* Qidx = idx ? idx->Qidx : nullptr;
  const void* Kidx = idx ? idx->Kidx : nullptr;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(Kbar) ||
      (Qidx && !aligned16(Qidx)) || (Kidx && !aligned16(Kidx)))
    return SGQA_ERR_ALIGNMENT;
  if (ws == nullptr || ws_bytes < sgqa_workspace_bytes(p, SGQA_WS_PREFILL))
    return SGQA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const SeqStride ss = seq_stride(dm);
  const int64_t qidx_bytes = dm.T * dm.Hkv * dm.d * dm.elem;
  for (int64_t b = 0; b < dm.batch; ++b) {
    rc = prefill_one(dm, at_bytes(Q, b, ss.q_bytes), at_bytes(K, b, ss.kv_bytes),
                     at_bytes(V, b, ss.kv_bytes), at_bytes(Qidx, b, qidx_bytes),
                     at_bytes(Kidx, b, ss.kv_bytes), at_b(page_table, b, ss.pt),
                     at_b(Kbar, b, ss.kbar), kbar_valid_blocks, at_bytes(O, b, ss.q_bytes),
                     at_b(lse, b, ss.lse), ws, status, st);
    if (rc != SGQA_OK) return rc;
  }
  return SGQA_OK;
}

SGQA_API int sgqa_prefill(const sgqa_params* p, const void* Q, const void* K, const void* V,
                          const int32_t* page_table, float* Kbar, int32_t kbar_valid_blocks,
                          void* O, float* lse, void* ws, size_t ws_bytes, int32_t* status,
                          sgqa_stream_t stream) {
  return sgqa_prefill_ex(p, Q, K, V, nullptr, page_table, Kbar, kbar_valid_blocks, O, lse, ws,
                         ws_bytes, status, stream);
}

SGQA_API int sgqa_decode(const sgqa_params* p, const void* Q, const void* K, const void* V,
                         const int32_t* page_table, sgqa_block_key_cache* cache, void* O,
                         float* lse, void* ws, size_t ws_bytes, int32_t* status,
                         sgqa_stream_t stream) {
  Dims dm;
  int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr || lse == nullptr ||
      cache == nullptr || cache->Kbar == nullptr || cache->Ksplit == nullptr ||
      cache->cap_blocks < dm.nblk || cache->valid_blocks < 0 ||
      ((dm.ps > 0) != (page_table != nullptr)))
    return SGQA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
      !aligned16(cache->Kbar) || !aligned16(cache->Ksplit))
    return SGQA_ERR_ALIGNMENT;
  if (((int64_t)cache->cap_blocks * dm.d * 2) % 16 != 0) return SGQA_ERR_ALIGNMENT;
  if (ws == nullptr || ws_bytes < sgqa_workspace_bytes(p, SGQA_WS_DECODE))
    return SGQA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carve c(align_ws(ws));
  AttnSplitWs sw;
  carve_decode(c, dm, nullptr, &sw);
  const int64_t cap = cache->cap_blocks;
  const int32_t valid = std::min<int32_t>(cache->valid_blocks, (int32_t)dm.nblk);
  KeyCache kc;
  kc.rows = cap;
  AttnSplit sp;
  sp.n = sw.n;
  sp.opart = sw.opart;
  sp.lpart = sw.lpart;
  const SeqStride ss = seq_stride(dm);
  const int64_t kcache = (int64_t)dm.Hkv * cap * dm.d;  // one sequence's cache rows
  for (int64_t b = 0; b < dm.batch; ++b) {
    __nv_bfloat16* hi = static_cast<__nv_bfloat16*>(cache->Ksplit) + b * 2 * kcache;
    kc.khi = hi;
    kc.klo = hi + kcache;
    rc = prefill_one(dm, at_bytes(Q, b, ss.q_bytes), at_bytes(K, b, ss.kv_bytes),
                     at_bytes(V, b, ss.kv_bytes), nullptr, nullptr, at_b(page_table, b, ss.pt),
                     cache->Kbar + b * kcache, valid, at_bytes(O, b, ss.q_bytes),
                     at_b(lse, b, ss.lse), ws, status, st, kc, sp);
    if (rc != SGQA_OK) return rc;
  }
  cache->valid_blocks = (int32_t)dm.nblk;
  return SGQA_OK;
}

SGQA_API int sgqa_prefill_plan(const sgqa_params* p, int64_t* chunk_queries, int32_t* launches) {
  Dims dm;
  const int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  const int64_t chunk = prefill_chunk(dm);
  if (chunk_queries) *chunk_queries = chunk;
  if (launches) {
    // with an empty block-key cache: merge, operand staging (fp32 rounding,
    // K/V block packing when use_pack), then per chunk the index query and indexer GEMM
    // (when there are blocks), the row selects (a CTA-per-row launch too when
    // the chunk has rows of more than 16384 blocks), tile union and attention;
    // where some rows select from threshold candidates, the sampled-key gather
    // once and per such chunk the sampled-block GEMM, the thresholds, the
    // candidate select (after zeroing its two counters and the row-tile
    // flags) and the refill GEMM of the row tiles it left (the rows it leaves
    // then all go through the warp-per-row select)
    const bool any_filt = dm.nblk > 0 && chunk_filtered(dm, 0, dm.T);
    const bool pack = use_pack(dm);
    int64_t n = (dm.nblk > 0 ? 1 : 0) + (dm.dtype == SGQA_FP32 ? (pack ? 1 : 3) : 0) +
                (pack ? 2 : 0) + (any_filt ? 1 : 0);
    for (int64_t q0 = 0; q0 < dm.T; q0 += chunk) {
      const int64_t q1 = std::min<int64_t>(dm.T, q0 + chunk);
      const bool filt = any_filt && chunk_filtered(dm, q0, q1);
      n += (dm.nblk > 0 ? 2 : 0) + 1 + (filt ? 4 + 2 + 2 : topk_union_launches(dm, q0, q1));
    }
    *launches = (int32_t)(n * dm.batch);
  }
  return SGQA_OK;
}

SGQA_API int sgqa_set_launch_log(sgqa_launch_log* log) {
  if (log != nullptr && (log->capacity < 0 || (log->capacity > 0 &&
                         (log->start == nullptr || log->stop == nullptr || log->kind == nullptr))))
    return SGQA_ERR_INVALID_ARG;
  g_log = log;
  return SGQA_OK;
}

SGQA_API int sgqa_reset_status(int32_t* status, sgqa_stream_t stream) {
  if (status == nullptr) return SGQA_ERR_INVALID_ARG;
  return cuda_rc(cudaMemsetAsync(status, 0, 4 * sizeof(int32_t),
                                 reinterpret_cast<cudaStream_t>(stream)));
}

SGQA_API int sgqa_read_status(const int32_t* status, int32_t* detail, sgqa_stream_t stream) {
  if (status == nullptr) return SGQA_ERR_INVALID_ARG;
  int32_t h[4] = {0, 0, 0, 0};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(h, status, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SGQA_ERR_CUDA;
  if (detail) *detail = h[1];
  return h[0];
}

}  // extern "C"
