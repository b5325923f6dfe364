// sgqa_topk_union_noalloc: the top-k + tile-union step for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// that runs inside another framework's memory pool (the pool owns every
// device byte and exposes no raw allocation to plugins), latency-critical
// serving loops where an allocation would synchronise the device or fragment
// a pre-carved arena, and embedded runtimes whose memory plan is fixed before
// the first request.  For them this entry point keeps its only scratch (the
// per-query selection lists that the union step reads back) in a file-scope
// device array of fixed size, so the caller passes just the scores and the
// union outputs.
#include <mutex>

#include "internal.h"

namespace sgqa {

// Largest scratch the entry point uses: Hkv * (q_end - q_begin) * (k / B)
// int32 selection entries.  Every GPU that loads the library holds this
// array (8 MiB) until the process exits.
constexpr int64_t kNoAllocSelEntries = int64_t(1) << 21;

static __device__ __align__(256) int32_t g_noalloc_sel[kNoAllocSelEntries];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
int32_t* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current.
int noalloc_scratch(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SGQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_sel) != cudaSuccess || p == nullptr)
      return SGQA_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return SGQA_OK;
}

}  // namespace
}  // namespace sgqa

using namespace sgqa;

extern "C" SGQA_API int sgqa_topk_union_noalloc(const sgqa_params* p, const float* scores,
                                                int32_t q_begin, int32_t q_end,
                                                int64_t* union_off, int32_t* union_len,
                                                int32_t* union_blk, uint64_t* union_mask,
                                                int64_t union_cap, int32_t* status,
                                                sgqa_stream_t stream) {
  Dims dm;
  const int rc = derive(p, &dm);
  if (rc != SGQA_OK) return rc;
  if (q_begin < 0 || q_end < q_begin || q_end > dm.T || q_begin % dm.W ||
      (q_end % dm.W && q_end != dm.T))
    return SGQA_ERR_INVALID_ARG;
  if ((dm.nblk > 0 && scores == nullptr) || union_off == nullptr || union_len == nullptr ||
      ((union_blk == nullptr || union_mask == nullptr) && sgqa_union_capacity(p) > 0))
    return SGQA_ERR_INVALID_ARG;
  if (scores && (reinterpret_cast<uintptr_t>(scores) & 15u)) return SGQA_ERR_ALIGNMENT;
  if (union_cap < sgqa_union_capacity(p)) return SGQA_ERR_WORKSPACE;
  // the selection lists of one sequence must fit the fixed scratch array
  // (the sequences of a batch reuse it one after another on the stream)
  const int64_t need = (int64_t)dm.Hkv * (q_end - q_begin) * (dm.Ks > 0 ? dm.Ks : 1);
  if (need > kNoAllocSelEntries) return SGQA_ERR_WORKSPACE;
  int32_t* sel = nullptr;
  const int src = noalloc_scratch(&sel);
  if (src != SGQA_OK) return src;
  // Every entry the union step reads is written first by the same launch, so
  // the array needs no clearing between calls.
  const int64_t nq = q_end - q_begin;
  const int64_t sc_stride = (int64_t)dm.Hkv * nq * dm.nblk;
  const int64_t tiles = (int64_t)dm.Hkv * dm.ntiles;
  const int64_t ucap_b = group_cap(dm) * dm.Hkv;
  for (int64_t b = 0; b < dm.batch; ++b) {
    const int rc2 = launch_topk_union(dm, scores ? scores + b * sc_stride : nullptr, q_begin, q_end,
                                      sel, union_off + b * tiles, union_len + b * tiles,
                                      union_blk + b * ucap_b, union_mask + b * ucap_b, ucap_b,
                                      status, reinterpret_cast<cudaStream_t>(stream));
    if (rc2 != SGQA_OK) return rc2;
  }
  return SGQA_OK;
}
