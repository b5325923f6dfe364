// Device pieces shared by the forward and backward block-sparse attention
// kernels: a stage's block list (MetaT) and the warp that builds it from a
// tile's union entries (gen_stage), the per-query slot bits and their key
// masks, bulk copies of block-packed K/V, and the Q tensor map.  Included by
// attn.cu and attn_bwd.cu (each translation unit keeps its own copy).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace sgqa {
namespace {

constexpr unsigned FULL = 0xffffffffu;

template <int NBPS>
struct MetaT {         // one stage's block list
  int32_t nb;          // blocks in the stage
  int32_t last;        // last stage of the work item
  int32_t diag;        // first slot holding a current block of the sub-tile (or nb)
  int32_t pad;
  int32_t blk[NBPS];
  uint64_t mask[NBPS]; // bit qi: query qi of the sub-tile may attend the block
  // B = 2, 4: qb[qi][w] bit j: query qi selected the historical block in slot
  // 32 w + j (slots before diag), the transpose of mask written once per stage
  static constexpr int N = NBPS;
  static constexpr int QW = NBPS == 32 || NBPS == 64 ? NBPS / 32 : 0;
  uint32_t qb[64][QW > 0 ? QW : 1];
};

// Bit bs (bs < diag): query qi of the sub-tile selected the historical block
// in slot bs of this stage (B >= 8: at most 16 slots, read per thread).
template <typename Meta>
__device__ __forceinline__ uint32_t qbits_of(const Meta& m, int qi) {
  constexpr int N = (int)(sizeof(m.blk) / sizeof(m.blk[0]));
  uint32_t hb = 0u;
#pragma unroll
  for (int bs = 0; bs < (N < 32 ? N : 32); ++bs)
    hb |= (uint32_t)((m.mask[bs] >> qi) & 1ull) << bs;
  const int diag = m.diag;
  return diag >= 32 ? hb : (hb & ((1u << diag) - 1u));
}

// Keys 32 w .. 32 w + 31 of a stage that query qi may attend among its
// historical blocks, from the query's slot bits hb (slots 32 w / B ..), each
// widened to the B keys of its block (a block never straddles a 32-key word).
template <int B>
__device__ __forceinline__ uint32_t hist_keys(uint32_t hb, int w) {
  if constexpr (B == 2) {
    uint32_t x = (hb >> ((w & 1) * 16)) & 0xFFFFu;  // hb: the slot word of keys 64 (w / 2) ..
    x = (x | (x << 8)) & 0x00FF00FFu;
    x = (x | (x << 4)) & 0x0F0F0F0Fu;
    x = (x | (x << 2)) & 0x33333333u;
    x = (x | (x << 1)) & 0x55555555u;  // bit i at 2 i
    return x * 3u;
  } else if constexpr (B == 4) {
    uint32_t x = (hb >> (w * 8)) & 0xFFu;
    x = (x | (x << 12)) & 0x000F000Fu;
    x = (x | (x << 6)) & 0x03030303u;
    x = (x | (x << 3)) & 0x11111111u;  // bit i at 4 i
    return x * 0xFu;
  } else if constexpr (B == 8) {
    return ((((hb >> (w * 4)) & 0xFu) * 0x00204081u) & 0x01010101u) * 0xFFu;
  } else {
    static_assert(B == 16, "block sizes 2, 4, 8, 16");
    const uint32_t x = hb >> (w * 2);
    return ((x & 1u) ? 0x0000FFFFu : 0u) | ((x & 2u) ? 0xFFFF0000u : 0u);
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// State of the block-list generator of one work item (kept by warp 0).
struct Gen {
  int64_t cur, end;  // cursor into the tile's union entries
  int64_t c0, c_last, nd;
  int phase;         // 0: historical union entries, 1: current blocks, 2: done
  int64_t pf_at;     // chunk start of the prefetched entries (-1: none)
  int32_t pf_b;      // this lane's prefetched entry pf_at + lane
  uint64_t pf_m;
};

// Load entry `idx` of the union list (lane-strided chunk), or a sentinel.
template <typename Args>
__device__ __forceinline__ void union_entry(const Args& a, int64_t idx, int64_t end,
                                            int32_t& b, uint64_t& m) {
  const bool valid = idx < end;
  b = valid ? a.ublk[idx] : 0x7fffffff;
  m = valid ? a.umask[idx] : 0ull;
}

// Fill `m` with up to nbps blocks.  Warp-cooperative (warp 0).
template <bool QB, typename Meta, typename Args>
__device__ void gen_stage(const Args& a, Gen& gs, Meta& m, int nbps, int sh, uint64_t qmask,
                          int nq) {
  const int lane = lane_id();
  int n = 0;
  while (gs.phase == 0 && n < nbps) {
    if (gs.cur >= gs.end) {
      gs.phase = 1;
      break;
    }
    const int64_t idx = gs.cur + lane;
    const bool valid = idx < gs.end;
    int32_t b;
    uint64_t um;
    if (gs.pf_at == gs.cur) {  // the chunk was prefetched by the previous step
      b = gs.pf_b;
      um = gs.pf_m;
    } else {
      union_entry(a, idx, gs.end, b, um);
    }
    const bool hist = valid && b < gs.c0;
    const uint64_t sub = a.mode == SGQA_UNION_MASKED ? ((um >> sh) & qmask) : ~0ull;
    const uint32_t nonhist = __ballot_sync(FULL, !hist);
    const int stop = nonhist ? __ffs(nonhist) - 1 : 32;  // first lane past the historical part
    const uint32_t below = stop == 32 ? FULL : ((1u << stop) - 1u);
    const uint32_t pm = __ballot_sync(FULL, hist && sub != 0ull) & below;
    const int cnt = __popc(pm);
    const int room = nbps - n;
    const int rank = __popc(pm & lanemask_lt());
    if (cnt <= room) {
      if ((pm >> lane) & 1u) {
        m.blk[n + rank] = b;
        m.mask[n + rank] = sub;
      }
      n += cnt;
      if (stop < 32) {
        gs.cur += stop;
        gs.phase = 1;
      } else {
        gs.cur += 32;
      }
    } else {
      // take the first `room` entries of this chunk only (cnt > room >= 1, so
      // exactly one lane holds the entry of rank room - 1)
      const int last_lane =
          __ffs(__ballot_sync(FULL, ((pm >> lane) & 1u) && rank == room - 1)) - 1;
      if (((pm >> lane) & 1u) && rank < room) {
        m.blk[n + rank] = b;
        m.mask[n + rank] = sub;
      }
      n += room;
      gs.cur += last_lane + 1;
    }
    // start loading the chunk the next step will read
    gs.pf_at = gs.cur;
    union_entry(a, gs.cur + lane, gs.end, gs.pf_b, gs.pf_m);
  }
  __syncwarp();
  if (gs.phase == 1 && n < nbps) {
    int64_t cur = gs.cur, nd = gs.nd;
    if (lane == 0) {
      while (n < nbps && nd <= gs.c_last) {
        while (cur < gs.end && a.ublk[cur] < nd) ++cur;
        const bool in_u = cur < gs.end && a.ublk[cur] == nd;
        const uint64_t um = in_u ? a.umask[cur] : 0ull;
        const uint64_t sub =
            a.mode == SGQA_UNION_MASKED ? ((um >> sh) & qmask) : (in_u ? ~0ull : 0ull);
        m.blk[n] = (int32_t)nd;
        m.mask[n] = sub;
        ++n;
        ++nd;
      }
    }
    n = __shfl_sync(FULL, n, 0);
    gs.cur = __shfl_sync(FULL, cur, 0);
    gs.nd = __shfl_sync(FULL, nd, 0);
    if (gs.nd > gs.c_last) gs.phase = 2;
  }
  if (lane == 0) {
    m.nb = n;
    m.last = gs.phase == 2 ? 1 : 0;
  }
  __syncwarp();
  // first slot holding a current block of the sub-tile: the slots before it
  // are historical; with QB each query's bits over them are transposed into
  // qb (one ballot per query and 32 slots) for the softmax threads
  // (B = 1 takes every slot block by block and needs neither)
  if constexpr (Meta::N > 64) return;
  int diag = n;
  for (int w0 = 0; w0 < n; w0 += 32) {
    const int bs = w0 + lane;
    const uint32_t cm = __ballot_sync(FULL, bs < n && m.blk[bs] >= gs.c0);
    if (cm) {
      diag = w0 + __ffs(cm) - 1;
      break;
    }
  }
  if (lane == 0) m.diag = diag;
  if constexpr (QB) {
#pragma unroll
    for (int w = 0; w < Meta::QW; ++w) {
      const int bs = w * 32 + lane;
      const uint64_t mk = bs < diag ? m.mask[bs] : 0ull;
#pragma unroll 1
      for (int qi = 0; qi < nq; ++qi) {
        const uint32_t bits = __ballot_sync(FULL, (mk >> qi) & 1ull);
        if (lane == (qi & 31)) m.qb[qi][w] = bits;
      }
    }
  }
  __syncwarp();
}

// Bulk-copy a stage's packed blocks into shared slots 0..NBPS-1 (warp-wide):
// lane bs copies block blk[bs] (the zero block `zb` past nb).  One copy per
// block measured faster than merging runs of neighbouring blocks into one
// copy or splitting blocks into smaller copies.
template <int NBPS>
__device__ __forceinline__ void copy_blocks(uint8_t* dst, const __nv_bfloat16* base,
                                            const int32_t* blk, int nb, int64_t zb,
                                            int blk_elems, uint64_t* bar) {
  static_assert(NBPS <= 32, "one lane per slot");
  const int lane = lane_id();
  if (lane < NBPS) {
    const int64_t b = lane < nb ? (int64_t)blk[lane] : zb;
    bulk_load(dst + (size_t)lane * blk_elems * 2, base + b * blk_elems,
              (uint32_t)blk_elems * 2u, bar);
  }
}

// Tensor map for Q [T][H][d] with box 64 x G x QS: one sub-tile's query heads.
bool make_qmap(const Dims& dm, int QS, const void* Q, CUtensorMap* mq) {
  auto fn = tmap_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t e = 2;
  const cuuint32_t estr[3] = {1, 1, 1};
  cuuint64_t dims[3] = {(cuuint64_t)dm.d, (cuuint64_t)dm.H, (cuuint64_t)dm.T};
  cuuint64_t str[2] = {dm.d * e, (cuuint64_t)dm.H * dm.d * e};
  cuuint32_t box[3] = {64, (cuuint32_t)dm.G, (cuuint32_t)QS};
  return fn(mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(Q), dims, str, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace sgqa
