// Indexer scores on tcgen05 tensor cores.
//
// "Inside Step 5 Preview" (StepFun blog), section Sparse GQA, paragraph
// "Reducing indexer's cost" and Figure 3: every query of a KV group is scored
// against every causal block representation of that group.  Here that is a
// GEMM per group, S = qt * Kbar^T, with qt the group's mean query and Kbar the
// mean-pooled block keys, both fp32.  To keep fp32-level accuracy on bf16
// tensor cores each operand is split as x = hi + lo (hi = bf16(x), lo =
// bf16(x - hi)) and S is accumulated in fp32 as hi*hi + hi*lo + lo*hi (the
// three-product scheme of Markidis et al., "NVIDIA Tensor Core
// Programmability, Performance & Precision", 2018).
//
// Work item = (128 queries, one group, 128 blocks): one 128x128 output tile.
// The items of a launch are split into equal contiguous ranges, one per SM
// (persistent CTAs), so every SM gets the same number of tiles however the
// causal row lengths vary; consecutive items share the query operand, which
// is reloaded only when the (row tile, group) pair changes.  Warp 0 issues
// the TMA loads (B double-buffered), warp 1 the MMAs into two TMEM
// accumulators (128 fp32 columns each), and warps 2-9 drain TMEM (one query
// row per thread, two warps per TMEM lane quadrant taking 64 columns each),
// apply the causal block mask and write the tile.  Stores go
// through a 128-byte-swizzled shared staging buffer and TMA, so each tile
// leaves as full 128-byte rows instead of 16-byte pieces of 32 rows.
//
// Three further modes serve the fused prefill.  Sampled mode scores only the
// sampled blocks (8 adjacent blocks of every 64, gathered into their own key
// array beforehand), so a row has (nh / 64) * 8 columns, with the single
// product hi*hi (the sampled scores only steer a threshold; every selection
// compares full-precision scores).  Filter mode compares each score with its
// row's candidate threshold (derived from the sampled scores) and appends
// every score at or above it, with its block index, to the row's candidate
// list instead of storing the score row: one list per 64-column half of the
// tile, and per half a front part (the CTA that starts the row tile, written
// upwards) and a back part (the CTA that finishes it, written downwards from
// the end of the list), so no two threads ever share a counter; rows without
// a threshold are stored in full.  Refill mode scores only listed row tiles
// (those whose candidates could not decide a row), counting its items on the
// device.
//
// The bf16 indexer (SGQA_INDEX_BF16) runs every mode with the single product
// hi * hi and rounds each score to bf16 (nearest even) as it leaves TMEM, so
// masks, thresholds, candidates and stored rows all see the rounded scores.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace sgqa {
namespace {

constexpr int IDX_BN = 128;  // blocks per output tile

template <int D>
struct IdxCfg {
  static constexpr int BM = 128, BN = IDX_BN, STAGES = 2, NACC = 2;
  static constexpr int KC = D / 64;          // 128-byte (64-element) chunks along d
  static constexpr int A_TILE = BM * 128;    // bytes of one chunk of A
  static constexpr int B_TILE = BN * 128;
  static constexpr int A_BYTES = KC * A_TILE;
  static constexpr int B_BYTES = KC * B_TILE;
  static constexpr int OFF_AHI = 0;
  static constexpr int OFF_ALO = A_BYTES;
  static constexpr int OFF_B = 2 * A_BYTES;
  static constexpr int STAGE_BYTES = 2 * B_BYTES;  // hi + lo
  static constexpr int STG_BYTES = 32 * 128;       // one 32 x 32 fp32 store box
  static constexpr int OFF_STG = OFF_B + STAGES * STAGE_BYTES;  // one per epilogue warp
  static constexpr int OFF_BAR = OFF_STG + 8 * STG_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t TMEM_COLS = NACC * BN;
  static constexpr int NTHREADS = 320;  // producer, MMA, 8 epilogue warps
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct IdxArgs {
  int64_t nq, q_begin, q_end, q_offset;
  int64_t nblk;       // columns of a score row
  int64_t krows;      // block-key rows per group in the B operand arrays
  int64_t nblk_full;  // complete blocks of the call (bounds nh)
  int B, Hkv;
  int sample;      // columns are the sampled blocks: a row has (nh / 64) * 8 of them
  int single;      // one product hi * hi (sampled mode, and the bf16 indexer)
  int round_bf16;  // scores rounded to bf16 (nearest even) before any use
  int64_t total;   // work items of the launch
  int fill_tail;   // write -inf for the columns past a row tile's last item
  int tma_store;   // scores rows are 16-byte multiples: store through the tensor map
  float* scores;
  // filter mode (tau != nullptr): candidates at or above the row's threshold
  const float* tau;  // [Hkv][nq]; NaN: the row takes no candidates
  uint2* cand;       // [Hkv][nq][2 halves][caph] (score bits, block)
  int32_t* ccnt;     // [Hkv][nq][2 halves][front, back] counts
  int caph;
  // refill mode (flist != nullptr): only the listed (group, row tile) pairs,
  // entries (g << 20) | rt, *nflist of them; the item count is found on the device
  const int32_t* flist;
  const int32_t* nflist;
  int nfl;
  int32_t* status;
};

// Valid columns of row t: its historical blocks, or in sampled mode the
// samples of its complete 64-block groups.
__device__ __forceinline__ int64_t bound_of(const IdxArgs& a, int64_t t) {
  int64_t nh = (a.q_offset + t) / a.B;
  if (nh > a.nblk_full) nh = a.nblk_full;
  return a.sample ? ((nh >> 6) << 3) : nh;
}

// Column tiles of row tile rt (at least one, so rows with no complete block
// still get their -inf row).
__device__ __forceinline__ int64_t ntiles_of(const IdxArgs& a, int64_t rt) {
  const int64_t t0 = a.q_begin + rt * 128;
  const int64_t t_last = (t0 + 128 < a.q_end ? t0 + 128 : a.q_end) - 1;
  const int64_t nh = bound_of(a, t_last);
  const int64_t nt = (nh + IDX_BN - 1) / IDX_BN;
  return nt > 0 ? nt : 1;
}

// Items are ordered by row tile, then group, then column tile (in refill
// mode: by list entry, then column tile).
struct Item {
  int64_t rt, n, nt;
  int g, li;
};
__device__ __forceinline__ void list_entry(const IdxArgs& a, Item& w) {
  const int32_t e = a.flist[w.li];
  w.g = e >> 20;
  w.rt = e & 0xfffff;
  w.nt = ntiles_of(a, w.rt);
}
__device__ Item item_at(const IdxArgs& a, int64_t i) {
  Item w;
  w.rt = 0;
  w.li = 0;
  if (a.flist != nullptr) {
    for (;; ++w.li) {
      list_entry(a, w);
      if (i < w.nt) {
        w.n = i;
        return w;
      }
      i -= w.nt;
    }
  }
  for (;;) {
    const int64_t nt = ntiles_of(a, w.rt);
    if (i < nt * a.Hkv) {
      w.g = (int)(i / nt);
      w.n = i % nt;
      w.nt = nt;
      return w;
    }
    i -= nt * a.Hkv;
    ++w.rt;
  }
}
__device__ __forceinline__ void item_next(const IdxArgs& a, Item& w) {
  if (++w.n < w.nt) return;
  w.n = 0;
  if (a.flist != nullptr) {
    if (++w.li < a.nfl) list_entry(a, w);
    return;
  }
  if (++w.g < a.Hkv) return;
  w.g = 0;
  ++w.rt;
  w.nt = ntiles_of(a, w.rt);
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    k_index_scores(const __grid_constant__ CUtensorMap mq_hi, const __grid_constant__ CUtensorMap mq_lo,
                   const __grid_constant__ CUtensorMap mk_hi, const __grid_constant__ CUtensorMap mk_lo,
                   const __grid_constant__ CUtensorMap ms, const IdxArgs a0) {
  IdxArgs a = a0;
  if (a.flist != nullptr) {  // refill mode: items of the listed row tiles
    a.nfl = *a.nflist;
    int64_t tot = 0;
    for (int i = 0; i < a.nfl; ++i) tot += ntiles_of(a, a.flist[i] & 0xfffff);
    a.total = tot;
    if (tot == 0) return;  // nothing listed: leave before any setup (uniform over the CTA)
  }
  using C = IdxCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* a_full = bars + 0;
  uint64_t* b_full = bars + 1;     // [STAGES]
  uint64_t* b_empty = bars + 5;    // [STAGES]
  uint64_t* acc_full = bars + 9;   // [NACC]
  uint64_t* acc_empty = bars + 13; // [NACC]
  uint64_t* mma_done = bars + 17;
  uint64_t* a_empty = bars + 18;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 19);
  int* abort_flag = reinterpret_cast<int*>(bars + 20);

  const int64_t lo = (int64_t)blockIdx.x * a.total / gridDim.x;
  const int64_t hi = (int64_t)(blockIdx.x + 1) * a.total / gridDim.x;
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < C::NACC; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 8);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag};
  int32_t* status = a.status;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && lo < hi) {
      tma_prefetch_desc(&mq_hi);
      tma_prefetch_desc(&mk_hi);
      Item w = item_at(a, lo);
      int64_t cur_rt = -1;
      int cur_g = -1, a_loads = 0;
      int issued[C::STAGES] = {};
      for (int64_t k = 0; k < hi - lo; ++k, item_next(a, w)) {
        const int s = (int)(k % C::STAGES);
        if (!mbar_wait(&b_empty[s], (uint32_t)((k / C::STAGES) & 1) ^ 1, ab, status, 101)) break;
        // one product: the hi halves only
        mbar_expect_tx(&b_full[s], a.single ? C::B_BYTES : C::STAGE_BYTES);
        uint8_t* sb = smem + C::OFF_B + s * C::STAGE_BYTES;
        const int32_t brow = (int32_t)(w.g * a.krows + w.n * C::BN);
        for (int c = 0; c < C::KC; ++c) {
          tma_load_2d(sb + c * C::B_TILE, &mk_hi, &b_full[s], c * 64, brow);
          if (!a.single) tma_load_2d(sb + C::B_BYTES + c * C::B_TILE, &mk_lo, &b_full[s], c * 64, brow);
        }
        ++issued[s];
        if (w.rt != cur_rt || w.g != cur_g) {  // new query operand
          if (a_loads > 0 && !mbar_wait(a_empty, (a_loads - 1) & 1, ab, status, 100)) break;
          mbar_expect_tx(a_full, a.single ? C::A_BYTES : 2 * C::A_BYTES);
          const int32_t arow = (int32_t)(w.g * a.nq + w.rt * C::BM);
          for (int c = 0; c < C::KC; ++c) {
            tma_load_2d(smem + C::OFF_AHI + c * C::A_TILE, &mq_hi, a_full, c * 64, arow);
            if (!a.single) tma_load_2d(smem + C::OFF_ALO + c * C::A_TILE, &mq_lo, a_full, c * 64, arow);
          }
          ++a_loads;
          cur_rt = w.rt;
          cur_g = w.g;
        }
      }
      if (ab.set()) {  // let every copy this CTA started land before it exits
        if (a_loads > 0) mbar_wait_drain(a_full, (a_loads - 1) & 1, status, 198);
        for (int s = 0; s < C::STAGES; ++s)
          if (issued[s] > 0) mbar_wait_drain(&b_full[s], (issued[s] - 1) & 1, status, 197);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && lo < hi) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::BM, C::BN, 0, 0);
      const uint32_t a_hi = smem_u32(smem + C::OFF_AHI);
      const uint32_t a_lo = smem_u32(smem + C::OFF_ALO);
      Item w = item_at(a, lo);
      int64_t cur_rt = -1;
      int cur_g = -1, a_uses = 0;
      for (int64_t k = 0; k < hi - lo; ++k, item_next(a, w)) {
        const int s = (int)(k % C::STAGES), acc = (int)(k % C::NACC);
        if (w.rt != cur_rt || w.g != cur_g) {
          if (a_uses > 0) umma_commit(a_empty);  // old operand free once its MMAs finish
          if (!mbar_wait(a_full, a_uses & 1, ab, status, 102)) break;
          ++a_uses;
          cur_rt = w.rt;
          cur_g = w.g;
        }
        if (!mbar_wait(&b_full[s], (uint32_t)((k / C::STAGES) & 1), ab, status, 103)) break;
        if (!mbar_wait(&acc_empty[acc], (uint32_t)((k / C::NACC) & 1) ^ 1, ab, status, 104)) break;
        tc_fence_after();
        const uint32_t b_hi = smem_u32(smem + C::OFF_B + s * C::STAGE_BYTES);
        const uint32_t b_lo = b_hi + C::B_BYTES;
        const uint32_t d_t = tmem + acc * C::BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::A_TILE + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * C::B_TILE + (kk & 3) * 32;
          const uint64_t ahi = sdesc_sw128(a_hi + off, 16, 1024);
          const uint64_t alo = sdesc_sw128(a_lo + off, 16, 1024);
          const uint64_t bhi = sdesc_sw128(b_hi + boff, 16, 1024);
          const uint64_t blo = sdesc_sw128(b_lo + boff, 16, 1024);
          umma_f16(d_t, ahi, bhi, idesc, kk > 0 ? 1u : 0u);
          if (!a.single) {
            umma_f16(d_t, ahi, blo, idesc, 1u);
            umma_f16(d_t, alo, bhi, idesc, 1u);
          }
        }
        umma_commit(&b_empty[s]);
        umma_commit(&acc_full[acc]);
      }
      umma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, status, 199);
    }
  } else {
    // --------------------------------------------------------------- epilogue
    const int q = warp & 3;           // TMEM lane quadrant of this warp
    const int eh = (warp - 2) >> 2;   // which 64 of the tile's 128 columns
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* stg = smem + C::OFF_STG + (warp - 2) * C::STG_BYTES;
    const float ninf = -__int_as_float(0x7f800000);
    const bool vec = (a.nblk & 3) == 0;
    const bool filt = a.tau != nullptr;
    if (lo < hi) {
      Item w = item_at(a, lo);
      float tau_r = 0.f;     // this thread's row threshold (filter mode)
      int64_t seg_n0 = 0;    // first column tile of the current segment
      int cn = 0;            // candidates of the current segment
      for (int64_t k = 0; k < hi - lo; ++k, item_next(a, w)) {
        const int acc = (int)(k % C::NACC);
        const int64_t tl_row = w.rt * C::BM + q * 32;  // first row of this warp, local
        const int64_t t = a.q_begin + tl_row + lane;
        const bool valid = t < a.q_end;
        const int64_t nh = bound_of(a, t);
        float* row = a.scores + ((int64_t)w.g * a.nq + tl_row + lane) * a.nblk;
        const int64_t crow = ((int64_t)w.g * a.nq + tl_row + lane) * 2 + eh;  // candidate list
        if (filt && (k == 0 || w.n == 0)) {  // a new (row tile, group) segment
          seg_n0 = w.n;
          cn = 0;
          tau_r = valid ? a.tau[(int64_t)w.g * a.nq + tl_row + lane] : __int_as_float(0x7fffffff);
        }
        // filter mode keeps full score rows only for rows without a threshold
        const bool keep = !filt || isnan(tau_r);
        const bool store_box = __any_sync(0xffffffffu, valid && keep);
        // outcome made warp-uniform: tcgen05.ld below is warp-collective
        const bool ok = mbar_wait(&acc_full[acc], (uint32_t)((k / C::NACC) & 1), ab, status, 105);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        // both 32-column pieces of this warp's half leave TMEM at once, and
        // the accumulator is released before they are processed
        static_assert(C::BN == 128, "two 32-column pieces per epilogue warp");
        uint32_t va[32], vb[32];
        tmem_ld32(tl + acc * C::BN + eh * 64, va);
        tmem_ld32(tl + acc * C::BN + eh * 64 + 32, vb);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        if (a.round_bf16) {  // the bf16 indexer: every score rounded before any use
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            va[i] = bf16_round_bits(va[i]);
            vb[i] = bf16_round_bits(vb[i]);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t(&v)[32] = h == 0 ? va : vb;
          const int cc = eh * 2 + h;
          const int64_t j0 = w.n * C::BN + cc * 32;
          if (j0 + 32 > nh) {  // the row's last tile: blocks past nh are not historical
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (j0 + i >= nh) v[i] = __float_as_uint(ninf);
          }
          uint32_t fm = 0u;  // this thread's candidates among the 32 columns
          if (filt) {        // (NaN thresholds and -inf scores take nothing)
#pragma unroll
            for (int i = 0; i < 32; ++i) fm |= (uint32_t)(__uint_as_float(v[i]) >= tau_r) << i;
          }
          bool staged = false;  // this thread's row of the tile is in its staging box
          if (a.tma_store) {
            if (store_box) {
              if (j0 >= a.nblk || tl_row >= a.nq) continue;  // box wholly outside (warp-uniform)
              uint8_t* buf = stg;
              if (lane == 0) bulk_wait_read<0>();  // the box last stored from `buf`
              __syncwarp();
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(buf + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                    make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&ms, buf, (int32_t)j0, (int32_t)tl_row, w.g);
                bulk_commit_group();
              }
              staged = true;
            }
          } else if (valid && keep) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const int64_t j = j0 + i;
              if (vec && j + 3 < a.nblk) {
                *reinterpret_cast<uint4*>(row + j) = make_uint4(v[i], v[i + 1], v[i + 2], v[i + 3]);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (j + e < a.nblk) row[j + e] = __uint_as_float(v[i + e]);
              }
            }
          }
          // the candidates' scores are read back from this thread's row of the
          // staging box (staged above when the box was stored, else here once
          // the box's last store has read it)
          uint8_t* mine = stg + lane * 128;
          if (!staged && __any_sync(0xffffffffu, fm != 0u)) {
            if (a.tma_store && lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(mine + ((c ^ (lane & 7)) << 4)) =
                  make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          }
          if (fm != 0u) {
            uint2* cl = a.cand + crow * a.caph;
            const bool front = seg_n0 == 0;
            do {
              const int i = __ffs(fm) - 1;
              fm &= fm - 1u;
              const uint32_t x =
                  *reinterpret_cast<const uint32_t*>(mine + (((i >> 2) ^ (lane & 7)) << 4) + (i & 3) * 4);
              if (cn < a.caph) cl[front ? cn : a.caph - 1 - cn] = make_uint2(x, (uint32_t)(j0 + i));
              ++cn;
            } while (fm != 0u);
          }
        }
        if (filt && valid && (w.n == w.nt - 1 || k == hi - lo - 1)) {  // segment ends
          int32_t* cc = a.ccnt + crow * 2;
          if (seg_n0 == 0) {
            cc[0] = cn;
            if (w.n == w.nt - 1) cc[1] = 0;  // one CTA covered the whole row tile
          } else {
            cc[1] = cn;
            if (w.n != w.nt - 1) report(status, SGQA_ERR_BOUNDS, (int)t);  // a third segment
          }
        }
        if (a.fill_tail && w.n == w.nt - 1 && eh == 0) {
          // columns past the row tile's last computed tile are never historical
          const int64_t jt = w.nt * C::BN;
          if (a.tma_store) {
            if (jt < a.nblk && tl_row < a.nq) {
              if (lane == 0) bulk_wait_read<0>();
              __syncwarp();
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<float4*>(stg + lane * 128 + c * 16) =
                    make_float4(ninf, ninf, ninf, ninf);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                for (int64_t j = jt; j < a.nblk; j += 32)
                  tma_store_3d(&ms, stg, (int32_t)j, (int32_t)tl_row, w.g);
                bulk_commit_group();
                bulk_wait_read<0>();
              }
              __syncwarp();
            }
          } else if (valid) {
            int64_t j = jt;
            if (vec)
              for (; j + 3 < a.nblk; j += 4)
                *reinterpret_cast<float4*>(row + j) = make_float4(ninf, ninf, ninf, ninf);
            for (; j < a.nblk; ++j) row[j] = ninf;
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all<0>();  // stores complete before the CTA's shared memory goes
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

bool make_tmap_scores(CUtensorMap* map, float* base, int64_t nblk, int64_t nq, int Hkv) {
  auto fn = tmap_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)nblk, (cuuint64_t)nq, (cuuint64_t)Hkv};
  cuuint64_t strides[2] = {(cuuint64_t)nblk * 4, (cuuint64_t)(nblk * nq * 4)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_impl(const Dims& dm, const __nv_bfloat16* qhi, const __nv_bfloat16* qlo,
                const __nv_bfloat16* khi, const __nv_bfloat16* klo, int64_t q_begin,
                int64_t q_end, float* scores, bool fill_tail, int32_t* status, cudaStream_t st,
                const IndexMode& mode) {
  using C = IdxCfg<D>;
  IdxArgs a;
  a.nq = q_end - q_begin;
  a.q_begin = q_begin;
  a.q_end = q_end;
  a.q_offset = dm.off;
  a.nblk_full = dm.nblk;
  a.sample = mode.sample ? 1 : 0;
  a.single = (mode.sample || dm.index_bf16) ? 1 : 0;
  a.round_bf16 = (!mode.sample && dm.index_bf16) ? 1 : 0;
  a.nblk = mode.sample ? sampled_cols(dm) : dm.nblk;
  a.krows = (!mode.sample && mode.krows > 0) ? mode.krows : a.nblk;
  a.B = dm.B;
  a.Hkv = dm.Hkv;
  a.fill_tail = fill_tail ? 1 : 0;
  a.tma_store = (a.nblk % 4 == 0 && (reinterpret_cast<uintptr_t>(scores) & 15u) == 0) ? 1 : 0;
  a.scores = scores;
  a.tau = mode.tau;
  a.cand = mode.cand;
  a.ccnt = mode.ccnt;
  a.caph = mode.caph;
  a.flist = mode.flist;
  a.nflist = mode.nflist;
  a.nfl = 0;
  a.status = status;
  // items: sum over row tiles of Hkv * column tiles (same count as the kernel)
  int64_t total = 0, max_nt = 1;
  for (int64_t t0 = q_begin; t0 < q_end; t0 += C::BM) {
    const int64_t t_last = std::min(t0 + C::BM, q_end) - 1;
    int64_t nh = std::min((dm.off + t_last) / dm.B, dm.nblk);
    if (a.sample) nh = (nh >> 6) << 3;
    const int64_t nt = std::max<int64_t>(1, (nh + C::BN - 1) / C::BN);
    total += dm.Hkv * nt;
    max_nt = std::max(max_nt, nt);
  }
  if (a.nblk == 0) return SGQA_OK;
  a.total = total;
  CUtensorMap m_qhi, m_qlo, m_khi, m_klo, m_s;
  const uint64_t row_bytes = (uint64_t)D * 2;
  if (!make_tmap_2d_bf16(&m_qhi, qhi, D, (uint64_t)dm.Hkv * a.nq, row_bytes, 64, C::BM) ||
      !make_tmap_2d_bf16(&m_qlo, qlo, D, (uint64_t)dm.Hkv * a.nq, row_bytes, 64, C::BM) ||
      !make_tmap_2d_bf16(&m_khi, khi, D, (uint64_t)dm.Hkv * a.krows, row_bytes, 64, C::BN) ||
      !make_tmap_2d_bf16(&m_klo, klo, D, (uint64_t)dm.Hkv * a.krows, row_bytes, 64, C::BN))
    return SGQA_ERR_CUDA;
  if (a.tma_store) {
    if (!make_tmap_scores(&m_s, scores, a.nblk, a.nq, dm.Hkv)) return SGQA_ERR_CUDA;
  } else {
    std::memset(&m_s, 0, sizeof(m_s));
  }
  if (cudaFuncSetAttribute(k_index_scores<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM) != cudaSuccess)
    return SGQA_ERR_CUDA;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0)
    return SGQA_ERR_CUDA;
  // refill mode: the items are counted on the device; one CTA per SM
  int64_t ctas = a.flist != nullptr ? nsm : std::min<int64_t>(total, nsm);
  // filter mode: every CTA takes at least a whole row tile's items, so a row
  // tile is split between at most two CTAs (front and back candidate parts)
  if (a.tau != nullptr) ctas = std::max<int64_t>(1, std::min<int64_t>(ctas, total / max_nt));
  const unsigned grid = (unsigned)ctas;
  log_begin(a.sample ? SGQA_K_SAMPLE_SCORES : SGQA_K_INDEX_SCORES, st);
  k_index_scores<D><<<grid, C::NTHREADS, C::SMEM, st>>>(m_qhi, m_qlo, m_khi, m_klo, m_s, a);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

}  // namespace

int launch_index_scores(const Dims& dm, const __nv_bfloat16* qhi, const __nv_bfloat16* qlo,
                        const __nv_bfloat16* khi, const __nv_bfloat16* klo, int64_t q_begin,
                        int64_t q_end, float* scores, bool fill_tail, int32_t* status,
                        cudaStream_t st, const IndexMode* mode) {
  if (q_end <= q_begin || dm.nblk == 0) return SGQA_OK;  // nothing to score
  const IndexMode plain{};
  const IndexMode& m = mode ? *mode : plain;
  if (m.tau != nullptr && (m.cand == nullptr || m.ccnt == nullptr || m.caph < 1))
    return SGQA_ERR_INVALID_ARG;
  if (dm.d == 128)
    return launch_impl<128>(dm, qhi, qlo, khi, klo, q_begin, q_end, scores, fill_tail, status, st,
                            m);
  if (dm.d == 64)
    return launch_impl<64>(dm, qhi, qlo, khi, klo, q_begin, q_end, scores, fill_tail, status, st,
                           m);
  return SGQA_ERR_UNSUPPORTED;
}

}  // namespace sgqa
