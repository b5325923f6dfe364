// Main-path block-sparse GQA attention on tcgen05 tensor cores.
//
// "Inside Step 5 Preview" (StepFun blog), section Sparse GQA, Figure 3
// caption: the main path reads the original K/V of the selected historical
// blocks plus the causally visible positions of the current block; paragraph
// "Efficient implementation of sparse attention": the top-k results of
// adjacent tokens are unioned so their overlapping work runs as dense matrix
// products.
//
// Work item = (KV group g, union tile tau, sub-tile s).  A sub-tile is QS =
// min(128 / G, W) consecutive queries of the tile; its QS * G query heads form
// the M = 128 rows of every MMA (row r = query r / G, head r % G).  The key
// list of a work item is every union block that some query of the sub-tile
// selected (mode MASKED; every union block in mode FULL) and lies before the
// sub-tile's first current block, followed by the sub-tile's current blocks.
// Keys are gathered 128 per stage.
//
// Warps 0-1 build each stage's block list and gather K/V rows into 128-byte
// swizzled shared tiles with cp.async; warp 2 issues S = Q K^T into a
// double-buffered TMEM tile and O += P V into a TMEM accumulator; warps 3-6
// hold one row each: they read S from TMEM, apply the per-query block mask
// and the causal cut of the current block, run the fp32 online softmax
// (rescaling O in TMEM only when the running maximum grows by more than 2^8),
// write P (bf16) to shared memory for the PV product, and finally normalise
// O and write O and the log-sum-exp.
#include "common.cuh"
#include "internal.h"

namespace sgqa {
namespace {

constexpr unsigned FULL = 0xffffffffu;

template <int D>
struct AttnCfg {
  static constexpr int BM = 128;  // rows per MMA
  static constexpr int KB = 128;  // keys per stage
  static constexpr int S = 2;     // K/V stages
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_TILE = KB * D * 2;
  static constexpr int P_BYTES = BM * KB * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + S * KV_TILE;
  static constexpr int OFF_P = OFF_V + S * KV_TILE;
  static constexpr int OFF_META = OFF_P + P_BYTES;
  static constexpr int OFF_BAR = OFF_META + S * 1552;  // sizeof(Meta) rounded
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;  // S[2] at 0 / 128, O at 256
  static constexpr int NTHREADS = 224;
};

struct Meta {          // one stage's block list
  int32_t nb;          // blocks in the stage
  int32_t last;        // last stage of the work item
  int32_t blk[128];
  uint64_t mask[128];  // bit qi: query qi of the sub-tile may attend the block
};
static_assert(sizeof(Meta) <= 1552, "meta size");

struct AttnArgs {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const int32_t* page_table;
  const int64_t* uoff;
  const int32_t* ulen;
  const int32_t* ublk;
  const uint64_t* umask;
  void* O;
  float* lse;
  int64_t T, Tkv, off, nblk, lay_tau0, lay_ntiles, tau_begin, tau_end;
  int H, Hkv, G, B, W, ps, QS, nsub, mode, out_f32;
  float scale_log2;
  int32_t* status;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
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

// Byte offset of 16-byte unit u (0..7) of row r inside a [rows][128 B] tile
// with the 128-byte swizzle that TMA and UMMA use.
__device__ __forceinline__ uint32_t sw128(int r, int u) {
  return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4));
}

// State of the block-list generator of one work item (kept by warp 0).
struct Gen {
  int64_t cur, end;  // cursor into the tile's union entries
  int64_t c0, c_last, nd;
  int phase;         // 0: historical union entries, 1: current blocks, 2: done
};

// Fill `m` with up to nbps blocks.  Warp-cooperative (warp 0).
__device__ void gen_stage(const AttnArgs& a, Gen& gs, Meta& m, int nbps, int sh, uint64_t qmask) {
  const int lane = lane_id();
  int n = 0;
  while (gs.phase == 0 && n < nbps) {
    if (gs.cur >= gs.end) {
      gs.phase = 1;
      break;
    }
    const int64_t idx = gs.cur + lane;
    const bool valid = idx < gs.end;
    const int32_t b = valid ? a.ublk[idx] : 0x7fffffff;
    const uint64_t um = valid ? a.umask[idx] : 0ull;
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
      // take the first `room` entries of this chunk only
      uint32_t mm = pm;
      for (int k = 1; k < room; ++k) mm &= mm - 1;
      const int last_lane = __ffs(mm) - 1;
      if (((pm >> lane) & 1u) && rank < room) {
        m.blk[n + rank] = b;
        m.mask[n + rank] = sub;
      }
      n += room;
      gs.cur += last_lane + 1;
    }
  }
  __syncwarp();
  if (gs.phase == 1 && n < nbps) {
    int64_t cur = gs.cur, nd = gs.nd;
    if (lane == 0) {
      while (n < nbps && nd <= gs.c_last) {
        while (cur < gs.end && a.ublk[cur] < nd) ++cur;
        const uint64_t um = (cur < gs.end && a.ublk[cur] == nd) ? a.umask[cur] : 0ull;
        uint64_t sub;
        if (a.mode == SGQA_UNION_MASKED)
          sub = (um >> sh) & qmask;
        else
          sub = (cur < gs.end && a.ublk[cur] == nd) ? ~0ull : 0ull;
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
}

template <int D>
__device__ __forceinline__ const __nv_bfloat16* kv_row(const AttnArgs& a, const __nv_bfloat16* base,
                                                       int g, int64_t p) {
  if (a.ps > 0) {
    const int64_t phys = a.page_table[p / a.ps];
    return base + ((phys * a.Hkv + g) * a.ps + (p % a.ps)) * (int64_t)D;
  }
  return base + (p * a.Hkv + g) * (int64_t)D;
}

template <int D, int B>
__global__ void __launch_bounds__(224, 1) k_sparse_attn(AttnArgs a) {
  using C = AttnCfg<D>;
  constexpr int NBPS = C::KB / B;  // blocks per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Meta* meta = reinterpret_cast<Meta*>(smem + C::OFF_META);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;    // [S]
  uint64_t* kv_empty = bars + 3;   // [S]
  uint64_t* meta_rdy = bars + 5;   // [S]
  uint64_t* s_full = bars + 7;     // [2]
  uint64_t* s_empty = bars + 9;    // [2]
  uint64_t* p_full = bars + 11;
  uint64_t* p_empty = bars + 12;
  uint64_t* mma_done = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  int* abort_flag = reinterpret_cast<int*>(bars + 15);

  // ---- work item
  const int64_t item = blockIdx.x;
  const int64_t per_tile = (int64_t)a.Hkv * a.nsub;
  const int64_t tau = a.tau_end - 1 - item / per_tile;  // heavy tiles first
  const int g = (int)((item % per_tile) / a.nsub);
  const int s = (int)(item % a.nsub);
  const int64_t tile_first = tau * a.W;
  const int64_t tile_len = (a.T - tile_first) < a.W ? (a.T - tile_first) : a.W;
  if ((int64_t)s * a.QS >= tile_len) return;  // uniform exit: empty sub-tile
  const int64_t tq0 = tile_first + (int64_t)s * a.QS;
  const int nq_sub = (int)((tile_len - (int64_t)s * a.QS) < a.QS ? (tile_len - (int64_t)s * a.QS) : a.QS);
  const int rows = nq_sub * a.G;
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 128);
    for (int i = 0; i < C::S; ++i) {
      mbar_init(&kv_full[i], 128);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&meta_rdy[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(p_empty, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag};

  if (warp < 2) {
    // ============================================================== producer
    const int pt = threadIdx.x;  // 0..63
    uint8_t* sQ = smem + C::OFF_Q;
    for (int idx = pt; idx < C::BM * (D / 8); idx += 64) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      uint8_t* dst = sQ + (c >> 3) * (C::BM * 128) + sw128(r, c & 7);
      if (r < rows) {
        const int qi = r / a.G, h = r % a.G;
        cp_async16(dst, a.Q + ((tq0 + qi) * a.H + (int64_t)g * a.G + h) * D + c * 8);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    mbar_arrive(q_full);
    cp_async_arrive(q_full);

    Gen gs;
    const int64_t lt = (int64_t)g * a.lay_ntiles + (tau - a.lay_tau0);
    gs.cur = a.uoff[lt];
    gs.end = gs.cur + a.ulen[lt];
    gs.c0 = (a.off + tq0) / B;
    gs.c_last = (a.off + tq0 + nq_sub - 1) / B;
    gs.nd = gs.c0;
    gs.phase = 0;
    const int sh = s * a.QS;
    const uint64_t qmask = nq_sub >= 64 ? ~0ull : ((1ull << nq_sub) - 1ull);

    for (int i = 0;; ++i) {
      const int st = i % C::S;
      const uint32_t ph = (uint32_t)((i / C::S) & 1);
      if (!mbar_wait(&kv_empty[st], ph ^ 1u, ab, a.status, 201)) break;
      Meta& m = meta[st];
      if (warp == 0) {
        gen_stage(a, gs, m, NBPS, sh, qmask);
        if (lane == 0) mbar_arrive(&meta_rdy[st]);
      } else {
        if (!mbar_wait(&meta_rdy[st], ph, ab, a.status, 202)) break;
      }
      const int nkeys = m.nb * B;
      const int last = m.last;
      uint8_t* sK = smem + C::OFF_K + st * C::KV_TILE;
      uint8_t* sV = smem + C::OFF_V + st * C::KV_TILE;
      for (int idx = pt; idx < C::KB * (D / 8); idx += 64) {
        const int k = idx / (D / 8), c = idx % (D / 8);
        const uint32_t o = (c >> 3) * (C::KB * 128) + sw128(k, c & 7);
        const int64_t p = k < nkeys ? (int64_t)m.blk[k / B] * B + (k % B) : a.Tkv;
        if (p < a.Tkv) {  // a partial current block ends at the last key
          cp_async16(sK + o, kv_row<D>(a, a.K, g, p) + c * 8);
          cp_async16(sV + o, kv_row<D>(a, a.V, g, p) + c * 8);
        } else {
          *reinterpret_cast<uint4*>(sK + o) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(sV + o) = make_uint4(0, 0, 0, 0);
        }
      }
      mbar_arrive(&kv_full[st]);
      cp_async_arrive(&kv_full[st]);
      if (last) break;
    }
    cp_async_wait_all();
  } else if (warp == 2) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(C::BM, C::KB, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(C::BM, D, 0, 1);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      const uint32_t sP = smem_u32(smem + C::OFF_P);
      const uint32_t tO = tmem + 256;
      bool ok = mbar_wait(q_full, 0, ab, a.status, 203);
      fence_proxy_async_smem();
      // S_j = Q K_j^T into TMEM buffer j % 2
      auto issue_qk = [&](int j) -> bool {
        const int st = j % C::S;
        if (!mbar_wait(&kv_full[st], (uint32_t)((j / C::S) & 1), ab, a.status, 204)) return false;
        fence_proxy_async_smem();
        if (!mbar_wait(&s_empty[j & 1], (uint32_t)(((j >> 1) & 1) ^ 1), ab, a.status, 205))
          return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + C::OFF_K + st * C::KV_TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * (C::KB * 128) + (kk & 3) * 32;
          umma_f16(tmem + (j & 1) * 128, sdesc_sw128(sQ + off, 16, 1024),
                   sdesc_sw128(sK + koff, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int i = 0; ok; ++i) {
        const int st = i % C::S;
        const bool last = meta[st].last != 0;
        if (!last && !issue_qk(i + 1)) break;
        if (!mbar_wait(p_full, (uint32_t)(i & 1), ab, a.status, 206)) break;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + C::OFF_V + st * C::KV_TILE);
#pragma unroll
        for (int kk = 0; kk < C::KB / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
          umma_f16(tO, sdesc_sw128(sP + poff, 16, 1024),
                   sdesc_sw128(sV + kk * 16 * 128, C::KB * 128, 1024), idesc_pv,
                   (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(p_empty);
        umma_commit(&kv_empty[st]);
        if (last) break;
      }
      umma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, a.status, 299);
    }
  } else {
    // =============================================================== softmax
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const bool row_ok = r < rows;
    const int qi = r / a.G, h = r % a.G;
    const int64_t t = tq0 + qi;
    const int64_t pos = a.off + t;
    const int64_t cur = pos / B;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float ninf = -__int_as_float(0x7f800000);
    uint8_t* sP = smem + C::OFF_P;
    float m_used = ninf, l = 0.0f;
    int i = 0;
    bool ok = true;
    for (;; ++i) {
      const int st = i % C::S;
      // waits are polled per thread but their outcome is made warp-uniform:
      // the tcgen05.ld/st below are warp-collective
      bool w = mbar_wait(&s_full[i & 1], (uint32_t)((i >> 1) & 1), ab, a.status, 207) &&
               mbar_wait(&kv_full[st], (uint32_t)((i / C::S) & 1), ab, a.status, 208);
      if (!__all_sync(FULL, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tl + (i & 1) * 128 + cc * 32, sv[cc]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[i & 1]);
      const Meta& m = meta[st];
      const int nb = m.nb;
      const bool last = m.last != 0;
      // mask and running maximum (log2 units)
      float smax = ninf;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int k = cc * 32 + e;
          const int bs = k / B;
          bool allowed = false;
          if (row_ok && bs < nb) {
            const int64_t b = m.blk[bs];
            const bool hist_ok = ((m.mask[bs] >> qi) & 1ull) && b < cur;
            const bool cur_ok = b == cur && (b * B + (k % B)) <= pos;
            allowed = hist_ok || cur_ok;
          }
          const float x = allowed ? __uint_as_float(sv[cc][e]) * a.scale_log2 : ninf;
          sv[cc][e] = __float_as_uint(x);
          smax = fmaxf(smax, x);
        }
      }
      // Raise the reference maximum when this stage exceeds it by more than 2^8.
      // O holds contributions under the old maximum, so it is rescaled once
      // PV_{i-1} is done; the whole warp takes that path together (rows that do
      // not need it scale by 1).
      const bool raise = smax > m_used + 8.0f;
      const bool rescale = raise && m_used != ninf;
      if (__any_sync(FULL, rescale)) {
        bool w2 = mbar_wait(p_empty, (uint32_t)((i - 1) & 1), ab, a.status, 209);
        if (!__all_sync(FULL, w2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = rescale ? ex2(m_used - smax) : 1.0f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          tmem_ld32(tl + 256 + cc * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
          tmem_st32(tl + 256 + cc * 32, ov);
        }
        tmem_wait_st();
        l *= f;
      }
      if (raise) m_used = smax;
      // probabilities -> bf16 pairs
      uint32_t pk[64];
      float rs = 0.0f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float x0 = __uint_as_float(sv[cc][e]), x1 = __uint_as_float(sv[cc][e + 1]);
          const float p0 = x0 == ninf ? 0.0f : ex2(x0 - m_used);
          const float p1 = x1 == ninf ? 0.0f : ex2(x1 - m_used);
          rs += p0 + p1;
          pk[(cc * 32 + e) / 2] = pack_bf16x2(p0, p1);
        }
      }
      l += rs;
      if (i > 0) {
        bool w3 = mbar_wait(p_empty, (uint32_t)((i - 1) & 1), ab, a.status, 210);
        if (!__all_sync(FULL, w3)) {
          ok = false;
          break;
        }
      }
      // P row r: keys 8u..8u+7 of chunk c at unit u (swizzled)
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = u >> 3;
        uint4 v = make_uint4(pk[u * 4 + 0], pk[u * 4 + 1], pk[u * 4 + 2], pk[u * 4 + 3]);
        *reinterpret_cast<uint4*>(sP + c * (C::BM * 128) + sw128(r, u & 7)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      if (last) break;
    }
    // ---- epilogue: O / l and the log-sum-exp
    bool fin = ok && mbar_wait(p_empty, (uint32_t)(i & 1), ab, a.status, 211);
    if (__all_sync(FULL, fin)) {
      tc_fence_after();
      const float inv = row_ok && l > 0.0f ? 1.0f / l : 0.0f;
      const int64_t hq = (int64_t)g * a.G + h;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        tmem_ld32(tl + 256 + cc * 32, ov);
        tmem_wait_ld();
        if (row_ok) {
          if (a.out_f32) {
            float* dst = static_cast<float*>(a.O) + (t * a.H + hq) * D + cc * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + e) =
                  make_float4(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                              __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.O) + (t * a.H + hq) * D + cc * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(ov[e + 4]) * inv, __uint_as_float(ov[e + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(ov[e + 6]) * inv, __uint_as_float(ov[e + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + e) = v;
            }
          }
        }
      }
      if (row_ok) a.lse[hq * a.T + t] = (m_used + __log2f(l)) * 0.69314718055994531f;
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int B>
int launch_db(const AttnArgs& a, int64_t items, cudaStream_t st) {
  using C = AttnCfg<D>;
  if (cudaFuncSetAttribute(k_sparse_attn<D, B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM) != cudaSuccess)
    return SGQA_ERR_CUDA;
  log_begin(SGQA_K_ATTN, st);
  k_sparse_attn<D, B><<<(unsigned)items, C::NTHREADS, C::SMEM, st>>>(a);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

template <int D>
int launch_d(const AttnArgs& a, int B, int64_t items, cudaStream_t st) {
  switch (B) {
    case 1: return launch_db<D, 1>(a, items, st);
    case 2: return launch_db<D, 2>(a, items, st);
    case 4: return launch_db<D, 4>(a, items, st);
    case 8: return launch_db<D, 8>(a, items, st);
    case 16: return launch_db<D, 16>(a, items, st);
    default: return SGQA_ERR_UNSUPPORTED;
  }
}

}  // namespace

int launch_sparse_attn_layout(const Dims& dm, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                              const __nv_bfloat16* V, const int32_t* page_table,
                              const int64_t* union_off, const int32_t* union_len,
                              const int32_t* union_blk, const uint64_t* union_mask, void* O,
                              float* lse, int64_t tau_begin, int64_t tau_end, int64_t lay_tau0,
                              int64_t lay_ntiles, int32_t* status, cudaStream_t st) {
  if (tau_end <= tau_begin) return SGQA_OK;
  if (dm.G > 128) return SGQA_ERR_UNSUPPORTED;
  AttnArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.page_table = page_table;
  a.uoff = union_off;
  a.ulen = union_len;
  a.ublk = union_blk;
  a.umask = union_mask;
  a.O = O;
  a.lse = lse;
  a.T = dm.T;
  a.Tkv = dm.Tkv;
  a.off = dm.off;
  a.nblk = dm.nblk;
  a.lay_tau0 = lay_tau0;
  a.lay_ntiles = lay_ntiles;
  a.tau_begin = tau_begin;
  a.tau_end = tau_end;
  a.H = dm.H;
  a.Hkv = dm.Hkv;
  a.G = dm.G;
  a.B = dm.B;
  a.W = dm.W;
  a.ps = dm.ps;
  a.QS = 128 / dm.G < dm.W ? 128 / dm.G : dm.W;
  a.nsub = (dm.W + a.QS - 1) / a.QS;
  a.mode = dm.mode;
  a.out_f32 = dm.dtype == SGQA_FP32;
  a.scale_log2 = dm.scale * 1.4426950408889634f;
  a.status = status;
  const int64_t items = (tau_end - tau_begin) * dm.Hkv * a.nsub;
  if (dm.d == 128) return launch_d<128>(a, dm.B, items, st);
  if (dm.d == 64) return launch_d<64>(a, dm.B, items, st);
  return SGQA_ERR_UNSUPPORTED;
}

int launch_sparse_attn(const Dims& dm, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                       const __nv_bfloat16* V, const int32_t* page_table,
                       const int64_t* union_off, const int32_t* union_len,
                       const int32_t* union_blk, const uint64_t* union_mask, void* O, float* lse,
                       int64_t tau_begin, int64_t tau_end, int32_t* status, cudaStream_t st) {
  return launch_sparse_attn_layout(dm, Q, K, V, page_table, union_off, union_len, union_blk,
                                   union_mask, O, lse, tau_begin, tau_end, 0, dm.ntiles, status,
                                   st);
}

}  // namespace sgqa
