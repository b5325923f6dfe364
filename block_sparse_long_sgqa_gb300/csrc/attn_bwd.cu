// Backward of the block-sparse GQA attention on tcgen05 tensor cores.
//
// "Inside Step 5 Preview" (StepFun blog), section Sparse GQA: the layer is
// used in training as well as inference, so the main path's attention needs
// its gradients.  With P the softmax over a row's allowed positions (the
// same key sets as the forward: Figure 3 caption, selected historical blocks
// plus the causal part of the current block), dO the gradient of the output
// and D = rowsum(dO * O):
//   dP = dO V^T,   dS = P * (dP - D),
//   dQ = scale * dS K,   dK = scale * dS^T Q,   dV = P^T dO.
// P is recomputed from the forward's log-sum-exp.  Two kernels write the
// three gradients, each exactly once, with no atomics on them (the results do
// not depend on scheduling):
//
//  k_attn_bwd_dq   query-major, one work item per (KV group, union tile,
//                  sub-tile) as in the forward, over the same stage lists of
//                  128 gathered keys; S and dP are computed in halves of 64
//                  keys into double-buffered TMEM so the MMAs of one half run
//                  while the softmax warps turn the other into dS, and
//                  dQ += dS K accumulates in TMEM.
//  k_attn_bwd_dkv  key-major, one work item per (KV group, key stage of 128
//                  consecutive keys); it walks, in tile order, the query
//                  sub-tiles that attend any of its keys (found through a
//                  per-stage bitmap of tiles and each tile's first union slot
//                  in the stage, built by k_bwd_index), computes S^T = K Q^T
//                  and dP^T = V dO^T in halves of 64 query rows, and
//                  accumulates dV += P^T dO and dK += dS^T Q in TMEM.
//
// K and V are read from the block-packed copies the forward uses (B >= 8).
#include "attn_common.cuh"

namespace sgqa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdArgs {
  // read by gen_stage / union_entry
  const int32_t* ublk;
  const uint64_t* umask;
  int mode;
  const int64_t* uoff;
  const int32_t* ulen;
  const __nv_bfloat16* Kp;  // block-packed K and V: [Hkv][nblkp + 1][B * D]
  const __nv_bfloat16* Vp;
  int64_t nblkp;            // packed blocks per head (the last one may be partial)
  const float* lse;         // [H][T] natural log
  const float* Dl;          // [H][T] rowsum(dO * O)
  float* dQ;                // [T][H][D]
  float* dK;                // [Tkv][Hkv][D]
  float* dV;
  const uint32_t* kbits;    // [Hkv][nks][nw]: tiles attending key stage ks
  const int32_t* first;     // [Hkv][ntiles][nks]: the tile's first union slot in the stage, -1
  int64_t T, Tkv, off, ntiles, nks, nw;
  int H, Hkv, G, lgG, B, W, QS, nsub;
  float scale, scale_log2;
  int32_t* status;
};

// ------------------------------------------------------------------ helpers
// D[h][t] = sum_i dO[t][h][i] O[t][h][i] (fp32), one warp per (t, h).
template <int D>
__global__ void k_bwd_delta(const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO,
                            int64_t T, int H, float* __restrict__ Dl) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= T * H) return;
  const int lane = threadIdx.x & 31;
  float acc = 0.0f;
#pragma unroll
  for (int i = lane * 4; i < D; i += 128) {
    const uint2 o = *reinterpret_cast<const uint2*>(O + row * D + i);
    const uint2 g = *reinterpret_cast<const uint2*>(dO + row * D + i);
    const __nv_bfloat162 o0 = *reinterpret_cast<const __nv_bfloat162*>(&o.x);
    const __nv_bfloat162 o1 = *reinterpret_cast<const __nv_bfloat162*>(&o.y);
    const __nv_bfloat162 g0 = *reinterpret_cast<const __nv_bfloat162*>(&g.x);
    const __nv_bfloat162 g1 = *reinterpret_cast<const __nv_bfloat162*>(&g.y);
    acc = fmaf(__low2float(o0), __low2float(g0), acc);
    acc = fmaf(__high2float(o0), __high2float(g0), acc);
    acc = fmaf(__low2float(o1), __low2float(g1), acc);
    acc = fmaf(__high2float(o1), __high2float(g1), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL, acc, o);
  if (lane == 0) {
    const int64_t t = row / H, h = row % H;
    Dl[h * T + t] = acc;
  }
}

// The key stages each union tile attends: bit tau of kbits[g][ks] and the
// tile's first union slot of the stage in first[g][tau][ks] (the union lists
// are sorted by block, so a stage's entries are consecutive); a tile's
// queries also attend their current blocks' stages.  One warp per (g, tau).
__global__ void k_bwd_index(BwdArgs a, int SB) {
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (wid >= (int64_t)a.Hkv * a.ntiles) return;
  const int lane = threadIdx.x & 31;
  const int g = (int)(wid / a.ntiles);
  const int64_t tau = wid % a.ntiles;
  const int64_t o = a.uoff[wid], n = a.ulen[wid];
  const uint32_t bit = 1u << (tau & 31);
  uint32_t* kb = const_cast<uint32_t*>(a.kbits) + (int64_t)g * a.nks * a.nw + (tau >> 5);
  int32_t* fs = const_cast<int32_t*>(a.first) + wid * a.nks;
  for (int64_t x0 = 0; x0 < n; x0 += 32) {
    const int64_t x = x0 + lane;
    if (x < n) {
      const int64_t ks = a.ublk[o + x] / SB;
      const int64_t kp = x > 0 ? a.ublk[o + x - 1] / SB : -1;
      if (ks != kp) {
        fs[ks] = (int32_t)(o + x);
        atomicOr(kb + ks * a.nw, bit);
      }
    }
  }
  const int64_t t0 = tau * a.W;
  const int64_t len = (a.T - t0) < a.W ? (a.T - t0) : a.W;
  const int64_t c0 = (a.off + t0) / a.B, cl = (a.off + t0 + len - 1) / a.B;
  for (int64_t ks = c0 / SB + lane; ks <= cl / SB; ks += 32) atomicOr(kb + ks * a.nw, bit);
}

// ===================================================================== dQ
template <int D, int B>
struct DqCfg {
  static constexpr int BM = 128, KB = 128, NBPS = KB / B;
  static constexpr int SK = 2, SV = 2, NM = 8, KC = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_TILE = KB * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + Q_BYTES;
  static constexpr int OFF_K = OFF_DO + Q_BYTES;
  static constexpr int OFF_V = OFF_K + SK * KV_TILE;
  static constexpr int OFF_META = OFF_V + SV * KV_TILE;
  static constexpr int META_BYTES = (int)((sizeof(MetaT<NBPS>) + 15) / 16 * 16);
  static constexpr int OFF_BAR = OFF_META + NM * META_BYTES;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;  // S[2] at 0/64, dP[2] at 128/192, dQ at 256
  static constexpr int NTHREADS = 384;
  static_assert(SMEM <= 232448, "shared memory plan");
};

template <int D, int B>
__global__ void __launch_bounds__(384, 1)
    k_attn_bwd_dq(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
                  BwdArgs a) {
  using C = DqCfg<D, B>;
  using Meta = MetaT<C::NBPS>;
  constexpr int NBPS = C::NBPS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  auto meta_at = [&](int i) -> Meta& {
    return *reinterpret_cast<Meta*>(smem + C::OFF_META + i * C::META_BYTES);
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [SK]
  uint64_t* k_empty = bars + 3;   // [SK]
  uint64_t* v_full = bars + 5;    // [SV]
  uint64_t* v_empty = bars + 7;   // [SV]
  uint64_t* m_full = bars + 9;    // [NM]
  uint64_t* m_empty = bars + 17;  // [NM]
  uint64_t* s_full = bars + 25;   // [2] S and dP of a half-stage computed
  uint64_t* ds_full = bars + 27;  // [2] dS of a half-stage written
  uint64_t* dq_done = bars + 29;
  uint64_t* mma_done = bars + 30;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 31);
  int* abort_flag = reinterpret_cast<int*>(bars + 32);
  volatile int* n_stages = reinterpret_cast<volatile int*>(bars + 33);

  const int64_t item = blockIdx.x;
  const int64_t per_tile = (int64_t)a.Hkv * a.nsub;
  const int64_t tau = a.ntiles - 1 - item / per_tile;  // heavy tiles first
  const int g = (int)((item % per_tile) / a.nsub);
  const int s = (int)(item % a.nsub);
  const int64_t tile_first = tau * a.W;
  const int64_t tile_len = (a.T - tile_first) < a.W ? (a.T - tile_first) : a.W;
  if ((int64_t)s * a.QS >= tile_len) return;  // uniform exit: empty sub-tile
  const int64_t tq0 = tile_first + (int64_t)s * a.QS;
  const int nq_sub =
      (int)((tile_len - (int64_t)s * a.QS) < a.QS ? (tile_len - (int64_t)s * a.QS) : a.QS);
  const int rows = nq_sub * a.G;
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::SK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < C::SV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < C::NM; ++i) {
      mbar_init(&m_full[i], 1);
      mbar_init(&m_empty[i], 10);  // both softmax groups (8 warps) + the K and V producers
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&ds_full[i], 4);
    }
    mbar_init(dq_done, 1);
    mbar_init(mma_done, 1);
    *n_stages = 0x7fffffff;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag};

  if (warp == 0) {
    // ============================================ block lists + Q and dO loads
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mdo);
      const uint32_t box = (uint32_t)(C::KC * 128 * a.G * a.QS);
      mbar_expect_tx(q_full, 2 * box);
      for (int c = 0; c < C::KC; ++c) {
        tma_load_3d(smem + C::OFF_Q + c * (C::BM * 128), &mq, q_full, c * 64, g * a.G, (int32_t)tq0);
        tma_load_3d(smem + C::OFF_DO + c * (C::BM * 128), &mdo, q_full, c * 64, g * a.G,
                    (int32_t)tq0);
      }
    }
    Gen gs;
    const int64_t lt = (int64_t)g * a.ntiles + tau;
    gs.cur = a.uoff[lt];
    gs.end = gs.cur + a.ulen[lt];
    gs.c0 = (a.off + tq0) / B;
    gs.c_last = (a.off + tq0 + nq_sub - 1) / B;
    gs.nd = gs.c0;
    gs.phase = 0;
    gs.pf_at = -1;
    const int sh = s * a.QS;
    const uint64_t qmask = nq_sub >= 64 ? ~0ull : ((1ull << nq_sub) - 1ull);
    for (int i = 0;; ++i) {
      const int ms = i % C::NM;
      const bool w = mbar_wait(&m_empty[ms], (uint32_t)(((i / C::NM) & 1) ^ 1), ab, a.status, 401);
      if (!__all_sync(FULL, w)) break;
      Meta& m = meta_at(ms);
      gen_stage<false>(a, gs, m, NBPS, sh, qmask, nq_sub);
      if (lane == 0 && m.last) {
        *n_stages = i + 1;
        __threadfence_block();
      }
      if (lane == 0) mbar_arrive(&m_full[ms]);
      if (m.last) break;
    }
    if (lane == 0 && ab.set()) mbar_wait_drain(q_full, 0, a.status, 491);
  } else if (warp == 11 || warp == 1) {
    // ================================================== K (warp 11), V (warp 1)
    const bool isK = warp == 11;
    const int SL = isK ? C::SK : C::SV;
    uint64_t* full = isK ? k_full : v_full;
    uint64_t* empty = isK ? k_empty : v_empty;
    const __nv_bfloat16* base = (isK ? a.Kp : a.Vp) + (int64_t)g * (a.nblkp + 1) * (B * D);
    int issued[2] = {0, 0};
    for (int i = 0;; ++i) {
      const int ms = i % C::NM, ks = i % SL;
      bool w = mbar_wait(&m_full[ms], (uint32_t)((i / C::NM) & 1), ab, a.status, 402) &&
               mbar_wait(&empty[ks], (uint32_t)(((i / SL) & 1) ^ 1), ab, a.status, 403);
      if (!__all_sync(FULL, w)) break;
      const Meta& m = meta_at(ms);
      const bool last = m.last != 0;
      uint8_t* dst = smem + (isK ? C::OFF_K : C::OFF_V) + ks * C::KV_TILE;
      if (lane == 0) mbar_expect_tx(&full[ks], C::KV_TILE);
      __syncwarp();
      copy_blocks<NBPS>(dst, base, m.blk, m.nb, a.nblkp, B * D, &full[ks]);
      ++issued[ks];
      __syncwarp();
      if (lane == 0) mbar_arrive(&m_empty[ms]);
      if (last) break;
    }
    if (lane == 0 && ab.set())
      for (int k = 0; k < SL; ++k)
        if (issued[k] > 0) mbar_wait_drain(&full[k], (issued[k] - 1) & 1, a.status, 492);
  } else if (warp == 2) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_h = idesc_bf16_f32(C::BM, 64, 0, 0);
      constexpr uint32_t idesc_dq = idesc_bf16_f32(C::BM, D, 0, 1);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sdO = smem_u32(smem + C::OFF_DO);
      bool ok = mbar_wait(q_full, 0, ab, a.status, 404);
      // S_h = Q K_h^T and dP_h = dO V_h^T for half-stage h (keys 64 e .. of stage h / 2)
      auto do_sdp = [&](int h) {
        const int i = h >> 1, e = h & 1;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + C::OFF_K + (i % C::SK) * C::KV_TILE);
        const uint32_t sV = smem_u32(smem + C::OFF_V + (i % C::SV) * C::KV_TILE);
        const uint32_t hoff = (uint32_t)e * 8u * (C::KC * 1024);  // 8 key groups of 8
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
          const uint32_t boff = hoff + (kk >> 2) * 1024 + (kk & 3) * 32;
          umma_f16(tmem + e * 64, sdesc_sw128(sQ + aoff, 16, 1024),
                   sdesc_sw128(sK + boff, 16, C::KC * 1024), idesc_h, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
          const uint32_t boff = hoff + (kk >> 2) * 1024 + (kk & 3) * 32;
          umma_f16(tmem + 128 + e * 64, sdesc_sw128(sdO + aoff, 16, 1024),
                   sdesc_sw128(sV + boff, 16, C::KC * 1024), idesc_h, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[e]);
        if (e == 1) umma_commit(&v_empty[i % C::SV]);
      };
      // dQ += dS_h K_h, dS read from TMEM (columns 0..31 of the half's S buffer)
      auto do_dq = [&](int h) {
        const int i = h >> 1, e = h & 1;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + C::OFF_K + (i % C::SK) * C::KV_TILE);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t kdesc =
              sdesc_sw128(sK + (uint32_t)(8 * e + 2 * kk) * (C::KC * 1024), 1024, C::KC * 1024);
          umma_f16_ts(tmem + 256, tmem + e * 64 + kk * 8, kdesc, idesc_dq,
                      (h > 0 || kk > 0) ? 1u : 0u);
        }
        if (e == 1) umma_commit(&k_empty[i % C::SK]);
      };
      int qn = 0, dn = 0, n_h = -1;
      uint64_t t_prog = globaltimer();
      uint32_t idle = 0;
      while (ok && (n_h < 0 || dn < n_h)) {
        bool progress = false;
        if (dn < qn && mbar_test(&ds_full[dn & 1], (uint32_t)((dn >> 1) & 1))) {
          do_dq(dn);
          ++dn;
          progress = true;
        }
        if ((n_h < 0 || qn < n_h) && qn < dn + 2) {
          const int i = qn >> 1;
          if (mbar_test(&m_full[i % C::NM], (uint32_t)((i / C::NM) & 1)) &&
              mbar_test(&k_full[i % C::SK], (uint32_t)((i / C::SK) & 1)) &&
              mbar_test(&v_full[i % C::SV], (uint32_t)((i / C::SV) & 1))) {
            if ((qn & 1) == 0 && meta_at(i % C::NM).last) n_h = 2 * i + 2;
            do_sdp(qn);
            ++qn;
            progress = true;
          }
        }
        if (progress) {
          t_prog = globaltimer();
          idle = 0;
        } else {
          __nanosleep(32);
          if ((++idle & 63) == 0) {
            if (ab.set()) break;
            if (globaltimer() - t_prog > kWaitLimitNs) {
              ab.raise(a.status, 405);
              break;
            }
          }
        }
      }
      umma_commit(dq_done);
      umma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, a.status, 499);
    }
  } else {
    // ============================================================ dS warps
    // Group grp (4 warps, one thread per query-head row) takes half grp of
    // every stage: keys 64 grp .. 64 grp + 63.
    const int q = warp & 3;
    const int grp = (warp - 3) >> 2;
    const int r = q * 32 + lane;
    const bool row_ok = r < rows;
    const int qi = r >> a.lgG, h = r & (a.G - 1);
    const int64_t t = tq0 + qi;
    const int64_t pos = a.off + t;
    const int64_t cur = pos / B;
    const int64_t hq = (int64_t)g * a.G + h;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t tS = tl + grp * 64, tP = tl + 128 + grp * 64;
    const float ninf = -__int_as_float(0x7f800000);
    const float nl2 = row_ok ? -a.lse[hq * a.T + t] * kLog2e : 0.0f;
    const float nD = row_ok ? -a.Dl[hq * a.T + t] : 0.0f;
    const uint64_t sl2x2 = f2_pack(a.scale_log2, a.scale_log2);
    const uint64_t nD2 = f2_pack(nD, nD);
    bool ok = true;
    for (int i = 0;; ++i) {
      const int ms = i % C::NM;
      bool have = true, w = true;
      {
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 0;; ++it) {
          if (mbar_try_wait_ns(&m_full[ms], (uint32_t)((i / C::NM) & 1), 500)) break;
          if (*n_stages <= i) {
            have = false;
            break;
          }
          if ((it & 15) == 15) {
            if (ab.set()) {
              w = false;
              break;
            }
            if (globaltimer() - t0 > kWaitLimitNs) {
              ab.raise(a.status, 412);
              w = false;
              break;
            }
          }
        }
      }
      if (!__all_sync(FULL, w)) {
        ok = false;
        break;
      }
      if (!__any_sync(FULL, have)) break;
      const bool ws = mbar_wait(&s_full[grp], (uint32_t)(i & 1), ab, a.status, 411);
      if (!__all_sync(FULL, ws)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const Meta& m = meta_at(ms);
      const int nb = m.nb;
      const bool last = m.last != 0;
      // allowed keys of this row among the half's 64 keys (two 32-key words);
      // in full union mode every union entry's mask is all ones, so the same
      // rules give the tile's union blocks before the query's own block
      uint32_t al0 = 0u, al1 = 0u;
      if (row_ok) {
        const uint32_t hb = qbits_of(m, qi);
        al0 = hist_keys<B>(hb, 2 * grp);
        al1 = hist_keys<B>(hb, 2 * grp + 1);
#pragma unroll 1
        for (int bs = m.diag; bs < nb; ++bs) {
          const int64_t b = m.blk[bs];
          int lim = 0;
          if (((m.mask[bs] >> qi) & 1ull) && b < cur)
            lim = B;
          else if (b == cur)
            lim = (int)(pos - b * B + 1);
          const int k0 = bs * B - 64 * grp;  // key within this half
          if (lim > 0 && k0 >= 0 && k0 < 64) {
            const uint32_t bits = lim >= 32 ? 0xffffffffu : ((1u << lim) - 1u);
            const uint32_t wv = bits << (uint32_t)(k0 & 31);
            al0 |= (k0 >> 5) == 0 ? wv : 0u;
            al1 |= (k0 >> 5) == 1 ? wv : 0u;
          }
        }
      }
      uint32_t sv[64], dp[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld32(tP, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_wait_ld();
      uint32_t pk[32];
#pragma unroll
      for (int e2 = 0; e2 < 64; e2 += 2) {
        const uint32_t aw = e2 < 32 ? al0 : al1;
        const float c0 = ((aw >> (e2 & 31)) & 1u) ? nl2 : ninf;
        const float c1 = ((aw >> ((e2 + 1) & 31)) & 1u) ? nl2 : ninf;
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e2]), __uint_as_float(sv[e2 + 1])), sl2x2,
                         f2_pack(c0, c1)),
                  x0, x1);
        const uint64_t p2 = f2_pack(ex2(x0), ex2(x1));
        const uint64_t t2 = f2_add(f2_pack(__uint_as_float(dp[e2]), __uint_as_float(dp[e2 + 1])), nD2);
        float d0, d1;
        f2_unpack(f2_mul(p2, t2), d0, d1);
        pk[e2 >> 1] = pack_bf16x2(d0, d1);
      }
      tmem_st32(tS, pk);  // dS over the S columns already read
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&m_empty[ms]);
        mbar_arrive(&ds_full[grp]);
      }
      if (last) break;
    }
    // ---- epilogue: dQ = scale * (dS K), this group's half of the columns
    bool fin = ok && *n_stages != 0x7fffffff;
    if (fin) fin = mbar_wait(dq_done, 0, ab, a.status, 415);
    if (__all_sync(FULL, fin)) {
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = grp * (D / 2) + cc * 32;
        uint32_t o[32];
        tmem_ld32(tl + 256 + col, o);
        tmem_wait_ld();
        if (row_ok) {
          float* dst = a.dQ + (t * a.H + hq) * D + col;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) =
                make_float4(__uint_as_float(o[e]) * a.scale, __uint_as_float(o[e + 1]) * a.scale,
                            __uint_as_float(o[e + 2]) * a.scale, __uint_as_float(o[e + 3]) * a.scale);
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ==================================================================== dK, dV
template <int D>
struct DkvCfg {
  static constexpr int BM = 128;             // keys per work item (M of every MMA)
  static constexpr int NQ = 2;               // Q / dO slots
  static constexpr int NM = 4;               // query-stage descriptors in flight
  static constexpr int KC = D / 64;
  static constexpr int KV_BYTES = BM * D * 2;
  static constexpr int Q_BYTES = 128 * D * 2;  // 128 query-head rows
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;
  static constexpr int OFF_DO = OFF_Q + NQ * Q_BYTES;
  static constexpr int OFF_META = OFF_DO + NQ * Q_BYTES;
  static constexpr int OFF_STG = OFF_META + NM * 2048;  // [32 tiles][16 blocks] union masks
  static constexpr int OFF_BAR = OFF_STG + 32 * 16 * 8;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;  // S^T[2] 0/64, dP^T[2] 128/192, dV 256, dK 256 + D
  static constexpr int NTHREADS = 352;        // builder, loader, MMA, 8 softmax warps
  static_assert(SMEM <= 232448, "shared memory plan");
};

// One query stage of a key-major work item: a sub-tile of a union tile.
struct QStage {
  int64_t tq0;           // first query of the sub-tile
  int32_t nq;            // its queries
  int32_t pad;
  uint64_t hm[16];       // per block of the key stage: the sub-tile's queries that selected it
  float nlse2[128];      // -lse * log2(e) of each query-head row (0 past the sub-tile)
  float nD[128];         // -D of each row
};
static_assert(sizeof(QStage) <= 2048, "descriptor slot");

template <int D, int B>
__global__ void __launch_bounds__(352, 1)
    k_attn_bwd_dkv(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
                   BwdArgs a) {
  using C = DkvCfg<D>;
  constexpr int SB = C::BM / B;  // blocks per key stage
  static_assert(SB <= 16, "one mask word per block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  auto qs_at = [&](int i) -> QStage& {
    return *reinterpret_cast<QStage*>(smem + C::OFF_META + i * 2048);
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;    // [NQ]
  uint64_t* q_empty = bars + 3;   // [NQ]
  uint64_t* m_full = bars + 5;    // [NM]
  uint64_t* m_empty = bars + 9;   // [NM]
  uint64_t* s_full = bars + 13;   // [2] S^T and dP^T of a half-stage computed
  uint64_t* p_full = bars + 15;   // [2] P^T and dS^T of a half-stage written
  uint64_t* mma_done = bars + 17;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  int* abort_flag = reinterpret_cast<int*>(bars + 19);
  volatile int* n_stages = reinterpret_cast<volatile int*>(bars + 20);
  uint64_t* ld_full = bars + 24;  // [NM] the stage's lse and D rows written (by the loader)
  uint64_t* stg = reinterpret_cast<uint64_t*>(smem + C::OFF_STG);  // [32][16]

  const int64_t item = blockIdx.x;
  const int g = (int)(item % a.Hkv);
  const int64_t ks = item / a.Hkv;  // early key stages (most attended) first
  const int64_t kb0 = ks * SB;
  const int64_t kb1 = (kb0 + SB) < a.nblkp ? (kb0 + SB) : a.nblkp;
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < C::NQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < C::NM; ++i) {
      mbar_init(&m_full[i], 1);
      mbar_init(&m_empty[i], 9);  // the loader + 8 softmax warps
      mbar_init(&ld_full[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    mbar_init(mma_done, 1);
    *n_stages = 0x7fffffff;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag};

  if (warp == 0) {
    // ========================================== query stages of this key stage
    // 32 tiles at a time: each lane fetches its tile's first slot in the
    // stage and the union entries there (at most one per block) into the
    // staging table, then the tiles are walked in order.
    int j = 0;
    bool ok = true;
    const uint32_t* row = a.kbits + ((int64_t)g * a.nks + ks) * a.nw;
    for (int64_t w0 = 0; w0 < a.nw && ok; ++w0) {
      uint32_t bits = row[w0];
      if (bits == 0u) continue;
      {
        const int64_t tau = w0 * 32 + lane;
        const bool act = (bits >> lane) & 1u;
        const int64_t lt = (int64_t)g * a.ntiles + tau;
        const int32_t fs = act ? a.first[lt * a.nks + ks] : -1;
        const int64_t end = act ? a.uoff[lt] + a.ulen[lt] : 0;
        uint64_t* my = stg + lane * 16;
        int64_t bx[SB];
#pragma unroll
        for (int x = 0; x < SB; ++x) {
          my[x] = 0ull;
          bx[x] = (fs >= 0 && fs + x < end) ? a.ublk[fs + x] : INT64_MAX;
        }
#pragma unroll
        for (int x = 0; x < SB; ++x)
          if (bx[x] < kb0 + SB) my[bx[x] - kb0] = a.umask[fs + x];
      }
      __syncwarp();
      while (bits != 0u && ok) {
        const int li = __ffs(bits) - 1;
        bits &= bits - 1u;
        const int64_t tau = w0 * 32 + li;
        const int64_t t0 = tau * a.W;
        const int64_t len = (a.T - t0) < a.W ? (a.T - t0) : a.W;
        const int nsub = (int)((len + a.QS - 1) / a.QS);
        const uint64_t um = lane < SB ? stg[li * 16 + lane] : 0ull;
        for (int sidx = 0; sidx < nsub; ++sidx) {
          const int64_t tq0 = t0 + (int64_t)sidx * a.QS;
          const int nq = (int)((len - (int64_t)sidx * a.QS) < a.QS ? (len - (int64_t)sidx * a.QS) : a.QS);
          const uint64_t qmask = nq >= 64 ? ~0ull : ((1ull << nq) - 1ull);
          const uint64_t hm =
              a.mode == SGQA_UNION_MASKED ? ((um >> (sidx * a.QS)) & qmask) : (um ? qmask : 0ull);
          const int64_t c0 = (a.off + tq0) / B, cl = (a.off + tq0 + nq - 1) / B;
          const bool has_cur = cl >= kb0 && c0 < kb0 + SB;
          if (!__any_sync(FULL, hm != 0ull) && !has_cur) continue;
          const int ms = j % C::NM;
          const bool wt = mbar_wait(&m_empty[ms], (uint32_t)(((j / C::NM) & 1) ^ 1), ab, a.status, 421);
          if (!__all_sync(FULL, wt)) {
            ok = false;
            break;
          }
          QStage& st = qs_at(ms);
          if (lane == 0) {
            st.tq0 = tq0;
            st.nq = nq;
          }
          if (lane < 16) st.hm[lane] = hm;
          __syncwarp();
          if (lane == 0) mbar_arrive(&m_full[ms]);
          ++j;
        }
      }
      __syncwarp();  // the staging table is rewritten for the next 32 tiles
    }
    if (lane == 0) {
      *n_stages = ok ? j : 0;
      __threadfence_block();
    }
  } else if (warp == 1) {
    // ========================================== K, V once; Q and dO per stage
    const int64_t hb = (int64_t)g * (a.nblkp + 1) * (B * D);
    if (lane == 0) mbar_expect_tx(kv_full, 2 * C::KV_BYTES);
    __syncwarp();
    if (lane < SB) {
      const int64_t b = kb0 + lane < kb1 ? kb0 + lane : a.nblkp;  // past the end: the zero block
      bulk_load(smem + C::OFF_K + lane * (B * D * 2), a.Kp + hb + b * (B * D), B * D * 2, kv_full);
      bulk_load(smem + C::OFF_V + lane * (B * D * 2), a.Vp + hb + b * (B * D), B * D * 2, kv_full);
    }
    int issued[C::NQ] = {0, 0};
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mdo);
    }
    const uint32_t box = (uint32_t)(C::KC * 128 * a.G * a.QS);
    for (int j = 0;; ++j) {
      const int ms = j % C::NM, qs = j % C::NQ;
      bool have = true;
      {
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 0;; ++it) {
          if (mbar_try_wait_ns(&m_full[ms], (uint32_t)((j / C::NM) & 1), 500)) break;
          if (*n_stages <= j) {
            have = false;
            break;
          }
          if ((it & 15) == 15) {
            if (ab.set()) {
              have = false;
              break;
            }
            if (globaltimer() - t0 > kWaitLimitNs) {
              ab.raise(a.status, 422);
              have = false;
              break;
            }
          }
        }
      }
      if (!__all_sync(FULL, have)) break;
      const bool wq = mbar_wait(&q_empty[qs], (uint32_t)(((j / C::NQ) & 1) ^ 1), ab, a.status, 423);
      if (!__all_sync(FULL, wq)) break;
      QStage& st = qs_at(ms);
      const int64_t tq0 = st.tq0;
      const int nq = st.nq;
      if (lane == 0) {
        mbar_expect_tx(&q_full[qs], 2 * box);
        for (int c = 0; c < C::KC; ++c) {
          tma_load_3d(smem + C::OFF_Q + qs * C::Q_BYTES + c * (128 * 128), &mq, &q_full[qs], c * 64,
                      g * a.G, (int32_t)tq0);
          tma_load_3d(smem + C::OFF_DO + qs * C::Q_BYTES + c * (128 * 128), &mdo, &q_full[qs],
                      c * 64, g * a.G, (int32_t)tq0);
        }
      }
      ++issued[qs];
      // -lse * log2(e) and -D of the stage's query-head rows (0 past its queries)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = lane + 32 * k;
        const int qi = r >> a.lgG, hh = r & (a.G - 1);
        float nl = 0.0f, nd = 0.0f;
        if (qi < nq) {
          const int64_t hq = (int64_t)g * a.G + hh, t = tq0 + qi;
          nl = -a.lse[hq * a.T + t] * kLog2e;
          nd = -a.Dl[hq * a.T + t];
        }
        st.nlse2[r] = nl;
        st.nD[r] = nd;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ld_full[ms]);
        mbar_arrive(&m_empty[ms]);
      }
    }
    if (lane == 0 && ab.set()) {
      mbar_wait_drain(kv_full, 0, a.status, 493);
      for (int k = 0; k < C::NQ; ++k)
        if (issued[k] > 0) mbar_wait_drain(&q_full[k], (issued[k] - 1) & 1, a.status, 494);
    }
  } else if (warp == 2) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_h = idesc_bf16_f32(C::BM, 64, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(C::BM, D, 0, 1);
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      bool ok = mbar_wait(kv_full, 0, ab, a.status, 424);
      // S^T_h = K Q_h^T and dP^T_h = V dO_h^T for query rows 64 e .. of stage h / 2
      auto do_sdp = [&](int h) {
        const int j = h >> 1, e = h & 1;
        tc_fence_after();
        const uint32_t sQ = smem_u32(smem + C::OFF_Q + (j % C::NQ) * C::Q_BYTES);
        const uint32_t sdO = smem_u32(smem + C::OFF_DO + (j % C::NQ) * C::Q_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 1024 + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (128 * 128) + (kk & 3) * 32 + e * (64 * 128);
          umma_f16(tmem + e * 64, sdesc_sw128(sK + koff, 16, C::KC * 1024),
                   sdesc_sw128(sQ + qoff, 16, 1024), idesc_h, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 1024 + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (128 * 128) + (kk & 3) * 32 + e * (64 * 128);
          umma_f16(tmem + 128 + e * 64, sdesc_sw128(sV + koff, 16, C::KC * 1024),
                   sdesc_sw128(sdO + qoff, 16, 1024), idesc_h, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[e]);
      };
      // dV += P^T_h dO_h, dK += dS^T_h Q_h (P^T, dS^T from TMEM; dO, Q MN-major)
      bool started = false;
      auto do_acc = [&](int h) {
        const int j = h >> 1, e = h & 1;
        tc_fence_after();
        const uint32_t sQ = smem_u32(smem + C::OFF_Q + (j % C::NQ) * C::Q_BYTES);
        const uint32_t sdO = smem_u32(smem + C::OFF_DO + (j % C::NQ) * C::Q_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t roff = (uint32_t)(64 * e + 16 * kk) * 128;
          umma_f16_ts(tmem + 256, tmem + e * 64 + kk * 8, sdesc_sw128(sdO + roff, 128 * 128, 1024),
                      idesc_o, (started || kk > 0) ? 1u : 0u);
          umma_f16_ts(tmem + 256 + D, tmem + 128 + e * 64 + kk * 8,
                      sdesc_sw128(sQ + roff, 128 * 128, 1024), idesc_o,
                      (started || kk > 0) ? 1u : 0u);
        }
        started = true;
        if (e == 1) umma_commit(&q_empty[j % C::NQ]);
      };
      int qn = 0, dn = 0, n_h = -1;
      uint64_t t_prog = globaltimer();
      uint32_t idle = 0;
      while (ok && (n_h < 0 || dn < n_h)) {
        bool progress = false;
        if (dn < qn && mbar_test(&p_full[dn & 1], (uint32_t)((dn >> 1) & 1))) {
          do_acc(dn);
          ++dn;
          progress = true;
        }
        if (n_h < 0) {
          const int ns = *n_stages;
          if (ns != 0x7fffffff) n_h = 2 * ns;
        }
        if ((n_h < 0 || qn < n_h) && qn < dn + 2) {
          const int j = qn >> 1;
          if (mbar_test(&q_full[j % C::NQ], (uint32_t)((j / C::NQ) & 1))) {
            do_sdp(qn);
            ++qn;
            progress = true;
          }
        }
        if (progress) {
          t_prog = globaltimer();
          idle = 0;
        } else {
          __nanosleep(32);
          if ((++idle & 63) == 0) {
            if (ab.set()) break;
            if (globaltimer() - t_prog > kWaitLimitNs) {
              ab.raise(a.status, 425);
              break;
            }
          }
        }
      }
      umma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, a.status, 498);
    }
  } else {
    // ===================================================== P^T and dS^T warps
    // Group grp (4 warps, one thread per key) takes query rows 64 grp .. of
    // every stage.
    const int q = warp & 3;
    const int grp = (warp - 3) >> 2;
    const int key = q * 32 + lane;
    const int64_t pk = kb0 * B + key;  // the key's position
    const int64_t blk = pk / B;
    const bool key_ok = blk < kb1 && pk < a.Tkv;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t tS = tl + grp * 64, tP = tl + 128 + grp * 64;
    const float ninf = -__int_as_float(0x7f800000);
    const uint64_t sl2x2 = f2_pack(a.scale_log2, a.scale_log2);
    bool ok = true;
    for (int j = 0;; ++j) {
      const int ms = j % C::NM;
      bool have = true, w = true;
      {
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 0;; ++it) {
          if (mbar_try_wait_ns(&ld_full[ms], (uint32_t)((j / C::NM) & 1), 500)) break;
          if (*n_stages <= j) {
            have = false;
            break;
          }
          if ((it & 15) == 15) {
            if (ab.set()) {
              w = false;
              break;
            }
            if (globaltimer() - t0 > kWaitLimitNs) {
              ab.raise(a.status, 432);
              w = false;
              break;
            }
          }
        }
      }
      if (!__all_sync(FULL, w)) {
        ok = false;
        break;
      }
      if (!__any_sync(FULL, have)) break;
      const bool ws = mbar_wait(&s_full[grp], (uint32_t)(j & 1), ab, a.status, 431);
      if (!__all_sync(FULL, ws)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const QStage& st = qs_at(ms);
      // the queries of the sub-tile that may attend this key
      const int64_t pos0 = a.off + st.tq0;
      uint64_t qa = 0ull;
      if (key_ok) {
        const uint64_t hm = st.hm[key / B];
        // historical: selected (masked mode), or in the tile's union and
        // before the query's own block (full mode)
        int64_t qc = (blk + 1) * B - pos0;  // first query whose own block is past this one
        qc = qc < 0 ? 0 : qc;
        const uint64_t after = qc >= 64 ? 0ull : (~0ull << qc);
        qa = a.mode == SGQA_UNION_MASKED ? hm : (hm & after);
        // current block: queries in this key's block at or after its position
        int64_t ca = pk - pos0;
        ca = ca < 0 ? 0 : ca;
        int64_t cb = (blk + 1) * B - pos0;
        cb = cb > st.nq ? st.nq : cb;
        if (ca < cb) {
          const uint64_t lo = ca >= 64 ? 0ull : (~0ull << ca);
          const uint64_t hi = cb >= 64 ? ~0ull : ((1ull << cb) - 1ull);
          qa |= lo & hi;
        }
        qa &= st.nq >= 64 ? ~0ull : ((1ull << st.nq) - 1ull);
      }
      // two passes of 32 rows; P^T and dS^T (bf16 pairs) go over the S^T and
      // dP^T columns already read (pass hh writes columns 16 hh .. 16 hh + 15,
      // which hold rows the earlier pass has read)
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tS + 32 * hh, sv);
        tmem_ld32(tP + 32 * hh, dp);
        tmem_wait_ld();
        uint32_t pp[16], pd[16];
        const float* nl = st.nlse2 + 64 * grp + 32 * hh;
        const float* nd = st.nD + 64 * grp + 32 * hh;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int r = 64 * grp + 32 * hh + c;
          const float c0 = ((qa >> (r >> a.lgG)) & 1ull) ? nl[c] : ninf;
          const float c1 = ((qa >> ((r + 1) >> a.lgG)) & 1ull) ? nl[c + 1] : ninf;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2,
                           f2_pack(c0, c1)),
                    x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          const uint64_t t2 = f2_add(f2_pack(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])),
                                     f2_pack(nd[c], nd[c + 1]));
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p0, p1), t2), d0, d1);
          pp[c >> 1] = pack_bf16x2(p0, p1);
          pd[c >> 1] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tS + 16 * hh, pp);
        tmem_st16(tP + 16 * hh, pd);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&m_empty[ms]);
        mbar_arrive(&p_full[grp]);
      }
    }
    // ---- epilogue: dV and dK (= scale * dS^T Q) of this key, half the columns
    const int ns = *n_stages;
    bool fin = ok && ns != 0x7fffffff;
    if (fin && ns > 0) fin = mbar_wait(mma_done, 0, ab, a.status, 435);
    if (__all_sync(FULL, fin)) {
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = grp * (D / 2) + cc * 32;
        uint32_t v[32], k[32];
        if (ns > 0) {
          tmem_ld32(tl + 256 + col, v);
          tmem_ld32(tl + 256 + D + col, k);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = k[e] = 0u;
        }
        if (key_ok) {
          float* dv = a.dV + (pk * a.Hkv + g) * D + col;
          float* dk = a.dK + (pk * a.Hkv + g) * D + col;
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            *reinterpret_cast<float4*>(dv + e) =
                make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                            __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
            *reinterpret_cast<float4*>(dk + e) =
                make_float4(__uint_as_float(k[e]) * a.scale, __uint_as_float(k[e + 1]) * a.scale,
                            __uint_as_float(k[e + 2]) * a.scale, __uint_as_float(k[e + 3]) * a.scale);
          }
        }
      }
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
int launch_bwd_db(const Dims& dm, const BwdArgs& a, const void* Q, const void* dO,
                  cudaStream_t st) {
  CUtensorMap mq, mdo;
  if (!make_qmap(dm, a.QS, Q, &mq) || !make_qmap(dm, a.QS, dO, &mdo)) return SGQA_ERR_CUDA;
  using CQ = DqCfg<D, B>;
  using CK = DkvCfg<D>;
  if (cudaFuncSetAttribute(k_attn_bwd_dq<D, B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CQ::SMEM) != cudaSuccess ||
      cudaFuncSetAttribute(k_attn_bwd_dkv<D, B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CK::SMEM) != cudaSuccess)
    return SGQA_ERR_CUDA;
  const int64_t items_q = dm.ntiles * dm.Hkv * a.nsub;
  log_begin(SGQA_K_ATTN_BWD, st);
  k_attn_bwd_dq<D, B><<<(unsigned)items_q, CQ::NTHREADS, CQ::SMEM, st>>>(mq, mdo, a);
  log_end(st);
  if (cudaGetLastError() != cudaSuccess) return SGQA_ERR_CUDA;
  const int64_t items_k = (int64_t)dm.Hkv * a.nks;
  log_begin(SGQA_K_ATTN_BWD, st);
  k_attn_bwd_dkv<D, B><<<(unsigned)items_k, CK::NTHREADS, CK::SMEM, st>>>(mq, mdo, a);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

}  // namespace

size_t attn_bwd_ws_bytes(const Dims& dm, size_t* off_D, size_t* off_bits, size_t* off_first) {
  const int SB = 128 / dm.B;
  const int64_t nblkp = (dm.Tkv + dm.B - 1) / dm.B;
  const int64_t nks = (nblkp + SB - 1) / SB, nw = (dm.ntiles + 31) / 32;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t o = 0;
  *off_D = o;
  o += up((size_t)dm.H * dm.T * 4);
  *off_bits = o;
  o += up((size_t)dm.Hkv * nks * nw * 4);
  *off_first = o;
  o += up((size_t)dm.Hkv * dm.ntiles * nks * 4);
  return o;
}

int launch_attn_bwd(const Dims& dm, const __nv_bfloat16* Q, const __nv_bfloat16* Kp,
                    const __nv_bfloat16* Vp, const int64_t* union_off, const int32_t* union_len,
                    const int32_t* union_blk, const uint64_t* union_mask, const void* O,
                    const float* lse, const void* dO, float* dQ, float* dK, float* dV, void* ws,
                    int32_t* status, cudaStream_t st) {
  if (dm.B < 8 || dm.dtype != SGQA_BF16 || (dm.G & (dm.G - 1)) != 0) return SGQA_ERR_UNSUPPORTED;
  size_t oD, oB, oF;
  attn_bwd_ws_bytes(dm, &oD, &oB, &oF);
  uint8_t* w = static_cast<uint8_t*>(ws);
  BwdArgs a;
  a.ublk = union_blk;
  a.umask = union_mask;
  a.mode = dm.mode;
  a.uoff = union_off;
  a.ulen = union_len;
  a.Kp = Kp;
  a.Vp = Vp;
  a.nblkp = (dm.Tkv + dm.B - 1) / dm.B;
  a.lse = lse;
  a.Dl = reinterpret_cast<float*>(w + oD);
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.kbits = reinterpret_cast<const uint32_t*>(w + oB);
  a.first = reinterpret_cast<const int32_t*>(w + oF);
  a.T = dm.T;
  a.Tkv = dm.Tkv;
  a.off = dm.off;
  a.ntiles = dm.ntiles;
  const int SB = 128 / dm.B;
  a.nks = (a.nblkp + SB - 1) / SB;
  a.nw = (dm.ntiles + 31) / 32;
  a.H = dm.H;
  a.Hkv = dm.Hkv;
  a.G = dm.G;
  a.lgG = __builtin_ctz((unsigned)dm.G);
  a.B = dm.B;
  a.W = dm.W;
  a.QS = 128 / dm.G < dm.W ? 128 / dm.G : dm.W;
  a.nsub = (dm.W + a.QS - 1) / a.QS;
  a.scale = dm.scale;
  a.scale_log2 = dm.scale * kLog2e;
  a.status = status;
  if (a.QS > 64) return SGQA_ERR_UNSUPPORTED;
  // D, then the key stages each tile attends
  const int64_t rows = dm.T * dm.H;
  const int grid_d = (int)((rows + 7) / 8);
  log_begin(SGQA_K_STAGE, st);
  if (dm.d == 128)
    k_bwd_delta<128><<<grid_d, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(O),
                                              static_cast<const __nv_bfloat16*>(dO), dm.T, dm.H,
                                              const_cast<float*>(a.Dl));
  else
    k_bwd_delta<64><<<grid_d, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(O),
                                             static_cast<const __nv_bfloat16*>(dO), dm.T, dm.H,
                                             const_cast<float*>(a.Dl));
  log_end(st);
  if (cudaGetLastError() != cudaSuccess) return SGQA_ERR_CUDA;
  log_begin(SGQA_K_STAGE, st);
  bool filled = fill_u32(w + oB, (int64_t)dm.Hkv * a.nks * a.nw, 0u, st) == cudaSuccess;
  log_end(st);
  log_begin(SGQA_K_STAGE, st);
  filled = filled &&
           fill_u32(w + oF, (int64_t)dm.Hkv * dm.ntiles * a.nks, 0xFFFFFFFFu, st) == cudaSuccess;
  log_end(st);
  if (!filled) return SGQA_ERR_CUDA;
  const int64_t warps = (int64_t)dm.Hkv * dm.ntiles;
  log_begin(SGQA_K_STAGE, st);
  k_bwd_index<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(a, SB);
  log_end(st);
  if (cudaGetLastError() != cudaSuccess) return SGQA_ERR_CUDA;
  if (dm.d == 128) return dm.B == 8 ? launch_bwd_db<128, 8>(dm, a, Q, dO, st)
                                    : launch_bwd_db<128, 16>(dm, a, Q, dO, st);
  if (dm.d == 64) return dm.B == 8 ? launch_bwd_db<64, 8>(dm, a, Q, dO, st)
                                   : launch_bwd_db<64, 16>(dm, a, Q, dO, st);
  return SGQA_ERR_UNSUPPORTED;
}

}  // namespace sgqa
