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
// Roles (12 warps):
//  warp 0   builds each stage's block list from the union entries (an
//           8-deep ring, so the lists run ahead of the loads);
//  warp 11  issues the K loads: for B >= 8 one contiguous bulk copy per block
//           from the block-packed, pre-swizzled K (see k_kv_pack), for B < 8
//           four-row TMA gathers (tile::gather4) from the original layout,
//           contiguous or paged;
//  warp 1   issues the V loads the same way;
//  warp 2   one thread issues S = Q K^T into a double-buffered TMEM tile
//           (K slots, three of them, are released as soon as their QK product
//           is done) and O += P V into the TMEM accumulator, with P read from
//           TMEM as the A operand and V from shared memory (MN-major);
//  warps 3-10 two softmax groups of 4 warps taking alternate stages, one
//           thread per query-head row and all 128 keys of the stage, each
//           group with its own S buffer, running maximum, sum and O
//           accumulator in TMEM: read S, apply the per-query block masks (the
//           causal cut only on current blocks), run the fp32 online softmax in
//           base 2 against a lazily raised reference maximum (O is rescaled in
//           TMEM only when it grows by more than 2^16), write P (bf16) into
//           TMEM over the S values already read (the S buffer is released by
//           the PV product); at the end the two groups' O, maxima and sums are
//           combined and O and the log-sum-exp written.
#include "attn_common.cuh"

namespace sgqa {
namespace {

// Lazy rescaling: the softmax keeps a row's reference maximum until a key
// exceeds it by more than 2^kLazy (log2 units), so P (bf16) stays below
// 2^kLazy and O (fp32) is rescaled only on such a jump.  bf16 and fp32 keep
// the same relative precision at any of these magnitudes; 2^16 leaves ample
// range for sums of a stage's products into fp32.
constexpr float kLazy = 16.0f;
// The one-pass check on 64 keys: their P values (relative to the reference
// maximum) are computed first and kept only when their sum stays at or below
// 2^kLazy, which bounds every one of them by 2^kLazy.  (A sum of many
// moderate values can trip it without any key exceeding the bound; the stage
// then takes the exact path below, which gives the same result.)
constexpr float kLazySum = 65536.0f;
static_assert(kLazySum == (float)(1 << 16) && kLazy == 16.0f, "the sum bound is 2^kLazy");

template <int D, int B>
struct AttnCfg {
  static constexpr int BM = 128;  // rows per MMA
  static constexpr int KB = 128;  // keys per stage
  static constexpr int NBPS = KB / B;
  static constexpr int SK = 3;            // K slots
  static constexpr int SV = 2;            // V slots
  static constexpr int NM = 8;            // stage block-list slots
  static constexpr int KC = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_TILE = KB * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + SK * KV_TILE;
  static constexpr int OFF_META = OFF_V + SV * KV_TILE;
  static constexpr int META_BYTES = (int)((sizeof(MetaT<NBPS>) + 15) / 16 * 16);
  static constexpr int OFF_X = OFF_META + NM * META_BYTES;  // epilogue max / sum exchange
  static constexpr int OFF_BAR = OFF_X + 2 * 2 * BM * 4;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;  // S[2] at 0 / 128, O[2] at 256 / 384
  static constexpr int NTHREADS = 384;        // 3 pipeline warps, 8 softmax warps, K loads
  static_assert(SMEM <= 232448, "shared memory plan");
};

struct AttnArgs {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const __nv_bfloat16* Kp;  // block-packed K and V (B >= 8)
  const __nv_bfloat16* Vp;
  int64_t nblkp;            // packed blocks per head, excluding the zero block
  const int32_t* page_table;
  const int64_t* uoff;
  const int32_t* ulen;
  const int32_t* ublk;
  const uint64_t* umask;
  void* O;
  float* lse;
  int64_t T, Tkv, off, nblk, lay_tau0, lay_ntiles, tau_begin, tau_end;
  int H, Hkv, G, B, W, ps, QS, nsub, mode, out_f32, npages;
  float scale_log2;
  int32_t* status;
  // split work items (few queries over long lists): nsplit > 1 splits each
  // item's historical union entries into nsplit ranges (the last also takes
  // the current blocks); each split writes its normalised partial O and its
  // log-sum-exp, merged by k_attn_combine
  int nsplit;
  float* opart;  // [nsplit][T][H][D]
  float* lpart;  // [nsplit][H][T]
};

// Gathers one stage's 128 key rows (bf16) of K or V for KV head g into the
// [head-dim half][key][128 B] swizzled layout the MMA reads: lane j brings keys
// 4j .. 4j + 3, one four-row TMA gather per 64-column half.  The map's rows
// are p * Hkv + g (contiguous cache) or (page * Hkv + g) * page_size + p %
// page_size (paged).  Keys past the stage's blocks read position 0 instead;
// the softmax gives them no weight.
template <int D, int B, int NBPS>
__device__ __forceinline__ void gather_stage(uint8_t* dst, const CUtensorMap* map,
                                             const AttnArgs& a, const MetaT<NBPS>& m, int g,
                                             int lane, uint64_t* bar) {
  constexpr int KB = 128;
  static_assert(KB == 4 * 32, "one four-row gather per lane and half");
  const int nkeys = m.nb * B;
  int32_t r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int k = lane * 4 + e;
    int64_t p = k < nkeys ? (int64_t)m.blk[k / B] * B + (k % B) : 0;
    if (p >= a.Tkv) p = 0;
    int64_t row = a.ps > 0 ? ((int64_t)a.page_table[p / a.ps] * a.Hkv + g) * a.ps + p % a.ps
                           : p * a.Hkv + g;
    if (row > 0x7fffffffll) {  // beyond the map's 32-bit row coordinate
      report(a.status, SGQA_ERR_BOUNDS, 230);
      row = 0;
    }
    r[e] = (int32_t)row;
  }
#pragma unroll
  for (int c = 0; c < D / 64; ++c)
    tma_gather4(dst + c * (KB * 128) + lane * 512, map, bar, c * 64, r[0], r[1], r[2], r[3]);
}

// A stage whose keys 64..127 exceed the softmax row's reference maximum by
// more than 2^kLazy after keys 0..63 passed and were written as P (TMEM columns
// 0..31 of the S buffer at tS) under it.  The S values of keys 64..127
// (columns 64..127) are still in place: their masked maximum mx is taken,
// the maximum raised to it (rows that need it) with O (at tOg, once the
// group's previous PV product is done: phase `parity` of p_empty), l, the
// stage's partial sums rs0/rs1 and the 32 P columns scaled by
// 2^(m_used - mx), and P of keys 64..127 written into columns 32..63.  Kept
// out of line: the path is rare, and inlined it slowed the common one.
// Warp-collective.
struct MidState {
  float m_used, l, rs0, rs1;
  bool ok;
};
template <int D>
__device__ __noinline__ MidState stage_second_half(uint32_t tS, uint32_t tOg, uint32_t al2,
                                                    uint32_t al3, float sl2, float m_used,
                                                    float l, float rs0, float rs1,
                                                    uint64_t* p_empty, uint32_t parity, Abort ab,
                                                    int32_t* status) {
  const float ninf = -__int_as_float(0x7f800000);
  tmem_wait_st();  // the P of keys 0..63 is read back below
  float mx = ninf;
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {  // keys 64 + 8 c ..
    uint32_t v[8];
    tmem_ld8(tS + 64 + 8 * c, v);
    tmem_wait_ld();
    const uint32_t am = ((c < 4 ? al2 : al3) >> ((c & 3) * 8)) & 0xffu;
#pragma unroll
    for (int e = 0; e < 8; ++e) mx = fmaxf(mx, ((am >> e) & 1u) ? __uint_as_float(v[e]) : ninf);
  }
  mx *= sl2;
  const bool raise = mx > m_used + kLazy;
  const float f = raise ? ex2(m_used - mx) : 1.0f;
  MidState r{m_used, l, rs0, rs1, false};
  if (!__all_sync(FULL, mbar_wait(p_empty, parity, ab, status, 214))) return r;
  tc_fence_after();
  // O, then the P of keys 0..63 (columns 0..31, bf16 pairs), scaled by f
#pragma unroll 1
  for (int c = 0; c < D / 8 + 4; ++c) {
    const bool isO = c < D / 8;
    const uint32_t ta = isO ? tOg + 8 * c : tS + 8 * (c - D / 8);
    uint32_t v[8];
    tmem_ld8(ta, v);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (isO) {
        v[e] = __float_as_uint(__uint_as_float(v[e]) * f);
      } else {
        const float lo = __uint_as_float(v[e] << 16);
        const float hi = __uint_as_float(v[e] & 0xffff0000u);
        v[e] = pack_bf16x2(lo * f, hi * f);
      }
    }
    tmem_st8(ta, v);
  }
  r.l = l * f;
  r.rs0 = rs0 * f;
  r.rs1 = rs1 * f;
  if (raise) r.m_used = mx;
  const float msub = r.m_used;
  // P of keys 64..127 into columns 32..63, 16 keys (8 columns) at a time
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t v0[8], v1[8], pk[8];
    tmem_ld8(tS + 64 + 16 * c, v0);
    tmem_ld8(tS + 72 + 16 * c, v1);
    tmem_wait_ld();
    const uint32_t am = ((c < 2 ? al2 : al3) >> ((c & 1) * 16)) & 0xffffu;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float p0 = ((am >> e) & 1u) ? ex2(fmaf(__uint_as_float(v0[e]), sl2, -msub)) : 0.0f;
      const float p1 = ((am >> (e + 1)) & 1u) ? ex2(fmaf(__uint_as_float(v0[e + 1]), sl2, -msub)) : 0.0f;
      const float p2 = ((am >> (8 + e)) & 1u) ? ex2(fmaf(__uint_as_float(v1[e]), sl2, -msub)) : 0.0f;
      const float p3 =
          ((am >> (9 + e)) & 1u) ? ex2(fmaf(__uint_as_float(v1[e + 1]), sl2, -msub)) : 0.0f;
      r.rs0 += p0 + p2;
      r.rs1 += p1 + p3;
      pk[e >> 1] = pack_bf16x2(p0, p1);
      pk[4 + (e >> 1)] = pack_bf16x2(p2, p3);
    }
    tmem_st8(tS + 32 + 8 * c, pk);
  }
  tmem_wait_st();
  r.ok = true;
  return r;
}

// PK: the K/V blocks come from the block-packed copy (B >= 8: whole 8-row
// swizzle atoms, one bulk copy each); otherwise keys are gathered four rows
// at a time (TMA tile::gather4) from the original contiguous or paged cache.
template <int D, int B, bool PK>
__global__ void __launch_bounds__(384, 1)
    k_sparse_attn(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mv, AttnArgs a) {
  using C = AttnCfg<D, B>;
  using Meta = MetaT<C::NBPS>;
  constexpr int NBPS = C::NBPS;  // blocks per stage
  constexpr bool kTma = PK;
  static_assert(!PK || B >= 8, "packed blocks are whole swizzle atoms");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  auto meta_at = [&](int i) -> Meta& {
    return *reinterpret_cast<Meta*>(smem + C::OFF_META + i * C::META_BYTES);
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;     // [SK]
  uint64_t* k_empty = bars + 4;    // [SK]
  uint64_t* v_full = bars + 7;     // [SV]
  uint64_t* v_empty = bars + 9;    // [SV]
  uint64_t* m_full = bars + 11;    // [NM]
  uint64_t* m_empty = bars + 19;   // [NM]
  uint64_t* s_full = bars + 27;    // [2]
  uint64_t* p_full = bars + 31;    // [2] P of a stage of softmax group g written
  uint64_t* mma_done = bars + 33;
  uint64_t* p_empty = bars + 34;   // [2] PV product into O[g] done
  uint64_t* l_bar = bars + 36;     // both groups' maxima and sums exchanged (epilogue)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 37);
  int* abort_flag = reinterpret_cast<int*>(bars + 38);
  volatile int* n_stages = reinterpret_cast<volatile int*>(bars + 39);  // set once known
  uint64_t* stall_bar = bars + 40;  // nothing arrives on it (the debug stall below)
  float* xmax = reinterpret_cast<float*>(smem + C::OFF_X);  // [2 group][BM]
  float* xsum = xmax + 2 * C::BM;                            // [2 group][BM]

  // ---- work item (and its split)
  const int sp = (int)(blockIdx.x % a.nsplit);
  const int64_t item = blockIdx.x / a.nsplit;
  const int64_t per_tile = (int64_t)a.Hkv * a.nsub;
  const int64_t tau = a.tau_end - 1 - item / per_tile;  // heavy tiles first
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
      mbar_init(&m_empty[i], 6);  // the stage's 4 softmax warps + the K and V producers
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(l_bar, 8);
    *n_stages = 0x7fffffff;
    mbar_init(mma_done, 1);
    mbar_init(stall_bar, 1);
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
    // ================================================ block lists + K loads
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      if constexpr (!kTma) {
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
      }
      // the Q box is G x QS rows (fewer than 128 when a sub-tile cannot fill M)
      mbar_expect_tx(q_full, (uint32_t)(C::KC * 128 * a.G * a.QS));
      for (int c = 0; c < C::KC; ++c)  // box (64, G, QS) lands as rows qi * G + h
        tma_load_3d(smem + C::OFF_Q + c * (C::BM * 128), &mq, q_full, c * 64, g * a.G,
                    (int32_t)tq0);
    }
    Gen gs;
    const int64_t lt = (int64_t)g * a.lay_ntiles + (tau - a.lay_tau0);
    gs.cur = a.uoff[lt];
    gs.end = gs.cur + a.ulen[lt];
    gs.c0 = (a.off + tq0) / B;
    gs.c_last = (a.off + tq0 + nq_sub - 1) / B;
    if (a.nsplit > 1) {
      // the historical entries (those before the first current block; the
      // entries at or past it are at most the last 64) are divided evenly
      const int64_t L = gs.end - gs.cur;
      int64_t trail = 0;
      for (int r0 = 0; r0 < 64 && r0 < L; r0 += 32) {
        const bool ge = r0 + lane < L && a.ublk[gs.end - 1 - r0 - lane] >= gs.c0;
        const uint32_t bal = __ballot_sync(FULL, ge);
        trail += __popc(bal);
        if (bal != FULL) break;
      }
      const int64_t h0 = gs.cur, lh = L - trail;
      gs.cur = h0 + lh * sp / a.nsplit;
      if (sp < a.nsplit - 1) {
        gs.end = h0 + lh * (sp + 1) / a.nsplit;
        gs.c_last = gs.c0 - 1;  // the current blocks go to the last split
      }
    }
    gs.nd = gs.c0;
    gs.phase = 0;
    gs.pf_at = -1;
    const int sh = s * a.QS;
    const uint64_t qmask = nq_sub >= 64 ? ~0ull : ((1ull << nq_sub) - 1ull);
    for (int i = 0;; ++i) {
      const int ms = i % C::NM;
      const bool w = mbar_wait(&m_empty[ms], (uint32_t)(((i / C::NM) & 1) ^ 1), ab, a.status, 201);
      if (!__all_sync(FULL, w)) break;
      Meta& m = meta_at(ms);
      gen_stage<B == 2 || B == 4>(a, gs, m, NBPS, sh, qmask, nq_sub);
      if (lane == 0 && m.last) {
        *n_stages = i + 1;  // lets the softmax group without a further stage stop
        __threadfence_block();
      }
      if (lane == 0) mbar_arrive(&m_full[ms]);
      if (m.last) break;
    }
    if (lane == 0 && ab.set()) mbar_wait_drain(q_full, 0, a.status, 291);
  } else if (warp == 11) {
    // ============================================================= K loads
    int issued_k[C::SK] = {};
    for (int i = 0;; ++i) {
      const int ms = i % C::NM, ks = i % C::SK;
      bool w = mbar_wait(&m_full[ms], (uint32_t)((i / C::NM) & 1), ab, a.status, 219) &&
               mbar_wait(&k_empty[ks], (uint32_t)(((i / C::SK) & 1) ^ 1), ab, a.status, 202);
      if (!__all_sync(FULL, w)) break;
      const Meta& m = meta_at(ms);
      const bool last = m.last != 0;
      uint8_t* sK = smem + C::OFF_K + ks * C::KV_TILE;
      if (lane == 0) mbar_expect_tx(&k_full[ks], C::KV_TILE);
      __syncwarp();
      if constexpr (kTma)  // lane bs copies block slot bs (one contiguous packed block each)
        copy_blocks<NBPS>(sK, a.Kp + (int64_t)g * (a.nblkp + 1) * (B * D), m.blk, m.nb,
                          a.nblkp, B * D, &k_full[ks]);
      else
        gather_stage<D, B, NBPS>(sK, &mk, a, m, g, lane, &k_full[ks]);
      ++issued_k[ks];
      __syncwarp();
      if (lane == 0) mbar_arrive(&m_empty[ms]);
      if (last) break;
    }
    if (lane == 0 && ab.set())  // let in-flight copies land before the CTA exits
      for (int k = 0; k < C::SK; ++k)
        if (issued_k[k] > 0) mbar_wait_drain(&k_full[k], (issued_k[k] - 1) & 1, a.status, 292);
  } else if (warp == 1) {
    // ============================================================= V loads
    int issued_v[C::SV] = {};
    for (int i = 0;; ++i) {
      const int ms = i % C::NM, vs = i % C::SV;
      bool w = mbar_wait(&m_full[ms], (uint32_t)((i / C::NM) & 1), ab, a.status, 203) &&
               mbar_wait(&v_empty[vs], (uint32_t)(((i / C::SV) & 1) ^ 1), ab, a.status, 204);
      if (!__all_sync(FULL, w)) break;
      const Meta& m = meta_at(ms);
      const bool last = m.last != 0;
      uint8_t* sV = smem + C::OFF_V + vs * C::KV_TILE;
      if (lane == 0) mbar_expect_tx(&v_full[vs], C::KV_TILE);
      __syncwarp();
      if constexpr (kTma)
        copy_blocks<NBPS>(sV, a.Vp + (int64_t)g * (a.nblkp + 1) * (B * D), m.blk, m.nb,
                          a.nblkp, B * D, &v_full[vs]);
      else
        gather_stage<D, B, NBPS>(sV, &mv, a, m, g, lane, &v_full[vs]);
      ++issued_v[vs];
      __syncwarp();
      if (lane == 0) mbar_arrive(&m_empty[ms]);
      if (last) break;
    }
    if (lane == 0 && ab.set())
      for (int k = 0; k < C::SV; ++k)
        if (issued_v[k] > 0) mbar_wait_drain(&v_full[k], (issued_v[k] - 1) & 1, a.status, 293);
  } else if (warp == 2) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(C::BM, C::KB, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(C::BM, D, 0, 1);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      bool ok = mbar_wait(q_full, 0, ab, a.status, 205);
      // Debug request (host-set status[3]): the first work item waits on a
      // barrier nothing arrives on, so the pipeline gives up (detail 220) while
      // its K and V copies are in flight.
      if (ok && blockIdx.x == 0 && debug_request(a.status) == SGQA_DEBUG_STALL)
        ok = mbar_wait(stall_bar, 0, ab, a.status, 220, kDebugStallNs);
      // S_j = Q K_j^T into TMEM buffer j % 2 (operands ready)
      auto do_qk = [&](int j) {
        const int ks = j % C::SK;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + C::OFF_K + ks * C::KV_TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (C::BM * 128) + (kk & 3) * 32;
          // packed stage: 8-key groups every KC KB, head-dim halves 1 KB apart;
          // gathered stage: halves KB*128 apart, groups every 1 KB
          const uint32_t koff = kTma ? (kk >> 2) * 1024 + (kk & 3) * 32
                                     : (kk >> 2) * (C::KB * 128) + (kk & 3) * 32;
          const uint32_t ksbo = kTma ? C::KC * 1024 : 1024;
          umma_f16(tmem + (j & 1) * 128, sdesc_sw128(sQ + off, 16, 1024),
                   sdesc_sw128(sK + koff, 16, ksbo), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
        umma_commit(&k_empty[ks]);  // the K slot is free once this product is done
      };
      // O[i % 2] += P_i V_i, P read from TMEM (operands ready)
      auto do_pv = [&](int i) {
        const int vs = i % C::SV;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + C::OFF_V + vs * C::KV_TILE);
#pragma unroll
        for (int kk = 0; kk < C::KB / 16; ++kk) {
          // P (bf16) fills columns 0..63 of S buffer i % 2: keys 16 kk .. 16 kk + 15
          // are 8 columns
          const uint32_t pt = tmem + (i & 1) * 128 + kk * 8;
          // V as an MN-major operand: LBO = stride between head-dim halves,
          // SBO = stride between 8-key groups
          const uint64_t vdesc =
              kTma ? sdesc_sw128(sV + kk * 2 * (C::KC * 1024), 1024, C::KC * 1024)
                   : sdesc_sw128(sV + kk * 16 * 128, C::KB * 128, 1024);
          // stage i accumulates into O[i % 2], the running sum of softmax group i % 2
          umma_f16_ts(tmem + 256 + (i & 1) * 128, pt, vdesc, idesc_pv, (i > 1 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&p_empty[i & 1]);
        umma_commit(&v_empty[vs]);
      };
      // Issue each product as soon as its operands are ready (the two softmax
      // groups' chains are independent), PV first.  QK_j overwrites the S/P
      // buffer that PV_{j-2} reads P from; it is issued once PV_{j-2} has been
      // issued, not once it has completed: tcgen05.mma operations of one
      // thread execute in issue order, so PV_{j-2} has read P before QK_j
      // writes S.  Every phase tested is at most one ahead of the last one
      // completed.  (Polling measured faster than sleeping in each barrier in
      // turn: the wake-up from a suspended wait lengthens every hand-off.)
      int qn = 0, pn = 0;  // next QK and PV to issue
      int n_st = -1;       // stages of the item, once the last list has been seen
      uint64_t t_prog = globaltimer();
      uint32_t idle = 0;
      while (ok && (n_st < 0 || pn < n_st)) {
        bool progress = false;
        if (pn < qn && mbar_test(&p_full[pn & 1], (uint32_t)((pn >> 1) & 1)) &&
            mbar_test(&v_full[pn % C::SV], (uint32_t)((pn / C::SV) & 1))) {
          do_pv(pn);
          ++pn;
          progress = true;
        }
        if ((n_st < 0 || qn < n_st) && qn <= pn + 1 &&
            mbar_test(&m_full[qn % C::NM], (uint32_t)((qn / C::NM) & 1)) &&
            mbar_test(&k_full[qn % C::SK], (uint32_t)((qn / C::SK) & 1))) {
          if (meta_at(qn % C::NM).last) n_st = qn + 1;
          do_qk(qn);
          ++qn;
          progress = true;
        }
        if (progress) {
          t_prog = globaltimer();
          idle = 0;
        } else {
          __nanosleep(32);
          if ((++idle & 63) == 0) {
            if (ab.set()) break;
            if (globaltimer() - t_prog > kWaitLimitNs) {
              ab.raise(a.status, 206);
              break;
            }
          }
        }
      }
      umma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, a.status, 299);
    }
  } else if (warp >= 3 && warp <= 10) {
    // =============================================================== softmax
    // Group grp (4 warps, one thread per query-head row) takes stages grp,
    // grp + 2, ...: all 128 keys of each, with its own running maximum and sum
    // and its own accumulator O[grp], so the two groups work independently and
    // are combined once at the end.
    const int q = warp & 3;           // TMEM lane quadrant of this warp
    const int grp = (warp - 3) >> 2;  // softmax group
    const int r = q * 32 + lane;
    const bool row_ok = r < rows;
    const int qi = r / a.G, h = r % a.G;
    const int64_t t = tq0 + qi;
    const int64_t pos = a.off + t;
    const int64_t cur = pos / B;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t tS = tl + grp * 128;         // this group's S buffer (P over its first 64 columns)
    const uint32_t tOg = tl + 256 + grp * 128;  // this group's O
    const float ninf = -__int_as_float(0x7f800000);
    const float sl2 = a.scale_log2;
    float m_used = ninf, l = 0.0f;
    bool ok = true;
    for (int i = grp;; i += 2) {
      const int ms = i % C::NM;
      // the block list of stage i, or the news that the item has no stage i
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
              ab.raise(a.status, 212);
              w = false;
              break;
            }
          }
        }
      }
      // outcomes made warp-uniform: the tcgen05.ld/st below are warp-collective
      if (!__all_sync(FULL, w)) {
        ok = false;
        break;
      }
      if (!__any_sync(FULL, have)) break;
      const bool ws = mbar_wait(&s_full[grp], (uint32_t)((i >> 1) & 1), ab, a.status, 211);
      if (!__all_sync(FULL, ws)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const Meta& m = meta_at(ms);
      const int nb = m.nb;
      const bool last = m.last != 0;
      // Allowed keys of this row among the stage's 128 keys (4 words): a whole
      // block when the query selected it and it is historical, the causal
      // prefix of the query's own block.
      uint32_t al0 = 0u, al1 = 0u, al2 = 0u, al3 = 0u;
      if (row_ok) {
        // historical blocks from the query's slot bits, widened to keys; then
        // the current blocks of the sub-tile block by block (the causal cut).
        // B = 1 takes every slot block by block.
        int bsd = 0;
        if constexpr (B >= 8) {
          const uint32_t hb = qbits_of(m, qi);
          al0 = hist_keys<B>(hb, 0);
          al1 = hist_keys<B>(hb, 1);
          al2 = hist_keys<B>(hb, 2);
          al3 = hist_keys<B>(hb, 3);
          bsd = m.diag;
        } else if constexpr (B >= 2) {
          constexpr int hw = B == 2 ? 1 : 0;  // slot word of keys 64 .. 127
          al0 = hist_keys<B>(m.qb[qi][0], 0);
          al1 = hist_keys<B>(m.qb[qi][0], 1);
          al2 = hist_keys<B>(m.qb[qi][hw], 2);
          al3 = hist_keys<B>(m.qb[qi][hw], 3);
          bsd = m.diag;
        }
#pragma unroll 1
        for (int bs = bsd; bs < nb; ++bs) {
          const int64_t b = m.blk[bs];
          int lim = 0;
          if (((m.mask[bs] >> qi) & 1ull) && b < cur)
            lim = B;
          else if (b == cur)
            lim = (int)(pos - b * B + 1);
          if (lim > 0) {
            const int k0 = bs * B;  // a block never straddles a 32-key word
            const uint32_t bits = lim >= 32 ? 0xffffffffu : ((1u << lim) - 1u);
            const uint32_t wv = bits << (uint32_t)(k0 & 31);
            const int wd = k0 >> 5;
            al0 |= wd == 0 ? wv : 0u;
            al1 |= wd == 1 ? wv : 0u;
            al2 |= wd == 2 ? wv : 0u;
            al3 |= wd == 3 ? wv : 0u;
          }
        }
      }
      // One pass when possible: p = 2^(s * scale * log2(e) - m_used) with the
      // running reference maximum, as long as the P values of each 64 keys
      // sum to at most 2^kLazy (checked before they are written).  When keys
      // 0..63 fail the check the stage is done in two passes below; when only
      // keys 64..127 do, the maximum is raised in place (stage_second_half),
      // since P of keys 0..63 already lies over their S values.  The exponent
      // arguments and the sums use packed f32x2 arithmetic.
      float rs0 = 0.0f, rs1 = 0.0f;
      bool fast = __all_sync(FULL, m_used != ninf || (al0 | al1 | al2 | al3) == 0u);
      bool mid = false;  // keys 64..127 need a higher maximum: the path below
      // Stages whose blocks are all historical (B >= 8) take the mask per
      // block: -m or -inf as the exponent's additive term.
      bool by_block = false;
      if constexpr (B >= 8) by_block = m.diag >= nb;
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      if (fast && by_block) {
        constexpr int BPHh = 64 / B;  // blocks per 64 keys
        const uint32_t hb = row_ok ? qbits_of(m, qi) : 0u;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[64];
          tmem_ld32(tS + (2 * hh) * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(tS + (2 * hh + 1) * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
          const uint32_t hbh = hb >> (hh * BPHh);
          uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
          uint32_t pk[32];
#pragma unroll
          for (int jj = 0; jj < BPHh; ++jj) {
            const float cbv = ((hbh >> jj) & 1u) ? -m_used : ninf;
            const uint64_t cb2 = f2_pack(cbv, cbv);
#pragma unroll
            for (int e = jj * B; e < jj * B + B; e += 2) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl2x2,
                               cb2),
                        x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              acc[(e >> 1) & 3] = f2_add(acc[(e >> 1) & 3], f2_pack(p0, p1));
              pk[e >> 1] = pack_bf16x2(p0, p1);
            }
          }
          float s0, s1;
          f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), s0, s1);
          const float hs = s0 + s1;
          if (__any_sync(FULL, !(hs <= kLazySum))) {
            if (hh == 0) {  // nothing written yet: the two passes below
              fast = false;
              break;
            }
            mid = true;
            break;
          }
          rs0 += hs;
          tmem_st32(tS + hh * 32, pk);  // S columns 0..63 have been read by now
        }
      } else if (fast) {
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v0[32], v1[32];
          tmem_ld32(tS + (2 * hh) * 32, v0);
          tmem_ld32(tS + (2 * hh + 1) * 32, v1);
          tmem_wait_ld();
          const uint32_t a0 = hh == 0 ? al0 : al2, a1 = hh == 0 ? al1 : al3;
          uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            // the additive term is -m for an allowed key and -inf otherwise
            float x0, x1, x2, x3;
            const float c0 = ((a0 >> e) & 1u) ? -m_used : ninf;
            const float c1 = ((a0 >> (e + 1)) & 1u) ? -m_used : ninf;
            const float c2 = ((a1 >> e) & 1u) ? -m_used : ninf;
            const float c3 = ((a1 >> (e + 1)) & 1u) ? -m_used : ninf;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v0[e]), __uint_as_float(v0[e + 1])), sl2x2,
                             f2_pack(c0, c1)),
                      x0, x1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v1[e]), __uint_as_float(v1[e + 1])), sl2x2,
                             f2_pack(c2, c3)),
                      x2, x3);
            const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
            acc[(e >> 1) & 1] = f2_add(acc[(e >> 1) & 1], f2_pack(p0, p1));
            acc[2 + ((e >> 1) & 1)] = f2_add(acc[2 + ((e >> 1) & 1)], f2_pack(p2, p3));
            pk[e >> 1] = pack_bf16x2(p0, p1);
            pk[16 + (e >> 1)] = pack_bf16x2(p2, p3);
          }
          float s0, s1;
          f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), s0, s1);
          const float hs = s0 + s1;
          if (__any_sync(FULL, !(hs <= kLazySum))) {
            if (hh == 0) {  // nothing written yet: the two passes below
              fast = false;
              break;
            }
            mid = true;
            break;
          }
          rs0 += hs;
          tmem_st32(tS + hh * 32, pk);  // S columns 0..63 have been read by now
        }
      }
      if (mid) {
        const MidState ms2 = stage_second_half<D>(tS, tOg, al2, al3, sl2, m_used, l, rs0, rs1,
                                                  &p_empty[grp], (uint32_t)(((i >> 1) - 1) & 1),
                                                  ab, a.status);
        m_used = ms2.m_used;
        l = ms2.l;
        rs0 = ms2.rs0;
        rs1 = ms2.rs1;
        if (!__all_sync(FULL, ms2.ok)) {
          ok = false;
          break;
        }
      }
      if (!fast) {
        tmem_wait_st();
        rs0 = 0.0f;
        rs1 = 0.0f;
        // pass 1: masked maximum over the 128 keys
        float mx0 = ninf, mx1 = ninf, mx2 = ninf, mx3 = ninf;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tmem_ld32(tS + cc * 32, v);
          tmem_wait_ld();
          const uint32_t am = cc == 0 ? al0 : cc == 1 ? al1 : cc == 2 ? al2 : al3;
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            mx0 = fmaxf(mx0, ((am >> e) & 1u) ? __uint_as_float(v[e]) : ninf);
            mx1 = fmaxf(mx1, ((am >> (e + 1)) & 1u) ? __uint_as_float(v[e + 1]) : ninf);
            mx2 = fmaxf(mx2, ((am >> (e + 2)) & 1u) ? __uint_as_float(v[e + 2]) : ninf);
            mx3 = fmaxf(mx3, ((am >> (e + 3)) & 1u) ? __uint_as_float(v[e + 3]) : ninf);
          }
        }
        const float smax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        // Raise the reference maximum when this stage exceeds it by more than
        // 2^kLazy.  O[grp] holds the group's earlier stages under the old maximum:
        // it is rescaled once the group's previous PV product (stage i - 2) is
        // done; each warp takes that path together (rows that do not need it
        // scale by 1).
        const bool raise = smax > m_used + kLazy;
        const bool rescale = raise && m_used != ninf;
        if (__any_sync(FULL, rescale)) {
          const bool w2 =
              mbar_wait(&p_empty[grp], (uint32_t)(((i >> 1) - 1) & 1), ab, a.status, 213);
          if (!__all_sync(FULL, w2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = rescale ? ex2(m_used - smax) : 1.0f;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(tOg + cc * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
            tmem_st32(tOg + cc * 32, ov);
          }
          tmem_wait_st();
          l *= f;
        }
        if (raise) m_used = smax;
        // pass 2: keys 64 hh .. 64 hh + 63 go to P columns 32 hh .. 32 hh + 31,
        // whose S values have been read by then.  A row with nothing allowed so
        // far has m_used = -inf and writes zeros.
        const float msub = m_used == ninf ? 0.0f : m_used;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v0[32], v1[32];
          tmem_ld32(tS + (2 * hh) * 32, v0);
          tmem_ld32(tS + (2 * hh + 1) * 32, v1);
          tmem_wait_ld();
          const uint32_t a0 = hh == 0 ? al0 : al2, a1 = hh == 0 ? al1 : al3;
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = ((a0 >> e) & 1u) ? ex2(fmaf(__uint_as_float(v0[e]), sl2, -msub)) : 0.0f;
            const float p1 =
                ((a0 >> (e + 1)) & 1u) ? ex2(fmaf(__uint_as_float(v0[e + 1]), sl2, -msub)) : 0.0f;
            const float p2 = ((a1 >> e) & 1u) ? ex2(fmaf(__uint_as_float(v1[e]), sl2, -msub)) : 0.0f;
            const float p3 =
                ((a1 >> (e + 1)) & 1u) ? ex2(fmaf(__uint_as_float(v1[e + 1]), sl2, -msub)) : 0.0f;
            rs0 += p0 + p2;
            rs1 += p1 + p3;
            pk[e >> 1] = pack_bf16x2(p0, p1);
            pk[16 + (e >> 1)] = pack_bf16x2(p2, p3);
          }
          tmem_st32(tS + hh * 32, pk);
        }
      }
      l += rs0 + rs1;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&m_empty[ms]);  // done with this stage's block list
        mbar_arrive(&p_full[grp]);
      }
      if (last) break;
    }
    // ---- epilogue: combine the groups, O / l and the log-sum-exp
    const int ns = *n_stages;
    const int n0 = (ns + 1) / 2, n1 = ns / 2;  // stages of group 0 and of group 1
    bool fin = ok && ns != 0x7fffffff;
    if (fin && n0 > 0) fin = mbar_wait(&p_empty[0], (uint32_t)((n0 - 1) & 1), ab, a.status, 215);
    if (fin && n1 > 0) fin = mbar_wait(&p_empty[1], (uint32_t)((n1 - 1) & 1), ab, a.status, 218);
    if (__all_sync(FULL, fin)) {
      xmax[grp * C::BM + r] = m_used;
      xsum[grp * C::BM + r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(l_bar);
      fin = mbar_wait(l_bar, 0, ab, a.status, 217);
    }
    if (__all_sync(FULL, fin)) {
      const float m0 = xmax[r], m1 = xmax[C::BM + r];
      const float mm = fmaxf(m0, m1);
      const float f0 = m0 == ninf ? 0.0f : ex2(m0 - mm);
      const float f1 = m1 == ninf ? 0.0f : ex2(m1 - mm);
      const float lt = xsum[r] * f0 + xsum[C::BM + r] * f1;
      tc_fence_after();
      const float inv = row_ok && lt > 0.0f ? 1.0f / lt : 0.0f;
      const float g0 = f0 * inv, g1 = f1 * inv;
      const int64_t hq = (int64_t)g * a.G + h;
      // this thread writes head-dim columns [grp * D / 2, grp * D / 2 + D / 2)
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = grp * (D / 2) + cc * 32;
        uint32_t o0[32], o1[32];
        tmem_ld32(tl + 256 + col, o0);
        if (n1 > 0) tmem_ld32(tl + 384 + col, o1);
        tmem_wait_ld();
        float ov[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          ov[e] = __uint_as_float(o0[e]) * g0 + (n1 > 0 ? __uint_as_float(o1[e]) * g1 : 0.0f);
        if (row_ok && a.nsplit > 1) {
          float* dst = a.opart + ((sp * a.T + t) * a.H + hq) * D + col;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
        } else if (row_ok) {
          if (a.out_f32) {
            float* dst = static_cast<float*>(a.O) + (t * a.H + hq) * D + col;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + e) = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.O) + (t * a.H + hq) * D + col;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 vv;
              vv.x = pack_bf16x2(ov[e], ov[e + 1]);
              vv.y = pack_bf16x2(ov[e + 2], ov[e + 3]);
              vv.z = pack_bf16x2(ov[e + 4], ov[e + 5]);
              vv.w = pack_bf16x2(ov[e + 6], ov[e + 7]);
              *reinterpret_cast<uint4*>(dst + e) = vv;
            }
          }
        }
      }
      if (row_ok && grp == 0) {
        const float l_e = (mm + __log2f(lt)) * 0.69314718055994531f;
        if (a.nsplit > 1)
          a.lpart[(sp * a.H + hq) * a.T + t] = lt > 0.0f ? l_e : ninf;
        else
          a.lse[hq * a.T + t] = l_e;
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


// Tensor map for gathering single key rows of K or V (bf16): a 2-d view
// [rows][d] with box 64 x 1 and the 128-byte swizzle.  Rows are p * Hkv + g
// for a contiguous cache; a paged cache's pool size is not passed, so its view
// spans every row a 32-bit coordinate can name and the page table bounds the
// rows actually read.
bool make_kvmap(const Dims& dm, const void* X, CUtensorMap* mx) {
  auto fn = tmap_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t e = 2;
  const cuuint32_t estr[2] = {1, 1};
  const cuuint64_t rows =
      dm.ps > 0 ? (cuuint64_t)0x7fffffff : (cuuint64_t)dm.Tkv * (cuuint64_t)dm.Hkv;
  cuuint64_t dims[2] = {(cuuint64_t)dm.d, rows};
  cuuint64_t str[1] = {dm.d * e};
  cuuint32_t box[2] = {64, 1};
  return fn(mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, str, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Merge of the splits of a work item (fixed order, so the result does not
// depend on scheduling): lse = log sum_s e^{lse_s}, O = sum_s e^{lse_s - lse}
// O_s.  One warp per (query, head) row.
template <int D>
__global__ void __launch_bounds__(256) k_attn_combine(const float* __restrict__ opart,
                                                      const float* __restrict__ lpart, int nsplit,
                                                      int64_t T, int H, void* O, float* lse,
                                                      int out_f32) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= T * H) return;
  const int lane = threadIdx.x & 31;
  const int64_t t = row / H, h = row % H;
  float mx = -__int_as_float(0x7f800000);
  for (int s2 = 0; s2 < nsplit; ++s2) mx = fmaxf(mx, lpart[(s2 * H + h) * T + t]);
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.0f;
  float sw = 0.0f;
  for (int s2 = 0; s2 < nsplit; ++s2) {
    const float l = lpart[(s2 * H + h) * T + t];
    const float w = l == mx ? 1.0f : expf(l - mx);  // e^{-inf} = 0 for an empty split
    sw += w;
    const float* src = opart + (s2 * T * H + row) * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(w, src[lane + 32 * i], acc[i]);
  }
  const float inv = 1.0f / sw;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const float v = acc[i] * inv;
    if (out_f32)
      static_cast<float*>(O)[row * D + lane + 32 * i] = v;
    else
      static_cast<__nv_bfloat16*>(O)[row * D + lane + 32 * i] = __float2bfloat16_rn(v);
  }
  if (lane == 0) lse[h * T + t] = mx + logf(sw);
}

template <int D, int B, bool PK>
int launch_db(const Dims& dm, const AttnArgs& a, const void* Q, int64_t items, cudaStream_t st) {
  using C = AttnCfg<D, B>;
  CUtensorMap mq, mk, mv;
  if (!make_qmap(dm, a.QS, Q, &mq)) return SGQA_ERR_CUDA;
  if constexpr (PK) {  // packed blocks: bulk copies, no gather maps
    memset(&mk, 0, sizeof(mk));
    memset(&mv, 0, sizeof(mv));
  } else {
    if (dm.ps == 0 && (int64_t)dm.Tkv * dm.Hkv > 0x7fffffffll) return SGQA_ERR_UNSUPPORTED;
    if (!make_kvmap(dm, a.K, &mk) || !make_kvmap(dm, a.V, &mv)) return SGQA_ERR_CUDA;
  }
  if (cudaFuncSetAttribute(k_sparse_attn<D, B, PK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM) != cudaSuccess)
    return SGQA_ERR_CUDA;
  log_begin(SGQA_K_ATTN, st);
  k_sparse_attn<D, B, PK><<<(unsigned)(items * a.nsplit), C::NTHREADS, C::SMEM, st>>>(mq, mk, mv, a);
  log_end(st);
  if (cudaGetLastError() != cudaSuccess) return SGQA_ERR_CUDA;
  if (a.nsplit > 1) {
    const int64_t rows = a.T * a.H;
    log_begin(SGQA_K_ATTN, st);
    k_attn_combine<D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(a.opart, a.lpart, a.nsplit, a.T,
                                                                  a.H, a.O, a.lse, a.out_f32);
    log_end(st);
  }
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

template <int D>
int launch_d(const Dims& dm, const AttnArgs& a, const void* Q, bool packed, int64_t items,
             cudaStream_t st) {
  switch (dm.B) {
    case 1: return launch_db<D, 1, false>(dm, a, Q, items, st);
    case 2: return launch_db<D, 2, false>(dm, a, Q, items, st);
    case 4: return launch_db<D, 4, false>(dm, a, Q, items, st);
    case 8:
      return packed ? launch_db<D, 8, true>(dm, a, Q, items, st)
                    : launch_db<D, 8, false>(dm, a, Q, items, st);
    case 16:
      return packed ? launch_db<D, 16, true>(dm, a, Q, items, st)
                    : launch_db<D, 16, false>(dm, a, Q, items, st);
    default: return SGQA_ERR_UNSUPPORTED;
  }
}

}  // namespace

int launch_sparse_attn_layout(const Dims& dm, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                              const __nv_bfloat16* V, const __nv_bfloat16* Kp,
                              const __nv_bfloat16* Vp, const int32_t* page_table,
                              const int64_t* union_off, const int32_t* union_len,
                              const int32_t* union_blk, const uint64_t* union_mask, void* O,
                              float* lse, int64_t tau_begin, int64_t tau_end, int64_t lay_tau0,
                              int64_t lay_ntiles, int32_t* status, cudaStream_t st, int nsplit,
                              float* opart, float* lpart) {
  if (tau_end <= tau_begin) return SGQA_OK;
  if (nsplit > 1 && (opart == nullptr || lpart == nullptr || tau_begin != 0 ||
                     tau_end != dm.ntiles))
    return SGQA_ERR_INVALID_ARG;
  if (dm.G > 128) return SGQA_ERR_UNSUPPORTED;
  AttnArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.Kp = Kp;
  a.Vp = Vp;
  a.nblkp = (dm.Tkv + dm.B - 1) / dm.B;
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
  a.npages = dm.ps > 0 ? (int)(dm.Tkv / dm.ps) : 0;
  a.QS = 128 / dm.G < dm.W ? 128 / dm.G : dm.W;
  a.nsub = (dm.W + a.QS - 1) / a.QS;
  a.mode = dm.mode;
  a.out_f32 = dm.dtype == SGQA_FP32;
  a.scale_log2 = dm.scale * 1.4426950408889634f;
  a.status = status;
  a.nsplit = nsplit > 1 ? nsplit : 1;
  a.opart = opart;
  a.lpart = lpart;
  const int64_t items = (tau_end - tau_begin) * dm.Hkv * a.nsub;
  // packed copies given: B >= 8 bulk copies; else key gathers from K and V
  const bool packed = Kp != nullptr && Vp != nullptr;
  if (packed && dm.B < 8) return SGQA_ERR_INVALID_ARG;
  if (dm.d == 128) return launch_d<128>(dm, a, Q, packed, items, st);
  if (dm.d == 64) return launch_d<64>(dm, a, Q, packed, items, st);
  return SGQA_ERR_UNSUPPORTED;
}

int launch_sparse_attn(const Dims& dm, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                       const __nv_bfloat16* V, const __nv_bfloat16* Kp, const __nv_bfloat16* Vp,
                       const int32_t* page_table, const int64_t* union_off,
                       const int32_t* union_len, const int32_t* union_blk,
                       const uint64_t* union_mask, void* O, float* lse, int64_t tau_begin,
                       int64_t tau_end, int32_t* status, cudaStream_t st) {
  return launch_sparse_attn_layout(dm, Q, K, V, Kp, Vp, page_table, union_off, union_len, union_blk,
                                   union_mask, O, lse, tau_begin, tau_end, 0, dm.ntiles, status,
                                   st, 1, nullptr, nullptr);
}

}  // namespace sgqa
