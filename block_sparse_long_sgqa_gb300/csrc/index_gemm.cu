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
// CTA = 128 queries x all causal blocks of one group, in steps of 128 blocks.
// Warp 0 issues TMA loads (A once, B double-buffered), warp 1 issues the
// MMAs into a double-buffered TMEM accumulator (2 x 128 fp32 columns), warps
// 2-5 drain TMEM (one query row per thread), apply the causal block mask and
// store the scores.
#include "common.cuh"
#include "internal.h"

namespace sgqa {
namespace {

template <int D>
struct IdxCfg {
  static constexpr int BM = 128, BN = 128, STAGES = 2;
  static constexpr int KC = D / 64;          // 128-byte (64-element) chunks along d
  static constexpr int A_TILE = BM * 128;    // bytes of one chunk of A
  static constexpr int B_TILE = BN * 128;
  static constexpr int A_BYTES = KC * A_TILE;
  static constexpr int B_BYTES = KC * B_TILE;
  static constexpr int OFF_AHI = 0;
  static constexpr int OFF_ALO = A_BYTES;
  static constexpr int OFF_B = 2 * A_BYTES;
  static constexpr int STAGE_BYTES = 2 * B_BYTES;  // hi + lo
  static constexpr int OFF_BAR = OFF_B + STAGES * STAGE_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr int NTHREADS = 192;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    k_index_scores(const __grid_constant__ CUtensorMap mq_hi, const __grid_constant__ CUtensorMap mq_lo,
                   const __grid_constant__ CUtensorMap mk_hi, const __grid_constant__ CUtensorMap mk_lo,
                   int64_t nq, int64_t q_begin, int64_t q_end, int64_t q_offset, int B, int64_t nblk,
                   float* __restrict__ scores, int32_t* status) {
  using C = IdxCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* a_full = bars + 0;
  uint64_t* b_full = bars + 1;     // [2]
  uint64_t* b_empty = bars + 3;    // [2]
  uint64_t* acc_full = bars + 5;   // [2]
  uint64_t* acc_empty = bars + 7;  // [2]
  uint64_t* mma_done = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  int* abort_flag = reinterpret_cast<int*>(bars + 11);

  const int g = blockIdx.y;
  const int64_t tl0 = (int64_t)(gridDim.x - 1 - blockIdx.x) * C::BM;  // heavy tiles first
  const int64_t t0 = q_begin + tl0;
  const int64_t t_last = (t0 + C::BM < q_end ? t0 + C::BM : q_end) - 1;
  int64_t nh_max = (q_offset + t_last) / B;
  if (nh_max > nblk) nh_max = nblk;
  const int n_tiles = (int)((nh_max + C::BN - 1) / C::BN);
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 4);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&mq_hi);
      tma_prefetch_desc(&mk_hi);
      const int32_t arow = (int32_t)(g * nq + tl0);
      mbar_expect_tx(a_full, 2 * C::A_BYTES);
      for (int c = 0; c < C::KC; ++c) {
        tma_load_2d(smem + C::OFF_AHI + c * C::A_TILE, &mq_hi, a_full, c * 64, arow);
        tma_load_2d(smem + C::OFF_ALO + c * C::A_TILE, &mq_lo, a_full, c * 64, arow);
      }
      int issued[2] = {0, 0};
      for (int n = 0; n < n_tiles; ++n) {
        const int s = n & 1;
        if (!mbar_wait(&b_empty[s], ((n >> 1) & 1) ^ 1, ab, status, 101)) break;
        mbar_expect_tx(&b_full[s], C::STAGE_BYTES);
        uint8_t* sb = smem + C::OFF_B + s * C::STAGE_BYTES;
        const int32_t brow = (int32_t)(g * nblk + (int64_t)n * C::BN);
        for (int c = 0; c < C::KC; ++c) {
          tma_load_2d(sb + c * C::B_TILE, &mk_hi, &b_full[s], c * 64, brow);
          tma_load_2d(sb + C::B_BYTES + c * C::B_TILE, &mk_lo, &b_full[s], c * 64, brow);
        }
        ++issued[s];
      }
      if (ab.set()) {  // let every copy this CTA started land before it exits
        mbar_wait_drain(a_full, 0, status, 198);
        for (int s = 0; s < 2; ++s)
          if (issued[s] > 0) mbar_wait_drain(&b_full[s], (issued[s] - 1) & 1, status, 197);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::BM, C::BN, 0, 0);
      const uint32_t a_hi = smem_u32(smem + C::OFF_AHI);
      const uint32_t a_lo = smem_u32(smem + C::OFF_ALO);
      if (mbar_wait(a_full, 0, ab, status, 102)) {
        for (int n = 0; n < n_tiles; ++n) {
          const int s = n & 1, acc = n & 1;
          if (!mbar_wait(&b_full[s], (n >> 1) & 1, ab, status, 103)) break;
          if (!mbar_wait(&acc_empty[acc], ((n >> 1) & 1) ^ 1, ab, status, 104)) break;
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
            umma_f16(d_t, ahi, blo, idesc, 1u);
            umma_f16(d_t, alo, bhi, idesc, 1u);
          }
          umma_commit(&b_empty[s]);
          umma_commit(&acc_full[acc]);
        }
      }
      umma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, status, 199);
    }
  } else {
    // --------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int r = q * 32 + lane;
    const int64_t t = t0 + r;
    const bool valid = t < q_end;
    int64_t nh = (q_offset + t) / B;
    if (nh > nblk) nh = nblk;
    float* row = scores + ((int64_t)g * nq + (t - q_begin)) * nblk;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool vec = (nblk & 3) == 0;
    const float ninf = -__int_as_float(0x7f800000);
    for (int n = 0; n < n_tiles; ++n) {
      const int acc = n & 1;
      // outcome made warp-uniform: tcgen05.ld below is warp-collective
      const bool w = mbar_wait(&acc_full[acc], (n >> 1) & 1, ab, status, 105);
      if (!__all_sync(0xffffffffu, w)) break;
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tl + acc * C::BN + cc * 32, v[cc]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (valid) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const int64_t j = (int64_t)n * C::BN + cc * 32 + i;
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = (j + e < nh) ? __uint_as_float(v[cc][i + e]) : ninf;
            if (vec && j + 3 < nblk) {
              *reinterpret_cast<float4*>(row + j) = make_float4(o[0], o[1], o[2], o[3]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (j + e < nblk) row[j + e] = o[e];
            }
          }
        }
      }
    }
    if (valid) {  // blocks past the last computed tile are never historical
      int64_t j = (int64_t)n_tiles * C::BN;
      if (vec) {
        for (; j + 3 < nblk; j += 4)
          *reinterpret_cast<float4*>(row + j) = make_float4(ninf, ninf, ninf, ninf);
      }
      for (; j < nblk; ++j) row[j] = ninf;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
int launch_impl(const Dims& dm, const __nv_bfloat16* qhi, const __nv_bfloat16* qlo,
                const __nv_bfloat16* khi, const __nv_bfloat16* klo, int64_t q_begin,
                int64_t q_end, float* scores, int32_t* status, cudaStream_t st) {
  using C = IdxCfg<D>;
  const int64_t nq = q_end - q_begin;
  CUtensorMap m_qhi, m_qlo, m_khi, m_klo;
  const uint64_t row_bytes = (uint64_t)D * 2;
  if (!make_tmap_2d_bf16(&m_qhi, qhi, D, (uint64_t)dm.Hkv * nq, row_bytes, 64, C::BM) ||
      !make_tmap_2d_bf16(&m_qlo, qlo, D, (uint64_t)dm.Hkv * nq, row_bytes, 64, C::BM) ||
      !make_tmap_2d_bf16(&m_khi, khi, D, (uint64_t)dm.Hkv * dm.nblk, row_bytes, 64, C::BN) ||
      !make_tmap_2d_bf16(&m_klo, klo, D, (uint64_t)dm.Hkv * dm.nblk, row_bytes, 64, C::BN))
    return SGQA_ERR_CUDA;
  if (cudaFuncSetAttribute(k_index_scores<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM) != cudaSuccess)
    return SGQA_ERR_CUDA;
  dim3 grid((unsigned)((nq + C::BM - 1) / C::BM), (unsigned)dm.Hkv);
  log_begin(SGQA_K_INDEX_SCORES, st);
  k_index_scores<D><<<grid, C::NTHREADS, C::SMEM, st>>>(m_qhi, m_qlo, m_khi, m_klo, nq, q_begin,
                                                         q_end, dm.off, dm.B, dm.nblk, scores,
                                                         status);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

}  // namespace

int launch_index_scores(const Dims& dm, const __nv_bfloat16* qhi, const __nv_bfloat16* qlo,
                        const __nv_bfloat16* khi, const __nv_bfloat16* klo, int64_t q_begin,
                        int64_t q_end, float* scores, int32_t* status, cudaStream_t st) {
  if (q_end <= q_begin || dm.nblk == 0) return SGQA_OK;  // nothing to score
  if (dm.d == 128) return launch_impl<128>(dm, qhi, qlo, khi, klo, q_begin, q_end, scores, status, st);
  if (dm.d == 64) return launch_impl<64>(dm, qhi, qlo, khi, klo, q_begin, q_end, scores, status, st);
  return SGQA_ERR_UNSUPPORTED;
}

}  // namespace sgqa
