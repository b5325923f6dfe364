// Streaming kernels of the path (HBM-bound, no tensor cores):
//  - block merge: the block representation of "Reducing indexer's cost"
//    (Inside Step 5 Preview, section Sparse GQA), the mean of B adjacent keys;
//  - the bf16 hi/lo split of the block keys and of the group index queries
//    that feeds the tensor-core indexer;
//  - fp32 -> bf16 staging of attention operands.
#include "common.cuh"
#include "internal.h"

namespace sgqa {
namespace {

template <typename T>
struct Vec8;  // 8 consecutive elements loaded as one 16- or 32-byte access

template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

__device__ __forceinline__ void split_store8(const float (&v)[8], __nv_bfloat16* hi,
                                             __nv_bfloat16* lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]);
    __nv_bfloat16 h1 = __float2bfloat16_rn(v[2 * i + 1]);
    float r0 = __fsub_rn(v[2 * i], __bfloat162float(h0));  // exact in fp32
    float r1 = __fsub_rn(v[2 * i + 1], __bfloat162float(h1));
    __nv_bfloat162 hh(h0, h1);
    h[i] = *reinterpret_cast<uint32_t*>(&hh);
    l[i] = pack_bf16x2(r0, r1);
  }
  *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

// One unit = one (block, group): CH = d / 8 threads, each 8 consecutive
// head-dim lanes of the block's B rows (B independent 16- or 32-byte loads).
// Sum of the B rows as adjacent pairs level by level, then times 1/B.  The
// unit's rows sit in one page (the page size is a multiple of B), so a paged
// cache costs one page-table read per unit.
template <typename T, int B, int CH>
__global__ void __launch_bounds__(256) k_block_merge(const T* __restrict__ K,
                                                     const int32_t* __restrict__ page_table,
                                                     int64_t blk_begin, int64_t nblocks, int Hkv,
                                                     int ps, int64_t nblk,
                                                     float* __restrict__ Kbar,
                                                     __nv_bfloat16* __restrict__ khi,
                                                     __nv_bfloat16* __restrict__ klo) {
  constexpr int D = CH * 8;
  constexpr int UPB = 256 / CH;  // units per CTA pass
  const int c = threadIdx.x % CH;
  const int64_t units = nblocks * Hkv;
  // rows of one (position run, group) are D apart in a page, Hkv * D apart
  // in a contiguous cache
  const int64_t rstride = ps > 0 ? D : (int64_t)Hkv * D;
  for (int64_t u = (int64_t)blockIdx.x * UPB + threadIdx.x / CH; u < units;
       u += (int64_t)gridDim.x * UPB) {
    const int64_t jr = u / Hkv;
    const int g = (int)(u - jr * Hkv);
    const int64_t j = blk_begin + jr;
    const int64_t p0 = j * B;
    const T* row;
    if (ps > 0) {
      const int64_t lp = p0 / ps;
      const int64_t phys = page_table[lp];
      row = K + ((phys * Hkv + g) * ps + (p0 - lp * ps)) * (int64_t)D + c * 8;
    } else {
      row = K + (p0 * Hkv + g) * (int64_t)D + c * 8;
    }
    float v[B][8];
#pragma unroll
    for (int r = 0; r < B; ++r) Vec8<T>::load(row + r * rstride, v[r]);
#pragma unroll
    for (int w = B; w > 1; w /= 2)
#pragma unroll
      for (int r = 0; r < w / 2; ++r)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[r][i] = __fadd_rn(v[2 * r][i], v[2 * r + 1][i]);
    const float inv = 1.0f / (float)B;  // exact: B is a power of two
#pragma unroll
    for (int i = 0; i < 8; ++i) v[0][i] = __fmul_rn(v[0][i], inv);
    const int64_t o = ((int64_t)g * nblk + j) * D + c * 8;
    float4* dst = reinterpret_cast<float4*>(Kbar + o);
    dst[0] = make_float4(v[0][0], v[0][1], v[0][2], v[0][3]);
    dst[1] = make_float4(v[0][4], v[0][5], v[0][6], v[0][7]);
    if (khi != nullptr) split_store8(v[0], khi + o, klo + o);
  }
}

__global__ void __launch_bounds__(256) k_split_kbar(const float* __restrict__ Kbar, int64_t n8,
                                                    __nv_bfloat16* __restrict__ khi,
                                                    __nv_bfloat16* __restrict__ klo) {
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < n8;
       x += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
    Vec8<float>::load(Kbar + x * 8, v);
    split_store8(v, khi + x * 8, klo + x * 8);
  }
}

// Group index query: qt[g][t] = (1/G) * sum of the G heads of group g, summed
// in head order in fp32, then split into bf16 hi/lo.  Output [Hkv][nq][d].
template <typename T>
__global__ void __launch_bounds__(256) k_index_query(const T* __restrict__ Q, int64_t q_begin,
                                                     int64_t nq, int H, int Hkv, int G, int d,
                                                     __nv_bfloat16* __restrict__ qhi,
                                                     __nv_bfloat16* __restrict__ qlo) {
  const int chunks = d / 8;
  const int64_t total = nq * Hkv * chunks;
  const float invG = 1.0f / (float)G;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(x % chunks);
    const int g = (int)((x / chunks) % Hkv);
    const int64_t tl = x / ((int64_t)chunks * Hkv);
    float acc[8], v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int h = 0; h < G; ++h) {
      Vec8<T>::load(Q + ((q_begin + tl) * H + g * G + h) * (int64_t)d + c * 8, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], v[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fmul_rn(acc[i], invG);
    const int64_t o = ((int64_t)g * nq + tl) * d + c * 8;
    split_store8(acc, qhi + o, qlo + o);
  }
}

__global__ void __launch_bounds__(256) k_to_bf16(const float* __restrict__ in, int64_t n8,
                                                 __nv_bfloat16* __restrict__ out) {
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < n8;
       x += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
    Vec8<float>::load(in + x * 8, v);
    uint4 u = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                         pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
    *reinterpret_cast<uint4*>(out + x * 8) = u;
  }
}

// fp32 K or V of a paged cache -> bf16 in the contiguous [Tkv][Hkv][d]
// layout: eight head-dim lanes of one (position, group) row per thread, the
// row found through the page table.
__global__ void __launch_bounds__(256) k_to_bf16_paged(const float* __restrict__ in,
                                                       const int32_t* __restrict__ page_table,
                                                       int ps, int64_t Tkv, int Hkv, int d,
                                                       __nv_bfloat16* __restrict__ out) {
  const int d8 = d / 8;
  const int64_t n8 = Tkv * Hkv * d8;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < n8;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = x / d8;
    const int c = (int)(x % d8);
    const int64_t p = row / Hkv;
    const int g = (int)(row % Hkv);
    const float* src =
        in + (((int64_t)page_table[p / ps] * Hkv + g) * ps + p % ps) * d + (int64_t)c * 8;
    float v[8];
    Vec8<float>::load(src, v);
    uint4 u = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                         pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
    *reinterpret_cast<uint4*>(out + x * 8) = u;
  }
}

// Eight consecutive elements as bf16 (16 bytes): copied as they are from a
// bf16 cache, rounded to nearest from an fp32 one.
__device__ __forceinline__ uint4 load_bf16x8(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint4 load_bf16x8(const float* p) {
  float v[8];
  Vec8<float>::load(p, v);
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// Block-packed K/V for the attention gathers: block j of KV head g becomes
// B/8 groups of 8 positions; each group holds its d/64 head-dim halves as
// 1 KB atoms of 8 rows x 128 B with the 128-byte swizzle (16-byte unit u of
// row r stored at unit u ^ r).  One block is then one contiguous copy that
// lands directly in the layout the tensor cores read.  Positions at or past
// Tkv (a partial last block) and the extra block at index nblkp are zero.
// Output [Hkv][nblkp + 1][B * d] bf16, nblkp = ceil(Tkv / B).
// One (group, block) = CH = d / 8 threads, each one 16-byte unit of the
// block's B rows (loaded up to eight rows at a time, then stored); the
// block's rows sit in one page (the page size is a multiple of B).
template <typename T, int B, int CH>
__global__ void __launch_bounds__(256) k_kv_pack(const T* __restrict__ X,
                                                 const int32_t* __restrict__ page_table,
                                                 int64_t Tkv, int Hkv, int ps, int64_t nblkp,
                                                 __nv_bfloat16* __restrict__ out) {
  constexpr int D = CH * 8, KC = D / 64;
  constexpr int UPB = 256 / CH;      // (group, block) pairs per CTA pass
  constexpr int RB = B < 8 ? B : 8;  // rows in flight per thread
  const int u = threadIdx.x % CH, c = u >> 3, uu = u & 7;
  const int64_t nbp = nblkp + 1;
  const int64_t pairs = (int64_t)Hkv * nbp;
  const int64_t rstride = ps > 0 ? D : (int64_t)Hkv * D;
  for (int64_t x = (int64_t)blockIdx.x * UPB + threadIdx.x / CH; x < pairs;
       x += (int64_t)gridDim.x * UPB) {
    const int64_t gq = x / nbp;
    const int g = (int)gq;
    const int64_t j = x - gq * nbp;
    const int64_t p0 = j * B;
    const T* row = nullptr;
    if (j < nblkp) {
      if (ps > 0) {
        const int64_t lp = p0 / ps;
        const int64_t phys = page_table[lp];
        row = X + ((phys * Hkv + g) * ps + (p0 - lp * ps)) * (int64_t)D + u * 8;
      } else {
        row = X + (p0 * Hkv + g) * (int64_t)D + u * 8;
      }
    }
    // rows of the block that exist (a partial last block, the zero block)
    const int nval = row == nullptr ? 0 : (Tkv - p0 < B ? (int)(Tkv - p0) : B);
    __nv_bfloat16* blk = out + x * (int64_t)(B * D);  // x = g * nbp + j
#pragma unroll
    for (int r0 = 0; r0 < B; r0 += RB) {
      uint4 w[RB];
#pragma unroll
      for (int k = 0; k < RB; ++k)
        w[k] = r0 + k < nval ? load_bf16x8(row + (r0 + k) * rstride) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int k = 0; k < RB; ++k) {
        const int rr = r0 + k, r8 = rr & 7, grp = rr >> 3;
        const int o = (grp * KC * 1024 + c * 1024 + r8 * 128 + ((uu ^ r8) << 4)) / 2;
        *reinterpret_cast<uint4*>(blk + o) = w[k];
      }
    }
  }
}

// Sampled block keys for the candidate thresholds of the fused prefill: of
// every 64 blocks of a group, the first 8 (the hi half, and the lo half when
// slo is given; 16 bytes per thread): out[g][s] = in[g][(s / 8) * 64 + s % 8].
__global__ void __launch_bounds__(256) k_sample_keys(const uint4* __restrict__ khi,
                                                     const uint4* __restrict__ klo, int64_t nblk,
                                                     int64_t ns, int Hkv, int c16,
                                                     uint4* __restrict__ shi,
                                                     uint4* __restrict__ slo) {
  const int64_t n = (int64_t)Hkv * ns * c16;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < n;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t c = x % c16, r = x / c16;
    const int64_t g = r / ns, si = r % ns;
    const int64_t src = (g * nblk + (si >> 3) * 64 + (si & 7)) * c16 + c;
    shi[x] = khi[src];
    if (slo != nullptr) slo[x] = klo[src];
  }
}

int grid_for(int64_t work) {
  // enough CTAs to cover every SM several times; grid-stride loops do the rest
  int64_t g = (work + 255) / 256;
  const int64_t cap = 152 * 16;
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

template <typename T>
cudaError_t merge_dispatch(const Dims& dm, const T* K, const int32_t* pt, int64_t b0, int64_t nb,
                           float* Kbar, __nv_bfloat16* khi, __nv_bfloat16* klo, cudaStream_t st) {
  if (dm.d != 128 && dm.d != 64) return cudaErrorInvalidValue;
  const int grid = grid_for(nb * dm.Hkv * (dm.d / 8));
  log_begin(SGQA_K_MERGE, st);
  bool known = true;
#define SGQA_MERGE_CASE(BB)                                                                   \
  case BB:                                                                                    \
    if (dm.d == 128)                                                                          \
      k_block_merge<T, BB, 16><<<grid, 256, 0, st>>>(K, pt, b0, nb, dm.Hkv, dm.ps, dm.nblk,   \
                                                     Kbar, khi, klo);                         \
    else                                                                                      \
      k_block_merge<T, BB, 8><<<grid, 256, 0, st>>>(K, pt, b0, nb, dm.Hkv, dm.ps, dm.nblk,    \
                                                    Kbar, khi, klo);                          \
    break;
  switch (dm.B) {
    SGQA_MERGE_CASE(1)
    SGQA_MERGE_CASE(2)
    SGQA_MERGE_CASE(4)
    SGQA_MERGE_CASE(8)
    SGQA_MERGE_CASE(16)
    default:
      known = false;
  }
#undef SGQA_MERGE_CASE
  log_end(st);
  if (!known) return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_merge(const Dims& dm, const void* K, const int32_t* page_table,
                               int64_t blk_begin, int64_t blk_end, float* Kbar,
                               __nv_bfloat16* khi, __nv_bfloat16* klo, cudaStream_t st) {
  const int64_t nb = blk_end - blk_begin;
  if (nb <= 0) return cudaSuccess;
  if (dm.dtype == SGQA_BF16)
    return merge_dispatch(dm, static_cast<const __nv_bfloat16*>(K), page_table, blk_begin, nb,
                          Kbar, khi, klo, st);
  return merge_dispatch(dm, static_cast<const float*>(K), page_table, blk_begin, nb, Kbar, khi,
                        klo, st);
}

cudaError_t launch_split_kbar(const Dims& dm, const float* Kbar, __nv_bfloat16* khi,
                              __nv_bfloat16* klo, cudaStream_t st) {
  const int64_t n8 = (int64_t)dm.Hkv * dm.nblk * dm.d / 8;
  if (n8 == 0) return cudaSuccess;
  log_begin(SGQA_K_SPLIT, st);
  k_split_kbar<<<grid_for(n8), 256, 0, st>>>(Kbar, n8, khi, klo);
  log_end(st);
  return cudaGetLastError();
}

cudaError_t launch_sample_keys(const Dims& dm, const __nv_bfloat16* khi, const __nv_bfloat16* klo,
                               __nv_bfloat16* shi, __nv_bfloat16* slo, cudaStream_t st,
                               int64_t krows) {
  const int64_t ns = sampled_cols(dm);
  const int c16 = dm.d / 8;
  const int64_t n = (int64_t)dm.Hkv * ns * c16;
  if (n == 0) return cudaSuccess;
  log_begin(SGQA_K_SPLIT, st);
  k_sample_keys<<<grid_for(n), 256, 0, st>>>(reinterpret_cast<const uint4*>(khi),
                                             reinterpret_cast<const uint4*>(klo),
                                             krows > 0 ? krows : dm.nblk, ns,
                                             dm.Hkv, c16, reinterpret_cast<uint4*>(shi),
                                             reinterpret_cast<uint4*>(slo));
  log_end(st);
  return cudaGetLastError();
}

cudaError_t launch_index_query(const Dims& dm, const void* Q, int64_t q_begin, int64_t q_end,
                               __nv_bfloat16* qhi, __nv_bfloat16* qlo, cudaStream_t st) {
  const int64_t nq = q_end - q_begin;
  if (nq <= 0) return cudaSuccess;
  const int grid = grid_for(nq * dm.Hkv * (dm.d / 8));
  log_begin(SGQA_K_INDEX_QUERY, st);
  if (dm.dtype == SGQA_BF16)
    k_index_query<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(Q), q_begin, nq, dm.H,
                                        dm.Hkv, dm.G, dm.d, qhi, qlo);
  else
    k_index_query<<<grid, 256, 0, st>>>(static_cast<const float*>(Q), q_begin, nq, dm.H, dm.Hkv,
                                        dm.G, dm.d, qhi, qlo);
  log_end(st);
  return cudaGetLastError();
}

namespace {

template <typename T>
cudaError_t kv_pack_dispatch(const Dims& dm, const T* X, const int32_t* pt, int64_t nblkp,
                             __nv_bfloat16* out, cudaStream_t st) {
  if (dm.d != 128 && dm.d != 64) return cudaErrorInvalidValue;
  const int grid = grid_for((int64_t)dm.Hkv * (nblkp + 1) * (dm.d / 8));
  bool known = true;
  log_begin(SGQA_K_STAGE, st);
#define SGQA_PACK_CASE(BB)                                                                      \
  case BB:                                                                                      \
    if (dm.d == 128)                                                                            \
      k_kv_pack<T, BB, 16><<<grid, 256, 0, st>>>(X, pt, dm.Tkv, dm.Hkv, dm.ps, nblkp, out);     \
    else                                                                                        \
      k_kv_pack<T, BB, 8><<<grid, 256, 0, st>>>(X, pt, dm.Tkv, dm.Hkv, dm.ps, nblkp, out);      \
    break;
  switch (dm.B) {
    SGQA_PACK_CASE(8)
    SGQA_PACK_CASE(16)
    default:
      known = false;
  }
#undef SGQA_PACK_CASE
  log_end(st);
  if (!known) return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_pack(const Dims& dm, const void* X, const int32_t* page_table,
                           __nv_bfloat16* out, cudaStream_t st) {
  const int64_t nblkp = (dm.Tkv + dm.B - 1) / dm.B;
  if (dm.dtype == SGQA_BF16)
    return kv_pack_dispatch(dm, static_cast<const __nv_bfloat16*>(X), page_table, nblkp, out, st);
  return kv_pack_dispatch(dm, static_cast<const float*>(X), page_table, nblkp, out, st);
}

cudaError_t launch_to_bf16(const float* in, __nv_bfloat16* out, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  log_begin(SGQA_K_STAGE, st);
  k_to_bf16<<<grid_for(n / 8), 256, 0, st>>>(in, n / 8, out);
  log_end(st);
  return cudaGetLastError();
}

cudaError_t launch_kv_to_bf16(const Dims& dm, const float* in, const int32_t* page_table,
                              __nv_bfloat16* out, cudaStream_t st) {
  if (dm.ps == 0) return launch_to_bf16(in, out, dm.Tkv * dm.Hkv * dm.d, st);
  const int64_t n8 = dm.Tkv * dm.Hkv * (dm.d / 8);
  if (n8 <= 0) return cudaSuccess;
  log_begin(SGQA_K_STAGE, st);
  k_to_bf16_paged<<<grid_for(n8), 256, 0, st>>>(in, page_table, dm.ps, dm.Tkv, dm.Hkv, dm.d,
                                                 out);
  log_end(st);
  return cudaGetLastError();
}

}  // namespace sgqa
