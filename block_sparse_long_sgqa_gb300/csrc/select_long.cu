// Exact top-k of long score rows, one CTA per row.
//
// "Inside Step 5 Preview" (StepFun blog), section Sparse GQA, paragraph
// "Trade-off between top-k and block size": each query keeps its k/B best
// historical blocks (this build: ties to the lower block index, the list in
// ascending block order, fp32 scores compared through the order-preserving
// map of their bit patterns).
//
// Rows of more than 16384 blocks (1M-token caches, small block sizes) are
// too long for one warp to stream quickly, so here a 512-thread CTA takes a
// row: an 11-bit histogram of the top key bits finds the bucket holding the
// k-th largest key.  When the keys at or above that bucket fit in shared
// memory (k/B plus the bucket, up to 6144) the second pass keeps them with
// their blocks, 11-bit radix levels among the bucket's resolve the k-th key
// exactly, and the taken blocks (above it, and of those equal to it the
// lowest-indexed) are marked in a bitmap over the row read out in block order
// by a CTA prefix sum: two passes over the row.  Otherwise the bucket's keys
// alone are compacted (or, for a bucket too large, the row is histogrammed
// again one digit lower), and a third pass over the row in block order writes
// every block above the k-th key and the lowest-indexed ones equal to it:
// each thread takes four consecutive blocks per step and one CTA-wide prefix
// sum per step (blocks above, blocks equal) gives every block its place.
#include "common.cuh"
#include "internal.h"

namespace sgqa {
namespace {

constexpr int SL_THREADS = 512;
constexpr int SL_WARPS = SL_THREADS / 32;
constexpr int SL_BINS = 2048;  // 11-bit digits
constexpr int SL_CAP = 4096;   // bucket members resolved in shared memory
constexpr int SL_CAP2 = 6144;  // keys at or above the bucket kept with their blocks
constexpr int SL_BMAX = 131072;  // longest row the bitmap emission covers

struct SLArgs {
  const float* scores;  // [Hkv][nq][nblk]
  int64_t nq, q_begin, off, nblk;
  int64_t r_first;      // rows r_first .. nq-1 (local) of every group
  int lgB, Ks;
  int32_t* sel;         // [Hkv][nq][Ks]
  int32_t* status;
};

struct SLShared {
  uint32_t hist[SL_BINS];
  uint32_t ckey[SL_CAP2];  // compacted keys (the bucket's, or all at or above it)
  uint32_t cidx[SL_CAP2];  // their blocks (two-pass form)
  uint32_t bmA[SL_BMAX / 32];  // taken blocks (two-pass form)
  uint32_t bmE[SL_BMAX / 32];  // blocks tied at the k-th key
  uint32_t wsum[SL_WARPS];
  uint32_t ccount;
  uint32_t b_bin, b_above, b_cnt;
};

// CTA-wide exclusive prefix sum of v (thread order); *total gets the sum.
__device__ uint32_t cta_excl_scan(SLShared& sm, uint32_t v, uint32_t* total) {
  const int lane = lane_id(), warp = warp_id();
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.wsum[warp] = incl;
  __syncthreads();
  uint32_t base = 0, tot = 0;
  for (int w = 0; w < SL_WARPS; ++w) {
    const uint32_t x = sm.wsum[w];
    if (w < warp) base += x;
    tot += x;
  }
  __syncthreads();  // wsum is reused by the next scan
  *total = tot;
  return base + incl - v;
}

// Bucket search over hist (SL_BINS bins) for the rem-th largest: the bin b,
// the count in bins above it and its own count (broadcast through sh).
__device__ void cta_find_bin(SLShared& sm, uint32_t rem) {
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  constexpr int PER = SL_BINS / SL_THREADS;  // 4 bins per thread, thread 0 the highest
  const int hi = SL_BINS - PER * tid;        // bins [hi - PER, hi)
  uint32_t s = 0;
#pragma unroll
  for (int i = 1; i <= PER; ++i) s += sm.hist[hi - i];
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.wsum[warp] = incl;
  __syncthreads();
  uint32_t wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += sm.wsum[w];
  const uint32_t excl = wbase + incl - s;  // keys in bins above this thread's
  if (excl < rem && rem <= excl + s) {
    uint32_t acc = excl;
#pragma unroll
    for (int i = 1; i <= PER; ++i) {
      const uint32_t h = sm.hist[hi - i];
      if (acc + h >= rem) {
        sm.b_bin = (uint32_t)(hi - i);
        sm.b_above = acc;
        sm.b_cnt = h;
        break;
      }
      acc += h;
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(SL_THREADS) k_select_long(SLArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SLShared& sm = *reinterpret_cast<SLShared*>(smem_raw);
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  const int64_t nlong = a.nq - a.r_first;
  const int g = (int)(blockIdx.x / nlong);
  const int64_t r = a.r_first + blockIdx.x % nlong;
  const int64_t t = a.q_begin + r;
  int64_t nh = (a.off + t) >> a.lgB;
  if (nh > a.nblk) nh = a.nblk;
  const uint32_t need = (uint32_t)(nh < a.Ks ? nh : a.Ks);
  int32_t* out = a.sel + ((int64_t)g * a.nq + r) * a.Ks;
  if ((int64_t)need == nh) {  // every historical block (or none)
    for (int64_t x = tid; x < a.Ks; x += SL_THREADS) out[x] = x < nh ? (int32_t)x : -1;
    return;
  }
  const float* row = a.scores + ((int64_t)g * a.nq + r) * a.nblk;
  const bool vec = (a.nblk & 3) == 0;
  const int64_t n4 = vec ? nh / 4 : 0;

  // ---- resolve the need-th largest key: prefix T of the keys at shift sh
  uint32_t T = 0, rem = need, cnt = (uint32_t)nh;
  int sh = 32;
  bool in_smem = false;  // the bucket's keys are in sm.ckey (ncand of them)
  uint32_t ncand = 0;
  auto match = [&](uint32_t key) { return sh >= 32 || (key >> sh) == T; };
  while (cnt != rem && sh > 0) {
    const int w = sh < 11 ? sh : 11;
    const int nsh = sh - w;
    const uint32_t dmask = (1u << w) - 1u;
    for (int i = tid; i < SL_BINS; i += SL_THREADS) sm.hist[i] = 0u;
    __syncthreads();
    if (in_smem) {
      for (uint32_t i = tid; i < ncand; i += SL_THREADS) {
        const uint32_t key = sm.ckey[i];
        if (match(key)) atomicAdd(&sm.hist[(key >> nsh) & dmask], 1u);
      }
    } else {
      for (int64_t x = tid; x < n4; x += SL_THREADS) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(row) + x);
        const uint32_t k0 = order_key(v.x), k1 = order_key(v.y), k2 = order_key(v.z),
                       k3 = order_key(v.w);
        if (match(k0)) atomicAdd(&sm.hist[(k0 >> nsh) & dmask], 1u);
        if (match(k1)) atomicAdd(&sm.hist[(k1 >> nsh) & dmask], 1u);
        if (match(k2)) atomicAdd(&sm.hist[(k2 >> nsh) & dmask], 1u);
        if (match(k3)) atomicAdd(&sm.hist[(k3 >> nsh) & dmask], 1u);
      }
      for (int64_t j = n4 * 4 + tid; j < nh; j += SL_THREADS) {
        const uint32_t key = order_key(__ldg(row + j));
        if (match(key)) atomicAdd(&sm.hist[(key >> nsh) & dmask], 1u);
      }
    }
    __syncthreads();
    cta_find_bin(sm, rem);
    T = (sh >= 32 ? 0u : (T << w)) | sm.b_bin;
    rem -= sm.b_above;
    cnt = sm.b_cnt;
    sh = nsh;
    if (!in_smem && sh == 21 && nh <= SL_BMAX && (need - rem) + cnt <= (uint32_t)SL_CAP2) {
      // ---- two-pass form: keep every key at or above the bucket with its
      // block, resolve the bucket among them, and emit from bitmaps over the
      // row's blocks (no third pass over the row)
      if (tid == 0) sm.ccount = 0u;
      __syncthreads();
      for (int64_t j = tid; j < nh; j += SL_THREADS) {
        const uint32_t key = order_key(__ldg(row + j));
        if ((key >> sh) >= T) {
          const uint32_t p = atomicAdd(&sm.ccount, 1u);
          if (p < (uint32_t)SL_CAP2) {
            sm.ckey[p] = key;
            sm.cidx[p] = (uint32_t)j;
          }
        }
      }
      __syncthreads();
      const uint32_t n2 = sm.ccount < (uint32_t)SL_CAP2 ? sm.ccount : (uint32_t)SL_CAP2;
      if (sm.ccount != (need - rem) + cnt && tid == 0) report(a.status, SGQA_ERR_BOUNDS, (int)t);
      while (cnt != rem && sh > 0) {  // the bucket's remaining digits
        const int w2 = sh < 11 ? sh : 11;
        const int nsh2 = sh - w2;
        const uint32_t m2 = (1u << w2) - 1u;
        for (int i = tid; i < SL_BINS; i += SL_THREADS) sm.hist[i] = 0u;
        __syncthreads();
        for (uint32_t i = tid; i < n2; i += SL_THREADS) {
          const uint32_t key = sm.ckey[i];
          if ((key >> sh) == T) atomicAdd(&sm.hist[(key >> nsh2) & m2], 1u);
        }
        __syncthreads();
        cta_find_bin(sm, rem);
        T = (T << w2) | sm.b_bin;
        rem -= sm.b_above;
        cnt = sm.b_cnt;
        sh = nsh2;
        __syncthreads();
      }
      const int nwords = (int)((nh + 31) >> 5);
      for (int i = tid; i < nwords; i += SL_THREADS) {
        sm.bmA[i] = 0u;
        sm.bmE[i] = 0u;
      }
      __syncthreads();
      const bool tie2 = cnt != rem;
      for (uint32_t i = tid; i < n2; i += SL_THREADS) {
        const uint32_t key = sm.ckey[i], j = sm.cidx[i];
        const uint32_t p = key >> sh;  // sh < 32 here
        const uint32_t bit = 1u << (j & 31);
        if (p > T || (p == T && !tie2)) atomicOr(&sm.bmA[j >> 5], bit);
        else if (p == T) atomicOr(&sm.bmE[j >> 5], bit);
      }
      __syncthreads();
      // each thread owns a contiguous run of bitmap words
      const int per = (nwords + SL_THREADS - 1) / SL_THREADS;
      const int w0 = tid * per, w1 = min(nwords, w0 + per);
      uint32_t tot = 0;
      if (tie2) {  // the first `rem` tied blocks in block order join the taken ones
        uint32_t c = 0;
        for (int w = w0; w < w1; ++w) c += __popc(sm.bmE[w]);
        int left = (int)rem - (int)cta_excl_scan(sm, c, &tot);
        for (int w = w0; w < w1 && left > 0; ++w) {
          const uint32_t e = sm.bmE[w];
          const int n = __popc(e);
          if (n <= left) {
            sm.bmA[w] |= e;
            left -= n;
          } else {
            sm.bmA[w] |= e & ((2u << __fns(e, 0, left)) - 1u);  // its lowest `left` bits
            left = 0;
          }
        }
        __syncthreads();
      }
      uint32_t c = 0;
      for (int w = w0; w < w1; ++w) c += __popc(sm.bmA[w]);
      uint32_t pos = cta_excl_scan(sm, c, &tot);
      for (int w = w0; w < w1; ++w) {
        uint32_t m = sm.bmA[w];
        while (m) {
          if (pos < need) out[pos] = w * 32 + (__ffs(m) - 1);
          ++pos;
          m &= m - 1u;
        }
      }
      for (int64_t x = need + tid; x < a.Ks; x += SL_THREADS) out[x] = -1;
      if (tid == 0 && tot != need) report(a.status, SGQA_ERR_BOUNDS, (int)t);
      return;
    }
    if (!in_smem && cnt != rem && sh > 0 && cnt <= (uint32_t)SL_CAP) {
      // compact the bucket's members (any order) for the remaining levels
      if (tid == 0) sm.ccount = 0u;
      __syncthreads();
      for (int64_t j = tid; j < nh; j += SL_THREADS) {
        const uint32_t key = order_key(__ldg(row + j));
        if ((key >> sh) == T) {
          const uint32_t p = atomicAdd(&sm.ccount, 1u);
          if (p < (uint32_t)SL_CAP) sm.ckey[p] = key;
        }
      }
      __syncthreads();
      ncand = sm.ccount < (uint32_t)SL_CAP ? sm.ccount : (uint32_t)SL_CAP;
      if (sm.ccount != cnt && tid == 0) report(a.status, SGQA_ERR_BOUNDS, (int)t);
      in_smem = true;
    }
    __syncthreads();  // hist and the broadcast slots are reused next level
  }

  // ---- emission in block order: keys above the prefix, and the first `rem`
  // keys equal to it (all of them when cnt == rem)
  const bool ties = cnt != rem;  // only possible at sh == 0: exact ties
  uint32_t g_run = 0, e_run = 0;  // taken-above and equal keys of earlier steps
  for (int64_t j0 = 0; j0 < nh; j0 += 4 * SL_THREADS) {
    const int64_t jb = j0 + 4 * tid;
    uint32_t kk[4];
    bool inb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      inb[u] = jb + u < nh;
      kk[u] = inb[u] ? order_key(__ldg(row + jb + u)) : 0u;
    }
    uint32_t gt = 0, eq = 0;
    int cls[4];  // 2: above, 1: equal, 0: below or past the row
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t p = sh >= 32 ? 0u : (kk[u] >> sh);
      cls[u] = !inb[u] ? 0 : (p > T ? 2 : (p == T ? 1 : 0));
      if (cls[u] == 1 && !ties) cls[u] = 2;  // every equal key is taken
      gt += cls[u] == 2;
      eq += cls[u] == 1;
    }
    const uint32_t mine = (eq << 16) | gt;
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sm.wsum[warp] = incl;
    __syncthreads();
    uint32_t wbase = 0, tot = 0;
    for (int w = 0; w < SL_WARPS; ++w) {
      const uint32_t v = sm.wsum[w];
      if (w < warp) wbase += v;
      tot += v;
    }
    __syncthreads();  // wsum is rewritten next step
    const uint32_t excl = wbase + incl - mine;
    uint32_t gb = g_run + (excl & 0xffffu), eb = e_run + (excl >> 16);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (cls[u] == 2) {
        const uint32_t pos = gb + (eb < rem ? eb : rem);
        if (pos < need) out[pos] = (int32_t)(jb + u);
        ++gb;
      } else if (cls[u] == 1) {
        if (eb < rem) {
          const uint32_t pos = gb + eb;
          if (pos < need) out[pos] = (int32_t)(jb + u);
        }
        ++eb;
      }
    }
    g_run += tot & 0xffffu;
    e_run += tot >> 16;
  }
  for (int64_t x = need + tid; x < a.Ks; x += SL_THREADS) out[x] = -1;
  if (tid == 0 && g_run + (e_run < rem ? e_run : rem) != need)
    report(a.status, SGQA_ERR_BOUNDS, (int)t);
}

}  // namespace

// First local row of [q_begin, q_end) whose select runs here (rows of more
// than kFiltMaxNh blocks that do not take every block); q_end - q_begin if none.
int64_t long_rows_first(const Dims& dm, int64_t q_begin, int64_t q_end) {
  int64_t lo = q_begin, hi = q_end;  // nh grows with the query: binary search
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    const int64_t nh = nh_of(dm, mid);
    if (nh > kFiltMaxNh && nh > dm.Ks)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo - q_begin;
}

int launch_select_long(const Dims& dm, const float* scores, int64_t q_begin, int64_t q_end,
                       int64_t r_first, int32_t* sel, int32_t* status, cudaStream_t st) {
  const int64_t nq = q_end - q_begin;
  if (r_first >= nq) return SGQA_OK;
  SLArgs a;
  a.scores = scores;
  a.nq = nq;
  a.q_begin = q_begin;
  a.off = dm.off;
  a.nblk = dm.nblk;
  a.r_first = r_first;
  a.lgB = __builtin_ctz((unsigned)dm.B);
  a.Ks = dm.Ks;
  a.sel = sel;
  a.status = status;
  const size_t smem = sizeof(SLShared);
  if (cudaFuncSetAttribute(k_select_long, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SGQA_ERR_CUDA;
  const int64_t ctas = (nq - r_first) * dm.Hkv;
  log_begin(SGQA_K_TOPK_UNION, st);
  k_select_long<<<(unsigned)ctas, SL_THREADS, smem, st>>>(a);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

}  // namespace sgqa
