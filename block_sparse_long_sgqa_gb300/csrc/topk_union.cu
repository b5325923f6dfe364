// Top-k block selection and tile union.
//
// "Inside Step 5 Preview" (StepFun blog), section Sparse GQA: each query keeps
// its k/B best historical blocks (paragraph "Trade-off between top-k and block
// size"), and the selections of adjacent queries are unioned so one gathered
// block list serves a whole tile (paragraph "Efficient implementation of
// sparse attention").
//
// Two kernels.  The row kernel runs an exact select per query row (one warp
// per row, persistent CTAs, rows dealt out in blocks of 8 consecutive
// queries) on the row's fp32 scores, compared through the order-preserving
// map of their bit patterns, and writes each list in ascending block order.
// Rows of 2048 .. 16384 blocks take the candidate path: a float threshold that
// a little more than k/B of the row's scores clear (predicted from the
// previous row of the same warp, else from a sample of 8 adjacent blocks in
// every 64), one pass that compacts the scores above it into shared memory in
// block order, and a radix select with ties to the lowest index on those
// candidates, so the row is read once.  Other rows, and rows whose candidates
// miss the selection or overflow, take the histogram path: an 11-bit
// histogram of the top key bits finds the bucket of the k-th largest key, the
// bucket is refined by further levels (in shared memory when it is small),
// and an ascending pass emits every block above the k-th key plus the
// lowest-indexed blocks equal to it.  The tile kernel (one CTA per tile and
// group) ORs the tile's lists into a block bitmask; the union is the set bits
// (ranks by a prefix sum of word popcounts), and a member mask per union slot
// is built from the lists with shared (or, for very long unions, global)
// atomic ORs.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace sgqa {
namespace {

constexpr int NB0 = 2048;        // bins of the level-0 histogram (top 11 key bits)
constexpr int NBR = 512;         // bins of the refinement histograms (9 bits)
constexpr int WARP_BYTES = 12288;  // per-warp scratch: histogram + candidate lists
constexpr int CAND_CAP = (WARP_BYTES - NBR * 4) / 8;  // 1280 (key, index) pairs
constexpr unsigned FULL = 0xffffffffu;
constexpr int BATCH = 8;         // 32-element groups loaded before use

struct TUArgs {
  const float* scores;  // [Hkv][nq][nblk], rows q_begin .. q_end-1 of the call
  int64_t nq, q_begin, q_end, T, off, nblk;
  int B, Ks, W, Hkv;
  int lgB;              // log2(B): block sizes are powers of two
  int32_t* sel;         // [Hkv][nq][Ks]
  int64_t* uoff;        // [Hkv][lay_ntiles]
  int32_t* ulen;
  int32_t* ublk;
  uint64_t* umask;
  int64_t ucap;         // slots available
  int64_t lay_tau0;     // first tile of the slot layout
  int64_t lay_ntiles;   // tiles in the slot layout
  int64_t capG;         // slots per group in the layout
  int64_t tau_begin;    // first tile of this launch
  int nwords;           // ceil(nblk / 32)
  int nw;               // warps per CTA
  const uint2* cand;    // fused prefill: threshold candidates [Hkv][nq][2][caph] (null: none)
  const int32_t* ccnt;  // their front / back counts per half [Hkv][nq][2][2]
  int caph;
  int32_t* rest;        // rows (g * nq + local row) left for the full-row select
  int32_t* nrest;       // their count
  int32_t* tflag;       // [Hkv][ceil(nq / 128)]: row tile has a row the candidates left
  int32_t* flist;       // flagged row tiles, (g << 20) | rt
  int32_t* nflist;      // their count
  int rb;               // row-select warps take blocks of rb consecutive queries
  int64_t r_end;        // the warp path selects local rows [0, r_end) (longer rows: one CTA each)
  int32_t* status;
};

__device__ __forceinline__ int64_t cap_of_tile(const TUArgs& a, int64_t tau) {
  const int64_t first = tau * a.W;
  int64_t len = a.T - first;
  if (len > a.W) len = a.W;
  int64_t nh = (a.off + first + len - 1) >> a.lgB;
  if (nh > a.nblk) nh = a.nblk;
  const int64_t k = len * a.Ks;
  return k < nh ? k : nh;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Warp-wide: in `hist` (nbins, a multiple of 32), find the bin holding the
// need-th largest element counting from the top bin down.  Returns the bin,
// the count strictly above it and the bin's count.
__device__ void find_bin(const uint32_t* hist, int nbins, uint32_t need, uint32_t& bin,
                         uint32_t& above, uint32_t& cnt) {
  const int lane = lane_id();
  const int per = nbins / 32;
  const int lo = lane * per;
  uint32_t s = 0;
  for (int i = 0; i < per; ++i) s += hist[lo + ((i + lane) & (per - 1))];  // rotated: no bank conflicts
  uint32_t incl = s;  // sum over lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(FULL, incl, o);
    if (lane + o < 32) incl += v;
  }
  const uint32_t excl = incl - s;
  const uint32_t who_m = __ballot_sync(FULL, excl < need && need <= incl);
  const int who = who_m ? __ffs(who_m) - 1 : 0;
  uint32_t b = 0, ab = 0, c = 0;
  if (lane == who) {
    uint32_t acc = excl;
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t h = hist[lo + i];
      if (acc + h >= need) {
        b = lo + i;
        ab = acc;
        c = h;
        break;
      }
      acc += h;
    }
  }
  bin = __shfl_sync(FULL, b, who);
  above = __shfl_sync(FULL, ab, who);
  cnt = __shfl_sync(FULL, c, who);
}

__device__ __forceinline__ void zero_hist(uint32_t* hist, int nbins) {
  for (int i = lane_id() * 4; i < nbins; i += 128)
    *reinterpret_cast<uint4*>(hist + i) = make_uint4(0, 0, 0, 0);
  __syncwarp();
}

// Histogram of (key >> shift) & (nbins-1) over row keys whose key >> pshift == pval
// (no filter when pshift == 32).  Loads 8 float4 per lane before using them.
__device__ __noinline__ void hist_row(const float* __restrict__ row, int64_t nh, bool vec, uint32_t* hist,
                         int shift, int nbins, int pshift, uint32_t pval) {
  const int lane = lane_id();
  const uint32_t bm = nbins - 1;
  auto add = [&](float v) {
    const uint32_t key = order_key(v);
    if (pshift == 32 || (key >> pshift) == pval) atomicAdd(&hist[(key >> shift) & bm], 1u);
  };
  int64_t done = 0;
  if (vec) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int64_t n4 = nh / 4;
    int64_t x = lane;
    for (; x + 7 * 32 < n4; x += 8 * 32) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(r4 + x + u * 32);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        add(v[u].x);
        add(v[u].y);
        add(v[u].z);
        add(v[u].w);
      }
    }
    for (; x < n4; x += 32) {
      const float4 v = __ldg(r4 + x);
      add(v.x);
      add(v.y);
      add(v.z);
      add(v.w);
    }
    done = n4 * 4;
  }
  for (int64_t j = done + lane; j < nh; j += 32) add(__ldg(row + j));
  __syncwarp();
}

__device__ void hist_cand(const uint2* cand, int n, uint32_t* hist, int shift, int nbins,
                          int pshift, uint32_t pval) {
  const uint32_t bm = nbins - 1;
  for (int i = lane_id(); i < n; i += 32) {
    const uint32_t key = cand[i].x;
    if ((key >> pshift) == pval) atomicAdd(&hist[(key >> shift) & bm], 1u);
  }
  __syncwarp();
}

// Visit row elements j = 0 .. nh-1 in ascending order, 32 at a time (lane l
// gets j = base + l), with BATCH groups of loads in flight.  f(j, valid, key)
// is called by all lanes for every group.
template <typename F>
__device__ __forceinline__ void ordered_pass(const float* __restrict__ row, int64_t nh, F f) {
  const int lane = lane_id();
  for (int64_t base = 0; base < nh; base += 32 * BATCH) {
    uint32_t keys[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int64_t j = base + u * 32 + lane;
      keys[u] = j < nh ? order_key(__ldg(row + j)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int64_t j0 = base + u * 32;
      if (j0 >= nh) break;  // warp-uniform
      f(j0, j0 + lane < nh, keys[u]);
    }
  }
}

// General path of a row's selection (any k/B, any row alignment, any bucket
// size), given the level-0 histogram result (bucket b0, `above0` keys above
// it, cnt0 keys in it).  Refines inside the bucket (from shared memory when
// the bucket fits, else by re-reading the row) and emits the list with a
// full ascending pass over the row.
__device__ __noinline__ void select_row_general(const TUArgs& a, const float* __restrict__ row, int64_t nh,
                                   uint32_t need, int32_t* out, bool vec, uint32_t b0,
                                   uint32_t above0, uint32_t cnt0, uint32_t* warp_smem,
                                   int64_t t) {
  const int lane = lane_id();
  // The selection is: every key above the threshold prefix Tp (compared on
  // key >> shift), plus the first `rem` keys equal to it in block order.
  uint32_t Tp = b0, rem = need - above0;
  int shift = 21;
  {
    uint32_t b = b0, above = above0, cnt = cnt0;
    if (cnt != rem) {
      // refine the remaining 21 bits in levels of 9, 9 and 3 bits
      uint2* cand = reinterpret_cast<uint2*>(warp_smem);          // reuses the histogram
      uint32_t* rh = warp_smem + CAND_CAP * 2;                     // refinement histogram
      const bool use_cand = cnt <= (uint32_t)CAND_CAP;
      int n = 0;
      __syncwarp();
      if (use_cand) {  // compact the bucket's members (order does not matter here)
        ordered_pass(row, nh, [&](int64_t j0, bool valid, uint32_t key) {
          const bool in = valid && (key >> 21) == b;
          const uint32_t m = __ballot_sync(FULL, in);
          if (in) cand[n + __popc(m & lanemask_lt())] = make_uint2(key, (uint32_t)(j0 + lane));
          n += __popc(m);
        });
        __syncwarp();
      }
      const int widths[3] = {9, 9, 3};
      for (int lv = 0; lv < 3 && cnt != rem; ++lv) {
        const int w = widths[lv];
        const int nb = 1 << w;
        const int nshift = shift - w;
        zero_hist(rh, nb < 128 ? 128 : nb);
        if (use_cand) hist_cand(cand, n, rh, nshift, nb, shift, Tp);
        else hist_row(row, nh, vec, rh, nshift, nb, shift, Tp);
        if (nb >= 32) {
          find_bin(rh, nb, rem, b, above, cnt);
        } else {  // tiny last level: scan serially on every lane
          uint32_t acc = 0;
          b = 0;
          above = 0;
          cnt = 0;
          for (int i = nb - 1; i >= 0; --i) {
            const uint32_t h = rh[i];
            if (acc + h >= rem) {
              b = i;
              above = acc;
              cnt = h;
              break;
            }
            acc += h;
          }
        }
        rem -= above;
        Tp = (Tp << w) | b;
        shift = nshift;
        __syncwarp();
      }
    }
  }

  // emission in ascending block order
  uint32_t eq_seen = 0, n_out = 0;
  ordered_pass(row, nh, [&](int64_t j0, bool valid, uint32_t key) {
    const uint32_t kp = key >> shift;
    const bool eq = valid && kp == Tp;
    const uint32_t meq = __ballot_sync(FULL, eq);
    const uint32_t rank = eq_seen + __popc(meq & lanemask_lt());
    const bool take = (valid && kp > Tp) || (eq && rank < rem);
    const uint32_t mt = __ballot_sync(FULL, take);
    if (take) out[n_out + __popc(mt & lanemask_lt())] = (int32_t)(j0 + lane);
    n_out += __popc(mt);
    eq_seen += __popc(meq);
  });
  for (int64_t x = n_out + lane; x < a.Ks; x += 32) out[x] = -1;
  if (lane == 0 && n_out != need) report(a.status, SGQA_ERR_BOUNDS, (int)t);
}

// Fast path of a row's selection: k/B <= 512, 16-byte aligned rows, and a
// level-0 bucket of at most 512 keys.  One vectorised pass in block order
// stores the blocks above the bucket (all selected) and the bucket's members
// in shared memory; the bucket is refined there; and the two ascending lists
// are merged into the output without another pass over the row.
constexpr int FAST_MAX = 512;
static_assert(4 * FAST_MAX * 4 <= WARP_BYTES, "fast-path lists must fit a warp's scratch");
static_assert(NBR <= FAST_MAX, "refinement histogram must fit its slot");

__device__ __forceinline__ int lower_bound_smem(const int32_t* v, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __noinline__ void select_row_fast(const TUArgs& a, const float* __restrict__ row, int64_t nh,
                                uint32_t need, int32_t* out, uint32_t b0, uint32_t above0,
                                uint32_t cnt0, uint32_t* warp_smem, int64_t t) {
  const int lane = lane_id();
  uint2* cand = reinterpret_cast<uint2*>(warp_smem);                  // [512] (key, block)
  int32_t* defs = reinterpret_cast<int32_t*>(warp_smem + 2 * FAST_MAX);  // [512] above the bucket
  uint32_t* rh = warp_smem + 3 * FAST_MAX;                             // [512] histogram, then
  int32_t* csel = reinterpret_cast<int32_t*>(rh);                      // selected bucket members
  __syncwarp();  // the level-0 histogram in the same space is no longer read
  const uint32_t lt = lanemask_lt();
  uint32_t n_def = 0, n_c = 0;
  // append the flagged elements of this lane's 4 consecutive blocks j0..j0+3, in order
  auto append = [&](int64_t j0, uint32_t fd, uint32_t fc, const uint32_t (&k)[4]) {
    const uint32_t nd = __popc(fd), nc = __popc(fc);
    uint32_t sd = nd, sc = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t td = __shfl_up_sync(FULL, sd, o), tc = __shfl_up_sync(FULL, sc, o);
      if (lane >= o) {
        sd += td;
        sc += tc;
      }
    }
    uint32_t pd = n_def + sd - nd, pc = n_c + sc - nc;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if ((fd >> e) & 1u) defs[pd++] = (int32_t)(j0 + e);
      if ((fc >> e) & 1u) cand[pc++] = make_uint2(k[e], (uint32_t)(j0 + e));
    }
    n_def += __shfl_sync(FULL, sd, 31);
    n_c += __shfl_sync(FULL, sc, 31);
  };
  const float4* r4 = reinterpret_cast<const float4*>(row);
  const int64_t n4 = nh / 4;
  for (int64_t base = 0; base < n4; base += 32 * BATCH) {
    float4 v[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int64_t x = base + u * 32 + lane;
      v[u] = x < n4 ? __ldg(r4 + x) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int64_t g0 = base + u * 32;
      if (g0 >= n4) break;  // warp-uniform
      const bool valid = g0 + lane < n4;
      const uint32_t k[4] = {order_key(v[u].x), order_key(v[u].y), order_key(v[u].z),
                             order_key(v[u].w)};
      uint32_t fd = 0, fc = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t bn = k[e] >> 21;
        fd |= (uint32_t)(valid && bn > b0) << e;
        fc |= (uint32_t)(valid && bn == b0) << e;
      }
      append(4 * (g0 + lane), fd, fc, k);
    }
  }
  {  // the last nh % 4 blocks, one per lane
    const int64_t j = n4 * 4 + lane;
    const bool valid = j < nh;
    const uint32_t key = valid ? order_key(__ldg(row + j)) : 0u;
    const uint32_t bn = key >> 21;
    const bool d = valid && bn > b0, c = valid && bn == b0;
    const uint32_t md = __ballot_sync(FULL, d), mc = __ballot_sync(FULL, c);
    if (d) defs[n_def + __popc(md & lt)] = (int32_t)j;
    if (c) cand[n_c + __popc(mc & lt)] = make_uint2(key, (uint32_t)j);
    n_def += __popc(md);
    n_c += __popc(mc);
  }
  __syncwarp();
  // refine the threshold inside the bucket: 9, 9 and 3 more key bits
  uint32_t Tp = b0, rem = need - above0, cnt = cnt0;
  int shift = 21;
  const int widths[3] = {9, 9, 3};
  for (int lv = 0; lv < 3 && cnt != rem; ++lv) {
    const int w = widths[lv];
    const int nb = 1 << w;
    const int nshift = shift - w;
    zero_hist(rh, nb < 128 ? 128 : nb);
    hist_cand(cand, (int)n_c, rh, nshift, nb, shift, Tp);
    uint32_t b, above;
    if (nb >= 32) {
      find_bin(rh, nb, rem, b, above, cnt);
    } else {
      uint32_t acc = 0;
      b = 0;
      above = 0;
      cnt = 0;
      for (int i = nb - 1; i >= 0; --i) {
        const uint32_t h = rh[i];
        if (acc + h >= rem) {
          b = i;
          above = acc;
          cnt = h;
          break;
        }
        acc += h;
      }
    }
    rem -= above;
    Tp = (Tp << w) | b;
    shift = nshift;
    __syncwarp();
  }
  // selected bucket members, in block order: above Tp, or equal and among the first `rem`
  uint32_t n_sel = 0, eq_seen = 0;
  for (uint32_t base = 0; base < n_c; base += 32) {
    const uint32_t i = base + lane;
    const bool valid = i < n_c;
    const uint2 cv = valid ? cand[i] : make_uint2(0u, 0u);
    const uint32_t kp = cv.x >> shift;
    const bool eq = valid && kp == Tp;
    const uint32_t meq = __ballot_sync(FULL, eq);
    const uint32_t rank = eq_seen + __popc(meq & lt);
    const bool take = (valid && kp > Tp) || (eq && rank < rem);
    const uint32_t mt = __ballot_sync(FULL, take);
    if (take) csel[n_sel + __popc(mt & lt)] = (int32_t)cv.y;
    n_sel += __popc(mt);
    eq_seen += __popc(meq);
  }
  __syncwarp();
  // merge the two ascending lists (disjoint block sets) into the output
  for (uint32_t i = lane; i < n_def; i += 32) {
    const int32_t v = defs[i];
    out[i + lower_bound_smem(csel, (int)n_sel, v)] = v;
  }
  for (uint32_t i = lane; i < n_sel; i += 32) {
    const int32_t v = csel[i];
    out[i + lower_bound_smem(defs, (int)n_def, v)] = v;
  }
  for (int x = (int)need + lane; x < a.Ks; x += 32) out[x] = -1;
  if (lane == 0 && n_def + n_sel != need) report(a.status, SGQA_ERR_BOUNDS, (int)t);
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Candidate path, for rows of 2048 .. 16384 blocks (16-byte aligned) that
// select at most CAND_NEED_MAX blocks.  A float threshold tf is chosen so that
// a little more than k/B of the row's scores clear it; one pass over the row
// compacts every score >= tf into shared memory in block order, and the exact
// k-th key and the emission are resolved on those candidates, so the row is
// read once.  {x >= tf} is an upper set of the key order (the key order only
// splits -0 below +0), so whenever it holds at least k/B blocks it holds the
// whole selection, ties included; the pass checks that and that the list did
// not overflow, and otherwise the row takes the histogram path.  The choice
// of tf only affects speed:
//  * predicted: from the previous row of the same warp (consecutive queries of
//    one group), tf = that row's k-th key minus a margin that a per-warp
//    controller keeps at about 1.3 k/B candidates;
//  * sampled: 8 adjacent blocks (one 32-byte sector) of every 64 are read and
//    a radix select on them picks the key ranked at the expected
//    count of the selection in the sample plus three standard deviations.
constexpr int CAND_NEED_MAX = 768;
constexpr int CAND_MAX = 1024;
constexpr int CAND_OFF = 1024;      // words: candidates / samples start 4 KB into the scratch
                                    // (the first 4 KB: pass staging, then select histogram)
constexpr int SAMP_MAX = 2048;
static_assert(CAND_OFF * 4 + CAND_MAX * 8 <= WARP_BYTES, "candidate path scratch");
static_assert(CAND_OFF * 4 + SAMP_MAX * 4 <= WARP_BYTES, "sample scratch");

struct Pred {         // per-warp threshold predictor
  float kappa;        // previous row's k-th key (as a float, rounded down)
  float margin;       // tf = kappa - margin
  bool valid;
};

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Radix select on n keys keys[i * stride] in shared memory (1 <= need <= n),
// with 8-bit digits from the highest bit at which the keys differ, for at most
// max_levels digits.  On return the need-th largest key has key >> sh == T;
// keys with a larger prefix rank above it, and `rem` of the `cnt` keys with
// prefix T complete the top `need` (cnt == rem once the digits resolve it).
struct Sel {
  uint32_t T, rem, cnt, kmin;
  int sh;
};
// kmin / kmax: this lane's minimum and maximum of the keys (any split of the
// keys over the lanes).
__device__ Sel radix_select_mm(const uint32_t* keys, int stride, uint32_t n, uint32_t need,
                               uint32_t* hist, int max_levels, uint32_t kmin, uint32_t kmax) {
  const int lane = lane_id();
  kmin = __reduce_min_sync(FULL, kmin);
  kmax = __reduce_max_sync(FULL, kmax);
  Sel s;
  s.rem = need;
  s.cnt = n;
  s.kmin = kmin;
  if (kmin == kmax) {
    s.T = kmin;
    s.sh = 0;
    return s;
  }
  const int hb = 31 - __clz(kmin ^ kmax);  // keys agree above bit hb
  s.sh = hb + 1;
  s.T = hb == 31 ? 0u : (kmax >> (hb + 1));
  for (int lv = 0; lv < max_levels && s.cnt != s.rem && s.sh > 0; ++lv) {
    const int w = s.sh < 8 ? s.sh : 8;
    const int nsh = s.sh - w;
    *reinterpret_cast<uint4*>(hist + lane * 8) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(hist + lane * 8 + 4) = make_uint4(0, 0, 0, 0);
    __syncwarp();
    for (uint32_t i = lane; i < n; i += 32) {
      const uint32_t k = keys[i * stride];
      if (s.sh >= 32 || (k >> s.sh) == s.T) atomicAdd(&hist[(k >> nsh) & ((1u << w) - 1u)], 1u);
    }
    __syncwarp();
    uint32_t b, above;
    find_bin(hist, 256, s.rem, b, above, s.cnt);
    s.rem -= above;
    s.T = (s.sh >= 32 ? 0u : (s.T << w)) | b;
    s.sh = nsh;
    __syncwarp();
  }
  return s;
}

__device__ Sel warp_radix_select(const uint32_t* keys, int stride, uint32_t n, uint32_t need,
                                 uint32_t* hist, int max_levels) {
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (uint32_t i = lane_id(); i < n; i += 32) {
    const uint32_t k = keys[i * stride];
    kmin = min(kmin, k);
    kmax = max(kmax, k);
  }
  return radix_select_mm(keys, stride, n, need, hist, max_levels, kmin, kmax);
}

// Threshold key from ns >= 1 sample keys in shared memory: the key ranked at
// the expected count of the selection in the sample plus nsd standard
// deviations, rounded down to the prefix the radix select resolved.
__device__ uint32_t sample_rank_key(const uint32_t* samp, int ns, int64_t nh, uint32_t need,
                                    uint32_t* hist, float nsd, uint32_t kmin, uint32_t kmax) {
  const float e = (float)need * (float)ns / (float)nh;
  uint32_t r = (uint32_t)ceilf(e + nsd * sqrtf(e));
  if (r > (uint32_t)ns) r = ns;
  if (r < 1) r = 1;
  const Sel sl = radix_select_mm(samp, 1, ns, r, hist, 2, kmin, kmax);
  return sl.sh >= 32 ? sl.kmin : (sl.T << sl.sh);
}

// Sampled threshold (as a key): 8 adjacent blocks of every 64 (two lanes per
// group) read from the row itself.
__device__ __noinline__ uint32_t sample_tau(const float* __restrict__ row, int64_t nh, uint32_t need,
                               uint32_t* hist, uint32_t* samp) {
  const int lane = lane_id();
  const float4* r4 = reinterpret_cast<const float4*>(row);
  const int nsg = (int)(nh / 64);
  const int ns = nsg * 8;
  for (int base = 0; base < nsg; base += 64) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = base + u * 16 + (lane >> 1);
      v[u] = q < nsg ? __ldg(r4 + q * 16 + (lane & 1)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = base + u * 16 + (lane >> 1);
      if (q < nsg)
        *reinterpret_cast<uint4*>(samp + q * 8 + (lane & 1) * 4) =
            make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z),
                       order_key(v[u].w));
    }
  }
  __syncwarp();
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int i = lane; i < ns; i += 32) {
    kmin = min(kmin, samp[i]);
    kmax = max(kmax, samp[i]);
  }
  return sample_rank_key(samp, ns, nh, need, hist, 3.f, kmin, kmax);
}

// Compact every block with score >= tf into cand (key, block), in block order.
// Returns the count (stops early once it exceeds CAND_MAX).  A batch gives
// each lane 32 consecutive blocks (8 float4), so a lane's candidates are
// contiguous in block order and one warp prefix sum per batch places them.
// The batch is staged in shared memory (rows swizzled by lane, so the 16-byte
// stores of 8 lanes hit distinct banks), and the warp then writes the
// batch's candidates 32 at a time, lane i taking the i-th: its source lane
// comes from a binary search over the prefix sums and its block from the
// source lane's flag word.  Loads run one batch ahead of their use.
__device__ uint32_t cand_pass(const float* __restrict__ row, int64_t nh, float tf, uint2* cand,
                              float* stage) {
  const int lane = lane_id();
  const uint32_t lt = lanemask_lt();
  const float4* r4 = reinterpret_cast<const float4*>(row);
  const int64_t n4 = nh / 4;
  const int64_t nbat = (n4 + 32 * BATCH - 1) / (32 * BATCH);
  const float qnan = __int_as_float(0x7fffffff);  // never >= tf
  uint32_t C = 0;
  auto load = [&](float4 (&v)[BATCH], int64_t bi) {
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int64_t x = bi * (32 * BATCH) + lane * BATCH + u;
      v[u] = x < n4 ? __ldg(r4 + x) : make_float4(qnan, qnan, qnan, qnan);
    }
  };
  auto proc = [&](const float4 (&v)[BATCH], int64_t bi) {
    uint32_t fl = 0;
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      fl |= (uint32_t)(v[u].x >= tf) << (4 * u);
      fl |= (uint32_t)(v[u].y >= tf) << (4 * u + 1);
      fl |= (uint32_t)(v[u].z >= tf) << (4 * u + 2);
      fl |= (uint32_t)(v[u].w >= tf) << (4 * u + 3);
    }
    if (!__any_sync(FULL, fl != 0u)) return;
    const uint32_t c = __popc(fl);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t tot = __shfl_sync(FULL, incl, 31);
#pragma unroll
    for (int u = 0; u < BATCH; ++u)
      *reinterpret_cast<float4*>(stage + lane * 32 + ((u ^ (lane & 7)) << 2)) = v[u];
    __syncwarp();
    const uint32_t jb = (uint32_t)(4 * bi * (32 * BATCH));
    for (uint32_t r0 = 0; r0 < tot; r0 += 32) {
      const uint32_t i = r0 + lane;  // the batch's i-th candidate
      int src = 0;                   // first lane whose inclusive count exceeds i
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint32_t pv = __shfl_sync(FULL, incl, src + o - 1);
        if (pv <= i) src += o;
      }
      const uint32_t ex = __shfl_sync(FULL, incl, src) - __shfl_sync(FULL, c, src);
      const uint32_t fs = __shfl_sync(FULL, fl, src);
      if (i < tot) {
        const uint32_t k = __fns(fs, 0, (int)(i - ex) + 1);  // bit of the (i-ex)-th set flag
        const float x = stage[src * 32 + (((k >> 2) ^ (src & 7)) << 2) + (k & 3)];
        if (C + i < (uint32_t)CAND_MAX)
          cand[C + i] = make_uint2(order_key(x), jb + (uint32_t)src * 32 + k);
      }
    }
    __syncwarp();
    C += tot;
  };
  // one copy of the batch body (a compact loop keeps the instruction cache warm)
  float4 cur[BATCH], nxt[BATCH];
  if (nbat > 0) load(cur, 0);
#pragma unroll 1
  for (int64_t bi = 0; bi < nbat && C <= (uint32_t)CAND_MAX; ++bi) {
    if (bi + 1 < nbat) load(nxt, bi + 1);
    proc(cur, bi);
#pragma unroll
    for (int u = 0; u < BATCH; ++u) cur[u] = nxt[u];
  }
  {  // the last nh % 4 blocks
    const int64_t j = n4 * 4 + lane;
    const float x = j < nh ? __ldg(row + j) : qnan;
    const bool f = x >= tf;
    const uint32_t m = __ballot_sync(FULL, f);
    const uint32_t pos = C + __popc(m & lt);
    if (f && pos < (uint32_t)CAND_MAX) cand[pos] = make_uint2(order_key(x), (uint32_t)j);
    C += __popc(m);
  }
  __syncwarp();
  return C;
}

// Exact selection among C candidates (need <= C <= CAND_MAX, block order):
// writes the list and returns the k-th key rounded down to its resolved prefix.
__device__ __noinline__ uint32_t cand_select(const TUArgs& a, const uint2* cand, uint32_t C, uint32_t need,
                                int32_t* out, uint32_t* hist, int64_t t) {
  const int lane = lane_id();
  const uint32_t lt = lanemask_lt();
  const Sel sl = warp_radix_select(reinterpret_cast<const uint32_t*>(cand), 2, C, need, hist, 4);
  // emission in block order: above the k-th key's prefix, or equal to it and
  // among the first `rem` such (all of them when cnt == rem)
  uint32_t n_out = 0, eq_seen = 0;
  const bool ties = sl.cnt != sl.rem;
  for (uint32_t base = 0; base < C; base += 32) {
    const uint32_t i = base + lane;
    const bool valid = i < C;
    const uint2 c = valid ? cand[i] : make_uint2(0u, 0u);
    const uint32_t kp = sl.sh >= 32 ? 0u : (c.x >> sl.sh);
    bool take;
    if (!ties) {
      take = valid && kp >= sl.T;
    } else {
      const bool eq = valid && kp == sl.T;
      const uint32_t meq = __ballot_sync(FULL, eq);
      take = (valid && kp > sl.T) || (eq && eq_seen + __popc(meq & lt) < sl.rem);
      eq_seen += __popc(meq);
    }
    const uint32_t mt = __ballot_sync(FULL, take);
    if (take) out[n_out + __popc(mt & lt)] = (int32_t)c.y;
    n_out += __popc(mt);
  }
  for (int64_t x = need + lane; x < a.Ks; x += 32) out[x] = -1;
  if (lane == 0 && n_out != need) report(a.status, SGQA_ERR_BOUNDS, (int)t);
  return sl.sh >= 32 ? sl.kmin : (sl.T << sl.sh);
}

// Select row t of group g and write its ascending list.  All lanes participate.
__device__ void select_row(const TUArgs& a, int g, int64_t t, uint32_t* warp_smem, Pred& pr) {
  const int lane = lane_id();
  const int64_t tl = t - a.q_begin;
  int64_t nh = (a.off + t) >> a.lgB;
  if (nh > a.nblk) nh = a.nblk;
  const uint32_t need = (uint32_t)(nh < a.Ks ? nh : a.Ks);
  const float* row = a.scores + ((int64_t)g * a.nq + tl) * a.nblk;
  int32_t* out = a.sel + ((int64_t)g * a.nq + tl) * a.Ks;
  const bool vec = (a.nblk & 3) == 0;
  if ((int64_t)need == nh) {  // every historical block (or none): no scores to read
    for (int64_t x = lane; x < a.Ks; x += 32) out[x] = x < nh ? (int32_t)x : -1;
    pr.valid = false;
    return;
  }
  if (vec && nh >= 2048 && nh <= 16384 && need <= (uint32_t)CAND_NEED_MAX) {
    uint32_t* hist = warp_smem;
    uint2* cand = reinterpret_cast<uint2*>(warp_smem + CAND_OFF);
    for (int attempt = 0; attempt < 2; ++attempt) {
      const bool predicted = attempt == 0 && pr.valid;
      if (attempt == 0 && !pr.valid) continue;
      float tf;
      if (predicted) {
        tf = pr.kappa - pr.margin;
      } else {
        tf = key_to_float(sample_tau(row, nh, need, hist, warp_smem + CAND_OFF));
      }
      const uint32_t C = cand_pass(row, nh, tf, cand, reinterpret_cast<float*>(warp_smem));
      if (C >= need && C <= (uint32_t)CAND_MAX) {
        const float kappa = key_to_float(cand_select(a, cand, C, need, out, hist, t));
        // keep about 1.3 k/B candidates for the next row
        float margin = predicted ? pr.margin : kappa - tf;
        if (!(margin > 0.f)) margin = fabsf(kappa) * 1e-3f + 1e-30f;
        const float ratio = (float)C / (float)need;
        if (ratio < 1.1f) margin *= 1.5f;
        else if (ratio > 1.6f) margin *= 0.7f;
        pr.kappa = kappa;
        pr.margin = margin;
        pr.valid = isfinite(kappa) && isfinite(margin);
        return;
      }
      if (predicted) pr.margin *= (C < need) ? 2.f : 0.5f;
    }
    pr.valid = false;
  }
  // histogram path: level 0, the top 11 key bits
  uint32_t b0, above0, cnt0;
  zero_hist(warp_smem, NB0);
  hist_row(row, nh, vec, warp_smem, 21, NB0, 32, 0);
  find_bin(warp_smem, NB0, need, b0, above0, cnt0);
  if (vec && need <= (uint32_t)FAST_MAX && cnt0 <= (uint32_t)FAST_MAX)
    select_row_fast(a, row, nh, need, out, b0, above0, cnt0, warp_smem, t);
  else
    select_row_general(a, row, nh, need, out, vec, b0, above0, cnt0, warp_smem, t);
}

// Slot base of tile tau of group g: g * capG + the caps of the layout's
// earlier tiles.  Every thread calls it; uses `red` (32 words) and one barrier.
__device__ int64_t tile_slot_base(const TUArgs& a, int g, int64_t tau, int64_t* red) {
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  const int nthr = blockDim.x;
  int64_t part = 0;
  for (int64_t x = a.lay_tau0 + tid; x < tau; x += nthr) part += cap_of_tile(a, x);
  for (int o = 16; o > 0; o >>= 1) part += __shfl_down_sync(FULL, part, o);
  if (lane == 0) red[warp] = part;
  __syncthreads();
  int64_t s = 0;
  for (int w = 0; w < (nthr >> 5); ++w) s += red[w];
  return (int64_t)g * a.capG + s;
}

// After every row of the tile has OR-ed its blocks into tile_bits: write the
// union list (ascending) and, per union slot, the mask of the tile's queries
// that selected it.  `mspace` (mask_pairs lo/hi word pairs) is shared scratch
// for the masks; longer unions use global atomics.  Starts with a barrier.
__device__ void finish_tile(const TUArgs& a, int g, int64_t tau, int64_t base, int len,
                            uint32_t* tile_bits, uint32_t* wprefix, uint32_t* mspace,
                            int64_t mask_pairs) {
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  const int nthr = blockDim.x, nw = nthr >> 5;
  __syncthreads();
  // ranks from a prefix sum of word popcounts
  if (warp == 0) {
    uint32_t carry = 0;
    for (int b0 = 0; b0 < a.nwords; b0 += 32) {
      const int w = b0 + lane;
      const uint32_t c = w < a.nwords ? __popc(tile_bits[w]) : 0u;
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += v;
      }
      if (w < a.nwords) wprefix[w] = carry + incl - c;
      carry += __shfl_sync(FULL, incl, 31);
    }
    if (lane == 0) wprefix[a.nwords] = carry;
  }
  __syncthreads();
  const int64_t U = wprefix[a.nwords];
  const int64_t cap = cap_of_tile(a, tau);
  const int64_t lt = (int64_t)g * a.lay_ntiles + (tau - a.lay_tau0);
  if (U > cap || base + U > a.ucap) {
    if (tid == 0) {
      report(a.status, SGQA_ERR_CAPACITY, (int)tau);
      a.uoff[lt] = base;
      a.ulen[lt] = 0;
    }
    return;
  }
  for (int w = tid; w < a.nwords; w += nthr) {
    uint32_t bits = tile_bits[w];
    uint32_t r = wprefix[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      a.ublk[base + r++] = w * 32 + b;
      bits &= bits - 1;
    }
  }
  // member masks
  const bool in_smem = U <= mask_pairs;
  uint32_t* mlo = mspace;
  uint32_t* mhi = mlo + (in_smem ? U : 0);
  if (in_smem) {
    for (int64_t s = tid; s < 2 * U; s += nthr) mlo[s] = 0;
  } else {
    for (int64_t s = tid; s < U; s += nthr) a.umask[base + s] = 0;
  }
  __syncthreads();
  const int64_t first = tau * a.W;
  for (int i = warp; i < len; i += nw) {
    const int64_t t = first + i;
    int64_t nh = (a.off + t) >> a.lgB;
    if (nh > a.nblk) nh = a.nblk;
    const int64_t need = nh < a.Ks ? nh : a.Ks;
    const int32_t* lst = a.sel + ((int64_t)g * a.nq + (t - a.q_begin)) * a.Ks;
    for (int64_t xb = 0; xb < need; xb += 32 * 8) {  // 8 coalesced loads in flight per lane
      int32_t jj[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t x = xb + u * 32 + lane;
        jj[u] = x < need ? lst[x] : -1;
      }
      // every slot first, then the updates (an update between two slot reads
      // would hold the second back)
      uint32_t sl[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int32_t j = jj[u] < 0 ? 0 : jj[u];
        const int w = j >> 5;
        sl[u] = wprefix[w] + __popc(tile_bits[w] & ((1u << (j & 31)) - 1u));
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (jj[u] < 0) continue;
        const int64_t slot = sl[u];
        if (in_smem) {
          atomicOr(i < 32 ? &mlo[slot] : &mhi[slot], 1u << (i & 31));
        } else {
          atomicOr(reinterpret_cast<unsigned long long*>(&a.umask[base + slot]), 1ull << i);
        }
      }
    }
  }
  __syncthreads();
  if (in_smem)
    for (int64_t s = tid; s < U; s += nthr)
      a.umask[base + s] = (static_cast<uint64_t>(mhi[s]) << 32) | mlo[s];
  if (tid == 0) {
    a.uoff[lt] = base;
    a.ulen[lt] = (int32_t)U;
  }
}

// Row kernel: the rows of every group are cut into blocks of rb consecutive
// queries (8 where the one-pass candidate path applies, else 1); warp w of
// the grid takes blocks w, w + (warps in the grid), ... (persistent CTAs, so
// all SMs stay busy however many tiles there are), and carries its threshold
// predictor from row to row within a block.
constexpr int ROW_BLOCK = 8;  // when the previous-row threshold can serve (else 1)

// Bulk prefetch into L2 of the scores of local row r of group g (the blocks
// the select reads, rounded up to 16 bytes; rows start 16-byte aligned when
// nblk % 4 == 0, otherwise nothing is prefetched).
__device__ __forceinline__ void prefetch_row_l2(const TUArgs& a, int g, int64_t r) {
  if (a.nblk & 3) return;
  int64_t nh = (a.off + a.q_begin + r) >> a.lgB;
  if (nh > a.nblk) nh = a.nblk;
  if (nh <= a.Ks) return;  // rows that take every block read no scores
  const uint32_t bytes = (uint32_t)(((nh + 3) & ~int64_t(3)) * 4);
  const float* p = a.scores + ((int64_t)g * a.nq + r) * a.nblk;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
constexpr int ROW_WARPS = 4;  // per CTA: 4 x 12 KB of scratch, four CTAs per SM

__global__ void __launch_bounds__(ROW_WARPS * 32, 4) k_topk_rows(TUArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = warp_id();
  uint32_t* wsm = reinterpret_cast<uint32_t*>(smem + (size_t)warp * WARP_BYTES);
  const int64_t nwt = (int64_t)gridDim.x * ROW_WARPS;
  if (a.rest != nullptr) {  // the rows the candidate select left, one at a time
    const int64_t nr = *a.nrest;
    for (int64_t i = (int64_t)blockIdx.x * ROW_WARPS + warp; i < nr; i += nwt) {
      const int64_t rr = a.rest[i];
      const int g = (int)(rr / a.nq);
      const int64_t lr = rr % a.nq;
      Pred pr;
      pr.valid = false;
      if (lane_id() == 0) prefetch_row_l2(a, g, lr);
      select_row(a, g, a.q_begin + lr, wsm, pr);
    }
    return;
  }
  const int64_t bpg = (a.r_end + a.rb - 1) / a.rb;  // row blocks per group
  for (int64_t b = (int64_t)blockIdx.x * ROW_WARPS + warp; b < bpg * a.Hkv; b += nwt) {
    const int g = (int)(b / bpg);
    const int64_t r0 = (b % bpg) * a.rb;
    const int64_t r1 = r0 + a.rb < a.r_end ? r0 + a.rb : a.r_end;
    Pred pr;
    pr.valid = false;
    if (lane_id() == 0) prefetch_row_l2(a, g, r0);
    for (int64_t r = r0; r < r1; ++r) {
      // the next row streams into L2 while this one is selected
      if (lane_id() == 0 && r + 1 < r1) prefetch_row_l2(a, g, r + 1);
      select_row(a, g, a.q_begin + r, wsm, pr);
    }
  }
}

// Tile kernel: one CTA per (tile, group) ORs the tile's lists into its block
// bitmask and writes the union and the member masks.
constexpr int UNION_THREADS = 256;

__global__ void __launch_bounds__(UNION_THREADS) k_tile_union(TUArgs a, int64_t mask_pairs) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int g = blockIdx.y;
  const int64_t tau = a.tau_begin + blockIdx.x;
  const int tid = threadIdx.x, warp = warp_id(), lane = lane_id();
  constexpr int nw = UNION_THREADS / 32;
  uint32_t* tile_bits = reinterpret_cast<uint32_t*>(smem);
  uint32_t* wprefix = tile_bits + ((a.nwords + 3) & ~3);          // nwords + 1 entries
  uint32_t* mspace = wprefix + ((a.nwords + 1 + 3) & ~3);         // mask_pairs lo/hi pairs
  __shared__ int64_t s_red[32];

  for (int i = tid; i < a.nwords; i += UNION_THREADS) tile_bits[i] = 0;
  const int64_t base = tile_slot_base(a, g, tau, s_red);  // ends with a barrier
  const int64_t first = tau * a.W;
  const int len = (int)((a.T - first) < a.W ? (a.T - first) : a.W);
  for (int i = warp; i < len; i += nw) {
    const int64_t t = first + i;
    int64_t nh = (a.off + t) >> a.lgB;
    if (nh > a.nblk) nh = a.nblk;
    const int need = (int)(nh < a.Ks ? nh : a.Ks);
    const int32_t* lst = a.sel + ((int64_t)g * a.nq + (t - a.q_begin)) * a.Ks;
    // each lane ORs a contiguous piece of the ascending list, one atomic per
    // word run; the piece's entries are loaded 16 at a time ahead of the
    // updates (an update between two loads would hold the second back)
    const int per = (need + 31) / 32;
    const int xa = lane * per, x1 = min(need, xa + per);
    uint32_t word = 0xffffffffu, bits = 0;
    for (int x0 = xa; x0 < x1; x0 += 16) {
      int32_t jj[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) jj[u] = x0 + u < x1 ? lst[x0 + u] : -1;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int32_t j = jj[u];
        if (j < 0) continue;
        if ((uint32_t)(j >> 5) != word) {
          if (bits) atomicOr(&tile_bits[word], bits);
          word = (uint32_t)(j >> 5);
          bits = 0;
        }
        bits |= 1u << (j & 31);
      }
    }
    if (bits) atomicOr(&tile_bits[word], bits);
  }
  finish_tile(a, g, tau, base, len, tile_bits, wprefix, mspace, mask_pairs);
}

}  // namespace

namespace {

// Candidate thresholds: one warp per row loads the row's sampled scores as
// keys into shared memory and ranks them (sample_rank_key).
constexpr int TAU_WARPS = 8;
constexpr float TAU_NSD = 5.f;
// five standard deviations: about 1.6 k/B candidates, and on the clustered
// 128K workload no row with fewer than k/B or more than 2.5 k/B of them
constexpr int TAU_SAMP = 2048;  // (kFiltMaxNh / 64) * 8 samples at most
constexpr int TAU_WARP_BYTES = 1024 + TAU_SAMP * 4;
static_assert((kFiltMaxNh >> 6) << 3 <= TAU_SAMP, "sample buffer");

__global__ void __launch_bounds__(TAU_WARPS * 32) k_row_tau(const float* __restrict__ ssc,
                                                            float* __restrict__ tau, int64_t nq,
                                                            int64_t q_begin, int64_t off,
                                                            int64_t nblk, int64_t ns_max, int lgB,
                                                            int Ks, int Hkv) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = warp_id(), lane = lane_id();
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + (size_t)warp * TAU_WARP_BYTES);
  uint32_t* samp = hist + 256;
  const int64_t rg = (int64_t)blockIdx.x * TAU_WARPS + warp;  // g * nq + local row
  if (rg >= nq * Hkv) return;
  const int64_t t = q_begin + rg % nq;
  int64_t nh = (off + t) >> lgB;
  if (nh > nblk) nh = nblk;
  const int64_t need = nh < Ks ? nh : Ks;
  float out = __int_as_float(0x7fffffff);
  if (filter_row(nh, need)) {
    const int ns = (int)((nh >> 6) << 3);
    const float4* r4 = reinterpret_cast<const float4*>(ssc + rg * ns_max);
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int i0 = 0; i0 < ns / 4; i0 += 128) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * 32 + lane;
        v[u] = i < ns / 4 ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * 32 + lane;
        if (i < ns / 4) {
          const uint4 k4 = make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z),
                                      order_key(v[u].w));
          *reinterpret_cast<uint4*>(samp + 4 * i) = k4;
          kmin = min(kmin, min(min(k4.x, k4.y), min(k4.z, k4.w)));
          kmax = max(kmax, max(max(k4.x, k4.y), max(k4.z, k4.w)));
        }
      }
    }
    __syncwarp();
    out = key_to_float(sample_rank_key(samp, ns, nh, (uint32_t)need, hist, TAU_NSD, kmin, kmax));
  }
  if (lane == 0) tau[rg] = out;
}

// Selection from the indexer's threshold candidates (fused prefill): one warp
// per row, rows dealt out round-robin.  The row's four candidate parts (front
// and back of each half-row list) are gathered into shared memory as keys and
// 16-bit block indices; a radix select finds the k-th key; the taken blocks
// (above it, and of those equal to it the lowest-indexed ones) are marked in a
// bitmap over the row's blocks; a prefix sum of the bitmap's word popcounts
// then gives each taken block its place in the ascending list.  While a row is
// selected, the next row's counts are loaded and its parts prefetched into L2.
// A row whose candidates cannot decide it (a half-row list overflowed, fewer
// than `need` or more than CR_CMAX of them), or that has too few or too many
// blocks for the candidate scheme, is appended to the rest list for the
// full-row select.
constexpr int CR_WARPS = 8;
constexpr int CR_CMAX = 1280;  // candidates a row can select from
// per-warp scratch (32-bit words): radix histogram, taken bitmap A and tie
// bitmap E (padded, one spare word per 32 so that a lane's 16 consecutive
// words sit in distinct banks), keys, then 16-bit block indices
constexpr int CR_HIST = 0, CR_A = 256, CR_E = CR_A + 528, CR_KEYS = CR_E + 528;
constexpr int CR_IDX = CR_KEYS + CR_CMAX;
constexpr int CR_WORDS = CR_IDX + CR_CMAX / 2;
static_assert(kFiltMaxNh / 32 <= 512, "bitmap words");

__device__ __forceinline__ int padw(int w) { return w + (w >> 5); }

// Lanes 0-3: L2 prefetch of part `lane` of row rn's candidate lists (16-byte
// rounded; the lists are 16-byte aligned and caph is even).
__device__ __forceinline__ void prefetch_cands(const TUArgs& a, int64_t rn, int32_t cnt) {
  const int lane = lane_id();
  if (lane >= 4 || cnt <= 0 || cnt > a.caph) return;
  const int start = (lane & 1) ? a.caph - cnt : 0;
  const int s0 = start & ~1, s1 = (start + cnt + 1) & ~1;
  const uint2* p = a.cand + (rn * 2 + (lane >> 1)) * a.caph + s0;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"((uint32_t)(s1 - s0) * 8u)
               : "memory");
}

__device__ __noinline__ bool cand_row(const TUArgs& a, int64_t r, int64_t nh, uint32_t need,
                                      int32_t cv, int64_t rn, int32_t cv_next, uint32_t* wsm,
                                      int32_t* out, int64_t t) {
  const int lane = lane_id();
  const int f0 = __shfl_sync(FULL, cv, 0), b0 = __shfl_sync(FULL, cv, 1);
  const int f1 = __shfl_sync(FULL, cv, 2), b1 = __shfl_sync(FULL, cv, 3);
  const int C = f0 + b0 + f1 + b1;
  if (min(min(f0, b0), min(f1, b1)) < 0 || f0 + b0 > a.caph || f1 + b1 > a.caph ||
      C < (int)need || C > CR_CMAX) {
    prefetch_cands(a, rn, cv_next);
    return false;
  }
  uint32_t* keys = wsm + CR_KEYS;
  uint16_t* idx = reinterpret_cast<uint16_t*>(wsm + CR_IDX);
  const uint2* l0 = a.cand + r * 2 * a.caph;
  // gather position i of part p reads list entry i + off_p (entries counted
  // from the row's half-0 list; half 1 follows it)
  const int e0 = f0, e1 = f0 + b0, e2 = e1 + f1;  // ends of the parts in gather order
  const int o1 = a.caph - b0 - e0, o2 = a.caph - e1, o3 = 2 * a.caph - b1 - e2;
  bool bad = false;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int base = 0; base < C; base += 512) {
    uint2 v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = base + u * 32 + lane;
      const int off = i < e0 ? 0 : i < e1 ? o1 : i < e2 ? o2 : o3;
      v[u] = i < C ? __ldg(l0 + (i + off)) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = base + u * 32 + lane;
      if (i < C) {
        bad |= v[u].y >= (uint32_t)nh;
        const uint32_t k = order_key(__uint_as_float(v[u].x));
        kmin = min(kmin, k);
        kmax = max(kmax, k);
        keys[i] = k;
        idx[i] = (uint16_t)v[u].y;
      }
    }
  }
  prefetch_cands(a, rn, cv_next);
  if (__any_sync(FULL, bad)) {  // not a list this indexer wrote
    if (lane == 0) report(a.status, SGQA_ERR_BOUNDS, (int)t);
    return false;
  }
  uint32_t* A = wsm + CR_A;
  uint32_t* E = wsm + CR_E;
  for (int w = lane; w < 528; w += 32) A[w] = 0u;
  __syncwarp();
  const Sel sl = radix_select_mm(keys, 1, (uint32_t)C, need, wsm + CR_HIST, 4, kmin, kmax);
  const bool ties = sl.cnt != sl.rem;
  if (ties)
    for (int w = lane; w < 528; w += 32) E[w] = 0u;
  __syncwarp();
  for (int i = lane; i < C; i += 32) {
    const uint32_t kp = sl.sh >= 32 ? 0u : (keys[i] >> sl.sh);
    const uint32_t j = idx[i];
    if (kp > sl.T || (kp == sl.T && !ties)) atomicOr(&A[padw(j >> 5)], 1u << (j & 31));
    else if (kp == sl.T) atomicOr(&E[padw(j >> 5)], 1u << (j & 31));
  }
  __syncwarp();
  if (ties) {  // the first sl.rem tied blocks in ascending order join A
    int left = (int)sl.rem;
    for (int w0 = 0; w0 < 512 && left > 0; w0 += 32) {
      const int w = padw(w0 + lane);
      const uint32_t e = E[w];
      const int n = __popc(e);
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
      }
      const int take = max(0, min(n, left - (incl - n)));
      if (take == n) {
        if (n) A[w] |= e;
      } else if (take > 0) {
        A[w] |= e & ((2u << __fns(e, 0, take)) - 1u);  // its lowest `take` set bits
      }
      left -= __shfl_sync(FULL, incl, 31);
    }
    __syncwarp();
  }
  // exclusive prefix of the word popcounts (lane: words 16 lane .. 16 lane + 15) into E
  uint32_t* P = E;
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) sum += __popc(A[padw(16 * lane + i)]);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  const int total = __shfl_sync(FULL, incl, 31);
  int run = incl - sum;
  __syncwarp();  // the tie pass's reads of E are done
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int w = padw(16 * lane + i);
    P[w] = (uint32_t)run;
    run += __popc(A[w]);
  }
  __syncwarp();
  for (int i = lane; i < C; i += 32) {
    const uint32_t j = idx[i];
    const int w = padw(j >> 5);
    const uint32_t m = A[w], bit = 1u << (j & 31);
    if (m & bit) {
      const uint32_t pos = P[w] + __popc(m & (bit - 1u));
      if (pos < need) out[pos] = (int32_t)j;
    }
  }
  for (int64_t x = need + lane; x < a.Ks; x += 32) out[x] = -1;
  if (lane == 0 && total != (int)need) report(a.status, SGQA_ERR_BOUNDS, (int)t);
  __syncwarp();
  return true;
}

__global__ void __launch_bounds__(CR_WARPS * 32, 2) k_cand_rows(TUArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = warp_id(), lane = lane_id();
  uint32_t* wsm = reinterpret_cast<uint32_t*>(smem) + warp * CR_WORDS;
  const int64_t W = (int64_t)gridDim.x * CR_WARPS;
  const int64_t nrows = a.nq * a.Hkv;
  int64_t r = (int64_t)blockIdx.x * CR_WARPS + warp;
  int32_t cv = (r < nrows && lane < 4) ? a.ccnt[r * 4 + lane] : 0;
  for (; r < nrows; r += W) {
    const int64_t rn = r + W;
    const int32_t cv_next = (rn < nrows && lane < 4) ? a.ccnt[rn * 4 + lane] : 0;
    const int64_t t = a.q_begin + r % a.nq;
    int64_t nh = (a.off + t) >> a.lgB;
    if (nh > a.nblk) nh = a.nblk;
    const uint32_t need = (uint32_t)(nh < a.Ks ? nh : a.Ks);
    int32_t* out = a.sel + r * a.Ks;
    bool done;
    if ((int64_t)need == nh) {  // every historical block (or none)
      for (int64_t x = lane; x < a.Ks; x += 32) out[x] = x < nh ? (int32_t)x : -1;
      prefetch_cands(a, rn, cv_next);
      done = true;
    } else if (filter_row(nh, need)) {
      done = cand_row(a, r, nh, need, cv, rn, cv_next, wsm, out, t);
    } else {
      prefetch_cands(a, rn, cv_next);
      done = false;
    }
    if (!done && lane == 0) {
      a.rest[atomicAdd(a.nrest, 1)] = (int32_t)r;
      if (filter_row(nh, need)) {  // its full score row is not stored: list its row tile
        const int g = (int)(r / a.nq);
        const int64_t rt = (r % a.nq) >> 7;
        if (atomicExch(&a.tflag[(int64_t)g * ((a.nq + 127) >> 7) + rt], 1) == 0)
          a.flist[atomicAdd(a.nflist, 1)] = (g << 20) | (int32_t)rt;
      }
    }
    cv = cv_next;
  }
}

}  // namespace

int topk_union_launches(const Dims& dm, int64_t q_begin, int64_t q_end) {
  return 2 + (long_rows_first(dm, q_begin, q_end) < q_end - q_begin ? 1 : 0);
}

int launch_cand_rows(const Dims& dm, int64_t q_begin, int64_t q_end, int32_t* sel,
                     const uint2* cand, const int32_t* ccnt, int caph, int32_t* rest,
                     int32_t* counters, int32_t* tflag, int32_t* flist, int32_t* status,
                     cudaStream_t st) {
  const int64_t nq = q_end - q_begin;
  if (nq <= 0) return SGQA_OK;
  if (caph < 2 || (caph & 1) || cand == nullptr || ccnt == nullptr) return SGQA_ERR_INVALID_ARG;
  TUArgs a;
  std::memset(&a, 0, sizeof(a));
  a.nq = nq;
  a.q_begin = q_begin;
  a.q_end = q_end;
  a.T = dm.T;
  a.off = dm.off;
  a.nblk = dm.nblk;
  a.B = dm.B;
  a.lgB = __builtin_ctz((unsigned)dm.B);
  a.Ks = dm.Ks;
  a.W = dm.W;
  a.Hkv = dm.Hkv;
  a.sel = sel;
  a.cand = cand;
  a.ccnt = ccnt;
  a.caph = caph;
  a.rest = rest;
  a.nrest = counters;
  a.nflist = counters + 1;
  a.tflag = tflag;
  a.flist = flist;
  a.status = status;
  const int64_t nrt = (nq + 127) / 128;
  log_begin(SGQA_K_TOPK_UNION, st);
  bool zeroed = fill_u32(counters, 2, 0u, st) == cudaSuccess;
  log_end(st);
  log_begin(SGQA_K_TOPK_UNION, st);
  zeroed = zeroed && fill_u32(tflag, (int64_t)dm.Hkv * nrt, 0u, st) == cudaSuccess;
  log_end(st);
  if (!zeroed) return SGQA_ERR_CUDA;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0)
    return SGQA_ERR_CUDA;
  const size_t smem = (size_t)CR_WARPS * CR_WORDS * 4;
  if (cudaFuncSetAttribute(k_cand_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SGQA_ERR_CUDA;
  const int64_t nrows = nq * dm.Hkv;
  const int64_t ctas = std::min<int64_t>((nrows + CR_WARPS - 1) / CR_WARPS, (int64_t)nsm * 2);
  log_begin(SGQA_K_TOPK_UNION, st);
  k_cand_rows<<<(unsigned)ctas, CR_WARPS * 32, smem, st>>>(a);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

int launch_row_tau(const Dims& dm, const float* sample_scores, int64_t q_begin, int64_t q_end,
                   float* tau, cudaStream_t st) {
  const int64_t nq = q_end - q_begin;
  if (nq <= 0) return SGQA_OK;
  const int64_t ns_max = sampled_cols(dm);
  if ((ns_max & 3) || (reinterpret_cast<uintptr_t>(sample_scores) & 15u)) return SGQA_ERR_ALIGNMENT;
  const int64_t rows = nq * dm.Hkv;
  const size_t smem = (size_t)TAU_WARPS * TAU_WARP_BYTES;
  if (cudaFuncSetAttribute(k_row_tau, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SGQA_ERR_CUDA;
  log_begin(SGQA_K_ROW_TAU, st);
  k_row_tau<<<(unsigned)((rows + TAU_WARPS - 1) / TAU_WARPS), TAU_WARPS * 32, smem, st>>>(
      sample_scores, tau, nq, q_begin, dm.off, dm.nblk, ns_max, __builtin_ctz((unsigned)dm.B),
      dm.Ks, dm.Hkv);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

size_t topk_union_ws_bytes(const Dims& dm, int64_t nq) {
  return (size_t)dm.Hkv * nq * (dm.Ks > 0 ? dm.Ks : 1) * sizeof(int32_t);
}

// Queries [q_begin, q_end) of the call; slot layout over tiles
// [lay_tau0, lay_tau0 + lay_ntiles) with capG slots per group.
int launch_topk_union_layout(const Dims& dm, const float* scores, int64_t q_begin, int64_t q_end,
                             int32_t* sel, int64_t* union_off, int32_t* union_len,
                             int32_t* union_blk, uint64_t* union_mask, int64_t union_cap,
                             int64_t lay_tau0, int64_t lay_ntiles, int64_t capG,
                             int32_t* status, cudaStream_t st, int32_t* rest,
                             int32_t* nrest) {
  if (q_end <= q_begin) return SGQA_OK;
  if ((rest == nullptr) != (nrest == nullptr)) return SGQA_ERR_INVALID_ARG;
  TUArgs a;
  std::memset(&a, 0, sizeof(a));
  a.rest = rest;
  a.nrest = nrest;
  a.scores = scores;
  a.nq = q_end - q_begin;
  a.q_begin = q_begin;
  a.q_end = q_end;
  a.T = dm.T;
  a.off = dm.off;
  a.nblk = dm.nblk;
  a.B = dm.B;
  a.lgB = __builtin_ctz((unsigned)dm.B);
  a.Ks = dm.Ks;
  a.W = dm.W;
  a.sel = sel;
  a.uoff = union_off;
  a.ulen = union_len;
  a.ublk = union_blk;
  a.umask = union_mask;
  a.ucap = union_cap;
  a.lay_tau0 = lay_tau0;
  a.lay_ntiles = lay_ntiles;
  a.capG = capG;
  a.tau_begin = q_begin / dm.W;
  a.nwords = (int)((dm.nblk + 31) / 32);
  a.status = status;
  a.Hkv = dm.Hkv;
  a.nw = ROW_WARPS;
  const int64_t tau_end = (q_end + dm.W - 1) / dm.W;
  // rows: persistent CTAs, at most four per SM
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0)
    return SGQA_ERR_CUDA;
  // blocks of 8 consecutive rows only where the one-pass candidate path (and
  // its previous-row threshold) can apply; longer rows go one per warp so
  // that many rows stream at once
  {
    const int64_t nh_lo = nh_of(dm, q_begin), nh_hi = nh_of(dm, q_end - 1);
    a.rb = (dm.Ks <= CAND_NEED_MAX && nh_hi >= 2048 && nh_lo <= 16384) ? ROW_BLOCK : 1;
  }
  a.r_end = rest == nullptr ? long_rows_first(dm, q_begin, q_end) : a.nq;
  const int64_t row_blocks = std::max<int64_t>(1, (a.r_end + a.rb - 1) / a.rb * dm.Hkv);
  const int64_t row_ctas =
      std::min<int64_t>((row_blocks + ROW_WARPS - 1) / ROW_WARPS, (int64_t)nsm * 4);
  const size_t row_smem = (size_t)ROW_WARPS * WARP_BYTES;
  // tiles: bitmask + word prefix + member masks (shared while they fit)
  const size_t fixed = (size_t)(((a.nwords + 3) & ~3) + ((a.nwords + 1 + 3) & ~3)) * 4;
  const size_t budget = 200 * 1024;
  if (fixed + 1024 > budget) return SGQA_ERR_UNSUPPORTED;
  const int64_t u_max = std::min<int64_t>((int64_t)dm.W * dm.Ks, dm.nblk);  // slots of a tile
  // (the lists are read twice, from L2; a small footprint keeps many CTAs per SM)
  const size_t mask_budget = budget - fixed;
  const int64_t mask_pairs =
      std::min<int64_t>(std::min<int64_t>(u_max, 4096), (int64_t)(mask_budget / 8));
  const size_t union_smem = fixed + (size_t)mask_pairs * 8;
  if (cudaFuncSetAttribute(k_topk_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)row_smem) != cudaSuccess ||
      cudaFuncSetAttribute(k_tile_union, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)union_smem) != cudaSuccess)
    return SGQA_ERR_CUDA;
  log_begin(SGQA_K_TOPK_UNION, st);
  k_topk_rows<<<(unsigned)row_ctas, ROW_WARPS * 32, row_smem, st>>>(a);
  log_end(st);
  if (cudaGetLastError() != cudaSuccess) return SGQA_ERR_CUDA;
  if (a.r_end < a.nq) {  // the long rows, one CTA each
    const int rc = launch_select_long(dm, scores, q_begin, q_end, a.r_end, sel, status, st);
    if (rc != SGQA_OK) return rc;
  }
  log_begin(SGQA_K_TILE_UNION, st);
  k_tile_union<<<dim3((unsigned)(tau_end - a.tau_begin), (unsigned)dm.Hkv), UNION_THREADS,
                 union_smem, st>>>(a, mask_pairs);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

int launch_topk_union(const Dims& dm, const float* scores, int64_t q_begin, int64_t q_end,
                      int32_t* sel, int64_t* union_off, int32_t* union_len, int32_t* union_blk,
                      uint64_t* union_mask, int64_t union_cap, int32_t* status, cudaStream_t st) {
  return launch_topk_union_layout(dm, scores, q_begin, q_end, sel, union_off, union_len,
                                  union_blk, union_mask, union_cap, 0, dm.ntiles, group_cap(dm),
                                  status, st, nullptr, nullptr);
}

}  // namespace sgqa
