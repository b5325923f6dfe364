// Top-k block selection and tile union.
//
// "Inside Step 5 Preview" (StepFun blog), section Sparse GQA: each query keeps
// its k/B best historical blocks (paragraph "Trade-off between top-k and block
// size"), and the selections of adjacent queries are unioned so one gathered
// block list serves a whole tile (paragraph "Efficient implementation of
// sparse attention").
//
// One CTA per (KV group, tile).  Each warp owns rows (queries) of the tile and
// runs an exact radix select on the row's fp32 scores, compared through the
// order-preserving map of their bit patterns: an 11-bit histogram of the top
// key bits finds the bucket of the k-th largest key, the bucket's members are
// compacted into shared memory, two more histogram levels (11 + 10 bits) pin
// the k-th key exactly, and a final pass in ascending block order emits every
// block above it plus the lowest-indexed blocks equal to it.  Emission uses
// warp ballots, so each list comes out sorted and each 32-block word of the
// tile's union bitmask is OR-ed in one shared atomic.  The union is then the
// set bits of that bitmask (ranks by a prefix sum of word popcounts), and a
// member mask per union slot is built from the rows' lists with shared (or,
// for very long unions, global) atomic ORs.
#include "common.cuh"
#include "internal.h"

namespace sgqa {
namespace {

constexpr int NB0 = 2048;        // bins of the level-0 histogram (top 11 key bits)
constexpr int NBR = 512;         // bins of the refinement histograms (9 bits)
constexpr int WARP_BYTES = NB0 * 4;  // per-warp scratch: level-0 histogram, then
                                     // bucket candidates + a refinement histogram
constexpr int CAND_CAP = (WARP_BYTES - NBR * 4) / 8;  // 768 (key, index) pairs
constexpr unsigned FULL = 0xffffffffu;
constexpr int BATCH = 8;         // 32-element groups loaded before use

struct TUArgs {
  const float* scores;  // [Hkv][nq][nblk], rows q_begin .. q_end-1 of the call
  int64_t nq, q_begin, q_end, T, off, nblk;
  int B, Ks, W;
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
  int32_t* status;
};

__device__ __forceinline__ int64_t cap_of_tile(const TUArgs& a, int64_t tau) {
  const int64_t first = tau * a.W;
  int64_t len = a.T - first;
  if (len > a.W) len = a.W;
  int64_t nh = (a.off + first + len - 1) / a.B;
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
__device__ void hist_row(const float* __restrict__ row, int64_t nh, bool vec, uint32_t* hist,
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
__device__ void select_row_general(const TUArgs& a, const float* __restrict__ row, int64_t nh,
                                   uint32_t need, int32_t* out, bool vec, uint32_t b0,
                                   uint32_t above0, uint32_t cnt0, uint32_t* warp_smem,
                                   uint32_t* tile_bits, int64_t t) {
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
    if (lane == 0 && mt) atomicOr(&tile_bits[j0 >> 5], mt);
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

__device__ void select_row_fast(const TUArgs& a, const float* __restrict__ row, int64_t nh,
                                uint32_t need, int32_t* out, uint32_t b0, uint32_t above0,
                                uint32_t cnt0, uint32_t* warp_smem, uint32_t* tile_bits,
                                int64_t t) {
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
    atomicOr(&tile_bits[v >> 5], 1u << (v & 31));
  }
  for (uint32_t i = lane; i < n_sel; i += 32) {
    const int32_t v = csel[i];
    out[i + lower_bound_smem(defs, (int)n_def, v)] = v;
    atomicOr(&tile_bits[v >> 5], 1u << (v & 31));
  }
  for (int x = (int)need + lane; x < a.Ks; x += 32) out[x] = -1;
  if (lane == 0 && n_def + n_sel != need) report(a.status, SGQA_ERR_BOUNDS, (int)t);
  __syncwarp();
}

// Select row t of group g, write its ascending list and OR it into the tile
// bitmask.  All lanes participate.
__device__ void select_row(const TUArgs& a, int g, int64_t t, uint32_t* warp_smem,
                           uint32_t* tile_bits) {
  const int lane = lane_id();
  const int64_t tl = t - a.q_begin;
  int64_t nh = (a.off + t) / a.B;
  if (nh > a.nblk) nh = a.nblk;
  const uint32_t need = (uint32_t)(nh < a.Ks ? nh : a.Ks);
  const float* row = a.scores + ((int64_t)g * a.nq + tl) * a.nblk;
  int32_t* out = a.sel + ((int64_t)g * a.nq + tl) * a.Ks;
  const bool vec = (a.nblk & 3) == 0;
  if (need == 0) {
    for (int64_t x = lane; x < a.Ks; x += 32) out[x] = -1;
    return;
  }
  if ((int64_t)need == nh) {  // every historical block: no scores to read
    for (int64_t x = lane; x < nh; x += 32) out[x] = (int32_t)x;
    for (int64_t w = lane; w < (nh + 31) / 32; w += 32) {
      const int64_t hi = (w + 1) * 32;
      atomicOr(&tile_bits[w], hi <= nh ? FULL : ((1u << (nh & 31)) - 1u));
    }
    for (int64_t x = nh + lane; x < a.Ks; x += 32) out[x] = -1;
    return;
  }
  // level 0: histogram of the top 11 key bits
  uint32_t b0, above0, cnt0;
  zero_hist(warp_smem, NB0);
  hist_row(row, nh, vec, warp_smem, 21, NB0, 32, 0);
  find_bin(warp_smem, NB0, need, b0, above0, cnt0);
  if (vec && need <= (uint32_t)FAST_MAX && cnt0 <= (uint32_t)FAST_MAX)
    select_row_fast(a, row, nh, need, out, b0, above0, cnt0, warp_smem, tile_bits, t);
  else
    select_row_general(a, row, nh, need, out, vec, b0, above0, cnt0, warp_smem, tile_bits, t);
}

__global__ void k_topk_union(TUArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int g = blockIdx.y;
  const int64_t tau = a.tau_begin + blockIdx.x;
  const int nthr = blockDim.x;
  const int tid = threadIdx.x, warp = warp_id(), lane = lane_id();
  uint32_t* tile_bits = reinterpret_cast<uint32_t*>(smem);
  uint32_t* wprefix = tile_bits + ((a.nwords + 3) & ~3);          // nwords + 1 entries
  uint8_t* wbase = reinterpret_cast<uint8_t*>(wprefix + ((a.nwords + 1 + 3) & ~3));
  __shared__ int64_t s_red[32];
  __shared__ int64_t s_base;

  for (int i = tid; i < a.nwords; i += nthr) tile_bits[i] = 0;

  // slot base of this tile: g * capG + sum of the caps of the layout's earlier tiles
  int64_t part = 0;
  for (int64_t x = a.lay_tau0 + tid; x < tau; x += nthr) part += cap_of_tile(a, x);
  for (int o = 16; o > 0; o >>= 1) part += __shfl_down_sync(FULL, part, o);
  if (lane == 0) s_red[warp] = part;
  __syncthreads();
  if (tid == 0) {
    int64_t s = 0;
    for (int w = 0; w < a.nw; ++w) s += s_red[w];
    s_base = (int64_t)g * a.capG + s;
  }

  // ---- per-row selection
  const int64_t first = tau * a.W;
  int len = (int)((a.T - first) < a.W ? (a.T - first) : a.W);
  uint32_t* wsm = reinterpret_cast<uint32_t*>(wbase + (size_t)warp * WARP_BYTES);
  for (int i = warp; i < len; i += a.nw) select_row(a, g, first + i, wsm, tile_bits);
  __syncthreads();

  // ---- union list: ranks from a prefix sum of word popcounts
  if (warp == 0) {
    uint32_t carry = 0;
    for (int base = 0; base < a.nwords; base += 32) {
      const int w = base + lane;
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
  const int64_t base = s_base;
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

  // ---- member masks
  const int64_t mask_words = (int64_t)a.nw * WARP_BYTES / 8;  // lo/hi pairs that fit
  const bool in_smem = U <= mask_words;
  uint32_t* mlo = reinterpret_cast<uint32_t*>(wbase);
  uint32_t* mhi = mlo + (in_smem ? U : 0);
  if (in_smem) {
    for (int64_t s = tid; s < 2 * U; s += nthr) mlo[s] = 0;
  } else {
    for (int64_t s = tid; s < U; s += nthr) a.umask[base + s] = 0;
  }
  __syncthreads();
  for (int i = warp; i < len; i += a.nw) {
    const int64_t t = first + i;
    int64_t nh = (a.off + t) / a.B;
    if (nh > a.nblk) nh = a.nblk;
    const int64_t need = nh < a.Ks ? nh : a.Ks;
    const int32_t* lst = a.sel + ((int64_t)g * a.nq + (t - a.q_begin)) * a.Ks;
    for (int64_t x = lane; x < need; x += 32) {
      const int32_t j = lst[x];
      const int w = j >> 5;
      const int64_t slot = wprefix[w] + __popc(tile_bits[w] & ((1u << (j & 31)) - 1u));
      if (in_smem) {
        atomicOr(i < 32 ? &mlo[slot] : &mhi[slot], 1u << (i & 31));
      } else {
        atomicOr(reinterpret_cast<unsigned long long*>(&a.umask[base + slot]),
                 1ull << i);
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

}  // namespace

size_t topk_union_ws_bytes(const Dims& dm, int64_t nq) {
  return (size_t)dm.Hkv * nq * (dm.Ks > 0 ? dm.Ks : 1) * sizeof(int32_t);
}

// Queries [q_begin, q_end) of the call; slot layout over tiles
// [lay_tau0, lay_tau0 + lay_ntiles) with capG slots per group.
int launch_topk_union_layout(const Dims& dm, const float* scores, int64_t q_begin, int64_t q_end,
                             int32_t* sel, int64_t* union_off, int32_t* union_len,
                             int32_t* union_blk, uint64_t* union_mask, int64_t union_cap,
                             int64_t lay_tau0, int64_t lay_ntiles, int64_t capG,
                             int32_t* status, cudaStream_t st) {
  if (q_end <= q_begin) return SGQA_OK;
  TUArgs a;
  a.scores = scores;
  a.nq = q_end - q_begin;
  a.q_begin = q_begin;
  a.q_end = q_end;
  a.T = dm.T;
  a.off = dm.off;
  a.nblk = dm.nblk;
  a.B = dm.B;
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
  const int64_t tau_end = (q_end + dm.W - 1) / dm.W;
  const size_t fixed = (size_t)(((a.nwords + 3) & ~3) + ((a.nwords + 1 + 3) & ~3)) * 4;
  const size_t budget = 200 * 1024;
  if (fixed + WARP_BYTES > budget) return SGQA_ERR_UNSUPPORTED;
  int nw = (int)((budget - fixed) / WARP_BYTES);
  if (nw > 8) nw = 8;  // 8 warps and ~70 KB: three CTAs share an SM
  if (nw > dm.W) nw = dm.W < 1 ? 1 : dm.W;
  if (nw < 1) nw = 1;
  a.nw = nw;
  const size_t smem = fixed + (size_t)nw * WARP_BYTES;
  if (cudaFuncSetAttribute(k_topk_union, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SGQA_ERR_CUDA;
  dim3 grid((unsigned)(tau_end - a.tau_begin), (unsigned)dm.Hkv);
  log_begin(SGQA_K_TOPK_UNION, st);
  k_topk_union<<<grid, nw * 32, smem, st>>>(a);
  log_end(st);
  return cudaGetLastError() == cudaSuccess ? SGQA_OK : SGQA_ERR_CUDA;
}

int launch_topk_union(const Dims& dm, const float* scores, int64_t q_begin, int64_t q_end,
                      int32_t* sel, int64_t* union_off, int32_t* union_len, int32_t* union_blk,
                      uint64_t* union_mask, int64_t union_cap, int32_t* status, cudaStream_t st) {
  return launch_topk_union_layout(dm, scores, q_begin, q_end, sel, union_off, union_len,
                                  union_blk, union_mask, union_cap, 0, dm.ntiles, group_cap(dm),
                                  status, st);
}

}  // namespace sgqa
