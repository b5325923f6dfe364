/*
 * CPU ORACLE for the block-wise Sparse GQA prefill path -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  It is a plain, slow, row-at-a-time statement of
 * what the path computes, in fp64 unless a function says otherwise, and it
 * shares no code, header or constant with the CUDA library.
 *
 * Source: "Inside Step 5 Preview: Architecture and Training for Agentic Work"
 * (StepFun blog), section "Sparse GQA": paragraph "Reducing indexer's cost"
 * (adjacent historical positions are compressed into one block
 * representation, B = 8), paragraph "Efficient implementation of sparse
 * attention" (the union of adjacent tokens' top-k results), paragraph
 * "Trade-off between top-k and block size" (k = 4096 tokens, k/B = 512
 * blocks), and the Figure 3 caption (each KV group selects independently;
 * the main path reads the selected historical blocks plus the causally
 * visible positions of the current block).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - merge operator: the mean of the B keys of a block;
 *  - indexer: per KV group, the dot product of the group's mean query with
 *    the block mean, no scale;
 *  - head h belongs to group h / G;
 *  - ties in the top-k go to the lower block index;
 *  - the k/B selected blocks are historical (strictly before the query's own
 *    block); the current block is always added, causally masked;
 *  - the union is a batching device (mode A): each query still attends to its
 *    own selection.  Mode B (every query of a tile attends to the tile's
 *    union, minus its future blocks) is kept as the alternative reading.
 *
 * Notation: T queries, query t sits at position pos(t) = q_offset + t, Tkv
 * keys, H query heads, Hkv KV groups, G = H / Hkv, d head dim, B block size,
 * nblk = floor(Tkv / B) complete blocks, nh(t) = floor(pos(t) / B)
 * historical blocks, Ks = topk_tokens / B blocks to select, W queries per
 * union tile.  Layouts: Q [T][H][d], K and V [Tkv][Hkv][d] (logical
 * positions), scores [Hkv][nrows][nblk], selections [Hkv][T][Ks].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define NEG_INF (-INFINITY)

/* ---------------------------------------------------------------------------
 * Step 1: block merge ("Reducing indexer's cost": adjacent historical
 * positions compressed into a single block representation).
 * Kbar[g][j] = (1/B) * sum_{i<B} K[jB+i][g], for j in [blk_begin, blk_end).
 * ------------------------------------------------------------------------- */

/* fp32 variant with a fixed summation order: adjacent pairs are added level by
 * level, ((k0+k1)+(k2+k3))+((k4+k5)+(k6+k7)) for B = 8, then the sum is
 * multiplied by 1/B (exact for a power-of-two B).  B must be a power of two
 * no larger than 64. */
int orc_merge_tree_f32(const float* K, int64_t Tkv, int Hkv, int d, int B,
                       int64_t blk_begin, int64_t blk_end, float* Kbar /* [Hkv][nblk][d] */) {
  if (B < 1 || B > 64 || (B & (B - 1))) return -1;
  const int64_t nblk = Tkv / B;
  const float inv = 1.0f / (float)B;
#pragma omp parallel for schedule(static)
  for (int64_t j = blk_begin; j < blk_end; ++j) {
    for (int g = 0; g < Hkv; ++g) {
      for (int i = 0; i < d; ++i) {
        float v[64];
        for (int r = 0; r < B; ++r) v[r] = K[((j * B + r) * Hkv + g) * (int64_t)d + i];
        for (int w = B; w > 1; w /= 2)
          for (int r = 0; r < w / 2; ++r) v[r] = v[2 * r] + v[2 * r + 1];
        Kbar[((int64_t)g * nblk + j) * d + i] = v[0] * inv;
      }
    }
  }
  return 0;
}

/* fp64 variant (the reference for scores): plain sum in position order. */
int orc_merge_f64(const float* K, int64_t Tkv, int Hkv, int d, int B,
                  double* Kbar /* [Hkv][nblk][d] */) {
  if (B < 1) return -1;
  const int64_t nblk = Tkv / B;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nblk; ++j)
    for (int g = 0; g < Hkv; ++g)
      for (int i = 0; i < d; ++i) {
        double s = 0.0;
        for (int r = 0; r < B; ++r) s += (double)K[((j * B + r) * Hkv + g) * (int64_t)d + i];
        Kbar[((int64_t)g * nblk + j) * d + i] = s / (double)B;
      }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Step 2: index query.  Each KV group scores history on its own (Figure 3
 * caption); the group's query is the mean of its G heads:
 * qt[r][g] = (1/G) * sum_{h = gG}^{gG+G-1} Q[t_r][h].
 * ------------------------------------------------------------------------- */
int orc_index_query(const float* Q, int64_t T, int H, int Hkv, int d, const int32_t* rows,
                    int64_t nrows, double* qt /* [nrows][Hkv][d] */) {
  if (Hkv < 1 || H % Hkv) return -1;
  const int G = H / Hkv;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t t = rows[r];
    for (int g = 0; g < Hkv; ++g)
      for (int i = 0; i < d; ++i) {
        double s = 0.0;
        for (int h = g * G; h < (g + 1) * G; ++h) s += (double)Q[(t * H + h) * (int64_t)d + i];
        qt[(r * Hkv + g) * (int64_t)d + i] = s / (double)G;
      }
  }
  (void)T;
  return 0;
}

/* ---------------------------------------------------------------------------
 * Step 3: indexer scores ("Reducing indexer's cost"; Figure 3: every causal
 * block is scored).  s[g][r][j] = qt[r][g] . Kbar[g][j] for j < nh(t_r),
 * -inf for j >= nh(t_r).
 * ------------------------------------------------------------------------- */
int orc_scores(const double* qt, const double* Kbar, int64_t nblk, int Hkv, int d, int B,
               int64_t q_offset, const int32_t* rows, int64_t nrows,
               double* S /* [Hkv][nrows][nblk] */) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t nh = (q_offset + rows[r]) / B;
    for (int g = 0; g < Hkv; ++g) {
      const double* q = qt + (r * Hkv + g) * (int64_t)d;
      for (int64_t j = 0; j < nblk; ++j) {
        double s = NEG_INF;
        if (j < nh) {
          const double* k = Kbar + ((int64_t)g * nblk + j) * d;
          s = 0.0;
          for (int i = 0; i < d; ++i) s += q[i] * k[i];
        }
        S[((int64_t)g * nrows + r) * nblk + j] = s;
      }
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Step 3, lower-precision variant: bf16 index scores.  The Step 5 pages leave
 * the indexer's precision open; the DeepSeek-V4 notes (section on FP4 QAT)
 * report that keeping index scores in bf16 instead of fp32 makes the top-k
 * twice as fast at 99.7% recall.  Here both operands are rounded to bf16
 * (nearest, ties to even) from their fp32 values, the products are summed
 * exactly (each product of two bf16 values is exact in fp64, and so is the
 * sum at these sizes), and the score is rounded to bf16 the same way.
 * qt32 [nrows][Hkv][d] and Kbar32 [Hkv][nblk][d] are fp32; S [Hkv][nrows][nblk]
 * is fp32 holding bf16 values, -inf where j >= nh(t_r).
 * ------------------------------------------------------------------------- */
static float round_bf16(double x) {
  /* nearest bf16 value of x, ties to even, decided on the exact value x
   * (its nearest fp32 value only locates the two bf16 neighbours) */
  float f = (float)x; /* nearest fp32 */
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint32_t base = u & 0xFFFF0000u;
  uint32_t down = base, up = base + 0x10000u;
  float fd, fu;
  memcpy(&fd, &down, 4);
  memcpy(&fu, &up, 4);
  /* the two bf16 neighbours of x (fd, fu share the sign of f); pick the
   * nearer by the exact distance, ties to the even mantissa */
  const double dd = fabs(x - (double)fd), du = fabs(x - (double)fu);
  if (dd < du) return fd;
  if (du < dd) return fu;
  return (down & 0x10000u) ? fu : fd;
}

int orc_scores_bf16(const float* qt32, const float* Kbar32, int64_t nblk, int Hkv, int d, int B,
                    int64_t q_offset, const int32_t* rows, int64_t nrows,
                    float* S /* [Hkv][nrows][nblk] */) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t nh = (q_offset + rows[r]) / B;
    for (int g = 0; g < Hkv; ++g) {
      const float* q = qt32 + (r * Hkv + g) * (int64_t)d;
      for (int64_t j = 0; j < nblk; ++j) {
        float s = NEG_INF;
        if (j < nh) {
          const float* k = Kbar32 + ((int64_t)g * nblk + j) * d;
          double acc = 0.0;
          for (int i = 0; i < d; ++i) acc += (double)round_bf16(q[i]) * (double)round_bf16(k[i]);
          s = round_bf16(acc);
        }
        S[((int64_t)g * nrows + r) * nblk + j] = s;
      }
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Step 4: top-k block selection ("Trade-off between top-k and block size":
 * k tokens = k/B blocks).  Row r keeps min(Ks, nh) blocks under the total
 * order "larger score first, equal scores: lower block index first", and
 * lists them in ascending block order, padded with -1.
 * For fp32 scores the comparison uses the order-preserving map of the bit
 * pattern (so -0.0 ranks below +0.0).
 * ------------------------------------------------------------------------- */
typedef struct {
  uint64_t key; /* larger is better */
  int32_t j;
} cand_t;

static int cmp_cand(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->key != y->key) return x->key > y->key ? -1 : 1;
  return x->j < y->j ? -1 : (x->j > y->j);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return x < y ? -1 : (x > y);
}

static uint64_t key_f32(float s) {
  uint32_t u;
  memcpy(&u, &s, 4);
  u ^= (u & 0x80000000u) ? 0xFFFFFFFFu : 0x80000000u;
  return u;
}

static uint64_t key_f64(double s) {
  uint64_t u;
  memcpy(&u, &s, 8);
  u ^= (u & 0x8000000000000000ull) ? 0xFFFFFFFFFFFFFFFFull : 0x8000000000000000ull;
  return u;
}

static void select_row(cand_t* c, int64_t nh, int64_t Ks, int32_t* out) {
  int64_t n = nh < Ks ? nh : Ks;
  qsort(c, (size_t)nh, sizeof(cand_t), cmp_cand);
  for (int64_t i = 0; i < n; ++i) out[i] = c[i].j;
  qsort(out, (size_t)n, sizeof(int32_t), cmp_i32);
  for (int64_t i = n; i < Ks; ++i) out[i] = -1;
}

/* is_f64: scores are double (else float).  S is [Hkv][nrows][nblk]; the output
 * is [Hkv][nrows][Ks]. */
int orc_select(const void* S, int is_f64, int64_t nblk, int Hkv, int B, int64_t q_offset,
               const int32_t* rows, int64_t nrows, int64_t Ks, int32_t* sel) {
  int err = 0;
#pragma omp parallel
  {
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(nblk > 0 ? nblk : 1));
    if (!c) {
#pragma omp atomic write
      err = -2;
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t rg = 0; rg < nrows * Hkv; ++rg) {
      if (!c) continue;
      const int64_t g = rg / nrows, r = rg % nrows;
      int64_t nh = (q_offset + rows[r]) / B;
      if (nh > nblk) nh = nblk;
      const int64_t base = (g * nrows + r) * nblk;
      for (int64_t j = 0; j < nh; ++j) {
        c[j].j = (int32_t)j;
        c[j].key = is_f64 ? key_f64(((const double*)S)[base + j]) : key_f32(((const float*)S)[base + j]);
      }
      select_row(c, nh, Ks, sel + (g * nrows + r) * Ks);
    }
    free(c);
  }
  return err;
}

/* ---------------------------------------------------------------------------
 * Step 5: union over a tile of adjacent queries ("Efficient implementation of
 * sparse attention").  Tiles are [tau W, min(tau W + W, T)).  For each group
 * and tile: U = ascending union of the members' selections; mask[u] bit i is
 * set when U[u] is in the selection of query tau W + i.  Output is CSR:
 * uoff [Hkv][ntiles + 1] (offsets into ublk / umask, global across groups:
 * group g's tile tau spans uoff[g][tau] .. uoff[g][tau + 1]).
 * sel is [Hkv][T][Ks] over all T queries.  ucap bounds the total length; the
 * return value is the total length, or -1 if ucap is too small.
 * ------------------------------------------------------------------------- */
int64_t orc_union(const int32_t* sel, int64_t T, int Hkv, int64_t Ks, int W, int64_t nblk,
                  int64_t ucap, int32_t* uoff, int32_t* ublk, uint64_t* umask) {
  const int64_t ntiles = (T + W - 1) / W;
  uint64_t* m = (uint64_t*)calloc((size_t)(nblk > 0 ? nblk : 1), sizeof(uint64_t));
  if (!m || W > 64) {
    free(m);
    return -1;
  }
  int64_t n = 0;
  for (int g = 0; g < Hkv; ++g) {
    for (int64_t tau = 0; tau < ntiles; ++tau) {
      uoff[(int64_t)g * (ntiles + 1) + tau] = (int32_t)n;
      memset(m, 0, sizeof(uint64_t) * (size_t)nblk);
      for (int i = 0; i < W && tau * W + i < T; ++i) {
        const int32_t* s = sel + ((int64_t)g * T + tau * W + i) * Ks;
        for (int64_t x = 0; x < Ks; ++x)
          if (s[x] >= 0) m[s[x]] |= (uint64_t)1 << i;
      }
      for (int64_t j = 0; j < nblk; ++j) {
        if (!m[j]) continue;
        if (n >= ucap) {
          free(m);
          return -1;
        }
        ublk[n] = (int32_t)j;
        umask[n] = m[j];
        ++n;
      }
    }
    uoff[(int64_t)g * (ntiles + 1) + ntiles] = (int32_t)n;
  }
  free(m);
  return n;
}

/* ---------------------------------------------------------------------------
 * Step 6: main-path attention (Figure 3 caption: the selected historical
 * blocks plus the causally visible positions of the current block).
 * For query t, head h, group g = h / G:
 *   mode 0 (A): allowed p: floor(p/B) in Sel[g][t], or floor(p/B) = floor(pos/B)
 *               and p <= pos.
 *   mode 1 (B): allowed p: floor(p/B) in U[g][tile(t)] and floor(p/B) < floor(pos/B),
 *               or the current-block part as in mode A.
 *   O = sum_p e^{z_p - m} V_p / sum_p e^{z_p - m}, z_p = scale * Q[t][h] . K[p][g],
 *   lse = m + ln sum_p e^{z_p - m}.
 * sel [Hkv][T][Ks] (mode A) or the union CSR of orc_union (mode B).
 * Outputs: O [nrows][H][d] and lse [H][nrows], fp64.
 * ------------------------------------------------------------------------- */
/* The allowed positions of a row: every position of its historical blocks,
 * then its own block up to pos.  Returns their number. */
static int64_t row_positions(int B, int64_t pos, const int32_t* blocks, int64_t nblocks,
                             int64_t* ps) {
  int64_t n = 0;
  for (int64_t x = 0; x < nblocks; ++x)
    for (int r = 0; r < B; ++r) ps[n++] = (int64_t)blocks[x] * B + r;
  for (int64_t p = (pos / B) * B; p <= pos; ++p) ps[n++] = p;
  return n;
}

/* The historical blocks a row attends: its selection (mode A), or its tile's
 * union blocks before its own block (mode B).  Returns their number. */
static int64_t row_blocks(int mode, int64_t T, int g, int64_t t, int64_t cur,
                          const int32_t* sel, int64_t Ks, const int32_t* uoff,
                          const int32_t* ublk, int W, int64_t ntiles, int32_t* blocks) {
  int64_t nb = 0;
  if (mode == 0) {
    const int32_t* s = sel + ((int64_t)g * T + t) * Ks;
    for (int64_t x = 0; x < Ks; ++x)
      if (s[x] >= 0) blocks[nb++] = s[x];
  } else {
    const int64_t tau = t / W;
    const int64_t a = uoff[(int64_t)g * (ntiles + 1) + tau];
    const int64_t b = uoff[(int64_t)g * (ntiles + 1) + tau + 1];
    for (int64_t x = a; x < b; ++x)
      if (ublk[x] < cur) blocks[nb++] = ublk[x];
  }
  return nb;
}

static void attend_row(const float* Q, const float* K, const float* V, int64_t t, int h, int g,
                       int H, int Hkv, int d, int B, int64_t pos, const int32_t* blocks,
                       int64_t nblocks, double scale, double* z, int64_t* ps, double* o,
                       double* lse) {
  const int64_t n = row_positions(B, pos, blocks, nblocks, ps);
  const float* q = Q + (t * H + h) * (int64_t)d;
  double mx = NEG_INF;
  for (int64_t a = 0; a < n; ++a) {
    const float* k = K + (ps[a] * Hkv + g) * (int64_t)d;
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += (double)q[i] * (double)k[i];
    z[a] = scale * s;
    if (z[a] > mx) mx = z[a];
  }
  double l = 0.0;
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int64_t a = 0; a < n; ++a) {
    const double e = exp(z[a] - mx);
    l += e;
    const float* v = V + (ps[a] * Hkv + g) * (int64_t)d;
    for (int i = 0; i < d; ++i) o[i] += e * (double)v[i];
  }
  for (int i = 0; i < d; ++i) o[i] /= l;
  *lse = mx + log(l);
}

int orc_sparse_attn(const float* Q, const float* K, const float* V, int64_t T, int64_t Tkv,
                    int64_t q_offset, int H, int Hkv, int d, int B, int mode,
                    const int32_t* sel, int64_t Ks, const int32_t* uoff, const int32_t* ublk,
                    int W, double scale, const int32_t* rows, int64_t nrows,
                    double* O /* [nrows][H][d] */, double* lse /* [H][nrows] */) {
  if (Hkv < 1 || H % Hkv) return -1;
  const int G = H / Hkv;
  const int64_t ntiles = (T + W - 1) / W;
  int64_t maxk = Ks;
  if (mode == 1) {
    for (int64_t x = 0; x < Hkv * (ntiles + 1) - 1; ++x) {
      int64_t len = (int64_t)uoff[x + 1] - uoff[x];
      if (len > maxk) maxk = len;
    }
  }
  const int64_t cap = maxk * B + B;
  int err = 0;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)cap);
    int64_t* ps = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
    int32_t* blocks = (int32_t*)malloc(sizeof(int32_t) * (size_t)(maxk > 0 ? maxk : 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)d);
    if (!z || !ps || !blocks || !o) {
#pragma omp atomic write
      err = -2;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t rh = 0; rh < nrows * H; ++rh) {
      if (!z || !ps || !blocks || !o) continue;
      const int64_t r = rh / H;
      const int h = (int)(rh % H), g = h / G;
      const int64_t t = rows[r], pos = q_offset + t, cur = pos / B;
      const int64_t nb = row_blocks(mode, T, g, t, cur, sel, Ks, uoff, ublk, W, ntiles, blocks);
      double l;
      attend_row(Q, K, V, t, h, g, H, Hkv, d, B, pos, blocks, nb, scale, z, ps,
                 O + (r * H + h) * (int64_t)d, &l);
      lse[(int64_t)h * nrows + r] = l;
    }
    free(z);
    free(ps);
    free(blocks);
    free(o);
  }
  (void)Tkv;
  return err;
}

/* ---------------------------------------------------------------------------
 * Backward of step 6 (the training side of the same layer: the pages apply
 * the sparse attention in training and inference alike, section Sparse GQA;
 * they give no backward, so this is the derivative of orc_sparse_attn written
 * out).  For the loss L = sum over the given rows and heads of dO . O, with
 * P_p = e^{z_p - lse} over the row's allowed positions (as in orc_sparse_attn):
 *   dV[p][g] += P_p dO
 *   dz_p      = P_p (dO . V[p][g] - dO . O)
 *   dQ[t][h]  = scale * sum_p dz_p K[p][g]
 *   dK[p][g] += scale * dz_p Q[t][h]
 * dO [nrows][H][d] and dQ [nrows][H][d]; dK and dV [Tkv][Hkv][d] are zeroed
 * here and accumulated over the rows (serially: rows share keys).
 * ------------------------------------------------------------------------- */
int orc_sparse_attn_bwd(const float* Q, const float* K, const float* V, const double* dO,
                        int64_t T, int64_t Tkv, int64_t q_offset, int H, int Hkv, int d, int B,
                        int mode, const int32_t* sel, int64_t Ks, const int32_t* uoff,
                        const int32_t* ublk, int W, double scale, const int32_t* rows,
                        int64_t nrows, double* dQ, double* dK, double* dV) {
  if (Hkv < 1 || H % Hkv) return -1;
  const int G = H / Hkv;
  const int64_t ntiles = (T + W - 1) / W;
  int64_t maxk = Ks;
  if (mode == 1) {
    for (int64_t x = 0; x < Hkv * (ntiles + 1) - 1; ++x) {
      int64_t len = (int64_t)uoff[x + 1] - uoff[x];
      if (len > maxk) maxk = len;
    }
  }
  const int64_t cap = maxk * B + B;
  double* z = (double*)malloc(sizeof(double) * (size_t)cap);
  double* pr = (double*)malloc(sizeof(double) * (size_t)cap);
  int64_t* ps = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
  int32_t* blocks = (int32_t*)malloc(sizeof(int32_t) * (size_t)(maxk > 0 ? maxk : 1));
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  int err = (!z || !pr || !ps || !blocks || !o) ? -2 : 0;
  const int64_t nkv = Tkv * Hkv * (int64_t)d;
  for (int64_t x = 0; x < nkv && !err; ++x) {
    dK[x] = 0.0;
    dV[x] = 0.0;
  }
  for (int64_t rh = 0; rh < nrows * H && !err; ++rh) {
    const int64_t r = rh / H;
    const int h = (int)(rh % H), g = h / G;
    const int64_t t = rows[r], pos = q_offset + t, cur = pos / B;
    const int64_t nb = row_blocks(mode, T, g, t, cur, sel, Ks, uoff, ublk, W, ntiles, blocks);
    const int64_t n = row_positions(B, pos, blocks, nb, ps);
    const float* q = Q + (t * H + h) * (int64_t)d;
    const double* go = dO + (r * H + h) * (int64_t)d;
    double mx = NEG_INF;
    for (int64_t a = 0; a < n; ++a) {
      const float* k = K + (ps[a] * Hkv + g) * (int64_t)d;
      double s = 0.0;
      for (int i = 0; i < d; ++i) s += (double)q[i] * (double)k[i];
      z[a] = scale * s;
      if (z[a] > mx) mx = z[a];
    }
    double l = 0.0;
    for (int64_t a = 0; a < n; ++a) {
      pr[a] = exp(z[a] - mx);
      l += pr[a];
    }
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    for (int64_t a = 0; a < n; ++a) {
      pr[a] /= l;
      const float* v = V + (ps[a] * Hkv + g) * (int64_t)d;
      for (int i = 0; i < d; ++i) o[i] += pr[a] * (double)v[i];
    }
    double dOO = 0.0;  /* dO . O */
    for (int i = 0; i < d; ++i) dOO += go[i] * o[i];
    double* gq = dQ + (r * H + h) * (int64_t)d;
    for (int i = 0; i < d; ++i) gq[i] = 0.0;
    for (int64_t a = 0; a < n; ++a) {
      const int64_t kv = (ps[a] * Hkv + g) * (int64_t)d;
      const float* k = K + kv;
      const float* v = V + kv;
      double dP = 0.0;
      for (int i = 0; i < d; ++i) dP += go[i] * (double)v[i];
      const double dz = pr[a] * (dP - dOO);
      for (int i = 0; i < d; ++i) {
        dV[kv + i] += pr[a] * go[i];
        gq[i] += scale * dz * (double)k[i];
        dK[kv + i] += scale * dz * (double)q[i];
      }
    }
  }
  free(z);
  free(pr);
  free(ps);
  free(blocks);
  free(o);
  return err;
}

/* Dense causal GQA attention (every p <= pos), the reference for coverage and
 * for the "all blocks selected" special case.  Outputs as orc_sparse_attn. */
int orc_dense_attn(const float* Q, const float* K, const float* V, int64_t T, int64_t Tkv,
                   int64_t q_offset, int H, int Hkv, int d, double scale, const int32_t* rows,
                   int64_t nrows, double* O, double* lse) {
  if (Hkv < 1 || H % Hkv) return -1;
  const int G = H / Hkv;
  int err = 0;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(Tkv > 0 ? Tkv : 1));
    if (!z) {
#pragma omp atomic write
      err = -2;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t rh = 0; rh < nrows * H; ++rh) {
      if (!z) continue;
      const int64_t r = rh / H;
      const int h = (int)(rh % H), g = h / G;
      const int64_t t = rows[r], pos = q_offset + t;
      const float* q = Q + (t * H + h) * (int64_t)d;
      double mx = NEG_INF;
      for (int64_t p = 0; p <= pos; ++p) {
        const float* k = K + (p * Hkv + g) * (int64_t)d;
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += (double)q[i] * (double)k[i];
        z[p] = scale * s;
        if (z[p] > mx) mx = z[p];
      }
      double l = 0.0;
      double* o = O + (r * H + h) * (int64_t)d;
      for (int i = 0; i < d; ++i) o[i] = 0.0;
      for (int64_t p = 0; p <= pos; ++p) {
        const double e = exp(z[p] - mx);
        l += e;
        const float* v = V + (p * Hkv + g) * (int64_t)d;
        for (int i = 0; i < d; ++i) o[i] += e * (double)v[i];
      }
      for (int i = 0; i < d; ++i) o[i] /= l;
      lse[(int64_t)h * nrows + r] = mx + log(l);
    }
    free(z);
  }
  return err;
}
