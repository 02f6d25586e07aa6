/*
 * mfd_oracle.c -- plain, slow CPU oracle for the Multi-Future Drafting (MFD)
 * drafting-and-verification round.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Sources (page title, section):
 *   [MC]  "MFD drafter for Qwen3.5-4B" model card, Model table (target LM head
 *         used at run time on the drafter's hidden states) and the first
 *         paragraph (B best prefixes by best-mode log-probability, standard
 *         tree verification, lossless).
 *   [PP]  "Multi-Future Drafting" project page: "How it works" step 1 (the
 *         expected accepted length is the covered mass, the best tree holds
 *         the most probable prefixes), step 2 (one distribution per position
 *         and mode, drafted in one pass), step 3 (every prefix scored by its
 *         best mode; the B best over all modes form one tree, the union of the
 *         per-mode trees, found by merging the K best-first searches into one
 *         heap), Figure 2 (c) (target verifies the tree in one pass).
 *   [SMDS] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *         1, 2, 3", SC'11 -- the Philox4x32 bijection with 10 rounds.
 *
 * Precision: logits and the log-sum-exp in double (the pages fix no
 * precision for them); prefix scores as an fp32 left fold in depth order and
 * the sampled-verification perturbation in fp32 (the method statement fixes
 * those).  Build with -O2 -fno-fast-math -ffp-contract=off so that every
 * float operation is a single IEEE-rounded step.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_L 16

/* ------------------------------------------------------------------------ */
/* bf16 -> float: a bf16 value is the upper 16 bits of an IEEE binary32.     */
static float bf16_to_float(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ------------------------------------------------------------------------ */
/* [MC] Model table: the target's LM head is applied to the drafter's hidden
 * states.  z[r][v] = sum_h h[r][h] * W[v][h], accumulated in double.
 * Rows are written for v in [v0, v1) into z[r * (v1 - v0) + (v - v0)]. */
void oracle_lmhead_logits(const uint16_t *h, int R, int H, const uint16_t *W,
                          int v0, int v1, double *z, int nthreads) {
  int nv = v1 - v0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (int v = v0; v < v1; ++v) {
    const uint16_t *w = W + (size_t)v * H;
    for (int r = 0; r < R; ++r) {
      const uint16_t *x = h + (size_t)r * H;
      double acc = 0.0;
      for (int k = 0; k < H; ++k)
        acc += (double)bf16_to_float(x[k]) * (double)bf16_to_float(w[k]);
      z[(size_t)r * nv + (v - v0)] = acc;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* [PP] step 2: one distribution per (mode, position): p = softmax(z).
 * log p_v = z_v - LSE, LSE = m + log sum_v exp(z_v - m), m = max_v z_v,
 * all in double; the table value is log p rounded once to fp32.
 * The top-k of a row is its first k entries after sorting by
 * (log p descending, token id ascending). */
typedef struct {
  float lp;
  int32_t tok;
} lp_tok;

static int cmp_lp_tok(const void *a, const void *b) {
  const lp_tok *x = (const lp_tok *)a, *y = (const lp_tok *)b;
  if (x->lp > y->lp) return -1;
  if (x->lp < y->lp) return 1;
  return (x->tok < y->tok) ? -1 : (x->tok > y->tok);
}

static void row_logsoftmax_topk(const double *z, int V, int topk, float *tk_logp,
                                int32_t *tk_tok, double *lse_out, lp_tok *scratch) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v)
    if (z[v] > m) m = z[v];
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp(z[v] - m);
  double lse = m + log(s);
  for (int v = 0; v < V; ++v) {
    scratch[v].lp = (float)(z[v] - lse);
    scratch[v].tok = v;
  }
  qsort(scratch, (size_t)V, sizeof(lp_tok), cmp_lp_tok);
  for (int j = 0; j < topk; ++j) {
    tk_logp[j] = scratch[j].lp;
    tk_tok[j] = scratch[j].tok;
  }
  if (lse_out) *lse_out = lse;
}

/* fp32 logits given directly (no LM head). */
int oracle_logits_topk(const float *logits, int R, int V, int topk, float *tk_logp,
                       int32_t *tk_tok, double *lse) {
  if (topk < 1 || topk > V) return 1;
  double *z = (double *)malloc(sizeof(double) * (size_t)V);
  lp_tok *scr = (lp_tok *)malloc(sizeof(lp_tok) * (size_t)V);
  if (!z || !scr) { free(z); free(scr); return 2; }
  for (int r = 0; r < R; ++r) {
    for (int v = 0; v < V; ++v) z[v] = (double)logits[(size_t)r * V + v];
    row_logsoftmax_topk(z, V, topk, tk_logp + (size_t)r * topk, tk_tok + (size_t)r * topk,
                        lse ? lse + r : NULL, scr);
  }
  free(z);
  free(scr);
  return 0;
}

/* LM head + log-softmax + top-k for R rows; rows run in parallel, each row
 * takes its logits over the full vocabulary from oracle_lmhead_logits'
 * definition. */
int oracle_lmhead_topk(const uint16_t *h, int R, int H, const uint16_t *W, int V, int topk,
                       float *tk_logp, int32_t *tk_tok, double *lse, int nthreads) {
  if (topk < 1 || topk > V) return 1;
  double *z = (double *)malloc(sizeof(double) * (size_t)R * V);
  if (!z) return 2;
  oracle_lmhead_logits(h, R, H, W, 0, V, z, nthreads);
  int err = 0;
#ifdef _OPENMP
#pragma omp parallel
#endif
  {
    lp_tok *scr = (lp_tok *)malloc(sizeof(lp_tok) * (size_t)V);
    if (!scr) {
      err = 2;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
      for (int r = 0; r < R; ++r)
        row_logsoftmax_topk(z + (size_t)r * V, V, topk, tk_logp + (size_t)r * topk,
                            tk_tok + (size_t)r * topk, lse ? lse + r : NULL, scr);
      free(scr);
    }
  }
  free(z);
  return err;
}

/* ------------------------------------------------------------------------ */
/* [PP] "In a serving engine", Figure 5 caption: the drafter's linear layers
 * run in FP8 with the serving engine's online option -- the weight quantized
 * once when it is loaded, the activations quantized on the fly -- and the
 * acceptance length does not change.  The pages name no format or scale
 * granularity; the reading here: FP8 E4M3 (4 exponent bits, bias 7, 3
 * mantissa bits, no infinities, largest finite 448), one scale for the whole
 * weight, one scale per hidden-state row, each the row's (tensor's) largest
 * magnitude over 448, values rounded to nearest-even and saturated at 448.
 *
 * Every fp32 step below is one IEEE-rounded float operation. */
#define E4M3_MAX 448.0f

/* float -> E4M3 byte, round to nearest even, saturating to +-448; NaN -> 0x7F.
 * Written from the format: normal numbers (1 + m/8) 2^(e-7) for exponent
 * fields e = 1..15 (0x7F and 0xFF are NaN), subnormals (m/8) 2^-6. */
uint8_t oracle_e4m3(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  double a = fabs((double)x);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);            /* a = f 2^e with f in [0.5, 1): a in [2^(e-1), 2^e) */
  int ex = e - 1;          /* unbiased exponent of a */
  if (ex < -6) ex = -6;    /* subnormal range shares the quantum of the smallest binade */
  double quantum = ldexp(1.0, ex - 3);
  double r = nearbyint(a / quantum) * quantum; /* exact scaling; ties to even (default mode) */
  if (r > (double)E4M3_MAX) r = (double)E4M3_MAX;
  if (r == 0.0) return sign;
  int er;
  double fr = frexp(r, &er);                  /* r = fr 2^er, fr in [0.5, 1) */
  int unb = er - 1;
  if (unb < -6) {                              /* subnormal: r = m 2^-9 */
    int m = (int)ldexp(r, 9);
    return (uint8_t)(sign | (uint8_t)m);
  }
  int mant = (int)ldexp(fr * 2.0 - 1.0, 3);    /* 3 mantissa bits */
  return (uint8_t)(sign | (uint8_t)((unb + 7) << 3) | (uint8_t)mant);
}

/* E4M3 byte -> its exact value. */
double oracle_e4m3_value(uint8_t b) {
  int sign = b & 0x80, ef = (b >> 3) & 15, m = b & 7;
  if (ef == 15 && m == 7) return NAN;
  double v = ef == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, ef - 7);
  return sign ? -v : v;
}

/* Quantize n bf16 values with one scale: amax = max |x|, inv = 448 / amax,
 * q = e4m3(x * inv), scale = amax / 448 (an all-zero input gives inv = 0 and
 * scale 0). */
void oracle_fp8_quantize(const uint16_t *x, size_t n, uint8_t *q, float *scale) {
  float amax = 0.0f;
  for (size_t i = 0; i < n; ++i) {
    float a = fabsf(bf16_to_float(x[i]));
    if (a > amax) amax = a;
  }
  float inv = amax > 0.0f ? E4M3_MAX / amax : 0.0f;
  for (size_t i = 0; i < n; ++i) q[i] = oracle_e4m3(bf16_to_float(x[i]) * inv);
  *scale = amax / E4M3_MAX;
}

/* The FP8 LM head, log-softmax and top-k: W quantized with one scale sW, each
 * hidden row r with its own scale t_r; z[r][v] = f_r * sum_h q_h[r][h] q_W[v][h]
 * with f_r = t_r * sW (one fp32 product), the sum of exact E4M3 products in
 * double; then the log-softmax and top-k of row_logsoftmax_topk.  Outputs as
 * oracle_lmhead_topk, plus the quantized weight's scale (sW) and the rows'
 * scales (t, [R]). */
int oracle_lmhead_fp8_topk(const uint16_t *h, int R, int H, const uint16_t *W, int V, int topk,
                           float *tk_logp, int32_t *tk_tok, double *lse, float *sW_out, float *t_out,
                           int nthreads) {
  if (topk < 1 || topk > V) return 1;
  uint8_t *qW = (uint8_t *)malloc((size_t)V * H);
  uint8_t *qh = (uint8_t *)malloc((size_t)R * H);
  double *z = (double *)malloc(sizeof(double) * (size_t)R * V);
  float *t = (float *)malloc(sizeof(float) * (size_t)R);
  double lut[256];
  if (!qW || !qh || !z || !t) { free(qW); free(qh); free(z); free(t); return 2; }
  for (int b = 0; b < 256; ++b) lut[b] = oracle_e4m3_value((uint8_t)b);
  float sW;
  oracle_fp8_quantize(W, (size_t)V * H, qW, &sW);
  for (int r = 0; r < R; ++r) oracle_fp8_quantize(h + (size_t)r * H, (size_t)H, qh + (size_t)r * H, &t[r]);
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (int v = 0; v < V; ++v) {
    const uint8_t *w = qW + (size_t)v * H;
    for (int r = 0; r < R; ++r) {
      const uint8_t *x = qh + (size_t)r * H;
      double acc = 0.0;
      for (int k = 0; k < H; ++k) acc += lut[x[k]] * lut[w[k]];
      const float f = t[r] * sW;
      z[(size_t)r * V + v] = (double)f * acc;
    }
  }
  int err = 0;
#ifdef _OPENMP
#pragma omp parallel
#endif
  {
    lp_tok *scr = (lp_tok *)malloc(sizeof(lp_tok) * (size_t)V);
    if (!scr) {
      err = 2;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
      for (int r = 0; r < R; ++r)
        row_logsoftmax_topk(z + (size_t)r * V, V, topk, tk_logp + (size_t)r * topk,
                            tk_tok + (size_t)r * topk, lse ? lse + r : NULL, scr);
      free(scr);
    }
  }
  if (sW_out) *sW_out = sW;
  if (t_out) memcpy(t_out, t, sizeof(float) * (size_t)R);
  free(qW); free(qh); free(z); free(t);
  return err;
}

/* ------------------------------------------------------------------------ */
/* [PP] step 3: mixture DDTree.
 *
 * Mode k scores a prefix x = (x_1..x_d) by the fp32 left fold of its
 * per-position table log-probabilities, in depth order; a token that is not
 * in mode k's top-k row at that position makes the prefix unreachable for
 * mode k (score -inf).  s(x) = max_k score_k(x).  Order: x before y iff
 * s(x) > s(y), or s(x) == s(y) and x's token ids are lexicographically
 * smaller (unsigned compare, a proper prefix first).  The tree keeps the B
 * first prefixes of depth 1..L with s > -inf.
 *
 * Algorithm, as the page states it: the K per-mode best-first searches merged
 * into one heap.  An entry is (mode, prefix, score_k).  Popping an entry
 * pushes all of its children in that mode.  A popped prefix that was already
 * kept (from another mode) is not kept again, but its children are still
 * pushed, because they belong to its own mode's search.  Ties between equal
 * (score, prefix) entries of different modes pop the smaller mode first, so
 * the recorded mode is the smallest one that attains s(x). */
typedef struct {
  float score;
  int32_t mode;
  int32_t depth;
  int32_t tok[ORACLE_MAX_L];
} heap_entry;

static int lex_cmp(const int32_t *a, int da, const int32_t *b, int db) {
  int n = da < db ? da : db;
  for (int i = 0; i < n; ++i) {
    uint32_t x = (uint32_t)a[i], y = (uint32_t)b[i];
    if (x != y) return x < y ? -1 : 1;
  }
  return (da > db) - (da < db);
}

/* returns nonzero iff a must pop before b */
static int entry_before(const heap_entry *a, const heap_entry *b) {
  if (a->score != b->score) return a->score > b->score;
  int c = lex_cmp(a->tok, a->depth, b->tok, b->depth);
  if (c != 0) return c < 0;
  return a->mode < b->mode;
}

typedef struct {
  heap_entry *e;
  size_t n, cap;
} heap_t;

static int heap_push(heap_t *hp, const heap_entry *x) {
  if (hp->n == hp->cap) {
    size_t nc = hp->cap ? hp->cap * 2 : 1024;
    heap_entry *ne = (heap_entry *)realloc(hp->e, nc * sizeof(heap_entry));
    if (!ne) return 2;
    hp->e = ne;
    hp->cap = nc;
  }
  size_t i = hp->n++;
  hp->e[i] = *x;
  while (i > 0) {
    size_t p = (i - 1) / 2;
    if (!entry_before(&hp->e[i], &hp->e[p])) break;
    heap_entry t = hp->e[i];
    hp->e[i] = hp->e[p];
    hp->e[p] = t;
    i = p;
  }
  return 0;
}

static heap_entry heap_pop(heap_t *hp) {
  heap_entry top = hp->e[0];
  hp->e[0] = hp->e[--hp->n];
  size_t i = 0;
  for (;;) {
    size_t l = 2 * i + 1, r = l + 1, b = i;
    if (l < hp->n && entry_before(&hp->e[l], &hp->e[b])) b = l;
    if (r < hp->n && entry_before(&hp->e[r], &hp->e[b])) b = r;
    if (b == i) break;
    heap_entry t = hp->e[i];
    hp->e[i] = hp->e[b];
    hp->e[b] = t;
    i = b;
  }
  return top;
}

/* One request.  tk_logp / tk_tok: [K][L][topk], row (k, i) holds mode k's
 * table for depth i+1.  Outputs sized for N = B + 1 nodes; mask has
 * W32 = ceil(N / 32) words per row.  Node 0 is the root (the anchor token at
 * depth 0); nodes 1.. are the kept prefixes in the order above, which is
 * topological because every prefix comes before its extensions.  Rows past
 * n_nodes are filled with -1 (ints), -inf (score) and zero mask words.
 * Returns 0, or 1 on bad arguments, 2 on allocation failure. */
int oracle_build_tree(const float *tk_logp, const int32_t *tk_tok, int K, int L, int topk,
                      int B, int32_t anchor, int32_t base_pos, int32_t *parent, int32_t *token,
                      int32_t *depth, float *score, int32_t *mode, uint32_t *mask, int32_t *pos,
                      int32_t *n_nodes) {
  if (K < 1 || L < 1 || L > ORACLE_MAX_L || topk < 1 || B < 1) return 1;
  const int N = B + 1, W32 = (N + 31) / 32;
  heap_t hp = {0};
  heap_entry *kept = (heap_entry *)malloc(sizeof(heap_entry) * (size_t)N);
  if (!kept) return 2;
  int err = 0;

  for (int k = 0; k < K && !err; ++k) {
    const float *lp = tk_logp + ((size_t)k * L + 0) * topk;
    const int32_t *tk = tk_tok + ((size_t)k * L + 0) * topk;
    for (int j = 0; j < topk && !err; ++j) {
      if (lp[j] == -INFINITY) continue;
      heap_entry e;
      memset(&e, 0, sizeof e);
      e.score = lp[j];
      e.mode = k;
      e.depth = 1;
      e.tok[0] = tk[j];
      err = heap_push(&hp, &e);
    }
  }

  int nk = 0;
  while (!err && hp.n > 0 && nk < B) {
    heap_entry e = heap_pop(&hp);
    int seen = 0;
    for (int i = 0; i < nk && !seen; ++i)
      seen = lex_cmp(kept[i].tok, kept[i].depth, e.tok, e.depth) == 0;
    if (!seen) kept[nk++] = e;
    if (e.depth < L) {
      const float *lp = tk_logp + ((size_t)e.mode * L + e.depth) * topk;
      const int32_t *tk = tk_tok + ((size_t)e.mode * L + e.depth) * topk;
      for (int j = 0; j < topk && !err; ++j) {
        if (lp[j] == -INFINITY) continue;
        heap_entry c = e;
        c.score = e.score + lp[j]; /* fp32 left fold, one rounding */
        c.tok[c.depth] = tk[j];
        c.depth = e.depth + 1;
        err = heap_push(&hp, &c);
      }
    }
  }
  free(hp.e);
  if (err) {
    free(kept);
    return err;
  }

  for (int i = 0; i < N; ++i) {
    parent[i] = -1;
    token[i] = -1;
    depth[i] = -1;
    score[i] = -INFINITY;
    mode[i] = -1;
    pos[i] = -1;
  }
  memset(mask, 0, sizeof(uint32_t) * (size_t)N * W32);
  parent[0] = -1;
  token[0] = anchor;
  depth[0] = 0;
  score[0] = 0.0f;
  mode[0] = -1;
  pos[0] = base_pos;
  for (int i = 0; i < nk; ++i) {
    int n = i + 1;
    token[n] = kept[i].tok[kept[i].depth - 1];
    depth[n] = kept[i].depth;
    score[n] = kept[i].score;
    mode[n] = kept[i].mode;
    pos[n] = base_pos + kept[i].depth;
    int par = 0;
    if (kept[i].depth > 1) {
      par = -1;
      for (int j = 0; j < i && par < 0; ++j)
        if (lex_cmp(kept[j].tok, kept[j].depth, kept[i].tok, kept[i].depth - 1) == 0) par = j + 1;
    }
    parent[n] = par;
  }
  /* mask row i: bit j set iff node j lies on the root->i path (inclusive). */
  for (int i = 0; i <= nk; ++i)
    for (int a = i; a >= 0; a = parent[a]) mask[(size_t)i * W32 + a / 32] |= 1u << (a % 32);
  *n_nodes = nk + 1;
  free(kept);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* [SMDS] Philox4x32 with 10 rounds.  One round maps the counter (c0,c1,c2,c3)
 * under key (k0,k1) to
 *   (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))
 * with the paper's multipliers M0 = 0xD2511F53, M1 = 0xCD9E8D57; between
 * rounds the key advances by the Weyl increments 0x9E3779B9 (golden ratio)
 * and 0xBB67AE85 (sqrt(3) - 1). */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

void oracle_philox_batch(const uint32_t *ctr, const uint32_t *key, int n, uint32_t *out) {
  for (int i = 0; i < n; ++i) oracle_philox4x32_10(ctr + 4 * i, key + 2 * i, out + 4 * i);
}

/* Gumbel noise for (seed, node, vocab id): word v mod 4 of the Philox4x32-10
 * block with counter (v div 4, node, 0, 0) and key (seed low 32 bits, seed
 * high 32 bits), so one block serves four consecutive vocabulary ids;
 * u = (2 * (x >> 9) + 1) * 2^-24, exact in fp32 and strictly inside (0, 1);
 * G = -log(-log(u)) with fp32 logarithms. */
float oracle_gumbel(uint64_t seed, int32_t node, int32_t v) {
  uint32_t ctr[4] = {(uint32_t)v / 4u, (uint32_t)node, 0u, 0u};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t o[4];
  oracle_philox4x32_10(ctr, key, o);
  float u = (float)(2u * (o[(uint32_t)v % 4u] >> 9) + 1u) * 0x1p-24f;
  return -logf(-logf(u));
}

void oracle_gumbel_batch(uint64_t seed, int32_t node, int V, float *g) {
  for (int v = 0; v < V; ++v) g[v] = oracle_gumbel(seed, node, v);
}

/* ------------------------------------------------------------------------ */
/* [MC] first paragraph, [PP] Figure 2 (c): standard tree verification.
 * From the root, the target picks a token y at the current node: greedy
 * (T == 0) y = argmax_v t[cur][v]; sampled (T > 0) y = argmax_v
 * (t[cur][v] / T + G(seed, cur, v)) in fp32, the Gumbel-max draw from
 * softmax(t / T).  Ties go to the smallest v.  If a child of cur carries
 * token y the walk moves there and continues, otherwise y is the bonus
 * token and the walk stops.
 * Outputs: accept_len = drafted tokens accepted; path_nodes[j] = node whose
 * row was read at step j (path_nodes[0] = 0); out_tokens[j] = y at step j
 * (accepted tokens, then the bonus last); gap[j] = top-1 minus top-2 score
 * at step j (the decision margin).  Entries past accept_len hold -1 / +inf.
 * Returns 0, or 1 on bad arguments. */
int oracle_verify(const float *t, int n_nodes, int V, int L, const int32_t *parent,
                  const int32_t *token, float temperature, uint64_t seed, int32_t *accept_len,
                  int32_t *path_nodes, int32_t *out_tokens, float *gap) {
  if (n_nodes < 1 || V < 2 || L < 1 || !(temperature >= 0.0f)) return 1;
  for (int j = 0; j <= L; ++j) {
    path_nodes[j] = -1;
    out_tokens[j] = -1;
    gap[j] = INFINITY;
  }
  int cur = 0, a = 0;
  for (int step = 0; step <= L; ++step) {
    const float *row = t + (size_t)cur * V;
    float best = -INFINITY, second = -INFINITY;
    int y = -1;
    for (int v = 0; v < V; ++v) {
      float sc = row[v];
      if (temperature > 0.0f) sc = row[v] / temperature + oracle_gumbel(seed, cur, v);
      if (y < 0 || sc > best) {
        second = best;
        best = sc;
        y = v;
      } else if (sc > second) {
        second = sc;
      }
    }
    path_nodes[step] = cur;
    out_tokens[step] = y;
    gap[step] = best - second;
    int next = -1;
    for (int c = 1; c < n_nodes && next < 0; ++c)
      if (parent[c] == cur && token[c] == y) next = c;
    if (next < 0) break;
    cur = next;
    ++a;
  }
  *accept_len = a;
  return 0;
}
