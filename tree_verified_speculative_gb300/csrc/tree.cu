// tree.cu -- the mixture DDTree of one round (project page "Multi-Future
// Drafting", How it works, step 3, and the Figure 1/2 caption): every prefix
// is scored by its best mode; the B best prefixes over all modes form one
// tree, which is the union of the per-mode trees at the common cut-off;
// shared prefixes are built once.
//
// One CTA (512 threads) builds one request's tree in shared memory.
//
// Keys.  A prefix is ordered by (s desc, token ids lexicographically asc, a
// proper prefix first).  For the lexicographic part every drafted position i
// gets the sorted union U_i of all modes' top-k tokens at i (at most 512),
// and a prefix is encoded as the tuple of its tokens' indices in U_i, 9 bits
// per position, zero-padded past its depth, followed by its depth: comparing
// these 149-bit keys as unsigned integers is exactly the lexicographic order
// of the token sequences, with a proper prefix first.  Equal keys mean equal
// sequences, so the key also identifies a node.
//
// Search.  The pool holds (mode, prefix) entries scored by their own mode.
// Level t expands the depth-t entries of the pool: the children of a mode-k
// entry come from mode k's row at depth t+1 in rank order, so their scores
// only fall.  A cut-off key kappa prunes the search: kappa = the best, over
// modes, of each mode's B-th best entry.  Each mode's entries are distinct
// prefixes, and a prefix's mixture score is at least its mode score, so at
// least B distinct prefixes are at least as good as kappa: the true B-th
// prefix of the mixture is never worse than kappa, and every entry that can
// reach the tree is kept.  kappa only improves as entries arrive.  When the
// pool fills up, kappa is recomputed, the pool pruned, and the expansion
// resumes where it stopped (each entry remembers its next child rank).
//
// Result.  After the last level the pool holds every (mode, prefix) entry
// that is at least as good as the final kappa, which includes the best-mode
// entry of every prefix in the tree.  A hash table on the prefix key keeps,
// per prefix, the entry with the best (score, then smallest mode); the B
// best of those are the tree.  Node order comes from rank counting, parents
// from a table lookup of the prefix key with its last position removed.
#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int THREADS = 512;
constexpr int NWARPS = THREADS / 32;
constexpr int TIE_CAP = 1024;
constexpr int MAX_PASSES = 256;

struct Entry {
  uint64_t g0, g1, g2;  // prefix key: positions 1-7, 8-14, 15-16 + depth
  float score;          // the entry's own-mode score (fp32 left fold)
  uint8_t mode, depth, next_j, pad;
};
static_assert(sizeof(Entry) == 32, "entry layout");

struct Key {
  uint32_t sk;  // desc_key(score)
  uint64_t g0, g1, g2;
};

__device__ __forceinline__ Key key_of(const Entry &e) { return Key{desc_key(e.score), e.g0, e.g1, e.g2}; }

__device__ __forceinline__ bool key_before(const Key &a, const Key &b) {
  if (a.sk != b.sk) return a.sk < b.sk;
  if (a.g0 != b.g0) return a.g0 < b.g0;
  if (a.g1 != b.g1) return a.g1 < b.g1;
  return a.g2 < b.g2;
}

__device__ __forceinline__ bool gk_less(uint64_t a0, uint64_t a1, uint64_t a2, uint64_t b0, uint64_t b1,
                                        uint64_t b2) {
  if (a0 != b0) return a0 < b0;
  if (a1 != b1) return a1 < b1;
  return a2 < b2;
}

// Position pos (1-based) of the key holds the token's index in U_pos.
__device__ __forceinline__ void gk_set(uint64_t &g0, uint64_t &g1, uint64_t &g2, int pos, uint32_t u) {
  const int w = (pos - 1) / 7, sl = (pos - 1) % 7;
  const int sh = 54 - 9 * sl;
  const uint64_t m = (uint64_t)0x1FF << sh, v = (uint64_t)(u & 0x1FF) << sh;
  if (w == 0)
    g0 = (g0 & ~m) | v;
  else if (w == 1)
    g1 = (g1 & ~m) | v;
  else
    g2 = (g2 & ~m) | v;
}
__device__ __forceinline__ uint32_t gk_get(uint64_t g0, uint64_t g1, uint64_t g2, int pos) {
  const int w = (pos - 1) / 7, sl = (pos - 1) % 7;
  const int sh = 54 - 9 * sl;
  const uint64_t g = (w == 0) ? g0 : (w == 1) ? g1 : g2;
  return (uint32_t)((g >> sh) & 0x1FF);
}
__device__ __forceinline__ void gk_set_depth(uint64_t &g2, int d) { g2 = (g2 & ~(uint64_t)31) | (uint64_t)d; }

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  x ^= x >> 30;
  x *= 0xBF58476D1CE4E5B9ull;
  x ^= x >> 27;
  x *= 0x94D049BB133111EBull;
  x ^= x >> 31;
  return x;
}
__device__ __forceinline__ uint64_t gk_hash(uint64_t g0, uint64_t g1, uint64_t g2, uint64_t seed) {
  uint64_t h = mix64(g0 ^ seed);
  h = mix64(h ^ g1 ^ 0x632BE59BD9B4E019ull);
  h = mix64(h ^ g2 ^ 0x8CB92BA72F3D8DD7ull);
  return h | 1ull;  // 0 marks an empty slot
}

__device__ __forceinline__ int warp_excl_scan(int x, int lane) {
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  return incl - x;
}

struct Params {
  const float *tk_logp;
  const int32_t *tk_tok;
  int K, L, topk, B;
  const int32_t *anchor, *base_pos;
  int32_t *parent, *token, *depth;
  float *score;
  int32_t *mode;
  uint32_t *mask;
  int32_t *pos, *n_nodes, *status;
  int32_t *union_ws;
  int cap, tsize;
};

struct Layout {
  size_t pool, live0, live1, freel, alive, nodeof, hslot, lp, gam, table, hist1, ties, par, nslot, total;
};

__host__ __device__ inline size_t al(size_t o, size_t a) { return (o + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int K, int L, int topk, int B, int cap, int tsize) {
  Layout y;
  size_t o = 0;
  const size_t klt = (size_t)K * L * topk;
  const size_t hist = (size_t)K * 256 * 4, tbl = (size_t)tsize * 16;
  y.pool = o;
  o += (size_t)cap * 32;
  y.live0 = o = al(o, 16);
  o += (size_t)cap * 2;
  y.live1 = o = al(o, 16);
  o += (size_t)cap * 2;
  y.freel = o = al(o, 16);
  o += (size_t)cap * 2;
  y.nodeof = o = al(o, 16);
  o += (size_t)cap * 2;
  y.hslot = o = al(o, 16);
  o += (size_t)cap * 2;
  y.alive = o = al(o, 16);
  o += (size_t)cap;
  y.lp = o = al(o, 16);
  o += klt * 4;
  y.gam = o = al(o, 16);
  o += klt * 2;
  y.table = o = al(o, 16);
  o += hist > tbl ? hist : tbl;
  y.hist1 = o = al(o, 16);
  o += 256 * 4;
  y.ties = o = al(o, 16);
  o += TIE_CAP * 2;
  y.par = o = al(o, 16);
  o += (size_t)(B + 1) * 2;
  y.nslot = o = al(o, 16);
  o += (size_t)(B + 1) * 2;
  y.total = al(o, 128);
  return y;
}

// Scalars shared by the whole CTA.
struct Shared {
  int n_live, n_new, tail, nfree, free_used, overflow, any_child, bad, has_kappa, nties, tie_over, coll;
  int n_sel, n_prim;
  int cur;  // which live buffer is current
  int cnt[16], active[16], rem[16], ntie[16];
  uint32_t pre[16];
  uint64_t kg[16][3];
  Key kappa;
};

// The B-th best key (score desc, prefix key asc) within each group.  Group
// of live entry i: grp(i) in [0, G) or -1 (ignored).  Sets sh.active[g] for
// groups with at least B members and, for those, sh.pre[g] (score key) and
// sh.kg[g] (prefix key) of their B-th best entry; sh.has_kappa = any active.
template <typename GroupFn>
__device__ void select_bth(Shared &sh, const Entry *pool, const uint16_t *live, int n_live, int G, int B,
                           uint32_t *hist, uint16_t *ties, GroupFn grp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 16) {
    sh.cnt[tid] = 0;
    sh.pre[tid] = 0;
    sh.rem[tid] = B;
    sh.ntie[tid] = 0;
  }
  if (tid == 0) {
    sh.nties = 0;
    sh.tie_over = 0;
  }
  __syncthreads();
  for (int i = tid; i < n_live; i += THREADS) {
    const int g = grp(i);
    if (g >= 0) atomicAdd(&sh.cnt[g], 1);
  }
  __syncthreads();
  if (tid < 16) sh.active[tid] = (tid < G && sh.cnt[tid] >= B);
  __syncthreads();
  if (tid == 0) {
    int any = 0;
    for (int g = 0; g < G; ++g) any |= sh.active[g];
    sh.has_kappa = any;
  }
  __syncthreads();
  if (!sh.has_kappa) return;

  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < G * 256; i += THREADS) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n_live; i += THREADS) {
      const int g = grp(i);
      if (g < 0 || !sh.active[g]) continue;
      const uint32_t sk = desc_key(pool[live[i]].score);
      if (pass == 0 || (sk >> (shift + 8)) == (sh.pre[g] >> (shift + 8)))
        atomicAdd(&hist[g * 256 + ((sk >> shift) & 255u)], 1u);
    }
    __syncthreads();
    for (int g = warp; g < G; g += NWARPS) {
      if (!sh.active[g]) continue;
      uint32_t c[8];
      int sum = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = hist[g * 256 + lane * 8 + b];
        sum += (int)c[b];
      }
      const int excl = warp_excl_scan(sum, lane);
      const int rem = sh.rem[g];
      int run = excl, fb = -1, fbefore = 0, fcnt = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (fb < 0 && run < rem && rem <= run + (int)c[b]) {
          fb = lane * 8 + b;
          fbefore = run;
          fcnt = (int)c[b];
        }
        run += (int)c[b];
      }
      if (fb >= 0) {
        sh.pre[g] |= (uint32_t)fb << shift;
        sh.rem[g] = rem - fbefore;
        sh.ntie[g] = fcnt;
      }
    }
    __syncthreads();
  }
  // Among the entries of group g whose score key equals pre[g], the B-th is
  // the rem[g]-th smallest prefix key.
  for (int i = tid; i < n_live; i += THREADS) {
    const int g = grp(i);
    if (g < 0 || !sh.active[g]) continue;
    const Entry &e = pool[live[i]];
    if (desc_key(e.score) != sh.pre[g]) continue;
    if (sh.ntie[g] == 1) {
      sh.kg[g][0] = e.g0;
      sh.kg[g][1] = e.g1;
      sh.kg[g][2] = e.g2;
    } else {
      const int k = atomicAdd(&sh.nties, 1);
      if (k < TIE_CAP)
        ties[k] = (uint16_t)i;
      else
        sh.tie_over = 1;
    }
  }
  __syncthreads();
  if (sh.nties > 0) {
    if (!sh.tie_over) {
      const int nt = sh.nties;
      for (int a = tid; a < nt; a += THREADS) {
        const int ia = ties[a];
        const int g = grp(ia);
        const Entry &e = pool[live[ia]];
        int r = 1;
        for (int b = 0; b < nt; ++b) {
          const int ib = ties[b];
          if (grp(ib) != g) continue;
          const Entry &f = pool[live[ib]];
          r += gk_less(f.g0, f.g1, f.g2, e.g0, e.g1, e.g2);
        }
        if (r == sh.rem[g]) {
          sh.kg[g][0] = e.g0;
          sh.kg[g][1] = e.g1;
          sh.kg[g][2] = e.g2;
        }
      }
    } else {
      // many exact score ties: rank against the whole live list
      for (int a = tid; a < n_live; a += THREADS) {
        const int g = grp(a);
        if (g < 0 || !sh.active[g] || sh.ntie[g] == 1) continue;
        const Entry &e = pool[live[a]];
        if (desc_key(e.score) != sh.pre[g]) continue;
        int r = 1;
        for (int b = 0; b < n_live; ++b) {
          if (grp(b) != g) continue;
          const Entry &f = pool[live[b]];
          if (desc_key(f.score) != sh.pre[g]) continue;
          r += gk_less(f.g0, f.g1, f.g2, e.g0, e.g1, e.g2);
        }
        if (r == sh.rem[g]) {
          sh.kg[g][0] = e.g0;
          sh.kg[g][1] = e.g1;
          sh.kg[g][2] = e.g2;
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    Key best{0xFFFFFFFFu, ~0ull, ~0ull, ~0ull};
    bool have = false;
    for (int g = 0; g < G; ++g) {
      if (!sh.active[g]) continue;
      const Key k{sh.pre[g], sh.kg[g][0], sh.kg[g][1], sh.kg[g][2]};
      if (!have || key_before(k, best)) {
        best = k;
        have = true;
      }
    }
    sh.kappa = best;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(THREADS, 1) build_tree_kernel(const Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Shared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = blockIdx.x;
  const int K = P.K, L = P.L, topk = P.topk, B = P.B;
  const int KT = K * topk;
  const int KLT = K * L * topk;
  const int cap = P.cap, tsize = P.tsize;
  const Layout lay = make_layout(K, L, topk, B, cap, tsize);
  Entry *pool = reinterpret_cast<Entry *>(smem + lay.pool);
  uint16_t *livebuf[2] = {reinterpret_cast<uint16_t *>(smem + lay.live0),
                          reinterpret_cast<uint16_t *>(smem + lay.live1)};
  uint16_t *freel = reinterpret_cast<uint16_t *>(smem + lay.freel);
  int16_t *nodeof = reinterpret_cast<int16_t *>(smem + lay.nodeof);
  uint16_t *hslot = reinterpret_cast<uint16_t *>(smem + lay.hslot);
  uint8_t *alive = smem + lay.alive;
  float *lp_s = reinterpret_cast<float *>(smem + lay.lp);
  uint16_t *gam_s = reinterpret_cast<uint16_t *>(smem + lay.gam);
  uint32_t *hist = reinterpret_cast<uint32_t *>(smem + lay.table);
  uint64_t *tag = reinterpret_cast<uint64_t *>(smem + lay.table);
  uint64_t *best = tag + tsize;
  uint32_t *hist1 = reinterpret_cast<uint32_t *>(smem + lay.hist1);
  uint16_t *ties = reinterpret_cast<uint16_t *>(smem + lay.ties);
  int16_t *par_s = reinterpret_cast<int16_t *>(smem + lay.par);
  uint16_t *nslot = reinterpret_cast<uint16_t *>(smem + lay.nslot);

  const float *glp = P.tk_logp + (size_t)q * KLT;
  const int32_t *gtk = P.tk_tok + (size_t)q * KLT;
  int32_t *U = P.union_ws + (size_t)q * 16 * 512;

  // ---------------------------------------------------- 0: tables, checks
  if (tid == 0) sh.bad = 0;
  __syncthreads();
  for (int e = tid; e < KLT; e += THREADS) {
    const float v = glp[e];
    lp_s[e] = v;
    const int j = e % topk;
    if (isnan(v) || v > 0.f || (j > 0 && !(glp[e - 1] >= v))) sh.bad = 1;
  }
  __syncthreads();

  // ---------------------------------------------------- 1: token unions
  {
    int up2 = 32;
    while (up2 < KT) up2 <<= 1;
    uint64_t *scratch = reinterpret_cast<uint64_t *>(smem + lay.pool);
    for (int i = warp; i < L; i += NWARPS) {
      uint64_t *arr = scratch + (size_t)warp * up2;
      for (int e = lane; e < up2; e += 32) {
        if (e < KT) {
          const int k = e / topk, j = e % topk;
          const uint32_t tk = (uint32_t)gtk[((size_t)k * L + i) * topk + j];
          arr[e] = ((uint64_t)tk << 32) | ((uint64_t)k << 16) | (uint64_t)j;
        } else {
          arr[e] = ~0ull;
        }
      }
      __syncwarp();
      for (int size = 2; size <= up2; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int e = lane; e < up2 / 2; e += 32) {
            const int lo = 2 * stride * (e / stride) + (e % stride), hi = lo + stride;
            const bool asc = (lo & size) == 0;
            const uint64_t a = arr[lo], b = arr[hi];
            if ((a > b) == asc) {
              arr[lo] = b;
              arr[hi] = a;
            }
          }
          __syncwarp();
        }
      const int seg = up2 / 32, beg = lane * seg;
      int cnt = 0;
      for (int e = beg; e < beg + seg; ++e)
        if (e < KT && (e == 0 || (arr[e] >> 32) != (arr[e - 1] >> 32))) ++cnt;
      int g = warp_excl_scan(cnt, lane) - 1;
      for (int e = beg; e < beg + seg && e < KT; ++e) {
        const uint64_t x = arr[e];
        const bool isnew = (e == 0) || ((x >> 32) != (arr[e - 1] >> 32));
        if (isnew) {
          ++g;
          U[i * 512 + g] = (int32_t)(uint32_t)(x >> 32);
        } else if (((arr[e - 1] >> 16) & 0xFFFF) == ((x >> 16) & 0xFFFF)) {
          sh.bad = 1;  // a token twice in one row
        }
        const int k = (int)((x >> 16) & 0xFFFF), j = (int)(x & 0xFFFF);
        gam_s[((size_t)k * L + i) * topk + j] = (uint16_t)g;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (sh.bad) {
    if (tid == 0) report(P.status, MFD_ERR_INPUT);
    return;
  }

  // ---------------------------------------------------- 2: depth-1 entries
  if (tid == 0) {
    sh.n_live = 0;
    sh.tail = 0;
    sh.nfree = 0;
    sh.free_used = 0;
    sh.cur = 0;
  }
  __syncthreads();
  for (int e = tid; e < KT; e += THREADS) {
    const int k = e / topk, j = e % topk;
    const float v = lp_s[((size_t)k * L) * topk + j];
    if (v == -INFINITY) continue;
    Entry en;
    en.g0 = (uint64_t)gam_s[((size_t)k * L) * topk + j] << 54;
    en.g1 = 0;
    en.g2 = 1;
    en.score = v;
    en.mode = (uint8_t)k;
    en.depth = 1;
    en.next_j = 0;
    en.pad = 0;
    const int slot = atomicAdd(&sh.tail, 1);
    pool[slot] = en;
    livebuf[0][atomicAdd(&sh.n_live, 1)] = (uint16_t)slot;
  }
  __syncthreads();

  // prune to the current kappa and rebuild the free list
  auto prune = [&]() {
    uint16_t *live = livebuf[sh.cur];
    uint16_t *nlive = livebuf[sh.cur ^ 1];
    const int n_live = sh.n_live, tail = sh.tail;
    const bool hk = sh.has_kappa;
    const Key kap = sh.kappa;
    for (int i = tid; i < tail; i += THREADS) alive[i] = 0;
    if (tid == 0) {
      sh.n_new = 0;
      sh.nfree = 0;
      sh.free_used = 0;
    }
    __syncthreads();
    for (int i = tid; i < n_live; i += THREADS) {
      const int slot = live[i];
      if (!hk || !key_before(kap, key_of(pool[slot]))) {
        alive[slot] = 1;
        nlive[atomicAdd(&sh.n_new, 1)] = (uint16_t)slot;
      }
    }
    __syncthreads();
    for (int i = tid; i < tail; i += THREADS)
      if (!alive[i]) freel[atomicAdd(&sh.nfree, 1)] = (uint16_t)i;
    __syncthreads();
    if (tid == 0) {
      sh.cur ^= 1;
      sh.n_live = sh.n_new;
    }
    __syncthreads();
  };

  auto kappa_by_mode = [&]() {
    const uint16_t *live = livebuf[sh.cur];
    select_bth(sh, pool, live, sh.n_live, K, B, hist, ties, [&](int i) { return (int)pool[live[i]].mode; });
  };

  // ---------------------------------------------------- 3: level expansion
  for (int t = 1; t < L; ++t) {
    if (tid == 0) sh.any_child = 0;
    int pass = 0;
    for (; pass < MAX_PASSES; ++pass) {
      kappa_by_mode();
      prune();
      if (tid == 0) sh.overflow = 0;
      __syncthreads();
      uint16_t *live = livebuf[sh.cur];
      const int n0 = sh.n_live;
      const bool hk = sh.has_kappa;
      const Key kap = sh.kappa;
      for (int i = tid; i < n0; i += THREADS) {
        const int slot = live[i];
        const Entry e = pool[slot];
        if (e.depth != t || e.next_j >= topk) continue;
        const int k = e.mode;
        const float *lprow = lp_s + ((size_t)k * L + t) * topk;
        const uint16_t *grow = gam_s + ((size_t)k * L + t) * topk;
        int j = e.next_j;
        while (j < topk) {
          const float lv = lprow[j];
          if (lv == -INFINITY) {
            j = topk;
            break;
          }
          const float cs = __fadd_rn(e.score, lv);
          uint64_t c0 = e.g0, c1 = e.g1, c2 = e.g2;
          gk_set(c0, c1, c2, t + 1, grow[j]);
          gk_set_depth(c2, t + 1);
          if (hk) {
            const uint32_t csk = desc_key(cs);
            if (csk > kap.sk) {
              j = topk;  // every later rank scores no better
              break;
            }
            if (csk == kap.sk && gk_less(kap.g0, kap.g1, kap.g2, c0, c1, c2)) {
              ++j;
              continue;
            }
          }
          int s2 = -1;
          const int f = atomicAdd(&sh.free_used, 1);
          if (f < sh.nfree) {
            s2 = freel[f];
          } else {
            const int tl = atomicAdd(&sh.tail, 1);
            if (tl < cap) s2 = tl;
          }
          if (s2 < 0) {
            sh.overflow = 1;
            break;
          }
          Entry c;
          c.g0 = c0;
          c.g1 = c1;
          c.g2 = c2;
          c.score = cs;
          c.mode = (uint8_t)k;
          c.depth = (uint8_t)(t + 1);
          c.next_j = 0;
          c.pad = 0;
          pool[s2] = c;
          live[atomicAdd(&sh.n_live, 1)] = (uint16_t)s2;
          sh.any_child = 1;
          ++j;
        }
        pool[slot].next_j = (uint8_t)j;
      }
      __syncthreads();
      if (tid == 0 && sh.tail > cap) sh.tail = cap;
      __syncthreads();
      if (!sh.overflow) break;
    }
    if (pass == MAX_PASSES) {
      if (tid == 0) report(P.status, MFD_ERR_TIMEOUT);
      return;
    }
    __syncthreads();
    if (!sh.any_child) break;
  }
  kappa_by_mode();
  prune();

  // ---------------------------------------------------- 4: one entry per prefix
  const uint16_t *live = livebuf[sh.cur];
  const int n_live = sh.n_live;
  uint64_t seed = 0x2545F4914F6CDD1Dull;
  for (int attempt = 0; attempt < 4; ++attempt) {
    for (int i = tid; i < tsize; i += THREADS) {
      tag[i] = 0;
      best[i] = ~0ull;
    }
    if (tid == 0) sh.coll = 0;
    __syncthreads();
    for (int i = tid; i < n_live; i += THREADS) {
      const Entry &e = pool[live[i]];
      const uint64_t h = gk_hash(e.g0, e.g1, e.g2, seed);
      uint32_t s = (uint32_t)h & (uint32_t)(tsize - 1);
      for (int probe = 0; probe < tsize; ++probe) {
        const unsigned long long prev =
            atomicCAS(reinterpret_cast<unsigned long long *>(&tag[s]), 0ull, (unsigned long long)h);
        if (prev == 0ull || prev == h) break;
        s = (s + 1) & (uint32_t)(tsize - 1);
      }
      hslot[i] = (uint16_t)s;
    }
    __syncthreads();
    for (int i = tid; i < n_live; i += THREADS) {
      const Entry &e = pool[live[i]];
      const uint64_t packed = ((uint64_t)desc_key(e.score) << 32) | ((uint64_t)e.mode << 16) | (uint64_t)i;
      atomicMin(reinterpret_cast<unsigned long long *>(&best[hslot[i]]), (unsigned long long)packed);
    }
    __syncthreads();
    for (int i = tid; i < n_live; i += THREADS) {
      const Entry &e = pool[live[i]];
      const Entry &r = pool[live[best[hslot[i]] & 0xFFFF]];
      if (r.g0 != e.g0 || r.g1 != e.g1 || r.g2 != e.g2) sh.coll = 1;
    }
    __syncthreads();
    if (!sh.coll) break;
    seed = mix64(seed + 0x9E3779B97F4A7C15ull);
    __syncthreads();
  }
  if (sh.coll) {
    if (tid == 0) report(P.status, MFD_ERR_UNSUPPORTED);
    return;
  }

  // ---------------------------------------------------- 5: the B best prefixes
  uint8_t *prim = alive;  // reused: prim[i] = live entry i is its prefix's best entry
  for (int i = tid; i < n_live; i += THREADS) prim[i] = (int)(best[hslot[i]] & 0xFFFF) == i;
  for (int i = tid; i < sh.tail; i += THREADS) nodeof[i] = -1;
  __syncthreads();
  select_bth(sh, pool, live, n_live, 1, B, hist1, ties, [&](int i) { return prim[i] ? 0 : -1; });
  uint16_t *sel = livebuf[sh.cur ^ 1];
  {
    const bool hk = sh.has_kappa;
    const Key kap = sh.kappa;
    if (tid == 0) sh.n_sel = 0;
    __syncthreads();
    for (int i = tid; i < n_live; i += THREADS)
      if (prim[i] && (!hk || !key_before(kap, key_of(pool[live[i]])))) sel[atomicAdd(&sh.n_sel, 1)] = live[i];
    __syncthreads();
  }
  const int n = sh.n_sel;  // min(B, number of distinct prefixes in the pool)
  for (int a = tid; a < n; a += THREADS) {
    const Key ka = key_of(pool[sel[a]]);
    int r = 0;
    for (int b = 0; b < n; ++b) r += key_before(key_of(pool[sel[b]]), ka);
    nslot[r + 1] = sel[a];
    nodeof[sel[a]] = (int16_t)(r + 1);
  }
  if (tid == 0) {
    par_s[0] = -1;
    sh.bad = 0;
  }
  __syncthreads();

  // ---------------------------------------------------- 6: parents
  for (int nd = 1 + tid; nd <= n; nd += THREADS) {
    const Entry &e = pool[nslot[nd]];
    const int d = e.depth;
    int par = 0;
    if (d > 1) {
      uint64_t p0 = e.g0, p1 = e.g1, p2 = e.g2;
      gk_set(p0, p1, p2, d, 0);
      gk_set_depth(p2, d - 1);
      const uint64_t h = gk_hash(p0, p1, p2, seed);
      uint32_t s = (uint32_t)h & (uint32_t)(tsize - 1);
      par = -1;
      for (int probe = 0; probe < tsize; ++probe) {
        const uint64_t tg = tag[s];
        if (tg == 0) break;
        if (tg == h) {
          const int ps = live[best[s] & 0xFFFF];
          const Entry &r = pool[ps];
          if (r.g0 == p0 && r.g1 == p1 && r.g2 == p2) {
            par = nodeof[ps];
            break;
          }
        }
        s = (s + 1) & (uint32_t)(tsize - 1);
      }
      if (par < 1 || par >= nd) sh.bad = 1;
    }
    par_s[nd] = (int16_t)par;
  }
  __syncthreads();
  if (sh.bad) {
    if (tid == 0) report(P.status, MFD_ERR_INPUT);
    return;
  }

  // ---------------------------------------------------- 7: outputs
  const int N = B + 1, W32 = (N + 31) / 32;
  const size_t ob = (size_t)q * N;
  const int anchor = P.anchor[q];
  const int bp = P.base_pos ? P.base_pos[q] : 0;
  for (int i = tid; i < N; i += THREADS) {
    int pa = -1, tk = -1, dp = -1, md = -1, ps = -1;
    float sc = -INFINITY;
    if (i == 0) {
      tk = anchor;
      dp = 0;
      sc = 0.f;
      ps = bp;
    } else if (i <= n) {
      const Entry &e = pool[nslot[i]];
      dp = e.depth;
      pa = par_s[i];
      tk = U[(dp - 1) * 512 + (int)gk_get(e.g0, e.g1, e.g2, dp)];
      sc = e.score;
      md = e.mode;
      ps = bp + dp;
    }
    P.parent[ob + i] = pa;
    P.token[ob + i] = tk;
    P.depth[ob + i] = dp;
    P.score[ob + i] = sc;
    P.mode[ob + i] = md;
    P.pos[ob + i] = ps;
  }
  for (int x = tid; x < N * W32; x += THREADS) {
    const int i = x / W32, w = x - (x / W32) * W32;
    uint32_t word = 0;
    if (i <= n)
      for (int a = i; a >= 0; a = (a == 0) ? -1 : par_s[a])
        if ((a >> 5) == w) word |= 1u << (a & 31);
    P.mask[(size_t)q * N * W32 + x] = word;
  }
  if (tid == 0) P.n_nodes[q] = n + 1;
}


int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

size_t tree_smem_bytes(int K, int L, int topk, int B, int *cap_out, int *tsize_out) {
  const int tsize = next_pow2(2 * K * B > 64 ? 2 * K * B : 64);
  const size_t budget = 232448 - sizeof(Shared) - 2048;
  int up2 = 32;
  while (up2 < K * topk) up2 <<= 1;
  const int warps_used = L < NWARPS ? L : NWARPS;
  for (int cap = 4096; cap >= 256; cap -= 128) {
    const Layout y = make_layout(K, L, topk, B, cap, tsize);
    if (y.total > budget) continue;
    if (cap < K * B + K * topk) return 0;
    if ((size_t)warps_used * up2 * 8 > (size_t)cap * 32) return 0;
    *cap_out = cap;
    *tsize_out = tsize;
    return y.total;
  }
  return 0;
}

cudaError_t launch_build_tree(const TreeLaunch &T, cudaStream_t stream) {
  int cap = 0, tsize = 0;
  const size_t bytes = tree_smem_bytes(T.K, T.L, T.topk, T.B, &cap, &tsize);
  if (bytes == 0) return cudaErrorInvalidValue;
  Params p;
  p.tk_logp = T.tk_logp;
  p.tk_tok = T.tk_tok;
  p.K = T.K;
  p.L = T.L;
  p.topk = T.topk;
  p.B = T.B;
  p.anchor = T.anchor;
  p.base_pos = T.base_pos;
  p.parent = T.parent;
  p.token = T.token;
  p.depth = T.depth;
  p.score = T.score;
  p.mode = T.mode;
  p.mask = T.mask;
  p.pos = T.pos;
  p.n_nodes = T.n_nodes;
  p.status = T.status;
  p.union_ws = T.union_ws;
  p.cap = cap;
  p.tsize = tsize;
  cudaError_t e = cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  build_tree_kernel<<<T.n_req, THREADS, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mfd
