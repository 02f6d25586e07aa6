// tree.cu -- the mixture DDTree of one round (project page "Multi-Future
// Drafting", How it works, step 3, and the Figure 1/2 caption): every prefix
// is scored by its best mode; the B best prefixes over all modes form one
// tree, which is the union of the per-mode trees at the common cut-off;
// shared prefixes are built once.
//
// One CTA (512 threads) builds one request's tree in shared memory.
//
// Entries.  The pool holds (mode, prefix) entries scored by their own mode.
// Within one mode a prefix is a tuple of ranks, one per position; replacing
// each rank by its token's rank inside that row (5 bits, token ids compared
// unsigned) turns the lexicographic token order into an unsigned compare of
// packed keys, depth last.  Across modes, prefixes are compared by their
// token ids (looked up through the rows).
//
// Search, level by level.  A per-mode score bound tau_k -- a value with at
// least B of mode k's entries scoring no worse -- comes from a two-digit
// radix select on the score key.  Each mode's entries are distinct
// prefixes and a prefix's mixture score is at least its mode score, so at
// least B distinct prefixes score no worse than min_k tau_k: the tree's
// cut-off is never worse, and every entry that can reach the tree, or lead
// to it, scores within the bound.  Level t expands the depth-t entries in
// rank order (child scores only fall) while the child is within the bound.
// When the pool fills, it is pruned to each mode's exact B best (radix
// select on the full score key, then the token order among equal scores)
// and expansion resumes where each entry stopped.
//
// Result.  The entries within the final bound are hashed by token sequence;
// a table keeps per sequence the entry with the best (score, smallest mode),
// equality checked on the full sequence (a collision reseeds the table).
// These primaries are distinct prefixes.  A radix bound over the primaries
// leaves about B of them; rank counting among those gives both the B best
// and their order.  Parents are looked up in the table by the hash of the
// sequence without its last token.
#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int THREADS = 512;
constexpr int NWARPS = THREADS / 32;
constexpr int MAX_PASSES = 64;
constexpr int PLIST = 1024;     // parents listed for pair-parallel expansion
constexpr int PAIR_MAX = 4096;  // (parent, rank) pairs expanded at once

// Pool entry (16 bytes).  k0: row ranks of positions 1..12, 5 bits each,
// position 1 highest (bits 59..55).  k1: depth at bits 4..0, positions
// 13..16 at bits 24..5, mode at bits 28..25.
struct PE {
  float score;
  uint32_t k1;
  uint64_t k0;
};
static_assert(sizeof(PE) == 16, "pool entry");

constexpr uint32_t K1_KEY = 0x01FFFFFFu;  // depth and positions 13..16

__device__ __forceinline__ void pk_set(uint64_t &k0, uint32_t &k1, int p, uint32_t s) {
  if (p <= 12) {
    const int sh = 55 - 5 * (p - 1);
    k0 = (k0 & ~((uint64_t)31 << sh)) | ((uint64_t)(s & 31u) << sh);
  } else {
    const int sh = 20 - 5 * (p - 13);
    k1 = (k1 & ~(31u << sh)) | ((s & 31u) << sh);
  }
}
__device__ __forceinline__ uint32_t pk_get(uint64_t k0, uint32_t k1, int p) {
  return p <= 12 ? (uint32_t)(k0 >> (55 - 5 * (p - 1))) & 31u : (k1 >> (20 - 5 * (p - 13))) & 31u;
}
__device__ __forceinline__ int pk_depth(uint32_t k1) { return (int)(k1 & 31u); }
__device__ __forceinline__ int pk_mode(uint32_t k1) { return (int)((k1 >> 25) & 15u); }

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  x ^= x >> 30;
  x *= 0xBF58476D1CE4E5B9ull;
  x ^= x >> 27;
  x *= 0x94D049BB133111EBull;
  x ^= x >> 31;
  return x;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
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

// Lanes hitting the same bin are merged first: one atomic per bin per warp.
__device__ __forceinline__ void warp_hist_add(int *hist, int bin) {
  const unsigned m = __match_any_sync(0xffffffffu, bin);
  if (bin >= 0 && (int)(threadIdx.x & 31) == __ffs(m) - 1) atomicAdd(&hist[bin], __popc(m));
}

// Warp-aggregated append: one atomic per warp; this lane's index or -1.
__device__ __forceinline__ int warp_append(int *ctr, bool pred) {
  const unsigned m = __ballot_sync(0xffffffffu, pred);
  if (m == 0) return -1;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if ((int)(threadIdx.x & 31) == leader) base = atomicAdd(ctr, __popc(m));
  base = __shfl_sync(0xffffffffu, base, leader);
  return pred ? base + __popc(m & lanemask_lt()) : -1;
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
  int cap;    // pool entries
  int nc;     // candidates hashed at the end
  int tsize;  // hash table slots (power of two)
};

struct Layout {
  size_t lp, tok, sig, inv, ent, nxt, flg, table, hist1, skk, sel, prim, hslot, nodeid, par, nslot, plist, total;
};

__host__ __device__ inline size_t al16(size_t o) { return (o + 15) & ~(size_t)15; }

__host__ __device__ inline Layout make_layout(int K, int L, int topk, int B, int cap, int nc, int tsize) {
  Layout y;
  size_t o = 0;
  const size_t klt = (size_t)K * L * topk;
  const size_t hist = (size_t)16 * 256 * 4, tbl = al16((size_t)tsize * 4) + (size_t)tsize * 8;
  y.ent = o;
  o += (size_t)cap * 16;
  y.table = o = al16(o);  // hash tags then best entries; the radix histograms overlay it
  o += hist > tbl ? hist : tbl;
  y.hist1 = o = al16(o);
  o += 256 * 4;
  y.lp = o = al16(o);
  o += klt * 4;
  y.tok = o = al16(o);
  o += klt * 4;
  y.skk = o = al16(o);
  o += (size_t)(nc + 4) * 4;  // padded to whole 16-byte words
  y.sel = o = al16(o);
  o += (size_t)nc * 2;
  y.hslot = o = al16(o);
  o += (size_t)nc * 2;
  y.nodeid = o = al16(o);
  o += (size_t)nc * 2;
  y.par = o = al16(o);
  o += (size_t)(B + 1) * 2;
  y.plist = o = al16(o);
  o += (size_t)PLIST * 2;
  y.nslot = o = al16(o);
  o += (size_t)(B + 1) * 2;
  y.nxt = o = al16(o);
  o += (size_t)cap;
  y.flg = o = al16(o);
  o += (size_t)cap;
  y.sig = o = al16(o);
  o += klt;
  y.inv = o = al16(o);
  o += klt;
  y.prim = o = al16(o);
  o += (size_t)nc;
  y.total = (o + 127) & ~(size_t)127;
  return y;
}

struct Shared {
  int n_ent, overflow, any, bad, coll, n_prim, n_sel, has_tau, n_par, wsum[NWARPS];
  int cnt[16], act[16], rem[16], ntie[16];
  uint32_t pre[16], tau;
};

struct Ctx {
  const float *lp;
  const int32_t *tok;
  const uint8_t *sig, *inv;
  int K, L, topk;
};

// token at position p (1-based) of an entry
__device__ __forceinline__ uint32_t token_at(const Ctx &c, const PE &e, int p) {
  const int row = (pk_mode(e.k1) * c.L + p - 1) * c.topk;
  return (uint32_t)c.tok[row + c.inv[row + pk_get(e.k0, e.k1, p)]];
}

// Token order of two prefixes of any modes (unsigned ids, a proper prefix
// first): <0, 0, >0.
__device__ int seq_cmp(const Ctx &c, const PE &a, const PE &b) {
  const int da = pk_depth(a.k1), db = pk_depth(b.k1);
  const int d = da < db ? da : db;
  for (int p = 1; p <= d; ++p) {
    const uint32_t ta = token_at(c, a, p), tb = token_at(c, b, p);
    if (ta != tb) return ta < tb ? -1 : 1;
  }
  return da - db;
}

__device__ __forceinline__ uint64_t seq_hash(const Ctx &c, const PE &e, int d, uint64_t seed) {
  uint64_t h = 0x2545F4914F6CDD1Dull ^ seed;
  for (int p = 1; p <= d; ++p) h = mix64(h ^ ((uint64_t)token_at(c, e, p) + ((uint64_t)p << 40)));
  return h;
}

// Per group g (grp(i) in [0, G), or -1 to skip), with at least B members
// among ent[0, n): digits of the B-th best score key, most significant
// first, over `passes` 8-bit passes.  Leaves sh.act[g], sh.pre[g] (the digits
// found, low bits zero), sh.rem[g] (rank of the B-th within that prefix) and
// sh.ntie[g] (members sharing the prefix).
template <typename GroupFn>
__device__ void radix_bound(Shared &sh, const PE *ent, int n, int G, int B, int passes, int *hist, GroupFn grp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 16) {
    sh.pre[tid] = 0;
    sh.rem[tid] = B;
    sh.ntie[tid] = 0;
    sh.act[tid] = tid < G;  // until the first pass has counted the group
  }
  for (int i = tid; i < G * 256; i += THREADS) hist[i] = 0;
  __syncthreads();
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 24 - 8 * pass;
    if (pass > 0) {
      for (int i = tid; i < G * 256; i += THREADS) hist[i] = 0;
      __syncthreads();
    }
    for (int base = warp * 32; base < n; base += THREADS) {
      const int i = base + lane;
      int bin = -1;
      if (i < n) {
        const int g = grp(i);
        if (g >= 0 && sh.act[g]) {
          const uint32_t sk = desc_key(ent[i].score);
          if (pass == 0 || (sk >> (shift + 8)) == (sh.pre[g] >> (shift + 8))) bin = g * 256 + (int)((sk >> shift) & 255u);
        }
      }
      warp_hist_add(hist, bin);
    }
    __syncthreads();
    for (int g = warp; g < G; g += NWARPS) {
      if (!sh.act[g]) continue;
      int c[8], sum = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = hist[g * 256 + lane * 8 + b];
        sum += c[b];
      }
      int run = warp_excl_scan(sum, lane);
      if (pass == 0) {
        const int total = __shfl_sync(0xffffffffu, run + sum, 31);
        if (total < B) {
          if (lane == 0) sh.act[g] = 0;
          continue;
        }
      }
      const int rem = sh.rem[g];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (run < rem && rem <= run + c[b]) {
          sh.pre[g] |= (uint32_t)(lane * 8 + b) << shift;
          sh.rem[g] = rem - run;
          sh.ntie[g] = c[b];
        }
        run += c[b];
      }
    }
    __syncthreads();
  }
}

// In-place stable compaction of ent/nxt[0, n) to the entries with keep(i).
template <typename KeepFn>
__device__ int block_compact(Shared &sh, PE *ent, uint8_t *nxt, int n, KeepFn keep) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int out = 0;
  for (int base = 0; base < n; base += THREADS) {
    const int i = base + tid;
    PE e;
    uint8_t nx = 0;
    bool kp = false;
    if (i < n) {
      e = ent[i];
      nx = nxt[i];
      kp = keep(i);
    }
    const unsigned m = __ballot_sync(0xffffffffu, kp);
    if (lane == 0) sh.wsum[warp] = __popc(m);
    __syncthreads();
    int woff = 0, tot = 0;
    for (int w = 0; w < NWARPS; ++w) {
      const int v = sh.wsum[w];
      woff += w < warp ? v : 0;
      tot += v;
    }
    if (kp) {
      const int d = out + woff + __popc(m & lanemask_lt());
      ent[d] = e;
      nxt[d] = nx;
    }
    out += tot;
    __syncthreads();
  }
  return out;
}

__global__ void __launch_bounds__(THREADS, 1) build_tree_kernel(const Params prm) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Shared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = blockIdx.x;
  const int K = prm.K, L = prm.L, topk = prm.topk, B = prm.B, CAP = prm.cap, NC = prm.nc, tsize = prm.tsize;
  const int KLT = K * L * topk;
  const Layout lay = make_layout(K, L, topk, B, CAP, NC, tsize);
  float *lp_s = reinterpret_cast<float *>(smem + lay.lp);
  int32_t *tok_s = reinterpret_cast<int32_t *>(smem + lay.tok);
  uint8_t *sig_s = smem + lay.sig;
  uint8_t *inv_s = smem + lay.inv;
  PE *ent = reinterpret_cast<PE *>(smem + lay.ent);
  uint8_t *nxt = smem + lay.nxt;
  uint8_t *flg = smem + lay.flg;
  int *hist1 = reinterpret_cast<int *>(smem + lay.hist1);
  uint32_t *tag = reinterpret_cast<uint32_t *>(smem + lay.table);
  uint64_t *best = reinterpret_cast<uint64_t *>(smem + lay.table + al16((size_t)tsize * 4));
  int *hist = reinterpret_cast<int *>(smem + lay.table);
  uint32_t *skk = reinterpret_cast<uint32_t *>(smem + lay.skk);
  uint16_t *sel = reinterpret_cast<uint16_t *>(smem + lay.sel);
  uint16_t *hslot = reinterpret_cast<uint16_t *>(smem + lay.hslot);
  int16_t *nodeid = reinterpret_cast<int16_t *>(smem + lay.nodeid);
  uint8_t *prim = smem + lay.prim;
  int16_t *par_s = reinterpret_cast<int16_t *>(smem + lay.par);
  uint16_t *nslot = reinterpret_cast<uint16_t *>(smem + lay.nslot);
  uint16_t *plist = reinterpret_cast<uint16_t *>(smem + lay.plist);

  const float *glp = prm.tk_logp + (size_t)q * KLT;
  const int32_t *gtk = prm.tk_tok + (size_t)q * KLT;
  pdl_wait();  // the tables may come from the grid launched just before
  pdl_launch_dependents();

  // ---------------------------------------------------- tables and checks
  if (tid == 0) {
    sh.bad = 0;
    sh.n_ent = 0;
  }
  __syncthreads();
  for (int e = tid; e < KLT; e += THREADS) {
    const float v = glp[e];
    lp_s[e] = v;
    tok_s[e] = gtk[e];
    const int j = e % topk;
    if (isnan(v) || v > 0.f || (j > 0 && !(glp[e - 1] >= v))) sh.bad = 1;
  }
  __syncthreads();
  for (int e = tid; e < KLT; e += THREADS) {
    const int j = e % topk, row = e - j;
    const uint32_t me = (uint32_t)tok_s[e];
    int s = 0, dup = 0;
    for (int f = 0; f < topk; ++f) {
      const uint32_t o = (uint32_t)tok_s[row + f];
      s += o < me;
      dup += (o == me) && f != j;
    }
    if (dup) sh.bad = 1;
    sig_s[e] = (uint8_t)s;
    inv_s[row + s] = (uint8_t)j;
  }
  __syncthreads();
  if (sh.bad) {
    if (tid == 0) report(prm.status, MFD_ERR_INPUT);
    return;
  }
  const Ctx c{lp_s, tok_s, sig_s, inv_s, K, L, topk};
  auto mode_of = [&](int i) { return pk_mode(ent[i].k1); };

  // ---------------------------------------------------- depth-1 entries
  for (int base = warp * 32; base < K * topk; base += THREADS) {
    const int e = base + lane;
    const int k = e / topk, j = e - (e / topk) * topk;
    const bool ok = e < K * topk && lp_s[(k * L) * topk + j] > -INFINITY;
    const int slot = warp_append(&sh.n_ent, ok);
    if (ok) {
      PE en;
      en.score = lp_s[(k * L) * topk + j];
      en.k0 = 0;
      en.k1 = 1u | ((uint32_t)k << 25);
      pk_set(en.k0, en.k1, 1, sig_s[(k * L) * topk + j]);
      ent[slot] = en;
      nxt[slot] = 0;
    }
  }
  __syncthreads();

  // the best (smallest) per-mode bound into sh.tau / sh.has_tau
  auto set_tau = [&](int passes) {
    radix_bound(sh, ent, sh.n_ent, K, B, passes, hist, mode_of);
    if (tid == 0) {
      uint32_t t = 0xFFFFFFFFu;
      int h = 0;
      for (int k = 0; k < K; ++k)
        if (sh.act[k]) {
          const uint32_t tk = sh.pre[k] | (passes >= 4 ? 0u : (0xFFFFFFFFu >> (8 * passes)));
          if (!h || tk < t) t = tk;
          h = 1;
        }
      sh.tau = t;
      sh.has_tau = h;
    }
    __syncthreads();
  };

  // prune to each mode's exact B best (only when the pool is full)
  auto prune_exact = [&]() {
    radix_bound(sh, ent, sh.n_ent, K, B, 4, hist, mode_of);
    const int n = sh.n_ent;
    // among a mode's entries tied at its B-th score, keep the first rem[k]
    // in token order; decided for every entry before any entry moves
    for (int i = tid; i < n; i += THREADS) {
      const PE e = ent[i];
      const int k = pk_mode(e.k1);
      bool kp = true;
      if (sh.act[k]) {
        const uint32_t sk = desc_key(e.score);
        if (sk != sh.pre[k]) {
          kp = sk < sh.pre[k];
        } else if (sh.ntie[k] != sh.rem[k]) {
          int r = 1;
          for (int f = 0; f < n; ++f) {
            const PE g = ent[f];
            if (pk_mode(g.k1) != k || desc_key(g.score) != sh.pre[k]) continue;
            r += (g.k0 < e.k0) || (g.k0 == e.k0 && (g.k1 & K1_KEY) < (e.k1 & K1_KEY));
          }
          kp = r <= sh.rem[k];
        }
      }
      flg[i] = kp;
    }
    __syncthreads();
    const int out = block_compact(sh, ent, nxt, n, [&](int i) { return flg[i] != 0; });
    if (tid == 0) sh.n_ent = out;
    __syncthreads();
  };

  // ---------------------------------------------------- level expansion
  bool failed = false, tau_current = false;
  for (int t = 1; t < L && !failed; ++t) {
    if (tid == 0) sh.any = 0;
    int pass = 0;
    for (; pass < MAX_PASSES; ++pass) {
      if (t == 1 && pass == 0 && topk < B) {
        if (tid == 0) sh.has_tau = 0;  // each mode holds only its topk depth-1 entries
      } else {
        set_tau(2);
      }
      tau_current = true;
      if (tid == 0) {
        sh.overflow = 0;
        sh.n_par = 0;
      }
      __syncthreads();
      const int n0 = sh.n_ent;
      const bool ht = sh.has_tau;
      const uint32_t tau = sh.tau;
      // the parents of this level that can still reach the bound
      for (int base = warp * 32; base < n0; base += THREADS) {
        const int i = base + lane;
        bool isp = false;
        if (i < n0) {
          const PE e = ent[i];
          isp = pk_depth(e.k1) == t && nxt[i] < topk && (!ht || desc_key(e.score) <= tau);
        }
        const int k = warp_append(&sh.n_par, isp);
        if (isp && k < PLIST) plist[k] = (uint16_t)i;
      }
      __syncthreads();
      const int np = sh.n_par;
      if (np <= PLIST && np * topk <= PAIR_MAX && n0 + np * topk <= CAP) {
        // few parents and room for every child: all (parent, rank) pairs at once
        for (int base = warp * 32; base < np * topk; base += THREADS) {
          const int x = base + lane;
          bool want = false;
          PE ch;
          if (x < np * topk) {
            const int i = plist[x / topk], j = x - (x / topk) * topk;
            const PE par = ent[i];
            const int row = (pk_mode(par.k1) * L + t) * topk;
            const float lv = lp_s[row + j];
            if (j >= nxt[i] && lv > -INFINITY) {
              ch.score = __fadd_rn(par.score, lv);
              if (!ht || desc_key(ch.score) <= tau) {
                ch.k0 = par.k0;
                ch.k1 = par.k1 & ~31u;
                pk_set(ch.k0, ch.k1, t + 1, sig_s[row + j]);
                ch.k1 |= (uint32_t)(t + 1);
                want = true;
              }
            }
          }
          const int slot = warp_append(&sh.n_ent, want);
          if (want) {
            ent[slot] = ch;
            nxt[slot] = 0;
          }
        }
        __syncthreads();
        for (int pi = tid; pi < np; pi += THREADS) nxt[plist[pi]] = (uint8_t)topk;
      } else {
        for (int base = warp * 32; base < n0; base += THREADS) {
          const int i = base + lane;
          PE par{0.f, 0u, 0ull};
          bool isp = false, act = false;
          int j = 0;
          if (i < n0) {
            par = ent[i];
            j = nxt[i];
            isp = pk_depth(par.k1) == t && j < topk && (!ht || desc_key(par.score) <= tau);
            act = isp;
          }
          const int row = (pk_mode(par.k1) * L + t) * topk;
          while (__any_sync(0xffffffffu, act)) {
            bool want = false;
            PE ch;
            if (act) {
              const float lv = lp_s[row + j];
              if (!(lv > -INFINITY)) {
                act = false;
                j = topk;
              } else {
                ch.score = __fadd_rn(par.score, lv);
                if (ht && desc_key(ch.score) > tau) {
                  act = false;  // every later rank scores no better
                  j = topk;
                } else {
                  ch.k0 = par.k0;
                  ch.k1 = par.k1 & ~31u;
                  pk_set(ch.k0, ch.k1, t + 1, sig_s[row + j]);
                  ch.k1 |= (uint32_t)(t + 1);
                  want = true;
                }
              }
            }
            const int slot = warp_append(&sh.n_ent, want);
            if (want) {
              if (slot < CAP) {
                ent[slot] = ch;
                nxt[slot] = 0;
                ++j;
                if (j >= topk) act = false;
              } else {
                act = false;  // j kept: resumed after the pool is pruned
                sh.overflow = 1;
              }
            }
          }
          if (isp) nxt[i] = (uint8_t)j;
        }
      }
      __syncthreads();
      if (tid == 0) {
        if (sh.n_ent > CAP) sh.n_ent = CAP;
        if (sh.n_ent > n0) sh.any = 1;
      }
      __syncthreads();
      if (sh.any) tau_current = false;
      if (!sh.overflow) break;
      prune_exact();
    }
    if (pass == MAX_PASSES) failed = true;
    if (!sh.any) break;
  }
  if (failed) {
    if (tid == 0) report(prm.status, MFD_ERR_UNSUPPORTED);
    return;
  }

  // ---------------------------------------------------- candidates
  if (!tau_current) set_tau(2);  // else: nothing was added since the last bound
  {
    const bool ht = sh.has_tau;
    const uint32_t tau = sh.tau;
    const int n = block_compact(sh, ent, nxt, sh.n_ent, [&](int i) { return !ht || desc_key(ent[i].score) <= tau; });
    if (tid == 0) sh.n_ent = n;
    __syncthreads();
  }
  if (sh.n_ent > NC) {  // many ties within the bound: keep each mode's exact B best
    prune_exact();
    if (sh.n_ent > NC) {
      if (tid == 0) report(prm.status, MFD_ERR_UNSUPPORTED);
      return;
    }
  }
  const int n = sh.n_ent;

  // ---------------------------------------------------- one entry per prefix
  uint64_t seed = 0;
  for (int attempt = 0; attempt < 4; ++attempt) {
    for (int s = tid; s < tsize; s += THREADS) {
      tag[s] = 0;
      best[s] = ~0ull;
    }
    if (tid == 0) sh.coll = 0;
    __syncthreads();
    for (int i = tid; i < n; i += THREADS) {
      const uint64_t h = seq_hash(c, ent[i], pk_depth(ent[i].k1), seed);
      const uint32_t tg = (uint32_t)(h >> 32) | 1u;
      uint32_t s = (uint32_t)h & (uint32_t)(tsize - 1);
      for (int probe = 0; probe < tsize; ++probe) {
        const uint32_t prev = atomicCAS(&tag[s], 0u, tg);
        if (prev == 0u || prev == tg) break;
        s = (s + 1) & (uint32_t)(tsize - 1);
      }
      hslot[i] = (uint16_t)s;
      const uint64_t packed = ((uint64_t)desc_key(ent[i].score) << 32) | ((uint64_t)pk_mode(ent[i].k1) << 16) | i;
      atomicMin(reinterpret_cast<unsigned long long *>(&best[s]), (unsigned long long)packed);
    }
    __syncthreads();
    for (int i = tid; i < n; i += THREADS) {
      const int r = (int)(best[hslot[i]] & 0xFFFF);
      if (r != i && seq_cmp(c, ent[i], ent[r]) != 0) sh.coll = 1;
    }
    __syncthreads();
    if (!sh.coll) break;
    seed = mix64(seed + 0x9E3779B97F4A7C15ull);
    __syncthreads();
  }
  if (sh.coll) {
    if (tid == 0) report(prm.status, MFD_ERR_UNSUPPORTED);
    return;
  }
  for (int i = tid; i < n; i += THREADS) {
    prim[i] = (int)(best[hslot[i]] & 0xFFFF) == i;
    nodeid[i] = -1;
  }
  __syncthreads();

  // ---------------------------------------------------- the B best prefixes
  radix_bound(sh, ent, n, 1, B, 2, hist1, [&](int i) { return prim[i] ? 0 : -1; });
  if (tid == 0) sh.n_sel = 0;
  __syncthreads();
  {
    const bool ht = sh.act[0];
    const uint32_t tau = sh.pre[0] | 0xFFFFu;
    for (int base = warp * 32; base < n; base += THREADS) {
      const int i = base + lane;
      const bool in = i < n && prim[i] && (!ht || desc_key(ent[i].score) <= tau);
      const int k = warp_append(&sh.n_sel, in);
      if (in) {
        sel[k] = (uint16_t)i;
        skk[k] = desc_key(ent[i].score);
      }
    }
  }
  __syncthreads();
  const int ns = sh.n_sel;
  const int ns4 = (ns + 3) & ~3;
  for (int b = ns + tid; b < ns4; b += THREADS) skk[b] = 0xFFFFFFFFu;  // never before a real key
  __syncthreads();
  // rank of each selected prefix = how many others come before it: score
  // keys first (four per load, two threads per prefix, each half of the
  // keys), then token order for the rare equal scores
  {
    const uint4 *s4 = reinterpret_cast<const uint4 *>(skk);
    const int nw = ns4 >> 2, h4 = nw >> 1;  // words of four keys; the first half
    for (int base = warp * 32; base < 2 * ns; base += THREADS) {
      const int a2 = base + lane;
      const bool valid = a2 < 2 * ns;
      const int a = valid ? a2 >> 1 : 0, half = a2 & 1;
      int lt = 0;
      if (valid) {
        const uint32_t ka = skk[a];
        const int w0 = half ? h4 : 0, w1 = half ? nw : h4;
        int eq = 0;
        for (int w = w0; w < w1; ++w) {
          const uint4 v = s4[w];
          lt += (v.x < ka) + (v.y < ka) + (v.z < ka) + (v.w < ka);
          eq += (v.x == ka) + (v.y == ka) + (v.z == ka) + (v.w == ka);
        }
        const int self = (a >= 4 * w0 && a < 4 * w1) ? 1 : 0;
        if (eq > self) {  // another prefix has the same score key
          const PE ea = ent[sel[a]];
          for (int b = 4 * w0; b < 4 * w1 && b < ns; ++b)
            if (b != a && skk[b] == ka && seq_cmp(c, ent[sel[b]], ea) < 0) ++lt;
        }
      }
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      if (valid && half == 0 && lt < B) {
        nslot[lt + 1] = sel[a];
        nodeid[sel[a]] = (int16_t)(lt + 1);
      }
    }
  }
  if (tid == 0) {
    par_s[0] = -1;
    sh.bad = 0;
  }
  __syncthreads();
  const int nn = ns < B ? ns : B;

  // ---------------------------------------------------- parents
  for (int nd = 1 + tid; nd <= nn; nd += THREADS) {
    const int i = nslot[nd];
    const PE e = ent[i];
    const int d = pk_depth(e.k1);
    int par = 0;
    if (d > 1) {
      par = -1;
      const uint64_t h = seq_hash(c, e, d - 1, seed);
      const uint32_t tg = (uint32_t)(h >> 32) | 1u;
      uint32_t s = (uint32_t)h & (uint32_t)(tsize - 1);
      for (int probe = 0; probe < tsize && par < 0; ++probe) {
        const uint32_t t0 = tag[s];
        if (t0 == 0u) break;
        if (t0 == tg) {
          const int r = (int)(best[s] & 0xFFFF);
          const PE g = ent[r];
          if (pk_depth(g.k1) == d - 1) {
            bool same = true;
            for (int p = 1; p < d && same; ++p) same = token_at(c, g, p) == token_at(c, e, p);
            if (same) par = nodeid[r];
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
    if (tid == 0) report(prm.status, MFD_ERR_INPUT);
    return;
  }

  // ---------------------------------------------------- outputs
  const int N = B + 1, W32 = (N + 31) / 32;
  const size_t ob = (size_t)q * N;
  const int anchor = prm.anchor[q];
  const int bp = prm.base_pos ? prm.base_pos[q] : 0;
  for (int nd = tid; nd < N; nd += THREADS) {
    int pa = -1, tk = -1, dp = -1, md = -1, ps = -1;
    float sc = -INFINITY;
    if (nd == 0) {
      tk = anchor;
      dp = 0;
      sc = 0.f;
      ps = bp;
    } else if (nd <= nn) {
      const PE e = ent[nslot[nd]];
      dp = pk_depth(e.k1);
      pa = par_s[nd];
      tk = (int)token_at(c, e, dp);
      sc = e.score;
      md = pk_mode(e.k1);
      ps = bp + dp;
    }
    prm.parent[ob + nd] = pa;
    prm.token[ob + nd] = tk;
    prm.depth[ob + nd] = dp;
    prm.score[ob + nd] = sc;
    prm.mode[ob + nd] = md;
    prm.pos[ob + nd] = ps;
  }
  for (int x = tid; x < N * W32; x += THREADS) {
    const int i = x / W32, w = x - (x / W32) * W32;
    uint32_t word = 0;
    if (i <= nn)
      for (int a = i; a >= 0; a = (a == 0) ? -1 : par_s[a])
        if ((a >> 5) == w) word |= 1u << (a & 31);
    prm.mask[(size_t)q * N * W32 + x] = word;
  }
  if (tid == 0) prm.n_nodes[q] = nn + 1;
}

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

size_t tree_smem_bytes(int K, int L, int topk, int B, int *cap_out, int *tsize_out) {
  const size_t budget = 232448 - sizeof(Shared) - 1024;
  const int need = K * B + K * topk + 64;
  for (int cap = 6144; cap >= need; cap -= 128) {
    const int nc = cap < K * B + 512 ? cap : K * B + 512;
    const int tsize = next_pow2(nc + nc / 2);
    const Layout y = make_layout(K, L, topk, B, cap, nc, tsize);
    if (y.total > budget) continue;
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
  p.cap = cap;
  p.nc = cap < T.K * T.B + 512 ? cap : T.K * T.B + 512;
  p.tsize = tsize;
  cudaError_t e = cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T.n_req);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, build_tree_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mfd
