// tree.cu -- the mixture DDTree of one round (project page "Multi-Future
// Drafting", How it works, step 3, and the Figure 1/2 caption): every prefix
// is scored by its best mode; the B best prefixes over all modes form one
// tree, which is the union of the per-mode trees at the common cut-off;
// shared prefixes are built once.
//
// One CTA (512 threads) builds one request's tree in shared memory, in two
// parts.
//
// Part 1, per mode (warp k = mode k, warp-synchronous only).  Mode k's B best
// prefixes under its own key (score_k desc, tokens lexicographically asc, a
// proper prefix first).  Within one mode a prefix is a tuple of ranks, one
// per position; replacing each rank by its token's rank inside that row
// (5 bits, token ids compared unsigned) turns the lexicographic token order
// into plain unsigned comparison of packed 80-bit keys, depth last.  The
// search is level by level: level t expands the depth-t entries in rank
// order (child scores only fall) while the child is not after the mode's
// current B-th best entry (kappa, from a 4-pass radix select on the score
// plus exact tie resolution on the key).  kappa only improves, so nothing
// that belongs to the mode's top-B is ever dropped.  If the pool fills,
// kappa is tightened, the pool pruned, and expansion resumes where each
// entry stopped.  The mode's top-B is then sorted (warp bitonic sort).
//
// Part 2, merge (all warps).  A prefix of the mixture tree is in the top-B
// list of every mode that attains its score, so the K sorted lists hold the
// tree.  Each list entry's token sequence is hashed; a hash table keeps, per
// sequence, the entry with the best (score, smallest mode) -- equality is
// checked on the full sequence, and a collision reseeds the table.  These
// "primary" entries are distinct prefixes keyed by (s, tokens).  A primary's
// node index is 1 + the number of primaries before it, summed over the K
// lists by binary search; the first B form the tree.  Parents come from the
// table (hash of the sequence without its last token).
#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int THREADS = 512;
constexpr int NWARPS = THREADS / 32;
constexpr int MAX_PASSES = 1024;

// Pool entry of one mode (16 bytes).  k0: row ranks of positions 1..12,
// 5 bits each, position 1 highest (bits 59..55).  k1: positions 13..16 at
// bits 24..5, depth at bits 4..0, next child rank at bits 31..26.
struct PE {
  float score;
  uint32_t k1;
  uint64_t k0;
};
static_assert(sizeof(PE) == 16, "pool entry");

constexpr uint32_t K1_KEY = 0x01FFFFFFu;

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
__device__ __forceinline__ int pk_next(uint32_t k1) { return (int)(k1 >> 26); }

struct MK {  // key within one mode
  uint32_t sk;
  uint64_t k0;
  uint32_t k1;
};
__device__ __forceinline__ MK mk_of(const PE &e) { return MK{desc_key(e.score), e.k0, e.k1 & K1_KEY}; }
__device__ __forceinline__ bool mk_before(const MK &a, const MK &b) {
  if (a.sk != b.sk) return a.sk < b.sk;
  if (a.k0 != b.k0) return a.k0 < b.k0;
  return a.k1 < b.k1;
}

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
  int pc;     // pool capacity per mode
  int tsize;  // hash table slots (power of two)
};

struct Layout {
  size_t lp, tok, sig, inv, pool, hv, hp, hslot, pcnt, nodeid, prim, table, par, nslot, total;
};

__host__ __device__ inline size_t al16(size_t o) { return (o + 15) & ~(size_t)15; }

__host__ __device__ inline Layout make_layout(int K, int L, int topk, int B, int pc, int tsize) {
  Layout y;
  size_t o = 0;
  const size_t klt = (size_t)K * L * topk, ne = (size_t)K * B;
  const size_t hist = (size_t)NWARPS * 256 * 4, tbl = al16((size_t)tsize * 4) + (size_t)tsize * 8;
  y.pool = o;
  o += (size_t)K * pc * 16;
  y.hv = o = al16(o);
  o += ne * 8;
  y.hp = o = al16(o);
  o += ne * 8;
  y.table = o = al16(o);  // hash tags (u32) then best (u64); the per-warp histograms overlay it
  o += hist > tbl ? hist : tbl;
  y.lp = o = al16(o);
  o += klt * 4;
  y.tok = o = al16(o);
  o += klt * 4;
  y.hslot = o = al16(o);
  o += ne * 2;
  y.pcnt = o = al16(o);
  o += ne * 2;
  y.nodeid = o = al16(o);
  o += ne * 2;
  y.par = o = al16(o);
  o += (size_t)(B + 1) * 2;
  y.nslot = o = al16(o);
  o += (size_t)(B + 1) * 2;
  y.sig = o = al16(o);
  o += klt;
  y.inv = o = al16(o);
  o += klt;
  y.prim = o = al16(o);
  o += ne;
  y.total = (o + 127) & ~(size_t)127;
  return y;
}

struct Shared {
  int bad, coll, total_prim;
  int cnt[16], off[17];
};

struct Ctx {
  const float *lp;
  const int32_t *tok;
  const uint8_t *sig, *inv;
  int K, L, topk, B, pc;
};

// token at position p (1-based) of a mode-k key
__device__ __forceinline__ uint32_t token_at(const Ctx &c, int k, uint64_t k0, uint32_t k1, int p) {
  const int row = (k * c.L + p - 1) * c.topk;
  return (uint32_t)c.tok[row + c.inv[row + pk_get(k0, k1, p)]];
}

// Lexicographic order of two prefixes of possibly different modes, by token
// ids (unsigned), a proper prefix first: <0, 0, >0.
__device__ int seq_cmp(const Ctx &c, int ka, const PE &a, int kb, const PE &b) {
  const int da = pk_depth(a.k1), db = pk_depth(b.k1);
  const int d = da < db ? da : db;
  for (int p = 1; p <= d; ++p) {
    const uint32_t ta = token_at(c, ka, a.k0, a.k1, p), tb = token_at(c, kb, b.k0, b.k1, p);
    if (ta != tb) return ta < tb ? -1 : 1;
  }
  return da - db;
}

// (s desc, tokens asc) across modes: true iff a is strictly before b.
__device__ __forceinline__ bool x_before(const Ctx &c, int ka, const PE &a, int kb, const PE &b) {
  const uint32_t sa = desc_key(a.score), sb = desc_key(b.score);
  if (sa != sb) return sa < sb;
  return seq_cmp(c, ka, a, kb, b) < 0;
}

// ---------------------------------------------------------------- part 1
// The B-th best entry of P[0, n) (warp-wide).  Returns false when n < B.
__device__ bool warp_kth(const PE *P, int n, int B, int *hist, MK &kap) {
  const int lane = threadIdx.x & 31;
  if (n < B) return false;
  uint32_t pre = 0;
  int rem = B, ntie = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      int bin = -1;
      if (i < n) {
        const uint32_t sk = desc_key(P[i].score);
        if (pass == 0 || (sk >> (shift + 8)) == (pre >> (shift + 8))) bin = (int)((sk >> shift) & 255u);
      }
      warp_hist_add(hist, bin);
    }
    __syncwarp();
    int c[8], sum = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      c[b] = hist[lane * 8 + b];
      sum += c[b];
    }
    int run = warp_excl_scan(sum, lane);
    int fb = -1, fbefore = 0, fcnt = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (fb < 0 && run < rem && rem <= run + c[b]) {
        fb = lane * 8 + b;
        fbefore = run;
        fcnt = c[b];
      }
      run += c[b];
    }
    const unsigned who = __ballot_sync(0xffffffffu, fb >= 0);
    const int src = __ffs(who) - 1;
    fb = __shfl_sync(0xffffffffu, fb, src);
    fbefore = __shfl_sync(0xffffffffu, fbefore, src);
    fcnt = __shfl_sync(0xffffffffu, fcnt, src);
    pre |= (uint32_t)fb << shift;
    rem -= fbefore;
    ntie = fcnt;
    __syncwarp();
  }
  // the rem-th smallest key among the entries whose score key is pre
  uint64_t b0 = 0;
  uint32_t b1 = 0;
  bool found = false;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    bool hit = false;
    if (i < n && desc_key(P[i].score) == pre) {
      if (ntie == 1) {
        hit = true;
      } else {
        const uint64_t e0 = P[i].k0;
        const uint32_t e1 = P[i].k1 & K1_KEY;
        int r = 1;
        for (int f = 0; f < n; ++f) {
          if (desc_key(P[f].score) != pre) continue;
          const uint64_t f0 = P[f].k0;
          const uint32_t f1 = P[f].k1 & K1_KEY;
          r += (f0 < e0) || (f0 == e0 && f1 < e1);
        }
        hit = (r == rem);
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      const int isrc = base + __ffs(m) - 1;
      b0 = P[isrc].k0;
      b1 = P[isrc].k1 & K1_KEY;
      found = true;
      break;
    }
  }
  kap = MK{pre, b0, b1};
  return found;
}

// Keep the entries not after kap; in place, order preserved.  Returns n.
__device__ int warp_prune(PE *P, int n, const MK &kap) {
  const int lane = threadIdx.x & 31;
  int out = 0;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    PE e;
    bool keep = false;
    if (i < n) {
      e = P[i];
      keep = !mk_before(kap, mk_of(e));
    }
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    __syncwarp();
    if (keep) P[out + __popc(m & lanemask_lt())] = e;
    out += __popc(m);
    __syncwarp();
  }
  return out;
}

// Expand the depth-t entries of P[0, n) in rank order (children appended
// after n).  Returns true when the pool filled before every child that can
// still make the cut was appended.
__device__ bool warp_expand(const Ctx &c, int k, int t, PE *P, int &n, bool hk, const MK &kap, bool &any) {
  const int lane = threadIdx.x & 31;
  const int n0 = n;
  const int row = (k * c.L + t) * c.topk;  // depth t+1 uses row index t
  bool overflow = false;
  for (int base = 0; base < n0 && !overflow; base += 32) {
    const int i = base + lane;
    PE par;
    bool isp = false, act = false;
    int j = 0;
    if (i < n0) {
      par = P[i];
      isp = pk_depth(par.k1) == t;
      j = pk_next(par.k1);
      act = isp && j < c.topk;
    }
    while (__any_sync(0xffffffffu, act)) {
      bool want = false;
      PE ch;
      if (act) {
        const float lv = c.lp[row + j];
        if (!(lv > -INFINITY)) {
          act = false;
          j = c.topk;
        } else {
          ch.score = __fadd_rn(par.score, lv);
          ch.k0 = par.k0;
          ch.k1 = par.k1 & ~(31u | (63u << 26));
          pk_set(ch.k0, ch.k1, t + 1, c.sig[row + j]);
          ch.k1 |= (uint32_t)(t + 1);
          if (!hk) {
            want = true;
          } else {
            const MK ck = mk_of(ch);
            if (ck.sk > kap.sk) {
              act = false;  // every later rank scores no better
              j = c.topk;
            } else if (mk_before(kap, ck)) {
              ++j;  // same score, after kappa in token order; a later rank may not be
              if (j >= c.topk) act = false;
            } else {
              want = true;
            }
          }
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, want);
      const int cnt = __popc(m);
      const int room = c.pc - n;
      const int r = __popc(m & lanemask_lt());
      if (want) {
        if (r < room) {
          P[n + r] = ch;
          ++j;
          if (j >= c.topk) act = false;
        } else {
          act = false;  // j kept: resumed in the next pass
          overflow = true;
        }
      }
      n += cnt < room ? cnt : room;
      if (cnt) any = true;
      overflow = __any_sync(0xffffffffu, overflow);
      if (overflow) act = false;
    }
    if (isp) P[i].k1 = (P[i].k1 & ~(63u << 26)) | ((uint32_t)j << 26);
    __syncwarp();
  }
  return overflow;
}

// Sort P[0, n) ascending by key (warp bitonic sort; P has room for the next
// power of two of n).  The padding sorts last.
__device__ void warp_sort(PE *P, int n) {
  const int lane = threadIdx.x & 31;
  int np2 = 1;
  while (np2 < n) np2 <<= 1;
  for (int i = n + lane; i < np2; i += 32) {
    P[i].score = -INFINITY;
    P[i].k0 = ~0ull;
    P[i].k1 = K1_KEY;
  }
  __syncwarp();
  for (int size = 2; size <= np2; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int ls = __ffs(stride) - 1;
      for (int e = lane; e < np2 / 2; e += 32) {
        const int lo = ((e >> ls) << (ls + 1)) | (e & (stride - 1)), hi = lo + stride;
        const bool asc = (lo & size) == 0;
        const PE a = P[lo], b = P[hi];
        if (mk_before(mk_of(b), mk_of(a)) == asc) {
          P[lo] = b;
          P[hi] = a;
        }
      }
      __syncwarp();
    }
}

__global__ void __launch_bounds__(THREADS, 1) build_tree_kernel(const Params prm) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Shared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = blockIdx.x;
  const int K = prm.K, L = prm.L, topk = prm.topk, B = prm.B, PC = prm.pc, tsize = prm.tsize;
  const int KLT = K * L * topk;
  const Layout lay = make_layout(K, L, topk, B, PC, tsize);
  float *lp_s = reinterpret_cast<float *>(smem + lay.lp);
  int32_t *tok_s = reinterpret_cast<int32_t *>(smem + lay.tok);
  uint8_t *sig_s = smem + lay.sig;
  uint8_t *inv_s = smem + lay.inv;
  PE *pools = reinterpret_cast<PE *>(smem + lay.pool);
  uint64_t *hv = reinterpret_cast<uint64_t *>(smem + lay.hv);
  uint64_t *hp = reinterpret_cast<uint64_t *>(smem + lay.hp);
  uint32_t *tag = reinterpret_cast<uint32_t *>(smem + lay.table);
  uint64_t *best = reinterpret_cast<uint64_t *>(smem + lay.table + al16((size_t)tsize * 4));
  int *hists = reinterpret_cast<int *>(smem + lay.table);
  uint16_t *hslot = reinterpret_cast<uint16_t *>(smem + lay.hslot);
  uint16_t *pcnt = reinterpret_cast<uint16_t *>(smem + lay.pcnt);
  int16_t *nodeid = reinterpret_cast<int16_t *>(smem + lay.nodeid);
  uint8_t *prim = smem + lay.prim;
  int16_t *par_s = reinterpret_cast<int16_t *>(smem + lay.par);
  uint16_t *nslot = reinterpret_cast<uint16_t *>(smem + lay.nslot);

  const float *glp = prm.tk_logp + (size_t)q * KLT;
  const int32_t *gtk = prm.tk_tok + (size_t)q * KLT;

  // ---------------------------------------------------- tables and checks
  if (tid == 0) sh.bad = 0;
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

  // ---------------------------------------------------- part 1: per mode
  const Ctx c{lp_s, tok_s, sig_s, inv_s, K, L, topk, B, PC};
  if (warp < K) {
    const int k = warp;
    PE *P = pools + (size_t)k * PC;
    int *hist = hists + warp * 256;
    int n = 0;
    for (int base = 0; base < topk; base += 32) {  // depth-1 entries
      const int j = base + lane;
      const int e = (k * L) * topk + j;
      const bool ok = j < topk && lp_s[e] > -INFINITY;
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      if (ok) {
        PE en;
        en.score = lp_s[e];
        en.k0 = 0;
        en.k1 = 1u;
        pk_set(en.k0, en.k1, 1, sig_s[e]);
        P[n + __popc(m & lanemask_lt())] = en;
      }
      n += __popc(m);
    }
    __syncwarp();
    bool failed = false;
    for (int t = 1; t < L && !failed; ++t) {
      bool any = false;
      int pass = 0;
      for (; pass < MAX_PASSES; ++pass) {
        MK kap{0, 0, 0};
        const bool hk = warp_kth(P, n, B, hist, kap);
        if (hk) n = warp_prune(P, n, kap);
        if (!warp_expand(c, k, t, P, n, hk, kap, any)) break;
      }
      if (pass == MAX_PASSES) failed = true;
      if (!any) break;
    }
    if (!failed) {
      MK kap{0, 0, 0};
      if (warp_kth(P, n, B, hist, kap)) n = warp_prune(P, n, kap);
      if (n > B) failed = true;  // the B-th entry was not found: impossible for valid tables
    }
    if (failed) {
      if (lane == 0) report(prm.status, MFD_ERR_UNSUPPORTED);
      n = 0;
    }
    warp_sort(P, n);
    if (lane == 0) sh.cnt[k] = n;
  }
  __syncthreads();

  // ---------------------------------------------------- part 2: merge
  if (tid == 0) {
    int o = 0;
    for (int k = 0; k < K; ++k) {
      sh.off[k] = o;
      o += sh.cnt[k];
    }
    sh.off[K] = o;
  }
  __syncthreads();
  const int NE = sh.off[K];
  auto entry_of = [&](int id, int &k, int &i) {
    k = 0;
    while (id >= sh.off[k + 1]) ++k;
    i = id - sh.off[k];
  };
  // hashes of each entry's token sequence and of its parent prefix
  for (int id = tid; id < NE; id += THREADS) {
    int k, i;
    entry_of(id, k, i);
    const PE e = pools[(size_t)k * PC + i];
    const int d = pk_depth(e.k1);
    uint64_t h = 0x2545F4914F6CDD1Dull, hpar = h;
    for (int p = 1; p <= d; ++p) {
      hpar = h;
      h = mix64(h ^ ((uint64_t)token_at(c, k, e.k0, e.k1, p) + ((uint64_t)p << 40)));
    }
    hv[id] = h;
    hp[id] = hpar;
  }
  uint64_t seed = 0;
  for (int attempt = 0; attempt < 4; ++attempt) {
    for (int s = tid; s < tsize; s += THREADS) {
      tag[s] = 0;
      best[s] = ~0ull;
    }
    if (tid == 0) sh.coll = 0;
    __syncthreads();
    for (int id = tid; id < NE; id += THREADS) {
      const uint64_t h = mix64(hv[id] ^ seed);
      const uint32_t tg = (uint32_t)(h >> 32) | 1u;
      uint32_t s = (uint32_t)h & (uint32_t)(tsize - 1);
      for (int probe = 0; probe < tsize; ++probe) {
        const uint32_t prev = atomicCAS(&tag[s], 0u, tg);
        if (prev == 0u || prev == tg) break;
        s = (s + 1) & (uint32_t)(tsize - 1);
      }
      hslot[id] = (uint16_t)s;
    }
    __syncthreads();
    for (int id = tid; id < NE; id += THREADS) {
      int k, i;
      entry_of(id, k, i);
      const PE e = pools[(size_t)k * PC + i];
      const uint64_t packed = ((uint64_t)desc_key(e.score) << 32) | ((uint64_t)k << 16) | (uint64_t)id;
      atomicMin(reinterpret_cast<unsigned long long *>(&best[hslot[id]]), (unsigned long long)packed);
    }
    __syncthreads();
    for (int id = tid; id < NE; id += THREADS) {
      const int rid = (int)(best[hslot[id]] & 0xFFFF);
      if (rid == id) continue;
      int k, i, rk, ri;
      entry_of(id, k, i);
      entry_of(rid, rk, ri);
      if (seq_cmp(c, k, pools[(size_t)k * PC + i], rk, pools[(size_t)rk * PC + ri]) != 0) sh.coll = 1;
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
  // primaries (one per distinct prefix) and their running counts per list
  for (int id = tid; id < NE; id += THREADS) {
    prim[id] = (int)(best[hslot[id]] & 0xFFFF) == id;
    nodeid[id] = -1;
  }
  __syncthreads();
  if (warp < K) {
    const int k = warp, o = sh.off[k], n = sh.cnt[k];
    int run = 0;
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      const int f = i < n ? prim[o + i] : 0;
      const int incl = warp_excl_scan(f, lane) + f;
      if (i < n) pcnt[o + i] = (uint16_t)(run + incl);
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int tot = 0;
    for (int k = 0; k < K; ++k)
      if (sh.cnt[k]) tot += pcnt[sh.off[k] + sh.cnt[k] - 1];
    sh.total_prim = tot;
  }
  // node index of a primary: 1 + the primaries before it, over every list
  for (int id = tid; id < NE; id += THREADS) {
    if (!prim[id]) continue;
    int k, i;
    entry_of(id, k, i);
    const PE e = pools[(size_t)k * PC + i];
    int before = pcnt[id] - 1;
    for (int k2 = 0; k2 < K && before < B; ++k2) {
      if (k2 == k) continue;
      const PE *P2 = pools + (size_t)k2 * PC;
      int lo = 0, hi = sh.cnt[k2];  // first entry of list k2 not before e
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (x_before(c, k2, P2[mid], k, e))
          lo = mid + 1;
        else
          hi = mid;
      }
      if (lo > 0) before += pcnt[sh.off[k2] + lo - 1];
    }
    if (before < B) {
      nodeid[id] = (int16_t)(before + 1);
      nslot[before + 1] = (uint16_t)id;
    }
  }
  if (tid == 0) {
    par_s[0] = -1;
    sh.bad = 0;
  }
  __syncthreads();
  const int nn = sh.total_prim < B ? sh.total_prim : B;
  // parents: the table entry of the sequence without its last token
  for (int nd = 1 + tid; nd <= nn; nd += THREADS) {
    const int id = nslot[nd];
    int k, i;
    entry_of(id, k, i);
    const PE e = pools[(size_t)k * PC + i];
    const int d = pk_depth(e.k1);
    int par = 0;
    if (d > 1) {
      par = -1;
      const uint64_t h = mix64(hp[id] ^ seed);
      const uint32_t tg = (uint32_t)(h >> 32) | 1u;
      uint32_t s = (uint32_t)h & (uint32_t)(tsize - 1);
      for (int probe = 0; probe < tsize && par < 0; ++probe) {
        const uint32_t t0 = tag[s];
        if (t0 == 0u) break;
        if (t0 == tg) {
          const int rid = (int)(best[s] & 0xFFFF);
          int rk, ri;
          entry_of(rid, rk, ri);
          const PE r = pools[(size_t)rk * PC + ri];
          if (pk_depth(r.k1) == d - 1) {
            bool same = true;
            for (int p = 1; p < d && same; ++p)
              same = token_at(c, rk, r.k0, r.k1, p) == token_at(c, k, e.k0, e.k1, p);
            if (same) par = nodeid[rid];
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
      int k, i;
      entry_of(nslot[nd], k, i);
      const PE e = pools[(size_t)k * PC + i];
      dp = pk_depth(e.k1);
      pa = par_s[nd];
      tk = (int)token_at(c, k, e.k0, e.k1, dp);
      sc = e.score;
      md = k;
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
  const int tsize = next_pow2(2 * K * B > 64 ? 2 * K * B : 64);
  const size_t budget = 232448 - sizeof(Shared) - 1024;
  const int need = next_pow2(B) > B + 2 * topk ? next_pow2(B) : B + 2 * topk;
  for (int pc = 4096; pc >= need; pc -= 32) {
    const Layout y = make_layout(K, L, topk, B, pc, tsize);
    if (y.total > budget) continue;
    *cap_out = pc;
    *tsize_out = tsize;
    return y.total;
  }
  return 0;
}

cudaError_t launch_build_tree(const TreeLaunch &T, cudaStream_t stream) {
  int pc = 0, tsize = 0;
  const size_t bytes = tree_smem_bytes(T.K, T.L, T.topk, T.B, &pc, &tsize);
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
  p.pc = pc;
  p.tsize = tsize;
  cudaError_t e = cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  build_tree_kernel<<<T.n_req, THREADS, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mfd
