// tree.cu -- the mixture DDTree of one round (project page "Multi-Future
// Drafting", How it works, step 3, and the Figure 1/2 caption): every prefix
// is scored by its best mode; the B best prefixes over all modes form one
// tree, which is the union of the per-mode trees at the common cut-off;
// shared prefixes are built once.
//
// One CTA (512 threads) builds one request's tree in shared memory.
//
// Entries.  The pool holds (mode, prefix) entries scored by their own mode;
// a prefix is packed as its tuple of row ranks (5 bits a position, depth
// last), and its tokens are read back through the rows.  Prefixes are
// compared by their token ids (unsigned, a proper prefix first).
//
// The bound.  Every first-row token is owned by one mode; entries whose
// first token their mode owns are pairwise distinct prefixes, and a prefix's
// mixture score is at least its mode score.  So with tau the B-th best score
// among the owned entries, at least B distinct prefixes score no worse than
// tau: the tree's cut-off is never worse, and an entry scoring worse than tau
// can neither be in the tree nor lead to it (scores only fall along a path).
// tau is found by a radix select of one or two 8-bit digits below the
// highest bit where the owned score keys differ, rounded to the worse end.
//
// Search, level by level.  Depth 1 and 2 are generated at once; then at
// each level the pool is cut to the bound and the entries of that depth are
// expanded in rank order (child scores only fall) while the child is within
// the bound.  When the pool fills, it is pruned to each mode's exact B best
// (radix select on the full score key, then the token order among equal
// scores) and expansion resumes where each entry stopped.
//
// Result.  The entries within the final bound are hashed by token sequence;
// a table keeps per sequence the entry with the best (score, smallest mode),
// equality checked on the full sequence (a collision reseeds the table).
// These primaries are distinct prefixes.  Their order comes from runs of 32
// sorted in registers and binary searches between the runs; a prefix's
// parent is the table slot of its sequence without the last token.
#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int THREADS = 512;
constexpr int NWARPS = THREADS / 32;

// Checked build (compiled with -DMFD_CHECKED): every shared-memory index the
// kernel computes from data is tested against its array's extent.  An index
// out of range is clamped into the array, so the access stays in bounds, and
// the CTA ends with MFD_ERR_CHECK in *status.  The ordinary build compiles
// CHK(i, n) to i.
#ifdef MFD_CHECKED
__shared__ int chk_bad_s;
__device__ __forceinline__ int chk_index(int i, int n) {
  if ((unsigned)i >= (unsigned)n) {
    chk_bad_s = 1;
    return i < 0 ? 0 : n - 1;
  }
  return i;
}
#define CHK(i, n) chk_index((int)(i), (int)(n))
#define CHK_INIT() \
  if (threadIdx.x == 0) chk_bad_s = 0
#define CHK_REPORT()                                                    \
  do {                                                                  \
    block_sync();                                                    \
    if (threadIdx.x == 0 && chk_bad_s) report(prm.status, MFD_ERR_CHECK); \
  } while (0)
#else
#define CHK(i, n) (i)
#define CHK_INIT() \
  do {             \
  } while (0)
#define CHK_REPORT() \
  do {               \
  } while (0)
#endif
constexpr int MAX_PASSES = 64;
constexpr int PLIST = 1024;     // parents listed for pair-parallel expansion
constexpr int PAIR_MAX = 4096;  // (parent, rank) pairs expanded at once
constexpr int MAX_GROUPS = 17;  // radix groups: one per mode, plus one across modes
constexpr int RANK_ALL = 1024;  // candidates up to which every primary is ranked
constexpr int MAX_MASK_WORDS = 17;  // 32-bit words of a mask row for B + 1 <= 513 nodes

// Pool entry (16 bytes).  k0: row ranks of positions 1..12, 5 bits each,
// position 1 highest (bits 59..55).  k1: depth at bits 4..0, positions
// 13..16 at bits 24..5, mode at bits 28..25.
struct PE {
  float score;
  uint32_t k1;
  uint64_t k0;
};
static_assert(sizeof(PE) == 16, "pool entry");

constexpr uint32_t K1_OWNED = 1u << 29;   // the entry's mode owns its first token

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
  size_t lp, tok, ent, nxt, flg, table, hist1, skk, ra, sel, prim, hslot, pslot, nodeid, par, nslot, plist,
      total;
};

__host__ __device__ inline size_t al16(size_t o) { return (o + 15) & ~(size_t)15; }

__host__ __device__ inline Layout make_layout(int K, int L, int topk, int B, int cap, int nc, int tsize) {
  Layout y;
  size_t o = 0;
  const size_t klt = (size_t)K * L * topk;
  const size_t hist = (size_t)2 * MAX_GROUPS * 256 * 4, tbl = (size_t)tsize * 14;
  y.ent = o;
  o += (size_t)cap * 16;
  y.table = o = al16(o);  // hash tags then best entries; the radix histograms overlay it
  o += hist > tbl ? hist : tbl;
  y.hist1 = o = al16(o);
  o += 2 * 256 * 4;
  y.lp = o = al16(o);
  o += klt * 4;
  y.tok = o = al16(o);
  o += klt * 4;
  y.skk = o = al16(o);
  o += (size_t)(nc + 32) * 4;  // padded to whole runs of 32
  y.sel = o = al16(o);
  o += (size_t)nc * 2;
  y.hslot = y.ra = o = al16(o);  // hash slots die with the primaries; the rank's run order reuses them
  o += (size_t)(nc + 32) * 2;
  y.pslot = o = al16(o);
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
  y.prim = o = al16(o);
  o += (size_t)nc;
  y.total = (o + 127) & ~(size_t)127;
  return y;
}

struct Shared {
  int n_ent, overflow, any, refine, bad, coll, n_prim, n_sel, has_tau, n_par, n_out, n_in, cut2, wbad[NWARPS];
  int cnt[MAX_GROUPS], act[MAX_GROUPS], rem[MAX_GROUPS], ntie[MAX_GROUPS];
  uint8_t u1[512];  // per first-row entry: its mode owns its token
  int f1[16], f2[16];
  float lo1[16], lo2[16];
  uint32_t kmin, kmax;
  uint32_t pre[MAX_GROUPS], tau;
};

struct Ctx {
  const float *lp;
  const int32_t *tok;
  int K, L, topk;
};

// token at position p (1-based) of an entry
__device__ __forceinline__ uint32_t token_at(const Ctx &c, const PE &e, int p) {
  const int row = (pk_mode(e.k1) * c.L + p - 1) * c.topk;
  return (uint32_t)c.tok[CHK(row + (int)pk_get(e.k0, e.k1, p), c.K * c.L * c.topk)];
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

// The hash of the whole sequence and (in *hp) of the sequence without its
// last token, which is the parent's hash.
__device__ __forceinline__ uint64_t seq_hash2(const Ctx &c, const PE &e, int d, uint64_t seed, uint64_t *hp) {
  uint64_t h = 0x2545F4914F6CDD1Dull ^ seed;
  *hp = h;
  for (int p = 1; p <= d; ++p) {
    *hp = h;
    h = mix64(h ^ ((uint64_t)token_at(c, e, p) + ((uint64_t)p << 40)));
  }
  return h;
}

// Per group g (grp(i) in [0, G), or -1 to skip), with at least B members
// among ent[0, n): digits of the B-th best score key, most significant
// first, over `passes` 8-bit passes.  Leaves sh.act[g], sh.pre[g] (the digits
// found, low bits zero), sh.rem[g] (rank of the B-th within that prefix) and
// sh.ntie[g] (members sharing the prefix).  With fold_tau, also the smallest
// bound over the groups, pre[g] with the undetermined low bits set, in
// sh.tau (sh.has_tau = 0 when no group has B members).  hA and hB hold G * 256
// counters each; a pass counts into one while the other is cleared.  An
// entry belongs to group grp(i) and, when grp2(i) >= 0, also to grp2(i).
template <typename GroupFn, typename Group2Fn>
__device__ void radix_bound(Shared &sh, const PE *ent, int n, int G, int B, int passes, int *hA, int *hB,
                            bool fold_tau, GroupFn grp, Group2Fn grp2) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < MAX_GROUPS) {
    sh.pre[tid] = 0;
    sh.rem[tid] = B;
    sh.ntie[tid] = 0;
    sh.act[tid] = tid < G;  // until the first pass has counted the group
  }
  if (fold_tau && tid == 0) {
    sh.tau = 0xFFFFFFFFu;
    sh.has_tau = 0;
  }
  for (int i = tid; i < G * 256; i += THREADS) hA[i] = 0;
  block_sync();
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 24 - 8 * pass;
    int *hist = (pass & 1) ? hB : hA;
    int *next = (pass & 1) ? hA : hB;
    for (int base = warp * 32; base < n; base += THREADS) {
      const int i = base + lane;
      int bin = -1, bin2 = -1;
      if (i < n) {
        const uint32_t sk = desc_key(ent[i].score);
        const int g = grp(i), g2 = grp2(i);
        if (g >= 0 && sh.act[g] && (pass == 0 || (sk >> (shift + 8)) == (sh.pre[g] >> (shift + 8))))
          bin = g * 256 + (int)((sk >> shift) & 255u);
        if (g2 >= 0 && sh.act[g2] && (pass == 0 || (sk >> (shift + 8)) == (sh.pre[g2] >> (shift + 8))))
          bin2 = g2 * 256 + (int)((sk >> shift) & 255u);
      }
      warp_hist_add(hist, bin);
      if (__any_sync(0xffffffffu, bin2 >= 0)) warp_hist_add(hist, bin2);
    }
    if (pass + 1 < passes)
      for (int i = tid; i < G * 256; i += THREADS) next[i] = 0;
    block_sync();
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
      // exactly one (lane, bin) holds the rem-th member
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (run < rem && rem <= run + c[b]) {
          const uint32_t pre = sh.pre[g] | ((uint32_t)(lane * 8 + b) << shift);
          sh.pre[g] = pre;
          sh.rem[g] = rem - run;
          sh.ntie[g] = c[b];
          if (fold_tau && pass + 1 == passes) {
            atomicMin(&sh.tau, pre | (passes >= 4 ? 0u : (0xFFFFFFFFu >> (8 * passes))));
            sh.has_tau = 1;
          }
        }
        run += c[b];
      }
    }
    block_sync();
  }
}

// In-place compaction of ent/nxt[0, n) to the entries with keep(e, i), order
// not kept.  Batches of THREADS * STAGE entries: every thread holds its
// entries of the batch in registers across a barrier, then appends the kept
// ones; a batch's writes land below the end of the batch, and the next
// batch's sources lie beyond it, so no entry is overwritten before it is read.
constexpr int STAGE = 6;
template <typename KeepFn>
__device__ int compact_pool(Shared &sh, PE *ent, uint8_t *nxt, int n, KeepFn keep) {
  const int tid = threadIdx.x;
  if (tid == 0) sh.n_out = 0;
  for (int b0 = 0; b0 < n; b0 += THREADS * STAGE) {
    PE e[STAGE];
    uint8_t nx[STAGE];
    bool kp[STAGE];
#pragma unroll
    for (int j = 0; j < STAGE; ++j) {
      const int i = b0 + tid + j * THREADS;
      kp[j] = false;
      if (i < n) {
        e[j] = ent[i];
        nx[j] = nxt[i];
        kp[j] = keep(e[j], i);
      }
    }
    block_sync();
#pragma unroll
    for (int j = 0; j < STAGE; ++j) {
      if (!__any_sync(0xffffffffu, kp[j])) continue;
      const int slot = warp_append(&sh.n_out, kp[j]);
      if (kp[j]) {
        ent[CHK(slot, n)] = e[j];
        nxt[CHK(slot, n)] = nx[j];
      }
    }
  }
  block_sync();
  return sh.n_out;
}

// The bound over the owned entries of ent[0, sh.n_ent): sh.tau, sh.has_tau.
// pre: the key range is in sh.kmin/kmax and the first digit's histogram was
// filled when the pool was generated.  Out of line: one copy of the code.
__device__ __noinline__ void bound_owned(Shared &sh, const PE *ent, int *hist, int B, bool pre) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    sh.tau = 0xFFFFFFFFu;
    sh.has_tau = 0;
  }
  const int n = sh.n_ent;
  if (!pre) {
    if (tid == 0) {
      sh.kmin = 0xFFFFFFFFu;
      sh.kmax = 0u;
    }
    if (tid < 256) hist[tid] = 0;
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;  // over the owned entries
    for (int i = tid; i < n; i += THREADS) {
      const PE e = ent[i];
      if (e.k1 & K1_OWNED) {
        const uint32_t k = desc_key(e.score);
        lo = min(lo, k);
        hi = max(hi, k);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    block_sync();
    if (lane == 0 && lo <= hi) {
      atomicMin(&sh.kmin, lo);
      atomicMax(&sh.kmax, hi);
    }
    block_sync();
  }
  const uint32_t kmin = sh.kmin, kmax = sh.kmax;
  const int hb = (kmin ^ kmax) ? 31 - __clz((int)(kmin ^ kmax)) : 0;
  // digits of 8 bits from the highest differing bit down; a second digit
  // only when the first leaves many entries in the boundary bin
  int shift = hb > 7 ? hb - 7 : 0;
  uint32_t prefix = shift + 8 >= 32 ? 0u : (kmin >> (shift + 8)) << (shift + 8);
  for (int digit = 0; digit < 2; ++digit) {
    const uint32_t hi_mask = shift + 8 >= 32 ? 0u : ~((1u << (shift + 8)) - 1u);
    if (!(pre && digit == 0)) {
    for (int base = warp * 32; base < n; base += THREADS) {
      const int i = base + lane;
      int bin = -1;
      if (i < n) {
        const PE e = ent[i];
        const uint32_t k = desc_key(e.score);
        if ((e.k1 & K1_OWNED) && (k & hi_mask) == prefix) bin = (int)((k >> shift) & 255u);
      }
      warp_hist_add(digit ? hist + 256 : hist, bin);
    }
    if (digit == 0 && tid < 256) hist[256 + tid] = 0;
    block_sync();
    }
    if (warp == 0) {
      const int *h = digit ? hist + 256 : hist;
      const int need = digit ? sh.rem[0] : B;
      int c8[8], sum = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c8[b] = h[lane * 8 + b];
        sum += c8[b];
      }
      int run = warp_excl_scan(sum, lane);
      const int total = __shfl_sync(0xffffffffu, run + sum, 31);
      if (lane == 0) sh.refine = 0;
      if (total >= need) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (run < need && need <= run + c8[b]) {
            const uint32_t pre = prefix | ((uint32_t)(lane * 8 + b) << shift);
            sh.tau = pre | ((1u << shift) - 1u);
            sh.has_tau = 1;
            sh.pre[0] = pre;
            sh.rem[0] = need - run;
            sh.refine = c8[b] > 64 && shift > 0;
          }
          run += c8[b];
        }
      }
    }
    block_sync();
    if (!sh.refine) break;
    prefix = sh.pre[0];
    shift = shift > 8 ? shift - 8 : 0;
  }
}

__device__ __noinline__ int compact_by_tau(Shared &sh, PE *ent, uint8_t *nxt, int n, uint32_t tau) {
  return compact_pool(sh, ent, nxt, n, [&](const PE &e, int) { return desc_key(e.score) <= tau; });
}
__device__ __noinline__ int compact_by_flag(Shared &sh, PE *ent, uint8_t *nxt, int n, const uint8_t *flg) {
  return compact_pool(sh, ent, nxt, n, [&](const PE &, int i) { return flg[i] != 0; });
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
  PE *ent = reinterpret_cast<PE *>(smem + lay.ent);
  uint8_t *nxt = smem + lay.nxt;
  uint8_t *flg = smem + lay.flg;
  int *hist1 = reinterpret_cast<int *>(smem + lay.hist1);
  uint32_t *tag = reinterpret_cast<uint32_t *>(smem + lay.table);
  uint32_t *bkey = tag + tsize;  // per slot: best score key, then (mode << 16 | entry) among those
  uint32_t *bsub = bkey + tsize;
  uint16_t *rep = reinterpret_cast<uint16_t *>(bsub + tsize);
  int *hist = reinterpret_cast<int *>(smem + lay.table);
  uint32_t *skk = reinterpret_cast<uint32_t *>(smem + lay.skk);
  uint16_t *sel = reinterpret_cast<uint16_t *>(smem + lay.sel);
  uint16_t *ra = reinterpret_cast<uint16_t *>(smem + lay.ra);
  uint16_t *hslot = reinterpret_cast<uint16_t *>(smem + lay.hslot);
  uint16_t *pslot = reinterpret_cast<uint16_t *>(smem + lay.pslot);
  int16_t *nodeid = reinterpret_cast<int16_t *>(smem + lay.nodeid);
  uint8_t *prim = smem + lay.prim;
  int16_t *par_s = reinterpret_cast<int16_t *>(smem + lay.par);
  uint16_t *nslot = reinterpret_cast<uint16_t *>(smem + lay.nslot);
  uint16_t *plist = reinterpret_cast<uint16_t *>(smem + lay.plist);

  const float *glp = prm.tk_logp + (size_t)q * KLT;
  const int32_t *gtk = prm.tk_tok + (size_t)q * KLT;
  CHK_INIT();
  pdl_wait();  // the tables may come from the grid launched just before
  pdl_launch_dependents();

  // ---------------------------------------------------- tables and checks
  // One row per segment of SEG lanes (SEG = topk rounded up to a power of
  // two).  Every warp first copies its own rows to shared memory (all loads
  // in flight at once), then checks them there: each entry against its left
  // neighbour (sorted, <= 0, not NaN) and against the row's other tokens.
  {
    int SEG = 1;
    while (SEG < topk) SEG <<= 1;
    const int rows = K * L, spw = 32 / SEG;  // rows per warp per round
    const int seg = lane / SEG, j = lane - seg * SEG;
    constexpr int RMAX = 16;                 // rounds: K * L <= 256 rows, 16 warps, >= 1 row a warp
    float v[RMAX];
    int32_t tk[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      const int row = (r * NWARPS + warp) * spw + seg;
      const bool in = row < rows && j < topk;
      v[r] = in ? __ldcg(glp + row * topk + j) : 0.f;  // L2: written by the kernel just before
      tk[r] = in ? __ldcg(gtk + row * topk + j) : 0;
    }
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      const int row = (r * NWARPS + warp) * spw + seg;
      if (row < rows && j < topk) {
        lp_s[row * topk + j] = v[r];
        tok_s[row * topk + j] = tk[r];
      }
    }
    if (tid == 0) sh.n_ent = 0;
    if (tid < 512) hist[tid] = 0;  // the first bound's two digit histograms
    if (tid < 256) hist[512 + tid] = 0;  // and the count of every depth-1 and depth-2 entry
  }
  block_sync();
  // The checks read only the warp's own rows; they run in the same interval
  // as the ownership scan below, and their verdict is acted on after the next
  // block barrier, before anything derived from the tables is used.
  {
    int SEG = 1;
    while (SEG < topk) SEG <<= 1;
    const int rows = K * L, spw = 32 / SEG;
    const int seg = lane / SEG, j = lane - seg * SEG;
    bool bad = false;
    for (int r = 0; (r * NWARPS + warp) * spw < rows; ++r) {
      const int row = (r * NWARPS + warp) * spw + seg;
      if (row < rows && j < topk) {
        const float *lr = lp_s + row * topk;
        const int32_t *tr = tok_s + row * topk;
        const float v = lr[j];
        const int32_t tk = tr[j];
        bad |= isnan(v) || v > 0.f || (j > 0 && !(lr[j - 1] >= v));
        int dup = 0;
#pragma unroll 4
        for (int f = 0; f < topk; ++f) dup += tr[f] == tk;
        bad |= dup != 1;
      }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) sh.wbad[warp] = bad;
  }
  const Ctx c{lp_s, tok_s, K, L, topk};
  auto mode_of = [&](int i) { return pk_mode(ent[i].k1); };

  // ---------------------------------------------------- depth-1 entries
  // Ownership: every first-row token is owned by one mode, the one with the
  // best value for it (smallest mode on ties).  Prefixes whose first token
  // their mode owns are pairwise distinct: two equal prefixes share their
  // first token, hence its owner, hence their mode.
  // With no bound possible yet (every mode holds only its topk first
  // entries), depth 2 is generated at once when it fits.
  // Depth 2 is made with depth 1 when every pair fits the pool (two).
  // Otherwise, with depth 2 present (pairs), the pairs are first only
  // counted: the owned ones into the first digit's histogram, all of them
  // into a second.  They are then made only within the bound that the first
  // histogram gives, when those fit (sh.cut2), else depth 1 alone.
  const bool two = L >= 2 && topk < B && K * topk * (1 + topk) <= CAP;
  const bool pairs = L >= 2 && topk < B;
  {
    // T1 threads per first-row entry look for its token in the other modes'
    // first rows, each through every T1-th mode
    const int n1 = K * topk;
    int T1 = 1;
    while (T1 < 32 && n1 * T1 * 2 <= THREADS) T1 <<= 1;
    for (int base = warp * 32; base < n1 * T1; base += THREADS) {
      const int x = base + lane;
      const int e = x / T1, part = x - e * T1;
      const bool in = e < n1;
      const int k = in ? e / topk : 0, j = in ? e - k * topk : 0;
      const int tkn = in ? tok_s[(k * L) * topk + j] : 0;
      const float v = in ? lp_s[(k * L) * topk + j] : 0.f;
      bool beaten = false;
      auto beats = [&](const float *lrow, int j2, int k2) { return lrow[j2] > v || (lrow[j2] == v && k2 < k); };
      if (in)
        for (int k2 = part; k2 < K; k2 += T1) {
          if (k2 == k) continue;
          const int32_t *row = tok_s + (k2 * L) * topk;
          const float *lrow = lp_s + (k2 * L) * topk;
          if ((topk & 3) == 0) {  // rows start on 16-byte boundaries
#pragma unroll 2
            for (int j4 = 0; j4 < topk; j4 += 4) {
              const int4 t4 = *reinterpret_cast<const int4 *>(row + j4);
              if (t4.x == tkn) beaten |= beats(lrow, j4, k2);
              if (t4.y == tkn) beaten |= beats(lrow, j4 + 1, k2);
              if (t4.z == tkn) beaten |= beats(lrow, j4 + 2, k2);
              if (t4.w == tkn) beaten |= beats(lrow, j4 + 3, k2);
            }
          } else {
            for (int j2 = 0; j2 < topk; ++j2)
              if (row[j2] == tkn) beaten |= beats(lrow, j2, k2);
          }
        }
      for (int o = T1 / 2; o > 0; o >>= 1) beaten |= __shfl_xor_sync(0xffffffffu, (int)beaten, o) != 0;
      if (in && part == 0) sh.u1[e] = beaten ? 0 : 1;
    }
    // finite entries of each mode's first two rows (the rows are sorted, so
    // they come first)
    // and their extremes, which bound every depth-1 and depth-2 score
    if (warp < K) {
      const float v1 = lane < topk ? lp_s[(warp * L) * topk + lane] : -INFINITY;
      const float v2 = lane < topk && L >= 2 ? lp_s[(warp * L + 1) * topk + lane] : -INFINITY;
      const bool f1 = v1 > -INFINITY, f2 = v2 > -INFINITY;
      const int c1 = __popc(__ballot_sync(0xffffffffu, f1)), c2 = __popc(__ballot_sync(0xffffffffu, f2));
      const float lo1 = -warp_max(f1 ? -v1 : -INFINITY), lo2 = -warp_max(f2 ? -v2 : -INFINITY);
      if (lane == 0) {
        sh.f1[warp] = c1;
        sh.f2[warp] = c2;
        sh.lo1[warp] = lo1;  // +inf when the row has no finite entry
        sh.lo2[warp] = lo2;
      }
    }
  }
  block_sync();
  {
    int any_bad = 0;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) any_bad |= sh.wbad[w];
    if (any_bad) {
      if (tid == 0) report(prm.status, MFD_ERR_INPUT);
      CHK_REPORT();
      return;
    }
  }
  {
    // fixed slots, mode-major: depth 1 first, then depth 2
    int N1 = 0, N2 = 0;
    bool full = true;
    float hi = -INFINITY, lo = INFINITY;  // bounds of every score counted here
    for (int k = 0; k < K; ++k) {
      const int f1 = sh.f1[k], f2 = sh.f2[k];
      N1 += f1;
      N2 += f1 * f2;
      full &= f1 == topk && f2 == topk;
      if (f1 > 0) {
        hi = fmaxf(hi, lp_s[(k * L) * topk]);
        lo = fminf(lo, sh.lo1[k]);
        if (pairs && f2 > 0) lo = fminf(lo, __fadd_rn(sh.lo1[k], sh.lo2[k]));
      }
    }
    if (!pairs) N2 = 0;
    // the owned entries are counted into the first digit's histogram as they
    // are made; the digit starts at the highest bit where the score keys of
    // [lo, hi] differ
    const uint32_t kmin = desc_key(hi), kmax = desc_key(lo);
    const int hb = (kmin ^ kmax) ? 31 - __clz((int)(kmin ^ kmax)) : 0;
    const int shift = hb > 7 ? hb - 7 : 0;
    if (tid == 0) {
      sh.kmin = kmin;
      sh.kmax = kmax;
      sh.cut2 = 0;
    }
    const int TT = topk * topk;
    // x / topk and x / TT as multiply-highs by ceil(2^32 / d): exact for
    // x < 2^16 and 1 < d <= 2^10 (d = 1 has no such multiplier)
    const uint32_t m1 = topk > 1 ? 0xFFFFFFFFu / (uint32_t)topk + 1u : 0u;
    const uint32_t m2 = TT > 1 ? 0xFFFFFFFFu / (uint32_t)TT + 1u : 0u;
    auto div1 = [&](int v) { return topk > 1 ? (int)__umulhi((uint32_t)v, m1) : v; };
    auto div2 = [&](int v) { return TT > 1 ? (int)__umulhi((uint32_t)v, m2) : v; };
    // entry x of the fixed order (x < N1: depth 1, else depth 2); returns
    // whether its mode owns its first token
    auto make = [&](int x, PE &en) {
      if (x < N1) {
        int k, j;
        if (full) {
          k = div1(x);
          j = x - k * topk;
        } else {
          int off = 0;
          k = 0;
          while (x - off >= sh.f1[k]) off += sh.f1[k++];
          j = x - off;
        }
        const bool own = sh.u1[CHK(k * topk + j, K * topk)];
        en.score = lp_s[CHK((k * L) * topk + j, KLT)];
        en.k0 = 0;
        en.k1 = 1u | ((uint32_t)k << 25) | (own ? K1_OWNED : 0u);
        pk_set(en.k0, en.k1, 1, (uint32_t)j);
        return own;
      }
      const int y = x - N1;
      int k, a, b2;
      if (full) {
        k = div2(y);
        const int r = y - k * TT;
        a = div1(r);
        b2 = r - a * topk;
      } else {
        int off = 0;
        k = 0;
        while (y - off >= sh.f1[k] * sh.f2[k]) {
          off += sh.f1[k] * sh.f2[k];
          ++k;
        }
        const int r = y - off, f2 = sh.f2[k];
        a = r / f2;
        b2 = r - a * f2;
      }
      const bool own = sh.u1[CHK(k * topk + a, K * topk)];
      en.score = __fadd_rn(lp_s[CHK((k * L) * topk + a, KLT)], lp_s[CHK((k * L + 1) * topk + b2, KLT)]);
      en.k0 = 0;
      en.k1 = 2u | ((uint32_t)k << 25) | (own ? K1_OWNED : 0u);
      pk_set(en.k0, en.k1, 1, (uint32_t)a);
      pk_set(en.k0, en.k1, 2, (uint32_t)b2);
      return own;
    };
    auto bin_of = [&](float score) { return (int)((desc_key(score) >> shift) & 255u); };
    if (pairs && !two) {
      int *hall = hist + 512;  // every pair and depth-1 entry, owned or not
      for (int x = tid; x < N1 + N2; x += THREADS) {
        PE en;
        const bool own = make(x, en);
        const int b = bin_of(en.score);
        if (own) atomicAdd(&hist[b], 1);
        atomicAdd(&hall[b], 1);
      }
      block_sync();
      if (warp == 0) {
        // the first digit's boundary bin for the B-th owned entry (as in
        // bound_owned), and how many entries lie within it
        int c8[8], sum = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          c8[b] = hist[lane * 8 + b];
          sum += c8[b];
        }
        int run = warp_excl_scan(sum, lane);
        const int total = __shfl_sync(0xffffffffu, run + sum, 31);
        int bs = 256;
        if (total >= B) {
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            if (run < B && B <= run + c8[b]) bs = lane * 8 + b;
            run += c8[b];
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bs = min(bs, __shfl_xor_sync(0xffffffffu, bs, o));
        int within = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) within += lane * 8 + b <= bs ? hall[lane * 8 + b] : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) within += __shfl_xor_sync(0xffffffffu, within, o);
        if (lane == 0 && bs < 256 && within <= CAP) {
          const uint32_t prefix = shift + 8 >= 32 ? 0u : (kmin >> (shift + 8)) << (shift + 8);
          sh.tau = prefix | ((uint32_t)bs << shift) | ((1u << shift) - 1u);
          sh.cut2 = 1;
        }
      }
      block_sync();
      if (sh.cut2) {
        // every entry within that first bound; the others can neither be in
        // the tree nor lead to it
        const uint32_t tau0 = sh.tau;
        for (int base = warp * 32; base < N1 + N2; base += THREADS) {
          const int x = base + lane;
          PE en;
          bool want = false;
          if (x < N1 + N2) {
            make(x, en);
            want = desc_key(en.score) <= tau0;
          }
          const int slot = warp_append(&sh.n_ent, want);
          if (want) {
            ent[CHK(slot, CAP)] = en;
            nxt[CHK(slot, CAP)] = x < N1 ? (uint8_t)topk : 0;
          }
        }
      } else {
        for (int x = tid; x < N1; x += THREADS) {
          PE en;
          make(x, en);
          ent[CHK(x, CAP)] = en;
          nxt[CHK(x, CAP)] = 0;
        }
        if (tid == 0) sh.n_ent = N1;
      }
    } else {
      for (int base = warp * 32; base < N1 + N2; base += THREADS) {
        const int x = base + lane;
        int bin = -1;
        if (x < N1 + N2) {
          PE en;
          const bool own = make(x, en);
          ent[CHK(x, CAP)] = en;
          nxt[CHK(x, CAP)] = x < N1 && two ? (uint8_t)topk : 0;
          if (own) bin = bin_of(en.score);
        }
        if (bin >= 0) atomicAdd(&hist[bin], 1);  // bins here are mostly distinct within a warp
      }
      if (tid == 0) sh.n_ent = N1 + N2;
    }
  }
  block_sync();
  const bool cut2 = sh.cut2;

  // The bound: the B-th best score key among the owned entries (distinct
  // prefixes, each scoring no better than its mixture score), found to 8
  // bits below the highest bit where the owned keys differ, rounded to the
  // worse end of its bin.  sh.has_tau = 0 while fewer than B entries are owned.
  auto no_group = [](int) { return -1; };
  auto set_tau = [&](bool pre) { bound_owned(sh, ent, hist, B, pre); };

  // prune to each mode's exact B best (only when the pool is full)
  auto prune_exact = [&]() {
    radix_bound(sh, ent, sh.n_ent, K, B, 4, hist, hist + MAX_GROUPS * 256, false, mode_of, no_group);
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
            r += seq_cmp(c, g, e) < 0;
          }
          kp = r <= sh.rem[k];
        }
      }
      flg[i] = kp;
    }
    block_sync();
    const int out = compact_by_flag(sh, ent, nxt, n, flg);
    if (tid == 0) sh.n_ent = out;
    block_sync();
  };

  // ---------------------------------------------------- level expansion
  bool failed = false, tau_current = false;
  int n_cut = -1;  // pool size right after the last cut to the bound (-1: none yet)
  for (int t = two || cut2 ? 2 : 1; t < L && !failed; ++t) {
    if (tid == 0) sh.any = 0;
    int pass = 0;
    for (; pass < MAX_PASSES; ++pass) {
      int n_pool = -1;
      if (t == 1 && pass == 0 && topk < B) {
        if (tid == 0) sh.has_tau = 0;  // each mode holds only its topk depth-1 entries
        tau_current = true;
      } else {
        // The bound only tightens as entries are added, so an earlier one stays
        // valid (only looser): it is recomputed, and the pool cut to it, once
        // the pool has grown by a quarter since the last cut, after a prune,
        // or while there is none.
        const int ne = sh.n_ent;
        if (n_cut < 0 || pass > 0 || !sh.has_tau || ne > n_cut + (n_cut >> 2) + 32) {
          set_tau(two && t == 2 && pass == 0);
          if (sh.has_tau) {
            // entries outside the bound can neither be in the tree nor lead to it
            const uint32_t tau = sh.tau;
            n_pool = compact_by_tau(sh, ent, nxt, sh.n_ent, tau);
            n_cut = n_pool;
          }
          tau_current = true;
        }
      }
      if (tid == 0) {
        if (n_pool >= 0) sh.n_ent = n_pool;
        sh.overflow = 0;
        sh.n_par = 0;
      }
      block_sync();
      const int n0 = sh.n_ent;
      const bool ht = sh.has_tau;
      const uint32_t tau = sh.tau;
      // the parents of this level that can still reach the bound
      for (int base = warp * 32; base < n0; base += THREADS) {
        const int i = base + lane;
        bool isp = false;
        if (i < n0) {
          const PE e = ent[i];
          const int j = nxt[i];
          if (pk_depth(e.k1) == t && j < topk) {
            // the next rank is the best remaining child: if it misses the
            // bound, so do the others
            const float lv = lp_s[CHK((pk_mode(e.k1) * L + t) * topk + j, KLT)];
            isp = lv > -INFINITY && (!ht || desc_key(__fadd_rn(e.score, lv)) <= tau);
          }
        }
        const int k = warp_append(&sh.n_par, isp);
        if (isp && k < PLIST) plist[k] = (uint16_t)i;
      }
      block_sync();
      const int np = sh.n_par;
      if (np <= PLIST && np * topk <= PAIR_MAX && n0 + np * topk <= CAP) {
        // few parents and room for every child: all (parent, rank) pairs at once
        for (int base = warp * 32; base < np * topk; base += THREADS) {
          const int x = base + lane;
          bool want = false;
          PE ch;
          if (x < np * topk) {
            const int i = CHK(plist[CHK(x / topk, PLIST)], n0);
            const int j = x - (x / topk) * topk;
            const PE par = ent[i];
            const int row = (pk_mode(par.k1) * L + t) * topk;
            const float lv = lp_s[CHK(row + j, KLT)];
            if (j >= nxt[i] && lv > -INFINITY) {
              ch.score = __fadd_rn(par.score, lv);
              if (!ht || desc_key(ch.score) <= tau) {
                ch.k0 = par.k0;
                ch.k1 = par.k1 & ~31u;
                pk_set(ch.k0, ch.k1, t + 1, (uint32_t)j);
                ch.k1 |= (uint32_t)(t + 1);
                want = true;
              }
            }
          }
          const int slot = warp_append(&sh.n_ent, want);
          if (want) {
            ent[CHK(slot, CAP)] = ch;
            nxt[CHK(slot, CAP)] = 0;
          }
        }
        block_sync();
        for (int pi = tid; pi < np; pi += THREADS) nxt[CHK(plist[pi], n0)] = (uint8_t)topk;
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
              const float lv = lp_s[CHK(row + j, KLT)];
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
                  pk_set(ch.k0, ch.k1, t + 1, (uint32_t)j);
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
      block_sync();
      if (tid == 0) {
        if (sh.n_ent > CAP) sh.n_ent = CAP;
        if (sh.n_ent > n0) sh.any = 1;
      }
      block_sync();
      if (sh.any) tau_current = false;
      if (!sh.overflow) break;
      prune_exact();
    }
    if (pass == MAX_PASSES) failed = true;
    if (!sh.any) break;
  }
  if (failed) {
    if (tid == 0) report(prm.status, MFD_ERR_UNSUPPORTED);
    CHK_REPORT();
    return;
  }

  // ---------------------------------------------------- candidates
  if (!tau_current) {  // else: the pool was cut to the bound and nothing was added since
    set_tau(false);
    if (sh.has_tau) {
      const uint32_t tau = sh.tau;
      const int n = compact_by_tau(sh, ent, nxt, sh.n_ent, tau);
      if (tid == 0) sh.n_ent = n;
      block_sync();
    }
  }
  if (sh.n_ent > NC) {  // many ties within the bound: keep each mode's exact B best
    prune_exact();
    if (sh.n_ent > NC) {
      if (tid == 0) report(prm.status, MFD_ERR_UNSUPPORTED);
      CHK_REPORT();
      return;
    }
  }
  const int n = sh.n_ent;

  // ---------------------------------------------------- one entry per prefix
  // Open addressing on the sequence hash: a slot's tag is claimed by CAS
  // (read first), its first claimant is the representative every other entry
  // of the slot is compared with (a different sequence is a collision: the
  // table is rebuilt with another seed), and the best (score key, then mode)
  // of the slot is found by two 32-bit atomicMins.
  // Each entry also finds the slot of its parent sequence (its prefix one
  // token shorter), from the hash taken on the way.
  uint64_t seed = 0;
  constexpr int JH = 5;  // entries a thread hashes: n <= NC <= THREADS * JH
  for (int attempt = 0; attempt < 4; ++attempt) {
    for (int s = tid; s < tsize; s += THREADS) {
      tag[s] = 0;
      bkey[s] = 0xFFFFFFFFu;
      bsub[s] = 0xFFFFFFFFu;
    }
    if (tid == 0) {
      sh.coll = 0;
      sh.n_sel = 0;
    }
    block_sync();
    uint64_t hpr[JH];
#pragma unroll
    for (int jj = 0; jj < JH; ++jj) {
      const int i = tid + jj * THREADS;
      hpr[jj] = 0;
      if (i >= n) continue;
      const PE e = ent[i];
      const uint64_t h = seq_hash2(c, e, pk_depth(e.k1), seed, &hpr[jj]);
      const uint32_t tg = (uint32_t)(h >> 32) | 1u;
      uint32_t s = (uint32_t)h & (uint32_t)(tsize - 1);
      for (int probe = 0; probe < tsize; ++probe) {
        const uint32_t t0 = tag[s];
        if (t0 == tg) break;
        if (t0 == 0u) {
          const uint32_t prev = atomicCAS(&tag[s], 0u, tg);
          if (prev == 0u) {
            rep[CHK(s, tsize)] = (uint16_t)i;
            break;
          }
          if (prev == tg) break;
        }
        s = (s + 1) & (uint32_t)(tsize - 1);
      }
      hslot[CHK(i, NC)] = (uint16_t)s;
      atomicMin(&bkey[CHK(s, tsize)], desc_key(e.score));
    }
    block_sync();
#pragma unroll
    for (int jj = 0; jj < JH; ++jj) {
      const int i = tid + jj * THREADS;
      if (i >= n) continue;
      const PE e = ent[i];
      const int s = CHK(hslot[i], tsize);
      const int r = CHK(rep[s], n);
      if (r != i && seq_cmp(c, e, ent[r]) != 0) sh.coll = 1;
      if (desc_key(e.score) == bkey[s]) atomicMin(&bsub[s], ((uint32_t)pk_mode(e.k1) << 16) | (uint32_t)i);
      // the parent's slot: same tag, a representative one token shorter
      // with the same tokens
      const int d = pk_depth(e.k1);
      uint16_t ps = 0xFFFFu;
      if (d > 1) {
        const uint32_t tg = (uint32_t)(hpr[jj] >> 32) | 1u;
        uint32_t q = (uint32_t)hpr[jj] & (uint32_t)(tsize - 1);
        for (int probe = 0; probe < tsize; ++probe) {
          const uint32_t t0 = tag[q];
          if (t0 == 0u) break;
          if (t0 == tg) {
            const PE g = ent[CHK(rep[q], n)];
            bool same = pk_depth(g.k1) == d - 1;
            for (int p = 1; p < d && same; ++p) same = token_at(c, g, p) == token_at(c, e, p);
            if (same) {
              ps = (uint16_t)q;
              break;
            }
          }
          q = (q + 1) & (uint32_t)(tsize - 1);
        }
      }
      pslot[CHK(i, NC)] = ps;
    }
    block_sync();
    if (!sh.coll) break;
    seed = mix64(seed + 0x9E3779B97F4A7C15ull);
    block_sync();
  }
  if (sh.coll) {
    if (tid == 0) report(prm.status, MFD_ERR_UNSUPPORTED);
    CHK_REPORT();
    return;
  }
  // primaries; with few candidates every primary is selected right away
  // (sh.n_sel was zeroed before the last barrier of the table rounds)
  for (int base = warp * 32; base < n; base += THREADS) {
    const int i = base + lane;
    bool pr = false;
    if (i < n) {
      pr = (int)(bsub[CHK(hslot[i], tsize)] & 0xFFFF) == i;
      prim[i] = pr;
      nodeid[i] = -1;
    }
    if (n <= RANK_ALL) {
      const int k = warp_append(&sh.n_sel, pr);
      if (pr) {
        sel[CHK(k, NC)] = (uint16_t)i;
        skk[CHK(k, NC)] = desc_key(ent[i].score);
      }
    }
  }
  block_sync();

  // ---------------------------------------------------- the B best prefixes
  // With few candidates every primary is ranked; otherwise a radix bound on
  // the primaries' score keys first leaves about B of them.
  if (n > RANK_ALL) {
    radix_bound(sh, ent, n, 1, B, 2, hist1, hist1 + 256, false, [&](int i) { return prim[i] ? 0 : -1; }, no_group);
    const bool ht_sel = sh.act[0];
    const uint32_t tau_sel = sh.pre[0] | 0xFFFFu;
    if (tid == 0) sh.n_sel = 0;
    block_sync();
    for (int base = warp * 32; base < n; base += THREADS) {
      const int i = base + lane;
      const bool in = i < n && prim[i] && (!ht_sel || desc_key(ent[i].score) <= tau_sel);
      const int k = warp_append(&sh.n_sel, in);
      if (in) {
        sel[CHK(k, NC)] = (uint16_t)i;
        skk[CHK(k, NC)] = desc_key(ent[i].score);
      }
    }
    block_sync();
  }
  const int ns = sh.n_sel;
  const int nruns = (ns + 31) >> 5;
  // rank of each selected prefix = how many others come before it.  Runs of
  // 32 are sorted by (score key, selection index) in registers; a prefix's
  // rank is its place in its run plus, per other run, the keys below its own
  // (a branch-free binary search).  Equal keys of different prefixes are
  // ordered by their token sequences instead, on a slow path.
  for (int r = warp; r < nruns; r += NWARPS) {
    const int a = r * 32 + lane;
    uint32_t key = a < ns ? skk[a] : 0xFFFFFFFFu;
    int ia = a;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const uint32_t ok = __shfl_xor_sync(0xffffffffu, key, j);
        const int oi = __shfl_xor_sync(0xffffffffu, ia, j);
        const bool other_less = ok < key || (ok == key && oi < ia);
        const bool keep_min = ((lane & j) == 0) == ((lane & k) == 0);
        if (keep_min == other_less) {
          key = ok;
          ia = oi;
        }
      }
    }
    skk[a] = key;
    ra[a] = (uint16_t)ia;
  }
  block_sync();
  for (int r = warp; r < nruns; r += NWARPS) {
    const int pos = r * 32 + lane;
    const uint32_t key = skk[pos];
    const int ia = ra[pos];
    const bool real = ia < ns;
    int lt = lane;  // the run's entries before this one
    bool tie = (__popc(__match_any_sync(0xffffffffu, key)) > 1) && real;
    for (int r0 = 0; r0 < nruns; r0 += 4) {
      // four independent searches in flight
      int cnt[4] = {0, 0, 0, 0};
      const uint32_t *run[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) run[u] = skk + (r0 + u < nruns ? r0 + u : r) * 32;
#pragma unroll
      for (int st = 16; st > 0; st >>= 1)
#pragma unroll
        for (int u = 0; u < 4; ++u) cnt[u] += run[u][cnt[u] + st - 1] < key ? st : 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        cnt[u] += run[u][cnt[u]] < key ? 1 : 0;
        if (r0 + u < nruns && r0 + u != r) {
          lt += cnt[u];
          tie |= cnt[u] < 32 && run[u][cnt[u]] == key;
        }
      }
    }
    if (real && tie) {
      // keys below, then token order among the equal keys: per run, the
      // keys below its lower bound, then its block of equal keys
      lt = 0;
      const PE ea = ent[CHK(sel[CHK(ia, NC)], n)];
      for (int u = 0; u < nruns; ++u) {
        const uint32_t *run = skk + u * 32;
        int lo = 0;
#pragma unroll
        for (int st = 16; st > 0; st >>= 1) lo += run[lo + st - 1] < key ? st : 0;
        lo += run[lo] < key ? 1 : 0;
        lt += lo;
        for (int p = lo; p < 32 && run[p] == key; ++p) {
          const int b = u * 32 + p;
          if (ra[b] != ia && ra[b] < ns && seq_cmp(c, ent[CHK(sel[ra[b]], n)], ea) < 0) ++lt;
        }
      }
    }
    if (real && lt < B) {
      nslot[CHK(lt + 1, B + 1)] = sel[CHK(ia, NC)];
      nodeid[CHK(sel[CHK(ia, NC)], NC)] = (int16_t)(lt + 1);
    }
  }
  if (tid == 0) {
    par_s[0] = -1;
    sh.bad = 0;
  }
  block_sync();
  const int nn = ns < B ? ns : B;

  // ---------------------------------------------------- parents
  for (int nd = 1 + tid; nd <= nn; nd += THREADS) {
    const int i = CHK(nslot[nd], n);
    int par = 0;
    if (pk_depth(ent[i].k1) > 1) {
      const int ps = pslot[i];
      par = ps == 0xFFFF ? -1 : nodeid[CHK(bsub[CHK(ps, tsize)] & 0xFFFF, NC)];
      if (par < 1 || par >= nd) sh.bad = 1;
    }
    par_s[nd] = (int16_t)par;
  }
  block_sync();
  if (sh.bad) {
    if (tid == 0) report(prm.status, MFD_ERR_INPUT);
    CHK_REPORT();
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
      const PE e = ent[CHK(nslot[nd], n)];
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
  // mask rows: one ancestor walk per node, its words gathered in a small
  // per-thread array (N <= 513 nodes: at most 17 words)
  for (int i = tid; i < N; i += THREADS) {
    uint32_t m[MAX_MASK_WORDS];
#pragma unroll
    for (int w = 0; w < MAX_MASK_WORDS; ++w) m[w] = 0u;
    if (i <= nn)
      for (int a = i; a >= 0; a = (a == 0) ? -1 : par_s[CHK(a, B + 1)]) m[CHK(a >> 5, MAX_MASK_WORDS)] |= 1u << (a & 31);
    uint32_t *row = prm.mask + ((size_t)q * N + i) * W32;
    for (int w = 0; w < W32; ++w) row[w] = m[w];
  }
  if (tid == 0) prm.n_nodes[q] = nn + 1;
  CHK_REPORT();
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
