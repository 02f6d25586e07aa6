// verify.cu -- the standard tree verification walk (model card "MFD drafter
// for Qwen3.5-4B", first paragraph; project page "Multi-Future Drafting",
// Figure 2 (c)): from the root, the target picks a token at the current node
// and the walk follows the child that carries it; the first miss gives the
// bonus token.  Greedy picks the argmax of the target's logits; sampled
// (temperature T > 0) picks argmax_v (t_v / T + G_v), a Gumbel-max draw from
// softmax(t / T) with counter-based noise, which keeps decoding lossless.
//
// Each step reduces one vocabulary row (V up to ~250K fp32) and the next
// step depends on its result, so the walk is a chain of short, wide
// reductions.  Two forms, one result:
//   - the grid walk (few requests): one cooperative grid covers the GPU; the
//     CTAs of a request's group split the row and publish (best value,
//     index) in tagged slots; the group's first CTA waits (bounded) for every
//     slot of the step, publishes the winner in one tagged word, and the
//     others wait (bounded) on that word.  A sampled row's Philox and
//     logarithms are spread over the whole GPU.
//   - the cluster walk (many requests): one thread-block cluster per
//     request; its CTAs exchange each step's results in their shared memory
//     behind a hardware cluster barrier, without polling memory.  Requests
//     run side by side, each on up to 16 SMs.
// Only rows on the walk are read.

#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int THREADS = 512;
constexpr int MAX_NODES = 513;
constexpr int NODE_SLOTS = (MAX_NODES + 31) / 32;  // node-table entries per lane

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11): the block
// at counter (c0, c1, 0, 0) and key (k0, k1).  A round maps (x0, x1, x2, x3)
// to (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)); the
// key advances by the two Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4(uint32_t c0, uint32_t c1, uint32_t k0, uint32_t k1) {
  uint32_t x0 = c0, x1 = c1, x2 = 0u, x3 = 0u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, x0), lo0 = 0xD2511F53u * x0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, x2), lo1 = 0xCD9E8D57u * x2;
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(x0, x1, x2, x3);
}

// G = -log(-log u), u = (2 (x >> 9) + 1) 2^-24 in (0, 1), for one word x.
__device__ __forceinline__ float gumbel_of(uint32_t x) {
  const float u = __fmul_rn((float)(2u * (x >> 9) + 1u), 0x1p-24f);
  return -logf(-logf(u));
}

// G(seed, node, v): word v mod 4 of the Philox block at counter (v div 4,
// node), key (seed low, seed high).
__device__ __forceinline__ float gumbel(uint64_t seed, int node, int v) {
  const uint4 b = philox4((uint32_t)v >> 2, (uint32_t)node, (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t j = (uint32_t)v & 3u;
  return gumbel_of(j == 0 ? b.x : j == 1 ? b.y : j == 2 ? b.z : b.w);
}

// ============================================================ grid walk

// A published step result: one 64-bit word, value in bits 63..32,
// vocabulary index in bits 31..2 (0x3FFFFFFF = none; V < 2^30), and a 2-bit
// tag in bits 1..0.  Result words are double-buffered by step parity; step e
// writes tag 1 + ((e >> 1) & 1), which differs from the tag step e - 2 left
// in the same word and from zero.
//
// No zeroing pass is needed before a call.  The workspace holds, per group, a
// generation word gen; every CTA reads it at the start (all read the same
// value, see below), and with G = gen + 1:
//   - each CTA clears the result words it will write, then stores G into its
//     ready word with release semantics;
//   - a reader waits until the writer's ready word holds G and takes it with
//     acquire semantics before it trusts that writer's result words: what it
//     then reads is the clear or a value of this call, never an earlier call's;
//   - the group's first CTA stores G into gen when it leaves, after it has
//     acquired every ready word of the group, so every CTA of the group read
//     gen before that store; the next call therefore uses G + 1, and a ready
//     word left by an earlier call never matches (also under graph replay).
// Workspace contents left by other calls only matter if a ready word happens
// to equal its group's gen + 1, which fresh, zeroed or pattern-filled memory
// does not.
constexpr uint32_t IDX_NONE = 0x3FFFFFFFu;

__device__ __forceinline__ unsigned long long slot_pack(float v, int i, unsigned tag) {
  const uint32_t ii = (i >= 0 && (uint32_t)i < IDX_NONE) ? (uint32_t)i : IDX_NONE;
  return ((unsigned long long)__float_as_uint(v) << 32) | ((unsigned long long)ii << 2) | tag;
}
__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_relaxed(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

struct GridParams {
  const float *t;
  int n_req, B, V, L;
  const int32_t *parent, *token, *n_nodes;
  const float *temperature;
  const uint64_t *seed;
  int32_t *accept_len, *path_nodes, *out_tokens, *status;
  unsigned long long *ws;  // [grid][8] words: see Ws
  int cpr;                    // CTAs per request group
  unsigned long long wait_ns;  // limit of every bounded wait
  int withhold;                // fault injection: CTAs other than a group's first never publish their slot
};

// Workspace words, 7 per CTA of the grid: per group g its gen, its leader's
// ready word and its result words; per CTA b its ready word and result words.
struct Ws {
  unsigned long long *base;
  int grid;
  __device__ unsigned long long *gen(int g) const { return base + g; }
  __device__ unsigned long long *lready(int g) const { return base + grid + g; }
  __device__ unsigned long long *res(int g, unsigned par) const { return base + 2 * grid + 2 * g + par; }
  __device__ unsigned long long *ready(int b) const { return base + 4 * grid + b; }
  __device__ unsigned long long *slot(int b, unsigned par) const { return base + 5 * grid + 2 * b + par; }
};

constexpr int POLL_SLOTS = 8;                       // group slots a lane polls (cpr <= 256)
constexpr int PRE = 4;                              // root-row entries a thread loads up front


// Per step: every thread scans its share of the row (loads first, then the
// arithmetic), the CTA reduces to one (value, index), warp 0 exchanges it
// with the group (above), takes the winner y and looks for the child of cur
// carrying y in the node table it holds in registers (tokens of a node's
// children are distinct, so at most one matches).  Two block barriers per
// step.
__global__ void __launch_bounds__(THREADS) verify_grid_kernel(const GridParams p) {
  __shared__ float red_v[THREADS / 32];
  __shared__ int red_i[THREADS / 32];
  __shared__ int s_next, s_ok;
  __shared__ unsigned long long s_G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cpr = p.cpr;
  const int grp = blockIdx.x / cpr, c = blockIdx.x - grp * cpr;
  const int n_groups = gridDim.x / cpr;
  unsigned epoch = 0;
  const int N = p.B + 1;
  const Ws ws{p.ws, (int)gridDim.x};
  // generation handshake (see the comment on the result words)
  // done by the last warp, so that warp 0's loads go out first; warp 0 takes
  // G from shared memory after the first block barrier
  // The tree and the target rows may come from the grids just before; the
  // next grid may start its prologue now (it waits for this one to end).
  // No CTA waits on another before the grid before has ended and freed its
  // SMs for the rest of this (cooperative) grid.
  pdl_wait();
  pdl_launch_dependents();
  bool acquired = false;  // this CTA has taken the ready words it reads
  unsigned long long rdy[POLL_SLOTS];  // ready words read early (warp 0)
#pragma unroll
  for (int j = 0; j < POLL_SLOTS; ++j) rdy[j] = 0ull;
  if (cpr > 1 && warp == THREADS / 32 - 1) {
    if (lane == 0) {
      const unsigned long long G = ld_relaxed(ws.gen(grp)) + 1ull;
      s_G = G;
      if (c == 0) {
        st_relaxed(ws.res(grp, 0), 0ull);
        st_relaxed(ws.res(grp, 1), 0ull);
        st_release(ws.lready(grp), G);
      } else {
        st_relaxed(ws.slot(blockIdx.x, 0), 0ull);
        st_relaxed(ws.slot(blockIdx.x, 1), 0ull);
        st_release(ws.ready(blockIdx.x), G);
      }
    }
  }

  for (int q = grp; q < p.n_req; q += n_groups) {
    const int v0 = (int)(((long long)c * p.V) / cpr), v1 = (int)(((long long)(c + 1) * p.V) / cpr);
    // the root's row and the node table do not depend on anything the walk
    // computes: their loads go out first, with the request's parameters
    float pre[PRE];
    {
      const float *row0 = p.t + (size_t)q * N * (size_t)p.V;
#pragma unroll
      for (int k = 0; k < PRE; ++k) {
        const int v = v0 + tid + k * THREADS;
        pre[k] = v < v1 ? __ldcs(row0 + v) : 0.f;
      }
    }
    int par_r[NODE_SLOTS], tok_r[NODE_SLOTS];
    if (warp == 0) {
#pragma unroll
      for (int j = 0; j < NODE_SLOTS; ++j) {
        const int i = j * 32 + lane;
        par_r[j] = i < N ? __ldg(p.parent + (size_t)q * N + i) : -2;
        tok_r[j] = i < N ? __ldg(p.token + (size_t)q * N + i) : -2;
      }
    }
    const int n = p.n_nodes[q];
    const float T = p.temperature[q];
    const uint64_t seed = p.seed[q];
    if (!(n >= 1 && n <= N) || !(T >= 0.f)) {
      if (c == 0 && tid == 0) {
        report(p.status, MFD_ERR_INPUT);
        p.accept_len[q] = 0;
      }
      continue;
    }
    if (warp == 0) {
#pragma unroll
      for (int j = 0; j < NODE_SLOTS; ++j)
        if (j * 32 + lane >= n) par_r[j] = -2;
      if (cpr > 1 && !acquired) {
        // read the ready words now; they are checked at the first exchange
        if (c == 0) {
#pragma unroll
          for (int j = 0; j < POLL_SLOTS; ++j) {
            const int k = 1 + lane + 32 * j;
            if (k < cpr) rdy[j] = ld_relaxed(ws.ready(grp * cpr + k));
          }
        } else if (lane == 0) {
          rdy[0] = ld_relaxed(ws.lready(grp));
        }
      }
    }
    int cur = 0, accepted = 0;
    for (int step = 0; step <= p.L; ++step) {
      const float *row = p.t + ((size_t)q * N + cur) * (size_t)p.V;
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
      int v = v0 + tid;
      if (step == 0) {
#pragma unroll
        for (int k = 0; k < PRE; ++k, v += THREADS) {
          if (v < v1) {
            const float a = T == 0.f ? pre[k] : __fadd_rn(__fdiv_rn(pre[k], T), gumbel(seed, cur, v));
            if (vi_before(a, v, bv, bi)) { bv = a; bi = v; }
          }
        }
      }
      if (T == 0.f) {
        for (; v + 3 * THREADS < v1; v += 4 * THREADS) {
          const float a0 = __ldcs(row + v), a1 = __ldcs(row + v + THREADS), a2 = __ldcs(row + v + 2 * THREADS),
                      a3 = __ldcs(row + v + 3 * THREADS);
          if (vi_before(a0, v, bv, bi)) { bv = a0; bi = v; }
          if (vi_before(a1, v + THREADS, bv, bi)) { bv = a1; bi = v + THREADS; }
          if (vi_before(a2, v + 2 * THREADS, bv, bi)) { bv = a2; bi = v + 2 * THREADS; }
          if (vi_before(a3, v + 3 * THREADS, bv, bi)) { bv = a3; bi = v + 3 * THREADS; }
        }
        for (; v < v1; v += THREADS) {
          const float a = __ldcs(row + v);
          if (vi_before(a, v, bv, bi)) { bv = a; bi = v; }
        }
      } else {
        for (; v + THREADS < v1; v += 2 * THREADS) {
          const float t0 = __ldcs(row + v), t1 = __ldcs(row + v + THREADS);
          const float a0 = __fadd_rn(__fdiv_rn(t0, T), gumbel(seed, cur, v));
          const float a1 = __fadd_rn(__fdiv_rn(t1, T), gumbel(seed, cur, v + THREADS));
          if (vi_before(a0, v, bv, bi)) { bv = a0; bi = v; }
          if (vi_before(a1, v + THREADS, bv, bi)) { bv = a1; bi = v + THREADS; }
        }
        for (; v < v1; v += THREADS) {
          const float a = __fadd_rn(__fdiv_rn(__ldcs(row + v), T), gumbel(seed, cur, v));
          if (vi_before(a, v, bv, bi)) { bv = a; bi = v; }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (vi_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) {
        red_v[warp] = bv;
        red_i[warp] = bi;
      }
      block_sync();
      if (warp == 0) {
        bv = lane < THREADS / 32 ? red_v[lane] : -INFINITY;
        bi = lane < THREADS / 32 ? red_i[lane] : 0x7FFFFFFF;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (vi_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        int ok = 1;
        if (cpr > 1) {
          // CTA 0 of the group gathers the other CTAs' slots and publishes
          // the winner in the group's result word; the others publish their
          // slot and poll that one word (a few pollers per cache line)
          const unsigned par = epoch & 1u, tag = 1u + ((epoch >> 1) & 1u);
          const unsigned long long t_start = globaltimer();
          const unsigned long long G = s_G;
          if (c == 0) {
            // tag and payload share one 64-bit word, so relaxed loads
            // suffice; a lane's slots are read at once and only the ones
            // without the tag are read again
            const int b0 = grp * cpr;
            if (!acquired) {
              // every other CTA of the group has cleared its result words
              for (;;) {
                bool all = true;
#pragma unroll
                for (int j = 0; j < POLL_SLOTS; ++j) all &= 1 + lane + 32 * j >= cpr || rdy[j] == G;
                if (all) break;
                if (globaltimer() - t_start > p.wait_ns) {
                  ok = 0;
                  break;
                }
#pragma unroll
                for (int j = 0; j < POLL_SLOTS; ++j)
                  if (1 + lane + 32 * j < cpr && rdy[j] != G) rdy[j] = ld_relaxed(ws.ready(b0 + 1 + lane + 32 * j));
              }
              fence_acq_rel();
              acquired = true;
            }
            const unsigned long long *sp = ws.slot(b0, par);
            unsigned long long w[POLL_SLOTS];
#pragma unroll
            for (int j = 0; j < POLL_SLOTS; ++j) {
              const int k = 1 + lane + 32 * j;
              w[j] = k < cpr ? ld_relaxed(sp + (size_t)k * 2) : (unsigned long long)tag;
            }
            for (; ok;) {
              bool all = true;
#pragma unroll
              for (int j = 0; j < POLL_SLOTS; ++j) all &= (unsigned)(w[j] & 3ull) == tag;
              if (all) break;
              if (globaltimer() - t_start > p.wait_ns) {
                ok = 0;
                break;
              }
#pragma unroll
              for (int j = 0; j < POLL_SLOTS; ++j) {
                const int k = 1 + lane + 32 * j;
                if ((unsigned)(w[j] & 3ull) != tag) w[j] = ld_relaxed(sp + (size_t)k * 2);
              }
            }
#pragma unroll
            for (int j = 0; j < POLL_SLOTS; ++j) {
              const int k = 1 + lane + 32 * j;
              if (k >= cpr) continue;
              const float wv = __uint_as_float((uint32_t)(w[j] >> 32));
              const uint32_t wi = (uint32_t)(w[j] >> 2) & IDX_NONE;
              const int wii = wi == IDX_NONE ? 0x7FFFFFFF : (int)wi;
              if (vi_before(wv, wii, bv, bi)) { bv = wv; bi = wii; }
            }
            ok = __all_sync(0xffffffffu, ok);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
              const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
              if (vi_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            if (lane == 0 && ok) st_relaxed(ws.res(grp, par), slot_pack(bv, bi, tag));
          } else {
            unsigned long long w = 0ull;
            if (lane == 0) {
              if (!p.withhold) st_relaxed(ws.slot(blockIdx.x, par), slot_pack(bv, bi, tag));
              if (!acquired) {
                // the group's first CTA has cleared the result words
                while (rdy[0] != G) {
                  if (globaltimer() - t_start > p.wait_ns) {
                    ok = 0;
                    break;
                  }
                  rdy[0] = ld_relaxed(ws.lready(grp));
                }
                fence_acq_rel();
              }
              w = ld_relaxed(ws.res(grp, par));
              while (ok && (unsigned)(w & 3ull) != tag) {
                if (globaltimer() - t_start > p.wait_ns) {
                  ok = 0;
                  break;
                }
                w = ld_relaxed(ws.res(grp, par));
              }
            }
            acquired = true;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            const uint32_t wi = (uint32_t)(__shfl_sync(0xffffffffu, w, 0) >> 2) & IDX_NONE;
            bi = wi == IDX_NONE ? 0x7FFFFFFF : (int)wi;
          }
          ++epoch;
        }
        // the child of cur that carries y = bi
        int nx = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < NODE_SLOTS; ++j) {
          const unsigned hit = __ballot_sync(0xffffffffu, par_r[j] == cur && tok_r[j] == bi && j * 32 + lane >= 1);
          if (hit && nx == 0x7FFFFFFF) nx = j * 32 + __ffs(hit) - 1;
        }
        if (lane == 0) {
          s_next = nx;
          s_ok = ok;
          if (c == 0 && ok) {
            p.path_nodes[(size_t)q * (p.L + 1) + step] = cur;
            p.out_tokens[(size_t)q * (p.L + 1) + step] = bi;
          }
        }
      }
      block_sync();
      if (!s_ok) {
        if (tid == 0) {
          report(p.status, MFD_ERR_TIMEOUT);
          if (c == 0) st_relaxed(ws.gen(grp), s_G);
        }
        return;
      }
      const int nx = s_next;
      if (nx == 0x7FFFFFFF || step == p.L) break;
      cur = nx;
      accepted = step + 1;
    }
    if (c == 0 && tid == 0) {
      p.accept_len[q] = accepted;
      for (int j = accepted + 1; j <= p.L; ++j) {
        p.path_nodes[(size_t)q * (p.L + 1) + j] = -1;
        p.out_tokens[(size_t)q * (p.L + 1) + j] = -1;
      }
    }
  }
  // the next call on this workspace uses the next generation
  if (c == 0 && tid == 0 && epoch > 0) st_relaxed(ws.gen(grp), s_G);
}

// ============================================================ cluster walk

constexpr int MAX_CLUSTER = 16;
constexpr int MAXG = 8;  // groups of four entries a thread loads at once (all in flight together)

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives, then waits: a hardware
// barrier over CTAs that are resident together by construction.  The
// .aligned forms want every thread of the warp to execute them together, so
// each first reconverges the warp.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  __syncwarp();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// `p` (this CTA's shared memory) as the address of the same variable in CTA
// `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// A step result: value bits 63..32, vocabulary index 31..0.
__device__ __forceinline__ unsigned long long pack_vi(float v, int i) {
  return ((unsigned long long)__float_as_uint(v) << 32) | (uint32_t)i;
}

struct ClusterParams {
  const float *t;
  int n_req, B, V, L;
  const int32_t *parent, *token, *n_nodes;
  const float *temperature;
  const uint64_t *seed;
  int32_t *accept_len, *path_nodes, *out_tokens, *status;
  int vec4;  // rows are 16-byte aligned (V % 4 == 0, t 16-byte aligned): float4 loads
};

// Entries 4g .. 4g + 3 of a row (-inf past V).
__device__ __forceinline__ float4 load4(const float *row, int g, int V, bool vec4) {
  if (vec4) return __ldcs(reinterpret_cast<const float4 *>(row) + g);
  const int v = 4 * g;
  float4 x;
  x.x = v < V ? __ldcs(row + v) : -INFINITY;
  x.y = v + 1 < V ? __ldcs(row + v + 1) : -INFINITY;
  x.z = v + 2 < V ? __ldcs(row + v + 2) : -INFINITY;
  x.w = v + 3 < V ? __ldcs(row + v + 3) : -INFINITY;
  return x;
}

// Folds entries 4g .. 4g + 3 into (bv, bi): the logit itself at T = 0, else
// t / T + G with the noise of word j of the Philox block (g, node).
__device__ __forceinline__ void fold4(float4 x, int g, int V, float T, int node, uint64_t seed, float &bv, int &bi) {
  const float xs[4] = {x.x, x.y, x.z, x.w};
  const int v = 4 * g;
  if (T == 0.f) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (v + j < V && vi_before(xs[j], v + j, bv, bi)) {
        bv = xs[j];
        bi = v + j;
      }
  } else {
    const uint4 w = philox4((uint32_t)g, (uint32_t)node, (uint32_t)seed, (uint32_t)(seed >> 32));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (v + j >= V) continue;
      // x / 1 = x exactly, so T = 1 needs no division
      const float tq = T == 1.f ? xs[j] : __fdiv_rn(xs[j], T);
      const float a = __fadd_rn(tq, gumbel_of(ws[j]));
      if (vi_before(a, v + j, bv, bi)) {
        bv = a;
        bi = v + j;
      }
    }
  }
}

__device__ __forceinline__ void warp_best(float &bv, int &bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (vi_before(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
}

// Per step: every thread scans its groups of four entries of the row, the
// CTA reduces to one (value, index) in warp 0, warp 0 writes it into slot
// [step parity][rank] of every CTA of the cluster, and after the cluster
// barrier every warp of every CTA reduces the cluster's slots to the same
// winner y and looks for the child of cur carrying y in the node table the
// CTA holds in shared memory (the tokens of a node's children are distinct).
// (Measured: with warp 0 alone doing this while the other warps waited at a
// block barrier, its shuffles and ballots took about 250 cycles each.)  The slots are
// double-buffered by step parity: a CTA writes step e + 1's slots only after
// step e's barrier, which every CTA reaches after reading step e - 1's.
// After the last barrier no CTA touches another's shared memory, so the CTAs
// may leave in any order.
__global__ void __launch_bounds__(THREADS, 1) verify_cluster_kernel(const ClusterParams p) {
  __shared__ float red_v[THREADS / 32];
  __shared__ int red_i[THREADS / 32];
  __shared__ unsigned long long xs[2][MAX_CLUSTER];
  __shared__ int par_s[NODE_SLOTS * 32], tok_s[NODE_SLOTS * 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = (int)cluster_count(), c = (int)cluster_rank();
  const int q = (int)cluster_index();
  const int N = p.B + 1, V = p.V;
  const bool vec4 = p.vec4 != 0;
  // groups of four entries; CTA c of the cluster scans groups [g0, g1)
  const int G4 = (V + 3) >> 2;
  const int g0 = (int)(((long long)c * G4) / C), g1 = (int)(((long long)(c + 1) * G4) / C);
  pdl_wait();  // the tree and the target rows may come from the grids just before
  pdl_launch_dependents();
  const int n = p.n_nodes[q];
  const float T = p.temperature[q];
  if (!(n >= 1 && n <= N) || !(T >= 0.f)) {
    // every CTA of the cluster reads the same n and T: all leave here,
    // before any barrier
    if (c == 0 && tid == 0) {
      report(p.status, MFD_ERR_INPUT);
      p.accept_len[q] = 0;
    }
    return;
  }
  const uint64_t seed = p.seed[q];
  // the node table: its loads go out first, next the first row's, and the
  // table is stored into shared memory after the first row is folded (it is
  // read after the first block barrier)
  int np_[2], nt_[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = tid + k * THREADS;
    np_[k] = i < n ? __ldg(p.parent + (size_t)q * N + i) : -2;
    nt_[k] = i < n ? __ldg(p.token + (size_t)q * N + i) : -2;
  }
  // this CTA has started: nothing is written into its shared memory by
  // another CTA before every CTA of the cluster has arrived here
  cluster_arrive_relaxed();
  float4 xv[MAXG];
  int cur = 0, accepted = 0;
  for (int step = 0; step <= p.L; ++step) {
    const float *row = p.t + ((size_t)q * N + cur) * (size_t)V;
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    // a thread's groups MAXG at a time: all loads first, one round trip
    for (int gb = g0 + tid; gb < g1; gb += MAXG * THREADS) {
#pragma unroll
      for (int k = 0; k < MAXG; ++k) {
        const int g = gb + k * THREADS;
        if (g < g1) xv[k] = load4(row, g, V, vec4);
      }
#pragma unroll
      for (int k = 0; k < MAXG; ++k) {
        const int g = gb + k * THREADS;
        if (g < g1) fold4(xv[k], g, V, T, cur, seed, bv, bi);
      }
    }
    if (step == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = tid + k * THREADS;
        if (i < NODE_SLOTS * 32) {
          par_s[i] = np_[k];
          tok_s[i] = nt_[k];
        }
      }
    }
    warp_best(bv, bi);
    if (lane == 0) {
      red_v[warp] = bv;
      red_i[warp] = bi;
    }
    block_sync();
    if (step == 0) cluster_wait();  // every CTA of the cluster has started
    const unsigned par = (unsigned)step & 1u;
    if (warp == 0) {
      bv = lane < THREADS / 32 ? red_v[lane] : -INFINITY;
      bi = lane < THREADS / 32 ? red_i[lane] : 0x7FFFFFFF;
      warp_best(bv, bi);
      if (lane < C) st_cluster_u64(cluster_addr(&xs[par][c], (uint32_t)lane), pack_vi(bv, bi));
    }
    cluster_arrive();
    cluster_wait();
    // every warp takes the winner and the next node itself: no warp waits
    // for another here
    {
      const unsigned long long w = lane < C ? xs[par][lane] : pack_vi(-INFINITY, 0x7FFFFFFF);
      bv = __uint_as_float((uint32_t)(w >> 32));
      bi = (int)(uint32_t)w;
    }
    warp_best(bv, bi);
    // the child of cur that carries y = bi
    int nx = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < NODE_SLOTS; ++j) {
      const int i = j * 32 + lane;
      const unsigned hit = __ballot_sync(0xffffffffu, par_s[i] == cur && tok_s[i] == bi && i >= 1);
      if (hit && nx == 0x7FFFFFFF) nx = j * 32 + __ffs(hit) - 1;
    }
    if (c == 0 && tid == 0) {
      p.path_nodes[(size_t)q * (p.L + 1) + step] = cur;
      p.out_tokens[(size_t)q * (p.L + 1) + step] = bi;
    }
    if (nx == 0x7FFFFFFF || step == p.L) break;
    cur = nx;
    accepted = step + 1;
  }
  if (c == 0 && tid == 0) {
    p.accept_len[q] = accepted;
    for (int j = accepted + 1; j <= p.L; ++j) {
      p.path_nodes[(size_t)q * (p.L + 1) + j] = -1;
      p.out_tokens[(size_t)q * (p.L + 1) + j] = -1;
    }
  }
}

}  // namespace

int verify_max_grid(int n_sm) { return n_sm < 256 ? n_sm : 256; }

// CTAs per request group: enough that each CTA scans at least 1024 entries
// of a row, at most the whole grid.
static int verify_cpr(int grid, int n_req, int V) {
  const int n_groups = n_req < grid ? n_req : grid;
  int cpr = grid / n_groups;
  const int want = (V + 1023) / 1024;
  if (want < cpr) cpr = want;
  return cpr < 1 ? 1 : cpr;
}

static cudaError_t launch_grid(const VerifyLaunch &V, cudaStream_t stream) {
  GridParams p;
  p.t = V.t;
  p.n_req = V.n_req;
  p.B = V.B;
  p.V = V.V;
  p.L = V.L;
  p.parent = V.parent;
  p.token = V.token;
  p.n_nodes = V.n_nodes;
  p.temperature = V.temperature;
  p.seed = V.seed;
  p.accept_len = V.accept_len;
  p.path_nodes = V.path_nodes;
  p.out_tokens = V.out_tokens;
  p.status = V.status;
  p.ws = V.ws;
  p.cpr = verify_cpr(V.grid, V.n_req, V.V);
  p.wait_ns = V.wait_ns ? V.wait_ns : kWaitLimitNs;
  p.withhold = V.withhold;
  const int n_groups = V.n_req < V.grid ? V.n_req : V.grid;
  const int grid = (n_groups < V.grid / p.cpr ? n_groups : V.grid / p.cpr) * p.cpr;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_grid_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// CTAs per request: the smallest power of two that gives each CTA at most
// 1024 groups of four entries, up to the largest cluster this device runs.
int verify_cluster_size(int V) {
  static int cmax = 0;
  if (cmax == 0) {
    int c = 8;
    if (cudaFuncSetAttribute(verify_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(MAX_CLUSTER);
      cfg.blockDim = dim3(THREADS);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = MAX_CLUSTER;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, verify_cluster_kernel, &cfg) == cudaSuccess && n >= 1) c = MAX_CLUSTER;
    }
    (void)cudaGetLastError();
    cmax = c;
  }
  const int groups = (V + 3) / 4;
  int c = 1;
  while (c < cmax && (groups + c - 1) / c > 1024) c <<= 1;
  return c;
}

static cudaError_t launch_cluster(const VerifyLaunch &V, cudaStream_t stream) {
  ClusterParams p;
  p.t = V.t;
  p.n_req = V.n_req;
  p.B = V.B;
  p.V = V.V;
  p.L = V.L;
  p.parent = V.parent;
  p.token = V.token;
  p.n_nodes = V.n_nodes;
  p.temperature = V.temperature;
  p.seed = V.seed;
  p.accept_len = V.accept_len;
  p.path_nodes = V.path_nodes;
  p.out_tokens = V.out_tokens;
  p.status = V.status;
  p.vec4 = (V.V % 4 == 0 && (reinterpret_cast<uintptr_t>(V.t) % 16) == 0) ? 1 : 0;
  const int C = verify_cluster_size(V.V);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(V.n_req * C);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_cluster_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The grid walk below VERIFY_CLUSTER_REQUESTS requests, where a request's
// group holds many CTAs (one request's sampled row: about 4 us of Philox and
// logarithms on a 16-SM cluster, well under 1 us over the whole GPU); the
// cluster walk from there on, where the requests' clusters fill the GPU side
// by side and no step waits on a global exchange (32 requests: 51 us
// against 88 us).
cudaError_t launch_verify(const VerifyLaunch &V, cudaStream_t stream) {
  // (the fault injection of the grid walk's waits always takes the grid walk)
  return V.n_req >= VERIFY_CLUSTER_REQUESTS && !V.withhold ? launch_cluster(V, stream) : launch_grid(V, stream);
}

}  // namespace mfd
