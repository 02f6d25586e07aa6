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
// reductions.  One cooperative grid covers the GPU; the CTAs of a request's
// group split the row, publish (best value, index), meet at a bounded
// grid-group barrier and all read the winner.  Only rows on the walk are read.
#include <cooperative_groups.h>

#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int THREADS = 512;
constexpr int MAX_NODES = 513;

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11), word 0 of
// the block at counter (c0, c1, 0, 0) and key (k0, k1).  A round maps
// (x0, x1, x2, x3) to (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1,
// lo(M0 x0)); the key advances by the two Weyl constants between rounds.
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t k0, uint32_t k1) {
  uint32_t x0 = c0, x1 = c1, x2 = 0u, x3 = 0u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, x0), lo0 = 0xD2511F53u * x0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, x2), lo1 = 0xCD9E8D57u * x2;
    const uint32_t y0 = hi1 ^ x1 ^ k0, y2 = hi0 ^ x3 ^ k1;
    x0 = y0;
    x1 = lo1;
    x2 = y2;
    x3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return x0;
}

// G(seed, node, v) = -log(-log u), u = (2 (x >> 9) + 1) 2^-24 in (0, 1).
__device__ __forceinline__ float gumbel(uint64_t seed, int node, int v) {
  const uint32_t x = philox_word0((uint32_t)v, (uint32_t)node, (uint32_t)seed, (uint32_t)(seed >> 32));
  const float u = __fmul_rn((float)(2u * (x >> 9) + 1u), 0x1p-24f);
  return -logf(-logf(u));
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct Params {
  const float *t;
  int n_req, B, V, L;
  const int32_t *parent, *token, *n_nodes;
  const float *temperature;
  const uint64_t *seed;
  int32_t *accept_len, *path_nodes, *out_tokens, *status;
  unsigned *bar;
  float2 *part;
  int cpr;  // CTAs per request group
};

__global__ void __launch_bounds__(THREADS) verify_kernel(const Params p) {
  __shared__ int32_t par_s[MAX_NODES], tok_s[MAX_NODES];
  __shared__ float red_v[THREADS / 32];
  __shared__ int red_i[THREADS / 32];
  __shared__ int s_next, s_ok;
  __shared__ float s_bv;
  __shared__ int s_bi;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cpr = p.cpr;
  const int grp = blockIdx.x / cpr, c = blockIdx.x - grp * cpr;
  const int n_groups = gridDim.x / cpr;
  unsigned epoch = 0;
  const int N = p.B + 1;

  for (int q = grp; q < p.n_req; q += n_groups) {
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
    for (int i = tid; i < n; i += THREADS) {
      par_s[i] = p.parent[(size_t)q * N + i];
      tok_s[i] = p.token[(size_t)q * N + i];
    }
    __syncthreads();
    const int v0 = (int)(((long long)c * p.V) / cpr), v1 = (int)(((long long)(c + 1) * p.V) / cpr);
    int cur = 0, accepted = 0;
    int step = 0;
    for (; step <= p.L; ++step) {
      const float *row = p.t + ((size_t)q * N + cur) * (size_t)p.V;
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
      if (T == 0.f) {
        int v = v0 + tid;
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
        for (int v = v0 + tid; v < v1; v += THREADS) {
          const float a = __fadd_rn(__fdiv_rn(__ldcs(row + v), T), gumbel(seed, cur, v));
          if (vi_before(a, v, bv, bi)) { bv = a; bi = v; }
        }
      }
      // CTA reduction
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
      __syncthreads();
      if (warp == 0) {
        bv = lane < THREADS / 32 ? red_v[lane] : -INFINITY;
        bi = lane < THREADS / 32 ? red_i[lane] : 0x7FFFFFFF;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (vi_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) {
          s_bv = bv;
          s_bi = bi;
          s_next = 0x7FFFFFFF;
        }
      }
      __syncthreads();
      if (cpr > 1) {
        // publish, meet, read every CTA of the group
        if (tid == 0) {
          p.part[(size_t)blockIdx.x * 2 + (epoch & 1u)] = make_float2(s_bv, __int_as_float(s_bi));
          __threadfence();
          unsigned *ctr = p.bar + grp;
          atomicAdd(ctr, 1u);
          const unsigned target = (epoch + 1u) * (unsigned)cpr;
          int ok = 1;
          if (ld_acquire(ctr) < target) {
            const unsigned long long t0 = globaltimer();
            while (ld_acquire(ctr) < target) {
              if (globaltimer() - t0 > kWaitLimitNs) {
                ok = 0;
                break;
              }
              __nanosleep(32);
            }
          }
          __threadfence();
          s_ok = ok;
        }
        __syncthreads();
        if (!s_ok) {
          if (tid == 0) report(p.status, MFD_ERR_TIMEOUT);
          return;
        }
        if (warp == 0) {
          bv = -INFINITY;
          bi = 0x7FFFFFFF;
          for (int k = lane; k < cpr; k += 32) {
            const float2 e = __ldcg(&p.part[(size_t)(grp * cpr + k) * 2 + (epoch & 1u)]);
            const int ei = __float_as_int(e.y);
            if (vi_before(e.x, ei, bv, bi)) { bv = e.x; bi = ei; }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (vi_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
          }
          if (lane == 0) s_bi = bi;
        }
        ++epoch;
        __syncthreads();
      }
      const int y = s_bi;
      for (int i = 1 + tid; i < n; i += THREADS)
        if (par_s[i] == cur && tok_s[i] == y) atomicMin(&s_next, i);
      __syncthreads();
      if (c == 0 && tid == 0) {
        p.path_nodes[(size_t)q * (p.L + 1) + step] = cur;
        p.out_tokens[(size_t)q * (p.L + 1) + step] = y;
      }
      const int nx = s_next;
      __syncthreads();
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
    __syncthreads();
  }
}

}  // namespace

int verify_max_grid(int n_sm) { return n_sm; }

cudaError_t launch_verify(const VerifyLaunch &V, cudaStream_t stream) {
  Params p;
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
  p.bar = V.bar;
  p.part = V.part;
  const int n_groups = V.n_req < V.grid ? V.n_req : V.grid;
  p.cpr = V.grid / n_groups;
  const int grid = n_groups * p.cpr;
  void *args[] = {&p};
  cudaError_t e = cudaLaunchCooperativeKernel((const void *)verify_kernel, dim3(grid), dim3(THREADS), args, 0, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mfd
