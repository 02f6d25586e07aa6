// topk.cu -- log-softmax and top-k: combining per-range partials of a row,
// and the partials themselves when fp32 logits are given directly.
//
// A row's distribution (project page "Multi-Future Drafting", How it works,
// step 2) is p_v = exp(z_v - LSE), LSE = M + log sum_ranges S_r exp(m_r - M),
// where range r contributed its max m_r and S_r = sum exp(z - m_r).  The
// row's top-k is the k best (z desc, id asc) among the ranges' own top-T
// lists (T >= k), which are sorted best first.
#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int MERGE_THREADS = 256;
constexpr int SURV_CAP = 256;  // survivors a warp gathers before falling back
constexpr int MAX_LISTS_PER_LANE = 8;  // P <= 256

struct Cand {
  float v;
  int i;
};

__device__ __forceinline__ Cand load_cand(const int2 *p) {
  const int2 c = __ldcg(p);
  return Cand{__int_as_float(c.x), c.y};
}

// Warp-wide best of (v, i) pairs; every lane gets the winner.
__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, c.v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, c.i, o);
    if (vi_before(ov, oi, c.v, c.i)) {
      c.v = ov;
      c.i = oi;
    }
  }
  return c;
}

// One CTA per row, one thread per list: the row's P lists (T candidates
// each, best first) and its P (max, sum exp) pairs are staged in shared
// memory with 16-byte loads, then every step is a parallel count:
//   LSE   = M + log sum_q S_q exp(m_q - M)
//   tau   = the topk-th best list head (ties ordered by list): at least topk
//           candidates are at least as good, so nothing worse can make it
//   top-k = survivors (the prefix of each list not worse than tau) ranked by
//           counting how many survivors beat each one
template <int T>
__global__ void __launch_bounds__(MERGE_THREADS)
    merge_topk_kernel(const float2 *__restrict__ part_ms, const int2 *__restrict__ part_cand, int R, int P,
                      int topk, float *__restrict__ tk_logp, int32_t *__restrict__ tk_tok, float *__restrict__ lse_out) {
  extern __shared__ int4 merge_smem[];
  __shared__ Cand surv[SURV_CAP];
  __shared__ Cand top[32];
  __shared__ int2 heads[MERGE_THREADS + 4];
  __shared__ float red[MERGE_THREADS / 32];
  __shared__ Cand tau_s;
  __shared__ int n_surv_s;
  __shared__ float lse_s, m_s;
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  if (row >= R) return;
  int2 *cs = reinterpret_cast<int2 *>(merge_smem);
  float2 *ms = reinterpret_cast<float2 *>(cs + (size_t)P * T);
  {
    const int4 *src = reinterpret_cast<const int4 *>(part_cand + (size_t)row * P * T);
    const int n4 = P * T / 2;
    for (int i = tid; i < n4; i += MERGE_THREADS) merge_smem[i] = __ldcg(src + i);
    for (int i = tid; i < P; i += MERGE_THREADS) ms[i] = __ldcg(part_ms + (size_t)row * P + i);
  }
  if (tid == 0) {
    n_surv_s = 0;
    tau_s = Cand{-INFINITY, 0x7FFFFFFF};
  }
  __syncthreads();
  auto cand_at = [&](int q, int c) {
    const int2 e = cs[q * T + c];
    return Cand{__int_as_float(e.x), e.y};
  };
  const int q = tid;  // this thread's list
  const bool has = q < P;

  // ---- log-sum-exp
  float x = has ? ms[q].x : -INFINITY;
  x = warp_max(x);
  if (lane == 0) red[warp] = x;
  __syncthreads();
  if (tid == 0) {
    float M = red[0];
    for (int w = 1; w < MERGE_THREADS / 32; ++w) M = fmaxf(M, red[w]);
    m_s = M;
  }
  __syncthreads();
  const float M = m_s;
  float sv = (has && ms[q].x > -INFINITY) ? ms[q].y * expf(ms[q].x - M) : 0.f;
  sv = warp_sum(sv);
  __syncthreads();
  if (lane == 0) red[warp] = sv;
  __syncthreads();
  if (tid == 0) {
    float S = 0.f;
    for (int w = 0; w < MERGE_THREADS / 32; ++w) S += red[w];
    lse_s = M + logf(S);
  }

  // ---- tau: rank of this list's head among all heads (heads copied to a
  // compact array; four independent counters keep the loads in flight)
  const int need = topk < P ? topk : P;
  if (has) heads[q] = cs[q * T];
  if (tid < 4) heads[P + tid] = make_int2(__float_as_int(-INFINITY), 0x7FFFFFFF);  // padding: never before
  __syncthreads();
  if (has) {
    const Cand h = cand_at(q, 0);
    int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
    const int P4 = (P + 3) & ~3;
    for (int o = 0; o < P4; o += 4) {
      const int2 g0 = heads[o], g1 = heads[o + 1], g2 = heads[o + 2], g3 = heads[o + 3];
      r0 += vi_before(__int_as_float(g0.x), g0.y, h.v, h.i) || (__int_as_float(g0.x) == h.v && g0.y == h.i && o < q);
      r1 += vi_before(__int_as_float(g1.x), g1.y, h.v, h.i) || (__int_as_float(g1.x) == h.v && g1.y == h.i && o + 1 < q);
      r2 += vi_before(__int_as_float(g2.x), g2.y, h.v, h.i) || (__int_as_float(g2.x) == h.v && g2.y == h.i && o + 2 < q);
      r3 += vi_before(__int_as_float(g3.x), g3.y, h.v, h.i) || (__int_as_float(g3.x) == h.v && g3.y == h.i && o + 3 < q);
    }
    // the padding heads equal (-inf, max) and sit after every list, so they
    // never count for a real head
    const int r = r0 + r1 + r2 + r3;
    if (r == need - 1 && need == topk) tau_s = h;
  }
  __syncthreads();
  const Cand tau = tau_s;  // (-inf, max) when there are fewer lists than topk: keep all

  // ---- survivors: the prefix of each list not worse than tau
  int c = 0;
  if (has)
    while (c < T) {
      const Cand e = cand_at(q, c);
      if (vi_before(tau.v, tau.i, e.v, e.i)) break;
      ++c;
    }
  const int slot = c ? atomicAdd(&n_surv_s, c) : 0;
  if (c && slot + c <= SURV_CAP)
    for (int k = 0; k < c; ++k) surv[slot + k] = cand_at(q, k);
  __syncthreads();
  const int n_surv = n_surv_s;
  if (n_surv <= SURV_CAP) {
    for (int a = tid; a < n_surv; a += MERGE_THREADS) {
      const Cand e = surv[a];
      int r = 0;
      for (int b = 0; b < n_surv; ++b) {
        const Cand f = surv[b];
        r += vi_before(f.v, f.i, e.v, e.i) || (f.v == e.v && f.i == e.i && b < a);
      }
      if (r < topk) top[r] = e;
    }
  } else if (warp == 0) {
    // many exact ties at the cut: topk rounds of "best remaining list head"
    int pos[MAX_LISTS_PER_LANE];
#pragma unroll
    for (int s2 = 0; s2 < MAX_LISTS_PER_LANE; ++s2) pos[s2] = 0;
    for (int r = 0; r < topk; ++r) {
      Cand b = Cand{-INFINITY, 0x7FFFFFFF};
      int bs = -1;
#pragma unroll
      for (int s2 = 0; s2 < MAX_LISTS_PER_LANE; ++s2) {
        const int qq = lane + 32 * s2;
        if (qq < P && pos[s2] < T) {
          const Cand e = cand_at(qq, pos[s2]);
          if (bs < 0 || vi_before(e.v, e.i, b.v, b.i)) {
            b = e;
            bs = s2;
          }
        }
      }
      const Cand w = warp_best(b);
      const unsigned owner = __ballot_sync(0xffffffffu, bs >= 0 && b.v == w.v && b.i == w.i);
      if (lane == __ffs(owner) - 1) {
#pragma unroll
        for (int s2 = 0; s2 < MAX_LISTS_PER_LANE; ++s2)
          if (s2 == bs) ++pos[s2];
      }
      if (lane == 0) top[r] = w;
    }
  }
  __syncthreads();

  // ---- log-probabilities, final order (log p desc, id asc)
  if (tid < topk) {
    const float lse = lse_s;
    const Cand e = top[tid];
    const float lp = e.v - lse;
    int r2 = 0;
    for (int o = 0; o < topk; ++o) {
      if (o == tid) continue;
      const float olp = top[o].v - lse;
      r2 += vi_before(olp, top[o].i, lp, e.i);
    }
    tk_logp[(size_t)row * topk + r2] = lp;
    tk_tok[(size_t)row * topk + r2] = e.i;
    if (tid == 0 && lse_out) lse_out[row] = lse;
  }
}

// One warp per (row, vocabulary chunk): lane-local online softmax and top-T,
// then a warp merge of the 32 lane lists into the chunk's top-T.
template <int T>
__global__ void __launch_bounds__(128)
    logits_partial_kernel(const float *__restrict__ logits, int R, int V, int P, int chunk,
                          float2 *__restrict__ part_ms, int2 *__restrict__ part_cand) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.y * 4 + warp;
  const int q = blockIdx.x;
  if (row >= R) return;
  const int v0 = q * chunk;
  const int v1 = min(V, v0 + chunk);
  const float *z = logits + (size_t)row * V;
  float m = -INFINITY, S = 0.f;
  float tv[T];
  int ti[T];
#pragma unroll
  for (int s = 0; s < T; ++s) {
    tv[s] = -INFINITY;
    ti[s] = 0x7FFFFFFF;
  }
  for (int v = v0 + lane; v < v1; v += 32) {
    const float x = __ldg(&z[v]);
    if (x > m) {
      S = (m == -INFINITY) ? 1.f : S * expf(m - x) + 1.f;
      m = x;
    } else if (x > -INFINITY) {
      S += expf(x - m);
    }
    if (vi_before(x, v, tv[T - 1], ti[T - 1])) {
      float cv = x;
      int ci = v;
#pragma unroll
      for (int s = 0; s < T; ++s) {
        const bool sw = vi_before(cv, ci, tv[s], ti[s]);
        const float ov = tv[s];
        const int oi = ti[s];
        tv[s] = sw ? cv : ov;
        ti[s] = sw ? ci : oi;
        cv = sw ? ov : cv;
        ci = sw ? oi : ci;
      }
    }
  }
  const float M = warp_max(m);
  const float Sw = warp_sum(m > -INFINITY ? S * expf(m - M) : 0.f);
  float out_v = -INFINITY;
  int out_i = 0x7FFFFFFF;
  for (int r = 0; r < T; ++r) {
    const Cand w = warp_best(Cand{tv[0], ti[0]});
    const unsigned owner = __ballot_sync(0xffffffffu, tv[0] == w.v && ti[0] == w.i);
    if (lane == __ffs(owner) - 1) {
#pragma unroll
      for (int s = 0; s < T - 1; ++s) {
        tv[s] = tv[s + 1];
        ti[s] = ti[s + 1];
      }
      tv[T - 1] = -INFINITY;
      ti[T - 1] = 0x7FFFFFFF;
    }
    if (lane == r) {
      out_v = w.v;
      out_i = w.i;
    }
  }
  const size_t base = (size_t)row * P + q;
  if (lane == 0) part_ms[base] = make_float2(M, Sw);
  if (lane < T) part_cand[base * T + lane] = make_int2(__float_as_int(out_v), out_i);
}

template <int T>
cudaError_t merge_t(const MergeLaunch &M, cudaStream_t s) {
  const size_t smem = (size_t)M.P * T * 8 + (size_t)M.P * 8;
  cudaError_t e = cudaFuncSetAttribute(merge_topk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M.R);
  cfg.blockDim = dim3(MERGE_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, merge_topk_kernel<T>, reinterpret_cast<const float2 *>(M.part_ms),
                         reinterpret_cast<const int2 *>(M.part_cand), M.R, M.P, M.topk, M.tk_logp, M.tk_tok, M.lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int T>
cudaError_t partial_t(const LogitsPartialLaunch &L, cudaStream_t s) {
  dim3 grid(L.P, (L.R + 3) / 4);
  logits_partial_kernel<T><<<grid, 128, 0, s>>>(L.logits, L.R, L.V, L.P, L.chunk,
                                               reinterpret_cast<float2 *>(L.part_ms),
                                               reinterpret_cast<int2 *>(L.part_cand));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge_topk(const MergeLaunch &M, cudaStream_t s) {
  if (M.P > 32 * MAX_LISTS_PER_LANE) return cudaErrorInvalidValue;
  switch (M.T) {
    case 8: return merge_t<8>(M, s);
    case 16: return merge_t<16>(M, s);
    case 32: return merge_t<32>(M, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_logits_partials(const LogitsPartialLaunch &L, cudaStream_t s) {
  switch (L.T) {
    case 8: return partial_t<8>(L, s);
    case 16: return partial_t<16>(L, s);
    case 32: return partial_t<32>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mfd
