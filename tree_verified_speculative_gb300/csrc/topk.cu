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

constexpr int MERGE_WARPS = 4;
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

template <int T>
__global__ void __launch_bounds__(MERGE_WARPS * 32)
    merge_topk_kernel(const float2 *__restrict__ part_ms, const int2 *__restrict__ part_cand, int R, int P,
                      int topk, float *__restrict__ tk_logp, int32_t *__restrict__ tk_tok, float *__restrict__ lse_out) {
  __shared__ Cand surv[MERGE_WARPS][SURV_CAP];
  __shared__ Cand park[MERGE_WARPS][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * MERGE_WARPS + warp;
  if (row >= R) return;
  const float2 *ms = part_ms + (size_t)row * P;
  const int2 *cand = part_cand + (size_t)row * P * T;

  // ---- log-sum-exp over the ranges
  float mloc = -INFINITY;
  for (int q = lane; q < P; q += 32) mloc = fmaxf(mloc, __ldcg(&ms[q]).x);
  const float M = warp_max(mloc);
  float sloc = 0.f;
  for (int q = lane; q < P; q += 32) {
    const float2 e = __ldcg(&ms[q]);
    if (e.x > -INFINITY) sloc += e.y * expf(e.x - M);
  }
  const float lse = M + logf(warp_sum(sloc));

  // ---- tau = the topk-th best list head: at least topk candidates are
  // at least as good, so nothing worse than tau can make the top-k.
  Cand head[MAX_LISTS_PER_LANE];
#pragma unroll
  for (int s = 0; s < MAX_LISTS_PER_LANE; ++s) {
    const int q = lane + 32 * s;
    head[s] = (q < P) ? load_cand(cand + (size_t)q * T) : Cand{-INFINITY, 0x7FFFFFFF};
  }
  Cand tau = Cand{-INFINITY, 0x7FFFFFFF};
  {
    Cand h2[MAX_LISTS_PER_LANE];
#pragma unroll
    for (int s = 0; s < MAX_LISTS_PER_LANE; ++s) h2[s] = head[s];
    const int rounds = topk < P ? topk : P;
    for (int r = 0; r < rounds; ++r) {
      Cand b = h2[0];
      int bs = 0;
#pragma unroll
      for (int s = 1; s < MAX_LISTS_PER_LANE; ++s)
        if (vi_before(h2[s].v, h2[s].i, b.v, b.i)) {
          b = h2[s];
          bs = s;
        }
      const Cand w = warp_best(b);
      const unsigned owner = __ballot_sync(0xffffffffu, b.v == w.v && b.i == w.i);
      if (lane == __ffs(owner) - 1) {
#pragma unroll
        for (int s = 0; s < MAX_LISTS_PER_LANE; ++s)
          if (s == bs) h2[s] = Cand{-INFINITY, 0x7FFFFFFF};
      }
      tau = w;
    }
    if (rounds < topk) tau = Cand{-INFINITY, 0x7FFFFFFF};  // fewer lists than topk: keep everything
  }

  // ---- gather survivors (a prefix of each list)
  int cnt[MAX_LISTS_PER_LANE];
  int total = 0;
#pragma unroll
  for (int s = 0; s < MAX_LISTS_PER_LANE; ++s) {
    const int q = lane + 32 * s;
    int c = 0;
    if (q < P) {
      const int2 *L = cand + (size_t)q * T;
      while (c < T) {
        const Cand e = load_cand(L + c);
        if (vi_before(tau.v, tau.i, e.v, e.i)) break;  // e is worse than tau
        ++c;
      }
    }
    cnt[s] = c;
    total += c;
  }
  int incl = total;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int n_surv = __shfl_sync(0xffffffffu, incl, 31);
  Cand mine = Cand{-INFINITY, 0x7FFFFFFF};
  int rank_mine = 1 << 30;
  const bool fast = n_surv <= SURV_CAP;
  if (fast) {
    int off = incl - total;
#pragma unroll
    for (int s = 0; s < MAX_LISTS_PER_LANE; ++s) {
      const int q = lane + 32 * s;
      for (int c = 0; c < cnt[s]; ++c) surv[warp][off++] = load_cand(cand + (size_t)q * T + c);
    }
    __syncwarp();
    // rank by counting; equal keys (padding only) are ordered by slot
    for (int a = lane; a < n_surv; a += 32) {
      const Cand e = surv[warp][a];
      int r = 0;
      for (int b = 0; b < n_surv; ++b) {
        const Cand f = surv[warp][b];
        r += vi_before(f.v, f.i, e.v, e.i) || (f.v == e.v && f.i == e.i && b < a);
      }
      if (r < topk) park[warp][r] = e;
    }
    __syncwarp();
    if (lane < topk) {
      mine = park[warp][lane];
      rank_mine = lane;
    }
  } else {
    // slow path: topk rounds of "best remaining list head", from memory
    int pos[MAX_LISTS_PER_LANE];
#pragma unroll
    for (int s = 0; s < MAX_LISTS_PER_LANE; ++s) pos[s] = 0;
    for (int r = 0; r < topk; ++r) {
      Cand b = Cand{-INFINITY, 0x7FFFFFFF};
      int bs = -1;
#pragma unroll
      for (int s = 0; s < MAX_LISTS_PER_LANE; ++s) {
        const int q = lane + 32 * s;
        if (q < P && pos[s] < T) {
          const Cand e = load_cand(cand + (size_t)q * T + pos[s]);
          if (bs < 0 || vi_before(e.v, e.i, b.v, b.i)) {
            b = e;
            bs = s;
          }
        }
      }
      const Cand w = warp_best(b);
      const unsigned owner = __ballot_sync(0xffffffffu, bs >= 0 && b.v == w.v && b.i == w.i);
      if (lane == __ffs(owner) - 1) {
#pragma unroll
        for (int s = 0; s < MAX_LISTS_PER_LANE; ++s)
          if (s == bs) ++pos[s];
      }
      if (lane == r) {
        mine = w;
        rank_mine = r;
      }
    }
  }

  // ---- log-probabilities, final order (log p desc, id asc)
  const float lp = mine.v - lse;
  int r2 = 0;
  for (int o = 0; o < 32; ++o) {
    const float olp = __shfl_sync(0xffffffffu, lp, o);
    const int oi = __shfl_sync(0xffffffffu, mine.i, o);
    const int orank = __shfl_sync(0xffffffffu, rank_mine, o);
    if (orank < topk && o != lane) r2 += vi_before(olp, oi, lp, mine.i);
  }
  if (rank_mine < topk) {
    tk_logp[(size_t)row * topk + r2] = lp;
    tk_tok[(size_t)row * topk + r2] = mine.i;
  }
  if (lane == 0 && lse_out) lse_out[row] = lse;
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
  const int grid = (M.R + MERGE_WARPS - 1) / MERGE_WARPS;
  merge_topk_kernel<T><<<grid, MERGE_WARPS * 32, 0, s>>>(reinterpret_cast<const float2 *>(M.part_ms),
                                                        reinterpret_cast<const int2 *>(M.part_cand), M.R, M.P,
                                                        M.topk, M.tk_logp, M.tk_tok, M.lse);
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
