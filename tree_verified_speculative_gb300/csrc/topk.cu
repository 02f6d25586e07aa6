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

constexpr int MERGE_THREADS = 128;       // one CTA per row
constexpr int MERGE_WARPS = MERGE_THREADS / 32;
constexpr int SURV_CAP = 512;            // survivors ranked before falling back
constexpr int LISTS_PER_THREAD = 2;      // P <= 256

struct Cand {
  float v;
  int i;
};

__device__ __forceinline__ Cand cand_of(int x, int y) { return Cand{__int_as_float(x), y}; }
__device__ __forceinline__ bool before(const Cand &a, const Cand &b) { return vi_before(a.v, a.i, b.v, b.i); }
__device__ __forceinline__ Cand shfl_cand(const Cand &c, int o) {
  return Cand{__shfl_xor_sync(0xffffffffu, c.v, o), __shfl_xor_sync(0xffffffffu, c.i, o)};
}

// Warp-wide best of (v, i) pairs; every lane gets the winner.
__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Cand d = shfl_cand(c, o);
    if (before(d, c)) c = d;
  }
  return c;
}

// One CTA of 128 threads per row; thread t owns lists t and t + 128 (P <=
// 256), each a range's T best (value desc, id asc) plus the range's (max,
// sum exp).  The steps are short and spread over the block so that the
// row's critical path stays a few hundred cycles past the loads:
//   LSE  = M + log sum_q S_q exp(m_q - M)
//   tau  = a candidate with at least topk candidates at or before it: the
//          threads are cut into G >= topk groups by t mod G (G a power of
//          two), and tau is the worst of the G group bests -- G distinct
//          candidates, each at or before tau.  Nothing after tau can be in
//          the top-k.
//   top  = the survivors (each list's prefix at or before tau, and not below
//          the LM head's row bound when there is one: the smallest of the
//          k residue-class maxima its ranges published, the value of k
//          distinct candidates or better) ranked by counting how many
//          survivors precede each one.
template <int T>
__global__ void __launch_bounds__(MERGE_THREADS)
    merge_topk_kernel(const float2 *__restrict__ part_ms, const int2 *__restrict__ part_cand, int R, int P,
                      int topk, float *__restrict__ tk_logp, int32_t *__restrict__ tk_tok, float *__restrict__ lse_out,
                      const int32_t *__restrict__ vocab_ids, int V_sub, int V_full, int32_t *status,
                      const int *__restrict__ rb, int G_rb) {
  __shared__ Cand surv[SURV_CAP];
  __shared__ Cand top[32];
  __shared__ int top_tok[32];  // a top entry's output token: its vocabulary id on a subset
  __shared__ Cand gbest[MERGE_WARPS][32];
  __shared__ float red_m[MERGE_WARPS], red_s[MERGE_WARPS];
  __shared__ int n_surv_s;
  __shared__ int bound_s;
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  if (row >= R) return;
  const float2 *ms = part_ms + (size_t)row * P;
  const int2 *cand = part_cand + (size_t)row * P * T;
  auto list_at = [&](int q, int j) {
    const int2 e = __ldcg(cand + (size_t)q * T + j);
    return cand_of(e.x, e.y);
  };
  if (tid == 0) n_surv_s = 0;
  // the row bound's class maxima: T / 4 lanes of warp 0, one 16-byte word each
  int bk = 0x7FFFFFFF;
  if (rb && warp == 0 && lane < T / 4) {
    const int4 q = __ldcg(reinterpret_cast<const int4 *>(rb + (size_t)row * T) + lane);
    const int c4 = 4 * lane;
    bk = c4 + 0 < G_rb ? min(bk, q.x) : bk;
    bk = c4 + 1 < G_rb ? min(bk, q.y) : bk;
    bk = c4 + 2 < G_rb ? min(bk, q.z) : bk;
    bk = c4 + 3 < G_rb ? min(bk, q.w) : bk;
  }

  // ---- (max, sum exp) and the first four candidates of each owned list, in
  // one round trip: a list rarely holds more than four of the row's top-k
  constexpr int HEAD = 4;  // T >= 8
  float m[LISTS_PER_THREAD], sx[LISTS_PER_THREAD];
  Cand hd[LISTS_PER_THREAD][HEAD];
#pragma unroll
  for (int s = 0; s < LISTS_PER_THREAD; ++s) {
    const int q = tid + MERGE_THREADS * s;
    m[s] = -INFINITY;
    sx[s] = 0.f;
#pragma unroll
    for (int j = 0; j < HEAD; ++j) hd[s][j] = Cand{-INFINITY, 0x7FFFFFFF};
    if (q < P) {
      const float2 x = __ldcg(ms + q);
      const int4 c0 = __ldcg(reinterpret_cast<const int4 *>(cand + (size_t)q * T));
      const int4 c1 = __ldcg(reinterpret_cast<const int4 *>(cand + (size_t)q * T) + 1);
      m[s] = x.x;
      sx[s] = x.y;
      hd[s][0] = cand_of(c0.x, c0.y);
      hd[s][1] = cand_of(c0.z, c0.w);
      hd[s][2] = cand_of(c1.x, c1.y);
      hd[s][3] = cand_of(c1.z, c1.w);
    }
  }

  // ---- per-warp partials of the LSE and of the group bests
  const float wm = warp_max(fmaxf(m[0], m[1]));
  float ls = 0.f;
#pragma unroll
  for (int s = 0; s < LISTS_PER_THREAD; ++s)
    if (m[s] > -INFINITY) ls += sx[s] * expf(m[s] - wm);
  ls = warp_sum(ls);
  int G = 1;
  while (G < topk) G <<= 1;
  Cand g = before(hd[1][0], hd[0][0]) ? hd[1][0] : hd[0][0];
  for (int o = 16; o >= G; o >>= 1) {
    const Cand d = shfl_cand(g, o);
    if (before(d, g)) g = d;
  }
  if (lane == 0) {
    red_m[warp] = wm;
    red_s[warp] = ls;
  }
  if (lane < G) gbest[warp][lane] = g;
  if (warp == 0) {
#pragma unroll
    for (int o = 1; o < T / 4; o <<= 1) bk = min(bk, __shfl_xor_sync(0xffffffffu, bk, o));
    if (lane == 0) bound_s = bk;
  }
  block_sync();

  float M = red_m[0];
#pragma unroll
  for (int w = 1; w < MERGE_WARPS; ++w) M = fmaxf(M, red_m[w]);
  float S = 0.f;
#pragma unroll
  for (int w = 0; w < MERGE_WARPS; ++w)
    if (red_m[w] > -INFINITY) S += red_s[w] * expf(red_m[w] - M);
  const float lse = M + logf(S);
  // group (lane mod G) best over the warps, then the worst over the groups
  Cand t = gbest[0][lane & (G - 1)];
#pragma unroll
  for (int w = 1; w < MERGE_WARPS; ++w) {
    const Cand d = gbest[w][lane & (G - 1)];
    if (before(d, t)) t = d;
  }
  for (int o = G >> 1; o > 0; o >>= 1) {
    const Cand d = shfl_cand(t, o);
    if (before(t, d)) t = d;
  }
  const Cand tau = t;  // (-inf, max) when a group owns no list: everything survives
  const float bnd = rb ? ord_val(bound_s) : -INFINITY;
  auto survives = [&](const Cand &e) { return !before(tau, e) && e.v >= bnd; };

  // ---- survivors: per owned list, the prefix at or before tau
  int cnt[LISTS_PER_THREAD];
  int c = 0;
#pragma unroll
  for (int s = 0; s < LISTS_PER_THREAD; ++s) {
    const int q = tid + MERGE_THREADS * s;
    int k = 0;
    if (q < P) {
#pragma unroll
      for (int j = 0; j < HEAD; ++j) k += (k == j && survives(hd[s][j])) ? 1 : 0;
      if (k == HEAD)
        while (k < T && survives(list_at(q, k))) ++k;
    }
    cnt[s] = k;
    c += k;
  }
  int off = c ? atomicAdd(&n_surv_s, c) : 0;
  if (c && off + c <= SURV_CAP) {
#pragma unroll
    for (int s = 0; s < LISTS_PER_THREAD; ++s) {
      const int q = tid + MERGE_THREADS * s;
#pragma unroll
      for (int j = 0; j < HEAD; ++j)
        if (j < cnt[s]) surv[off++] = hd[s][j];
      for (int k = HEAD; k < cnt[s]; ++k) surv[off++] = list_at(q, k);
    }
  }
  block_sync();
  const int n_surv = n_surv_s;

  if (n_surv <= SURV_CAP) {
    // rank = survivors before this one (equal pairs, only the padding, are
    // ordered by slot)
    for (int a = tid; a < n_surv; a += MERGE_THREADS) {
      const Cand e = surv[a];
      // a subset row's vocabulary id, loaded while the rank is counted
      const int tok = vocab_ids ? ((e.i >= 0 && e.i < V_sub) ? __ldg(vocab_ids + e.i) : -1) : e.i;
      int r0 = 0, r1 = 0;
      int b = 0;
      for (; b + 1 < n_surv; b += 2) {
        const Cand f0 = surv[b], f1 = surv[b + 1];
        r0 += before(f0, e) || (f0.v == e.v && f0.i == e.i && b < a);
        r1 += before(f1, e) || (f1.v == e.v && f1.i == e.i && b + 1 < a);
      }
      if (b < n_surv) {
        const Cand f = surv[b];
        r0 += before(f, e) || (f.v == e.v && f.i == e.i && b < a);
      }
      const int r = r0 + r1;
      if (r < topk) {
        top[r] = e;
        top_tok[r] = tok;
      }
    }
  } else if (warp == 0) {
    // many exact ties at the cut: topk rounds of "best remaining list head"
    int pos[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) pos[s] = 0;
    for (int r = 0; r < topk; ++r) {
      Cand b = Cand{-INFINITY, 0x7FFFFFFF};
      int bs = -1;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int q = lane + 32 * s;
        if (q < P && pos[s] < T) {
          const Cand e = list_at(q, pos[s]);
          if (bs < 0 || before(e, b)) {
            b = e;
            bs = s;
          }
        }
      }
      const Cand w = warp_best(b);
      const unsigned owner = __ballot_sync(0xffffffffu, bs >= 0 && b.v == w.v && b.i == w.i);
      if (lane == __ffs(owner) - 1) {
#pragma unroll
        for (int s = 0; s < 8; ++s)
          if (s == bs) ++pos[s];
      }
      if (lane == 0) {
        top[r] = w;
        top_tok[r] = vocab_ids ? ((w.i >= 0 && w.i < V_sub) ? __ldg(vocab_ids + w.i) : -1) : w.i;
      }
    }
  }
  block_sync();

  // ---- log-probabilities, final order (log p desc, id asc)
  if (tid < topk) {
    const Cand e = top[tid];
    const float lp = e.v - lse;
    int r2 = 0;
    for (int o = 0; o < topk; ++o) {
      if (o == tid) continue;
      r2 += vi_before(top[o].v - lse, top[o].i, lp, e.i);
    }
    // on a subset, the row index's vocabulary id; the table is increasing,
    // so (log p desc, subset index asc) is (log p desc, id asc)
    int tok = top_tok[tid];
    if (vocab_ids && (tok < 0 || tok >= V_full)) {
      report(status, MFD_ERR_INPUT);
      tok = -1;
    }
    tk_logp[(size_t)row * topk + r2] = lp;
    tk_tok[(size_t)row * topk + r2] = tok;
  }
  if (tid == 0 && lse_out) lse_out[row] = lse;
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M.R);
  cfg.blockDim = dim3(MERGE_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, merge_topk_kernel<T>, reinterpret_cast<const float2 *>(M.part_ms),
                         reinterpret_cast<const int2 *>(M.part_cand), M.R, M.P, M.topk, M.tk_logp, M.tk_tok, M.lse,
                         M.vocab_ids, M.V_sub, M.V_full, M.status, M.rb, M.rb ? M.G : 0);
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
  if (M.P > MERGE_THREADS * LISTS_PER_THREAD) return cudaErrorInvalidValue;
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
