// analytics.cu -- what a tree spends its budget on (project page "Multi-Future
// Drafting", TL;DR and Abstract: chimeras, prefixes spliced from different
// futures that the target never produces; How it works, step 1, and "What the
// modes are", Figure 3: the expected accepted length is the probability mass
// the tree covers, which is read depth by depth).
//
// For trees in mfd_build_tree's format, the planted futures and the target's
// per-node logits:
//   class[n] = ON_FUTURE (the root, or a prefix of some future), CHIMERA (at
//              every position the token is some future's token there, yet the
//              prefix is no future's), OTHER (some token no future has there);
//   reach[n] = the probability that the walk arrives at n: the product along
//              the root -> n path of the target's probability of each next
//              token, softmax(t[parent] / T) for T > 0 and the greedy choice
//              (probability 1 for the argmax, smallest id on ties) for T = 0;
//   mass[d]  = the sum of reach over the nodes at depth d (mass[0] = 1), so
//              that sum_{d >= 1} mass[d] is the expected accepted length.
// Probabilities are computed in double.  Two kernels: one CTA per target row
// that has children (its log-sum-exp or argmax), then one CTA per request.
#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int ROW_THREADS = 512;
constexpr int NODE_THREADS = 512;
constexpr int MAX_NODES = 513;
constexpr int MAX_L = 16;

// Per (request q, node n) whose row is some node's parent row:
//   T > 0: lse[q][n] = max_v (t_v / T) + log sum_v exp(t_v / T - max)
//   T = 0: amax[q][n] = argmax_v t_v (smallest v on ties)
__global__ void __launch_bounds__(ROW_THREADS)
    analytics_rows_kernel(const float *__restrict__ t, int N, int V, const int32_t *__restrict__ parent,
                          const int32_t *__restrict__ n_nodes, const float *__restrict__ temperature,
                          double *__restrict__ lse, int32_t *__restrict__ amax) {
  __shared__ int has_child;
  __shared__ double red_d[ROW_THREADS / 32];
  __shared__ float red_f[ROW_THREADS / 32];
  __shared__ int red_i[ROW_THREADS / 32];
  const int q = blockIdx.y, n = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nn = n_nodes[q];
  if (nn < 1 || nn > N || n >= nn) return;
  if (tid == 0) has_child = 0;
  block_sync();
  for (int c = 1 + tid; c < nn; c += ROW_THREADS)
    if (parent[(size_t)q * N + c] == n) has_child = 1;
  block_sync();
  if (!has_child) return;
  const float T = temperature[q];
  const float *row = t + ((size_t)q * N + n) * (size_t)V;
  // the row's max (value desc, id asc), shared by both cases
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  for (int v = tid; v < V; v += ROW_THREADS) {
    const float a = __ldg(row + v);
    if (vi_before(a, v, bv, bi)) {
      bv = a;
      bi = v;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (vi_before(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  if (lane == 0) {
    red_f[warp] = bv;
    red_i[warp] = bi;
  }
  block_sync();
  if (tid == 0) {
    for (int w = 1; w < ROW_THREADS / 32; ++w)
      if (vi_before(red_f[w], red_i[w], red_f[0], red_i[0])) {
        red_f[0] = red_f[w];
        red_i[0] = red_i[w];
      }
  }
  block_sync();
  if (!(T > 0.f)) {
    if (tid == 0) amax[(size_t)q * N + n] = red_i[0];
    return;
  }
  const double Td = (double)T;
  const double zmax = (double)red_f[0] / Td;
  double s = 0.0;
  for (int v = tid; v < V; v += ROW_THREADS) s += exp((double)__ldg(row + v) / Td - zmax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) red_d[warp] = s;
  block_sync();
  if (tid == 0) {
    double tot = 0.0;
    for (int w = 0; w < ROW_THREADS / 32; ++w) tot += red_d[w];
    lse[(size_t)q * N + n] = zmax + log(tot);
  }
}

// One CTA per request: classes, reach, mass by depth.
__global__ void __launch_bounds__(NODE_THREADS)
    analytics_nodes_kernel(const float *__restrict__ t, int N, int V, int L, const int32_t *__restrict__ parent,
                           const int32_t *__restrict__ token, const int32_t *__restrict__ depth,
                           const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ futures, int F,
                           const float *__restrict__ temperature, const double *__restrict__ lse,
                           const int32_t *__restrict__ amax, int32_t *__restrict__ node_class,
                           double *__restrict__ reach, double *__restrict__ mass, int32_t *status) {
  __shared__ int par_s[MAX_NODES], tok_s[MAX_NODES], dep_s[MAX_NODES];
  __shared__ double edge_s[MAX_NODES], reach_s[MAX_NODES];
  __shared__ int bad;
  const int q = blockIdx.x, tid = threadIdx.x;
  const int nn = n_nodes[q];
  const float T = temperature[q];
  if (tid == 0) bad = !(nn >= 1 && nn <= N) || !(T >= 0.f);
  block_sync();
  if (bad) {
    if (tid == 0) report(status, MFD_ERR_INPUT);
    return;
  }
  for (int n = tid; n < nn; n += NODE_THREADS) {
    par_s[n] = parent[(size_t)q * N + n];
    tok_s[n] = token[(size_t)q * N + n];
    dep_s[n] = depth[(size_t)q * N + n];
  }
  block_sync();
  // the tree's own shape: parents first, depth one more than the parent's
  for (int n = tid; n < nn; n += NODE_THREADS) {
    const bool ok = n == 0 ? (dep_s[0] == 0) : (par_s[n] >= 0 && par_s[n] < n && dep_s[n] == dep_s[par_s[n]] + 1 &&
                                                  dep_s[n] <= L && tok_s[n] >= 0 && tok_s[n] < V);
    if (!ok) bad = 1;
  }
  block_sync();
  if (bad) {
    if (tid == 0) report(status, MFD_ERR_INPUT);
    return;
  }
  const int32_t *fut = futures + (size_t)q * F * L;
  for (int n = tid; n < nn; n += NODE_THREADS) {
    // the path's tokens, root first
    int seq[MAX_L];
    const int d = dep_s[n];
    for (int a = n; a > 0; a = par_s[a]) seq[dep_s[a] - 1] = tok_s[a];
    int cls = 0;  // ON_FUTURE
    if (d > 0) {
      bool prefix_of = false, splice = true;
      for (int f = 0; f < F && !prefix_of; ++f) {
        bool same = true;
        for (int i = 0; i < d && same; ++i) same = fut[f * L + i] == seq[i];
        prefix_of = same;
      }
      for (int i = 0; i < d && splice; ++i) {
        bool any = false;
        for (int f = 0; f < F && !any; ++f) any = fut[f * L + i] == seq[i];
        splice = any;
      }
      cls = prefix_of ? 0 : (splice ? 1 : 2);
    }
    node_class[(size_t)q * N + n] = cls;
    // the edge into n: the target's probability of n's token at its parent
    double e = 1.0;
    if (n > 0) {
      const int p = par_s[n];
      if (T > 0.f) {
        const float tv = __ldg(t + ((size_t)q * N + p) * (size_t)V + tok_s[n]);
        e = exp((double)tv / (double)T - lse[(size_t)q * N + p]);
      } else {
        e = tok_s[n] == amax[(size_t)q * N + p] ? 1.0 : 0.0;
      }
    }
    edge_s[n] = e;
  }
  block_sync();
  for (int n = tid; n < nn; n += NODE_THREADS) {
    // reach: the edges multiplied from the root down
    int path[MAX_L + 1];
    const int d = dep_s[n];
    for (int a = n; a > 0; a = par_s[a]) path[dep_s[a]] = a;
    double r = 1.0;
    for (int i = 1; i <= d; ++i) r *= edge_s[path[i]];
    reach_s[n] = r;
    reach[(size_t)q * N + n] = r;
  }
  for (int n = nn + tid; n < N; n += NODE_THREADS) {
    node_class[(size_t)q * N + n] = -1;
    reach[(size_t)q * N + n] = 0.0;
  }
  block_sync();
  // mass by depth, summed in node order
  if (tid <= L) {
    double s = 0.0;
    for (int n = 0; n < nn; ++n)
      if (dep_s[n] == tid) s += reach_s[n];
    mass[(size_t)q * (L + 1) + tid] = s;
  }
}

}  // namespace

cudaError_t launch_tree_analytics(const AnalyticsLaunch &A, cudaStream_t stream) {
  const int N = A.B + 1;
  if (N > MAX_NODES || A.L > MAX_L || A.F < 1) return cudaErrorInvalidValue;
  dim3 g1(N, A.n_req);
  analytics_rows_kernel<<<g1, ROW_THREADS, 0, stream>>>(A.t, N, A.V, A.parent, A.n_nodes, A.temperature, A.lse,
                                                       A.amax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  analytics_nodes_kernel<<<A.n_req, NODE_THREADS, 0, stream>>>(A.t, N, A.V, A.L, A.parent, A.token, A.depth,
                                                               A.n_nodes, A.futures, A.F, A.temperature, A.lse,
                                                               A.amax, A.node_class, A.reach, A.mass, A.status);
  return cudaGetLastError();
}

}  // namespace mfd
