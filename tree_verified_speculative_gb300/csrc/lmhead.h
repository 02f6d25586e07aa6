// lmhead.h -- internal launch interface of the fused LM-head kernel.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mfd {

struct LmheadLaunch {
  const CUtensorMap *tmap_h;  // bf16 [R][H], box 64 x 128, 128-byte swizzle
  const CUtensorMap *tmap_w;  // bf16 [V][H], box 64 x 256, 128-byte swizzle
  int R, H, V;
  int T;     // candidates kept per (row, range): 8, 16 or 32
  int P;     // vocabulary ranges (<= number of 256-row tiles)
  int n_sm;  // persistent grid size
  int tile_rows;  // lmhead_tile_rows(R, V, n_sm)
  void *part_ms;    // float2 [R][P]
  void *part_cand;  // int2 [R][P][T]
  int32_t *status;
  const void *w_packed;  // packed weight (lmhead_packed_bytes), or null: use tmap_w
  bool fp8 = false;                 // E4M3 packed weight (lmhead_packed_fp8_bytes), tmap_h over E4M3 rows
  const float *row_scale = nullptr;  // FP8: t_r per hidden row
  const float *w_amax = nullptr;     // FP8: the weight's largest magnitude (in the packed buffer's trailer)
  bool withhold = false;             // fault injection for tests of the bounded waits
  // row bound (R <= 128): lmhead_bound_bytes(R, T) of scratch that no other
  // launch touches while this one runs -- its generation and ready words,
  // then the class maxima -- and G residue classes (the top-k, <= T); null:
  // every range keeps its own top-T
  void *rb = nullptr;
  int G = 0;
};

size_t lmhead_bound_bytes(int R, int T);  // scratch of the row bound (0 when R > 128)
constexpr size_t LMHEAD_BOUND_HEADER = 256;  // generation and ready words; the class maxima follow
// vocabulary rows per tile for R hidden rows, V vocabulary rows and n_sm
// CTAs: 256, unless R fits one M tile and 256-row tiles would leave CTAs
// without a tile (then 128)
int lmhead_tile_rows(int R, int V, int n_sm);
int lmhead_m_rows();     // hidden rows per M tile (128)
int lmhead_k_chunk();    // K elements per pipeline stage (64)
cudaError_t launch_lmhead_partials(const LmheadLaunch &L, cudaStream_t stream);
size_t lmhead_packed_bytes(int V, int H);  // bytes of the packed weight
cudaError_t launch_pack_w(const void *W, int V, int H, void *Wp, cudaStream_t stream);
// E4M3 packed weight: 32 KB blocks of 256 rows x 128 K elements, then a
// 256-byte trailer whose first word is the weight's largest magnitude
size_t lmhead_packed_fp8_bytes(int V, int H);
cudaError_t launch_pack_w_fp8(const void *W, int V, int H, void *Wp, cudaStream_t stream);
// online E4M3 of bf16 rows x [R][H] (H % 8 == 0): q [rows][stride] bytes
// (rows >= R; rows past R zero; 0 = R rows of H bytes), scale [R]
cudaError_t launch_quant_rows(const void *x, int R, int H, void *q, float *scale, cudaStream_t stream,
                              int rows = 0, size_t stride = 0);

// Hidden rows as the LM head reads them.  Every CTA reads the same hidden
// rows at about the same time; rows that span too few bytes of address
// space are staged into scratch first, padded with zero rows (and, for
// narrow rows, spaced further apart), so that they span more.
struct HiddenStage {
  bool staged;    // copied into scratch before the LM head
  int rows;       // rows the hidden operand spans (>= R; rows past R are zero)
  size_t stride;  // bytes from one row to the next
  size_t bytes;   // scratch bytes of the staged copy (0 unless staged)
};
HiddenStage lmhead_hidden_stage(int R, size_t row_bytes);
size_t lmhead_stage_max_bytes();  // bound on HiddenStage::bytes over every R and row size
// bf16 rows x [R][row_bytes] -> dst [s.rows][s.stride] (rows past R zero)
cudaError_t launch_stage_rows(const void *x, int R, size_t row_bytes, void *dst, const HiddenStage &s,
                              cudaStream_t stream);

// topk.cu
struct MergeLaunch {
  const void *part_ms;    // float2 [R][P]
  const void *part_cand;  // int2 [R][P][T]
  int R, P, T, topk;
  float *tk_logp;
  int32_t *tk_tok;
  float *lse;  // may be NULL
  int32_t *status;
  // draft-vocabulary subset: candidate ids are rows of the subset weight and
  // are written as vocab_ids[id] (ids in [0, V_full)); null: written as is
  const int32_t *vocab_ids;
  int V_sub, V_full;
  // the LM head's row bound (int [R][T] class maxima as order keys, classes
  // 0..G-1 used), or null: candidates below it cannot be in the top-k
  const int *rb = nullptr;
  int G = 0;
};
cudaError_t launch_merge_topk(const MergeLaunch &M, cudaStream_t stream);

struct LogitsPartialLaunch {
  const float *logits;  // [R][V]
  int R, V, T, P, chunk;
  void *part_ms;
  void *part_cand;
};
cudaError_t launch_logits_partials(const LogitsPartialLaunch &L, cudaStream_t stream);

// tree.cu
struct TreeLaunch {
  const float *tk_logp;
  const int32_t *tk_tok;
  int n_req, K, L, topk, B;
  const int32_t *anchor, *base_pos;
  int32_t *parent, *token, *depth;
  float *score;
  int32_t *mode;
  uint32_t *mask;
  int32_t *pos, *n_nodes, *status;
};
size_t tree_smem_bytes(int K, int L, int topk, int B, int *cap_out, int *tsize_out);
cudaError_t launch_build_tree(const TreeLaunch &T, cudaStream_t stream);

// verify.cu
struct VerifyLaunch {
  const float *t;
  int n_req, B, V, L;
  const int32_t *parent, *token, *n_nodes;
  const float *temperature;
  const uint64_t *seed;
  int32_t *accept_len, *path_nodes, *out_tokens, *status;
  // the grid walk (n_req < VERIFY_CLUSTER_REQUESTS) only:
  unsigned long long *ws;  // [grid][8] exchange words (generation-tagged, no zeroing needed)
  int grid;                   // largest cooperative grid
  unsigned long long wait_ns = 0;  // bounded-wait limit (0: the library's default)
  int withhold = 0;                // fault injection for tests of the bounded waits
};
// requests from which a round is walked by clusters (one per request)
// instead of the cooperative grid
constexpr int VERIFY_CLUSTER_REQUESTS = 8;
int verify_max_grid(int n_sm);
int verify_cluster_size(int V);  // CTAs of the cluster that walks one request
cudaError_t launch_verify(const VerifyLaunch &V, cudaStream_t stream);

// analytics.cu
struct AnalyticsLaunch {
  const float *t;  // target logits [n_req][B + 1][V]
  int n_req, B, V, L;
  const int32_t *parent, *token, *depth, *n_nodes;
  const int32_t *futures;  // [n_req][F][L]
  int F;
  const float *temperature;
  double *lse;     // scratch [n_req][B + 1]
  int32_t *amax;   // scratch [n_req][B + 1]
  int32_t *node_class;
  double *reach, *mass;
  int32_t *status;
};
cudaError_t launch_tree_analytics(const AnalyticsLaunch &A, cudaStream_t stream);

}  // namespace mfd
