// mfd_api.cu -- the extern "C" entry points of libmfd (declared and
// documented in include/mfd.h): argument checks, scratch layout, TMA
// descriptor encoding, kernel launches.  No allocation, no host sync.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/mfd.h"
#include "lmhead.h"

namespace {

struct DeviceInfo {
  int n_sm = 0, major = 0, minor = 0;
  bool ok = false;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_dev;

int current_device_info(DeviceInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MFD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MFD_ERR_CUDA;
    d.ok = true;
    it = g_dev.emplace(dev, d).first;
  }
  *out = it->second;
  return MFD_OK;
}

bool is_sm103(const DeviceInfo &d) { return d.major == 10 && d.minor == 3; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int cand_width(int topk) { return topk <= 8 ? 8 : (topk <= 16 ? 16 : 32); }

// ---------------------------------------------------------------- TMA maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

using MapKey = std::tuple<int, const void *, int, int, int, int, size_t>;  // device, ptr, rows, cols, box rows, bytes/elem, row stride
std::map<MapKey, CUtensorMap> g_maps;

// bf16 (elem = 2) or 8-bit (elem = 1) [rows][cols] row-major, rows `stride`
// bytes apart (0: cols * elem), box = 128 bytes of columns x box_rows rows,
// 128B swizzle, out-of-range rows read as zero.  The descriptor is copied
// into *out while the lock is held: another thread may clear the cache right
// after.
int tensor_map(const void *ptr, int rows, int cols, int box_rows, CUtensorMap *out, int elem = 2, size_t stride = 0) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MFD_ERR_CUDA;
  if (stride == 0) stride = (size_t)cols * (size_t)elem;
  std::lock_guard<std::mutex> lk(g_mu);
  const MapKey key{dev, ptr, rows, cols, box_rows, elem, stride};
  auto it = g_maps.find(key);
  if (it == g_maps.end()) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return MFD_ERR_CUDA;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)stride};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / elem), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(&m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                          const_cast<void *>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MFD_ERR_CUDA;
    if (g_maps.size() > 4096) g_maps.clear();
    it = g_maps.emplace(key, m).first;
  }
  *out = it->second;
  return MFD_OK;
}

// ---------------------------------------------------------------- layouts
struct TopkLayout {
  int P, T, chunk;
  size_t ms_bytes, cand_bytes, total;
  size_t stage_off = 0;  // LM head: room for the staged hidden rows (lmhead_hidden_stage)
  size_t part_off = 0;   // LM head: the partials follow the row bound, which starts the scratch
};

// Fewest weight tiles for the busiest CTA when n_groups M tiles share
// `workers` CTAs: over P vocabulary ranges, a CTA takes
// ceil(n_groups * P / workers) items of ceil(tiles / P) tiles.  Among equal
// costs the fewest ranges win: fewer partials to merge and fewer top-T
// restarts per row.
static long long best_ranges(int tiles, int n_groups, int workers, int *P_out) {
  long long best = -1;
  const int pmax = tiles < 256 ? tiles : 256;
  for (int P = 1; P <= pmax; ++P) {
    const long long rounds = ((long long)n_groups * P + workers - 1) / workers;
    const long long cost = rounds * ((tiles + P - 1) / P);
    if (best < 0 || cost < best) {
      best = cost;
      *P_out = P;
    }
  }
  return best;
}

TopkLayout lmhead_layout(int R, int V, int topk, int n_sm) {
  TopkLayout y;
  const int tile_rows = mfd::lmhead_tile_rows(R, V, n_sm);
  const int tiles = (V + tile_rows - 1) / tile_rows;
  const int n_mt = (R + mfd::lmhead_m_rows() - 1) / mfd::lmhead_m_rows();
  y.P = tiles < n_sm ? tiles : n_sm;
  if (y.P > 256) y.P = 256;
  if (n_mt > 1) {
    best_ranges(tiles, n_mt, n_sm, &y.P);  // work items are (range, M tile)
  } else {
    // When at most three quarters of the ranges hold the largest share, the
    // last wave leaves many SMs idle: take the fewest ranges with the same
    // largest range instead, so that every CTA that streams streams as many
    // tiles (measured: 65,536 rows 64.2 -> 61.5 us, 248,320 rows at H = 5120
    // 384 -> 377 us; with 151,936 rows, 138 of 152 ranges hold four tiles,
    // and 149 ranges were slower)
    const int most = (tiles + y.P - 1) / y.P;
    const int at_most = tiles - (most - 1) * y.P;  // ranges holding `most` tiles
    if (4 * at_most <= 3 * y.P) y.P = (tiles + most - 1) / most;
  }
  y.T = cand_width(topk);
  y.chunk = 0;
  // the row bound's generation words sit at offset 0 for every shape, so a
  // call of another shape finds them where the last one left them
  y.part_off = mfd::lmhead_bound_bytes(R, y.T);
  y.ms_bytes = align256((size_t)R * y.P * 8);
  y.cand_bytes = align256((size_t)R * y.P * y.T * 8);
  y.total = y.part_off + y.ms_bytes + y.cand_bytes;
  // one M tile: room for the hidden rows staged when they span few bytes
  y.stage_off = y.total;
  if (R <= mfd::lmhead_m_rows()) y.total += align256(mfd::lmhead_stage_max_bytes());
  return y;
}

// FP8 LM head scratch: the partials of lmhead_layout, then the E4M3 hidden
// rows (R rows of H bytes, or the padded rows of lmhead_hidden_stage) and
// their scales [R].
struct Fp8Layout {
  TopkLayout y;
  size_t hq_off, sc_off, total;
};
Fp8Layout fp8_layout(int R, int H, int V, int topk, int n_sm) {
  Fp8Layout f;
  f.y = lmhead_layout(R, V, topk, n_sm);
  f.hq_off = f.y.total;
  const mfd::HiddenStage hs = mfd::lmhead_hidden_stage(R, (size_t)H);
  f.sc_off = f.hq_off + align256(hs.staged ? hs.bytes : (size_t)R * H);
  f.total = f.sc_off + align256((size_t)R * 4);
  return f;
}

TopkLayout logits_layout(int R, int V, int topk) {
  TopkLayout y;
  int chunk = (V + 255) / 256;
  chunk = (chunk + 31) / 32 * 32;
  if (chunk < 1024) chunk = 1024;
  y.chunk = chunk;
  y.P = (V + chunk - 1) / chunk;
  y.T = cand_width(topk);
  y.ms_bytes = align256((size_t)R * y.P * 8);
  y.cand_bytes = align256((size_t)R * y.P * y.T * 8);
  y.total = y.ms_bytes + y.cand_bytes;
  return y;
}

size_t verify_bytes(int n_sm) { return align256((size_t)mfd::verify_max_grid(n_sm) * 8 * 8); }

size_t analytics_bytes(int n_req, int B) { return align256((size_t)n_req * (B + 1) * 8) + align256((size_t)n_req * (B + 1) * 4); }

size_t tree_bytes(int n_req) {
  (void)n_req;
  return 256;  // the tree is built in shared memory; the scratch is not used
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MFD_OK : MFD_ERR_CUDA; }

// Scratch of mfd_logits_topk_noalloc: one static array per device, kept
// for the life of the process.  Host code cannot use its name as a device
// address, so its address is looked up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MFD_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
std::map<int, void *> g_noalloc_ptr;

int noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MFD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  auto it = g_noalloc_ptr.find(dev);
  if (it == g_noalloc_ptr.end()) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MFD_ERR_CUDA;
    it = g_noalloc_ptr.emplace(dev, p).first;
  }
  *out = it->second;
  return MFD_OK;
}

}  // namespace

extern "C" {

const char *mfd_status_string(int status) {
  switch (status) {
    case MFD_OK: return "ok";
    case MFD_ERR_INVALID_ARG: return "invalid argument (NULL pointer, size out of range or misaligned pointer)";
    case MFD_ERR_UNSUPPORTED: return "unsupported: outside the library limits or not an sm_103a device";
    case MFD_ERR_WORKSPACE: return "workspace missing or smaller than mfd_workspace_size";
    case MFD_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case MFD_ERR_TIMEOUT: return "a bounded device wait ran out; the kernel stopped early";
    case MFD_ERR_INPUT: return "input values break the contract (see mfd.h)";
    case MFD_ERR_CHECK: return "bounds-checked build: an index out of range was clamped";
    default: return "unknown status";
  }
}

int mfd_tree_analytics(const int32_t *parent, const int32_t *token, const int32_t *depth, const int32_t *n_nodes,
                       int n_req, int B, int L, const int32_t *futures, int F, const float *target_logits, int V,
                       const float *temperature, int32_t *node_class, double *reach, double *mass, int32_t *status,
                       void *ws, size_t ws_bytes, mfd_stream_t stream) {
  if (!parent || !token || !depth || !n_nodes || !futures || !target_logits || !temperature || !node_class ||
      !reach || !mass || !status)
    return MFD_ERR_INVALID_ARG;
  if (n_req < 1 || B < 1 || L < 1 || F < 1 || V < 1) return MFD_ERR_INVALID_ARG;
  if (B > 512 || L > 16 || F > 64 || V >= (1 << 30)) return MFD_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < analytics_bytes(n_req, B) || !aligned(ws, 256)) return MFD_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  mfd::AnalyticsLaunch A;
  A.t = target_logits;
  A.n_req = n_req;
  A.B = B;
  A.V = V;
  A.L = L;
  A.parent = parent;
  A.token = token;
  A.depth = depth;
  A.n_nodes = n_nodes;
  A.futures = futures;
  A.F = F;
  A.temperature = temperature;
  A.lse = reinterpret_cast<double *>(base);
  A.amax = reinterpret_cast<int32_t *>(base + align256((size_t)n_req * (B + 1) * 8));
  A.node_class = node_class;
  A.reach = reach;
  A.mass = mass;
  A.status = status;
  return cuda_status(mfd::launch_tree_analytics(A, reinterpret_cast<cudaStream_t>(stream)));
}

int mfd_mfdd_modes(int n_req, int K) {
  if (n_req < 1 || K < 1 || K > 16) return 0;
  return n_req < MFD_MFDD_SWITCH_REQUESTS ? K : 1;
}

size_t mfd_workspace_size(int op, int n_req, int K, int L, int topk, int B, int R, int V) {
  (void)K;
  (void)L;
  (void)B;
  DeviceInfo d;
  switch (op) {
    case MFD_OP_LMHEAD_TOPK:
      if (R < 1 || V < 16 || topk < 1 || topk > 32 || topk > V) return 0;
      if (current_device_info(&d) != MFD_OK) return 0;
      return lmhead_layout(R, V, topk, d.n_sm).total;
    case MFD_OP_LOGITS_TOPK:
      if (R < 1 || V < 16 || topk < 1 || topk > 32 || topk > V) return 0;
      return logits_layout(R, V, topk).total;
    case MFD_OP_BUILD_TREE:
      if (n_req < 1) return 0;
      return tree_bytes(n_req);
    case MFD_OP_VERIFY:
      if (n_req < 1) return 0;
      if (current_device_info(&d) != MFD_OK) return 0;
      return verify_bytes(d.n_sm);
    case MFD_OP_TREE_ANALYTICS:
      if (n_req < 1 || B < 1 || B > 512) return 0;
      return analytics_bytes(n_req, B);
    default:
      return 0;
  }
}

}  // extern "C"

namespace {
// The LM head call, from the row-major weight (W, through its tensor map) or
// from the packed weight (Wp).
// vocab_ids: null, or the draft-vocabulary subset (V rows of the weight are
// vocabulary ids vocab_ids[0..V), increasing, below V_full)
int lmhead_call(const void *h, int R, int H, const void *W, const void *Wp, int V, int topk, float *tk_logp,
                int32_t *tk_tok, float *lse, int32_t *status, void *ws, size_t ws_bytes, mfd_stream_t stream,
                const int32_t *vocab_ids = nullptr, int V_full = 0, bool fp8 = false, bool withhold = false) {
  if (!h || (!W && !Wp) || !tk_logp || !tk_tok || !status || R < 1 || H < 1 || V < 1 || topk < 1)
    return MFD_ERR_INVALID_ARG;
  if (!aligned(h, 16) || (W && !aligned(W, 16)) || (Wp && !aligned(Wp, 256))) return MFD_ERR_INVALID_ARG;
  if (H % ((fp8 ? 2 : 1) * mfd::lmhead_k_chunk()) != 0 || topk > 32 || V < 16 || topk > V || V >= (1 << 30))
    return MFD_ERR_UNSUPPORTED;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MFD_OK) return rc;
  if (!is_sm103(d)) return MFD_ERR_UNSUPPORTED;
  const TopkLayout y = lmhead_layout(R, V, topk, d.n_sm);
  const Fp8Layout f8 = fp8_layout(R, H, V, topk, d.n_sm);
  if (!ws || ws_bytes < (fp8 ? f8.total : y.total) || !aligned(ws, 256)) return MFD_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap mh, mw;
  // hidden rows that span few bytes are read from a padded copy
  const mfd::HiddenStage hs = mfd::lmhead_hidden_stage(R, (size_t)H * (fp8 ? 1 : 2));
  if (fp8) {
    // the hidden rows in E4M3 with their scales, then the E4M3 head over them
    if ((rc = cuda_status(mfd::launch_quant_rows(h, R, H, base + f8.hq_off, reinterpret_cast<float *>(base + f8.sc_off),
                                                 s, hs.rows, hs.stride))) != MFD_OK)
      return rc;
    if ((rc = tensor_map(base + f8.hq_off, hs.rows, H, mfd::lmhead_m_rows(), &mh, 1, hs.stride)) != MFD_OK) return rc;
  } else if (hs.staged) {
    char *hstage = base + y.stage_off;
    if ((rc = cuda_status(mfd::launch_stage_rows(h, R, (size_t)H * 2, hstage, hs, s))) != MFD_OK) return rc;
    if ((rc = tensor_map(hstage, hs.rows, H, mfd::lmhead_m_rows(), &mh, 2, hs.stride)) != MFD_OK) return rc;
  } else if ((rc = tensor_map(h, R, H, mfd::lmhead_m_rows(), &mh)) != MFD_OK) {
    return rc;
  }
  if (W && (rc = tensor_map(W, V, H, mfd::lmhead_tile_rows(R, V, d.n_sm), &mw)) != MFD_OK) return rc;
  mfd::LmheadLaunch L;
  L.tmap_h = &mh;
  L.tmap_w = W ? &mw : nullptr;
  L.w_packed = W ? nullptr : Wp;
  L.R = R;
  L.H = H;
  L.V = V;
  L.T = y.T;
  L.P = y.P;
  L.n_sm = d.n_sm;
  L.tile_rows = mfd::lmhead_tile_rows(R, V, d.n_sm);
  L.part_ms = base + y.part_off;
  L.part_cand = base + y.part_off + y.ms_bytes;
  L.status = status;
  L.withhold = withhold;
  L.rb = y.part_off ? base : nullptr;
  L.G = topk;
  if (fp8) {
    L.fp8 = true;
    L.row_scale = reinterpret_cast<const float *>(base + f8.sc_off);
    L.w_amax = reinterpret_cast<const float *>(static_cast<const char *>(Wp) + mfd::lmhead_packed_fp8_bytes(V, H) - 256);
  }
  if ((rc = cuda_status(mfd::launch_lmhead_partials(L, s))) != MFD_OK) return rc;
  mfd::MergeLaunch M;
  M.part_ms = L.part_ms;
  M.part_cand = L.part_cand;
  M.R = R;
  M.P = y.P;
  M.T = y.T;
  M.topk = topk;
  M.tk_logp = tk_logp;
  M.tk_tok = tk_tok;
  M.lse = lse;
  M.status = status;
  M.vocab_ids = vocab_ids;
  M.V_sub = V;
  M.V_full = vocab_ids ? V_full : V;
  M.rb = L.rb ? reinterpret_cast<const int *>(base + mfd::LMHEAD_BOUND_HEADER) : nullptr;
  M.G = topk;
  return cuda_status(mfd::launch_merge_topk(M, s));
}
}  // namespace

extern "C" {

int mfd_lmhead_topk(const void *h, int R, int H, const void *W, int V, int topk, float *tk_logp,
                    int32_t *tk_tok, float *lse, int32_t *status, void *ws, size_t ws_bytes,
                    mfd_stream_t stream) {
  if (!W) return MFD_ERR_INVALID_ARG;
  return lmhead_call(h, R, H, W, nullptr, V, topk, tk_logp, tk_tok, lse, status, ws, ws_bytes, stream);
}

size_t mfd_lmhead_packed_bytes(int V, int H) {
  if (V < 16 || V >= (1 << 30) || H < 1 || H % mfd::lmhead_k_chunk() != 0) return 0;
  return mfd::lmhead_packed_bytes(V, H);
}

int mfd_lmhead_pack(const void *W, int V, int H, void *W_packed, size_t packed_bytes, mfd_stream_t stream) {
  if (!W || !W_packed || V < 1 || H < 1) return MFD_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(W_packed, 256)) return MFD_ERR_INVALID_ARG;
  const size_t need = mfd_lmhead_packed_bytes(V, H);
  if (need == 0) return MFD_ERR_UNSUPPORTED;
  if (packed_bytes < need) return MFD_ERR_WORKSPACE;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MFD_OK) return rc;
  if (!is_sm103(d)) return MFD_ERR_UNSUPPORTED;
  return cuda_status(mfd::launch_pack_w(W, V, H, W_packed, reinterpret_cast<cudaStream_t>(stream)));
}

int mfd_lmhead_topk_packed(const void *h, int R, int H, const void *W_packed, int V, int topk, float *tk_logp,
                           int32_t *tk_tok, float *lse, int32_t *status, void *ws, size_t ws_bytes,
                           mfd_stream_t stream) {
  if (!W_packed) return MFD_ERR_INVALID_ARG;
  return lmhead_call(h, R, H, nullptr, W_packed, V, topk, tk_logp, tk_tok, lse, status, ws, ws_bytes, stream);
}

int mfd_lmhead_withheld_test(const void *h, int R, int H, const void *W_packed, int V, int topk, float *tk_logp,
                             int32_t *tk_tok, float *lse, int32_t *status, void *ws, size_t ws_bytes,
                             mfd_stream_t stream) {
  if (!W_packed) return MFD_ERR_INVALID_ARG;
  return lmhead_call(h, R, H, nullptr, W_packed, V, topk, tk_logp, tk_tok, lse, status, ws, ws_bytes, stream,
                     nullptr, 0, false, true);
}

size_t mfd_lmhead_packed_fp8_bytes(int V, int H) {
  if (V < 16 || V >= (1 << 30) || H < 1 || H % (2 * mfd::lmhead_k_chunk()) != 0) return 0;
  return mfd::lmhead_packed_fp8_bytes(V, H);
}

int mfd_lmhead_pack_fp8(const void *W, int V, int H, void *W_packed, size_t packed_bytes, mfd_stream_t stream) {
  if (!W || !W_packed || V < 1 || H < 1) return MFD_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(W_packed, 256)) return MFD_ERR_INVALID_ARG;
  const size_t need = mfd_lmhead_packed_fp8_bytes(V, H);
  if (need == 0) return MFD_ERR_UNSUPPORTED;
  if (packed_bytes < need) return MFD_ERR_WORKSPACE;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MFD_OK) return rc;
  if (!is_sm103(d)) return MFD_ERR_UNSUPPORTED;
  return cuda_status(mfd::launch_pack_w_fp8(W, V, H, W_packed, reinterpret_cast<cudaStream_t>(stream)));
}

int mfd_fp8_quantize_rows(const void *x, int R, int H, void *q, float *scale, mfd_stream_t stream) {
  if (!x || !q || !scale || R < 1 || H < 8 || H % 8 != 0) return MFD_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q, 8) || !aligned(scale, 4)) return MFD_ERR_INVALID_ARG;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MFD_OK) return rc;
  if (!is_sm103(d)) return MFD_ERR_UNSUPPORTED;
  return cuda_status(mfd::launch_quant_rows(x, R, H, q, scale, reinterpret_cast<cudaStream_t>(stream)));
}

size_t mfd_lmhead_fp8_workspace_bytes(int R, int H, int V, int topk) {
  if (R < 1 || H < 1 || H % (2 * mfd::lmhead_k_chunk()) != 0 || V < 16 || topk < 1 || topk > 32 || topk > V)
    return 0;
  DeviceInfo d;
  if (current_device_info(&d) != MFD_OK) return 0;
  return fp8_layout(R, H, V, topk, d.n_sm).total;
}

int mfd_lmhead_topk_fp8(const void *h, int R, int H, const void *W_packed_fp8, int V, int topk, float *tk_logp,
                        int32_t *tk_tok, float *lse, int32_t *status, void *ws, size_t ws_bytes,
                        mfd_stream_t stream) {
  if (!W_packed_fp8) return MFD_ERR_INVALID_ARG;
  return lmhead_call(h, R, H, nullptr, W_packed_fp8, V, topk, tk_logp, tk_tok, lse, status, ws, ws_bytes, stream,
                     nullptr, 0, true);
}

int mfd_lmhead_topk_subset(const void *h, int R, int H, const void *W_packed, int V_sub, const int32_t *vocab_ids,
                           int V_full, int topk, float *tk_logp, int32_t *tk_tok, float *lse, int32_t *status,
                           void *ws, size_t ws_bytes, mfd_stream_t stream) {
  if (!W_packed || !vocab_ids || !aligned(vocab_ids, 4)) return MFD_ERR_INVALID_ARG;
  if (V_full < V_sub || V_full >= (1 << 30)) return MFD_ERR_INVALID_ARG;
  return lmhead_call(h, R, H, nullptr, W_packed, V_sub, topk, tk_logp, tk_tok, lse, status, ws, ws_bytes, stream,
                     vocab_ids, V_full);
}

int mfd_logits_topk(const float *logits, int R, int V, int topk, float *tk_logp, int32_t *tk_tok, float *lse,
                    int32_t *status, void *ws, size_t ws_bytes, mfd_stream_t stream) {
  if (!logits || !tk_logp || !tk_tok || !status || R < 1 || V < 1 || topk < 1) return MFD_ERR_INVALID_ARG;
  if (topk > 32 || V < 16 || topk > V || V >= (1 << 30)) return MFD_ERR_UNSUPPORTED;
  const TopkLayout y = logits_layout(R, V, topk);
  if (!ws || ws_bytes < y.total || !aligned(ws, 256)) return MFD_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mfd::LogitsPartialLaunch L;
  L.logits = logits;
  L.R = R;
  L.V = V;
  L.T = y.T;
  L.P = y.P;
  L.chunk = y.chunk;
  L.part_ms = base;
  L.part_cand = base + y.ms_bytes;
  int rc = cuda_status(mfd::launch_logits_partials(L, s));
  if (rc != MFD_OK) return rc;
  mfd::MergeLaunch M;
  M.part_ms = L.part_ms;
  M.part_cand = L.part_cand;
  M.R = R;
  M.P = y.P;
  M.T = y.T;
  M.topk = topk;
  M.tk_logp = tk_logp;
  M.tk_tok = tk_tok;
  M.lse = lse;
  M.status = status;
  M.vocab_ids = nullptr;
  M.V_sub = M.V_full = V;
  return cuda_status(mfd::launch_merge_topk(M, s));
}

int mfd_logits_topk_noalloc(const float *logits, int R, int V, int topk, float *tk_logp, int32_t *tk_tok,
                            float *lse, int32_t *status, mfd_stream_t stream) {
  if (!logits || !tk_logp || !tk_tok || !status || R < 1 || V < 1 || topk < 1) return MFD_ERR_INVALID_ARG;
  if (topk > 32 || V < 16 || topk > V || V >= (1 << 30)) return MFD_ERR_UNSUPPORTED;
  const TopkLayout y = logits_layout(R, V, topk);
  if (y.total > MFD_NOALLOC_SCRATCH_BYTES) return MFD_ERR_WORKSPACE;  // too large for the fixed scratch
  void *scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != MFD_OK) return rc;
  char *base = static_cast<char *>(scratch);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mfd::LogitsPartialLaunch L;
  L.logits = logits;
  L.R = R;
  L.V = V;
  L.T = y.T;
  L.P = y.P;
  L.chunk = y.chunk;
  L.part_ms = base;
  L.part_cand = base + y.ms_bytes;
  rc = cuda_status(mfd::launch_logits_partials(L, s));
  if (rc != MFD_OK) return rc;
  mfd::MergeLaunch M;
  M.part_ms = L.part_ms;
  M.part_cand = L.part_cand;
  M.R = R;
  M.P = y.P;
  M.T = y.T;
  M.topk = topk;
  M.tk_logp = tk_logp;
  M.tk_tok = tk_tok;
  M.lse = lse;
  M.status = status;
  M.vocab_ids = nullptr;
  M.V_sub = M.V_full = V;
  return cuda_status(mfd::launch_merge_topk(M, s));
}

int mfd_build_tree(const float *tk_logp, const int32_t *tk_tok, int n_req, int K, int L, int topk, int B,
                   const int32_t *anchor_tok, const int32_t *base_pos, int32_t *parent, int32_t *token,
                   int32_t *depth, float *score, int32_t *mode, uint32_t *mask, int32_t *pos, int32_t *n_nodes,
                   int32_t *status, void *ws, size_t ws_bytes, mfd_stream_t stream) {
  if (!tk_logp || !tk_tok || !anchor_tok || !parent || !token || !depth || !score || !mode || !mask || !pos ||
      !n_nodes || !status)
    return MFD_ERR_INVALID_ARG;
  if (n_req < 1 || K < 1 || L < 1 || topk < 1 || B < 1) return MFD_ERR_INVALID_ARG;
  if (K > 16 || L > 16 || topk > 32 || B > 512 || K * B > 2048) return MFD_ERR_UNSUPPORTED;
  int cap = 0, tsize = 0;
  if (mfd::tree_smem_bytes(K, L, topk, B, &cap, &tsize) == 0) return MFD_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < tree_bytes(n_req) || !aligned(ws, 256)) return MFD_ERR_WORKSPACE;
  mfd::TreeLaunch T;
  T.tk_logp = tk_logp;
  T.tk_tok = tk_tok;
  T.n_req = n_req;
  T.K = K;
  T.L = L;
  T.topk = topk;
  T.B = B;
  T.anchor = anchor_tok;
  T.base_pos = base_pos;
  T.parent = parent;
  T.token = token;
  T.depth = depth;
  T.score = score;
  T.mode = mode;
  T.mask = mask;
  T.pos = pos;
  T.n_nodes = n_nodes;
  T.status = status;
  return cuda_status(mfd::launch_build_tree(T, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
int verify_call(const float *target_logits, int n_req, int B, int V, int L, const int32_t *parent,
                const int32_t *token, const int32_t *n_nodes, const float *temperature, const uint64_t *seed,
                int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens, int32_t *status, void *ws,
                size_t ws_bytes, mfd_stream_t stream, unsigned long long wait_ns, int withhold) {
  if (!target_logits || !parent || !token || !n_nodes || !temperature || !seed || !accept_len || !path_nodes ||
      !out_tokens || !status)
    return MFD_ERR_INVALID_ARG;
  if (n_req < 1 || B < 1 || V < 2 || L < 1) return MFD_ERR_INVALID_ARG;
  if (B > 512 || L > 16 || V >= (1 << 30)) return MFD_ERR_UNSUPPORTED;
  DeviceInfo d;
  int rc = current_device_info(&d);
  if (rc != MFD_OK) return rc;
  if (!ws || ws_bytes < verify_bytes(d.n_sm) || !aligned(ws, 256)) return MFD_ERR_WORKSPACE;
  // the target logits: device memory, or page-locked host memory mapped into
  // the device's address space, which the walk reads in place (only the rows
  // on the walk cross the host link)
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, target_logits) != cudaSuccess) {
    (void)cudaGetLastError();
    return MFD_ERR_INVALID_ARG;
  }
  const float *t = target_logits;
  if (pa.type == cudaMemoryTypeHost) {
    if (!pa.devicePointer) return MFD_ERR_INVALID_ARG;
    t = static_cast<const float *>(pa.devicePointer);
  } else if (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged) {
    return MFD_ERR_INVALID_ARG;  // pageable host memory
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mfd::VerifyLaunch Vl;
  Vl.t = t;
  Vl.n_req = n_req;
  Vl.B = B;
  Vl.V = V;
  Vl.L = L;
  Vl.parent = parent;
  Vl.token = token;
  Vl.n_nodes = n_nodes;
  Vl.temperature = temperature;
  Vl.seed = seed;
  Vl.accept_len = accept_len;
  Vl.path_nodes = path_nodes;
  Vl.out_tokens = out_tokens;
  Vl.status = status;
  Vl.ws = static_cast<unsigned long long *>(ws);
  Vl.grid = mfd::verify_max_grid(d.n_sm);
  Vl.wait_ns = wait_ns;
  Vl.withhold = withhold;
  return cuda_status(mfd::launch_verify(Vl, s));
}
}  // namespace

extern "C" {

int mfd_verify(const float *target_logits, int n_req, int B, int V, int L, const int32_t *parent,
               const int32_t *token, const int32_t *n_nodes, const float *temperature, const uint64_t *seed,
               int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens, int32_t *status, void *ws,
               size_t ws_bytes, mfd_stream_t stream) {
  return verify_call(target_logits, n_req, B, V, L, parent, token, n_nodes, temperature, seed, accept_len,
                     path_nodes, out_tokens, status, ws, ws_bytes, stream, 0ull, 0);
}

int mfd_verify_withheld_test(const float *target_logits, int n_req, int B, int V, int L, const int32_t *parent,
                             const int32_t *token, const int32_t *n_nodes, const float *temperature,
                             const uint64_t *seed, int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens,
                             int32_t *status, void *ws, size_t ws_bytes, uint64_t wait_limit_ns,
                             mfd_stream_t stream) {
  if (wait_limit_ns < 1000ull || wait_limit_ns > 100000000ull) return MFD_ERR_INVALID_ARG;
  return verify_call(target_logits, n_req, B, V, L, parent, token, n_nodes, temperature, seed, accept_len,
                     path_nodes, out_tokens, status, ws, ws_bytes, stream, wait_limit_ns, 1);
}

}  // extern "C"
