/*
 * mfd.h -- C ABI of libmfd: the per-round drafting-and-verification hot path
 * of Multi-Future Drafting (MFD) on one GB300 (sm_103a).
 *
 * A round (project page "Multi-Future Drafting", How it works, steps 2-3, and
 * Figure 2; model card "MFD drafter for Qwen3.5-4B", Model table and first
 * paragraph) is three calls on one CUDA stream:
 *
 *   mfd_lmhead_topk  the K modes' drafter hidden states for the L drafted
 *                    positions go through the target's LM head; per row an
 *                    online log-softmax over the vocabulary and the top-k.
 *   mfd_build_tree   the mixture DDTree: the B prefixes with the highest
 *                    best-mode log-probability, shared prefixes built once;
 *                    parent/token/depth arrays and the tree-attention mask.
 *   mfd_verify       the standard tree verification walk against the
 *                    target's per-node logits: greedy, or lossless sampled
 *                    with a counter-based Gumbel-max.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory owned by the caller, contiguous
 *     row-major, unless marked "host".  The library allocates nothing and
 *     keeps no per-call state; it only caches TMA descriptors (see
 *     mfd_lmhead_topk) and per-device attributes.
 *   - Work is enqueued on `stream` and never synchronises the host.
 *   - The return value reports argument and launch errors synchronously.
 *     Errors found on the device are stored into `*status` (one int32 in
 *     device memory).  The caller sets *status to MFD_OK before the round;
 *     a kernel that finds a problem stores its code only if *status is still
 *     MFD_OK (the first error wins) and no kernel ever clears it.
 *   - Scratch memory is the caller's: `ws` / `ws_bytes`, at least
 *     mfd_workspace_size(...) bytes, 256-byte aligned, reused freely
 *     between calls that do not overlap on the GPU.
 *   - Rows of the drafted block: r = (q * K + k) * L + i for request q, mode
 *     k in [0, K) and drafted position i in [0, L) (depth i + 1).
 *
 * Limits: 1 <= K <= 16, 1 <= L <= 16, 1 <= topk <= 32, 1 <= B <= 512,
 * K * B <= 2048, H % 64 == 0, 16 <= V < 2^30 (and V >= topk).
 */
#ifndef MFD_H_
#define MFD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same type as cudaStream_t); NULL is the legacy stream. */
typedef struct CUstream_st *mfd_stream_t;

typedef enum {
  MFD_OK = 0,
  MFD_ERR_INVALID_ARG = 1, /* NULL pointer, size out of range, misalignment */
  MFD_ERR_UNSUPPORTED = 2, /* valid but outside the limits above, or no sm_103a device */
  MFD_ERR_WORKSPACE = 3,   /* ws NULL or smaller than mfd_workspace_size */
  MFD_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  MFD_ERR_TIMEOUT = 5,     /* device: a bounded wait ran out (kernel exited early) */
  MFD_ERR_INPUT = 6,       /* device: input values break the contract (see each call) */
  MFD_ERR_CHECK = 7        /* device, bounds-checked build (libmfd_checked) only: an index
                              computed from data fell outside its array; the access was
                              clamped into the array and the results are not to be trusted */
} mfd_status;

/* Static English text for a status code; never NULL. */
const char *mfd_status_string(int status);

/* Operation ids for mfd_workspace_size. */
enum {
  MFD_OP_LMHEAD_TOPK = 0,
  MFD_OP_LOGITS_TOPK = 1,
  MFD_OP_BUILD_TREE = 2,
  MFD_OP_VERIFY = 3,
  MFD_OP_TREE_ANALYTICS = 4
};

/* Bytes of scratch that `op` needs for the given sizes on the CURRENT CUDA
 * device (the LM-head and verify splits follow its SM count).  Arguments an
 * op does not use are ignored: LMHEAD_TOPK uses (R, V, topk); LOGITS_TOPK
 * uses (R, V, topk); BUILD_TREE uses (n_req); VERIFY uses (n_req);
 * TREE_ANALYTICS uses (n_req, B).
 * Returns 0 for an unknown op or sizes outside the limits. */
size_t mfd_workspace_size(int op, int n_req, int K, int L, int topk, int B, int R, int V);

/* LM head, log-softmax and top-k.
 * Model card "MFD drafter for Qwen3.5-4B", Model table: the drafter uses the
 * target's LM head at run time; project page, How it works, step 2: each
 * (mode, position) gives one distribution over the vocabulary.
 *
 *   z[r][v]     = sum_h h[r][h] * W[v][h]        (bf16 x bf16, fp32 accumulate)
 *   lse[r]      = log sum_v exp(z[r][v])          (natural log)
 *   tk_tok[r][] = the topk token ids of largest z[r][.], ties to the smaller id
 *   tk_logp[r][j] = z[r][tk_tok[r][j]] - lse[r]   (fp32)
 * Each output row is sorted by (tk_logp descending, token id ascending).
 * The logits never reach global memory.
 *
 *   h        bf16 [R][H], 16-byte aligned (TMA source)
 *   W        bf16 [V][H], 16-byte aligned (TMA source); streamed once
 *   tk_logp  fp32 [R][topk]      out
 *   tk_tok   int32 [R][topk]     out
 *   lse      fp32 [R]            out, may be NULL
 *   status   int32 [1]           device status word (MFD_ERR_TIMEOUT on a
 *                                bounded pipeline wait running out)
 * Requires an sm_103a device.  TMA descriptors for (h, W, R, H, V) are
 * encoded on the first call and cached by (pointer, shape); the cache is
 * thread-safe.  Hidden rows that span 144 KB or less (R * H * 2 bytes) are
 * first copied into ws, padded with zero rows: every CTA reads them, and on
 * GB300 rows within so few bytes of address space are served by few L2
 * slices.  The copy changes no result.  With R <= 128 the vocabulary
 * ranges also share, through ws, a lower bound on each row's topk-th best
 * logit (the smallest of topk per-residue-class maxima of published
 * candidates, token id mod topk), and a range skips a column below it; the
 * bound changes no result.  ws needs no zeroing for it: its first 16 bytes
 * hold a generation word and a ready word, each call advances the
 * generation, clears the bound and only then stores ready = the splitmix64
 * finalizer of the new generation, and the CTAs trust the bound only after
 * they read that value.  Contents left by other calls are mistaken for a
 * cleared bound only if the ready word already equals that value, which
 * fresh, zeroed or pattern-filled memory does not hold.  Errors: INVALID_ARG
 * (NULL, R < 1, misaligned h/W), UNSUPPORTED (limits, device), WORKSPACE,
 * CUDA. */
int mfd_lmhead_topk(const void *h, int R, int H, const void *W, int V, int topk,
                    float *tk_logp, int32_t *tk_tok, float *lse, int32_t *status, void *ws,
                    size_t ws_bytes, mfd_stream_t stream);

/* The LM-head weight packed for streaming.  The weight is fixed for a model
 * (model card "MFD drafter for Qwen3.5-4B", Model table: the target's LM
 * head), so it can be laid out once, when the model is loaded, in the order
 * mfd_lmhead_topk_packed streams it: per vocabulary tile of 256 rows and per
 * 64-element K slice, one 32 KB block holding that slice of the 256 rows in
 * the MMA's 128-byte-swizzled shared-memory order; rows past V are zero.
 * Every pipeline stage then reads one contiguous piece of memory.
 *
 * mfd_lmhead_packed_bytes: bytes of the packed weight for (V, H), or 0 outside
 *   the limits of mfd_lmhead_topk.
 * mfd_lmhead_pack: W bf16 [V][H] (16-byte aligned) -> W_packed (device,
 *   256-byte aligned, packed_bytes >= mfd_lmhead_packed_bytes(V, H)).  Errors:
 *   INVALID_ARG (NULL, V or H < 1, misaligned), UNSUPPORTED (limits, device),
 *   WORKSPACE (W_packed too small), CUDA.  Enqueued on `stream`.
 * mfd_lmhead_topk_packed: mfd_lmhead_topk with the packed weight in place of
 *   W; same arguments, workspace (MFD_OP_LMHEAD_TOPK), outputs and errors, and
 *   bit-identical results. */
size_t mfd_lmhead_packed_bytes(int V, int H);
int mfd_lmhead_pack(const void *W, int V, int H, void *W_packed, size_t packed_bytes, mfd_stream_t stream);
int mfd_lmhead_topk_packed(const void *h, int R, int H, const void *W_packed, int V, int topk,
                           float *tk_logp, int32_t *tk_tok, float *lse, int32_t *status, void *ws,
                           size_t ws_bytes, mfd_stream_t stream);

/* FP8 drafter head (project page "Multi-Future Drafting", In a serving
 * engine, Figure 5 caption: MFD runs its drafter's linear layers in FP8, the
 * serving engine's online option, and the acceptance length is unchanged;
 * decoding stays lossless because the walk verifies against the target's own
 * logits).  The pages name no format or scale granularity; this library's
 * reading: E4M3 values (round to nearest even, saturating at +-448), one
 * scale for the whole weight, one scale per hidden row computed on the fly:
 *   s_W = max|W| / 448,   Wq = e4m3(W * (448 / max|W|))        (once, at load)
 *   t_r = max|h[r]| / 448, hq = e4m3(h[r] * (448 / max|h[r]|)) (every call)
 *   z[r][v] = (t_r * s_W) * sum_h hq[r][h] Wq[v][h]   (exact E4M3 products,
 *                                                       fp32 accumulation)
 * then the log-softmax and top-k of mfd_lmhead_topk.  An all-zero row or
 * weight has scale 0.  Every fp32 step is one IEEE-rounded operation.
 *
 * mfd_lmhead_packed_fp8_bytes: bytes of the E4M3 packed weight for (V, H):
 *   per 256-row vocabulary tile and 128-element K slice one 32 KB block of
 *   the 128-byte-swizzled shared-memory image (as mfd_lmhead_pack, 128 values
 *   a row), rows past V zero, then a 256-byte trailer whose first word is
 *   max|W| (fp32).  0 unless H % 128 == 0 and V within the limits.
 * mfd_lmhead_pack_fp8: W bf16 [V][H] (16-byte aligned) -> W_packed (device,
 *   256-byte aligned).  Errors as mfd_lmhead_pack.  Enqueued on `stream`.
 * mfd_fp8_quantize_rows: x bf16 [R][H] (16-byte aligned, H % 8 == 0) ->
 *   q uint8 [R][H] (E4M3, 8-byte aligned) and scale fp32 [R] = t_r.
 *   Errors: INVALID_ARG, UNSUPPORTED (device), CUDA.
 * mfd_lmhead_fp8_workspace_bytes: scratch of mfd_lmhead_topk_fp8 (the
 *   LM head's partials plus the E4M3 hidden rows and their scales) on the
 *   current device; 0 outside the limits (H % 128 != 0 included).
 * mfd_lmhead_topk_fp8: mfd_lmhead_topk_packed with the E4M3 packed weight;
 *   h stays bf16 (quantized inside the call); ws_bytes >=
 *   mfd_lmhead_fp8_workspace_bytes(R, H, V, topk).  Outputs and errors as
 *   mfd_lmhead_topk. */
size_t mfd_lmhead_packed_fp8_bytes(int V, int H);
int mfd_lmhead_pack_fp8(const void *W, int V, int H, void *W_packed, size_t packed_bytes, mfd_stream_t stream);
int mfd_fp8_quantize_rows(const void *x, int R, int H, void *q, float *scale, mfd_stream_t stream);
size_t mfd_lmhead_fp8_workspace_bytes(int R, int H, int V, int topk);
int mfd_lmhead_topk_fp8(const void *h, int R, int H, const void *W_packed_fp8, int V, int topk,
                        float *tk_logp, int32_t *tk_tok, float *lse, int32_t *status, void *ws,
                        size_t ws_bytes, mfd_stream_t stream);

/* Draft-vocabulary subset head (project page "Multi-Future Drafting", In a
 * serving engine: the serving build drafts only over the target's most
 * frequent tokens, about 64K of them, while the walk still checks against
 * every token, so the output distribution is the target's).  As
 * mfd_lmhead_topk_packed over the subset:
 *   W_packed     the packed (mfd_lmhead_pack) weight of the V_sub subset rows
 *   vocab_ids    int32 [V_sub] device: the vocabulary id of each subset row,
 *                strictly increasing, each in [0, V_full)
 * The log-softmax and top-k are over the subset (the drafter's
 * distribution); tk_tok holds vocabulary ids (vocab_ids[row]), in the order
 * (log p desc, id asc).  A mapped id outside [0, V_full) sets MFD_ERR_INPUT
 * in *status and is written as -1; a table that is not increasing gives ties
 * in subset order.  Workspace: mfd_workspace_size(MFD_OP_LMHEAD_TOPK, ...)
 * with V = V_sub.  Errors: as mfd_lmhead_topk_packed; NULL vocab_ids or
 * V_full < V_sub -> MFD_ERR_INVALID_ARG. */
int mfd_lmhead_topk_subset(const void *h, int R, int H, const void *W_packed, int V_sub, const int32_t *vocab_ids,
                           int V_full, int topk, float *tk_logp, int32_t *tk_tok, float *lse, int32_t *status,
                           void *ws, size_t ws_bytes, mfd_stream_t stream);

/* Log-softmax and top-k of fp32 logits given directly (no LM head): the
 * same outputs as mfd_lmhead_topk with z = logits [R][V].  Non-finite logits
 * are the caller's responsibility. */
int mfd_logits_topk(const float *logits, int R, int V, int topk, float *tk_logp,
                    int32_t *tk_tok, float *lse, int32_t *status, void *ws, size_t ws_bytes,
                    mfd_stream_t stream);

/* Log-softmax and top-k of given fp32 logits, like mfd_logits_topk, for
 * callers that cannot allocate device memory at the point where they call
 * (for instance code that runs after its memory budget is fixed, or that
 * must not pay the implicit synchronisation of cudaMalloc): it takes no
 * workspace.  The paper has no counterpart to this entry point; it is a
 * library convenience.
 *
 * Scratch comes from one array of MFD_NOALLOC_SCRATCH_BYTES bytes that the
 * library reserves as a static device variable on every GPU that loads it,
 * for the life of the process.  The scratch needed is
 * mfd_workspace_size(MFD_OP_LOGITS_TOPK, ...) for the same R, V and topk;
 * larger problems are rejected with MFD_ERR_WORKSPACE (use mfd_logits_topk).
 * The first call on a device looks up that array's device address (once per
 * device); make that first call before any stream capture.  The address is
 * kept for the life of the process: after cudaDeviceReset it is stale, so a
 * caller that resets a device must not call this entry point on it again.  All calls share
 * the one array and it keeps the last call's contents: calls that may
 * overlap on the GPU (different streams, or different host threads) race on
 * it, so serialise them.  Arguments and results are those of
 * mfd_logits_topk; no allocation is made. */
#define MFD_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)
int mfd_logits_topk_noalloc(const float *logits, int R, int V, int topk, float *tk_logp,
                            int32_t *tk_tok, float *lse, int32_t *status, mfd_stream_t stream);

/* Mixture DDTree (project page, How it works, step 3, and the Figure 1/2
 * caption): mode k scores a prefix x = (x_1..x_d) by the fp32 left fold,
 * in depth order, of its per-position table log-probabilities; a token not
 * in mode k's top-k row at that position makes x unreachable for mode k.
 * s(x) = max_k score_k(x).  Order: x before y iff s(x) > s(y), or s(x) ==
 * s(y) and x's token ids are lexicographically smaller (unsigned, a proper
 * prefix first).  The tree keeps the first B prefixes of depth 1..L with
 * finite s, which is the union of the per-mode trees at the common cut-off.
 *
 *   tk_logp, tk_tok  [n_req][K][L][topk], rows as mfd_lmhead_topk writes
 *                    them: log-probabilities (<= 0, not NaN) sorted
 *                    descending with distinct tokens; otherwise *status =
 *                    MFD_ERR_INPUT.  -inf entries are never used.
 *   anchor_tok       int32 [n_req]  token of the root (node 0)
 *   base_pos         int32 [n_req]  position of the root, may be NULL (0)
 * Outputs, N = B + 1 nodes per request, W32 = ceil(N / 32):
 *   parent  int32 [n_req][N]       parent node (-1 for the root)
 *   token   int32 [n_req][N]       node token (anchor for the root)
 *   depth   int32 [n_req][N]       0 for the root, 1..L otherwise
 *   score   fp32  [n_req][N]       s(x) (0 for the root)
 *   mode    int32 [n_req][N]       smallest mode attaining s(x) (-1 root)
 *   mask    uint32 [n_req][N][W32] bit j of word j/32 of row i set iff node j
 *                                  is on the root->i path (inclusive)
 *   pos     int32 [n_req][N]       base_pos + depth
 *   n_nodes int32 [n_req]          1 + number of kept prefixes (<= N)
 * Node 0 is the root; nodes 1.. follow the order above (so parent[i] < i).
 * Rows at and past n_nodes hold -1 (ints), -inf (score) and 0 (mask). */
int mfd_build_tree(const float *tk_logp, const int32_t *tk_tok, int n_req, int K, int L,
                   int topk, int B, const int32_t *anchor_tok, const int32_t *base_pos,
                   int32_t *parent, int32_t *token, int32_t *depth, float *score,
                   int32_t *mode, uint32_t *mask, int32_t *pos, int32_t *n_nodes,
                   int32_t *status, void *ws, size_t ws_bytes, mfd_stream_t stream);

/* Tree verification walk (model card, first paragraph; project page,
 * Figure 2 (c)): from the root, the target picks a token y at the current
 * node -- greedy (temperature 0): y = argmax_v t[cur][v]; sampled
 * (temperature T > 0): y = argmax_v (t[cur][v] / T + G(seed, cur, v)), a
 * Gumbel-max draw from softmax(t / T), where G = -log(-log(u)),
 * u = (2 * (x >> 9) + 1) * 2^-24 and x is word v mod 4 of the Philox4x32-10
 * block (Salmon et al., SC'11) at counter (v div 4, cur, 0, 0), key (seed
 * low, seed high).  Ties go to the smaller v.  If a child of cur carries y the walk moves there,
 * otherwise y is the bonus token and the walk stops.
 *
 *   target_logits fp32 [n_req][B + 1][V]; only the rows on the walk are read.
 *                 Device memory, or page-locked host memory mapped into the
 *                 device's address space (cudaHostAlloc, or cudaHostRegister
 *                 with mapping), which the walk reads in place: then only the
 *                 rows on the walk cross the host link (NVLink-C2C on GB300).
 *                 Pageable host memory -> MFD_ERR_INVALID_ARG.
 *   parent, token int32 [n_req][B + 1] and n_nodes int32 [n_req] from
 *                 mfd_build_tree (or any tree in that format)
 *   temperature   fp32 [n_req]  0 = greedy; < 0 or NaN -> MFD_ERR_INPUT
 *   seed          uint64 [n_req]
 *   accept_len    int32 [n_req]         drafted tokens accepted (0..L)
 *   path_nodes    int32 [n_req][L + 1]  node read at step j (path_nodes[0] = 0)
 *   out_tokens    int32 [n_req][L + 1]  y at step j: accepted tokens, bonus last
 * Entries past accept_len hold -1.  Below 8 requests the walk is one
 * cooperative grid with a bounded grid-wide wait per step (MFD_ERR_TIMEOUT if
 * it runs out); its CTAs exchange step results through ws, which needs no
 * zeroing: its words carry a generation counter that each call advances, so
 * ws may be shared with other calls and replayed in CUDA graphs (only calls
 * overlapping on the GPU must not share it).  From 8 requests on, each
 * request is walked by one thread-block cluster (up to 16 CTAs) whose CTAs
 * exchange each step's result in their shared memory behind a hardware
 * cluster barrier; ws is then not written.  Both forms give the same
 * results. */
int mfd_verify(const float *target_logits, int n_req, int B, int V, int L,
               const int32_t *parent, const int32_t *token, const int32_t *n_nodes,
               const float *temperature, const uint64_t *seed, int32_t *accept_len,
               int32_t *path_nodes, int32_t *out_tokens, int32_t *status, void *ws,
               size_t ws_bytes, mfd_stream_t stream);

/* Tree analytics: what a tree spends its budget on (project page "Multi-Future
 * Drafting", TL;DR and Abstract: chimeras -- prefixes spliced from different
 * futures that the target never produces; How it works, step 1, and "What the
 * modes are", Figure 3: the expected number of accepted tokens is the
 * probability mass the tree covers, read depth by depth).  Not part of a
 * round: an analysis of trees against known futures and target logits.
 *
 *   parent, token, depth int32 [n_req][B + 1], n_nodes int32 [n_req]: trees
 *                 in mfd_build_tree's format (parents before children)
 *   futures       int32 [n_req][F][L]: the futures a chimera splices
 *   target_logits fp32 [n_req][B + 1][V] (device memory); temperature fp32
 *                 [n_req] (0 = greedy)
 * Outputs:
 *   node_class int32 [n_req][B + 1]: MFD_NODE_ON_FUTURE (the root, or a prefix
 *              of some future), MFD_NODE_CHIMERA (every token is some future's
 *              token at that position, yet the prefix is no future's),
 *              MFD_NODE_OTHER; -1 past n_nodes
 *   reach  double [n_req][B + 1]: probability that the verification walk
 *              arrives at the node: the product, root first, of the target's
 *              probability of each next token -- softmax(t[parent] / T)[token]
 *              for T > 0, 1 or 0 for the greedy choice (argmax, smallest id on
 *              ties) at T = 0; 0 past n_nodes
 *   mass   double [n_req][L + 1]: sum of reach over the nodes at each depth
 *              (mass[0] = 1); summed over depths >= 1 it is the expected
 *              accepted length
 * Probabilities are computed in double.  Limits: B <= 512, L <= 16, F >= 1.
 * ws: mfd_workspace_size(MFD_OP_TREE_ANALYTICS, n_req, .., B, ..) bytes.
 * Errors: INVALID_ARG, UNSUPPORTED (limits), WORKSPACE, CUDA; a tree that is
 * not topological, a depth that is not its parent's plus one, a token outside
 * [0, V) or a negative temperature set MFD_ERR_INPUT in *status. */
enum { MFD_NODE_ON_FUTURE = 0, MFD_NODE_CHIMERA = 1, MFD_NODE_OTHER = 2 };
int mfd_tree_analytics(const int32_t *parent, const int32_t *token, const int32_t *depth,
                       const int32_t *n_nodes, int n_req, int B, int L, const int32_t *futures, int F,
                       const float *target_logits, int V, const float *temperature, int32_t *node_class,
                       double *reach, double *mass, int32_t *status, void *ws, size_t ws_bytes,
                       mfd_stream_t stream);

/* MFD-D, the single-mode default path (project page "Multi-Future Drafting",
 * In a serving engine, the MFD-D paragraph and Figure 5): the same drafter
 * drafts all K modes while few requests are in flight and switches to its
 * single-mode default path from three requests on, where the draft cost of
 * K modes grows with the batch while the acceptance length does not.  The
 * returned count is the K to pass to the round's calls (the single-mode
 * round is the same three calls with K = 1: its tree is the product-ranked
 * one).  Host only; no device work.
 *   returns K for 1 <= n_req < MFD_MFDD_SWITCH_REQUESTS, 1 for n_req at or
 *   above it, and 0 for n_req < 1 or K outside [1, 16]. */
#define MFD_MFDD_SWITCH_REQUESTS 3
int mfd_mfdd_modes(int n_req, int K);

/* Fault injection for the LM head's bounded waits, for tests (the pages have
 * no counterpart: it exists so that the kernel's timeout path can be
 * exercised without faulting or hanging a GPU).  Arguments and outputs as
 * mfd_lmhead_topk_packed; every CTA's producer stops after the CTA's first
 * weight tile, so the MMA warp's next wait gives up after the kernel's wait
 * limit (1 s): it stores MFD_ERR_TIMEOUT in *status and raises the CTA's
 * abort flag, the epilogue warps leave their waits, the MMAs already issued
 * drain, tensor memory is released and every CTA returns.  The outputs are
 * then not meaningful; the next call on the same buffers is exact.  Errors:
 * those of mfd_lmhead_topk_packed. */
int mfd_lmhead_withheld_test(const void *h, int R, int H, const void *W_packed, int V, int topk,
                             float *tk_logp, int32_t *tk_tok, float *lse, int32_t *status, void *ws,
                             size_t ws_bytes, mfd_stream_t stream);

/* Fault injection for the walk's bounded waits, for tests (the pages have no
 * counterpart: it exists so that the timeout path can be exercised without
 * faulting or hanging a GPU).  Arguments and outputs as mfd_verify, always
 * walked by the cooperative grid (the form with waits), plus
 * wait_limit_ns in [1e3, 1e8]: every bounded wait of this call gives up after
 * that long.  In every request group of more than one CTA (V >= 2048), the
 * CTAs other than the group's first never publish their step result, so the
 * first CTA's gather runs out, nobody publishes a winner, and the others' waits
 * run out too: every CTA returns and *status = MFD_ERR_TIMEOUT.  The
 * workspace's generation still advances, so the next mfd_verify on the same
 * workspace is correct.  Errors: those of mfd_verify; INVALID_ARG for a limit
 * outside the range. */
int mfd_verify_withheld_test(const float *target_logits, int n_req, int B, int V, int L,
                             const int32_t *parent, const int32_t *token, const int32_t *n_nodes,
                             const float *temperature, const uint64_t *seed, int32_t *accept_len,
                             int32_t *path_nodes, int32_t *out_tokens, int32_t *status, void *ws,
                             size_t ws_bytes, uint64_t wait_limit_ns, mfd_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MFD_H_ */
