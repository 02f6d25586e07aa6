// lmhead.cu -- the target's LM head on the drafter's hidden states, with the
// log-softmax and per-row top-k fused into the epilogue (model card "MFD
// drafter for Qwen3.5-4B", Model table: the target LM head is applied at run
// time; project page "Multi-Future Drafting", How it works, step 2: one
// distribution per mode and position).
//
// Shape of the work: R hidden rows (K modes x L positions per request) times
// a V x H bf16 weight.  At R <= 128 the weight stream (V*H*2 bytes) is the
// whole cost, so the kernel reads W exactly once, with TMA, and keeps the
// logits in tensor memory: they never reach global memory.
//
//   D[128 x BN] (TMEM, fp32) = h_tile[128 x H] . W_tile[BN x H]^T
//
// A = 128 hidden rows (one M tile, zero-filled past R), B = BN vocabulary
// rows (256, or 128 when 256-row tiles would leave SMs idle), K streamed
// through a shared-memory ring of one 64-element (128-byte, swizzled) K atom
// per stage.  Each TMEM lane is one hidden row, so the
// epilogue thread that owns lane r reads its row's logits column by column
// and keeps the row's running max, running sum of exp and a sorted top-T in
// registers -- no cross-thread reduction.
//
// Grid: persistent, one CTA per SM.  The vocabulary is split into P
// contiguous ranges of BN-row tiles; work item = (range, M tile).  A CTA
// writes, per row and range, (max, sum exp) and its T best (logit, id)
// pairs; merge_topk (topk.cu) combines the P partials of a row.
//
// Many M tiles (R > 128): the work items of one vocabulary range are its M
// tiles; the host orders items range-major, so the CTAs of a range stream the
// same weight tiles at about the same time and each weight tile comes from
// HBM about once and from L2 for the other M tiles.  Every CTA loads only
// into its own shared memory.
//
// Roles (224 threads): warp 0 = TMA producer, warp 1 = MMA issuer (one
// thread each), warps 2-5 = epilogue (warp w reads TMEM lanes 32*(w%4)..),
// warp 6 = the row bound's upkeep (one M tile; see the row bound below).
// TMEM holds 512 / BN fp32 accumulators, so that the MMAs run ahead of the
// epilogue while a range's first tile, where the row's top-T fills, is
// worked through.
//
// FP8 form (project page, In a serving engine, Figure 5 caption: the
// drafter's linear layers in FP8, quantized online): the weight is packed
// once as E4M3 with one scale for the whole tensor, the hidden rows are
// quantized per call with one scale per row (quant_rows_kernel), and the MMA
// is tcgen05 kind::f8f6f4 with an fp32 accumulator.  A stage then holds a
// 128-element K slice (the same 128-byte swizzled rows, the same 48 KB), so
// the weight stream is half the bytes; the epilogue scales the accumulator
// by the row's factor f_r = t_r * s_W before the softmax and top-k.
#include <cuda_fp8.h>

#include "lmhead.h"
#include "mfd_device.cuh"

namespace mfd {
namespace {

constexpr int BM = 128;
constexpr int PK = 256;           // vocabulary rows of a packed weight block
constexpr int BK = 64;            // one 128-byte swizzle atom of bf16
constexpr int BK8 = 128;          // one 128-byte swizzle atom of E4M3
constexpr int KSUB = 1;           // K atoms per pipeline stage
constexpr int A_SUB = BM * BK * 2;  // one K atom of the hidden tile
constexpr int PK_SUB = PK * BK * 2;  // one K atom of a packed block
constexpr int A_BYTES = KSUB * A_SUB;
constexpr int THREADS = 224;
constexpr int TMEM_COLS = 512;

// Tile shape.  BN = 256: two 256-column accumulators and a 4-stage ring of
// 48 KB stages, two thirds of them weight.  A CTA streams about as many
// bytes at once whatever the split, and at one M tile the weight's share of
// them sets its rate.  Several M tiles also load the hidden tile half as
// often per weight byte.  BN = 128: four 128-column accumulators and a
// 6-stage ring of 32 KB stages, half of them weight, for vocabularies too
// small to give every SM a 256-row tile.
template <int BN_>
struct Tile {
  static constexpr int BN = BN_;
  static constexpr int NACC = TMEM_COLS / BN;
  static constexpr int STAGES = BN == 128 ? 6 : 4;
  static constexpr int B_SUB = BN * BK * 2;  // one K atom of the weight tile
  static constexpr int B_BYTES = KSUB * B_SUB;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
};
constexpr float LOG2E = 1.4426950408889634f;
constexpr int STAGE_STRIDE = 36;  // floats per staged row (16-byte aligned rows)
constexpr int STAGE_ROW_BYTES = 32 * STAGE_STRIDE * 4;  // one epilogue warp's 32 rows

template <int BN>
constexpr int smem_bytes() {
  using TL = Tile<BN>;
  return 1024 /* alignment slack */ + TL::STAGES * TL::STAGE_BYTES + 4 * STAGE_ROW_BYTES +
         8 * (2 * TL::STAGES + 2 * TL::NACC + 1) + 16 + 4 * BM + 16;
}

// Row bound (one M tile).  A column below the row's k-th best logit over the
// whole vocabulary cannot reach the row's top-k, so a range need not insert
// it.  Such a bound: split the vocabulary ids into G = k residue classes
// (id mod k) and let every range publish its list's first two entries into
// their classes' slots (an integer max of the value's order key); the
// smallest of the k class maxima is then the value of k distinct columns at
// least, so at most the k-th best.  A range inserts a column only if it
// beats both its own T-th entry and that bound; every column of the final
// top-k still enters its range's list, and the lists stay real, sorted
// candidates, which is all the merge needs.  The slots live in the
// workspace, cleared per call by CTA 0 behind a generation handshake (the
// same scheme as the verify walk's): every CTA reads gen, expects
// ready == mix(gen + 1), and trusts the slots only after seeing that;
// CTA 0 clears them, stores ready with release semantics, and writes
// gen + 1 into gen when it leaves.  A seventh warp keeps this CTA's copy of
// the bounds (shared memory) current; publications need no handshake, since
// a clear can only lose one, never make one wrong.
constexpr int KEY_NEG_INF = (int)0x807FFFFF;  // ord_key(-inf)
constexpr int RB_READY_POLLS = 1 << 16;       // x ~128 ns before a CTA gives up on the bound
constexpr int RB_PASSES = 1 << 22;
constexpr unsigned RB_SLEEP_NS = 256;
constexpr int RB_BATCH = 8;  // 16-byte slot loads a lane has in flight at once

// the largest float below g (-inf for -inf), so that x >= g is x > below(g)
// for every non-NaN x; denormals are compared as they are (no flush to zero)
__device__ __forceinline__ float below(float g) {
  if (!(g > -INFINITY)) return -INFINITY;
  if (g == 0.f) return __int_as_float((int)0x80000001);
  const int b = __float_as_int(g);
  return __int_as_float(g > 0.f ? b - 1 : b + 1);
}

// splitmix64's finalizer (Steele, Lea, Flood, OOPSLA'14): a bijection, so
// distinct generations give distinct ready words
__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ int4 ld_relaxed_v4(const int *p) {
  int4 v;
  asm volatile("ld.relaxed.gpu.global.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void red_max(int *p, int v) {
  asm volatile("red.relaxed.gpu.global.max.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct Params {
  int R, H, V;
  int n_mt;     // M tiles of 128 rows
  int n_vt;     // vocabulary tiles of 256 rows
  int P;        // vocabulary ranges
  int n_items;  // n_mt * P
  float2 *part_ms;  // [R][P]      (running max, sum exp(z - max))
  int2 *part_cand;  // [R][P][T]   (logit bits, token id), best first
  int32_t *status;
  const uint8_t *w_packed;  // packed weight (see pack_w_kernel), or null
  const float *row_scale;   // FP8: t_r per hidden row [R]
  const float *w_amax;      // FP8: the weight's largest magnitude (s_W = w_amax / 448)
  int withhold;             // fault injection for tests: the producer stops after each CTA's first tile
  int *rb;                  // row bound (one M tile): int [R][T] class maxima (order keys), or null
  unsigned long long *rb_gen, *rb_ready;
  int G;                    // residue classes of the row bound (the top-k)
};

// Work item -> (M tile, vocabulary tiles [t0, t1), range); items are
// range-major.
__device__ __forceinline__ void item_range(const Params &p, int item, int &mt, int &t0, int &t1, int &range) {
  range = item / p.n_mt;
  mt = item - range * p.n_mt;
  t0 = (int)(((long long)range * p.n_vt) / p.P);
  t1 = (int)(((long long)(range + 1) * p.n_vt) / p.P);
}

// The packed weight holds 256-row blocks (pack_w_kernel).  The K atom kc of
// 256-row tile t is block (t, kc); that of 128-row tile t is half of block
// (t / 2, kc): its first 16 KB for an even tile, its second for an odd one.
// A half is self-contained: the swizzle repeats every 8 rows.
template <int BN>
__device__ __forceinline__ const uint8_t *packed_at(const uint8_t *w, int t, int kc, int nk) {
  if (BN == PK) return w + ((size_t)t * nk + kc) * PK_SUB;
  return w + ((size_t)(t >> 1) * nk + kc) * PK_SUB + (size_t)(t & 1) * Tile<BN>::B_SUB;
}

// Insert (x, v) into the sorted (value desc, id asc) list; the caller has
// checked that x beats the last entry.  b[s] = entry s stays before (x, v);
// the b's are true up to x's place and false after it, so entry s keeps its
// place when b[s], takes (x, v) when b[s - 1] alone holds, and takes entry
// s - 1 otherwise: T independent compares and two selects per entry, with no
// position to count or compare.  A row's columns come in increasing id
// order, so every listed id is below v (the empty list's entries are -inf,
// which x beats): entry s stays before (x, v) exactly when its value is at
// least x, one compare.
template <int T>
__device__ __forceinline__ void topk_insert(float (&tv)[T], int (&ti)[T], float x, int v) {
  bool b[T];
#pragma unroll
  for (int s = 0; s < T; ++s) b[s] = tv[s] >= x;
#pragma unroll
  for (int s = T - 1; s > 0; --s) {  // tv[s - 1] is still the old entry here
    tv[s] = b[s] ? tv[s] : (b[s - 1] ? x : tv[s - 1]);
    ti[s] = b[s] ? ti[s] : (b[s - 1] ? v : ti[s - 1]);
  }
  tv[0] = b[0] ? tv[0] : x;
  ti[0] = b[0] ? ti[0] : v;
}

// Sort 32 (value, id) pairs best first (value desc, id asc) with a bitonic
// network: 15 stages of 16 independent compare-exchanges, all in registers.
__device__ __forceinline__ void sort32_best_first(float (&sv)[32], int (&si)[32]) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int l = i ^ j;
        if (l > i) {
          // blocks with (i & k) == 0 put the better pair first, the others last
          const bool sw = (i & k) == 0 ? vi_before(sv[l], si[l], sv[i], si[i]) : vi_before(sv[i], si[i], sv[l], si[l]);
          const float a = sv[i], b = sv[l];
          const int ia = si[i], ib = si[l];
          sv[i] = sw ? b : a;
          sv[l] = sw ? a : b;
          si[i] = sw ? ib : ia;
          si[l] = sw ? ia : ib;
        }
      }
    }
  }
}

// PACKED: the weight comes as pack_w_kernel lays it out, so a stage's
// weight bytes are one contiguous 1-D bulk copy instead of KSUB 2-D boxes of
// 256 rows x 128 bytes (rows 2H bytes apart), which stream markedly slower.
template <int T, bool PACKED, bool FP8, int BN>
__global__ void __launch_bounds__(THREADS, 1)
    lmhead_topk_kernel(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
                       const Params p) {
  using TL = Tile<BN>;
  constexpr int NACC = TL::NACC, STAGES = TL::STAGES, B_SUB = TL::B_SUB, B_BYTES = TL::B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  float *stage_all = reinterpret_cast<float *>(sB + STAGES * B_BYTES);
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES + 4 * STAGE_ROW_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + NACC;
  uint64_t *drain = tempty + NACC;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *never = abort_flag + 1;
  volatile int *epi_left = never + 1;  // epilogue warps still running
  volatile float *bnd_s = reinterpret_cast<volatile float *>(epi_left + 1);  // row bounds [BM]
  volatile int *rb_stop = reinterpret_cast<volatile int *>(bnd_s + BM);     // upkeep may stop

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta0 = (int)blockIdx.x;
  const int ncta = (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *never = 0;
    *epi_left = 4;
    *rb_stop = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_h);
    if (!PACKED) prefetch_tmap(&tmap_w);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 6)
    for (int i = lane; i < BM; i += 32) bnd_s[i] = -INFINITY;
  tc_fence_before();
  block_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  static_assert(!FP8 || PACKED, "the FP8 weight is always packed");
  constexpr int KEL = FP8 ? BK8 : BK;  // K elements per stage
  const int nk = p.H / KEL;
  if (PACKED && warp == 0 && lane == 0 && cta0 < p.n_items) {
    // The weight is no product of the previous grid, so the first stages of
    // this CTA's weight go to L2 while that grid finishes.  A prefetch moves
    // nothing into the CTA: the loads below still read W after the wait.
    int mt, t0, t1, range;
    item_range(p, cta0, mt, t0, t1, range);
    if (t0 < t1)
      for (int kc = 0; kc < nk && kc < STAGES * KSUB; ++kc) bulk_prefetch_l2(packed_at<BN>(p.w_packed, t0, kc, nk), (uint32_t)B_SUB);
  }
  // The prologue above may overlap the previous grid; the CTA reads global
  // memory only after it has finished.
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------- producer
      // a weight tile is read once per M tile: streamed past L2 when there
      // is one M tile, kept at normal priority for the other M tiles' reuse
      const uint64_t pol_w = p.n_mt == 1 ? policy_evict_first() : policy_evict_normal();
      const uint64_t pol_h = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      bool ok = true, stop = false;
      for (int item = cta0; item < p.n_items && ok && !stop; item += ncta) {
        int mt, t0, t1, range;
        item_range(p, item, mt, t0, t1, range);
        for (int t = t0; t < t1 && ok; ++t) {
          if (p.withhold && (t > t0 || item != cta0)) {
            // fault injection: nothing more is loaded, so the MMA warp's next
            // wait runs out and the CTA takes its timeout path
            stop = true;
            break;
          }
          if (p.n_mt > 1) {
            // Every M tile of a range reads the same weight tiles at about
            // the same time, so a weight tile missing in L2 stalls them all.
            // One tile ahead, the CTAs of the range bring the next weight
            // tile into L2 between them: M tile mt takes K atoms mt,
            // mt + n_mt, ...
            int tn = t + 1;
            if (tn >= t1) {
              tn = -1;
              if (item + ncta < p.n_items) {
                int mt2, t2, t3, r2;
                item_range(p, item + ncta, mt2, t2, t3, r2);
                tn = t2 < t3 ? t2 : -1;
              }
            }
            if (tn >= 0)
              for (int kb = mt; kb < nk; kb += p.n_mt) {
                if (PACKED)
                  bulk_prefetch_l2(packed_at<BN>(p.w_packed, tn, kb, nk), (uint32_t)B_SUB);
                else
                  tma_prefetch_2d(&tmap_w, kb * KEL, tn * BN);
              }
          }
          for (int kc = 0; kc < nk; kc += KSUB) {
            const int nsub = nk - kc < KSUB ? nk - kc : KSUB;
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], (uint32_t)(nsub * (A_SUB + B_SUB)));
            if (PACKED)
              bulk_load_1d(sB + stage * B_BYTES, packed_at<BN>(p.w_packed, t, kc, nk), (uint32_t)(nsub * B_SUB), &full[stage],
                           pol_w);
            else
              for (int sub = 0; sub < nsub; ++sub)
                tma_load_2d(sB + stage * B_BYTES + sub * B_SUB, &tmap_w, (kc + sub) * KEL, t * BN, &full[stage],
                            pol_w);
            for (int sub = 0; sub < nsub; ++sub)
              tma_load_2d(sA + stage * A_BYTES + sub * A_SUB, &tmap_h, (kc + sub) * KEL, mt * BM, &full[stage], pol_h);
            issued |= 1u << stage;
            issued_par = phase ? (issued_par | (1u << stage)) : (issued_par & ~(1u << stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        if (!*abort_flag) report(p.status, MFD_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // Every load issued must land before the CTA may exit.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(&full[s], (issued_par >> s) & 1u, never);
    }
    // The block barrier below is an aligned one: the warp's idle lanes wait
    // here for lane 0 so that all 32 reach it together.  Arriving there apart
    // from lane 0 held the warp for 10-27 us at the end of the kernel.
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = FP8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int item = cta0; item < p.n_items && ok; item += ncta) {
        int mt, t0, t1, range;
        item_range(p, item, mt, t0, t1, range);
        for (int t = t0; t < t1 && ok; ++t) {
          if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          for (int kc = 0; kc < nk; kc += KSUB) {
            const int nsub = nk - kc < KSUB ? nk - kc : KSUB;
            if (!mbar_wait(&full[stage], phase, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int sub = 0; sub < nsub; ++sub) {
              const uint64_t ad = smem_desc_sw128(smem_u32(sA + stage * A_BYTES + sub * A_SUB));
              const uint64_t bd = smem_desc_sw128(smem_u32(sB + stage * B_BYTES + sub * B_SUB));
              // four MMAs of 32 bytes of K each (16 bf16 or 32 E4M3 elements):
              // the descriptor's start address advances by 32 bytes (>> 4 = 2)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                if (FP8)
                  tc_mma_f8(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kc | sub | kk) != 0);
                else
                  tc_mma_f16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kc | sub | kk) != 0);
              }
            }
            tc_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(&tfull[acc]);
          if (++acc == NACC) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
      }
      if (!ok) {
        if (!*abort_flag) report(p.status, MFD_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // All MMAs must finish before TMEM is released.
      tc_commit(drain);
      mbar_wait(drain, 0, never);
    }
    __syncwarp();  // as the producer warp: reconverge before the block barrier
  } else if (warp == 6) {
    // ------------------------------------------------------ row bound
    if (p.rb) {
      const unsigned long long G = __shfl_sync(0xffffffffu, ld_relaxed_u64(p.rb_gen), 0) + 1ull;
      const unsigned long long want = mix64(G);
      if (cta0 == 0) {
        for (int i = lane; i < p.R * T; i += 32) p.rb[i] = KEY_NEG_INF;
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          st_release_u64(p.rb_ready, want);
        }
        __syncwarp();
      }
      // loop conditions are taken by lane 0 for the whole warp (the loops
      // hold full-warp shuffles)
      auto running = [&]() { return __shfl_sync(0xffffffffu, (int)(!*abort_flag && !*rb_stop && *epi_left > 0), 0) != 0; };
      bool trusted = false;
      for (int it = 0; it < RB_READY_POLLS && running(); ++it) {
        trusted = __all_sync(0xffffffffu, ld_relaxed_u64(p.rb_ready) == want);
        if (trusted) break;
        __nanosleep(128);
      }
      if (trusted) {
        __threadfence();  // every lane saw the ready word: its later loads see the clear
        // A pass reads the slots as 16-byte words, RB_BATCH of them in flight
        // per lane: word i holds classes 4 (i mod T/4) .. + 3 of row
        // i div (T/4), so the T/4 lanes of one row reduce by shuffles.
        constexpr int QR = T / 4;
        const int nq = p.R * QR;
        const int c4 = 4 * (lane % QR);
        for (int pass = 0; pass < RB_PASSES && running(); ++pass) {
          for (int i0 = 0; i0 < nq && running(); i0 += 32 * RB_BATCH) {
            int4 q[RB_BATCH];
#pragma unroll
            for (int k = 0; k < RB_BATCH; ++k) {
              const int i = i0 + 32 * k + lane;
              q[k] = i < nq ? ld_relaxed_v4(p.rb + 4 * (size_t)i) : make_int4(0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF, 0x7FFFFFFF);
            }
#pragma unroll
            for (int k = 0; k < RB_BATCH; ++k) {
              int m = 0x7FFFFFFF;
              m = c4 + 0 < p.G ? min(m, q[k].x) : m;
              m = c4 + 1 < p.G ? min(m, q[k].y) : m;
              m = c4 + 2 < p.G ? min(m, q[k].z) : m;
              m = c4 + 3 < p.G ? min(m, q[k].w) : m;
#pragma unroll
              for (int o = 1; o < QR; o <<= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
              const int i = i0 + 32 * k + lane;
              if (c4 == 0 && i < nq) {
                const float b = ord_val(m);
                if (b > bnd_s[i / QR]) bnd_s[i / QR] = b;
              }
            }
          }
          __nanosleep(RB_SLEEP_NS);
        }
      }
      __syncwarp();
      // every CTA read gen when it started; the next call takes G + 1
      if (cta0 == 0 && lane == 0) st_relaxed_u64(p.rb_gen, G);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    float *stage = stage_all + (warp - 2) * (STAGE_ROW_BYTES / 4);
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const float s_w = FP8 ? __fdiv_rn(__ldg(p.w_amax), 448.0f) : 1.f;
    for (int item = cta0; item < p.n_items && ok; item += ncta) {
      int mt, t0, t1, range;
      item_range(p, item, mt, t0, t1, range);
      // FP8: z = f_r * acc with f_r = t_r * s_W, one fp32 product
      const int my_row = mt * BM + row_in_tile;
      const float f_r = FP8 ? (my_row < p.R ? __fmul_rn(__ldg(p.row_scale + my_row), s_w) : 0.f) : 1.f;
      float m = -INFINITY, S = 0.f;
      float tv[T];
      int ti[T];
#pragma unroll
      for (int s = 0; s < T; ++s) {
        tv[s] = -INFINITY;
        ti[s] = 0x7FFFFFFF;
      }
      int pub0 = -1, pub1 = -1;  // ids of entries 0 and 1 when last published
      const bool pub_row = p.rb != nullptr && my_row < p.R;
      int *rb_row = pub_row ? p.rb + (size_t)my_row * T : nullptr;
      // publishes the list's first two entries when they have changed and
      // beat the bound in use (a slot already holds at least the bound)
      auto publish = [&]() {
        if (!pub_row) return;
        const float gb = bnd_s[row_in_tile];
        if (ti[0] != pub0 && ti[0] != 0x7FFFFFFF && tv[0] > gb) red_max(rb_row + ti[0] % p.G, ord_key(tv[0]));
        if (ti[1] != pub1 && ti[1] != 0x7FFFFFFF && tv[1] > gb) red_max(rb_row + ti[1] % p.G, ord_key(tv[1]));
        pub0 = ti[0];
        pub1 = ti[1];
      };
      for (int t = t0; t < t1; ++t) {
        // the bound changes little from here on: its upkeep ends now rather
        // than hold up the CTA's exit with a pass in flight
        if (t == t1 - 1 && item + ncta >= p.n_items) *rb_stop = 1;
        if (!mbar_wait(&tfull[acc], acc_phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_addr + (uint32_t)(acc * BN);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float x[32];
          tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), x);
          if (FP8) {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __fmul_rn(x[j], f_r);
          }
          const int v0 = t * BN + c * 32;
          if (v0 + 32 > p.V) {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = (v0 + j < p.V) ? x[j] : -INFINITY;
          }
          float cmax = x[0];
#pragma unroll
          for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, x[j]);
          if (cmax > -INFINITY) {
            if (cmax > m) {
              S *= exp2f((m - cmax) * LOG2E);
              m = cmax;
            }
            const float mb = m * LOG2E;
#pragma unroll
            for (int j = 0; j < 32; ++j) S += exp2f(fmaf(x[j], LOG2E, -mb));
          }
          if (t == t0 && c == 0) {
            // the range's first chunk meets an empty list: its T best, by a
            // sort of the chunk, are the list (columns past V, at -inf, stay
            // (-inf, none) as the empty list's entries)
            float sv[32];
            int si[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {  // as the insert path: only columns above -inf enter
              const bool in = x[j] > -INFINITY;
              sv[j] = in ? x[j] : -INFINITY;
              si[j] = in ? v0 + j : 0x7FFFFFFF;
            }
            sort32_best_first(sv, si);
#pragma unroll
            for (int s = 0; s < T; ++s) {
              tv[s] = sv[s];
              ti[s] = si[s];
            }
            publish();
            continue;
          }
          // Top-T: one bit per column that beats this row's current T-th
          // entry (a later column never ties its way in: its id is larger).
          // Only the set bits are visited, so the warp pays for the largest
          // candidate count among its 32 rows, not for every column.
          // ... and is not below the row bound (x >= bound: x > below(bound))
          const float thr = fmaxf(tv[T - 1], below(bnd_s[row_in_tile]));
          uint32_t cm = 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) cm |= (x[j] > thr ? 1u : 0u) << j;
          if (__any_sync(0xffffffffu, cm != 0)) {
            float *st = stage + lane * STAGE_STRIDE;
#pragma unroll
            for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4 *>(st + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
            while (__any_sync(0xffffffffu, cm != 0)) {
              if (cm) {
                const int j = __ffs(cm) - 1;
                cm &= cm - 1;
                const float xv = st[j];
                if (xv > tv[T - 1]) topk_insert<T>(tv, ti, xv, v0 + j);
              }
            }
            publish();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        if (++acc == NACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) break;
      const int row = mt * BM + row_in_tile;
      if (row < p.R) {
        const size_t base = (size_t)row * p.P + range;
        p.part_ms[base] = make_float2(m, S);
        int2 *c = p.part_cand + base * T;
#pragma unroll
        for (int s = 0; s < T; ++s) c[s] = make_int2(__float_as_int(tv[s]), ti[s]);
      }
    }
    if (!ok) {
      if (!*abort_flag) report(p.status, MFD_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    __syncwarp();
    if (lane == 0) atomicAdd(const_cast<int *>(epi_left), -1);
  }

  block_sync();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Packed weight: for vocabulary tile t (256 rows) and K atom a (64 elements)
// a 32 KB block at ((t * H/64) + a) * 32 KB holding exactly the shared-memory
// image a 2-D box load of those 256 rows x 64 elements writes with the
// 128-byte swizzle: row r at r * 128 bytes, its 16-byte chunk j at position
// j ^ (r % 8).  Rows past V are zero (as the box load's fill).
__global__ void pack_w_kernel(const uint4 *__restrict__ W, int V, int H, uint4 *__restrict__ Wp, size_t n16) {
  const int nk = H / BK;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n16; q += stride) {
    const size_t blk = q / (PK_SUB / 16);
    const int c = (int)(q - blk * (PK_SUB / 16));
    const int t = (int)(blk / nk), a = (int)(blk - (size_t)t * nk);
    const int r = c >> 3, j = (c & 7) ^ (r & 7);
    const int row = t * PK + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < V) v = __ldg(W + (size_t)row * (H / 8) + a * 8 + j);
    Wp[q] = v;
  }
}

// FP8 weight, pass 1: the largest magnitude of W (bf16 [V][H], n16 chunks of
// 8 values) into *amax (zeroed before; non-negative floats order as their
// bit patterns, so an integer max suffices).
__global__ void amax_bf16_kernel(const uint4 *__restrict__ W, size_t n16, unsigned int *amax_bits) {
  float m = 0.f;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n16; q += stride) {
    const uint4 v = __ldg(W + q);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));
}

// E4M3 of x, rounding to nearest even and saturating at +-448.
__device__ __forceinline__ uint32_t to_e4m3(float x) {
  return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// FP8 weight, pass 2: for vocabulary tile t (256 rows) and K slice a (128
// elements) a 32 KB block at ((t * H/128) + a) * 32 KB, row r at r * 128
// bytes, its 16-byte chunk j (elements 16 j .. 16 j + 15 of the slice) at
// chunk position j ^ (r % 8): the shared-memory image of the MMA's 128-byte
// swizzle.  Each value is e4m3(w * (448 / amax)); rows past V are zero.
__global__ void pack_w_fp8_kernel(const uint4 *__restrict__ W, int V, int H, const float *amax, uint4 *__restrict__ Wp,
                                  size_t n16) {
  const int nk = H / BK8;
  const float a = __ldg(amax);
  const float inv = a > 0.f ? __fdiv_rn(448.0f, a) : 0.f;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n16; q += stride) {
    const size_t blk = q / (PK_SUB / 16);
    const int c = (int)(q - blk * (PK_SUB / 16));
    const int t = (int)(blk / nk), s = (int)(blk - (size_t)t * nk);
    const int r = c >> 3, j = (c & 7) ^ (r & 7);
    const int row = t * PK + r;
    uint32_t o[4] = {0u, 0u, 0u, 0u};
    if (row < V) {
      const uint4 *src = W + ((size_t)row * H + (size_t)s * BK8 + (size_t)j * 16) / 8;
      const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t bits = (e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16);
        o[e >> 2] |= to_e4m3(__fmul_rn(__uint_as_float(bits), inv)) << (8 * (e & 3));
      }
    }
    Wp[q] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Online FP8 of the hidden rows: one warp per row of x (bf16 [R][H]):
// amax = max |x|, q = e4m3(x * (448 / amax)), scale[r] = amax / 448 (0 and
// zero bytes for an all-zero row).  q has `rows` rows `stride` bytes apart;
// rows R..rows-1 are written as zero bytes.
__global__ void __launch_bounds__(128) quant_rows_kernel(const uint16_t *__restrict__ x, int R, int H,
                                                        uint8_t *__restrict__ q, float *__restrict__ scale,
                                                        int rows, size_t stride) {
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 4 + warp;
  if (r >= rows) return;
  if (r >= R) {
    for (int k = lane * 8; k < H; k += 256) *reinterpret_cast<uint2 *>(q + (size_t)r * stride + k) = make_uint2(0u, 0u);
    return;
  }
  const uint16_t *xr = x + (size_t)r * H;
  float m = 0.f;
  for (int k = lane * 8; k < H; k += 256) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr + k));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
  m = warp_max(m);
  const float inv = m > 0.f ? __fdiv_rn(448.0f, m) : 0.f;
  for (int k = lane * 8; k < H; k += 256) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr + k));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t bits = (e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16);
      o[e >> 2] |= to_e4m3(__fmul_rn(__uint_as_float(bits), inv)) << (8 * (e & 3));
    }
    *reinterpret_cast<uint2 *>(q + (size_t)r * stride + k) = make_uint2(o[0], o[1]);
  }
  if (lane == 0) scale[r] = __fdiv_rn(m, 448.0f);
}

// Staged hidden rows: row r of x (row16 16-byte words) to row r of dst
// (stride16 words apart), zeros for rows R..rows-1.  One CTA per row.
__global__ void __launch_bounds__(128) stage_rows_kernel(const uint4 *__restrict__ x, int R, int row16,
                                                        uint4 *__restrict__ dst, int stride16) {
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x;
  uint4 *d = dst + (size_t)r * stride16;
  if (r < R) {
    const uint4 *s = x + (size_t)r * row16;
    for (int i = threadIdx.x; i < row16; i += 128) d[i] = __ldg(s + i);
  } else {
    for (int i = threadIdx.x; i < row16; i += 128) d[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int T, bool PACKED, bool FP8, int BN>
cudaError_t launch_t(const LmheadLaunch &L, cudaStream_t stream) {
  static_assert(smem_bytes<BN>() <= 232448, "shared memory budget");
  Params p;
  p.R = L.R;
  p.H = L.H;
  p.V = L.V;
  p.n_mt = (L.R + BM - 1) / BM;
  p.n_vt = (L.V + BN - 1) / BN;
  p.P = L.P;
  p.n_items = p.n_mt * p.P;
  p.part_ms = reinterpret_cast<float2 *>(L.part_ms);
  p.part_cand = reinterpret_cast<int2 *>(L.part_cand);
  p.status = L.status;
  p.w_packed = static_cast<const uint8_t *>(L.w_packed);
  p.row_scale = L.row_scale;
  p.w_amax = L.w_amax;
  p.withhold = L.withhold ? 1 : 0;
  const bool rb = L.rb != nullptr;
  if (rb && !(p.n_mt == 1 && L.G >= 1 && L.G <= T)) return cudaErrorInvalidValue;
  p.rb = rb ? reinterpret_cast<int *>(static_cast<char *>(L.rb) + LMHEAD_BOUND_HEADER) : nullptr;
  p.rb_gen = rb ? static_cast<unsigned long long *>(L.rb) : nullptr;
  p.rb_ready = rb ? static_cast<unsigned long long *>(L.rb) + 1 : nullptr;
  p.G = rb ? L.G : 0;
  cudaError_t e = cudaFuncSetAttribute(lmhead_topk_kernel<T, PACKED, FP8, BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<BN>());
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < L.n_sm ? p.n_items : L.n_sm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem_bytes<BN>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, lmhead_topk_kernel<T, PACKED, FP8, BN>, *L.tmap_h, PACKED ? *L.tmap_h : *L.tmap_w, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int lmhead_tile_rows(int R, int V, int n_sm) { return R > BM || (V + 255) / 256 >= n_sm ? 256 : 128; }
size_t lmhead_bound_bytes(int R, int T) {
  return R <= BM ? LMHEAD_BOUND_HEADER + ((size_t)R * T * 4 + 255) / 256 * 256 : 0;
}
int lmhead_m_rows() { return BM; }
int lmhead_k_chunk() { return BK; }

template <int BN>
cudaError_t launch_bn(const LmheadLaunch &L, cudaStream_t stream) {
  const bool pk = L.w_packed != nullptr;
  if (L.fp8) {
    if (!pk || !L.row_scale || !L.w_amax) return cudaErrorInvalidValue;
    switch (L.T) {
      case 8: return launch_t<8, true, true, BN>(L, stream);
      case 16: return launch_t<16, true, true, BN>(L, stream);
      case 32: return launch_t<32, true, true, BN>(L, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (L.T) {
    case 8: return pk ? launch_t<8, true, false, BN>(L, stream) : launch_t<8, false, false, BN>(L, stream);
    case 16: return pk ? launch_t<16, true, false, BN>(L, stream) : launch_t<16, false, false, BN>(L, stream);
    case 32: return pk ? launch_t<32, true, false, BN>(L, stream) : launch_t<32, false, false, BN>(L, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_lmhead_partials(const LmheadLaunch &L, cudaStream_t stream) {
  if (L.tile_rows != lmhead_tile_rows(L.R, L.V, L.n_sm)) return cudaErrorInvalidValue;
  return L.tile_rows == 128 ? launch_bn<128>(L, stream) : launch_bn<256>(L, stream);
}

size_t lmhead_packed_bytes(int V, int H) { return (size_t)((V + PK - 1) / PK) * PK * (size_t)H * 2; }

size_t lmhead_packed_fp8_bytes(int V, int H) { return (size_t)((V + PK - 1) / PK) * PK * (size_t)H + 256; }

cudaError_t launch_pack_w_fp8(const void *W, int V, int H, void *Wp, cudaStream_t stream) {
  const size_t body = lmhead_packed_fp8_bytes(V, H) - 256;
  unsigned int *amax = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(Wp) + body);
  cudaError_t e = cudaMemsetAsync(amax, 0, 256, stream);
  if (e != cudaSuccess) return e;
  amax_bf16_kernel<<<4 * 152, 256, 0, stream>>>(static_cast<const uint4 *>(W), (size_t)V * H / 8, amax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  pack_w_fp8_kernel<<<4 * 152, 256, 0, stream>>>(static_cast<const uint4 *>(W), V, H,
                                                 reinterpret_cast<const float *>(amax), static_cast<uint4 *>(Wp),
                                                 body / 16);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const void *x, int R, int H, void *q, float *scale, cudaStream_t stream, int rows,
                              size_t stride) {
  if (rows < R) rows = R;
  if (stride == 0) stride = (size_t)H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, quant_rows_kernel, static_cast<const uint16_t *>(x), R, H,
                                     static_cast<uint8_t *>(q), scale, rows, stride);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Every CTA of the LM head reads the same hidden rows at about the same
// time.  Measured on GB300: while those rows span 128 KB of addresses or
// less, wherever they sit, their L2 requests gather on a few L2 slices (the
// busiest slice serves about 5x the mean instead of 2x) and one M tile's
// kernel takes 1.45x as long (172-182 us instead of 120 us at V = 151,936,
// H = 2560, for 1 to 25 rows).  Such rows are copied into scratch first:
// zero rows are appended until they span more than kHiddenSpread bytes, and
// when even a full M tile of rows would not, the rows are spaced further
// apart.  The zero rows change no result: each MMA row is independent and
// rows past R are never written out.
constexpr size_t kHiddenSpread = 144 * 1024;

HiddenStage lmhead_hidden_stage(int R, size_t row_bytes) {
  HiddenStage s{false, R, row_bytes, 0};
  if (R > BM || (size_t)R * row_bytes > kHiddenSpread) return s;
  const size_t need = kHiddenSpread + 1;
  size_t rows = (need + row_bytes - 1) / row_bytes;
  if (rows > (size_t)BM) rows = BM;
  if (rows < (size_t)R) rows = R;
  size_t stride = ((need + rows - 1) / rows + 127) / 128 * 128;
  if (stride < row_bytes) stride = row_bytes;
  s.staged = true;
  s.rows = (int)rows;
  s.stride = stride;
  s.bytes = rows * stride;
  return s;
}

// Staged only when R * row_bytes <= kHiddenSpread: either rows * row_bytes
// <= kHiddenSpread + row_bytes (stride = row_bytes), or rows = BM and stride
// <= (kHiddenSpread + 1) / BM + 128.
size_t lmhead_stage_max_bytes() { return 2 * kHiddenSpread + 1 + (size_t)BM * 128 + 256; }

cudaError_t launch_stage_rows(const void *x, int R, size_t row_bytes, void *dst, const HiddenStage &s,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.rows);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, stage_rows_kernel, static_cast<const uint4 *>(x), R, (int)(row_bytes / 16),
                                     static_cast<uint4 *>(dst), (int)(s.stride / 16));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_pack_w(const void *W, int V, int H, void *Wp, cudaStream_t stream) {
  const size_t n16 = lmhead_packed_bytes(V, H) / 16;
  pack_w_kernel<<<4 * 152, 256, 0, stream>>>(static_cast<const uint4 *>(W), V, H, static_cast<uint4 *>(Wp), n16);
  return cudaGetLastError();
}

}  // namespace mfd
