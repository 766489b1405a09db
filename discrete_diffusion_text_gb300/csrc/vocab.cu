// Fused LM head + posterior statistics + Gumbel-max sampling over the vocabulary.
//
// z = y W^T (rows = canvas positions, columns = vocabulary) is computed on the 5th-generation
// tensor cores tile by tile; no logit ever leaves the SM.  Each CTA is persistent over "units"
// = (128-row tile, contiguous vocabulary chunk):
//   warp 0       TMA: k-blocks of y (128 x 64) and W (256 x 64) into a 4-stage ring;
//   warp 1       one thread issues tcgen05.mma M=128, N=256, K=16 into one of two TMEM
//                accumulators (2 x 256 columns), so the next tile's MMA overlaps this epilogue;
//   warps 2..17  epilogue: four groups of four warps, each group one 64-column quarter of the
//                tile, one thread per row: tempered logits z~ = z / tau, online (max, sum exp)
//                for the log-sum-exp, the top-1 (lowest index on ties), and the exact
//                two-level posterior sample: Gumbel-max over aligned 32-entry chunks scored
//                by their log-sum-exps, then Gumbel-max over the winning chunk's entries.
// Only rows' partial tuples are written; a finalisation kernel merges them in a fixed order and
// applies the Euler step (the chunk scores merge like any Gumbel-max scores).  With many row
// tiles the CTAs run as clusters of two that share each weight k-block by TMA multicast.  With
// separate weight and y rings (single-wave passes) the first weight stages are requested
// before the wait for the previous kernel, which only y depends on.
#include <algorithm>
#include <type_traits>

#include "kernels.cuh"
#include "sm103.cuh"

namespace dg {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;      // TMA warp + MMA warp + epilogue
constexpr int kGroups = kEpiWarps / 4;          // column groups of the tile
constexpr int kGroupCols = kBN / kGroups;       // 64 columns per group
constexpr int kManyRowTiles = 16;  // from this many row tiles: multicast clusters, W kept in L2

struct VocabParams {
  int R, L, d, V;
  int num_mt, nvt, per, S, units;
  float inv_tau;
  uint32_t k0, k1, c3, c3_pick;  // Philox key; counter word 3 (stream tag | step) of the
                                 // chunk Gumbel and of the within-chunk pick
  const int32_t* targets;  // cross-entropy mode: the target token of each row (or NULL)
  uint16_t* sc_p;          // self-conditioning: bf16 exp(z~ - m_ref) [R, V]
  float* sc_m;             // and m_ref per row and 32-column chunk [R, V / 32]
  VocabPart* parts;
  uint32_t* bar;           // sampling: per row, the best chunk score published so far in this
                           // launch (order-preserving key; 0 = none), zeroed before the launch
  uint32_t* status;
  const int* n_active;
  uint64_t wait_ns;  // limit of every on-chip wait
  int skip_loads;    // nonzero: the load warps issue nothing (tests of the timeout path)
  int w_keep;        // nonzero: W tiles use the normal L2 policy (many row tiles share them);
                     // zero: evict-first (each W tile is read once, by a few CTAs at a time)
};

// Shared memory.  Unified ring: kStages stages of (y k-block, W k-block).  Split rings (one
// wave of CTAs, i.e. one canvas): kWStages W k-blocks from the TMA warp and kYStages y
// k-blocks from a second TMA warp, so more of the memory holds the weight stream from DRAM
// (the y tiles come from L2).
template <bool kSplit>
struct VocabLayout {
  static constexpr int kABytes = kBM * kBK * 2;   // 16 KiB: a y k-block
  static constexpr int kBBytes = kBN * kBK * 2;   // 32 KiB: a W k-block
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kWStages = kSplit ? 5 : kStages;
  static constexpr int kYStages = kSplit ? 3 : 0;
  static constexpr int kYOff = kWStages * kBBytes;  // split rings only
  static constexpr int kRingBytes =
      kSplit ? kWStages * kBBytes + kYStages * kABytes : kStages * kStageBytes;
  static constexpr int kScratchOff = kRingBytes;
  static constexpr int kScratchBytes = (kGroups - 1) * kBM * sizeof(VocabPart);
  static constexpr int kBarOff = kScratchOff + kScratchBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
  static constexpr int kThreadsT = kThreads + (kSplit ? 32 : 0);  // + the y TMA warp
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(!kSplit || kYOff + kYStages * kABytes == kRingBytes, "y ring after the W ring");
};

constexpr float kLog2e = 1.4426950408889634f;

// Running per-row state of one epilogue thread.
struct RowState {
  float m;       // running max of z~ (natural units)
  float s;       // sum of exp(z~ - m)
  float t;       // sum of exp(z~ - m) * (z~ - m): entropy = log s - t / s
  float top_z;
  int top_idx;
  float best;    // best chunk score lse_c + g_c
  int best_idx;  // the entry picked inside that chunk
  float best_z;  // and its tempered logit
};

// Three-operand maximum (one instruction for two new elements of a running max).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float open_unit(uint32_t u) {
  // W = (u + 1/2) / 2^32, rounded to fp32 (full relative precision near 0)
  return fmaf(__uint2float_rn(u), 2.3283064365386963e-10f, 1.1641532182693481e-10f);
}

// Order-preserving 32-bit key of a float (a < b iff key(a) < key(b)); key 0 is below every
// float, so a zeroed word means "no score published".
__device__ __forceinline__ uint32_t score_key(float x) {
  const uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float score_from_key(uint32_t k) {
  if (k == 0u) return -INFINITY;
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One 32-column chunk of raw logits z (tempered here: z~ = z * inv_tau, inv_tau > 0); the
// chunk is one of the aligned 32-entry chunks of the two-level posterior sample.
//  - The chunk max is taken on raw z: rounding is monotone, so max(fl(z * c)) = fl(max(z) * c).
//  - exp(z~ - m) is one FFMA into ex2: exp2(z * c log2 e - m log2 e); the sum of the chunk's 32
//    values, sc, is also the chunk's mass relative to the running max.
//  - Sampling (not kCE): the chunk's score is lse_c + g_c = m + log(sc) + g_c with g_c the chunk
//    Gumbel (word c&3 of counter (c>>2, pos, canvas, c3)); a chunk that beats the row's best so
//    far (strictly: an earlier chunk keeps ties) picks its entry at once by Gumbel-max over its
//    32 tempered logits with Gumbels from the pick stream.  The draws cost one Philox call
//    and three logarithms per 32 logits, plus the pick of each chunk that takes the lead.
// kCE (cross-entropy mode): no draws; instead the tempered logit of the row's target token is
// captured (in the best-sample fields, which that mode does not otherwise use).
// kEnt: also accumulate t = sum exp(z~ - m)(z~ - m) for the entropy (one FMA per logit).
// kSC: also store the chunk's exp(z~ - m) as bf16 (32 values, 64 bytes at sc_dst) with the
// reference m it was taken against (at *sc_mdst); NULL pointers for rows past the end.  The
// normalised posterior of the self-conditioning contraction is that value times
// exp(m - lse), applied once lse is known.  Sixteen values go out per store: one 32-byte
// store (a whole sector: the 32 lanes of a warp write 32 different rows) when sc_v8 (the
// buffer is 32-byte aligned), else two 16-byte stores.
// u_gumbel: the chunk's Gumbel draw, word c & 3 of Philox(c >> 2, pos, canvas, c3) for chunk
// c = vbase / 32 (computed by the caller, once for the chunks that share a counter).
// bar / bar_ptr: the row's best chunk score published by any thread of the launch so far (as
// read at the start of this tile) and the row's word to publish to.  A chunk that leads this
// thread's sequence but scores below the bar cannot be the row's sample (some chunk of the row
// scores strictly higher), so its entry is not picked; the leading state records the score
// with no entry, which loses every merge against the published chunk.  Only chunks at or above
// the bar pick (and publish), which keeps the costly pick to about one per warp and unit
// instead of one per lane that leads (the 32 lanes of a warp hold 32 different rows).
template <bool kCE, bool kEnt, bool kSC>
__device__ __forceinline__ void process_chunk(RowState& st, const float (&z)[32], int vbase,
                                              float inv_tau, uint32_t pos, uint32_t canvas,
                                              const PhiloxKeys& keys, uint32_t u_gumbel,
                                              uint32_t c3_pick, int target, uint16_t* sc_dst,
                                              float* sc_mdst, bool sc_v8, float bar,
                                              uint32_t* bar_ptr) {
  float mx[4] = {z[0], z[1], z[2], z[3]};  // four partial maxima: short dependency chains
#pragma unroll
  for (int e = 4; e < 32; e += 2) mx[(e >> 1) & 3] = fmax3(mx[(e >> 1) & 3], z[e], z[e + 1]);
  const float cmr = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
  const float cm = cmr * inv_tau;
  // strictly greater: an equal value seen earlier (a lower index) keeps the top-1; within the
  // chunk the first position holding the maximum wins
  if (cm > st.top_z) {
    uint32_t eq = 0;
#pragma unroll
    for (int e = 0; e < 32; ++e) eq |= (z[e] * inv_tau == cm ? 1u : 0u) << e;
    st.top_z = cm;
    st.top_idx = vbase + __ffs(eq) - 1;
  }
  if (cm > st.m) {
    const float f = ex2_approx((st.m - cm) * kLog2e);
    if (kEnt) st.t = st.s > 0.f ? f * fmaf(st.s, st.m - cm, st.t) : 0.f;  // re-reference
    st.s *= f;
    st.m = cm;
  }
  const float scale = inv_tau * kLog2e;
  const float mlog2 = st.m * kLog2e;
  float ps[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums of exp(z~ - m)
  float pt[4] = {0.f, 0.f, 0.f, 0.f};  // and of exp(z~ - m) (z~ - m) log2(e)
  if (kSC && sc_mdst) *sc_mdst = st.m;
  uint32_t pk[8];
#pragma unroll
  for (int e = 0; e < 32; e += 2) {  // two logits per packed fp32 instruction
    float a0, a1;
    ffma2(a0, a1, z[e], z[e + 1], scale, scale, -mlog2, -mlog2);
    const float p0 = ex2_approx(a0);
    const float p1 = ex2_approx(a1);
    const int q = (e >> 1) & 1;
    fadd2(ps[2 * q], ps[2 * q + 1], ps[2 * q], ps[2 * q + 1], p0, p1);
    if (kEnt) ffma2(pt[2 * q], pt[2 * q + 1], p0, p1, a0, a1, pt[2 * q], pt[2 * q + 1]);
    if (kSC) {  // sixteen values (32 bytes) per store
      pk[(e >> 1) & 7] = pack_bf16x2(p0, p1);
      if ((e & 15) == 14 && sc_dst) {
        uint16_t* d = sc_dst + (e - 14);
        if (sc_v8) {
          st_global_v8(d, pk);
        } else {
          reinterpret_cast<uint4*>(d)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          reinterpret_cast<uint4*>(d)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
  }
  const float sc = (ps[0] + ps[1]) + (ps[2] + ps[3]);
  st.s += sc;
  if (kEnt) st.t += ((pt[0] + pt[1]) + (pt[2] + pt[3])) * 0.6931471805599453f;
  if (kCE) {
    const int e = target - vbase;
    if (e >= 0 && e < 32) {
      float ze = z[0];
#pragma unroll
      for (int k = 1; k < 32; ++k) ze = e == k ? z[k] : ze;  // static indices only
      st.best = 0.f;
      st.best_idx = target;
      st.best_z = ze * inv_tau;
    }
    return;
  }
  const float score = st.m + logf(sc) - logf(-log1pf(-open_unit(u_gumbel)));
  if (score > st.best) {
    st.best = score;
    if (score < bar) {  // another chunk of the row scores higher: no entry needed
      st.best_idx = 0x7FFFFFFF;
      st.best_z = -INFINITY;
      return;
    }
    // The chunk leads the row so far: pick its entry by Gumbel-max over z~_v + g'_v with the
    // pick stream's Gumbels (entry v: word v & 3 of Philox(v >> 2, pos, canvas, c3_pick)),
    // lowest entry on ties.  The draws depend only on v, so the entry is the same whichever
    // thread, and whenever, the chunk is picked.
    float bs = -INFINITY, zj = 0.f;
    int j = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const Words4 w = philox4x32_10((static_cast<uint32_t>(vbase) >> 2) + q, pos, canvas,
                                     c3_pick, keys);
      const uint32_t wq[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float zt = z[4 * q + r] * inv_tau;
        const float se = zt - logf(-log1pf(-open_unit(wq[r])));
        if (se > bs) {
          bs = se;
          j = 4 * q + r;
          zj = zt;
        }
      }
    }
    st.best_idx = vbase + j;
    st.best_z = zj;
    if (bar_ptr) atomicMax(bar_ptr, score_key(score));
  }
}

// kMc (unified ring only): the kernel runs as clusters of two CTAs that take row tiles 2k and
// 2k + 1 of the same vocabulary chunk in lockstep.  Each CTA loads its own y k-block and one
// 128-row half of the W k-block, multicast into both CTAs' stage (tmB then addresses 128-row
// boxes), so the W tile is read from L2 once per two row tiles; a stage is refilled only after
// both CTAs' MMAs have read it (each MMA commit arrives on both CTAs' empty barrier).
template <bool kCE, bool kEnt, bool kSC, bool kSplit, bool kMc>
__global__ void __launch_bounds__(VocabLayout<kSplit>::kThreadsT, 1)
    vocab_posterior_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, VocabParams p) {
  static_assert(!(kMc && kSplit), "multicast with the unified ring only");
  using Lay = VocabLayout<kSplit>;
  constexpr int kWS = Lay::kWStages;
  constexpr int kYS = Lay::kYStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  VocabPart* scratch = reinterpret_cast<VocabPart*>(smem + Lay::kScratchOff);
  // full/empty: the unified stages, or the W stages of the split rings; yfull/yempty: the y
  // stages of the split rings (none otherwise)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* empty = full + kWS;
  uint64_t* yfull = empty + kWS;
  uint64_t* yempty = yfull + kYS;
  uint64_t* tfull = yempty + kYS;  // [2]
  uint64_t* tempty = tfull + 2;    // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = p.d / kBK;
  const uint32_t rank = kMc ? cluster_ctarank() : 0u;

  // W stages started before the wait for the previous kernel (split rings: the W ring holds
  // the weight alone, which no kernel of the stream writes); thread 0 is the W producer
  int pre = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kMc ? 2 : 1);
    }
    for (int s = 0; s < kYS; ++s) {
      mbar_init(&yfull[s], 1);
      mbar_init(&yempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpiThreads);
    }
    *abort_flag = 0;
    fence_barrier_init();
    if (kSplit && blockIdx.x < p.units && !p.skip_loads) {
      tma_prefetch_map(&tmB);
      const uint64_t pol = p.w_keep ? l2_policy_evict_normal() : l2_policy_evict_first();
      const int vt = (static_cast<int>(blockIdx.x) / p.num_mt) * p.per;  // the first unit's
      pre = nkb < kWS ? nkb : kWS;
      for (int kb = 0; kb < pre; ++kb) {
        mbar_arrive_expect_tx(&full[kb], Lay::kBBytes);
        tma_load_2d_hint(smem + kb * Lay::kBBytes, &tmB, &full[kb], kb * kBK, vt * kBN, pol);
      }
    }
  }
  pdl_wait();
  if (p.n_active && *p.n_active == 0) {  // the same for every CTA of the grid
    if (threadIdx.x == 0)  // let the started copies land before the CTA leaves
      for (int s = 0; s < pre; ++s) mbar_wait_drain(&full[s], 0);
    return;
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (kMc) {  // the peer's barriers are initialised before any multicast data or commit arrives
    cluster_arrive();
    cluster_wait();
  }
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&tmA);
      tma_prefetch_map(&tmB);
      // y is read by every vocabulary tile: it stays in L2 (evict-last).  W: see w_keep.
      const uint64_t stream_once = p.w_keep ? l2_policy_evict_normal() : l2_policy_evict_first();
      const uint64_t y_pol = l2_policy_evict_last();
      uint32_t g = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && !p.skip_loads && u < p.units; u += gridDim.x) {
        const int mt = u % p.num_mt;
        const int chunk = u / p.num_mt;
        const int vt0 = chunk * p.per;
        const int vt1 = min(vt0 + p.per, p.nvt);
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          for (int kb = 0; kb < nkb; ++kb, ++g) {
            if (g < static_cast<uint32_t>(pre)) continue;  // started before the wait
            const int s = g % kWS;
            if (!mbar_wait(&empty[s], ((g / kWS) & 1) ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
            if constexpr (kSplit) {  // the W k-block alone (warp 18 loads y)
              uint8_t* sb = smem + s * Lay::kBBytes;
              mbar_arrive_expect_tx(&full[s], Lay::kBBytes);
              tma_load_2d_hint(sb, &tmB, &full[s], kb * kBK, vt * kBN, stream_once);
            } else {
              uint8_t* sa = smem + s * Lay::kStageBytes;
              mbar_arrive_expect_tx(&full[s], Lay::kStageBytes);  // y + both W halves
              tma_load_2d_hint(sa, &tmA, &full[s], kb * kBK, mt * kBM, y_pol);
              if constexpr (kMc)
                tma_load_2d_multicast(sa + Lay::kABytes + rank * (Lay::kBBytes / 2), &tmB,
                                      &full[s], kb * kBK, vt * kBN + rank * (kBN / 2), 0x3,
                                      stream_once);
              else
                tma_load_2d_hint(sa + Lay::kABytes, &tmB, &full[s], kb * kBK, vt * kBN,
                                 stream_once);
            }
          }
        }
      }
      if (!ok) {
        for (uint32_t q = (g > kWS ? g - kWS : 0); q < g; ++q)
          mbar_wait_drain(&full[q % kWS], (q / kWS) & 1);
      } else if (kMc) {
        // every stage this CTA filled has been released by both MMAs, so no commit of the
        // peer is still on its way to this CTA's barriers when it leaves
        for (uint32_t q = (g > kWS ? g - kWS : 0); ok && q < g; ++q)
          ok = mbar_wait(&empty[q % kWS], (q / kWS) & 1, abort_flag, p.wait_ns);
      }
    }
  } else if (kSplit && warp == kThreads / 32) {
    // ------------------------------------------- y producer (split rings only) -----
    if constexpr (kSplit) {
    if (lane == 0) {
      const uint64_t y_pol = l2_policy_evict_last();  // y is read by every vocabulary tile
      uint32_t g = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && !p.skip_loads && u < p.units; u += gridDim.x) {
        const int mt = u % p.num_mt;
        const int chunk = u / p.num_mt;
        const int vt0 = chunk * p.per;
        const int vt1 = min(vt0 + p.per, p.nvt);
        for (int vt = vt0; ok && vt < vt1; ++vt) {
          for (int kb = 0; kb < nkb; ++kb, ++g) {
            const int s = g % kYS;
            if (!mbar_wait(&yempty[s], ((g / kYS) & 1) ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
            uint8_t* sa = smem + Lay::kYOff + s * Lay::kABytes;
            mbar_arrive_expect_tx(&yfull[s], Lay::kABytes);
            tma_load_2d_hint(sa, &tmA, &yfull[s], kb * kBK, mt * kBM, y_pol);
          }
        }
      }
      if (!ok) {
        for (uint32_t q = (g > kYS ? g - kYS : 0); q < g; ++q)
          mbar_wait_drain(&yfull[q % kYS], (q / kYS) & 1);
      }
    }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, kBN, false);
      uint32_t g = 0, j = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        const int chunk = u / p.num_mt;
        const int vt0 = chunk * p.per;
        const int vt1 = min(vt0 + p.per, p.nvt);
        for (int vt = vt0; ok && vt < vt1; ++vt, ++j) {
          const int buf = j & 1;
          if (!mbar_wait(&tempty[buf], ((j >> 1) & 1) ^ 1, abort_flag, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem + buf * kBN;
          for (int kb = 0; kb < nkb; ++kb, ++g) {
            const int s = g % kWS;
            if (!mbar_wait(&full[s], (g / kWS) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
            uint32_t sa, sb;
            int ys = 0;
            if constexpr (kSplit) {
              ys = g % kYS;
              if (!mbar_wait(&yfull[ys], (g / kYS) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
              sa = smem_u32(smem + Lay::kYOff + ys * Lay::kABytes);
              sb = smem_u32(smem + s * Lay::kBBytes);
            } else {
              sa = smem_u32(smem + s * Lay::kStageBytes);
              sb = sa + Lay::kABytes;
            }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_bf16_ss(d_tmem, sdesc_sw128(sa + k * 32, 16, 1024),
                          sdesc_sw128(sb + k * 32, 16, 1024), idesc, (kb | k) != 0);
            if constexpr (kMc)
              mma_commit_multicast(&empty[s], 0x3);  // both CTAs' copy of this stage
            else
              mma_commit(&empty[s]);
            if constexpr (kSplit) mma_commit(&yempty[ys]);
          }
          if (ok) mma_commit(&tfull[buf]);
        }
      }
      if (!ok) {
        mma_commit(&tfull[0]);
        mbar_wait_drain(&tfull[0], 0);
        mbar_wait_drain(&tfull[0], 1);
      }
    }
  } else {
    // --------------------------------------------------------------- epilogue -----
    const int ew = warp - 2;
    const int grp = ew >> 2;                        // which 64-column quarter of the tile
    const int row_in = (warp & 3) * 32 + lane;      // TMEM lane quarter of this warp
    const uint32_t lane_base = tmem_lane_base(warp);
    const PhiloxKeys keys = philox_round_keys(p.k0, p.k1);
    // After an abort the loop structure is kept (every epilogue warp still reaches each
    // unit's named barriers); only the waits, loads and stores are skipped.
    uint32_t j = 0;
    bool ok = true;
    // rows start 2V bytes apart and chunks 64 bytes apart: the base's alignment decides
    const bool sc_v8 = kSC && (reinterpret_cast<uintptr_t>(p.sc_p) & 31) == 0 && (p.V & 15) == 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      const int mt = u % p.num_mt;
      const int chunk = u / p.num_mt;
      const int vt0 = chunk * p.per;
      const int vt1 = min(vt0 + p.per, p.nvt);
      const int row = mt * kBM + row_in;
      const uint32_t canvas = static_cast<uint32_t>(row / p.L);
      const uint32_t pos = static_cast<uint32_t>(row % p.L);
      const int target = kCE && p.targets && row < p.R ? p.targets[row] : -1;
      uint16_t* sc_row = kSC && row < p.R ? p.sc_p + static_cast<int64_t>(row) * p.V : nullptr;
      float* scm_row = kSC && row < p.R ? p.sc_m + static_cast<int64_t>(row) * (p.V / 32)
                                        : nullptr;
      uint32_t* bar_row = !kCE && p.bar && row < p.R ? p.bar + row : nullptr;
      RowState st;
      st.m = -INFINITY;
      st.s = 0.f;
      st.t = 0.f;
      st.top_z = -INFINITY;
      st.top_idx = 0x7FFFFFFF;
      st.best = -INFINITY;
      st.best_idx = 0x7FFFFFFF;
      st.best_z = -INFINITY;
      for (int vt = vt0; vt < vt1; ++vt, ++j) {
        const int buf = j & 1;
        // the row's published best, read before the wait so the load's latency is hidden
        const float bar = bar_row ? score_from_key(ld_relaxed(bar_row)) : -INFINITY;
        if (ok) ok = warp_wait(&tfull[buf], (j >> 1) & 1, abort_flag, p.wait_ns);
        if (!ok) continue;
        tc_fence_after();
        // this thread's 64 columns, 32 at a time (fewer live registers); the accumulator
        // buffer goes back to the MMA warp after the second read, which leaves it a whole tile
        // of slack (the MMA needs this buffer again only after the other one)
        const int col = grp * kGroupCols;
        // this thread's two chunks, 8 vt + 2 grp and the next, share the Gumbel counter
        // (chunk >> 2): one Philox call gives both draws
        static_assert(kGroupCols == 64, "two 32-column chunks per thread and tile");
        uint32_t ug[2] = {0u, 0u};
        if (!kCE) {
          const uint32_t c0 = static_cast<uint32_t>(vt * kBN + col) >> 5;  // even
          const Words4 w = philox4x32_10(c0 >> 2, pos, canvas, p.c3, keys);
          ug[0] = (c0 & 2) ? w.z : w.x;
          ug[1] = (c0 & 2) ? w.w : w.y;
        }
#pragma unroll 1
        for (int c = 0; c < kGroupCols / 32; ++c) {
          float z[32];
          tmem_ld32(tmem + lane_base + buf * kBN + col + c * 32, z);
          if (c == kGroupCols / 32 - 1) {
            tc_fence_before();
            mbar_arrive(&tempty[buf]);
          }
          const int vb = vt * kBN + col + c * 32;
          process_chunk<kCE, kEnt, kSC>(st, z, vb, p.inv_tau, pos, canvas, keys,
                                        c == 0 ? ug[0] : ug[1], p.c3_pick, target,
                                        sc_row ? sc_row + vb : nullptr,
                                        scm_row ? scm_row + (vb >> 5) : nullptr, sc_v8, bar,
                                        bar_row);
        }
      }
      // Merge the column groups of each row through shared memory, in group order.
      VocabPart mine;
      mine.m = st.m;
      mine.s = st.s;
      mine.top_z = st.top_z;
      mine.top_idx = st.top_idx;
      mine.best_score = st.best;
      mine.best_idx = st.best_idx;
      mine.best_z = st.best_z;
      mine.t = st.t;
      named_bar_sync(1, kEpiThreads);
      if (grp > 0) scratch[(grp - 1) * kBM + row_in] = mine;
      named_bar_sync(1, kEpiThreads);
      if (grp == 0) {
#pragma unroll
        for (int q = 1; q < kGroups; ++q) merge_part(mine, scratch[(q - 1) * kBM + row_in]);
        if (ok && row < p.R) p.parts[static_cast<int64_t>(u) * kBM + row_in] = mine;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (kMc) {  // neither CTA leaves while the other may still write to it
    cluster_arrive();
    cluster_wait();
  }
  // every warp of this CTA is done: the next kernel in the stream may be scheduled (not
  // earlier: its waiting CTAs would share the SM with this kernel's epilogue)
  pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, kStatusTimeout);
}

}  // namespace

VocabPlan plan_vocab(int R, int V) {
  VocabPlan pl;
  pl.num_mt = (R + kBM - 1) / kBM;
  pl.nvt = V / kBN;
  const int sms = num_sms();
  // Choose the number of vocabulary chunks S: minimise the tiles of the busiest CTA
  // (waves x tiles per chunk) plus a small cost per chunk for the merge (each row's tuples are
  // merged by one warp, 32 per round); units stay within 16 waves so the tuple workspace stays
  // bounded (at most 16 x SMs x 4 KiB unless there are more row tiles than that).
  int bestS = 1, best_per = pl.nvt;
  double best_cost = -1.0;
  for (int S = 1; S <= pl.nvt; ++S) {
    const int per = (pl.nvt + S - 1) / S;
    const int S2 = (pl.nvt + per - 1) / per;
    if (S2 != S) continue;
    const int64_t units = static_cast<int64_t>(pl.num_mt) * S2;
    if (S2 > 1 && units > 16ll * sms) break;
    const int64_t waves = (units + sms - 1) / sms;
    const double cost = static_cast<double>(waves * per) + S2 / 8.0;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      bestS = S2;
      best_per = per;
    }
  }
  pl.S = bestS;
  pl.per = best_per;
  pl.units = pl.num_mt * pl.S;
  pl.grid = pl.units < sms ? pl.units : sms;
  // the partial tuples, then one 32-bit bar word per row (16-byte aligned)
  pl.part_bytes = static_cast<size_t>(pl.units) * kBM * sizeof(VocabPart) +
                  ((static_cast<size_t>(R) * 4 + 15) & ~static_cast<size_t>(15));
  return pl;
}

uint32_t* vocab_bars(VocabPart* parts, int R, int V) {
  return reinterpret_cast<uint32_t*>(parts + static_cast<size_t>(plan_vocab(R, V).units) * kBM);
}

cudaError_t launch_vocab_pass(const uint16_t* y, const uint16_t* W, int R, int L, int d, int V,
                              float inv_tau, uint64_t seed, int step, VocabPart* parts,
                              uint32_t* status, const int* n_active, cudaStream_t st,
                              const int32_t* targets, bool entropy, uint16_t* sc_p,
                              float* sc_m, bool ce_only, bool bars_clear) {
  const VocabPlan pl = plan_vocab(R, V);
  CUtensorMap ta, tb;
  const uint64_t dA[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(R)};
  const uint64_t sA[1] = {static_cast<uint64_t>(d) * 2};
  const uint32_t bA[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kBM)};
  const uint64_t dB[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(V)};
  const uint32_t bB[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kBN)};
  if (!make_tmap_bf16(&ta, y, 2, dA, sA, bA)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, W, 2, dB, sA, bB)) return cudaErrorInvalidValue;

  VocabParams p;
  p.R = R;
  p.L = L;
  p.d = d;
  p.V = V;
  p.num_mt = pl.num_mt;
  p.nvt = pl.nvt;
  p.per = pl.per;
  p.S = pl.S;
  p.units = pl.units;
  p.inv_tau = inv_tau;
  p.k0 = static_cast<uint32_t>(seed);
  p.k1 = static_cast<uint32_t>(seed >> 32);
  p.c3 = kStreamGumbel | (static_cast<uint32_t>(step) & 0xFFFFFFu);
  p.c3_pick = kStreamPick | (static_cast<uint32_t>(step) & 0xFFFFFFu);
  p.targets = targets;
  p.sc_p = sc_p;
  p.sc_m = sc_m;
  p.parts = parts;
  p.bar = nullptr;
  p.status = status;
  p.n_active = n_active;
  p.wait_ns = wait_limit_ns();
  p.skip_loads = wait_test_skip_loads() ? 1 : 0;
  // With many row tiles each W tile is read by every row tile's CTA over a window in which
  // the L2 also holds y: evict-first W lines left the L2 before most readers came (64
  // canvases: 12.4 GB of DRAM reads per launch for 1.14 GB of data); the normal policy with y
  // kept (evict-last) reads 2.7 GB and runs 9.5 % faster (5.2 % at 16 canvases, 7.0 % at 32).
  // With few row tiles a W tile is read once, by a few CTAs together: evict-first keeps the
  // stream from displacing the other kernels' weights and caches.
  p.w_keep = pl.num_mt >= kManyRowTiles ? 1 : 0;

  static int configured_device = -1;
  static int max_pairs = 0;  // clusters of two multicast CTAs that can be resident at once
  const int dev = device_id();
  if (configured_device != dev) {
    cudaError_t e = cudaSuccess;
    for (auto fn : {vocab_posterior_kernel<false, false, false, false, false>,
                    vocab_posterior_kernel<false, true, false, false, false>,
                    vocab_posterior_kernel<true, false, false, false, false>,
                    vocab_posterior_kernel<false, false, true, false, false>,
                    vocab_posterior_kernel<false, true, true, false, false>,
                    vocab_posterior_kernel<true, false, true, false, false>,
                    vocab_posterior_kernel<false, false, false, false, true>,
                    vocab_posterior_kernel<false, true, false, false, true>,
                    vocab_posterior_kernel<true, false, false, false, true>,
                    vocab_posterior_kernel<false, false, true, false, true>,
                    vocab_posterior_kernel<false, true, true, false, true>,
                    vocab_posterior_kernel<true, false, true, false, true>})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 VocabLayout<false>::kSmemBytes);
    for (auto fn : {vocab_posterior_kernel<false, false, false, true, false>,
                    vocab_posterior_kernel<false, true, false, true, false>,
                    vocab_posterior_kernel<true, false, false, true, false>,
                    vocab_posterior_kernel<false, false, true, true, false>,
                    vocab_posterior_kernel<false, true, true, true, false>,
                    vocab_posterior_kernel<true, false, true, true, false>})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 VocabLayout<true>::kSmemBytes);
    if (e != cudaSuccess) return e;
    {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(2 * (num_sms() / 2));
      cfg.blockDim = dim3(VocabLayout<false>::kThreadsT);
      cfg.dynamicSmemBytes = VocabLayout<false>::kSmemBytes;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, vocab_posterior_kernel<false, false, false, false, true>,
                                         &cfg) != cudaSuccess)
        n = 0;
      cudaGetLastError();  // an unsupported query leaves no sticky error; the pass runs unpaired
      max_pairs = n;
    }
    configured_device = dev;
  }
  // cross-entropy mode (targets, or the self-conditioning pass alone: no sampling), or
  // sampling with or without the entropy accumulator; each with or without the
  // self-conditioning store.  Split rings when the pass is a single wave (one unit per CTA:
  // one canvas), except with the entropy accumulator: measured at one canvas, cross-entropy
  // 0.1998 -> 0.1922 ms, the self-conditioning store 0.269 -> 0.256 ms, sampling 0.2112 ->
  // 0.2098 ms (once its epilogue became light), but the entropy accumulator's loop 0.7 %
  // slower (the extra TMA warp takes issue slots from the heavier epilogue); with several
  // waves the unified ring is faster (-7 % at 16 canvases).
  const bool sc = sc_p != nullptr;
  const bool ce = targets != nullptr || ce_only;
  if (!ce) {  // every sampling launch starts with no bar published
    p.bar = vocab_bars(parts, R, V);
    if (!bars_clear) {
      const cudaError_t em = cudaMemsetAsync(p.bar, 0, static_cast<size_t>(R) * 4, st);
      if (em != cudaSuccess) return em;
    }
  }
  // Multicast clusters from 16 row tiles (eight canvases) up, where the pass runs under the
  // power cap: halving the W reads from L2 lowers its power, and the clock rises more than the
  // clusters' lockstep costs (measured: 64 canvases +3.7 % throughput at 1,725 against 1,627 MHz,
  // 16 canvases +3.0 %); at one canvas (not power-bound) it was 0.7 % slower.
  const bool split = pl.units <= pl.grid && (ce || sc || !entropy);
  const bool mc = !split && max_pairs > 0 && pl.num_mt % 2 == 0 && pl.num_mt >= kManyRowTiles;
  timer_begin(0, st);
  cudaError_t e;
  auto pick = [&](auto split_tag, auto mc_tag) {
    constexpr bool kS = decltype(split_tag)::value;
    constexpr bool kM = decltype(mc_tag)::value;
    return ce ? (sc ? vocab_posterior_kernel<true, false, true, kS, kM>
                    : vocab_posterior_kernel<true, false, false, kS, kM>)
              : entropy ? (sc ? vocab_posterior_kernel<false, true, true, kS, kM>
                              : vocab_posterior_kernel<false, true, false, kS, kM>)
                        : (sc ? vocab_posterior_kernel<false, false, true, kS, kM>
                              : vocab_posterior_kernel<false, false, false, kS, kM>);
  };
  if (mc) {
    // W in 128-row boxes (each CTA of a cluster loads one half of a 256-row k-block)
    const uint32_t bH[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kBN / 2)};
    CUtensorMap th;
    if (!make_tmap_bf16(&th, W, 2, dB, sA, bH)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(std::min(pl.units, 2 * max_pairs));
    cfg.blockDim = dim3(VocabLayout<false>::kThreadsT);
    cfg.dynamicSmemBytes = VocabLayout<false>::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 2;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, pick(std::false_type{}, std::true_type{}), ta, th, p);
  } else if (split) {
    e = launch_dependent(pick(std::true_type{}, std::false_type{}), dim3(pl.grid),
                         dim3(VocabLayout<true>::kThreadsT), VocabLayout<true>::kSmemBytes, st,
                         ta, tb, p);
  } else {
    e = launch_dependent(pick(std::false_type{}, std::false_type{}), dim3(pl.grid),
                         dim3(VocabLayout<false>::kThreadsT), VocabLayout<false>::kSmemBytes, st,
                         ta, tb, p);
  }
  timer_end(0, st);
  return e;
}

}  // namespace dg
