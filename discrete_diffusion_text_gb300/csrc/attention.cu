// Canvas attention on the 5th-generation tensor cores.
//
// One CTA serves two "slots" that read the same keys and values: the two query heads of a GQA
// group for one 128-query tile (or, when a group has one query head, two query tiles of that
// head).  Keys and values come in tiles of 64 keys, staged once for both slots through a deep
// ring.
//   warp 0       TMA: Q of both slots once, then K_0, V_0, K_1, V_1, ... (ring of 10 tiles at
//                hd=128);
//   warps 1, 2   one thread each issues S_s(j) = Q_s K_j^T (M=128, N=64) of slot s = warp - 1
//                into one of the slot's two TMEM score buffers;
//   warp 3       one thread issues O_s += P_s(j) V_j for both slots, with P_s(j) read straight
//                from TMEM (A operand in tensor memory, V as an MN-major operand);
//   warps 4..7   softmax of slot 0, warps 8..11 softmax of slot 1: one thread per query row
//                reads its 64 scores from TMEM, masks, exponentiates against a running
//                reference max and writes P as bf16 pairs over the first 32 columns of the
//                same score buffer.
// TMEM: S of (slot s, buffer b) at [(2s + b) * 64, +64), O of slot s at [256 + 128 s, +128).
// With two score buffers per slot, S_s(j+2) is computed while the softmax of tile j+1 runs, so
// a slot's softmax warps go from tile to tile without waiting for its P.V or score MMAs; the
// only ordering is that S_s(j+2) waits for O_s += P_s(j) V_j, which reads the buffer's P.
// An issuing thread is held in each tcgen05.mma for about the MMA's own duration, so a single
// issuer leaves the pipe idle during every barrier wait and commit; three issuers with about
// equal shares (scores of slot 0, scores of slot 1, both P.V) cover each other's waits.
// The reference max is only raised when a row's max grows by more than 2^8 (log2 units):
// p <= 256 is exact enough in fp32 accumulation and bf16, and O and l use the same reference,
// so the result is unchanged while O (in TMEM) is rescaled rarely.
// With several key splits, each writes unnormalised fp32 partials (O, m, l) and a merge kernel
// combines them with the log-sum-exp rule.
// A second kernel (canvas_attn1_kernel, below) takes one query head per CTA with 128-key
// tiles; plan_attention picks it where the K/V work is short (see there).  Its 2..8 key
// splits of a unit run as one thread-block cluster and merge there (attn1_cluster_merge).
// Both kernels request their first prefix K/V tiles before waiting for the previous kernel.
#include <array>
#include <mutex>
#include <vector>

#include "kernels.cuh"
#include "sm103.cuh"

namespace dg {
namespace {

constexpr int kQTile = 128;  // queries per slot
constexpr int kKTile = 64;   // keys per tile
constexpr float kRescaleLog2 = 8.f;
constexpr float kRaiseSum = 256.f;  // 2^kRescaleLog2: a row sum above it may hide a p above it
constexpr int kRingMax = 16;
constexpr int kThreads = 384;      // warpgroup 0: TMA + MMA warps; warpgroups 1, 2: softmax
constexpr int kRegsControl = 104;  // registers per thread of warpgroup 0 after the split
constexpr int kRegsSoftmax = 192;  // registers per thread of the softmax warpgroups
// 128 x 104 + 256 x 192 = 62,464 registers: needs a launch allocation of >= 163 per thread.

struct AttnParams {
  int B, L, P, H, Hkv, hd, window;
  float scale_log2;  // scale * log2(e)
  int n_pre_tiles, n_can_tiles, n_qtiles, splits;
  int units;         // CTAs per split
  uint16_t* out;
  float* lse;
  float* part_o;   // [splits][B*H*L][hd]
  float* part_ml;  // [splits][B*H*L][2]
  uint32_t* status;
  const int* n_active;
  uint64_t wait_ns;  // limit of every on-chip wait
  int cluster_merge;  // one-slot kernel: the key splits of a unit form a cluster and merge there
};

template <int HD>
struct AttnLayout {
  static constexpr int kRing = HD == 128 ? 10 : 16;  // K/V ring slots (K_j and V_j alternate)
  static constexpr int kQChunk = kQTile * 128;        // [128 rows][64 bf16] swizzled chunk
  static constexpr int kKVChunk = kKTile * 128;       // [64 keys][64 bf16]
  static constexpr int kQBytes = (HD / 64) * kQChunk;    // one slot's Q tile
  static constexpr int kKVBytes = (HD / 64) * kKVChunk;  // one K or V tile
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + 2 * kQBytes;
  static constexpr int kBarOff = kKVOff + kRing * kKVBytes;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static_assert(kRing <= kRingMax, "barrier array");
};

// The two slots of a CTA: (head, query tile) each, sharing one KV head and key range.
struct Slots {
  int b, g, h0, h1, qt0, qt1;
  bool valid1;
};

__device__ __forceinline__ Slots cta_slots(int u, const AttnParams& p) {
  Slots s;
  const int r = p.H / p.Hkv;
  if ((r & 1) == 0) {  // two query heads of one group, same query tile
    const int pairs = p.H / 2;
    const int qt = u % p.n_qtiles;
    const int pr = (u / p.n_qtiles) % pairs;
    s.b = u / (p.n_qtiles * pairs);
    s.h0 = 2 * pr;
    s.h1 = 2 * pr + 1;
    s.qt0 = s.qt1 = qt;
    s.valid1 = true;
  } else {  // one head, two consecutive query tiles
    const int nqp = (p.n_qtiles + 1) / 2;
    const int qp = u % nqp;
    const int h = (u / nqp) % p.H;
    s.b = u / (nqp * p.H);
    s.h0 = s.h1 = h;
    s.qt0 = 2 * qp;
    s.qt1 = 2 * qp + 1;
    s.valid1 = s.qt1 < p.n_qtiles;
  }
  s.g = (s.h0 * p.Hkv) / p.H;
  return s;
}

// Three-operand maximum (one instruction for two new elements of a running max).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    canvas_attn_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmKp,
                       const __grid_constant__ CUtensorMap tmVp,
                       const __grid_constant__ CUtensorMap tmKc,
                       const __grid_constant__ CUtensorMap tmVc, AttnParams p) {
  using Lay = AttnLayout<HD>;
  constexpr int kRing = Lay::kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                  // [kRing]
  uint64_t* kv_empty = bars + 1 + kRingMax;      // [kRing]
  uint64_t* s_full = bars + 1 + 2 * kRingMax;    // [slot * 2 + buffer]
  uint64_t* p_full = s_full + 4;                 // [slot * 2 + buffer]
  uint64_t* pv_done = s_full + 8;                // [slot * 2 + buffer]
  uint64_t* drain = s_full + 12;                 // [issuer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Slots sl = cta_slots(blockIdx.x, p);
  const int split = blockIdx.y;
  const int nslots = sl.valid1 ? 2 : 1;

  // Key tiles: prefix tiles from the first one any query of either slot can see (slot 0 holds
  // the lower query tile), then the canvas tiles; this split takes a contiguous share.
  int t_lo = 0;
  if (p.window > 0) {
    const int kmin = p.P + sl.qt0 * kQTile - p.window + 1;
    t_lo = kmin > 0 ? kmin / kKTile : 0;
    if (t_lo > p.n_pre_tiles) t_lo = p.n_pre_tiles;
  }
  const int n_pre = p.n_pre_tiles - t_lo;
  const int nt_all = n_pre + p.n_can_tiles;
  // Even partition: with splits <= nt_all every split gets at least one tile.  (CTAs that
  // find no work and exit at once were measured to delay the whole launch by ~12 us.)
  const int t_begin = static_cast<int>(static_cast<int64_t>(split) * nt_all / p.splits);
  const int t_end = static_cast<int>(static_cast<int64_t>(split + 1) * nt_all / p.splits);
  const int nt = t_end > t_begin ? t_end - t_begin : 0;

  // softmax role of this thread (warps 4..11)
  const int slot = warp >= 8 ? 1 : 0;
  const int row_in = (warp & 3) * 32 + lane;  // TMEM lane quarter of this warp
  const int qi = (slot ? sl.qt1 : sl.qt0) * kQTile + row_in;
  const int hq = slot ? sl.h1 : sl.h0;
  const int64_t out_row = (static_cast<int64_t>(sl.b) * p.H + hq) * p.L + qi;  // (b, h, i)
  const int64_t part_rows = static_cast<int64_t>(p.B) * p.H * p.L;
  auto q_buf = [&](int s) { return smem + Lay::kQOff + s * Lay::kQBytes; };
  auto kv_buf = [&](int i) { return smem + Lay::kKVOff + (i % kRing) * Lay::kKVBytes; };

  // Before the wait for the previous kernel: the barriers, and the prefix K/V tiles of the
  // first ring slots (the cache, which the kernels of a denoising step do not write); thread
  // 0 is the producer.
  int n_early = 0;
  if (threadIdx.x == 0 && nt > 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], (s & 1) ? 1 : nslots);  // K slots: each score thread; V slots: the P.V thread
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4);  // one arrival per softmax warp
      mbar_init(&pv_done[s], 1);
    }
    for (int s = 0; s < 3; ++s) mbar_init(&drain[s], 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmKp);
    tma_prefetch_map(&tmVp);
    for (int i = 0; i < 2 * nt && i < kRing; ++i) {
      const int t = t_begin + (i >> 1);
      if (t >= n_pre) break;
      const CUtensorMap* m = (i & 1) ? &tmVp : &tmKp;
      mbar_arrive_expect_tx(&kv_full[i], Lay::kKVBytes);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_4d(kv_buf(i) + c * Lay::kKVChunk, m, &kv_full[i], c * 64, sl.g,
                    (t_lo + t) * kKTile, sl.b);
      ++n_early;
    }
  }
  pdl_wait();
  if (p.n_active && *p.n_active == 0) {  // the same for every CTA of the grid
    if (threadIdx.x == 0)  // let the started copies land before the CTA leaves
      for (int i = 0; i < n_early; ++i) mbar_wait_drain(&kv_full[i], 0);
    return;
  }
  pdl_trigger();  // the next kernel's CTAs may start their own prologue on idle SMs

  if (nt == 0) {  // nothing to do: empty partials (only when splits > 1)
    if (warp >= 4 && (slot == 0 || sl.valid1) && qi < p.L) {
      float* ml = p.part_ml + (split * part_rows + out_row) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
      float* po = p.part_o + (split * part_rows + out_row) * HD;
      for (int c = 0; c < HD; ++c) po[c] = 0.f;
    }
    return;
  }

  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto tm_s = [&](int s, int b) { return tmem + (2 * s + b) * kKTile; };
  auto tm_o = [&](int s) { return tmem + 256 + s * 128; };

  // Register split (each warpgroup changes its budget in its own branch): the control
  // warpgroup (TMA and MMA warps) needs few registers, each softmax thread holds a score row.
  // 128 x kRegsControl + 256 x kRegsSoftmax fits the launch allocation (checked on the host
  // before the first launch).
  if (warp < 4) {
    regs_decrease<kRegsControl>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------------ producer -----
      tma_prefetch_map(&tmQ);
      mbar_arrive_expect_tx(q_full, nslots * Lay::kQBytes);
      for (int s = 0; s < nslots; ++s)
        for (int c = 0; c < HD / 64; ++c)
          tma_load_4d(q_buf(s) + c * Lay::kQChunk, &tmQ, q_full, c * 64, s ? sl.h1 : sl.h0,
                      (s ? sl.qt1 : sl.qt0) * kQTile, sl.b);
      // load index i: K_j for i = 2j, V_j for i = 2j + 1, into ring slot i % kRing
      int issued = 0;
      for (int i = 0; i < 2 * nt; ++i) {
        if (i < n_early) {  // requested before the wait
          ++issued;
          continue;
        }
        const int rs = i % kRing;
        if (!mbar_wait(&kv_empty[rs], ((i / kRing) & 1) ^ 1, abort_flag, p.wait_ns)) break;
        const int t = t_begin + (i >> 1);
        const bool pre = t < n_pre;
        const int kb = pre ? (t_lo + t) * kKTile : (t - n_pre) * kKTile;
        const CUtensorMap* m = (i & 1) ? (pre ? &tmVp : &tmVc) : (pre ? &tmKp : &tmKc);
        uint8_t* dst = kv_buf(i);
        mbar_arrive_expect_tx(&kv_full[rs], Lay::kKVBytes);
        for (int c = 0; c < HD / 64; ++c)
          tma_load_4d(dst + c * Lay::kKVChunk, m, &kv_full[rs], c * 64, sl.g, kb, sl.b);
        ++issued;
      }
      if (*abort_flag) {
        mbar_wait_drain(q_full, 0);
        for (int i = (issued > kRing ? issued - kRing : 0); i < issued; ++i)
          mbar_wait_drain(&kv_full[i % kRing], (i / kRing) & 1);
      }
    } else if (lane == 0 && (warp == 3 || warp - 1 < nslots)) {
      // ------------------------------------------------------------------ MMA issuers -----
      // warp 1 + s (s < 2): the score MMAs of slot s; warp 3: the P.V MMAs of both slots
      constexpr uint32_t idesc_s = idesc_bf16(128, kKTile, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, HD, true);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.wait_ns);
      auto wait_kv = [&](int i) {
        return mbar_wait(&kv_full[i % kRing], (i / kRing) & 1, abort_flag, p.wait_ns);
      };
      if (warp < 3) {
        const int s = warp - 1;
        const uint32_t qa = smem_u32(q_buf(s));
        for (int j = 0; ok && j < nt; ++j) {
          if (!(ok = wait_kv(2 * j))) break;
          // S_s(j) overwrites the buffer whose first columns hold P_s(j-2)
          if (j >= 2 && !(ok = mbar_wait(&pv_done[2 * s + (j & 1)], ((j - 2) >> 1) & 1, abort_flag, p.wait_ns)))
            break;
          tc_fence_after();
          const uint32_t ka = smem_u32(kv_buf(2 * j));
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            mma_bf16_ss(tm_s(s, j & 1),
                        sdesc_sw128(qa + (kk >> 2) * Lay::kQChunk + (kk & 3) * 32, 16, 1024),
                        sdesc_sw128(ka + (kk >> 2) * Lay::kKVChunk + (kk & 3) * 32, 16, 1024),
                        idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[2 * s + (j & 1)]);
          mma_commit(&kv_empty[(2 * j) % kRing]);  // this slot's read of K_j
        }
      } else {
        for (int j = 0; ok && j < nt; ++j) {
          if (!(ok = wait_kv(2 * j + 1))) break;
          const uint32_t va = smem_u32(kv_buf(2 * j + 1));
          for (int s = 0; ok && s < nslots; ++s) {
            if (!(ok = mbar_wait(&p_full[2 * s + (j & 1)], (j >> 1) & 1, abort_flag, p.wait_ns))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kKTile / 16; ++kk) {
              mma_bf16_ts(tm_o(s), tm_s(s, j & 1) + kk * 8,
                          sdesc_sw128(va + kk * 2048, Lay::kKVChunk, 1024), idesc_o,
                          (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&pv_done[2 * s + (j & 1)]);
          }
          if (!ok) break;
          mma_commit(&kv_empty[(2 * j + 1) % kRing]);  // V_j read by both slots
        }
      }
      if (*abort_flag) {  // make sure no MMA is still writing TMEM before it is released
        mma_commit(&drain[warp - 1]);
        mbar_wait_drain(&drain[warp - 1], 0);
      }
    }
  } else {
    regs_increase<kRegsSoftmax>();
    if (slot == 0 || sl.valid1) {
      // ------------------------------------------------------------- softmax warps -----
      const uint32_t lane_base = tmem_lane_base(warp);
      float m_ref = -INFINITY;
      float l = 0.f;
      bool ok = true;
      const int kmin = p.window > 0 ? p.P + qi - p.window + 1 : 0;
      const float c = p.scale_log2;
      for (int j = 0; j < nt; ++j) {
        const int b = j & 1;
        if (!warp_wait(&s_full[2 * slot + b], (j >> 1) & 1, abort_flag, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        const int t = t_begin + j;
        const bool pre = t < n_pre;
        const int kb = pre ? (t_lo + t) * kKTile : (t - n_pre) * kKTile;
        const int klim = pre ? p.P : p.L;
        const int klo = pre ? kmin : 0;
        float sv[kKTile];
        tmem_ld64(tm_s(slot, b) + lane_base, sv);  // the score row in one TMEM round trip
        // raw scores; the scale (> 0) is folded into the exponent, so the max is taken on raw
        // values (rounding is monotone)
        if (!(kb >= klo && kb + kKTile <= klim)) {
#pragma unroll
          for (int e = 0; e < kKTile; ++e) {
            const int key = kb + e;
            if (!(key < klim && key >= klo)) sv[e] = -INFINITY;
          }
        }
        // P = exp2(s * c - m_ref).  With a reference already set the tile is exponentiated
        // against it at once (no row-max reduction on the common path): the reference is raised
        // only when some p would exceed 2^8, which the row sum of p then also exceeds; such a
        // rare tile is redone against its own max.  The first tile of a row (no reference yet)
        // takes the max first.
        float ps[8];
        uint32_t pk[kKTile / 2];
        float f = 1.f;
        bool need = false;
        auto exp_tile = [&](float m_use) {  // two scores per packed fp32 instruction
#pragma unroll
          for (int q = 0; q < 8; ++q) ps[q] = 0.f;
#pragma unroll
          for (int e = 0; e < kKTile; e += 2) {
            float xa, xb;
            ffma2(xa, xb, sv[e], sv[e + 1], c, c, -m_use, -m_use);
            const float a = ex2_approx(xa);
            const float bb = ex2_approx(xb);
            const int q = (e >> 1) & 3;
            fadd2(ps[2 * q], ps[2 * q + 1], ps[2 * q], ps[2 * q + 1], a, bb);
            pk[e >> 1] = pack_bf16x2(a, bb);
          }
          return ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        };
        auto tile_max = [&]() {
          float mx[8];  // eight partial maxima: short dependency chains
#pragma unroll
          for (int q = 0; q < 8; ++q) mx[q] = sv[q];
#pragma unroll
          for (int e = 8; e < kKTile; e += 2)
            mx[(e >> 1) & 7] = fmax3(mx[(e >> 1) & 7], sv[e], sv[e + 1]);
          return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        };
        float rs;
        if (m_ref == -INFINITY) {
          m_ref = tile_max() * c;  // stays -inf for a fully masked tile
          rs = exp_tile(m_ref == -INFINITY ? 0.f : m_ref);
        } else {
          rs = exp_tile(m_ref);
          if (rs > kRaiseSum) {  // some p may exceed 2^8: raise the reference to this tile's max
            const float m_new = fmaxf(m_ref, tile_max() * c);
            if (m_new > m_ref) {
              need = true;
              f = ex2_approx(m_ref - m_new);
              m_ref = m_new;
              rs = exp_tile(m_ref);
            }
          }
        }
        tmem_st32(tm_s(slot, b) + lane_base, pk);
        l = l * f + rs;
        if (__any_sync(0xFFFFFFFFu, need)) {  // O *= f once PV of tile j - 1 has completed
          if (!warp_wait(&pv_done[2 * slot + ((j - 1) & 1)], ((j - 1) >> 1) & 1, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < HD / 32; ++cc) {
            float o[32];
            tmem_ld32(tm_o(slot) + lane_base + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tmem_st32(tm_o(slot) + lane_base + cc * 32, o);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[2 * slot + b]);
      }
      if (ok)
        ok = warp_wait(&pv_done[2 * slot + ((nt - 1) & 1)], ((nt - 1) >> 1) & 1, abort_flag, p.wait_ns);
      tc_fence_after();
      const bool write = ok && qi < p.L;
      if (p.splits == 1) {
        const float inv_l = 1.f / l;
        uint16_t* dst = p.out + ((static_cast<int64_t>(sl.b) * p.L + qi) * p.H + hq) * HD;
#pragma unroll 1
        for (int cc = 0; cc < HD / 32; ++cc) {
          float o[32];
          tmem_ld32(tm_o(slot) + lane_base + cc * 32, o);
          if (write) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              d4[q] = make_uint4(pack_bf16x2(o[q * 8 + 0] * inv_l, o[q * 8 + 1] * inv_l),
                                 pack_bf16x2(o[q * 8 + 2] * inv_l, o[q * 8 + 3] * inv_l),
                                 pack_bf16x2(o[q * 8 + 4] * inv_l, o[q * 8 + 5] * inv_l),
                                 pack_bf16x2(o[q * 8 + 6] * inv_l, o[q * 8 + 7] * inv_l));
          }
        }
        if (write && p.lse) p.lse[out_row] = (m_ref + __log2f(l)) * 0.6931471805599453f;
      } else {
        const int64_t prow = split * part_rows + out_row;
        float* po = p.part_o + prow * HD;
#pragma unroll 1
        for (int cc = 0; cc < HD / 32; ++cc) {
          float o[32];
          tmem_ld32(tm_o(slot) + lane_base + cc * 32, o);
          if (write) {
            float4* d4 = reinterpret_cast<float4*>(po + cc * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              d4[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
        }
        if (write) {
          p.part_ml[prow * 2] = m_ref;
          p.part_ml[prow * 2 + 1] = l;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, kStatusTimeout);
}

// ------------------------------------------------------------ one query head per CTA -----
// For long prefixes: one CTA serves one (canvas, query head, 128-query tile) over one key
// split, in key tiles of 128.  Every MMA is 128 wide (S = Q K^T: M128 N128; O += P V: M128,
// N = hd, K = 128 keys), where the two-slot kernel's 64-key score MMAs run at three quarters
// of the pipe's rate.  TMEM: two 128-column score buffers and O (hd columns), so S(j+1) is
// computed while the softmax of tile j runs and S(j+2) waits only for P(j).V.
//   warp 0       TMA: Q once, then K_0, V_0, K_1, ... (128-key tiles, 32 KiB at hd = 128)
//   warp 1       one thread issues the score MMAs, warp 2 one thread the P.V MMAs
//   warps 4..7   softmax of keys 0..63 of each tile, warps 8..11 of keys 64..127: a thread
//                owns one query row's half tile; the two halves exchange their row maxima
//                through shared memory, so both apply the same reference max, and each writes
//                its P half as bf16 pairs into the buffer's first 64 columns (keys 0..63 in
//                columns 0..31, keys 64..127 in 32..63: the A operand of P.V); each half keeps
//                its own running sum l and rescales its half of O.
constexpr int kKT1 = 128;  // keys per tile

template <int HD>
struct Attn1Layout {
  static constexpr int kRing = 5;                    // K/V tiles (K_j and V_j alternate)
  static constexpr int kQChunk = kQTile * 128;       // [128 rows][64 bf16]
  static constexpr int kKVChunk = kKT1 * 128;        // [128 keys][64 bf16]
  static constexpr int kQBytes = (HD / 64) * kQChunk;
  static constexpr int kKVBytes = (HD / 64) * kKVChunk;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQBytes;
  static constexpr int kXOff = kKVOff + kRing * kKVBytes;  // row-max exchange [2][2][128] f32
  static constexpr int kLOff = kXOff + 2 * 2 * kQTile * 4;  // l exchange [128] f32
  static constexpr int kBarOff = kLOff + kQTile * 4;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory");
  // Cluster merge, in the idle K/V ring: the rows this CTA merges, as received from every
  // split, [split][row][kPitch] fp32 (O unnormalised; the padded pitch puts a warp's 32 rows
  // on distinct banks), and each received row's (reference max, sum) [split][row].  A CTA
  // merges at most ceil(128 / S) rows, so S splits need at most 128 + S row slots.
  static constexpr int kPitch = HD + 4;  // floats
  static constexpr int kStageOff = kKVOff;
  static constexpr int kMLOff = kStageOff + (kQTile + 8) * kPitch * 4;
  static_assert(kMLOff + (kQTile + 8) * 8 <= kKVOff + kRing * kKVBytes, "merge staging");
};

// The split-KV merge inside a cluster (the splits of one unit, cluster rank = split).  CTA q
// merges rows [q 128 / S, (q + 1) 128 / S) of the query tile.  Three steps, every thread of
// every CTA taking part in the two cluster barriers:
//   1. barrier: every CTA of the cluster is past its main loop, so every K/V ring is idle;
//   2. each CTA stores every row of its partial (O unnormalised; the row's reference max m and
//      sum l, base 2) into the ring of the CTA that merges the row (remote stores, no round
//      trip); barrier: all rows have arrived;
//   3. each CTA combines its rows from its own shared memory in rank order (the same order for
//      every row): O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, M = max_s m_s.  No CTA
//      touches another's shared memory after the second barrier.
__device__ __forceinline__ int merge_owner(int row, int S) { return ((row + 1) * S - 1) / kQTile; }

// One softmax thread's half row (HD / 2 columns at column half * HD / 2) of its partial into
// the merging CTA's receive slot; the half-0 thread also sends (m, l).
template <int HD>
__device__ __forceinline__ void attn1_push(uint8_t* smem, int S, int split, int row, int half,
                                           const float* o, float m, float l) {
  using Lay = Attn1Layout<HD>;
  const int q = merge_owner(row, S);
  const int rpo = (kQTile + S - 1) / S;  // row slots per split
  const int slot = split * rpo + (row - q * kQTile / S);
  const uint32_t dst = dsmem_addr(
      smem_u32(smem + Lay::kStageOff) + (slot * Lay::kPitch + half * (HD / 2)) * 4, q);
#pragma unroll
  for (int c = 0; c < HD / 2; c += 4)
    st_dsmem_f4(dst + c * 4, make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]));
  if (half == 0) st_dsmem_f2(dsmem_addr(smem_u32(smem + Lay::kMLOff) + slot * 8, q),
                             make_float2(m, l));
}

__device__ __forceinline__ void cluster_sync_all() {
  __syncwarp();  // the cluster barrier is warp-aligned
  cluster_arrive();
  cluster_wait();
}

// Step 3 (with the second barrier); called by every thread of the CTA once its softmax
// threads have pushed their rows.
template <int HD>
__device__ __forceinline__ void attn1_cluster_merge(const AttnParams& p, uint8_t* smem, int b,
                                                    int hq, int qt) {
  using Lay = Attn1Layout<HD>;
  constexpr int kCG = HD / 16;  // 16-column groups of a row
  cluster_sync_all();  // every CTA's rows are in their merging CTAs
  const int S = p.splits;
  const int q = static_cast<int>(cluster_ctarank());
  const int r0 = q * kQTile / S, r1 = (q + 1) * kQTile / S;
  const int rpo = (kQTile + S - 1) / S;
  const float* stage = reinterpret_cast<const float*>(smem + Lay::kStageOff);
  const float2* mls = reinterpret_cast<const float2*>(smem + Lay::kMLOff);
  for (int i = static_cast<int>(threadIdx.x) - 128; i >= 0 && i < (r1 - r0) * kCG; i += 256) {
    const int lr = i / kCG;
    const int cg = i % kCG;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, mls[s * rpo + lr].x);
    float L = 0.f;
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int s = 0; s < S; ++s) {
      const float2 ml = mls[s * rpo + lr];
      if (ml.x == -INFINITY) continue;  // an empty partial (or one given up) adds nothing
      const float w = ex2_approx(ml.x - M);
      L += w * ml.y;
      const float4* src =
          reinterpret_cast<const float4*>(stage + (s * rpo + lr) * Lay::kPitch + cg * 16);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = src[k];
        acc[4 * k] += w * v.x;
        acc[4 * k + 1] += w * v.y;
        acc[4 * k + 2] += w * v.z;
        acc[4 * k + 3] += w * v.w;
      }
    }
    const int qi = qt * kQTile + r0 + lr;
    if (qi < p.L) {
      const float inv_l = 1.f / L;
      uint4* dst = reinterpret_cast<uint4*>(
          p.out + ((static_cast<int64_t>(b) * p.L + qi) * p.H + hq) * HD + cg * 16);
#pragma unroll
      for (int k = 0; k < 2; ++k)
        dst[k] = make_uint4(pack_bf16x2(acc[8 * k + 0] * inv_l, acc[8 * k + 1] * inv_l),
                            pack_bf16x2(acc[8 * k + 2] * inv_l, acc[8 * k + 3] * inv_l),
                            pack_bf16x2(acc[8 * k + 4] * inv_l, acc[8 * k + 5] * inv_l),
                            pack_bf16x2(acc[8 * k + 6] * inv_l, acc[8 * k + 7] * inv_l));
      if (cg == 0 && p.lse)
        p.lse[(static_cast<int64_t>(b) * p.H + hq) * p.L + qi] =
            (M + __log2f(L)) * 0.6931471805599453f;
    }
  }
}

__device__ __forceinline__ void attn1_unit(int u, const AttnParams& p, int& b, int& h, int& qt) {
  qt = u % p.n_qtiles;
  h = (u / p.n_qtiles) % p.H;
  b = u / (p.n_qtiles * p.H);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    canvas_attn1_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmKp,
                        const __grid_constant__ CUtensorMap tmVp,
                        const __grid_constant__ CUtensorMap tmKc,
                        const __grid_constant__ CUtensorMap tmVc, AttnParams p) {
  using Lay = Attn1Layout<HD>;
  constexpr int kRing = Lay::kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* xmax = reinterpret_cast<float*>(smem + Lay::kXOff);  // [tile parity][half][row]
  float* xl = reinterpret_cast<float*>(smem + Lay::kLOff);    // [row]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;             // [kRing]
  uint64_t* kv_empty = bars + 1 + kRing;    // [kRing]
  uint64_t* s_full = bars + 1 + 2 * kRing;  // [buffer]
  uint64_t* p_full = s_full + 2;            // [buffer]
  uint64_t* pv_done = s_full + 4;           // [buffer]
  uint64_t* drain = s_full + 6;             // [issuer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int b, hq, qt;
  attn1_unit(blockIdx.x, p, b, hq, qt);
  const int g = (hq * p.Hkv) / p.H;
  const int split = blockIdx.y;

  int t_lo = 0;  // first 128-key prefix tile a query of this tile can see
  if (p.window > 0) {
    const int kmin = p.P + qt * kQTile - p.window + 1;
    t_lo = kmin > 0 ? kmin / kKT1 : 0;
    if (t_lo > p.n_pre_tiles) t_lo = p.n_pre_tiles;
  }
  const int n_pre = p.n_pre_tiles - t_lo;
  const int nt_all = n_pre + p.n_can_tiles;
  const int t_begin = static_cast<int>(static_cast<int64_t>(split) * nt_all / p.splits);
  const int t_end = static_cast<int>(static_cast<int64_t>(split + 1) * nt_all / p.splits);
  const int nt = t_end > t_begin ? t_end - t_begin : 0;

  const int half = warp >= 8 ? 1 : 0;         // softmax warps: which 64 keys of a tile
  const int row_in = (warp & 3) * 32 + lane;  // TMEM lane quarter of this warp
  const int qi = qt * kQTile + row_in;
  const int64_t out_row = (static_cast<int64_t>(b) * p.H + hq) * p.L + qi;  // (b, h, i)
  const int64_t part_rows = static_cast<int64_t>(p.B) * p.H * p.L;
  uint8_t* q_buf = smem + Lay::kQOff;
  auto kv_buf = [&](int i) { return smem + Lay::kKVOff + (i % kRing) * Lay::kKVBytes; };

  // Before the wait for the previous kernel: the barriers, and the prefix K/V tiles of the
  // first ring slots (the cache, which the kernels of a denoising step do not write); thread
  // 0 is the producer.
  int n_early = 0;
  if (threadIdx.x == 0 && nt > 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);  // K slots: the score thread; V slots: the P.V thread
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 8);  // one arrival per softmax warp
      mbar_init(&pv_done[s], 1);
      mbar_init(&drain[s], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmKp);
    tma_prefetch_map(&tmVp);
    for (int i = 0; i < 2 * nt && i < kRing; ++i) {
      const int t = t_begin + (i >> 1);
      if (t >= n_pre) break;
      const CUtensorMap* m = (i & 1) ? &tmVp : &tmKp;
      mbar_arrive_expect_tx(&kv_full[i], Lay::kKVBytes);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_4d(kv_buf(i) + c * Lay::kKVChunk, m, &kv_full[i], c * 64, g, (t_lo + t) * kKT1,
                    b);
      ++n_early;
    }
  }
  pdl_wait();
  if (p.n_active && *p.n_active == 0) {  // the same for every CTA of the grid
    if (threadIdx.x == 0)  // let the started copies land before the CTA leaves
      for (int i = 0; i < n_early; ++i) mbar_wait_drain(&kv_full[i], 0);
    return;
  }
  pdl_trigger();  // the next kernel's CTAs may start their own prologue on idle SMs

  if (nt == 0) {  // nothing to do: empty partials (only when splits > 1)
    if (p.cluster_merge) {  // an empty partial for the cluster's merge, which every CTA joins
      cluster_sync_all();  // every ring of the cluster is idle
      if (warp >= 4) {
        float o[HD / 2];
        for (int c = 0; c < HD / 2; ++c) o[c] = 0.f;
        attn1_push<HD>(smem, p.splits, split, row_in, half, o, -INFINITY, 0.f);
      }
      attn1_cluster_merge<HD>(p, smem, b, hq, qt);
      return;
    }
    if (warp >= 4 && qi < p.L) {
      if (half == 0) {
        float* ml = p.part_ml + (split * part_rows + out_row) * 2;
        ml[0] = -INFINITY;
        ml[1] = 0.f;
      }
      float* po = p.part_o + (split * part_rows + out_row) * HD + half * (HD / 2);
      for (int c = 0; c < HD / 2; ++c) po[c] = 0.f;
    }
    return;
  }

  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto tm_s = [&](int bf) { return tmem + bf * kKT1; };
  const uint32_t tm_o = tmem + 2 * kKT1;

  if (warp < 4) {
    regs_decrease<kRegsControl>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------------ producer -----
      tma_prefetch_map(&tmQ);
      mbar_arrive_expect_tx(q_full, Lay::kQBytes);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_4d(q_buf + c * Lay::kQChunk, &tmQ, q_full, c * 64, hq, qt * kQTile, b);
      int issued = 0;
      for (int i = 0; i < 2 * nt; ++i) {
        if (i < n_early) {  // requested before the wait
          ++issued;
          continue;
        }
        const int rs = i % kRing;
        if (!mbar_wait(&kv_empty[rs], ((i / kRing) & 1) ^ 1, abort_flag, p.wait_ns)) break;
        const int t = t_begin + (i >> 1);
        const bool pre = t < n_pre;
        const int kb = pre ? (t_lo + t) * kKT1 : (t - n_pre) * kKT1;
        const CUtensorMap* m = (i & 1) ? (pre ? &tmVp : &tmVc) : (pre ? &tmKp : &tmKc);
        uint8_t* dst = kv_buf(i);
        mbar_arrive_expect_tx(&kv_full[rs], Lay::kKVBytes);
        for (int c = 0; c < HD / 64; ++c)
          tma_load_4d(dst + c * Lay::kKVChunk, m, &kv_full[rs], c * 64, g, kb, b);
        ++issued;
      }
      if (*abort_flag) {
        mbar_wait_drain(q_full, 0);
        for (int i = (issued > kRing ? issued - kRing : 0); i < issued; ++i)
          mbar_wait_drain(&kv_full[i % kRing], (i / kRing) & 1);
      }
    } else if ((warp == 1 || warp == 2) && lane == 0) {
      // ------------------------------------------------------------------ MMA issuers -----
      constexpr uint32_t idesc_s = idesc_bf16(128, kKT1, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, HD, true);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.wait_ns);
      auto wait_kv = [&](int i) {
        return mbar_wait(&kv_full[i % kRing], (i / kRing) & 1, abort_flag, p.wait_ns);
      };
      if (warp == 1) {
        const uint32_t qa = smem_u32(q_buf);
        for (int j = 0; ok && j < nt; ++j) {
          if (!(ok = wait_kv(2 * j))) break;
          // S(j) overwrites the buffer whose first columns hold P(j-2)
          if (j >= 2 && !(ok = mbar_wait(&pv_done[j & 1], ((j - 2) >> 1) & 1, abort_flag,
                                         p.wait_ns)))
            break;
          tc_fence_after();
          const uint32_t ka = smem_u32(kv_buf(2 * j));
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            mma_bf16_ss(tm_s(j & 1),
                        sdesc_sw128(qa + (kk >> 2) * Lay::kQChunk + (kk & 3) * 32, 16, 1024),
                        sdesc_sw128(ka + (kk >> 2) * Lay::kKVChunk + (kk & 3) * 32, 16, 1024),
                        idesc_s, kk > 0 ? 1u : 0u);
          mma_commit(&s_full[j & 1]);
          mma_commit(&kv_empty[(2 * j) % kRing]);
        }
      } else {
        for (int j = 0; ok && j < nt; ++j) {
          if (!(ok = wait_kv(2 * j + 1))) break;
          if (!(ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, p.wait_ns))) break;
          tc_fence_after();
          const uint32_t va = smem_u32(kv_buf(2 * j + 1));
#pragma unroll
          for (int kk = 0; kk < kKT1 / 16; ++kk)
            mma_bf16_ts(tm_o, tm_s(j & 1) + kk * 8,
                        sdesc_sw128(va + kk * 2048, Lay::kKVChunk, 1024), idesc_o,
                        (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&pv_done[j & 1]);
          mma_commit(&kv_empty[(2 * j + 1) % kRing]);
        }
      }
      if (*abort_flag) {  // make sure no MMA is still writing TMEM before it is released
        mma_commit(&drain[warp - 1]);
        mbar_wait_drain(&drain[warp - 1], 0);
      }
    }
  } else {
    regs_increase<kRegsSoftmax>();
    // --------------------------------------------------------------- softmax warps -----
    const uint32_t lane_base = tmem_lane_base(warp);
    float m_ref = -INFINITY;
    float l = 0.f;  // this half's running sum
    bool ok = true;
    const int kmin = p.window > 0 ? p.P + qi - p.window + 1 : 0;
    const float c = p.scale_log2;
    for (int j = 0; j < nt; ++j) {
      const int bf = j & 1;
      // both halves take every step of the loop (the exchange barrier below), even after an
      // abort; only the waits, loads and stores are skipped
      if (ok) ok = warp_wait(&s_full[bf], (j >> 1) & 1, abort_flag, p.wait_ns);
      tc_fence_after();
      const int t = t_begin + j;
      const bool pre = t < n_pre;
      const int kb = (pre ? (t_lo + t) * kKT1 : (t - n_pre) * kKT1) + half * 64;
      const int klim = pre ? p.P : p.L;
      const int klo = pre ? kmin : 0;
      float sv[64];
      if (ok) {
        tmem_ld64(tm_s(bf) + lane_base + half * 64, sv);
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[e] = -INFINITY;
      }
      if (!(kb >= klo && kb + 64 <= klim)) {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int key = kb + e;
          if (!(key < klim && key >= klo)) sv[e] = -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) mx[q] = sv[q];
#pragma unroll
      for (int e = 8; e < 64; e += 2) mx[(e >> 1) & 7] = fmax3(mx[(e >> 1) & 7], sv[e], sv[e + 1]);
      float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // the row's max over both halves (the exchange slot of this tile's parity is free: the
      // other half passed the previous tile's barrier only after reading it)
      xmax[(bf * 2 + half) * kQTile + row_in] = mt;
      named_bar_sync(1, 256);
      mt = fmaxf(mt, xmax[(bf * 2 + (half ^ 1)) * kQTile + row_in]);
      const float m_new = fmaxf(m_ref, mt * c);
      const bool need = j > 0 && m_new > m_ref + kRescaleLog2;
      const float f = need ? ex2_approx(m_ref - m_new) : 1.f;
      if (j == 0 || need) m_ref = m_new;
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
      float ps[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) ps[q] = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 64; e += 2) {  // two scores per packed fp32 instruction
        float xa, xb;
        ffma2(xa, xb, sv[e], sv[e + 1], c, c, -m_use, -m_use);
        const float a = ex2_approx(xa);
        const float bb = ex2_approx(xb);
        const int q = (e >> 1) & 3;
        fadd2(ps[2 * q], ps[2 * q + 1], ps[2 * q], ps[2 * q + 1], a, bb);
        pk[e >> 1] = pack_bf16x2(a, bb);
      }
      // P of this half: columns half * 32 .. + 32 (the other half's raw scores there were
      // read before the exchange barrier)
      if (ok) tmem_st32(tm_s(bf) + lane_base + half * 32, pk);
      const float rs = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      l = l * f + rs;
      if (ok && __any_sync(0xFFFFFFFFu, need)) {  // O *= f (this half's columns) after P(j-1).V
        if (!warp_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.wait_ns)) {
          ok = false;
        } else {
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < HD / 64; ++cc) {
            float o[32];
            tmem_ld32(tm_o + lane_base + half * (HD / 2) + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tmem_st32(tm_o + lane_base + half * (HD / 2) + cc * 32, o);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[bf]);
    }
    if (ok) ok = warp_wait(&pv_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, abort_flag, p.wait_ns);
    tc_fence_after();
    // the row's sum over both halves
    if (half == 1) xl[row_in] = l;
    named_bar_sync(1, 256);
    const float lt = half == 0 ? l + xl[row_in] : 0.f;
    if (half == 0) xl[row_in] = lt;
    named_bar_sync(1, 256);
    const float l_row = xl[row_in];
    const bool write = ok && qi < p.L;
    if (p.splits == 1) {
      const float inv_l = 1.f / l_row;
      uint16_t* dst = p.out + ((static_cast<int64_t>(b) * p.L + qi) * p.H + hq) * HD +
                      half * (HD / 2);
#pragma unroll 1
      for (int cc = 0; cc < HD / 64; ++cc) {
        float o[32];
        tmem_ld32(tm_o + lane_base + half * (HD / 2) + cc * 32, o);
        if (write) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack_bf16x2(o[q * 8 + 0] * inv_l, o[q * 8 + 1] * inv_l),
                               pack_bf16x2(o[q * 8 + 2] * inv_l, o[q * 8 + 3] * inv_l),
                               pack_bf16x2(o[q * 8 + 4] * inv_l, o[q * 8 + 5] * inv_l),
                               pack_bf16x2(o[q * 8 + 6] * inv_l, o[q * 8 + 7] * inv_l));
        }
      }
      if (write && half == 0 && p.lse)
        p.lse[out_row] = (m_ref + __log2f(l_row)) * 0.6931471805599453f;
    } else if (p.cluster_merge) {
      // this row's partial into the CTA that merges it, once every CTA of the cluster is past
      // its main loop (the control warps take the same barrier in the common tail); a CTA
      // that gave up waiting contributes nothing
      float o[HD / 2];
#pragma unroll
      for (int cc = 0; cc < HD / 64; ++cc) {
        float t[32];
        tmem_ld32(tm_o + lane_base + half * (HD / 2) + cc * 32, t);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[cc * 32 + e] = ok ? t[e] : 0.f;
      }
      cluster_sync_all();  // every ring of the cluster is idle
      attn1_push<HD>(smem, p.splits, split, row_in, half, o, ok ? m_ref : -INFINITY,
                     ok ? l_row : 0.f);
    } else {
      const int64_t prow = split * part_rows + out_row;
      float* po = p.part_o + prow * HD + half * (HD / 2);
#pragma unroll 1
      for (int cc = 0; cc < HD / 64; ++cc) {
        float o[32];
        tmem_ld32(tm_o + lane_base + half * (HD / 2) + cc * 32, o);
        if (write) {
          float4* d4 = reinterpret_cast<float4*>(po + cc * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            d4[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
      if (write && half == 0) {
        p.part_ml[prow * 2] = m_ref;
        p.part_ml[prow * 2 + 1] = l_row;
      }
    }
  }

  if (p.cluster_merge) {
    if (warp < 4) cluster_sync_all();  // the softmax warps took this barrier before their pushes
    attn1_cluster_merge<HD>(p, smem, b, hq, qt);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, kStatusTimeout);
}

// Combines split partials: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.  One warp per
// (b, h, i) row; lane s holds the (m, l) of splits s and s + 32, so the weights need one load
// round trip, and the O loads of consecutive splits are independent.
template <int HD>
__global__ void attn_merge_kernel(AttnParams p) {
  pdl_wait();
  pdl_trigger();
  if (p.n_active && *p.n_active == 0) return;
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.L;
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
  if (lane < p.splits) {
    m0 = p.part_ml[(lane * rows + row) * 2];
    l0 = p.part_ml[(lane * rows + row) * 2 + 1];
  }
  if (lane + 32 < p.splits) {
    m1 = p.part_ml[((lane + 32) * rows + row) * 2];
    l1 = p.part_ml[((lane + 32) * rows + row) * 2 + 1];
  }
  float M = fmaxf(m0, m1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  const float w0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - M);
  const float w1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - M);
  float l = w0 * l0 + w1 * l1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
  float acc[HD / 32];
#pragma unroll
  for (int e = 0; e < HD / 32; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int s = 0; s < p.splits; ++s) {
    const float w = __shfl_sync(0xFFFFFFFFu, s < 32 ? w0 : w1, s & 31);
    const float* po = p.part_o + (s * rows + row) * HD;
#pragma unroll
    for (int e = 0; e < HD / 32; ++e) acc[e] += w * po[e * 32 + lane];
  }
  const int i = static_cast<int>(row % p.L);
  const int64_t bh = row / p.L;
  const int h = static_cast<int>(bh % p.H);
  const int64_t b = bh / p.H;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + ((b * p.L + i) * p.H + h) * HD;
  const float inv_l = 1.f / l;
#pragma unroll
  for (int e = 0; e < HD / 32; ++e) dst[e * 32 + lane] = __float2bfloat16_rn(acc[e] * inv_l);
  if (p.lse && lane == 0) p.lse[row] = (M + __log2f(l)) * 0.6931471805599453f;
}

// How many clusters of S one-slot CTAs (cluster along the key splits) can be resident at once
// on this device (0: none); asked once per device and S.
template <int HD>
int attn1_max_clusters(int S) {
  static std::mutex mu;
  static std::vector<std::array<int, 9>> known;  // per device and S: -1 unknown
  const int dev = device_id();
  std::lock_guard<std::mutex> lk(mu);
  while (static_cast<int>(known.size()) <= dev) {
    std::array<int, 9> a;
    a.fill(-1);
    known.push_back(a);
  }
  int& n = known[dev][S];
  if (n < 0) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, S, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Attn1Layout<HD>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = S;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaFuncSetAttribute(canvas_attn1_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Attn1Layout<HD>::kSmemBytes) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c, canvas_attn1_kernel<HD>, &cfg) != cudaSuccess) {
      cudaGetLastError();  // clear the query's error: the launch then uses the merge kernel
      c = 0;
    }
    n = c;
  }
  return n;
}

template <int HD>
cudaError_t launch_hd(const CUtensorMap* maps, const AttnParams& p_in, bool one,
                      cudaStream_t st) {
  using Lay = AttnLayout<HD>;
  using Lay1 = Attn1Layout<HD>;
  static int configured_device = -1;
  const int dev = device_id();
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(canvas_attn_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(canvas_attn1_kernel<HD>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, Lay1::kSmemBytes);
    if (e != cudaSuccess) return e;
    // The register split must fit the block's launch allocation, or an increase would never
    // be granted: refuse to launch a build where it does not.
    for (auto fn : {canvas_attn_kernel<HD>, canvas_attn1_kernel<HD>}) {
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      if (static_cast<long>(fa.numRegs) * kThreads < 128L * kRegsControl + 256L * kRegsSoftmax)
        return cudaErrorInvalidConfiguration;
    }
    configured_device = dev;
  }
  // One-slot kernel with 2..8 key splits: the splits of a unit run as one cluster and merge
  // in it, when every cluster of the launch can be resident at once; otherwise the split
  // partials go through the workspace to attn_merge_kernel.
  AttnParams p = p_in;
  p.cluster_merge = one && p.splits >= 2 && p.splits <= 8 &&
                    attn1_max_clusters<HD>(p.splits) >= p.units;
  dim3 grid(p.units, p.splits);
  timer_begin(1, st);
  cudaError_t e;
  if (p.cluster_merge) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay1::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = p.splits;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, canvas_attn1_kernel<HD>, maps[0], maps[1], maps[2], maps[3],
                           maps[4], p);
  } else {
    e = one ? launch_dependent(canvas_attn1_kernel<HD>, grid, dim3(kThreads), Lay1::kSmemBytes,
                               st, maps[0], maps[1], maps[2], maps[3], maps[4], p)
            : launch_dependent(canvas_attn_kernel<HD>, grid, dim3(kThreads), Lay::kSmemBytes, st,
                               maps[0], maps[1], maps[2], maps[3], maps[4], p);
  }
  if (e != cudaSuccess) return e;
  if (p.splits > 1 && !p.cluster_merge) {
    const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.L;
    const int warps_per_block = 8;
    e = launch_dependent(attn_merge_kernel<HD>,
                         dim3(static_cast<int>((rows + warps_per_block - 1) / warps_per_block)),
                         dim3(32 * warps_per_block), 0, st, p);
  }
  timer_end(1, st);
  return e;
}

int attn_units(int B, int L, int H, int Hkv) {
  const int n_q = (L + kQTile - 1) / kQTile;
  const int r = H / Hkv;
  return (r % 2 == 0) ? B * (H / 2) * n_q : B * H * ((n_q + 1) / 2);
}

}  // namespace

AttnPlan plan_attention(int B, int L, int P, int H, int Hkv, int hd, int window) {
  // Kernel: the two-slot kernel (two query heads of a GQA group share each 64-key K/V tile,
  // half the K/V bytes per FLOP) keeps long K/V streams fed; where the work is short (at most
  // ~32 of its key tiles per SM) fixed per-CTA costs and latency dominate, and the one-slot
  // kernel (128-key tiles, full-rate MMAs, twice the CTAs) is faster.  Measured: window1k
  // 0.0234 -> 0.0193 ms, one canvas with a 4,096-key prefix 0.029 -> 0.025 ms; but long128k
  // 0.234 -> 0.260 ms, 16 canvases at 8,192 keys 0.277 -> 0.308 ms, 64 canvases at 4,096 keys
  // 0.537 -> 0.607 ms (there the one-slot kernel waits on its K/V stream).
  const int eff_p = (window > 0 && window < P) ? window + L : P;  // keys a query tile may see
  const int sms = num_sms();
  const int64_t two_slot_tiles = static_cast<int64_t>(attn_units(B, L, H, Hkv)) *
                                 ((eff_p + kKTile - 1) / kKTile + (L + kKTile - 1) / kKTile);
  const bool one = hd == 128 && two_slot_tiles <= 32ll * sms;
  const int kt = one ? kKT1 : kKTile;
  const int units = one ? B * H * ((L + kQTile - 1) / kQTile) : attn_units(B, L, H, Hkv);
  const int nt_all = (eff_p + kt - 1) / kt + (L + kt - 1) / kt;
  // Cost in units of one key tile of a CTA: waves x (tiles per split + a fixed cost per CTA
  // for start-up, pipeline fill and the partial write: ~6 64-key tiles, ~3 128-key tiles),
  // plus the same for the merge kernel when keys are split; ties go to fewer splits.  With at
  // least one CTA per SM already, keys are not split.
  const int fixed = one ? 3 : 6;
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= nt_all && s <= 64 && (s == 1 || units < sms); ++s) {
    const int per = (nt_all + s - 1) / s;
    const int64_t ctas = static_cast<int64_t>(units) * s;
    const int64_t waves = (ctas + sms - 1) / sms;
    const int64_t cost = waves * (per + fixed) + (s > 1 ? fixed : 0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  AttnPlan pl;
  pl.splits = best;
  pl.one = one ? 1 : 0;
  pl.units = units;
  pl.part_bytes = best > 1 ? static_cast<size_t>(best) * B * H * L * (hd + 2) * sizeof(float) : 0;
  return pl;
}

cudaError_t launch_attention(const uint16_t* q, const uint16_t* k_pre, const uint16_t* v_pre,
                             const uint16_t* k_can, const uint16_t* v_can, uint16_t* out,
                             float* lse, int B, int L, int P, int H, int Hkv, int hd, int window,
                             float scale, void* part_ws, uint32_t* status, const int* n_active,
                             cudaStream_t st, int pre_stride) {
  if (pre_stride < 0) pre_stride = P;
  const AttnPlan pl = plan_attention(B, L, P, H, Hkv, hd, window);
  CUtensorMap maps[5];
  {
    const uint32_t box[4] = {64u, 1u, static_cast<uint32_t>(kQTile), 1u};
    const uint64_t dims[4] = {static_cast<uint64_t>(hd), static_cast<uint64_t>(H),
                              static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
    const uint64_t str[3] = {static_cast<uint64_t>(hd) * 2, static_cast<uint64_t>(H) * hd * 2,
                             static_cast<uint64_t>(L) * H * hd * 2};
    if (!make_tmap_bf16(&maps[0], q, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  const int kt = pl.one ? kKT1 : kKTile;
  const uint32_t kvbox[4] = {64u, 1u, static_cast<uint32_t>(kt), 1u};
  const uint16_t* kv_src[4] = {k_pre, v_pre, k_can, v_can};
  for (int m = 0; m < 4; ++m) {
    const int rows = m < 2 ? (P > 0 ? P : 1) : L;
    const uint16_t* base = kv_src[m];
    if (m < 2 && P == 0) base = k_can;  // never read: the prefix has no tiles
    const uint64_t dims[4] = {static_cast<uint64_t>(hd), static_cast<uint64_t>(Hkv),
                              static_cast<uint64_t>(rows), static_cast<uint64_t>(B)};
    const uint64_t str[3] = {static_cast<uint64_t>(hd) * 2, static_cast<uint64_t>(Hkv) * hd * 2,
                             static_cast<uint64_t>(m < 2 ? (P > 0 ? pre_stride : L) : L) * Hkv *
                                 hd * 2};
    if (!make_tmap_bf16(&maps[1 + m], base, 4, dims, str, kvbox)) return cudaErrorInvalidValue;
  }
  AttnParams p;
  p.B = B;
  p.L = L;
  p.P = P;
  p.H = H;
  p.Hkv = Hkv;
  p.hd = hd;
  p.window = window;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.n_pre_tiles = (P + kt - 1) / kt;
  p.n_can_tiles = (L + kt - 1) / kt;
  p.n_qtiles = (L + kQTile - 1) / kQTile;
  p.splits = pl.splits;
  p.units = pl.units;
  p.out = out;
  p.lse = lse;
  p.part_o = reinterpret_cast<float*>(part_ws);
  p.part_ml = pl.splits > 1 ? p.part_o + static_cast<size_t>(pl.splits) * B * H * L * hd : nullptr;
  p.status = status;
  p.n_active = n_active;
  p.wait_ns = wait_limit_ns();
  p.cluster_merge = 0;
  return hd == 64 ? launch_hd<64>(maps, p, pl.one != 0, st)
                  : launch_hd<128>(maps, p, pl.one != 0, st);
}

}  // namespace dg
