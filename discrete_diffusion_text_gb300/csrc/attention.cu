// Canvas attention on the 5th-generation tensor cores: 128 canvas queries of one head
// against the visible prefix keys and all canvas keys, in key tiles of 128.
//
// Per CTA = (canvas b, query head h, query tile, key split):
//   warp 0     TMA: the Q tile once, then K/V tiles into a 2-stage ring (128-byte swizzle);
//   warp 1     one thread issues S_j = Q K_j^T (tcgen05, M=128, N=128) into one of two TMEM
//              score buffers, and O += P_{j-1} V_{j-1} (M=128, N=hd) once P_{j-1} is ready;
//   warps 2..5 one thread per query row: read S_j from TMEM, mask, exponentiate against a
//              running reference max, write P_j (bf16) to shared memory in the swizzled
//              K-major layout the tensor core reads.
// The reference max is only raised when a row's max grows by more than 2^8 (log2 units):
// p <= 256 stays exact in fp32 accumulation and bf16, and O/l use the same reference, so the
// result is unchanged while O (in TMEM) is rescaled rarely.
// With several key splits, each writes unnormalised fp32 partials (O, m, l) and a merge
// kernel combines them with the log-sum-exp rule.
#include "kernels.cuh"
#include "sm103.cuh"

namespace dg {
namespace {

constexpr int kTile = 128;         // queries per CTA and keys per tile
constexpr float kRescaleLog2 = 8.f;

struct AttnParams {
  int B, L, P, H, Hkv, hd, window;
  float scale_log2;  // scale * log2(e)
  int n_pre_tiles, n_can_tiles, n_qtiles, splits;
  uint16_t* out;
  float* lse;
  float* part_o;   // [splits][B*H*L][hd]
  float* part_ml;  // [splits][B*H*L][2]
  uint32_t* status;
  const int* n_active;
};

template <int HD>
struct AttnLayout {
  static constexpr int kChunk = kTile * 64 * 2;      // one [128][64] bf16 swizzled chunk
  static constexpr int kQBytes = (HD / 64) * kChunk;
  static constexpr int kKVBytes = (HD / 64) * kChunk;  // one of K or V
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kPBytes = 2 * kChunk;          // [128 queries][128 keys]
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQBytes;
  static constexpr int kPOff = kKVOff + 2 * kStageBytes;
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
};

__device__ __forceinline__ void write_p_row(uint8_t* pbuf, int row, const float* p) {
  // 128 bf16 of one query row into two [128 rows][64 keys] chunks, 16-byte units swizzled by
  // (row % 8), matching the 128-byte-swizzle K-major operand layout.
#pragma unroll
  for (int u16 = 0; u16 < 16; ++u16) {
    const int chunk = u16 >> 3;
    const int u = u16 & 7;
    const int phys = u ^ (row & 7);
    uint4 v;
    v.x = pack_bf16x2(p[u16 * 8 + 0], p[u16 * 8 + 1]);
    v.y = pack_bf16x2(p[u16 * 8 + 2], p[u16 * 8 + 3]);
    v.z = pack_bf16x2(p[u16 * 8 + 4], p[u16 * 8 + 5]);
    v.w = pack_bf16x2(p[u16 * 8 + 6], p[u16 * 8 + 7]);
    *reinterpret_cast<uint4*>(pbuf + chunk * (kTile * 128) + row * 128 + phys * 16) = v;
  }
}

template <int HD>
__global__ void __launch_bounds__(192, 1)
    canvas_attn_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmKp,
                       const __grid_constant__ CUtensorMap tmVp,
                       const __grid_constant__ CUtensorMap tmKc,
                       const __grid_constant__ CUtensorMap tmVc, AttnParams p) {
  using Lay = AttnLayout<HD>;
  if (p.n_active && *p.n_active == 0) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;    // [2]
  uint64_t* pv_done = bars + 9;   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int idx = blockIdx.x;
  const int qt = idx % p.n_qtiles;
  idx /= p.n_qtiles;
  const int h = idx % p.H;
  const int b = idx / p.H;
  const int g = (h * p.Hkv) / p.H;
  const int split = blockIdx.y;
  const int q0 = qt * kTile;

  // Key tiles of this query tile: prefix tiles from the first one any of its queries can see,
  // then the canvas tiles; this split takes a contiguous share of them.
  int t_lo = 0;
  if (p.window > 0) {
    const int kmin = p.P + q0 - p.window + 1;
    t_lo = kmin > 0 ? kmin / kTile : 0;
    if (t_lo > p.n_pre_tiles) t_lo = p.n_pre_tiles;
  }
  const int n_pre = p.n_pre_tiles - t_lo;
  const int nt_all = n_pre + p.n_can_tiles;
  const int per = (nt_all + p.splits - 1) / p.splits;
  const int t_begin = split * per;
  const int t_end = min(nt_all, t_begin + per);
  const int nt = t_end > t_begin ? t_end - t_begin : 0;

  const int row_in = (warp & 3) * 32 + lane;  // softmax warps 2..5 -> quarters 2,3,0,1
  const int qi = q0 + row_in;
  const int64_t out_row = (static_cast<int64_t>(b) * p.H + h) * p.L + qi;  // (b, h, i)

  if (nt == 0) {  // nothing to do: an empty partial (only when splits > 1)
    if (warp >= 2 && qi < p.L) {
      float* ml = p.part_ml + (static_cast<int64_t>(split) * p.B * p.H * p.L + out_row) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
      float* po = p.part_o + (static_cast<int64_t>(split) * p.B * p.H * p.L + out_row) * HD;
      for (int c = 0; c < HD; ++c) po[c] = 0.f;
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 128);
      mbar_init(&pv_done[s], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_s0 = tmem;         // scores, buffer 0: columns [0, 128)
  const uint32_t tm_o = tmem + 256;    // output accumulator: columns [256, 256 + HD)

  uint8_t* sQ = smem + Lay::kQOff;
  auto kv_stage = [&](int s) { return smem + Lay::kKVOff + s * Lay::kStageBytes; };
  auto p_buf = [&](int s) { return smem + Lay::kPOff + s * Lay::kPBytes; };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      mbar_arrive_expect_tx(q_full, Lay::kQBytes);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_4d(sQ + c * Lay::kChunk, &tmQ, q_full, c * 64, h, q0, b);
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&kv_empty[s], ((j >> 1) & 1) ^ 1, abort_flag)) break;
        const int t = t_begin + j;
        const bool pre = t < n_pre;
        const int kb = pre ? (t_lo + t) * kTile : (t - n_pre) * kTile;
        const CUtensorMap* mk = pre ? &tmKp : &tmKc;
        const CUtensorMap* mv = pre ? &tmVp : &tmVc;
        uint8_t* st = kv_stage(s);
        mbar_arrive_expect_tx(&kv_full[s], Lay::kStageBytes);
        for (int c = 0; c < HD / 64; ++c) {
          tma_load_4d(st + c * Lay::kChunk, mk, &kv_full[s], c * 64, g, kb, b);
          tma_load_4d(st + Lay::kKVBytes + c * Lay::kChunk, mv, &kv_full[s], c * 64, g, kb, b);
        }
        ++issued;
      }
      if (*abort_flag) {
        mbar_wait_drain(q_full, 0);
        for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
          mbar_wait_drain(&kv_full[j & 1], (j >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, kTile, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, HD, true);
      const uint32_t q_addr = smem_u32(sQ);
      bool ok = mbar_wait(q_full, 0, abort_flag);
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj & 1;
        if (!mbar_wait(&p_full[s], (jj >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(p_buf(s));
        const uint32_t va = smem_u32(kv_stage(s) + Lay::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(pa + (kk >> 2) * Lay::kChunk + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(va + kk * 2048, Lay::kChunk, 1024);
          mma_bf16_ss(tm_o, ad, bd, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&pv_done[s]);
        mma_commit(&kv_empty[s]);
        return true;
      };
      for (int j = 0; ok && j < nt; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&kv_full[s], (j >> 1) & 1, abort_flag)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(&p_full[s], ((j - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t ka = smem_u32(kv_stage(s));
        const uint32_t tm_s = tm_s0 + s * kTile;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Lay::kChunk + (kk & 3) * 32;
          mma_bf16_ss(tm_s, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                      idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[s]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(nt - 1);
      if (*abort_flag) {  // make sure no MMA is still writing TMEM before it is released
        uint64_t* last = &pv_done[0];
        mma_commit(last);
        mbar_wait_drain(last, 0);
        mbar_wait_drain(last, 1);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps -----
    const uint32_t lane_base = tmem_lane_base(warp);
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    const int kmin = p.window > 0 ? p.P + qi - p.window + 1 : 0;
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1;
      if (!warp_wait(&s_full[s], (j >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const int t = t_begin + j;
      const bool pre = t < n_pre;
      const int kb = pre ? (t_lo + t) * kTile : (t - n_pre) * kTile;
      const int klim = pre ? p.P : p.L;
      const int klo = pre ? kmin : 0;
      float sv[kTile];
#pragma unroll
      for (int c = 0; c < kTile / 32; ++c) {
        float v[32];
        tmem_ld32(tm_s0 + lane_base + s * kTile + c * 32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int key = kb + c * 32 + e;
          sv[c * 32 + e] = (key < klim && key >= klo) ? v[e] * p.scale_log2 : -INFINITY;
        }
      }
      float mt = -INFINITY;
#pragma unroll
      for (int e = 0; e < kTile; ++e) mt = fmaxf(mt, sv[e]);
      const float m_new = fmaxf(m_ref, mt);
      if (j == 0) {
        m_ref = m_new;
      } else {
        const bool need = m_new > m_ref + kRescaleLog2;
        if (__any_sync(0xFFFFFFFFu, need)) {
          if (!warp_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const float f = need ? ex2_approx(m_ref - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            float o[32];
            tmem_ld32(tm_o + lane_base + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tmem_st32(tm_o + lane_base + c * 32, o);
          }
          if (need) {
            l *= f;
            m_ref = m_new;
          }
        }
      }
      if (j >= 2 && !warp_wait(&pv_done[s], ((j - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
      float rs = 0.f;
#pragma unroll
      for (int e = 0; e < kTile; ++e) {
        sv[e] = ex2_approx(sv[e] - m_use);
        rs += sv[e];
      }
      l += rs;
      write_p_row(p_buf(s), row_in, sv);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[s]);
    }
    if (ok) ok = warp_wait(&pv_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, abort_flag);
    tc_fence_after();
    const bool write = ok && qi < p.L;
    if (p.splits == 1) {
      const float inv_l = 1.f / l;
      uint16_t* dst = p.out + ((static_cast<int64_t>(b) * p.L + qi) * p.H + h) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        tmem_ld32(tm_o + lane_base + c * 32, o);
        if (write) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
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
      const int64_t prow = static_cast<int64_t>(split) * p.B * p.H * p.L + out_row;
      float* po = p.part_o + prow * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        tmem_ld32(tm_o + lane_base + c * 32, o);
        if (write) {
          float4* d4 = reinterpret_cast<float4*>(po + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q) d4[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
      if (write) {
        p.part_ml[prow * 2] = m_ref;
        p.part_ml[prow * 2 + 1] = l;
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

// Combines split partials: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.  One warp per
// (b, h, i) row.
template <int HD>
__global__ void attn_merge_kernel(AttnParams p) {
  if (p.n_active && *p.n_active == 0) return;
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.L;
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float M = -INFINITY;
  for (int s = 0; s < p.splits; ++s) M = fmaxf(M, p.part_ml[(s * rows + row) * 2]);
  float acc[HD / 32];
#pragma unroll
  for (int e = 0; e < HD / 32; ++e) acc[e] = 0.f;
  float l = 0.f;
  for (int s = 0; s < p.splits; ++s) {
    const float ms = p.part_ml[(s * rows + row) * 2];
    if (ms == -INFINITY) continue;
    const float w = ex2_approx(ms - M);
    l += w * p.part_ml[(s * rows + row) * 2 + 1];
    const float* po = p.part_o + (s * rows + row) * HD;
#pragma unroll
    for (int e = 0; e < HD / 32; ++e) acc[e] += w * po[e * 32 + lane];
  }
  const int64_t hrow = row;  // (b, h, i)
  const int i = static_cast<int>(hrow % p.L);
  const int64_t bh = hrow / p.L;
  const int h = static_cast<int>(bh % p.H);
  const int64_t b = bh / p.H;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + ((b * p.L + i) * p.H + h) * HD;
  const float inv_l = 1.f / l;
#pragma unroll
  for (int e = 0; e < HD / 32; ++e) dst[e * 32 + lane] = __float2bfloat16_rn(acc[e] * inv_l);
  if (p.lse && lane == 0) p.lse[row] = (M + __log2f(l)) * 0.6931471805599453f;
}

template <int HD>
cudaError_t launch_hd(const CUtensorMap* maps, const AttnParams& p, cudaStream_t st) {
  using Lay = AttnLayout<HD>;
  static int configured_device = -1;
  const int dev = device_id();
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(canvas_attn_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  dim3 grid(p.B * p.H * p.n_qtiles, p.splits);
  timer_begin(1, st);
  canvas_attn_kernel<HD><<<grid, 192, Lay::kSmemBytes, st>>>(maps[0], maps[1], maps[2], maps[3],
                                                             maps[4], p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.splits > 1) {
    const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.L;
    const int warps_per_block = 8;
    attn_merge_kernel<HD><<<static_cast<int>((rows + warps_per_block - 1) / warps_per_block),
                            32 * warps_per_block, 0, st>>>(p);
    e = cudaGetLastError();
  }
  timer_end(1, st);
  return e;
}

}  // namespace

AttnPlan plan_attention(int B, int L, int P, int H, int hd, int window) {
  const int n_q = (L + kTile - 1) / kTile;
  const int units = B * H * n_q;
  const int eff_p = (window > 0 && window < P) ? window + L : P;  // keys a query tile may see
  const int nt_all = (eff_p + kTile - 1) / kTile + n_q;
  const int sms = num_sms();
  // Minimise waves x tiles-per-split, then prefer fewer splits (less merge traffic).  With
  // at least one CTA per SM already, keys are not split.
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= nt_all && s <= 64 && (s == 1 || units < sms); ++s) {
    const int per = (nt_all + s - 1) / s;
    const int64_t ctas = static_cast<int64_t>(units) * s;
    const int64_t waves = (ctas + sms - 1) / sms;
    const int64_t cost = waves * (per + 1);  // +1: per-CTA setup, roughly one tile
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  AttnPlan pl;
  pl.splits = best;
  pl.part_bytes = best > 1 ? static_cast<size_t>(best) * B * H * L * (hd + 2) * sizeof(float) : 0;
  return pl;
}

cudaError_t launch_attention(const uint16_t* q, const uint16_t* k_pre, const uint16_t* v_pre,
                             const uint16_t* k_can, const uint16_t* v_can, uint16_t* out,
                             float* lse, int B, int L, int P, int H, int Hkv, int hd, int window,
                             float scale, void* part_ws, uint32_t* status, const int* n_active,
                             cudaStream_t st) {
  const AttnPlan pl = plan_attention(B, L, P, H, hd, window);
  CUtensorMap maps[5];
  const uint32_t box[4] = {64u, 1u, static_cast<uint32_t>(kTile), 1u};
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(hd), static_cast<uint64_t>(H),
                              static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
    const uint64_t str[3] = {static_cast<uint64_t>(hd) * 2, static_cast<uint64_t>(H) * hd * 2,
                             static_cast<uint64_t>(L) * H * hd * 2};
    if (!make_tmap_bf16(&maps[0], q, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  const uint16_t* kv_src[4] = {k_pre, v_pre, k_can, v_can};
  for (int m = 0; m < 4; ++m) {
    const int rows = m < 2 ? (P > 0 ? P : 1) : L;
    const uint16_t* base = kv_src[m];
    if (m < 2 && P == 0) base = k_can;  // never read: the prefix has no tiles
    const uint64_t dims[4] = {static_cast<uint64_t>(hd), static_cast<uint64_t>(Hkv),
                              static_cast<uint64_t>(rows), static_cast<uint64_t>(B)};
    const uint64_t str[3] = {static_cast<uint64_t>(hd) * 2, static_cast<uint64_t>(Hkv) * hd * 2,
                             static_cast<uint64_t>(m < 2 ? (P > 0 ? P : L) : L) * Hkv * hd * 2};
    if (!make_tmap_bf16(&maps[1 + m], base, 4, dims, str, box)) return cudaErrorInvalidValue;
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
  p.n_pre_tiles = (P + kTile - 1) / kTile;
  p.n_can_tiles = (L + kTile - 1) / kTile;
  p.n_qtiles = (L + kTile - 1) / kTile;
  p.splits = pl.splits;
  p.out = out;
  p.lse = lse;
  p.part_o = reinterpret_cast<float*>(part_ws);
  p.part_ml = pl.splits > 1 ? p.part_o + static_cast<size_t>(pl.splits) * B * H * L * hd : nullptr;
  p.status = status;
  p.n_active = n_active;
  return hd == 64 ? launch_hd<64>(maps, p, st) : launch_hd<128>(maps, p, st);
}

}  // namespace dg
