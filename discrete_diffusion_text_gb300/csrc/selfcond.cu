// Self-conditioning signal s = FFW(p_hat_0 . E) on GB300
// [TR "디노이징 반복과 self-conditioning": s_(t-h) = FFW(p_hat_0 . E)].
//
// The vocabulary pass (vocab.cu, self-conditioning instantiation) leaves, for every row r and
// vocabulary entry v, P~[r, v] = bf16(exp(z~ - m_ref)) together with the reference m_ref of
// each 32-entry chunk; its finalisation gives lse[r].  Here:
//   1. sc_gemm_kernel      fp32 partials of e = P_hat E over vocabulary splits: a 128 x 256
//                          tile per CTA on the tensor cores (tcgen05.mma, TMEM accumulator),
//                          A = P~ rows (K-major), B = E rows read MN-major (E is [V, d], so a
//                          64-row slab of E is the K x N operand as stored).  Each A stage is
//                          normalised on its way from shared to tensor memory: the four
//                          epilogue warps (idle until the accumulator is done) read row r's
//                          64 entries, multiply them by exp(m_ref - lse[r]), re-round to bf16
//                          and store them into a TMEM ring that the MMA reads as its A operand
//                          (row r in lane r), so P_hat = bf16(P~ exp(m_ref - lse)) never goes
//                          back to HBM or to shared memory;
//   2. sc_reduce_kernel    e = bf16(sum of the partials, in split order);
//   3. two projection GEMMs: u = bf16(gelu(e Wsc1^T)), s = bf16(u Wsc2^T).
// The contraction over the 262,144-entry vocabulary is split across CTAs (split-K) so that
// one canvas still fills the GPU; the CTAs of one split are adjacent in launch order (n tile
// fastest, then m tile), so the slab of E they share and the rows of P_hat each n tile
// re-reads are served from L2.
#include "kernels.cuh"
#include "sm103.cuh"

namespace dg {
namespace {

constexpr int kScBM = 128;
constexpr int kScBN = 256;
constexpr int kScBK = 64;
constexpr int kScStages = 4;
constexpr int kScABytes = kScBM * kScBK * 2;          // 16 KiB
constexpr int kScBChunk = kScBK * 64 * 2;             // 64 vocab rows x 64 columns: 8 KiB
constexpr int kScBBytes = kScBChunk * (kScBN / 64);   // 32 KiB
constexpr int kScStageBytes = kScABytes + kScBBytes;
constexpr int kScBarOff = kScStages * kScStageBytes;
constexpr int kScSmemBytes = kScBarOff + 256 + 1024;
static_assert(kScStageBytes % 1024 == 0, "stages must keep the 1 KiB swizzle alignment");
constexpr float kScLog2e = 1.4426950408889634f;

struct ScGemmParams {
  int R, d, V, nkb, per;
  const float* m_ref;  // [R, V / 32]
  const float* lse;    // [R]
  float* part;         // [S, R, d]
  uint32_t* status;
  const int* n_active;
  uint64_t wait_ns;  // limit of every on-chip wait
};

__global__ void __launch_bounds__(192, 1)
    sc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   ScGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kScBarOff);
  uint64_t* empty = full + kScStages;
  uint64_t* scaled = empty + kScStages;  // [kScStages]: A slot in TMEM written, MMA may read
  uint64_t* acc_full = scaled + kScStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kScBN;
  const int m0 = blockIdx.y * kScBM;
  const int kb0 = blockIdx.z * p.per;
  const int kb1 = min(kb0 + p.per, p.nkb);  // the plan leaves no split empty

  // Before the wait for the previous kernel (the finalisation, which writes lse): the barriers
  // and the first stages' copies.  P~ and m_ref come from the vocabulary pass before it, which
  // has completed once this kernel can start; E is the model's.  Thread 0 is the producer.
  const uint64_t stream_once = l2_policy_evict_first();
  auto load_stage = [&](int s, int kb) {
    uint8_t* sa = smem + s * kScStageBytes;
    mbar_arrive_expect_tx(&full[s], kScStageBytes);
    tma_load_2d(sa, &tmA, &full[s], kb * kScBK, m0);
#pragma unroll
    for (int c = 0; c < kScBN / 64; ++c)
      tma_load_2d_hint(sa + kScABytes + c * kScBChunk, &tmB, &full[s], n0 + c * 64, kb * kScBK,
                       stream_once);
  };
  int pre = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&scaled[s], 4);  // one arrival per transform warp
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    for (; pre < kScStages && kb0 + pre < kb1; ++pre) load_stage(pre, kb0 + pre);
  }
  pdl_wait();
  if (p.n_active && *p.n_active == 0) {  // the same for every CTA of the grid
    if (threadIdx.x == 0)  // let the started copies land before the CTA leaves
      for (int s = 0; s < pre; ++s) mbar_wait_drain(&full[s], 0);
    return;
  }
  pdl_trigger();  // the next kernel's CTAs may start their own prologue on idle SMs
  // TMEM: the fp32 accumulator in columns [0, 256); the normalised A operand in a ring of
  // kScStages slots of 32 columns (64 bf16 per lane) from column 256.
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued = pre;  // the first stages were started before the wait
      for (int kb = kb0 + pre; kb < kb1; ++kb, ++issued) {
        const int s = issued % kScStages;
        const uint32_t r = issued / kScStages;
        if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, p.wait_ns)) break;
        load_stage(s, kb);
      }
      if (*abort_flag) {  // let copies already in flight land before the CTA exits
        for (int q = (issued > kScStages ? issued - kScStages : 0); q < issued; ++q)
          mbar_wait_drain(&full[q % kScStages], (q / kScStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kScBM, kScBN, true);
      int q = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++q) {
        const int s = q % kScStages;
        if (!mbar_wait(&scaled[s], (q / kScStages) & 1, abort_flag, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t sb = smem_u32(smem + s * kScStageBytes) + kScABytes;
        const uint32_t ta = tmem + kScBN + s * 32;
#pragma unroll
        for (int k = 0; k < kScBK / 16; ++k)
          mma_bf16_ts(tmem, ta + k * 8, sdesc_sw128(sb + k * 2048, kScBChunk, 1024), idesc,
                      (q | k) != 0);
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);
      if (*abort_flag) mbar_wait_drain(acc_full, 0);
    }
  } else {
    // Normalise each A stage: row r's 64 entries (128 bytes in shared memory, its eight
    // 16-byte chunks permuted by the 128-byte swizzle: logical chunk j sits at j ^ (r & 7))
    // times exp(m_ref - lse) of their 32-entry chunk, packed in k order into this lane's slot
    // of the TMEM ring.  The reference maxima are fetched one k-block ahead.
    const int r_in = (warp & 3) * 32 + lane;
    const int row = m0 + r_in;
    const bool live = row < p.R;  // rows past the end are zero-filled by TMA; scaled by 0
    const float lse = live ? p.lse[row] : 0.f;
    const float* mrow = p.m_ref + static_cast<int64_t>(live ? row : 0) * (p.V / 32);
    const uint32_t sw = static_cast<uint32_t>(r_in & 7);
    const uint32_t lane_base = tmem_lane_base(warp);
    bool ok = true;
    float2 mr_next = live ? *reinterpret_cast<const float2*>(mrow + kb0 * 2) : make_float2(0, 0);
    int q = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++q) {
      const int s = q % kScStages;
      const float2 mr = mr_next;
      if (live && kb + 1 < kb1) mr_next = *reinterpret_cast<const float2*>(mrow + kb * 2 + 2);
      if (ok) ok = warp_wait(&full[s], (q / kScStages) & 1, abort_flag, p.wait_ns);
      if (ok) {
        const float c0 = live ? ex2_approx((mr.x - lse) * kScLog2e) : 0.f;
        const float c1 = live ? ex2_approx((mr.y - lse) * kScLog2e) : 0.f;
        const uint4* rowp = reinterpret_cast<const uint4*>(
            smem + s * kScStageBytes + (r_in >> 3) * 1024 + (r_in & 7) * 128);
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float c = j < 4 ? c0 : c1;
          const uint4 w = rowp[j ^ sw];
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
            pk[j * 4 + e] = pack_bf16x2(x.x * c, x.y * c);
          }
        }
        tmem_st32(tmem + lane_base + kScBN + s * 32, pk);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&scaled[s]);
    }
    ok = ok && warp_wait(acc_full, 0, abort_flag, p.wait_ns);
    tc_fence_after();
    float* dst = p.part + (static_cast<int64_t>(blockIdx.z) * p.R + row) * p.d + n0;
    // one thread per row: 32-byte stores write whole L2 sectors when the base allows them
    const bool v8 = (reinterpret_cast<uintptr_t>(p.part) & 31) == 0;
#pragma unroll 1
    for (int c = 0; c < kScBN / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + tmem_lane_base(warp) + c * 32, v);
      if (!ok || row >= p.R) continue;
      if (v8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(v[q * 8 + e]);
          st_global_v8(dst + c * 32 + q * 8, w);
        }
      } else {
        float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          d4[q] = make_float4(v[q * 4], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
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

// e = bf16(sum_z part[z]) with the splits added in order (deterministic).
__global__ void sc_reduce_kernel(const float4* __restrict__ part, uint2* __restrict__ e, int S,
                                 int64_t n4, const int* n_active) {
  pdl_wait();
  pdl_trigger();
  if (n_active && *n_active == 0) return;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = part[i];
    for (int z = 1; z < S; ++z) {
      const float4 b = part[z * n4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    e[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
  }
}

int stream_grid(int64_t items, int threads) {
  const int64_t want = (items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

ScPlan plan_selfcond(int R, int V, int d) {
  ScPlan pl;
  pl.mt = (R + kScBM - 1) / kScBM;
  pl.nt = d / kScBN;
  pl.nkb = V / kScBK;
  const int64_t tiles = static_cast<int64_t>(pl.mt) * pl.nt;
  const int sms = num_sms();
  // Splits of the vocabulary: minimise (waves x k-blocks per split) plus the partial-sum
  // traffic (each split writes and re-reads R x d fp32 values: about the time of 12 k-blocks
  // of one tile per 1 MiB per SM, counted crudely as S / 4 here).
  int best_per = pl.nkb;
  double best_cost = -1.0;
  for (int S = 1; S <= pl.nkb && S <= 256; ++S) {
    const int per = (pl.nkb + S - 1) / S;
    const int Sx = (pl.nkb + per - 1) / per;  // splits actually used (none empty)
    if (Sx != S) continue;
    const int64_t waves = (tiles * S + sms - 1) / sms;
    const double cost = static_cast<double>(waves * per) + S / 4.0;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_per = per;
    }
  }
  pl.per = best_per;
  pl.S = (pl.nkb + best_per - 1) / best_per;
  pl.part_bytes = static_cast<size_t>(pl.S) * R * d * sizeof(float);
  return pl;
}

cudaError_t launch_self_condition(const uint16_t* p_til, const float* m_ref, const float* lse,
                                  const uint16_t* E, const uint16_t* W1, const uint16_t* W2,
                                  int R, int V, int d, int dsc, float* part, uint16_t* e,
                                  uint16_t* u, uint16_t* s, uint32_t* status,
                                  const int* n_active, cudaStream_t st) {
  if (d % kScBN != 0 || V % kScBK != 0 || V % 32 != 0 || dsc % 64 != 0)
    return cudaErrorInvalidValue;
  const ScPlan pl = plan_selfcond(R, V, d);
  CUtensorMap ta, tb;
  const uint64_t dA[2] = {static_cast<uint64_t>(V), static_cast<uint64_t>(R)};
  const uint64_t sA[1] = {static_cast<uint64_t>(V) * 2};
  const uint32_t bA[2] = {static_cast<uint32_t>(kScBK), static_cast<uint32_t>(kScBM)};
  const uint64_t dB[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(V)};
  const uint64_t sB[1] = {static_cast<uint64_t>(d) * 2};
  const uint32_t bB[2] = {64u, static_cast<uint32_t>(kScBK)};
  if (!make_tmap_bf16(&ta, p_til, 2, dA, sA, bA)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, E, 2, dB, sB, bB)) return cudaErrorInvalidValue;
  static int configured_device = -1;
  const int dev = device_id();
  if (configured_device != dev) {
    const cudaError_t err = cudaFuncSetAttribute(
        sc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScSmemBytes);
    if (err != cudaSuccess) return err;
    configured_device = dev;
  }
  ScGemmParams gp;
  gp.R = R;
  gp.d = d;
  gp.V = V;
  gp.m_ref = m_ref;
  gp.lse = lse;
  gp.nkb = pl.nkb;
  gp.per = pl.per;
  gp.part = part;
  gp.status = status;
  gp.n_active = n_active;
  gp.wait_ns = wait_limit_ns();
  timer_begin(2, st);
  cudaError_t err = launch_dependent(sc_gemm_kernel, dim3(pl.nt, pl.mt, pl.S), dim3(192),
                                     kScSmemBytes, st, ta, tb, gp);
  timer_end(2, st);
  if (err != cudaSuccess) return err;
  {
    const int64_t n4 = static_cast<int64_t>(R) * d / 4;
    err = launch_dependent(sc_reduce_kernel, dim3(stream_grid(n4, 256)), dim3(256), 0, st,
                           reinterpret_cast<const float4*>(part), reinterpret_cast<uint2*>(e),
                           pl.S, n4, n_active);
    if (err != cudaSuccess) return err;
  }
  GemmOut o1{};
  o1.nseg = 1;
  o1.seg_begin[0] = 0;
  o1.seg_begin[1] = dsc;
  o1.ptr[0] = u;
  o1.ld[0] = dsc;
  // the contraction's partials are consumed: their buffer takes the GEMMs' split partials
  err = launch_gemm(e, W1, R, dsc, d, o1, nullptr, 0, status, n_active, st, kActGeluTanh, part,
                    pl.part_bytes);
  if (err != cudaSuccess) return err;
  GemmOut o2{};
  o2.nseg = 1;
  o2.seg_begin[0] = 0;
  o2.seg_begin[1] = d;
  o2.ptr[0] = s;
  o2.ld[0] = d;
  return launch_gemm(u, W2, R, d, dsc, o2, nullptr, 0, status, n_active, st, kActNone, part,
                     pl.part_bytes);
}

}  // namespace dg
