// Projection GEMM of the stand-in decoder on the 5th-generation tensor cores:
//   C[M, N] = A[M, K] W[N, K]^T (+ residual), bf16 in, fp32 accumulate in tensor memory,
//   bf16 out.
// One 128 x BN output tile per CTA.  Warp 0 streams A/W k-blocks with TMA into a 4-stage
// shared-memory ring (128-byte swizzle); one thread of warp 1 issues tcgen05.mma
// (M = 128, N = BN, K = 16 per instruction) into a TMEM accumulator; warps 2..5 read the
// accumulator back with tcgen05.ld and write bf16 rows.
#include "kernels.cuh"
#include "sm103.cuh"

namespace dg {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;

struct GemmParams {
  int M, N, K;
  GemmOut out;
  const uint16_t* residual;
  int ld_res;
  uint32_t* status;
  const int* n_active;
  int act;  // kActNone or kActGeluTanh, applied after the residual
};

// GELU, tanh form: x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
__device__ __forceinline__ float gelu_tanh(float x) {
  const float k = 0.7978845608028654f;
  return 0.5f * x * (1.f + tanhf(k * fmaf(0.044715f * x, x * x, x)));
}

// As many pipeline stages as fit in ~192 KiB: with one or two waves of CTAs that each run a
// few dozen k-blocks, the copies in flight per SM (not the MMA) set the GEMM's speed.
template <int BN>
struct GemmLayout {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (192 * 1024) / kStageBytes;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + 1 KiB alignment slack
};

template <int BN>
__global__ void __launch_bounds__(192, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, GemmParams p) {
  using Lay = GemmLayout<BN>;
  pdl_wait();
  if (p.n_active && *p.n_active == 0) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* empty = full + Lay::kStages;
  uint64_t* acc_full = empty + Lay::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * kBM;
  const int nkb = p.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Lay::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&tmA);
      tma_prefetch_map(&tmB);
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % Lay::kStages;
        const uint32_t r = kb / Lay::kStages;
        if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag)) break;
        uint8_t* sa = smem + s * Lay::kStageBytes;
        mbar_arrive_expect_tx(&full[s], Lay::kStageBytes);
        tma_load_2d(sa, &tmA, &full[s], kb * kBK, m0);
        tma_load_2d(sa + Lay::kABytes, &tmB, &full[s], kb * kBK, n0);
        ++issued;
      }
      if (*abort_flag) {  // let copies already in flight land before the CTA exits
        for (int kb = (issued > Lay::kStages ? issued - Lay::kStages : 0); kb < issued; ++kb)
          mbar_wait_drain(&full[kb % Lay::kStages], (kb / Lay::kStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, BN, false);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % Lay::kStages;
        const uint32_t r = kb / Lay::kStages;
        if (!mbar_wait(&full[s], r & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * Lay::kStageBytes);
        const uint32_t sb = sa + Lay::kABytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          mma_bf16_ss(tmem, sdesc_sw128(sa + k * 32, 16, 1024), sdesc_sw128(sb + k * 32, 16, 1024),
                      idesc, (kb | k) != 0);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);
      if (*abort_flag) mbar_wait_drain(acc_full, 0);
    }
  } else {
    const bool ok = warp_wait(acc_full, 0, abort_flag);
    tc_fence_after();
    const int row = m0 + (warp & 3) * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + tmem_lane_base(warp) + c * 32, v);
      if (!ok || row >= p.M) continue;
      const int col = n0 + c * 32;
      if (p.residual) {
        const uint4* rp = reinterpret_cast<const uint4*>(
            p.residual + static_cast<int64_t>(row) * p.ld_res + col);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = rp[q];
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&ws[e]);
            const float2 f = __bfloat1622float2(b2);
            v[q * 8 + 2 * e] += f.x;
            v[q * 8 + 2 * e + 1] += f.y;
          }
        }
      }
      if (p.act == kActGeluTanh) {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = gelu_tanh(v[e]);
      }
      // output segment of this column (static indices only: no local-memory copy of params)
      uint16_t* base = p.out.ptr[0];
      int ld = p.out.ld[0];
      int beg = p.out.seg_begin[0];
      if (p.out.nseg > 1 && col >= p.out.seg_begin[1]) {
        base = p.out.ptr[1];
        ld = p.out.ld[1];
        beg = p.out.seg_begin[1];
      }
      if (p.out.nseg > 2 && col >= p.out.seg_begin[2]) {
        base = p.out.ptr[2];
        ld = p.out.ld[2];
        beg = p.out.seg_begin[2];
      }
      uint16_t* dst = base + static_cast<int64_t>(row) * ld + (col - beg);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        d4[q] = make_uint4(pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]),
                           pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]),
                           pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]),
                           pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]));
      }
    }
  }

  // this CTA's work is done: the next kernel in the stream may be scheduled
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.status, kStatusTimeout);
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                      cudaStream_t st) {
  using Lay = GemmLayout<BN>;
  static int configured_device = -1;  // attribute is per device; set on first use of each
  const int dev = device_id();
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  dim3 grid(p.N / BN, (p.M + kBM - 1) / kBM);
  return launch_dependent(gemm_bf16_kernel<BN>, grid, dim3(192), Lay::kSmemBytes, st, ta, tb, p);
}

}  // namespace

cudaError_t launch_gemm(const uint16_t* A, const uint16_t* W, int M, int N, int K,
                        const GemmOut& out, const uint16_t* residual, int ld_res,
                        uint32_t* status, const int* n_active, cudaStream_t st, int act) {
  // Largest N tile that divides every output-segment boundary (a tile never straddles two
  // outputs) and still gives at least two CTAs per SM; 64 otherwise.
  if (N % 64 != 0 || K % kBK != 0) return cudaErrorInvalidValue;
  for (int s = 0; s <= out.nseg; ++s)
    if (out.seg_begin[s] % 64 != 0) return cudaErrorInvalidValue;
  const int mt = (M + kBM - 1) / kBM;
  auto fits = [&](int bn) {
    for (int s = 0; s <= out.nseg; ++s)
      if (out.seg_begin[s] % bn != 0) return false;
    return static_cast<int64_t>(mt) * (N / bn) >= 2 * num_sms();
  };
  int BN = 64;
  if (fits(256)) BN = 256;
  else if (fits(128)) BN = 128;

  CUtensorMap ta, tb;
  const uint64_t dA[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint64_t sA[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t bA[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kBM)};
  const uint64_t dB[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
  const uint32_t bB[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(BN)};
  if (!make_tmap_bf16(&ta, A, 2, dA, sA, bA)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb, W, 2, dB, sA, bB)) return cudaErrorInvalidValue;

  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.out = out;
  p.residual = residual;
  p.ld_res = ld_res;
  p.status = status;
  p.n_active = n_active;
  p.act = act;
  timer_begin(3, st);
  cudaError_t e;
  switch (BN) {
    case 256: e = launch_bn<256>(ta, tb, p, st); break;
    case 128: e = launch_bn<128>(ta, tb, p, st); break;
    default: e = launch_bn<64>(ta, tb, p, st); break;
  }
  timer_end(3, st);
  return e;
}

}  // namespace dg
