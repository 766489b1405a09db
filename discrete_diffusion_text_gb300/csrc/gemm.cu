// Projection GEMM of the stand-in decoder on the 5th-generation tensor cores:
//   C[M, N] = A[M, K] W[N, K]^T (+ residual), bf16 in, fp32 accumulate in tensor memory,
//   bf16 out.
// Warp 0 streams A/W k-blocks with TMA into a shared-memory ring (128-byte swizzle); one
// thread of warp 1 issues tcgen05.mma (M = 128, N = BN, K = 16 per instruction) into a TMEM
// accumulator; warps 2..5 read the accumulator back with tcgen05.ld.  The W halves of the
// first stages are requested before the wait for the previous kernel (gemm_start): the weights
// are never written by the stream's kernels, only A (the activations) has to wait.
//
// Two kernels share that main loop:
//  * gemm_bf16_kernel: one 128 x BN output tile per CTA over the whole K (many tiles: a
//    canvas batch);
//  * gemm_splitk_kernel: one tile per cluster of S CTAs, each CTA taking 1/S of the K range
//    (few tiles: one canvas).  The issuing thread is held about as long in one tcgen05.mma
//    for N = 64 as for N = 256 (where a single issuer keeps the pipe busy), so with few tiles
//    the per-CTA chain of K/16 instructions, not bandwidth, sets the time; splitting K
//    shortens it.  CTA q of the cluster owns rows [q 128/S, (q+1) 128/S) of the
//    tile: it keeps its own partial of those rows in shared memory, writes the other rows'
//    partials to an fp32 workspace, and after a cluster barrier sums the S partials of its
//    rows in rank order (deterministic), adds the residual and writes bf16.
#include <mutex>
#include <vector>

#include "kernels.cuh"
#include "sm103.cuh"

namespace dg {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreadsG = 192;  // TMA warp, MMA warp, four epilogue warps

struct GemmParams {
  int M, N, K;
  GemmOut out;
  const uint16_t* residual;
  int ld_res;
  uint32_t* status;
  const int* n_active;
  int act;  // kActNone or kActGeluTanh, applied after the residual
  uint64_t wait_ns;  // limit of every on-chip wait
};

// GELU, tanh form: x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
__device__ __forceinline__ float gelu_tanh(float x) {
  const float k = 0.7978845608028654f;
  return 0.5f * x * (1.f + tanhf(k * fmaf(0.044715f * x, x * x, x)));
}

// As many pipeline stages as fit in ~192 KiB.
template <int BN>
struct GemmLayout {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (192 * 1024) / kStageBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + 1 KiB alignment slack
};

// Destination of the output columns starting at col (a tile never straddles two segments).
struct SegDst {
  uint16_t* base;
  int ld, beg;
};
__device__ __forceinline__ SegDst segment_of(const GemmOut& out, int col) {
  // static indices only: no local-memory copy of the parameters
  SegDst d{out.ptr[0], out.ld[0], out.seg_begin[0]};
  if (out.nseg > 1 && col >= out.seg_begin[1]) d = SegDst{out.ptr[1], out.ld[1], out.seg_begin[1]};
  if (out.nseg > 2 && col >= out.seg_begin[2]) d = SegDst{out.ptr[2], out.ld[2], out.seg_begin[2]};
  return d;
}

// Producer (one thread), before the previous kernel's writes are visible: the W halves (the
// weights, which no kernel of the stream writes) of the first stages, each stage's barrier
// armed for the whole stage.  Returns the number of stages started.
template <int BN>
__device__ __forceinline__ int gemm_prefetch_w(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                               uint8_t* smem, uint64_t* full, int kb0, int nk,
                                               int n0) {
  using Lay = GemmLayout<BN>;
  tma_prefetch_map(tmA);
  tma_prefetch_map(tmB);
  const int n = nk < Lay::kStages ? nk : Lay::kStages;
  for (int i = 0; i < n; ++i) {
    mbar_arrive_expect_tx(&full[i], Lay::kStageBytes);
    tma_load_2d(smem + i * Lay::kStageBytes + Lay::kABytes, tmB, &full[i], (kb0 + i) * kBK, n0);
  }
  return n;
}

// Producer (one thread): k-blocks kb0 .. kb0 + nk - 1 of A rows m0.. and W rows n0.. into the
// ring; the first `pre` stages already hold their W copies (gemm_prefetch_w) and get A only.
// After an abort it waits (briefly) for the copies already in flight to land.
template <int BN>
__device__ __forceinline__ void gemm_produce(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                             uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             int kb0, int nk, int m0, int n0, int pre,
                                             volatile int* abort_flag, uint64_t wait_ns) {
  using Lay = GemmLayout<BN>;
  int issued = 0;
  for (int i = 0; i < nk; ++i) {
    const int s = i % Lay::kStages;
    const uint32_t r = i / Lay::kStages;
    uint8_t* sa = smem + s * Lay::kStageBytes;
    if (i < pre) {
      tma_load_2d(sa, tmA, &full[s], (kb0 + i) * kBK, m0);
      ++issued;
      continue;
    }
    if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, wait_ns)) break;
    mbar_arrive_expect_tx(&full[s], Lay::kStageBytes);
    tma_load_2d(sa, tmA, &full[s], (kb0 + i) * kBK, m0);
    tma_load_2d(sa + Lay::kABytes, tmB, &full[s], (kb0 + i) * kBK, n0);
    ++issued;
  }
  if (*abort_flag) {
    for (int i = (issued > Lay::kStages ? issued - Lay::kStages : 0); i < issued; ++i)
      mbar_wait_drain(&full[i % Lay::kStages], (i / Lay::kStages) & 1);
  }
}

// MMA issuer (one thread): nk k-blocks into the accumulator, then one arrival on acc_full.
template <int BN>
__device__ __forceinline__ void gemm_mma(uint32_t tmem, uint8_t* smem, uint64_t* full,
                                         uint64_t* empty, uint64_t* acc_full, int nk,
                                         volatile int* abort_flag, uint64_t wait_ns) {
  using Lay = GemmLayout<BN>;
  constexpr uint32_t idesc = idesc_bf16(kBM, BN, false);
  for (int i = 0; i < nk; ++i) {
    const int s = i % Lay::kStages;
    const uint32_t r = i / Lay::kStages;
    if (!mbar_wait(&full[s], r & 1, abort_flag, wait_ns)) break;
    tc_fence_after();
    const uint32_t sa = smem_u32(smem + s * Lay::kStageBytes);
    const uint32_t sb = sa + Lay::kABytes;
#pragma unroll
    for (int k = 0; k < kBK / 16; ++k)
      mma_bf16_ss(tmem, sdesc_sw128(sa + k * 32, 16, 1024), sdesc_sw128(sb + k * 32, 16, 1024),
                  idesc, (i | k) != 0);
    mma_commit(&empty[s]);
  }
  mma_commit(acc_full);
  if (*abort_flag) mbar_wait_drain(acc_full, 0);
}

// Barriers and flags after the data region: full[kStages], empty[kStages], acc_full, the TMEM
// base address and the abort flag.
struct GemmSync {
  uint64_t *full, *empty, *acc_full;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};
template <int kStages>
__device__ __forceinline__ GemmSync gemm_sync_at(uint8_t* p) {
  GemmSync g;
  g.full = reinterpret_cast<uint64_t*>(p);
  g.empty = g.full + kStages;
  g.acc_full = g.empty + kStages;
  g.tmem_slot = reinterpret_cast<uint32_t*>(g.acc_full + 1);
  g.abort_flag = reinterpret_cast<volatile int*>(g.tmem_slot + 1);
  return g;
}

// The start of both GEMM kernels, up to the tensor-memory allocation: barriers initialised,
// the weight copies of the first stages started, then the wait for the previous kernel in the
// stream (everything before it touches no memory that kernel writes).  Returns false when the
// denoising loop has no active canvas left: the CTA then only lets its weight copies land and
// leaves (every thread returns).
template <int BN>
__device__ __forceinline__ bool gemm_start(const GemmSync& g, const CUtensorMap* tmA,
                                           const CUtensorMap* tmB, uint8_t* smem, int kb0, int nk,
                                           int m0, int n0, const int* n_active, int& pre) {
  using Lay = GemmLayout<BN>;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Lay::kStages; ++s) {
      mbar_init(&g.full[s], 1);
      mbar_init(&g.empty[s], 1);
    }
    mbar_init(g.acc_full, 1);
    *g.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pre = 0;
  if (threadIdx.x == 0) pre = gemm_prefetch_w<BN>(tmA, tmB, smem, g.full, kb0, nk, n0);
  pdl_wait();
  if (n_active && *n_active == 0) {  // the same for every CTA of the grid
    if (threadIdx.x == 0) {  // complete the started stages (A is readable), let them land
      for (int i = 0; i < pre; ++i) {
        tma_load_2d(smem + i * Lay::kStageBytes, tmA, &g.full[i], (kb0 + i) * kBK, m0);
        mbar_wait_drain(&g.full[i], 0);
      }
    }
    return false;
  }
  if ((threadIdx.x >> 5) == 1) {
    tmem_alloc(g.tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return true;
}

template <int BN>
__global__ void __launch_bounds__(kThreadsG, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, GemmParams p) {
  using Lay = GemmLayout<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const GemmSync g = gemm_sync_at<Lay::kStages>(smem + Lay::kBarOff);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * kBM;
  int pre;
  if (!gemm_start<BN>(g, &tmA, &tmB, smem, 0, p.K / kBK, m0, n0, p.n_active, pre)) return;
  pdl_trigger();  // the next kernel's CTAs may start their own prologue on idle SMs
  const uint32_t tmem = *g.tmem_slot;

  if (warp == 0) {
    if (lane == 0)
      gemm_produce<BN>(&tmA, &tmB, smem, g.full, g.empty, 0, p.K / kBK, m0, n0, pre,
                       g.abort_flag, p.wait_ns);
  } else if (warp == 1) {
    if (lane == 0) gemm_mma<BN>(tmem, smem, g.full, g.empty, g.acc_full, p.K / kBK, g.abort_flag,
                                    p.wait_ns);
  } else {
    const bool ok = warp_wait(g.acc_full, 0, g.abort_flag, p.wait_ns);
    tc_fence_after();
    const int row = m0 + (warp & 3) * 32 + lane;
    const SegDst dst = segment_of(p.out, n0);
    // one thread per row: 32-byte stores write whole L2 sectors (rows lie ld apart) when the
    // segment's base and row pitch allow them
    const bool v8 = (reinterpret_cast<uintptr_t>(dst.base) & 31) == 0 && (dst.ld & 15) == 0;
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
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
            v[q * 8 + 2 * e] += f.x;
            v[q * 8 + 2 * e + 1] += f.y;
          }
        }
      }
      if (p.act == kActGeluTanh) {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = gelu_tanh(v[e]);
      }
      uint16_t* d = dst.base + static_cast<int64_t>(row) * dst.ld + (col - dst.beg);
      uint32_t pk[2][8];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e >> 3][e & 7] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
      if (v8) {
        st_global_v8(d, pk[0]);
        st_global_v8(d + 16, pk[1]);
      } else {
        uint4* d4 = reinterpret_cast<uint4*>(d);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          d4[q] = make_uint4(pk[q >> 1][4 * (q & 1)], pk[q >> 1][4 * (q & 1) + 1],
                             pk[q >> 1][4 * (q & 1) + 2], pk[q >> 1][4 * (q & 1) + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
  if (threadIdx.x == 0 && *g.abort_flag) atomicOr(p.status, kStatusTimeout);
}

// Split-K layout: the ring as above; once the main loop is done the ring's memory holds this
// CTA's own rows ([kR][BN] fp32, 16-byte chunks XOR-swizzled by row so that the row-per-thread
// writes and the column-per-thread reads are both free of bank conflicts) and the fp32 sums of
// those rows ([kR][BN + 4], padded for the same reason).
template <int BN, int S>
struct SplitLayout {
  using Ring = GemmLayout<BN>;
  static constexpr int kR = kBM / S;  // rows of the tile summed by one CTA
  static constexpr int kOwnOff = 0;
  static constexpr int kOwnBytes = kR * BN * 4;
  static constexpr int kSumLd = BN + 4;
  static constexpr int kSumOff = kOwnBytes;
  static constexpr int kSumBytes = kR * kSumLd * 4;
  static_assert(kSumOff + kSumBytes <= Ring::kRingBytes, "split-K scratch exceeds the ring");
};

// grid (S, N / BN, M tiles), cluster (S, 1, 1); part: [tiles][S][BN / 4][128] float4.
template <int BN, int S>
__global__ void __launch_bounds__(kThreadsG, 1)
    gemm_splitk_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, GemmParams p,
                       float4* __restrict__ part) {
  using Lay = SplitLayout<BN, S>;
  using Ring = GemmLayout<BN>;
  constexpr int c4n = BN / 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const GemmSync g = gemm_sync_at<Ring::kStages>(smem + Ring::kBarOff);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q = static_cast<int>(cluster_ctarank());
  const int n0 = blockIdx.y * BN;
  const int m0 = blockIdx.z * kBM;
  const int nkb = p.K / kBK;
  const int kb0 = q * nkb / S;
  const int nk = (q + 1) * nkb / S - kb0;
  float4* tile_part =
      part + static_cast<int64_t>(blockIdx.z * gridDim.y + blockIdx.y) * S * c4n * kBM;
  int pre;
  // n_active is the same for every CTA of the grid, so a cluster leaves (or stays) whole
  if (!gemm_start<BN>(g, &tmA, &tmB, smem, kb0, nk, m0, n0, p.n_active, pre)) return;
  pdl_trigger();  // the next kernel's CTAs may start their own prologue on idle SMs
  const uint32_t tmem = *g.tmem_slot;

  if (warp == 0) {
    if (lane == 0)
      gemm_produce<BN>(&tmA, &tmB, smem, g.full, g.empty, kb0, nk, m0, n0, pre, g.abort_flag,
                       p.wait_ns);
  } else if (warp == 1) {
    if (lane == 0) gemm_mma<BN>(tmem, smem, g.full, g.empty, g.acc_full, nk, g.abort_flag, p.wait_ns);
  } else {
    // partial accumulator: own rows to shared memory, the others to the workspace in a
    // [chunk][row] layout so that a warp's 32 rows of one 16-byte chunk are 512 contiguous
    // bytes (the ring is idle: every MMA that read it has completed)
    warp_wait(g.acc_full, 0, g.abort_flag, p.wait_ns);
    tc_fence_after();
    const int row = (warp & 3) * 32 + lane;
    const bool own = row / Lay::kR == q;
    float4* gp = tile_part + static_cast<int64_t>(q) * c4n * kBM + row;
    uint8_t* orow = smem + Lay::kOwnOff + (row - q * Lay::kR) * (BN * 4);
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      float v[64];
      tmem_ld64(tmem + tmem_lane_base(warp) + c * 64, v);
      if (own) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int ch = (c * 16 + j) ^ (row & 7);
          *reinterpret_cast<float4*>(orow + ch * 16) =
              make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          __stcg(gp + static_cast<int64_t>(c * 16 + j) * kBM,
                 make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
      }
    }
  }
  tc_fence_before();
  __syncwarp();
  cluster_arrive();  // this CTA's partials are written (and its TMEM reads are done)
  cluster_wait();    // ... and so are every other CTA's of the cluster
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }

  // this CTA's kR rows: the S partials summed in rank order (the same order for every row,
  // whichever CTA sums it), into fp32 sums in shared memory
  constexpr int nitems = Lay::kR * c4n;
  constexpr int kU = 4;  // items in flight per thread
  float* sums = reinterpret_cast<float*>(smem + Lay::kSumOff);
  for (int i0 = threadIdx.x; i0 < nitems; i0 += kU * kThreadsG) {
    float4 v[kU][S];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * kThreadsG < nitems ? i0 + u * kThreadsG : i0;
      const int rr = i % Lay::kR, c4 = i / Lay::kR;
      const int trow = q * Lay::kR + rr;
#pragma unroll
      for (int j = 0; j < S; ++j) {
        if (j == q)
          v[u][j] = *reinterpret_cast<const float4*>(smem + Lay::kOwnOff + rr * (BN * 4) +
                                                     ((c4 ^ (trow & 7)) * 16));
        else
          v[u][j] = __ldcg(tile_part + (static_cast<int64_t>(j) * c4n + c4) * kBM + trow);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * kThreadsG;
      if (i < nitems) {
        const int rr = i % Lay::kR, c4 = i / Lay::kR;
        float4 a = v[u][0];
#pragma unroll
        for (int j = 1; j < S; ++j) {
          a.x += v[u][j].x;
          a.y += v[u][j].y;
          a.z += v[u][j].z;
          a.w += v[u][j].w;
        }
        *reinterpret_cast<float4*>(sums + rr * Lay::kSumLd + c4 * 4) = a;
      }
    }
  }
  __syncthreads();

  // residual, activation, bf16: eight columns a thread, consecutive threads along a row
  const bool good = !*g.abort_flag;
  const SegDst dst = segment_of(p.out, n0);
  constexpr int c8n = BN / 8;
#pragma unroll 2
  for (int i = threadIdx.x; i < Lay::kR * c8n; i += kThreadsG) {
    const int rr = i / c8n, c8 = i % c8n;
    const int row = m0 + q * Lay::kR + rr;
    if (!good || row >= p.M) continue;
    const float4 s0 = *reinterpret_cast<const float4*>(sums + rr * Lay::kSumLd + c8 * 8);
    const float4 s1 = *reinterpret_cast<const float4*>(sums + rr * Lay::kSumLd + c8 * 8 + 4);
    float o[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const int col = n0 + c8 * 8;
    if (p.residual) {
      const uint4 rv =
          *reinterpret_cast<const uint4*>(p.residual + static_cast<int64_t>(row) * p.ld_res + col);
      const uint32_t w[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
        o[2 * e] += f.x;
        o[2 * e + 1] += f.y;
      }
    }
    if (p.act == kActGeluTanh) {
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = gelu_tanh(o[e]);
    }
    *reinterpret_cast<uint4*>(dst.base + static_cast<int64_t>(row) * dst.ld + (col - dst.beg)) =
        make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                   pack_bf16x2(o[6], o[7]));
  }
  if (threadIdx.x == 0 && *g.abort_flag) atomicOr(p.status, kStatusTimeout);
}

template <typename Kernel>
cudaError_t set_smem_once(Kernel kernel, int bytes, int* configured_device) {
  const int dev = device_id();
  if (*configured_device == dev) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) *configured_device = dev;
  return e;
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                      cudaStream_t st) {
  using Lay = GemmLayout<BN>;
  static int configured_device = -1;  // the attribute is per device; set on first use of each
  cudaError_t e = set_smem_once(gemm_bf16_kernel<BN>, Lay::kSmemBytes, &configured_device);
  if (e != cudaSuccess) return e;
  dim3 grid(p.N / BN, (p.M + kBM - 1) / kBM);
  return launch_dependent(gemm_bf16_kernel<BN>, grid, dim3(kThreadsG), Lay::kSmemBytes, st, ta,
                          tb, p);
}

template <int BN, int S>
cudaError_t launch_split(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                         float* part, cudaStream_t st) {
  using Lay = GemmLayout<BN>;
  static int configured_device = -1;
  cudaError_t e =
      set_smem_once(gemm_splitk_kernel<BN, S>, Lay::kSmemBytes, &configured_device);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(S, p.N / BN, (p.M + kBM - 1) / kBM);
  cfg.blockDim = dim3(kThreadsG);
  cfg.dynamicSmemBytes = Lay::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_splitk_kernel<BN, S>, ta, tb, p,
                            reinterpret_cast<float4*>(part));
}

// Whether a cluster of S split-K CTAs (each with the whole ring of shared memory) can be
// resident on this device at all (a partitioned GPU may not offer it); asked once per device.
template <int BN, int S>
bool split_cluster_fits() {
  static std::mutex mu;
  static std::vector<int> known;  // per device: 0 unknown, 1 fits, 2 does not
  const int dev = device_id();
  std::lock_guard<std::mutex> lk(mu);
  if (static_cast<int>(known.size()) <= dev) known.resize(dev + 1, 0);
  if (known[dev] == 0) {
    using Lay = GemmLayout<BN>;
    int n = 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3(kThreadsG);
    cfg.dynamicSmemBytes = Lay::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool ok =
        cudaFuncSetAttribute(gemm_splitk_kernel<BN, S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay::kSmemBytes) == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&n, gemm_splitk_kernel<BN, S>, &cfg) == cudaSuccess &&
        n > 0;
    if (!ok) cudaGetLastError();  // clear the query's error, if any
    known[dev] = ok ? 1 : 2;
  }
  return known[dev] == 1;
}

bool split_fits(int bn, int s) {
  if (bn == 256) return s == 4 ? split_cluster_fits<256, 4>() : split_cluster_fits<256, 2>();
  return s == 4 ? split_cluster_fits<128, 4>() : split_cluster_fits<128, 2>();
}

bool divides_segments(const GemmOut& out, int N, int bn) {
  if (N % bn != 0) return false;
  for (int s = 0; s <= out.nseg; ++s)
    if (out.seg_begin[s] % bn != 0) return false;
  return true;
}

}  // namespace

namespace {
GemmPlan plan_gemm_impl(int M, int N, int K, const GemmOut& out, bool allow_split) {
  // Cost in units of one k-block of one CTA (~0.3 us): the issuing thread spends about the
  // same time on an MMA whatever N <= 256, so a CTA's time is its k-block count whatever the
  // tile width, and the cost is waves x k-blocks per CTA (one CTA per SM: the ring fills its
  // shared memory).  A K split adds the write-out and sum of its fp32 partials: measured
  // ~10 k-blocks per 96 KiB a CTA writes ((S - 1)/S of its 128 x BN partial).  Ties: more
  // CTAs (the narrower tiles' smaller epilogues and spread loads measured slightly faster).
  GemmPlan pl{};
  pl.BN = 64;
  pl.S = 1;
  const int mt = (M + kBM - 1) / kBM;
  const int nkb = K / kBK;
  const int64_t nsm = num_sms();
  if (mt <= 0 || nkb <= 0) return pl;
  double best = -1.0;
  int64_t best_ctas = 0;
  for (int bn : {256, 128, 64}) {
    if (!divides_segments(out, N, bn)) continue;
    for (int s : {1, 2, 4}) {
      if (s > 1 && (!allow_split || bn == 64 || s > nkb || !split_fits(bn, s))) continue;
      const int64_t ctas = static_cast<int64_t>(mt) * (N / bn) * s;
      const int64_t waves = (ctas + nsm - 1) / nsm;
      const double written_kib = (s - 1) * (kBM / s) * bn * 4 / 1024.0;
      const double cost = static_cast<double>(waves) * ((nkb + s - 1) / s + written_kib / 9.6);
      if (best < 0 || cost < best - 1e-9 || (cost < best + 1e-9 && ctas > best_ctas)) {
        best = cost;
        best_ctas = ctas;
        pl.BN = bn;
        pl.S = s;
      }
    }
  }
  pl.part_bytes =
      pl.S > 1 ? static_cast<size_t>(mt) * (N / pl.BN) * pl.S * kBM * pl.BN * 4 : 0;
  return pl;
}
}  // namespace

GemmPlan plan_gemm(int M, int N, int K, const GemmOut& out) {
  return plan_gemm_impl(M, N, K, out, true);
}

cudaError_t launch_gemm(const uint16_t* A, const uint16_t* W, int M, int N, int K,
                        const GemmOut& out, const uint16_t* residual, int ld_res,
                        uint32_t* status, const int* n_active, cudaStream_t st, int act,
                        void* part_ws, size_t part_ws_bytes) {
  if (N % 64 != 0 || K % kBK != 0) return cudaErrorInvalidValue;
  for (int s = 0; s <= out.nseg; ++s)
    if (out.seg_begin[s] % 64 != 0) return cudaErrorInvalidValue;
  GemmPlan pl = plan_gemm(M, N, K, out);
  if (pl.S > 1 && (part_ws == nullptr || part_ws_bytes < pl.part_bytes ||
                   (reinterpret_cast<uintptr_t>(part_ws) & 15) != 0)) {
    // no room for the split partials: one CTA per tile over the whole K
    pl = plan_gemm_impl(M, N, K, out, false);
  }

  CUtensorMap ta, tb;
  const uint64_t dA[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint64_t sA[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t bA[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(kBM)};
  const uint64_t dB[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
  const uint32_t bB[2] = {static_cast<uint32_t>(kBK), static_cast<uint32_t>(pl.BN)};
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
  p.wait_ns = wait_limit_ns();
  p.act = act;
  float* part = static_cast<float*>(part_ws);
  timer_begin(3, st);
  cudaError_t e;
  switch (pl.S * 1000 + pl.BN) {
    case 4256: e = launch_split<256, 4>(ta, tb, p, part, st); break;
    case 2256: e = launch_split<256, 2>(ta, tb, p, part, st); break;
    case 4128: e = launch_split<128, 4>(ta, tb, p, part, st); break;
    case 2128: e = launch_split<128, 2>(ta, tb, p, part, st); break;
    case 1256: e = launch_bn<256>(ta, tb, p, st); break;
    case 1128: e = launch_bn<128>(ta, tb, p, st); break;
    default: e = launch_bn<64>(ta, tb, p, st); break;
  }
  timer_end(3, st);
  return e;
}

}  // namespace dg
