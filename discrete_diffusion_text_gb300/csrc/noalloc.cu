// Allocation-free entry point: dg_vocab_posterior_step_noalloc.
//
// Some callers cannot hand this library a workspace allocation.  A plugin or custom operator
// inside a host framework typically receives only its input and output buffers, with no
// handle to the framework's memory pool; a serving process may reserve its whole device
// budget up front, so an extra cudaMalloc fails or breaks the budget; and cudaMalloc /
// cudaFree can synchronise the device, which a latency-bound serving loop must not do.
// For such callers this variant of dg_vocab_posterior_step keeps its scratch (the
// per-canvas counters of the finalisation and the split-vocabulary partial tuples) in one
// file-scope device array of fixed size, and allocates nothing itself.
#include <cmath>
#include <mutex>
#include <string>
#include <vector>

#include "dg_common.cuh"
#include "kernels.cuh"

namespace dg {
namespace {

// 16 MiB, held by every GPU that loads the library until the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch for the current device, looked up once per device.
// (In host code the symbol is only a host-side stand-in, never a device address.)
bool scratch_address(unsigned char** out) {
  static std::mutex mu;
  static std::vector<unsigned char*> by_device;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (static_cast<int>(by_device.size()) <= dev) by_device.resize(dev + 1, nullptr);
  if (by_device[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return false;
    by_device[dev] = static_cast<unsigned char*>(p);
  }
  *out = by_device[dev];
  return true;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" dg_status dg_vocab_posterior_step_noalloc(
    const uint16_t* y, const uint16_t* W, int B, int L, int d, int V, float inv_tau,
    uint64_t seed, int step, const int32_t* x_in, int32_t* x_out, uint8_t* lock, uint8_t* jump,
    uint8_t* done, uint64_t jump_thr, float lock_logthr, const dg_posterior_out* out,
    void* stream) {
  if (B < 0 || L <= 0 || d <= 0 || V <= 0) return fail(DG_EINVAL, "vocab_posterior_noalloc: bad sizes");
  if (d % 64 != 0) return fail(DG_ENOTSUP, "vocab_posterior_noalloc: d must be a multiple of 64");
  if (V % 256 != 0) return fail(DG_ENOTSUP, "vocab_posterior_noalloc: V must be a multiple of 256");
  if (L > 256 || L % 64 != 0)
    return fail(DG_ENOTSUP, "vocab_posterior_noalloc: L must be 64..256, multiple of 64");
  if (step < 0 || step >= (1 << 24)) return fail(DG_EINVAL, "vocab_posterior_noalloc: step out of range");
  if (!(inv_tau > 0.f) || !std::isfinite(inv_tau))
    return fail(DG_EINVAL, "vocab_posterior_noalloc: bad inv_tau");
  if (jump_thr > (1ull << 32)) return fail(DG_EINVAL, "vocab_posterior_noalloc: jump_thr above 2^32");
  if (static_cast<int64_t>(B) * L >= (1ll << 31))
    return fail(DG_ENOTSUP, "vocab_posterior_noalloc: too many rows");
  if (B == 0) return DG_OK;
  if (y == nullptr || W == nullptr || !aligned16(y) || !aligned16(W))
    return fail(DG_EINVAL, "vocab_posterior_noalloc: NULL or misaligned y / W");
  if (x_in && !x_out) return fail(DG_EINVAL, "vocab_posterior_noalloc: x_out required with x_in");

  const VocabPlan vp = plan_vocab(B * L, V);
  const size_t counter_bytes = round256(2 * sizeof(int) * static_cast<size_t>(B));
  const size_t need = counter_bytes + vp.part_bytes;
  if (need > kNoAllocScratchBytes)
    return fail(DG_ENOTSUP, "vocab_posterior_noalloc: this size needs " + std::to_string(need) +
                                " bytes of scratch, above the fixed 16 MiB (use "
                                "dg_vocab_posterior_step with a workspace)");
  unsigned char* scratch = nullptr;
  if (!scratch_address(&scratch))
    return fail(DG_ECUDA, "vocab_posterior_noalloc: cannot resolve the scratch array's device address");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* counters = reinterpret_cast<int*>(scratch);
  VocabPart* parts = reinterpret_cast<VocabPart*>(scratch + counter_bytes);
  // The array keeps the previous call's contents: the finalisation counters must start at 0.
  cudaError_t e = cudaMemsetAsync(counters, 0, 2 * sizeof(int) * static_cast<size_t>(B), st);
  if (e != cudaSuccess) return cuda_fail(e, "vocab_posterior_noalloc: clearing counters");
  uint32_t* status = status_or_fallback(nullptr);
  e = launch_vocab_pass(y, W, B * L, L, d, V, inv_tau, seed, step, parts, status, nullptr, st,
                        nullptr, out && out->entropy);
  if (e != cudaSuccess) return cuda_fail(e, "vocab_posterior_noalloc: vocab pass launch");
  FinalizeParams fp{};
  fp.parts = parts;
  fp.num_mt = vp.num_mt;
  fp.S = vp.S;
  fp.L = L;
  if (out) {
    fp.out_x0hat = out->x0hat;
    fp.out_top1 = out->top1;
    fp.out_logp_top1 = out->logp_top1;
    fp.out_lse = out->lse;
    fp.out_logp_x0hat = out->logp_x0hat;
    fp.out_entropy = out->entropy;
  }
  fp.x_in = x_in;
  fp.x_out = x_out;
  fp.lock = lock;
  fp.jump = jump;
  fp.done = done;
  fp.jump_thr = jump_thr;
  fp.lock_logthr = lock_logthr;
  fp.k0 = static_cast<uint32_t>(seed);
  fp.k1 = static_cast<uint32_t>(seed >> 32);
  fp.step = static_cast<uint32_t>(step);
  fp.ticket = reinterpret_cast<unsigned long long*>(counters);
  launch_vocab_finalize(fp, B, st);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "vocab_posterior_noalloc: finalize launch");
  return DG_OK;
}
