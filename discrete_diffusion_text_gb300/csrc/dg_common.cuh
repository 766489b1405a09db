// Internal declarations shared by the library's translation units: the counter-based
// generator, the per-position Euler decision, the split-vocabulary partial tuple, status
// reporting and the host helpers (error text, tensor maps, device properties).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "dgcanvas.h"

namespace dg {

// ------------------------------------------------------------- Philox4x32-10 -----------
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): ten
// rounds of two 32x32->64-bit multiplies with the round key xored into the high halves;
// the key is bumped by two Weyl constants between rounds.

struct Words4 {
  uint32_t x, y, z, w;
};

// One 32 x 32 -> 64-bit product (its high and low words in one multiply).
__device__ __forceinline__ uint64_t mul_wide_u32(uint32_t a, uint32_t b) {
  uint64_t p;
  asm("mul.wide.u32 %0, %1, %2;" : "=l"(p) : "r"(a), "r"(b));
  return p;
}

__device__ __forceinline__ Words4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = mul_wide_u32(0xD2511F53u, c0);
    const uint64_t p1 = mul_wide_u32(0xCD9E8D57u, c2);
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ k1;
    c0 = n0;
    c1 = static_cast<uint32_t>(p1);
    c2 = n2;
    c3 = static_cast<uint32_t>(p0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return {c0, c1, c2, c3};
}

// The same generator with the ten round keys computed once (k0 + r*W0, k1 + r*W1) by the
// caller, for loops that draw many counters under one key.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

__device__ __forceinline__ PhiloxKeys philox_round_keys(uint32_t k0, uint32_t k1) {
  PhiloxKeys k;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = k0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
    k.k1[r] = k1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
  }
  return k;
}

__device__ __forceinline__ Words4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                uint32_t c3, const PhiloxKeys& k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = mul_wide_u32(0xD2511F53u, c0);
    const uint64_t p1 = mul_wide_u32(0xCD9E8D57u, c2);
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ k.k0[r];
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ k.k1[r];
    c0 = n0;
    c1 = static_cast<uint32_t>(p1);
    c2 = n2;
    c3 = static_cast<uint32_t>(p0);
  }
  return {c0, c1, c2, c3};
}

// Stream tags in the top byte of counter word 3 (the step index sits in the low 24 bits).
constexpr uint32_t kStreamNoise = 1u << 24;
constexpr uint32_t kStreamGumbel = 2u << 24;
constexpr uint32_t kStreamJump = 3u << 24;
constexpr uint32_t kStreamRenoise = 4u << 24;
constexpr uint32_t kStreamPick = 5u << 24;

// A draw as a token uniform over [0, V): floor(u * V / 2^32).
__device__ __forceinline__ int32_t draw_token(uint32_t u, uint32_t V) {
  return static_cast<int32_t>((static_cast<uint64_t>(u) * V) >> 32);
}

// ---------------------------------------------------- Euler step with locking ---------
// Per position: locked -> unchanged; else if top-1 log-probability >= log(theta) -> lock and
// commit the top-1 token; else jump to the posterior sample when the jump draw falls under
// the integer threshold floor(lambda_n * 2^32).  lock_logthr = +inf disables locking.

struct EulerOut {
  int32_t x;
  bool lock;
  bool jump;
};

__device__ __forceinline__ EulerOut euler_decide(int32_t x_in, int32_t x0hat, int32_t top1,
                                                 float logp_top1, bool locked, uint32_t u_jump,
                                                 uint64_t jump_thr, float lock_logthr) {
  if (locked) return {x_in, true, false};
  if (logp_top1 >= lock_logthr) return {top1, true, false};
  const bool j = static_cast<uint64_t>(u_jump) < jump_thr;
  return {j ? x0hat : x_in, false, j};
}

__device__ __forceinline__ uint32_t jump_draw(uint32_t pos, uint32_t canvas, uint32_t step,
                                              uint32_t k0, uint32_t k1) {
  return philox4x32_10(0u, pos, canvas, kStreamJump | step, k0, k1).x;
}

// ------------------------------------------------- split-vocabulary partial tuple -----
// What one CTA knows about one row after scanning a contiguous range of the vocabulary:
// running max m, s = sum of exp(z - m) and t = sum of exp(z - m) (z - m) of the tempered
// logits (the entropy of the row is log s - t / s), the top-1 logit and index, and the best
// Gumbel-perturbed score with its index and logit.  Ties go to the lower index.

struct alignas(16) VocabPart {
  float m, s, top_z, best_score;
  float best_z;
  int32_t top_idx, best_idx;
  float t;
};

__device__ __forceinline__ void merge_part(VocabPart& a, const VocabPart& b) {
  const float M = fmaxf(a.m, b.m);
  float s = 0.f, t = 0.f;
  if (a.m != -INFINITY) {  // re-reference to M: (z - M) = (z - m_a) + (m_a - M)
    const float f = __expf(a.m - M);
    s += a.s * f;
    t += f * fmaf(a.s, a.m - M, a.t);
  }
  if (b.m != -INFINITY) {
    const float f = __expf(b.m - M);
    s += b.s * f;
    t += f * fmaf(b.s, b.m - M, b.t);
  }
  a.m = M;
  a.s = s;
  a.t = t;
  if (b.top_z > a.top_z || (b.top_z == a.top_z && b.top_idx < a.top_idx)) {
    a.top_z = b.top_z;
    a.top_idx = b.top_idx;
  }
  if (b.best_score > a.best_score ||
      (b.best_score == a.best_score && b.best_idx < a.best_idx)) {
    a.best_score = b.best_score;
    a.best_idx = b.best_idx;
    a.best_z = b.best_z;
  }
}

__device__ __forceinline__ VocabPart empty_part() {
  VocabPart p;
  p.m = -INFINITY;
  p.s = 0.f;
  p.top_z = -INFINITY;
  p.best_score = -INFINITY;
  p.best_z = -INFINITY;
  p.top_idx = 0x7FFFFFFF;
  p.best_idx = 0x7FFFFFFF;
  p.t = 0.f;
  return p;
}

// --------------------------------------------------------------- device status -----------
// Bit flags OR-ed into a device word by kernels that give up on a wait.
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBadIndex = 2u;

// Device status word for calls made without a workspace (a library-owned __device__ word;
// read through dg_workspace_status(NULL)).  Launchers pass it when the caller gave none, so
// kernels always receive a valid status pointer.
uint32_t* status_or_fallback(uint32_t* status);

// ------------------------------------------------------------------- host helpers -----

// The limit of every on-chip wait of kernels the calling thread enqueues (set with
// dg_set_wait_control; 2 s by default), and the LM-head kernel's test switch that makes its
// load warps issue nothing (so its waits run out with no copy or tensor-core work in flight).
uint64_t wait_limit_ns();
bool wait_test_skip_loads();

void set_error(const std::string& msg);
dg_status fail(dg_status code, const std::string& msg);
dg_status cuda_fail(cudaError_t e, const char* what);
int num_sms();
int device_id();

// Tiled tensor map over a bf16 array with 128-byte swizzle.  dims[0] is the contiguous
// dimension; strides_bytes[i] is the byte stride of dims[i+1].
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace dg
