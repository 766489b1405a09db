// Integer-decision kernels: forward noising, the Euler jump/lock/commit step, and the
// finalisation of the fused vocabulary pass (split merge + posterior outputs + Euler step).
#include "dg_common.cuh"
#include "kernels.cuh"
#include "sm103.cuh"

namespace dg {

// ------------------------------------------------------------------ forward noising ----
// [TR "Forward Process"]: x_t = x_0 when the keep draw passes kappa's threshold, else a
// uniform token.  One Philox call per position; four positions per thread with 16-byte
// loads and stores when the four lie in the array.
__global__ void forward_noise_kernel(const int32_t* __restrict__ x0, int32_t* __restrict__ xt,
                                     const uint64_t* __restrict__ keep_thr, int B, int L,
                                     uint32_t V, uint32_t k0, uint32_t k1) {
  const int64_t n = static_cast<int64_t>(B) * L;
  const int64_t n4 = (n + 3) / 4;
  for (int64_t i4 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i4 < n4;
       i4 += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p0 = i4 * 4;
    int32_t in[4] = {0, 0, 0, 0}, out[4];
    const bool full = p0 + 3 < n;
    if (full) {
      const int4 v = *reinterpret_cast<const int4*>(x0 + p0);
      in[0] = v.x;
      in[1] = v.y;
      in[2] = v.z;
      in[3] = v.w;
    } else {
      for (int e = 0; e < 4; ++e)
        if (p0 + e < n) in[e] = x0[p0 + e];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t p = p0 + e;
      const uint32_t canvas = static_cast<uint32_t>(p / L);
      const uint32_t pos = static_cast<uint32_t>(p % L);
      const Words4 w = philox4x32_10(pos, canvas, 0u, kStreamNoise, k0, k1);
      const bool keep = p < n && static_cast<uint64_t>(w.x) < keep_thr[p < n ? canvas : 0];
      out[e] = keep ? in[e] : draw_token(w.y, V);
    }
    if (full) {
      *reinterpret_cast<int4*>(xt + p0) = make_int4(out[0], out[1], out[2], out[3]);
    } else {
      for (int e = 0; e < 4; ++e)
        if (p0 + e < n) xt[p0 + e] = out[e];
    }
  }
}

void launch_forward_noise(const int32_t* x0, int32_t* xt, const uint64_t* keep_thr, int B, int L,
                          int V, uint64_t seed, cudaStream_t st) {
  const int64_t n4 = (static_cast<int64_t>(B) * L + 3) / 4;
  const int threads = 256;
  int64_t blocks = (n4 + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  forward_noise_kernel<<<static_cast<int>(blocks), threads, 0, st>>>(
      x0, xt, keep_thr, B, L, static_cast<uint32_t>(V), static_cast<uint32_t>(seed),
      static_cast<uint32_t>(seed >> 32));
}

// --------------------------------------------------------------- Euler update ----------
// One CTA per canvas, one thread per position; `done` is a block-wide AND of the locks.
__global__ void euler_update_kernel(const int32_t* __restrict__ x_in,
                                    const int32_t* __restrict__ x0hat,
                                    const int32_t* __restrict__ top1,
                                    const float* __restrict__ logp_top1, int32_t* x_out,
                                    uint8_t* lock, uint8_t* jump, uint8_t* done, int L,
                                    uint32_t k0, uint32_t k1, uint32_t step, uint64_t jump_thr,
                                    float lock_logthr) {
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  bool locked_after = true;
  if (i < L) {
    const int64_t r = static_cast<int64_t>(b) * L + i;
    const uint32_t u = jump_draw(static_cast<uint32_t>(i), static_cast<uint32_t>(b), step, k0, k1);
    const EulerOut o = euler_decide(x_in[r], x0hat[r], top1[r], logp_top1[r], lock[r] != 0, u,
                                    jump_thr, lock_logthr);
    x_out[r] = o.x;
    lock[r] = o.lock ? 1 : 0;
    if (jump) jump[r] = o.jump ? 1 : 0;
    locked_after = o.lock;
  }
  const int all = __syncthreads_and(locked_after ? 1 : 0);
  if (done && i == 0) done[b] = all ? 1 : 0;
}

void launch_euler_update(const int32_t* x_in, const int32_t* x0hat, const int32_t* top1,
                         const float* logp_top1, int32_t* x_out, uint8_t* lock, uint8_t* jump,
                         uint8_t* done, int B, int L, uint64_t seed, int step, uint64_t jump_thr,
                         float lock_logthr, cudaStream_t st) {
  const int threads = ((L + 31) / 32) * 32;
  euler_update_kernel<<<B, threads, 0, st>>>(x_in, x0hat, top1, logp_top1, x_out, lock, jump,
                                             done, L, static_cast<uint32_t>(seed),
                                             static_cast<uint32_t>(seed >> 32),
                                             static_cast<uint32_t>(step), jump_thr, lock_logthr);
}

// ------------------------------------------------- vocabulary-pass finalisation -------
// One warp per position (eight positions per CTA, all of one canvas).  The lanes merge the
// position's partial tuples from the vocabulary chunks (lane l takes chunks l, l + 32, ...),
// then a fixed xor-butterfly combines the lanes: the reduction order never changes, so the
// result is deterministic.  Lane 0 writes the posterior outputs and applies the Euler step.
// Per canvas, the CTAs count the positions left unlocked; the last CTA of the canvas to
// finish (an atomic ticket, no waiting) sets `done`, updates the loop bookkeeping and resets
// the counters for the next call.
constexpr int kFinRows = 8;

__device__ __forceinline__ VocabPart shfl_xor_part(const VocabPart& a, int off) {
  VocabPart o;
  o.m = __shfl_xor_sync(0xFFFFFFFFu, a.m, off);
  o.s = __shfl_xor_sync(0xFFFFFFFFu, a.s, off);
  o.top_z = __shfl_xor_sync(0xFFFFFFFFu, a.top_z, off);
  o.best_score = __shfl_xor_sync(0xFFFFFFFFu, a.best_score, off);
  o.best_z = __shfl_xor_sync(0xFFFFFFFFu, a.best_z, off);
  o.top_idx = __shfl_xor_sync(0xFFFFFFFFu, a.top_idx, off);
  o.best_idx = __shfl_xor_sync(0xFFFFFFFFu, a.best_idx, off);
  o.t = __shfl_xor_sync(0xFFFFFFFFu, a.t, off);
  return o;
}

// What the Euler step of one position reads besides the posterior: the token and the lock it
// had, whether its canvas is active, and the position's jump uniform (Philox).  None of it is
// written by the vocabulary pass, so the fused kernel reads it before waiting for that pass.
struct RowIn {
  int32_t x_old;
  bool was_locked, is_active;
  uint32_t u;
};
__device__ __forceinline__ RowIn row_inputs(const FinalizeParams& p, int row) {
  const int b = row / p.L;
  const int i = row % p.L;
  RowIn in;
  in.is_active = p.active == nullptr || p.active[b] != 0;
  in.x_old = p.x_in != nullptr ? p.x_in[row] : 0;
  in.was_locked = p.lock != nullptr && p.lock[row] != 0;
  in.u = jump_draw(static_cast<uint32_t>(i), static_cast<uint32_t>(b), p.step, p.k0, p.k1);
  return in;
}

// One position: the lanes of a warp merge its tuples (each lane its own in order c = lane,
// lane + 32, ..., four loads in flight, then a butterfly); lane 0 writes the posterior outputs
// and applies the Euler step.  Returns (valid in lane 0) whether the position is locked after
// the step and its token.
struct RowFinal {
  bool locked_after;
  bool changed;  // the position's token differs from the one it had before the step
  int32_t token;
};

__device__ __forceinline__ RowFinal finalize_row(const FinalizeParams& p, int row, int lane,
                                                const RowIn& in) {
  constexpr int kB = 4;  // tuple loads in flight per lane
  const bool is_active = in.is_active;
  const int mt = row >> 7;
  const int row_in = row & 127;
  VocabPart acc = empty_part();
  for (int c0 = lane; c0 < p.S; c0 += 32 * kB) {
    VocabPart t[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const int c = c0 + 32 * k;
      t[k] = c < p.S ? p.parts[(static_cast<int64_t>(c) * p.num_mt + mt) * 128 + row_in]
                     : empty_part();
    }
#pragma unroll
    for (int k = 0; k < kB; ++k)
      if (c0 + 32 * k < p.S) merge_part(acc, t[k]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const VocabPart o = shfl_xor_part(acc, off);
    // both lanes of a pair combine (lower lane's tuple first) and get identical results
    if (lane & off) {
      VocabPart t = o;
      merge_part(t, acc);
      acc = t;
    } else {
      merge_part(acc, o);
    }
  }

  RowFinal r{false, false, 0};
  if (lane == 0) {
    if (p.bar) p.bar[row] = 0u;  // the row's tuples are merged: clear its bar for the next pass
    const float lse = acc.m + logf(acc.s);
    const float lp_top1 = acc.top_z - lse;
    if (p.out_x0hat) p.out_x0hat[row] = acc.best_idx;
    if (p.out_top1) p.out_top1[row] = acc.top_idx;
    if (p.out_logp_top1) p.out_logp_top1[row] = lp_top1;
    if (p.out_lse) p.out_lse[row] = lse;
    if (p.out_logp_x0hat) p.out_logp_x0hat[row] = acc.best_z - lse;
    // entropy = log s - t / s (both relative to the max), clamped at 0 against rounding
    if (p.out_entropy) p.out_entropy[row] = fmaxf(0.f, logf(acc.s) - acc.t / acc.s);
    // cross-entropy mode: the best-sample fields carry the target's tempered logit
    if (p.out_loss) p.out_loss[row] = acc.best_idx != 0x7FFFFFFF ? lse - acc.best_z : NAN;
    if (p.x_in != nullptr && is_active) {
      const int32_t x_old = in.x_old;  // read before the step (x_out may be x_in)
      const EulerOut o = euler_decide(x_old, acc.best_idx, acc.top_idx, lp_top1, in.was_locked,
                                      in.u, p.jump_thr, p.lock_logthr);
      p.x_out[row] = o.x;
      if (p.lock) p.lock[row] = o.lock ? 1 : 0;
      if (p.jump) p.jump[row] = o.jump ? 1 : 0;
      r.locked_after = o.lock && p.lock != nullptr;
      r.changed = o.x != x_old;
      r.token = o.x;
    } else if (p.x_in != nullptr) {
      const int32_t x = in.x_old;
      if (p.x_out != p.x_in) p.x_out[row] = x;
      if (p.jump) p.jump[row] = 0;
      r.locked_after = in.was_locked;
      r.token = x;
    }
  }
  return r;
}

// One thread per CTA, after the CTA's positions of canvas b are final: one 64-bit atomic adds
// their unlocked count (high word) and takes a ticket (low word); the CTA that draws the
// canvas's last ticket (no waiting) sees the canvas's whole unlocked count in the value it got
// back, sets `done`, updates the loop bookkeeping and resets the word.  (Nothing the other
// CTAs wrote is read here, so no fence is needed; the next kernel sees all of it.)
__device__ __forceinline__ void finalize_ticket(const FinalizeParams& p, int b, int unlocked,
                                                int ctas_per_canvas) {
  const bool is_active = p.active == nullptr || p.active[b] != 0;
  const unsigned long long old =
      atomicAdd(&p.ticket[b], (static_cast<unsigned long long>(unlocked) << 32) | 1ull);
  if (static_cast<int>(old & 0xFFFFFFFFull) == ctas_per_canvas - 1) {  // the last CTA
    const bool all = static_cast<int>(old >> 32) + unlocked == 0;
    if (p.done) p.done[b] = all ? 1 : 0;
    if (is_active && p.x_in != nullptr) {
      if (p.steps_taken) p.steps_taken[b] += 1;
      if (p.active && p.stop_when_all_locked && all) {
        p.active[b] = 0;
        if (p.n_active) atomicSub(p.n_active, 1);
      }
    }
    p.ticket[b] = 0ull;
  }
}

__global__ void __launch_bounds__(kFinRows * 32) vocab_finalize_kernel(FinalizeParams p) {
  pdl_wait();
  pdl_trigger();
  if (p.n_active && *p.n_active == 0) return;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kFinRows + warp;  // L is a multiple of kFinRows
  const RowFinal r = finalize_row(p, row, lane, row_inputs(p, row));
  const int unlocked = __syncthreads_count(lane == 0 && !r.locked_after ? 1 : 0);
  if (threadIdx.x == 0) finalize_ticket(p, row / p.L, unlocked, p.L / kFinRows);
}

// The previous step's finalisation fused with this step's embedding gather: eight positions
// per CTA (one warp each finalises its position, as above), then the CTA gathers E at those of
// the eight new tokens that changed, 16 bytes per thread: h already holds E[x] of every
// position whose token the step kept (the loop's first step gathers all of them, and only
// this kernel writes h in between).  Each thread issues its loads before any store, and the
// per-canvas ticket's atomics run while those loads are in flight.
__global__ void __launch_bounds__(kFinRows * 32) embed_finalize_kernel(FinalizeParams p,
                                                                       const uint4* __restrict__ E,
                                                                       uint4* __restrict__ h, int V,
                                                                       int d16) {
  constexpr int32_t kKept = -2;  // s_token of a position whose token the step kept
  constexpr int kU = 8;          // 16-byte loads in flight per thread
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kFinRows;  // L is a multiple of kFinRows
  // the canvas, the locks and the active flags were last written by the previous step's
  // launch of this kernel, long complete: read them before waiting for the vocabulary pass
  const RowIn in = row_inputs(p, row0 + warp);
  pdl_wait();
  pdl_trigger();
  if (p.n_active && *p.n_active == 0) return;
  __shared__ int32_t s_token[kFinRows];
  const RowFinal r = finalize_row(p, row0 + warp, lane, in);
  if (lane == 0) s_token[warp] = r.changed ? r.token : kKept;
  const int unlocked = __syncthreads_count(lane == 0 && !r.locked_after ? 1 : 0);
  const int n16 = kFinRows * d16;
  for (int q0 = threadIdx.x; q0 < n16; q0 += kU * blockDim.x) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = q0 + u * blockDim.x;
      const int rr = q / d16;
      const int id = q < n16 ? s_token[rr] : kKept;
      v[u] = id >= 0 && id < V ? E[static_cast<int64_t>(id) * d16 + (q - rr * d16)]
                               : make_uint4(0, 0, 0, 0);
    }
    if (q0 == threadIdx.x && threadIdx.x == 0)
      finalize_ticket(p, row0 / p.L, unlocked, p.L / kFinRows);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = q0 + u * blockDim.x;
      const int rr = q / d16;
      const int id = q < n16 ? s_token[rr] : kKept;
      if (id == kKept) continue;
      const int c = q - rr * d16;
      if (!(id >= 0 && id < V) && c == 0) atomicOr(p.status, kStatusBadIndex);
      h[static_cast<int64_t>(row0 + rr) * d16 + c] = v[u];
    }
  }
}

// Entropy-bounded step [TR "DiffusionGemma 샘플러"]: one CTA per canvas, one thread per
// position.  Each position's rank in (entropy, position) order is counted against the
// canvas's entropies in shared memory; one thread then forms the running float32 sum in that
// order and the mean in position order, exactly as the definition states them (no parallel
// reduction, so the acceptance count and the stop test are bit-reproducible).
__global__ void __launch_bounds__(1024) entropy_bounded_kernel(EBParams p) {
  pdl_wait();
  pdl_trigger();
  if (p.n_active && *p.n_active == 0) return;
  const int b = blockIdx.x;
  if (p.active && p.active[b] == 0) return;  // uniform over the CTA
  __shared__ float sH[1024];
  __shared__ float sSorted[1024];
  __shared__ int s_k;
  __shared__ float s_mean;
  const int i = threadIdx.x;
  const bool valid = i < p.L;
  const int64_t r = static_cast<int64_t>(b) * p.L + i;
  const bool have_prev = p.prev_top1 != nullptr && p.prev_valid != 0;
  float Hi = 0.f;
  int32_t t1 = 0, prev = 0;
  if (valid) {
    Hi = p.entropy[r];
    sH[i] = Hi;
    t1 = p.top1[r];
    if (have_prev) prev = p.prev_top1[r];
  }
  __syncthreads();
  int rank = 0;
  if (valid) {
    for (int j = 0; j < p.L; ++j) {
      const float Hj = sH[j];
      rank += (Hj < Hi || (Hj == Hi && j < i)) ? 1 : 0;
    }
    sSorted[rank] = Hi;
  }
  const int all_same = __syncthreads_and((!valid || (have_prev && prev == t1)) ? 1 : 0);
  if (i == 0) {
    float run = 0.f;
    int k = 0;
    for (int j = 0; j < p.L; ++j) {
      run = __fadd_rn(run, sSorted[j]);
      if (run > p.gamma) break;
      k = j + 1;
    }
    float acc = 0.f;
    for (int j = 0; j < p.L; ++j) acc = __fadd_rn(acc, sH[j]);
    s_k = k;
    s_mean = __fdiv_rn(acc, static_cast<float>(p.L));
  }
  __syncthreads();
  const bool done = s_mean < p.stop_entropy && have_prev && all_same != 0;
  if (valid) {
    const bool acc_i = rank < s_k;
    int32_t x;
    if (done || p.final_step) {
      x = t1;
    } else if (acc_i) {
      x = p.x0hat[r];
    } else {
      const uint32_t u = philox4x32_10(static_cast<uint32_t>(i), static_cast<uint32_t>(b), 0u,
                                       kStreamRenoise | p.step, p.k0, p.k1).x;
      x = draw_token(u, static_cast<uint32_t>(p.V));
    }
    p.x_out[r] = x;
    if (p.accept) p.accept[r] = acc_i ? 1 : 0;
    if (p.prev_top1) p.prev_top1[r] = t1;
  }
  if (i == 0) {
    if (p.done) p.done[b] = done ? 1 : 0;
    if (p.mean_out) p.mean_out[b] = s_mean;
    if (p.steps_taken) p.steps_taken[b] += 1;
    if (p.active && done) {
      p.active[b] = 0;
      if (p.n_active) atomicSub(p.n_active, 1);
    }
  }
}

void launch_entropy_bounded(const EBParams& p, int B, cudaStream_t st) {
  const int threads = (p.L + 31) / 32 * 32;
  launch_dependent(entropy_bounded_kernel, dim3(B), dim3(threads), 0, st, p);
}

void launch_vocab_finalize(const FinalizeParams& p, int B, cudaStream_t st) {
  const int rows = B * p.L;
  timer_begin(4, st);
  launch_dependent(vocab_finalize_kernel, dim3(rows / kFinRows), dim3(kFinRows * 32), 0, st, p);
  timer_end(4, st);
}

void launch_embed_finalize(const FinalizeParams& p0, int B, const uint16_t* E, uint16_t* h,
                           int V, int d, cudaStream_t st) {
  FinalizeParams p = p0;
  p.status = status_or_fallback(p.status);
  const int d16 = d / 8;
  timer_begin(4, st);
  launch_dependent(embed_finalize_kernel, dim3(B * p.L / kFinRows), dim3(kFinRows * 32), 0, st, p,
                   reinterpret_cast<const uint4*>(E), reinterpret_cast<uint4*>(h), V, d16);
  timer_end(4, st);
}

// Loop bookkeeping: active[b] = 1 unless the canvas is already fully locked and stopping is
// on, or it is not generating any more (gen_active[b] == 0); n_active = number of active
// canvases; steps_taken = 0.
__global__ void loop_init_kernel(const uint8_t* lock, const uint8_t* gen_active, uint8_t* active,
                                 int* n_active, int32_t* steps_taken, int L,
                                 int stop_when_all_locked) {
  const int b = blockIdx.x;
  bool locked = lock != nullptr;  // no lock state: nothing is locked
  for (int i = threadIdx.x; locked && i < L; i += blockDim.x)
    locked = lock[static_cast<int64_t>(b) * L + i] != 0;
  const int all = __syncthreads_and(locked ? 1 : 0);
  if (threadIdx.x == 0) {
    const bool act = !(stop_when_all_locked && all) && (gen_active == nullptr || gen_active[b]);
    active[b] = act ? 1 : 0;
    steps_taken[b] = 0;
    if (act) atomicAdd(n_active, 1);
  }
}

void launch_loop_init(const uint8_t* lock, uint8_t* active, int* n_active, int32_t* steps_taken,
                      int B, int L, int stop_when_all_locked, cudaStream_t st) {
  loop_init_kernel<<<B, 256, 0, st>>>(lock, nullptr, active, n_active, steps_taken, L,
                                      stop_when_all_locked);
}

void launch_loop_init_masked(const uint8_t* lock, const uint8_t* gen_active, uint8_t* active,
                             int* n_active, int32_t* steps_taken, int B, int L,
                             int stop_when_all_locked, cudaStream_t st) {
  loop_init_kernel<<<B, 256, 0, st>>>(lock, gen_active, active, n_active, steps_taken, L,
                                      stop_when_all_locked);
}

// Encode-append: the canvas's K and V rows (kv_row_elems bf16 each) into cache rows P .. P+L-1
// of every active canvas; cache [B, P_cap, row].  16 bytes per thread.
__global__ void kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 uint4* __restrict__ kc, uint4* __restrict__ vc,
                                 const uint8_t* active, int L, int P, int P_cap, int row16) {
  const int r = blockIdx.x;  // canvas row b * L + i
  const int b = r / L, i = r % L;
  if (active && active[b] == 0) return;
  const int64_t src = static_cast<int64_t>(r) * row16;
  const int64_t dst = (static_cast<int64_t>(b) * P_cap + P + i) * row16;
  for (int c = threadIdx.x; c < row16; c += blockDim.x) {
    kc[dst + c] = k[src + c];
    vc[dst + c] = v[src + c];
  }
}

void launch_kv_append(const uint16_t* k, const uint16_t* v, uint16_t* k_cache, uint16_t* v_cache,
                      const uint8_t* active, int B, int L, int P, int P_cap, int kv_row_elems,
                      cudaStream_t st) {
  kv_append_kernel<<<B * L, 128, 0, st>>>(reinterpret_cast<const uint4*>(k),
                                          reinterpret_cast<const uint4*>(v),
                                          reinterpret_cast<uint4*>(k_cache),
                                          reinterpret_cast<uint4*>(v_cache), active, L, P, P_cap,
                                          kv_row_elems / 8);
}

// A finished block j of every generating canvas: out[b, j, :] = canvas, steps added, blocks =
// j + 1; the first end-of-turn token (if any) fixes the response length and ends the canvas.
__global__ void block_init_kernel(uint8_t* gen_active, int* gen_count, int32_t* blocks,
                                  int32_t* n_tokens, int32_t* steps_total, int B) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    gen_active[b] = 1;
    blocks[b] = 0;
    n_tokens[b] = 0;
    steps_total[b] = 0;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *gen_count = B;
}

void launch_block_init(uint8_t* gen_active, int* gen_count, int32_t* blocks, int32_t* n_tokens,
                       int32_t* steps_total, int B, cudaStream_t st) {
  const int blocks_n = std::min((B + 255) / 256, 1024);
  block_init_kernel<<<blocks_n, 256, 0, st>>>(gen_active, gen_count, blocks, n_tokens,
                                              steps_total, B);
}

__global__ void block_record_kernel(const int32_t* canvas, const int32_t* steps_taken,
                                    int32_t* out, uint8_t* active, int* gen_count,
                                    int32_t* blocks, int32_t* n_tokens, int32_t* steps_total,
                                    int L, int NB, int j, int32_t eos) {
  const int b = blockIdx.x;
  if (active[b] == 0) return;  // uniform over the CTA
  __shared__ int first;
  if (threadIdx.x == 0) first = 0x7FFFFFFF;
  __syncthreads();
  for (int i = threadIdx.x; i < L; i += blockDim.x) {
    const int32_t x = canvas[static_cast<int64_t>(b) * L + i];
    out[(static_cast<int64_t>(b) * NB + j) * L + i] = x;
    if (x == eos) atomicMin(&first, i);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    blocks[b] = j + 1;
    steps_total[b] += steps_taken[b];
    if (first != 0x7FFFFFFF) {
      n_tokens[b] = j * L + first + 1;
      active[b] = 0;
      atomicSub(gen_count, 1);
    } else {
      n_tokens[b] = (j + 1) * L;
    }
  }
}

void launch_block_record(const int32_t* canvas, const int32_t* steps_taken, int32_t* out,
                         uint8_t* active, int* gen_count, int32_t* blocks, int32_t* n_tokens,
                         int32_t* steps_total, int B, int L, int NB, int j, int32_t eos,
                         cudaStream_t st) {
  block_record_kernel<<<B, 256, 0, st>>>(canvas, steps_taken, out, active, gen_count, blocks,
                                         n_tokens, steps_total, L, NB, j, eos);
}

// h[r, :] = E[x[r], :]; ids outside [0, V) give a zero row.  16 bytes per thread.
// h = E[x] (+ s, the self-conditioning signal, summed in fp32 and rounded to bf16).
__global__ void embed_gather_kernel(const int32_t* __restrict__ x, const uint4* __restrict__ E,
                                    const uint4* __restrict__ s, uint4* __restrict__ h, int V,
                                    int d16, const int* n_active, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  if (n_active && *n_active == 0) return;
  const int r = blockIdx.x;
  const int id = x[r];
  const bool ok = id >= 0 && id < V;
  if (!ok && threadIdx.x == 0) atomicOr(status, kStatusBadIndex);
  for (int c = threadIdx.x; c < d16; c += blockDim.x) {
    uint4 w = ok ? E[static_cast<int64_t>(id) * d16 + c] : make_uint4(0, 0, 0, 0);
    if (s) {
      const uint4 a = s[static_cast<int64_t>(r) * d16 + c];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      uint32_t ew[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
        const float2 fe = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ew[e]));
        ew[e] = pack_bf16x2(fe.x + fa.x, fe.y + fa.y);
      }
      w = make_uint4(ew[0], ew[1], ew[2], ew[3]);
    }
    h[static_cast<int64_t>(r) * d16 + c] = w;
  }
}

void launch_embed_gather(const int32_t* x, const uint16_t* E, uint16_t* h, int BL, int V, int d,
                         const int* n_active, cudaStream_t st, uint32_t* status,
                         const uint16_t* s) {
  const int d16 = d / 8;
  const int threads = d16 < 256 ? ((d16 + 31) / 32) * 32 : 256;
  launch_dependent(embed_gather_kernel, dim3(BL), dim3(threads), 0, st, x,
                   reinterpret_cast<const uint4*>(E), reinterpret_cast<const uint4*>(s),
                   reinterpret_cast<uint4*>(h), V, d16, n_active, status_or_fallback(status));
}

}  // namespace dg
