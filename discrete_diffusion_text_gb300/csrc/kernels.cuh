// Launch interfaces of the library's kernels (host side of each translation unit).
#pragma once

#include <utility>

#include "dg_common.cuh"

namespace dg {

struct FinalizeParams {
  const VocabPart* parts;  // [S * num_mt * 128]
  int num_mt, S, L;
  int32_t* out_x0hat;
  int32_t* out_top1;
  float* out_logp_top1;
  float* out_lse;
  float* out_logp_x0hat;
  float* out_entropy;
  float* out_loss;      // cross-entropy mode: lse - z~[target]
  const int32_t* x_in;  // NULL: posterior only
  int32_t* x_out;
  uint8_t* lock;
  uint8_t* jump;
  uint8_t* done;
  uint64_t jump_thr;
  float lock_logthr;
  uint32_t k0, k1, step;
  uint8_t* active;       // loop only
  int32_t* steps_taken;  // loop only
  int* n_active;         // loop only
  int stop_when_all_locked;
  // [B] per canvas: (positions left unlocked << 32) + CTAs done, zero before the first call;
  // reset by the kernel (8-byte aligned)
  unsigned long long* ticket;
  uint32_t* bar;  // the vocabulary pass's sampling bars: zeroed per row once merged (or NULL)
  uint32_t* status;  // embed_finalize_kernel: kStatusBadIndex for a token outside [0, V)
};

// One step of the entropy-bounded sampler for every canvas (one CTA per canvas).
struct EBParams {
  const int32_t* x0hat;
  const int32_t* top1;
  const float* entropy;
  int32_t* prev_top1;  // NULL: no previous prediction
  int prev_valid;
  int32_t* x_out;
  uint8_t* accept;
  uint8_t* done;
  float* mean_out;
  int L, V;
  uint32_t k0, k1, step;
  float gamma, stop_entropy;
  int final_step;
  uint8_t* active;       // loop only
  int32_t* steps_taken;  // loop only
  int* n_active;         // loop only
};
void launch_entropy_bounded(const EBParams& p, int B, cudaStream_t st);

// Block-AR helpers: K/V of the canvas into cache rows [P, P + L) of each active canvas, and
// the record of a finished block (output, end-of-turn test, counts).
void launch_kv_append(const uint16_t* k, const uint16_t* v, uint16_t* k_cache, uint16_t* v_cache,
                      const uint8_t* active, int B, int L, int P, int P_cap, int kv_row_elems,
                      cudaStream_t st);
void launch_block_init(uint8_t* gen_active, int* gen_count, int32_t* blocks, int32_t* n_tokens,
                       int32_t* steps_total, int B, cudaStream_t st);
void launch_block_record(const int32_t* canvas, const int32_t* steps_taken, int32_t* out,
                         uint8_t* active, int* gen_count, int32_t* blocks, int32_t* n_tokens,
                         int32_t* steps_total, int B, int L, int NB, int j, int32_t eos,
                         cudaStream_t st);
void launch_loop_init_masked(const uint8_t* lock, const uint8_t* gen_active, uint8_t* active,
                             int* n_active, int32_t* steps_taken, int B, int L,
                             int stop_when_all_locked, cudaStream_t st);

void launch_forward_noise(const int32_t* x0, int32_t* xt, const uint64_t* keep_thr, int B, int L,
                          int V, uint64_t seed, cudaStream_t st);
void launch_euler_update(const int32_t* x_in, const int32_t* x0hat, const int32_t* top1,
                         const float* logp_top1, int32_t* x_out, uint8_t* lock, uint8_t* jump,
                         uint8_t* done, int B, int L, uint64_t seed, int step, uint64_t jump_thr,
                         float lock_logthr, cudaStream_t st);
void launch_vocab_finalize(const FinalizeParams& p, int B, cudaStream_t st);
// The finalisation of p (the previous step) fused with the embedding gather h = E[x_out] of
// the next step (no self-conditioning signal); p.x_in and p.x_out must be set.
void launch_embed_finalize(const FinalizeParams& p, int B, const uint16_t* E, uint16_t* h, int V,
                           int d, cudaStream_t st);
void launch_loop_init(const uint8_t* lock, uint8_t* active, int* n_active, int32_t* steps_taken,
                      int B, int L, int stop_when_all_locked, cudaStream_t st);
// h = E[x] (+ s when s != NULL: the self-conditioning signal, bf16 [BL, d]).  An id outside
// [0, V) gives a zero row and sets kStatusBadIndex in *status (NULL: the library's word).
void launch_embed_gather(const int32_t* x, const uint16_t* E, uint16_t* h, int BL, int V, int d,
                         const int* n_active, cudaStream_t st, uint32_t* status,
                         const uint16_t* s = nullptr);

// Launch with programmatic stream serialisation: the kernel may be scheduled while the
// previous kernel in the stream finishes (its launch latency hidden behind that kernel); it
// must call pdl_wait() before touching memory that kernel writes (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- projection GEMM -----
// C[M, N] = A[M, K] W[N, K]^T (+ R[M, N]) in bf16 with fp32 accumulation; the N columns are
// routed to up to three output tensors (column ranges [seg_begin[i], seg_begin[i+1])).
struct GemmOut {
  int nseg;
  int seg_begin[4];
  uint16_t* ptr[3];
  int ld[3];
};

constexpr int kActNone = 0;
constexpr int kActGeluTanh = 1;
// Tile width and K split chosen for a shape; part_bytes: the fp32 workspace the split needs
// (0 without a split).
struct GemmPlan {
  int BN, S;
  size_t part_bytes;
};
GemmPlan plan_gemm(int M, int N, int K, const GemmOut& out);
// part_ws: workspace for the split partials (16-byte aligned); without one, or with fewer than
// plan_gemm(...).part_bytes bytes, every tile runs on one CTA over the whole K.
cudaError_t launch_gemm(const uint16_t* A, const uint16_t* W, int M, int N, int K,
                        const GemmOut& out, const uint16_t* residual, int ld_res,
                        uint32_t* status, const int* n_active, cudaStream_t st,
                        int act = kActNone, void* part_ws = nullptr, size_t part_ws_bytes = 0);

// ------------------------------------------------------------ self-conditioning -----
struct ScPlan {
  int mt, nt, nkb, per, S;
  size_t part_bytes;  // fp32 partials [S, R, d]
};
ScPlan plan_selfcond(int R, int V, int d);
// From the vocabulary pass's bf16 exp(z~ - m_ref) [R, V] (normalised to the posterior on its
// way through shared memory), m_ref [R, V/32] and lse [R]: e = p_hat E (bf16 [R, d]),
// u = gelu(e W1^T) (bf16 [R, dsc]), s = u W2^T (bf16 [R, d]).  d % 256 == 0, V % 64 == 0,
// dsc % 64 == 0.
cudaError_t launch_self_condition(const uint16_t* p_til, const float* m_ref, const float* lse,
                                  const uint16_t* E, const uint16_t* W1, const uint16_t* W2,
                                  int R, int V, int d, int dsc, float* part, uint16_t* e,
                                  uint16_t* u, uint16_t* s, uint32_t* status,
                                  const int* n_active, cudaStream_t st);

// ------------------------------------------------------------------- attention -----
struct AttnPlan {
  int splits;
  int one;    // 1: one query head per CTA with 128-key tiles; 0: two heads per CTA, 64-key tiles
  int units;  // CTAs per split
  size_t part_bytes;  // fp32 partials for split > 1
};
AttnPlan plan_attention(int B, int L, int P, int H, int Hkv, int hd, int window);
// pre_stride: prefix rows allocated per canvas in k_pre / v_pre (-1: P).
cudaError_t launch_attention(const uint16_t* q, const uint16_t* k_pre, const uint16_t* v_pre,
                             const uint16_t* k_can, const uint16_t* v_can, uint16_t* out,
                             float* lse, int B, int L, int P, int H, int Hkv, int hd, int window,
                             float scale, void* part_ws, uint32_t* status, const int* n_active,
                             cudaStream_t st, int pre_stride = -1);

// -------------------------------------------------------------- vocabulary pass -----
struct VocabPlan {
  int num_mt, nvt, per, S, units, grid;
  size_t part_bytes;  // the partial tuples, then one 32-bit sampling bar per row
};
VocabPlan plan_vocab(int R, int V);
// The per-row sampling bars inside a partials area of plan_vocab(R, V).part_bytes bytes: the
// best chunk score published so far in a sampling launch; zero before each sampling launch.
uint32_t* vocab_bars(VocabPart* parts, int R, int V);
// targets != NULL: cross-entropy mode (no Gumbel draws; the tuples carry the target's logit).
// entropy: the tuples also carry the entropy accumulator (otherwise it stays 0).
// sc_p, sc_m != NULL: also store bf16 exp(z~ - m_ref) [R, V] and m_ref [R, V / 32] for the
// self-conditioning contraction.  ce_only: no sampling even without targets (lse only).
// bars_clear: the caller guarantees the sampling bars are zero (a finalisation since the last
// sampling launch reset them, or the caller cleared them); otherwise the launch clears them.
cudaError_t launch_vocab_pass(const uint16_t* y, const uint16_t* W, int R, int L, int d, int V,
                              float inv_tau, uint64_t seed, int step, VocabPart* parts,
                              uint32_t* status, const int* n_active, cudaStream_t st,
                              const int32_t* targets = nullptr, bool entropy = false,
                              uint16_t* sc_p = nullptr, float* sc_m = nullptr,
                              bool ce_only = false, bool bars_clear = false);

// Optional CUDA-event timing around kernels (kind 0: vocabulary pass, 1: attention with its
// merge, 2: self-conditioning contraction, 3: projection GEMM, 4: finalisation).
constexpr int kTimerKinds = 5;
void timer_begin(int kind, cudaStream_t st);
void timer_end(int kind, cudaStream_t st);

}  // namespace dg
