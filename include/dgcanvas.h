/*
 * libdgcanvas: the per-step canvas-denoising core of a block-diffusion text model
 * (DiffusionGemma-style uniform-source discrete diffusion), for NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [TR]   "DiffusionGemma Technical Report 정리": "이산 디퓨전 정식화", "Forward Process",
 *          "Backward Denoising Process", "블록 자기회귀(Block-AR) 생성",
 *          "디노이징 반복과 self-conditioning", "DiffusionGemma 샘플러",
 *          "1단계: Supervised Finetuning", "CPU-GPU 동기화 제거".
 *   [BLOG] "DiffusionGemma 완전분석": "스펙 정리" (canvas 256, vocabulary 262k, window 1,024).
 *   [PBD]  "Google DiffusionGemma 출시: 병렬 블록 디코딩": glossary "Iterative denoising",
 *          FAQ (confident tokens are locked in, the rest re-evaluated).
 *   [P11]  Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11 (Philox4x32-10).
 *
 * Conventions shared by every call
 *   - Time runs from t = 1 (uniform noise) to t = 0 (clean) [TR "이산 디퓨전 정식화"]; step n
 *     of T maps t_n = (T - n)/T to t_n - h with h = 1/T [TR "디노이징 반복과 self-conditioning"].
 *   - Tokens are int32; activations and weights are bfloat16 passed as uint16_t bit patterns;
 *     every matrix is row-major; arithmetic accumulates in fp32.
 *   - Pointers are DEVICE pointers unless marked "host".  The caller owns every buffer; no
 *     call allocates device memory.  Device pointers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Device-side calls are
 *     stream-ordered and asynchronous; they return after enqueueing work.
 *   - Random draws are Philox4x32-10 [P11] keyed by the 64-bit seed (low word = key 0) with
 *     counters that depend only on (stream, step, canvas, position, vocab index):
 *       noising / canvas init: (position, canvas, 0, 1<<24); word 0 = keep draw, word 1 = token
 *       chunk Gumbel:          (c >> 2, position, canvas, (2<<24) | step); the 32-entry
 *                              vocabulary chunk c = v / 32 uses word c & 3
 *       Euler jump:            (0, position, canvas, (3<<24) | step); word 0
 *       re-noising:            (position, canvas, 0, (4<<24) | step); word 0
 *       within-chunk Gumbel:   (v >> 2, position, canvas, (5<<24) | step); vocab v uses word v & 3
 *     so results do not depend on launch shape, and a run can be resumed at any step.
 *   - A probability p is passed as the integer threshold floor(p * 2^32) (p = 1 -> 2^32); a
 *     32-bit draw u "passes" iff u < threshold.  Decisions are therefore exact integer tests.
 *   - Errors: every call validates its arguments on the host and returns DG_EINVAL /
 *     DG_ENOTSUP before launching anything; a CUDA launch or API failure returns DG_ECUDA.
 *     dg_last_error() returns a thread-local message for the last non-OK status.  Kernels
 *     that wait on on-chip barriers never spin without limit: a wait that exceeds the call's
 *     limit (2 s unless dg_set_wait_control set another) sets a flag in the call's
 *     workspace, read by dg_workspace_status().  A kernel that meets a token id outside
 *     [0, V) where it gathers an embedding row uses a zero row instead of reading out of
 *     bounds and sets another flag, reported as DG_EKERNEL.
 *   - Threading: calls are thread-compatible; the only global state is the thread-local error
 *     text, a per-device cache of device properties and the optional kernel timer.
 */
#ifndef DGCANVAS_H
#define DGCANVAS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DG_OK = 0,
  DG_EINVAL = 1,   /* bad argument (null pointer, negative size, misaligned pointer, ...) */
  DG_ENOTSUP = 2,  /* valid but unsupported shape (see each call's limits) */
  DG_ECUDA = 3,    /* a CUDA runtime call or kernel launch failed */
  DG_EKERNEL = 4,  /* a kernel reported an out-of-range index it skipped */
  DG_ETIMEOUT = 5  /* a kernel gave up waiting on an on-chip barrier */
} dg_status;

typedef enum { DG_SCHED_LINEAR = 0, DG_SCHED_COSINE = 1 } dg_schedule;

/* Thread-local text of the last non-OK status (never NULL). */
const char* dg_last_error(void);

/* Version of this ABI (increments on incompatible change). */
int dg_abi_version(void);

/* ------------------------------------------------------------------ schedules (host) ----
 * kappa_t falls monotonically from kappa_0 = 1 to kappa_1 = 0 [TR "Forward Process"]; the pages
 * fix no family, so two are offered: linear kappa = 1 - t and cosine kappa = cos^2(pi t / 2).
 * The discrete Euler step of the factorised mixture path [TR "Backward Denoising Process"]
 * replaces a token by a fresh posterior sample with probability
 *     lambda_n = min(1, h * (-kappa'(t_n)) / (1 - kappa(t_n)))
 * (linear: 1/(T - n); cosine: h*pi*cot(pi t_n / 2), so lambda_0 = 0 and lambda_{T-1} = 1).
 *
 * dg_schedule_thresholds: keep_thr[n] = floor(kappa(t_n) * 2^32) for n = 0..T (host array of
 * T + 1; t_T = 0) and jump_thr[n] = floor(lambda_n * 2^32) for n = 0..T-1 (host array of T).
 * Either output may be NULL.  Computed in double precision.  Errors: DG_EINVAL if T < 1 or
 * the schedule is unknown.
 */
dg_status dg_schedule_thresholds(int schedule, int T, uint64_t* keep_thr, uint64_t* jump_thr);

/* keep_thr[b] = floor(kappa(t[b]) * 2^32) for noise levels t[b] in [0, 1] (host arrays of B).
 * Errors: DG_EINVAL on NULL arrays, B < 0, t outside [0, 1] or an unknown schedule. */
dg_status dg_keep_thresholds(int schedule, const double* t, int B, uint64_t* keep_thr);

/* ------------------------------------------------------------------- forward noising ----
 * Closed-form forward process [TR "Forward Process"; "1단계: Supervised Finetuning"]:
 *     x_t^i = x_0^i if the keep draw of position i passes keep_thr[canvas], else a token uniform
 *     over [0, V) (word 1 of the same draw), independently per position,
 * so P(x_t^i = x_0^i) = kappa_t + (1 - kappa_t)/V.  keep_thr = 0 gives the uniform prior x_1
 * used to initialise a canvas [TR "블록 자기회귀(Block-AR) 생성"].
 *
 *   x0 [B, L] int32 (values are copied through, not range-checked); xt [B, L] int32 (may alias
 *   x0); keep_thr [B] uint64 (device).  Limits: B, L >= 0, B * L < 2^31, 1 <= V < 2^31.
 *   Errors: DG_EINVAL on NULL or misaligned pointers or bad sizes.
 */
dg_status dg_forward_noise(const int32_t* x0, int32_t* xt, const uint64_t* keep_thr, int B, int L,
                           int V, uint64_t seed, void* stream);

/* ------------------------------------------------- stand-in decoder: embedding + QKV ----
 * First half of logits = Decoder(x_t, KV) [TR "디노이징 반복과 self-conditioning"] for a
 * one-layer stand-in decoder: h = E[x_t]; [q | k_c | v_c] = h Wqkv^T (rounded to bf16).
 *
 *   x [B*L] int32 token ids in [0, V) (ids outside read as a zero row); E [V, d] bf16;
 *   Wqkv [(H + 2*Hkv)*hd, d] bf16 (rows: the H query heads, then the Hkv key heads, then the Hkv
 *   value heads, each hd rows); outputs h [B*L, d], q [B*L, H*hd], k [B*L, Hkv*hd],
 *   v [B*L, Hkv*hd] bf16 (q, k, v are [B, L, heads, hd] in memory).
 *   Limits: d % 64 == 0, hd in {64, 128}, H % Hkv == 0.  Errors: DG_EINVAL / DG_ENOTSUP.
 */
dg_status dg_embed_qkv(const int32_t* x, const uint16_t* E, const uint16_t* Wqkv, uint16_t* h,
                       uint16_t* q, uint16_t* k, uint16_t* v, int BL, int V, int d, int H,
                       int Hkv, int hd, void* stream);

/* ------------------------------------------------------------------- canvas attention ----
 * The decoder's attention over a cached prefix plus the whole canvas [TR "블록 자기회귀(Block-AR)
 * 생성": bidirectional inside the canvas, cross-attention to the KV cache; BLOG "스펙 정리":
 * sliding-window layers of 1,024 tokens]:
 *     O[b, i, h] = softmax_k( q[b, i, h] . K[b, k, g] * scale ) V[b, k, g],   g = floor(h*Hkv/H)
 * over keys k = the visible prefix keys followed by all L canvas keys.  Canvas query i sits at
 * absolute position P + i; prefix key k is visible iff window == 0 or P + i - k < window.
 *
 *   q [B, L, H, hd]; k_pre, v_pre [B, P, Hkv, hd] (each canvas has its own prefix);
 *   k_can, v_can [B, L, Hkv, hd]; out [B, L, H, hd] bf16; lse [B, H, L] fp32 natural-log
 *   log-sum-exp of the scaled scores, or NULL.  ws: workspace of at least
 *   dg_canvas_attn_workspace(...) bytes (its first 256 bytes hold the status word).
 *   Limits: 1 <= L <= 256, L % 64 == 0, P >= 0, hd in {64, 128}, H % Hkv == 0, window >= 0.
 *   Errors: DG_EINVAL / DG_ENOTSUP; DG_EINVAL if ws_bytes is too small.
 */
size_t dg_canvas_attn_workspace(int B, int L, int P, int H, int Hkv, int hd, int window);
dg_status dg_canvas_attn(const uint16_t* q, const uint16_t* k_pre, const uint16_t* v_pre,
                         const uint16_t* k_can, const uint16_t* v_can, uint16_t* out, float* lse,
                         int B, int L, int P, int H, int Hkv, int hd, int window, float scale,
                         void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------- output projection with residual ----
 * y = h + O Wo^T, rounded to bf16 (the stand-in decoder's attention output projection).
 *   h [BL, d]; O [BL, H*hd]; Wo [d, H*hd]; y [BL, d] bf16 (y must not alias h).
 *   Limits: d % 64 == 0, (H*hd) % 64 == 0.
 */
dg_status dg_out_proj(const uint16_t* h, const uint16_t* O, const uint16_t* Wo, uint16_t* y, int BL,
                      int d, int Hhd, void* stream);

/* ---------------------------------------- fused LM head, posterior and Euler update ----
 * p_hat_0 = Softmax(logits / tau) with logits = y W^T (LM head tied to the embedding), then
 * x_(t-h) ~ Step(x_t, p_hat_0) [TR "디노이징 반복과 self-conditioning", "Backward Denoising
 * Process"], with the reverse step factorised per position.  Per row r (canvas r / L,
 * position r % L), with z~ = z * inv_tau:
 *     lse        = log sum_v exp(z~_v)
 *     top1       = argmax_v z~_v (lowest index on ties);   logp_top1 = z~_top1 - lse
 *     x0hat      = an exact sample of Softmax(z~), by Gumbel-max at two levels over the aligned
 *                  32-entry chunks c of the vocabulary: c* = argmax_c (lse_c + g_c) with
 *                  lse_c = log sum_{v in c} exp(z~_v) and g_c from the chunk Gumbel stream,
 *                  then x0hat = argmax_{v in c*} (z~_v + g'_v) with g'_v from the within-chunk
 *                  Gumbel stream (lowest index on ties at both levels); P(x0hat = v) = p_v.
 *                                                          logp_x0hat = z~_x0hat - lse
 *     entropy    = -sum_v p_v log p_v of p = Softmax(z~) [TR "DiffusionGemma 샘플러"], accumulated
 *                  online in the same pass (log s - t / s with s = sum exp(z~ - m),
 *                  t = sum exp(z~ - m) (z~ - m)), clamped at 0
 * and, when x_in != NULL, the Euler step of dg_euler_update at `step`.  No [rows, V] logit
 * tensor is written to memory.
 *
 *   y [B*L, d] bf16; W [V, d] bf16; x_in [B*L] int32 or NULL (posterior only); x_out [B*L] (may
 *   alias x_in); lock [B*L] uint8 in/out (NULL = nothing locked, no lock state kept);
 *   jump [B*L] uint8 out or NULL; done [B] uint8 out (1 = every position locked) or NULL;
 *   out: optional per-row outputs (each field may be NULL).  jump_thr = floor(lambda * 2^32);
 *   lock_logthr = log(theta) as float, +INFINITY disables locking.  ws: at least
 *   dg_vocab_posterior_workspace(B, L, V) bytes.
 *   Limits: d % 64 == 0, V % 256 == 0, L % 64 == 0, 1 <= L <= 256.
 */
typedef struct {
  int32_t* x0hat;
  int32_t* top1;
  float* logp_top1;
  float* lse;
  float* logp_x0hat;
  float* entropy; /* -sum_v p_v log p_v of Softmax(z~), clamped at 0 */
} dg_posterior_out;

size_t dg_vocab_posterior_workspace(int B, int L, int V);
dg_status dg_vocab_posterior_step(const uint16_t* y, const uint16_t* W, int B, int L, int d, int V,
                                  float inv_tau, uint64_t seed, int step, const int32_t* x_in,
                                  int32_t* x_out, uint8_t* lock, uint8_t* jump, uint8_t* done,
                                  uint64_t jump_thr, float lock_logthr,
                                  const dg_posterior_out* out, void* ws, size_t ws_bytes,
                                  void* stream);

/* Allocation-free variant of dg_vocab_posterior_step.  (The pages have no counterpart: this is
 * a deployment convenience, not a step of the method.)  It is for callers that cannot supply
 * a workspace: code that receives only input and output buffers from a host framework with
 * no handle to its memory pool, processes whose device memory is reserved up front, and
 * loops that must not risk the device synchronisation of cudaMalloc / cudaFree.
 *   - Same arguments, layouts, results and errors as dg_vocab_posterior_step, without ws.
 *   - Scratch lives in one file-scope device array of 16 MiB.  The call allocates nothing (no
 *     cudaMalloc, cudaFree or allocating library routine); it clears the part of the array
 *     that must start at zero.
 *   - The array belongs to a module that CUDA loads lazily (the default module loading): the
 *     first call on each device loads it, which is when the driver reserves the 16 MiB on that
 *     device (held until the process exits), and looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  So that first call can still fail for
 *     lack of memory, or synchronise the device: make it at start-up, before the process
 *     reserves the rest of its device memory and before any stream capture.
 *   - Sizes whose scratch exceeds 16 MiB (about 1,800 canvases of 256 positions or more at a
 *     262,144-token vocabulary on a 152-SM GPU; the need is the dg_vocab_posterior_workspace
 *     size less 256 bytes) return DG_ENOTSUP with a message; use dg_vocab_posterior_step with
 *     a workspace for those.
 *   - Every call shares the one array: calls that may overlap on the GPU (different streams
 *     without ordering between them) race on it.  Order them on one stream.
 *   - Kernel timeouts and out-of-range indices are reported through the library's status word
 *     that every call made without a workspace shares; dg_workspace_status(NULL, stream) reads
 *     and clears it, so read it on the same stream right after the call (another caller's read
 *     would otherwise consume the report, or this call's read could see another call's).
 */
dg_status dg_vocab_posterior_step_noalloc(const uint16_t* y, const uint16_t* W, int B, int L,
                                          int d, int V, float inv_tau, uint64_t seed, int step,
                                          const int32_t* x_in, int32_t* x_out, uint8_t* lock,
                                          uint8_t* jump, uint8_t* done, uint64_t jump_thr,
                                          float lock_logthr, const dg_posterior_out* out,
                                          void* stream);

/* ----------------------------------------------------- Euler jump + lock + commit ----
 * The reverse Step [TR "Backward Denoising Process"] with optional confidence locking
 * [PBD glossary "Iterative denoising"]: per position of every canvas,
 *     already locked                          -> unchanged
 *     logp_top1 >= lock_logthr (float32)      -> lock; x <- top1
 *     jump draw < jump_thr                    -> x <- x0hat, jump = 1
 *     otherwise                               -> unchanged
 * and done[b] = 1 iff every position of canvas b is locked afterwards.
 *
 *   x_in, x0hat, top1 [B, L] int32; logp_top1 [B, L] fp32; x_out [B, L] (may alias x_in);
 *   lock [B, L] uint8 in/out (0/1); jump [B, L] uint8 out or NULL; done [B] uint8 out or NULL.
 *   Limits: 1 <= L <= 1024.
 */
dg_status dg_euler_update(const int32_t* x_in, const int32_t* x0hat, const int32_t* top1,
                          const float* logp_top1, int32_t* x_out, uint8_t* lock, uint8_t* jump,
                          uint8_t* done, int B, int L, uint64_t seed, int step, uint64_t jump_thr,
                          float lock_logthr, void* stream);

/* ------------------------------------------------------- fused SFT cross-entropy ----
 * The training-side twin of the fused LM head [TR "1단계: Supervised Finetuning": L(theta) =
 * - sum_i log p_theta(x_0^i | x_t, c)]: per row r, with z~ = (y W^T) * inv_tau,
 *     loss[r] = lse_r - z~_r[targets[r]]   (= -log Softmax(z~_r)[targets[r]])
 * in one pass over the vocabulary (no Gumbel draws, no [rows, V] logit tensor).
 *   y [B*L, d] bf16; W [V, d] bf16; targets [B*L] int32 in [0, V) (a target outside gives NaN);
 *   loss [B*L] fp32 out; lse [B*L] fp32 out or NULL.  ws: at least
 *   dg_vocab_posterior_workspace(B, L, V) bytes.  Limits: those of dg_vocab_posterior_step.
 */
dg_status dg_cross_entropy_step(const uint16_t* y, const uint16_t* W, int B, int L, int d, int V,
                                float inv_tau, const int32_t* targets, float* loss, float* lse,
                                void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------ entropy-bounded update ----
 * One step of the entropy-bounded sampler [TR "DiffusionGemma 샘플러": "Entropy-bounded 토큰
 * 정제", "Adaptive stopping"], per canvas b:
 *   - positions taken in increasing (entropy, position) order are accepted while the running
 *     float32 sum of their entropies stays <= gamma (possibly none); accepted positions take
 *     x0hat, every other position a fresh uniform token (Philox counter (pos, canvas, 0,
 *     4<<24 | step), word 0, mapped to [0, V) by multiply-shift);
 *   - done[b] = mean entropy < stop_entropy, and prev_top1 != NULL with prev_valid != 0 and
 *     top1 == prev_top1 at every position; the mean is the float32 sum in position order,
 *     divided by L;
 *   - when done[b], or when final_step != 0, the canvas's x_out is its top1 sequence instead;
 *   - prev_top1 (when not NULL) is overwritten with top1 for the next step.
 *
 *   x0hat, top1 [B, L] int32; entropy [B, L] fp32; prev_top1 [B, L] int32 in/out or NULL;
 *   x_out [B, L] int32 (may alias x0hat or top1); accept [B, L] uint8 out or NULL; done [B]
 *   uint8 out or NULL; mean_entropy [B] fp32 out or NULL.  Limits: 1 <= L <= 1024, V >= 1.
 */
dg_status dg_entropy_bounded_update(const int32_t* x0hat, const int32_t* top1,
                                    const float* entropy, int32_t* prev_top1, int prev_valid,
                                    int32_t* x_out, uint8_t* accept, uint8_t* done,
                                    float* mean_entropy, int B, int L, int V, uint64_t seed,
                                    int step, float gamma, float stop_entropy, int final_step,
                                    void* stream);

/* -------------------------------------------------------------------- denoising loop ----
 * Steps n = start_step .. end_step-1 of at most T [TR "디노이징 반복과 self-conditioning";
 * "DiffusionGemma 샘플러": cap T] of
 *     h = E[x]; q,k,v = h Wqkv^T; O = attention(q, prefix KV, canvas KV); y = h + O Wo^T;
 *     posterior + Euler step with jump threshold floor(lambda_n * 2^32),
 * entirely on the device with no host synchronisation between steps [TR "CPU-GPU 동기화
 * 제거"].  When stop_when_all_locked is set, a canvas whose positions are all locked stops
 * (its later steps are skipped), and once every canvas has stopped the remaining kernels
 * return at once.
 * With cfg->sampler = DG_SAMPLER_ENTROPY_BOUNDED the step is instead the posterior at the
 * annealed temperature tau_n followed by dg_entropy_bounded_update; a canvas stops at the first
 * step whose stop test holds, and every canvas ends holding its last top-1 sequence (lock is
 * not used and may be NULL; the run must start at step 0 and cover all T steps).
 *
 *   m: device pointers to the weights (E [V, d] also serves as the LM head) and the sizes;
 *   k_pre, v_pre [B, P, Hkv, hd]; canvas [B, L] int32 in: x_1 (or the state at start_step),
 *   out: final state; lock [B, L] uint8 in/out; steps_taken [B] int32 out (steps applied by
 *   this call).  ws: at least dg_denoise_loop_workspace(m, B, L, P, window) bytes.
 *   Limits: those of the calls above.  end_step <= 0 means T.
 */
typedef struct {
  const uint16_t* E;
  const uint16_t* Wqkv;
  const uint16_t* Wo;
  int V, d, H, Hkv, hd;
  /* Self-conditioning feed-forward [TR "디노이징 반복과 self-conditioning"]: Wsc1 [d_sc, d],
   * Wsc2 [d, d_sc] bf16, or both NULL (and d_sc = 0) for a decoder without it.  With it, each
   * step's tempered posterior p_hat gives s = bf16(bf16(gelu(bf16(p_hat E) Wsc1^T)) Wsc2^T)
   * (tanh-form GELU), and the next step's embeddings are h = bf16(E[x] + s); s is zero at
   * step 0.  Needs d % 256 == 0 and d_sc % 64 == 0. */
  const uint16_t* Wsc1;
  const uint16_t* Wsc2;
  int d_sc;
} dg_model;

typedef enum {
  DG_SAMPLER_EULER = 0,           /* Euler step with optional locking (the fields above) */
  DG_SAMPLER_ENTROPY_BOUNDED = 1  /* entropy-bounded sampler with annealing and stopping */
} dg_sampler;

typedef struct {
  int T;                    /* number of steps of the schedule (h = 1/T); the cap for EB */
  int schedule;             /* dg_schedule (Euler) */
  float inv_tau;            /* 1 / temperature (Euler) */
  float lock_logthr;        /* log(theta) as float; +INFINITY disables locking (Euler) */
  uint64_t seed;
  int start_step;           /* first step to run (resume; 0 for the entropy-bounded sampler) */
  int end_step;             /* one past the last step to run; <= 0 means T */
  int stop_when_all_locked; /* nonzero: a fully locked canvas stops (Euler) */
  int sampler;              /* dg_sampler */
  double tau_start;         /* entropy-bounded: temperature of step 0 ... */
  double tau_end;           /* ... and of step T-1; tau_n = tau_start + (tau_end - tau_start) * n
                               / (T - 1) in double, handed to the kernels as float(1 / tau_n) */
  float gamma;              /* entropy budget of the accepted positions */
  float stop_entropy;       /* adaptive-stopping threshold on the mean entropy */
} dg_sampler_cfg;

/* Bytes of device workspace dg_denoise_loop (and dg_sft_loss, dg_block_generate's loop part)
 * needs: the status word, activations, attention and vocabulary partials, the fp32 partials of
 * the split-K projections (present when one launch of them would not fill the GPU, as for one
 * canvas) and, with self-conditioning, its buffers.  Depends on the device's SM count.  Host
 * only. */
size_t dg_denoise_loop_workspace(const dg_model* m, int B, int L, int P, int window);

/* Number of kernels one dg_denoise_loop call with the Euler sampler launches for `steps` steps
 * on this device (its launch plan depends on the SM count); -1 on invalid arguments.  (The
 * entropy-bounded sampler adds its update kernel per step and, without self-conditioning,
 * steps - 1 finalisation launches that the Euler loop folds into its embedding launches.)
 * Host only. */
int dg_denoise_loop_kernel_count(const dg_model* m, int B, int L, int P, int window, int steps);
dg_status dg_denoise_loop(const dg_model* m, const uint16_t* k_pre, const uint16_t* v_pre, int B,
                          int L, int P, int window, int32_t* canvas, uint8_t* lock,
                          int32_t* steps_taken, const dg_sampler_cfg* cfg, void* ws,
                          size_t ws_bytes, void* stream);

/* ------------------------------------------------------- SFT loss on noised canvases ----
 * The SFT loss on noised canvases: x_t = dg_forward_noise(x_0, keep_thr, seed) (per-canvas keep
 * thresholds floor(kappa(t_b) * 2^32); the report draws t_b ~ Unif[0, 1]), the stand-in decoder
 * on x_t with the prefix KV, and loss = dg_cross_entropy_step against x_0.
 *   x0 [B, L] int32; keep_thr [B] uint64 (device); xt [B, L] int32 out; loss [B, L] fp32 out.
 *   ws: at least dg_denoise_loop_workspace(m, B, L, P, window) bytes.  Limits: those of
 *   dg_denoise_loop.
 */
dg_status dg_sft_loss(const dg_model* m, const uint16_t* k_pre, const uint16_t* v_pre, int B,
                      int L, int P, int window, const int32_t* x0, const uint64_t* keep_thr,
                      uint64_t seed, float inv_tau, int32_t* xt, float* loss, void* ws,
                      size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ self-conditioning ----
 * s_(t-h) = FFW(p_hat_0 . E) [TR "디노이징 반복과 self-conditioning"], alone (the denoising loop
 * runs the same kernels when the model carries Wsc1/Wsc2):
 *   p_hat = Softmax(y E^T * inv_tau) per row; e = bf16(p_hat E); u = bf16(gelu(e Wsc1^T))
 *   (tanh-form GELU); s = bf16(u Wsc2^T).
 * The LM-head pass stores bf16 exp(z~ - m) (m: its running maximum, recorded per 32 entries),
 * rescales it by exp(m - lse) once lse is known, and contracts it with E on the tensor cores
 * (split over the vocabulary, partial sums added in a fixed order: deterministic).
 *   y [B*L, d], E [V, d], Wsc1 [d_sc, d], Wsc2 [d, d_sc] bf16 (device); s_out [B*L, d] bf16
 *   out; e_out [B*L, d] bf16 out or NULL.  ws: at least dg_self_condition_workspace(B, L, d,
 *   V, d_sc) bytes (status word first; it holds B*L*V*2 bytes of posterior).
 *   Limits: d % 256 == 0, V % 256 == 0, d_sc % 64 == 0, L a multiple of 64 up to 256.
 */
size_t dg_self_condition_workspace(int B, int L, int d, int V, int d_sc);
dg_status dg_self_condition(const uint16_t* y, const uint16_t* E, const uint16_t* Wsc1,
                            const uint16_t* Wsc2, int B, int L, int d, int V, int d_sc,
                            float inv_tau, uint16_t* s_out, uint16_t* e_out, void* ws,
                            size_t ws_bytes, void* stream);

/* ------------------------------------------------- encode-append and block-AR loop ----
 * [TR "블록 자기회귀(Block-AR) 생성": context encoding, denoising loop, encode-append, repeated
 * until the end-of-turn token; "추론 효율 지표": one extra forward between canvases.]
 *
 * dg_encode_append: the finished canvas goes through the causal encoder and its keys and
 * values are appended to the prefix cache.  For the one-layer stand-in decoder a token's key
 * and value are its own projections, k = E[x] Wk^T, v = E[x] Wv^T (bf16; Wk, Wv are the K and
 * V row blocks of Wqkv), so the causal pass is the K/V part of the fused projection.  They are
 * written at cache rows P .. P+L-1 of every canvas b with active[b] != 0 (all when active is
 * NULL); other rows are not touched.
 *   canvas [B, L] int32 (device); k_cache, v_cache [B, P_cap, Hkv, hd] bf16 in/out; active [B]
 *   uint8 or NULL.  ws: at least dg_encode_append_workspace(m, B, L) bytes, status word first.
 *   Limits: P + L <= P_cap; B * P_cap < 2^31; the model limits of dg_denoise_loop.
 *
 * dg_block_generate: block-AR generation for B independent conversations.  On entry cache rows
 * 0 .. P0-1 hold the encoded context.  For block j = 0 .. NB-1, while the conversation has not
 * ended:
 *   - the canvas starts from the uniform prior x_1 drawn with key cfg->seed + j (dg_forward_noise
 *     with keep threshold 0);
 *   - dg_denoise_loop runs all T steps of cfg (either sampler, key cfg->seed + j, lock cleared)
 *     with the P0 + j*L cache rows as prefix;
 *   - the finished canvas is written to out[b, j, :] and encode-appended at rows P0 + j*L;
 *   - if it holds the end-of-turn token `eos`, the conversation ends: its response is the
 *     tokens up to and including the first `eos`.
 * Outputs: out [B, NB, L] int32 (-1 in blocks never generated); blocks [B] = canvases
 * generated; n_tokens [B] = response length (j*L + i + 1 for the first eos at position i of
 * block j, else blocks * L); steps [B] = denoising steps summed over the canvases (the
 * sum s_k of the throughput metrics).  All device, int32.  Everything stays on the device;
 * the host enqueues NB blocks and does not wait: blocks after every conversation ended
 * return at once.
 *   k_cache, v_cache [B, P_cap, Hkv, hd] bf16 in/out (rows P0 .. P0 + blocks*L - 1 written).
 *   ws: at least dg_block_generate_workspace(m, B, L, P0, NB, window) bytes, status word first.
 *   Limits: P0 + NB*L <= P_cap; cfg runs steps 0 .. T-1; those of dg_denoise_loop.
 */
size_t dg_encode_append_workspace(const dg_model* m, int B, int L);
dg_status dg_encode_append(const dg_model* m, const int32_t* canvas, uint16_t* k_cache,
                           uint16_t* v_cache, int B, int L, int P, int P_cap,
                           const uint8_t* active, void* ws, size_t ws_bytes, void* stream);
size_t dg_block_generate_workspace(const dg_model* m, int B, int L, int P0, int NB, int window);
dg_status dg_block_generate(const dg_model* m, uint16_t* k_cache, uint16_t* v_cache, int B, int P0,
                            int P_cap, int L, int NB, int window, int32_t eos,
                            const dg_sampler_cfg* cfg, int32_t* out, int32_t* blocks,
                            int32_t* n_tokens, int32_t* steps, void* ws, size_t ws_bytes,
                            void* stream);

/* ----------------------------------------------------------------- status and timing ----
 * dg_workspace_status: synchronises `stream`, reads and clears the status word at the start
 * of a workspace used by dg_canvas_attn, dg_vocab_posterior_step, dg_denoise_loop,
 * dg_encode_append, dg_block_generate or dg_self_condition (ws = NULL: the library's word
 * shared by every call made without a workspace), and returns DG_OK, DG_ETIMEOUT (a kernel
 * gave up waiting on an on-chip barrier) or DG_EKERNEL (a kernel met an out-of-range token
 * id) accordingly, DG_ECUDA if the stream failed.
 *
 * dg_set_wait_control: the limit, in nanoseconds, of every on-chip barrier wait in the
 * kernels the calling thread enqueues from now on (0 = the default 2 s; at most 60 s, else
 * DG_EINVAL).  A wait that runs out raises the CTA's abort flag; the CTA's other waits then
 * give up at once, the kernel drains what it has in flight (bounded), frees its tensor memory
 * and returns, and the status word reports DG_ETIMEOUT.  skip_loads != 0 (for tests of that
 * path) makes the LM-head kernel's load warps issue nothing, so its consumers' waits run out
 * with no copy or tensor-core operation in flight; its results are then meaningless.  The
 * setting is thread-local and stays until changed.
 *
 * dg_kernel_timer_enable(1) makes the library record CUDA events on the launching stream
 * around every launch of its LM-head/posterior kernel (kind 0), attention kernels (kind 1),
 * self-conditioning contraction (kind 2), projection GEMMs (kind 3) and posterior
 * finalisation (kind 4);
 * dg_kernel_timer_read synchronises those events and returns the summed milliseconds and the
 * number of launches since the last reset; dg_kernel_timer_enable(0) stops and resets.
 */
dg_status dg_workspace_status(const void* ws, void* stream);
dg_status dg_set_wait_control(uint64_t limit_ns, int skip_loads);
dg_status dg_kernel_timer_enable(int enable);
dg_status dg_kernel_timer_read(int kind, double* total_ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* DGCANVAS_H */
