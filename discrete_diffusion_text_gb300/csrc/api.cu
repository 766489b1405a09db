// C ABI of libdgcanvas: argument validation, workspace layout, schedules and the denoising
// loop.  Every step of the path runs in the library's own kernels.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "dg_common.cuh"
#include "kernels.cuh"

namespace dg {

// --------------------------------------------------------------------- errors -----

static thread_local std::string g_last_error = "ok";

void set_error(const std::string& msg) { g_last_error = msg; }

dg_status fail(dg_status code, const std::string& msg) {
  set_error(msg);
  return code;
}

dg_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DG_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// ------------------------------------------------------------- device properties -----

int device_id() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

int num_sms() {
  static std::mutex mu;
  static std::vector<int> cache;
  const int d = device_id();
  std::lock_guard<std::mutex> lk(mu);
  if (static_cast<int>(cache.size()) <= d) cache.resize(d + 1, 0);
  if (cache[d] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0)
      n = 1;
    cache[d] = n;
  }
  return cache[d];
}

// ----------------------------------------------------------------- bounded waits -----

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
constexpr uint64_t kMaxWaitNs = 60000000000ull;     // 60 s
static thread_local uint64_t g_wait_limit_ns = kDefaultWaitNs;
static thread_local bool g_wait_skip_loads = false;

uint64_t wait_limit_ns() { return g_wait_limit_ns; }
bool wait_test_skip_loads() { return g_wait_skip_loads; }

// Library-owned status word for calls that take no workspace.
__device__ uint32_t g_fallback_status_word;

uint32_t* status_or_fallback(uint32_t* status) {
  if (status) return status;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fallback_status_word) != cudaSuccess) return nullptr;
  return static_cast<uint32_t*>(p);
}

// -------------------------------------------------------------------- tensor maps -----

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5];
  cuuint32_t es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                        const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------- kernel timer -----

namespace {
struct TimerRec {
  int kind;
  cudaEvent_t start, stop;
};
std::mutex g_timer_mu;
bool g_timer_on = false;
std::vector<cudaEvent_t> g_timer_pool;
std::vector<TimerRec> g_timer_recs;
cudaEvent_t g_timer_open[kTimerKinds] = {};

cudaEvent_t timer_event() {
  if (!g_timer_pool.empty()) {
    cudaEvent_t e = g_timer_pool.back();
    g_timer_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void timer_reset_locked() {
  for (auto& r : g_timer_recs) {
    g_timer_pool.push_back(r.start);
    g_timer_pool.push_back(r.stop);
  }
  g_timer_recs.clear();
  for (auto& e : g_timer_open)
    if (e) {
      g_timer_pool.push_back(e);
      e = nullptr;
    }
}
}  // namespace

void timer_begin(int kind, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_timer_mu);
  if (!g_timer_on) return;
  cudaEvent_t e = timer_event();
  cudaEventRecord(e, st);
  g_timer_open[kind] = e;
}

void timer_end(int kind, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_timer_mu);
  if (!g_timer_on || !g_timer_open[kind]) return;
  cudaEvent_t e = timer_event();
  cudaEventRecord(e, st);
  g_timer_recs.push_back({kind, g_timer_open[kind], e});
  g_timer_open[kind] = nullptr;
}

// ------------------------------------------------------------------ schedules -----

static bool schedule_rate(int schedule, int T, int n, double* lam) {
  const double t = static_cast<double>(T - n) / T;
  const double h = 1.0 / T;
  double v;
  if (schedule == DG_SCHED_LINEAR) {
    v = h / t;  // -kappa' = 1, 1 - kappa = t
  } else if (schedule == DG_SCHED_COSINE) {
    const double x = 0.5 * M_PI * t;
    v = h * (M_PI * std::cos(x) * std::sin(x)) / (std::sin(x) * std::sin(x));
  } else {
    return false;
  }
  *lam = v < 1.0 ? (v > 0.0 ? v : 0.0) : 1.0;
  return true;
}

static bool schedule_kappa(int schedule, double t, double* k) {
  if (schedule == DG_SCHED_LINEAR) {
    *k = 1.0 - t;
  } else if (schedule == DG_SCHED_COSINE) {
    const double c = std::cos(0.5 * M_PI * t);
    *k = c * c;
  } else {
    return false;
  }
  return true;
}

static uint64_t prob_threshold(double p) {
  if (!(p > 0.0)) return 0;
  if (p >= 1.0) return 1ull << 32;
  return static_cast<uint64_t>(std::floor(p * 4294967296.0));
}

}  // namespace dg

using namespace dg;

namespace {

constexpr size_t kStatusBytes = 256;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool bad_ptr(const void* p) { return p == nullptr || !aligned16(p); }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

dg_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DG_OK;
}

// Loop workspace regions (all 256-byte aligned).
struct LoopWs {
  uint32_t* status;
  uint8_t* active;
  int* n_active;
  int* counters;  // [2B]: the finalisation's per-canvas tickets (B 64-bit words)
  uint16_t *h, *q, *k, *v, *o, *y;
  void* attn;
  void* gemm_part;  // fp32 split-K partials of the projections
  size_t gemm_part_bytes;
  VocabPart* parts;
  int32_t *x0hat, *top1, *prev_top1;  // entropy-bounded sampler
  float* entropy;
  // self-conditioning (empty without it): bf16 exp(z~ - m_ref) [BL, V], m_ref [BL, V/32],
  // lse [BL], split partials, e [BL, d], u [BL, d_sc] and the signal s [BL, d], which stays
  // in the workspace between calls so that a split run resumes with it
  uint16_t* sc_p;
  float *sc_m, *sc_lse, *sc_part;
  uint16_t *sc_e, *sc_u, *sc_s;
  size_t total;
};

bool has_sc(const dg_model* m) { return m->Wsc1 != nullptr; }

GemmOut qkv_segments(const dg_model* m) {
  GemmOut o{};
  o.nseg = 3;
  o.seg_begin[0] = 0;
  o.seg_begin[1] = m->H * m->hd;
  o.seg_begin[2] = (m->H + m->Hkv) * m->hd;
  o.seg_begin[3] = (m->H + 2 * m->Hkv) * m->hd;
  return o;
}

// Workspace of the split-K partials of the two projections of BL canvas rows.
size_t proj_part_bytes(const dg_model* m, int BL) {
  const int Hhd = m->H * m->hd;
  const GemmOut qkv = qkv_segments(m);
  GemmOut yo{};
  yo.nseg = 1;
  yo.seg_begin[1] = m->d;
  return std::max(plan_gemm(BL, qkv.seg_begin[3], m->d, qkv).part_bytes,
                  plan_gemm(BL, m->d, Hhd, yo).part_bytes);
}

LoopWs loop_layout(const dg_model* m, int B, int L, int P, int window, uint8_t* base) {
  LoopWs w{};
  const size_t BL = static_cast<size_t>(B) * L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off += align256(bytes);
    return p;
  };
  w.status = reinterpret_cast<uint32_t*>(take(kStatusBytes));
  w.active = take(B);
  w.n_active = reinterpret_cast<int*>(take(sizeof(int)));
  w.counters = reinterpret_cast<int*>(take(2 * sizeof(int) * static_cast<size_t>(B)));
  w.h = reinterpret_cast<uint16_t*>(take(BL * m->d * 2));
  w.q = reinterpret_cast<uint16_t*>(take(BL * m->H * m->hd * 2));
  w.k = reinterpret_cast<uint16_t*>(take(BL * m->Hkv * m->hd * 2));
  w.v = reinterpret_cast<uint16_t*>(take(BL * m->Hkv * m->hd * 2));
  w.o = reinterpret_cast<uint16_t*>(take(BL * m->H * m->hd * 2));
  w.y = reinterpret_cast<uint16_t*>(take(BL * m->d * 2));
  const AttnPlan ap = plan_attention(B, L, P, m->H, m->Hkv, m->hd, window);
  w.attn = take(ap.part_bytes > 0 ? ap.part_bytes : 16);
  w.gemm_part_bytes = proj_part_bytes(m, static_cast<int>(BL));
  w.gemm_part = take(w.gemm_part_bytes > 0 ? w.gemm_part_bytes : 16);
  const VocabPlan vp = plan_vocab(static_cast<int>(BL), m->V);
  w.parts = reinterpret_cast<VocabPart*>(take(vp.part_bytes));
  w.x0hat = reinterpret_cast<int32_t*>(take(BL * 4));
  w.top1 = reinterpret_cast<int32_t*>(take(BL * 4));
  w.prev_top1 = reinterpret_cast<int32_t*>(take(BL * 4));
  w.entropy = reinterpret_cast<float*>(take(BL * 4));
  if (has_sc(m)) {
    const ScPlan sp = plan_selfcond(static_cast<int>(BL), m->V, m->d);
    w.sc_s = reinterpret_cast<uint16_t*>(take(BL * m->d * 2));
    w.sc_p = reinterpret_cast<uint16_t*>(take(BL * m->V * 2));
    w.sc_m = reinterpret_cast<float*>(take(BL * (m->V / 32) * 4));
    w.sc_lse = reinterpret_cast<float*>(take(BL * 4));
    w.sc_part = reinterpret_cast<float*>(take(sp.part_bytes));
    w.sc_e = reinterpret_cast<uint16_t*>(take(BL * m->d * 2));
    w.sc_u = reinterpret_cast<uint16_t*>(take(BL * m->d_sc * 2));
  }
  w.total = off;
  return w;
}

dg_status check_attn_dims(int B, int L, int P, int H, int Hkv, int hd, int window) {
  if (B < 0 || L <= 0 || P < 0 || H <= 0 || Hkv <= 0 || window < 0)
    return fail(DG_EINVAL, "attention: negative or zero size");
  if (L > 256 || L % 64 != 0) return fail(DG_ENOTSUP, "attention: L must be 64, 128, 192 or 256");
  if (hd != 64 && hd != 128) return fail(DG_ENOTSUP, "attention: hd must be 64 or 128");
  if (H % Hkv != 0) return fail(DG_EINVAL, "attention: H must be a multiple of Hkv");
  if (static_cast<int64_t>(B) * H * ((L + 127) / 128) > 0x7FFFFFFF)
    return fail(DG_ENOTSUP, "attention: too many query tiles");
  return DG_OK;
}

dg_status check_model(const dg_model* m) {
  if (!m) return fail(DG_EINVAL, "model: NULL");
  if (bad_ptr(m->E) || bad_ptr(m->Wqkv) || bad_ptr(m->Wo))
    return fail(DG_EINVAL, "model: NULL or misaligned weight pointer");
  if (m->V <= 0 || m->d <= 0 || m->H <= 0 || m->Hkv <= 0)
    return fail(DG_EINVAL, "model: non-positive size");
  if (m->d % 64 != 0) return fail(DG_ENOTSUP, "model: d must be a multiple of 64");
  if (m->V % 256 != 0) return fail(DG_ENOTSUP, "model: V must be a multiple of 256");
  if (m->hd != 64 && m->hd != 128) return fail(DG_ENOTSUP, "model: hd must be 64 or 128");
  if (m->H % m->Hkv != 0) return fail(DG_EINVAL, "model: H must be a multiple of Hkv");
  if (m->Wsc1 != nullptr || m->Wsc2 != nullptr || m->d_sc != 0) {
    if (bad_ptr(m->Wsc1) || bad_ptr(m->Wsc2) || m->d_sc <= 0)
      return fail(DG_EINVAL, "model: self-conditioning needs Wsc1, Wsc2 and d_sc > 0");
    if (m->d_sc % 64 != 0) return fail(DG_ENOTSUP, "model: d_sc must be a multiple of 64");
    if (m->d % 256 != 0)
      return fail(DG_ENOTSUP, "model: self-conditioning needs d to be a multiple of 256");
  }
  return DG_OK;
}

}  // namespace

extern "C" {

const char* dg_last_error(void) { return g_last_error.c_str(); }

int dg_abi_version(void) { return 3; }

dg_status dg_schedule_thresholds(int schedule, int T, uint64_t* keep_thr, uint64_t* jump_thr) {
  if (T < 1) return fail(DG_EINVAL, "schedule: T must be >= 1");
  if (schedule != DG_SCHED_LINEAR && schedule != DG_SCHED_COSINE)
    return fail(DG_EINVAL, "schedule: unknown schedule");
  for (int n = 0; n <= T; ++n) {
    double k;
    schedule_kappa(schedule, static_cast<double>(T - n) / T, &k);
    if (keep_thr) keep_thr[n] = prob_threshold(k);
    if (jump_thr && n < T) {
      double lam;
      schedule_rate(schedule, T, n, &lam);
      jump_thr[n] = prob_threshold(lam);
    }
  }
  return DG_OK;
}

dg_status dg_keep_thresholds(int schedule, const double* t, int B, uint64_t* keep_thr) {
  if (B < 0 || (B > 0 && (!t || !keep_thr))) return fail(DG_EINVAL, "keep thresholds: bad arrays");
  if (schedule != DG_SCHED_LINEAR && schedule != DG_SCHED_COSINE)
    return fail(DG_EINVAL, "keep thresholds: unknown schedule");
  for (int b = 0; b < B; ++b) {
    if (!(t[b] >= 0.0 && t[b] <= 1.0)) return fail(DG_EINVAL, "keep thresholds: t outside [0, 1]");
    double k;
    schedule_kappa(schedule, t[b], &k);
    keep_thr[b] = prob_threshold(k);
  }
  return DG_OK;
}

dg_status dg_forward_noise(const int32_t* x0, int32_t* xt, const uint64_t* keep_thr, int B, int L,
                           int V, uint64_t seed, void* stream) {
  if (B < 0 || L < 0 || V < 1) return fail(DG_EINVAL, "forward_noise: bad sizes");
  if (static_cast<int64_t>(B) * L >= (1ll << 31)) return fail(DG_ENOTSUP, "forward_noise: too large");
  if (static_cast<int64_t>(B) * L == 0) return DG_OK;
  if (bad_ptr(x0) || bad_ptr(xt) || keep_thr == nullptr || (reinterpret_cast<uintptr_t>(keep_thr) & 7))
    return fail(DG_EINVAL, "forward_noise: NULL or misaligned pointer");
  launch_forward_noise(x0, xt, keep_thr, B, L, V, seed, as_stream(stream));
  return check_launch("forward_noise launch");
}

dg_status dg_embed_qkv(const int32_t* x, const uint16_t* E, const uint16_t* Wqkv, uint16_t* h,
                       uint16_t* q, uint16_t* k, uint16_t* v, int BL, int V, int d, int H,
                       int Hkv, int hd, void* stream) {
  if (BL < 0 || V <= 0 || d <= 0 || H <= 0 || Hkv <= 0) return fail(DG_EINVAL, "embed_qkv: bad sizes");
  if (d % 64 != 0) return fail(DG_ENOTSUP, "embed_qkv: d must be a multiple of 64");
  if (hd != 64 && hd != 128) return fail(DG_ENOTSUP, "embed_qkv: hd must be 64 or 128");
  if (H % Hkv != 0) return fail(DG_EINVAL, "embed_qkv: H must be a multiple of Hkv");
  if (BL == 0) return DG_OK;
  if (bad_ptr(x) || bad_ptr(E) || bad_ptr(Wqkv) || bad_ptr(h) || bad_ptr(q) || bad_ptr(k) || bad_ptr(v))
    return fail(DG_EINVAL, "embed_qkv: NULL or misaligned pointer");
  cudaStream_t st = as_stream(stream);
  launch_embed_gather(x, E, h, BL, V, d, nullptr, st, nullptr);
  dg_status s = check_launch("embed gather launch");
  if (s != DG_OK) return s;
  GemmOut out{};
  out.nseg = 3;
  out.seg_begin[0] = 0;
  out.seg_begin[1] = H * hd;
  out.seg_begin[2] = (H + Hkv) * hd;
  out.seg_begin[3] = (H + 2 * Hkv) * hd;
  out.ptr[0] = q;
  out.ptr[1] = k;
  out.ptr[2] = v;
  out.ld[0] = H * hd;
  out.ld[1] = Hkv * hd;
  out.ld[2] = Hkv * hd;
  const cudaError_t e = launch_gemm(h, Wqkv, BL, (H + 2 * Hkv) * hd, d, out, nullptr, 0,
                                    status_or_fallback(nullptr), nullptr, st);
  if (e != cudaSuccess) return cuda_fail(e, "qkv gemm launch");
  return DG_OK;
}

size_t dg_canvas_attn_workspace(int B, int L, int P, int H, int Hkv, int hd, int window) {
  if (B < 0 || L <= 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || (hd != 64 && hd != 128))
    return kStatusBytes;
  return kStatusBytes + align256(plan_attention(B, L, P, H, Hkv, hd, window).part_bytes);
}

dg_status dg_canvas_attn(const uint16_t* q, const uint16_t* k_pre, const uint16_t* v_pre,
                         const uint16_t* k_can, const uint16_t* v_can, uint16_t* out, float* lse,
                         int B, int L, int P, int H, int Hkv, int hd, int window, float scale,
                         void* ws, size_t ws_bytes, void* stream) {
  dg_status s = check_attn_dims(B, L, P, H, Hkv, hd, window);
  if (s != DG_OK) return s;
  if (B == 0) return DG_OK;
  if (bad_ptr(q) || bad_ptr(k_can) || bad_ptr(v_can) || bad_ptr(out) || bad_ptr(ws))
    return fail(DG_EINVAL, "attention: NULL or misaligned pointer");
  if (P > 0 && (bad_ptr(k_pre) || bad_ptr(v_pre)))
    return fail(DG_EINVAL, "attention: NULL or misaligned prefix pointer");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3)) return fail(DG_EINVAL, "attention: misaligned lse");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(DG_EINVAL, "attention: bad scale");
  if (ws_bytes < dg_canvas_attn_workspace(B, L, P, H, Hkv, hd, window))
    return fail(DG_EINVAL, "attention: workspace too small");
  uint8_t* w = static_cast<uint8_t*>(ws);
  const cudaError_t e = launch_attention(q, k_pre, v_pre, k_can, v_can, out, lse, B, L, P, H, Hkv,
                                         hd, window, scale, w + kStatusBytes,
                                         reinterpret_cast<uint32_t*>(w), nullptr, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return DG_OK;
}

dg_status dg_out_proj(const uint16_t* h, const uint16_t* O, const uint16_t* Wo, uint16_t* y, int BL,
                      int d, int Hhd, void* stream) {
  if (BL < 0 || d <= 0 || Hhd <= 0) return fail(DG_EINVAL, "out_proj: bad sizes");
  if (d % 64 != 0 || Hhd % 64 != 0) return fail(DG_ENOTSUP, "out_proj: sizes must be multiples of 64");
  if (BL == 0) return DG_OK;
  if (bad_ptr(h) || bad_ptr(O) || bad_ptr(Wo) || bad_ptr(y)) return fail(DG_EINVAL, "out_proj: bad pointer");
  if (y == h) return fail(DG_EINVAL, "out_proj: y must not alias h");
  GemmOut out{};
  out.nseg = 1;
  out.seg_begin[0] = 0;
  out.seg_begin[1] = d;
  out.ptr[0] = y;
  out.ld[0] = d;
  const cudaError_t e = launch_gemm(O, Wo, BL, d, Hhd, out, h, d, status_or_fallback(nullptr),
                                    nullptr, as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "out_proj gemm launch");
  return DG_OK;
}

size_t dg_vocab_posterior_workspace(int B, int L, int V) {
  if (B <= 0 || L <= 0 || V < 256) return kStatusBytes;
  return kStatusBytes + align256(2 * sizeof(int) * static_cast<size_t>(B)) +
         align256(plan_vocab(B * L, V).part_bytes);
}

dg_status dg_vocab_posterior_step(const uint16_t* y, const uint16_t* W, int B, int L, int d, int V,
                                  float inv_tau, uint64_t seed, int step, const int32_t* x_in,
                                  int32_t* x_out, uint8_t* lock, uint8_t* jump, uint8_t* done,
                                  uint64_t jump_thr, float lock_logthr,
                                  const dg_posterior_out* out, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (B < 0 || L <= 0 || d <= 0 || V <= 0) return fail(DG_EINVAL, "vocab_posterior: bad sizes");
  if (d % 64 != 0) return fail(DG_ENOTSUP, "vocab_posterior: d must be a multiple of 64");
  if (V % 256 != 0) return fail(DG_ENOTSUP, "vocab_posterior: V must be a multiple of 256");
  if (L > 256 || L % 64 != 0) return fail(DG_ENOTSUP, "vocab_posterior: L must be 64..256, multiple of 64");
  if (step < 0 || step >= (1 << 24)) return fail(DG_EINVAL, "vocab_posterior: step out of range");
  if (!(inv_tau > 0.f) || !std::isfinite(inv_tau)) return fail(DG_EINVAL, "vocab_posterior: bad inv_tau");
  if (jump_thr > (1ull << 32)) return fail(DG_EINVAL, "vocab_posterior: jump_thr above 2^32");
  if (static_cast<int64_t>(B) * L >= (1ll << 31)) return fail(DG_ENOTSUP, "vocab_posterior: too many rows");
  if (B == 0) return DG_OK;
  if (bad_ptr(y) || bad_ptr(W) || bad_ptr(ws)) return fail(DG_EINVAL, "vocab_posterior: bad pointer");
  if (x_in && !x_out) return fail(DG_EINVAL, "vocab_posterior: x_out required with x_in");
  if (ws_bytes < dg_vocab_posterior_workspace(B, L, V))
    return fail(DG_EINVAL, "vocab_posterior: workspace too small");
  cudaStream_t st = as_stream(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(w);
  int* counters = reinterpret_cast<int*>(w + kStatusBytes);
  VocabPart* parts = reinterpret_cast<VocabPart*>(
      w + kStatusBytes + align256(2 * sizeof(int) * static_cast<size_t>(B)));
  {
    const cudaError_t em = cudaMemsetAsync(counters, 0, 2 * sizeof(int) * B, st);
    if (em != cudaSuccess) return cuda_fail(em, "vocab_posterior: memset");
  }
  const VocabPlan vp = plan_vocab(B * L, V);
  cudaError_t e = launch_vocab_pass(y, W, B * L, L, d, V, inv_tau, seed, step, parts, status,
                                    nullptr, st, nullptr, out && out->entropy);
  if (e != cudaSuccess) return cuda_fail(e, "vocab pass launch");
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
  return check_launch("vocab finalize launch");
}

dg_status dg_cross_entropy_step(const uint16_t* y, const uint16_t* W, int B, int L, int d, int V,
                                float inv_tau, const int32_t* targets, float* loss, float* lse,
                                void* ws, size_t ws_bytes, void* stream) {
  if (B < 0 || L <= 0 || d <= 0 || V <= 0) return fail(DG_EINVAL, "cross_entropy: bad sizes");
  if (d % 64 != 0) return fail(DG_ENOTSUP, "cross_entropy: d must be a multiple of 64");
  if (V % 256 != 0) return fail(DG_ENOTSUP, "cross_entropy: V must be a multiple of 256");
  if (L > 256 || L % 64 != 0) return fail(DG_ENOTSUP, "cross_entropy: L must be 64..256, multiple of 64");
  if (!(inv_tau > 0.f) || !std::isfinite(inv_tau)) return fail(DG_EINVAL, "cross_entropy: bad inv_tau");
  if (static_cast<int64_t>(B) * L >= (1ll << 31)) return fail(DG_ENOTSUP, "cross_entropy: too many rows");
  if (B == 0) return DG_OK;
  if (bad_ptr(y) || bad_ptr(W) || bad_ptr(ws) || bad_ptr(targets) || !loss)
    return fail(DG_EINVAL, "cross_entropy: NULL or misaligned pointer");
  if (ws_bytes < dg_vocab_posterior_workspace(B, L, V))
    return fail(DG_EINVAL, "cross_entropy: workspace too small");
  cudaStream_t st = as_stream(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(w);
  int* counters = reinterpret_cast<int*>(w + kStatusBytes);
  VocabPart* parts = reinterpret_cast<VocabPart*>(
      w + kStatusBytes + align256(2 * sizeof(int) * static_cast<size_t>(B)));
  const cudaError_t em = cudaMemsetAsync(counters, 0, 2 * sizeof(int) * B, st);
  if (em != cudaSuccess) return cuda_fail(em, "cross_entropy: memset");
  const VocabPlan vp = plan_vocab(B * L, V);
  cudaError_t e = launch_vocab_pass(y, W, B * L, L, d, V, inv_tau, 0, 0, parts, status, nullptr,
                                    st, targets);
  if (e != cudaSuccess) return cuda_fail(e, "cross_entropy: vocab pass launch");
  FinalizeParams fp{};
  fp.parts = parts;
  fp.num_mt = vp.num_mt;
  fp.S = vp.S;
  fp.L = L;
  fp.out_lse = lse;
  fp.out_loss = loss;
  fp.ticket = reinterpret_cast<unsigned long long*>(counters);
  launch_vocab_finalize(fp, B, st);
  return check_launch("cross_entropy: finalize launch");
}

dg_status dg_sft_loss(const dg_model* m, const uint16_t* k_pre, const uint16_t* v_pre, int B,
                      int L, int P, int window, const int32_t* x0, const uint64_t* keep_thr,
                      uint64_t seed, float inv_tau, int32_t* xt, float* loss, void* ws,
                      size_t ws_bytes, void* stream) {
  dg_status s = check_model(m);
  if (s != DG_OK) return s;
  s = check_attn_dims(B, L, P, m->H, m->Hkv, m->hd, window);
  if (s != DG_OK) return s;
  if (!(inv_tau > 0.f) || !std::isfinite(inv_tau)) return fail(DG_EINVAL, "sft_loss: bad inv_tau");
  if (static_cast<int64_t>(B) * L >= (1ll << 31)) return fail(DG_ENOTSUP, "sft_loss: too many rows");
  if (B == 0) return DG_OK;
  if (bad_ptr(x0) || bad_ptr(xt) || bad_ptr(ws) || !loss || keep_thr == nullptr ||
      (reinterpret_cast<uintptr_t>(keep_thr) & 7))
    return fail(DG_EINVAL, "sft_loss: NULL or misaligned pointer");
  if (P > 0 && (bad_ptr(k_pre) || bad_ptr(v_pre))) return fail(DG_EINVAL, "sft_loss: bad prefix pointer");
  if (ws_bytes < dg_denoise_loop_workspace(m, B, L, P, window))
    return fail(DG_EINVAL, "sft_loss: workspace too small");
  cudaStream_t st = as_stream(stream);
  const LoopWs w = loop_layout(m, B, L, P, window, static_cast<uint8_t*>(ws));
  const int BL = B * L;
  const int Hhd = m->H * m->hd;
  const int KVhd = m->Hkv * m->hd;
  cudaError_t e = cudaMemsetAsync(w.counters, 0, 2 * sizeof(int) * B, st);
  if (e != cudaSuccess) return cuda_fail(e, "sft_loss: memset");
  // x_t = forward noising of x_0 at each canvas's keep threshold
  launch_forward_noise(x0, xt, keep_thr, B, L, m->V, seed, st);
  if ((s = check_launch("sft_loss: noise launch")) != DG_OK) return s;
  launch_embed_gather(xt, m->E, w.h, BL, m->V, m->d, nullptr, st, w.status);
  if ((s = check_launch("sft_loss: embed launch")) != DG_OK) return s;
  GemmOut qkv = qkv_segments(m);  // the segments the workspace's split-K plan was sized for
  qkv.ptr[0] = w.q;
  qkv.ptr[1] = w.k;
  qkv.ptr[2] = w.v;
  qkv.ld[0] = Hhd;
  qkv.ld[1] = KVhd;
  qkv.ld[2] = KVhd;
  e = launch_gemm(w.h, m->Wqkv, BL, Hhd + 2 * KVhd, m->d, qkv, nullptr, 0, w.status, nullptr, st,
                  kActNone, w.gemm_part, w.gemm_part_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "sft_loss: qkv gemm launch");
  e = launch_attention(w.q, k_pre, v_pre, w.k, w.v, w.o, nullptr, B, L, P, m->H, m->Hkv, m->hd,
                       window, 1.0f / std::sqrt(static_cast<float>(m->hd)), w.attn, w.status,
                       nullptr, st);
  if (e != cudaSuccess) return cuda_fail(e, "sft_loss: attention launch");
  GemmOut yo{};
  yo.nseg = 1;
  yo.seg_begin[0] = 0;
  yo.seg_begin[1] = m->d;
  yo.ptr[0] = w.y;
  yo.ld[0] = m->d;
  e = launch_gemm(w.o, m->Wo, BL, m->d, Hhd, yo, w.h, m->d, w.status, nullptr, st, kActNone,
                  w.gemm_part, w.gemm_part_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "sft_loss: out_proj gemm launch");
  // fused LM head + cross-entropy against x_0
  e = launch_vocab_pass(w.y, m->E, BL, L, m->d, m->V, inv_tau, 0, 0, w.parts, w.status, nullptr,
                        st, x0);
  if (e != cudaSuccess) return cuda_fail(e, "sft_loss: vocab pass launch");
  const VocabPlan vp = plan_vocab(BL, m->V);
  FinalizeParams fp{};
  fp.parts = w.parts;
  fp.num_mt = vp.num_mt;
  fp.S = vp.S;
  fp.L = L;
  fp.out_loss = loss;
  fp.ticket = reinterpret_cast<unsigned long long*>(w.counters);
  launch_vocab_finalize(fp, B, st);
  return check_launch("sft_loss: finalize launch");
}

dg_status dg_entropy_bounded_update(const int32_t* x0hat, const int32_t* top1,
                                    const float* entropy, int32_t* prev_top1, int prev_valid,
                                    int32_t* x_out, uint8_t* accept, uint8_t* done,
                                    float* mean_entropy, int B, int L, int V, uint64_t seed,
                                    int step, float gamma, float stop_entropy, int final_step,
                                    void* stream) {
  if (B < 0 || L <= 0 || L > 1024 || V < 1)
    return fail(DG_EINVAL, "entropy_bounded_update: bad sizes (1 <= L <= 1024, V >= 1)");
  if (step < 0 || step >= (1 << 24)) return fail(DG_EINVAL, "entropy_bounded_update: bad step");
  if (std::isnan(gamma) || std::isnan(stop_entropy))
    return fail(DG_EINVAL, "entropy_bounded_update: NaN threshold");
  if (B == 0) return DG_OK;
  if (!x0hat || !top1 || !entropy || !x_out)
    return fail(DG_EINVAL, "entropy_bounded_update: NULL pointer");
  EBParams p{};
  p.x0hat = x0hat;
  p.top1 = top1;
  p.entropy = entropy;
  p.prev_top1 = prev_top1;
  p.prev_valid = prev_valid;
  p.x_out = x_out;
  p.accept = accept;
  p.done = done;
  p.mean_out = mean_entropy;
  p.L = L;
  p.V = V;
  p.k0 = static_cast<uint32_t>(seed);
  p.k1 = static_cast<uint32_t>(seed >> 32);
  p.step = static_cast<uint32_t>(step);
  p.gamma = gamma;
  p.stop_entropy = stop_entropy;
  p.final_step = final_step;
  launch_entropy_bounded(p, B, as_stream(stream));
  return check_launch("entropy_bounded_update launch");
}

dg_status dg_euler_update(const int32_t* x_in, const int32_t* x0hat, const int32_t* top1,
                          const float* logp_top1, int32_t* x_out, uint8_t* lock, uint8_t* jump,
                          uint8_t* done, int B, int L, uint64_t seed, int step, uint64_t jump_thr,
                          float lock_logthr, void* stream) {
  if (B < 0 || L <= 0 || L > 1024) return fail(DG_EINVAL, "euler_update: bad sizes (1 <= L <= 1024)");
  if (step < 0 || step >= (1 << 24)) return fail(DG_EINVAL, "euler_update: step out of range");
  if (jump_thr > (1ull << 32)) return fail(DG_EINVAL, "euler_update: jump_thr above 2^32");
  if (B == 0) return DG_OK;
  if (!x_in || !x0hat || !top1 || !logp_top1 || !x_out || !lock)
    return fail(DG_EINVAL, "euler_update: NULL pointer");
  launch_euler_update(x_in, x0hat, top1, logp_top1, x_out, lock, jump, done, B, L, seed, step,
                      jump_thr, lock_logthr, as_stream(stream));
  return check_launch("euler_update launch");
}

size_t dg_denoise_loop_workspace(const dg_model* m, int B, int L, int P, int window) {
  if (!m || B <= 0 || L <= 0 || m->d <= 0 || m->H <= 0 || m->Hkv <= 0 ||
      (m->hd != 64 && m->hd != 128) || m->V < 256)
    return kStatusBytes;
  return loop_layout(m, B, L, P, window, nullptr).total;
}

int dg_denoise_loop_kernel_count(const dg_model* m, int B, int L, int P, int window, int steps) {
  if (!m || B <= 0 || L <= 0 || steps < 0 || m->H <= 0 || (m->hd != 64 && m->hd != 128))
    return -1;
  const AttnPlan ap = plan_attention(B, L, P, m->H, m->Hkv, m->hd, window);
  // loop init, then per step: embedding gather, QKV GEMM, attention (+ split merge),
  // output projection, vocabulary pass, finalisation (Euler sampler).  Without
  // self-conditioning a step's finalisation shares the next step's embedding launch, so the
  // call's last step alone adds one.  With self-conditioning, every step but the run's last
  // (counted here as the last of these `steps`) adds the rescale, the contraction, its
  // reduction and the two feed-forward GEMMs.
  const bool sc = m->Wsc1 != nullptr;
  const int sc_steps = sc && steps > 0 ? steps - 1 : 0;
  const int per_step = 5 + (ap.splits > 1 ? 1 : 0) + (sc ? 1 : 0);
  return 1 + steps * per_step + (!sc && steps > 0 ? 1 : 0) + 5 * sc_steps;
}

}  // extern "C"

namespace {

// Checks a sampler configuration; on success *end is the last step + 1 and, for the
// entropy-bounded sampler, eb_inv_tau holds 1/tau_n for every step (double, then rounded).
dg_status check_cfg(const dg_sampler_cfg* cfg, int* end, std::vector<float>* eb_inv_tau) {
  if (!cfg) return fail(DG_EINVAL, "loop: NULL cfg");
  if (cfg->T < 1 || cfg->T >= (1 << 24)) return fail(DG_EINVAL, "loop: T out of range");
  const bool eb = cfg->sampler == DG_SAMPLER_ENTROPY_BOUNDED;
  if (!eb && cfg->sampler != DG_SAMPLER_EULER) return fail(DG_EINVAL, "loop: unknown sampler");
  if (!eb && cfg->schedule != DG_SCHED_LINEAR && cfg->schedule != DG_SCHED_COSINE)
    return fail(DG_EINVAL, "loop: unknown schedule");
  if (!eb && (!(cfg->inv_tau > 0.f) || !std::isfinite(cfg->inv_tau)))
    return fail(DG_EINVAL, "loop: bad inv_tau");
  *end = cfg->end_step > 0 ? cfg->end_step : cfg->T;
  if (cfg->start_step < 0 || *end > cfg->T || cfg->start_step > *end)
    return fail(DG_EINVAL, "loop: bad start/end step");
  eb_inv_tau->clear();
  if (eb) {
    if (cfg->start_step != 0 || *end != cfg->T)
      return fail(DG_ENOTSUP, "loop: the entropy-bounded sampler runs from step 0 to T");
    if (!(cfg->tau_start > 0.0) || !(cfg->tau_end > 0.0) || !std::isfinite(cfg->tau_start) ||
        !std::isfinite(cfg->tau_end) || std::isnan(cfg->gamma) || std::isnan(cfg->stop_entropy))
      return fail(DG_EINVAL, "loop: bad entropy-bounded sampler parameters");
    for (int n = 0; n < cfg->T; ++n) {
      const double tau = cfg->T == 1 ? cfg->tau_start
                                     : cfg->tau_start + (cfg->tau_end - cfg->tau_start) * n /
                                                            (cfg->T - 1);
      eb_inv_tau->push_back(static_cast<float>(1.0 / tau));
    }
  }
  return DG_OK;
}

// One canvas denoising run on the stream: loop bookkeeping, then steps start .. end-1 of the
// sampler.  The prefix holds P rows per canvas at a stride of pre_stride rows; gen_active (or
// NULL) leaves canvases out; seed is the run's key.  Arguments are already checked.
struct RunArgs {
  const dg_model* m;
  const uint16_t* k_pre;
  const uint16_t* v_pre;
  int B, L, P, pre_stride, window;
  int32_t* canvas;
  uint8_t* lock;  // NULL for the entropy-bounded sampler
  int32_t* steps_taken;
  const uint8_t* gen_active;
  uint64_t seed;
  int start, end;
};

dg_status run_denoise(const RunArgs& a, const dg_sampler_cfg* cfg,
                      const std::vector<float>& eb_inv_tau, const std::vector<uint64_t>& jump,
                      const LoopWs& w, cudaStream_t st) {
  const dg_model* m = a.m;
  const bool eb = cfg->sampler == DG_SAMPLER_ENTROPY_BOUNDED;
  const int B = a.B, L = a.L;
  const int BL = B * L;
  const int Hhd = m->H * m->hd;
  const int KVhd = m->Hkv * m->hd;
  const VocabPlan vp = plan_vocab(BL, m->V);
  dg_status s;

  // the vocabulary pass's sampling bars are cleared once here; each step's finalisation clears
  // them again for the next step
  uint32_t* bars = vocab_bars(w.parts, BL, m->V);
  cudaError_t e = cudaMemsetAsync(w.n_active, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(w.counters, 0, 2 * sizeof(int) * B, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(bars, 0, static_cast<size_t>(BL) * 4, st);
  if (e != cudaSuccess) return cuda_fail(e, "loop: memset");
  launch_loop_init_masked(a.lock, a.gen_active, w.active, w.n_active, a.steps_taken, B, L,
                          eb ? 0 : cfg->stop_when_all_locked, st);
  if ((s = check_launch("loop init launch")) != DG_OK) return s;

  GemmOut qkv = qkv_segments(m);  // the segments the workspace's split-K plan was sized for
  qkv.ptr[0] = w.q;
  qkv.ptr[1] = w.k;
  qkv.ptr[2] = w.v;
  qkv.ld[0] = Hhd;
  qkv.ld[1] = KVhd;
  qkv.ld[2] = KVhd;
  GemmOut yo{};
  yo.nseg = 1;
  yo.seg_begin[0] = 0;
  yo.seg_begin[1] = m->d;
  yo.ptr[0] = w.y;
  yo.ld[0] = m->d;
  const float scale = 1.0f / std::sqrt(static_cast<float>(m->hd));
  const uint32_t k0 = static_cast<uint32_t>(a.seed), k1 = static_cast<uint32_t>(a.seed >> 32);

  const bool sc = has_sc(m);
  // Euler without self-conditioning: each step's finalisation runs inside the next step's
  // embedding launch (one kernel boundary fewer per step); the call's last step is finalised
  // on its own at the end.
  const bool fuse = !eb && !sc;
  FinalizeParams pending{};
  for (int n = a.start; n < a.end; ++n) {
    if (fuse && n > a.start) {
      launch_embed_finalize(pending, B, m->E, w.h, m->V, m->d, st);
      if ((s = check_launch("loop: embed + finalize launch")) != DG_OK) return s;
    } else {
      // the signal of the previous step (none at step 0; a resumed run reads the one its
      // previous call left in the workspace)
      launch_embed_gather(a.canvas, m->E, w.h, BL, m->V, m->d, w.n_active, st, w.status,
                          sc && n > 0 ? w.sc_s : nullptr);
      if ((s = check_launch("loop: embed launch")) != DG_OK) return s;
    }
    e = launch_gemm(w.h, m->Wqkv, BL, Hhd + 2 * KVhd, m->d, qkv, nullptr, 0, w.status, w.n_active,
                    st, kActNone, w.gemm_part, w.gemm_part_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "loop: qkv gemm launch");
    e = launch_attention(w.q, a.k_pre, a.v_pre, w.k, w.v, w.o, nullptr, B, L, a.P, m->H, m->Hkv,
                         m->hd, a.window, scale, w.attn, w.status, w.n_active, st, a.pre_stride);
    if (e != cudaSuccess) return cuda_fail(e, "loop: attention launch");
    e = launch_gemm(w.o, m->Wo, BL, m->d, Hhd, yo, w.h, m->d, w.status, w.n_active, st, kActNone,
                    w.gemm_part, w.gemm_part_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "loop: out_proj gemm launch");
    const bool sc_next = sc && n < cfg->T - 1;  // the last step's signal is never used
    const float inv_tau = eb ? eb_inv_tau[n] : cfg->inv_tau;
    e = launch_vocab_pass(w.y, m->E, BL, L, m->d, m->V, inv_tau, a.seed, n, w.parts, w.status,
                          w.n_active, st, nullptr, eb, sc_next ? w.sc_p : nullptr,
                          sc_next ? w.sc_m : nullptr, false, /*bars_clear=*/true);
    if (e != cudaSuccess) return cuda_fail(e, "loop: vocab pass launch");
    FinalizeParams fp{};
    fp.parts = w.parts;
    fp.bar = bars;
    fp.status = w.status;
    fp.num_mt = vp.num_mt;
    fp.S = vp.S;
    fp.L = L;
    if (sc_next) fp.out_lse = w.sc_lse;
    if (eb) {  // posterior only; the entropy-bounded kernel makes the step
      fp.out_x0hat = w.x0hat;
      fp.out_top1 = w.top1;
      fp.out_entropy = w.entropy;
      fp.n_active = w.n_active;
      fp.ticket = reinterpret_cast<unsigned long long*>(w.counters);
      launch_vocab_finalize(fp, B, st);
      if ((s = check_launch("loop: finalize launch")) != DG_OK) return s;
      EBParams ep{};
      ep.x0hat = w.x0hat;
      ep.top1 = w.top1;
      ep.entropy = w.entropy;
      ep.prev_top1 = w.prev_top1;
      ep.prev_valid = n > 0 ? 1 : 0;
      ep.x_out = a.canvas;
      ep.L = L;
      ep.V = m->V;
      ep.k0 = k0;
      ep.k1 = k1;
      ep.step = static_cast<uint32_t>(n);
      ep.gamma = cfg->gamma;
      ep.stop_entropy = cfg->stop_entropy;
      ep.final_step = n == cfg->T - 1 ? 1 : 0;
      ep.active = w.active;
      ep.steps_taken = a.steps_taken;
      ep.n_active = w.n_active;
      launch_entropy_bounded(ep, B, st);
      if ((s = check_launch("loop: entropy-bounded launch")) != DG_OK) return s;
    } else {
      fp.x_in = a.canvas;
      fp.x_out = a.canvas;
      fp.lock = a.lock;
      fp.jump_thr = jump[n];
      fp.lock_logthr = cfg->lock_logthr;
      fp.k0 = k0;
      fp.k1 = k1;
      fp.step = static_cast<uint32_t>(n);
      fp.active = w.active;
      fp.steps_taken = a.steps_taken;
      fp.n_active = w.n_active;
      fp.stop_when_all_locked = cfg->stop_when_all_locked;
      fp.ticket = reinterpret_cast<unsigned long long*>(w.counters);
      if (fuse) {
        pending = fp;
      } else {
        launch_vocab_finalize(fp, B, st);
        if ((s = check_launch("loop: finalize launch")) != DG_OK) return s;
      }
    }
    if (sc_next) {
      e = launch_self_condition(w.sc_p, w.sc_m, w.sc_lse, m->E, m->Wsc1, m->Wsc2, BL, m->V,
                                m->d, m->d_sc, w.sc_part, w.sc_e, w.sc_u, w.sc_s, w.status,
                                w.n_active, st);
      if (e != cudaSuccess) return cuda_fail(e, "loop: self-conditioning launch");
    }
  }
  if (fuse && a.end > a.start) {
    launch_vocab_finalize(pending, B, st);
    if ((s = check_launch("loop: finalize launch")) != DG_OK) return s;
  }
  return DG_OK;
}

// Encode-append scratch: status word, embeddings, K and V of the canvas.
struct AppendWs {
  uint32_t* status;
  uint16_t *h, *k, *v;
  size_t total;
};

AppendWs append_layout(const dg_model* m, int B, int L, uint8_t* base) {
  AppendWs w{};
  const size_t BL = static_cast<size_t>(B) * L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off += align256(bytes);
    return p;
  };
  w.status = reinterpret_cast<uint32_t*>(take(kStatusBytes));
  w.h = reinterpret_cast<uint16_t*>(take(BL * m->d * 2));
  w.k = reinterpret_cast<uint16_t*>(take(BL * m->Hkv * m->hd * 2));
  w.v = reinterpret_cast<uint16_t*>(take(BL * m->Hkv * m->hd * 2));
  w.total = off;
  return w;
}

// K and V of the canvas tokens (embedding gather, then the K/V rows of the fused projection
// only), copied to cache rows P .. P+L-1 of every canvas with active[b] != 0 (all if NULL).
// n_run (or NULL) lets the kernels skip the pass when no canvas is generating.
dg_status run_encode_append(const dg_model* m, const int32_t* canvas, uint16_t* k_cache,
                            uint16_t* v_cache, int B, int L, int P, int P_cap,
                            const uint8_t* active, const int* n_run, uint16_t* h, uint16_t* k,
                            uint16_t* v, uint32_t* status, cudaStream_t st) {
  const int BL = B * L;
  const int Hhd = m->H * m->hd;
  const int KVhd = m->Hkv * m->hd;
  dg_status s;
  launch_embed_gather(canvas, m->E, h, BL, m->V, m->d, n_run, st, status);
  if ((s = check_launch("encode-append: embed launch")) != DG_OK) return s;
  GemmOut kv{};
  kv.nseg = 2;
  kv.seg_begin[0] = 0;
  kv.seg_begin[1] = KVhd;
  kv.seg_begin[2] = 2 * KVhd;
  kv.ptr[0] = k;
  kv.ptr[1] = v;
  kv.ld[0] = KVhd;
  kv.ld[1] = KVhd;
  const cudaError_t e = launch_gemm(h, m->Wqkv + static_cast<size_t>(Hhd) * m->d, BL, 2 * KVhd,
                                    m->d, kv, nullptr, 0, status, n_run, st);
  if (e != cudaSuccess) return cuda_fail(e, "encode-append: kv gemm launch");
  launch_kv_append(k, v, k_cache, v_cache, active, B, L, P, P_cap, KVhd, st);
  return check_launch("encode-append: copy launch");
}

// Block-autoregressive generation scratch: the denoising loop's workspace first (so that its
// status word is the workspace's first word), sized for the longest prefix, then the block
// state.
struct BlockWs {
  LoopWs loop;
  size_t loop_bytes;
  int32_t *canvas, *zeros, *steps_taken;
  uint64_t* keep_zero;
  uint8_t *lock, *gen_active;
  int* gen_count;
  size_t total;
};

BlockWs block_layout(const dg_model* m, int B, int L, int P0, int NB, int window, uint8_t* base) {
  BlockWs w{};
  size_t loop_bytes = 0;
  for (int j = 0; j < NB; ++j)
    loop_bytes = std::max(loop_bytes,
                          loop_layout(m, B, L, P0 + j * L, window, nullptr).total);
  const size_t app = append_layout(m, B, L, nullptr).total;
  loop_bytes = std::max(loop_bytes, app);
  w.loop_bytes = loop_bytes;
  const size_t BL = static_cast<size_t>(B) * L;
  size_t off = loop_bytes;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off += align256(bytes);
    return p;
  };
  w.canvas = reinterpret_cast<int32_t*>(take(BL * 4));
  w.zeros = reinterpret_cast<int32_t*>(take(BL * 4));
  w.steps_taken = reinterpret_cast<int32_t*>(take(static_cast<size_t>(B) * 4));
  w.keep_zero = reinterpret_cast<uint64_t*>(take(static_cast<size_t>(B) * 8));
  w.lock = take(BL);
  w.gen_active = take(B);
  w.gen_count = reinterpret_cast<int*>(take(sizeof(int)));
  w.total = off;
  return w;
}

}  // namespace

extern "C" {

dg_status dg_denoise_loop(const dg_model* m, const uint16_t* k_pre, const uint16_t* v_pre, int B,
                          int L, int P, int window, int32_t* canvas, uint8_t* lock,
                          int32_t* steps_taken, const dg_sampler_cfg* cfg, void* ws,
                          size_t ws_bytes, void* stream) {
  dg_status s = check_model(m);
  if (s != DG_OK) return s;
  s = check_attn_dims(B, L, P, m->H, m->Hkv, m->hd, window);
  if (s != DG_OK) return s;
  int end = 0;
  std::vector<float> eb_inv_tau;
  if ((s = check_cfg(cfg, &end, &eb_inv_tau)) != DG_OK) return s;
  const bool eb = cfg->sampler == DG_SAMPLER_ENTROPY_BOUNDED;
  if (static_cast<int64_t>(B) * L >= (1ll << 31)) return fail(DG_ENOTSUP, "loop: too many rows");
  if (B == 0) return DG_OK;
  if (bad_ptr(canvas) || (!eb && bad_ptr(lock)) || bad_ptr(steps_taken) || bad_ptr(ws))
    return fail(DG_EINVAL, "loop: NULL or misaligned canvas/lock/steps/workspace");
  if (eb) lock = nullptr;
  if (P > 0 && (bad_ptr(k_pre) || bad_ptr(v_pre))) return fail(DG_EINVAL, "loop: bad prefix pointer");
  if (ws_bytes < dg_denoise_loop_workspace(m, B, L, P, window))
    return fail(DG_EINVAL, "loop: workspace too small");

  std::vector<uint64_t> jump(cfg->T);
  dg_schedule_thresholds(cfg->schedule, cfg->T, nullptr, jump.data());
  RunArgs a{};
  a.m = m;
  a.k_pre = k_pre;
  a.v_pre = v_pre;
  a.B = B;
  a.L = L;
  a.P = P;
  a.pre_stride = P;
  a.window = window;
  a.canvas = canvas;
  a.lock = lock;
  a.steps_taken = steps_taken;
  a.gen_active = nullptr;
  a.seed = cfg->seed;
  a.start = cfg->start_step;
  a.end = end;
  return run_denoise(a, cfg, eb_inv_tau, jump, loop_layout(m, B, L, P, window,
                                                           static_cast<uint8_t*>(ws)),
                     as_stream(stream));
}

size_t dg_self_condition_workspace(int B, int L, int d, int V, int d_sc) {
  if (B <= 0 || L <= 0 || d <= 0 || V < 256 || d_sc <= 0) return kStatusBytes;
  const size_t BL = static_cast<size_t>(B) * L;
  const VocabPlan vp = plan_vocab(static_cast<int>(BL), V);
  const ScPlan sp = plan_selfcond(static_cast<int>(BL), V, d);
  return kStatusBytes + align256(2 * sizeof(int) * static_cast<size_t>(B)) +
         align256(vp.part_bytes) + align256(BL * V * 2) +
         align256(BL * (V / 32) * 4) + align256(BL * 4) + align256(sp.part_bytes) +
         align256(BL * d * 2) + align256(BL * d_sc * 2);
}

dg_status dg_self_condition(const uint16_t* y, const uint16_t* E, const uint16_t* Wsc1,
                            const uint16_t* Wsc2, int B, int L, int d, int V, int d_sc,
                            float inv_tau, uint16_t* s_out, uint16_t* e_out, void* ws,
                            size_t ws_bytes, void* stream) {
  if (B < 0 || L <= 0 || d <= 0 || V <= 0 || d_sc <= 0)
    return fail(DG_EINVAL, "self-condition: bad sizes");
  if (d % 256 != 0 || V % 256 != 0 || d_sc % 64 != 0)
    return fail(DG_ENOTSUP, "self-condition: needs d % 256 == 0, V % 256 == 0, d_sc % 64 == 0");
  if (L > 256 || L % 64 != 0)
    return fail(DG_ENOTSUP, "self-condition: L must be 64..256, multiple of 64");
  if (!(inv_tau > 0.f) || !std::isfinite(inv_tau))
    return fail(DG_EINVAL, "self-condition: bad inv_tau");
  if (static_cast<int64_t>(B) * L >= (1ll << 31) / 128)
    return fail(DG_ENOTSUP, "self-condition: too many rows");
  if (B == 0) return DG_OK;
  if (bad_ptr(y) || bad_ptr(E) || bad_ptr(Wsc1) || bad_ptr(Wsc2) || bad_ptr(s_out) ||
      bad_ptr(ws) || (e_out && !aligned16(e_out)))
    return fail(DG_EINVAL, "self-condition: NULL or misaligned pointer");
  if (ws_bytes < dg_self_condition_workspace(B, L, d, V, d_sc))
    return fail(DG_EINVAL, "self-condition: workspace too small");
  cudaStream_t st = as_stream(stream);
  const int BL = B * L;
  const VocabPlan vp = plan_vocab(BL, V);
  const ScPlan sp = plan_selfcond(BL, V, d);
  uint8_t* p = static_cast<uint8_t*>(ws);
  uint32_t* status = reinterpret_cast<uint32_t*>(p);
  p += kStatusBytes;
  int* counters = reinterpret_cast<int*>(p);
  p += align256(2 * sizeof(int) * static_cast<size_t>(B));
  VocabPart* parts = reinterpret_cast<VocabPart*>(p);
  p += align256(vp.part_bytes);
  uint16_t* sc_p = reinterpret_cast<uint16_t*>(p);
  p += align256(static_cast<size_t>(BL) * V * 2);
  float* sc_m = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(BL) * (V / 32) * 4);
  float* lse = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(BL) * 4);
  float* part = reinterpret_cast<float*>(p);
  p += align256(sp.part_bytes);
  uint16_t* e_ws = reinterpret_cast<uint16_t*>(p);
  p += align256(static_cast<size_t>(BL) * d * 2);
  uint16_t* u = reinterpret_cast<uint16_t*>(p);
  // the LM head pass without sampling (lse only), storing the exponentials
  cudaError_t e = launch_vocab_pass(y, E, BL, L, d, V, inv_tau, 0, 0, parts, status, nullptr, st,
                                    nullptr, false, sc_p, sc_m, true);
  if (e != cudaSuccess) return cuda_fail(e, "self-condition: vocab pass launch");
  FinalizeParams fp{};
  fp.parts = parts;
  fp.num_mt = vp.num_mt;
  fp.S = vp.S;
  fp.L = L;
  fp.out_lse = lse;
  dg_status s;
  e = cudaMemsetAsync(counters, 0, 2 * sizeof(int) * B, st);  // finalisation counters
  if (e != cudaSuccess) return cuda_fail(e, "self-condition: memset");
  fp.ticket = reinterpret_cast<unsigned long long*>(counters);
  launch_vocab_finalize(fp, B, st);
  if ((s = check_launch("self-condition: finalize launch")) != DG_OK) return s;
  e = launch_self_condition(sc_p, sc_m, lse, E, Wsc1, Wsc2, BL, V, d, d_sc, part,
                            e_out ? e_out : e_ws, u, s_out, status, nullptr, st);
  if (e != cudaSuccess) return cuda_fail(e, "self-condition: launch");
  return DG_OK;
}

size_t dg_encode_append_workspace(const dg_model* m, int B, int L) {
  if (!m || B <= 0 || L <= 0 || m->d <= 0 || m->Hkv <= 0 || m->hd <= 0) return kStatusBytes;
  return append_layout(m, B, L, nullptr).total;
}

dg_status dg_encode_append(const dg_model* m, const int32_t* canvas, uint16_t* k_cache,
                           uint16_t* v_cache, int B, int L, int P, int P_cap,
                           const uint8_t* active, void* ws, size_t ws_bytes, void* stream) {
  dg_status s = check_model(m);
  if (s != DG_OK) return s;
  if (B < 0 || L <= 0 || P < 0 || P_cap < P + L)
    return fail(DG_EINVAL, "encode-append: bad sizes (need P + L <= P_cap)");
  if (static_cast<int64_t>(B) * L >= (1ll << 31) || static_cast<int64_t>(B) * P_cap >= (1ll << 31))
    return fail(DG_ENOTSUP, "encode-append: too many rows");
  if (B == 0) return DG_OK;
  if (bad_ptr(canvas) || bad_ptr(k_cache) || bad_ptr(v_cache) || bad_ptr(ws))
    return fail(DG_EINVAL, "encode-append: NULL or misaligned canvas/cache/workspace");
  if (ws_bytes < dg_encode_append_workspace(m, B, L))
    return fail(DG_EINVAL, "encode-append: workspace too small");
  const AppendWs w = append_layout(m, B, L, static_cast<uint8_t*>(ws));
  return run_encode_append(m, canvas, k_cache, v_cache, B, L, P, P_cap, active, nullptr, w.h, w.k,
                           w.v, w.status, as_stream(stream));
}

size_t dg_block_generate_workspace(const dg_model* m, int B, int L, int P0, int NB, int window) {
  if (!m || B <= 0 || L <= 0 || P0 < 0 || NB <= 0 || m->d <= 0 || m->H <= 0 || m->Hkv <= 0 ||
      (m->hd != 64 && m->hd != 128) || m->V < 256)
    return kStatusBytes;
  return block_layout(m, B, L, P0, NB, window, nullptr).total;
}

dg_status dg_block_generate(const dg_model* m, uint16_t* k_cache, uint16_t* v_cache, int B, int P0,
                            int P_cap, int L, int NB, int window, int32_t eos,
                            const dg_sampler_cfg* cfg, int32_t* out, int32_t* blocks,
                            int32_t* n_tokens, int32_t* steps, void* ws, size_t ws_bytes,
                            void* stream) {
  dg_status s = check_model(m);
  if (s != DG_OK) return s;
  if (NB < 0 || P0 < 0) return fail(DG_EINVAL, "block generate: negative size");
  if (static_cast<int64_t>(P0) + static_cast<int64_t>(NB) * L > P_cap)
    return fail(DG_EINVAL, "block generate: cache too small (need P0 + NB * L <= P_cap)");
  s = check_attn_dims(B, L, P0, m->H, m->Hkv, m->hd, window);
  if (s != DG_OK) return s;
  int end = 0;
  std::vector<float> eb_inv_tau;
  if ((s = check_cfg(cfg, &end, &eb_inv_tau)) != DG_OK) return s;
  if (cfg->start_step != 0 || end != cfg->T)
    return fail(DG_ENOTSUP, "block generate: every block runs steps 0 .. T-1");
  const bool eb = cfg->sampler == DG_SAMPLER_ENTROPY_BOUNDED;
  if (static_cast<int64_t>(B) * P_cap >= (1ll << 31) ||
      static_cast<int64_t>(B) * NB * L >= (1ll << 31))
    return fail(DG_ENOTSUP, "block generate: too many rows");
  if (B == 0 || NB == 0) return DG_OK;
  if (bad_ptr(k_cache) || bad_ptr(v_cache) || bad_ptr(out) || bad_ptr(blocks) ||
      bad_ptr(n_tokens) || bad_ptr(steps) || bad_ptr(ws))
    return fail(DG_EINVAL, "block generate: NULL or misaligned pointer");
  if (ws_bytes < dg_block_generate_workspace(m, B, L, P0, NB, window))
    return fail(DG_EINVAL, "block generate: workspace too small");

  std::vector<uint64_t> jump(cfg->T);
  dg_schedule_thresholds(cfg->schedule, cfg->T, nullptr, jump.data());
  cudaStream_t st = as_stream(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const BlockWs bw = block_layout(m, B, L, P0, NB, window, base);
  const int BL = B * L;
  cudaError_t e = cudaMemsetAsync(out, 0xFF, static_cast<size_t>(BL) * NB * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(bw.zeros, 0, static_cast<size_t>(BL) * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(bw.keep_zero, 0, static_cast<size_t>(B) * 8, st);
  if (e != cudaSuccess) return cuda_fail(e, "block generate: memset");
  launch_block_init(bw.gen_active, bw.gen_count, blocks, n_tokens, steps, B, st);
  if ((s = check_launch("block generate: init launch")) != DG_OK) return s;

  for (int j = 0; j < NB; ++j) {
    const int P = P0 + j * L;
    const uint64_t seed = cfg->seed + static_cast<uint64_t>(j);
    // x_1 of block j: the uniform prior under the block's own key
    launch_forward_noise(bw.zeros, bw.canvas, bw.keep_zero, B, L, m->V, seed, st);
    if ((s = check_launch("block generate: prior launch")) != DG_OK) return s;
    if (!eb) {
      e = cudaMemsetAsync(bw.lock, 0, BL, st);
      if (e != cudaSuccess) return cuda_fail(e, "block generate: lock memset");
    }
    RunArgs a{};
    a.m = m;
    a.k_pre = k_cache;
    a.v_pre = v_cache;
    a.B = B;
    a.L = L;
    a.P = P;
    a.pre_stride = P_cap;
    a.window = window;
    a.canvas = bw.canvas;
    a.lock = eb ? nullptr : bw.lock;
    a.steps_taken = bw.steps_taken;
    a.gen_active = bw.gen_active;
    a.seed = seed;
    a.start = 0;
    a.end = cfg->T;
    const LoopWs lw = loop_layout(m, B, L, P, window, base);
    if ((s = run_denoise(a, cfg, eb_inv_tau, jump, lw, st)) != DG_OK) return s;
    const AppendWs aw = append_layout(m, B, L, base);
    if ((s = run_encode_append(m, bw.canvas, k_cache, v_cache, B, L, P, P_cap, bw.gen_active,
                               bw.gen_count, aw.h, aw.k, aw.v, aw.status, st)) != DG_OK)
      return s;
    launch_block_record(bw.canvas, bw.steps_taken, out, bw.gen_active, bw.gen_count, blocks,
                        n_tokens, steps, B, L, NB, j, eos, st);
    if ((s = check_launch("block generate: record launch")) != DG_OK) return s;
  }
  return DG_OK;
}

dg_status dg_set_wait_control(uint64_t limit_ns, int skip_loads) {
  if (limit_ns > kMaxWaitNs) return fail(DG_EINVAL, "wait control: limit above 60 s");
  g_wait_limit_ns = limit_ns ? limit_ns : kDefaultWaitNs;
  g_wait_skip_loads = skip_loads != 0;
  return DG_OK;
}

dg_status dg_workspace_status(const void* ws, void* stream) {
  cudaStream_t st = as_stream(stream);
  uint32_t* word = ws ? static_cast<uint32_t*>(const_cast<void*>(ws)) : status_or_fallback(nullptr);
  if (!word) return fail(DG_ECUDA, "status: no status word");
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, sizeof(v), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "status: read");
  if (v & kStatusTimeout) return fail(DG_ETIMEOUT, "a kernel gave up waiting on an on-chip barrier");
  if (v & kStatusBadIndex) return fail(DG_EKERNEL, "a kernel skipped an out-of-range index");
  return DG_OK;
}

dg_status dg_kernel_timer_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_timer_mu);
  timer_reset_locked();
  g_timer_on = enable != 0;
  return DG_OK;
}

dg_status dg_kernel_timer_read(int kind, double* total_ms, int* launches) {
  if (!total_ms || !launches || kind < 0 || kind >= kTimerKinds) return fail(DG_EINVAL, "timer: bad arguments");
  std::lock_guard<std::mutex> lk(g_timer_mu);
  double tot = 0.0;
  int n = 0;
  for (auto& r : g_timer_recs) {
    if (r.kind != kind) continue;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e != cudaSuccess) return cuda_fail(e, "timer: event sync");
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) return cuda_fail(e, "timer: elapsed");
    tot += ms;
    ++n;
  }
  *total_ms = tot;
  *launches = n;
  return DG_OK;
}

}  // extern "C"
