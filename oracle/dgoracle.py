"""Plain CPU oracle of the canvas-denoising core of a block-diffusion text model.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library and its Python
binding never import it, and it imports nothing from them: the two sides share no code,
headers, tables or constants.  The only thing they share is the seeded input generator
module (``discrete_diffusion_text_gb300.synth``), which holds none of the method's arithmetic.

Everything here is numpy in float64 (integer work in uint64/int64), written so that each
function can be checked against the passage it follows by eye.  A library matmul, a
logsumexp or an argmax serves as a step where the definition is that operation; there is no
blocking, fusion or reordering beyond what the definitions state.  Long rows are processed
in row chunks purely to bound memory; each row's arithmetic is unchanged by that.

Sources (web pages on DiffusionGemma; cited by title and section):
  [TR]  "DiffusionGemma Technical Report 정리" (juhoplayground), sections
        "이산 디퓨전 정식화", "Forward Process", "Backward Denoising Process",
        "블록 자기회귀(Block-AR) 생성", "디노이징 반복과 self-conditioning",
        "DiffusionGemma 샘플러", "추론 효율 지표", "1단계: Supervised Finetuning".
  [BLOG] "DiffusionGemma 완전분석" (cell-devlog), section "스펙 정리".
  [PBD] "Google DiffusionGemma 출시: 병렬 블록 디코딩" (molayo), glossary entry
        "Iterative denoising" and the FAQ.
  [P11] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11
        (the Philox4x32-10 counter-based generator).

Readings taken where the pages are silent (each listed in the design notes):
  * time runs from t=1 (noise) to t=0 (clean); step n of T maps t_n=(T-n)/T to t_n-h, h=1/T;
  * the Euler step of the factorised uniform-source mixture path jumps to a fresh sample
    of the posterior with probability lambda_n = min(1, h * (-kappa'(t_n)) / (1 - kappa(t_n)));
  * schedules: linear kappa(t)=1-t and cosine kappa(t)=cos^2(pi t / 2);
  * confidence locking (optional): a position whose top-1 posterior log-probability is at
    least log(theta) is locked to its top-1 token and frozen; the lock test precedes the jump;
  * the decoder is a one-layer stand-in: embedding, one bidirectional attention layer over
    [prefix KV ; canvas] with GQA and an optional sliding window, output projection with a
    residual, and an LM head tied to the embedding; no norm, no RoPE, no time input;
  * intermediate activations (q, k, v, attention output, y) are rounded to bfloat16;
  * self-conditioning (when the model carries Wsc1, Wsc2): the expected embedding
    e = p_hat_0 E under the step's tempered posterior, rounded to bfloat16, goes through a
    two-layer feed-forward s = Wsc2 gelu(Wsc1 e) (tanh-form GELU, bfloat16 after each layer);
    s is added to the token embeddings of the next step, h = bf16(E[x] + s), and is zero at
    the first step of a canvas.

Counter-based random numbers (Philox4x32-10 keyed by the 64-bit seed) replace every random
draw the method makes, so that both implementations see identical random bits:
  noising / canvas init : counter (pos, canvas, 0, 1<<24); word 0 = keep draw, word 1 = token
  chunk Gumbel noise    : counter (c>>2, pos, canvas, (2<<24)|step); chunk c uses word c&3
  Euler jump            : counter (0, pos, canvas, (3<<24)|step); word 0
  re-noising (entropy-bounded sampler) : counter (pos, canvas, 0, (4<<24)|step); word 0
  within-chunk Gumbel   : counter (v>>2, pos, canvas, (5<<24)|step); entry v uses word v&3

Posterior sample x_hat_0 ~ p_hat_0 (exact, Gumbel-max at two levels): the vocabulary is cut
into aligned chunks of 32 entries; a chunk is chosen by Gumbel-max over the chunks'
log-sum-exps (so chunk c is chosen with probability sum_{v in c} p_v), then an entry of that
chunk by Gumbel-max over its tempered logits with an independent family of Gumbels
(probability p_v / sum_{v' in c} p_v').  The product is p_v.

Entropy-bounded sampler [TR "DiffusionGemma 샘플러"], readings taken where the section is silent:
  * the entropy of a position is that of the tempered posterior used for sampling at the step,
    -sum_v p_v log p_v with p = Softmax(z / tau_n);
  * tau_n = tau_start + (tau_end - tau_start) * n / (T - 1) over steps n = 0..T-1, so the first
    step uses 0.8 and the last possible step 0.4 (the section's two endpoints);
  * positions are ordered by (entropy, position); k is the length of the longest prefix of that
    order whose running float32 sum stays <= gamma (k may be 0); the first k positions take
    their posterior sample, every other position a fresh uniform token;
  * a canvas stops after step n when its mean entropy (float32 sum in position order / L) is
    below the threshold and its top-1 sequence equals that of step n-1; the returned canvas is
    the top-1 sequence of the last evaluated posterior (also when the cap T is reached).
"""

from __future__ import annotations

import math

import numpy as np

MASK32 = np.uint64(0xFFFFFFFF)
TWO32 = 1 << 32

# [P11] Philox4x32 round multipliers and Weyl key increments.
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint64(0x9E3779B9)
_PHILOX_W1 = np.uint64(0xBB67AE85)

STREAM_NOISE = 1
STREAM_GUMBEL = 2
STREAM_JUMP = 3
STREAM_RENOISE = 4
STREAM_PICK = 5
SAMPLE_CHUNK = 32  # entries per chunk of the two-level posterior sample

SCHED_LINEAR = 0
SCHED_COSINE = 1


# ----------------------------------------------------------------------------------------
# Counter-based generator [P11]
# ----------------------------------------------------------------------------------------

def seed_key(seed: int) -> tuple[np.uint64, np.uint64]:
    """Split a 64-bit seed into the two 32-bit Philox key words (low word first)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return np.uint64(seed & 0xFFFFFFFF), np.uint64(seed >> 32)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds [P11].

    One round: (hi0, lo0) = M0*c0, (hi1, lo1) = M1*c2 as 64-bit products;
    the new counter is (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0); then the key is bumped by
    the Weyl constants.  Inputs broadcast; every word is a 32-bit value held in uint64.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & MASK32 for c in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & MASK32
    k1 = np.asarray(k1, dtype=np.uint64) & MASK32
    for _ in range(10):
        p0 = _PHILOX_M0 * c0
        p1 = _PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + _PHILOX_W0) & MASK32
        k1 = (k1 + _PHILOX_W1) & MASK32
    return c0, c1, c2, c3


def u32_to_token(u, V: int):
    """Map a 32-bit draw to a token uniform over [0, V): floor(u * V / 2^32)."""
    return ((np.asarray(u, dtype=np.uint64) * np.uint64(V)) >> np.uint64(32)).astype(np.int64)


def u32_to_open_unit(u):
    """Map a 32-bit draw to W = (u + 1/2) / 2^32, uniform on the open interval (0, 1)."""
    return (np.asarray(u, dtype=np.uint64).astype(np.float64) + 0.5) / float(TWO32)


def gumbel_from_u32(u):
    """Standard Gumbel variate from a draw: g = -log(E), E = -log(1 - W) ~ Exp(1).

    1 - W is itself uniform on (0, 1), so this is the textbook g = -log(-log U).  Writing
    E through log1p keeps full relative precision for the large-g tail (W near 0).
    """
    W = u32_to_open_unit(u)
    E = -np.log1p(-W)
    return -np.log(E)


# ----------------------------------------------------------------------------------------
# Schedules [TR "Forward Process"; reading: linear and cosine families]
# ----------------------------------------------------------------------------------------

def kappa(schedule: int, t):
    """kappa_t, monotone from kappa_0 = 1 to kappa_1 = 0 [TR "Forward Process"]."""
    t = np.asarray(t, dtype=np.float64)
    if schedule == SCHED_LINEAR:
        return 1.0 - t
    if schedule == SCHED_COSINE:
        return np.cos(0.5 * math.pi * t) ** 2
    raise ValueError("unknown schedule")


def neg_dkappa(schedule: int, t):
    """-d kappa / dt for the two schedule families."""
    t = np.asarray(t, dtype=np.float64)
    if schedule == SCHED_LINEAR:
        return np.ones_like(t)
    if schedule == SCHED_COSINE:
        return math.pi * np.cos(0.5 * math.pi * t) * np.sin(0.5 * math.pi * t)
    raise ValueError("unknown schedule")


def one_minus_kappa(schedule: int, t):
    """1 - kappa_t written in closed form (t for linear, sin^2(pi t / 2) for cosine), so
    that no cancellation enters the Euler rate near t = 0."""
    t = np.asarray(t, dtype=np.float64)
    if schedule == SCHED_LINEAR:
        return t.copy()
    if schedule == SCHED_COSINE:
        return np.sin(0.5 * math.pi * t) ** 2
    raise ValueError("unknown schedule")


def step_times(T: int):
    """t_n = (T - n) / T for n = 0..T-1, step size h = 1/T [TR "디노이징 반복과 self-conditioning"]."""
    n = np.arange(T, dtype=np.float64)
    return (T - n) / T, 1.0 / T


def jump_rate(schedule: int, T: int):
    """lambda_n = min(1, h * (-kappa'(t_n)) / (1 - kappa(t_n))): the probability that the
    discrete Euler step at t_n replaces a token by a fresh posterior sample.

    Reading of [TR "Backward Denoising Process"] (the Euler update of the mixture path): the
    factorised velocity is u_t = (-kappa'/(1-kappa)) * (p_hat - delta_{x_t}); one Euler step
    of size h moves a token to a posterior sample with probability h times that rate.
    """
    t, h = step_times(T)
    lam = h * neg_dkappa(schedule, t) / one_minus_kappa(schedule, t)
    return np.minimum(1.0, lam)


def probability_threshold(p):
    """A probability p in [0, 1] as the integer threshold floor(p * 2^32); a 32-bit draw u
    passes iff u < threshold, so p = 1 gives 2^32 (always) and p = 0 gives 0 (never)."""
    p = np.clip(np.asarray(p, dtype=np.float64), 0.0, 1.0)
    return np.floor(p * float(TWO32)).astype(np.uint64)


def schedule_thresholds(schedule: int, T: int):
    """keep_thr[n] = floor(kappa(t_n) * 2^32) for n = 0..T (t_T = 0) and
    jump_thr[n] = floor(lambda_n * 2^32) for n = 0..T-1."""
    t_all = (T - np.arange(T + 1, dtype=np.float64)) / T
    keep = probability_threshold(kappa(schedule, t_all))
    jump = probability_threshold(jump_rate(schedule, T))
    return keep, jump


def keep_threshold_from_t(schedule: int, t):
    """Per-canvas keep threshold for noising a clean canvas to level t."""
    return probability_threshold(kappa(schedule, t))


# ----------------------------------------------------------------------------------------
# Forward noising [TR "Forward Process", eq. p_t(x_t|x_0); "1단계: Supervised Finetuning"]
# ----------------------------------------------------------------------------------------

def forward_noise(x0, keep_thr, V: int, seed: int):
    """x_t^i = x_0^i with probability kappa_t, else a token uniform over V (positions
    independent).  Because the uniform replacement may hit x_0^i itself, the marginal is
    P(x_t^i = x_0^i) = kappa_t + (1 - kappa_t)/|V|, as in the closed form.

    x0: int [B, L]; keep_thr: uint64 [B] (floor(kappa_t * 2^32) per canvas).
    """
    x0 = np.asarray(x0, dtype=np.int64)
    B, L = x0.shape
    k0, k1 = seed_key(seed)
    pos = np.arange(L, dtype=np.uint64)[None, :]
    canvas = np.arange(B, dtype=np.uint64)[:, None]
    u_keep, u_tok, _, _ = philox4x32_10(pos, canvas, 0, STREAM_NOISE << 24, k0, k1)
    keep = u_keep < np.asarray(keep_thr, dtype=np.uint64)[:, None]
    return np.where(keep, x0, u32_to_token(u_tok, V))


def initial_canvas(B: int, L: int, V: int, seed: int):
    """x_1: every position uniform over the vocabulary [TR "블록 자기회귀(Block-AR) 생성"]
    (the noising stream with kappa = 0)."""
    return forward_noise(np.zeros((B, L), np.int64), np.zeros(B, np.uint64), V, seed)


# ----------------------------------------------------------------------------------------
# Stand-in decoder [TR "디노이징 반복과 self-conditioning"; "블록 자기회귀(Block-AR) 생성"]
# ----------------------------------------------------------------------------------------

def round_bf16(x):
    """Round to the nearest bfloat16 (ties to even) and return float64."""
    import torch  # library conversion routine only

    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.float64)))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def attention_mask(L: int, P: int, window: int):
    """Boolean [L, P + L]: query i (absolute position P + i) sees every canvas key
    (bidirectional inside the canvas) and prefix key k iff window == 0 or P + i - k < window
    [TR "블록 자기회귀(Block-AR) 생성": bidirectional canvas, cross-attention to the cache;
    BLOG "스펙 정리": sliding window of 1,024]."""
    i = np.arange(L)[:, None]
    k = np.arange(P)[None, :]
    pre = np.ones((L, P), dtype=bool) if window == 0 else ((P + i - k) < window)
    return np.concatenate([pre, np.ones((L, L), dtype=bool)], axis=1)


def canvas_attention(q, k_pre, v_pre, k_can, v_can, window: int, scale: float):
    """O = softmax(q K^T * scale + mask) V over keys = [prefix ; canvas], per canvas and head.

    q [B, L, H, hd]; k_pre/v_pre [B, P, Hkv, hd]; k_can/v_can [B, L, Hkv, hd].
    Query head hq reads KV head floor(hq * Hkv / H) (grouped-query attention).
    Returns O [B, L, H, hd] and the natural-log log-sum-exp of the scaled scores [B, H, L].
    """
    q = np.asarray(q, np.float64)
    B, L, H, hd = q.shape
    P, Hkv = k_pre.shape[1], k_pre.shape[2]
    mask = attention_mask(L, P, window)
    O = np.zeros((B, L, H, hd))
    lse = np.zeros((B, H, L))
    for b in range(B):
        for hq in range(H):
            g = (hq * Hkv) // H
            K = np.concatenate([k_pre[b, :, g, :], k_can[b, :, g, :]], axis=0).astype(np.float64)
            Vv = np.concatenate([v_pre[b, :, g, :], v_can[b, :, g, :]], axis=0).astype(np.float64)
            s = (q[b, :, hq, :] @ K.T) * scale
            s = np.where(mask, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            den = e.sum(axis=1, keepdims=True)
            O[b, :, hq, :] = (e / den) @ Vv
            lse[b, hq, :] = (m + np.log(den))[:, 0]
    return O, lse


def decoder_front(x, E, Wqkv, H: int, Hkv: int, hd: int, s=None):
    """h = E[x_t] (+ s_t, rounded to bfloat16, when a self-conditioning signal is given);
    [q | k_c | v_c] = h Wqkv^T, each rounded to bfloat16.

    x [B, L] int; E [V, d]; Wqkv [(H + 2 Hkv) hd, d] (rows: q heads, then k heads, then v);
    s [B, L, d] or None.
    """
    x = np.asarray(x, np.int64)
    B, L = x.shape
    h = np.asarray(E, np.float64)[x]                       # [B, L, d]
    if s is not None:
        h = round_bf16(h + np.asarray(s, np.float64).reshape(h.shape))
    qkv = round_bf16(h.reshape(B * L, -1) @ np.asarray(Wqkv, np.float64).T)
    q = qkv[:, : H * hd].reshape(B, L, H, hd)
    k = qkv[:, H * hd:(H + Hkv) * hd].reshape(B, L, Hkv, hd)
    v = qkv[:, (H + Hkv) * hd:].reshape(B, L, Hkv, hd)
    return h, q, k, v


def decoder_back(h, O, Wo):
    """y = h + O Wo^T, rounded to bfloat16.  h [B, L, d]; O [B, L, H, hd]; Wo [d, H hd]."""
    B, L, d = h.shape
    O = round_bf16(O).reshape(B * L, -1)
    y = h.reshape(B * L, d) + O @ np.asarray(Wo, np.float64).T
    return round_bf16(y).reshape(B, L, d)


# ----------------------------------------------------------------------------------------
# Posterior, sample, top-1 [TR "디노이징 반복과 self-conditioning": p_hat_0 = Softmax(logits /
# tau); x_(t-h) ~ Step(x_t, p_hat_0) draws from p_hat_0]
# ----------------------------------------------------------------------------------------

def two_level_sample(z, pos, canvas, step: int, seed: int):
    """One exact draw from Softmax(z) per row of tempered logits z [c, V] (float64), by
    Gumbel-max at two levels over the aligned 32-entry chunks c of the vocabulary:

      lse_c  = log sum_{v in c} exp(z_v)
      c*     = argmax_c (lse_c + g_c)             (chunk c is chosen with probability
                                                   sum_{v in c} p_v; lowest c on ties)
      x0hat  = argmax_{v in c*} (z_v + g'_v)      (entry v of c* with probability
                                                   p_v / sum_{v' in c*} p_v'; lowest v on ties)

    The two Gumbel families are independent, so x0hat = v with probability p_v exactly.  g_c
    comes from the chunk Gumbel stream (word c&3 of counter (c>>2, pos, canvas, 2<<24 | step)),
    g'_v from the pick stream (word v&3 of counter (v>>2, pos, canvas, 5<<24 | step)); only the
    winning chunk's g'_v are ever needed.  Returns x0hat and, for the parity bars, the
    decision's margin: the smaller of the gaps between the two largest perturbed scores at
    either level (chunk scores; perturbed logits inside c*)."""
    n, V = z.shape
    nc = (V + SAMPLE_CHUNK - 1) // SAMPLE_CHUNK
    pad = np.full((n, nc * SAMPLE_CHUNK), -np.inf)
    pad[:, :V] = z
    zc = pad.reshape(n, nc, SAMPLE_CHUNK)
    mc = zc.max(axis=2, keepdims=True)
    lse_c = (mc + np.log(np.exp(zc - mc).sum(axis=2, keepdims=True)))[:, :, 0]
    k0, k1 = seed_key(seed)

    def word_of(counter0, sel, tag):
        words = philox4x32_10(counter0, pos, canvas, (tag << 24) | int(step), k0, k1)
        return np.choose(np.broadcast_to(sel, counter0.shape), words)

    def top2_gap(score):
        if score.shape[1] < 2:
            return np.full(score.shape[0], np.inf)
        two = -np.partition(-score, 1, axis=1)[:, :2]
        return two[:, 0] - two[:, 1]

    c = np.arange(nc, dtype=np.uint64)[None, :]
    chunk_score = lse_c + gumbel_from_u32(
        word_of(np.broadcast_to(c >> np.uint64(2), (n, nc)), (c & np.uint64(3)).astype(np.int64),
                STREAM_GUMBEL))
    cstar = np.argmax(chunk_score, axis=1)
    v = cstar.astype(np.uint64)[:, None] * np.uint64(SAMPLE_CHUNK) + \
        np.arange(SAMPLE_CHUNK, dtype=np.uint64)[None, :]            # [n, 32] entries of c*
    g_pick = gumbel_from_u32(word_of(v >> np.uint64(2), (v & np.uint64(3)).astype(np.int64),
                                     STREAM_PICK))
    entry_score = zc[np.arange(n), cstar] + g_pick                    # -inf past the end
    j = np.argmax(entry_score, axis=1)
    margin = np.minimum(top2_gap(chunk_score), top2_gap(entry_score))
    return cstar * SAMPLE_CHUNK + j, margin


def posterior(y, E, inv_tau: float, seed: int, step: int, L: int, rows=None, chunk=None):
    """Per row r (canvas r // L, position r % L) of y [R, d], with logits z = y E^T
    (LM head tied to the embedding) and z~ = z * inv_tau:

      lse        = log sum_v exp(z~_v)
      top1       = argmax_v z~_v                     (lowest index on ties)
      logp_top1  = z~_top1 - lse
      x0hat      = two_level_sample(z~)                (an exact sample of Softmax(z~))
      logp_x0hat = z~_x0hat - lse
      entropy    = -sum_v p_v log p_v,  p = Softmax(z~)   (clamped at 0 against rounding)

    Also returned, for the parity bars: the sample's margin (gap_perturbed: see
    two_level_sample) and the gap between the two largest logits.  ``rows`` selects a subset
    of rows (default: all).
    """
    y = np.asarray(y, np.float64)
    E64 = np.asarray(E, np.float64)
    R = y.shape[0]
    V = E64.shape[0]
    rows = np.arange(R) if rows is None else np.asarray(rows, np.int64)
    if chunk is None:  # rows per batch, so that one [rows, V] float64 block stays ~128 MiB
        chunk = max(1, (1 << 24) // V)
    out = {k: np.zeros(len(rows), np.float64) for k in
           ("lse", "logp_top1", "logp_x0hat", "gap_perturbed", "gap_logit", "entropy")}
    out["top1"] = np.zeros(len(rows), np.int64)
    out["x0hat"] = np.zeros(len(rows), np.int64)
    for s in range(0, len(rows), chunk):
        rr = rows[s:s + chunk]
        z = (y[rr] @ E64.T) * inv_tau                      # [c, V]
        m = z.max(axis=1, keepdims=True)
        lse = (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]
        canvas = (rr // L).astype(np.uint64)[:, None]
        pos = (rr % L).astype(np.uint64)[:, None]
        x0hat, margin = two_level_sample(z, pos, canvas, step, seed)
        top1 = np.argmax(z, axis=1)
        idx = np.arange(len(rr))
        sl = slice(s, s + len(rr))
        out["lse"][sl] = lse
        out["top1"][sl] = top1
        out["x0hat"][sl] = x0hat
        out["logp_top1"][sl] = z[idx, top1] - lse
        out["logp_x0hat"][sl] = z[idx, x0hat] - lse
        logp = z - lse[:, None]
        out["entropy"][sl] = np.maximum(0.0, -(np.exp(logp) * logp).sum(axis=1))
        out["gap_perturbed"][sl] = margin
        twz = -np.partition(-z, 1, axis=1)[:, :2]
        out["gap_logit"][sl] = twz[:, 0] - twz[:, 1]
    return out


# ----------------------------------------------------------------------------------------
# Self-conditioning [TR "디노이징 반복과 self-conditioning": s_(t-h) = FFW(p_hat_0 . E)]
# ----------------------------------------------------------------------------------------

def gelu_tanh(x):
    """GELU in its tanh form: x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))."""
    x = np.asarray(x, np.float64)
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


def expected_embedding(y, E, inv_tau: float, chunk=None):
    """e = p_hat_0 . E per row: sum_v Softmax(y E^T * inv_tau)_v E[v].  y [R, d]; returns
    float64 [R, d] (not rounded)."""
    y = np.asarray(y, np.float64)
    E64 = np.asarray(E, np.float64)
    R, V = y.shape[0], E64.shape[0]
    if chunk is None:
        chunk = max(1, (1 << 24) // V)
    e = np.zeros((R, E64.shape[1]))
    for s0 in range(0, R, chunk):
        z = (y[s0:s0 + chunk] @ E64.T) * inv_tau
        m = z.max(axis=1, keepdims=True)
        w = np.exp(z - m)
        p = w / w.sum(axis=1, keepdims=True)
        e[s0:s0 + chunk] = p @ E64
    return e


def self_condition(y, E, inv_tau: float, Wsc1, Wsc2, chunk=None):
    """s = FFW(p_hat_0 . E): e = bf16(p_hat_0 E), u = bf16(gelu(e Wsc1^T)), s = bf16(u Wsc2^T).
    y [R, d]; Wsc1 [d_sc, d]; Wsc2 [d, d_sc].  Returns a dict with e_exact (float64, not
    rounded), e, u and s."""
    e_exact = expected_embedding(y, E, inv_tau, chunk)
    e = round_bf16(e_exact)
    u = round_bf16(gelu_tanh(e @ np.asarray(Wsc1, np.float64).T))
    s = round_bf16(u @ np.asarray(Wsc2, np.float64).T)
    return {"e_exact": e_exact, "e": e, "u": u, "s": s}


def has_self_cond(model) -> bool:
    return model.get("Wsc1") is not None


# ----------------------------------------------------------------------------------------
# Discrete Euler step with optional confidence locking
# [TR "Backward Denoising Process": x_(t-h) ~ Step(x_t, p_theta(.|x_t)), factorised per
# position; PBD glossary "Iterative denoising": confident tokens are locked in]
# ----------------------------------------------------------------------------------------

def euler_update(x_in, x0hat, top1, logp_top1, lock, seed: int, step: int, jump_thr: int,
                 lock_logthr: float):
    """One reverse step at every position of every canvas (arrays [B, L]):

      locked already                      -> unchanged
      lock on and logp_top1 >= log theta  -> lock, x <- top1
      jump draw u < jump_thr              -> x <- x0hat (jump = 1)
      otherwise                           -> unchanged

    lock_logthr = +inf switches locking off; the comparison is made in float32 on float32
    inputs.  Returns x_out, lock_out (uint8), jump (uint8), done (uint8 [B], all locked).
    """
    x_in = np.asarray(x_in, np.int64)
    B, L = x_in.shape
    lock = np.asarray(lock, np.uint8).astype(bool)
    k0, k1 = seed_key(seed)
    pos = np.arange(L, dtype=np.uint64)[None, :]
    canvas = np.arange(B, dtype=np.uint64)[:, None]
    u, _, _, _ = philox4x32_10(0, pos, canvas, (STREAM_JUMP << 24) | int(step), k0, k1)
    lp = np.asarray(logp_top1, np.float32)
    new_lock = (~lock) & (lp >= np.float32(lock_logthr))
    jump = (~lock) & (~new_lock) & (u < np.uint64(jump_thr))
    x_out = np.where(new_lock, np.asarray(top1, np.int64),
                     np.where(jump, np.asarray(x0hat, np.int64), x_in))
    lock_out = lock | new_lock
    done = lock_out.all(axis=1)
    return x_out, lock_out.astype(np.uint8), jump.astype(np.uint8), done.astype(np.uint8)


# ----------------------------------------------------------------------------------------
# One denoising step and the loop [TR "디노이징 반복과 self-conditioning"]
# ----------------------------------------------------------------------------------------

def decoder_posterior(model, k_pre, v_pre, window: int, x, n: int, inv_tau: float, seed: int,
                      s=None):
    """logits = Decoder(x_t, KV, s_t); the posterior tuple of every row at inverse temperature
    inv_tau; with self-conditioning weights in the model, also s_(t-h) = FFW(p_hat_0 . E) in
    post["s"] ([B, L, d]).  s: this step's signal (None = zero)."""
    E, H, Hkv, hd = model["E"], model["H"], model["Hkv"], model["hd"]
    B, L = np.asarray(x).shape
    h, q, kc, vc = decoder_front(x, E, model["Wqkv"], H, Hkv, hd, s)
    O, _ = canvas_attention(q, k_pre, v_pre, kc, vc, window, hd ** -0.5)
    y = decoder_back(h, O, model["Wo"])
    post = posterior(y.reshape(B * L, -1), E, inv_tau, seed, n, L)
    if has_self_cond(model):
        post["s"] = self_condition(y.reshape(B * L, -1), E, inv_tau, model["Wsc1"],
                                   model["Wsc2"])["s"].reshape(B, L, -1)
    return post


def denoise_step(model, k_pre, v_pre, window: int, x, lock, n: int, jump_thr: int,
                 inv_tau: float, lock_logthr: float, seed: int, s=None):
    """logits = Decoder(x_t, KV, s_t); p_hat_0 = Softmax(logits / tau); x_(t-h) ~ Step(x_t,
    p_hat_0); s_(t-h) = FFW(p_hat_0 . E) when the model self-conditions.

    model: dict with E [V, d], Wqkv, Wo, H, Hkv, hd (and optionally Wsc1, Wsc2).  Returns
    (x_out, lock_out, jump, done, diagnostics) where diagnostics holds the posterior tuple per
    row (and the next signal under "s").
    """
    B, L = np.asarray(x).shape
    post = decoder_posterior(model, k_pre, v_pre, window, x, n, inv_tau, seed, s)
    shape = (B, L)
    x_out, lock_out, jump, done = euler_update(
        x, post["x0hat"].reshape(shape), post["top1"].reshape(shape),
        post["logp_top1"].reshape(shape).astype(np.float32), lock, seed, n, jump_thr,
        lock_logthr)
    return x_out, lock_out, jump, done, post


def denoise_loop(model, k_pre, v_pre, window: int, x, lock, T: int, schedule: int,
                 inv_tau: float, lock_logthr: float, seed: int, start_step: int = 0,
                 stop_when_all_locked: bool = False, end_step: int | None = None,
                 state: dict | None = None):
    """Steps n = start_step .. end_step-1 (default T-1) of at most T [TR "DiffusionGemma 샘플러":
    cap T].  A canvas whose positions are all locked stops when ``stop_when_all_locked``.
    Returns the final canvas, the lock mask and the number of steps applied per canvas.
    With self-conditioning, the signal starts at zero at step 0; ``state`` (a dict) carries
    it across calls that split the run (read as state["s"] when start_step > 0, written at
    the end)."""
    x = np.asarray(x, np.int64).copy()
    lock = np.asarray(lock, np.uint8).copy()
    B = x.shape[0]
    s = None
    if start_step > 0 and state is not None:
        s = state.get("s")
    _, jump_thr = schedule_thresholds(schedule, T)
    steps = np.zeros(B, np.int64)
    active = np.ones(B, bool)
    if stop_when_all_locked:
        active &= ~lock.astype(bool).all(axis=1)
    end = T if end_step is None else end_step
    for n in range(start_step, end):
        if not active.any():
            break
        x_new, lock_new, _, done, post = denoise_step(model, k_pre, v_pre, window, x, lock, n,
                                                      int(jump_thr[n]), inv_tau, lock_logthr,
                                                      seed, s)
        x[active] = x_new[active]
        lock[active] = lock_new[active]
        steps[active] += 1
        if "s" in post:
            s = post["s"] if s is None else np.where(active[:, None, None], post["s"], s)
        if stop_when_all_locked:
            active &= ~done.astype(bool)
    if state is not None:
        state["s"] = s
    return x, lock, steps


# ----------------------------------------------------------------------------------------
# Entropy-bounded sampler with temperature annealing and adaptive stopping
# [TR "DiffusionGemma 샘플러": "Entropy-bounded 토큰 정제", "Temperature annealing",
# "Adaptive stopping"; hyper-parameters T = 48, gamma = 0.1, stop threshold 0.005,
# tau 0.8 -> 0.4]
# ----------------------------------------------------------------------------------------

def annealed_temperature(T: int, tau_start: float = 0.8, tau_end: float = 0.4):
    """tau_n for n = 0..T-1: linear in the step index from tau_start to tau_end."""
    n = np.arange(T, dtype=np.float64)
    if T == 1:
        return np.array([tau_start])
    return tau_start + (tau_end - tau_start) * n / (T - 1)


def entropy_bounded_select(entropy, gamma: float):
    """Accept positions in increasing (entropy, position) order while the running float32 sum
    of their entropies stays <= gamma.  entropy: float32 [B, L].  Returns accept (uint8 [B, L])
    and the accepted count k [B]."""
    H = np.asarray(entropy, np.float32)
    B, L = H.shape
    g = np.float32(gamma)
    accept = np.zeros((B, L), np.uint8)
    k = np.zeros(B, np.int64)
    for b in range(B):
        order = sorted(range(L), key=lambda i: (H[b, i], i))
        run = np.float32(0.0)
        for cnt, i in enumerate(order):
            run = np.float32(run + H[b, i])
            if run > g:
                break
            accept[b, i] = 1
            k[b] = cnt + 1
    return accept, k


def renoise_tokens(B: int, L: int, V: int, seed: int, step: int):
    """A fresh uniform token per position from the re-noising stream of the step."""
    k0, k1 = seed_key(seed)
    pos = np.arange(L, dtype=np.uint64)[None, :]
    canvas = np.arange(B, dtype=np.uint64)[:, None]
    u, _, _, _ = philox4x32_10(pos, canvas, 0, (STREAM_RENOISE << 24) | int(step), k0, k1)
    return u32_to_token(u, V)


def mean_entropy(entropy):
    """Per canvas: float32 sum over positions in position order, divided by L in float32."""
    H = np.asarray(entropy, np.float32)
    B, L = H.shape
    out = np.zeros(B, np.float32)
    for b in range(B):
        acc = np.float32(0.0)
        for i in range(L):
            acc = np.float32(acc + H[b, i])
        out[b] = np.float32(acc / np.float32(L))
    return out


def entropy_bounded_update(x0hat, top1, entropy, prev_top1, seed: int, step: int, V: int,
                           gamma: float, stop_entropy: float, final_step: bool = False):
    """One step of the entropy-bounded sampler on every canvas (arrays [B, L]):

      accepted positions (entropy_bounded_select) -> their posterior sample x0hat
      all other positions                         -> a fresh uniform token (re-noising)
      done = mean entropy < stop_entropy  and  top1 == prev_top1 at every position
             (prev_top1 None: no previous prediction, never done)
      a canvas that is done, or any canvas at the final step, returns its top-1 sequence.

    Returns x_out, accept (uint8), done (uint8 [B]), mean entropy (float32 [B])."""
    x0hat = np.asarray(x0hat, np.int64)
    top1 = np.asarray(top1, np.int64)
    B, L = x0hat.shape
    accept, _ = entropy_bounded_select(entropy, gamma)
    x_out = np.where(accept.astype(bool), x0hat, renoise_tokens(B, L, V, seed, step))
    mh = mean_entropy(entropy)
    if prev_top1 is None:
        stable = np.zeros(B, bool)
    else:
        stable = (np.asarray(prev_top1, np.int64) == top1).all(axis=1)
    done = (mh < np.float32(stop_entropy)) & stable
    finish = done | bool(final_step)
    x_out = np.where(finish[:, None], top1, x_out)
    return x_out, accept, done.astype(np.uint8), mh


def eb_denoise_step(model, k_pre, v_pre, window: int, x, n: int, inv_tau: float,
                    prev_top1, seed: int, gamma: float, stop_entropy: float,
                    final_step: bool, s=None):
    """logits = Decoder(x_t, KV, s_t); p_hat = Softmax(logits / tau_n); entropy-bounded
    update (and the next self-conditioning signal in post["s"] when the model has one)."""
    E = model["E"]
    B, L = np.asarray(x).shape
    post = decoder_posterior(model, k_pre, v_pre, window, x, n, inv_tau, seed, s)
    shape = (B, L)
    x_out, accept, done, mh = entropy_bounded_update(
        post["x0hat"].reshape(shape), post["top1"].reshape(shape),
        post["entropy"].reshape(shape).astype(np.float32), prev_top1, seed, n, E.shape[0],
        gamma, stop_entropy, final_step)
    return x_out, accept, done, mh, post


def eb_inv_tau(T: int, tau_start: float, tau_end: float):
    """Per-step inverse temperature as handed to the kernels: float32(1 / tau_n)."""
    return [float(np.float32(1.0 / t)) for t in annealed_temperature(T, tau_start, tau_end)]


def eb_denoise_loop(model, k_pre, v_pre, window: int, x, T: int, tau_start: float,
                    tau_end: float, gamma: float, stop_entropy: float, seed: int):
    """The entropy-bounded sampler for at most T steps.  Returns the final canvas (the top-1
    sequence of each canvas's last posterior), the steps taken per canvas and the per-step
    mean entropies of step 0 (diagnostic)."""
    x = np.asarray(x, np.int64).copy()
    B, L = x.shape
    inv = eb_inv_tau(T, tau_start, tau_end)
    steps = np.zeros(B, np.int64)
    active = np.ones(B, bool)
    prev = None
    s = None
    for n in range(T):
        if not active.any():
            break
        x_new, _, done, _, post = eb_denoise_step(model, k_pre, v_pre, window, x, n, inv[n],
                                                  prev, seed, gamma, stop_entropy, n == T - 1,
                                                  s)
        x[active] = x_new[active]
        steps[active] += 1
        if "s" in post:
            s = post["s"] if s is None else np.where(active[:, None, None], post["s"], s)
        top1 = post["top1"].reshape(B, L)
        prev = top1 if prev is None else np.where(active[:, None], top1, prev)
        active &= ~done.astype(bool)
    return x, steps



# ----------------------------------------------------------------------------------------
# Fused SFT cross-entropy on noised canvases [TR "1단계: Supervised Finetuning":
# canvases noised at t ~ Unif[0, 1] (each token replaced by a uniform draw with probability t),
# loss L = - sum_i log p_theta(x_0^i | x_t, c)]
# ----------------------------------------------------------------------------------------

def cross_entropy(y, E, inv_tau: float, targets, chunk=None):
    """Per row r of y [R, d] (logits z = y E^T, tempered z~ = z * inv_tau):
    loss_r = -log Softmax(z~)[target_r] = lse_r - z~_r[target_r].  Returns (loss, lse)."""
    y = np.asarray(y, np.float64)
    E64 = np.asarray(E, np.float64)
    tgt = np.asarray(targets, np.int64)
    R, V = y.shape[0], E64.shape[0]
    if chunk is None:
        chunk = max(1, (1 << 24) // V)
    loss = np.zeros(R)
    lse = np.zeros(R)
    for s in range(0, R, chunk):
        z = (y[s:s + chunk] @ E64.T) * inv_tau
        m = z.max(axis=1, keepdims=True)
        l = (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]
        lse[s:s + chunk] = l
        loss[s:s + chunk] = l - z[np.arange(len(l)), tgt[s:s + chunk]]
    return loss, lse


def sft_loss(model, k_pre, v_pre, window: int, x0, keep_thr, seed: int, inv_tau: float = 1.0):
    """Noise x0 [B, L] with per-canvas keep thresholds (forward process), run the stand-in decoder
    on x_t and return the per-position loss [B, L] = -log p(x_0 | x_t, KV) and x_t."""
    E, H, Hkv, hd = model["E"], model["H"], model["Hkv"], model["hd"]
    x0 = np.asarray(x0, np.int64)
    B, L = x0.shape
    xt = forward_noise(x0, keep_thr, E.shape[0], seed)
    h, q, kc, vc = decoder_front(xt, E, model["Wqkv"], H, Hkv, hd)
    O, _ = canvas_attention(q, k_pre, v_pre, kc, vc, window, hd ** -0.5)
    y = decoder_back(h, O, model["Wo"])
    loss, _ = cross_entropy(y.reshape(B * L, -1), E, inv_tau, x0.reshape(-1))
    return loss.reshape(B, L), xt


# ----------------------------------------------------------------------------------------
# Encode-append and the block-autoregressive outer loop [TR "블록 자기회귀(Block-AR) 생성":
# context encoding -> denoising loop over a 256-token canvas -> the finished canvas passes
# through the causal encoder and is appended to the KV cache; repeat until the end-of-turn
# token; the response is the concatenation of the canvases]
# ----------------------------------------------------------------------------------------

def encode_append(model, canvas, k_cache, v_cache, P: int, rows=None):
    """For the one-layer stand-in, the keys and values a token contributes to later attention are
    its own projections (bf16): k = E[x] Wk^T, v = E[x] Wv^T; a causal encoder over the canvas
    therefore reduces to them.  They are written at cache rows P .. P+L-1 of each canvas (or of
    the canvases in ``rows``).  k_cache, v_cache: float64 [B, P_cap, Hkv, hd], modified."""
    E, H, Hkv, hd = model["E"], model["H"], model["Hkv"], model["hd"]
    canvas = np.asarray(canvas, np.int64)
    B, L = canvas.shape
    _, _, k, v = decoder_front(canvas, E, model["Wqkv"], H, Hkv, hd)
    sel = np.arange(B) if rows is None else np.asarray(rows, np.int64)
    k_cache[sel, P:P + L] = k[sel]
    v_cache[sel, P:P + L] = v[sel]
    return k_cache, v_cache


def block_generate(model, k_ctx, v_ctx, window: int, L: int, NB: int, eos: int, seed: int,
                   T: int, schedule: int = SCHED_LINEAR, inv_tau: float = 1.0,
                   lock_logthr: float = math.inf, stop_when_all_locked: bool = False,
                   sampler: str = "euler", tau_start: float = 0.8, tau_end: float = 0.4,
                   gamma: float = 0.1, stop_entropy: float = 0.005):
    """Blocks j = 0 .. NB-1: the canvas starts from the uniform prior of seed + j, the denoising
    loop (Euler or entropy-bounded, with seed + j) runs with the context plus every earlier
    canvas as prefix KV, the finished canvas is recorded and encode-appended.  A canvas stops
    at the first block whose canvas contains `eos` (its response length counts the tokens up to
    and including it) or after NB blocks.  Returns out [B, NB, L] (-1 where never generated),
    blocks [B], n_tokens [B], steps [B] (denoising steps summed over blocks) and the caches."""
    k_ctx = np.asarray(k_ctx, np.float64)
    v_ctx = np.asarray(v_ctx, np.float64)
    B, P0 = k_ctx.shape[:2]
    V = model["E"].shape[0]
    cap = P0 + NB * L
    k_cache = np.zeros((B, cap) + k_ctx.shape[2:])
    v_cache = np.zeros((B, cap) + v_ctx.shape[2:])
    k_cache[:, :P0] = k_ctx
    v_cache[:, :P0] = v_ctx
    out = np.full((B, NB, L), -1, np.int64)
    blocks = np.zeros(B, np.int64)
    n_tokens = np.zeros(B, np.int64)
    steps = np.zeros(B, np.int64)
    active = np.ones(B, bool)
    for j in range(NB):
        if not active.any():
            break
        P = P0 + j * L
        x = initial_canvas(B, L, V, seed + j)
        kp, vp = k_cache[:, :P], v_cache[:, :P]
        if sampler == "euler":
            xf, _, st = denoise_loop(model, kp, vp, window, x, np.zeros((B, L), np.uint8), T,
                                     schedule, inv_tau, lock_logthr, seed + j,
                                     stop_when_all_locked=stop_when_all_locked)
        else:
            xf, st = eb_denoise_loop(model, kp, vp, window, x, T, tau_start, tau_end, gamma,
                                     stop_entropy, seed + j)
        rows = np.nonzero(active)[0]
        out[rows, j] = xf[rows]
        steps[rows] += st[rows]
        blocks[rows] = j + 1
        encode_append(model, xf, k_cache, v_cache, P, rows)
        for b in rows:
            hit = np.nonzero(xf[b] == eos)[0]
            if len(hit):
                n_tokens[b] = j * L + int(hit[0]) + 1
                active[b] = False
            else:
                n_tokens[b] = (j + 1) * L
    return out, blocks, n_tokens, steps, k_cache, v_cache
