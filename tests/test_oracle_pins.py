"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every test here runs on the CPU.  Each one checks the oracle against something other than
itself: an independent library routine, a closed form, an invariant of the definition, or a
brute-force / statistical consequence, chosen so that a plausible slip (a dropped term, a
wrong sign or index, a swapped word) fails at least one of them.
"""

import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
from scipy import stats
from scipy.special import logsumexp

from oracle import dgoracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# ------------------------------------------------------------------ Philox4x32-10 -----

_TRITON_SCRIPT = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl

@triton.jit
def kern(out_ptr, c_ptr, seed, N: tl.constexpr):
    i = tl.arange(0, N)
    c0 = tl.load(c_ptr + 4 * i)
    c1 = tl.load(c_ptr + 4 * i + 1)
    c2 = tl.load(c_ptr + 4 * i + 2)
    c3 = tl.load(c_ptr + 4 * i + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + 4 * i, a)
    tl.store(out_ptr + 4 * i + 1, b)
    tl.store(out_ptr + 4 * i + 2, c)
    tl.store(out_ptr + 4 * i + 3, d)

req = json.loads(sys.stdin.read())
res = []
for seed, ctr in zip(req["seeds"], req["counters"]):
    c = torch.tensor(ctr, dtype=torch.int64).to(torch.int32)
    out = torch.zeros_like(c)
    kern[(1,)](out, c, seed, N=len(ctr) // 4)
    res.append([v & 0xFFFFFFFF for v in out.tolist()])
print(json.dumps(res))
"""


def test_philox_matches_triton_reference_implementation():
    """Bit-identical to Triton's Philox4x32-10 (run by its CPU interpreter), an implementation
    independent of the oracle, over random counters and 64-bit seeds."""
    pytest.importorskip("triton")
    rng = np.random.default_rng(123)
    seeds = [0, 1, 0xDEADBEEF, int(rng.integers(0, 2**63 - 1)), 2**63 - 1]
    counters = []
    for _ in seeds:
        c = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64)
        c[0] = 0
        c[1] = 0xFFFFFFFF
        counters.append(c)
    req = {"seeds": seeds,
           "counters": [[int(v) - (1 << 32) if v >= (1 << 31) else int(v) for v in c.reshape(-1)]
                        for c in counters]}
    env = dict(os.environ, TRITON_INTERPRET="1")
    p = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(req),
                       capture_output=True, text=True, env=env, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    got = json.loads(p.stdout.strip().splitlines()[-1])
    for seed, c, ref in zip(seeds, counters, got):
        k0, k1 = O.seed_key(seed)
        w = O.philox4x32_10(c[:, 0], c[:, 1], c[:, 2], c[:, 3], k0, k1)
        mine = np.stack(w, axis=1).reshape(-1)
        assert np.array_equal(mine, np.asarray(ref, dtype=np.uint64)), seed


def test_philox_words_are_uniform_and_decorrelated():
    k0, k1 = O.seed_key(7)
    n = np.arange(200000, dtype=np.uint64)
    w = O.philox4x32_10(n, 0, 0, 0, k0, k1)
    for word in w:
        bins = np.bincount((word >> np.uint64(24)).astype(np.int64), minlength=256)
        assert stats.chisquare(bins).pvalue > 1e-4
    r = np.corrcoef(w[0].astype(np.float64), w[1].astype(np.float64))[0, 1]
    assert abs(r) < 0.02


# ---------------------------------------------------------------- draw conversions -----

@pytest.mark.parametrize("V", [16, 4096, 262144, 1000])
def test_u32_to_token_edges(V):
    u = np.array([0, 1, 2**31, 2**32 - 1], dtype=np.uint64)
    t = O.u32_to_token(u, V)
    assert t[0] == 0 and t[1] == 0
    assert t[2] == V // 2 if V % 2 == 0 else True
    assert t[3] == V - 1
    if V & (V - 1) == 0:  # power of two: the top log2(V) bits
        uu = np.random.default_rng(0).integers(0, 2**32, 10000, dtype=np.uint64)
        shift = 32 - int(math.log2(V))
        assert np.array_equal(O.u32_to_token(uu, V), (uu >> np.uint64(shift)).astype(np.int64))


def test_open_unit_interval_and_gumbel_distribution():
    u = np.array([0, 2**32 - 1], dtype=np.uint64)
    W = O.u32_to_open_unit(u)
    assert 0.0 < W[0] < 1e-9 and 1.0 - 1e-9 < W[1] < 1.0
    k0, k1 = O.seed_key(11)
    draws = O.philox4x32_10(np.arange(250000, dtype=np.uint64), 5, 6, 7, k0, k1)
    g = O.gumbel_from_u32(np.concatenate(draws))
    # standard Gumbel: mean = Euler-Mascheroni constant, variance = pi^2 / 6
    assert abs(g.mean() - np.euler_gamma) < 5 * math.sqrt(math.pi**2 / 6 / g.size)
    assert abs(g.var() - math.pi**2 / 6) < 0.02
    assert stats.kstest(g, stats.gumbel_r.cdf).pvalue > 1e-3


# --------------------------------------------------------------------- schedules -----

@pytest.mark.parametrize("T", [1, 2, 12, 48, 192])
def test_linear_jump_rate_is_one_over_remaining_steps(T):
    _, jump = O.schedule_thresholds(O.SCHED_LINEAR, T)
    for n in range(T):
        assert int(jump[n]) == (1 << 32) // (T - n)   # floor(2^32 / (T - n)), exact integers
    keep, _ = O.schedule_thresholds(O.SCHED_LINEAR, T)
    assert int(keep[0]) == 0 and int(keep[T]) == 1 << 32


@pytest.mark.parametrize("T", [2, 12, 48])
def test_cosine_rate_endpoints_and_derivative(T):
    lam = O.jump_rate(O.SCHED_COSINE, T)
    assert lam[0] == pytest.approx(0.0, abs=1e-15)      # kappa'(1) = 0: first step never jumps
    assert lam[-1] == 1.0                                # last step is clamped to 1
    _, thr = O.schedule_thresholds(O.SCHED_COSINE, T)
    assert int(thr[0]) == 0 and int(thr[-1]) == 1 << 32
    # -kappa' against a central finite difference of kappa itself
    t, h = O.step_times(T)
    eps = 1e-6
    fd = -(O.kappa(O.SCHED_COSINE, t + eps) - O.kappa(O.SCHED_COSINE, t - eps)) / (2 * eps)
    lam_fd = np.minimum(1.0, h * fd / (1.0 - O.kappa(O.SCHED_COSINE, t)))
    assert np.allclose(lam_fd, lam, atol=1e-6)
    k = O.kappa(O.SCHED_COSINE, np.array([0.0, 1.0]))
    assert k[0] == 1.0 and k[1] == pytest.approx(0.0, abs=1e-15)


@pytest.mark.parametrize("T", [4, 12, 48])
def test_linear_euler_matches_exact_bridge_and_forward_marginal(T):
    """For linear kappa the Euler jump probability equals the exact mixture-path bridge
    (kappa_{t-h} - kappa_t) / (1 - kappa_t), so the reverse chain driven by the true one-hot
    posterior reproduces the forward marginal: P(not yet jumped after n steps) = 1 - kappa(t_n)."""
    lam = O.jump_rate(O.SCHED_LINEAR, T)
    t, h = O.step_times(T)
    bridge = (O.kappa(O.SCHED_LINEAR, t - h) - O.kappa(O.SCHED_LINEAR, t)) / (1 - O.kappa(O.SCHED_LINEAR, t))
    assert np.allclose(lam, bridge, rtol=1e-12)
    stay = np.cumprod(1.0 - lam)
    assert np.allclose(stay, 1.0 - O.kappa(O.SCHED_LINEAR, t - h), atol=1e-12)


# ------------------------------------------------------------------ forward noise -----

@pytest.mark.parametrize("V", [4096, 262144])
@pytest.mark.parametrize("t", [0.1, 0.5, 0.9])
def test_noising_marginal_matches_closed_form(V, t):
    """P(x_t = x_0) = kappa_t + (1 - kappa_t)/|V| per position (Forward Process closed form);
    with linear kappa, each token is replaced by a uniform draw with probability t."""
    B, L = 256, 256
    x0 = np.random.default_rng(1).integers(0, V, (B, L))
    thr = O.keep_threshold_from_t(O.SCHED_LINEAR, np.full(B, t))
    xt = O.forward_noise(x0, thr, V, seed=99)
    k = 1.0 - t
    p = k + (1.0 - k) / V
    n = B * L
    assert abs((xt == x0).mean() - p) < 5 * math.sqrt(p * (1 - p) / n)
    # replaced tokens are uniform over the vocabulary
    rep = xt[xt != x0]
    bins = np.bincount(rep * 64 // V, minlength=64)
    assert stats.chisquare(bins).pvalue > 1e-4


def test_noising_extremes_and_independence():
    V, B, L = 4096, 4, 256
    x0 = np.random.default_rng(2).integers(0, V, (B, L))
    assert np.array_equal(O.forward_noise(x0, np.full(B, 1 << 32, np.uint64), V, 5), x0)
    a = O.forward_noise(x0, np.zeros(B, np.uint64), V, 5)
    b = O.forward_noise(np.zeros_like(x0), np.zeros(B, np.uint64), V, 5)
    assert np.array_equal(a, b)                                # independent of x_0 at kappa = 0
    assert np.array_equal(a, O.initial_canvas(B, L, V, 5))
    assert (a == x0).mean() < 0.01
    c = O.forward_noise(x0, np.zeros(B, np.uint64), V, 6)
    assert (a != c).mean() > 0.99                              # the seed changes the draws


# ---------------------------------------------------------------------- attention -----

def _sdpa(q, K, V, scale):
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None],
        scale=scale)[0].numpy()


@pytest.mark.parametrize("P", [0, 1, 37, 256])
@pytest.mark.parametrize("window", [0, 16, 100])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (2, 2)])
def test_attention_equals_sdpa_on_visible_keys(P, window, H, Hkv):
    """Per query, the oracle equals torch's float64 scaled-dot-product attention over exactly
    the visible keys: the prefix keys k >= P + i - window + 1 (all of them when window = 0)
    followed by every canvas key, with KV head floor(h * Hkv / H)."""
    B, L, hd = 2, 64, 16
    rng = np.random.default_rng(P * 100 + window + H)
    q = rng.standard_normal((B, L, H, hd))
    kp, vp = rng.standard_normal((2, B, P, Hkv, hd))
    kc, vc = rng.standard_normal((2, B, L, Hkv, hd))
    scale = hd ** -0.5
    out, lse = O.canvas_attention(q, kp, vp, kc, vc, window, scale)
    for b in range(B):
        for h in range(H):
            g = h // (H // Hkv)
            for i in range(L):
                lo = 0 if window == 0 else max(0, P + i - window + 1)
                K = np.concatenate([kp[b, lo:, g], kc[b, :, g]])
                Vv = np.concatenate([vp[b, lo:, g], vc[b, :, g]])
                ref = _sdpa(q[b, i:i + 1, h], K, Vv, scale)
                assert np.allclose(out[b, i, h], ref[0], atol=1e-10)
                s = (K @ q[b, i, h]) * scale
                assert lse[b, h, i] == pytest.approx(logsumexp(s), abs=1e-10)


def test_attention_is_bidirectional_in_the_canvas():
    """Changing a later canvas value changes earlier canvas outputs (no causal mask)."""
    B, L, H, hd, P = 1, 64, 2, 16, 8
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, L, H, hd))
    kp, vp = rng.standard_normal((2, B, P, H, hd))
    kc, vc = rng.standard_normal((2, B, L, H, hd))
    o1, _ = O.canvas_attention(q, kp, vp, kc, vc, 0, 0.25)
    vc2 = vc.copy()
    vc2[0, L - 1] += 1.0
    o2, _ = O.canvas_attention(q, kp, vp, kc, vc2, 0, 0.25)
    assert np.abs(o1[0, 0] - o2[0, 0]).max() > 1e-4


# ------------------------------------------------------------- stand-in decoder -----

def test_decoder_front_selects_the_right_segments():
    """With Wqkv rows that are unit vectors, q / k / v are chosen coordinates of h = E[x]:
    a transposed weight, a swapped q|k|v segment or a wrong head split fails this."""
    V, d, H, Hkv, hd, B, L = 32, 64, 2, 1, 8, 2, 4
    rng = np.random.default_rng(0)
    E = O.round_bf16(rng.standard_normal((V, d)))
    cols = rng.permutation(d)[: (H + 2 * Hkv) * hd]
    Wqkv = np.zeros(((H + 2 * Hkv) * hd, d))
    Wqkv[np.arange(len(cols)), cols] = 1.0
    x = rng.integers(0, V, (B, L))
    h, q, k, v = O.decoder_front(x, E, Wqkv, H, Hkv, hd)
    assert np.array_equal(h, E[x])
    hq = h[..., cols[: H * hd]].reshape(B, L, H, hd)
    hk = h[..., cols[H * hd:(H + Hkv) * hd]].reshape(B, L, Hkv, hd)
    hv = h[..., cols[(H + Hkv) * hd:]].reshape(B, L, Hkv, hd)
    assert np.array_equal(q, hq) and np.array_equal(k, hk) and np.array_equal(v, hv)


def test_decoder_back_is_residual_plus_projection():
    B, L, d, H, hd = 1, 3, 16, 2, 8
    rng = np.random.default_rng(1)
    h = O.round_bf16(rng.standard_normal((B, L, d)))
    Oa = O.round_bf16(rng.standard_normal((B, L, H, hd)))
    assert np.array_equal(O.decoder_back(h, Oa, np.zeros((d, H * hd))), h)
    Wo = np.zeros((d, H * hd))
    Wo[np.arange(d), np.arange(d)[::-1]] = 1.0                 # y_j = h_j + O_flat[d - 1 - j]
    y = O.decoder_back(h, Oa, Wo)
    ref = O.round_bf16(h + Oa.reshape(B, L, -1)[..., ::-1])
    assert np.array_equal(y, ref)


# ---------------------------------------------------------------------- posterior -----

def test_posterior_uniform_logits():
    """All logits equal: lse = log V, top-1 is the lowest index, log p = -log V, and the
    posterior sample is uniform over the vocabulary."""
    V, d, R, L = 64, 8, 4096, 256
    E = np.random.default_rng(0).standard_normal((V, d))
    y = np.zeros((R, d))
    post = O.posterior(y, E, 1.0, seed=3, step=0, L=L)
    assert np.allclose(post["lse"], math.log(V), atol=1e-12)
    assert np.all(post["top1"] == 0)
    assert np.allclose(post["logp_top1"], -math.log(V), atol=1e-12)
    bins = np.bincount(post["x0hat"], minlength=V)
    assert stats.chisquare(bins).pvalue > 1e-4


def test_posterior_normalisation_and_temperature():
    V, d, R, L = 512, 32, 64, 16
    rng = np.random.default_rng(1)
    E = rng.standard_normal((V, d)) * 0.5
    y = rng.standard_normal((R, d))
    p1 = O.posterior(y, E, 2.0, seed=4, step=3, L=L)
    p2 = O.posterior(2.0 * y, E, 1.0, seed=4, step=3, L=L)
    for k in ("lse", "logp_top1", "logp_x0hat"):
        assert np.allclose(p1[k], p2[k], atol=1e-9)
    for k in ("top1", "x0hat"):
        assert np.array_equal(p1[k], p2[k])
    z = (y @ E.T) * 2.0
    # sum_v exp(logp_v) = 1, with logp_v = z_v - lse
    assert np.allclose(np.exp(z - p1["lse"][:, None]).sum(axis=1), 1.0, atol=1e-12)
    assert np.allclose(p1["lse"], logsumexp(z, axis=1), atol=1e-10)
    assert np.array_equal(p1["top1"], np.argmax(z, axis=1))
    assert np.all(p1["logp_x0hat"] <= p1["logp_top1"] + 1e-12)


def test_posterior_sample_is_the_softmax():
    """The posterior sample over 10^6 rows with distinct counters (one chunk: the within-chunk
    Gumbel-max alone) is a categorical draw from Softmax(z / tau): chi-square against the
    exact probabilities."""
    V, d = 16, 16
    z_target = np.linspace(-1.5, 1.0, V)
    E = np.eye(V, d)
    tau = 0.7
    R, L = 1_000_000, 1000
    y = np.broadcast_to(z_target, (R, d))
    post = O.posterior(y, E, 1.0 / tau, seed=2024, step=5, L=L, chunk=250000)
    counts = np.bincount(post["x0hat"], minlength=V)
    p = np.exp(z_target / tau - logsumexp(z_target / tau))
    assert stats.chisquare(counts, p * R).pvalue > 1e-3


def test_two_level_sample_over_many_chunks_is_the_softmax():
    """With 8 chunks of different masses (and uneven probabilities inside them), 4 x 10^5
    draws with distinct counters follow Softmax(z / tau): chi-square against the exact
    probabilities, per entry and per chunk."""
    V = 256
    rng = np.random.default_rng(77)
    z_target = rng.standard_normal(V) * 1.2
    z_target[64:96] += 1.5          # one heavy chunk
    z_target[160:192] -= 2.0        # one light chunk
    tau = 0.8
    R, L = 400_000, 1000
    y = np.broadcast_to(z_target, (R, V))
    post = O.posterior(y, np.eye(V), 1.0 / tau, seed=99, step=7, L=L, chunk=20000)
    p = np.exp(z_target / tau - logsumexp(z_target / tau))
    counts = np.bincount(post["x0hat"], minlength=V)
    assert stats.chisquare(counts, p * R).pvalue > 1e-3
    chunk_counts = counts.reshape(8, 32).sum(axis=1)
    assert stats.chisquare(chunk_counts, p.reshape(8, 32).sum(axis=1) * R).pvalue > 1e-3


def test_two_level_sample_hand_cases():
    """(a) All mass on one entry: always that entry.
    (b) Two equal entries in different chunks: the chunk whose Gumbel is larger wins (the
    lower chunk on an exact tie); inside a chunk with one live entry that entry is taken.
    (c) Two equal entries in one chunk: the entry whose own Gumbel (word v&3 of the pick
    stream's counter v>>2) is larger wins.
    (d) The reported margin is the smaller of the two levels' top-2 gaps, counted by brute
    force over the perturbed scores."""
    V, L = 64, 16
    z = np.full((6, V), -1e4)
    z[:, 21] = 3.0
    x, _ = O.two_level_sample(z, np.arange(6, dtype=np.uint64)[:, None] % L,
                              np.arange(6, dtype=np.uint64)[:, None] // L, 4, 8)
    assert np.all(x == 21)
    z = np.full((40, V), -1e4)
    z[:, 5] = 0.0
    z[:, 40] = 0.0
    pos = np.arange(40, dtype=np.uint64)[:, None] % L
    can = np.arange(40, dtype=np.uint64)[:, None] // L
    x, _ = O.two_level_sample(z, pos, can, 2, 31)
    k0, k1 = O.seed_key(31)
    w = O.philox4x32_10(0, pos[:, 0], can[:, 0], (O.STREAM_GUMBEL << 24) | 2, k0, k1)
    g0, g1 = O.gumbel_from_u32(w[0]), O.gumbel_from_u32(w[1])   # chunks 0 and 1: words 0, 1
    assert np.array_equal(x, np.where(g0 >= g1, 5, 40))
    assert 5 < (x == 5).sum() < 35
    # (c) entries 5 and 10 of chunk 0: counters 1 and 2, words 1 and 2 of the pick stream
    z = np.full((40, V), -1e4)
    z[:, 5] = 0.0
    z[:, 10] = 0.0
    x, _ = O.two_level_sample(z, pos, can, 6, 17)
    k0, k1 = O.seed_key(17)
    tag = (O.STREAM_PICK << 24) | 6
    g5 = O.gumbel_from_u32(O.philox4x32_10(1, pos[:, 0], can[:, 0], tag, k0, k1)[1])
    g10 = O.gumbel_from_u32(O.philox4x32_10(2, pos[:, 0], can[:, 0], tag, k0, k1)[2])
    assert np.array_equal(x, np.where(g5 >= g10, 5, 10))
    assert 5 < (x == 5).sum() < 35
    # (d) margins by brute force over every chunk score and the winning chunk's entries
    rng = np.random.default_rng(5)
    z = rng.standard_normal((40, V)) * 0.3
    x, margin = O.two_level_sample(z, pos, can, 3, 11)
    k0, k1 = O.seed_key(11)
    for r in range(40):
        cs = []
        for c in range(V // 32):
            u = O.philox4x32_10(c // 4, pos[r, 0], can[r, 0], (O.STREAM_GUMBEL << 24) | 3, k0, k1)
            cs.append(logsumexp(z[r, 32 * c:32 * c + 32]) + O.gumbel_from_u32(u[c % 4]))
        cstar = int(np.argmax(cs))
        es = []
        for v in range(32 * cstar, 32 * cstar + 32):
            u = O.philox4x32_10(v // 4, pos[r, 0], can[r, 0], (O.STREAM_PICK << 24) | 3, k0, k1)
            es.append(z[r, v] + O.gumbel_from_u32(u[v % 4]))
        assert x[r] == 32 * cstar + int(np.argmax(es))
        gaps = [np.diff(np.sort(a)[-2:])[0] for a in (np.array(cs), np.array(es))]
        assert math.isclose(margin[r], min(gaps), rel_tol=1e-12)


def test_posterior_rows_subset_equals_full():
    V, d, R, L = 256, 16, 48, 16
    rng = np.random.default_rng(9)
    E, y = rng.standard_normal((V, d)), rng.standard_normal((R, d))
    full = O.posterior(y, E, 1.0, 1, 2, L)
    rows = np.array([0, 5, 17, 47])
    sub = O.posterior(y, E, 1.0, 1, 2, L, rows=rows)
    for k in full:
        assert np.allclose(full[k][rows], sub[k])


# -------------------------------------------------------------------- Euler step -----

def test_euler_one_hot_posterior_at_last_step_returns_x0():
    """With the posterior one-hot at x_0 and h = t (the last step, lambda = 1) every position
    lands on x_0."""
    V, B, L, T = 4096, 3, 256, 12
    rng = np.random.default_rng(3)
    x0 = rng.integers(0, V, (B, L))
    xt = rng.integers(0, V, (B, L))
    _, jump = O.schedule_thresholds(O.SCHED_COSINE, T)
    lock = np.zeros((B, L), np.uint8)
    x, lk, jmp, done = O.euler_update(xt, x0, x0, np.zeros((B, L), np.float32), lock, 1, T - 1,
                                      int(jump[T - 1]), float("inf"))
    assert np.array_equal(x, x0) and jmp.all() and not lk.any() and not done.any()


def test_euler_delta_posterior_is_a_fixed_point_and_rate_matches():
    V, B, L, T, n = 4096, 64, 256, 12, 4
    rng = np.random.default_rng(4)
    xt = rng.integers(0, V, (B, L))
    x0hat = rng.integers(0, V, (B, L))
    lock = np.zeros((B, L), np.uint8)
    _, jump = O.schedule_thresholds(O.SCHED_LINEAR, T)
    x, _, jmp, _ = O.euler_update(xt, xt, xt, np.full((B, L), -9.0, np.float32), lock, 3, n,
                                  int(jump[n]), float("inf"))
    assert np.array_equal(x, xt)                               # posterior delta_{x_t}: no move
    x, _, jmp, _ = O.euler_update(xt, x0hat, x0hat, np.full((B, L), -9.0, np.float32), lock, 3,
                                  n, int(jump[n]), float("inf"))
    lam = 1.0 / (T - n)
    N = B * L
    assert abs(jmp.mean() - lam) < 5 * math.sqrt(lam * (1 - lam) / N)
    assert np.array_equal(x, np.where(jmp.astype(bool), x0hat, xt))


def test_euler_lock_precedes_jump_and_locked_positions_freeze():
    V, B, L = 100, 2, 64
    rng = np.random.default_rng(5)
    xt = rng.integers(0, V, (B, L))
    x0hat = (xt + 1) % V
    top1 = (xt + 2) % V
    lp = np.full((B, L), -5.0, np.float32)
    lp[:, ::3] = -0.01                                          # confident positions
    lock = np.zeros((B, L), np.uint8)
    lock[:, 1] = 1                                              # already locked
    thr = np.float32(math.log(0.9))
    x, lk, jmp, done = O.euler_update(xt, x0hat, top1, lp, lock, 8, 0, 1 << 32, float(thr))
    conf = np.zeros((B, L), bool)
    conf[:, ::3] = True
    assert np.array_equal(x[:, 1], xt[:, 1]) and lk[:, 1].all()
    assert np.array_equal(x[conf], top1[conf]) and lk[conf].all() and not jmp[conf].any()
    rest = ~conf
    rest[:, 1] = False
    assert np.array_equal(x[rest], x0hat[rest]) and jmp[rest].all() and not lk[rest].any()
    assert not done.any()
    lock_all = np.ones((B, L), np.uint8)
    _, _, _, done = O.euler_update(xt, x0hat, top1, lp, lock_all, 8, 0, 1 << 32, float(thr))
    assert done.all()


# ------------------------------------------------------------------------- loop -----

def _planted_model(V, d, H, Hkv, hd, scale=8.0):
    """A decoder whose posterior is (numerically) delta at the input token: orthogonal
    embeddings of norm `scale` and a zero output projection, so y = E[x_t] and the logits
    are scale^2 at x_t and 0 elsewhere."""
    rng = np.random.default_rng(0)
    E = np.zeros((V, d))
    E[np.arange(V), np.arange(V)] = scale
    return {"E": E, "Wqkv": rng.standard_normal(((H + 2 * Hkv) * hd, d)) * 0.02,
            "Wo": np.zeros((d, H * hd)), "H": H, "Hkv": Hkv, "hd": hd}


def test_loop_with_delta_posterior_keeps_canvas_and_locks_at_once():
    V, d, H, Hkv, hd, B, L, P, T = 64, 64, 2, 1, 16, 2, 64, 16, 6
    m = _planted_model(V, d, H, Hkv, hd)
    rng = np.random.default_rng(1)
    kp, vp = rng.standard_normal((2, B, P, Hkv, hd))
    x1 = O.initial_canvas(B, L, V, 42)
    lock = np.zeros((B, L), np.uint8)
    x, lk, steps = O.denoise_loop(m, kp, vp, 0, x1, lock, T, O.SCHED_LINEAR, 1.0,
                                  float("inf"), 42)
    assert np.array_equal(x, x1) and not lk.any() and np.all(steps == T)
    x, lk, steps = O.denoise_loop(m, kp, vp, 0, x1, lock, T, O.SCHED_LINEAR, 1.0,
                                  float(np.float32(math.log(0.9))), 42, stop_when_all_locked=True)
    assert np.array_equal(x, x1) and lk.all() and np.all(steps == 1)


def test_loop_resume_is_deterministic():
    """Running steps 0..5 and then 6..11 equals running 0..11 (counters depend only on
    seed, step, canvas and position)."""
    V, d, H, Hkv, hd, B, L, P, T = 512, 64, 4, 2, 16, 2, 64, 32, 12
    rng = np.random.default_rng(2)
    m = {"E": O.round_bf16(rng.standard_normal((V, d)) * 0.3),
         "Wqkv": O.round_bf16(rng.standard_normal(((H + 2 * Hkv) * hd, d)) * 0.2),
         "Wo": O.round_bf16(rng.standard_normal((d, H * hd)) * 0.2), "H": H, "Hkv": Hkv, "hd": hd}
    kp, vp = O.round_bf16(rng.standard_normal((2, B, P, Hkv, hd)))
    x1 = O.initial_canvas(B, L, V, 7)
    lock = np.zeros((B, L), np.uint8)
    thr = float(np.float32(math.log(0.3)))
    xa, la, sa = O.denoise_loop(m, kp, vp, 24, x1, lock, T, O.SCHED_COSINE, 1.0, thr, 7)
    xh, lh, sh = O.denoise_loop(m, kp, vp, 24, x1, lock, T, O.SCHED_COSINE, 1.0, thr, 7,
                                end_step=6)
    xb, lb, sb = O.denoise_loop(m, kp, vp, 24, xh, lh, T, O.SCHED_COSINE, 1.0, thr, 7,
                                start_step=6)
    assert np.array_equal(xa, xb) and np.array_equal(la, lb)
    assert np.array_equal(sa, sh + sb)
    assert (xa != x1).mean() > 0.2                              # the canvas did move
    assert 0 < la.mean() < 1                                    # and some positions locked


# ---------------------------------------------------------------------- metrics -----

def _golden(name):
    vals = {}
    for line in open(os.path.join(ROOT, "tests", "golden", name), encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            k, *v = line.split()
            vals[k] = [float(x) for x in v]
    return vals


def test_metrics_match_the_pages():
    from discrete_diffusion_text_gb300 import metrics as M

    g = _golden("tps_batch1.txt")
    tps = M.tokens_per_second(g["tpf"][0], g["t_fwd_ms"][0] / 1000.0)
    assert round(tps) == g["tps"][0]
    for k in ("aime2026", "gpqa_diamond", "gsm8k"):
        tpf, tps_k = g[k]
        assert 0.010 < tpf / tps_k < 0.020
    # hand-made two-canvas example: n = (256, 100), s = (12, 6)
    n, s = [256, 100], [12, 6]
    assert M.total_tokens(n) == 356 and M.total_denoising_steps(s) == 18
    assert M.effective_denoising_steps(n, s) == pytest.approx((256 * 12 + 100 * 6) / 356)
    assert M.tokens_per_forward(n, s) == pytest.approx(356 / 19)
    assert M.valid_tokens([5, 7, 1, 9]) == 2 and M.valid_tokens([5, 7]) == 2


# ------------------------------------------------------- entropy-bounded sampler -----

def test_posterior_entropy_matches_scipy_and_closed_forms():
    """Entropy of the tempered posterior: scipy.stats.entropy on random logits, log V for
    uniform logits, log 4 for four equal dominant logits, and the binary closed form
    H = -p log p - (1-p) log(1-p) with p = sigmoid(delta / tau)."""
    V, d, R, L = 300, 300, 24, 8
    rng = np.random.default_rng(7)
    E = np.eye(V, d)
    y = rng.standard_normal((R, d)) * 2.0
    tau = 0.6
    post = O.posterior(y, E, 1.0 / tau, seed=1, step=0, L=L)
    ref = stats.entropy(np.exp((y / tau) - logsumexp(y / tau, axis=1, keepdims=True)), axis=1)
    assert np.allclose(post["entropy"], ref, atol=1e-10)
    uni = O.posterior(np.zeros((2, d)), E, 1.0, seed=1, step=0, L=L)
    assert np.allclose(uni["entropy"], math.log(V), atol=1e-12)
    four = np.full((1, d), -60.0)
    four[0, [3, 50, 51, 299]] = 5.0
    assert abs(O.posterior(four, E, 1.0, seed=1, step=0, L=L)["entropy"][0] - math.log(4)) < 1e-9
    for delta in (0.0, 0.3, 2.0, 9.0):
        two = np.full((1, d), -80.0)
        two[0, 0], two[0, 1] = delta, 0.0
        p = 1.0 / (1.0 + math.exp(-delta / tau))
        h = -(p * math.log(p) + (1 - p) * math.log(1 - p))
        got = O.posterior(two, E, 1.0 / tau, seed=1, step=0, L=L)["entropy"][0]
        assert abs(got - h) < 1e-9, (delta, got, h)


def test_annealed_temperature_endpoints_and_linearity():
    """0.8 at the first step, 0.4 at the last possible step, equal decrements in between."""
    for T in (2, 12, 48):
        tau = O.annealed_temperature(T)
        assert tau[0] == 0.8 and abs(tau[-1] - 0.4) < 1e-15
        assert np.allclose(np.diff(tau), -0.4 / (T - 1), atol=1e-15)
    assert O.annealed_temperature(1)[0] == 0.8
    inv = O.eb_inv_tau(48, 0.8, 0.4)
    assert inv[0] == float(np.float32(1.25)) and inv[-1] == float(np.float32(2.5))


def test_entropy_bounded_select_hand_examples():
    """Worked cases: ordering by (entropy, position), a running sum equal to gamma is still
    accepted, k = 0 when the smallest entropy exceeds gamma, all-zero entropies accept all."""
    cases = [
        ([0.05, 0.0, 0.03, 0.04, 0.0], 0.1, [0, 1, 1, 1, 1], 4),
        ([0.2, 0.3, 0.11], 0.1, [0, 0, 0], 0),
        ([0.0, 0.0, 0.0, 0.0], 0.1, [1, 1, 1, 1], 4),
        ([0.05, 0.05, 0.05], 0.1, [1, 1, 0], 2),          # tie broken by position
        ([0.0625, 0.03125, 0.0625], 0.09375, [1, 1, 0], 2),  # exact dyadic sum == gamma
        ([0.1, 0.0], 0.1, [1, 1], 2),
    ]
    for H, g, want, k in cases:
        acc, kk = O.entropy_bounded_select(np.array([H], np.float32), g)
        assert acc[0].tolist() == want and int(kk[0]) == k, (H, g, acc, kk)


def test_renoise_stream_is_uniform_and_distinct():
    """Re-noised tokens are uniform over V (chi-square) and differ from the noising and jump
    streams of the same counters."""
    V, B, L = 64, 400, 256
    tok = O.renoise_tokens(B, L, V, seed=11, step=3)
    assert stats.chisquare(np.bincount(tok.reshape(-1), minlength=V)).pvalue > 1e-4
    init = O.initial_canvas(B, L, V, seed=11)
    assert (tok != init).mean() > 0.9
    assert (O.renoise_tokens(B, L, V, seed=11, step=4) != tok).mean() > 0.9


def test_entropy_bounded_update_decisions():
    """Accepted positions take x0hat and the rest fresh tokens; done needs both the entropy
    test and an unchanged top-1 sequence; done canvases and the final step return top-1."""
    B, L, V = 3, 6, 50
    x0hat = np.arange(B * L).reshape(B, L) % V
    top1 = (np.arange(B * L).reshape(B, L) * 7) % V
    H = np.array([[0.0] * 6, [0.001] * 6, [0.0, 0.5, 0.5, 0.5, 0.5, 0.0]], np.float32)
    prev = top1.copy()
    prev[1, 2] += 1  # canvas 1 changed its prediction
    x_out, acc, done, mh = O.entropy_bounded_update(x0hat, top1, H, prev, 5, 2, V, 0.1, 0.005)
    assert done.tolist() == [1, 0, 0]
    assert np.array_equal(x_out[0], top1[0])                      # done -> top-1
    assert acc[1].tolist() == [1] * 6 and np.array_equal(x_out[1], x0hat[1])
    rn = O.renoise_tokens(B, L, V, 5, 2)
    assert acc[2].tolist() == [1, 0, 0, 0, 0, 1]
    assert np.array_equal(x_out[2], np.where(acc[2] == 1, x0hat[2], rn[2]))
    assert abs(float(mh[2]) - 2.0 / 6.0) < 1e-7
    _, _, done0, _ = O.entropy_bounded_update(x0hat, top1, H, None, 5, 2, V, 0.1, 0.005)
    assert done0.tolist() == [0, 0, 0]                            # no previous prediction
    xf, _, _, _ = O.entropy_bounded_update(x0hat, top1, H, None, 5, 2, V, 0.1, 0.005, True)
    assert np.array_equal(xf, top1)                               # final step


def _peaked_model(V, d, H, Hkv, hd, scale, seed):
    rng = np.random.default_rng(seed)
    E = rng.standard_normal((V, d))
    E = E / np.linalg.norm(E, axis=1, keepdims=True) * scale
    E = O.round_bf16(E)
    Wqkv = O.round_bf16(rng.standard_normal(((H + 2 * Hkv) * hd, d)) * 0.02)
    Wo = O.round_bf16(rng.standard_normal((d, H * hd)) * 0.02)
    return {"E": E, "Wqkv": Wqkv, "Wo": Wo, "H": H, "Hkv": Hkv, "hd": hd}


def test_entropy_bounded_loop_fixed_point_stops_after_two_steps():
    """With large, nearly orthogonal embedding rows the posterior at each position is
    concentrated on the token already there: entropies ~0, every position is accepted with its
    (identical) sample, the prediction is unchanged at the second step, and the loop stops
    there returning the initial canvas."""
    V, d, H, Hkv, hd, B, L, P = 512, 128, 2, 2, 64, 2, 16, 8
    model = _peaked_model(V, d, H, Hkv, hd, 20.0, 3)
    rng = np.random.default_rng(4)
    k_pre = O.round_bf16(rng.standard_normal((B, P, Hkv, hd)))
    v_pre = O.round_bf16(rng.standard_normal((B, P, Hkv, hd)))
    x = O.initial_canvas(B, L, V, seed=9)
    out, steps = O.eb_denoise_loop(model, k_pre, v_pre, 0, x, 48, 0.8, 0.4, 0.1, 0.005, 9)
    assert steps.tolist() == [2, 2]
    assert np.array_equal(out, x)


def test_entropy_bounded_loop_uninformed_model_runs_to_the_cap():
    """Near-uniform posteriors (entropy ~ log V > gamma): nothing is accepted, every position is
    re-noised each step, and the loop runs all T steps, returning the last top-1 sequence."""
    V, d, H, Hkv, hd, B, L, P, T = 256, 64, 2, 1, 64, 2, 16, 4, 5
    rng = np.random.default_rng(5)
    model = {"E": O.round_bf16(rng.standard_normal((V, d)) * 0.02),
             "Wqkv": O.round_bf16(rng.standard_normal(((H + 2 * Hkv) * hd, d)) * 0.02),
             "Wo": O.round_bf16(rng.standard_normal((d, H * hd)) * 0.02), "H": H, "Hkv": Hkv, "hd": hd}
    k_pre = O.round_bf16(rng.standard_normal((B, P, Hkv, hd)))
    v_pre = O.round_bf16(rng.standard_normal((B, P, Hkv, hd)))
    x = O.initial_canvas(B, L, V, seed=6)
    out, steps = O.eb_denoise_loop(model, k_pre, v_pre, 0, x, T, 0.8, 0.4, 0.1, 0.005, 6)
    assert steps.tolist() == [T, T]
    # the last step's canvas: re-noised tokens of steps 0..T-2, then top-1 at the last step
    xs = x.copy()
    inv = O.eb_inv_tau(T, 0.8, 0.4)
    for n in range(T - 1):
        xs, acc, _, _, _ = O.eb_denoise_step(model, k_pre, v_pre, 0, xs, n, inv[n], None, 6,
                                             0.1, 0.005, False)
        assert acc.sum() == 0
        assert np.array_equal(xs, O.renoise_tokens(B, L, V, 6, n))
    _, _, _, _, post = O.eb_denoise_step(model, k_pre, v_pre, 0, xs, T - 1, inv[T - 1], None, 6,
                                         0.1, 0.005, True)
    assert np.array_equal(out, post["top1"].reshape(B, L))


# --------------------------------------------------------------- SFT cross-entropy -----

def test_cross_entropy_matches_torch_and_closed_forms():
    """Against torch.nn.functional.cross_entropy in float64 (an independent implementation), log V
    for uniform logits, and ~0 for a dominant correct logit."""
    V, d, R = 500, 64, 40
    rng = np.random.default_rng(21)
    E = rng.standard_normal((V, d)) * 0.3
    y = rng.standard_normal((R, d))
    tgt = rng.integers(0, V, R)
    loss, lse = O.cross_entropy(y, E, 1.7, tgt)
    z = torch.tensor((y @ E.T) * 1.7)
    ref = torch.nn.functional.cross_entropy(z, torch.tensor(tgt), reduction="none").numpy()
    assert np.allclose(loss, ref, atol=1e-10)
    assert np.allclose(lse, torch.logsumexp(z, dim=1).numpy(), atol=1e-10)
    uni, _ = O.cross_entropy(np.zeros((3, d)), E, 1.0, [0, 7, 499])
    assert np.allclose(uni, math.log(V), atol=1e-12)
    Ei = np.eye(V, d)
    yy = np.zeros((2, d))
    yy[0, 5], yy[1, 9] = 60.0, 60.0
    sharp, _ = O.cross_entropy(yy, Ei, 1.0, [5, 9])
    assert np.all(sharp < 1e-20)
    wrong, _ = O.cross_entropy(yy, Ei, 1.0, [6, 10])
    assert np.allclose(wrong, 60.0, atol=1e-9)


def test_sft_loss_is_the_cross_entropy_of_the_noised_canvas():
    """keep = 1 (t = 0) leaves x_0 unchanged; the loss equals the cross-entropy of the decoder on
    x_0; with t = 1 every token is redrawn; per-canvas thresholds act per canvas."""
    V, d, H, Hkv, hd, B, L, P = 256, 64, 2, 1, 64, 2, 16, 4
    rng = np.random.default_rng(22)
    model = {"E": O.round_bf16(rng.standard_normal((V, d)) * 0.5),
             "Wqkv": O.round_bf16(rng.standard_normal(((H + 2 * Hkv) * hd, d)) * 0.02),
             "Wo": O.round_bf16(rng.standard_normal((d, H * hd)) * 0.02), "H": H, "Hkv": Hkv, "hd": hd}
    k_pre = O.round_bf16(rng.standard_normal((B, P, Hkv, hd)))
    v_pre = O.round_bf16(rng.standard_normal((B, P, Hkv, hd)))
    x0 = rng.integers(0, V, (B, L))
    full = np.array([1 << 32, 0], np.uint64)  # canvas 0 kept (kappa = 1), canvas 1 fully noised
    loss, xt = O.sft_loss(model, k_pre, v_pre, 0, x0, full, seed=3)
    assert np.array_equal(xt[0], x0[0])
    assert np.mean(xt[1] != x0[1]) > 0.9
    h, q, kc, vc = O.decoder_front(x0, model["E"], model["Wqkv"], H, Hkv, hd)
    Oa, _ = O.canvas_attention(q, k_pre, v_pre, kc, vc, 0, hd ** -0.5)
    y = O.decoder_back(h, Oa, model["Wo"])
    ref, _ = O.cross_entropy(y.reshape(B * L, -1)[:L], model["E"], 1.0, x0[0])
    # canvas 0's decoder input is x_0 itself, but its attention sees canvas 0 only: compare it
    assert np.allclose(loss[0], ref, atol=1e-9)


# ------------------------------------------------------ encode-append + block-AR loop -----

def _delta_model(V, d, H, Hkv, hd, seed):
    """Embedding 8 * I (V = d): the posterior is a delta at the token already there, so every
    denoising loop returns its initial canvas."""
    rng = np.random.default_rng(seed)
    return {"E": np.eye(V, d) * 8.0,
            "Wqkv": O.round_bf16(rng.standard_normal(((H + 2 * Hkv) * hd, d)) * 0.02),
            "Wo": np.zeros((d, H * hd)), "H": H, "Hkv": Hkv, "hd": hd}


def test_encode_append_writes_the_key_and_value_projections():
    """Rows P..P+L-1 become E[x] Wk^T and E[x] Wv^T (Wk, Wv: the key and value row blocks of
    Wqkv, rounded to bf16); other rows and other canvases are untouched."""
    V, d, H, Hkv, hd, B, L, P = 64, 64, 2, 1, 64, 3, 8, 5
    m = _delta_model(V, d, H, Hkv, hd, 1)
    rng = np.random.default_rng(2)
    canvas = rng.integers(0, V, (B, L))
    kc = rng.standard_normal((B, P + L + 4, Hkv, hd))
    vc = rng.standard_normal((B, P + L + 4, Hkv, hd))
    k0, v0 = kc.copy(), vc.copy()
    O.encode_append(m, canvas, kc, vc, P, rows=[0, 2])
    Wk = m["Wqkv"][H * hd:(H + Hkv) * hd]
    Wv = m["Wqkv"][(H + Hkv) * hd:]
    for b in (0, 2):
        emb = m["E"][canvas[b]]
        assert np.allclose(kc[b, P:P + L], O.round_bf16(emb @ Wk.T).reshape(L, Hkv, hd), atol=0)
        assert np.allclose(vc[b, P:P + L], O.round_bf16(emb @ Wv.T).reshape(L, Hkv, hd), atol=0)
    assert np.array_equal(kc[1], k0[1]) and np.array_equal(vc[1], v0[1])
    assert np.array_equal(kc[:, :P], k0[:, :P]) and np.array_equal(kc[:, P + L:], k0[:, P + L:])


def test_block_generate_with_delta_posterior_and_eos():
    """Each block returns its own uniform-prior canvas (seed + j); a canvas stops at the first
    block containing the end-of-turn token, with the response length counted up to it; the KV
    cache grows by one canvas per generated block."""
    V, d, H, Hkv, hd, B, L, P0, NB, T = 256, 256, 2, 1, 64, 3, 16, 8, 4, 3
    m = _delta_model(V, d, H, Hkv, hd, 3)
    rng = np.random.default_rng(4)
    k_ctx = O.round_bf16(rng.standard_normal((B, P0, Hkv, hd)))
    v_ctx = O.round_bf16(rng.standard_normal((B, P0, Hkv, hd)))
    seed = 10
    inits = [O.initial_canvas(B, L, V, seed + j) for j in range(NB)]
    eos = int(inits[1][0, 5])  # canvas 0 meets it in block 1 (if not already in block 0)
    out, blocks, n_tok, steps, kc, vc = O.block_generate(m, k_ctx, v_ctx, 0, L, NB, eos, seed, T)
    for b in range(B):
        stop = next((j for j in range(NB) if eos in inits[j][b]), None)
        nb = NB if stop is None else stop + 1
        assert blocks[b] == nb
        for j in range(nb):
            assert np.array_equal(out[b, j], inits[j][b])
        assert np.all(out[b, nb:] == -1)
        n_exp = NB * L if stop is None else stop * L + int(np.nonzero(inits[stop][b] == eos)[0][0]) + 1
        assert n_tok[b] == n_exp
        assert steps[b] == nb * T
        assert np.array_equal(kc[b, :P0], k_ctx[b])
    assert blocks[0] <= 2


# ------------------------------------------------------------- self-conditioning -----

def test_gelu_tanh_matches_torch_and_its_symmetry():
    """The tanh-form GELU against torch's independent implementation, its values at 0 and in
    the tails, and gelu(x) - gelu(-x) = x (the gate and its mirror add up to one)."""
    x = np.linspace(-12.0, 12.0, 4001)
    ref = torch.nn.functional.gelu(torch.tensor(x), approximate="tanh").numpy()
    assert np.abs(O.gelu_tanh(x) - ref).max() <= 1e-15
    assert O.gelu_tanh(0.0) == 0.0
    assert abs(O.gelu_tanh(12.0) - 12.0) < 1e-12 and abs(O.gelu_tanh(-12.0)) < 1e-12
    assert np.abs(O.gelu_tanh(x) - O.gelu_tanh(-x) - x).max() <= 1e-13


def test_expected_embedding_closed_forms():
    """p_hat . E for (a) E = c I: the softmax itself scaled by c (scipy); (b) y = 0: the mean
    embedding row; (c) one logit ahead by 60 nats: that row of E; (d) brute force over a
    5-token vocabulary with explicit loops."""
    from scipy.special import softmax

    rng = np.random.default_rng(11)
    V = d = 32
    c = 1.7
    E = c * np.eye(V)
    y = rng.standard_normal((6, d))
    e = O.expected_embedding(y, E, 0.8)
    assert np.abs(e - c * softmax(y @ E.T * 0.8, axis=1)).max() <= 1e-14
    E2 = rng.standard_normal((50, 8))
    assert np.abs(O.expected_embedding(np.zeros((3, 8)), E2, 1.3) - E2.mean(axis=0)).max() < 1e-14
    y3 = np.zeros((1, 8))
    y3[0, 2] = 1.0
    E3 = rng.standard_normal((50, 8)) * 0.01
    E3[17, 2] = 60.0
    assert np.abs(O.expected_embedding(y3, E3, 1.0)[0] - E3[17]).max() < 1e-20 + 1e-24 * 60
    E4 = rng.standard_normal((5, 3))
    y4 = rng.standard_normal((2, 3))
    for r in range(2):
        w = [math.exp(0.5 * sum(y4[r, k] * E4[v, k] for k in range(3))) for v in range(5)]
        tot = sum(w)
        want = [sum(w[v] / tot * E4[v, j] for v in range(5)) for j in range(3)]
        assert np.allclose(O.expected_embedding(y4[r:r + 1], E4, 0.5)[0], want, rtol=1e-13,
                           atol=1e-15)


def test_expected_embedding_is_invariant_to_vocabulary_order():
    """Relabelling the vocabulary (a permutation of E's rows) changes nothing."""
    rng = np.random.default_rng(12)
    E = rng.standard_normal((300, 16))
    y = rng.standard_normal((4, 16))
    perm = rng.permutation(300)
    a = O.expected_embedding(y, E, 1.25)
    b = O.expected_embedding(y, E[perm], 1.25)
    assert np.abs(a - b).max() < 1e-13


def test_self_condition_feed_forward_layers():
    """With identity layers s = bf16(gelu(bf16(e))) (torch's GELU); a zero second layer gives
    s = 0; the first layer acts on e, the second on gelu of the first (a swapped order or a
    transposed weight fails the rectangular case, checked with torch matmuls)."""
    rng = np.random.default_rng(13)
    V, d = 64, 16
    E = O.round_bf16(rng.standard_normal((V, d)))
    y = O.round_bf16(rng.standard_normal((5, d)))
    r = O.self_condition(y, E, 1.0, np.eye(d), np.eye(d))
    e_b = O.round_bf16(O.expected_embedding(y, E, 1.0))
    g = torch.nn.functional.gelu(torch.tensor(e_b), approximate="tanh").numpy()
    assert np.array_equal(r["e"], e_b)
    assert np.array_equal(r["s"], O.round_bf16(O.round_bf16(g)))
    assert not O.self_condition(y, E, 1.0, np.eye(d), np.zeros((d, d)))["s"].any()
    W1 = O.round_bf16(rng.standard_normal((24, d)) * 0.3)
    W2 = O.round_bf16(rng.standard_normal((d, 24)) * 0.3)
    r = O.self_condition(y, E, 0.7, W1, W2)
    tu = torch.nn.functional.gelu(torch.tensor(r["e"]) @ torch.tensor(W1).T, approximate="tanh")
    u = O.round_bf16(tu.numpy())
    assert np.array_equal(r["u"], u)
    assert np.array_equal(r["s"], O.round_bf16((torch.tensor(u) @ torch.tensor(W2).T).numpy()))
    assert r["s"].shape == (5, d) and r["u"].shape == (5, 24)


def _sc_model(V, d, H, Hkv, hd, dsc, seed, w2_scale=0.5):
    rng = np.random.default_rng(seed)
    return {"E": O.round_bf16(rng.standard_normal((V, d)) * 0.3),
            "Wqkv": O.round_bf16(rng.standard_normal(((H + 2 * Hkv) * hd, d)) * 0.2),
            "Wo": O.round_bf16(rng.standard_normal((d, H * hd)) * 0.2), "H": H, "Hkv": Hkv,
            "hd": hd, "Wsc1": O.round_bf16(rng.standard_normal((dsc, d)) * 0.3),
            "Wsc2": O.round_bf16(rng.standard_normal((d, dsc)) * w2_scale)}


def test_self_conditioning_signal_enters_the_embedding():
    """With zero attention weights the decoder output is h itself, so the step's logits are
    bf16(E[x] + s) E^T: the posterior of a step given s equals the posterior of that y."""
    V, d, H, Hkv, hd, B, L, P = 128, 32, 2, 1, 16, 2, 8, 4
    m = _sc_model(V, d, H, Hkv, hd, 32, 14)
    m["Wqkv"] = np.zeros_like(m["Wqkv"])
    m["Wo"] = np.zeros_like(m["Wo"])
    rng = np.random.default_rng(15)
    kp, vp = rng.standard_normal((2, B, P, Hkv, hd))
    x = rng.integers(0, V, (B, L))
    s = O.round_bf16(rng.standard_normal((B, L, d)))
    post = O.decoder_posterior(m, kp, vp, 0, x, 3, 1.1, 5, s)
    y = O.round_bf16(m["E"][x] + s).reshape(B * L, d)
    ref = O.posterior(y, m["E"], 1.1, 5, 3, L)
    assert np.array_equal(post["x0hat"], ref["x0hat"]) and np.allclose(post["lse"], ref["lse"])
    want_s = O.self_condition(y, m["E"], 1.1, m["Wsc1"], m["Wsc2"])["s"].reshape(B, L, d)
    assert np.array_equal(post["s"], want_s)
    post0 = O.decoder_posterior(m, kp, vp, 0, x, 3, 1.1, 5, None)
    assert not np.allclose(post0["lse"], post["lse"])


def test_self_conditioning_loop_wiring():
    """A zero second layer makes every signal zero, so the loop equals the loop of the model
    without self-conditioning; with a real signal the loop differs from it, and splitting the
    run at step 4 (carrying the signal) reproduces the whole run, for both samplers."""
    V, d, H, Hkv, hd, B, L, P, T = 256, 32, 2, 1, 16, 2, 16, 8, 8
    m = _sc_model(V, d, H, Hkv, hd, 32, 16)
    rng = np.random.default_rng(17)
    kp, vp = O.round_bf16(rng.standard_normal((2, B, P, Hkv, hd)))
    x1 = O.initial_canvas(B, L, V, 3)
    lock = np.zeros((B, L), np.uint8)
    plain = {k: v for k, v in m.items() if k not in ("Wsc1", "Wsc2")}
    zero2 = dict(m, Wsc2=np.zeros_like(m["Wsc2"]))
    args = (kp, vp, 0, x1, lock, T, O.SCHED_LINEAR, 1.0, float("inf"), 3)
    xp, _, _ = O.denoise_loop(plain, *args)
    xz, _, _ = O.denoise_loop(zero2, *args)
    xs, _, ss = O.denoise_loop(m, *args)
    assert np.array_equal(xp, xz)
    assert (xs != xp).mean() > 0.05
    st = {}
    xh, lh, sh = O.denoise_loop(m, *args, end_step=4, state=st)
    assert st["s"] is not None and st["s"].any()
    xb, _, sb = O.denoise_loop(m, kp, vp, 0, xh, lh, T, O.SCHED_LINEAR, 1.0, float("inf"), 3,
                               start_step=4, state=st)
    assert np.array_equal(xb, xs) and np.array_equal(sh + sb, ss)
    ep, _ = O.eb_denoise_loop(plain, kp, vp, 0, x1, T, 0.8, 0.4, 0.1, 0.005, 3)
    ez, _ = O.eb_denoise_loop(zero2, kp, vp, 0, x1, T, 0.8, 0.4, 0.1, 0.005, 3)
    es, _ = O.eb_denoise_loop(m, kp, vp, 0, x1, T, 0.8, 0.4, 0.1, 0.005, 3)
    assert np.array_equal(ep, ez) and not np.array_equal(ep, es)
