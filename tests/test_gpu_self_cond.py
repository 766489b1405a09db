"""GPU parity of self-conditioning (s = FFW(p_hat . E)) against the CPU oracle: the standalone
call, and the denoising loop with the signal fed back.  Every call goes through the C ABI."""

import dataclasses
import math

import numpy as np
import pytest
import torch

from discrete_diffusion_text_gb300 import synth
from oracle import dgoracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"
U = 2.0 ** -8  # unit roundoff of bf16 (round to nearest)
GUMBEL_TIE = 1e-3


@pytest.fixture(scope="module")
def dgc():
    import os

    from discrete_diffusion_text_gb300 import dgcanvas

    if not os.path.exists(dgcanvas.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build()
    dgcanvas.load()
    return dgcanvas


def f64(t):
    return t.double().cpu().numpy()


def _run_sc(dgc, y, E, W1, W2, B, L, inv_tau):
    R, d = y.shape
    s = torch.empty((R, d), dtype=torch.bfloat16, device=DEV)
    e = torch.empty((R, d), dtype=torch.bfloat16, device=DEV)
    ws = dgc.workspace(dgc.dg_self_condition_workspace(B, L, d, E.shape[0], W1.shape[0]))
    dgc.dg_self_condition(y.to(DEV), E.to(DEV), W1.to(DEV), W2.to(DEV), B, L, inv_tau, s, ws,
                          e_out=e)
    dgc.dg_workspace_status(ws)
    return f64(e), f64(s)


def _check_e(e_gpu, y, E, inv_tau, rows=None):
    """|e_gpu - e| <= 2u * sum_v p_v |E_vj| (the stored and the rescaled bf16 posterior) + u |e|
    (the final rounding) + 1e-7, elementwise; e, p in float64 from the oracle."""
    y64, E64 = f64(y), f64(E)
    if rows is not None:
        y64 = y64[rows]
        e_gpu = e_gpu[rows]
    e = O.expected_embedding(y64, E64, inv_tau)
    z = y64 @ E64.T * inv_tau
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    bound = 2 * U * (p @ np.abs(E64)) + U * np.abs(e) + 1e-7
    err = np.abs(e_gpu - e)
    assert np.all(err <= bound), float((err / bound).max())
    return e


def _check_ffw(s_gpu, e_gpu, W1, W2):
    """s against the oracle's feed-forward applied to the GPU's own e: the first layer's output
    may round to a neighbouring bf16 value (fp32 vs float64 sums), which moves s by at most
    u sum_k |u_k W2_jk|; then one more rounding."""
    W1_64, W2_64 = f64(W1), f64(W2)
    u = O.round_bf16(O.gelu_tanh(e_gpu @ W1_64.T))
    s = O.round_bf16(u @ W2_64.T)
    bound = 2 * U * (np.abs(u) @ np.abs(W2_64).T) + U * np.abs(s) + 1e-7
    err = np.abs(s_gpu - s)
    assert np.all(err <= bound), float((err / bound).max())
    assert (s_gpu == s).mean() > 0.9


def _check_s_end_to_end(s_gpu, y, E, W1, W2, inv_tau):
    """s against the oracle's own s = bf16(bf16(gelu(bf16(e) W1^T)) W2^T): the GPU's e is
    within the _check_e bound of the exact e and the oracle rounds e once more (u |e|); that
    difference passes through |W1|, the GELU's slope (at most 1.13 for the tanh form; 1.15
    used), a bf16 rounding of u on each side (2u |u|), |W2| and a rounding of s (2u |s|)."""
    y64, E64, W1_64, W2_64 = f64(y), f64(E), f64(W1), f64(W2)
    ref = O.self_condition(y64, E64, inv_tau, W1_64, W2_64)
    z = y64 @ E64.T * inv_tau
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    de = 2 * U * (p @ np.abs(E64)) + 2 * U * np.abs(ref["e_exact"]) + 1e-7
    du = 1.15 * (de @ np.abs(W1_64).T) + 2 * U * np.abs(ref["u"]) + 1e-7
    bound = du @ np.abs(W2_64).T + 2 * U * np.abs(ref["s"]) + 1e-7
    err = np.abs(s_gpu - ref["s"])
    assert np.all(err <= bound), float((err / bound).max())


@pytest.mark.parametrize("B,L,V,d,dsc,ystd,inv_tau", [
    (2, 128, 4096, 256, 128, 0.05, 1.0),    # near-uniform posterior
    (1, 256, 8192, 512, 192, 1.0, 2.0),     # sharp posterior
    (3, 64, 4096, 256, 64, 0.5, 1.25),      # in between, three canvases
    (8, 256, 4096, 256, 128, 0.5, 1.25),    # 16 row tiles: the multicast LM-head pass
])
def test_self_condition_matches_oracle(dgc, B, L, V, d, dsc, ystd, inv_tau):
    E = synth.normal_bf16((V, d), 0.1, 81)
    y = synth.normal_bf16((B * L, d), ystd, 82)
    W1 = synth.normal_bf16((dsc, d), 0.1, 83)
    W2 = synth.normal_bf16((d, dsc), 0.1, 84)
    e_gpu, s_gpu = _run_sc(dgc, y, E, W1, W2, B, L, inv_tau)
    _check_e(e_gpu, y, E, inv_tau)
    _check_ffw(s_gpu, e_gpu, W1, W2)
    _check_s_end_to_end(s_gpu, y, E, W1, W2, inv_tau)


@pytest.mark.parametrize("B", [1, 2])
def test_self_condition_window1k_sampled_rows(dgc, B):
    """window1k shapes at full size (vocabulary 262,144, d 2,048, d_sc 1,920: 7.9M feed-forward
    parameters) for one and two canvases, whose feed-forward GEMMs take different K splits
    (4-way over 30 or 32 k-blocks; 2- and 4-way); the oracle computes 8 sampled rows."""
    w = synth.WINDOW1K
    m = synth.make_model(w, DEV)
    W1 = synth.normal_bf16((1920, w.d), 0.02, 85)
    W2 = synth.normal_bf16((w.d, 1920), 0.02, 86)
    y = synth.normal_bf16((B * w.L, w.d), 0.5, 87)
    e_gpu, s_gpu = _run_sc(dgc, y, m["E"], W1, W2, B, w.L, 1.0)
    rows = np.sort(np.random.default_rng(3).choice(B * w.L, 8, replace=False))
    _check_e(e_gpu, y, m["E"].cpu(), 1.0, rows)
    _check_ffw(s_gpu[rows], e_gpu[rows], W1, W2)


def _sc_model(w, dsc, seed):
    """The workload's N(0, 0.02) decoder with N(0, 1) and N(0, 16) feed-forward layers: the
    near-uniform posteriors give e ~ the mean embedding row, and the signal comes out at ~5x
    the embeddings' scale, enough to move a few percent of the samples."""
    m = synth.make_model(w)
    m["Wsc1"] = synth.normal_bf16((dsc, w.d), 1.0, seed)
    m["Wsc2"] = synth.normal_bf16((w.d, dsc), 4.0, seed + 1)
    return m


def _oracle_model(m):
    om = {k: (f64(v) if torch.is_tensor(v) else v) for k, v in m.items()}
    return om


def _gpu_loop(dgc, w, m, kp, vp, canvas, cfg, lock=None, ws=None, sampler_eb=False):
    md = dgc.make_model(*(m[k].to(DEV) for k in ("E", "Wqkv", "Wo")), w.H, w.Hkv, w.hd,
                        *((m["Wsc1"].to(DEV), m["Wsc2"].to(DEV)) if "Wsc1" in m else ()))
    c = torch.tensor(canvas, dtype=torch.int32, device=DEV)
    lk = None if sampler_eb else torch.tensor(
        np.zeros((w.B, w.L), np.uint8) if lock is None else lock, device=DEV)
    st = torch.zeros(w.B, dtype=torch.int32, device=DEV)
    if ws is None:
        ws = dgc.workspace(dgc.dg_denoise_loop_workspace(md, w.B, w.L, w.P, w.window))
    dgc.dg_denoise_loop(md, kp.to(DEV), vp.to(DEV), w.window, c, lk, st, cfg, ws)
    dgc.dg_workspace_status(ws)
    return (c.cpu().numpy(), None if lk is None else lk.cpu().numpy(), st.cpu().numpy(), ws)


TINY_SC = dataclasses.replace(synth.TINY, B=2, L=128, P=192, d=256, H=4, Hkv=2, hd=64,
                              V=4096, T=6)


def test_loop_zero_second_layer_equals_plain_loop(dgc):
    """A zero second feed-forward layer makes every signal zero: the loop with
    self-conditioning is bit-identical to the loop without it."""
    w = TINY_SC
    m = _sc_model(w, 128, 91)
    m["Wsc2"] = torch.zeros_like(m["Wsc2"])
    plain = {k: v for k, v in m.items() if k not in ("Wsc1", "Wsc2")}
    kp, vp = synth.make_prefix_kv(w)
    x1 = O.initial_canvas(w.B, w.L, w.V, 4)
    cfg = dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 4)
    a = _gpu_loop(dgc, w, m, kp, vp, x1, cfg)
    b = _gpu_loop(dgc, w, plain, kp, vp, x1, cfg)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])


def test_loop_with_self_conditioning_matches_oracle_and_resumes(dgc):
    """Two steps (the second one sees the first one's signal) against the oracle up to Gumbel
    near-ties; the whole loop agrees on >= 99 % of the tokens and differs from the loop without
    the signal (on ~1.5 % of them); a run split at step 3 with the same workspace reproduces the whole run."""
    w = TINY_SC
    m = _sc_model(w, 128, 92)
    kp, vp = synth.make_prefix_kv(w)
    om = _oracle_model(m)
    okp, ovp = f64(kp), f64(vp)
    x1 = O.initial_canvas(w.B, w.L, w.V, 5)
    lock = np.zeros((w.B, w.L), np.uint8)
    g2 = _gpu_loop(dgc, w, m, kp, vp, x1, dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 5,
                                                       end_step=2))[0]
    st = {}
    r1, l1, _ = O.denoise_loop(om, okp, ovp, w.window, x1, lock, w.T, w.schedule, 1.0, math.inf,
                               5, end_step=1, state=st)
    _, jumps = O.schedule_thresholds(w.schedule, w.T)
    r2, _, _, _, post = O.denoise_step(om, okp, ovp, w.window, r1, l1, 1, int(jumps[1]), 1.0,
                                       math.inf, 5, st["s"])
    diff = (g2 != r2).reshape(-1)
    assert not np.any(diff & (post["gap_perturbed"] >= GUMBEL_TIE)), int(diff.sum())
    cfg = dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 5)
    full, _, steps, _ = _gpu_loop(dgc, w, m, kp, vp, x1, cfg)
    ref, _, _ = O.denoise_loop(om, okp, ovp, w.window, x1, lock, w.T, w.schedule, 1.0, math.inf,
                               5)
    assert (full == ref).mean() >= 0.99 and np.all(steps == w.T)
    plain = {k: v for k, v in m.items() if k not in ("Wsc1", "Wsc2")}
    assert (full != _gpu_loop(dgc, w, plain, kp, vp, x1, cfg)[0]).mean() > 0.005
    h, lh, _, ws = _gpu_loop(dgc, w, m, kp, vp, x1,
                             dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 5, end_step=3))
    b, _, _, _ = _gpu_loop(dgc, w, m, kp, vp, h, dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 5,
                                                              start_step=3), lock=lh, ws=ws)
    assert np.array_equal(b, full)


def _ulp_bf16(x):
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def test_entropy_bounded_loop_with_self_conditioning(dgc):
    """The entropy-bounded sampler with the signal fed back (near-uniform posteriors: nothing
    is accepted, every step re-noises, and the result is the top-1 of the last posterior).
    Steps taken equal the oracle's.  The signal the GPU feeds back is one bf16 rounding away
    from the oracle's (its expected embedding sums bf16 probabilities), which moves each
    coordinate of the last step's y by up to a few bf16 ulps; so where the top-1 tokens differ,
    the oracle's logit of the GPU's token must lie within inv_tau * sum_j 3 ulp(y_j)
    (|E_a,j| + |E_b,j|) of its best, and differences stay rare."""
    w = dataclasses.replace(TINY_SC, T=5)
    m = _sc_model(w, 64, 93)
    kp, vp = synth.make_prefix_kv(w)
    x1 = O.initial_canvas(w.B, w.L, w.V, 6)
    cfg = dgc.make_cfg(w.T, 0, seed=6, sampler=dgc.DG_SAMPLER_ENTROPY_BOUNDED)
    g, _, steps, _ = _gpu_loop(dgc, w, m, kp, vp, x1, cfg, sampler_eb=True)
    om, okp, ovp = _oracle_model(m), f64(kp), f64(vp)
    ref, rsteps = O.eb_denoise_loop(om, okp, ovp, w.window, x1, w.T, 0.8, 0.4, 0.1, 0.005, 6)
    assert np.array_equal(steps, rsteps) and np.all(rsteps == w.T)  # nothing stops early
    # the oracle's loop once more, by hand, keeping the input of the last step
    inv = O.eb_inv_tau(w.T, 0.8, 0.4)
    x, prev, sig = x1.copy(), None, None
    for n in range(w.T - 1):
        x, _, _, _, post = O.eb_denoise_step(om, okp, ovp, w.window, x, n, inv[n], prev, 6, 0.1,
                                             0.005, False, sig)
        prev, sig = post["top1"].reshape(w.B, w.L), post["s"]
    h, q, k, v = O.decoder_front(x, om["E"], om["Wqkv"], w.H, w.Hkv, w.hd, sig)
    Oa, _ = O.canvas_attention(q, okp, ovp, k, v, w.window, w.hd ** -0.5)
    y = O.decoder_back(h, Oa, om["Wo"]).reshape(w.B * w.L, w.d)
    z = y @ om["E"].T * inv[-1]
    top = np.argmax(z, axis=1)
    assert np.array_equal(top.reshape(w.B, w.L), ref)
    gf = g.reshape(-1)
    diff = np.nonzero(gf != top)[0]
    for r in diff:
        a, b = top[r], gf[r]
        tol = inv[-1] * np.sum(3 * _ulp_bf16(y[r]) * (np.abs(om["E"][a]) + np.abs(om["E"][b])))
        assert z[r, a] - z[r, b] <= tol, (r, z[r, a] - z[r, b], tol)
    assert len(diff) <= 0.03 * gf.size
