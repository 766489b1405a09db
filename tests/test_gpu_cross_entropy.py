"""GPU parity of the fused SFT cross-entropy (LM head + log-sum-exp + target logit in one pass)
and of the SFT loss on noised canvases, against the CPU oracle, through the C ABI."""

import dataclasses

import numpy as np
import pytest
import torch

from discrete_diffusion_text_gb300 import synth
from oracle import dgoracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"
LOSS_TOL = 2e-3  # the log-probability bar of the posterior tests


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


@pytest.mark.parametrize("B,L,V,d,ystd,inv_tau", [
    (1, 256, 4096, 256, 0.05, 1.0),     # near-uniform: loss ~ log V
    (3, 192, 4096, 256, 1.0, 20.0),     # ragged row tile, sharp posteriors
    (2, 128, 8192, 512, 0.5, 2.0),
    (16, 256, 4096, 256, 0.3, 1.0),
])
def test_cross_entropy_matches_oracle(dgc, B, L, V, d, ystd, inv_tau):
    R = B * L
    E = synth.normal_bf16((V, d), 0.1, 81).to(DEV)
    y = synth.normal_bf16((R, d), ystd, 82)
    rng = np.random.default_rng(83)
    tgt = rng.integers(0, V, R)
    # make some targets the row's argmax so that small losses are covered too
    z = f64(y) @ f64(E).T
    tgt[::3] = np.argmax(z[::3], axis=1)
    loss = torch.empty(R, dtype=torch.float32, device=DEV)
    lse = torch.empty(R, dtype=torch.float32, device=DEV)
    ws = dgc.workspace(dgc.dg_vocab_posterior_workspace(B, L, V))
    dgc.dg_cross_entropy_step(y.to(DEV), E, B, L, inv_tau, torch.tensor(tgt, dtype=torch.int32,
                                                                        device=DEV), loss, lse, ws)
    dgc.dg_workspace_status(ws)
    ref, rlse = O.cross_entropy(f64(y), f64(E), inv_tau, tgt)
    assert np.abs(loss.cpu().numpy() - ref).max() <= LOSS_TOL
    assert np.abs(lse.cpu().numpy() - rlse).max() <= LOSS_TOL


def test_cross_entropy_full_vocabulary_sampled_rows(dgc):
    w = synth.WINDOW1K
    E = synth.make_model(w, DEV)["E"]
    y = synth.normal_bf16((w.L, w.d), 0.05, 84)
    tgt = np.random.default_rng(85).integers(0, w.V, w.L)
    loss = torch.empty(w.L, dtype=torch.float32, device=DEV)
    ws = dgc.workspace(dgc.dg_vocab_posterior_workspace(1, w.L, w.V))
    dgc.dg_cross_entropy_step(y.to(DEV), E, 1, w.L, 1.0, torch.tensor(tgt, dtype=torch.int32,
                                                                      device=DEV), loss, None, ws)
    dgc.dg_workspace_status(ws)
    rows = np.sort(np.random.default_rng(3).choice(w.L, 16, replace=False))
    ref, _ = O.cross_entropy(f64(y)[rows], f64(E), 1.0, tgt[rows])
    assert np.abs(loss.cpu().numpy()[rows] - ref).max() <= LOSS_TOL


def test_sft_loss_on_noised_canvases_matches_oracle(dgc):
    """Zipf(1.1) clean canvases noised at per-canvas t (keep thresholds from t), the stand-in
    decoder over them with the prefix KV, and the cross-entropy against x_0."""
    w = dataclasses.replace(synth.TINY, B=4)
    m = synth.make_model(w)
    kp, vp = synth.make_prefix_kv(w)
    x0 = synth.zipf_tokens(w.B, w.L, w.V, 1.1, 86)
    t = synth.uniform_times(w.B, 87)
    keep = O.keep_threshold_from_t(O.SCHED_LINEAR, t)
    md = dgc.make_model(m["E"].to(DEV), m["Wqkv"].to(DEV), m["Wo"].to(DEV), w.H, w.Hkv, w.hd)
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(md, w.B, w.L, w.P, w.window))
    x0d = torch.tensor(x0, dtype=torch.int32, device=DEV)
    xt = torch.empty_like(x0d)
    loss = torch.empty((w.B, w.L), dtype=torch.float32, device=DEV)
    keep_d = torch.tensor(keep.astype(np.int64), device=DEV)
    dgc.dg_sft_loss(md, kp.to(DEV), vp.to(DEV), w.window, x0d, keep_d, 91, xt, loss, 1.0, ws)
    dgc.dg_workspace_status(ws)
    om = {"E": f64(m["E"]), "Wqkv": f64(m["Wqkv"]), "Wo": f64(m["Wo"]), "H": w.H, "Hkv": w.Hkv,
          "hd": w.hd}
    ref, rxt = O.sft_loss(om, f64(kp), f64(vp), w.window, x0, keep, 91)
    assert np.array_equal(xt.cpu().numpy(), rxt)
    assert np.abs(loss.cpu().numpy() - ref).max() <= LOSS_TOL


@pytest.mark.parametrize("B,L", [(1, 256), (2, 256), (1, 192)])
def test_sft_loss_window1k_sampled_rows(dgc, B, L):
    """SFT loss at the window1k dims (d_model 2,048, 16q/8kv x 128, vocabulary 262,144, prefix
    1,024 in a 1,024 window) for one and two canvases and a 192-position canvas (a ragged last
    row tile), whose projections run as cluster split-K (QKV 4- or 2-way, the output projection
    4-way at 128 or 256 columns): noising bit-exact for every canvas; the oracle recomputes the
    decoder for every canvas and the loss at 16 sampled positions.  With the tied head a kept position's loss is
    lse - 2 y.E[x_t] at 1/tau = 2: a projection that dropped a quarter of its K range would move
    it by ~1e-2, while the attention's bf16 probabilities in P.V move y.E[x_t] by ~3e-4 (so
    1/tau = 20 would put legitimate rounding at the tolerance)."""
    w = dataclasses.replace(synth.WINDOW1K, B=B, L=L)
    m = synth.make_model(w, DEV)
    kp, vp = synth.make_prefix_kv(w, DEV)
    x0 = synth.zipf_tokens(w.B, w.L, w.V, 1.1, 96)
    keep = O.keep_threshold_from_t(O.SCHED_LINEAR, synth.uniform_times(w.B, 97))
    md = dgc.make_model(m["E"], m["Wqkv"], m["Wo"], w.H, w.Hkv, w.hd)
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(md, w.B, w.L, w.P, w.window))
    x0d = torch.tensor(x0, dtype=torch.int32, device=DEV)
    xt = torch.empty_like(x0d)
    loss = torch.empty((w.B, w.L), dtype=torch.float32, device=DEV)
    keep_d = torch.tensor(keep.astype(np.int64), device=DEV)
    dgc.dg_sft_loss(md, kp, vp, w.window, x0d, keep_d, 98, xt, loss, 2.0, ws)
    dgc.dg_workspace_status(ws)
    E = f64(m["E"])
    rxt = O.forward_noise(x0, keep, w.V, 98)
    assert np.array_equal(xt.cpu().numpy(), rxt)
    h, q, kc, vc = O.decoder_front(rxt, E, f64(m["Wqkv"]), w.H, w.Hkv, w.hd)
    Oa, _ = O.canvas_attention(q, f64(kp), f64(vp), kc, vc, w.window, w.hd ** -0.5)
    y = O.decoder_back(h, Oa, f64(m["Wo"])).reshape(w.B * w.L, w.d)
    rows = np.sort(np.random.default_rng(99).choice(w.B * w.L, 16, replace=False))
    ref, _ = O.cross_entropy(y[rows], E, 2.0, x0.reshape(-1)[rows])
    got = loss.cpu().numpy().reshape(-1)[rows]
    assert np.std(ref) > 0.05  # the loss varies from row to row
    assert np.abs(got - ref).max() <= LOSS_TOL
