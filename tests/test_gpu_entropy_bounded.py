"""GPU parity of the entropy-bounded sampler (entropy in the fused posterior, the update
kernel, and the loop) against the CPU oracle.  Every call goes through the C ABI."""

import math

import numpy as np
import pytest
import torch

from discrete_diffusion_text_gb300 import synth
from oracle import dgoracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"
ENT_TOL = 1e-3       # absolute, on entropies of O(1)-O(10) nats computed in fp32 online
GUMBEL_TIE = 1e-3
LOGIT_TIE = 1e-4


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


def _i32(a):
    return torch.tensor(np.asarray(a), dtype=torch.int32, device=DEV)


def _eb_inputs(B, L, V, seed):
    """Entropies with exact zeros, repeated values (ordering ties), a few tiny canvases (mean
    below the stop threshold) and large values; top-1 equal to the previous prediction on some
    canvases."""
    rng = np.random.default_rng(seed)
    H = rng.exponential(0.02, size=(B, L)).astype(np.float32)
    H[rng.random((B, L)) < 0.15] = 0.0
    H[rng.random((B, L)) < 0.1] = np.float32(0.0125)
    H[:, : L // 8] = rng.exponential(3.0, size=(B, L // 8)).astype(np.float32)
    H[::4] = (rng.random((len(H[::4]), L)) * 1e-3).astype(np.float32)
    x0hat = rng.integers(0, V, size=(B, L))
    top1 = rng.integers(0, V, size=(B, L))
    prev = top1.copy()
    prev[1::3, 0] = (prev[1::3, 0] + 1) % V
    return x0hat, top1, H, prev


@pytest.mark.parametrize("B,L,V", [(16, 256, 262144), (5, 100, 1000), (3, 1024, 4096), (2, 1, 7)])
@pytest.mark.parametrize("mode", ["prev", "no_prev", "final"])
def test_entropy_bounded_update_bit_exact(dgc, B, L, V, mode):
    x0hat, top1, H, prev = _eb_inputs(B, L, V, 100 + L)
    gamma, stop = 0.1, 0.005
    x_out = torch.empty((B, L), dtype=torch.int32, device=DEV)
    accept = torch.empty((B, L), dtype=torch.uint8, device=DEV)
    done = torch.empty(B, dtype=torch.uint8, device=DEV)
    mean = torch.empty(B, dtype=torch.float32, device=DEV)
    g_prev = _i32(prev)
    dgc.dg_entropy_bounded_update(_i32(x0hat), _i32(top1), torch.tensor(H, device=DEV), x_out,
                                  seed=77, step=9, V=V, gamma=gamma, stop_entropy=stop,
                                  prev_top1=g_prev, prev_valid=mode == "prev", accept=accept,
                                  done=done, mean_entropy=mean, final_step=mode == "final")
    torch.cuda.synchronize()
    rx, racc, rdone, rmean = O.entropy_bounded_update(
        x0hat, top1, H, prev if mode == "prev" else None, 77, 9, V, gamma, stop,
        final_step=mode == "final")
    assert np.array_equal(x_out.cpu().numpy(), rx)
    assert np.array_equal(accept.cpu().numpy(), racc)
    assert np.array_equal(done.cpu().numpy(), rdone)
    assert np.array_equal(mean.cpu().numpy(), rmean)
    assert np.array_equal(g_prev.cpu().numpy(), top1)  # overwritten for the next step
    if L >= 8:  # the inputs exercise both outcomes (L = 1 is the degenerate case)
        if mode == "prev":
            assert rdone.any() and not rdone.all()
        assert racc.any() and not racc.all()


def _posterior_with_entropy(dgc, y, E, B, L, inv_tau, seed, step):
    R = B * L
    out = {k: torch.empty(R, dtype=torch.int32 if k in ("x0hat", "top1") else torch.float32,
                          device=DEV) for k in ("x0hat", "top1", "lse", "entropy")}
    ws = dgc.workspace(dgc.dg_vocab_posterior_workspace(B, L, E.shape[0]))
    dgc.dg_vocab_posterior_step(y.to(DEV), E, B, L, inv_tau, seed, step, out=out, ws=ws)
    dgc.dg_workspace_status(ws)
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("B,L,V,d,ystd,inv_tau", [
    (1, 256, 4096, 256, 0.05, 1.25),    # near-uniform: entropy ~ log V
    (3, 192, 4096, 256, 1.0, 50.0),     # sharp posteriors: entropy ~ 0
    (2, 128, 8192, 512, 0.5, 2.5),      # in between
    (16, 256, 4096, 256, 0.5, 2.5),     # 32 row tiles: the multicast LM-head pass
])
def test_posterior_entropy_matches_oracle(dgc, B, L, V, d, ystd, inv_tau):
    E = synth.normal_bf16((V, d), 0.02 if ystd < 0.5 else 0.1, 51).to(DEV)
    y = synth.normal_bf16((B * L, d), ystd, 52)
    got = _posterior_with_entropy(dgc, y, E, B, L, inv_tau, 99, 2)
    ref = O.posterior(f64(y), f64(E), inv_tau, 99, 2, L)
    err = np.abs(got["entropy"] - ref["entropy"])
    assert err.max() <= ENT_TOL + 1e-4 * ref["entropy"].max(), err.max()
    assert np.all(got["entropy"] >= 0.0)


def test_posterior_entropy_window1k_sampled_rows(dgc):
    w = synth.WINDOW1K
    E = synth.make_model(w, DEV)["E"]
    y = synth.normal_bf16((w.L, w.d), 0.05, 53)
    got = _posterior_with_entropy(dgc, y, E, 1, w.L, 1.25, w.seed, 0)
    rows = np.sort(np.random.default_rng(2).choice(w.L, 16, replace=False))
    ref = O.posterior(f64(y), f64(E), 1.25, w.seed, 0, w.L, rows=rows)
    assert np.abs(got["entropy"][rows] - ref["entropy"]).max() <= ENT_TOL


def test_entropy_bounded_decisions_on_gpu_posteriors(dgc):
    """The fused chain: GPU entropies (and samples) feed the update; decisions equal the
    oracle's except where the oracle's own margin is within the entropy tolerance."""
    B, L, V, d = 4, 256, 4096, 256
    rng = np.random.default_rng(8)
    # rows of very different sharpness: some positions get entropies far below gamma
    E = synth.normal_bf16((V, d), 0.1, 54).to(DEV)
    scale = torch.tensor(np.where(rng.random(B * L) < 0.5, 3.0, 0.05), dtype=torch.float32)
    y = (synth.normal_bf16((B * L, d), 1.0, 55).float() * scale[:, None]).to(torch.bfloat16)
    got = _posterior_with_entropy(dgc, y, E, B, L, 2.5, 5, 4)
    ref = O.posterior(f64(y), f64(E), 2.5, 5, 4, L)
    shape = (B, L)
    gx = torch.empty(shape, dtype=torch.int32, device=DEV)
    gacc = torch.empty(shape, dtype=torch.uint8, device=DEV)
    dgc.dg_entropy_bounded_update(_i32(got["x0hat"].reshape(shape)),
                                  _i32(got["top1"].reshape(shape)),
                                  torch.tensor(got["entropy"].reshape(shape), device=DEV), gx,
                                  seed=5, step=4, V=V, gamma=0.1, stop_entropy=0.005,
                                  prev_top1=None, prev_valid=False, accept=gacc)
    torch.cuda.synchronize()
    H = ref["entropy"].reshape(shape).astype(np.float32)
    _, racc, _, _ = O.entropy_bounded_update(ref["x0hat"].reshape(shape),
                                             ref["top1"].reshape(shape), H, None, 5, 4, V, 0.1,
                                             0.005)
    gacc = gacc.cpu().numpy()
    assert racc.sum() > 0 and racc.sum() < racc.size
    for b in range(B):
        order = np.lexsort((np.arange(L), H[b]))
        cum = np.cumsum(H[b][order].astype(np.float64))
        k_ref, k_gpu = int(racc[b].sum()), int(gacc[b].sum())
        if k_ref != k_gpu:  # only allowed when the running sum passes gamma within tolerance
            lo, hi = min(k_ref, k_gpu), max(k_ref, k_gpu)
            assert np.all(np.abs(cum[lo:hi] - 0.1) <= ENT_TOL * hi), (b, k_ref, k_gpu)
        diff = np.nonzero(racc[b] != gacc[b])[0]
        for i in diff:  # a position on the acceptance boundary of a near-tie in entropy
            kth = H[b][order[min(k_ref, k_gpu) - 1]] if min(k_ref, k_gpu) > 0 else 0.0
            assert abs(H[b, i] - kth) <= 2 * ENT_TOL or k_ref != k_gpu, (b, i)


def _gpu_eb_loop(dgc, w, m, kp, vp, canvas, cfg):
    md = dgc.make_model(m["E"].to(DEV), m["Wqkv"].to(DEV), m["Wo"].to(DEV), w.H, w.Hkv, w.hd)
    c = _i32(canvas)
    st = torch.zeros(w.B, dtype=torch.int32, device=DEV)
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(md, w.B, w.L, w.P, w.window))
    dgc.dg_denoise_loop(md, kp.to(DEV), vp.to(DEV), w.window, c, None, st, cfg, ws)
    dgc.dg_workspace_status(ws)
    return c.cpu().numpy(), st.cpu().numpy()


def _peaked_model(V, d, H, Hkv, hd, scale, seed):
    g = torch.Generator().manual_seed(seed)
    E = torch.randn((V, d), generator=g, dtype=torch.float64)
    E = (E / E.norm(dim=1, keepdim=True) * scale).to(torch.bfloat16)
    Wqkv = (torch.randn(((H + 2 * Hkv) * hd, d), generator=g) * 0.02).to(torch.bfloat16)
    Wo = (torch.randn((d, H * hd), generator=g) * 0.02).to(torch.bfloat16)
    return {"E": E, "Wqkv": Wqkv, "Wo": Wo, "H": H, "Hkv": Hkv, "hd": hd}


def test_entropy_bounded_loop_fixed_point(dgc):
    """Concentrated posteriors at the tokens already there: every canvas stops after two steps
    and returns its initial tokens, as the oracle does."""
    import dataclasses

    w = dataclasses.replace(synth.TINY, B=3, L=64, P=64, d=128, H=2, Hkv=2, hd=64, V=512, T=48)
    m = _peaked_model(w.V, w.d, w.H, w.Hkv, w.hd, 20.0, 3)
    kp = synth.normal_bf16((w.B, w.P, w.Hkv, w.hd), 1.0, 71)
    vp = synth.normal_bf16((w.B, w.P, w.Hkv, w.hd), 1.0, 72)
    x = O.initial_canvas(w.B, w.L, w.V, 9)
    cfg = dgc.make_cfg(w.T, 0, seed=9, sampler=dgc.DG_SAMPLER_ENTROPY_BOUNDED)
    gx, st = _gpu_eb_loop(dgc, w, m, kp, vp, x, cfg)
    om = {"E": f64(m["E"]), "Wqkv": f64(m["Wqkv"]), "Wo": f64(m["Wo"]), "H": w.H, "Hkv": w.Hkv,
          "hd": w.hd}
    rx, rst = O.eb_denoise_loop(om, f64(kp), f64(vp), 0, x, w.T, 0.8, 0.4, 0.1, 0.005, 9)
    assert st.tolist() == rst.tolist() == [2, 2, 2]
    assert np.array_equal(gx, rx) and np.array_equal(gx, x)


def test_entropy_bounded_loop_uninformed_runs_to_the_cap(dgc):
    """tiny workload (near-uniform posteriors): nothing accepted, every step re-noises, T steps;
    the returned top-1 sequence matches the oracle's up to logit near-ties."""
    import dataclasses

    w = dataclasses.replace(synth.TINY, T=6)
    m = synth.make_model(w)
    kp, vp = synth.make_prefix_kv(w)
    x = O.initial_canvas(w.B, w.L, w.V, w.seed)
    cfg = dgc.make_cfg(w.T, 0, seed=w.seed, sampler=dgc.DG_SAMPLER_ENTROPY_BOUNDED)
    gx, st = _gpu_eb_loop(dgc, w, m, kp, vp, x, cfg)
    assert st.tolist() == [w.T] * w.B
    om = {"E": f64(m["E"]), "Wqkv": f64(m["Wqkv"]), "Wo": f64(m["Wo"]), "H": w.H, "Hkv": w.Hkv,
          "hd": w.hd}
    # the state before the last step is the re-noise of step T-2; the last step returns top-1
    xs = O.renoise_tokens(w.B, w.L, w.V, w.seed, w.T - 2)
    inv = O.eb_inv_tau(w.T, 0.8, 0.4)
    _, _, _, _, post = O.eb_denoise_step(om, f64(kp), f64(vp), w.window, xs, w.T - 1, inv[-1],
                                         None, w.seed, 0.1, 0.005, True)
    ref = post["top1"].reshape(w.B, w.L)
    diff = (gx != ref).reshape(-1)
    assert not np.any(diff & (post["gap_logit"] >= LOGIT_TIE)), int(diff.sum())
