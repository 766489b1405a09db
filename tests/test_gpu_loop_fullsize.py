"""GPU parity of the denoising loop at full size (vocabulary 262,144, d_model 2,048, 16q/8kv x
128) against the oracle's own trajectory, through the C ABI.

  * window1k: all 12 cosine steps in one dg_denoise_loop call (each step's finalisation runs
    inside the next step's embedding launch; lambda_n < 1 jump decisions until the last step).
  * four canvases with planted confident positions: locks at theta = 0.95 fire inside the
    loop, and a canvas whose positions all lock stops (stop-when-all-locked).
  * two canvases with an 8,192-token global prefix (the batch16 dimensions), one step.

Decisions are bit-exact except at the oracle's near-ties (two best perturbed scores within
1e-3 at a position that jumps; top-1 log-probability within 2e-3 of log(theta)).  A canvas
with no near-tie along the oracle's trajectory must come out identical; every step is also
replayed on the GPU from the oracle's own state, and the one-call run must equal the same steps
run one call at a time.
"""

import math

import numpy as np
import pytest
import torch

from discrete_diffusion_text_gb300 import synth
from oracle import dgoracle as O

from loop_reference import trajectory

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def dgc():
    import os

    from discrete_diffusion_text_gb300 import dgcanvas

    if not os.path.exists(dgcanvas.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build()
    dgcanvas.load()
    return dgcanvas


class Side:
    """The same model and prefix on both sides: drawn on the host, copied to the device."""

    def __init__(self, dgc, w, B):
        m = synth.make_model(w)
        kp, vp = synth.make_prefix_kv(w, B=B)
        self.om = {"E": m["E"].double().numpy(), "Wqkv": m["Wqkv"].double().numpy(),
                   "Wo": m["Wo"].double().numpy(), "H": w.H, "Hkv": w.Hkv, "hd": w.hd}
        self.okp, self.ovp = kp.double().numpy(), vp.double().numpy()
        self.E = m["E"]
        self.dE, self.dWqkv, self.dWo = m["E"].to(DEV), m["Wqkv"].to(DEV), m["Wo"].to(DEV)
        self.kp, self.vp = kp.to(DEV), vp.to(DEV)
        self.model = dgc.make_model(self.dE, self.dWqkv, self.dWo, w.H, w.Hkv, w.hd)
        self.ws = dgc.workspace(dgc.dg_denoise_loop_workspace(self.model, B, w.L, w.P, w.window))
        self.w, self.B, self.dgc = w, B, dgc

    def run(self, x, lock, cfg):
        c = torch.tensor(x, dtype=torch.int32, device=DEV)
        lk = torch.tensor(lock, dtype=torch.uint8, device=DEV)
        st = torch.zeros(self.B, dtype=torch.int32, device=DEV)
        self.dgc.dg_denoise_loop(self.model, self.kp, self.vp, self.w.window, c, lk, st, cfg,
                                 self.ws)
        self.dgc.dg_workspace_status(self.ws)
        return c.cpu().numpy().astype(np.int64), lk.cpu().numpy(), st.cpu().numpy()


def _check_loop(dgc, side, x0, lock0, T, schedule, inv_tau, lock_logthr, seed, stop):
    """Oracle trajectory vs (a) one GPU call over all steps, (b) the GPU one step at a time from
    the oracle's states, (c) the GPU one step at a time from its own states.  Returns the
    number of near-tie positions met along the trajectory and the number of positions that
    differ in (a)."""
    B, L = x0.shape
    states, ties = trajectory(side.om, side.okp, side.ovp, side.w.window, x0, lock0, T, schedule,
                              inv_tau, lock_logthr, seed, stop_when_all_locked=stop)

    def cfg(start=0, end=0):
        return dgc.make_cfg(T, schedule, inv_tau, lock_logthr, seed, start_step=start,
                            end_step=end, stop_when_all_locked=stop)

    # (b) each step from the oracle's own state: only near-ties of that step may differ
    for n in range(T):
        xs, ls, _, _ = states[n]
        gx, gl, _ = side.run(xs, ls, cfg(n, n + 1))
        rx, rl, _, _ = states[n + 1]
        diff = (gx != rx) | (gl != rl)
        assert not np.any(diff & ~ties[n]), f"step {n}: {int(diff.sum())} positions differ"
    # (a) the whole run in one call
    fx, fl, fs = side.run(x0, lock0, cfg())
    rx, rl, _, rs = states[-1]
    tie_any = np.zeros((B, L), bool)
    for t in ties:
        tie_any |= t
    clean = ~tie_any.any(axis=1)  # canvases with no near-tie anywhere along the trajectory
    assert np.array_equal(fx[clean], rx[clean]) and np.array_equal(fl[clean], rl[clean])
    assert np.array_equal(fs[clean], rs[clean])
    differ = int(((fx != rx) | (fl != rl)).sum())
    assert differ <= max(2, int(0.02 * B * L)), differ
    # (c) the one-call run equals the same steps run one call at a time on the GPU
    x, lk = x0, lock0
    steps = np.zeros(B, np.int64)
    for n in range(T):
        x, lk, st = side.run(x, lk, cfg(n, n + 1))
        steps += st
    assert np.array_equal(x, fx) and np.array_equal(lk, fl) and np.array_equal(steps, fs)
    return int(tie_any.sum()), differ


def test_loop_window1k_twelve_cosine_steps_in_one_call(dgc):
    """window1k at full size: seed 1 (the workload's), whose oracle trajectory has no near-tie,
    so the 12-step one-call run must equal the oracle's canvas exactly."""
    w = synth.WINDOW1K
    side = Side(dgc, w, 1)
    x0 = O.initial_canvas(1, w.L, w.V, w.seed)
    lock0 = np.zeros((1, w.L), np.uint8)
    ties, differ = _check_loop(dgc, side, x0, lock0, w.T, w.schedule, 1.0, math.inf, w.seed,
                               False)
    assert ties == 0 and differ == 0


def test_loop_planted_locks_four_canvases(dgc):
    """Four canvases at the window1k dimensions, 4 linear steps, inverse temperature 20 and
    locking at theta = 0.95 with stop-when-all-locked.  The stand-in decoder's residual keeps a
    token's own logit at |E_x|^2, so the tokens with the largest embedding norms are confident:
    canvas 0 holds the 256 largest (every position locks at step 0 and the canvas stops after
    one step), canvas 1 alternates the largest and the smallest, canvas 2 is the uniform prior,
    canvas 3 holds the 256 smallest (confidence ~0.9: no lock at step 0)."""
    import dataclasses

    w = dataclasses.replace(synth.WINDOW1K, B=4)
    side = Side(dgc, w, 4)
    norms = (side.E.double() ** 2).sum(1).numpy()
    order = np.argsort(-norms, kind="stable")
    top, bot = order[:w.L], order[-w.L:]
    x0 = O.initial_canvas(4, w.L, w.V, 11)
    x0[0] = top
    x0[1, ::2], x0[1, 1::2] = top[:w.L // 2], bot[:w.L // 2]
    x0[3] = bot
    lock0 = np.zeros((4, w.L), np.uint8)
    thr = float(np.float32(math.log(0.95)))
    T = 4
    _check_loop(dgc, side, x0, lock0, T, synth.SCHED_LINEAR, 20.0, thr, 11, True)
    fx, fl, fs = side.run(x0, lock0, dgc.make_cfg(T, synth.SCHED_LINEAR, 20.0, thr, 11,
                                                  stop_when_all_locked=True))
    assert fl[0].all() and fs[0] == 1 and np.array_equal(fx[0], x0[0])  # locked to its top-1
    assert 0.3 < fl[1].mean() < 0.8 and fs[1] == T
    assert fl[2].mean() > 0.5 and not fl[2].all()
    assert fl[3].mean() < 0.5 and fs[3] == T


def test_loop_step_prefix_8192_two_canvases(dgc):
    """The batch16 dimensions (8,192-token global prefix, lock at 0.9) with two canvases: the
    loop's last step (lambda = 1) from the uniform prior; the oracle recomputes the decoder for
    both canvases and the posterior for 16 sampled positions of each."""
    import dataclasses

    w = dataclasses.replace(synth.BATCH16, B=2)
    side = Side(dgc, w, 2)
    x0 = O.initial_canvas(2, w.L, w.V, w.seed)
    lock0 = np.zeros((2, w.L), np.uint8)
    thr = float(np.float32(math.log(w.lock_theta)))
    n = w.T - 1
    gx, gl, st = side.run(x0, lock0, dgc.make_cfg(w.T, w.schedule, 1.0, thr, w.seed,
                                                  start_step=n, end_step=n + 1))
    assert np.all(st == 1) and not gl.any()  # near-uniform posteriors never reach 0.9
    om = side.om
    h, q, k, v = O.decoder_front(x0, om["E"], om["Wqkv"], w.H, w.Hkv, w.hd)
    Oa, _ = O.canvas_attention(q, side.okp, side.ovp, k, v, w.window, w.hd ** -0.5)
    y = O.decoder_back(h, Oa, om["Wo"]).reshape(2 * w.L, w.d)
    rng = np.random.default_rng(8)
    rows = np.sort(np.concatenate([rng.choice(w.L, 16, replace=False),
                                   w.L + rng.choice(w.L, 16, replace=False)]))
    post = O.posterior(y, om["E"], 1.0, w.seed, n, w.L, rows=rows)
    diff = gx.reshape(-1)[rows] != post["x0hat"]
    assert not np.any(diff & (post["gap_perturbed"] >= 1e-3)), int(diff.sum())


def test_loop_step_eight_canvases_multicast_lm_head(dgc):
    """The window1k dimensions with eight canvases (16 row tiles: the LM head runs as two-CTA
    clusters sharing each weight k-block by multicast): the loop's last step from the uniform
    prior; the oracle recomputes the decoder and the posterior of 4 positions per canvas."""
    import dataclasses

    w = dataclasses.replace(synth.WINDOW1K, B=8)
    side = Side(dgc, w, 8)
    x0 = O.initial_canvas(8, w.L, w.V, 21)
    lock0 = np.zeros((8, w.L), np.uint8)
    n = w.T - 1
    gx, gl, st = side.run(x0, lock0, dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 21,
                                                  start_step=n, end_step=n + 1))
    assert np.all(st == 1)
    om = side.om
    h, q, k, v = O.decoder_front(x0, om["E"], om["Wqkv"], w.H, w.Hkv, w.hd)
    Oa, _ = O.canvas_attention(q, side.okp, side.ovp, k, v, w.window, w.hd ** -0.5)
    y = O.decoder_back(h, Oa, om["Wo"]).reshape(8 * w.L, w.d)
    rng = np.random.default_rng(9)
    rows = np.sort(np.concatenate([b * w.L + rng.choice(w.L, 4, replace=False)
                                   for b in range(8)]))
    post = O.posterior(y, om["E"], 1.0, 21, n, w.L, rows=rows)
    diff = gx.reshape(-1)[rows] != post["x0hat"]
    assert not np.any(diff & (post["gap_perturbed"] >= 1e-3)), int(diff.sum())
