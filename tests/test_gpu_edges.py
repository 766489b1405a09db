"""Empty and degenerate calls on the GPU, through the C ABI: zero canvases, zero steps, a single
step, the smallest vocabulary (one 256-entry tile) and the shortest canvas (64 positions)."""

import dataclasses
import math

import numpy as np
import pytest
import torch

from discrete_diffusion_text_gb300 import synth
from oracle import dgoracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"
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


def _model(w):
    m = synth.make_model(w)
    om = {k: (f64(v) if torch.is_tensor(v) else v) for k, v in m.items()}
    return m, om


def test_zero_canvases_are_no_ops(dgc):
    """B = 0 everywhere: DG_OK, nothing launched, nothing written."""
    w = dataclasses.replace(synth.TINY, B=0)
    m, _ = _model(w)
    md = dgc.make_model(*(m[k].to(DEV) for k in ("E", "Wqkv", "Wo")), w.H, w.Hkv, w.hd)
    empty = torch.empty((0, w.L), dtype=torch.int32, device=DEV)
    dgc.dg_forward_noise(empty, empty, torch.empty(0, dtype=torch.int64, device=DEV), w.V, 1)
    kp = torch.empty((0, w.P, w.Hkv, w.hd), dtype=torch.bfloat16, device=DEV)
    ws = dgc.workspace(256)
    dgc.dg_denoise_loop(md, kp, kp, w.window, empty, torch.empty((0, w.L), dtype=torch.uint8,
                                                                 device=DEV),
                        torch.empty(0, dtype=torch.int32, device=DEV),
                        dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 1), ws)
    dgc.dg_workspace_status(ws)


def test_zero_steps_leave_the_canvas(dgc):
    """start_step == end_step: the canvas and locks are unchanged and no step is counted."""
    w = synth.TINY
    m, _ = _model(w)
    kp, vp = synth.make_prefix_kv(w)
    md = dgc.make_model(*(m[k].to(DEV) for k in ("E", "Wqkv", "Wo")), w.H, w.Hkv, w.hd)
    x1 = O.initial_canvas(w.B, w.L, w.V, 4)
    c = torch.tensor(x1, dtype=torch.int32, device=DEV)
    lk = torch.zeros((w.B, w.L), dtype=torch.uint8, device=DEV)
    st = torch.full((w.B,), 9, dtype=torch.int32, device=DEV)
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(md, w.B, w.L, w.P, w.window))
    dgc.dg_denoise_loop(md, kp.to(DEV), vp.to(DEV), w.window, c, lk, st,
                        dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 4, start_step=5,
                                     end_step=5), ws)
    dgc.dg_workspace_status(ws)
    assert np.array_equal(c.cpu().numpy(), x1) and not lk.cpu().numpy().any()
    assert st.cpu().tolist() == [0] * w.B


@pytest.mark.parametrize("V,L", [(256, 256), (4096, 64)])
def test_single_step_loop_small_shapes(dgc, V, L):
    """T = 1 (one step with lambda = 1: every position takes its sample), with the smallest
    vocabulary (a single 256-entry tile) or the shortest canvas (64 positions): equal to the
    oracle except at near-ties of the sample."""
    w = dataclasses.replace(synth.TINY, B=3, L=L, V=V, T=1)
    m, om = _model(w)
    kp, vp = synth.make_prefix_kv(w)
    md = dgc.make_model(*(m[k].to(DEV) for k in ("E", "Wqkv", "Wo")), w.H, w.Hkv, w.hd)
    x1 = O.initial_canvas(w.B, w.L, w.V, 6)
    c = torch.tensor(x1, dtype=torch.int32, device=DEV)
    lk = torch.zeros((w.B, w.L), dtype=torch.uint8, device=DEV)
    st = torch.zeros(w.B, dtype=torch.int32, device=DEV)
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(md, w.B, w.L, w.P, w.window))
    dgc.dg_denoise_loop(md, kp.to(DEV), vp.to(DEV), w.window, c, lk, st,
                        dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 6), ws)
    dgc.dg_workspace_status(ws)
    _, jumps = O.schedule_thresholds(w.schedule, w.T)
    assert int(jumps[0]) == 1 << 32
    rx, _, _, _, post = O.denoise_step(om, f64(kp), f64(vp), w.window, x1,
                                       np.zeros((w.B, w.L), np.uint8), 0, int(jumps[0]), 1.0,
                                       math.inf, 6)
    diff = (c.cpu().numpy() != rx).reshape(-1)
    assert not np.any(diff & (post["gap_perturbed"] >= GUMBEL_TIE)), int(diff.sum())
    assert st.cpu().tolist() == [1] * w.B


def test_block_generate_zero_blocks(dgc):
    """NB = 0: DG_OK; the outputs and the cache are not touched."""
    w = synth.TINY
    m, _ = _model(w)
    md = dgc.make_model(*(m[k].to(DEV) for k in ("E", "Wqkv", "Wo")), w.H, w.Hkv, w.hd)
    kc = torch.ones((w.B, w.P, w.Hkv, w.hd), dtype=torch.bfloat16, device=DEV)
    vc = torch.ones_like(kc)
    out = torch.zeros((w.B, 0, w.L), dtype=torch.int32, device=DEV)
    blocks, n_tok, steps = (torch.full((w.B,), 5, dtype=torch.int32, device=DEV)
                            for _ in range(3))
    ws = dgc.workspace(256)
    dgc.dg_block_generate(md, kc, vc, w.P, w.L, w.window, -1,
                          dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 1), out, blocks, n_tok,
                          steps, ws)
    torch.cuda.synchronize()
    assert blocks.cpu().tolist() == n_tok.cpu().tolist() == steps.cpu().tolist() == [5] * w.B
    assert bool((kc == 1).all()) and bool((vc == 1).all())
