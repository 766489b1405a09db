"""Failure reporting of libdgcanvas on the GPU, made without faulting the GPU.

  * An out-of-range token id where an embedding row is gathered: the kernel uses a zero row
    (no out-of-bounds read) and the status word reports DG_EKERNEL.
  * A bounded on-chip wait that runs out: with a 1 us limit and the LM-head kernel's load warps
    told to issue nothing (so that no copy or tensor-core operation is in flight when the waits
    give up), the status word reports DG_ETIMEOUT; the next call with the default limit on the
    same workspace is correct again.
"""

import math

import numpy as np
import pytest
import torch

from discrete_diffusion_text_gb300 import synth
from oracle import dgoracle as O

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
    dgcanvas.dg_workspace_status(None)  # start from a clean library status word
    return dgcanvas


def test_out_of_range_token_reports_kernel_error(dgc):
    w = synth.TINY
    m = synth.make_model(w, DEV)
    x = torch.tensor(O.initial_canvas(1, w.L, w.V, 3), dtype=torch.int32, device=DEV)
    x[0, 5] = w.V + 7
    x[0, 9] = -1
    BL = w.L
    h = torch.empty((BL, w.d), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((BL, w.H * w.hd), dtype=torch.bfloat16, device=DEV)
    k = torch.empty((BL, w.Hkv * w.hd), dtype=torch.bfloat16, device=DEV)
    v = torch.empty_like(k)
    dgc.dg_embed_qkv(x, m["E"], m["Wqkv"], h, q, k, v, w.H, w.Hkv, w.hd)
    with pytest.raises(dgc.DGError) as e:
        dgc.dg_workspace_status(None)
    assert e.value.status == dgc.DG_EKERNEL
    assert not h[5].any() and not h[9].any() and h[4].any()
    dgc.dg_workspace_status(None)  # the word was cleared by the read

    # inside the denoising loop: reported through the loop's workspace
    model = dgc.make_model(m["E"], m["Wqkv"], m["Wo"], w.H, w.Hkv, w.hd)
    kp, vp = synth.make_prefix_kv(w, DEV)
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(model, 1, w.L, w.P, w.window))
    lock = torch.zeros((1, w.L), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dgc.dg_denoise_loop(model, kp, vp, w.window, x, lock, st,
                        dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 3), ws)
    with pytest.raises(dgc.DGError) as e:
        dgc.dg_workspace_status(ws)
    assert e.value.status == dgc.DG_EKERNEL
    assert int(st[0]) == w.T
    # the last step (lambda = 1) replaced every position by a sample from the vocabulary
    xs = x.cpu().numpy()
    assert xs.min() >= 0 and xs.max() < w.V
    dgc.dg_workspace_status(ws)


def test_wait_timeout_is_reported_and_the_next_call_is_correct(dgc):
    B, L, V, d = 1, 64, 4096, 256
    y = synth.normal_bf16((B * L, d), 0.5, 71)
    E = synth.normal_bf16((V, d), 0.5, 72)
    ws = dgc.workspace(dgc.dg_vocab_posterior_workspace(B, L, V))

    def run():
        out = {kk: torch.empty(B * L, dtype=torch.int32 if kk in ("x0hat", "top1")
                               else torch.float32, device=DEV)
               for kk in ("x0hat", "top1", "logp_top1", "lse")}
        dgc.dg_vocab_posterior_step(y.to(DEV), E.to(DEV), B, L, 1.0, 5, 2, out=out, ws=ws)
        return out

    try:
        dgc.dg_set_wait_control(1000, skip_loads=True)  # 1 us, and nothing is loaded
        run()
    finally:
        dgc.dg_set_wait_control(0, skip_loads=False)
    with pytest.raises(dgc.DGError) as e:
        dgc.dg_workspace_status(ws)
    assert e.value.status == dgc.DG_ETIMEOUT

    out = run()
    dgc.dg_workspace_status(ws)
    ref = O.posterior(y.double().numpy(), E.double().numpy(), 1.0, 5, 2, L)
    assert np.abs(out["lse"].cpu().numpy() - ref["lse"]).max() <= 2e-3
    assert np.abs(out["logp_top1"].cpu().numpy() - ref["logp_top1"]).max() <= 2e-3
    d_top = out["top1"].cpu().numpy() != ref["top1"]
    assert not np.any(d_top & (ref["gap_logit"] >= 1e-4))
    d_x = out["x0hat"].cpu().numpy() != ref["x0hat"]
    assert not np.any(d_x & (ref["gap_perturbed"] >= 1e-3))


def test_wait_control_rejects_a_limit_above_a_minute(dgc):
    with pytest.raises(dgc.DGError) as e:
        dgc.dg_set_wait_control(61 * 10 ** 9)
    assert e.value.status == dgc.DG_EINVAL
    dgc.dg_set_wait_control(0)
