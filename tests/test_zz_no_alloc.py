"""The allocation-free variant of the fused vocabulary step.

Some callers of this library cannot allocate device memory for a workspace (an operator inside
a host framework that only receives its input and output buffers, a process whose device
memory is reserved up front, a loop that must not risk cudaMalloc's device synchronisation).
dg_vocab_posterior_step_noalloc serves them from a fixed device array inside the library.
This file checks, through the C ABI, that two calls in a row give the same results as the
workspace entry point, that the second call leaves the device's free memory and torch's
allocations unchanged, and that a size beyond the array is refused.  It is collected last and
also runs on its own in a fresh process.
"""

import math

import numpy as np
import pytest
import torch

from discrete_diffusion_text_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
LOGP_TOL = 2e-3  # the log-probability tolerance of the parity tests


@pytest.fixture(scope="module")
def dgc():
    import os

    from discrete_diffusion_text_gb300 import dgcanvas

    if not os.path.exists(dgcanvas.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build()
    dgcanvas.load()
    return dgcanvas


def _outputs(R):
    return {k: torch.full((R,), -7, dtype=torch.int32 if k in ("x0hat", "top1") else torch.float32,
                          device=DEV) for k in ("x0hat", "top1", "logp_top1", "lse", "logp_x0hat")}


def _run(dgc, fn, y, E, B, L, inv_tau, seed, step, x_in, lock_in, jump_thr, thr, ws=None):
    R = B * L
    out = _outputs(R)
    x = x_in.clone()
    lk = lock_in.clone()
    jp = torch.zeros(R, dtype=torch.uint8, device=DEV)
    dn = torch.zeros(B, dtype=torch.uint8, device=DEV)
    kw = dict(x_in=x, x_out=x, lock=lk, jump=jp, done=dn, jump_thr=jump_thr, lock_logthr=thr,
              out=out)
    if ws is None:
        fn(y, E, B, L, inv_tau, seed, step, **kw)
    else:
        fn(y, E, B, L, inv_tau, seed, step, ws=ws, **kw)
    dgc.dg_workspace_status(ws)
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res.update(x=x.cpu().numpy(), lock=lk.cpu().numpy(), jump=jp.cpu().numpy(),
               done=dn.cpu().numpy())
    return res


def _run_bare(dgc, y, E, B, L, inv_tau, seed, step, x_in, lock_in, jump_thr, thr):
    """The allocation-free call alone, with every buffer made beforehand (the caller's)."""
    R = B * L
    bufs = dict(out=_outputs(R), x=x_in.clone(), lock=lock_in.clone(),
                jump=torch.zeros(R, dtype=torch.uint8, device=DEV),
                done=torch.zeros(B, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    dgc.dg_vocab_posterior_step_noalloc(y, E, B, L, inv_tau, seed, step, x_in=bufs["x"],
                                        x_out=bufs["x"], lock=bufs["lock"], jump=bufs["jump"],
                                        done=bufs["done"], jump_thr=jump_thr, lock_logthr=thr,
                                        out=bufs["out"])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0  # the device's free memory (driver view)
    assert torch.cuda.memory_allocated() == alloc0
    return bufs


def _collect(dgc, bufs):
    dgc.dg_workspace_status(None)
    res = {k: v.cpu().numpy() for k, v in bufs["out"].items()}
    res.update(x=bufs["x"].cpu().numpy(), lock=bufs["lock"].cpu().numpy(),
               jump=bufs["jump"].cpu().numpy(), done=bufs["done"].cpu().numpy())
    return res


def _same(a, b):
    for k in ("lse", "logp_top1", "logp_x0hat"):
        assert np.abs(a[k] - b[k]).max() <= LOGP_TOL, k
    for k in ("x0hat", "top1", "x", "lock", "jump", "done"):
        assert np.array_equal(a[k], b[k]), k


def test_noalloc_matches_workspace_entry_point_on_two_calls(dgc):
    B, L, V, d = 3, 256, 8192, 256
    E = synth.normal_bf16((V, d), 0.1, 71).to(DEV)
    thr = float(np.float32(math.log(0.9)))
    _, jumps = dgc.dg_schedule_thresholds(0, 12)
    rng = np.random.default_rng(5)
    x0 = torch.tensor(rng.integers(0, V, B * L).astype(np.int32), device=DEV)
    lock0 = torch.tensor((rng.random(B * L) < 0.1).astype(np.uint8), device=DEV)
    ws = dgc.workspace(dgc.dg_vocab_posterior_workspace(B, L, V))
    # two calls in a row with different inputs, each checked against the workspace call
    for call, (ystd, inv_tau, step) in enumerate(((1.0, 20.0, 4), (0.05, 1.0, 9))):
        y = synth.normal_bf16((B * L, d), ystd, 72 + call).to(DEV)
        if call == 1:  # the first call loaded the array's module; from now on nothing is taken
            a = _collect(dgc, _run_bare(dgc, y, E, B, L, inv_tau, 99, step, x0, lock0,
                                        int(jumps[step]), thr))
        else:
            a = _run(dgc, dgc.dg_vocab_posterior_step_noalloc, y, E, B, L, inv_tau, 99, step, x0,
                     lock0, int(jumps[step]), thr)
        b = _run(dgc, dgc.dg_vocab_posterior_step, y, E, B, L, inv_tau, 99, step, x0, lock0,
                 int(jumps[step]), thr, ws=ws)
        _same(a, b)
        assert (a["x0hat"] >= 0).all() and (a["x0hat"] < V).all()
        if call == 0:
            assert a["lock"].mean() > 0.1  # the sharp first call does lock positions


def test_noalloc_refuses_sizes_beyond_its_array(dgc):
    # 2,050 canvases of 256 positions need more than 16 MiB of scratch (host-side query first);
    # the buffers passed are really that large, so the call could not read out of bounds even
    # if it were accepted.
    B, L, V, d = 2050, 256, 256, 64
    assert dgc.dg_vocab_posterior_workspace(B, L, V) - 256 > 16 << 20
    y = torch.zeros((B * L, d), dtype=torch.bfloat16, device=DEV)
    E = torch.zeros((V, d), dtype=torch.bfloat16, device=DEV)
    so = dgc.load()
    st = so.dg_vocab_posterior_step_noalloc(y.data_ptr(), E.data_ptr(), B, L, d, V, 1.0, 0, 0,
                                            None, None, None, None, None, 0, math.inf, None, None)
    assert st == dgc.DG_ENOTSUP
    assert "16 MiB" in so.dg_last_error().decode()
