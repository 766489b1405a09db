"""GPU parity of encode-append and the block-autoregressive outer loop against the CPU oracle.
Every call goes through the C ABI."""

import dataclasses
import math

import numpy as np
import pytest
import torch

from discrete_diffusion_text_gb300 import synth
from oracle import dgoracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16_REL = 2.0 ** -7  # two bf16 roundings of the same exact value are at most one ulp apart


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


def _oracle_model(m):
    return {"E": f64(m["E"]), "Wqkv": f64(m["Wqkv"]), "Wo": f64(m["Wo"]), "H": m["H"],
            "Hkv": m["Hkv"], "hd": m["hd"]}


def _dev_model(dgc, m):
    E, Wqkv, Wo = (m[k].to(DEV) for k in ("E", "Wqkv", "Wo"))
    md = dgc.make_model(E, Wqkv, Wo, m["H"], m["Hkv"], m["hd"])
    md._keep = (E, Wqkv, Wo)  # the struct holds raw pointers
    return md


def _close_bf16(got, ref, abs_sum=None):
    """Element-wise: equal, or one bf16 rounding apart; with abs_sum (the sum of the absolute
    values of the products that form each element), also the fp32 accumulation error of a
    sum that cancels down to a tiny value (2^-20 of abs_sum: generous for 256-2048 terms)."""
    err = np.abs(got - ref)
    tol = BF16_REL * np.abs(ref) + 1e-30
    if abs_sum is not None:
        tol = tol + 2.0 ** -20 * abs_sum
    return err <= tol


def _kv_abs_sums(om, tokens):
    """sum_k |E[x]_k W_jk| for the key and value rows of the given tokens: [n, Hkv, hd] each."""
    H, Hkv, hd = om["H"], om["Hkv"], om["hd"]
    h = np.abs(om["E"][np.asarray(tokens).reshape(-1)])
    W = np.abs(om["Wqkv"])
    ak = h @ W[H * hd:(H + Hkv) * hd].T
    av = h @ W[(H + Hkv) * hd:].T
    return ak.reshape(-1, Hkv, hd), av.reshape(-1, Hkv, hd)


def _random_model(V, d, H, Hkv, hd, seed):
    return {"E": synth.normal_bf16((V, d), 0.5, seed), "Wqkv":
            synth.normal_bf16(((H + 2 * Hkv) * hd, d), 0.05, seed + 1),
            "Wo": synth.normal_bf16((d, H * hd), 0.02, seed + 2), "H": H, "Hkv": Hkv, "hd": hd}


@pytest.mark.parametrize("with_mask", [False, True])
def test_encode_append_rows_and_mask(dgc, with_mask):
    """K/V of the canvas land at rows P .. P+L-1 of the selected canvases (one bf16 rounding
    of the oracle's projections); every other cache byte is untouched."""
    B, L, P, V, d, H, Hkv, hd = 3, 128, 100, 1024, 256, 4, 2, 64
    cap = P + L + 64
    m = _random_model(V, d, H, Hkv, hd, 11)
    canvas = np.random.default_rng(4).integers(0, V, size=(B, L))
    kc = synth.normal_bf16((B, cap, Hkv, hd), 1.0, 12)
    vc = synth.normal_bf16((B, cap, Hkv, hd), 1.0, 13)
    gk, gv = kc.to(DEV), vc.to(DEV)
    active = np.array([1, 0, 1], np.uint8)
    md = _dev_model(dgc, m)
    ws = dgc.workspace(dgc.dg_encode_append_workspace(md, B, L))
    dgc.dg_encode_append(md, torch.tensor(canvas, dtype=torch.int32, device=DEV), gk, gv, P, ws,
                         active=torch.tensor(active, device=DEV) if with_mask else None)
    dgc.dg_workspace_status(ws)
    rows = np.nonzero(active)[0] if with_mask else None
    om = _oracle_model(m)
    rk, rv = O.encode_append(om, canvas, f64(kc), f64(vc), P, rows=rows)
    ak, av = _kv_abs_sums(om, canvas)
    for got, ref, before, asum in ((f64(gk), rk, f64(kc), ak), (f64(gv), rv, f64(vc), av)):
        written = np.zeros(got.shape, bool)
        sel = rows if with_mask else np.arange(B)
        written[sel, P:P + L] = True
        bound = np.zeros(got.shape)
        bound[:, P:P + L] = asum.reshape(B, L, Hkv, hd)
        assert np.all(_close_bf16(got[written], ref[written], bound[written]))
        assert (got[written] == ref[written]).mean() > 0.99
        assert np.array_equal(got[~written], before[~written])


def _delta_model(V, d, H, Hkv, hd):
    """Posterior a delta at the input token: E = 8 I, Wo = 0, so y = E[x] and the logits are
    64 at x and 0 elsewhere."""
    return {"E": (torch.eye(V, d) * 8.0).to(torch.bfloat16),
            "Wqkv": synth.normal_bf16(((H + 2 * Hkv) * hd, d), 0.02, 61),
            "Wo": torch.zeros((d, H * hd), dtype=torch.bfloat16), "H": H, "Hkv": Hkv, "hd": hd}


def _eos_in_second_block(B, L, V, seed):
    """A token of canvas 0's second prior that its first prior does not hold."""
    x0 = O.initial_canvas(B, L, V, seed)[0]
    x1 = O.initial_canvas(B, L, V, seed + 1)[0]
    for i in range(10, L):
        if x1[i] not in x0 and x1[i] not in x1[:i]:
            return int(x1[i]), i
    raise AssertionError("no usable end-of-turn token")


def _gpu_block_generate(dgc, m, kctx, vctx, cap, L, NB, window, eos, cfg):
    B, P0 = kctx.shape[:2]
    kc = torch.zeros((B, cap) + tuple(kctx.shape[2:]), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kc[:, :P0] = kctx.to(DEV)
    vc[:, :P0] = vctx.to(DEV)
    md = _dev_model(dgc, m)
    out = torch.zeros((B, NB, L), dtype=torch.int32, device=DEV)
    blocks, n_tok, steps = (torch.full((B,), 7, dtype=torch.int32, device=DEV) for _ in range(3))
    ws = dgc.workspace(dgc.dg_block_generate_workspace(md, B, L, P0, NB, window))
    dgc.dg_block_generate(md, kc, vc, P0, L, window, eos, cfg, out, blocks, n_tok, steps, ws)
    dgc.dg_workspace_status(ws)
    return (out.cpu().numpy(), blocks.cpu().numpy(), n_tok.cpu().numpy(), steps.cpu().numpy(),
            f64(kc), f64(vc))


@pytest.mark.parametrize("sampler", ["euler", "eb"])
def test_block_generate_delta_model_exact(dgc, sampler):
    """With a delta posterior every block returns its own prior x_1 (key seed + j); canvas 0
    meets the end-of-turn token in its second block and stops, the others run all blocks.
    Outputs equal the oracle's; the appended cache rows are one bf16 rounding from it."""
    B, L, P0, NB, V, d, H, Hkv, hd, T, seed = 3, 64, 100, 4, 256, 256, 2, 1, 64, 6, 21
    m = _delta_model(V, d, H, Hkv, hd)
    eos, pos = _eos_in_second_block(B, L, V, seed)
    kctx = synth.normal_bf16((B, P0, Hkv, hd), 1.0, 62)
    vctx = synth.normal_bf16((B, P0, Hkv, hd), 1.0, 63)
    thr = float(np.float32(math.log(0.9)))
    if sampler == "euler":
        cfg = dgc.make_cfg(T, 0, 1.0, thr, seed, stop_when_all_locked=True)
        okw = dict(lock_logthr=thr, stop_when_all_locked=True)
    else:
        cfg = dgc.make_cfg(T, 0, seed=seed, sampler=dgc.DG_SAMPLER_ENTROPY_BOUNDED)
        okw = dict(sampler="eb")
    cap = P0 + NB * L + 32
    got = _gpu_block_generate(dgc, m, kctx, vctx, cap, L, NB, 0, eos, cfg)
    out, blocks, n_tok, steps, rk, rv = O.block_generate(_oracle_model(m), f64(kctx), f64(vctx), 0,
                                                         L, NB, eos, seed, T, **okw)
    assert np.array_equal(got[0], out)
    assert np.array_equal(got[1], blocks) and np.array_equal(got[2], n_tok)
    assert np.array_equal(got[3], steps)
    assert blocks[0] == 2 and n_tok[0] == L + pos + 1
    for b in range(B):
        for j in range(blocks[b]):
            assert np.array_equal(out[b, j], O.initial_canvas(B, L, V, seed + j)[b])
    assert np.all(steps == blocks * (1 if sampler == "euler" else 2))
    for g, r in ((got[4], rk), (got[5], rv)):
        r_full = np.zeros_like(g)
        r_full[:, :r.shape[1]] = r
        assert np.all(_close_bf16(g, r_full))
        for b in range(B):  # rows past the generated blocks stay as they were (zero)
            assert not g[b, P0 + blocks[b] * L:].any()


@pytest.mark.parametrize("window", [0, 96])
def test_block_generate_tiny_random_model(dgc, window):
    """tiny-model shapes with a ragged context (P0 = 192 + 37), three blocks of 128 tokens, the
    Euler sampler: tokens agree with the oracle except at rare Gumbel near-ties, and the
    cache rows of the blocks that agree are one bf16 rounding from it."""
    w = dataclasses.replace(synth.TINY, B=2, L=128, P=229, d=256, H=4, Hkv=2, hd=64, V=4096, T=5)
    NB = 3
    m = synth.make_model(w)
    kctx, vctx = synth.make_prefix_kv(w)
    om = _oracle_model(m)
    cfg = dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, 5)
    args = (om, f64(kctx), f64(vctx), window, w.L, NB)
    # pick an end-of-turn token inside block 1 of canvas 1 (generation does not depend on eos)
    full = O.block_generate(*args, -1, 5, w.T, w.schedule)[0]
    eos = int(full[1, 1, 40])
    out, blocks, n_tok, steps, rk, rv = O.block_generate(*args, eos, 5, w.T, w.schedule)
    cap = w.P + NB * w.L
    g = _gpu_block_generate(dgc, m, kctx, vctx, cap, w.L, NB, window, eos, cfg)
    gen = out >= 0
    assert np.array_equal(g[0] >= 0, gen)
    assert (g[0][gen] == out[gen]).mean() >= 0.99
    assert np.array_equal(g[1], blocks) and np.array_equal(g[2], n_tok)
    assert np.all(g[3] == blocks * w.T)
    for b in range(w.B):
        for j in range(blocks[b]):
            if not np.array_equal(g[0][b, j], out[b, j]):
                break
            r0 = w.P + j * w.L
            ak, av = _kv_abs_sums(om, out[b, j])
            for gc, rc, asum in ((g[4], rk, ak), (g[5], rv, av)):
                assert np.all(_close_bf16(gc[b, r0:r0 + w.L], rc[b, r0:r0 + w.L], asum))


def test_block_generate_window1k_blocks_equal_standalone_loops(dgc):
    """window1k shapes at full size (1,024-token context, 262,144-token vocabulary), two
    blocks: each block's canvas is what dg_denoise_loop gives alone on the same prefix and
    key, the appended rows are dg_encode_append of it, and 16 sampled appended rows match the
    oracle's projections of the generated tokens."""
    w = dataclasses.replace(synth.WINDOW1K, T=3)
    NB = 2
    m = synth.make_model(w, DEV)
    kctx, vctx = synth.make_prefix_kv(w, DEV)
    cap = w.P + NB * w.L
    eos = -1
    cfg = dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, w.seed)
    out, blocks, n_tok, steps, gk, gv = _gpu_block_generate(dgc, m, kctx, vctx, cap, w.L, NB,
                                                            w.window, eos, cfg)
    assert blocks.tolist() == [NB] and n_tok.tolist() == [NB * w.L]
    assert steps.tolist() == [NB * w.T]
    md = _dev_model(dgc, m)
    kp = torch.tensor(gk, dtype=torch.bfloat16, device=DEV)
    vp = torch.tensor(gv, dtype=torch.bfloat16, device=DEV)
    for j in range(NB):
        P = w.P + j * w.L
        c = torch.tensor(O.initial_canvas(1, w.L, w.V, w.seed + j), dtype=torch.int32,
                         device=DEV)
        lock = torch.zeros((1, w.L), dtype=torch.uint8, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        ws = dgc.workspace(dgc.dg_denoise_loop_workspace(md, 1, w.L, P, w.window))
        dgc.dg_denoise_loop(md, kp[:, :P].contiguous(), vp[:, :P].contiguous(), w.window, c,
                            lock, st, dgc.make_cfg(w.T, w.schedule, 1.0, math.inf, w.seed + j),
                            ws)
        dgc.dg_workspace_status(ws)
        assert np.array_equal(c.cpu().numpy()[0], out[0, j])
    # the appended rows: one bf16 rounding from the oracle's k = E[x] Wk^T, v = E[x] Wv^T
    om_E = m["E"].double().cpu()
    Wqkv = m["Wqkv"].double().cpu()
    Hhd, KVhd = w.H * w.hd, w.Hkv * w.hd
    rows = np.sort(np.random.default_rng(6).choice(NB * w.L, 16, replace=False))
    toks = out[0].reshape(-1)[rows]
    h = om_E[torch.tensor(toks)]
    k = O.round_bf16((h @ Wqkv[Hhd:Hhd + KVhd].T).numpy()).reshape(16, w.Hkv, w.hd)
    v = O.round_bf16((h @ Wqkv[Hhd + KVhd:].T).numpy()).reshape(16, w.Hkv, w.hd)
    ak = (h.abs() @ Wqkv[Hhd:Hhd + KVhd].abs().T).numpy().reshape(16, w.Hkv, w.hd)
    av = (h.abs() @ Wqkv[Hhd + KVhd:].abs().T).numpy().reshape(16, w.Hkv, w.hd)
    assert np.all(_close_bf16(gk[0, w.P + rows], k, ak))
    assert np.all(_close_bf16(gv[0, w.P + rows], v, av))


def test_block_generate_with_self_conditioning(dgc):
    """Block-AR generation with a self-conditioning decoder: every block's loop starts from a
    zero signal; tokens agree with the oracle except at rare near-ties."""
    w = dataclasses.replace(synth.TINY, B=2, L=128, P=192, d=256, H=4, Hkv=2, hd=64, V=4096, T=4)
    NB = 2
    m = synth.make_model(w)
    m["Wsc1"] = synth.normal_bf16((64, w.d), 1.0, 301)
    m["Wsc2"] = synth.normal_bf16((w.d, 64), 4.0, 302)
    kctx, vctx = synth.make_prefix_kv(w)
    om = {k: (f64(v) if torch.is_tensor(v) else v) for k, v in m.items()}
    out, blocks, n_tok, steps, _, _ = O.block_generate(om, f64(kctx), f64(vctx), 0, w.L, NB, -1,
                                                       11, w.T, w.schedule)
    kc = torch.zeros((w.B, w.P + NB * w.L, w.Hkv, w.hd), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kc[:, :w.P] = kctx.to(DEV)
    vc[:, :w.P] = vctx.to(DEV)
    md = dgc.make_model(*(m[k].to(DEV) for k in ("E", "Wqkv", "Wo")), w.H, w.Hkv, w.hd,
                        m["Wsc1"].to(DEV), m["Wsc2"].to(DEV))
    g_out = torch.zeros((w.B, NB, w.L), dtype=torch.int32, device=DEV)
    g_b, g_n, g_s = (torch.zeros(w.B, dtype=torch.int32, device=DEV) for _ in range(3))
    ws = dgc.workspace(dgc.dg_block_generate_workspace(md, w.B, w.L, w.P, NB, 0))
    dgc.dg_block_generate(md, kc, vc, w.P, w.L, 0, -1, dgc.make_cfg(w.T, w.schedule, 1.0,
                                                                     math.inf, 11),
                          g_out, g_b, g_n, g_s, ws)
    dgc.dg_workspace_status(ws)
    assert g_b.cpu().tolist() == blocks.tolist() == [NB, NB]
    assert g_s.cpu().tolist() == steps.tolist()
    assert (g_out.cpu().numpy() == out).mean() >= 0.99
