"""Thin Python binding of libdgcanvas (argument marshalling only).

Each function has the name of the C entry point it calls, takes torch tensors (device memory
for device arguments) or numpy arrays (host arguments), passes raw pointers and sizes through
ctypes, and raises DGError on a non-OK status.  No step of the method runs here: if the
library is missing, loading fails loudly; there is no fallback.
"""

from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdgcanvas.so")

DG_OK, DG_EINVAL, DG_ENOTSUP, DG_ECUDA, DG_EKERNEL, DG_ETIMEOUT = range(6)
DG_SCHED_LINEAR, DG_SCHED_COSINE = 0, 1
DG_SAMPLER_EULER, DG_SAMPLER_ENTROPY_BOUNDED = 0, 1
_STATUS_NAMES = {0: "DG_OK", 1: "DG_EINVAL", 2: "DG_ENOTSUP", 3: "DG_ECUDA", 4: "DG_EKERNEL",
                 5: "DG_ETIMEOUT"}

# C entry points and their signatures, as declared in include/dgcanvas.h.
_P = ctypes.c_void_p
_I = ctypes.c_int
_U64 = ctypes.c_uint64
_F = ctypes.c_float
_D = ctypes.c_double
_SZ = ctypes.c_size_t


class DGError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn}: {_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class dg_model(ctypes.Structure):
    _fields_ = [("E", _P), ("Wqkv", _P), ("Wo", _P), ("V", _I), ("d", _I), ("H", _I),
                ("Hkv", _I), ("hd", _I), ("Wsc1", _P), ("Wsc2", _P), ("d_sc", _I)]


class dg_sampler_cfg(ctypes.Structure):
    _fields_ = [("T", _I), ("schedule", _I), ("inv_tau", _F), ("lock_logthr", _F),
                ("seed", _U64), ("start_step", _I), ("end_step", _I),
                ("stop_when_all_locked", _I), ("sampler", _I), ("tau_start", _D),
                ("tau_end", _D), ("gamma", _F), ("stop_entropy", _F)]


class dg_posterior_out(ctypes.Structure):
    _fields_ = [("x0hat", _P), ("top1", _P), ("logp_top1", _P), ("lse", _P),
                ("logp_x0hat", _P), ("entropy", _P)]


_POST_FIELDS = ("x0hat", "top1", "logp_top1", "lse", "logp_x0hat", "entropy")


SIGNATURES = {
    "dg_last_error": (ctypes.c_char_p, []),
    "dg_abi_version": (_I, []),
    "dg_schedule_thresholds": (_I, [_I, _I, _P, _P]),
    "dg_keep_thresholds": (_I, [_I, _P, _I, _P]),
    "dg_forward_noise": (_I, [_P, _P, _P, _I, _I, _I, _U64, _P]),
    "dg_embed_qkv": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "dg_canvas_attn_workspace": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "dg_canvas_attn": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _SZ,
                            _P]),
    "dg_out_proj": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "dg_vocab_posterior_workspace": (_SZ, [_I, _I, _I]),
    "dg_vocab_posterior_step": (_I, [_P, _P, _I, _I, _I, _I, _F, _U64, _I, _P, _P, _P, _P, _P,
                                     _U64, _F, _P, _P, _SZ, _P]),
    "dg_vocab_posterior_step_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _F, _U64, _I, _P, _P, _P,
                                             _P, _P, _U64, _F, _P, _P]),
    "dg_euler_update": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _U64, _I, _U64, _F, _P]),
    "dg_cross_entropy_step": (_I, [_P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _SZ, _P]),
    "dg_sft_loss": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _U64, _F, _P, _P, _P, _SZ, _P]),
    "dg_entropy_bounded_update": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _U64, _I,
                                       _F, _F, _I, _P]),
    "dg_denoise_loop_workspace": (_SZ, [_P, _I, _I, _I, _I]),
    "dg_denoise_loop_kernel_count": (_I, [_P, _I, _I, _I, _I, _I]),
    "dg_denoise_loop": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "dg_self_condition_workspace": (_SZ, [_I, _I, _I, _I, _I]),
    "dg_self_condition": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _SZ, _P]),
    "dg_encode_append_workspace": (_SZ, [_P, _I, _I]),
    "dg_encode_append": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "dg_block_generate_workspace": (_SZ, [_P, _I, _I, _I, _I, _I]),
    "dg_block_generate": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                               _SZ, _P]),
    "dg_workspace_status": (_I, [_P, _P]),
    "dg_set_wait_control": (_I, [_U64, _I]),
    "dg_kernel_timer_enable": (_I, [_I]),
    "dg_kernel_timer_read": (_I, [_I, _P, _P]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libdgcanvas.so (built in-tree); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int, fn: str):
    if status != DG_OK:
        raise DGError(status, fn, load().dg_last_error().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dev(t: torch.Tensor, dtype, name: str):
    if t is None:
        return None
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}")
    return t


def _bf16(t, name):
    return _dev(t, torch.bfloat16, name)


# ------------------------------------------------------------------------- host calls ---

def dg_abi_version() -> int:
    return load().dg_abi_version()


def dg_schedule_thresholds(schedule: int, T: int):
    keep = np.zeros(T + 1, np.uint64)
    jump = np.zeros(T, np.uint64)
    _check(load().dg_schedule_thresholds(schedule, T, keep.ctypes.data, jump.ctypes.data),
           "dg_schedule_thresholds")
    return keep, jump


def dg_keep_thresholds(schedule: int, t) -> np.ndarray:
    t = np.ascontiguousarray(t, np.float64)
    out = np.zeros(t.size, np.uint64)
    _check(load().dg_keep_thresholds(schedule, t.ctypes.data, t.size, out.ctypes.data),
           "dg_keep_thresholds")
    return out


# ----------------------------------------------------------------------- device calls ---

def dg_forward_noise(x0, xt, keep_thr, V: int, seed: int, stream=None):
    """x0, xt: int32 [B, L] CUDA; keep_thr: int64 [B] CUDA holding floor(kappa * 2^32)."""
    _dev(x0, torch.int32, "x0")
    _dev(xt, torch.int32, "xt")
    _dev(keep_thr, torch.int64, "keep_thr")
    B, L = x0.shape
    _check(load().dg_forward_noise(_ptr(x0), _ptr(xt), _ptr(keep_thr), B, L, V, seed,
                                   _stream(stream)), "dg_forward_noise")


def dg_embed_qkv(x, E, Wqkv, h, q, k, v, H: int, Hkv: int, hd: int, stream=None):
    _dev(x, torch.int32, "x")
    for t, n in ((E, "E"), (Wqkv, "Wqkv"), (h, "h"), (q, "q"), (k, "k"), (v, "v")):
        _bf16(t, n)
    V, d = E.shape
    _check(load().dg_embed_qkv(_ptr(x), _ptr(E), _ptr(Wqkv), _ptr(h), _ptr(q), _ptr(k), _ptr(v),
                               x.numel(), V, d, H, Hkv, hd, _stream(stream)), "dg_embed_qkv")


def dg_canvas_attn_workspace(B, L, P, H, Hkv, hd, window) -> int:
    return load().dg_canvas_attn_workspace(B, L, P, H, Hkv, hd, window)


def dg_canvas_attn(q, k_pre, v_pre, k_can, v_can, out, lse, window: int, scale: float | None,
                   ws, stream=None):
    """q [B, L, H, hd]; k_pre/v_pre [B, P, Hkv, hd]; k_can/v_can [B, L, Hkv, hd]; out like q;
    lse fp32 [B, H, L] or None; ws uint8 CUDA workspace."""
    for t, n in ((q, "q"), (k_can, "k_can"), (v_can, "v_can"), (out, "out")):
        _bf16(t, n)
    B, L, H, hd = q.shape
    P, Hkv = k_pre.shape[1], k_pre.shape[2]
    if P > 0:
        _bf16(k_pre, "k_pre")
        _bf16(v_pre, "v_pre")
    if lse is not None:
        _dev(lse, torch.float32, "lse")
    scale = hd ** -0.5 if scale is None else scale
    _check(load().dg_canvas_attn(_ptr(q), _ptr(k_pre) if P > 0 else None,
                                 _ptr(v_pre) if P > 0 else None, _ptr(k_can), _ptr(v_can),
                                 _ptr(out), _ptr(lse), B, L, P, H, Hkv, hd, window, scale,
                                 _ptr(ws), ws.numel(), _stream(stream)), "dg_canvas_attn")


def dg_out_proj(h, O, Wo, y, stream=None):
    for t, n in ((h, "h"), (O, "O"), (Wo, "Wo"), (y, "y")):
        _bf16(t, n)
    d = Wo.shape[0]
    BL = h.numel() // d
    _check(load().dg_out_proj(_ptr(h), _ptr(O), _ptr(Wo), _ptr(y), BL, d, Wo.shape[1],
                              _stream(stream)), "dg_out_proj")


def dg_vocab_posterior_workspace(B, L, V) -> int:
    return load().dg_vocab_posterior_workspace(B, L, V)


def dg_vocab_posterior_step(y, W, B: int, L: int, inv_tau: float, seed: int, step: int,
                            x_in=None, x_out=None, lock=None, jump=None, done=None,
                            jump_thr: int = 0, lock_logthr: float = math.inf, out=None,
                            ws=None, stream=None):
    """y [B*L, d] bf16; W [V, d] bf16; x_in/x_out int32 [B*L] or None; lock/jump uint8 [B*L];
    done uint8 [B]; out: dict with optional int32/fp32 [B*L] tensors x0hat, top1, logp_top1,
    lse, logp_x0hat, entropy."""
    _bf16(y, "y")
    _bf16(W, "W")
    V, d = W.shape
    po = None
    if out is not None:
        po = dg_posterior_out(*(_ptr(out.get(k)) for k in _POST_FIELDS))
    _check(load().dg_vocab_posterior_step(
        _ptr(y), _ptr(W), B, L, d, V, inv_tau, seed, step, _ptr(x_in), _ptr(x_out), _ptr(lock),
        _ptr(jump), _ptr(done), jump_thr, lock_logthr,
        ctypes.addressof(po) if po is not None else None, _ptr(ws), ws.numel(), _stream(stream)),
        "dg_vocab_posterior_step")


def dg_vocab_posterior_step_noalloc(y, W, B: int, L: int, inv_tau: float, seed: int, step: int,
                                    x_in=None, x_out=None, lock=None, jump=None, done=None,
                                    jump_thr: int = 0, lock_logthr: float = math.inf, out=None,
                                    stream=None):
    """dg_vocab_posterior_step without a workspace: the library's fixed device scratch array
    is used instead (for callers that cannot allocate); same arguments otherwise."""
    _bf16(y, "y")
    _bf16(W, "W")
    V, d = W.shape
    po = None
    if out is not None:
        po = dg_posterior_out(*(_ptr(out.get(k)) for k in _POST_FIELDS))
    _check(load().dg_vocab_posterior_step_noalloc(
        _ptr(y), _ptr(W), B, L, d, V, inv_tau, seed, step, _ptr(x_in), _ptr(x_out), _ptr(lock),
        _ptr(jump), _ptr(done), jump_thr, lock_logthr,
        ctypes.addressof(po) if po is not None else None, _stream(stream)),
        "dg_vocab_posterior_step_noalloc")


def dg_euler_update(x_in, x0hat, top1, logp_top1, x_out, lock, jump, done, seed: int, step: int,
                    jump_thr: int, lock_logthr: float, stream=None):
    B, L = x_in.shape
    _check(load().dg_euler_update(_ptr(x_in), _ptr(x0hat), _ptr(top1), _ptr(logp_top1),
                                  _ptr(x_out), _ptr(lock), _ptr(jump), _ptr(done), B, L, seed,
                                  step, jump_thr, lock_logthr, _stream(stream)),
           "dg_euler_update")


def dg_cross_entropy_step(y, W, B: int, L: int, inv_tau: float, targets, loss, lse=None,
                          ws=None, stream=None):
    """y [B*L, d] bf16; W [V, d] bf16; targets int32 [B*L]; loss (and lse) fp32 [B*L] out."""
    _bf16(y, "y")
    _bf16(W, "W")
    V, d = W.shape
    _dev(targets, torch.int32, "targets")
    _dev(loss, torch.float32, "loss")
    _check(load().dg_cross_entropy_step(_ptr(y), _ptr(W), B, L, d, V, inv_tau, _ptr(targets),
                                        _ptr(loss), _ptr(lse), _ptr(ws), ws.numel(),
                                        _stream(stream)), "dg_cross_entropy_step")


def dg_sft_loss(m, k_pre, v_pre, window: int, x0, keep_thr, seed: int, xt, loss,
                inv_tau: float = 1.0, ws=None, stream=None):
    """x0, xt int32 [B, L]; keep_thr int64/uint64 [B] (device); loss fp32 [B, L] out."""
    _dev(x0, torch.int32, "x0")
    _dev(xt, torch.int32, "xt")
    _dev(loss, torch.float32, "loss")
    B, L = x0.shape
    P = k_pre.shape[1]
    _check(load().dg_sft_loss(ctypes.byref(m), _ptr(k_pre) if P > 0 else None,
                              _ptr(v_pre) if P > 0 else None, B, L, P, window, _ptr(x0),
                              _ptr(keep_thr), seed, inv_tau, _ptr(xt), _ptr(loss), _ptr(ws),
                              ws.numel(), _stream(stream)), "dg_sft_loss")


def dg_entropy_bounded_update(x0hat, top1, entropy, x_out, seed: int, step: int, V: int,
                              gamma: float, stop_entropy: float, prev_top1=None,
                              prev_valid: bool = True, accept=None, done=None,
                              mean_entropy=None, final_step: bool = False, stream=None):
    """x0hat, top1, x_out, prev_top1 int32 [B, L]; entropy fp32 [B, L]; accept uint8 [B, L];
    done uint8 [B]; mean_entropy fp32 [B]."""
    B, L = x0hat.shape
    _check(load().dg_entropy_bounded_update(
        _ptr(x0hat), _ptr(top1), _ptr(entropy), _ptr(prev_top1), 1 if prev_valid else 0,
        _ptr(x_out), _ptr(accept), _ptr(done), _ptr(mean_entropy), B, L, V, seed, step, gamma,
        stop_entropy, 1 if final_step else 0, _stream(stream)), "dg_entropy_bounded_update")


def make_model(E, Wqkv, Wo, H: int, Hkv: int, hd: int, Wsc1=None, Wsc2=None) -> dg_model:
    """Weights of the stand-in decoder (device bf16); Wsc1 [d_sc, d] and Wsc2 [d, d_sc] turn on
    self-conditioning."""
    for t, n in ((E, "E"), (Wqkv, "Wqkv"), (Wo, "Wo")):
        _bf16(t, n)
    if (Wsc1 is None) != (Wsc2 is None):
        raise ValueError("Wsc1 and Wsc2 go together")
    d_sc = 0
    if Wsc1 is not None:
        _bf16(Wsc1, "Wsc1")
        _bf16(Wsc2, "Wsc2")
        d_sc = Wsc1.shape[0]
    V, d = E.shape
    m = dg_model(_ptr(E), _ptr(Wqkv), _ptr(Wo), V, d, H, Hkv, hd, _ptr(Wsc1), _ptr(Wsc2), d_sc)
    m._keep = (E, Wqkv, Wo, Wsc1, Wsc2)
    return m


def make_cfg(T: int, schedule: int, inv_tau: float = 1.0, lock_logthr: float = math.inf,
             seed: int = 0, start_step: int = 0, end_step: int = 0,
             stop_when_all_locked: bool = False, sampler: int = DG_SAMPLER_EULER,
             tau_start: float = 0.8, tau_end: float = 0.4, gamma: float = 0.1,
             stop_entropy: float = 0.005) -> dg_sampler_cfg:
    return dg_sampler_cfg(T, schedule, inv_tau, lock_logthr, seed, start_step, end_step,
                          1 if stop_when_all_locked else 0, sampler, tau_start, tau_end, gamma,
                          stop_entropy)


def dg_denoise_loop_workspace(m: dg_model, B, L, P, window) -> int:
    return load().dg_denoise_loop_workspace(ctypes.byref(m), B, L, P, window)


def dg_denoise_loop_kernel_count(m: dg_model, B, L, P, window, steps) -> int:
    return load().dg_denoise_loop_kernel_count(ctypes.byref(m), B, L, P, window, steps)


def dg_denoise_loop(m: dg_model, k_pre, v_pre, window: int, canvas, lock, steps_taken,
                    cfg: dg_sampler_cfg, ws, stream=None):
    """canvas int32 [B, L] (in/out); lock uint8 [B, L] (in/out; may be None with the
    entropy-bounded sampler); steps_taken int32 [B] (out)."""
    _dev(canvas, torch.int32, "canvas")
    if lock is not None:
        _dev(lock, torch.uint8, "lock")
    _dev(steps_taken, torch.int32, "steps_taken")
    B, L = canvas.shape
    P = k_pre.shape[1]
    _check(load().dg_denoise_loop(ctypes.byref(m), _ptr(k_pre) if P > 0 else None,
                                  _ptr(v_pre) if P > 0 else None, B, L, P, window, _ptr(canvas),
                                  _ptr(lock), _ptr(steps_taken), ctypes.byref(cfg), _ptr(ws),
                                  ws.numel(), _stream(stream)), "dg_denoise_loop")


def dg_self_condition_workspace(B, L, d, V, d_sc) -> int:
    return load().dg_self_condition_workspace(B, L, d, V, d_sc)


def dg_self_condition(y, E, Wsc1, Wsc2, B: int, L: int, inv_tau: float, s_out, ws, e_out=None,
                      stream=None):
    """y bf16 [B*L, d]; E bf16 [V, d]; Wsc1 bf16 [d_sc, d]; Wsc2 bf16 [d, d_sc]; s_out bf16
    [B*L, d] (out); e_out bf16 [B*L, d] (out, optional: the expected embedding p_hat . E)."""
    for t, n in ((y, "y"), (E, "E"), (Wsc1, "Wsc1"), (Wsc2, "Wsc2"), (s_out, "s_out")):
        _bf16(t, n)
    if e_out is not None:
        _bf16(e_out, "e_out")
    V, d = E.shape
    _check(load().dg_self_condition(_ptr(y), _ptr(E), _ptr(Wsc1), _ptr(Wsc2), B, L, d, V,
                                    Wsc1.shape[0], inv_tau, _ptr(s_out), _ptr(e_out), _ptr(ws),
                                    ws.numel(), _stream(stream)), "dg_self_condition")


def dg_encode_append_workspace(m: dg_model, B, L) -> int:
    return load().dg_encode_append_workspace(ctypes.byref(m), B, L)


def dg_encode_append(m: dg_model, canvas, k_cache, v_cache, P: int, ws, active=None,
                     stream=None):
    """canvas int32 [B, L]; k_cache, v_cache bf16 [B, P_cap, Hkv, hd] (rows P .. P+L-1 written
    for canvases with active[b] != 0, all if active is None)."""
    _dev(canvas, torch.int32, "canvas")
    if active is not None:
        _dev(active, torch.uint8, "active")
    B, L = canvas.shape
    P_cap = k_cache.shape[1]
    _check(load().dg_encode_append(ctypes.byref(m), _ptr(canvas), _ptr(k_cache), _ptr(v_cache),
                                   B, L, P, P_cap, _ptr(active), _ptr(ws), ws.numel(),
                                   _stream(stream)), "dg_encode_append")


def dg_block_generate_workspace(m: dg_model, B, L, P0, NB, window) -> int:
    return load().dg_block_generate_workspace(ctypes.byref(m), B, L, P0, NB, window)


def dg_block_generate(m: dg_model, k_cache, v_cache, P0: int, L: int, window: int, eos: int,
                      cfg: dg_sampler_cfg, out, blocks, n_tokens, steps, ws, stream=None):
    """k_cache, v_cache bf16 [B, P_cap, Hkv, hd] (rows 0 .. P0-1 the context; generated canvases
    appended); out int32 [B, NB, L]; blocks, n_tokens, steps int32 [B] (all outputs)."""
    _dev(out, torch.int32, "out")
    for t, name in ((blocks, "blocks"), (n_tokens, "n_tokens"), (steps, "steps")):
        _dev(t, torch.int32, name)
    B, NB, Lo = out.shape
    if Lo != L:
        raise ValueError("out must be [B, NB, L]")
    P_cap = k_cache.shape[1]
    _check(load().dg_block_generate(ctypes.byref(m), _ptr(k_cache), _ptr(v_cache), B, P0, P_cap,
                                    L, NB, window, eos, ctypes.byref(cfg), _ptr(out),
                                    _ptr(blocks), _ptr(n_tokens), _ptr(steps), _ptr(ws),
                                    ws.numel(), _stream(stream)), "dg_block_generate")


def dg_workspace_status(ws=None, stream=None):
    _check(load().dg_workspace_status(_ptr(ws), _stream(stream)), "dg_workspace_status")


def dg_set_wait_control(limit_ns: int = 0, skip_loads: bool = False):
    """Limit (ns) of every on-chip wait of the calls this thread enqueues next (0 = 2 s);
    skip_loads makes the LM-head kernel's load warps issue nothing (timeout-path tests)."""
    _check(load().dg_set_wait_control(int(limit_ns), 1 if skip_loads else 0),
           "dg_set_wait_control")


def dg_kernel_timer_enable(on: bool):
    _check(load().dg_kernel_timer_enable(1 if on else 0), "dg_kernel_timer_enable")


def dg_kernel_timer_read(kind: int):
    ms = ctypes.c_double()
    n = ctypes.c_int()
    _check(load().dg_kernel_timer_read(kind, ctypes.byref(ms), ctypes.byref(n)),
           "dg_kernel_timer_read")
    return ms.value, n.value


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed uint8 device buffer (the caller owns workspace memory)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
