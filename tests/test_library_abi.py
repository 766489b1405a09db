"""The C-ABI library loads, exports every symbol include/dgcanvas.h declares, and its host-side
logic (schedule thresholds, argument validation) behaves without a GPU."""

import ctypes
import math
import os
import re

import numpy as np
import pytest

from oracle import dgoracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dgcanvas.h")


@pytest.fixture(scope="module")
def lib():
    from discrete_diffusion_text_gb300 import dgcanvas as dgc

    if not os.path.exists(dgc.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build()
    return dgc


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_calls_of_the_path():
    names = declared_functions()
    for f in ("dg_forward_noise", "dg_canvas_attn", "dg_vocab_posterior_step", "dg_euler_update",
              "dg_denoise_loop"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing
    assert set(declared_functions()) == set(lib.SIGNATURES), \
        "binding signatures and header declarations differ"


def test_abi_version(lib):
    assert lib.dg_abi_version() == 3


@pytest.mark.parametrize("T", [1, 2, 12, 48])
def test_linear_thresholds_equal_oracle(lib, T):
    keep, jump = lib.dg_schedule_thresholds(lib.DG_SCHED_LINEAR, T)
    ok, oj = O.schedule_thresholds(O.SCHED_LINEAR, T)
    assert np.array_equal(keep, ok) and np.array_equal(jump, oj)


@pytest.mark.parametrize("T", [2, 12, 48])
def test_cosine_thresholds_equal_oracle(lib, T):
    """Both sides evaluate the schedule in double precision; the libm's cos/sin may round one
    ulp differently, so a threshold may differ by one count out of 2^32 (a draw would have to
    hit that single value to change a decision)."""
    keep, jump = lib.dg_schedule_thresholds(lib.DG_SCHED_COSINE, T)
    ok, oj = O.schedule_thresholds(O.SCHED_COSINE, T)
    assert np.abs(keep.astype(np.int64) - ok.astype(np.int64)).max() <= 1
    assert np.abs(jump.astype(np.int64) - oj.astype(np.int64)).max() <= 1
    assert jump[0] == 0 and jump[-1] == 1 << 32


def test_keep_thresholds_from_t(lib):
    t = np.random.default_rng(0).random(64)
    t[:3] = [0.0, 1.0, 0.5]
    for s in (lib.DG_SCHED_LINEAR, lib.DG_SCHED_COSINE):
        got = lib.dg_keep_thresholds(s, t)
        ref = O.keep_threshold_from_t(s, t)
        assert np.abs(got.astype(np.int64) - ref.astype(np.int64)).max() <= 1
    with pytest.raises(lib.DGError):
        lib.dg_keep_thresholds(0, np.array([1.5]))


def test_argument_validation_without_gpu(lib):
    so = lib.load()
    assert so.dg_forward_noise(None, None, None, 2, 8, 16, 0, None) == lib.DG_EINVAL
    assert "NULL" in so.dg_last_error().decode()
    assert so.dg_forward_noise(None, None, None, -1, 8, 16, 0, None) == lib.DG_EINVAL
    assert so.dg_schedule_thresholds(7, 12, None, None) == lib.DG_EINVAL
    assert so.dg_schedule_thresholds(0, 0, None, None) == lib.DG_EINVAL
    assert so.dg_canvas_attn(None, None, None, None, None, None, None, 1, 100, 0, 4, 4, 64, 0,
                             0.125, None, 0, None) == lib.DG_ENOTSUP
    assert so.dg_canvas_attn(None, None, None, None, None, None, None, 1, 256, 0, 4, 4, 96, 0,
                             0.125, None, 0, None) == lib.DG_ENOTSUP
    assert so.dg_canvas_attn(None, None, None, None, None, None, None, 1, 256, 0, 6, 4, 64, 0,
                             0.125, None, 0, None) == lib.DG_EINVAL
    assert so.dg_vocab_posterior_step(None, None, 1, 256, 256, 1000, 1.0, 0, 0, None, None, None,
                                      None, None, 0, math.inf, None, None, 0, None) == lib.DG_ENOTSUP
    assert so.dg_vocab_posterior_step(None, None, 1, 256, 256, 4096, 1.0, 0, 0, None, None, None,
                                      None, None, (1 << 32) + 1, math.inf, None, None, 0,
                                      None) == lib.DG_EINVAL
    assert so.dg_euler_update(None, None, None, None, None, None, None, None, 1, 2000, 0, 0, 0,
                              0.0, None) == lib.DG_EINVAL
    m = lib.dg_model(None, None, None, 4096, 256, 4, 4, 64)
    cfg = lib.make_cfg(12, 0)
    assert so.dg_denoise_loop(ctypes.byref(m), None, None, 1, 256, 0, 0, None, None, None,
                              ctypes.byref(cfg), None, 0, None) == lib.DG_EINVAL


def test_workspace_sizes_are_host_only_and_monotone(lib):
    a = lib.dg_vocab_posterior_workspace(1, 256, 4096)
    assert a >= 256
    assert lib.dg_canvas_attn_workspace(1, 256, 1024, 16, 8, 128, 1024) >= 256


def test_argument_validation_of_the_later_rows_without_gpu(lib):
    """Self-conditioning, encode-append and block-AR generation refuse bad arguments before
    any device work."""
    so = lib.load()
    # self-conditioning: d not a multiple of 256, then NULL pointers
    assert so.dg_self_condition(None, None, None, None, 1, 256, 192, 4096, 64, 1.0, None, None,
                                None, 0, None) == lib.DG_ENOTSUP
    assert so.dg_self_condition(None, None, None, None, 1, 256, 256, 4096, 64, 1.0, None, None,
                                None, 0, None) == lib.DG_EINVAL
    assert so.dg_self_condition(None, None, None, None, 1, 256, 256, 4096, 64, 0.0, None, None,
                                None, 0, None) == lib.DG_EINVAL
    # a model that names one self-conditioning layer but not the other
    m = lib.dg_model(None, None, None, 4096, 256, 4, 4, 64, None, None, 128)
    cfg = lib.make_cfg(12, 0)
    assert so.dg_denoise_loop(ctypes.byref(m), None, None, 1, 256, 0, 0, None, None, None,
                              ctypes.byref(cfg), None, 0, None) == lib.DG_EINVAL
    # encode-append: the appended rows must fit the cache
    m = lib.dg_model(16, 16, 16, 4096, 256, 4, 4, 64, None, None, 0)
    assert so.dg_encode_append(ctypes.byref(m), None, None, None, 1, 256, 100, 300, None, None, 0,
                               None) == lib.DG_EINVAL
    # block generation: the cache must hold P0 + NB * L rows; every block runs steps 0 .. T-1
    assert so.dg_block_generate(ctypes.byref(m), None, None, 1, 64, 64 + 3 * 256 - 1, 256, 3, 0,
                                2, ctypes.byref(cfg), None, None, None, None, None, 0,
                                None) == lib.DG_EINVAL
    part = lib.make_cfg(12, 0, start_step=2)
    assert so.dg_block_generate(ctypes.byref(m), None, None, 1, 64, 64 + 3 * 256, 256, 3, 0, 2,
                                ctypes.byref(part), None, None, None, None, None, 0,
                                None) == lib.DG_ENOTSUP


def test_later_rows_workspace_sizes_are_host_only(lib):
    m = lib.dg_model(16, 16, 16, 4096, 256, 4, 4, 64, 16, 16, 128)
    B, L, V, d = 2, 256, 4096, 256
    loop = lib.dg_denoise_loop_workspace(m, B, L, 512, 0)
    plain = lib.dg_denoise_loop_workspace(lib.dg_model(16, 16, 16, 4096, 256, 4, 4, 64, None,
                                                       None, 0), B, L, 512, 0)
    # the self-conditioning buffers: at least the bf16 exponentials, B * L * V * 2 bytes
    assert loop - plain >= B * L * V * 2
    assert lib.dg_self_condition_workspace(B, L, d, V, 128) >= B * L * V * 2
    assert lib.dg_encode_append_workspace(m, B, L) >= B * L * d * 2
    one = lib.dg_block_generate_workspace(m, B, L, 512, 1, 0)
    four = lib.dg_block_generate_workspace(m, B, L, 512, 4, 0)
    assert four >= one >= loop
