"""Oracle trajectories of the denoising loop for the GPU parity tests (test helper).

The trajectory runs the oracle's own steps (decoder, posterior, Euler step with locking) and
records, per step, which positions an arithmetic difference far below the parity tolerances
could still decide differently: a position that jumps to its posterior sample whose two best
perturbed scores are within 1e-3 (the sample's near-tie), and an unlocked position whose
top-1 log-probability is within 2e-3 of the lock threshold.
"""

from __future__ import annotations

import numpy as np

from oracle import dgoracle as O

GUMBEL_TIE = 1e-3
LOCK_TIE = 2e-3


def trajectory(om, k_pre, v_pre, window, x, lock, T, schedule, inv_tau, lock_logthr, seed,
               stop_when_all_locked=False, start=0, end=None):
    """Steps start .. end-1 of the loop from (x, lock).  Returns the list of states
    [(x_n, lock_n, active_n, steps_n)] for n = start .. end, and per step the boolean [B, L]
    mask of positions whose decision is a near-tie."""
    x = np.asarray(x, np.int64).copy()
    lock = np.asarray(lock, np.uint8).copy()
    B, L = x.shape
    _, jump_thr = O.schedule_thresholds(schedule, T)
    end = T if end is None else end
    active = np.ones(B, bool)
    if stop_when_all_locked:
        active &= ~lock.astype(bool).all(axis=1)
    steps = np.zeros(B, np.int64)
    states = [(x.copy(), lock.copy(), active.copy(), steps.copy())]
    ties = []
    for n in range(start, end):
        x_new, lock_new, jump, done, post = O.denoise_step(
            om, k_pre, v_pre, window, x, lock, n, int(jump_thr[n]), inv_tau, lock_logthr, seed)
        was_locked = lock.astype(bool)
        sample_tie = (post["gap_perturbed"] < GUMBEL_TIE).reshape(B, L) & jump.astype(bool)
        lock_tie = ~was_locked & (np.abs(post["logp_top1"].reshape(B, L) - lock_logthr)
                                  < LOCK_TIE)
        ties.append((sample_tie | lock_tie) & active[:, None])
        x[active] = x_new[active]
        lock[active] = lock_new[active]
        steps[active] += 1
        if stop_when_all_locked:
            active &= ~done.astype(bool)
        states.append((x.copy(), lock.copy(), active.copy(), steps.copy()))
    return states, ties
