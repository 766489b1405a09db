"""Benchmark of the canvas-denoising core on GB300.

One benchmark step = one pass of the whole hot path over one batch of synthetic canvases:
the canvas is initialised from the uniform prior with the forward-noising kernel, then
dg_denoise_loop runs all T Euler steps (embedding + QKV, canvas attention, output projection,
fused LM head / posterior / Gumbel-max / Euler update).  Metric: canvas tokens/s.step =
L x B x T / (seconds per benchmark step).

  python bench.py [--gpus N --steps K --warmup W --workload window1k --impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own canvases (no data
exchange), the timed region is bracketed by barriers, and the slowest rank's time is used.
--impl reference times the CPU oracle (on this machine's cores) on a bounded sample of the
same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "canvas tokens/sec·step (256×batch×steps/s) at 1 GB300; % of tensor/HBM roofline"
UNIT = "canvas_token_steps/s"
PROFILE_DIR = os.path.join(ROOT, "profiles")
DEFAULT_WORKLOAD = "sweep4k"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (default: 64 for sweep4k, the largest "
                         "batch of its sweep; the workload's own otherwise)")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the other configurations (window1k, batch16, long128k) that the "
                         "default run times under 'workloads'")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", default="denoise", choices=["denoise", "sft", "blockar"],
                    help="sft: one step = the SFT loss (noising at t ~ U(0,1), decoder, fused "
                         "cross-entropy) over the workload's batch of Zipf(1.1) canvases; "
                         "blockar: one step = block-AR generation of --blocks canvases after "
                         "the workload's context (denoising loops + encode-append)")
    ap.add_argument("--blocks", type=int, default=4, help="canvases per blockar step")
    ap.add_argument("--selfcond", type=int, default=0, metavar="D_SC",
                    help="denoise mode: add a self-conditioning feed-forward of width D_SC "
                         "(N(0, 0.02) weights; 1920 gives the pages' 7.8M parameters at d 2048)")
    ap.add_argument("--sampler", default="euler", choices=["euler", "eb"],
                    help="euler: the workload's Euler step; eb: entropy-bounded sampler with "
                         "annealing 0.8->0.4, gamma 0.1, stop at mean entropy 0.005, cap T")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d["bf16_tflops_sustained"], "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        # the raw samples go to DG_CLOCKS_DIR (default: the system temporary directory)
        out_dir = os.environ.get("DG_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.fh.close()
        return self.parse(self.path)

    @staticmethod
    def parse(path):
        """Median SM clock, the maximum clock, the throttle reasons seen and the median board
        power (W) of the samples in the csv file."""
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            try:
                power.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
               "reasons": sorted(reasons), "samples": len(sm)}
        if power:
            out["power_w"] = statistics.median(power)
        return out


def traffic_from_profile(kernel_file: str, workload: str):
    """DRAM bytes per launch of the kernel at the workload, from the committed ncu summary,
    if it was taken on the current source of the kernel (the summary records the kernel
    source's sha256); else None."""
    p = os.path.join(PROFILE_DIR, "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    src = os.path.join(ROOT, "discrete_diffusion_text_gb300", "csrc", kernel_file)
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    e = d.get(kernel_file, {}).get(workload)
    if not e or e.get("source_sha256") != h:
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------ oracle arm -----

class OracleSample:
    """One denoising step of one canvas of the workload by the CPU oracle: the decoder over
    the whole 256-token canvas, then the posterior over the whole vocabulary and the Euler
    step for every position.  The seeded inputs (one canvas: model and prefix drawn on the
    host) are made once; each call returns the seconds of one canvas-step, the posterior and
    the canvas it started from."""

    def __init__(self, w):
        from discrete_diffusion_text_gb300 import synth

        self.w = w
        self.m = synth.make_model(w)
        self.kp, self.vp = synth.make_prefix_kv(w, B=1)
        self.om = {k: (v.double().numpy() if hasattr(v, "double") else v)
                   for k, v in self.m.items()}
        self.okp, self.ovp = self.kp.double().numpy(), self.vp.double().numpy()

    def __call__(self, seed_shift: int = 0):
        import numpy as np

        from oracle import dgoracle as O

        w, om = self.w, self.om
        x = O.initial_canvas(1, w.L, w.V, w.seed + seed_shift)
        _, jump = O.schedule_thresholds(w.schedule, w.T)
        n = w.T - 1
        t0 = time.perf_counter()
        h, q, k, v = O.decoder_front(x, om["E"], om["Wqkv"], w.H, w.Hkv, w.hd)
        Oa, _ = O.canvas_attention(q, self.okp, self.ovp, k, v, w.window, w.hd ** -0.5)
        y = O.decoder_back(h, Oa, om["Wo"]).reshape(w.L, w.d)
        post = O.posterior(y, om["E"], w.inv_tau, w.seed + seed_shift, n, w.L)
        O.euler_update(x, post["x0hat"][None], post["top1"][None],
                       post["logp_top1"][None].astype(np.float32), np.zeros((1, w.L), np.uint8),
                       w.seed + seed_shift, n, int(jump[n]), math.inf)
        return time.perf_counter() - t0, post, x


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample_text(w) -> str:
    return (f"one canvas-step of the {w.name} workload per benchmark step (decoder over the "
            f"{w.L}-token canvas, posterior over all {w.V:,} tokens and Euler step for all "
            f"{w.L} positions), numpy float64 with threaded BLAS; the metric is per canvas-step "
            f"and extrapolates linearly to the workload's {w.B} canvases x {w.T} steps")


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    sample_step = OracleSample(w)
    for i in range(args.warmup):
        sample_step(i)
    ts = [sample_step(100 + i)[0] for i in range(args.steps)]
    sec = sum(ts) / len(ts)
    value = w.L / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1000, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.describe(), "global_batch": w.B, "seq_len": w.L,
                       "prefix": w.P, "parallelism": "cpu"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": oracle_sample_text(w)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------------- GPU arm -----

def attention_work(w):
    """Algorithmic FLOPs and prefix K/V bytes of one canvas attention launch: every canvas
    query of every head against its visible prefix keys and the whole canvas."""
    if w.window:
        vis = sum(min(w.P, max(0, w.window - 1 - i)) for i in range(w.L))  # keys k > P + i - W
        rows = min(w.P, w.window - 1)
    else:
        vis = w.P * w.L
        rows = w.P
    flops = 4.0 * w.B * w.H * w.hd * (vis + w.L * w.L)
    kv_bytes = 4.0 * w.B * rows * w.Hkv * w.hd
    return flops, kv_bytes


def measure_denoise(w, dev, steps, warmup, *, rank=0, world=1, dist=None, sc=0, eb=False,
                    e2e=True, timer_steps=None, noising=0):
    """Times `steps` benchmark steps of workload w.  One step: (with `noising` = n canvases)
    forward noising of n Zipf(1.1) clean canvases at t ~ U(0, 1), then the uniform-prior
    canvases and dg_denoise_loop over all of the sampler's steps.  Returns a dict of results."""
    import numpy as np
    import torch

    from discrete_diffusion_text_gb300 import dgcanvas as dgc
    from discrete_diffusion_text_gb300 import replicas, synth

    B = w.B
    m = synth.make_model(w, dev)
    kp, vp = synth.make_prefix_kv(w, dev)
    if sc:
        m["Wsc1"] = synth.normal_bf16((sc, w.d), 0.02, 1000 * w.seed + 6, dev)
        m["Wsc2"] = synth.normal_bf16((w.d, sc), 0.02, 1000 * w.seed + 7, dev)
    model = dgc.make_model(m["E"], m["Wqkv"], m["Wo"], w.H, w.Hkv, w.hd, m.get("Wsc1"),
                           m.get("Wsc2"))
    lock_thr = math.log(w.lock_theta) if w.lock_theta else math.inf
    lock_thr = float(np.float32(lock_thr))
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(model, B, w.L, w.P, w.window), dev)
    canvas = torch.zeros((B, w.L), dtype=torch.int32, device=dev)
    lock = torch.zeros((B, w.L), dtype=torch.uint8, device=dev)
    steps_taken = torch.zeros(B, dtype=torch.int32, device=dev)
    keep0 = torch.zeros(B, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    if noising:  # training-style noising of clean canvases (the workload's Zipf(1.1) tokens)
        x0_h = torch.tensor(synth.zipf_tokens(noising, w.L, w.V, 1.1, w.seed), dtype=torch.int32)
        t = synth.uniform_times(noising, w.seed)
        keep_h = torch.tensor(dgc.dg_keep_thresholds(synth.SCHED_LINEAR, t).astype(np.int64))
        x0_d, keep_d = x0_h.to(dev), keep_h.to(dev)
        xt_d = torch.empty_like(x0_d)

    def make_cfg(seed):
        if eb:
            return dgc.make_cfg(w.T, w.schedule, seed=seed, sampler=dgc.DG_SAMPLER_ENTROPY_BOUNDED,
                                tau_start=0.8, tau_end=0.4, gamma=0.1, stop_entropy=0.005)
        return dgc.make_cfg(w.T, w.schedule, w.inv_tau, lock_thr, seed,
                            stop_when_all_locked=w.stop_when_all_locked)

    def step(i, kpd=kp, vpd=vp, x0=None, keep=None):
        seed = replicas.replica_seed(w.seed, rank, i)
        if noising:
            dgc.dg_forward_noise(x0_d if x0 is None else x0, xt_d,
                                 keep_d if keep is None else keep, w.V, seed)
        dgc.dg_forward_noise(canvas, canvas, keep0, w.V, seed)        # x_1: uniform prior
        lock.zero_()
        dgc.dg_denoise_loop(model, kpd, vpd, w.window, canvas, lock, steps_taken, make_cfg(seed),
                            ws)

    for i in range(warmup):
        step(i)
    dgc.dg_workspace_status(ws)
    torch.cuda.synchronize()

    # ---- device-timed region (the library's kernel timer off: its events between kernels
    # would stop each kernel from being scheduled while its predecessor finishes)
    clocks = ClockSampler(int(str(dev).split(":")[-1]) if ":" in str(dev) else 0)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    dgc.dg_workspace_status(ws)
    # state of the last benchmark step's canvases
    st_last = steps_taken.cpu().numpy().astype(np.float64)
    lock_frac = float(lock.float().mean().item())
    ms = replicas.max_over_ranks(ms)
    ms_per_step = ms / steps
    denoise_steps = float(st_last.mean()) if st_last.sum() else float(w.T)
    value = replicas.job_throughput(world, w.L, B, denoise_steps, ms_per_step / 1000.0)

    res = {"value": value, "ms_per_step": ms_per_step, "clocks": clk,
           "steps_per_canvas": denoise_steps,
           "steps_per_canvas_max": float(st_last.max()) if B else 0.0,
           # tokens per forward of one canvas (no canvas is appended to a cache here, so the
           # pages' K - 1 encode term is 0) and effective denoising steps
           "tpf": w.L / denoise_steps, "eds": denoise_steps, "lock_fraction": lock_frac}

    # ---- end to end through the public API with host buffers: the prefix KV of the step's
    # requests (and the clean canvases and keep thresholds of the noising leg) go host ->
    # device; the final canvases, their step counts (and the noised canvases) come back.  The
    # inputs are double-buffered on the device: a copy stream brings step i + 1's inputs while
    # step i computes (every copy is inside the timed region; a step starts only once its own
    # inputs have landed, and a buffer is refilled only after the step that read it is done).
    if e2e:
        kp_h = kp.cpu().pin_memory()
        vp_h = vp.cpu().pin_memory()
        out_h = torch.empty((B, w.L), dtype=torch.int32).pin_memory()
        st_h = torch.empty(B, dtype=torch.int32).pin_memory()
        bufs = [(torch.empty_like(kp), torch.empty_like(vp)) for _ in range(2)]
        if noising:
            x0_hp, keep_hp = x0_h.pin_memory(), keep_h.pin_memory()
            nbufs = [(torch.empty_like(x0_d), torch.empty_like(keep_d)) for _ in range(2)]
            xt_h = torch.empty_like(x0_h).pin_memory()
        copy_stream = torch.cuda.Stream(dev)
        landed = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]

        def issue_copy(i):  # step i's inputs into buffer i % 2, on the copy stream
            k = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(consumed[k])
                bufs[k][0].copy_(kp_h, non_blocking=True)
                bufs[k][1].copy_(vp_h, non_blocking=True)
                if noising:
                    nbufs[k][0].copy_(x0_hp, non_blocking=True)
                    nbufs[k][1].copy_(keep_hp, non_blocking=True)
                landed[k].record(copy_stream)

        def e2e_run(n, first):
            copy_stream.wait_event(first)  # no copy before the region starts
            issue_copy(0)
            for i in range(n):
                if i + 1 < n:
                    issue_copy(i + 1)
                k = i % 2
                stream.wait_event(landed[k])
                step(7777 + i, bufs[k][0], bufs[k][1], nbufs[k][0] if noising else None,
                     nbufs[k][1] if noising else None)
                consumed[k].record(stream)
                out_h.copy_(canvas, non_blocking=True)
                st_h.copy_(steps_taken, non_blocking=True)
                if noising:
                    xt_h.copy_(xt_d, non_blocking=True)

        w0 = torch.cuda.Event()
        w0.record(stream)
        e2e_run(min(warmup, 3), w0)
        torch.cuda.synchronize()
        e2e_clocks = ClockSampler(int(str(dev).split(":")[-1]) if ":" in str(dev) else 0)
        e2e_clocks.start()
        if dist:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(steps, e0)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_clk = e2e_clocks.stop()
        e2e_ms = replicas.max_over_ranks(e0.elapsed_time(e1))
        e2e_steps = float(st_h.sum().item()) / B if int(st_h.sum().item()) else w.T
        h2d = kp.numel() * 2 * 2 + (x0_h.numel() * 4 + keep_h.numel() * 8 if noising else 0)
        d2h = out_h.numel() * 4 + st_h.numel() * 4 + (x0_h.numel() * 4 if noising else 0)
        res["e2e"] = {"value": replicas.job_throughput(world, w.L, B, e2e_steps,
                                                       e2e_ms / steps / 1000.0),
                      "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "clocks": e2e_clk}

    # ---- the same steps again with the kernel timer on: per-launch durations of the LM-head,
    # attention and self-conditioning kernels (CUDA events on the launching stream)
    tsteps = steps if timer_steps is None else timer_steps
    dgc.dg_kernel_timer_enable(True)
    for i in range(tsteps):
        step(warmup + steps + i)
    torch.cuda.synchronize()
    vocab_ms, vocab_n = dgc.dg_kernel_timer_read(0)
    attn_ms, attn_n = dgc.dg_kernel_timer_read(1)
    sc_ms, sc_n = dgc.dg_kernel_timer_read(2)
    dgc.dg_kernel_timer_enable(False)
    dgc.dg_workspace_status(ws)
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    flops_per_launch = 2.0 * B * w.L * w.d * w.V
    vocab_avg_s = vocab_ms / max(vocab_n, 1) / 1000.0
    achieved = flops_per_launch / vocab_avg_s / 1e12
    res["lm_head"] = {
        "kernel": "vocab_posterior_kernel (fused LM head + posterior + two-level Gumbel-max "
                  "sample)",
        "bound": "tensor", "achieved": achieved, "peak": tf_burst, "unit": "TFLOP/s",
        "frac": achieved / tf_burst, "peak_sustained": tf_sust,
        "frac_sustained": achieved / tf_sust, "peak_kind": f"{peak_kind} bf16 (burst; sustained "
                                                          f"beside)",
        "traffic": traffic_from_profile("vocab.cu", w.name),
        "launches": vocab_n, "avg_ms": vocab_avg_s * 1000.0,
        "hbm_frac": (2.0 * w.V * w.d + 2.0 * B * w.L * w.d) / vocab_avg_s / 1e9 / hbm}
    a_flops, a_bytes = attention_work(w)
    attn_avg_s = attn_ms / max(attn_n, 1) / 1000.0
    res["attention"] = {
        "kernel": "canvas_attn_kernel + attn_merge_kernel", "avg_ms": attn_avg_s * 1000.0,
        "launches": attn_n, "achieved_tflops": a_flops / attn_avg_s / 1e12 if attn_n else None,
        "frac_burst": a_flops / attn_avg_s / 1e12 / tf_burst if attn_n else None,
        "frac_sustained": a_flops / attn_avg_s / 1e12 / tf_sust if attn_n else None,
        "kv_gbs": a_bytes / attn_avg_s / 1e9 if attn_n else None,
        "hbm_frac": a_bytes / attn_avg_s / 1e9 / hbm if attn_n else None}
    if sc:  # the self-conditioning contraction p_hat E: the same FLOPs as the LM head
        sc_avg_s = sc_ms / max(sc_n, 1) / 1000.0
        res["selfcond_contraction"] = {
            "kernel": "sc_gemm_kernel", "avg_ms": sc_avg_s * 1000.0, "launches": sc_n,
            "achieved_tflops": flops_per_launch / sc_avg_s / 1e12 if sc_n else None,
            "hbm_gbs_algorithmic": (2.0 * w.V * w.d + 2.0 * B * w.L * w.V) / sc_avg_s / 1e9
            if sc_n else None}
    # the count is the Euler sampler's; the entropy-bounded sampler launches one more kernel
    # (its update) per denoising step and, without self-conditioning, keeps every step's
    # finalisation as its own launch (the Euler loop folds all but the last into the next
    # step's embedding launch)
    eb_extra = (w.T + (w.T - 1 if not sc else 0)) if eb else 0
    per_step = (1 + (1 if noising else 0) + dgc.dg_denoise_loop_kernel_count(
        model, B, w.L, w.P, w.window, int(round(denoise_steps))) + eb_extra)
    res["gpu_launches"] = steps * per_step
    del model, ws, m, kp, vp
    torch.cuda.empty_cache()
    return res


def parity_probe(w, dev, oracle: "OracleSample", seed_shift: int, result):
    """The oracle sample's canvas-step on the GPU: the same canvas, model and prefix (one
    canvas), the loop's last step (lambda = 1, so every position takes its posterior sample);
    counts positions whose sampled token differs from the oracle's and the oracle's near-ties
    (two best perturbed scores within 1e-3 at either level of the sample)."""
    import torch

    from discrete_diffusion_text_gb300 import dgcanvas as dgc

    _, post, x = result
    md = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in oracle.m.items()}
    model = dgc.make_model(md["E"], md["Wqkv"], md["Wo"], w.H, w.Hkv, w.hd)
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(model, 1, w.L, w.P, w.window), dev)
    c = torch.tensor(x, dtype=torch.int32, device=dev)
    lk = torch.zeros((1, w.L), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    n = w.T - 1
    cfg = dgc.make_cfg(w.T, w.schedule, w.inv_tau, math.inf, w.seed + seed_shift,
                       start_step=n, end_step=n + 1)
    dgc.dg_denoise_loop(model, oracle.kp.to(dev), oracle.vp.to(dev), w.window, c, lk, st, cfg,
                        ws)
    dgc.dg_workspace_status(ws)
    got = c.cpu().numpy().reshape(-1)
    diff = got != post["x0hat"]
    near = post["gap_perturbed"] < 1e-3
    del model, ws, md
    torch.cuda.empty_cache()
    return {"positions": int(w.L), "sampled_token_mismatches": int(diff.sum()),
            "mismatches_off_near_tie": int((diff & ~near).sum()),
            "oracle_near_ties": int(near.sum()),
            "near_tie_rule": "two best perturbed scores within 1e-3 at either level of the "
                             "sample (chunk scores, or perturbed logits in the chosen chunk)"}


def run_ours(args, w):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from discrete_diffusion_text_gb300 import dgcanvas as dgc
    from discrete_diffusion_text_gb300 import synth

    dgc.load()
    sc = args.selfcond
    eb = args.sampler == "eb"
    noising = w.B if w.name.startswith("sweep4k") else 0   # the sweep's noising leg

    # the other full-size configurations, same contract, fewer steps (at N = 1); the light
    # one-canvas workloads first, before the power-capped batched ones warm the GPU
    subs = {}
    if world == 1 and not args.no_sub and args.workload == DEFAULT_WORKLOAD and not sc and not eb:
        for name, k in (("window1k", args.steps), ("long128k", args.steps),
                        ("batch16", max(3, args.steps // 4))):
            sw = synth.WORKLOADS[name]
            r = measure_denoise(sw, dev, k, 3, e2e=False, timer_steps=min(k, 3))
            subs[name] = {"workload": sw.describe(), "value": r["value"], "unit": UNIT,
                          "steps": k, "warmup": 3, "ms_per_step": r["ms_per_step"],
                          "steps_per_canvas": r["steps_per_canvas"],
                          "lock_fraction": r["lock_fraction"], "clocks": r["clocks"],
                          "lm_head": r["lm_head"], "attention": r["attention"],
                          "gpu_launches": r["gpu_launches"]}

    main = measure_denoise(w, dev, args.steps, args.warmup, rank=rank, world=world, dist=dist,
                           sc=sc, eb=eb, noising=noising)

    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        oracle = OracleSample(w)
        res = oracle(0)
        cpu = {"value": w.L / res[0], "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": oracle_sample_text(w)}
        parity = parity_probe(w, dev, oracle, 0, res)

    if rank == 0:
        roofline = dict(main["lm_head"])
        roofline["attention"] = main["attention"]
        if sc:
            roofline["selfcond_contraction"] = main["selfcond_contraction"]
        line = {"metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) prefix KV, "
                                         "uniform-prior canvases"
                                         + ("; Zipf(1.1) clean canvases noised at t ~ U(0,1)"
                                            if noising else "") + ")",
                "config": {"workload": w.describe() + (
                               "; entropy-bounded sampler (tau 0.8->0.4, gamma 0.1, stop at mean "
                               "entropy 0.005, cap T)" if eb else "") + (
                               f"; self-conditioning FFW d_sc {sc}" if sc else "") + (
                               f"; each step also noises {noising} x {w.L} Zipf(1.1) clean "
                               f"tokens at t ~ U(0,1)" if noising else ""),
                           "global_batch": w.B * world, "seq_len": w.L,
                           "prefix": w.P, "denoise_steps_cap": w.T,
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                           "l2": "inputs larger than L2: the 1 GiB LM-head weight and the prefix "
                                 "KV are streamed every denoising step; no flush"},
                "clocks": main["clocks"], "e2e": main["e2e"],
                "gpu_launches": main["gpu_launches"], "roofline": roofline,
                "steps_per_canvas": main["steps_per_canvas"],
                "steps_per_canvas_max": main["steps_per_canvas_max"],
                "tpf": main["tpf"], "eds": main["eds"], "lock_fraction": main["lock_fraction"],
                "parity_probe": parity, "cpu_baseline": cpu}
        if subs:
            line["workloads"] = subs
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_sft(args, w):
    """SFT loss throughput: canvas tokens whose loss is computed per second (one bench step =
    noising + decoder + fused LM head / cross-entropy over the batch)."""
    import numpy as np
    import torch

    from discrete_diffusion_text_gb300 import dgcanvas as dgc
    from discrete_diffusion_text_gb300 import synth

    dev = torch.device("cuda", 0)
    dgc.load()
    B = w.B
    m = synth.make_model(w, dev)
    kp, vp = synth.make_prefix_kv(w, dev)
    model = dgc.make_model(m["E"], m["Wqkv"], m["Wo"], w.H, w.Hkv, w.hd)
    ws = dgc.workspace(dgc.dg_denoise_loop_workspace(model, B, w.L, w.P, w.window), dev)
    x0 = torch.tensor(synth.zipf_tokens(B, w.L, w.V, 1.1, w.seed), dtype=torch.int32, device=dev)
    t = synth.uniform_times(B, w.seed)
    keep = torch.tensor(np.floor((1.0 - t) * 2.0 ** 32).astype(np.int64), device=dev)
    xt = torch.empty_like(x0)
    loss = torch.empty((B, w.L), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        dgc.dg_sft_loss(model, kp, vp, w.window, x0, keep, w.seed + i, xt, loss, 1.0, ws)

    for i in range(args.warmup):
        step(i)
    dgc.dg_workspace_status(ws)
    clocks = ClockSampler(0)
    clocks.start()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    # kernel durations from a second pass with the library's timer on (its events between
    # kernels stop the dependent launches, so the throughput pass runs without them)
    dgc.dg_kernel_timer_enable(True)
    for i in range(args.steps):
        step(args.warmup + args.steps + i)
    torch.cuda.synchronize()
    vocab_ms, vocab_n = dgc.dg_kernel_timer_read(0)
    dgc.dg_kernel_timer_enable(False)
    dgc.dg_workspace_status(ws)
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    vocab_avg_s = vocab_ms / max(vocab_n, 1) / 1000.0
    achieved = 2.0 * B * w.L * w.d * w.V / vocab_avg_s / 1e12
    print(json.dumps({
        "metric": "SFT loss tokens/sec (noising + decoder + fused LM head cross-entropy)",
        "value": B * w.L / (ms / 1000.0), "unit": "canvas_tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (Zipf(1.1) clean canvases, t ~ U(0,1) per canvas)",
        "config": {"workload": w.describe() + "; SFT loss", "global_batch": B, "seq_len": w.L},
        "clocks": clk, "mean_loss": float(loss.mean().item()),
        "roofline": {"kernel": "vocab_posterior_kernel, cross-entropy mode", "bound": "tensor",
                     "achieved": achieved, "peak": tf_sust, "unit": "TFLOP/s",
                     "frac": achieved / tf_sust, "avg_ms": vocab_avg_s * 1000.0,
                     "peak_kind": f"{peak_kind} sustained bf16"}}), flush=True)


def run_blockar(args, w):
    """Block-AR generation throughput: generated tokens per second when one bench step is
    dg_block_generate of NB canvases (all T steps each, then encode-append) after the workload's
    context; no end-of-turn token, so every step generates B x NB x L tokens."""
    import torch

    from discrete_diffusion_text_gb300 import dgcanvas as dgc
    from discrete_diffusion_text_gb300 import synth

    dev = torch.device("cuda", 0)
    dgc.load()
    B, L, NB = w.B, w.L, args.blocks
    m = synth.make_model(w, dev)
    kctx, vctx = synth.make_prefix_kv(w, dev)
    cap = w.P + NB * L
    kc = torch.zeros((B, cap, w.Hkv, w.hd), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kc[:, :w.P] = kctx
    vc[:, :w.P] = vctx
    del kctx, vctx
    model = dgc.make_model(m["E"], m["Wqkv"], m["Wo"], w.H, w.Hkv, w.hd)
    ws = dgc.workspace(dgc.dg_block_generate_workspace(model, B, L, w.P, NB, w.window), dev)
    out = torch.empty((B, NB, L), dtype=torch.int32, device=dev)
    blocks, n_tok, steps = (torch.empty(B, dtype=torch.int32, device=dev) for _ in range(3))
    lock_logthr = math.log(w.lock_theta) if w.lock_theta else math.inf
    stream = torch.cuda.current_stream(dev)

    def step(i):
        cfg = dgc.make_cfg(w.T, w.schedule, 1.0, lock_logthr, w.seed + 1000 * i,
                           stop_when_all_locked=w.stop_when_all_locked)
        dgc.dg_block_generate(model, kc, vc, w.P, L, w.window, -1, cfg, out, blocks, n_tok, steps,
                              ws)

    for i in range(args.warmup):
        step(i)
    dgc.dg_workspace_status(ws)
    clocks = ClockSampler(0)
    clocks.start()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    tokens = int(n_tok.sum().item())
    total_steps = int(steps.sum().item())
    # kernel durations from a second pass with the library's timer on
    dgc.dg_kernel_timer_enable(True)
    for i in range(args.steps):
        step(args.warmup + args.steps + i)
    torch.cuda.synchronize()
    vocab_ms, vocab_n = dgc.dg_kernel_timer_read(0)
    attn_ms, attn_n = dgc.dg_kernel_timer_read(1)
    dgc.dg_kernel_timer_enable(False)
    dgc.dg_workspace_status(ws)
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    vocab_avg_s = vocab_ms / max(vocab_n, 1) / 1000.0
    achieved = 2.0 * B * L * w.d * w.V / vocab_avg_s / 1e12
    print(json.dumps({
        "metric": "block-AR generated tokens/sec (denoising loops + encode-append)",
        "value": tokens / (ms / 1000.0), "unit": "generated_tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (random weights, random context KV, no end-of-turn token)",
        "config": {"workload": w.describe() + f"; block-AR, {NB} canvases of {L}",
                   "global_batch": B, "seq_len": L, "blocks": NB,
                   "context": w.P, "cache_rows": cap},
        "clocks": clk,
        "tokens_per_step": tokens, "denoising_steps_per_canvas": total_steps / max(B, 1),
        "tpf": (tokens / B) / (total_steps / B + NB - 1),
        "ms_per_block": ms / NB,
        "attn_ms_per_step": attn_ms / args.steps, "vocab_ms_per_step": vocab_ms / args.steps,
        "roofline": {"kernel": "vocab_posterior_kernel", "bound": "tensor",
                     "achieved": achieved, "peak": tf_sust, "unit": "TFLOP/s",
                     "frac": achieved / tf_sust, "avg_ms": vocab_avg_s * 1000.0,
                     "peak_kind": f"{peak_kind} sustained bf16"}}), flush=True)


def main():
    args = parse()
    from discrete_diffusion_text_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    batch = args.batch or (max(synth.SWEEP_BATCHES) if args.workload == "sweep4k" else 0)
    if batch:
        w = w.with_batch(batch)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.mode == "sft":
        run_sft(args, w)
    elif args.mode == "blockar":
        run_blockar(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
