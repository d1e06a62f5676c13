#!/usr/bin/env python
"""Benchmark: one Llama-7B-shaped decoder block (q, k, v, o 4096x4096; gate, up 4096x11008;
down 11008x4096; bf16), 131072 calibration tokens per site, compressed to 50% of the
block's parameters under global allocation.  One step = the whole path over one batch:
K-FAC factors of the 11 calibration sites (tcgen05 SYRK), Cholesky factors and whitening of
the 7 weights, their spectra (Gram + blocked Jacobi), global sort-and-truncate allocation,
and the rank-r factors U, V.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kfsvd|reference]
                    [--score half_sigma2|energy_ratio|empirical_fisher] [--route whitened|activation_only]

Prints one JSON line.  `value` is calibration tokens per second through the whole step with
inputs resident in HBM (17.2 GB of synthetic bf16 rows, larger than L2, so no L2 flush is
needed between steps); `e2e` is the same metric when every step also copies its inputs
from pinned host memory and reads the factors back.  --impl reference times the fp64 CPU
oracle on a bounded sample of the same workload.  Under torchrun each rank runs its own
replica of the workload (the path has no data exchange): scaling is weak, value sums ranks.
--score picks the allocation key (LASER's empirical-Fisher score adds a second pass over the
rows, timed as its own kernel entry); --route activation_only times Swift-SVD's route over
the same block (activation rows only: output covariance, one eigendecomposition per matrix,
W V_k V_k^T).  The default line is the whitened path with 1/2 sigma^2.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "calib tokens/s into K-FAC covariances; whitened-SVD layers/s; % bf16/HBM roof"
WORKLOAD = "llama7b_block: q,k,v,o 4096x4096, gate,up 4096x11008, down 11008x4096 bf16; N=131072; rho=0.5 global"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kfsvd", choices=["kfsvd", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--score", default="half_sigma2", choices=["half_sigma2", "energy_ratio", "empirical_fisher"],
                    help="allocation key: 1/2 sigma^2 (default), UniRank's energy ratio, or LASER's "
                         "empirical-Fisher score (adds a second pass over the calibration rows)")
    ap.add_argument("--route", default="whitened", choices=["whitened", "activation_only"],
                    help="whitened: the K-FAC path (default); activation_only: Swift-SVD's route "
                         "(output covariance W^T X W, one eigendecomposition, W V_k V_k^T)")
    ap.add_argument("--no-alloc-scaled", action="store_true",
                    help="skip the allocation timed at 2^28 components (its HBM roofline)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="calibration tokens per site (default: the workload's 131072); a smaller N "
                         "keeps every matrix shape and is meant for profiler captures")
    ap.add_argument("--workloads", default="all",
                    help="comma-separated extra workloads timed once each after the main line, at N=1 on "
                         "rank 0: single_linear, llama70b_block, llama7b_model, vlm; 'all' (default) or "
                         "'none'")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), "kfsvd_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), r[2:]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------- workload
def cost_tail(m, n):
    s = min(m, n)
    return m * n * s + (m ** 3 + n ** 3) / 3.0 + m * m * n + m * n * n


# DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) of one jac_apply_tc_kernel
# launch in which every task ran (7 problems of 4096, the 16384-token case, whose Jacobi shapes
# are those of every N): 728,819,968 read + 908,009,984 written, against 1,651,507,200
# algorithmic bytes for such a launch (per problem 528 C super-tiles: 64 KB read, 128 KB or
# on the diagonal 64 KB written; 2048 Qt half-panels: 32 KB read + 32 KB written).  Traffic
# grows with the tasks a launch runs, so the bench reports it per average launch as this
# ratio times the launch's algorithmic bytes.
JAC_APPLY_DRAM_PER_ALG_BYTE = (728819968 + 908009984) / 1651507200


# ALGORITHMIC bytes per component of one score_and_allocate call (a model of the minimum
# traffic, not measured DRAM bytes): sigma read (4) and key written (8); four stable radix
# passes over the score word, each reading and writing the 8-byte key (4 x 16); one read of
# the sorted keys for the cost prefix and the cut (8).
ALLOC_BYTES_PER_KEY = 12 + 4 * 16 + 8
# Measured DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum over every kernel of one
# call) per component on a 2^24-component call in units of 4096: 766,178,304 read + 437,207,040
# written.  Below the algorithmic 84 at that size because part of the written keys end in L2
# (126 MB) before the call finishes; the reads alone are 45.7 B per component.
ALLOC_DRAM_BYTES_PER_KEY_2E24 = round((766178304 + 437207040) / (1 << 24), 1)


def alloc_scaled(ctx, torch, K, hbm_peak, log2n=28, unit_len=1 << 17, reps=5):
    """score_and_allocate over 2^log2n components (units of unit_len descending values, m + n
    = 2 unit_len each, budget half of everything), timed with CUDA events on the launching
    stream after two warm-up calls.  ``achieved`` is algorithmic bytes per second."""
    n = 1 << log2n
    n_units = n // unit_len
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    sig = torch.sort(torch.rand((n_units, unit_len), generator=g, device="cuda"), dim=1, descending=True)[0]
    sig = sig.reshape(-1).contiguous()
    off = torch.arange(0, n + 1, unit_len, dtype=torch.int64, device="cuda")
    cost = torch.full((n_units,), 2 * unit_len, dtype=torch.int64, device="cuda")
    budget = int(n * 2 * unit_len // 2)
    ranks = torch.empty(n_units, dtype=torch.int32, device="cuda")
    cut = torch.empty(2, device="cuda")
    used = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = torch.empty(K.score_and_allocate_workspace_size(n, n_units), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(2):
        K.score_and_allocate(ctx, sig, off, cost, budget, ranks, cut=cut, used=used, workspace=ws, stream=st)
    ctx.sync_status()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        K.score_and_allocate(ctx, sig, off, cost, budget, ranks, cut=cut, used=used, workspace=ws, stream=st)
    e1.record(st)
    torch.cuda.synchronize()
    ctx.sync_status()
    ms = e0.elapsed_time(e1) / reps
    gbs = ALLOC_BYTES_PER_KEY * n / (ms / 1e3) / 1e9
    kept = int(ranks.sum().item())
    del sig, ws
    torch.cuda.empty_cache()
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(gbs / hbm_peak, 4), "ms": round(ms, 3), "components": n, "units": n_units,
            "kept": kept, "algorithmic_bytes_per_key": ALLOC_BYTES_PER_KEY,
            "dram_bytes_per_key_measured_at_2e24": ALLOC_DRAM_BYTES_PER_KEY_2E24,
            "peak_kind": "HBM copy, of measured"}


def fp32_peak_probe(ctx, torch, K, iters=1 << 19):
    """FP32 FMA roof of this device, measured: the library's probe kernel (every SM's FMA pipes
    busy with independent fma chains) timed with CUDA events on the launching stream; best of
    three after a warm-up launch."""
    sink = torch.zeros(8, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    K.kf_fp32_fma_probe(ctx, 1 << 12, sink, stream=st)
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(3):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        f = K.kf_fp32_fma_probe(ctx, iters, sink, stream=st)
        e1.record(st)
        torch.cuda.synchronize()
        best = max(best, f / (e0.elapsed_time(e1) / 1e3) / 1e12)
    return best


def streaming_kernels(ctx, torch, K, hbm_peak, reps=5):
    """The HBM-bound streaming steps on a VLM-sized stream (147456 tokens x 3584 bf16
    channels, 1.06 GB, larger than L2): the seeded generator's device twin (writes 2 B per
    element) and the per-token INT8 fake quantisation of quantisation-aware whitening (reads 2 B
    and writes 2 B per element), each timed with CUDA events over `reps` launches."""
    from synth import device, recipes
    wl = recipes.vlm()
    site = wl.sites["lm.b0.attn_in"]
    N, d = wl.n_tokens, site.d
    st = torch.cuda.current_stream()
    out = {}
    rows = device.stream_on_device(wl, site, 0, N, torch)
    q = torch.empty_like(rows)
    K.fake_quant_rows(ctx, rows, q, stream=st)
    torch.cuda.synchronize()
    for name, fn, nbytes in (("synthetic generator (libkfsynth, 2 B written per element)",
                              lambda: device.stream_on_device(wl, site, 0, N, torch), 2 * N * d),
                             ("fake_quant_kernel (INT8 per token, 2 B read + 2 B written per element)",
                              lambda: K.fake_quant_rows(ctx, rows, q, stream=st), 4 * N * d)):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            fn()
        e1.record(st)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(gbs / hbm_peak, 4), "ms": round(ms, 3), "elements": N * d,
                     "peak_kind": "HBM copy, of measured"}
    ctx.sync_status()
    del rows, q
    torch.cuda.empty_cache()
    return out


def run_workloads(ctx, torch, K, names, fp32_peak):
    """One end-to-end pass of each named workload through the streaming pipeline (calibration
    rows generated on the device chunk by chunk, the way a data loader feeds them; blocks one
    after another for the multi-block workloads), with wall-clock seconds, the pipeline's phase
    times from CUDA events, and the SM clocks sampled during the pass."""
    from synth import device, recipes
    from vlm_compression_fac_b300 import pipeline
    makers = {"single_linear": recipes.single_linear, "llama70b_block": recipes.llama70b_block,
              "llama7b_model": recipes.llama7b_model, "vlm": recipes.vlm}
    out = {}
    for name in names:
        wl = makers[name]()
        units = pipeline.unit_specs(wl)
        weights = device.weights_on_device(wl, torch)
        groups = None
        if len({u.block for u in wl.units}) > 1:
            groups = [[i for i, u in enumerate(wl.units) if u.block == b] for b in sorted({u.block for u in wl.units})]
        st = torch.cuda.current_stream()
        ev = []

        def mark(tag):
            e = torch.cuda.Event(enable_timing=True)
            e.record(st)
            ev.append((tag, e))

        torch.cuda.synchronize()
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        t0 = time.perf_counter()
        mark("start")
        res = pipeline.compress(ctx, units, weights, device.rows_fn(wl, torch), None, wl.n_tokens, lam=wl.lam,
                                budget=None if wl.fixed_rank is not None else wl.budget, fixed_rank=wl.fixed_rank,
                                quant=wl.quant == "int8_token", site_dims={n: s.d for n, s in wl.sites.items()},
                                act_sites=[n for n, s in wl.sites.items() if s.kind == "act"], groups=groups,
                                chunk_tokens=32768, keep_covs=False, keep_whitened=False, sync_timer=mark)
        ctx.sync_status()
        torch.cuda.synchronize()
        secs = time.perf_counter() - t0
        clk = clocks.stop()
        ph, syrk_ms, prev = {}, 0.0, ev[0][1]
        open_s = None
        for tag, e in ev[1:]:
            if tag == "syrk<":
                open_s = e
                continue
            if tag == "syrk>":
                syrk_ms += open_s.elapsed_time(e)
                continue
            ph[tag] = ph.get(tag, 0.0) + prev.elapsed_time(e)
            prev = e
        blocks = len({u.block for u in wl.units})
        svd_ms = ph.get("whiten", 0.0) + ph.get("svd", 0.0)
        out[name] = {
            "workload": "%s: %d units, N=%d per site%s, %s" % (
                wl.name, len(wl.units), wl.n_tokens, ", INT8 per-token fake-quantised activations"
                if wl.quant == "int8_token" else "", "fixed r=%d" % wl.fixed_rank if wl.fixed_rank is not None
                else "rho=%.2f global" % wl.rho),
            "seconds_end_to_end": round(secs, 3),
            "calib_tokens_per_s": round(wl.n_tokens * blocks / (ph.get("kfac", 0.0) / 1e3), 1),
            "syrk_ms": round(syrk_ms, 2),
            "layers_per_s": round(len(wl.units) / (svd_ms / 1e3), 3) if svd_ms > 0 else None,
            "phases_ms": {k: round(v, 2) for k, v in ph.items()},
            "ranks_sum": int(res.ranks.sum().item()), "used": int(res.used.item()),
            "budget": None if wl.fixed_rank is not None else int(wl.budget),
            "sweeps_max": max(u.sweeps for u in res.units), "clocks": clk,
            "inputs": "calibration rows generated on the device by the seeded generator inside the timed pass"}
        del res, weights
        torch.cuda.empty_cache()
    return out


class SitePrefetch:
    """Calibration rows for the pipeline's streamed-rows interface, copied from pinned host
    memory on a side stream one site ahead: while the compute stream accumulates a site's
    covariance, the next site's rows are already on their way (the copy engine and the
    tensor cores overlap).  ``order`` is the order in which the pipeline asks for the sites; a
    site asked for out of that order is copied when asked."""

    def __init__(self, torch, host, order, compute):
        self.torch = torch
        self.host = host
        self.order = list(order)
        self.compute = compute
        self.copy = torch.cuda.Stream()
        self.ready = {}
        self._start(0)

    def _start(self, i):
        if i >= len(self.order) or self.order[i] in self.ready:
            return
        name = self.order[i]
        with self.torch.cuda.stream(self.copy):
            t = self.host[name].to("cuda", non_blocking=True)
            ev = self.torch.cuda.Event()
            ev.record(self.copy)
        self.ready[name] = (t, ev, i)

    def __call__(self, name, t0, t1):
        if name not in self.ready:
            self.order.append(name)
            self._start(len(self.order) - 1)
        t, ev, i = self.ready.pop(name)
        self.compute.wait_event(ev)
        t.record_stream(self.compute)
        self._start(i + 1)
        return t[t0:t1]


def syrk_flops(n_tokens, d):
    return 2.0 * n_tokens * d * (d + 1) / 2.0


def run_kfsvd(args):
    import torch
    import torch.distributed as dist

    from synth import device as sdev, recipes
    from vlm_compression_fac_b300 import kfsvd as K, pipeline

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    wl = recipes.llama7b_block() if args.tokens is None else recipes.llama7b_block(n_tokens=args.tokens)
    ctx = K.Context(local)
    K.kf_svd_profile_enable(ctx, True)
    units = [pipeline.UnitSpec(u.name, u.m, u.n, u.x_site, u.g_site) for u in wl.units]
    acts = {n: sdev.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "act"}
    grads = {} if args.route == "activation_only" else \
        {n: sdev.stream_on_device(wl, s, 0, wl.n_tokens, torch) for n, s in wl.sites.items() if s.kind == "grad"}
    weights = {u.name: sdev.weight_on_device(wl, u, torch) for u in wl.units}
    torch.cuda.synchronize()
    in_bytes = sum(t.numel() * t.element_size() for t in list(acts.values()) + list(grads.values()))
    w_bytes = sum(t.numel() * t.element_size() for t in weights.values())

    stream = torch.cuda.current_stream()
    rec = []

    def mark(tag):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        rec.append((tag, e))

    swift = args.route == "activation_only"

    def run(a, g, w, timer=None):
        if swift:
            return pipeline.compress_activation_only(ctx, units, w, a, wl.n_tokens, wl.budget, sync_timer=timer)
        return pipeline.compress(ctx, units, w, a, g, wl.n_tokens, lam=wl.lam, budget=wl.budget, sync_timer=timer,
                                 score=args.score)

    def run_rows(rows, w):
        """The same step with the calibration rows from a callable (whole sites per call)."""
        dims = {n: s.d for n, s in wl.sites.items()}
        if swift:
            return pipeline.compress_activation_only(ctx, units, w, rows, wl.n_tokens, wl.budget, site_dims=dims,
                                                     chunk_tokens=wl.n_tokens)
        return pipeline.compress(ctx, units, w, rows, None, wl.n_tokens, lam=wl.lam, budget=wl.budget,
                                 score=args.score, site_dims=dims,
                                 act_sites=[n for n, s in wl.sites.items() if s.kind == "act"],
                                 chunk_tokens=wl.n_tokens)

    def one_step(a, g, w):
        return run(a, g, w, mark)

    for _ in range(args.warmup):
        rec.clear()
        res = one_step(acts, grads, weights)
    ctx.sync_status()
    torch.cuda.synchronize()

    # ---------------- timed region (device-resident inputs)
    phases = {k: 0.0 for k in (("kfac", "cov", "eig", "allocate", "factors") if swift else
                               ("kfac", "whiten", "svd", "score", "allocate", "unwhiten"))}
    syrk_ms, jac_ms, jac_flops, jac_bytes, svd_prof = 0.0, 0.0, 0.0, 0.0, None
    fisher_ms, n_fisher = 0.0, 0
    apply_ms, solve_ms, apply_launches = 0.0, 0.0, 0
    n_syrk = 0
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    l0 = K.kf_launch_count()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    per_step_marks = []
    for _ in range(args.steps):
        rec.clear()
        mark("start")
        res = one_step(acts, grads, weights)
        per_step_marks.append(list(rec))
        p = K.kf_svd_profile_read(ctx)
        jac_ms += p["jacobi_ms"]
        jac_flops += p["jacobi_apply_flops"]
        jac_bytes += p["jacobi_apply_bytes"]
        apply_ms += p["jacobi_apply_ms"]
        solve_ms += p["jacobi_solve_ms"]
        apply_launches += p["jacobi_apply_launches"]
        svd_prof = p
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    launches = K.kf_launch_count() - l0
    ctx.sync_status()
    total_ms = t0.elapsed_time(t1)
    if world > 1:
        tt = torch.tensor([total_ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    for marks in per_step_marks:
        prev = marks[0][1]
        open_syrk = open_fisher = None
        for tag, e in marks[1:]:
            if tag == "syrk<":
                open_syrk = e
                continue
            if tag == "syrk>":
                syrk_ms += open_syrk.elapsed_time(e)
                n_syrk += 1
                continue
            if tag == "fisher<":
                open_fisher = e
                continue
            if tag == "fisher>":
                fisher_ms += open_fisher.elapsed_time(e)
                n_fisher += 1
                continue
            phases[tag] += prev.elapsed_time(e)
            prev = e
    K_ = args.steps
    ms_step = total_ms / K_
    tokens = wl.n_tokens * world
    value = tokens / (ms_step / 1e3)

    # ---------------- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        h_acts = {k: v.cpu().pin_memory() for k, v in acts.items()}
        h_grads = {k: v.cpu().pin_memory() for k, v in grads.items()}
        h_w = {k: v.cpu().pin_memory() for k, v in weights.items()}
        torch.cuda.synchronize()
        out_bytes = 0
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        h_rows = dict(h_acts)
        h_rows.update(h_grads)
        order = []                  # the order in which the pipeline asks for the sites
        for u in units:
            for sn in ((u.x_site,) if swift else (u.x_site, u.g_site)):
                if sn not in order:
                    order.append(sn)
        e0.record(stream)
        for _ in range(K_):
            w = {k: v.to("cuda", non_blocking=True) for k, v in h_w.items()}
            rows = SitePrefetch(torch, h_rows, order, stream)
            r = run_rows(rows, w)
            outs = [u.U.cpu() for u in r.units] + [u.V.cpu() for u in r.units] + [r.ranks.cpu()]
            out_bytes = sum(o.numel() * o.element_size() for o in outs)
            del w, r, rows
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
        if world > 1:
            tt = torch.tensor([e2e_ms], device="cuda")
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e2e_ms = float(tt.item())
        e2e = {"value": tokens / (e2e_ms / K_ / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": in_bytes + w_bytes,
               "d2h_bytes_per_step": out_bytes}
        del h_acts, h_grads, h_w

    # ---------------- roofline of the dominant kernel
    pk = peaks() or {}
    bf16_peak = pk.get("bf16_tflops_sustained", 1400.0)
    sm_max = (clk or {}).get("sm_max_mhz") or pk.get("sm_max_mhz", 2032.0)
    n_sm = torch.cuda.get_device_properties(local).multi_processor_count
    fp32_derived = n_sm * 128 * 2 * sm_max * 1e6 / 1e12
    fp32_measured = fp32_peak_probe(ctx, torch, K)
    fp32_peak = fp32_measured
    sites = list(acts.values()) + list(grads.values())
    syrk_total_flops = sum(syrk_flops(wl.n_tokens, t.shape[1]) for t in sites) * K_
    syrk_tf = syrk_total_flops / (syrk_ms / 1e3) / 1e12 if syrk_ms > 0 else 0.0
    apply_tf = jac_flops / (apply_ms / 1e3) / 1e12 if apply_ms > 0 else 0.0
    apply_gbs = jac_bytes / (apply_ms / 1e3) / 1e9 if apply_ms > 0 else 0.0
    hbm_peak = pk.get("hbm_gbs", 6400.0)
    bf16_burst = pk.get("bf16_tflops", 1800.0)
    kern = {
        "tc_gemm_kernel (covariance SYRK)": {
            "bound": "tensor", "achieved": round(syrk_tf, 2), "peak": bf16_peak, "unit": "TFLOP/s",
            "frac": round(syrk_tf / bf16_peak, 4), "ms_per_step": round(syrk_ms / K_, 3),
            "launches_per_step": n_syrk // K_, "peak_kind": "bf16 dense, sustained, of measured"},
        "jac_apply_tc_kernel (Jacobi rotations, tcgen05)": {
            "bound": "hbm", "achieved": round(apply_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(apply_gbs / hbm_peak, 4), "ms_per_step": round(apply_ms / K_, 3),
            "launches_per_step": apply_launches // K_,
            "avg_launch_ms": round(apply_ms / max(apply_launches, 1), 4),
            "algorithmic_bytes_per_step": round(jac_bytes / K_),
            "traffic": round(JAC_APPLY_DRAM_PER_ALG_BYTE * jac_bytes / max(apply_launches, 1)),
            "tensor_tflops_executed": round(apply_tf, 2),
            "tensor_frac_of_bf16_burst": round(apply_tf / bf16_burst, 4),
            "peak_kind": "HBM copy, of measured; algorithmic bytes = C and Qt read and written once per executed "
                         "task"},
        "jac_solve_kernel (Jacobi pair problems)": {
            "bound": "latency", "ms_per_step": round(solve_ms / K_, 3),
            "launches_per_step": apply_launches // K_},
    }
    if n_fisher:
        # projections P = A U, Q = Gr V^T over every component: one bf16 activation plane times
        # the hi and lo planes of U (and of V), 2 x 2 N s (m + n) flop per unit
        f_flops = sum(4.0 * wl.n_tokens * min(u.m, u.n) * (u.m + u.n) for u in wl.units) * K_
        f_tf = f_flops / (fisher_ms / 1e3) / 1e12
        kern["empirical-Fisher pass (tc_gemm_kernel projections + fisher_reduce_kernel)"] = {
            "bound": "tensor", "achieved": round(f_tf, 2), "peak": bf16_peak, "unit": "TFLOP/s",
            "frac": round(f_tf / bf16_peak, 4), "ms_per_step": round(fisher_ms / K_, 3),
            "calls_per_step": n_fisher // K_, "peak_kind": "bf16 dense, sustained, of measured"}
    if not args.no_alloc_scaled:
        kern["score_and_allocate (2^28 components, 2048 units of 2^17)"] = alloc_scaled(ctx, torch, K,
                                                                                       pk.get("hbm_gbs", 6400.0))
        kern["score_and_allocate (2^28 components, 65536 units of 4096)"] = alloc_scaled(
            ctx, torch, K, pk.get("hbm_gbs", 6400.0), unit_len=4096)
    if rank == 0 and world == 1:
        kern.update(streaming_kernels(ctx, torch, K, pk.get("hbm_gbs", 6400.0)))
    dom = max(("tc_gemm_kernel (covariance SYRK)", syrk_ms),
              ("jac_apply_tc_kernel (Jacobi rotations, tcgen05)", apply_ms), key=lambda kv: kv[1])[0]
    roof = {k: v for k, v in kern[dom].items() if k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof["kernel"] = dom
    roof.setdefault("traffic", None)

    # ---------------- CPU baseline (oracle on a bounded sample), rank 0 only at N=1
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1 and not swift:
        cpu = oracle_sample(wl, sample_tokens=1024)
        cpu["single_linear_in_full"] = oracle_single_linear()

    # ---------------- the other workloads, one pass each (N=1, rank 0)
    wls = None
    names = [] if args.workloads == "none" else (
        ["single_linear", "llama70b_block", "llama7b_model", "vlm"] if args.workloads == "all"
        else [x for x in args.workloads.split(",") if x])
    if names and rank == 0 and world == 1:
        K.kf_svd_profile_enable(ctx, False)
        wls = run_workloads(ctx, torch, K, names, fp32_peak)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K_,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic: seeded Philox4x32-10 streams and weights generated on the device",
        "config": {"workload": WORKLOAD, "route": args.route, "score": None if swift else args.score,
                   "global_batch": wl.n_tokens * world, "seq_len": wl.n_tokens,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs (%.1f GB) larger than L2; no flush" % (in_bytes / 1e9)},
        "layers_per_s": round(len(units) * world / ((phases["cov"] + phases["eig"]) if swift else
                                                     (phases["whiten"] + phases["svd"])) * K_ * 1e3, 3),
        "kfac_tokens_per_s": round(tokens / ((phases["kfac"]) / K_ / 1e3), 1),
        "phases_ms": {k: round(v / K_, 3) for k, v in phases.items()},
        "svd_profile": svd_prof, "ranks": [int(x) for x in res.ranks.cpu().tolist()],
        "jacobi_sweeps": [int(u.sweeps) for u in res.units],
        "units_larger_than_dense": res.larger_than_dense(),
        "roofline": roof, "kernels": kern, "clocks": clk, "e2e": e2e, "gpu_launches": int(launches),
        "cpu_baseline": cpu, "fp32_peak_tflops": {"measured": round(fp32_measured, 2),
                                                  "derived": round(fp32_derived, 2), "sm_count": n_sm},
        "workloads": wls,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------- oracle arm
_SAMPLE_WEIGHTS = {}


def oracle_sample(wl, sample_tokens=1024, tail_unit="q"):
    """fp64 oracle on a bounded sample of the workload, extrapolated to one full step:
    covariance sums of `sample_tokens` rows of every site (scaled by N / sample_tokens) plus
    the per-unit tail (factors, whitening, SVD, factors U V) of one unit, scaled to all
    units by m n min(m,n) + (m^3 + n^3)/3 + m^2 n + m n^2."""
    import numpy as np
    import oracle as O
    from synth import recipes

    cores = os.cpu_count()
    t0 = time.perf_counter()
    for s in wl.sites.values():
        A = recipes.gen_stream(wl, s, 0, sample_tokens).astype(np.float64)
        O.covariance_sum(A)
    t_cov = time.perf_counter() - t0
    u = [x for x in wl.units if x.name == tail_unit][0]
    r = np.random.default_rng(0)
    t1 = time.perf_counter()
    Ax = recipes.gen_stream(wl, wl.sites[u.x_site], 0, 256).astype(np.float64)
    Ag = recipes.gen_stream(wl, wl.sites[u.g_site], 0, 256).astype(np.float64)
    t_gen = time.perf_counter() - t1
    X = O.finalize_covariance(O.covariance_sum(Ax), 256, wl.lam)
    G = O.finalize_covariance(O.covariance_sum(Ag), 256, wl.lam)
    key = (wl.name, u.name)
    if key not in _SAMPLE_WEIGHTS:   # input generation, outside the timed tail: made once per run
        _SAMPLE_WEIGHTS[key] = recipes.gen_weight(wl, u).astype(np.float64)
    W = _SAMPLE_WEIGHTS[key]
    t2 = time.perf_counter()
    Sx, Sg = O.cholesky_factors(X, G)
    Wt = O.whiten(W, Sx, Sg)
    Ut, s, Vt = O.whitened_svd(Wt)
    O.unwhiten(Sx, Sg, Ut, s, Vt, min(u.m, u.n) // 2)
    t_tail = time.perf_counter() - t2
    scale = sum(cost_tail(x.m, x.n) for x in wl.units) / cost_tail(u.m, u.n)
    est = t_cov * (wl.n_tokens / sample_tokens) + t_tail * scale
    return {"value": round(wl.n_tokens / est, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "covariance sums of %d of %d tokens on all %d sites (%.1f s, scaled by N) + factor/whiten/"
                      "SVD/unwhiten tail of unit %s (%.1f s, scaled by the tail cost model to all %d units); "
                      "extrapolated step %.1f s" % (sample_tokens, wl.n_tokens, len(wl.sites), t_cov, tail_unit,
                                                    t_tail, len(wl.units), est)}


def oracle_single_linear():
    """The fp64 oracle over the whole single 256 x 512 layer workload (2048 float32 tokens,
    rank 64), in full: no sample, no extrapolation."""
    import oracle as O
    from synth import recipes
    wl = recipes.single_linear()
    t0 = time.perf_counter()
    O.compress_workload(wl)
    secs = time.perf_counter() - t0
    return {"value": round(wl.n_tokens / secs, 1), "unit": "tokens/s", "seconds": round(secs, 3),
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": "the whole single_linear workload (256x512 float32 layer, N=2048, r=64), not extrapolated"}


def run_reference(args):
    rank, local, world = dist_env()
    if rank != 0:
        return
    from synth import recipes
    wl = recipes.llama7b_block()
    for _ in range(args.warmup):
        oracle_sample(wl, sample_tokens=64)
    t = []
    res = None
    for _ in range(args.steps):
        res = oracle_sample(wl, sample_tokens=256)
        t.append(wl.n_tokens / res["value"])
    ms = 1e3 * sum(t) / len(t)
    v = wl.n_tokens / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": wl.n_tokens, "seq_len": wl.n_tokens,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "cores": res["cores"], "kind": "oracle",
                             "sample": res["sample"]},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_kfsvd(a)
