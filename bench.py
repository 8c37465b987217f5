"""Benchmark: one step = forward + backward attention over one batch.

Default workload: the GPT-2-medium-shaped causal attention (B=64, H=16,
N=1024, d=64, bf16).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

FLOP convention (FlashAttention pages; exact count of unmasked (i, j) pairs):
  forward = 4 d per visible pair (Q K^T and P V);
  "fwd+bwd" headline = 2.5 x forward (the literal reading of the metric);
  executed fwd+bwd = forward + backward (10 d per pair: S recompute, dP, dV,
  dK, dQ) = 3.5 x forward, reported beside it.
Multi-GPU: every rank runs its own full copy of the workload (independent
heads, no collective on the data path); value = all ranks' FLOPs / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd attention TFLOP/s & % of BF16 tensor peak, GPT-2-medium shape"
METRIC_FP8 = "FP8 (E4M3) attention forward TFLOP/s, quantiser included"


def visible_pairs(wl) -> int:
    """Exact number of visible (query, key) pairs summed over all heads."""
    N, T = wl.N, 128
    nb = -(-N // T)
    if wl.block_mask is not None:
        blocks = np.argwhere(wl.block_mask != 0)
    else:
        blocks = np.array([(I, J) for I in range(nb) for J in range(nb)])
    Ls = [N] * wl.B if wl.seqlens is None else [int(min(max(x, 0), N)) for x in wl.seqlens]
    total = 0
    for L in Ls:
        cnt = 0
        for I, J in blocks:
            i = np.arange(I * T, min(N, I * T + T))
            jlo, jhi = J * T, min(N, L, J * T + T)          # keys [jlo, jhi)
            if jhi <= jlo:
                continue
            if wl.causal:
                lo = np.maximum(jlo, i - wl.window + 1) if wl.window > 0 else jlo   # sliding window
                cnt += int(np.clip(np.minimum(i + 1, jhi) - lo, 0, None).sum())
            else:
                cnt += i.size * (jhi - jlo)
        total += cnt * wl.H
    return total


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.proc = None
        self.lines = []
        self.idx = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        time.sleep(0.1)
        sm, smax, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [x for x in sm if smax is None or x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "sm_mhz_min": min(loaded) if loaded else None,
                "power_w_median": statistics.median(pw) if pw else None, "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(ws, step_flops, ms_max):
    """Whole-job TFLOP/s: every one of the ws ranks did step_flops per step; the
    step time is the slowest rank's (max over ranks)."""
    return ws * step_flops / (ms_max * 1e-3) / 1e12


def is_fp8(wl) -> bool:
    return "_fp8" in wl.name


def oracle_sample(wl, budget_s, inputs=None):
    """Time the float64 oracle (as it stands) on whole heads of `wl` for ~budget_s.

    FP8 workloads time the oracle's FP8 forward (quantise one head, then the
    forward on its codes); the others time the exact forward + backward."""
    from oracle import attention as A
    from oracle import fp8 as F
    from exact_io_aware_tiled_gb300 import workloads as W
    spec = A.Spec(B=wl.B, H=wl.H, N=wl.N, d=wl.d, causal=wl.causal,
                  seqlens_k=None if wl.seqlens is None else np.asarray(wl.seqlens),
                  block_mask=None if wl.block_mask is None else wl.block_mask.astype(bool),
                  dropout_p=wl.dropout_p, seed=wl.dropout_seed, offset=wl.dropout_offset, H_kv=wl.H_kv,
                  window=wl.window)
    one = wl.with_(B=1, H=1, H_kv=None, seqlens=None if wl.seqlens is None else wl.seqlens[:1])
    inp = W.make_inputs(one) if inputs is None else inputs
    q, k, v, do = (inp[n][0, 0].float().numpy().astype(np.float64) for n in ("q", "k", "v", "do"))
    fp8 = is_fp8(wl)
    head_flops = (1.0 if fp8 else 2.5) * 4 * wl.d * visible_pairs(one)
    signs = W.rotation_signs(wl.d, wl.seed)
    t0 = time.perf_counter()
    heads = 0
    while True:
        if fp8:
            qz = [F.quantize(x[None, None], signs) for x in (q, k, v)]
            F.head_forward(spec, 0, 0, qz[0][0][0, 0], qz[0][1][0, 0], qz[1][0][0, 0], qz[1][1][0, 0],
                           qz[2][0][0, 0], qz[2][1][0, 0], signs)
        else:
            A.head_forward(spec, 0, 0, q, k, v)
            A.head_backward(spec, 0, 0, q, k, v, do)
        heads += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return heads * head_flops / dt / 1e12, heads, dt


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, wl):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample(wl, 0.0)
    vals = []
    t0 = time.perf_counter()
    heads_total = 0
    for _ in range(args.steps):
        v, heads, _ = oracle_sample(wl, 0.0)
        vals.append(v)
        heads_total += heads
    dt = time.perf_counter() - t0
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC_FP8 if is_fp8(wl) else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d, "causal": wl.causal,
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": "one (b=0,h=0) head %s per step, float64 numpy, %d heads total"
                                   % ("FP8 quantise + forward" if is_fp8(wl) else "fwd+bwd", heads_total)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gpt2_medium_causal")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--batch", type=int, default=0, help="override B (small profiling cases)")
    ap.add_argument("--soak", type=float, default=2.0, help="seconds of back-to-back steps for the per-step "
                    "distribution and the clocks under load (0: skip)")
    ap.add_argument("--cold-iters", type=int, default=50, help="steps timed one by one after a 512 MB write "
                    "(cold L2; 0: skip)")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-config table")
    ap.add_argument("--config-steps", type=int, default=20, help="timed steps per config of the table")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    from exact_io_aware_tiled_gb300 import workloads as W
    wl = W.CONFIGS[args.workload]
    if args.batch > 0:
        wl = wl.with_(B=args.batch, name=wl.name + "_B%d" % args.batch,
                      seqlens=None if wl.seqlens is None else wl.seqlens[:args.batch])
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import exact_io_aware_tiled_gb300 as fa
    fa.load()

    host = W.make_inputs(wl)
    R = Runner(wl, host, dev)
    t, kw, step = R.t, R.kw, R.step
    fp8 = R.fp8
    fwd_flops, bwd_flops = R.fwd_flops, R.bwd_flops
    step_flops_headline, step_flops_exec = R.step_flops_headline, R.step_flops_exec
    stream = torch.cuda.current_stream(dev)
    if fp8:
        kw8, signs, fp8_buf = R.kw8, R.signs, R.fp8_buf

    R.warmup(args.warmup)

    K = args.steps
    clk = ClockSampler(dev.index)
    clk.start()
    time.sleep(0.3)
    _barrier(ws)
    torch.cuda.synchronize()
    ms, fwd_ms, bwd_ms, _ = R.timed(K)
    torch.cuda.synchronize()
    _barrier(ws)
    timed_region_s = ms * K * 1e-3
    ms_max = _max_over_ranks(ms, ws, dev)
    # soak: the same step back to back for >= soak_s seconds (per-step events),
    # so that the clock sampler sees the GPU under load and the per-step
    # distribution (median, p10, p90) rests on many iterations
    soak = None
    if args.soak > 0:
        soak = R.soak(args.soak)
    clocks = clk.stop()
    cold = R.cold_l2(args.cold_iters) if args.cold_iters > 0 else None

    # end to end: pinned host inputs -> device, fwd + bwd, O, LSE and the
    # gradients back to pinned host memory, every step.  Consecutive steps
    # are pipelined the way a caller streaming batches would run them: the
    # host-to-device copy of step i+1 and the device-to-host copy of step
    # i-1 run on their own streams while step i computes (two device input
    # sets, two host output sets).
    e2e = None
    if not args.no_e2e:
        ins = ("q", "k", "v") if fp8 else ("q", "k", "v", "do")
        outs = ("o",) if fp8 else ("o", "dq", "dk", "dv")
        hp = {k: host[k].pin_memory() for k in ins}
        kv_like = lambda n: "k" if n in ("dk", "dv") else "q"
        hout = [{n: torch.empty_like(hp[kv_like(n)]).pin_memory() for n in outs}
                for _ in range(2)]
        for ho in hout:
            ho["lse"] = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32).pin_memory()
        dsets = [{k: torch.empty_like(hp[k], device=dev) for k in ins} for _ in range(2)]
        # device outputs (two sets) and workspaces allocated once: allocating
        # them per call from the caching allocator, with the copies out still
        # pending on another stream, made it fall back to cudaMalloc while the
        # host ran ahead, which could serialise the whole pipeline
        douts = [{n: torch.empty_like(hout[0][n], device=dev) for n in hout[0]} for _ in range(2)]
        p_ = fa.make_params(t["q"], k=t["k"], causal=wl.causal, window=wl.window, dropout_p=wl.dropout_p,
                            seqlens_k=kw["seqlens_k"], block_mask=kw["block_mask"])
        lib = fa.load()
        import ctypes
        ws_f = torch.empty(lib.fa_fwd_workspace_size(ctypes.byref(p_)), device=dev, dtype=torch.uint8)
        ws_b = None if fp8 else torch.empty(lib.fa_bwd_workspace_size(ctypes.byref(p_)), device=dev,
                                            dtype=torch.uint8)
        buf8 = fp8_buf if fp8 else None
        h2d = sum(v.numel() * v.element_size() for v in hp.values())
        d2h = sum(v.numel() * v.element_size() for v in hout[0].values())
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        # per-step durations of the three parts (timed loop only)
        KE = max(6, K // 2)
        tev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(KE)]
        timing = [None]

        def e2e_step(i):
            x = i % 2
            d, do_ = dsets[x], douts[x]
            te = timing[0][i] if timing[0] is not None else None
            s_in.wait_event(ev_cmp[x])          # step i-2 has finished reading this input set
            with torch.cuda.stream(s_in):
                if te: te[0].record(s_in)
                for k in d:
                    d[k].copy_(hp[k], non_blocking=True)
                if te: te[1].record(s_in)
                ev_in[x].record(s_in)
            s_cmp.wait_event(ev_in[x])
            s_cmp.wait_event(ev_out[x])         # step i-2's outputs have been copied out
            with torch.cuda.stream(s_cmp):
                if te: te[2].record(s_cmp)
                if fp8:
                    fa.fwd_fp8(d["q"], d["k"], d["v"], signs=signs, buf=buf8, out=(do_["o"], do_["lse"]),
                               workspace=ws_f, **kw8)
                else:
                    fa.fwd(d["q"], d["k"], d["v"], out=(do_["o"], do_["lse"]), workspace=ws_f, **kw)
                    fa.bwd(d["q"], d["k"], d["v"], do_["o"], d["do"], do_["lse"],
                           out=(do_["dq"], do_["dk"], do_["dv"]), workspace=ws_b, **kw)
                if te: te[3].record(s_cmp)
                ev_cmp[x].record(s_cmp)
            s_out.wait_event(ev_cmp[x])
            with torch.cuda.stream(s_out):
                if te: te[4].record(s_out)
                for n in hout[x]:
                    hout[x][n].copy_(do_[n], non_blocking=True)
                if te: te[5].record(s_out)
                ev_out[x].record(s_out)

        for i in range(4):                      # both buffer sets, twice
            e2e_step(i)
        torch.cuda.synchronize()
        _barrier(ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        timing[0] = tev
        a.record(s_in)
        for i in range(KE):
            e2e_step(i)
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_cmp)
        b.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = _max_over_ranks(a.elapsed_time(b) / KE, ws, dev)
        parts = {n: round(sum(te[j].elapsed_time(te[j + 1]) for te in tev) / KE, 3)
                 for n, j in (("h2d_ms", 0), ("compute_ms", 2), ("d2h_ms", 4))}
        e2e = {"value": replica_value(ws, step_flops_headline, e2e_ms), "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "parts_mean": parts,
               "pipelined": "H2D of step i+1 and D2H of step i-1 overlap step i's kernels; "
                            "device outputs and workspaces allocated once"}

    peaks, peak_kind = _peaks()
    # The K-step timed region lasts well under a second: its kernels run at
    # the burst clock, so their fractions are taken of the burst peak.  The
    # soak (seconds back to back, under the power cap) is compared with the
    # sustained peak.
    burst_region = timed_region_s < 1.0
    peak_name = "bf16_tflops" if burst_region else "bf16_tflops_sustained"
    peak = float(peaks[peak_name])
    peak_src = "%s %s (timed region %.3f s)" % (peak_kind, peak_name, timed_region_s)
    if fp8:     # E4M3 products: the bf16 peak x the nominal dense FP8 / BF16 ratio (4.5 / 2.25)
        peak *= 2.0
        peak_src += " x 2 (nominal fp8 / bf16 dense ratio)"
    dominant = "bwd" if bwd_ms >= fwd_ms else "fwd"
    kern_ms = bwd_ms if dominant == "bwd" else fwd_ms
    kern_flops = bwd_flops if dominant == "bwd" else fwd_flops
    achieved = kern_flops / (kern_ms * 1e-3) / 1e12
    kern_name = ("attn_%s_tc" % dominant) if not fp8 else "attn_fwd_fp8"
    traffic = _recorded_traffic(wl.name, "fwd_fp8" if fp8 else dominant)
    if soak is not None:
        sus = float(peaks["bf16_tflops_sustained"]) * (2.0 if fp8 else 1.0)
        soak["fwd_frac_of_sustained"] = fwd_flops / (soak["fwd_ms"]["median"] * 1e-3) / 1e12 / sus
        if not fp8:
            soak["bwd_frac_of_sustained"] = bwd_flops / (soak["bwd_ms"]["median"] * 1e-3) / 1e12 / sus
        soak["value_median"] = replica_value(ws, step_flops_headline, soak["step_ms"]["median"])

    per_config = None
    if ws == 1 and not args.no_per_config:
        per_config = {}
        for name in PER_CONFIG:
            if name == wl.name:
                rr = R
            else:
                rr = Runner(W.CONFIGS[name], W.make_inputs(W.CONFIGS[name]), dev)
                rr.warmup(3)
            m, f, b_, _ = rr.timed(args.config_steps)
            per_config[name] = rr.summary(m, f, b_, peaks, args.config_steps)
            if rr is not R:
                rr.release()
            del rr
            torch.cuda.empty_cache()

    if rank != 0:
        return
    cpu = None
    if ws == 1 and args.cpu_budget > 0:
        v, heads, dt = oracle_sample(wl, args.cpu_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
               "sample": "%d whole (b=0,h=0) heads %s in %.1f s, float64 numpy"
                         % (heads, "FP8 quantise + forward" if fp8 else "fwd+bwd", dt)}
    value = replica_value(ws, step_flops_headline, ms_max)
    line = {
        "metric": METRIC_FP8 if fp8 else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 (from %s inputs)" % wl.dtype if fp8 else wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "H_kv": wl.hkv, "N": wl.N, "d": wl.d,
                   "causal": wl.causal, "window": wl.window,
                   "dropout_p": wl.dropout_p, "parallelism": "replicas" if ws > 1 else "single",
                   "l2": "inputs exceed L2 (%.0f MB per step); cold-L2 run separately" %
                         (sum(v.numel() * v.element_size() for v in host.values()) / 1e6)},
        "pct_of_bf16_peak": 100.0 * value / float(peaks[peak_name]) / ws,
        "value_executed_flops": replica_value(ws, step_flops_exec, ms_max),
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "roofline": {"kernel": kern_name, "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_src},
        "roofline_fwd": {"achieved": fwd_flops / (fwd_ms * 1e-3) / 1e12, "peak": peak,
                         "frac": fwd_flops / (fwd_ms * 1e-3) / 1e12 / peak},
        "clocks": clocks,
        "soak": soak,
        "cold_l2": cold,
        "per_config": per_config,
        "gpu_launches": _launches_per_step(wl) * K,
        "cpu_baseline": cpu,
        "e2e": e2e,
    }
    print(json.dumps(line, default=_json_default), flush=True)


def _json_default(o):
    """numpy scalars (e.g. the pair counts) as plain numbers."""
    if hasattr(o, "item"):
        return o.item()
    raise TypeError("not JSON serialisable: %r" % (o,))


# The five workloads the per-config table covers (one line each in the JSON
# object ``per_config``).
PER_CONFIG = ("tiny_f32", "gpt2_medium_causal", "bert_large_pad_dropout", "long_ragged_causal_f16",
              "butterfly_sparse_64k")


def _pct(xs, q):
    xs = sorted(xs)
    if not xs:
        return None
    k = (len(xs) - 1) * q
    lo = int(k)
    hi = min(lo + 1, len(xs) - 1)
    return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)


def _dist_stats(xs):
    return {"median": _pct(xs, 0.5), "p10": _pct(xs, 0.1), "p90": _pct(xs, 0.9), "n": len(xs)}


class Runner:
    """One workload resident on the device and its fwd(+bwd) step."""

    def __init__(self, wl, host, dev):
        import torch
        import exact_io_aware_tiled_gb300 as fa
        from exact_io_aware_tiled_gb300 import workloads as W
        self.torch, self.fa, self.wl, self.dev = torch, fa, wl, dev
        self.t = {k: v.to(dev) for k, v in host.items()}
        self.kw = dict(causal=wl.causal, dropout_p=wl.dropout_p, seed=wl.dropout_seed, offset=wl.dropout_offset,
                       window=wl.window,
                       seqlens_k=None if wl.seqlens is None else
                       torch.from_numpy(np.asarray(wl.seqlens, np.int32)).to(dev),
                       block_mask=None if wl.block_mask is None else
                       torch.from_numpy(wl.block_mask.astype(np.uint8)).to(dev))
        self.pairs = visible_pairs(wl)
        self.fp8 = is_fp8(wl)
        self.fwd_flops = 4.0 * wl.d * self.pairs
        self.bwd_flops = 0.0 if self.fp8 else 10.0 * wl.d * self.pairs
        # FP8 workloads are forward only (quantise + forward): their step counts the forward FLOPs
        self.step_flops_headline = self.fwd_flops if self.fp8 else 2.5 * self.fwd_flops
        self.step_flops_exec = self.fwd_flops + self.bwd_flops
        self.stream = torch.cuda.current_stream(dev)
        if self.fp8:
            self.kw8 = {k_: v_ for k_, v_ in self.kw.items() if k_ not in ("dropout_p", "seed", "offset")}
            self.signs = torch.from_numpy(W.rotation_signs(wl.d, wl.seed)).to(dev)
            self.fp8_buf = torch.empty(fa.fp8_layout(fa.make_params(self.t["q"], k=self.t["k"]))["total"],
                                       device=dev, dtype=torch.uint8)

    def step(self, prof_f=None, prof_b=None, src=None):
        fa, src = self.fa, (self.t if src is None else src)
        if self.fp8:
            o, lse = fa.fwd_fp8(src["q"], src["k"], src["v"], signs=self.signs, prof=prof_f, buf=self.fp8_buf,
                                **self.kw8)
            return o, lse, None
        o, lse = fa.fwd(src["q"], src["k"], src["v"], prof=prof_f, **self.kw)
        dq, dk, dv = fa.bwd(src["q"], src["k"], src["v"], o, src["do"], lse, prof=prof_b, **self.kw)
        return o, lse, dq

    def check_status(self, when):
        """Exit if the last forward / backward left an error in its status word."""
        fa = self.fa
        st_f = fa.check_status(fa.fwd_fp8.last_workspace if self.fp8 else fa.fwd.last_workspace)
        st_b = 0 if self.fp8 else fa.check_status(fa.bwd.last_workspace)
        if st_f or st_b:
            raise SystemExit("device status after %s (%s): fwd %d bwd %d" % (when, self.wl.name, st_f, st_b))

    def warmup(self, n):
        for _ in range(n):
            self.step()
        self.torch.cuda.synchronize()
        self.check_status("warm-up")

    def _events(self, n):
        torch = self.torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for e in ev:            # materialise the events so their handles can be passed down
            for x in e:
                x.record(self.stream)
        torch.cuda.synchronize()
        return ev

    def timed(self, K, ev=None, between=None):
        """K steps back to back (or with ``between()`` before each, untimed):
        mean step ms over the whole region, mean fwd / bwd kernel ms, and the
        per-step kernel times.  Events inside the calls bracket the main
        kernels on the launching stream."""
        torch = self.torch
        ev = self._events(K) if ev is None else ev
        steps = []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if between is None:
            e0.record(self.stream)
            for s in range(K):
                self.step((ev[s][0].cuda_event, ev[s][1].cuda_event), (ev[s][2].cuda_event, ev[s][3].cuda_event))
            e1.record(self.stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / K
        else:
            marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
            for s in range(K):
                between()
                marks[s][0].record(self.stream)
                self.step((ev[s][0].cuda_event, ev[s][1].cuda_event), (ev[s][2].cuda_event, ev[s][3].cuda_event))
                marks[s][1].record(self.stream)
            torch.cuda.synchronize()
            steps = [a.elapsed_time(b) for a, b in marks]
            ms = sum(steps) / K
        self.check_status("the timed steps")
        fw = [e[0].elapsed_time(e[1]) for e in ev[:K]]
        bw = [0.0 if self.fp8 else e[2].elapsed_time(e[3]) for e in ev[:K]]
        return ms, sum(fw) / K, sum(bw) / K, dict(step=steps, fwd=fw, bwd=bw)

    def soak(self, seconds, chunk=50, max_steps=5000):
        """Steps back to back for about ``seconds``; per-step distributions."""
        torch = self.torch
        ev = self._events(chunk)
        step_ms, fw, bw = [], [], []
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < seconds and n < max_steps:
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(chunk + 1)]
            marks[0].record(self.stream)
            for s in range(chunk):
                self.step((ev[s][0].cuda_event, ev[s][1].cuda_event), (ev[s][2].cuda_event, ev[s][3].cuda_event))
                marks[s + 1].record(self.stream)
            torch.cuda.synchronize()
            step_ms += [marks[s].elapsed_time(marks[s + 1]) for s in range(chunk)]
            fw += [e[0].elapsed_time(e[1]) for e in ev]
            bw += [0.0 if self.fp8 else e[2].elapsed_time(e[3]) for e in ev]
            n += chunk
        out = {"seconds": round(time.perf_counter() - t0, 3), "step_ms": _dist_stats(step_ms),
               "fwd_ms": _dist_stats(fw)}
        if not self.fp8:
            out["bwd_ms"] = _dist_stats(bw)
        return out

    def cold_l2(self, iters, scratch_mb=512):
        """Each step preceded (untimed) by a write of a buffer four times the
        L2, so the step starts with none of its inputs in L2."""
        torch = self.torch
        buf = torch.empty(scratch_mb << 20, dtype=torch.uint8, device=self.dev)
        flip = [0]

        def between():
            flip[0] ^= 1
            buf.fill_(flip[0])

        ms, f, b_, per = self.timed(iters, between=between)
        del buf
        out = {"scratch_mb_between_steps": scratch_mb, "step_ms": _dist_stats(per["step"]),
               "fwd_ms": _dist_stats(per["fwd"])}
        if not self.fp8:
            out["bwd_ms"] = _dist_stats(per["bwd"])
        out["value_median"] = self.step_flops_headline / (out["step_ms"]["median"] * 1e-3) / 1e12
        return out

    def summary(self, ms, fwd_ms, bwd_ms, peaks, K):
        burst = float(peaks["bf16_tflops"])
        wl = self.wl
        out = {"shape": "B%d H%d%s N%d d%d %s%s%s%s%s" % (
            wl.B, wl.H, "" if wl.hkv == wl.H else " H_kv%d" % wl.hkv, wl.N, wl.d, wl.dtype,
            " causal" if wl.causal else "", " window%d" % wl.window if wl.window else "",
            " padding" if wl.seqlens is not None else "", " butterfly" if wl.block_mask is not None else "")
            + (" dropout%.2g" % wl.dropout_p if wl.dropout_p else ""),
            "steps": K, "ms": ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "tflops_literal": self.step_flops_headline / (ms * 1e-3) / 1e12,
            "tflops_executed": self.step_flops_exec / (ms * 1e-3) / 1e12,
            "visible_pairs": int(self.pairs)}
        if wl.dtype == "f32":
            out["note"] = "float32 path on CUDA cores (FFMA); no tensor-core fraction"
        else:
            out["fwd_frac_of_burst"] = self.fwd_flops / (fwd_ms * 1e-3) / 1e12 / burst
            out["bwd_frac_of_burst"] = self.bwd_flops / (bwd_ms * 1e-3) / 1e12 / burst
        return out

    def release(self):
        self.t = None


def _launches_per_step(wl):
    # fwd: [block lists] + attention; bwd: [block lists] + prep + attention + dq convert (16-bit)
    # FP8: quantiser (one pass with block scales) + [block lists] + attention
    sparse = 1 if wl.block_mask is not None else 0
    if is_fp8(wl):
        return 1 + sparse + 1
    fwd = sparse + 1
    bwd = sparse + 2 + (0 if wl.dtype == "f32" else 1)
    return fwd + bwd


def _source_hash(which):
    import hashlib
    m = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_io_aware_tiled_gb300", "csrc")
    if which == "fwd_fp8":
        files = ["fwd_fp8.cu", "fp8.cuh", "fwd_plan.cuh", "common.cuh"]
    elif which == "fwd":
        files = ["fwd_tc.cu", "fwd_tc1.cu", "fwd_plan.cuh", "common.cuh"]
    else:
        files = ["bwd_tc.cu", "common.cuh", "bwd_items.cuh"]
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            m.update(fh.read())
    return m.hexdigest()[:16]


def _recorded_traffic(workload, which):
    """DRAM bytes per launch recorded from an ncu capture (profiles/traffic.json), or None
    when there is none for this workload or the kernel sources changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(workload, {})
    if which not in rec or rec.get("source_sha256", {}).get(which) != _source_hash(which):
        return None
    return rec[which]


if __name__ == "__main__":
    main()
