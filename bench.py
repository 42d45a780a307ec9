"""Benchmark of one fused SSD round (verify + fan-out cache build + lookup) on GB300.

Workload: B=256 sequences, K=4 drafted tokens, V=128256, bf16 logits, half the
sequences greedy (tau=0) and half sampled (tau=1), cache budget 32 with the
geometric fan-out a_p=0.75, r=0.5 -- the largest of the five synthetic
workloads.  A step is one ssd_round call over the whole batch; the metric is
verified speculation rounds per second (whole job), with the achieved HBM
bandwidth of the kernel against the measured copy bandwidth.

Arms:
  (default)          libssd through its Python binding (C ABI, CUDA kernels)
  --impl reference   the float64 CPU oracle on the host cores (the only other
                     implementation of this path; there is no upstream code)

Multi-GPU (torchrun): every rank runs its own batch of 256 sequences (weak
scaling, no collective on the data path); a barrier and a max over ranks
bracket the timed region.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = "c5"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--workloads", default="c1,c2,c3,c4",
                    help="further workloads timed after the headline one (one GPU only), "
                         "comma-separated, or 'none'")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (greedy share scaled); for profiling")
    ap.add_argument("--two-pass-sigma", action="store_true",
                    help="workloads with a sigma_{F,C} draft: find the descriptors in a separate "
                         "pass (ssd_reshape_draft) before ssd_verify instead of in the same pass")
    ap.add_argument("--study", choices=["fanout", "csweep"], default=None,
                    help="fanout: cache hit rate of the geometric and the uniform fan-out at "
                         "several temperatures, with the batch all-hit rate p_hit^b; "
                         "csweep: draft-only cache keys with sigma_{F_k,C} drafting, hit rate "
                         "and acceptance as C goes from 1 to 0")
    ap.add_argument("--study-draws", type=int, default=4,
                    help="independent draft-token draws per temperature (study mode)")
    ap.add_argument("--study-rounds", type=int, default=64,
                    help="rounds with fresh uniforms per draft-token draw (study mode)")
    return ap.parse_args()


def chosen_workload(args):
    wl = synth.WORKLOADS[args.workload]
    if args.batch:
        g = wl.greedy_first * args.batch // wl.B if wl.greedy_first else 0
        wl = wl.replace(B=args.batch, greedy_first=g)
    return wl


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(name: str, rank: int) -> int:
    """Seed of a rank's batch: every rank draws its own batch of the workload (weak
    scaling: the same per-GPU work on every rank, no data shared between ranks)."""
    return synth.BENCH_SEED[name] + rank


def max_over_ranks(x: float, pg, device) -> float:
    """The slowest rank's value (a timed region bracketed by barriers ends when the
    slowest rank does)."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world: int, elapsed_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the (max-over-ranks) time."""
    return world * units_per_rank / (elapsed_ms * 1e-3)


def kernel_label(kind: str, wl) -> str:
    tag = "F32Tag" if wl.dtype == synth.F32 else "BF16Tag"
    return {"stream": f"ssd_stream_kernel<{tag}>", "cluster": f"ssd_unit_kernel<{tag}>",
            "reshape+cluster": f"ssd_reshape_kernel<{tag}> + ssd_unit_kernel<{tag}>"}.get(kind, kind)


def workload_config(wl) -> dict:
    return {"workload": f"{wl.name}: {wl.description}", "B": wl.B, "K": wl.K, "V": wl.V,
            "logits": wl.dtype, "mode": wl.mode, "greedy_sequences": min(wl.greedy_first, wl.B),
            "budget": wl.budget, "a_p": wl.a_p, "r": wl.r,
            "l2": "inputs larger than L2 (logits %.0f MB vs 129 MB L2), no flush" %
                  ((wl.B * (2 * wl.K + 1) * wl.V * wl.elem_bytes) / 1e6)}


def metric_name():
    return "verified speculation rounds/sec (HBM GB/s vs measured copy bandwidth)"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# Clock sampling (nvidia-smi, during the timed region).
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for (t, r) in self.rows if t0 <= t <= t1]
        window = "timed"
        if not inside:
            inside = [r for (_, r) in self.rows]
            window = "run"
        mhz, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(mhz), "window": window}


# ---------------------------------------------------------------------------
# Our arm.
# ---------------------------------------------------------------------------
def to_device(inp, torch, dev):
    wl = inp["workload"]

    def logits(a):
        if wl.dtype == synth.F32:
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    return {"tgt": logits(inp["tgt"]), "drf": logits(inp["drf"]),
            "tokens": torch.from_numpy(inp["tokens"]).to(dev),
            "uniforms": torch.from_numpy(inp["uniforms"]).to(dev),
            "temperature": torch.from_numpy(inp["temperature"]).to(dev)}


def traffic_record(kernel_digest: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken of this build."""
    path = os.path.join(ROOT, "profiles", "ssd_stream_kernel_c5_traffic.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    if d.get("source_digest") != kernel_digest:
        return None
    return d.get("dram_bytes_per_launch")


def cpu_baseline(inp, wl, off, sample_per_half: int = 128):
    import oracle
    B = wl.B
    g = min(wl.greedy_first, B)
    idx = np.concatenate([np.arange(0, min(g, sample_per_half)),
                          np.arange(g, min(B, g + sample_per_half))])
    sub = {k: inp[k][idx] for k in ("tgt", "drf", "tokens", "uniforms", "temperature")}
    threads = oracle.default_threads()
    reps = 0
    t0 = time.perf_counter()
    while True:  # repeat the sample until about 10 s of host time (at most 30 rounds)
        oracle.round_(sub["tgt"], sub["drf"], sub["tokens"], sub["uniforms"], sub["temperature"],
                      wl.dtype, off, wl.budget, threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 10.0 or reps >= 30:
            break
    rounds = reps * len(idx) / B
    return {"value": rounds / dt, "unit": "rounds/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(idx)} of {B} sequences of one round ({len(idx)//2} greedy, "
                      f"{len(idx) - len(idx)//2} sampled) x {reps} repetitions, float64 C oracle, "
                      f"{threads} host threads; {dt:.2f} s wall"}


def prepare(wl, seed: int, ssd, torch, dev, two_pass_sigma: bool = False) -> dict:
    """Inputs of one workload on the device and its step (one call of the path over
    the whole batch).  Workloads with a sigma_{F,C} draft redraw their drafted tokens
    from sigma_{F,C} on the device (input synthesis, not a step of the method)."""
    inp = synth.make_inputs(wl, seed)
    F, off = ssd.ssd_fanout(wl.K, max(wl.budget, 0), wl.a_p or 0.5, wl.r, wl.V) if wl.budget else (
        np.zeros(wl.K + 1, np.int32), np.zeros(wl.K + 2, np.int32))
    d = to_device(inp, torch, dev)
    ws = ssd.workspace(wl.B, wl.K, dev)
    stream = torch.cuda.current_stream(dev)
    sig = wl.reshape_F > 0
    sig_F = [wl.reshape_F] * wl.K
    desc = torch.zeros((wl.B * wl.K, 4), dtype=torch.int32, device=dev)
    if sig:
        ssd.ssd_reshape_draft(d["drf"], wl.reshape_F, wl.reshape_C, desc=desc)
        thr_val, thr_id, _, _ = ssd.desc_fields(desc)
        zd = d["drf"].float()
        ids = torch.arange(wl.V, device=dev).view(1, 1, wl.V)
        mem = (zd > thr_val.view(wl.B, wl.K, 1)) | ((zd == thr_val.view(wl.B, wl.K, 1)) &
                                                     (ids <= thr_id.view(wl.B, wl.K, 1)))
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed + 7)
        gum = -torch.log(-torch.log(torch.rand(zd.shape, generator=gen, device=dev).clamp_min(1e-30)))
        tau = d["temperature"].view(wl.B, 1, 1)
        score = zd / tau.clamp_min(1e-30) + mem.float() * float(np.log(wl.reshape_C)) + gum
        d["tokens"] = torch.where(tau.view(wl.B, 1) > 0, torch.argmax(score, dim=-1),
                                  torch.argmax(zd, dim=-1)).to(torch.int32).contiguous()
        del zd, mem, gum, score
    box = {"out": None}

    def step():
        out = box["out"]
        if wl.mode == "round":
            r = ssd.ssd_round(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"], F,
                              wl.budget, out=out, probs=False, workspace=ws, stream=stream)
        elif sig and two_pass_sigma:
            ssd.ssd_reshape_draft(d["drf"], wl.reshape_F, wl.reshape_C, desc=desc, stream=stream)
            r = ssd.ssd_verify(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"],
                               reshape=desc, probs=False, workspace=ws, stream=stream)
        elif sig:
            r = ssd.ssd_verify_sigma(d["tgt"], d["drf"], d["tokens"], d["uniforms"],
                                     d["temperature"], sig_F, wl.reshape_C, desc_out=desc,
                                     probs=False, workspace=ws, stream=stream)
        else:
            r = ssd.ssd_verify(d["tgt"], d["drf"], d["tokens"], d["uniforms"], d["temperature"],
                               probs=False, workspace=ws, stream=stream)
        box["out"] = r if wl.mode == "round" else None
        return r

    return {"wl": wl, "inp": inp, "F": F, "off": off, "d": d, "ws": ws, "stream": stream,
            "sig": sig, "sig_F": sig_F, "desc": desc, "step": step,
            "launches_per_step": 2 if (sig and two_pass_sigma) else 1}


def back_to_back_ms(step, stream, torch, dev, n: int) -> float:
    """Device time of n launches issued back to back (CUDA events on the launching
    stream around them, none between: the streaming kernel may start while the
    previous launch drains)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b)


def isolated_ms(step, stream, torch, dev, n: int) -> list:
    """Per-launch device time with an event on each side of every launch."""
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize(dev)
    return [x.elapsed_time(y) for x, y in zip(ev0, ev1)]


def measure_workload(name: str, ssd, torch, dev, peak: float) -> dict:
    """One line per further workload: the whole path over its batch, timed with CUDA
    events over back-to-back launches (at least 200; 2000 for the single-sequence
    one), isolated launch times, algorithmic bytes from the actual accepted lengths
    and the fraction of the measured copy bandwidth."""
    wl = synth.WORKLOADS[name]
    pr = prepare(wl, synth.BENCH_SEED[name], ssd, torch, dev)
    out = pr["step"]()
    torch.cuda.synchronize(dev)
    kernel = ssd.ssd_last_kernel()
    acc = out["accept_len"].cpu().numpy()
    tau = pr["inp"]["temperature"]
    alg = synth.algorithmic_bytes(wl, tau, acc)
    # a sigma draft: the bytes of the rows the verification needs (the pass finds each
    # row's descriptor while it reads it; rows after the first rejection are not needed)
    rows_bytes = synth.algorithmic_bytes(wl.replace(reshape_F=0), tau, acc)
    n = 2000 if wl.B == 1 else 300
    for _ in range(20):
        pr["step"]()
    ms = back_to_back_ms(pr["step"], pr["stream"], torch, dev, n) / n
    iso = isolated_ms(pr["step"], pr["stream"], torch, dev, 200)
    basis = rows_bytes if pr["sig"] else alg
    achieved = basis / (ms * 1e-3) / 1e9
    entry = {
        "workload": f"{wl.name}: {wl.description}", "B": wl.B, "K": wl.K, "V": wl.V,
        "logits": wl.dtype, "call": ("ssd_round" if wl.mode == "round" else
                                     "ssd_verify_sigma" if pr["sig"] else "ssd_verify"),
        "kernel": kernel, "launches_timed": n,
        "us_per_round": ms * 1e3, "rounds_per_s": 1e3 / ms, "sequence_rounds_per_s": wl.B * 1e3 / ms,
        "isolated_us": {"mean": statistics.mean(iso) * 1e3, "p10": float(np.percentile(iso, 10)) * 1e3,
                        "p90": float(np.percentile(iso, 90)) * 1e3},
        "algorithmic_bytes_per_round": alg,
        "hbm_gbs": achieved, "frac": achieved / peak,
        "accept_mean": float(np.mean(acc[acc >= 0])) if (acc >= 0).any() else None,
    }
    if pr["sig"]:
        entry["bytes_basis"] = ("rows the verification reads (2(a+1) rows per sequence below a "
                                "full accept); algorithmic_bytes_per_round adds the separate "
                                "reshape pass over every draft row")
        entry["verify_row_bytes_per_round"] = rows_bytes
    if wl.mode == "round":
        entry["hit_rate"] = float(out["hit"].float().mean().item())
    del pr, out
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    import speculative_decoding_verification_ssd_gb300 as ssd
    from speculative_decoding_verification_ssd_gb300 import _build

    wl = chosen_workload(args)
    pr = prepare(wl, rank_seed(wl.name, rank), ssd, torch, dev, args.two_pass_sigma)
    inp, F, off, d, ws, stream = pr["inp"], pr["F"], pr["off"], pr["d"], pr["ws"], pr["stream"]
    sig, sig_F, desc, step = pr["sig"], pr["sig_F"], pr["desc"], pr["step"]
    launches_per_step = pr["launches_per_step"]

    out = step()
    torch.cuda.synchronize(dev)
    acc = out["accept_len"].cpu().numpy()
    alg_bytes = synth.algorithmic_bytes(wl, inp["temperature"], acc)
    if sig and not args.two_pass_sigma:
        # descriptors found while the rows are read: the bytes are the rows verification needs
        alg_bytes = synth.algorithmic_bytes(wl.replace(reshape_F=0), inp["temperature"], acc)
    dense_bytes = wl.B * (2 * wl.K + 1) * wl.V * wl.elem_bytes

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    # launches back to back (no event between them: the streaming kernel may start
    # while the previous one drains)
    start.record(stream)
    for i in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if pg:
        pg.barrier()
    time.sleep(0.05)
    sampler.stop()
    elapsed_ms = max_over_ranks(start.elapsed_time(end), pg, dev)
    clocks = sampler.summary(t_wall0, t_wall1)
    # isolated launch durations (an event on each side of every launch), after the timed region
    n_iso = min(args.steps, 200)
    kernel_ms = isolated_ms(step, stream, torch, dev, n_iso)
    kernel_name = ssd.ssd_last_kernel()

    # end to end: pinned host inputs -> device, round, outputs -> host, every step
    host = {k: v.cpu().pin_memory() for k, v in d.items()}
    res_keys = ["accept_len", "bonus"] + (["cache_tok", "hit", "slot"] if wl.mode == "round" else [])
    host_out = {k: torch.empty(out[k].shape, dtype=out[k].dtype).pin_memory() for k in res_keys}
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    if wl.mode == "round":
        # the library's host-buffer round: it copies the target logits and only the
        # sampled sequences' draft rows, runs the round and copies the results back
        staging = torch.empty(ssd.ssd_host_staging_size(ssd._logit_dtype(d["tgt"]), wl.B, wl.K, wl.V,
                                                        wl.budget), dtype=torch.uint8, device=dev)
        h2d_box = [0]

        def e2e_step():
            _, h2d_box[0] = ssd.ssd_round_host(host["tgt"], host["drf"], host["tokens"], host["uniforms"],
                                               host["temperature"], F, wl.budget, out=host_out,
                                               staging=staging, workspace=ws, stream=stream)
    else:
        dev_in = {k: torch.empty_like(v) for k, v in d.items()}
        h2d_box = [sum(v.numel() * v.element_size() for v in host.values())]

        def e2e_step():
            for k in dev_in:
                dev_in[k].copy_(host[k], non_blocking=True)
            if sig:
                o = ssd.ssd_verify_sigma(dev_in["tgt"], dev_in["drf"], dev_in["tokens"],
                                         dev_in["uniforms"], dev_in["temperature"], sig_F,
                                         wl.reshape_C, desc_out=desc, probs=False, workspace=ws,
                                         stream=stream)
            else:
                o = ssd.ssd_verify(dev_in["tgt"], dev_in["drf"], dev_in["tokens"], dev_in["uniforms"],
                                   dev_in["temperature"], probs=False, workspace=ws, stream=stream)
            for k in res_keys:
                host_out[k].copy_(o[k], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)

    peak, peak_kind = measured_peak()
    kmean = statistics.mean(kernel_ms)
    # time per step in the timed region: one launch of the streaming kernel per step
    # of the default round (two launches with --two-pass-sigma, whose bytes both count)
    launch_ms = elapsed_ms / args.steps
    achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
    value = job_rate(args.steps, world, elapsed_ms)
    line = {
        "metric": metric_name(), "value": value, "unit": "rounds/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Gaussian + Zipf log-bias logits; no datasets, no weights)",
        "config": workload_config(wl),
        "sequence_rounds_per_s": value * wl.B,
        "hbm_gbs_algorithmic": achieved,
        "algorithmic_bytes_per_round": alg_bytes, "dense_logit_bytes_per_round": dense_bytes,
        "kernel_ms": {"mean": kmean, "p10": float(np.percentile(kernel_ms, 10)),
                      "median": float(np.median(kernel_ms)), "p90": float(np.percentile(kernel_ms, 90)),
                      "launches": n_iso, "timing": "isolated launches, an event on each side"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": traffic_record(_build.stream_kernel_digest()),
                     "kernel": kernel_label(kernel_name, wl)},
        "e2e": {"value": job_rate(args.e2e_steps, world, e2e_ms), "unit": "rounds/s",
                "h2d_bytes_per_step": h2d_box[0], "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
        "accept_mean": float(np.mean(acc[acc >= 0])) if (acc >= 0).any() else None,
        "hit_rate": float(out["hit"].float().mean().item()) if wl.mode == "round" else None,
    }
    if sig:
        line["config"]["sigma"] = {
            "F": wl.reshape_F, "C": wl.reshape_C,
            "descriptors": ("separate pass (ssd_reshape_draft, then ssd_verify)" if args.two_pass_sigma
                            else "found in the verification pass (ssd_verify_sigma)"),
            "drafted_tokens": "drawn from sigma_{F,C} of the draft (Gumbel-max on the device)"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, wl, off)
    others = [w for w in args.workloads.split(",") if w and w != "none" and w != wl.name]
    if world == 1 and others and not args.batch:
        line["workloads"] = {w: measure_workload(w, ssd, torch, dev, peak) for w in others}
        line["gpu_launches_workloads"] = sum(
            e["launches_timed"] + 220 for e in line["workloads"].values())
    if pg:
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Reference arm: the float64 oracle on the host cores.
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    wl = chosen_workload(args)
    inp = synth.make_inputs(wl, synth.BENCH_SEED[wl.name])
    F, off, _ = oracle.fanout(wl.K, wl.budget, wl.a_p, wl.r, wl.V) if wl.budget else (
        None, np.zeros(wl.K + 2, np.int32), None)
    threads = oracle.default_threads()
    g = min(wl.greedy_first, wl.B)
    # each step: one sequence per host thread, alternating greedy / sampled, cycling the batch
    order = np.ravel(np.column_stack([np.arange(0, g), np.arange(g, 2 * g)])) if 0 < g < wl.B \
        else np.arange(wl.B)
    per_step = max(1, min(threads, wl.B))
    cursor = [0]

    def step():
        idx = np.array([order[(cursor[0] + j) % len(order)] for j in range(per_step)])
        cursor[0] += per_step
        sub = {k: inp[k][idx] for k in ("tgt", "drf", "tokens", "uniforms", "temperature")}
        if wl.mode == "round":
            oracle.round_(sub["tgt"], sub["drf"], sub["tokens"], sub["uniforms"], sub["temperature"],
                          wl.dtype, off, wl.budget, threads=threads)
        else:
            oracle.verify(sub["tgt"], sub["drf"], sub["tokens"], sub["uniforms"], sub["temperature"],
                          wl.dtype, wl.reshape_F, wl.reshape_C, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps * per_step / wl.B / dt
    line = {
        "impl": "reference", "metric": metric_name(), "value": value, "unit": "rounds/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Gaussian + Zipf log-bias logits; no datasets, no weights)",
        "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": "rounds/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {per_step} of {wl.B} sequences of one round "
                                   "(alternating greedy / sampled), float64 C oracle"},
        "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_fanout_study(args):
    """Cache-topology comparison of the Saguaro notes ("关键设计" item 1 and the
    component analysis): the same synthetic round (the workload's shapes, every
    sequence at one temperature) is run with the geometric and with the uniform
    fan-out of the same budget, and the share of sequences whose true outcome
    (a, t*) was cached is counted.  For a batch of b sequences the round only
    avoids the fallback when all b hit (item 3): the empirical all-hit rate of
    consecutive groups of b is reported beside p_hit^b."""
    import torch
    import speculative_decoding_verification_ssd_gb300 as ssd
    wl = chosen_workload(args).replace(greedy_first=0)
    if wl.budget == 0:
        wl = synth.WORKLOADS["c5"].replace(B=wl.B, K=wl.K, V=wl.V, dtype=wl.dtype)
    B, K, V = wl.B, wl.K, wl.V
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(synth.BENCH_SEED[WORKLOAD] + 17)
    tgt, drf = synth.make_logits(wl, rng)
    tt = torch.from_numpy(tgt.view(np.int16) if wl.dtype == synth.BF16 else tgt).to(dev)
    td = torch.from_numpy(drf.view(np.int16) if wl.dtype == synth.BF16 else drf).to(dev)
    if wl.dtype == synth.BF16:
        tt, td = tt.view(torch.bfloat16), td.view(torch.bfloat16)
    drf_f32 = synth.stored_to_f32(drf, wl.dtype)
    sizes = [b for b in (1, 2, 4, 8, 16, 32, 64, 128, 256) if b <= B]
    ws = ssd.workspace(B, K, dev)
    rows = []
    for tau in (0.0, 0.7, 1.0):
        taus = np.full(B, tau, np.float32)
        t_dev = torch.from_numpy(taus).to(dev)
        draws = [(torch.from_numpy(synth.sample_draft_tokens(rng, drf_f32, taus)).to(dev),
                  [torch.from_numpy(rng.random((B, K + 1), dtype=np.float32)).to(dev)
                   for _ in range(args.study_rounds)]) for _ in range(args.study_draws)]
        # the acceptance rate seen at this temperature (maximum likelihood of a geometric
        # accepted length truncated at K: accepted positions / tested positions) gives
        # the fan-out's a_p its fitted value
        a = torch.cat([ssd.ssd_round(tt, td, tok, draws[0][1][0], t_dev,
                                     ssd.ssd_fanout_uniform(K, wl.budget, V)[0], wl.budget,
                                     probs=False, workspace=ws)["accept_len"] for tok, _ in draws])
        a = a.cpu().numpy()
        tested = int((a + (a < K)).sum())
        a_fit = min(max(float(a.sum()) / max(tested, 1), 0.01), 0.99)
        shapes = {"geometric": (ssd.ssd_fanout(K, wl.budget, wl.a_p, wl.r, V), wl.a_p),
                  "geometric_fitted": (ssd.ssd_fanout(K, wl.budget, a_fit, wl.r, V), a_fit),
                  "uniform": (ssd.ssd_fanout_uniform(K, wl.budget, V), None)}
        hits = {name: [] for name in shapes}
        acc = {name: [] for name in shapes}
        for tokens, us in draws:
            for u in us:
                for name, ((F, _), _) in shapes.items():
                    o = ssd.ssd_round(tt, td, tokens, u, t_dev, F, wl.budget, probs=False,
                                      workspace=ws)
                    hits[name].append(o["hit"])
                    acc[name].append(o["accept_len"])
        torch.cuda.synchronize()
        for name, ((F, _), a_p) in shapes.items():
            H = torch.stack(hits[name]).cpu().numpy().astype(bool)      # [rounds, B]
            A = torch.stack(acc[name]).cpu().numpy()
            p_hat = float(H.mean())
            all_hit = {}
            for b in sizes:
                g = H[:, : (B // b) * b].reshape(H.shape[0], B // b, b).all(axis=2)
                all_hit[str(b)] = {"empirical": float(g.mean()), "p_hit^b": p_hat ** b}
            rows.append({"tau": tau, "fanout": name, "a_p": a_p, "F": [int(f) for f in F],
                         "hit_rate": p_hat, "accept_mean": float(A.mean()),
                         "hit_rate_by_accept_len": {
                             str(k): float(H[A == k].mean()) if (A == k).any() else None
                             for k in range(K + 1)},
                         "batch_all_hit": all_hit})
    line = {"study": "fanout", "workload": f"{wl.name}-shaped: B={B}, K={K}, V={V} {wl.dtype}, "
            f"budget {wl.budget}, geometric a_p={wl.a_p} r={wl.r}",
            "data": "synthetic (seeded Gaussian + Zipf log-bias logits; no datasets, no weights)",
            "rounds_per_temperature": args.study_draws * args.study_rounds,
            "rows": rows}
    print(json.dumps(line), flush=True)


def run_csweep_study(args):
    """The acceptance / cache-hit trade-off of SAGUARO sampling (the Saguaro notes,
    "关键设计" item 2): the cache keys of outcome k are the F_k best draft tokens of
    draft row k (the drafted token left out), and the draft samples x~_k from
    sigma_{F_k,C}, which scales the weight of those same tokens by C.  Lower C moves
    residual mass onto the cached tokens (more hits) and moves q away from p (fewer
    acceptances).  Per C: draft keys and descriptors (ssd_draft_cache), drafting by
    Gumbel-max on the device (input synthesis, not a step of the method), then
    rounds of ssd_verify on the reshaped q and ssd_cache_lookup."""
    import torch
    import speculative_decoding_verification_ssd_gb300 as ssd
    wl = chosen_workload(args).replace(greedy_first=0)
    if wl.budget == 0:
        wl = synth.WORKLOADS["c5"].replace(B=wl.B, K=wl.K, V=wl.V, dtype=wl.dtype)
    B, K, V = wl.B, wl.K, wl.V
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(synth.BENCH_SEED[WORKLOAD] + 29)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(rng.integers(1 << 62)))
    tgt, drf = synth.make_logits(wl, rng, draft_rows=K + 1)

    def logits(a):
        if wl.dtype == synth.F32:
            return torch.from_numpy(a).to(dev)
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    tt, td = logits(tgt), logits(drf)
    zd = td[:, :K].float()
    F, _ = ssd.ssd_fanout(K, wl.budget, wl.a_p, wl.r, V)
    ids = torch.arange(V, device=dev)
    sizes = [b for b in (1, 4, 16, 64) if b <= B]
    rows = []
    for tau in (0.7, 1.0):
        taus = torch.full((B,), tau, dtype=torch.float32, device=dev)
        for C in (1.0, 0.75, 0.5, 0.25, 0.1, 0.0):
            _, desc = ssd.ssd_draft_cache(td, None, F, wl.budget, C, cache=False, reshape=True)
            thr_val, thr_id, _, _ = ssd.desc_fields(desc)
            thr_val = thr_val.view(B, K, 1)
            thr_id = thr_id.view(B, K, 1)
            member = (zd > thr_val) | ((zd == thr_val) & (ids.view(1, 1, V) <= thr_id))
            logc = torch.where(member, torch.tensor(float(np.log(C)) if C > 0 else -float("inf"),
                                                    device=dev), torch.zeros((), device=dev))
            H, A = [], []
            for _ in range(args.study_draws):
                g = -torch.log(-torch.log(torch.rand(zd.shape, generator=gen, device=dev)
                                          .clamp_min(1e-30)))
                tokens = torch.argmax(zd / tau + logc + g, dim=-1).to(torch.int32).contiguous()
                cache, desc = ssd.ssd_draft_cache(td, tokens, F, wl.budget, C, reshape=True)
                for _ in range(args.study_rounds):
                    u = torch.rand((B, K + 1), generator=gen, device=dev)
                    v = ssd.ssd_verify(tt, td, tokens, u, taus, reshape=desc, probs=False)
                    h, _ = ssd.ssd_cache_lookup(cache, F, v["accept_len"], v["bonus"])
                    H.append(h)
                    A.append(v["accept_len"])
            H = torch.stack(H).cpu().numpy().astype(bool)
            A = torch.stack(A).cpu().numpy()
            tested = int((A + (A < K)).sum())
            p_hat = float(H.mean())
            rows.append({
                "tau": tau, "C": C, "hit_rate": p_hat, "accept_mean": float(A.mean()),
                "acceptance_rate": float(A.sum()) / max(tested, 1),
                "tokens_per_round": float(A.mean()) + 1.0,
                "batch_all_hit": {str(b): {
                    "empirical": float(H[:, : (B // b) * b].reshape(H.shape[0], B // b, b)
                                       .all(axis=2).mean()),
                    "p_hit^b": p_hat ** b} for b in sizes}})
    line = {"study": "csweep", "workload": f"{wl.name}-shaped: B={B}, K={K}, V={V} {wl.dtype}, "
            f"K+1 draft rows, budget {wl.budget}, geometric F={[int(f) for f in F]}",
            "data": "synthetic (seeded Gaussian + Zipf log-bias logits; no datasets, no weights)",
            "rounds_per_point": args.study_draws * args.study_rounds, "rows": rows}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.study == "fanout":
        run_fanout_study(args)
    elif args.study == "csweep":
        run_csweep_study(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
