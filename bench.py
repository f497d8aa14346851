"""Throughput of LRMoE's backward recalibration path on GB300.

One step = one pass of the whole path over one layer batch, through the C
ABI: route stats -> LRM score -> per-expert top-Q select -> compaction ->
grouped dgrad -> grouped wgrad.  The metric is retained token-expert pairs per
second (sum of the quotas over the step time).  Inputs are seeded synthetic
tensors shaped like a Qwen3-30B-A3B MoE layer (T=32768, E=128, k=8, h=2048,
I=768, bf16) unless --workload names another one; they are resident in HBM
and larger than L2, so no L2 flush is done between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the path's correctness
reference) on the host cores, on a bounded token slice of the same workload.
Under torchrun every rank runs an independent replica of the layer (the path
has no data exchange); rank 0 prints one JSON line.
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

DEFAULT_WORKLOAD = "qwen3_30b_a3b_T32768_E128_k8_h2048_I768"
METRIC = "retained pairs/s through score->select->compact->grouped GEMM"
UNIT = "pairs/s"
KERNELS = ("route_stats", "score", "select", "compact", "dgrad", "wgrad")
# kernels of one step: route stats 3 (count, finalize, scatter), score 1,
# select 1 (one cluster of CTAs per expert), compact 1, dgrad 1, wgrad 1
LAUNCHES_PER_STEP = 8


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # LRMoE sec. 4.1 times 50 warm-up and 1000 measured iterations (--warmup 50 --steps 1000);
    # the defaults are shorter so that the reference arm (the fp64 oracle, about 0.2 s a
    # step at its smallest sample) also ends within a couple of minutes
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-comparator", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other layers and the comparator sweep")
    ap.add_argument("--cpu-steps-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--ref-tokens", type=int, default=0, help="token slice of the reference arm's step")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def _snapshot(self):
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
            for line in out.stdout.strip().splitlines():
                self.rows.append([x.strip() for x in line.split(",")])
        except (OSError, subprocess.SubprocessError):
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.rows.append([x.strip() for x in line.split(",")])

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)
        if not self.rows:
            self._snapshot()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in self.rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# algorithmic work per launch (bytes or flop)


def algorithmic_work(w, retained, active_experts):
    """Per launch: (bytes, flop) of the work the method must do.

    Bytes are the HBM traffic a perfect kernel needs (each input read once,
    each output written once); flop counts only the retained rows, never the
    padding the method avoids.  A GEMM is bound by whichever roof takes
    longer: its flop at the bf16 peak or its bytes at the HBM peak.
    """
    T, E, k, h, I = w.T, w.E, w.k, w.h, w.I
    N = T * k
    gemm_flop = 2 * retained * h * I
    rows_bytes = 2 * retained * (h + I)
    return {
        "route_stats": (T * (4 * E + 4 * k) + 4 * N, 0),
        "score": (2 * T * h + N * (2 * I + 8), 0),
        "select": (8 * N + 4 * retained, 0),
        "compact": (retained * (4 * (h + I) + 8), 0),
        "dgrad": (rows_bytes + 2 * active_experts * h * I, gemm_flop),
        "wgrad": (rows_bytes + 4 * E * h * I, gemm_flop),
    }


def roofline_entry(nbytes, flop, ms, pk):
    """Roofline of one kernel from its mean per-call CUDA-event time.  Every
    such time is of a single launch well under a millisecond, so the tensor
    roof is the burst bf16 peak (the sustained one applies to seconds-long
    loops of one GEMM under the power cap)."""
    t_hbm = nbytes / (pk["hbm"] * 1e9)
    tc_peak = pk["bf16"]
    t_tc = flop / (tc_peak * 1e12)
    sec = ms * 1e-3
    if t_tc > t_hbm:
        achieved, peak, unit, kind = flop / sec / 1e12, tc_peak, "TFLOP/s", "tensor"
    else:
        achieved, peak, unit, kind = nbytes / sec / 1e9, pk["hbm"], "GB/s", "hbm"
    ent = {"bound": kind, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
           "frac": round(achieved / peak, 4), "hbm_frac": round(t_hbm / sec, 4), "bytes": nbytes}
    if flop:
        ent.update(tensor_frac=round(t_tc / sec, 4), flop=flop)
    return ent


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the
    kernel's source has not changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    try:
        with open(src, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    return rec["dram_bytes"] if digest == rec["source_sha256"] else None


# ---------------------------------------------------------------------------
# our arm


def issue_step(rec, d, ev=None, stream=None):
    """One step issued call by call; with `ev` (seven CUDA events) an event is
    recorded before the first and after every kernel call."""
    if ev is None:
        rec.run(d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"])
        return
    calls = (lambda: rec.route_stats(d["logits"], d["expert_idx"]), lambda: rec.score(d["g"], d["phi"], d["alpha"]),
             rec.select, lambda: rec.compact(d["g"], d["phi"], d["alpha"]), lambda: rec.dgrad(d["W"]), rec.wgrad)
    ev[0].record(stream)
    for i, call in enumerate(calls):
        call()
        ev[i + 1].record(stream)


def per_kernel_times(rec, d, K):
    """Per-kernel CUDA-event times (ms) of K steps issued call by call, and
    the eager step time."""
    import torch

    stream = torch.cuda.current_stream()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        issue_step(rec, d, evs[i], stream)
    torch.cuda.synchronize()
    eager_ms = evs[0][0].elapsed_time(evs[-1][6])
    per = {name: [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)] for j, name in enumerate(KERNELS)}
    return per, eager_ms


def graph_kernel_times(rec, d, n=20, reps=3):
    """Per-kernel time (ms) without host launch cost: n back-to-back calls of
    one step's kernel captured in a CUDA graph, replayed `reps` times after a
    warm replay.  Back-to-back calls find their small inputs in L2, so these
    are a lower bound for the latency-bound kernels' time inside the step."""
    import torch

    calls = dict(route_stats=lambda s: rec.route_stats(d["logits"], d["expert_idx"], s),
                 score=lambda s: rec.score(d["g"], d["phi"], d["alpha"], s), select=lambda s: rec.select(s),
                 compact=lambda s: rec.compact(d["g"], d["phi"], d["alpha"], s),
                 dgrad=lambda s: rec.dgrad(d["W"], s), wgrad=lambda s: rec.wgrad(s))
    out = {}
    for name in KERNELS:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for _ in range(n):
                    calls[name](side)
        torch.cuda.current_stream().wait_stream(side)
        graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        e1.synchronize()
        out[name] = round(e0.elapsed_time(e1) / (reps * n), 5)
        del graph
    return out


def kernel_table(w, retained, active, per, pk):
    """Per-kernel mean time, percentiles, share of the step and roofline."""
    work = algorithmic_work(w, retained, active)
    total = sum(sum(v) for v in per.values())
    kernels = {}
    for name in KERNELS:
        ms = statistics.mean(per[name])
        nbytes, flop = work[name]
        ent = roofline_entry(nbytes, flop, ms, pk)
        q = np.percentile(per[name], [10, 50, 90])
        ent.update(ms=round(ms, 5), ms_p10=round(float(q[0]), 5), ms_median=round(float(q[1]), 5),
                   ms_p90=round(float(q[2]), 5), share=round(sum(per[name]) / total, 4))
        kernels[name] = ent
    return kernels, work


def graph_steps(rec, d, K, sampler=None, dist=None):
    """K whole steps replayed as one CUDA graph, timed with CUDA events on the
    current stream with a synchronize (and a barrier under torchrun) on both
    sides; returns (total ms, host seconds)."""
    import torch

    from backward_token_expert_gb300.pipeline import StepGraph

    graph = StepGraph(rec, d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"])
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_host0 = time.perf_counter()
    e_start.record(stream)
    for _ in range(K):
        graph.replay()
    e_end.record(stream)
    torch.cuda.synchronize()
    t_host = time.perf_counter() - t_host0
    if sampler:
        sampler.stop()
    if dist:
        dist.barrier()
    return e_start.elapsed_time(e_end), t_host


def prepare_layer(w, inp, local, warmup):
    """Device inputs and buffers of one layer, warmed up and checked."""
    import torch

    from backward_token_expert_gb300.pipeline import Recalibration, to_device_inputs

    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho, device=local)
    d = to_device_inputs(inp, f"cuda:{local}")
    for _ in range(max(3, warmup)):
        issue_step(rec, d)
    torch.cuda.synchronize()
    flags = rec.device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} on {w.name}")
    return rec, d


def run_ours(args, rank, world, local):
    import torch

    from backward_token_expert_gb300 import build as B
    from backward_token_expert_gb300.replicas import job_totals, replica_seed
    from workloads import generate, get_workload

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        B.build()
    if dist:
        dist.barrier()

    # independent replicas: rank r draws its own layer batch
    w = get_workload(args.workload, seed=replica_seed(rank))
    inp = generate(w)
    rec, d = prepare_layer(w, inp, local, args.warmup)
    summ = rec.summary()
    retained = int(summ["retained"])

    # the timed steps: the whole step as one CUDA graph (StepGraph), replayed
    K = args.steps
    sampler = ClockSampler(local) if rank == 0 else None
    total_ms, t_host = graph_steps(rec, d, K, sampler, dist)
    # whole job: pairs of every replica over the slowest replica's time
    job_pairs, job_s = job_totals(retained * K, total_ms * 1e-3, device=f"cuda:{local}")
    total_ms = job_s * 1e3

    # per-kernel times: the same step issued call by call, events between the calls
    per, eager_ms = per_kernel_times(rec, d, K)
    in_graph = graph_kernel_times(rec, d) if rank == 0 else None
    flags = rec.device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} after the timed steps")

    result = None
    if rank == 0:
        pk = peaks()
        so = rec.buf.sel_offsets.cpu().numpy()
        active = int((np.diff(so) > 0).sum())
        kernels, work = kernel_table(w, retained, active, per, pk)
        dominant = max(KERNELS, key=lambda n: kernels[n]["ms"])
        top = {k2: kernels[dominant][k2] for k2 in ("bound", "achieved", "peak", "unit", "frac")}
        top.update(kernel=dominant, traffic=measured_traffic(dominant) if w.name == DEFAULT_WORKLOAD else None,
                   algorithmic_bytes=kernels[dominant]["bytes"],
                   peak_kind="burst bf16 (of measured)" if top["bound"] == "tensor" else "hbm copy (of measured)",
                   peak_source=pk["source"])
        value = job_pairs / job_s
        in_bytes = w.N * w.I * 2 + w.E * w.h * w.I * 2 + w.T * w.h * 2
        # pipeline fraction: the time every step would take at its binding roof,
        # over the measured time of the steps
        ideal_s = sum(max(work[n][0] / (pk["hbm"] * 1e9), work[n][1] / (pk["bf16"] * 1e12)) for n in KERNELS)
        steps_s = sum(kernels[n]["ms"] for n in KERNELS) * 1e-3
        excl_rs_s = sum(kernels[n]["ms"] for n in KERNELS if n != "route_stats") * 1e-3
        result = {
            "metric": METRIC,
            "value": value,
            "unit": UNIT,
            "n_gpus": world,
            "steps": K,
            "warmup": max(3, args.warmup),
            "ms_per_step": total_ms / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": f"synthetic (seeded {w.name} layer, random-init weights)",
            "config": {
                "workload": w.name, "T": w.T, "E": w.E, "k": w.k, "h": w.h, "I": w.I,
                "zipf_s": w.zipf_s, "rho": str(w.rho), "CF": str(w.cf), "retained_pairs": retained,
                "routed_pairs": w.N, "C": summ["C"], "max_over_mean": round(summ["max_over_mean"], 3),
                "drop_rate": round(summ["drop_rate"], 5), "parallelism": f"replicas x{world}",
                "l2": (f"no flush: inputs {'larger than' if in_bytes > 129e6 else 'within'} L2 "
                       f"(phi {w.N * w.I * 2 / 2**20:.0f} MiB, W {w.E * w.h * w.I * 2 / 2**20:.0f} MiB, "
                       f"g {w.T * w.h * 2 / 2**20:.0f} MiB; L2 129 MB)"),
            },
            "roofline": top,
            "launch": "CUDA graph of the whole step (StepGraph.replay; route stats a branch beside score); "
                      "per-kernel times from the same step issued call by call with events between the calls",
            "eager": {"ms_per_step": round(eager_ms / K, 5), "value": round(retained * K / (eager_ms * 1e-3), 1)},
            "pipeline_frac": round(ideal_s / steps_s, 4),
            "score_select_compact": {
                "what": "score, select and compact as one aggregate: their algorithmic bytes over their summed "
                        "times, against the HBM copy peak",
                "ms": round(sum(kernels[n]["ms"] for n in ("score", "select", "compact")), 5),
                "hbm_frac": round(sum(work[n][0] for n in ("score", "select", "compact")) / (pk["hbm"] * 1e9)
                                  / (sum(kernels[n]["ms"] for n in ("score", "select", "compact")) * 1e-3), 4)},
            "score_to_gemm": {
                "what": "the metric as its name defines it: retained pairs over the mean time of score, select, "
                        "compact, dgrad and wgrad (route stats reported apart)",
                "value": round(retained / excl_rs_s, 1), "unit": UNIT,
                "route_stats_ms": kernels["route_stats"]["ms"]},
            "kernels": kernels,
            "kernels_in_graph_ms": dict(in_graph, what="each kernel alone, 20 back-to-back calls captured in one "
                                        "CUDA graph: no host launch cost, small inputs warm in L2"),
            "gpu_launches": LAUNCHES_PER_STEP * K,
            "host_s": round(t_host, 4),
            "clocks": sampler.summary() if sampler else None,
        }
        if not args.no_comparator:
            result["comparator"] = comparator(rec, d, w, retained, pk)
            result["inverse_mapping"] = inverse_mapping(rec, d, w, retained, pk)
            result["bf16_dW"] = bf16_dw_step(rec, d, w, retained, pk, work, min(K, 100))
            result["fc1_backward"] = fc1_backward(rec, w, retained, pk)
    if not args.no_e2e:
        # every replica runs its end-to-end loop at the same time, before the
        # CPU baseline keeps the host cores busy
        if dist:
            dist.barrier()
        ent = e2e(rec, inp, w, retained, min(K, 20), local)
        if result is not None:
            result["e2e"] = ent
    rec.close()
    del rec, d
    if result is not None and not args.no_configs:
        # the other layers of the scope, each with its own timed steps and clocks
        torch.cuda.empty_cache()
        result["comparator_sweep"] = comparator_sweep(local, peaks())
        result["configs"] = {}
        for name in OTHER_CONFIGS:
            result["configs"][name] = other_config(name, local, min(K, 20), args.warmup, peaks())
    if result is not None and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, tokens=args.ref_tokens or 8192)
        result["cpu_baseline"]["per_step"] = cpu_per_step(inp.workload.name, tokens=4096)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return result


# the layers measured next to the headline one (configs of the scope besides
# the tiny one and the sweep)
OTHER_CONFIGS = ("glm45_air_T32768_E128_k8_h4096_I1408", "stress_T131072_E128_k8_h4096_I1408",
                 "deepseek_v2_T32768_E160_k6_h5120_I1536")


def other_config(name, local, K, warmup, pk):
    """The step on another layer: graph-replayed steps with clocks sampled
    during them, and per-kernel times with their rooflines."""
    import torch

    from workloads import generate, get_workload

    w = get_workload(name)
    inp = generate(w)
    rec, d = prepare_layer(w, inp, local, warmup)
    del inp
    try:
        summ = rec.summary()
        retained = int(summ["retained"])
        sampler = ClockSampler(local)
        total_ms, _ = graph_steps(rec, d, K, sampler)
        per, _ = per_kernel_times(rec, d, K)
        flags = rec.device_status()
        if flags:
            raise RuntimeError(f"device status flags {flags:#x} on {name}")
        so = rec.buf.sel_offsets.cpu().numpy()
        kernels, _ = kernel_table(w, retained, int((np.diff(so) > 0).sum()), per, pk)
        return {
            "value": round(retained * K / (total_ms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(total_ms / K, 5),
            "steps": K, "retained_pairs": retained, "routed_pairs": w.N, "C": summ["C"],
            "max_over_mean": round(summ["max_over_mean"], 3), "empty_experts": w.E - summ["nonempty"],
            "experts_over_C": int((rec.buf.counts > summ["C"]).sum().item()),
            "kernels": {n: {k2: kernels[n][k2] for k2 in ("ms", "bound", "achieved", "unit", "frac", "hbm_frac")
                            + (("tensor_frac",) if "tensor_frac" in kernels[n] else ())} for n in KERNELS},
            "clocks": sampler.summary(),
        }
    finally:
        rec.close()
        del rec, d
        torch.cuda.empty_cache()


def comparator_sweep(local, pk, iters=10):
    """Compacted GEMMs against the zero-masked capacity-padded ones at every
    point of the skew / retention sweep, on identical tensors (the sweep
    points share one seed, so g, phi and W are drawn and uploaded once)."""
    import torch

    from backward_token_expert_gb300.pipeline import to_device_inputs
    from workloads import generate, get_workload
    from workloads.generate import Inputs

    names = [f"qwen3_sweep_s{s:g}_rho{r}" for s in (0.0, 0.8, 1.2, 1.6) for r in ("1_1", "3_4", "1_2")]
    base = generate(get_workload(names[0]))
    shared = None
    points = {}
    for name in names:
        w = get_workload(name)
        r = generate(w, parts=())
        inp = Inputs(w, r.logits, r.expert_idx, r.alpha, base.g, base.phi, base.W, r.bias)
        if shared is None:
            shared = to_device_inputs(inp, f"cuda:{local}")
            d = shared
        else:
            d = dict(shared, logits=torch.from_numpy(r.logits).to(shared["g"].device),
                     expert_idx=torch.from_numpy(r.expert_idx).to(shared["g"].device),
                     alpha=torch.from_numpy(r.alpha).to(shared["g"].device))
        from backward_token_expert_gb300.pipeline import Recalibration

        rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho, device=local)
        try:
            issue_step(rec, d)
            torch.cuda.synchronize()
            summ = rec.summary()
            ent = comparator(rec, d, w, int(summ["retained"]), pk, iters=iters)
            ent.update(zipf_s=w.zipf_s, rho=str(w.rho), retained_pairs=int(summ["retained"]),
                       max_over_mean=round(summ["max_over_mean"], 3))
            for key in ("what", "padded_slots"):
                ent.pop(key, None)
            points[name] = ent
        finally:
            rec.close()
    del shared
    torch.cuda.empty_cache()
    return {"what": "compact+dgrad+wgrad on the retained rows vs compact_padded+dgrad+wgrad at M=C per expert "
                    "(E*C = 327680 slots), same kernels and tensors, every (zipf s, rho) point",
            "points": points}


def bf16_dw_step(rec, d, w, retained, pk, work, iters):
    """The same step with the weight gradient stored as bf16
    (lrm_grouped_wgrad_bf16; the BF16 gradient of the pages' mixed-precision
    training): the whole step as a CUDA graph timed again, and the wgrad alone
    with its roofline (its bytes drop from 4 to 2 per dW element)."""
    import torch

    from backward_token_expert_gb300.pipeline import StepGraph

    s = torch.cuda.current_stream()
    graph = StepGraph(rec, d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"], dw_bf16=True)
    out = {}
    for name, fn in (("step", graph.replay), ("wgrad", rec.wgrad_bf16)):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(iters):
            fn()
        e1.record(s)
        e1.synchronize()
        out[name + "_ms"] = e0.elapsed_time(e1) / iters
    flags = rec.device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} in the bf16-dW step")
    nbytes = work["wgrad"][0] - 2 * w.E * w.h * w.I
    ent = roofline_entry(nbytes, work["wgrad"][1], out["wgrad_ms"], pk)
    return {"what": "the timed step (CUDA graph) with dW stored as bf16",
            "value": round(retained / (out["step_ms"] * 1e-3), 1), "unit": UNIT,
            "ms_per_step": round(out["step_ms"], 5), "steps": iters,
            "wgrad": dict(ms=round(out["wgrad_ms"], 5), **ent)}


def inverse_mapping(rec, d, w, retained, pk, iters=20):
    """The inverse mapping (ScatterWithZeros): dgrad written through the
    selection into the [N, I] pair-major layout plus the zeroing of the dropped
    rows, against the compacted dgrad alone."""
    import torch

    rows = torch.empty(w.N, w.I, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream()
    out = {}
    for name, fn in (("dgrad_compacted", lambda: rec.dgrad(d["W"])),
                     ("dgrad_scatter", lambda: rec.dgrad_scatter(d["W"], rows, zero_dropped=False)),
                     ("scatter_with_zeros", lambda: rec.dgrad_scatter(d["W"], rows, zero_dropped=True))):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(iters):
            fn()
        e1.record(s)
        e1.synchronize()
        out[name + "_ms"] = round(e0.elapsed_time(e1) / iters, 5)
    zero_bytes = (w.N - retained) * w.I * 2
    out.update(what="dgrad into the compacted rows vs through the selection into [N, I] (+ zeros for dropped rows)",
               zeroed_bytes=zero_bytes,
               zeroing_hbm_frac=round(zero_bytes / (pk["hbm"] * 1e9) /
                                      max((out["scatter_with_zeros_ms"] - out["dgrad_scatter_ms"]) * 1e-3, 1e-9), 4))
    flags = rec.device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} in the inverse mapping")
    return out


def fc1_backward(rec, w, retained, pk, iters=20):
    """The FC1 side of the expert backward on the retained pairs (SwiGLU read),
    after the timed FC2 steps have left their compacted input gradient: each of
    its five library calls timed alone, with its roofline from the algorithmic
    bytes (and flop) per launch."""
    import torch

    from backward_token_expert_gb300 import lrm as L
    from workloads import fc1_inputs

    f1 = fc1_inputs(w)

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()

    x, ab, W1 = dev(f1.x), dev(f1.ab), dev(f1.W1)
    del f1
    rec.fc1_backward(x, ab, W1)  # allocates the FC1 buffers
    f, b, ctx, mr = rec.fc1, rec.buf, rec.ctx, rec.max_rows
    T, E, k, h, I = w.T, w.E, w.k, w.h, w.I
    d_in, d_fc1 = L.Dims(T, E, k, h, 2 * I), L.Dims(T, E, k, 2 * I, h)
    act = int((b.sel_offsets[1:] > b.sel_offsets[:-1]).sum().item())
    gemm_flop = 2 * retained * 2 * I * h
    calls = {
        "compact": (lambda: L.lrm_compact(ctx, x, ab, f.ones, b.sel_offsets, b.sel_ids, d_in, mr, f.xc, f.abc, None),
                    (retained * (4 * h + 8 * I + 8), 0)),
        "swiglu_backward": (lambda: L.lrm_swiglu_backward(ctx, b.dphi_c, f.abc, b.sel_offsets, rec.dims, mr, f.dh1),
                            (retained * 10 * I, 0)),
        "dgrad": (lambda: L.lrm_grouped_dgrad(ctx, f.dh1, W1, b.sel_offsets, d_fc1, mr, f.dxc),
                  (retained * 2 * (2 * I + h) + act * 4 * I * h, gemm_flop)),
        "wgrad": (lambda: L.lrm_grouped_wgrad(ctx, f.dh1, f.xc, b.sel_offsets, d_fc1, mr, 0, f.dW1),
                  (retained * 2 * (2 * I + h) + E * 8 * I * h, gemm_flop)),
        "combine": (lambda: L.lrm_combine_rows(ctx, f.dxc, b.sel_offsets, b.sel_ids, rec.dims, mr, h, f.dx, f.ws,
                                               f.ws.numel()),
                    (8 * w.N + 8 * retained + retained * 2 * h + T * 2 * h, 0)),
    }
    s = torch.cuda.current_stream()
    out = {}
    for name, (fn, (nbytes, flop)) in calls.items():
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(iters):
            fn()
        e1.record(s)
        e1.synchronize()
        ms = e0.elapsed_time(e1) / iters
        out[name] = dict(ms=round(ms, 5), **roofline_entry(nbytes, flop, ms, pk))
    for _ in range(3):
        rec.fc1_backward(x, ab, W1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(iters):
        rec.fc1_backward(x, ab, W1)
    e1.record(s)
    e1.synchronize()
    total = e0.elapsed_time(e1) / iters
    flags = rec.device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} in the FC1 backward")
    return {"what": "compact x and [a|b], SwiGLU backward, FC1 dgrad and wgrad (K = 2I), combine per token",
            "ms": round(total, 5), "pairs_per_s": round(retained / (total * 1e-3), 1), "kernels": out}


def comparator(rec, d, w, retained, pk, iters=20):
    """Zero-masked fixed-shape (capacity-padded) GEMMs on the same retained rows."""
    import torch

    from backward_token_expert_gb300 import lrm as L

    E, C = w.E, rec.C
    dpad = torch.empty(E * C, w.h, dtype=torch.bfloat16, device="cuda")
    ppad = torch.empty(E * C, w.I, dtype=torch.bfloat16, device="cuda")
    poff = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dphi = torch.empty(E * C, w.I, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(E, w.h, w.I, dtype=torch.float32, device="cuda")
    b = rec.buf
    s = torch.cuda.current_stream()

    def padded():
        L.lrm_compact_padded(rec.ctx, b.delta_c, b.phi_c, b.sel_offsets, rec.dims, C, dpad, ppad, poff)
        L.lrm_grouped_dgrad(rec.ctx, dpad, d["W"], poff, rec.dims, E * C, dphi)
        L.lrm_grouped_wgrad(rec.ctx, dpad, ppad, poff, rec.dims, E * C, 0, dW)

    def compacted():
        rec.compact(d["g"], d["phi"], d["alpha"])
        rec.dgrad(d["W"])
        rec.wgrad()

    out = {}
    for name, fn in (("compacted", compacted), ("zero_masked", padded)):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(iters):
            fn()
        e1.record(s)
        e1.synchronize()
        out[name + "_ms"] = round(e0.elapsed_time(e1) / iters, 5)
    flops_alg = 4 * retained * w.h * w.I
    flops_pad = 4 * E * C * w.h * w.I
    out.update(
        what="compact+dgrad+wgrad on the retained rows vs compact_padded+dgrad+wgrad at M=C per expert",
        algorithmic_flop=flops_alg, padded_flop=flops_pad, padded_slots=E * C,
        speedup=round(out["zero_masked_ms"] / out["compacted_ms"], 3),
        zero_masked_algorithmic_tflops=round(flops_alg / (out["zero_masked_ms"] * 1e-3) / 1e12, 2),
        zero_masked_padded_tflops=round(flops_pad / (out["zero_masked_ms"] * 1e-3) / 1e12, 2),
        compacted_algorithmic_tflops=round(flops_alg / (out["compacted_ms"] * 1e-3) / 1e12, 2))
    flags = rec.device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} in the comparator")
    return out


def e2e(rec, inp, w, retained, iters, local):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory, runs the path and copies its results
    back (HostPipeline: the copies of neighbouring steps overlap the compute
    on their own streams)."""
    import torch

    from backward_token_expert_gb300.pipeline import HostPipeline
    from backward_token_expert_gb300.replicas import job_totals

    def pinned(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            t = t.view(dtype)
        return t.pin_memory()

    h_in = dict(logits=pinned(inp.logits), expert_idx=pinned(inp.expert_idx), alpha=pinned(inp.alpha),
                g=pinned(inp.g.view(np.int16), torch.bfloat16), phi=pinned(inp.phi.view(np.int16), torch.bfloat16),
                W=pinned(inp.W.view(np.int16), torch.bfloat16))
    pipe = HostPipeline(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho, device=local)
    h_out = [pipe.host_outputs(), pipe.host_outputs()]
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    try:
        for i in range(3):
            pipe.submit(h_in, h_out[i % 2])
        pipe.synchronize()
        b0 = pipe.d2h_bytes
        t0 = time.perf_counter()
        for i in range(iters):
            pipe.submit(h_in, h_out[i % 2])
        pipe.synchronize()
        dt = time.perf_counter() - t0
        d2h = (pipe.d2h_bytes - b0) // iters  # dW, the selection, the summary and the retained dphi_c rows
        flags = pipe.device_status()
        if flags:
            raise RuntimeError(f"device status flags {flags:#x} in the end-to-end loop")
        got = int(np.frombuffer(h_out[(iters - 1) % 2]["sel_offsets"].numpy().tobytes(), dtype=np.int32)[-1])
        if got != retained:
            raise RuntimeError(f"end-to-end loop retained {got} pairs, the device-timed step {retained}")
    finally:
        pipe.close()
    pairs, slowest = job_totals(retained * iters, dt, device=f"cuda:{local}")
    return {"value": pairs / slowest, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": iters, "ms_per_step": slowest * 1e3 / iters,
            "api": "backward_token_expert_gb300.pipeline.HostPipeline.submit (C ABI), pinned host buffers, "
                   "copies on their own streams overlapping the neighbouring steps' compute; of dphi_c only the "
                   "retained rows are copied back"}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores (cpu_baseline leg and the reference arm)


def token_slice(inp, tokens):
    import dataclasses

    from workloads.generate import Inputs

    w = inp.workload
    T = min(tokens, w.T)
    ws = dataclasses.replace(w, T=T)
    return Inputs(ws, inp.logits[:T], inp.expert_idx[:T], inp.alpha[: T * w.k], inp.g[:T], inp.phi[: T * w.k],
                  inp.W, inp.bias)


def oracle_step(sl):
    import oracle as O

    out = O.backward_recalibration(sl)
    return int(out["stats"]["retained"])


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name and architecture, as the kernel reports them."""
    import platform

    model, impl, part = "", "", ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" not in line:
                    continue
                key, val = (x.strip() for x in line.split(":", 1))
                key = key.lower()
                if key in ("model name", "cpu model", "hardware") and not model:
                    model = val
                elif key == "cpu implementer" and not impl:
                    impl = val
                elif key == "cpu part" and not part:
                    part = val
    except OSError:
        pass
    if not model and impl:  # Arm cores report an implementer and a part number instead of a name
        model = f"Arm CPU implementer {impl} part {part}"
    return {"model": model or platform.processor() or "unknown", "arch": platform.machine()}


def cpu_baseline(inp, tokens, target_s=15.0):
    """The oracle as it stands on a bounded token slice, repeated until about
    `target_s` seconds of timed CPU work have run (at least two passes)."""
    sl = token_slice(inp, tokens)
    t0 = time.perf_counter()
    oracle_step(sl)  # warm-up, also sizes the repetition count
    first = time.perf_counter() - t0
    steps = max(2, min(50, int(target_s / max(first, 1e-3))))
    t0 = time.perf_counter()
    retained = 0
    for _ in range(steps):
        retained += oracle_step(sl)
    dt = time.perf_counter() - t0
    w = inp.workload
    return {"value": retained / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"whole path (fp64 numpy oracle) on the first {sl.workload.T} tokens of the "
                      f"{w.name} layer ({sl.workload.N} routed pairs, same E/k/h/I/CF/rho); "
                      f"{steps} timed passes after 1 warm-up; BLAS may use all {cpu_cores()} cores, "
                      "the rest of numpy one",
            "seconds": round(dt, 3), "host": cpu_model()}


CPU_STEPS = ("route_stats", "score", "select", "compact", "dgrad", "wgrad")
BLAS_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                    "GOTO_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")


def cpu_steps_child(workload, tokens, runs=3):
    """Run in a child process whose BLAS thread count its environment fixed:
    each step of the oracle timed alone on a token slice (one warm-up, then
    `runs` timed runs; the median is reported)."""
    import oracle as O
    from workloads import generate, get_workload

    inp = token_slice(generate(get_workload(workload)), tokens)
    w = inp.workload
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
    R = O.score(inp.g, inp.phi, inp.alpha, w.k)
    so, ids = O.select(R, inp.expert_idx, w.E, st["quota"])
    steps = {
        "route_stats": lambda: O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho),
        "score": lambda: O.score(inp.g, inp.phi, inp.alpha, w.k),
        "select": lambda: O.select(R, inp.expert_idx, w.E, st["quota"]),
        "compact": lambda: O.compact(inp.g, inp.phi, inp.alpha, ids, w.k),
        "dgrad": lambda: O.grouped_dgrad(inp.g, inp.W, inp.alpha, so, ids, w.E, w.k),
        "wgrad": lambda: O.grouped_wgrad(inp.g, inp.phi, inp.alpha, so, ids, w.E, w.k),
    }
    out = {}
    for name in CPU_STEPS:
        steps[name]()
        times = []
        for _ in range(runs):
            t0 = time.perf_counter()
            steps[name]()
            times.append(time.perf_counter() - t0)
        out[name] = round(statistics.median(times), 5)
    retained = int(so[-1])
    total = sum(out[n] for n in CPU_STEPS if n != "route_stats")
    return {"seconds": out, "retained_pairs": retained, "routed_pairs": w.N, "tokens": w.T,
            "value": round(retained / total, 1), "unit": UNIT}


def cpu_per_step(workload, tokens):
    """The oracle per step at one thread and at all host cores, each in a child
    process with the BLAS thread variables set before numpy loads."""
    out = {"what": f"fp64 numpy oracle per step on the first {tokens} tokens of {workload}; median of 3 timed runs "
                   "after 1 warm-up; value = retained pairs over score..wgrad seconds (route stats apart)",
           "host": cpu_model()}
    for label, threads in (("threads_1", 1), ("threads_all", cpu_cores())):
        env = dict(os.environ, **{v: str(threads) for v in BLAS_THREAD_VARS})
        try:
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-steps-child", "--workload", workload,
                                "--ref-tokens", str(tokens)], env=env, capture_output=True, text=True, timeout=600)
            ent = json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else {"error": r.stderr[-300:]}
        except (subprocess.SubprocessError, ValueError, IndexError) as ex:
            ent = {"error": str(ex)[:300]}
        ent["threads"] = threads
        out[label] = ent
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from workloads import generate, get_workload

    w = get_workload(args.workload)
    inp = generate(w)
    K, W = args.steps, max(3, args.warmup)
    # size the token slice so that K + W passes take about two minutes
    tokens = args.ref_tokens
    if not tokens:
        probe = token_slice(inp, 256)
        oracle_step(probe)
        t0 = time.perf_counter()
        oracle_step(probe)
        per256 = time.perf_counter() - t0
        budget = 120.0 / (K + W)
        tokens = int(max(64, min(w.T, 256 * budget / max(per256, 1e-3))))
        tokens = max(64, (tokens // 64) * 64)
    sl = token_slice(inp, tokens)
    for _ in range(W):
        oracle_step(sl)
    t0 = time.perf_counter()
    retained = 0
    for _ in range(K):
        retained += oracle_step(sl)
    dt = time.perf_counter() - t0
    value = retained / dt
    sample = (f"whole path (fp64 numpy oracle) on the first {sl.workload.T} tokens of the {w.name} layer "
              f"({sl.workload.N} routed pairs per step, same E/k/h/I/CF/rho)")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": dt * 1e3 / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": w.name, "T": w.T, "E": w.E, "k": w.k, "h": w.h, "I": w.I,
                   "sample_tokens": sl.workload.T},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample,
                         "host": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.cpu_steps_child:
        print(json.dumps(cpu_steps_child(args.workload, args.ref_tokens or 4096)))
        return
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
