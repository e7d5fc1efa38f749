#!/usr/bin/env python
"""Benchmark of the Domino draft-block rollout on GB300.

Default workload: Qwen3-8B-shaped rollout (V=151936, H=4096, E=G=F=1024,
bf16 weights, fp32 accumulation), B=1 request, full-vocabulary correction
(K0), 15 proposals per block.  One JSON line on stdout (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-sweep] [--no-cpu-baseline]

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events
on the launching stream; a 512 MiB buffer is written between timed steps so
that every step starts with a cold L2.  Multi-GPU (torchrun): every rank runs
an independent replica on its own requests (no collective on the data path);
the step time is the max over ranks.
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

from speculative_decoding_draft_lm_gb300 import inputs  # noqa: E402

METRIC = "Domino rollout µs/block & proposals/s at B=1/8/64; % HBM/tensor roofline"
UNIT = "proposals/s"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SWEEP = ("qwen3_8b_b1_k0", "qwen3_8b_b8_k0", "qwen3_8b_b64_k0",
         "qwen3_8b_b1_k2048", "qwen3_8b_b8_k2048", "qwen3_8b_b64_k2048")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_8b_b1_k0", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--no-sweep", action="store_true", help="skip the B=1/8/64 x K0/K2048 table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0, help="wall budget of the oracle sample")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---- algorithmic bytes / flops -------------------------------------------

def alg_bytes(sh: inputs.Shape, B: int, K: int, n_prop: int = 15, s_in_library: bool = False) -> dict:
    """Algorithmic bytes per launch of each phase and per block; ``n_prop``
    proposals take max(2, n_prop) GRU updates and n_prop - 1 corrected steps;
    ``s_in_library`` adds W_hid and the s rows to the LM-head launch."""
    e = 2 if sh.dtype == "bf16" else 4
    V, H, E, G, F = sh.V, sh.H, sh.E, sh.G, sh.F
    full = K == 0 or K >= V
    lm = V * H * e + B * 16 * H * e + B * 16 * V * 4
    lm_flop = 2.0 * B * 16 * V * H
    if s_in_library:
        lm += F * H * e + B * 15 * F * e
        lm_flop += 2.0 * B * 16 * F * H
    if full:
        corr = V * F * e + V * e + B * V * 4 + B * F * 4
    else:
        corr = B * K * (F * e + e + 4 + 4) + B * F * 4
    # GRU: W_hh, plus per request one row of the token table (3G fp32: the
    # input side W_ih emb[t], built at load time) and the state in and out
    gru = 3 * G * G * e + B * (3 * G * 4 + G * 4 * 2)
    fc1 = F * G * e + B * (G * 4 + F * e + F * 4 * 2)
    pool = 0 if full else B * 15 * V * 4 + B * V * 4 * 5 + B * K * 4
    # persistent driver: the GRU seed and the corrected steps in one launch.
    # A tensor counts once per launch when its working set over the whole
    # rollout fits in 64 MB of L2, else once per step: W_hh and fc1 always
    # fit; the pool's gathered rows fit for small B*K; fc2 over the full
    # vocabulary does not.  Per-step rows (token table, base logits, state,
    # s, activations) always count per step.
    n_upd, n_corr = max(2, n_prop), n_prop - 1
    l2_fit = 64 << 20
    per_upd = B * (3 * G * 4 + G * 4 * 2)
    per_fc1 = B * (G * 4 + F * e + F * 4 * 2)
    if full:
        corr_once, corr_step = 0, corr
    else:
        rows = B * K * (F * e + e + 4)
        corr_once, corr_step = (rows, corr - rows) if rows <= l2_fit else (0, corr)
    steps = (3 * G * G * e + F * G * e + corr_once + n_upd * per_upd +
             n_corr * (per_fc1 + corr_step))
    per_block = lm + pool + steps
    return {"lmhead": lm, "correct": corr, "gru": gru, "fc1": fc1, "pool": pool, "steps": steps,
            "block": per_block, "lmhead_flop": lm_flop}


# ---- clocks sampler ---------------------------------------------------------

class Clocks:
    """SM clock and clock-event reasons sampled during the timed region.

    Reads NVML through ctypes every ~2 ms from a background thread (read-only
    queries); falls back to `nvidia-smi -lms 200` when NVML is unavailable.
    """
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.nvml = None
        self.handle = None
        self.samples = []
        self.stop_flag = False
        self.thread = None
        self._init_nvml()

    def _init_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            import torch
            props = torch.cuda.get_device_properties(self.dev)
            handle = ctypes.c_void_p()
            ok = False
            bus = getattr(props, "pci_bus_id", None)
            if bus is not None:
                dom = getattr(props, "pci_domain_id", 0)
                devid = getattr(props, "pci_device_id", 0)
                busid = ("%08x:%02x:%02x.0" % (dom, bus, devid)).encode()
                ok = lib.nvmlDeviceGetHandleByPciBusId_v2(busid, ctypes.byref(handle)) == 0
            if not ok:
                ok = lib.nvmlDeviceGetHandleByIndex_v2(self.dev, ctypes.byref(handle)) == 0
            if ok:
                self.nvml, self.handle = lib, handle
        except (OSError, AttributeError):
            self.nvml = None

    def _poll(self):
        import ctypes
        lib, h = self.nvml, self.handle
        clk = ctypes.c_uint()
        mw = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag:
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                p_ok = lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0
                r_ok = get_reasons(h, ctypes.byref(rs)) == 0
                self.samples.append((clk.value, mw.value / 1000.0 if p_ok else None, rs.value if r_ok else 0))
            time.sleep(0.002)

    def start(self):
        if self.nvml is not None:
            import threading
            self.samples = []
            self.stop_flag = False
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.nvml is not None:
            import ctypes
            self.stop_flag = True
            self.thread.join()
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))
            sm = [x[0] for x in self.samples]
            pw = [x[1] for x in self.samples if x[1] is not None]
            reasons = set()
            for _, _, r in self.samples:
                for bit, name in self.REASONS.items():
                    if r & bit:
                        reasons.add(name)
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx.value or None,
                    "power_w_max": max(pw) if pw else None, "samples": len(sm), "source": "nvml, 2 ms",
                    "reasons": sorted(reasons)}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "source": "nvidia-smi, 200 ms",
                "reasons": sorted(reasons)}


# ---- distributed plumbing ---------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_seeds(wl: inputs.Workload, rank: int) -> list:
    """Request seeds of one replica: every rank runs its own B requests."""
    return [s + rank * 100000 for s in wl.request_seeds]


def max_over_ranks(x: float, dist, device: str) -> float:
    """The slowest rank's value (identity without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(B: int, world: int, ms_per_step: float) -> float:
    """Proposals per second of all replicas: 15 per request per block."""
    return 15.0 * B * world / (ms_per_step * 1e-3)


# ---- CPU oracle leg ------------------------------------------------------------

class OracleSample:
    """The CPU oracle, as it stands, timed on a bounded slice of the workload.

    The oracle's cost is linear in the vocabulary (LM-head and correction), so
    a sample keeps the first V_s vocabulary rows of lm_head/emb/fc2/b and one
    request, and its time is scaled by V / V_s to one block.  V_s is the whole
    vocabulary when one block fits the per-step budget.  Widening the weights
    to fp64 is the oracle's "load" and is done once, untimed.
    """

    def __init__(self, wl: inputs.Workload, weights: dict, requests: dict, budget_s: float):
        import numpy as np
        import oracle
        self.oracle = oracle
        self.wl = wl
        sh = wl.shape
        req = {k: v[:1] for k, v in requests.items()}
        Vs = min(sh.V, 8192)
        t = self._prepare_and_time(weights, req, Vs)
        target = max(Vs, min(sh.V, int(Vs * budget_s / max(t, 1e-3))))
        if target > Vs:
            Vs = target
            self._prepare_and_time(weights, req, Vs)
        self.Vs = Vs
        self.cores = len(os.sched_getaffinity(0))
        self.sample = (f"1 request, vocabulary rows 0..{Vs - 1} of {sh.V} ({Vs / sh.V:.1%}), fp64 numpy/OpenBLAS, "
                       f"time scaled by V/V_s to one block of {wl.B} request(s)")

    def _prepare_and_time(self, weights, req, Vs):
        import numpy as np
        w = dict(weights)
        for n in ("lm_head", "emb", "fc2", "b"):
            w[n] = weights[n][:Vs]
        r = dict(req)
        r["verified"] = (req["verified"] % Vs).astype(np.int32)
        self.Vs = Vs
        self.ow = self.oracle.OracleWeights(w)
        self.r = r
        self.K = self.wl.K if self.wl.K < Vs else 0
        return self.time_block() * Vs / self.wl.shape.V / self.wl.B

    def time_block(self) -> float:
        """Seconds for one block of the workload (all B requests), scaled."""
        t0 = time.perf_counter()
        self.oracle.rollout(self.ow, self.r["hidden"], self.r["s"], self.r["verified"], self.K)
        t = time.perf_counter() - t0
        return t * self.wl.shape.V / self.Vs * self.wl.B


def oracle_sample(wl: inputs.Workload, weights: dict, requests: dict, budget_s: float) -> dict:
    samp = OracleSample(wl, weights, requests, budget_s)
    ts = [samp.time_block() for _ in range(2)]
    s_block = min(ts)
    return {"value": 15.0 * wl.B / s_block, "unit": UNIT, "s_per_block": s_block, "cores": samp.cores,
            "kind": "oracle", "sample": samp.sample}


def run_reference(args):
    """The reference arm: the CPU oracle timed as it stands on the host cores."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = inputs.WORKLOADS[args.workload]
    weights, requests = inputs.make(wl, B=1)
    per_step = max(0.2, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    samp = OracleSample(wl, weights, requests, per_step)
    for _ in range(args.warmup):
        samp.time_block()
    ts = [samp.time_block() for _ in range(args.steps)]
    s_per_block = statistics.median(ts)
    value = 15.0 * wl.B / s_per_block
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": s_per_block * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": samp.cores, "kind": "oracle",
                             "sample": samp.sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl: inputs.Workload) -> dict:
    sh = wl.shape
    return {"workload": wl.name, "B": wl.B, "K": wl.K, "block": 16, "proposals": 15, "V": sh.V, "H": sh.H,
            "E": sh.E, "G": sh.G, "F": sh.F, "weights": sh.dtype, "accumulate": "fp32",
            "l2": "flushed between timed steps (512 MiB write)", "parallelism": "replicas (one per GPU)"}


# ---- our arm -------------------------------------------------------------------

def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    from speculative_decoding_draft_lm_gb300.rollout import DominoRollout, to_device

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()

    wl = inputs.WORKLOADS[args.workload]
    sh = wl.shape
    sweep = [] if args.no_sweep or rank != 0 else [n for n in SWEEP if inputs.WORKLOADS[n].shape == sh]
    max_B = max([wl.B] + [inputs.WORKLOADS[n].B for n in sweep])
    max_K = max([wl.K] + [inputs.WORKLOADS[n].K for n in sweep])
    weights = inputs.make_weights(sh, wl.weight_seed, wl.scales)
    # every rank runs its own requests (weak scaling of independent replicas)
    requests = inputs.make_requests(sh, replica_seeds(wl, rank))

    eng = DominoRollout(sh.V, sh.H, sh.E, sh.G, sh.F, max_B=max_B, max_K=max_K, dtype=sh.dtype, device=local)
    dw = {k: to_device(v) for k, v in weights.items()}
    eng.load_weights(dw)
    hid, s, ver = to_device(requests["hidden"]), to_device(requests["s"]), \
        torch.from_numpy(requests["verified"]).cuda()
    out = torch.empty((wl.B, 15), dtype=torch.int32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(h_, s_, v_, B, K):
        eng.run(h_, s_, v_, K=K, out=out[:B])

    # warm-up
    for _ in range(max(3, args.warmup)):
        step(hid, s, ver, wl.B, wl.K)
    torch.cuda.synchronize()
    if eng.status() != 0:
        raise RuntimeError("device error during warm-up")

    # timed region: K steps, each bracketed by CUDA events on the launching
    # stream, a 512 MiB write between steps so every step starts with a cold L2
    times = []
    launches = 0
    clocks = Clocks(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(hid, s, ver, wl.B, wl.K)
        e1.record(stream)
        launches += eng.last_launch_count()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    if eng.status() != 0:
        raise RuntimeError("device error during the timed steps")
    # second timed region of K steps with the library's per-launch events (they
    # separate consecutive launches, so they are kept out of the step time)
    eng.enable_timing(True)
    eng.read_timing()
    phase_ms = {}
    phase_n = {}
    for _ in range(args.steps):
        flush.zero_()
        step(hid, s, ver, wl.B, wl.K)
        torch.cuda.synchronize()
        for p_, (ms, n) in eng.read_timing().items():
            phase_ms[p_] = phase_ms.get(p_, 0.0) + ms
            phase_n[p_] = phase_n.get(p_, 0) + n
    eng.enable_timing(False)
    ms_step = max_over_ranks(sum(times) / len(times), dist, "cuda")
    value = whole_job_rate(wl.B, ws, ms_step)

    # end to end through the public API: pinned host inputs -> run -> tokens back
    h_host = torch.from_numpy(requests["hidden"].view(np.int16) if requests["hidden"].dtype == np.uint16
                              else requests["hidden"]).pin_memory()
    s_host = torch.from_numpy(requests["s"].view(np.int16) if requests["s"].dtype == np.uint16
                              else requests["s"]).pin_memory()
    v_host = torch.from_numpy(requests["verified"]).pin_memory()
    o_host = torch.empty((wl.B, 15), dtype=torch.int32).pin_memory()
    h_dev = torch.empty(h_host.shape, dtype=h_host.dtype, device="cuda")
    s_dev = torch.empty(s_host.shape, dtype=s_host.dtype, device="cuda")
    v_dev = torch.empty(v_host.shape, dtype=v_host.dtype, device="cuda")
    e2e_times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h_dev.copy_(h_host, non_blocking=True)
        s_dev.copy_(s_host, non_blocking=True)
        v_dev.copy_(v_host, non_blocking=True)
        hv = h_dev.view(torch.bfloat16) if sh.dtype == "bf16" else h_dev
        sv = s_dev.view(torch.bfloat16) if sh.dtype == "bf16" else s_dev
        eng.run(hv, sv, v_dev, K=wl.K, out=out)
        o_host.copy_(out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            e2e_times.append(e0.elapsed_time(e1))
    e2e_ms = max_over_ranks(sum(e2e_times) / len(e2e_times), dist, "cuda")
    h2d = h_host.numel() * h_host.element_size() + s_host.numel() * s_host.element_size() + v_host.numel() * 4
    d2h = o_host.numel() * 4

    # roofline of the dominant kernel (largest share of the timed phases)
    peaks, peak_src = load_peaks()
    ab = alg_bytes(sh, wl.B, wl.K)
    total_phase = sum(phase_ms.values()) or 1.0
    dom = max((p for p in phase_ms if phase_n.get(p)), key=lambda p: phase_ms[p])
    avg_ms = phase_ms[dom] / phase_n[dom]
    shares = {p: round(phase_ms[p] / total_phase, 4) for p in phase_ms if phase_n.get(p)}
    traffic = read_traffic(dom, wl.name)
    if dom == "lmhead" and wl.B >= 64:
        achieved = ab["lmhead_flop"] / (avg_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        per_launch = ab.get(dom, 0)
        achieved = per_launch / (avg_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    roof.update({"frac": roof["achieved"] / roof["peak"], "traffic": traffic, "kernel": dom,
                 "launches_per_step": phase_n[dom] / args.steps, "avg_launch_us": avg_ms * 1e3,
                 "timing": "CUDA events around each launch on the run's stream, second timed region of K steps",
                 "alg_bytes_per_launch": ab.get(dom), "peak_source": peak_src + " (MEASURED_PEAKS.json)"
                 if peak_src == "measured" else "fallback"})
    step_roof = {"alg_bytes_per_block": ab["block"],
                 "achieved_gbs": ab["block"] / (ms_step * 1e-3) / 1e9 * 1.0,
                 "hbm_peak_gbs": peaks["hbm_gbs"],
                 "frac": ab["block"] / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"],
                 "frac_of_8tbs": ab["block"] / (ms_step * 1e-3) / 1e9 / 8000.0}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "us_per_block": ms_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": sh.dtype,
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) hidden/s, uniform verified token)",
            "config": workload_config(wl),
            "e2e": {"value": whole_job_rate(wl.B, ws, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches, "clocks": clk, "roofline": roof, "step_roofline": step_roof,
            "phase_share": shares,
            "phase_us_per_step": {p: phase_ms[p] * 1e3 / args.steps for p in phase_ms if phase_n.get(p)},
            "context": {"pages_a100_tp1_ms": {"B1_K0": 2.363, "B8_K0": 2.881, "B64_K0": 7.808,
                                              "B1_K2048": 1.618, "B8_K2048": 2.122, "B64_K2048": 7.188},
                        "note": "A100 numbers at the pages' checkpoint shapes; context only"}}

    # B = 1/8/64 x K0/K2048 table on the same weights (rank 0), then the
    # early-stopped b8 variant (7 proposals) of the B = 1/8 workloads, then
    # K0 with s derived in the library from the backbone hidden rows
    if sweep:
        table = {}
        # (workload, proposals, s in the library, vocabulary shards of the pool)
        runs = ([(n, 15, False, 1) for n in sweep] +
                [(n, 7, False, 1) for n in sweep if inputs.WORKLOADS[n].B <= 8] +
                [(n, 15, True, 1) for n in sweep if inputs.WORKLOADS[n].K == 0] +
                [(n, 15, False, 2) for n in sweep if inputs.WORKLOADS[n].K > 0])
        if any(r_[2] for r_ in runs):
            w_hid = to_device(inputs.make_fc1_hidden(sh, seed=5))
            eng.load_backbone_proj(w_hid)
        for name, n_prop, own_s, parts in runs:
            w2 = inputs.WORKLOADS[name]
            eng.set_proposals(n_prop)
            eng.set_vocab_partitions(parts)
            rq = inputs.make_requests(sh, list(w2.request_seeds))
            h2, s2, v2 = to_device(rq["hidden"]), to_device(rq["s"]), torch.from_numpy(rq["verified"]).cuda()
            if own_s:
                s2 = None
            for _ in range(3):
                step(h2, s2, v2, w2.B, w2.K)
            n_sweep = max(5, args.steps // 2)
            # clean step times: no per-launch events (they would serialise the
            # programmatically dependent launches of the batched driver)
            tt = []
            for _ in range(n_sweep):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                step(h2, s2, v2, w2.B, w2.K)
                e1.record(stream)
                e1.synchronize()
                tt.append(e0.elapsed_time(e1))
            # separate pass for the per-phase breakdown
            eng.enable_timing(True)
            eng.read_timing()
            lm_ms, lm_n = 0.0, 0
            ph_ms = {}
            for _ in range(n_sweep):
                flush.zero_()
                step(h2, s2, v2, w2.B, w2.K)
                torch.cuda.synchronize()
                ph = eng.read_timing()
                lm_ms += ph["lmhead"][0]
                lm_n += ph["lmhead"][1]
                for k_, (m_, n_) in ph.items():
                    if n_:
                        ph_ms[k_] = ph_ms.get(k_, 0.0) + m_
            eng.enable_timing(False)
            ms = sum(tt) / len(tt)
            ab2 = alg_bytes(sh, w2.B, w2.K, n_prop, own_s)
            lm_avg = lm_ms / max(1, lm_n)
            label = (name + ("" if n_prop == 15 else f"_n{n_prop}") + ("_s_in_library" if own_s else "") +
                     ("" if parts == 1 else f"_compact_pool_p{parts}"))
            table[label] = {
                "us_per_block": ms * 1e3, "proposals": n_prop, "s": "in library" if own_s else "input",
                "vocab_partitions": parts,
                "proposals_per_s": float(n_prop) * w2.B / (ms * 1e-3),
                "hbm_frac_block": ab2["block"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "lmhead_us": lm_avg * 1e3,
                "lmhead_tensor_frac": ab2["lmhead_flop"] / (lm_avg * 1e-3) / 1e12 / peaks["bf16_tflops"],
                "phase_us_timed_pass": {k_: m_ * 1e3 / n_sweep for k_, m_ in ph_ms.items()}}
        eng.set_proposals(15)
        eng.set_vocab_partitions(1)
        torch.cuda.synchronize()
        if eng.status() != 0:
            raise RuntimeError("device error during the sweep")
        line["by_workload"] = table

    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample(wl, weights, requests, args.cpu_budget_s)
    if rank == 0:
        print(json.dumps(line), flush=True)
    eng.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def read_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it matches the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    ent = t.get(workload, {}).get(kernel)
    if not ent:
        return None
    if ent.get("source_hash") != source_hash(ent.get("files")):
        return None
    return ent.get("dram_bytes_per_launch")


def source_hash(files=None) -> str:
    """Hash of the kernel sources (all of them, or the listed files of the
    captured kernel) with // comments and blank lines dropped, so that a
    comment edit, or an edit of another kernel, does not orphan the committed
    counters."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_draft_lm_gb300", "csrc")
    for f in sorted(files or os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                code = [re.sub(r"\s*//.*$", "", ln).rstrip() for ln in fh]
            h.update(f.encode() + b"\0" + "\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    sys.exit(main())
