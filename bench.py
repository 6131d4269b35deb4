#!/usr/bin/env python3
"""Attention throughput on GB300: one step = forward + backward (D pre-pass, then
the dK/dV and dQ kernels for d = 64, 128, or the one launch of dK, dV and dQ CTAs
for d = 256) of exact causal attention over one batch.

Workload (default): B=2, H=16, N=8192, d=128, bf16, causal, Q/K/V = 0.5*N(0,1),
dO = N(0,1) (seeded, synthetic).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

FLOP accounting: forward 4*B*H*N^2*d, backward 2.5x that, both halved under the
causal mask.  ``value`` is forward+backward TFLOP/s with inputs resident in
device memory; ``e2e`` is the same metric through the C-ABI with host buffers
(pinned host->device copies of Q, K, V, dO and device->host copies of O, L, dQ,
dK, dV inside the timed region).  L2 is flushed (a 256 MB write) before every
timed step.  The secondary bound, the exponentials (one per visible pair in each
pass), is reported as exp/s and as a fraction of the MUFU rate at the sampled SM
clock.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

METRIC = "attention TFLOP/s fwd and fwd+bwd (bf16, causal/non-causal) and % of GB300 peak"
UNIT = "TFLOP/s"


def attention_flops(w, backward=True):
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    if w.causal:
        f /= 2
    return f * (3.5 if backward else 1.0)


def load_peaks():
    p = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def sources_sha256(paths):
    """sha256 over the listed files' bytes, in order (paths relative to the repo root)."""
    import hashlib

    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(HERE, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic(kernel_tag):
    """DRAM bytes per launch of a kernel from its committed ncu summary, if none of the
    sources the kernel was built from has changed since the capture (else None).

    The summary lists ``- source: `a`, `b` ...`` (comma-separated, repo-relative),
    ``- source_sha256: `...` `` (over those files in order) and
    ``- traffic_bytes_per_launch: `...` ``.
    """
    summ = os.path.join(HERE, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(summ):
        return None
    fields = {}
    for line in open(summ):
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip()
    srcs = [x.strip().strip("`") for x in fields.get("source", "").split(",") if x.strip()]
    want = fields.get("source_sha256", "").strip("`")
    tb = fields.get("traffic_bytes_per_launch", "").strip("`")
    if not (srcs and want and tb):
        return None
    if not all(os.path.exists(os.path.join(HERE, x)) for x in srcs) or sources_sha256(srcs) != want:
        return None
    try:
        return float(tb)
    except ValueError:
        return None


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, sampled every few
    milliseconds by a host thread through NVML (the driver's libnvidia-ml, read
    only), from before the warm-up until after the e2e leg.  Samples taken while
    ``busy`` is set (a timed region is running) are the ones under load.  Falls
    back to an ``nvidia-smi --query-gpu`` loop if NVML cannot be opened."""

    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    QUERY = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, pci_bus_id, uuid=None, period_s=0.004):
        self.pci = pci_bus_id
        self.uuid = uuid
        self.period = period_s
        self.samples = []  # (busy, sm_mhz, reason bits)
        self.max_mhz = None
        self.busy = False
        self.source = None
        self._stop = False
        self._thread = None
        self._proc = None

    def _nvml(self):
        import ctypes

        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        found = lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci.encode(), ctypes.byref(h)) == 0
        if not found and self.uuid:
            found = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not found:
            raise OSError("no NVML handle for " + self.pci)
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = SM clock
            self.max_mhz = float(mx.value)
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, get_reasons

    def __enter__(self):
        import threading

        try:
            lib, h, get_reasons = self._nvml()
            self.source = "nvml"

            def run():
                import ctypes

                mhz, bits = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop:
                    busy = self.busy
                    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                        r = get_reasons(h, ctypes.byref(bits))
                        self.samples.append((busy, float(mhz.value), int(bits.value) if r == 0 else 0))
                    time.sleep(self.period)

            self._thread = threading.Thread(target=run, daemon=True)
            self._thread.start()
        except Exception:
            self._start_smi()
        return self

    def _start_smi(self):
        import threading

        try:
            self._proc = subprocess.Popen(["nvidia-smi", "-i", self.pci, f"--query-gpu={self.QUERY}",
                                           "--format=csv,noheader,nounits", "-lms", "20"],
                                          stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self._proc = None
            return
        self.source = "nvidia-smi"
        bits = (0x8, 0x40, 0x20, 0x4)

        def run():
            for line in self._proc.stdout:
                parts = [p.strip() for p in line.split(",")]
                try:
                    mhz, self.max_mhz = float(parts[0]), float(parts[1])
                except (ValueError, IndexError):
                    continue
                r = sum(b for b, v in zip(bits, parts[2:6]) if v.lower() == "active")
                self.samples.append((self.busy, mhz, r))

        self._thread = threading.Thread(target=run, daemon=True)
        self._thread.start()

    def __exit__(self, *exc):
        self._stop = True
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no clock samples"], "samples": 0}
        load = [s for s in self.samples if s[0]] or self.samples
        reasons = sorted({n for _, _, r in load for b, n in self.REASONS.items() if r & b})
        return {"sm_mhz": statistics.median(m for _, m, _ in load), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(m for _, m, _ in load), "reasons": reasons, "samples": len(load),
                "samples_total": len(self.samples), "source": self.source}


def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(x, world, device):
    """Max of a float over ranks (control plane only; the attention work exchanges nothing)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ex2.approx.f32 throughput measured on this part (one probe CTA per SM): the
# secondary bound of the method, one exponential per visible (query, key) pair.
MUFU_EX2_PER_CLK_PER_SM = 32


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (the model name, or on Arm the
    implementer and part codes), for the CPU baseline's record."""
    import platform

    try:
        lines = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.processor() or platform.machine()
    for key in ("model name", "Model"):
        for line in lines:
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    found = {}
    for line in lines:
        for key in ("CPU implementer", "CPU part"):
            if line.startswith(key) and ":" in line and key not in found:
                found[key] = line.split(":", 1)[1].strip()
    return f"{platform.machine()}, implementer {found.get('CPU implementer', '?')}, part {found.get('CPU part', '?')}"


def visible_pairs(w, rows):
    """(query, key) pairs the mask leaves visible in the given query rows of one head."""
    import numpy as np

    rows = np.asarray(rows, dtype=np.int64)
    if not w.causal:
        return int(rows.size) * w.kv_len
    return int(np.clip(rows + (w.kv_len - w.N) + 1, 0, w.kv_len).sum())


def oracle_rows(w, q, k, v, do, bh, rows, backward, chunk=1024):
    """Run the oracle (as it stands) on some query rows of one head, `chunk` rows at a time;
    returns the algorithmic FLOPs of those rows (4d per visible pair forward, 10d backward)."""
    import numpy as np

    import oracle

    b, h = divmod(bh, w.H)
    g = h // (w.H // w.kv_heads)
    for r0 in range(0, len(rows), chunk):
        rr = np.asarray(rows[r0:r0 + chunk])
        oracle.forward_rows(q[b, h], k[b, g], v[b, g], w.scale, w.causal, rr)
        if backward:
            oracle.head_backward_rows(q[b, h], k[b, g], v[b, g], do[b, h], w.scale, w.causal, rr)
    return visible_pairs(w, rows) * w.d * (14 if backward else 4)


def cpu_oracle_sample(w, q, k, v, do, backward=True, min_seconds=10.0):
    """Time the oracle on whole heads of the workload, head after head, until at least
    `min_seconds` of CPU work; returns (TFLOP/s, seconds, heads)."""
    import numpy as np

    rows = np.arange(w.N)
    flops, heads = 0, 0
    t0 = time.perf_counter()
    while True:
        flops += oracle_rows(w, q, k, v, do, heads % (w.B * w.H), rows, backward)
        heads += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            return flops / dt / 1e12, dt, heads


def run_reference(args, w, backward):
    """The reference arm: the fp64 oracle as it stands, on the host cores.  Each step is a
    strided sample of query rows of one head (forward, and backward if the workload has
    one), sized so that warm-up plus timed steps take about two minutes in all."""
    import numpy as np

    from exact_attention_37_gb300.synth import make_inputs

    world, rank, _ = dist_setup()
    if rank != 0:
        return
    q, k, v, do = make_inputs(w.with_(B=1, H=min(w.H, 4), H_kv=None if w.H_kv is None else 1), with_dout=True)
    ws = w.with_(B=1, H=q.shape[1], H_kv=None if w.H_kv is None else 1)
    budget = 120.0 / (args.steps + args.warmup)
    t0 = time.perf_counter()
    oracle_rows(ws, q, k, v, do, 0, np.arange(0, w.N, max(1, w.N // 64)), backward)
    per_row = (time.perf_counter() - t0) / len(range(0, w.N, max(1, w.N // 64)))
    R = int(min(w.N, max(8, budget / max(per_row, 1e-9))))
    spread = max(1, w.N // R)

    def one(i):
        rows = np.unique((i % spread + (np.arange(R) * w.N) // R) % w.N)
        t = time.perf_counter()
        f = oracle_rows(ws, q, k, v, do, i % (ws.B * ws.H), rows, backward)
        return f, time.perf_counter() - t

    for i in range(args.warmup):
        one(i)
    flops, secs = 0, []
    for i in range(args.steps):
        f, dt = one(args.warmup + i)
        flops += f
        secs.append(dt)
    value = flops / sum(secs) / 1e12
    sample = (f"{R} evenly spaced query rows of one head per step, forward"
              f"{' + backward' if backward else ''}, fp64 numpy; FLOPs of the rows' visible pairs")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "input_dtype": w.dtype, "step": "fwd + bwd" if backward else "fwd"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "cpu": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_B2_H16_N8192_d128_bf16_causal")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--causal", type=int, choices=[0, 1], default=None, help="override the workload's mask")
    ap.add_argument("--fwd-only", action="store_true", help="time the forward pass alone (default for forward-only workloads)")
    ap.add_argument("--chunks", type=int, default=0, help="head chunks of the host-buffer (e2e) pipeline; 0 = library default")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from exact_attention_37_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    profile_key = w.name.split("_")[0]
    if args.causal is not None and bool(args.causal) != w.causal:
        base = w.name[: -len("_causal")] if w.name.endswith("_causal") else w.name
        w = w.with_(causal=bool(args.causal), name=base + ("_causal" if args.causal else ""))
        profile_key += "_causal" if args.causal else "_full"
    fwd_only = args.fwd_only or not w.backward
    if args.impl == "reference":
        run_reference(args, w, backward=not fwd_only)
        return

    import torch

    import exact_attention_37_gb300 as fa
    from exact_attention_37_gb300 import build

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    fa.load()

    q, k, v, do = synth.make_inputs(w, with_dout=True)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    B, H, N, d = qd.shape
    od = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    if fwd_only:
        dq = dk = dv = ws = None
    else:
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def run_bwd():
        if not fwd_only:
            fa.fa_bwd(qd, kd, vd, od, dod, lse, dq, dk, dv, ws, w.scale, w.causal)

    def step():
        fa.fa_fwd(qd, kd, vd, od, lse, w.scale, w.causal)
        run_bwd()

    props = torch.cuda.get_device_properties(dev)
    pci = getattr(props, "pci_bus_id", None)
    pci = (f"{getattr(props, 'pci_domain_id', 0):08x}:{pci:02x}:{getattr(props, 'pci_device_id', 0):02x}.0"
           if isinstance(pci, int) else str(local))
    uuid = getattr(props, "uuid", None)
    uuid = None if uuid is None else (str(uuid) if str(uuid).startswith("GPU-") else f"GPU-{uuid}")
    clocks = ClockSampler(pci, uuid)
    clocks.__enter__()
    try:
        for _ in range(args.warmup):
            flush.zero_()
            step()
        fa.fa_check_device_status()

        K = args.steps
        n_launch = 1 if fwd_only else (3 if d in (64, 128) else 2)  # main-kernel launches per step
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        fa.fa_profile_begin(n_launch * K)
        barrier(world)
        torch.cuda.synchronize()
        clocks.busy = True
        for i in range(K):
            flush.zero_()
            e0, e1, e2 = ev[i]
            e0.record(stream)
            fa.fa_fwd(qd, kd, vd, od, lse, w.scale, w.causal)
            e1.record(stream)
            run_bwd()
            e2.record(stream)
        torch.cuda.synchronize()
        clocks.busy = False
        barrier(world)
        kernels = fa.fa_profile_end()
        fa.fa_check_device_status()
        step_ms = [e[0].elapsed_time(e[2]) for e in ev]
        fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
        bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
        per_kind = {}
        for kind, ms in kernels:
            per_kind.setdefault(kind, []).append(ms)
        total_ms = reduce_max(sum(step_ms), world, dev)
        ms_per_step = total_ms / K

        flops_fwd = attention_flops(w, backward=False)
        flops_step = flops_fwd if fwd_only else attention_flops(w)
        value = world * flops_step * K / (total_ms / 1e3) / 1e12

        # ---- end to end through the C ABI with host buffers: fa_fwd_host / fa_fwd_bwd_host take
        # pinned host tensors and pipeline head chunks (copies in, kernels, copies out) on the
        # library's streams; the caller's stream waits for the whole step
        pin = lambda t: t.pin_memory()
        qh, kh, vh, doh = (pin(x) for x in (q, k, v, do))
        oh = torch.empty_like(q).pin_memory()
        lseh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        host_in = [qh, kh, vh] + ([] if fwd_only else [doh])
        host_out = [oh, lseh]
        if not fwd_only:
            dqh, dkh, dvh = (torch.empty_like(x).pin_memory() for x in (q, k, v))
            host_out += [dqh, dkh, dvh]
        h2d = sum(x.numel() * x.element_size() for x in host_in)
        d2h = sum(x.numel() * x.element_size() for x in host_out)
        scratch = torch.empty(fa.fa_host_scratch_size(B, H, N, d, not fwd_only), dtype=torch.uint8, device=dev)

        def host_step():
            if fwd_only:
                fa.fa_fwd_host(qh, kh, vh, oh, lseh, scratch, w.scale, w.causal, args.chunks)
            else:
                fa.fa_fwd_bwd_host(qh, kh, vh, doh, oh, lseh, dqh, dkh, dvh, scratch, w.scale, w.causal,
                                   args.chunks)

        for _ in range(2):
            host_step()
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        torch.cuda.synchronize()
        barrier(world)
        clocks.busy = True
        for i in range(K):
            flush.zero_()
            e2e_ev[i][0].record(stream)
            host_step()
            e2e_ev[i][1].record(stream)
        torch.cuda.synchronize()
        clocks.busy = False
        barrier(world)
        fa.fa_check_device_status()
    finally:
        clocks.__exit__(None, None, None)
    e2e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_ev), world, dev)
    e2e_value = world * flops_step * K / (e2e_ms / 1e3) / 1e12
    # spread of the single steps (rank 0): the host copies' speed varies from run to run
    e2e_steps = sorted(a.elapsed_time(b) for a, b in e2e_ev)

    # ---- roofline: every main kernel on its own, the dominant one as the `roofline` entry.
    # Algorithmic FLOPs (forward 4d per visible pair, backward 10d: the five products S, dP,
    # dV, dK, dQ at 2d each) are attributed to the kernel that produces the product's
    # result for an output: the dK/dV kernel owns S, dP, dV, dK (4 of the 5), the dQ
    # kernel only dQ (its S and dP are recomputation: executed, not algorithmic); the
    # single d = 256 backward launch owns all five.  `executed_tflops` counts every
    # product a kernel runs: 3 of 5 for the dQ kernel; for d = 256, 8 of 5 (S in the
    # dK, dV and dQ CTAs, dP in the dK and dQ CTAs, and the three gradients).
    peaks, peak_src = load_peaks()
    timed_s = total_ms / 1e3
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    # a timed region under a second is a burst; seconds-long loops settle at the sustained rate
    peak, peak_kind = (burst, "burst") if timed_s < 1.0 else (sustained, "sustained")
    flops_bwd = attention_flops(w) - flops_fwd
    own = {"fwd": (flops_fwd, flops_fwd), "bwd_kv": (0.8 * flops_bwd, 0.8 * flops_bwd),
           "bwd_q": (0.2 * flops_bwd, 0.6 * flops_bwd), "bwd_fused": (flops_bwd, 1.6 * flops_bwd)}
    names = {"fwd": "fa_fwd_kernel", "bwd_kv": "fa_bwd_kv_kernel", "bwd_q": "fa_bwd_q_kernel",
             "bwd_fused": "fa_bwd256_kernel"}
    kern = {}
    for kind, lst in per_kind.items():
        ms = statistics.mean(lst)
        alg, exe = own[kind]
        kern[names[kind]] = {"ms": ms, "launches": len(lst), "algorithmic_tflop": alg / 1e12,
                             "tflops": alg / (ms / 1e3) / 1e12, "frac": alg / (ms / 1e3) / 1e12 / peak,
                             "executed_tflops": exe / (ms / 1e3) / 1e12}
    dom = max(kern, key=lambda n: kern[n]["ms"])
    fwd_avg = kern["fa_fwd_kernel"]["ms"]
    bwd_main_avg = sum(kern[n]["ms"] for n in kern if n != "fa_fwd_kernel")
    tag = f"{dom}_{profile_key}"
    roofline = {"bound": "tensor", "kernel": dom, "achieved": kern[dom]["tflops"], "peak": peak,
                "unit": "TFLOP/s", "frac": kern[dom]["frac"], "traffic": profile_traffic(tag),
                "peak_source": f"{peak_src} bf16 {peak_kind} ({peak_kind} peak: the timed region is "
                               f"{timed_s:.2f} s)",
                "frac_of_sustained": kern[dom]["tflops"] / sustained, "kernels": kern}
    if not fwd_only:
        pair = flops_bwd / (bwd_main_avg / 1e3) / 1e12
        roofline["bwd_main"] = {"ms": bwd_main_avg, "tflops": pair, "frac": pair / peak,
                                "kernels": [n for n in kern if n != "fa_fwd_kernel"]}
    fwd_tflops = flops_fwd / (fwd_avg / 1e3) / 1e12

    # Exponentials: one per visible pair in the forward pass and the same again in
    # the backward pass (algorithmic counts; the backward kernels evaluate them more
    # than once).  Peak: the MUFU rate at the SM clock sampled under load.
    clk = clocks.summary()
    sm_mhz = clk.get("sm_mhz") or clk.get("sm_max_mhz")
    if sm_mhz:
        clk["ms_x_mhz_per_step"] = ms_per_step * sm_mhz
    n_sms = props.multi_processor_count
    mufu_peak = MUFU_EX2_PER_CLK_PER_SM * n_sms * sm_mhz * 1e6 if sm_mhz else None
    exps = B * H * visible_pairs(w, range(w.N))

    def exp_rate(ms):
        r = exps / (ms / 1e3)
        return {"exp_per_s": r, "exp_frac_of_mufu": (r / mufu_peak) if mufu_peak else None}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cv, cdt, heads = cpu_oracle_sample(w, q, k, v, do, backward=not fwd_only)
        cpu = {"value": cv, "unit": UNIT, "cores": os.cpu_count(), "cpu": cpu_model(), "kind": "oracle",
               "sample": f"{heads} head(s) of the {w.B * w.H}, forward{'' if fwd_only else ' + backward'}, "
                         f"fp64 numpy, {cdt:.1f} s; FLOPs of the visible pairs"}

    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": d, "causal": w.causal,
                       "step": "fwd" if fwd_only else ("fwd + bwd (pre, dK/dV kernel, dQ kernel)" if d in (64, 128)
                                                        else "fwd + bwd (pre, one launch of dK, dV and dQ CTAs)"),
                       "l2": "256 MB flush write before every step", "parallelism": f"replicas x{world}"},
            "fwd": {"tflops": fwd_tflops, "ms": fwd_avg, "frac_of_peak_burst": fwd_tflops / burst,
                    **exp_rate(fwd_avg)},
            "bwd": None if fwd_only else {
                "tflops": flops_bwd / (statistics.mean(bwd_ms) / 1e3) / 1e12, "ms": statistics.mean(bwd_ms),
                "main_kernels_ms": bwd_main_avg,
                "main_kernels_frac_of_peak_burst": flops_bwd / (bwd_main_avg / 1e3) / 1e12 / burst,
                **exp_rate(bwd_main_avg)},
            "mufu_peak_exp_per_s": mufu_peak,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms / K,
                    "step_ms_min_median_max": [e2e_steps[0], statistics.median(e2e_steps), e2e_steps[-1]],
                    "path": f"{'fa_fwd_host' if fwd_only else 'fa_fwd_bwd_host'} (C ABI, pinned host buffers, "
                            f"{args.chunks if args.chunks > 0 else 'default'} head chunks)"},
            "gpu_launches": (1 if fwd_only else n_launch + 1) * K,  # + the D pre-pass
            "clocks": clk,
        }
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
