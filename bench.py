"""Benchmark of the attention hot path on GB300, one JSON line on stdout.

Step = one forward + one backward (fa_fwd, fa_bwd) of the workload the metric
is quoted on: causal bf16 attention, B=2, H=16, S=8192, d=128, Q drawn x8 so
raw logits reach ~+-100, batch row 0 with keys 0..63 padded (its first 64
query rows see no key).  Inputs are seeded synthetic tensors from
io_aware_exact_tcgen05_gb300.workloads.  FLOPs follow the metric's formula:
forward 4*B*H*Sq*Sk*d / 2 (causal), backward 2.5x that.

The same run also times the Sq=1 decode path (fa_decode) on the ragged KV
cache workload (B=32, Hq=32, Hkv=8, d=128, Sk in [1024, 32768]) and reports
its GB/s against the HBM roofline, and the CPU oracle on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With N > 1 (torchrun), every rank runs an independent replica of the step
(the path shards by batch/head with no exchange), value = all ranks' FLOPs /
max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from io_aware_exact_tcgen05_gb300 import workloads  # noqa: E402

METRIC = "attention TFLOP/s fwd & fwd+bwd, causal bf16 d=128 S=8192; % of BF16 tensor peak"
WORKLOAD = "prefill_8k_masked"
DECODE = "decode_ragged"
L2_BYTES = 129 * 1024 * 1024
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

THROTTLE_BITS = {
    0x0000000000000001: "gpu_idle",
    0x0000000000000002: "applications_clocks_setting",
    0x0000000000000004: "sw_power_cap",
    0x0000000000000008: "hw_slowdown",
    0x0000000000000010: "sync_boost",
    0x0000000000000020: "sw_thermal_slowdown",
    0x0000000000000040: "hw_thermal_slowdown",
    0x0000000000000080: "hw_power_brake_slowdown",
    0x0000000000000100: "display_clock_setting",
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled every 5 ms through
    NVML while the timed region runs (read-only queries; nothing is set)."""

    NVML_CLOCK_SM = 1

    def __init__(self, cuda_index: int, period_s: float = 0.005):
        self.cuda_index = cuda_index
        self.period = period_s
        self.samples = []  # (sm_mhz, reasons_bitmask)
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._lib = None
        self._dev = None

    def _open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        props = torch.cuda.get_device_properties(self.cuda_index)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        dev = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(dev)) != 0:
            raise RuntimeError(f"no NVML handle for {bus}")
        mx = ctypes.c_uint(0)
        if lib.nvmlDeviceGetMaxClockInfo(dev, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._lib, self._dev = lib, dev

    def _loop(self):
        import ctypes
        lib, dev = self._lib, self._dev
        clk = ctypes.c_uint(0)
        rs = ctypes.c_ulonglong(0)
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            ok = lib.nvmlDeviceGetClockInfo(dev, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0
            okr = get_reasons(dev, ctypes.byref(rs)) == 0
            if ok:
                self.samples.append((float(clk.value), int(rs.value) if okr else 0))
            time.sleep(self.period)

    def __enter__(self):
        try:
            self._open()
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        except (OSError, RuntimeError, AttributeError) as e:
            self.error = str(e)
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz,
                    "reasons": [f"unavailable: {self.error}" if self.error else "no samples"]}
        reasons = set()
        for _, mask in self.samples:
            for bit, name in THROTTLE_BITS.items():
                if mask & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "NVML, 5 ms, during the timed steps"}


def _kernel_source_hash(name: str) -> str:
    path = os.path.join(ROOT, "io_aware_exact_tcgen05_gb300", "csrc", name)
    with open(path, "rb") as f:
        h = hashlib.sha256(f.read())
    with open(os.path.join(ROOT, "io_aware_exact_tcgen05_gb300", "csrc", "sm103_ptx.cuh"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str, source: str):
    """DRAM bytes per launch from the committed ncu summary, only when the
    summary was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = _kernel_source_hash(source)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and parts[0] == kernel and parts[1] == want:
                return float(parts[2])
    return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _sync_max(value: float, ws: int) -> float:
    """Max over ranks (the slowest replica sets the job time)."""
    if ws == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def job_tflops(flops_per_rank: float, ms_per_step_max: float, ws: int) -> float:
    """Whole-job throughput: every replica processes the same step, the job
    takes as long as the slowest rank."""
    return ws * flops_per_rank / (ms_per_step_max * 1e-3) / 1e12


# --------------------------------------------------------------- CPU oracle --

def cpu_oracle_sample(w, budget_s: float = 12.0):
    """Time the FP64 oracle's forward + backward on whole heads of the workload
    (batch row 0, heads 0, 1, ...) until `budget_s` has elapsed (at least one
    head).  Returns (TFLOP/s by the metric's formula, threads, sample text)."""
    from oracle import oracle as orc
    t = w.tensors
    flops = 0.0
    heads = 0
    t0 = time.perf_counter()
    ks = t.get("k_start")
    ke = t.get("k_end")
    while heads < w.Hq:
        b, h = 0, heads
        hk = h // (w.Hq // w.Hkv)
        q = t["q"][b:b + 1, h:h + 1]
        k = t["k"][b:b + 1, hk:hk + 1]
        v = t["v"][b:b + 1, hk:hk + 1]
        do = t["dout"][b:b + 1, h:h + 1]
        kst = None if ks is None else ks[b:b + 1]
        ken = None if ke is None else ke[b:b + 1]
        orc.fwd(q, k, v, w.causal, w.scale, k_start=kst, k_end=ken)
        orc.bwd(q, k, v, do, w.causal, w.scale, k_start=kst, k_end=ken)
        heads += 1
        flops += 3.5 * 4.0 * w.Sq * w.Sk * w.d / (2 if w.causal else 1)
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, orc.num_threads(), (
        f"oracle fwd+bwd of {heads} whole head(s) (batch row 0) of the "
        f"{WORKLOAD} workload, {dt:.1f} s")


def oracle_step_sample(w, i: int, rows: int = 2048):
    """One bounded sample of the workload for the reference arm: the last
    `rows` query rows of head i (batch row 0) against all keys, forward and
    backward on the FP64 oracle.  Under the causal rule aligned to the
    bottom-right corner these rows see exactly the keys they see in the full
    problem.  Returns (seconds, FLOPs by the metric's formula)."""
    from oracle import oracle as orc
    t = w.tensors
    h = i % w.Hq
    hk = h // (w.Hq // w.Hkv)
    q = t["q"][0:1, h:h + 1, w.Sq - rows:]
    k = t["k"][0:1, hk:hk + 1]
    v = t["v"][0:1, hk:hk + 1]
    do = t["dout"][0:1, h:h + 1, w.Sq - rows:]
    ks = t.get("k_start")
    ke = t.get("k_end")
    kst = None if ks is None else ks[0:1]
    ken = None if ke is None else ke[0:1]
    t0 = time.perf_counter()
    orc.fwd(q, k, v, w.causal, w.scale, k_start=kst, k_end=ken)
    orc.bwd(q, k, v, do, w.causal, w.scale, k_start=kst, k_end=ken)
    dt = time.perf_counter() - t0
    off = w.Sk - w.Sq
    visible = sum(min(w.Sk, i2 + off + 1) for i2 in range(w.Sq - rows, w.Sq))
    return dt, 3.5 * 4.0 * visible * w.d


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    w = workloads.make(WORKLOAD)
    from oracle import oracle as orc
    orc.build()
    for i in range(args.warmup):
        oracle_step_sample(w, i)
    vals = []
    t0 = time.perf_counter()
    for i in range(args.steps):
        dt, fl = oracle_step_sample(w, args.warmup + i)
        vals.append(fl / dt / 1e12)
    dt = time.perf_counter() - t0
    value = statistics.median(vals)
    threads = orc.num_threads()
    sample = (f"per step: oracle fwd+bwd of the last 2048 query rows of one head (batch "
              f"row 0) of the {WORKLOAD} workload against all 8192 keys")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1000 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: {workloads.DESCRIPTIONS[WORKLOAD]}",
                   "step": "last 2048 query rows of one head, fwd+bwd, on the host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm --

def run_ours(args):
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import io_aware_exact_tcgen05_gb300 as fa
    fa.load_library()
    dev = torch.device("cuda", local)
    peaks, peak_src = _peaks()

    w = workloads.make(WORKLOAD)
    t = w.tensors
    q, k, v, do = (t[n].to(dev) for n in ("q", "k", "v", "dout"))
    kst = t["k_start"].to(dev)
    ken = t["k_end"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = torch.empty(fa.fa_bwd_workspace_size(w.B, w.Hq, w.Sq, w.d), dtype=torch.uint8,
                      device=dev)
    f_fwd, f_bwd = w.flops_fwd(), w.flops_bwd()
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            fa.fa_profile_next_launch(ev[0], ev[1])
        fa.fa_fwd(q, k, v, True, w.scale, k_start=kst, k_end=ken, o=o, lse=lse)
        if ev is not None:
            fa.fa_profile_next_launch(ev[2], ev[3])
        fa.fa_bwd(q, k, v, o, do, lse, True, w.scale, k_start=kst, k_end=ken, dq=dq, dk=dk,
                  dv=dv, workspace=wsb)

    launches_per_step = 1 + 3  # fa_fwd: 1 kernel; fa_bwd: preprocess, main, convert

    for _ in range(max(3, args.warmup)):
        step()
    st, word = fa.fa_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {word:#x}")

    evs = []
    for _ in range(args.steps):
        e4 = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in e4:
            e.record()  # creates the event; the library records it again
        evs.append(e4)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    _barrier(ws)
    with ClockSampler(local) as clocks:
        _barrier(ws)
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        stop.record(stream)
        _barrier(ws)
    total_ms = _sync_max(start.elapsed_time(stop), ws)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    st, word = fa.fa_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {word:#x}")

    ms_per_step = total_ms / args.steps
    value = job_tflops(f_fwd + f_bwd, ms_per_step, ws)
    peak_t = peaks["bf16_tflops"]
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12

    # ---- end to end through the public API: pinned host -> device, compute,
    #      device -> host of the step's results
    host_in = {n: t[n].pin_memory() for n in ("q", "k", "v", "dout")}
    host_out = {"o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                "lse": torch.empty(lse.shape, dtype=lse.dtype).pin_memory(),
                "dq": torch.empty(dq.shape, dtype=dq.dtype).pin_memory(),
                "dk": torch.empty(dk.shape, dtype=dk.dtype).pin_memory(),
                "dv": torch.empty(dv.shape, dtype=dv.dtype).pin_memory()}
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in host_out.values())

    # Two device copies of every input and result, so that step i+1's inputs
    # are copied in (stream s_in) and step i-1's results copied out (stream
    # s_out) while step i computes: every step still moves its own inputs in
    # from pinned host memory and its own results back out.
    dev_in = [{"q": q, "k": k, "v": v, "dout": do},
              {n: torch.empty_like(x) for n, x in (("q", q), ("k", k), ("v", v), ("dout", do))}]
    dev_out = [{"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv},
               {n: torch.empty_like(x) for n, x in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk),
                                                    ("dv", dv))}]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def copy_in(b):
        for n in ("q", "k", "v", "dout"):
            dev_in[b][n].copy_(host_in[n], non_blocking=True)

    def copy_out(b):
        for n in host_out:
            host_out[n].copy_(dev_out[b][n], non_blocking=True)

    def compute(b):
        x, y = dev_in[b], dev_out[b]
        fa.fa_fwd(x["q"], x["k"], x["v"], True, w.scale, k_start=kst, k_end=ken, o=y["o"],
                  lse=y["lse"])
        fa.fa_bwd(x["q"], x["k"], x["v"], y["o"], x["dout"], y["lse"], True, w.scale,
                  k_start=kst, k_end=ken, dq=y["dq"], dk=y["dk"], dv=y["dv"], workspace=wsb)

    def e2e_serial(n_steps):
        for _ in range(n_steps):
            copy_in(0)
            compute(0)
            copy_out(0)

    def e2e_overlapped(n_steps):
        in_ready = [torch.cuda.Event(), torch.cuda.Event()]
        comp_done = [torch.cuda.Event(), torch.cuda.Event()]
        out_done = [torch.cuda.Event(), torch.cuda.Event()]
        used = [False, False]
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        with torch.cuda.stream(s_in):
            copy_in(0)
            in_ready[0].record(s_in)
        for i in range(n_steps):
            b = i % 2
            stream.wait_event(in_ready[b])
            if used[b]:
                stream.wait_event(out_done[b])  # step i-2's results have left buffer b
            compute(b)
            comp_done[b].record(stream)
            if i + 1 < n_steps:
                nb = 1 - b
                if used[nb]:
                    s_in.wait_event(comp_done[nb])  # step i-1 has read buffer nb
                with torch.cuda.stream(s_in):
                    copy_in(nb)
                    in_ready[nb].record(s_in)
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                copy_out(b)
                out_done[b].record(s_out)
            used[b] = True
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    def timed(fn):
        fn(max(3, args.warmup))
        _barrier(ws)
        s2 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        fn(args.steps)
        e2.record(stream)
        _barrier(ws)
        return _sync_max(s2.elapsed_time(e2), ws) / args.steps

    e2e_serial_ms = timed(e2e_serial)
    e2e_ms = timed(e2e_overlapped)
    e2e_value = job_tflops(f_fwd + f_bwd, e2e_ms, ws)

    # ---- the widened rows (key masks, dropout, packed varlen), timed alone
    nxt = None
    if not args.skip_next:
        nxt = next_rows_bench(fa, dev, peaks, w, q, k, v, do, kst, ken, o, lse, dq, dk, dv, wsb)

    # ---- decode (Sq = 1 over the ragged cache), timed alone
    dec = None
    if not args.skip_decode:
        dec = decode_bench(fa, dev, peaks, args, ws)

    del host_in, host_out
    line = None
    if rank == 0:
        cpu = None
        if ws == 1 and not args.skip_cpu:
            v_cpu, threads, sample = cpu_oracle_sample(w, budget_s=args.cpu_budget)
            cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": sample}
        trafficb = _traffic("fa_bwd_main", "fa_bwd.cu")
        trafficf = _traffic("fa_fwd_kernel", "fa_fwd.cu")
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {
                "workload": f"{WORKLOAD}: {workloads.DESCRIPTIONS[WORKLOAD]}",
                "step": "fa_fwd + fa_bwd",
                "l2": "inputs larger than L2: Q, K, V, dO, O = 335 MB read per step, no flush",
                "seed": 0, "parallelism": f"replicas x{ws}",
            },
            "fwd_tflops": fwd_tf, "fwd_frac_of_peak": fwd_tf / peak_t,
            "bwd_tflops": bwd_tf, "bwd_frac_of_peak": bwd_tf / peak_t,
            "fwd_bwd_tflops": value / ws,
            "roofline": {"kernel": "fa_bwd_main", "bound": "tensor", "achieved": bwd_tf,
                         "peak": peak_t, "unit": "TFLOP/s", "frac": bwd_tf / peak_t,
                         "traffic": trafficb, "peak_source": f"bf16_tflops ({peak_src}, burst)",
                         "algorithmic": f"{f_bwd:.4g} FLOP per launch (2.5 x causal fwd)"},
            "roofline_fwd": {"kernel": "fa_fwd_kernel", "bound": "tensor", "achieved": fwd_tf,
                             "peak": peak_t, "unit": "TFLOP/s", "frac": fwd_tf / peak_t,
                             "traffic": trafficf,
                             "algorithmic": f"{f_fwd:.4g} FLOP per launch"},
            "decode": dec,
            "next_rows": nxt,
            "clocks": clocks.summary(),
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "overlap": "step i+1's inputs copied in and step i-1's results copied out "
                               "on two more streams while step i computes (double-buffered "
                               "device tensors)",
                    "serial": {"value": job_tflops(f_fwd + f_bwd, e2e_serial_ms, ws),
                               "ms_per_step": e2e_serial_ms}},
            "gpu_launches": launches_per_step * args.steps,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def next_rows_bench(fa, dev, peaks, w, q, k, v, do, kst, ken, o, lse, dq, dk, dv, wsb):
    """The widened rows measured on the same shapes: a per-key boolean mask
    (10% of keys hidden, seeded), dropout p = 0.1, a packed varlen batch
    (16 causal sequences, lengths uniform in [1024, 8192], seeded) and the
    FP8 forward (per-tensor e4m3 quantisation of the same Q, K, V).  TFLOP/s
    use the metric's formula on each problem's own sizes (masked keys and
    dropped weights are not discounted)."""
    peak_t = peaks["bf16_tflops"]

    def timed(fn, reps=5):
        for _ in range(2):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        b.synchronize()
        return a.elapsed_time(b) / reps

    out = {}
    g = torch.Generator().manual_seed(1)
    km = (torch.rand(w.B, w.Sk, generator=g) >= 0.1).to(dev)
    bits = fa.fa_pack_key_mask(km)
    f_f, f_b = w.flops_fwd(), w.flops_bwd()
    ms_f = timed(lambda: fa.fa_fwd(q, k, v, True, w.scale, k_start=kst, k_end=ken, o=o, lse=lse,
                                   key_mask=bits))
    ms_b = timed(lambda: fa.fa_bwd(q, k, v, o, do, lse, True, w.scale, k_start=kst, k_end=ken,
                                   dq=dq, dk=dk, dv=dv, workspace=wsb, key_mask=bits))
    out["key_mask"] = {"workload": f"{WORKLOAD} + 10% of keys hidden by a boolean mask",
                       "fwd_tflops": f_f / ms_f / 1e9, "fwd_frac": f_f / ms_f / 1e9 / peak_t,
                       "bwd_tflops": f_b / ms_b / 1e9, "bwd_frac": f_b / ms_b / 1e9 / peak_t}
    ms_f = timed(lambda: fa.fa_fwd(q, k, v, True, w.scale, k_start=kst, k_end=ken, o=o, lse=lse,
                                   dropout_p=0.1, seed=1, offset=0))
    ms_b = timed(lambda: fa.fa_bwd(q, k, v, o, do, lse, True, w.scale, k_start=kst, k_end=ken,
                                   dq=dq, dk=dk, dv=dv, workspace=wsb, dropout_p=0.1, seed=1,
                                   offset=0))
    out["dropout"] = {"workload": f"{WORKLOAD} + dropout p = 0.1",
                      "fwd_tflops": f_f / ms_f / 1e9, "fwd_frac": f_f / ms_f / 1e9 / peak_t,
                      "bwd_tflops": f_b / ms_b / 1e9, "bwd_frac": f_b / ms_b / 1e9 / peak_t}
    lens = torch.randint(1024, 8193, (16,), generator=g)
    cu = torch.zeros(17, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    total, H, d = int(cu[-1]), w.Hq, w.d
    gd = torch.Generator(device=dev).manual_seed(2)
    vq, vk, vv, vdo = (torch.randn(H, total, d, generator=gd, device=dev).bfloat16()
                       for _ in range(4))
    cud = cu.to(dev)
    L = int(lens.max())
    vo, vl = fa.fa_fwd_varlen(vq, vk, vv, cud, cud, L, L, True, w.scale)
    ws_v = torch.empty(fa.fa_bwd_workspace_size(1, H, total, d), dtype=torch.uint8, device=dev)
    vgq, vgk, vgv = torch.empty_like(vq), torch.empty_like(vk), torch.empty_like(vv)
    f_vf = sum(4.0 * H * int(n) * int(n) * d / 2 for n in lens)
    ms_f = timed(lambda: fa.fa_fwd_varlen(vq, vk, vv, cud, cud, L, L, True, w.scale, o=vo, lse=vl))
    ms_b = timed(lambda: fa.fa_bwd_varlen(vq, vk, vv, vo, vdo, vl, cud, cud, L, L, True, w.scale,
                                          dq=vgq, dk=vgk, dv=vgv, workspace=ws_v))
    out["varlen"] = {"workload": f"16 packed causal sequences, {total} tokens, H={H} d={d}",
                     "fwd_tflops": f_vf / ms_f / 1e9, "fwd_frac": f_vf / ms_f / 1e9 / peak_t,
                     "bwd_tflops": 2.5 * f_vf / ms_b / 1e9,
                     "bwd_frac": 2.5 * f_vf / ms_b / 1e9 / peak_t}
    # FP8 (e4m3) forward on the same shapes; per-tensor descale = max|x| / 448
    if getattr(torch, "float8_e4m3fn", None) is not None:
        q8, qd, k8, kd, vt8, vd = _fp8_inputs(q, k, v)
        peak8 = 2.0 * peak_t  # the nominal FP8 : BF16 dense ratio (4.5 : 2.25 PFLOP/s)
        ms_f = timed(lambda: fa.fa_fwd_fp8(q8, k8, vt8, True, w.scale, qd, kd, vd, k_start=kst,
                                           k_end=ken, o=o, lse=lse))
        out["fp8_fwd"] = {"workload": f"{WORKLOAD}, Q/K/V in e4m3 (V transposed)",
                          "fwd_tflops": f_f / ms_f / 1e9, "fwd_frac": f_f / ms_f / 1e9 / peak8,
                          "peak": peak8, "peak_source": "2 x measured bf16 (nominal FP8:BF16)"}
    st, word = fa.fa_device_status()
    if st != 0:
        raise RuntimeError(f"device status after the widened rows: {word:#x}")
    return out


def _fp8_inputs(q, k, v):
    """e4m3 Q, K and V^T ([B, Hkv, d, Sk]) with per-tensor descales max|x| / 448."""
    f8 = torch.float8_e4m3fn

    def quant(x):
        ds = float(x.float().abs().max()) / 448.0
        return (x.float() / ds).to(f8), ds
    q8, qd = quant(q)
    k8, kd = quant(k)
    v8, vd = quant(v)
    return q8, qd, k8, kd, v8.transpose(-1, -2).contiguous(), vd


def decode_bench(fa, dev, peaks, args, ws):
    w = workloads.make(DECODE)
    t = w.tensors
    q = t["q"].to(dev)
    kc = t["k"].to(dev)
    vc = t["v"].to(dev)
    sl = t["seqlens_k"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device=dev)
    wsd = torch.empty(fa.fa_decode_workspace_size(w.B, w.Hq, w.Sk, w.d), dtype=torch.uint8,
                      device=dev)
    n_keys = int(t["seqlens_k"].sum())
    algo_bytes = n_keys * w.Hkv * w.d * 2 * 2 + q.numel() * 2 * 2 + lse.numel() * 4
    for _ in range(max(3, args.warmup)):
        fa.fa_decode(q, kc, vc, sl, w.scale, o=o, lse=lse, workspace=wsd)
    reps = max(10, args.steps)
    evs = []
    for _ in range(reps):
        e4 = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in e4:
            e.record()
        evs.append(e4)
    _barrier(ws)
    for e4 in evs:
        e4[0].record()
        fa.fa_profile_next_launch(e4[2], e4[3])
        fa.fa_decode(q, kc, vc, sl, w.scale, o=o, lse=lse, workspace=wsd)
        e4[1].record()
    _barrier(ws)
    call_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    part_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    peak = peaks["hbm_gbs"]
    gbs = algo_bytes / (call_ms * 1e-3) / 1e9
    part_gbs = (n_keys * w.Hkv * w.d * 2 * 2 + q.numel() * 2) / (part_ms * 1e-3) / 1e9
    st, word = fa.fa_device_status()
    if st != 0:
        raise RuntimeError(f"device status after decode: {word:#x}")
    return {"workload": f"{DECODE}: {workloads.DESCRIPTIONS[DECODE]}",
            "value": gbs, "unit": "GB/s", "us_per_call": call_ms * 1e3,
            "algorithmic_bytes": algo_bytes, "frac_of_hbm": gbs / peak,
            "l2": "KV bytes read per call 1.76e9+ > L2",
            "roofline": {"kernel": "fa_decode_partial", "bound": "hbm", "achieved": part_gbs,
                         "peak": peak, "unit": "GB/s", "frac": part_gbs / peak,
                         "traffic": _traffic("fa_decode_partial", "fa_decode.cu")},
            "gpu_launches_per_call": 2}


def run_only(args):
    """Profiling aid: run just one call kind (fwd, bwd, decode, the FP8
    forward or the dropout forward at p = 0.1 on the step's workload)
    `--warmup` + `--steps` times, no timing JSON.  Used as the command an ncu
    capture of a single kernel runs."""
    import io_aware_exact_tcgen05_gb300 as fa
    fa.load_library()
    dev = torch.device("cuda", 0)
    n = args.warmup + args.steps
    if args.only == "decode":
        w = workloads.make(DECODE, **({"B": args.decode_batch} if args.decode_batch else {}))
        t = w.tensors
        q, kc, vc, sl = (t[x].to(dev) for x in ("q", "k", "v", "seqlens_k"))
        for _ in range(n):
            fa.fa_decode(q, kc, vc, sl, w.scale)
    elif args.only == "fp8":
        w = workloads.make(WORKLOAD)
        t = w.tensors
        q, k, v = (t[x].to(dev) for x in ("q", "k", "v"))
        kst, ken = t["k_start"].to(dev), t["k_end"].to(dev)
        q8, qd, k8, kd, vt8, vd = _fp8_inputs(q, k, v)
        for _ in range(n):
            fa.fa_fwd_fp8(q8, k8, vt8, True, w.scale, qd, kd, vd, k_start=kst, k_end=ken)
    else:
        w = workloads.make(WORKLOAD)
        t = w.tensors
        q, k, v, do = (t[x].to(dev) for x in ("q", "k", "v", "dout"))
        kst, ken = t["k_start"].to(dev), t["k_end"].to(dev)
        o, lse = fa.fa_fwd(q, k, v, True, w.scale, k_start=kst, k_end=ken)
        for _ in range(n):
            if args.only == "fwd":
                fa.fa_fwd(q, k, v, True, w.scale, k_start=kst, k_end=ken, o=o, lse=lse)
            elif args.only == "fwd_dropout":
                fa.fa_fwd(q, k, v, True, w.scale, k_start=kst, k_end=ken, o=o, lse=lse,
                          dropout_p=0.1, seed=1, offset=0)
            else:
                fa.fa_bwd(q, k, v, o, do, lse, True, w.scale, k_start=kst, k_end=ken)
    st, word = fa.fa_device_status()
    print(json.dumps({"only": args.only, "calls": n, "status": st, "word": word}))
    return 0 if st == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-next", action="store_true",
                    help="skip the key-mask / dropout / varlen measurements")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--only", choices=["fwd", "bwd", "decode", "fp8", "fwd_dropout"], default=None)
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="with --only decode: fewer sequences (a smaller profiling case)")
    args = ap.parse_args()
    if args.only:
        return run_only(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
