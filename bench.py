"""Throughput of the Ulysses low-precision quantize -> pack -> unpack path.

A step is one pass of the whole path (boundary min/max, derive, then pack
with the amax fused in and the exchange folded into its stores, then unpack;
launch-bound workloads fold the derive into pack too) over every rank of an emulated Ulysses group held on one
GPU, on seeded synthetic inputs shaped like the long non-aligned workload
(B=1, H=40, D=128, P=8, L=9360, bf16, used 74800).  Prints one JSON line.

Workloads whose inputs fit in a few times the L2 (``--workload`` tiny or
padding) are launch-bound: their line also times the step four ways (eager
launches or one CUDA-graph replay, L2 flushed before each step or not), and
``value`` is the eager step with the L2 flushed before it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun, one process per GPU) every GPU runs its own replica of
the emulated group (no collective on the data path), so per-GPU work is fixed
(weak scaling); value = bytes of all ranks / the slowest rank's time.
``--impl reference`` times the CPU oracle instead, on rank 0 only.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s (amax+pack+unpack) & % of GB300 HBM peak; tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="workload name (default: the headline one)")
    ap.add_argument("--mode", choices=["fused", "unfused"], default="fused")
    ap.add_argument("--q-group", type=int, choices=[64, 128], default=128,
                    help="Q group rows (64: Q groups are the K groups)")
    ap.add_argument("--derive", choices=["auto", "folded", "separate"], default="auto",
                    help="boundary derive inside pack (three launches) or its own launch (four); "
                         "auto: inside pack for launch-bound workloads")
    ap.add_argument("--launch", choices=["single", "multi"], default="multi",
                    help="the step as three or four launches (multi, the default) or as one "
                         "cooperative launch (single)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum CPU time spent on the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense fp16 tensor TFLOP/s: the measured bf16 burst figure (fp16 runs at
    the bf16 rate), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16 burst (cuBLAS); fp16 rate = bf16 rate"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback bf16 burst; fp16 rate = bf16 rate"


# ------------------------------------------------------- recorded traffic

PACK_SOURCES = ["quantize_pack_gb300/csrc/ulp_pack.cu", "quantize_pack_gb300/csrc/ulp_pack.cuh",
                "quantize_pack_gb300/csrc/ulp_internal.cuh"]
# the DRAM bytes of one pack launch, from one ncu capture (written by hand from
# its output, with the digest of the pack sources it was taken on)
TRAFFIC_RECORD = "profiles/pack_traffic.json"


def pack_source_digest():
    import hashlib
    h = hashlib.sha256()
    for rel in PACK_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload_name):
    """DRAM bytes (read + write) per pack launch from the committed ncu
    record, or None when it was taken on other kernel sources or another
    workload."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_RECORD)) as f:
            rec = json.load(f)
        if rec.get("source_sha256") != pack_source_digest() or rec.get("workload") != workload_name:
            return None
        return int(rec["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) with host
    timestamps; only samples inside [t0, t1] of the timed region are kept."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str | None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if gpu_index is not None:
            cmd += ["-i", gpu_index]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def wait_first(self, timeout=5.0):
        t = time.monotonic()
        while self.proc and not self.samples and time.monotonic() - t < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            if t0 - 0.06 <= ts <= t1 + 0.06:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == 8:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in timed region"],
                    "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((float(r[2]) for r in rows
                                    if r[2].replace(".", "").isdigit()), default=None)}


# ------------------------------------------------------------- CPU oracle

def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo), or on Arm its implementer
    and part numbers, or the machine type."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    for key in ("model name", "cpu model", "hardware"):
        if key in fields:
            return fields[key]
    if "cpu part" in fields:
        return (f"{platform.machine()} implementer {fields.get('cpu implementer', '?')} "
                f"part {fields['cpu part']}")
    return platform.machine()


def oracle_sample(wl):
    """A bounded sample of one step for the CPU oracle: rank 0's sender work
    (k_grouped_amax, boundary min/max of every rank, derive, pack) and
    destination 0's receiver work (unpack_for_sage), on the workload with one
    head per destination (H = P; L, P, D, dtype and padding unchanged).  The
    receiver is fed rank 0's chunk in every source slot (the oracle's loops do
    the same work whatever the bytes).  Returns (callable, algorithmic bytes)."""
    import numpy as np

    from oracle import oracle as O
    from quantize_pack_gb300 import metrics, synth

    swl = wl.replace(H=wl.P, name=wl.name + "_h1")
    inp = synth.make_inputs(swl)
    q, k, v = inp.shards("q"), inp.shards("k"), inp.shards("v")
    P, L = swl.P, swl.L

    def run():
        a = O.k_grouped_amax(k[0], inp.k_mean, swl.dtype, rank=0, world_size=P,
                             used_sequence=swl.used_sequence)
        mm, qb = zip(*[O.boundary_minmax(k[r], q[r], swl.dtype, rank=r, world_size=P,
                                         used_sequence=swl.used_sequence, q_group=swl.q_group)
                       for r in range(P)])
        g = np.ascontiguousarray(np.stack(mm))
        gq = np.ascontiguousarray(np.stack(qb))
        O.derive_k_boundary_amax(a, g, inp.k_mean, swl.dtype, rank=0, local_sequence=L,
                                 world_size=P)
        send = O.pack(q[0], k[0], v[0], inp.k_mean, swl.dtype, a, gq, inp.v_scale, rank=0,
                      world_size=P, q_group=swl.q_group)
        recv0 = np.ascontiguousarray(np.broadcast_to(send[0], send.shape))
        O.unpack_for_sage(recv0, batch_size=swl.B, local_sequence=L, local_heads=1,
                          head_dim=swl.D, world_size=P, scale_sequence=swl.scale_sequence,
                          q_group=swl.q_group)

    return run, metrics.step_bytes(swl) / P, swl


def run_reference(args, wl, rank):
    if rank != 0:
        return
    run, nbytes, swl = oracle_sample(wl)
    for _ in range(args.warmup):
        run()
    t = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t) / args.steps
    value = nbytes / dt / 1e9
    sample = (f"per step: rank 0 sender + destination 0 receiver of {swl.name} "
              f"(H={swl.H}, one head per destination), {nbytes / 1e6:.1f} MB algorithmic")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, **{k: v for k, v in wl.describe().items() if k != "workload"}},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "nproc": os.cpu_count(), "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ multi-rank

def max_over_ranks(dist, values, device=None):
    """Element-wise max of a list of floats over every rank (identity when
    dist is None).  The bench's timings are the slowest rank's."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_value(step_bytes, world, ms):
    """Whole-job effective bandwidth in GB/s: every rank's bytes over the
    slowest rank's time per step."""
    return step_bytes * world / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ GPU arm

def step_modes(torch, path, inputs, stream, dev, steps, l2_bytes):
    """The step of a launch-bound workload timed four ways: eager launches or
    the replay of one captured CUDA graph; with the L2 flushed before each
    step (a write of twice the L2 size, outside the timed events; median of
    per-step events) or hot (back-to-back steps in one event pair; mean).
    Returns {mode: {"ms": ...}}."""
    flush = torch.empty(max(2 * l2_bytes, 1 << 20), dtype=torch.uint8, device=dev)
    graph = path.capture(*inputs)

    def eager():
        path.run(*inputs)

    def replay():
        graph.replay()

    out = {}
    for name, run in (("eager", eager), ("graph", replay)):
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        out[f"{name}_hot"] = {"ms": e0.elapsed_time(e1) / steps}
        evs = []
        for i in range(steps):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        out[f"{name}_cold"] = {"ms": statistics.median(a.elapsed_time(b) for a, b in evs)}
    for v in out.values():
        v["launches"] = path.launches_per_step
    del flush
    return out


def run_ours(args, wl, rank, world, dist):
    import numpy as np
    import torch

    from quantize_pack_gb300 import metrics, synth, ulp
    from quantize_pack_gb300.path import UlyssesLowpPath

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ulp.lib()                                               # fail loudly if not built
    dt = torch.bfloat16 if wl.dtype == 0 else torch.float16

    inp = synth.make_inputs(wl)
    host = {n: torch.from_numpy(np.ascontiguousarray(inp.shards(n)).view(np.int16)).view(dt)
            for n in "qkv"}
    km_h = torch.from_numpy(inp.k_mean.view(np.int16)).view(dt)
    vs_h = torch.from_numpy(inp.v_scale)
    q, k, v = (host[n].to(dev) for n in "qkv")
    km, vs = km_h.to(dev), vs_h.to(dev)
    path = UlyssesLowpPath(B=wl.B, L=wl.L, H=wl.H, D=wl.D, world_size=wl.P, dtype=dt,
                           used_sequence=wl.used_sequence, scale_sequence=wl.scale_sequence,
                           aligned=wl.aligned, q_group=wl.q_group, fused=(args.mode == "fused"),
                           fold_exchange=True, fold_derive={"auto": None, "folded": True, "separate": False}[args.derive],
                           single_launch=args.launch == "single" and args.derive != "separate",
                           device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        path.run(q, k, v, km, vs)
    torch.cuda.synchronize()

    gpu_id = None
    try:
        props = torch.cuda.get_device_properties(dev)
        u = str(getattr(props, "uuid", ""))
        if u:
            gpu_id = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    sampler.wait_first()

    K = args.steps
    ev_pack = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    ev_end = [torch.cuda.Event(enable_timing=True) for _ in range(K)]    # after unpack
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    start.record(stream)
    for i in range(K):
        e0, e1 = ev_pack[i]
        path.run(q, k, v, km, vs, on_pack=(lambda e=e0: e.record(stream), lambda e=e1: e.record(stream)))
        ev_end[i].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    barrier()
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    ms = start.elapsed_time(end) / K
    pack_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev_pack)
    unpack_ms = statistics.mean(e1.elapsed_time(e2) for (_, e1), e2 in zip(ev_pack, ev_end))
    ms, pack_ms, unpack_ms = max_over_ranks(dist, [ms, pack_ms, unpack_ms], dev)

    # ---- launch-bound workloads: eager vs graph replay, cold vs hot L2
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 0)
    small = 6 * wl.N <= 4 * max(l2_bytes, 1)
    modes = None
    if small:
        modes = step_modes(torch, path, (q, k, v, km, vs), stream, dev, max(K, 50), l2_bytes)
        (cold_ms,) = max_over_ranks(dist, [modes["eager_cold"]["ms"]], dev)

    # ---- the emulated all-to-all on its own (the step folds it into pack's
    # stores): the permutation copy recv[p][s] = send[s][p] of every chunk
    a2a_src, a2a_dst = torch.empty_like(path.recv), torch.empty_like(path.recv)
    for _ in range(3):
        ulp.alltoall_emulate(a2a_src, a2a_dst)
    ta0, ta1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    KX = max(10, K // 10)
    ta0.record(stream)
    for _ in range(KX):
        ulp.alltoall_emulate(a2a_src, a2a_dst)
    ta1.record(stream)
    torch.cuda.synchronize()
    a2a_ms = ta0.elapsed_time(ta1) / KX
    a2a_bytes = 2 * a2a_src.numel()
    del a2a_src, a2a_dst

    # ---- the step before the path: k_mean_global production (not in the step)
    kmean_out = torch.empty_like(km)
    kmean_ws = torch.empty(ulp.k_mean_workspace_bytes(wl.B, wl.L, wl.H, wl.D, wl.P),
                           dtype=torch.uint8, device=dev)
    for _ in range(3):
        ulp.k_mean_global(k, used_sequence=wl.used_sequence, workspace=kmean_ws, out=kmean_out)
    ks0, ks1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    KM = max(10, K // 10)
    ks0.record(stream)
    for _ in range(KM):
        ulp.k_mean_global(k, used_sequence=wl.used_sequence, workspace=kmean_ws, out=kmean_out)
    ks1.record(stream)
    torch.cuda.synchronize()
    kmean_ms = ks0.elapsed_time(ks1) / KM

    # ---- the standalone k_grouped_amax of every rank (the public call and
    # the unfused mode; the fused step computes it inside pack): reads K once
    amax_out = torch.empty((wl.P, wl.B, wl.H, ulp.slots(wl.L, 64)), dtype=torch.float32, device=dev)
    for _ in range(3):
        ulp.k_grouped_amax(k, km, rank=None, world_size=wl.P, used_sequence=wl.used_sequence, out=amax_out)
    kg0, kg1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kg0.record(stream)
    for _ in range(KM):
        ulp.k_grouped_amax(k, km, rank=None, world_size=wl.P, used_sequence=wl.used_sequence, out=amax_out)
    kg1.record(stream)
    torch.cuda.synchronize()
    kgamax_ms = kg0.elapsed_time(kg1) / KM

    # ---- the step after the path: attention over destination 0's outputs
    n_att = wl.used_sequence or wl.S
    q8, k8, v8, qsc, ksc = (o[0] for o in path.out)
    vs0 = vs[:, :wl.h].contiguous()
    att_ws = torch.empty(ulp.sage_attention_workspace_bytes(wl.B, wl.S, wl.h, wl.D, n_att),
                         dtype=torch.uint8, device=dev)
    att_out = torch.empty((wl.B, n_att, wl.h, wl.D), dtype=dt, device=dev)
    att_status = torch.zeros(1, dtype=torch.int32, device=dev)

    def attend():
        ulp.sage_attention(q8, k8, v8, qsc, ksc, vs0, n=n_att, q_group=wl.q_group,
                           out=att_out, workspace=att_ws, status=att_status)

    def attend8():
        ulp.sage_attention(q8, k8, v8, qsc, ksc, vs0, n=n_att, q_group=wl.q_group,
                           out=att_out, workspace=att_ws, status=att_status, pv_fp8=True)

    def time_calls(fn, calls):
        for _ in range(2):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(calls):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / calls

    KA = 5
    att_ms = time_calls(attend, KA)
    att8_ms = time_calls(attend8, KA)
    att_flops = 4.0 * wl.B * wl.h * n_att * n_att * wl.D

    # ---- end to end through the public API with host buffers: E steps from
    # pinned host inputs to pinned host outputs (UlyssesLowpPath.run_host:
    # step i + 1's upload overlaps step i's kernels and download)
    E = max(2, args.e2e_steps)
    pin = {n: host[n].pin_memory() for n in "qkv"}
    km_p, vs_p = km_h.pin_memory(), vs_h.pin_memory()
    hin = [(pin["q"], pin["k"], pin["v"], km_p, vs_p)] * E
    outs_h = [tuple(torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in path.out)
              for _ in range(2)]
    hout = [outs_h[i % 2] for i in range(E)]
    pipe = path.host_pipe()
    path.run_host(hin[:2], hout[:2], pipe)               # warm the pipeline's buffers
    torch.cuda.synchronize()
    barrier()
    # the host link and host memory are shared with other jobs on the
    # machine: five timed runs of E steps each, the median reported
    e2e_runs = []
    for _ in range(5):
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es.record(stream)
        pipe["up"].wait_stream(stream)                    # the first upload starts after es
        path.run_host(hin, hout, pipe)
        ee.record(stream)                                 # run_host ends waiting for the downloads
        torch.cuda.synchronize()
        e2e_runs.append(es.elapsed_time(ee) / E)
    e2e_ms = statistics.median(e2e_runs)
    (e2e_ms,) = max_over_ranks(dist, [e2e_ms], dev)
    h2d = sum(t.numel() * t.element_size() for t in hin[0])
    d2h = sum(t.numel() * t.element_size() for t in hout[0])

    if rank != 0:
        return
    step_bytes = metrics.step_bytes(wl)
    vms = cold_ms if small else ms          # the step time that value reports
    value = whole_job_value(step_bytes, world, vms)
    peak, peak_kind = peaks()
    mhz = clocks.get("sm_mhz") or None

    def cycles(t_ms):
        """The kernel time in SM clock cycles at the median clock of the
        timed region (for comparing runs whose clocks differ)."""
        return None if mhz is None else t_ms * 1e-3 * mhz * 1e6
    pack_gbs = metrics.pack_bytes(wl) / (pack_ms * 1e-3) / 1e9
    if path.single_launch:
        # one launch a step: the events around it time the whole step, whose
        # algorithmic bytes are the step's
        step_gbs = step_bytes / (pack_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": "group_step_kernel", "achieved": step_gbs, "peak": peak,
                    "peak_kind": f"{peak_kind} (STREAM copy)", "unit": "GB/s", "frac": step_gbs / peak,
                    "traffic": None, "algorithmic_bytes_per_launch": step_bytes, "launch_ms": pack_ms}
        kernels = {"group_step": {"ms": pack_ms, "gbs": step_gbs, "frac": step_gbs / peak,
                                  "algorithmic_bytes": step_bytes, "sm_cycles": cycles(pack_ms)}}
        path_desc = (f"{args.mode} amax+pack (exchange folded into the stores) + unpack, one cooperative "
                     "launch/step (boundary min/max, pack with the derive folded in, unpack; grid barriers)")
    else:
        roofline = {"bound": "hbm", "kernel": "pack_kernel", "achieved": pack_gbs, "peak": peak,
                    "peak_kind": f"{peak_kind} (STREAM copy)", "unit": "GB/s",
                    "frac": pack_gbs / peak, "traffic": recorded_traffic(wl.name),
                    "algorithmic_bytes_per_launch": metrics.pack_bytes(wl),
                    "launch_ms": pack_ms}
        kernels = {
            "pack": {"ms": pack_ms, "gbs": pack_gbs, "frac": pack_gbs / peak,
                     "algorithmic_bytes": metrics.pack_bytes(wl), "sm_cycles": cycles(pack_ms)},
            "unpack": {"ms": unpack_ms,
                       "gbs": metrics.unpack_bytes(wl) / (unpack_ms * 1e-3) / 1e9,
                       "frac": metrics.unpack_bytes(wl) / (unpack_ms * 1e-3) / 1e9 / peak,
                       "algorithmic_bytes": metrics.unpack_bytes(wl), "sm_cycles": cycles(unpack_ms)},
            "boundary_minmax" + ("" if path.fold_derive else "+derive"): {
                "ms": max(0.0, ms - pack_ms - unpack_ms), "sm_cycles": cycles(max(0.0, ms - pack_ms - unpack_ms))},
        }
        path_desc = (f"{args.mode} amax+pack (exchange folded into the stores) + unpack, "
                     f"{path.launches_per_step} launches/step")
    kernels["note"] = ("CUDA events around each launch inside the timed steps (means); sm_cycles = "
                       "ms x the median SM clock sampled in the timed region")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": vms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": wl.name, **{k_: v_ for k_, v_ in wl.describe().items() if k_ != "workload"},
            "path": path_desc,
            "l2": (f"value: L2 ({l2_bytes / 1e6:.0f} MB) flushed before each timed step (a {2 * l2_bytes / 1e6:.0f} MB "
                   f"write, not timed)" if small else f"inputs {6 * wl.N / 1e9:.2f} GB > 129 MB L2; no flush"),
            "parallelism": f"{world} independent replica(s) of a P={wl.P} emulated Ulysses group",
        },
        "tokens_per_s": wl.tokens * world / (vms * 1e-3),
        "hbm_frac": value / world / peak,
        "step_bytes": step_bytes,
        "roofline": roofline,
        "e2e": {"value": whole_job_value(step_bytes, world, e2e_ms), "unit": "GB/s",
                "ms_per_step": e2e_ms, "steps": E, "runs_ms_per_step": e2e_runs,
                "timing": "median of 5 timed runs of E pipelined steps (UlyssesLowpPath.run_host)",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "kernels": kernels,
        "alltoall_emulate": {"ms": a2a_ms, "calls": KX, "bytes": a2a_bytes,
                             "gbs": a2a_bytes / (a2a_ms * 1e-3) / 1e9,
                             "frac": a2a_bytes / (a2a_ms * 1e-3) / 1e9 / peak, "sm_cycles": cycles(a2a_ms),
                             "note": "the emulated all-to-all as its own device copy (read + write of "
                                     "every chunk, 6N bytes); the step folds it into pack's stores; "
                                     "not in value"},
        "gpu_launches": K * path.launches_per_step,
        "k_mean_global": {"ms": kmean_ms, "steps": KM, "sm_cycles": cycles(kmean_ms),
                          "achieved_gbs": 2 * wl.N / (kmean_ms * 1e-3) / 1e9,
                          "frac": 2 * wl.N / (kmean_ms * 1e-3) / 1e9 / peak,
                          "note": "the step before the path (reads K once); not in value"},
        "k_grouped_amax": {"ms": kgamax_ms, "calls": KM, "sm_cycles": cycles(kgamax_ms),
                           "achieved_gbs": 2 * wl.N / (kgamax_ms * 1e-3) / 1e9,
                           "frac": 2 * wl.N / (kgamax_ms * 1e-3) / 1e9 / peak,
                           "note": "the standalone call over all ranks (2N bytes: K read once); "
                                   "the fused step does this inside pack; not in value"},
        "attention": {"ms": att_ms, "calls": KA, "tflops": att_flops / (att_ms * 1e-3) / 1e12,
                      "peak": tensor_peak()[0], "peak_kind": tensor_peak()[1],
                      "frac": att_flops / (att_ms * 1e-3) / 1e12 / tensor_peak()[0],
                      "flops_per_call": att_flops, "status": int(att_status.item()),
                      "note": "the step after the path: softmax attention of destination 0 "
                              f"({wl.h} heads, {n_att} live rows, D={wl.D}) on its unpacked "
                              "INT8/E4M3 tensors, fp16 tensor cores; 4 n^2 D flops per head; "
                              "not in value"},
        "attention_e4m3_pv": {
            "ms": att8_ms, "calls": KA, "tflops": att_flops / (att8_ms * 1e-3) / 1e12,
            "peak": tensor_peak()[0] * 4 / 3,
            "peak_kind": "mixed: QK^T at the measured fp16 (= bf16) burst rate, PV at twice it "
                         "(E4M3, kind::f8f6f4): 4/3 of the fp16 peak for 4 n^2 D flops",
            "frac": att_flops / (att8_ms * 1e-3) / 1e12 / (tensor_peak()[0] * 4 / 3),
            "status": int(att_status.item()),
            "note": "the same call with the PV product in E4M3 (P rounded to E4M3, V read from "
                    "v8 itself); not in value"},
        "clocks": clocks,
    }
    if small:
        line["step_modes"] = modes
        line["hot_eager_ms_per_step"] = ms
    if not args.no_cpu_baseline:
        run, nbytes, swl = oracle_sample(wl)
        n, t = 0, time.perf_counter()
        while True:
            run()
            n += 1
            if time.perf_counter() - t >= args.cpu_seconds:
                break
        dtc = (time.perf_counter() - t) / n
        line["cpu_baseline"] = {
            "value": nbytes / dtc / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "nproc": os.cpu_count(), "cpu_model": cpu_model(),
            "sample": f"{n} x (rank 0 sender + destination 0 receiver of {swl.name}, "
                      f"{nbytes / 1e6:.1f} MB algorithmic each)"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    from quantize_pack_gb300 import configs
    wl = configs.BY_NAME[args.workload] if args.workload else configs.HEADLINE
    if args.q_group != wl.q_group:
        wl = wl.replace(q_group=args.q_group, name=f"{wl.name}_gq{args.q_group}")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, wl, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist_
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist_.init_process_group(backend)
        dist = dist_
    try:
        run_ours(args, wl, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
