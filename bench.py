"""Benchmark: attention backward TFLOP/s on GB300 through libfab's C ABI.

One step = one fab_backward call over the workload (what a user calls:
on the tensor-core path the query pass, which forms D_i and dQ, then the
key/value pass for dK and dV), inputs resident in HBM, L2 flushed before
every step (256 MiB written, then another 256 MiB read, so the written lines
are back in HBM before the timed call), CUDA events on the launching stream
around the call.  Throughput counts 10*B*H*N*M*D flops per backward, halved for a
causal mask.  A second loop, outside the timed region, calls the two passes
through their own entry points with an event between them, which gives each
kernel's launch time (stages_ms) and the dominant kernel's roofline against
the measured dense bf16 peak.  Also reported: two end-to-end numbers with
host buffers (pinned H2D copies of the inputs, fab_backward, D2H of the
packed gradients; once with the saved o and lse, once with the op's own
operands q, k, v, the mask and d, the forward then recomputed inside), the
forward kernel's TFLOP/s, fab_backward without o and lse on resident inputs,
the two-phase API's D_i kernel in GB/s (each of these three after at least
three warm-up calls, the L2 flushed before every call, median of the timed
calls), and the fp64 CPU oracle on the workload's (batch, key/value head)
units.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl fab|reference]

Under torchrun every rank runs the same workload on its own GPU (replicas; no
collective on the data path) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from attention_backward_tcgen05_gb300 import inputs  # noqa: E402

METRIC = "attn-backward TFLOP/s (dQ,dK,dV) and fraction of GB300 dense BF16 peak"
DEFAULT_WORKLOAD = "gqa_causal_d128"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM read + write bytes of one launch of each tensor-core pass from an ncu
# capture (profiles/query_pass_*.md, profiles/key_pass_*.md), keyed by
# (workload, pass); entries are removed when the kernel changes after the
# capture.
MEASURED_TRAFFIC = {
    ("gqa_causal_d128", "query"): 252111616 + 98254848,
    ("gqa_causal_d128", "key"): 305679616 + 33606912,
}


def backward_flops(w: inputs.Workload) -> float:
    f = 10.0 * w.B * w.H * w.N * w.M * w.DK
    return f / 2 if w.causal else f


def pass_flops(w: inputs.Workload, gemms: int) -> float:
    """Flops of a kernel that runs `gemms` of the backward's N x M x D
    contractions (the query pass runs 3: S, dP, dQ; the key pass 4: S, dP,
    dV, dK), halved for a causal mask."""
    f = 2.0 * gemms * w.B * w.H * w.N * w.M * w.DK
    return f / 2 if w.causal else f


def executed_tile_fraction(w: inputs.Workload, mask, gemms: int) -> float:
    """The share of its tiles a tensor-core pass runs when the mask's live
    spans let it skip the rest: per row of 128 x 128 tiles (query tiles for
    the query pass, gemms = 3; key tiles for the key pass, gemms = 4) the
    tiles from the first to the last one holding an entry other than -inf,
    within the causal bound; a query tile with none still runs one.  1.0
    without a mask."""
    if mask is None:
        return 1.0
    qt, kt = -(-w.N // 128), -(-w.M // 128)
    live = torch.zeros((qt * 128, kt * 128), dtype=torch.bool)
    live[:w.N, :w.M] = mask.float() != float("-inf")
    live = live.reshape(qt, 128, kt, 128).any(3).any(1)
    done = dense = 0
    rows = live if gemms == 3 else live.t()
    for i in range(rows.shape[0]):
        if gemms == 3:
            lo, hi = 0, (min(kt, (i * 128 + 127) // 128 + 1) if w.causal else kt)
        else:
            lo, hi = (min(qt, i) if w.causal else 0), qt
        idx = torch.nonzero(rows[i]).flatten()
        s0, s1 = (int(idx[0]), int(idx[-1]) + 1) if idx.numel() else (rows.shape[1], 0)
        a, b = max(lo, s0), min(hi, s1)
        done += (b - a) if b > a else (1 if gemms == 3 else 0)
        dense += hi - lo
    return done / dense if dense else 1.0


def preprocess_bytes(w: inputs.Workload) -> int:
    """Algorithmic DRAM bytes of the D_i kernel: dO and O read once (the input
    type), D_i written (f32), the packed result's padding zeroed."""
    elem = 4 if w.dtype == "f32" else 2
    rows = w.B * w.H * w.N
    pad16 = lambda n: (n + 3) // 4 * 4  # floats, to 16 bytes
    nq, nk, nv = rows * w.DK, w.B * w.Hkv * w.M * w.DK, w.B * w.Hkv * w.M * w.DV
    pad = (pad16(nq) - nq) + (pad16(nk) - nk) + (pad16(nv) - nv)
    return 2 * rows * w.DV * elem + rows * 4 + pad * 4


def forward_flops(w: inputs.Workload) -> float:
    f = 4.0 * w.B * w.H * w.N * w.M * w.DK
    return f / 2 if w.causal else f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return FALLBACK_PEAKS, "fallback"


# ----------------------------------------------------------------------------- distributed plumbing


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index
        self.out = os.path.join("/tmp", f"fab_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.dev)], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.out):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.out)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle sample


def oracle_sample(w: inputs.Workload, x: dict, target_s: float = 15.0):
    """Times the fp64 oracle, one (batch, kv-head) unit per host thread.

    Every unit of the workload when that is expected to take at most
    `target_s` on this host (about 4.5 counted GFLOP/s per core), else the
    first units, a whole number of rounds over the cores, sized to about
    `target_s`.  Returns (TFLOP/s, threads used, sample text, seconds)."""
    import oracle

    cores = os.cpu_count() or 1
    units_total = w.B * w.Hkv
    per_unit = backward_flops(w) / units_total
    est_s = per_unit * units_total / (4.5e9 * cores)
    if est_s <= target_s:
        n_units = units_total
    else:
        rounds = max(1, int(target_s / (per_unit / 4.5e9)))
        n_units = min(units_total, rounds * cores)
    threads = min(cores, n_units)
    units = None if n_units == units_total else list(range(n_units))
    t0 = time.perf_counter()
    oracle.backward(x["q"], x["k"], x["v"], x["d"], x["mask"], w.causal, w.scale, units=units, threads=threads)
    dt = time.perf_counter() - t0
    tflops = per_unit * n_units / dt / 1e12
    what = "all" if units is None else f"{n_units} of"
    sample = (f"{what} {units_total} (batch, kv-head) units of {w.name} in {dt:.1f} s on {threads} threads; "
              f"counted 10*B*H*N*M*D{'/2' if w.causal else ''} flops per unit")
    return tflops, threads, sample, dt


# ----------------------------------------------------------------------------- reference arm (the oracle)


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    x = inputs.make(w)
    times, vals = [], []
    sample, c = "", 1
    for i in range(args.warmup + args.steps):
        v, c, sample, dt = oracle_sample(w, x, target_s=6.0)
        if i >= args.warmup:
            times.append(dt)
            vals.append(v)
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.mean(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "N": w.N, "M": w.M, "D": w.DK,
                   "causal": w.causal, "mask": w.mask, "seed": w.seed},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": c,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- the fab arm


def run_fab(args, rank, world, local):
    from attention_backward_tcgen05_gb300 import binding

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = inputs.WORKLOADS[args.workload]
    xc = inputs.make(w)
    x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in xc.items()}
    q, k, v, d, mask = x["q"], x["k"], x["v"], x["d"], x["mask"]
    dims = binding.dims_of(q, k, v)
    dt = binding.dtype_code(q)
    stream = torch.cuda.current_stream()

    ws, packed = binding.alloc_backward(dims, dt, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(val=0.0):
        # a buffer larger than L2 written, then another one read: the written
        # lines leave L2 (written back to HBM) here, not inside the timed call
        flush.fill_(val)
        flush_rd.amax()

    def time_calls(call, n_timed):
        # the side measurements: untimed warm-up calls, then n_timed calls,
        # each after an L2 flush, timed with CUDA events on the stream
        n_warm = max(3, args.warmup)
        ms = []
        for i in range(n_warm + n_timed):
            flush_l2(float(i))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            if i >= n_warm:
                ms.append(e0.elapsed_time(e1))
        return ms

    # the forward (saved O and LSE), timed on its own
    o, lse = binding.forward(q, k, v, mask, w.causal, w.scale)
    fwd_ms = []
    if args.forward_steps:
        fwd_ms = time_calls(lambda: binding.fab_forward_lse(q, k, v, mask, w.causal, w.scale, o, lse), 10)
    tensor_core = w.dtype in ("bf16", "f16") and w.DK == w.DV and w.DK in (64, 128)

    # fab_backward without o and lse (the op's own operands only): the forward
    # is recomputed into the workspace first; timed on its own, L2 flushed
    rec_ms = []
    if args.forward_steps:
        ws_r, packed_r = binding.alloc_backward(dims, dt, dev, recompute=True)
        rec_ms = time_calls(lambda: binding.fab_backward(q, k, v, d, None, None, mask, w.causal, w.scale,
                                                         ws_r, packed_r), 5)
        del ws_r, packed_r

    # the two-phase API's D_i kernel (fab_backward computes D_i inside the
    # query pass instead): HBM-bound, timed on its own between L2 flushes
    pre_ms = []
    if args.forward_steps:
        pre_ms = time_calls(lambda: binding.fab_backward_preprocess(d, o, dims, ws, packed), 5)

    def step():
        binding.fab_backward(q, k, v, d, o, lse, mask, w.causal, w.scale, ws, packed)

    # kernels one fab_backward call launches: the mask scan (with a mask), the
    # query pass and the key/value pass; on the CUDA-core path the D_i
    # kernel, then dq_simt and dkdv_simt
    launches_per_step = (2 + (1 if mask is not None else 0)) if tensor_core else 3

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    status = binding.fab_last_device_error()
    if status != binding.FAB_OK:
        raise RuntimeError(f"device error during warm-up: {binding.status_string(status)}")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    clk = clocks.stop()
    status = binding.fab_last_device_error()
    if status != binding.FAB_OK:
        raise RuntimeError(f"device error in the timed region: {binding.status_string(status)}")
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world)
    flops = backward_flops(w)
    value = flops * world / (ms_max / 1e3) / 1e12

    # each kernel's launch time: the same work through the two entry points
    # fab_backward is made of, with an event between them (outside the timed
    # region above; with a mask each entry point also scans it)
    if tensor_core:
        stage_names = ("query_pass", "key_pass")

        def first():
            binding.fab_backward_query_pass(q, k, v, d, o, lse, mask, w.causal, w.scale, ws, packed)

        def second():
            binding.fab_backward_key_pass(q, k, v, d, lse, mask, w.causal, w.scale, ws, packed)
    else:
        stage_names = ("preprocess", "main")

        def first():
            binding.fab_backward_preprocess(d, o, dims, ws, packed)

        def second():
            binding.fab_backward_main(q, k, v, d, lse, mask, w.causal, w.scale, ws, packed)

    for _ in range(args.warmup):
        flush_l2()
        first()
        second()
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2()
        sev[i][0].record(stream)
        first()
        sev[i][1].record(stream)
        second()
        sev[i][2].record(stream)
    torch.cuda.synchronize()
    first_ms = [e[0].elapsed_time(e[1]) for e in sev]
    second_ms = [e[1].elapsed_time(e[2]) for e in sev]

    # end to end through the public call with host buffers: every step copies
    # its inputs from pinned host memory, runs fab_backward and reads the packed
    # gradients back.  Steps overlap (H2D of step i+1 and D2H of step i-1 run
    # on their own streams while step i computes, two buffer sets); "serial"
    # runs the three phases of each step back to back on one stream.  The
    # headline copies the saved forward output and LSE with the inputs;
    # "op_operands" copies only ggml_flash_attn_back's operands (q, k, v, the
    # mask, d) and lets fab_backward recompute O and LSE on the device.
    e2e = None
    if not args.no_e2e:
        host = {kk: vv.pin_memory() for kk, vv in xc.items() if isinstance(vv, torch.Tensor)}
        host["o"] = o.cpu().pin_memory()
        host["lse"] = lse.cpu().pin_memory()
        d2h = packed.numel() * 4
        s_h2d, s_cmp, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_variant(saved: bool):
            names = [n for n in ("q", "k", "v", "d", "mask") + (("o", "lse") if saved else ()) if n in host]
            h2d = sum(host[n].numel() * host[n].element_size() for n in names)
            sets = []
            for _ in range(2):
                bufs = {n: torch.empty_like(host[n], device=dev) for n in names}
                wsb, pkb = binding.alloc_backward(dims, dt, dev, recompute=not saved)
                sets.append((bufs, wsb, pkb, torch.empty(packed.numel(), dtype=torch.float32).pin_memory()))

            def call(bufs, wsb, pkb, strm):
                binding.fab_backward(bufs["q"], bufs["k"], bufs["v"], bufs["d"], bufs.get("o"), bufs.get("lse"),
                                     bufs.get("mask"), w.causal, w.scale, wsb, pkb, stream=strm)

            def run_pipelined(nsteps):
                ev_in = [torch.cuda.Event() for _ in range(2)]
                ev_cmp = [torch.cuda.Event() for _ in range(2)]
                ev_out = [torch.cuda.Event() for _ in range(2)]
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(s_h2d)
                for i in range(nsteps):
                    bufs, wsb, pkb, outh = sets[i % 2]
                    if i >= 2:
                        s_h2d.wait_event(ev_cmp[i % 2])  # inputs of step i-2 consumed
                    with torch.cuda.stream(s_h2d):
                        for n in names:
                            bufs[n].copy_(host[n], non_blocking=True)
                        ev_in[i % 2].record(s_h2d)
                    s_cmp.wait_event(ev_in[i % 2])
                    if i >= 2:
                        s_cmp.wait_event(ev_out[i % 2])  # packed of step i-2 read back
                    call(bufs, wsb, pkb, s_cmp)
                    ev_cmp[i % 2].record(s_cmp)
                    s_d2h.wait_event(ev_cmp[i % 2])
                    with torch.cuda.stream(s_d2h):
                        outh.copy_(pkb, non_blocking=True)
                        ev_out[i % 2].record(s_d2h)
                s_d2h.wait_event(ev_out[(nsteps - 1) % 2])
                t1.record(s_d2h)
                t1.synchronize()
                return t0.elapsed_time(t1) / nsteps

            def run_serial(nsteps):
                bufs, wsb, pkb, outh = sets[0]
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                for _ in range(nsteps):
                    for n in names:
                        bufs[n].copy_(host[n], non_blocking=True)
                    call(bufs, wsb, pkb, stream)
                    outh.copy_(pkb, non_blocking=True)
                t1.record(stream)
                t1.synchronize()
                return t0.elapsed_time(t1) / nsteps

            run_pipelined(max(2, args.warmup))
            run_serial(max(1, args.warmup))
            torch.cuda.synchronize()
            barrier(world)
            pipe_ms = max_over_ranks(run_pipelined(args.steps), world)
            barrier(world)
            ser_ms = max_over_ranks(run_serial(args.steps), world)
            status = binding.fab_last_device_error()
            if status != binding.FAB_OK:
                raise RuntimeError(f"device error in the e2e region: {binding.status_string(status)}")
            del sets
            return {"value": round(flops * world / (pipe_ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
                    "ms_per_step": round(pipe_ms, 3), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "serial": {"value": round(flops * world / (ser_ms / 1e3) / 1e12, 3),
                               "ms_per_step": round(ser_ms, 3)}}

        e2e = e2e_variant(True)
        e2e["mode"] = "two buffer sets, H2D / backward / D2H on three streams, steps overlapped; o and lse copied in"
        e2e["op_operands"] = e2e_variant(False)
        e2e["op_operands"]["mode"] = ("as above, copying q, k, v, the mask and d only; fab_backward with o = lse = "
                                      "NULL recomputes the forward on the device (backward flops counted)")

    peaks, peak_src = load_peaks()
    first_mean, second_mean = statistics.mean(first_ms), statistics.mean(second_ms)
    peak = float(peaks["bf16_tflops"])
    if tensor_core:
        # the dominant kernel of the two, with the contractions it runs itself
        if second_mean >= first_mean:
            kname, kms, kflops, kkey = "bwd_tc_kernel (key pass: S, dP, dV, dK)", second_mean, pass_flops(w, 4), "key"
        else:
            kname, kms, kflops, kkey = "dq_tc_kernel (query pass: S, dP, dQ, D_i)", first_mean, pass_flops(w, 3), "query"
    else:
        kname, kms, kflops, kkey = "dq_simt_kernel+dkdv_simt_kernel", second_mean, flops, None
    # with a mask, only the tiles the kernel runs (the live spans) count
    frac_run = executed_tile_fraction(w, xc["mask"], 4 if kkey == "key" else 3) if tensor_core else 1.0
    kflops *= frac_run
    achieved = kflops / (kms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "traffic": args.traffic_bytes if args.traffic_bytes is not None else MEASURED_TRAFFIC.get((w.name, kkey)),
                "kernel": kname, "kernel_ms": round(kms, 4), "kernel_flops": kflops,
                "tiles_run": round(frac_run, 4),
                "peak_source": (f"{peak_src} bf16_tflops (burst: the kernel is timed alone between L2 flushes)"
                                + ("; f16 has the same nominal dense rate as bf16 (ratio 1)" if w.dtype == "f16" else ""))}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample, _ = oracle_sample(w, xc)
        cpu = {"value": round(v_cpu, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
            "ms_step_median": round(statistics.median(step_ms), 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "N": w.N, "M": w.M, "D": w.DK,
                       "causal": w.causal, "mask": w.mask, "seed": w.seed, "parallelism": f"replicas x{world}",
                       "l2": "flushed before every step (256 MiB written, then another 256 MiB read so the written lines leave L2 before the timed call)",
                       "timed": "one fab_backward call per step (CUDA events on its stream)"},
            "frac_of_peak": round(value / world / peak, 4),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "stages_ms": {stage_names[0]: round(first_mean, 4), stage_names[1]: round(second_mean, 4),
                          "note": "each entry point timed on its own, outside the timed region"},
            "wall_s": round(wall, 4),
            "forward": ({"tflops": round(forward_flops(w) / (statistics.median(fwd_ms) / 1e3) / 1e12, 2),
                         "ms": round(statistics.median(fwd_ms), 4), "timed_calls": len(fwd_ms),
                         "kernel": "fwd_tc_kernel" if tensor_core else "fwd_simt_kernel"}
                        if fwd_ms else None),
            "preprocess": ({"gbps": round(preprocess_bytes(w) / (statistics.median(pre_ms) / 1e3) / 1e9, 1),
                            "ms": round(statistics.median(pre_ms), 4), "bytes": preprocess_bytes(w),
                            "peak_gbps": float(peaks["hbm_gbs"]),
                            "frac": round(preprocess_bytes(w) / (statistics.median(pre_ms) / 1e3) / 1e9
                                          / float(peaks["hbm_gbs"]), 4),
                            "kernel": "preprocess_kernel (fab_backward_preprocess: D_i and the packed padding)",
                            "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
                           if pre_ms else None),
            "recompute": ({"ms": round(statistics.median(rec_ms), 3),
                           "tflops_fwd_plus_bwd": round((forward_flops(w) + flops) / (statistics.median(rec_ms) / 1e3)
                                                        / 1e12, 2),
                           "note": "fab_backward with o and lse NULL: forward recomputed, then the backward"}
                          if rec_ms else None),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["fab", "reference"], default="fab")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(inputs.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--forward-steps", type=int, default=1)
    ap.add_argument("--traffic-bytes", type=float, default=None,
                    help="dram read+write bytes per main-kernel launch from an ncu capture")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_fab(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
