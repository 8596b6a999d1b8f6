"""Benchmark: the im2col convolution pipeline (page "DirectCompute Neural Network
Engine", section "Convolution: The im2col Approach"), forward + backward, on the
AlexNet-shaped conv1-5 layers at batch 128, one GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
for every layer conv_fwd, (max-pool forward + backward after conv1 and conv2),
conv_bwd_data, conv_bwd_filter, conv_bwd_bias and an SGD step on the filters
and bias.  The metric is algorithmic TFLOP/s of the three convolution GEMMs
(2 * outC * inC*k*k * batch*outH*outW each) over the whole step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload alexnet|lenet]

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead (host cores only).
`--workload lenet` times the LeNet-5 training step (batch 64) instead: the
whole step captured as one CUDA graph, in training images/s.  `--math tf32`
runs the contractions as one TF32 product (the fast mode) and reports them
against the TF32 roofline.  `--workload direct` times the direct (CUDA-core)
convolution kernels against the implicit-GEMM path (an ablation);
`--workload matmul` times the flagged matmul on shapes of its sweep.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "conv fwd+bwd TFLOP/s per layer at batch 128 and % of tensor roofline"
UNIT = "TFLOP/s"
WORKLOAD = "AlexNet conv1-5 fwd+bwd (fwd, input grad, filter grad, bias grad, pools, SGD), batch 128, fp32 NCHW"
LAYERS = synthetic.ALEXNET
L2_BYTES = 126 * 1024 * 1024
TF32_OVER_BF16 = 1.1 / 2.25      # nominal dense TF32 : BF16 tensor rate on GB300
SPLIT_PRODUCTS = 3               # 3xTF32: three tensor-core products per fp32 product


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return float(m["bf16_tflops"]), float(m["hbm_gbs"]), "measured"
    return 1900.0, 6800.0, "fallback"


def max_over_ranks(x, dist=None) -> float:
    """The largest value of x over all ranks (x itself on one process): every
    rank's timed region must be done before the job's is."""
    if dist is None:
        return float(x)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, ms_max, world) -> float:
    """Whole-job throughput of independent replicas (weak scaling): every rank
    processes units_per_rank per step, the job's step takes the slowest rank's
    time.  Units per second."""
    return world * units_per_rank / (ms_max * 1e-3)


STEP_TRAFFIC = os.path.join(ROOT, "profiles", "step_traffic_alexnet_b128.json")


def gemm_sources_digest(names) -> str:
    """sha256 over the named GEMM kernel sources (name, then bytes, in order)."""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        h.update(n.encode())
        with open(os.path.join(ROOT, "im2col_convolution_tiled_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def gemm_traffic_per_step():
    """DRAM bytes (read + write) of the conv GEMM kernels in one step, from the
    ncu counters stored in profiles/ -- or None when they are absent or were
    taken on GEMM sources other than the ones built now (stale)."""
    if not os.path.exists(STEP_TRAFFIC):
        return None
    with open(STEP_TRAFFIC) as f:
        rec = json.load(f)
    if gemm_sources_digest(rec["gemm_sources"]) != rec["gemm_sources_sha256"]:
        return None
    return int(rec["conv_gemm_dram_bytes_per_step"])


def step_flops(layers) -> int:
    return sum(3 * L.gemm_flops for L in layers)


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on a bounded sample

def oracle_sample_run(layers, batch):
    import oracle
    orc = oracle.get()
    flops = 0
    inputs = []
    for L in layers:   # input generation is not part of the timed work
        l = L.with_batch(batch)
        inputs.append((l, l.make()))
    t0 = time.perf_counter()
    for l, (x, w, b, dy) in inputs:
        orc.conv_fwd(x, w, b, l.stride, l.pad)
        orc.conv_bwd_data(w, dy, x.shape, l.stride, l.pad)
        orc.conv_bwd_filter(x, dy, w.shape, l.stride, l.pad)
        orc.conv_bwd_bias(dy)
        flops += 3 * l.gemm_flops
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, orc.threads()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    batch = args.ref_batch
    for _ in range(args.warmup):
        oracle_sample_run(LAYERS, batch)
    vals, times = [], []
    cores = 1
    for _ in range(args.steps):
        v, dt, cores = oracle_sample_run(LAYERS, batch)
        vals.append(v)
        times.append(dt)
    value = len(vals) * step_flops([L.with_batch(batch) for L in LAYERS]) / sum(times) / 1e12
    sample = "AlexNet conv1-5 fwd + input/filter/bias grads at batch %d (of 128) per step" % batch
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_batch": batch},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        # nvidia-smi's start-up queries the driver; let it finish (first sample
        # written, at most 5 s) before the timed launches begin
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        except OSError:
            rows = []
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx = max(mx, float(r[1]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if self.path:
            os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm

class ParamStore:
    """Every layer's filters and bias in one flat device buffer and their
    gradients in another (each tensor a view starting on a 16-byte boundary),
    so that one SGD call updates all parameters of the step.  The padding slots
    between views hold 0 in both buffers, so SGD leaves them unchanged."""

    def __init__(self, layers, torch):
        shapes = []
        for L in layers:
            shapes += [L.w_shape, (L.outC,)]
        sizes = [int(np.prod(sh)) for sh in shapes]
        offs, n = [], 0
        for sz in sizes:
            offs.append(n)
            n += (sz + 3) // 4 * 4
        self.p = torch.zeros(n, device="cuda")
        self.g = torch.zeros(n, device="cuda")
        self.views = [(self.p[o:o + sz].view(sh), self.g[o:o + sz].view(sh))
                      for o, sz, sh in zip(offs, sizes, shapes)]


class LayerBufs:
    def __init__(self, L, torch, cb, params):
        """params: (w, dw, b, db) views of a ParamStore."""
        self.L = L
        x, w, b, dy = L.make()
        self.host = {"x": x, "w": w, "b": b, "dy": dy}
        dev = lambda a: torch.from_numpy(a).cuda()
        self.x, self.dy = dev(x), dev(dy)
        self.w, self.dw, self.b, self.db = params
        self.w.copy_(torch.from_numpy(w))
        self.b.copy_(torch.from_numpy(b))
        self.y = torch.empty(L.y_shape, device="cuda")
        self.dx = torch.empty(L.x_shape, device="cuda")
        self.pool = None
        if L.pool:
            k, s = L.pool
            P = (L.outH - k) // s + 1
            self.pool = (k, s)
            self.yp = torch.empty((L.batch, L.outC, P, P), device="cuda")
            self.idx = torch.empty((L.batch, L.outC, P, P), dtype=torch.int32, device="cuda")
            self.host["dyp"] = synthetic.pool_grad((L.batch, L.outC, P, P), L.seed_base + 20)
            self.dyp = dev(self.host["dyp"])
            self.dxp = torch.empty(L.y_shape, device="cuda")
        s = cb.shape_of(L.x_shape, L.w_shape, L.stride, L.pad)
        self.ws_bytes = max(cb.workspace_bytes(op, s) for op in range(3))

    def bytes_in(self):
        return sum(a.nbytes for a in self.host.values())

    def bytes_out(self):
        n = self.y.numel() + self.dx.numel() + self.dw.numel() + self.db.numel()
        if self.pool:
            n += self.dxp.numel()
        return 4 * n


def run_ours(args):
    import torch
    import im2col_convolution_tiled_gb300 as cb

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    if not os.path.exists(cb.LIB_PATH):
        from im2col_convolution_tiled_gb300 import build
        build.build()
    cb.load()
    fast = args.math == "tf32"
    cb.set_math_mode(cb.CONV_MATH_TF32 if fast else cb.CONV_MATH_FP32)

    def make_set():
        store = ParamStore(LAYERS, torch)
        v = store.views
        return store, [LayerBufs(L, torch, cb, (v[2 * i][0], v[2 * i][1], v[2 * i + 1][0], v[2 * i + 1][1]))
                       for i, L in enumerate(LAYERS)]

    store, bufs = make_set()
    ws = torch.empty(max(b.ws_bytes for b in bufs) + 16, dtype=torch.uint8, device="cuda")
    lr, clip = synthetic.SGD_LR_CLIP
    stream = torch.cuda.current_stream()
    ops = ["fwd", "pool", "dgrad", "wgrad"]   # wgrad includes the bias gradient; SGD runs once per step
    rec = {}   # (layer, op) -> list of (start_event, end_event)

    def timed(key, fn):
        if key is None:
            fn()
            return
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        rec.setdefault(key, []).append((e0, e1))

    def run_layer(b, record):
        L = b.L
        key = (lambda op: (L.name, op)) if record else (lambda op: None)
        timed(key("fwd"), lambda: cb.conv_fwd(b.x, b.w, b.b, L.stride, L.pad, y=b.y, workspace=ws))
        if b.pool:
            k, s = b.pool
            timed(key("pool"), lambda: (cb.maxpool2d_fwd(b.y, k, s, y=b.yp, idx=b.idx),
                                        cb.maxpool2d_bwd(b.dyp, b.idx, L.y_shape, k, s, dx=b.dxp)))
        timed(key("dgrad"), lambda: cb.conv_bwd_data(b.w, b.dy, L.x_shape, L.stride, L.pad, dx=b.dx,
                                                     workspace=ws))
        # filter and bias gradients from one pass over dy (conv_bwd_filter_bias)
        timed(key("wgrad"), lambda: cb.conv_bwd_filter_bias(b.x, b.dy, L.w_shape, L.stride, L.pad, dw=b.dw,
                                                            db=b.db, workspace=ws))

    def sgd(st_, record):
        # SGD on every filter and bias of the step, one launch over the flat store
        timed(("step", "sgd") if record else None, lambda: cb.sgd_step(st_.p, st_.g, lr, clip))

    def step(record):
        for b in bufs:
            run_layer(b, record)
        sgd(store, record)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    # The clock sampler starts before the warm-up, so that whatever its start
    # costs the driver lands in untimed steps; its samples cover warm-up and
    # timed steps.
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            step(False)
        cb.check()

        # --- device-resident timed region ---------------------------------
        # The step is timed as a whole, with nothing between its launches (an
        # event record between two calls would keep the second call's first
        # kernel from overlapping the first call's tail); the per-operation
        # table and the roofline come from as many further steps that record
        # an event pair around every call.
        barrier()
        n0 = cb.launch_count()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            step(False)
        t_end.record(stream)
        launches = cb.launch_count() - n0
        # no synchronisation here: the instrumented steps queue up behind the
        # timed ones, so none of their calls waits on the host to be issued
        for _ in range(args.steps):
            step(True)
        barrier()
    cb.check()
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, dist)
    ms_step = ms_total / args.steps
    flops = step_flops(LAYERS)
    value = job_rate(flops, ms_step, world) / 1e12

    times = {k: sorted(a.elapsed_time(b) for a, b in v) for k, v in rec.items()}
    avg = {k: sum(v) / len(v) for k, v in times.items()}
    per_layer = []
    gemm_ms = 0.0
    for b in bufs:
        L = b.L
        g = L.gemm_flops
        d = {"layer": L.name}
        for op in ops:
            if (L.name, op) in avg:
                v = times[(L.name, op)]
                d[op + "_ms"] = round(avg[(L.name, op)], 4)
                d[op + "_ms_median_min_max"] = [round(statistics.median(v), 4), round(v[0], 4), round(v[-1], 4)]
        for op in ("fwd", "dgrad", "wgrad"):
            d[op + "_tflops"] = round(g / (avg[(L.name, op)] * 1e-3) / 1e12, 2)
            gemm_ms += avg[(L.name, op)]
        d["fwd_bwd_tflops"] = round(3 * g / ((avg[(L.name, "fwd")] + avg[(L.name, "dgrad")] +
                                              avg[(L.name, "wgrad")]) * 1e-3) / 1e12, 2)
        per_layer.append(d)

    bf16, hbm, peak_kind = peaks()
    products = 1 if fast else SPLIT_PRODUCTS
    peak = bf16 * TF32_OVER_BF16 / products
    achieved = flops / (gemm_ms * 1e-3) / 1e12
    traffic = None if fast else gemm_traffic_per_step()

    # --- end to end through the public API with host buffers ---------------
    # As a training loop runs it: every step uploads its batch -- each layer's
    # input x, its upstream gradient dy and the pool gradients -- from pinned
    # host memory, and reads the step's result back: the parameters (every
    # filter and bias) after the SGD update, one flat buffer.  Parameters stay
    # resident on the device between steps.  `e2e_full_readback` additionally
    # uploads the parameters and reads every output of every call back (y, dx,
    # dw, db, pool input gradients).  Two sets of device buffers alternate
    # between steps, as a training loop double-buffers its batches: step i + 1's
    # uploads run on one copy stream and step i - 1's read-backs on another
    # while step i computes.  Within a step, layer i's compute waits only for
    # layer i's uploads.
    pin = lambda a: torch.from_numpy(a).pin_memory()
    host_in = [{k: pin(v) for k, v in b.host.items()} for b in bufs]
    host_out = [{"y": torch.empty(b.L.y_shape).pin_memory(), "dx": torch.empty(b.L.x_shape).pin_memory(),
                 "dw": torch.empty(b.L.w_shape).pin_memory(), "db": torch.empty((b.L.outC,)).pin_memory(),
                 "dxp": torch.empty(b.L.y_shape).pin_memory() if b.pool else None} for b in bufs]
    sets = [(store, bufs), make_set()]
    host_params = torch.empty(store.p.shape).pin_memory()
    batch_keys = ("x", "dy", "dyp")
    h2d_full = sum(b.bytes_in() for b in bufs)
    d2h_full = sum(b.bytes_out() for b in bufs)
    h2d_batch = sum(a.nbytes for b in bufs for k, a in b.host.items() if k in batch_keys)
    d2h_result = host_params.numel() * 4
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_free_in = [torch.cuda.Event() for _ in sets]     # compute of the set's last step is done
    ev_free_out = [torch.cuda.Event() for _ in sets]    # read-back of the set's last step is done
    for e_ in ev_free_in + ev_free_out:
        e_.record(stream)

    def e2e_step(i, full):
        cur_store, cur = sets[i % 2]
        ev_in = [torch.cuda.Event() for _ in cur]
        ev_out = [torch.cuda.Event() for _ in cur]
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(ev_free_in[i % 2])
            for j, (b, hi) in enumerate(zip(cur, host_in)):
                b.x.copy_(hi["x"], non_blocking=True)
                if full:
                    b.w.copy_(hi["w"], non_blocking=True)
                    b.b.copy_(hi["b"], non_blocking=True)
                b.dy.copy_(hi["dy"], non_blocking=True)
                if b.pool:
                    b.dyp.copy_(hi["dyp"], non_blocking=True)
                ev_in[j].record(s_h2d)
        stream.wait_event(ev_free_out[i % 2])
        for j, b in enumerate(cur):
            stream.wait_event(ev_in[j])
            run_layer(b, None)
            if j == len(cur) - 1:
                sgd(cur_store, False)
            ev_out[j].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_out[j])
                if full:
                    ho = host_out[j]
                    ho["y"].copy_(b.y, non_blocking=True)
                    ho["dx"].copy_(b.dx, non_blocking=True)
                    ho["dw"].copy_(b.dw, non_blocking=True)
                    ho["db"].copy_(b.db, non_blocking=True)
                    if b.pool:
                        ho["dxp"].copy_(b.dxp, non_blocking=True)
                elif j == len(cur) - 1:
                    host_params.copy_(cur_store.p, non_blocking=True)
        ev_free_in[i % 2].record(stream)
        ev_free_out[i % 2].record(s_d2h)

    def e2e_run(n, full):
        for i in range(n):
            e2e_step(i, full)
        s_h2d.synchronize()
        s_d2h.synchronize()
        stream.synchronize()

    def e2e_time(full):
        steps = max(3, args.steps // 4)
        e2e_run(2, full)
        barrier()
        t0 = time.perf_counter()
        e2e_run(steps, full)
        barrier()
        return max_over_ranks((time.perf_counter() - t0) * 1e3 / steps, dist)

    e2e_ms = e2e_time(False)
    e2e_full_ms = e2e_time(True)
    cb.check()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, cores = oracle_sample_run(LAYERS, args.cpu_batch)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "AlexNet conv1-5 fwd + input/filter/bias grads at batch %d (of 128), %.1f s"
                         % (args.cpu_batch, dt)}

    working_set = sum(b.bytes_in() + b.bytes_out() for b in bufs)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "tf32" if fast else "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 128, "layers": [L.name for L in LAYERS],
                   "precision": ("one TF32 product on tcgen05 (fast mode), fp32 accumulation" if fast else
                                 "fp32-faithful 3xTF32 on tcgen05, fp32 accumulation"),
                   "step_gflop": round(flops / 1e9, 2),
                   "l2": "no flush: one step streams %.2f GB of distinct tensors (> %d MB L2)"
                         % (working_set / 1e9, L2_BYTES >> 20),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": UNIT,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "conv GEMMs (conv_fwd + conv_bwd_data + conv_bwd_filter, all layers)",
                     "peak_basis": ("%s bf16 %.1f TFLOP/s x %.3f (TF32/BF16)" % (peak_kind, bf16, TF32_OVER_BF16) +
                                    ("" if fast else " / 3 (3xTF32)"))},
        "per_layer": per_layer,
        "sgd_ms_per_step": round(avg[("step", "sgd")], 4),
        "e2e": {"value": round(job_rate(flops, e2e_ms, world) / 1e12, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d_batch, "d2h_bytes_per_step": d2h_result, "ms_per_step": round(e2e_ms, 3),
                "copies": "up: every layer's x and dy and the pool gradients; back: the parameters after SGD"},
        "e2e_full_readback": {"value": round(job_rate(flops, e2e_full_ms, world) / 1e12, 3), "unit": UNIT,
                              "h2d_bytes_per_step": h2d_full, "d2h_bytes_per_step": d2h_full,
                              "ms_per_step": round(e2e_full_ms, 3),
                              "copies": "up: also the parameters; back: every output of every call"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# LeNet-5 training step (--workload lenet): the whole step -- forward, loss,
# backward, SGD over 61,706 parameters -- as one CUDA graph

LENET_METRIC = "LeNet-5 training step (fwd + softmax-CE + bwd + SGD), batch 64: training images/s"
LENET_WORKLOAD = ("LeNet-5, batch 64, 1x28x28 fp32: conv 6@5x5 p2, ReLU, pool 2/2, conv 16@5x5, ReLU, pool 2/2, "
                  "linear 400-120-84-10 with ReLU, softmax cross-entropy, SGD lr 0.01 clip 1.0")


def lenet_step_flops(batch=64) -> int:
    """Algorithmic FLOPs of the step's contractions: conv1 forward and filter
    gradient (its input needs no gradient), conv2 forward, input and filter
    gradients, and three GEMMs per linear layer."""
    c1, c2 = synthetic.LENET
    f = 2 * c1.with_batch(batch).gemm_flops + 3 * c2.with_batch(batch).gemm_flops
    f += sum(3 * 2 * batch * fin * fout for fin, fout in synthetic.LENET_FC)
    return f


def oracle_lenet_run(steps):
    import oracle.lenet as olenet
    params = synthetic.lenet_params()
    x, labels = synthetic.lenet_batch()
    t0 = time.perf_counter()
    for _ in range(steps):
        params, _, _ = olenet.step(params, x, labels)
    return time.perf_counter() - t0


def run_lenet_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    oracle_lenet_run(args.warmup)
    dt = oracle_lenet_run(args.steps)
    value = args.steps * 64 / dt
    line = {
        "impl": "reference", "metric": LENET_METRIC, "value": value, "unit": "images/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": LENET_WORKLOAD},
        "cpu_baseline": {"value": value, "unit": "images/s", "cores": oracle.get().threads(), "kind": "oracle",
                         "sample": "the full batch-64 step"},
        "e2e": {"value": value, "unit": "images/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_lenet(args):
    import torch
    import im2col_convolution_tiled_gb300 as cb
    from im2col_convolution_tiled_gb300.lenet import LeNet5

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if not os.path.exists(cb.LIB_PATH):
        from im2col_convolution_tiled_gb300 import build
        build.build()
    cb.load()

    B = 64
    x, labels = synthetic.lenet_batch(B)
    net = LeNet5(synthetic.lenet_params(), batch=B)
    net.load_batch(x, labels)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    # eager (one library call per operation from Python), for comparison
    for _ in range(args.warmup):
        net.run()
    barrier()
    n0 = cb.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        net.run()
    e1.record(stream)
    barrier()
    launches_per_step = (cb.launch_count() - n0) // args.steps
    eager_ms = e0.elapsed_time(e1) / args.steps

    # graph: capture once, replay
    net.capture()
    with ClockSampler(local) as clk:   # started before the warm-up replays (see run_ours)
        for _ in range(args.warmup):
            net.replay()
        barrier()
        e0.record(stream)
        for _ in range(args.steps):
            net.replay()
        e1.record(stream)
        barrier()
    cb.check()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, dist)
    value = job_rate(B, ms, world)

    # end to end: each step's batch goes up from pinned host memory and its loss comes back
    hx = torch.from_numpy(x).pin_memory()
    hl = torch.from_numpy(labels).pin_memory()
    hloss = torch.empty(1).pin_memory()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        net.t["x"].copy_(hx, non_blocking=True)
        net.t["labels"].copy_(hl, non_blocking=True)
        net.replay()
        hloss.copy_(net.t["loss"], non_blocking=True)
    stream.synchronize()
    barrier()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.steps, dist)
    cb.check()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = 20
        dt = oracle_lenet_run(n)
        import oracle
        cpu = {"value": n * B / dt, "unit": "images/s", "cores": oracle.get().threads(), "kind": "oracle",
               "sample": "%d full batch-64 steps, %.1f s" % (n, dt)}
    flops = lenet_step_flops(B)
    line = {
        "metric": LENET_METRIC, "value": round(value, 1), "unit": "images/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": LENET_WORKLOAD, "batch": B, "params": 61706,
                   "step_gflop": round(flops / 1e9, 4), "l2": "no flush: the whole step (about 10 MB) is L2-resident",
                   "eager_ms_per_step": round(eager_ms, 4),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "latency", "launches_per_step": launches_per_step,
                     "us_per_launch": round(1e3 * ms / launches_per_step, 2),
                     "achieved": round(flops / (ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s", "peak": None,
                     "frac": None, "traffic": None,
                     "note": "dependent launches of small kernels; the graph removes the host issue cost"},
        "e2e": {"value": round(job_rate(B, e2e_ms, world), 1), "unit": "images/s",
                "h2d_bytes_per_step": int(x.nbytes + labels.nbytes), "d2h_bytes_per_step": 4,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# direct convolution vs implicit GEMM (--workload direct): the page's legacy
# direct kernels as an ablation on small-channel and large layers

DIRECT_METRIC = "direct (CUDA-core) vs implicit-GEMM (tcgen05) convolution time, fwd + input grad + filter grad"


def run_direct(args):
    import torch
    import im2col_convolution_tiled_gb300 as cb

    if int(os.environ.get("RANK", "0")) != 0:
        return
    if not os.path.exists(cb.LIB_PATH):
        from im2col_convolution_tiled_gb300 import build
        build.build()
    cb.load()
    layers = [synthetic.SINGLE] + list(synthetic.LENET) + [synthetic.ALEXNET_CONV1]
    stream = torch.cuda.current_stream()

    def timed(fn, reps):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    rows = []
    total = {"gemm": 0.0, "direct": 0.0}
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        for L in layers:
            x, w, b, dy = (torch.from_numpy(a).cuda() for a in L.make())
            s = cb.shape_of(L.x_shape, L.w_shape, L.stride, L.pad)
            ws = torch.empty(max(cb.workspace_bytes(op, s) for op in range(3)) + 16, dtype=torch.uint8, device="cuda")
            y, dx, dw = torch.empty(L.y_shape, device="cuda"), torch.empty(L.x_shape, device="cuda"), \
                torch.empty(L.w_shape, device="cuda")
            gemm = lambda: (cb.conv_fwd(x, w, b, L.stride, L.pad, y=y, workspace=ws),
                            cb.conv_bwd_data(w, dy, L.x_shape, L.stride, L.pad, dx=dx, workspace=ws),
                            cb.conv_bwd_filter(x, dy, L.w_shape, L.stride, L.pad, dw=dw, workspace=ws))
            direct = lambda: (cb.conv_fwd_direct(x, w, b, L.stride, L.pad, y=y),
                              cb.conv_bwd_data_direct(w, dy, L.x_shape, L.stride, L.pad, dx=dx),
                              cb.conv_bwd_filter_direct(x, dy, L.w_shape, L.stride, L.pad, dw=dw))
            reps = max(2, args.steps if L.batch < 128 else args.steps // 10)
            tg, td = timed(gemm, reps), timed(direct, reps)
            total["gemm"] += tg
            total["direct"] += td
            rows.append({"layer": L.name, "gemm_ms": round(tg, 4), "direct_ms": round(td, 4),
                         "direct_over_gemm": round(td / tg, 3),
                         "gemm_tflops": round(3 * L.gemm_flops / (tg * 1e-3) / 1e12, 3),
                         "direct_tflops": round(3 * L.gemm_flops / (td * 1e-3) / 1e12, 3)})
    cb.check()
    line = {
        "metric": DIRECT_METRIC, "value": round(total["direct"] / total["gemm"], 3), "unit": "time ratio",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "single conv b4, LeNet conv1/conv2 b64, AlexNet conv1 b128; each layer's three "
                               "convolution calls", "layers": rows},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# flagged matmul (--workload matmul): shapes of the matmul sweep, every flag

MATMUL_METRIC = "flagged fp32 matmul C = op(A) op(B): TFLOP/s (3xTF32 on tcgen05) and % of tensor roofline"
MATMUL_SHAPES = [(9216, 9216, 4096), (4096, 4096, 4096), (9216, 9216, 363), (1024, 1024, 1600), (128, 9216, 2304),
                 (16, 4096, 4096), (127, 127, 150)]


def run_matmul(args):
    import torch
    import im2col_convolution_tiled_gb300 as cb

    if int(os.environ.get("RANK", "0")) != 0:
        return
    if not os.path.exists(cb.LIB_PATH):
        from im2col_convolution_tiled_gb300 import build
        build.build()
    cb.load()
    bf16, hbm, peak_kind = peaks()
    tf32 = args.math == "tf32"
    cb.set_math_mode(cb.CONV_MATH_TF32 if tf32 else cb.CONV_MATH_FP32)
    peak = bf16 * TF32_OVER_BF16 / (1 if tf32 else SPLIT_PRODUCTS)
    stream = torch.cuda.current_stream()
    rows = []
    flops_all, ms_all = 0, 0.0
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        for M, N, K in MATMUL_SHAPES:
            for flags in range(4):
                A, B = synthetic.matmul_case(M, K, N, flags)
                a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
                c = torch.empty((M, N), device="cuda")
                reps = args.steps if M * N * K < 2 ** 32 else max(3, args.steps // 5)
                for _ in range(args.warmup):
                    cb.matmul(a, b, flags, C=c)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                for _ in range(reps):
                    cb.matmul(a, b, flags, C=c)
                e1.record(stream)
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / reps
                f = 2 * M * N * K
                flops_all += f
                ms_all += ms
                bn, pieces, fed = cb.matmul_tiling(M, K, N, flags, a, b, with_tma=True)
                rows.append({"M": M, "N": N, "K": K, "flags": flags, "ms": round(ms, 4), "tma_fed": fed,
                             "tflops": round(f / (ms * 1e-3) / 1e12, 2), "frac": round(f / (ms * 1e-3) / 1e12 / peak, 4),
                             "frac_attainable": round(f / (ms * 1e-3) / 1e12 / attainable_tflops(M, N, K, peak, hbm), 4),
                             "tile_cols": bn, "k_pieces": pieces})
    cb.check()
    big = [r for r in rows if (r["M"], r["N"], r["K"]) == MATMUL_SHAPES[0]]
    value = sum(2 * r["M"] * r["N"] * r["K"] for r in big) / (sum(r["ms"] for r in big) * 1e-3) / 1e12
    line = {
        "metric": MATMUL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "tf32" if tf32 else "f32",
        "data": "synthetic",
        "config": {"workload": "largest sweep shape M=N=9216, K=4096, all four flags (value); the table covers "
                               "further sweep shapes", "shapes": rows,
                   "all_shapes_tflops": round(flops_all / (ms_all * 1e-3) / 1e12, 2), "math": args.math,
                   "l2": "no flush: operands of the value's shape are 0.6 GB (> 126 MB L2)"},
        "roofline": {"bound": "tensor", "achieved": round(value, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(value / peak, 4), "traffic": None,
                     "peak_basis": "%s bf16 %.1f TFLOP/s x %.3f (TF32/BF16)%s"
                                   % (peak_kind, bf16, TF32_OVER_BF16, "" if tf32 else " / 3 (3xTF32)")},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# helpers shared by the per-kernel workloads below

def _load_lib():
    import im2col_convolution_tiled_gb300 as cb
    if not os.path.exists(cb.LIB_PATH):
        from im2col_convolution_tiled_gb300 import build
        build.build()
    cb.load()
    return cb


def graph_time_ms(run, reps, warmup=3):
    """Mean device time of one run() over `reps` calls captured once into a
    CUDA graph and replayed between CUDA events on the launching stream (host
    issue cost cannot hide short kernels).  run() must allocate nothing."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):
            run()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            run()
    g.replay()   # one untimed replay
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def layer_tensors(cb, L):
    """Device tensors of one layer workload plus preallocated outputs and one
    workspace large enough for its three convolution calls."""
    import torch
    x, w, b, dy = (torch.from_numpy(a).cuda() for a in L.make())
    s = cb.shape_of(L.x_shape, L.w_shape, L.stride, L.pad)
    ws = torch.empty(max(cb.workspace_bytes(op, s) for op in range(3)) + 16, dtype=torch.uint8, device="cuda")
    return {"x": x, "w": w, "b": b, "dy": dy, "ws": ws, "y": torch.empty(L.y_shape, device="cuda"),
            "dx": torch.empty(L.x_shape, device="cuda"), "dw": torch.empty(L.w_shape, device="cuda"),
            "db": torch.empty(L.outC, device="cuda")}


# ---------------------------------------------------------------------------
# the single convolution layer (--workload single): batch 4, 1x28x28, six 5x5
# filters -- the forward and the three gradients of one ConvLayer

SINGLE_METRIC = "single conv layer fwd+bwd (batch 4, 1x28x28 -> 6@5x5): TFLOP/s of the three GEMMs"


def run_single(args):
    import torch
    cb = _load_lib()
    if int(os.environ.get("RANK", "0")) != 0:
        return
    L = synthetic.SINGLE
    t = layer_tensors(cb, L)

    def step():
        cb.conv_fwd(t["x"], t["w"], t["b"], L.stride, L.pad, y=t["y"], workspace=t["ws"])
        cb.conv_bwd_data(t["w"], t["dy"], L.x_shape, L.stride, L.pad, dx=t["dx"], workspace=t["ws"])
        cb.conv_bwd_filter_bias(t["x"], t["dy"], L.w_shape, L.stride, L.pad, dw=t["dw"], db=t["db"],
                                workspace=t["ws"])

    n0 = cb.launch_count()
    step()
    launches = cb.launch_count() - n0
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        ms = graph_time_ms(step, args.steps, args.warmup)
    cb.check()
    flops = 3 * L.gemm_flops
    value = flops / (ms * 1e-3) / 1e12

    # end to end: x and dy up from pinned host memory, y, dx, dw, db back, per step
    hx, hdy = (torch.from_numpy(a).pin_memory() for a in L.make()[0:4:3])
    outs = {k: torch.empty(t[k].shape).pin_memory() for k in ("y", "dx", "dw", "db")}
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        t["x"].copy_(hx, non_blocking=True)
        t["dy"].copy_(hdy, non_blocking=True)
        step()
        for k, v in outs.items():
            v.copy_(t[k], non_blocking=True)
    stream.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    cb.check()

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        orc = oracle.get()
        x, w, b, dy = L.make()
        n = 200
        t0 = time.perf_counter()
        for _ in range(n):
            orc.conv_fwd(x, w, b, L.stride, L.pad)
            orc.conv_bwd_data(w, dy, x.shape, L.stride, L.pad)
            orc.conv_bwd_filter(x, dy, w.shape, L.stride, L.pad)
            orc.conv_bwd_bias(dy)
        dt = time.perf_counter() - t0
        cpu = {"value": n * flops / dt / 1e12, "unit": "TFLOP/s", "cores": orc.threads(), "kind": "oracle",
               "sample": "the whole layer (forward and the three gradients) %d times, %.2f s" % (n, dt)}
    line = {
        "metric": SINGLE_METRIC, "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "single conv layer, batch 4, 1x28x28 U[0,1) -> 6 filters 5x5, stride 1, pad 0: "
                               "conv_fwd, conv_bwd_data, conv_bwd_filter_bias, one CUDA graph",
                   "gflop_per_step": round(flops / 1e9, 5), "l2": "no flush: the layer is 0.1 MB, L2-resident"},
        "roofline": {"bound": "latency", "launches_per_step": launches,
                     "us_per_launch": round(1e3 * ms / max(launches, 1), 2), "achieved": round(value, 4),
                     "unit": "TFLOP/s", "peak": None, "frac": None, "traffic": None,
                     "note": "2.1 MFLOP over dependent launches: far below any throughput roofline"},
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(hx.numel() * 4 + hdy.numel() * 4),
                "d2h_bytes_per_step": int(sum(v.numel() * 4 for v in outs.values())),
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# HBM-bound kernels (--workload hbm): im2col, col2im, max pooling, the
# standalone bias gradient and SGD on the AlexNet batch-128 shapes, each
# timed alone (graph-replayed) against the measured copy bandwidth

HBM_METRIC = "HBM-bound kernels on AlexNet batch-128 shapes: GB/s of algorithmic bytes and fraction of copy bandwidth"


def hbm_cases(cb, torch):
    """(name, algorithmic bytes, run) for every HBM-bound kernel measured."""
    cases = []
    for L in synthetic.ALEXNET:
        x = torch.from_numpy(L.make()[0]).cuda()
        ncol = L.inC * L.k * L.k * L.batch * L.outH * L.outW
        col = torch.empty(ncol, device="cuda").view(L.inC * L.k * L.k, -1)
        dx = torch.empty(L.x_shape, device="cuda")
        nb = 4 * (x.numel() + ncol)
        cases.append(("im2col " + L.name, nb, lambda x=x, col=col, L=L: cb.im2col(x, L.k, L.stride, L.pad, col=col)))
        cases.append(("col2im " + L.name, nb, lambda col=col, dx=dx, L=L:
                      cb.col2im(col, L.x_shape, L.k, L.stride, L.pad, dx=dx)))
        dy = torch.from_numpy(synthetic.normal(L.y_shape, L.seed_base + 4)).cuda()
        db = torch.empty(L.outC, device="cuda")
        cases.append(("bias_grad " + L.name, 4 * dy.numel(), lambda dy=dy, db=db: cb.conv_bwd_bias(dy, db=db)))
        if L.pool:
            k, st = L.pool
            xp = torch.from_numpy(synthetic.pool_input(L)).cuda()
            yp, idx = cb.maxpool2d_fwd(xp, k, st)
            dyp = torch.from_numpy(synthetic.pool_grad(tuple(yp.shape), 5)).cuda()
            dxp = torch.empty(L.y_shape, device="cuda")
            fwd_b = 4 * (xp.numel() + 2 * yp.numel())
            bwd_b = 4 * (2 * yp.numel() + xp.numel())
            cases.append(("maxpool_fwd %dx%d/%d after %s" % (k, k, st, L.name), fwd_b,
                          lambda xp=xp, yp=yp, idx=idx, k=k, st=st: cb.maxpool2d_fwd(xp, k, st, y=yp, idx=idx)))
            cases.append(("maxpool_bwd %dx%d/%d after %s" % (k, k, st, L.name), bwd_b,
                          lambda dyp=dyp, idx=idx, dxp=dxp, k=k, st=st, L=L:
                          cb.maxpool2d_bwd(dyp, idx, L.y_shape, k, st, dx=dxp)))
    n = sum(L.outC * L.inC * L.k * L.k + L.outC for L in synthetic.ALEXNET)
    for count, what in ((n, "AlexNet conv1-5 filters and biases"), (1 << 26, "64 M parameters")):
        p = torch.from_numpy(synthetic.normal((count,), 71)).cuda()
        g = torch.from_numpy(synthetic.normal((count,), 72)).cuda()
        cases.append(("sgd_step " + what, 12 * count, lambda p=p, g=g: cb.sgd_step(p, g, 0.01, 1.0)))
    return cases


def run_hbm(args):
    import torch
    cb = _load_lib()
    if int(os.environ.get("RANK", "0")) != 0:
        return
    _, hbm, peak_kind = peaks()
    rows = []
    n0 = cb.launch_count()
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        for name, nbytes, run in hbm_cases(cb, torch):
            reps = max(5, min(args.steps, 50))
            ms = graph_time_ms(run, reps, args.warmup)
            gbs = nbytes / (ms * 1e-3) / 1e9
            rows.append({"kernel": name, "mb": round(nbytes / 1e6, 2), "us": round(ms * 1e3, 2),
                         "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4)})
            torch.cuda.empty_cache()
    cb.check()
    launches = cb.launch_count() - n0
    big = [r for r in rows if r["mb"] >= 100]
    tot_b = sum(r["mb"] for r in big) * 1e6
    tot_s = sum(r["us"] for r in big) * 1e-6
    value = tot_b / tot_s / 1e9
    dom = max(rows, key=lambda r: r["us"])
    line = {
        "metric": HBM_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "im2col, col2im, bias gradient (AlexNet conv1-5, batch 128), max pool fwd / bwd "
                               "(3x3 stride 2 after conv1 and conv2), SGD; value = algorithmic bytes / time over "
                               "the kernels moving >= 100 MB per call",
                   "kernels": rows,
                   "l2": "no flush: every kernel of >= 100 MB streams more than L2; smaller ones are listed "
                         "but left out of the value"},
        "roofline": {"bound": "hbm", "kernel": dom["kernel"], "achieved": dom["gbs"], "peak": round(hbm, 1),
                     "unit": "GB/s", "frac": dom["frac"], "traffic": None,
                     "peak_basis": "%s copy bandwidth" % peak_kind},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# one entry point on one workload (--workload case): a small fixed command for
# a profiler to attach to; nothing is timed or checked

def run_case(args):
    import torch
    cb = _load_lib()
    cb.set_math_mode(cb.CONV_MATH_TF32 if args.math == "tf32" else cb.CONV_MATH_FP32)
    layers = {L.name: L for L in synthetic.ALEXNET + synthetic.LENET + (synthetic.SINGLE,)}
    if args.op == "matmul":
        M, N, K = (int(v) for v in args.mnk.split(","))
        A, B = synthetic.matmul_case(M, K, N, args.flags)
        At, Bt = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        C = torch.empty((M, N), device="cuda")
        run = lambda: cb.matmul(At, Bt, args.flags, C=C)
    else:
        L = layers[args.layer]
        t = layer_tensors(cb, L)
        if args.op == "fwd":
            run = lambda: cb.conv_fwd(t["x"], t["w"], t["b"], L.stride, L.pad, y=t["y"], workspace=t["ws"])
        elif args.op == "dgrad":
            run = lambda: cb.conv_bwd_data(t["w"], t["dy"], L.x_shape, L.stride, L.pad, dx=t["dx"], workspace=t["ws"])
        elif args.op == "wgrad":
            run = lambda: cb.conv_bwd_filter_bias(t["x"], t["dy"], L.w_shape, L.stride, L.pad, dw=t["dw"],
                                                  db=t["db"], workspace=t["ws"])
        elif args.op == "bias":
            run = lambda: cb.conv_bwd_bias(t["dy"], db=t["db"])
        elif args.op in ("pool", "poolfwd", "poolbwd"):
            k, st = L.pool or (2, 2)
            xp = torch.from_numpy(synthetic.pool_input(L)).cuda()
            yp, idx = cb.maxpool2d_fwd(xp, k, st)
            dyp = torch.from_numpy(synthetic.pool_grad(tuple(yp.shape), 5)).cuda()
            dxp = torch.empty(L.y_shape, device="cuda")
            f = lambda: cb.maxpool2d_fwd(xp, k, st, y=yp, idx=idx)
            bw = lambda: cb.maxpool2d_bwd(dyp, idx, L.y_shape, k, st, dx=dxp)
            run = {"pool": lambda: (f(), bw()), "poolfwd": f, "poolbwd": bw}[args.op]
        elif args.op == "im2col":
            col = torch.empty((L.inC * L.k * L.k, L.batch * L.outH * L.outW), device="cuda")
            run = lambda: cb.im2col(t["x"], L.k, L.stride, L.pad, col=col)
        elif args.op == "col2im":
            col = torch.from_numpy(synthetic.normal((L.inC * L.k * L.k, L.batch * L.outH * L.outW), 6)).cuda()
            run = lambda: cb.col2im(col, L.x_shape, L.k, L.stride, L.pad, dx=t["dx"])
        elif args.op == "sgd":
            p = torch.from_numpy(synthetic.normal((1 << 26,), 71)).cuda()
            g = torch.from_numpy(synthetic.normal((1 << 26,), 72)).cuda()
            run = lambda: cb.sgd_step(p, g, 0.01, 1.0)
        else:
            raise SystemExit("unknown --op %s" % args.op)
    for _ in range(args.steps):
        run()
    cb.check()
    print("case done: %s %s x%d" % (args.mnk if args.op == "matmul" else args.layer, args.op, args.steps))


# ---------------------------------------------------------------------------
# the whole flagged-matmul sweep (--workload matmul_sweep): every one of the
# 1176 (M, N, K, flags) cases timed on its own

def attainable_tflops(M, N, K, peak_tflops, hbm_gbs):
    """Roofline of one case: the tensor peak, or the HBM bandwidth times the
    arithmetic intensity at minimal traffic (read A and B once, write C once),
    whichever is lower."""
    ai = 2.0 * M * N * K / (4.0 * (M * K + K * N + M * N))
    return min(peak_tflops, ai * hbm_gbs * 1e-3)


def run_matmul_sweep(args):
    import torch
    import im2col_convolution_tiled_gb300 as cb

    if int(os.environ.get("RANK", "0")) != 0:
        return
    if not os.path.exists(cb.LIB_PATH):
        from im2col_convolution_tiled_gb300 import build
        build.build()
    cb.load()
    bf16, hbm, peak_kind = peaks()
    tf32 = args.math == "tf32"
    cb.set_math_mode(cb.CONV_MATH_TF32 if tf32 else cb.CONV_MATH_FP32)
    peak = bf16 * TF32_OVER_BF16 / (1 if tf32 else SPLIT_PRODUCTS)
    stream = torch.cuda.current_stream()
    pools = [torch.from_numpy(synthetic.matmul_pool(i)).cuda() for i in (0, 1)]
    big = max(synthetic.MATMUL_MN)
    cbuf = torch.empty(big * big, dtype=torch.float32, device="cuda")
    rows = []
    flops_all, ms_all = 0, 0.0
    n0 = cb.launch_count()
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        for M, K, N, flags in synthetic.matmul_sweep():
            oa, ob = synthetic.matmul_sweep_offsets(M, K, N, flags)
            a = pools[0][oa:oa + M * K].view(*((K, M) if flags & 1 else (M, K)))
            b = pools[1][ob:ob + K * N].view(*((N, K) if flags & 2 else (K, N)))
            c = cbuf[:M * N].view(M, N)
            f = 2 * M * N * K
            est_ms = f / 150e12 * 1e3 + 0.005
            reps = int(min(50, max(3, 1.0 / est_ms)))
            cb.matmul(a, b, flags, C=c)   # warm-up
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                cb.matmul(a, b, flags, C=c)
            e1.record(stream)
            e1.synchronize()
            ms = e0.elapsed_time(e1) / reps
            flops_all += f
            ms_all += ms
            att = attainable_tflops(M, N, K, peak, hbm)
            tfl = f / (ms * 1e-3) / 1e12
            bn, pieces, fed = cb.matmul_tiling(M, K, N, flags, a, b, with_tma=True)
            rows.append({"M": M, "N": N, "K": K, "flags": flags, "ms": round(ms, 5), "tflops": round(tfl, 2),
                         "frac": round(tfl / peak, 4), "frac_attainable": round(tfl / att, 4),
                         "tile_cols": bn, "k_pieces": pieces, "tma_fed": fed})
    cb.check()
    launches = cb.launch_count() - n0
    small = [r for r in rows if min(r["M"], r["N"]) < 128]
    large = [r for r in rows if min(r["M"], r["N"]) >= 128]

    def agg(rs):
        fl = sum(2 * r["M"] * r["N"] * r["K"] for r in rs)
        ms = sum(r["ms"] for r in rs)
        return {"cases": len(rs), "tflops": round(fl / (ms * 1e-3) / 1e12, 2),
                "median_frac_attainable": round(statistics.median(r["frac_attainable"] for r in rs), 4),
                "min_frac_attainable": min(r["frac_attainable"] for r in rs)}

    value = flops_all / (ms_all * 1e-3) / 1e12
    worst = sorted(rows, key=lambda r: r["frac_attainable"])[:12]
    if args.table:
        with open(args.table, "w") as fh:
            json.dump(rows, fh)
    line = {
        "metric": MATMUL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": 1,
        "warmup": 1, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "tf32" if tf32 else "f32", "data": "synthetic",
        "config": {"workload": "the whole flagged-matmul sweep: M, N in %s, K in %s, flags 0-3 (1176 cases); "
                               "value = total sweep FLOP / summed per-case time"
                               % (list(synthetic.MATMUL_MN), list(synthetic.MATMUL_K)),
                   "math": args.math, "small_regime": agg(small), "large_regime": agg(large),
                   "worst_cases": worst, "table": args.table,
                   "l2": "no flush; each case repeated on the same operands (small cases run from L2)"},
        "roofline": {"bound": "tensor", "achieved": round(value, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(value / peak, 4), "traffic": None,
                     "peak_basis": "%s bf16 %.1f TFLOP/s x %.3f (TF32/BF16)%s; frac_attainable per case uses "
                                   "min(peak, intensity x %.1f GB/s)"
                                   % (peak_kind, bf16, TF32_OVER_BF16, "" if tf32 else " / 3 (3xTF32)", hbm)},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-batch", type=int, default=64)
    ap.add_argument("--ref-batch", type=int, default=1)
    ap.add_argument("--workload", choices=["alexnet", "lenet", "single", "direct", "matmul", "matmul_sweep",
                                           "hbm", "case"], default="alexnet")
    ap.add_argument("--layer", default="alexnet_conv2_b128", help="case: the layer workload")
    ap.add_argument("--op", default="fwd", help="case: fwd, dgrad, wgrad, bias, pool, poolfwd, poolbwd, im2col, "
                                                "col2im, sgd or matmul")
    ap.add_argument("--mnk", default="4096,4096,4096", help="case --op matmul: M,N,K")
    ap.add_argument("--flags", type=int, default=0, help="case --op matmul: transpose flags")
    ap.add_argument("--table", default=None, help="matmul_sweep: write the per-case table (JSON) here")
    ap.add_argument("--math", choices=["fp32", "tf32"], default="fp32",
                    help="contractions in fp32-faithful 3xTF32 (default) or one TF32 product")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps, always
    if args.workload == "lenet":
        (run_lenet_reference if args.impl == "reference" else run_lenet)(args)
    elif args.workload == "direct":
        run_direct(args)
    elif args.workload == "matmul":
        run_matmul(args)
    elif args.workload == "matmul_sweep":
        run_matmul_sweep(args)
    elif args.workload == "single":
        run_single(args)
    elif args.workload == "hbm":
        run_hbm(args)
    elif args.workload == "case":
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
