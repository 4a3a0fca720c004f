#!/usr/bin/env python
"""Benchmark of the INT8 convrot linear on one GB300 (or N, one process each).

One step is one pass of the whole hot path over one batch: pack the
activations (rotate + row absmax + quantize, one kernel) and run the linear
(integer GEMM + fused scale/bias epilogue, one kernel) for the DiT MLP
up-projection M=4096, K=3072, N=12288, G=256. Weights are quantized once,
offline, before timing (the page "INT8 Convrot Safetensors" stores them
quantized). Inputs are seeded synthetic tensors resident in HBM.

Prints one JSON line (rank 0). ``--impl reference`` times the oracle (the
plain fp64 CPU statement of the layer) on the host cores instead.
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

from int8_hadamard_rotated_convrot_gb300.inputs import stage_shapes  # noqa: E402  (seeded shapes only)

METRIC = "convrot linear INT8 TOPS + pack GB/s at 4096x3072x12288, % of roofline"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mlp_up")
    ap.add_argument("--codes", choices=["auto", "i8", "bf16"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused-pack", action="store_true",
                    help="MLP pair: pack the up projection's output in its epilogue (convrot_linear_act_pack) "
                         "instead of a separate pack launch")
    ap.add_argument("--eager", action="store_true",
                    help="launch the timed steps one call at a time instead of replaying them as one CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="approximate CPU time budget of the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def slowest_rank(values, pg, device):
    """Each per-rank time replaced by its maximum over all ranks: the slowest
    rank sets the job's time. Works over gloo (CPU tensors) or NCCL."""
    if pg is None:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_tops(world: int, ops_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own full workload per step."""
    return world * ops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def measured_traffic(workload: str, codes: str):
    """DRAM bytes per GEMM launch from the committed ncu summary, if the kernel is unchanged since."""
    import hashlib

    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tpath):
        return None
    entry = json.load(open(tpath)).get(f"{workload}/{codes}")
    if not entry:
        return None
    h = hashlib.sha256()
    for rel in entry["sources"]:  # the kernel's file and the headers it is built from, in order
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    if h.hexdigest()[:16] != entry["sha256_16"]:
        return None
    return entry["gemm_bytes"]


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.uuid and parts[0] != self.uuid:
                    continue
                rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- CPU baseline (the oracle)
def oracle_sample_run(wl, rows: int, packed_w, X, split=None):
    """One oracle pass over `rows` rows of the workload: for each stage pack,
    integer GEMM and reconstruct (with the stage's activation). `split`, if
    given, accumulates the seconds spent in the packs and in GEMM + reconstruct."""
    import oracle

    H = X[:rows]
    for (Qw, sw, b), st in zip(packed_w, stage_shapes(wl)):
        t0 = time.perf_counter()
        Qx, sx, _ = oracle.pack_rows(H, wl.G, want_pre_round=False)
        t1 = time.perf_counter()
        A = oracle.gemm_i32(Qx, Qw, st.k)
        H, _ = oracle.reconstruct(A, sx, sw, b, st.act)
        if split is not None:
            split["pack"] += t1 - t0
            split["gemm"] += time.perf_counter() - t1


def cpu_baseline(wl, budget_s: float, steps: int = 1, warmup: int = 0):
    """Times the oracle as it stands on this host's cores on a bounded row sample."""
    import oracle
    from int8_hadamard_rotated_convrot_gb300 import inputs

    oracle.build()
    X = inputs.activations(wl)
    packed_w = []
    for s_i, _ in enumerate(stage_shapes(wl)):  # offline, untimed
        Ws, b = inputs.stage_weights(wl, s_i)
        Qw, sw, _ = oracle.pack_rows(np.concatenate(Ws), wl.G, want_pre_round=False)
        packed_w.append((Qw, sw, b))
    per_row, trial = 1.0, 2
    for _ in range(2):  # calibrate on a small, then a larger trial
        t0 = time.perf_counter()
        oracle_sample_run(wl, trial, packed_w, X)
        per_row = max((time.perf_counter() - t0) / trial, 1e-6)
        trial = int(max(2, min(X.shape[0], 0.2 * budget_s / max(steps, 1) / per_row)))
    rows = int(max(2, min(X.shape[0], budget_s / max(steps, 1) / per_row)))
    for _ in range(warmup):
        oracle_sample_run(wl, rows, packed_w, X)
    times = []
    split = {"pack": 0.0, "gemm": 0.0}
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle_sample_run(wl, rows, packed_w, X, split)
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    ops = wl.step_ops * rows / wl.m
    pack_bytes = sum(rows * (5 * st.k + 4) for st in stage_shapes(wl))
    what = " then ".join(f"pack + int GEMM vs {st.n} weight rows + reconstruct" for st in stage_shapes(wl))
    scope = ("the full shape" if rows == wl.m else
             f"a {rows}-row subset; rows are independent, so the rate stands for all {wl.m} rows (extrapolated)")
    return {"value": ops / t / 1e12, "unit": "TOPS", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} of {wl.m} rows of {wl.name} ({what}), fp64 oracle, "
                      f"{len(times)} step(s) of {t:.2f} s: {scope}",
            "seconds_per_step": t,
            "pack_gbs": pack_bytes * steps / max(split["pack"], 1e-9) / 1e9,
            "gemm_tops": ops * steps / max(split["gemm"], 1e-9) / 1e12}


def workload_name(wl) -> str:
    if wl.lora_r:
        return f"{wl.name} M{wl.m} K{wl.k} N{wl.n} G{wl.G} + LoRA r{wl.lora_r} scale {wl.lora_scale:g}"
    if wl.down_n:
        return f"{wl.name} M{wl.m} K{wl.k} N{wl.n} (GELU in the epilogue) -> K{wl.n} N{wl.down_n} G{wl.G}"
    grouped = f"x{wl.linears} (one grouped GEMM)" if wl.linears > 1 else ""
    return f"{wl.name} M{wl.m} K{wl.k} N{wl.n}{grouped} G{wl.G}"


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from int8_hadamard_rotated_convrot_gb300 import inputs

    wl = inputs.WORKLOADS[args.workload]
    if world > 1:
        # torch.distributed.run sets OMP_NUM_THREADS=1 in every rank; rank 0 is the only
        # one working here, so the oracle gets this process's cores (read before it loads)
        os.environ["OMP_NUM_THREADS"] = str(len(os.sched_getaffinity(0)))
    budget = max(1.0, min(args.cpu_seconds, 120.0 / max(args.steps + args.warmup, 1)))
    cb = cpu_baseline(wl, budget * (args.steps), steps=args.steps, warmup=args.warmup)
    line = {
        "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "TOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["seconds_per_step"] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(wl), "sample": cb["sample"]},
        "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "pack_gbs", "gemm_tops")},
        "e2e": {"value": cb["value"], "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    from int8_hadamard_rotated_convrot_gb300 import build, inputs
    from int8_hadamard_rotated_convrot_gb300 import convrot as cr

    build.build()
    cr.load()
    wl = inputs.WORKLOADS[args.workload]
    codes = {"i8": cr.CODES_I8, "bf16": cr.CODES_BF16, "auto": cr.CODES_BF16}[args.codes]

    # inputs: every rank runs the full workload on its own GPU (weak scaling; rows are independent)
    stages = stage_shapes(wl)
    X = torch.from_numpy(inputs.activations(wl)).to(dev)
    code_b = 1 if codes == cr.CODES_I8 else 2
    touched = wl.m * wl.k * 4 + sum(st.n * st.k * code_b + wl.m * st.n * 4 + wl.m * st.k * code_b for st in stages)
    R = max(2, -(-3 * L2_BYTES // touched) + 1)  # rotating sets so a reuse is > 2 L2s away
    R = min(R, 6)
    Xs = [X] + [X.clone() for _ in range(R - 1)]
    pws, biases, pxs, Ys = [], [], [], []
    for s_i, st in enumerate(stages):
        # linears sharing the packed input (q, k, v) run as one grouped GEMM over concatenated weights
        Ws_np, b_np = inputs.stage_weights(wl, s_i)
        Ws = [torch.from_numpy(W).to(dev) for W in Ws_np]
        pws.append([cr.quantize_weights_grouped(Ws, wl.G, codes) for _ in range(R)])
        biases.append(torch.from_numpy(b_np).to(dev))
        pxs.append([cr.empty_packed(wl.m, st.k, codes, dev) for _ in range(R)])
        Ys.append([torch.empty((wl.m, st.n), dtype=torch.float32, device=dev) for _ in range(R)])
        del Ws
    n_out = stages[-1].n
    # a stream of its own: the timed steps are captured into a CUDA graph on it
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    # MLP pair with --fused-pack: the down projection's pack fused into the up projection
    # (rotation and row absmax in its epilogue, then a light quantize launch)
    fused = bool(wl.down_n) and args.fused_pack
    if fused:
        works = [torch.empty((cr.linear_pack_work_bytes(wl.m, stages[0].n),), dtype=torch.uint8, device=dev)
                 for _ in range(R)]
    if wl.lora_r:  # runtime LoRA on the first linear: T from the unrotated X, one extra GEMM chunk
        A_l, B_l = inputs.lora_weights(wl)
        A_l = cr.convrot_lora_prepare_down(torch.from_numpy(A_l).to(dev))
        B_ext = cr.convrot_lora_prepare(torch.from_numpy(B_l).to(dev), wl.lora_scale)
        T_ext = [torch.empty((wl.m, cr.lora_cols(wl.lora_r)), dtype=torch.bfloat16, device=dev) for _ in range(R)]

    def step_ops(x_in, j):
        """One step as its kernel launches, in order: (tag, launch) pairs."""
        ops = []
        h = x_in
        for s_i, st in enumerate(stages):
            def pack(h=h, s_i=s_i):
                cr.convrot_pack_activations(h, wl.G, codes, out=pxs[s_i][j], stream=stream)
            if fused and s_i == 1:
                ops.append(("gemm", lambda s_i=s_i, st=st: cr.convrot_linear_act(
                    pxs[s_i][j], pws[s_i][j], biases[s_i], st.act, out=Ys[s_i][j], stream=stream)))
            elif fused and s_i == 0:
                ops.append(("pack", pack))
                ops.append(("gemm_pack", lambda st=st: cr.convrot_linear_act_pack(
                    pxs[0][j], pws[0][j], biases[0], st.act, wl.G, codes, out=pxs[1][j], work=works[j],
                    stream=stream)))
            elif wl.lora_r and s_i == 0:
                # T = X A^T first: the pack then finds X in L2 (it reads X with an evict-first
                # hint, so X would not wait in L2 for lora_down the other way round)
                ops.append(("lora_down", lambda h=h: cr.convrot_lora_down(h, A_l, out=T_ext[j], stream=stream)))
                ops.append(("pack", pack))
                ops.append(("gemm", lambda s_i=s_i, st=st: cr.convrot_linear_lora(
                    pxs[s_i][j], pws[s_i][j], biases[s_i], st.act, T_ext[j], B_ext, wl.lora_r, out=Ys[s_i][j],
                    stream=stream)))
            else:
                ops.append(("pack", pack))
                ops.append(("gemm", lambda s_i=s_i, st=st: cr.convrot_linear_act(
                    pxs[s_i][j], pws[s_i][j], biases[s_i], st.act, out=Ys[s_i][j], stream=stream)))
            h = Ys[s_i][j]
        return ops, h

    def run_stages(x_in, j):
        ops, y = step_ops(x_in, j)
        for _, launch in ops:
            launch()
        return y

    def step(i):
        run_stages(Xs[i % R], i % R)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    # The K timed steps as one CUDA graph: the same kernels on the same buffers,
    # launched without the host between them. Replayed once untimed so that the
    # graph's upload is not in the timed region.
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(args.steps):
                step(i)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            graph.replay()
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # The timed region holds no events between kernels: each one serialises the
    # stream (~2.4 us), so the per-kernel durations are measured apart (below).
    t_start.record(stream)
    if graph is not None:
        with torch.cuda.stream(stream):
            graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    total_ms = t_start.elapsed_time(t_end)
    # Per-kernel durations: each launch of the step repeated K times back to back
    # over the rotating sets (as one CUDA graph unless --eager), with an event
    # pair around the batch: its average launch duration, free of the stream
    # serialisation that an event between two kernels costs.
    kern_ms = {}
    n_ops = len(step_ops(Xs[0], 0)[0])
    for q in range(n_ops):
        tag = step_ops(Xs[0], 0)[0][q][0]

        def batch(q=q):
            for i in range(args.steps):
                step_ops(Xs[i % R], i % R)[0][q][1]()
        g = None
        if graph is not None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                batch()
            with torch.cuda.stream(stream):
                g.replay()
        else:
            batch()
        torch.cuda.synchronize(dev)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        if g is not None:
            with torch.cuda.stream(stream):
                g.replay()
        else:
            batch()
        b1.record(stream)
        torch.cuda.synchronize(dev)
        kern_ms[tag] = kern_ms.get(tag, 0.0) + b0.elapsed_time(b1) / args.steps
        if tag == "pack" and "pack_first" not in kern_ms:
            kern_ms["pack_first"] = b0.elapsed_time(b1) / args.steps
        del g
    # Context for the pack's roofline: torch's own elementwise conversion of the same
    # activations to the code type (the same bytes: 4 read and 1 or 2 written per
    # element), timed the same way. Not part of a step and not counted in gpu_launches.
    code_dtype = torch.int8 if codes == cr.CODES_I8 else torch.bfloat16
    conv_out = [torch.empty((wl.m, wl.k), dtype=code_dtype, device=dev) for _ in range(R)]

    def conv_batch():
        for i in range(args.steps):
            conv_out[i % R].copy_(Xs[i % R])
    def conv_run(g):
        with torch.cuda.stream(stream):
            if g is not None:
                g.replay()
            else:
                conv_batch()

    conv_run(None)
    g = None
    if graph is not None:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            conv_batch()
    conv_run(g)
    torch.cuda.synchronize(dev)
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    conv_run(g)
    b1.record(stream)
    torch.cuda.synchronize(dev)
    conv_ms = b0.elapsed_time(b1) / args.steps
    del g, conv_out
    # keep the GPU busy a little longer with the same steps for the clock record
    t_keep = time.time()
    i = 0
    while time.time() - t_keep < 1.0:
        step(i)
        i += 1
    torch.cuda.synchronize(dev)
    clk = clocks.stop()

    # end to end through the public API: every step copies its X from pinned host memory
    # and its Y back to pinned host memory. Steps are pipelined as a throughput user would:
    # step i's Y goes to the host on one copy stream while step i+1's X comes in on another
    # and step i+1 computes; two device and two host buffer sets alternate.
    e2e_steps = max(4, min(args.steps, 10))
    Xh = torch.from_numpy(inputs.activations(wl)).pin_memory()
    Yh = [torch.empty((wl.m, n_out), dtype=torch.float32).pin_memory() for _ in range(2)]
    Xd = [torch.empty_like(Xs[0]) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]   # compute of the set finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # its Y is on the host
    for e in ev_done + ev_out:
        e.record(stream)

    def e2e_step(i):
        j = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_done[j])          # the set's previous X is no longer read
            Xd[j].copy_(Xh, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])             # the set's previous Y has left for the host
        y = run_stages(Xd[j], j)
        ev_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[j])
            Yh[j].copy_(y, non_blocking=True)
            ev_out[j].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    for j in range(2):
        stream.wait_event(ev_out[j])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    ms_step, e2e_ms = slowest_rank([total_ms / args.steps, e2e_ms], pg, dev)

    ops = float(wl.step_ops)
    value = job_tops(world, ops, ms_step)
    gemm_avg = kern_ms["gemm"]
    pack_avg = kern_ms["pack"]
    fused_avg = kern_ms.get("gemm_pack")
    pk = peaks()
    gemm_tops = ops / (gemm_avg * 1e-3) / 1e12
    # algorithmic bytes of a pack: 4 B read + 1 B code written per element + 4 B scale per row
    # (the page's I8 codes); the bytes this launch actually stores (bf16 codes: 2 B) beside them
    # (fused MLP pair: only the activation pack is a pack launch; the hidden one is in gemm_pack)
    pack_stages = stages[:1] if fused else stages
    pack_bytes = sum(wl.m * (5 * st.k + 4) for st in pack_stages)
    stored_pack_bytes = sum(wl.m * (4 * st.k + code_b * st.k + 4) for st in pack_stages)
    if fused:  # the GEMM figure covers the down projection alone; the up one is inside gemm_pack
        gemm_tops = 2 * wl.m * stages[1].n * stages[1].k / (gemm_avg * 1e-3) / 1e12
    pack_gbs = pack_bytes / (pack_avg * 1e-3) / 1e9
    stored_pack_gbs = stored_pack_bytes / (pack_avg * 1e-3) / 1e9
    first_pack_bytes = wl.m * (5 * stages[0].k + 4)
    first_pack_ms = kern_ms["pack_first"]
    conv_gbs = wl.m * stages[0].k * (4 + code_b) / (conv_ms * 1e-3) / 1e9
    traffic = measured_traffic(wl.name, "i8" if codes == cr.CODES_I8 else "bf16")

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s8" if codes == cr.CODES_I8 else "bf16-coded s8",
        "data": "synthetic (seeded N(0,1) activations with 0.1% outlier channels x50, N(0,0.02^2) weights)",
        "config": {"workload": workload_name(wl), "global_batch": wl.m * world,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "codes": "i8" if codes == cr.CODES_I8 else "bf16",
                   "l2": f"{R} rotating input/output sets, {touched / 1e6:.2f} MB touched per step "
                         + ("(> L2)" if touched > L2_BYTES else
                            "(all sets fit in L2: L2-warm timing, a parity-size workload)"),
                   "launch": ("eager, one C-ABI call per kernel" if graph is None else
                              "the K timed steps replayed as one CUDA graph of the same C-ABI launches"),
                   "kernel_timing": "each launch of the step repeated K times back to back over the rotating "
                                    "sets, CUDA events around the batch (pack_ms, gemm_ms and the rooflines)"},
        "pack_gbs": pack_gbs, "pack_ms": pack_avg, "gemm_ms": gemm_avg, "gemm_tops": gemm_tops,
        **({"gemm_pack_ms": fused_avg,
            "fused": "up projection + GELU + the down projection's rotation and row absmax in one GEMM, then a "
                     "quantize launch (gemm_pack_ms, both); gemm_ms and gemm_tops: the down projection"}
           if fused else {}),
        **({"lora_down_ms": kern_ms["lora_down"],
            "lora": f"rank {wl.lora_r}, scale {wl.lora_scale:g}: T = X A^T in its own kernel (lora_down_ms), "
                    "the correction as an extra fp32 chunk of the GEMM (in gemm_ms); its own "
                    "multiply-adds are not counted in value"} if wl.lora_r else {}),
        "roofline": {"bound": "tensor", "achieved": gemm_tops, "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": gemm_tops / pk["bf16_tflops"], "traffic": traffic,
                     "kernel": "gemm", "peak_source": f"{pk['source']} dense bf16 burst",
                     **({"note": "I8 codes run the legacy mma.sync s8 kernel, whose own ceiling on this "
                                 "part is ~150 TOPS (a register-only microbenchmark); the bf16 peak is the "
                                 "denominator of the default bf16-code path"}
                        if codes == cr.CODES_I8 else {})},
        "roofline_pack": {"bound": "hbm", "achieved": pack_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                          "frac": pack_gbs / pk["hbm_gbs"], "bytes_per_launch": pack_bytes,
                          "bytes": "algorithmic: 4 B read + 1 B code per element, 4 B scale per row",
                          "peak_source": f"{pk['source']} copy bandwidth",
                          "stored": {"bytes_per_launch": stored_pack_bytes, "gbs": stored_pack_gbs,
                                     "frac": stored_pack_gbs / pk["hbm_gbs"],
                                     "what": f"the bytes the launch moves with {code_b}-byte codes"},
                          "same_bytes_conversion": {
                              "what": f"torch fp32 -> {str(code_dtype).replace('torch.', '')} copy_ of the "
                                      "same activations, timed like the pack (context, not a step kernel)",
                              "ms": conv_ms, "gbs": conv_gbs,
                              "pack_ms": first_pack_ms,
                              "pack_gbs": first_pack_bytes / (first_pack_ms * 1e-3) / 1e9}},
        "e2e": {"value": job_tops(world, ops, e2e_ms), "unit": "TOPS",
                "pipelining": "H2D of step i+1 and D2H of step i overlap compute on separate streams",
                "h2d_bytes_per_step": wl.m * wl.k * 4, "d2h_bytes_per_step": wl.m * n_out * 4,
                "ms_per_step": e2e_ms},
        # (fused MLP pair: pack, GEMM, quantize, GEMM; its cudaMemsetAsync is a runtime memset node)
        "gpu_launches": (2 * len(stages) + (1 if wl.lora_r else 0)) * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline and world == 1:
        cb = cpu_baseline(wl, args.cpu_seconds)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "pack_gbs",
                                                   "gemm_tops")}
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
