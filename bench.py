"""Benchmark: one 7B-shaped decode step of quantised projections on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--batch B]

A step is one pass of the whole hot path over one batch of synthetic input: for each of 32
layers and each projection {q|k|v Q4_K 6144x4096, o Q4_K 4096x4096, gate|up Q4_K 28672x4096,
down Q6_K 4096x14336}, the q8_K pack of that projection's activation and the mat-vec of its
weight.  By default one or two vectors run one launch per projection (qmd_qmatvec_x_ws, which
packs inside the kernel and hands the last rows of deep launches to warps as they free up) and
larger batches qmd_q8k_pack followed by qmd_qmatvec_ws (every CTA of a fused launch packs the
whole input for itself, which costs more than the extra launch once the input holds three or
more vectors); --fused and --unfused force one form everywhere.  Each launch depends on the
previous one in stream order, as in a real decode where a projection's input comes from the
layer before.  The step's launches are captured once into a CUDA graph and replayed.  Weights
(4.41 GB) exceed L2 many times over, so consecutive steps read them from HBM.

Throughput is quoted on algorithmic bytes: every weight byte, the f32 activations read and the
f32 outputs written, once per step (4.419 GB at batch 1).

Printed (rank 0, one JSON line): the step's algorithmic bytes / time as GB/s (value), the
same through host buffers (e2e: inputs copied in and outputs copied out every step), the
dominant kernel's roofline against the measured copy peak and the measured read-only ceiling,
the oracle's throughput on the host cores (cpu_baseline), SM clocks sampled during the timed
region, launch counts, (steps) the same step at batches 2, 4 and 8 over the same weights, and
(configs) each of configs 0-3 as a single mat-vec on packed input, timed apart from the step.

--impl reference times the CPU oracle on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs an independent replica of the step (replicas only; the
path needs no exchange); value is the bytes all ranks processed / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (% of GB300 peak) and rows/s for Q4_K/Q6_K×q8_K decode mat-vec"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.txt")
KERNEL_SOURCES = ["quantised_decode_mat_gb300/csrc/qmv.cuh", "quantised_decode_mat_gb300/csrc/qmv_rl.cuh",
                  "quantised_decode_mat_gb300/csrc/qmv_q4k.cu", "quantised_decode_mat_gb300/csrc/qmv_q6k.cu",
                  "quantised_decode_mat_gb300/csrc/ptx.cuh", "quantised_decode_mat_gb300/csrc/pack.cu",
                  "quantised_decode_mat_gb300/csrc/q8k.cuh"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    try:
        vals = {}
        with open(PROFILE_TRAFFIC) as f:
            for line in f:
                line = line.split("#", 1)[0].strip()
                if ":" in line:
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
        if vals.get("source_hash") != kernel_source_hash():
            return None
        v = vals.get(f"{kernel}_dram_bytes_per_launch")
        return float(v) if v else None
    except FileNotFoundError:
        return None


# ---- clocks sampled during the timed region ------------------------------------------------------
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.lines: list[str] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except FileNotFoundError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
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
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def alu_roofline(q, step, batch: int, ms_per_launch: float, dp4a_rate: float, mma_rate: float) -> dict:
    """The Q4_K mat-vec against the measured issue rate of the unit doing its multiply-adds:
    dp4a (64 per 256-value block-row per vector) on the dp4a kernel, or mma.sync (one
    m16n8k16, 4096 FLOP with the batch padded to 8, per block-row) on the tensor-core kernel."""
    q4 = [p for p in step.projs if p.fmt == q.Q4_K]
    block_rows = sum(p.rows * (p.K // 256) for p in q4) / len(q4)
    tc = q.launch_kernel(q.Q4_K, q4[0].rows, q4[0].K, batch) == "qmv_tc_kernel"
    if tc:
        ops, peak, unit, op = block_rows * 4096.0, mma_rate, "TFLOP/s", "mma.sync.m16n8k16 f16->f32"
    else:
        ops, peak, unit, op = block_rows * 64.0 * batch, dp4a_rate, "Tdp4a/s", "dp4a"
    achieved = ops / (ms_per_launch * 1e-3)
    return {"bound": "alu", "kernel": kernel_name(q, q.Q4_K, q4[0].rows, q4[0].K, batch), "op": op,
            "achieved": achieved / 1e12, "peak": peak / 1e12, "unit": unit, "frac": achieved / peak,
            "ops_per_launch": ops, "peak_kind": "measured (qmd_measure_alu, register-only kernels)"}


def gpu_uuid(torch, dev_index: int):
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---- distributed helpers (timing only: replicas exchange no data) ---------------------------------
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- the oracle on the host cores ------------------------------------------------------------------
def oracle_step_sample(layers, batch: int, row_fraction: float = 1.0, threads: int = 1, passes: int = 1):
    """Run the oracle (pack + mat-vec, its default sequential order) over the given layers of the
    decode step, the first row_fraction of each projection's rows, those rows split across
    `threads` host threads (the oracle is C called through ctypes, which releases the
    interpreter lock).  Inputs are generated before the clock starts; the work is timed `passes`
    times over.  Returns (wall seconds, algorithmic bytes, rows), summed over the passes."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle as O
    from quantised_decode_mat_gb300 import synth
    work = []
    for layer in layers:
        for t, (name, fmt, rows, K) in enumerate(synth.STEP_PROJECTIONS):
            r = max(1, int(rows * row_fraction))
            W = synth.weights(fmt, synth.step_seed(layer), rows, K, layer, t)[:r]
            x = synth.activations(synth.step_seed(layer), batch, K, layer, t)
            work.append((O.FMT_Q4_K if fmt == "q4k" else O.FMT_Q6_K, W, x, r, K))
    nbytes = sum(r * (K // 256) * (144 if f == O.FMT_Q4_K else 210) + batch * K * 4 + batch * r * 4
                 for (f, _, _, r, K) in work)  # weights + f32 activations + f32 outputs
    nrows = sum(r for (_, _, _, r, _) in work)
    with ThreadPoolExecutor(max(1, threads)) as ex:
        t0 = time.perf_counter()
        for (f, W, x, r, K) in work * max(1, passes):
            qs, xd, bs = O.q8k_pack(x)
            if threads <= 1:
                O.qmatvec(f, W, qs, xd, bs)
                continue
            cuts = [r * i // threads for i in range(threads + 1)]
            futs = [ex.submit(O.qmatvec, f, W[cuts[i]:cuts[i + 1]], qs, xd, bs)
                    for i in range(threads) if cuts[i + 1] > cuts[i]]
            for fu in futs:
                fu.result()
        secs = time.perf_counter() - t0
    return secs, nbytes * max(1, passes), nrows * max(1, passes)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from quantised_decode_mat_gb300 import synth
    import oracle
    oracle.build()
    layer_bytes = sum((rows * (K // 256) * (144 if f == "q4k" else 210)) for (_, f, rows, K) in synth.STEP_PROJECTIONS)
    # bound the whole run to about two minutes at the oracle's ~0.15 GB/s
    ncores = os.cpu_count() or 1
    # bound the whole run to about two minutes on the host cores
    budget_bytes = 18e9 * min(ncores, 8)
    frac = min(1.0, budget_bytes / max(1, args.steps + args.warmup) / layer_bytes)
    frac = max(frac, 1.0 / 4096)
    for i in range(args.warmup):
        oracle_step_sample([i % synth.STEP_LAYERS], args.batch, frac, ncores)
    tot_s = tot_b = 0.0
    for i in range(args.steps):
        s, b, _ = oracle_step_sample([i % synth.STEP_LAYERS], args.batch, frac, ncores)
        tot_s += s
        tot_b += b
    gbs = tot_b / tot_s / 1e9
    sample = (f"per step: the first {frac:.4%} of every projection's rows of one layer (layer = step index mod 32) "
              f"of the 32-layer step, batch {args.batch}; oracle pack + mat-vec, rows split over {ncores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 dot / f32 epilogue",
        "data": "synthetic", "config": workload_config(args),
        "cpu_baseline": {"value": gbs, "unit": UNIT, "cores": ncores, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": gbs, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def use_fused(args):
    """True / False when a flag forces one launch form everywhere; None for the per-projection
    default (quantised_decode_mat_gb300.step.fuse_pack)."""
    if getattr(args, "fused", False):
        return True
    if getattr(args, "unfused", False):
        return False
    return None


def launch_form(args) -> str:
    from quantised_decode_mat_gb300 import synth
    from quantised_decode_mat_gb300.step import fuse_pack
    f = use_fused(args)
    fused = [n for (n, _, _, K) in synth.STEP_PROJECTIONS if (fuse_pack(args.batch, K) if f is None else f)]
    if len(fused) == len(synth.STEP_PROJECTIONS):
        return "pack fused into the mat-vec (one kernel per projection)"
    if not fused:
        return "pack+mat-vec as two kernels"
    return f"pack fused into the mat-vec for {', '.join(fused)}; pack+mat-vec as two kernels for the rest"


def workload_config(args):
    from quantised_decode_mat_gb300 import synth
    layers = getattr(args, "layers", synth.STEP_LAYERS)
    return {"workload": f"decode_step_7b_q4k_q6k_{layers}layers_b{args.batch}",
            "launch": launch_form(args),
            "schedule": ("rows split evenly over the SMs" if getattr(args, "no_workspace", False) else
                         "rows split evenly, the last quarter of each 1-2 vector launch handed out to warps as "
                         "they free up (scheduling workspace)"),
            "layers": layers,
            "projections": [f"{n}:{f}:{r}x{k}" for (n, f, r, k) in synth.STEP_PROJECTIONS],
            "batch": args.batch,
            "l2": f"inputs larger than L2 ({layers * 0.1378:.2f} GB of weights streamed per step; no flush needed)",
            "parallelism": "replicas" if args.gpus > 1 else "single"}


# ---- our path ----------------------------------------------------------------------------------------
def time_graph(torch, g, reps: int, stream) -> float:
    """ms per replay of graph g, CUDA events on the replay stream."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def kernel_name(q, fmt: int, rows: int, K: int, batch: int) -> str:
    """The mat-vec kernel qmd_qmatvec runs for these sizes (qmd_qmatvec_launch_kernel)."""
    return q.launch_kernel(fmt, rows, K, batch)


def time_configs(torch, q, device, peak: float, peak_kind: str = "measured") -> dict:
    """Configs 0-3 as single mat-vecs on packed input (the batches each config names): a
    CUDA-graph chain of launches rotating over seeded weight copies that together exceed 3 x L2,
    so every launch reads its weights from HBM.  Bytes per launch as the workload tables count
    them: weights + q8_K blocks (276 B each) + f32 outputs."""
    from quantised_decode_mat_gb300 import synth
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    out = {}
    for cid in (0, 1, 2, 3):
        c = synth.CONFIGS[cid]
        rows, K, fmt = c["rows"], c["K"], c["fmt"]
        nb = K // 256
        g = torch.from_numpy(synth.weights(fmt, c["seed"], rows, K).reshape(rows, -1)).to(device)
        if fmt == "q6k":
            W, Wa = q.bind_q6k(g, rows, K)
            wbytes, f = rows * nb * 210, q.Q6_K_SPLIT
        else:
            W, Wa = g, None
            wbytes, f = rows * nb * 144, q.Q4_K
        ncopy = min(2000, max(2, -(-3 * l2 // wbytes)))
        copies = [(W.clone(), None if Wa is None else Wa.clone()) for _ in range(ncopy)]
        del g, W, Wa
        ws = q.workspace(device)  # every launch of a chain is ordered in one stream: one workspace
        for B in c["batches"]:
            xq = q.q8k_pack(torch.from_numpy(synth.activations(c["seed"], B, K)).to(device))
            y = torch.empty((B, rows), dtype=torch.float32, device=device)
            # the default plan; for the short one-vector configs also the split-K form at each
            # split count the rows allow (qmd_debug_set_split_k), so its cost is on record beside it
            splits = [0] + ([ks for ks in (2, 3, 4) if ks <= nb // 4] if cid in (0, 1) and B == 1 else [])
            for ks in splits:
                q.debug_set_split_k(ks)
                try:
                    s = torch.cuda.Stream(device)
                    s.wait_stream(torch.cuda.current_stream(device))
                    with torch.cuda.stream(s):
                        for (Wc, Ac) in copies:  # first launches set kernel attributes outside capture
                            q.qmatvec(f, Wc, Ac, xq, y, rows, s, workspace=ws)
                    torch.cuda.synchronize(device)
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr, stream=s):
                        for (Wc, Ac) in copies:
                            q.qmatvec(f, Wc, Ac, xq, y, rows, s, workspace=ws)
                    info = q.launch_info(f, rows, K, B)
                    kname = kernel_name(q, f, rows, K, B)
                finally:
                    q.debug_set_split_k(0)
                for _ in range(3):
                    gr.replay()
                ms = time_graph(torch, gr, 10, torch.cuda.current_stream(device)) / ncopy  # replays go there
                alg = wbytes + B * nb * 276 + B * rows * 4
                gbs = alg / (ms * 1e-3) / 1e9
                out[f"config{cid}_b{B}" + (f"_splitk{ks}" if ks else "")] = {
                    "shape": f"{fmt} {rows}x{K} batch {B}", "us_per_launch": ms * 1e3, "gbs": gbs,
                    "frac_of_peak": gbs / peak, "peak_kind": peak_kind, "frac_of_nominal_8TBps": gbs / NOMINAL_HBM_GBS,
                    "bytes_per_launch": alg, "weight_copies_rotated": ncopy, "kernel": kname,
                    "grid": info["grid"], "threads": info["threads"]}
                del gr
        del copies
        torch.cuda.empty_cache()
    q.get_device_error()
    return out


def time_step_at(torch, q, step, batch: int, steps: int, warmup: int, stream, peak: float) -> dict:
    """The decode step over the same weights at another batch: its own graph, timed like the
    headline step, plus its Q4_K mat-vecs as a chain (the roofline kernel at that batch)."""
    st = step.with_batch(batch)
    g = st.capture()
    for _ in range(warmup):
        g.replay()
    ms = time_graph(torch, g, steps, stream)
    nq4 = sum(1 for p in st.projs if p.fmt == q.Q4_K)
    g4 = st.capture(lambda: st.run_matvecs(q.Q4_K))
    g4.replay()
    ms4 = time_graph(torch, g4, max(3, steps), stream) / nq4
    per = lambda p: p.algorithmic_bytes() if p.fused else p.matvec_bytes()
    b4 = sum(per(p) for p in st.projs if p.fmt == q.Q4_K) / nq4
    nb = st.bytes()
    q.get_device_error()
    out = {"value": nb["algorithmic"] / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms, "steps": steps,
           "frac_of_peak": nb["algorithmic"] / (ms * 1e-3) / 1e9 / peak,
           "row_vectors_per_s": sum(p.rows for p in st.projs) * batch / (ms * 1e-3),
           "launch": "pack fused into the mat-vec" if all(p.fused for p in st.projs) else "pack+mat-vec",
           "q4k_kernel": kernel_name(q, q.Q4_K, st.projs[0].rows, st.projs[0].K, batch),
           "q4k_us_per_launch": ms4 * 1e3,
           "q4k_roofline_frac": b4 / (ms4 * 1e-3) / 1e9 / peak}
    del g, g4, st
    return out


def run_ours(args):
    import torch
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local_rank)
    if rank == 0:
        from quantised_decode_mat_gb300 import build as qbuild
        qbuild.build()
    barrier(world)
    import quantised_decode_mat_gb300 as q
    from quantised_decode_mat_gb300 import step as qstep
    q.lib()  # fails loudly if the CUDA library is missing

    step = qstep.make_step(args.batch, layers=args.layers, device=f"cuda:{local_rank}", fused=use_fused(args),
                           workspace=not getattr(args, "no_workspace", False))
    dp4a_rate, mma_rate = q.measure_alu()  # before the timed region
    nbytes = step.bytes()
    stream = torch.cuda.current_stream()

    g = step.capture()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_uuid(torch, local_rank))
    barrier(world)
    sampler.start()
    ms = time_graph(torch, g, args.steps, stream)
    clocks = sampler.stop()
    barrier(world)
    ms_max = max_over_ranks(ms, world)
    q.get_device_error()

    # the dominant kernel and the others, each timed as a graph of its launches in step order
    nq4 = sum(1 for p in step.projs if p.fmt == q.Q4_K)
    nq6 = len(step.projs) - nq4
    reps = max(3, min(args.steps, 200))
    g4 = step.capture(lambda: step.run_matvecs(q.Q4_K))
    g6 = step.capture(lambda: step.run_matvecs(q.Q6_K_SPLIT))
    gp = step.capture(step.run_packs)
    for gg in (g4, g6, gp):
        gg.replay()
    ms4 = time_graph(torch, g4, reps, stream) / nq4
    ms6 = time_graph(torch, g6, reps, stream) / nq6
    msp = time_graph(torch, gp, reps, stream) / len(step.projs)
    per = lambda p: p.algorithmic_bytes() if p.fused else p.matvec_bytes()
    q4_fused = all(p.fused for p in step.projs if p.fmt == q.Q4_K)
    b4 = sum(per(p) for p in step.projs if p.fmt == q.Q4_K) / nq4
    b6 = sum(per(p) for p in step.projs if p.fmt == q.Q6_K_SPLIT) / nq6
    bp = nbytes["pack"] / len(step.projs)

    # RMSNorm + residual + pack (qmd_rmsnorm_q8k_pack) on the inputs of q|k|v and gate|up (the two
    # projections that read a normalised residual stream in a decode step), a chain of launches
    rms = [p for p in step.projs if p.name in ("qkv", "gate_up")]
    gain = torch.full((4096,), 1.0, dtype=torch.float32, device=stream.device)
    resid = [torch.zeros_like(p.x) for p in rms]

    def run_rms():
        for p, r in zip(rms, resid):
            q.rmsnorm_q8k_pack(p.x, r, gain, 1e-6, h_out=r, out=p.xq)

    gr = step.capture(run_rms)
    gr.replay()
    msr = time_graph(torch, gr, reps, stream) / len(rms)
    br = sum(4 * p.x.numel() * 3 + 4 * 4096 + p.xq.batch * (4096 + 16 * 4 + 16 * 16) for p in rms) / len(rms)

    # the same normalised inputs feeding their mat-vecs: RMSNorm + pack, then the mat-vec (two
    # launches), against qmd_qmatvec_rmsnorm_x (one launch); h written to its own buffer in both
    hbuf = [torch.empty_like(p.x) for p in rms]

    def run_norm_two():
        for p, r, h in zip(rms, resid, hbuf):
            q.rmsnorm_q8k_pack(p.x, r, gain, 1e-6, h_out=h, out=p.xq)
            q.qmatvec(p.fmt, p.W, p.W_aux, p.xq, p.y, p.rows)

    def run_norm_one():
        for p, r, h in zip(rms, resid, hbuf):
            q.qmatvec_rmsnorm_x(p.fmt, p.W, p.W_aux, p.x, r, gain, 1e-6, h_out=h, y=p.y, rows=p.rows)

    gn2 = step.capture(run_norm_two)
    gn1 = step.capture(run_norm_one)
    gn2.replay()
    gn1.replay()
    msn2 = time_graph(torch, gn2, reps, stream) / len(rms)
    msn1 = time_graph(torch, gn1, reps, stream) / len(rms)
    bn = sum(p.weight_bytes + 4 * p.x.numel() * 3 + 4 * 4096 + 4 * p.xq.batch * p.rows for p in rms) / len(rms)

    # end to end: inputs from pinned host memory in, outputs to pinned host memory out, every step
    x_host = torch.empty(step.x_all.shape, dtype=step.x_all.dtype, pin_memory=True)
    y_host = torch.empty(step.y_all.shape, dtype=step.y_all.dtype, pin_memory=True)
    x_host.copy_(step.x_all)

    def e2e_step():
        step.run_through_host(x_host, y_host)

    ge = step.capture(e2e_step)
    for _ in range(max(1, args.warmup)):
        ge.replay()
    barrier(world)
    ms_e2e = max_over_ranks(time_graph(torch, ge, args.steps, stream), world)
    q.get_device_error()

    peak, peak_kind = measured_peak()
    gbs = world * nbytes["algorithmic"] / (ms_max * 1e-3) / 1e9
    # the read-only ceiling: bulk-copy streaming of a buffer 16 x the L2, measured here
    rbuf = torch.empty(16 * torch.cuda.get_device_properties(local_rank).L2_cache_size // 16 * 16,
                       dtype=torch.uint8, device=stream.device)
    read_gbs = q.measure_read_bw(rbuf) / 1e9
    del rbuf
    q.get_device_error()
    rows_per_step = sum(p.rows for p in step.projs)
    ach4 = b4 / (ms4 * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 dot / f32 epilogue", "data": "synthetic",
        "config": workload_config(args),
        "pct_of_peak": {"of_" + peak_kind: gbs / world / peak, "of_nominal_8TBps": gbs / world / NOMINAL_HBM_GBS,
                        "of_read_ceiling": gbs / world / read_gbs},
        "read_ceiling": {"value": read_gbs, "unit": "GB/s",
                         "how": "qmd_measure_read_bw: one CTA per SM streams a buffer of 16 x L2 into shared "
                                "memory with 1-D bulk copies and discards it; 5 passes after a warm-up"},
        "rows_per_s": world * rows_per_step / (ms_max * 1e-3),
        "row_vectors_per_s": world * rows_per_step * args.batch / (ms_max * 1e-3),
        "bytes_per_step": nbytes,
        "gbs_by_bytes": {"algorithmic": gbs,
                         "weights_only": world * nbytes["weights"] / (ms_max * 1e-3) / 1e9,
                         "matvec_only": world * nbytes["matvec"] / (ms_max * 1e-3) / 1e9,
                         "pack_inclusive": world * (nbytes["matvec"] + nbytes["pack"]) / (ms_max * 1e-3) / 1e9},
        "roofline": {"bound": "hbm",
                     "kernel": "%s<Q4_K, batch %d, %s>" % (kernel_name(q, q.Q4_K, 4096, 4096, args.batch),
                                                            args.batch,
                                                            "fused pack" if q4_fused else "packed input"),
                     "achieved": ach4, "peak": peak,
                     "unit": "GB/s", "frac": ach4 / peak, "peak_kind": peak_kind,
                     "frac_of_read_ceiling": ach4 / read_gbs, "frac_of_nominal_8TBps": ach4 / NOMINAL_HBM_GBS,
                     # the committed capture is of the batch-1 fused-pack launches only
                     "traffic": profiled_traffic("qmv_q4k") if args.batch == 1 and q4_fused else None,
                     "algorithmic_bytes_per_launch": b4, "ms_per_launch": ms4},
        "alu_roofline": alu_roofline(q, step, args.batch, ms4, dp4a_rate, mma_rate),
        "kernels": {
            "qmv_q4k": {"launches_per_step": nq4, "us_per_launch": ms4 * 1e3, "gbs": ach4},
            "qmv_q6k": {"launches_per_step": nq6, "us_per_launch": ms6 * 1e3, "gbs": b6 / (ms6 * 1e-3) / 1e9},
            "q8k_pack": {"launches_per_step": sum(1 for p in step.projs if not p.fused),
                         "us_per_launch": msp * 1e3, "gbs": bp / (msp * 1e-3) / 1e9,
                         "note": "stand-alone pack kernel, timed as a chain of its launches"},
            "rmsnorm_q8k_pack": {"launches_per_step": 0, "us_per_launch": msr * 1e3, "gbs": br / (msr * 1e-3) / 1e9,
                                 "note": "RMSNorm + residual add + pack of a 4096-wide input (x, residual in "
                                         "place, gain read; codes, scales, sums written), timed as a chain of "
                                         "its launches beside the step"},
            "qmv_rmsnorm": {"launches_per_step": 0, "us_per_launch": msn1 * 1e3, "gbs": bn / (msn1 * 1e-3) / 1e9,
                            "two_launch_us": msn2 * 1e3, "two_launch_gbs": bn / (msn2 * 1e-3) / 1e9,
                            "note": "residual add + RMSNorm + pack + mat-vec in one launch (qmd_qmatvec_rmsnorm_x) "
                                    "on the 4096-wide projections (q|k|v, gate|up), against RMSNorm-pack then "
                                    "mat-vec; bytes = weights + x, residual, h + gain + y; chains beside the step"},
        },
        "e2e": {"value": world * nbytes["algorithmic"] / (ms_e2e * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": step.x_all.numel() * 4, "d2h_bytes_per_step": step.y_all.numel() * 4,
                "ms_per_step": ms_e2e},
        "clocks": clocks,
        "gpu_launches": step.launches * args.steps,
    }
    del g, g4, g6, gp, ge, gr, gn1, gn2
    if rank == 0 and not args.no_batches:
        # the same step at the other batches the workload names (4) and the batched range's ends
        line["steps"] = {f"batch{b}": time_step_at(torch, q, step, b, min(args.steps, 20), 3, stream, peak)
                         for b in (2, 4, 8) if b != args.batch}
    if rank == 0 and not args.no_configs:
        line["configs"] = time_configs(torch, q, torch.device(f"cuda:{local_rank}"), peak, peak_kind)
    if rank == 0 and args.cpu_layers > 0:
        import oracle
        oracle.build()
        # about 10 s of CPU work each: 3 passes on one thread, 4 x the cores over all threads
        secs, ob, orows = oracle_step_sample(range(args.cpu_layers), args.batch, passes=3)
        ncores = os.cpu_count() or 1
        tsecs, tb, _ = oracle_step_sample(range(args.cpu_layers), args.batch, 1.0, ncores, passes=4)
        line["cpu_baseline"] = {"value": tb / tsecs / 1e9, "unit": UNIT, "cores": ncores, "kind": "oracle",
                                "sample": f"layers 0-{args.cpu_layers - 1} of 32, all four projections, batch "
                                          f"{args.batch}: oracle q8_K pack + mat-vec, rows split over {ncores} "
                                          f"threads, 4 passes, {tsecs:.1f} s wall",
                                "single_thread": {"value": ob / secs / 1e9, "cores": 1, "seconds": secs},
                                "cpu_model": cpu_model()}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--batch", type=int, default=1, choices=range(1, 9))
    ap.add_argument("--unfused", action="store_true",
                    help="run each projection as qmd_q8k_pack + qmd_qmatvec (two launches; the default above batch 1)")
    ap.add_argument("--fused", action="store_true",
                    help="run each projection as one qmd_qmatvec_x launch (the default at batch 1)")
    ap.add_argument("--layers", type=int, default=32,
                    help="decoder layers in the step (32 for the 7B-shaped step; fewer only for profiling "
                         "captures, which must stay small)")
    ap.add_argument("--no-workspace", action="store_true",
                    help="run the mat-vecs without a scheduling workspace (every row split evenly over the SMs)")
    ap.add_argument("--no-batches", action="store_true",
                    help="skip the step at batches 2, 4 and 8 reported beside the headline (steps)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config mat-vec timings (configs 0-3) reported beside the step")
    ap.add_argument("--cpu-layers", type=int, default=8,
                    help="layers of the step the oracle is timed on for cpu_baseline (0: skip)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
