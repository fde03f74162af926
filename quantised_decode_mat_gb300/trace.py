"""Per-phase breakdown of a decode step, from the traced build's per-CTA time stamps.

    python -m quantised_decode_mat_gb300.trace [--layers 8] [--batch 1] [--reps 5] [--fused|--unfused]

Builds libqmd_trace.so (the same kernels compiled with -DQMD_TRACE, include/qmd_trace.h), makes
the decode step of `--layers` layers as bench.py does, captures it as a CUDA graph with every
launch recording its CTAs' global-timer stamps, replays it, and prints for each projection
(median over its layers) where a launch's time goes on the critical path:

  period    this launch's last CTA exit minus the previous launch's last CTA exit
  release   previous launch's last exit -> the first of this launch's CTAs released by the
            dependency wait (the programmatic-launch hand-off)
  spread    first -> median CTA released (CTAs that start late, e.g. waiting for an SM to free)
  acts      median over CTAs of: wait released -> activations ready (the fused pack, or the
            packed activations' scales and sums read)
  first     median over CTAs of: activations ready -> first weight stage landed (0 when it had
            landed already)
  stream    median over CTAs of: first stage landed -> the CTA's last rows written
  tail      median CTA exit -> last CTA exit (imbalance at the end)
and, per CTA, launch entry -> first weight copies requested (`issue`) and entry relative to the
previous launch's last exit (`entry`, negative when the CTA became resident before the previous
launch ended).  Times in microseconds.  The numbers come from a traced build: each CTA stores a
few stamps, so they are close to, but not exactly, the product library's.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import statistics
import sys


def _median(v):
    return statistics.median(v) if v else float("nan")


def analyse(rec, launches, names):
    """rec: uint64 [n][8] stamp records; launches: [(first, ctas)]; names: launch labels."""
    out = []
    prev_end = None
    for (first, ctas), name in zip(launches, names):
        rows = [rec[first + i] for i in range(ctas)]
        rows = [r for r in rows if int(r[7]) != 0 and int(r[0]) != 0]
        if not rows:
            out.append({"name": name, "ctas": 0})
            continue
        e0 = [int(r[0]) for r in rows]
        rel = [int(r[2]) for r in rows]
        ex = [int(r[6]) for r in rows]
        end = max(ex)
        kind = int(rows[0][7]) >> 48
        d = {"name": name, "kind": {1: "fused", 2: "packed", 3: "pack"}.get(kind, str(kind)), "ctas": len(rows)}
        if prev_end is not None:
            d["period"] = (end - prev_end) / 1e3
            d["release"] = (min(rel) - prev_end) / 1e3
            d["entry"] = (_median(e0) - prev_end) / 1e3
        d["spread"] = (_median(rel) - min(rel)) / 1e3
        d["tail"] = (end - _median(ex)) / 1e3
        if kind != 3:
            d["issue"] = _median([int(r[1]) - int(r[0]) for r in rows]) / 1e3
            d["acts"] = _median([int(r[3]) - int(r[2]) for r in rows]) / 1e3
            d["first"] = _median([max(0, int(r[4]) - int(r[3])) for r in rows]) / 1e3
            d["stream"] = _median([int(r[5]) - max(int(r[4]), int(r[3])) for r in rows]) / 1e3
        else:
            d["work"] = _median([int(r[6]) - int(r[2]) for r in rows]) / 1e3
        out.append(d)
        prev_end = end
    return out


def summarise(per_launch):
    """Median of each field over the launches with the same label."""
    by = {}
    for d in per_launch:
        by.setdefault(d["name"], []).append(d)
    out = {}
    for name, ds in by.items():
        keys = [k for k in ds[-1] if k not in ("name", "kind")]
        out[name] = {"kind": ds[-1].get("kind"), "launches": len(ds)}
        for k in keys:
            vals = [d[k] for d in ds if k in d]
            out[name][k] = round(_median(vals), 3) if vals else None
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--fused", action="store_true")
    ap.add_argument("--unfused", action="store_true")
    ap.add_argument("--json", action="store_true", help="print the per-launch records as JSON too")
    ap.add_argument("--flags", type=int, default=0,
                    help="qmd_debug_set_launch_flags value for the captured step (e.g. 4: batches of 3..8 "
                         "on the tensor-core kernel wherever it fits)")
    ap.add_argument("--detail", default=None,
                    help="a projection name: print one of its launches CTA by CTA (SM id, times from the "
                         "previous launch's last exit)")
    args = ap.parse_args(argv)

    import numpy as np
    import torch

    from . import build as qbuild
    import quantised_decode_mat_gb300 as q
    from . import step as qstep

    L = q.lib(qbuild.build(trace=True))
    if not hasattr(L, "qmd_debug_trace"):
        raise RuntimeError("the loaded library is not the traced build")
    fused = True if args.fused else False if args.unfused else None
    step = qstep.make_step(args.batch, layers=args.layers, fused=fused)
    n_rec = 1 << 16
    buf = torch.zeros(n_rec * 8, dtype=torch.int64, device="cuda")

    # warm (kernel attributes are set outside the capture), then capture with recording on
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    q.debug_set_launch_flags(args.flags)
    try:
        with torch.cuda.stream(s):
            step.run()
        torch.cuda.synchronize()
        q._check(L.qmd_debug_trace(buf.data_ptr(), n_rec))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step.run()
    finally:
        q.debug_set_launch_flags(0)
    n = L.qmd_debug_trace_launches(None, None, 0)
    first = (ctypes.c_int64 * n)()
    ctas = (ctypes.c_int32 * n)()
    L.qmd_debug_trace_launches(first, ctas, n)
    q._check(L.qmd_debug_trace(None, 0))
    for _ in range(max(1, args.reps)):
        buf.zero_()
        g.replay()
    torch.cuda.synchronize()
    q.get_device_error()
    rec = buf.view(n_rec, 8).cpu().numpy().view(np.uint64)

    names = []
    for p in step.projs:
        if not p.fused:
            names.append(p.name + ":pack")
        names.append(p.name)
    if len(names) != n:
        raise RuntimeError(f"{n} launches recorded, {len(names)} expected")
    per = analyse(rec, list(zip(first, ctas)), names)
    per = per[len(names) // args.layers:]  # drop the first layer (its first launch has no predecessor in the graph)
    summ = summarise(per)
    periods = [d["period"] for d in per if "period" in d]
    print(json.dumps({"workload": f"decode step, {args.layers} layers, batch {args.batch}, form {step.form}, launch flags {args.flags}",
                      "reps": args.reps, "per_projection_us": summ,
                      "layer_us": round(sum(periods) / (args.layers - 1), 3)}, indent=1))
    if args.json:
        print(json.dumps(per))
    if args.detail:
        k = [i for i, nm in enumerate(names) if nm == args.detail][1]  # its launch in layer 1
        pf, pc = first[k - 1], ctas[k - 1]
        prev_end = max(int(rec[pf + j][6]) for j in range(pc) if int(rec[pf + j][7]) != 0)
        rows = sorted((int(rec[first[k] + j][7]) & 0xffff, j) for j in range(ctas[k]) if int(rec[first[k] + j][7]) != 0)
        print(f"launch {k} ({args.detail}): per CTA, microseconds after the previous launch's last exit")
        print("  sm  cta   entry  release   acts  first   last   exit")
        for sm, j in rows:
            r = [int(v) for v in rec[first[k] + j]]
            f = lambda i: (r[i] - prev_end) / 1e3 if r[i] else float("nan")
            print(f"  {sm:3d} {j:4d} {f(0):7.2f} {f(2):7.2f} {f(3):7.2f} {f(4):6.2f} {f(5):7.2f} {f(6):7.2f}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
