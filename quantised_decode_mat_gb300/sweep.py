"""Launch-plan sweep of one projection of the decode step, or of the whole step under launch flags.

    python -m quantised_decode_mat_gb300.sweep [--projection down] [--batch 1] [--layers 8]
        [--warps 8,12,16] [--stages 1,2,3,4] [--pre 1,2,3] [--reps 20]
    python -m quantised_decode_mat_gb300.sweep --step-flags 0,32 [--batch 1] [--layers 32]
    python -m quantised_decode_mat_gb300.sweep --in-step --projection down [--layers 32] [grid as above]
    python -m quantised_decode_mat_gb300.sweep --projection o --split-k 2,3,4 --warps "" [--in-step]

Makes the decode step of `--layers` layers as bench.py does and, for the default plan and then
every forced plan of the grid (qmd_debug_set_plan: ring warps per CTA, ring slots per warp, and
slots requested before the dependency wait -- the row-lane kernel's parameters), captures the
chosen projection's launches over all layers, in the step's launch form, as one CUDA graph and
times its replays with CUDA events on the replay stream.  Prints one markdown row per plan: µs
per launch and GB/s over the algorithmic bytes (weights + f32 x + f32 y), with the plan the
library actually used (a forced depth that does not fit is cut to the deepest that does).
Every forced plan's outputs are compared with the default plan's, bit for bit.

With --step-flags, the whole step (every projection, in the step's launch forms) is captured
once per value of qmd_debug_set_launch_flags and the graphs are timed in turn, three rounds
interleaved, 200 replays each; printed as GB/s over the step's algorithmic bytes.  With
--in-step, the grid of plans is applied to the chosen projection's launches only, inside the
whole step (a plan is fixed when a launch is captured, so the other projections keep their
default plans), each plan's step timed the same way.  --split-k adds the split-K form at each
of the given cluster sizes (qmd_debug_set_split_k), with each --pre value as its slots requested
before the dependency wait, to either mode.
"""
from __future__ import annotations

import argparse
import itertools
import sys


def _ints(s: str) -> list[int]:
    return [int(v) for v in s.split(",") if v.strip()]


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--projection", default="down", choices=["qkv", "o", "gate_up", "down"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--warps", default="8,12,16")
    ap.add_argument("--stages", default="1,2,3,4")
    ap.add_argument("--pre", default="1,2,3")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--step-flags", default=None, help="time the whole step under each of these launch-flag values")
    ap.add_argument("--in-step", action="store_true", help="force the plans on one projection inside the whole step")
    ap.add_argument("--split-k", default="", help="also the split-K form at these CTAs per cluster")
    args = ap.parse_args(argv)

    import torch
    from . import (debug_set_launch_flags, debug_set_plan, debug_set_split_k, get_device_error, launch_info, lib,
                   q8k_pack, qmatvec, qmatvec_x)
    from .step import make_step

    lib()
    st = make_step(args.batch, layers=args.layers)
    if args.step_flags is not None:
        nbytes = st.bytes()["algorithmic"]
        graphs = {}
        try:
            for fl in _ints(args.step_flags):
                debug_set_launch_flags(fl)
                graphs[fl] = st.capture()
        finally:
            debug_set_launch_flags(0)
        res = {fl: [] for fl in graphs}
        stream = torch.cuda.current_stream()
        for _ in range(3):
            for fl, g in graphs.items():
                for _ in range(5):
                    g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                for _ in range(200):
                    g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                res[fl].append(nbytes / (e0.elapsed_time(e1) / 200 * 1e-3) / 1e9)
        get_device_error()
        print(f"{args.layers}-layer step, batch {args.batch}, {nbytes / 1e9:.3f} GB a step")
        print()
        print("| launch flags | GB/s, three rounds |")
        print("|---|---|")
        for fl, v in res.items():
            print(f"| {fl} | " + ", ".join(f"{x:.0f}" for x in v) + " |")
        return 0
    if args.in_step:
        return _in_step(args, st, torch)
    ps = [p for p in st.projs if p.name == args.projection]
    alg = sum(p.algorithmic_bytes() for p in ps) / len(ps)

    def run():
        for p in ps:
            if p.fused:
                qmatvec_x(p.fmt, p.W, p.W_aux, p.x, p.y, p.rows, workspace=st.ws)
            else:
                q8k_pack(p.x, p.xq)
                qmatvec(p.fmt, p.W, p.W_aux, p.xq, p.y, p.rows, workspace=st.ws)

    def time_plan():
        g = st.capture(run)
        stream = torch.cuda.current_stream()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        get_device_error()
        del g
        return e0.elapsed_time(e1) * 1e3 / args.reps / len(ps)

    p0 = ps[0]
    info = launch_info(p0.fmt, p0.rows, p0.K, args.batch)
    us = time_plan()
    ref = torch.cat([p.y.reshape(-1) for p in ps]).clone()
    print(f"{args.projection}: {p0.rows} x {p0.K}, batch {args.batch}, {len(ps)} layers, "
          f"{'fused pack' if p0.fused else 'pack + mat-vec'}, {alg / 1e6:.2f} MB a launch")
    print()
    print("| plan (warps, slots, before wait) | used: grid x threads, slots | µs / launch | GB/s |")
    print("|---|---|---:|---:|")
    print(f"| default | {info['grid']} x {info['threads']}, {info['stages']} | {us:.2f} | {alg / us / 1e3:.0f} |")
    rows = []
    grid = [(0, w, s, pre) for w, s, pre in itertools.product(_ints(args.warps), _ints(args.stages), _ints(args.pre))
            if pre <= s]
    grid += [(ks, 0, 0, pre) for ks, pre in itertools.product(_ints(args.split_k), _ints(args.pre))]
    try:
        for ks, w, s, pre in grid:
            debug_set_split_k(ks)
            debug_set_plan(w, pre, s, 0)
            info = launch_info(p0.fmt, p0.rows, p0.K, args.batch)
            us = time_plan()
            same = torch.equal(torch.cat([p.y.reshape(-1) for p in ps]).view(torch.int32), ref.view(torch.int32))
            rows.append((us, w, s, pre))
            name = f"split-K {ks}, {info['stages']}, {pre}" if ks else f"{w}, {s}, {pre}"
            print(f"| {name} | {info['grid']} x {info['threads']}, {info['stages']} | {us:.2f} | "
                  f"{alg / us / 1e3:.0f} |" + ("" if same else " OUTPUTS DIFFER"), flush=True)
            if not same:
                return 1
    finally:
        debug_set_plan()
        debug_set_split_k(0)
    if rows:
        best = min(rows)
        print(f"\nfastest forced plan: {best[1]} warps, {best[2]} slots, {best[3]} before the wait: {best[0]:.2f} µs")
    return 0


def _launch(p, ws):
    from . import q8k_pack, qmatvec, qmatvec_x
    if p.fused:
        qmatvec_x(p.fmt, p.W, p.W_aux, p.x, p.y, p.rows, workspace=ws)
    else:
        q8k_pack(p.x, p.xq)
        qmatvec(p.fmt, p.W, p.W_aux, p.xq, p.y, p.rows, workspace=ws)


def _in_step(args, st, torch) -> int:
    """The whole step with the grid's plans forced on one projection's launches only."""
    from . import debug_set_plan, debug_set_split_k, get_device_error, launch_info
    nbytes = st.bytes()["algorithmic"]
    p0 = [p for p in st.projs if p.name == args.projection][0]
    # (ring warps, slots before the wait, ring slots, split-K CTAs per cluster)
    plans = [None] + [(w, pre, s, 0) for w, s, pre in itertools.product(_ints(args.warps), _ints(args.stages),
                                                                         _ints(args.pre)) if pre <= s]
    plans += [(0, pre, 0, ks) for ks, pre in itertools.product(_ints(args.split_k), _ints(args.pre))]

    def force(plan):
        if plan is None:
            debug_set_plan()
            debug_set_split_k(0)
        else:
            debug_set_plan(plan[0], plan[1], plan[2], 0)
            debug_set_split_k(plan[3])

    def capture(plan):
        def run():
            try:
                for p in st.projs:
                    force(plan if p.name == args.projection else None)
                    _launch(p, st.ws)
            finally:
                force(None)
        return st.capture(run)

    graphs, used = {}, {}
    for plan in plans:
        force(plan)
        info = launch_info(p0.fmt, p0.rows, p0.K, args.batch)
        force(None)
        used[plan] = f"{info['grid']} x {info['threads']}, {info['stages']}"
        graphs[plan] = capture(plan)
    res = {plan: [] for plan in plans}
    stream = torch.cuda.current_stream()
    for _ in range(3):
        for plan, g in graphs.items():
            for _ in range(5):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(100):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            res[plan].append(nbytes / (e0.elapsed_time(e1) / 100 * 1e-3) / 1e9)
    get_device_error()
    print(f"{args.layers}-layer step, batch {args.batch}, plans forced on {args.projection} only "
          f"({p0.rows} x {p0.K}), {nbytes / 1e9:.3f} GB a step")
    print()
    print("| plan on it (warps, slots, before wait) | used: grid x threads, slots | step GB/s, three rounds |")
    print("|---|---|---|")
    for plan in plans:
        name = ("default" if plan is None else f"split-K {plan[3]}, -, {plan[1]}" if plan[3]
                else f"{plan[0]}, {plan[2]}, {plan[1]}")
        print(f"| {name} | {used[plan]} | " + ", ".join(f"{x:.0f}" for x in res[plan]) + " |")
    return 0


if __name__ == "__main__":
    sys.exit(main())
