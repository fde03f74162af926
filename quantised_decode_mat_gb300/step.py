"""A decode step of quantised projections, run through the C ABI and replayable as a CUDA graph.

Each projection is: q8_K pack of its f32 activation (qmd_q8k_pack), then the mat-vec of its
weight against the packed bytes (qmd_qmatvec).  A 7B-shaped decode step is 32 layers of
{q|k|v fused Q4_K 6144x4096, o Q4_K 4096x4096, gate|up fused Q4_K 28672x4096, down Q6_K
4096x14336} ("Language models on the device: the cajeta-llm kernels", §1 fused q|k|v and §3.3
fused gate|up launches).  Capturing the step's launches once and replaying them is the CUDA
form of the pages' deferred streams ("One kernel, any device", §1; "The scheduler: what runs
when, beside what", §3), which issue a whole decode step as one graph.

All activations of the step live in one device buffer and all outputs in another, so an
end-to-end step moves its inputs in with one host-to-device copy and its outputs out with one
device-to-host copy.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

from . import Q4_K, Q6_K_SPLIT, QMD_QK, Q8K, bind_q6k, q6k_prefix_stride, q8k_pack, qmatvec, qmatvec_x
from . import synth


@dataclass
class Projection:
    name: str
    layer: int
    fmt: int
    rows: int
    K: int
    W: "object"            # device uint8: Q4_K blocks or Q6_K bodies
    W_aux: "object"        # device Q6_K prefix or None
    x: "object"            # device f32 [B, K] (view into DecodeStep.x_all)
    xq: Q8K
    y: "object"            # device f32 [B, rows] (view into DecodeStep.y_all)
    weight_bytes: int
    fused: bool = True     # one launch that packs inside the mat-vec, or pack + mat-vec

    def act_bytes(self) -> int:
        """q8_K bytes the mat-vec reads: codes + scale (+ the eight sums for Q4_K) per block."""
        nb = self.K // QMD_QK
        per = 256 + 4 + (16 if self.fmt == Q4_K else 0)
        return self.xq.batch * nb * per

    def matvec_bytes(self) -> int:
        """Bytes the mat-vec kernel must read and write given packed activations."""
        return self.weight_bytes + self.act_bytes() + self.xq.batch * self.rows * 4

    def pack_bytes(self) -> int:
        """Bytes the stand-alone pack kernel reads and writes."""
        nb = self.K // QMD_QK
        B = self.xq.batch
        return B * self.K * 4 + B * (self.K + nb * 4 + nb * 16)

    def algorithmic_bytes(self) -> int:
        """What the projection must move whatever the kernel split: its weights, its f32
        activations and its f32 outputs (packed activations are an intermediate)."""
        B = self.xq.batch
        return self.weight_bytes + B * self.K * 4 + B * self.rows * 4


# Most vectors whose q8_K pack the default step fuses into the mat-vec.
FUSE_MAX_BATCH = 2


def fuse_pack(batch: int, K: int) -> bool:
    """Default launch form of a projection: one launch that packs inside the mat-vec
    (qmd_qmatvec_x) for one or two vectors (the row-lane kernel, whose CTAs pack with all their
    warps: the fused form was as fast as or faster than pack + mat-vec on every 7B shape, the
    14336-wide down projection included); the stand-alone pack followed by the mat-vec for more
    vectors, where every CTA of a fused launch would pack the whole batch for itself after the
    dependency wait (67 / 95 / 109 against 45 / 80 / 92 us per layer at 2 / 4 / 8 vectors on the
    older kernels)."""
    return batch <= FUSE_MAX_BATCH


@dataclass
class DecodeStep:
    batch: int
    projs: list = field(default_factory=list)
    x_all: "object" = None
    y_all: "object" = None
    host_weights: dict = field(default_factory=dict)  # (layer, name) -> canonical GGUF bytes, if kept
    ws: "object" = None    # the scheduling workspace every mat-vec of the step uses (one stream), or None

    @property
    def form(self) -> str:
        """'fused' (every projection one launch), 'two-kernel' (pack + mat-vec everywhere) or
        'mixed'."""
        f = {p.fused for p in self.projs}
        return "fused" if f == {True} else "two-kernel" if f == {False} else "mixed"

    def run(self, stream=None) -> None:
        for p in self.projs:
            if p.fused:
                qmatvec_x(p.fmt, p.W, p.W_aux, p.x, p.y, p.rows, stream=stream, workspace=self.ws)
            else:
                q8k_pack(p.x, p.xq, stream)
                qmatvec(p.fmt, p.W, p.W_aux, p.xq, p.y, p.rows, stream, workspace=self.ws)

    def run_matvecs(self, fmt: int | None = None, stream=None) -> int:
        """The step's mat-vec launches only (fused form: each packs its own activations)."""
        n = 0
        for p in self.projs:
            if fmt is None or p.fmt == fmt:
                if p.fused:
                    qmatvec_x(p.fmt, p.W, p.W_aux, p.x, p.y, p.rows, stream=stream, workspace=self.ws)
                else:
                    qmatvec(p.fmt, p.W, p.W_aux, p.xq, p.y, p.rows, stream, workspace=self.ws)
                n += 1
        return n

    def run_through_host(self, x_host, y_host, chunks: int = 16, in_chunks: int = 1) -> None:
        """One step with its inputs copied in from pinned host memory (x_host, shaped like
        x_all) and its outputs copied out (y_host, shaped like y_all), the copies overlapped
        with the mat-vecs on two side streams: layer 0's inputs first, then the other layers' in
        `in_chunks` groups (the first layer of each group waits for its group's copy); the outputs
        in `chunks` groups of layers, each as soon as its group has run.  The current stream
        waits for every copy before it continues.  (Measured on the 32-layer step at batch 1:
        4, 8, 16, 32 output groups 4455, 4493, 4495, 4488 GB/s; input groups beyond layer 0's
        each add a wait to the launch chain: 4 groups 4427, 8 groups 4357.)"""
        import torch
        cur = torch.cuda.current_stream()
        if not hasattr(self, "_copy_streams"):
            self._copy_streams = (torch.cuda.Stream(), torch.cuda.Stream())
        h2d, d2h = self._copy_streams
        layers = sorted({p.layer for p in self.projs})
        span = {l: [p for p in self.projs if p.layer == l] for l in layers}

        def x_range(ls):
            ps = [p for l in ls for p in span[l]]
            lo = ps[0].x.data_ptr() - self.x_all.data_ptr()
            hi = ps[-1].x.data_ptr() + ps[-1].x.numel() * 4 - self.x_all.data_ptr()
            return lo // 4, hi // 4

        def y_range(ls):
            ps = [p for l in ls for p in span[l]]
            lo = ps[0].y.data_ptr() - self.y_all.data_ptr()
            hi = ps[-1].y.data_ptr() + ps[-1].y.numel() * 4 - self.y_all.data_ptr()
            return lo // 4, hi // 4

        h2d.wait_stream(cur)
        d2h.wait_stream(cur)
        n = len(layers)
        rest = layers[1:]
        m = len(rest)
        in_groups = [layers[:1]] + [g for g in (rest[k * m // in_chunks:(k + 1) * m // in_chunks]
                                                for k in range(max(1, in_chunks))) if g]
        x_ready = {}  # the first layer of each input group -> its copy's event
        with torch.cuda.stream(h2d):
            for ls in in_groups:
                a, b = x_range(ls)
                self.x_all[a:b].copy_(x_host[a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(h2d)
                x_ready[ls[0]] = e
        groups = [g for g in (layers[k * n // chunks:(k + 1) * n // chunks] for k in range(chunks)) if g]
        for i, l in enumerate(layers):
            if l in x_ready:
                cur.wait_event(x_ready[l])
            for p in span[l]:
                if p.fused:
                    qmatvec_x(p.fmt, p.W, p.W_aux, p.x, p.y, p.rows, stream=cur, workspace=self.ws)
                else:
                    q8k_pack(p.x, p.xq, cur)
                    qmatvec(p.fmt, p.W, p.W_aux, p.xq, p.y, p.rows, cur, workspace=self.ws)
            for g in groups:
                if g[-1] == l:
                    done = torch.cuda.Event()
                    done.record(cur)
                    d2h.wait_event(done)
                    a, b = y_range(g)
                    if g is groups[-1]:
                        b = self.y_all.numel()  # through the last output's padding
                    with torch.cuda.stream(d2h):
                        y_host[a:b].copy_(self.y_all[a:b], non_blocking=True)
        cur.wait_stream(h2d)
        cur.wait_stream(d2h)

    def with_batch(self, batch: int, fused: bool | None = None, workspace: bool = True) -> "DecodeStep":
        """The same step (the same weight tensors, shared) for `batch` activation vectors: new
        activations from the same seeds, new outputs and packed buffers, the launch forms
        fuse_pack picks for that batch (or `fused`), and its own scheduling workspace."""
        import torch
        from . import workspace as new_workspace
        dev = self.x_all.device
        names = [n for (n, _, _, _) in synth.STEP_PROJECTIONS]
        st = DecodeStep(batch=batch)
        st.ws = new_workspace(dev) if workspace else None
        st.x_all = torch.empty(sum(batch * p.K for p in self.projs), dtype=torch.float32, device=dev)
        st.y_all = torch.empty(sum((batch * p.rows + 3) // 4 * 4 for p in self.projs), dtype=torch.float32,
                               device=dev)
        xo = yo = 0
        for p in self.projs:
            x = st.x_all[xo: xo + batch * p.K].view(batch, p.K)
            x.copy_(torch.from_numpy(synth.activations(synth.step_seed(p.layer), batch, p.K, p.layer,
                                                       names.index(p.name))))
            xo += batch * p.K
            y = st.y_all[yo: yo + batch * p.rows].view(batch, p.rows)
            yo += (batch * p.rows + 3) // 4 * 4
            st.projs.append(Projection(p.name, p.layer, p.fmt, p.rows, p.K, p.W, p.W_aux, x,
                                       Q8K.empty(batch, p.K, dev), y, p.weight_bytes,
                                       fuse_pack(batch, p.K) if fused is None else bool(fused)))
        torch.cuda.synchronize(dev)
        return st

    def run_packs(self, stream=None) -> int:
        for p in self.projs:
            q8k_pack(p.x, p.xq, stream)
        return len(self.projs)

    def capture(self, fn=None):
        """Capture fn() (default: the whole step) into a CUDA graph on a side stream."""
        import torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            (fn or self.run)()  # warm: first launches set kernel attributes outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            (fn or self.run)()
        torch.cuda.synchronize()
        return g

    @property
    def launches(self) -> int:
        return sum(1 if p.fused else 2 for p in self.projs)

    def bytes(self) -> dict:
        """algorithmic: weights + f32 activations + f32 outputs of every projection (the
        figure the throughput is quoted on); matvec/pack: what the two-kernel form moves."""
        mv = sum(p.matvec_bytes() for p in self.projs)
        pk = sum(p.pack_bytes() for p in self.projs)
        w = sum(p.weight_bytes for p in self.projs)
        alg = sum(p.algorithmic_bytes() for p in self.projs)
        return dict(algorithmic=alg, matvec=mv, pack=pk, weights=w)


def _gen_layer(layer: int, projections, batch: int, seed_fn):
    out = []
    for t, (name, fmt, rows, K) in enumerate(projections):
        seed = seed_fn(layer)
        W = synth.weights(fmt, seed, rows, K, layer, t)
        x = synth.activations(seed, batch, K, layer, t)
        out.append((name, fmt, rows, K, W, x))
    return out


def make_step(batch: int, layers: int = synth.STEP_LAYERS, projections=synth.STEP_PROJECTIONS,
              device="cuda", seed_fn=synth.step_seed, keep_host_layers=(), threads: int = 8,
              fused: bool | None = None, workspace: bool = True) -> DecodeStep:
    """Generate the seeded weights and activations of a decode step and place them on the device.

    keep_host_layers: layers whose canonical GGUF weight bytes stay in host memory (for the
    oracle).  Q6_K weights are bound (split) on the device.  fused: True for one launch per
    projection (qmd_qmatvec_x), False for pack + mat-vec, None for the faster of the two per
    projection (fuse_pack).  workspace: the mat-vecs share one scheduling workspace (the step
    runs in one stream), which hands the last rows of each launch to warps as they free up."""
    import torch
    from . import workspace as new_workspace
    dev = torch.device(device)
    step = DecodeStep(batch=batch)
    step.ws = new_workspace(dev) if workspace else None
    x_sizes = [batch * K for (_, _, _, K) in projections] * layers
    y_sizes = [(batch * rows + 3) // 4 * 4 for (_, _, rows, _) in projections] * layers
    step.x_all = torch.empty(sum(x_sizes), dtype=torch.float32, device=dev)
    step.y_all = torch.empty(sum(y_sizes), dtype=torch.float32, device=dev)
    xo = yo = 0
    with ThreadPoolExecutor(max(1, threads)) as ex:
        futs = [ex.submit(_gen_layer, l, projections, batch, seed_fn) for l in range(layers)]
        for l, fut in enumerate(futs):
            for (name, fmt, rows, K, Wh, xh) in fut.result():
                nb = K // QMD_QK
                x = step.x_all[xo: xo + batch * K].view(batch, K)
                x.copy_(torch.from_numpy(xh))
                xo += batch * K
                y = step.y_all[yo: yo + batch * rows].view(batch, rows)
                yo += (batch * rows + 3) // 4 * 4
                if fmt == "q4k":
                    W = torch.from_numpy(Wh.reshape(rows, -1)).to(dev)
                    Wa = None
                    wbytes = rows * nb * 144
                    qfmt = Q4_K
                else:
                    g = torch.from_numpy(Wh.reshape(rows, -1)).to(dev)
                    W, Wa = bind_q6k(g, rows, K)
                    del g
                    wbytes = rows * nb * 208 + rows * q6k_prefix_stride(K) * 2
                    qfmt = Q6_K_SPLIT
                if l in keep_host_layers:
                    step.host_weights[(l, name)] = Wh
                step.projs.append(Projection(name, l, qfmt, rows, K, W, Wa, x, Q8K.empty(batch, K, dev), y,
                                             wbytes, fuse_pack(batch, K) if fused is None else bool(fused)))
    torch.cuda.synchronize(dev)
    return step


def host_activation(step: DecodeStep, p: Projection) -> np.ndarray:
    """The activation a projection was given (regenerated on the host from its seed)."""
    names = [n for (n, _, _, _) in synth.STEP_PROJECTIONS]
    return synth.activations(synth.step_seed(p.layer), step.batch, p.K, p.layer, names.index(p.name))
