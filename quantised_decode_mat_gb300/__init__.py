"""Thin Python binding of libqmd (ctypes): decode-time Q4_K / Q6_K x q8_K mat-vec on GB300.

Argument marshalling only.  Every step of the computation runs in the library's CUDA kernels;
torch supplies device memory and streams.  The functions here carry the C ABI's names
(qmd_q8k_pack -> q8k_pack, qmd_qmatvec -> qmatvec, ...) and raise QmdError on any status
other than QMD_OK.  There is no CPU path: if libqmd.so is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqmd.so")

QMD_QK = 256
QMD_MAX_BATCH = 8
QMD_WORKSPACE_BYTES = 4096
Q4_K = 12
Q5_K = 13
Q6_K_SPLIT = 14

STATUS = {
    0: "QMD_OK",
    1: "QMD_ERR_NULL",
    2: "QMD_ERR_FORMAT",
    3: "QMD_ERR_K_NOT_MULTIPLE_OF_256",
    4: "QMD_ERR_BATCH",
    5: "QMD_ERR_MISALIGNED",
    6: "QMD_ERR_SHAPE",
    7: "QMD_ERR_LAUNCH",
    8: "QMD_ERR_DEVICE_TIMEOUT",
    9: "QMD_ERR_DEVICE",
    10: "QMD_ERR_VALUE",
}


class QmdError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(self.name + (f": {detail}" if detail else ""))


class Q8KPtrs(ctypes.Structure):
    _fields_ = [("qs", ctypes.c_void_p), ("d", ctypes.c_void_p), ("bsums", ctypes.c_void_p)]


_lib = None


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load libqmd.so (raises if it has not been built).  `path` loads another build of the same
    library instead (the traced build, libqmd_trace.so); it must come before the first load."""
    global _lib
    if _lib is not None and path is not None and path != _lib._name:
        raise RuntimeError(f"{_lib._name} is already loaded")
    if _lib is None:
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "or `python -m quantised_decode_mat_gb300.build`")
        L = ctypes.CDLL(path)
        i64, i32, vp, u64 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64
        ip = ctypes.POINTER(ctypes.c_int)
        sizep = ctypes.POINTER(ctypes.c_size_t)
        sigs = {
            "qmd_q8k_pack": ([vp, Q8KPtrs, i64, i32, vp], i32),
            "qmd_rmsnorm_q8k_pack": ([vp, vp, vp, ctypes.c_float, vp, Q8KPtrs, i64, i32, vp], i32),
            "qmd_qmatvec": ([i32, vp, vp, Q8KPtrs, vp, i64, i64, i32, vp], i32),
            "qmd_qmatvec_x": ([i32, vp, vp, vp, Q8KPtrs, vp, i64, i64, i32, vp], i32),
            "qmd_qmatvec_ws": ([i32, vp, vp, Q8KPtrs, vp, i64, i64, i32, vp, vp], i32),
            "qmd_qmatvec_x_ws": ([i32, vp, vp, vp, Q8KPtrs, vp, i64, i64, i32, vp, vp], i32),
            "qmd_qmatvec_x_static": ([i32, vp, vp, vp, Q8KPtrs, vp, i64, i64, i32, vp], i32),
            "qmd_qmatvec_rmsnorm_x": ([i32, vp, vp, vp, vp, vp, ctypes.c_float, vp, Q8KPtrs, vp, i64, i64, i32, vp],
                                      i32),
            "qmd_q6k_prefix_stride": ([i64], i64),
            "qmd_q6k_split_bytes": ([i64, i64, sizep, sizep], i32),
            "qmd_bind_q6k": ([vp, vp, vp, i64, i64, vp], i32),
            "qmd_bind_q4k": ([vp, i64, i64], i32),
            "qmd_bind_q5k": ([vp, i64, i64], i32),
            "qmd_status_str": ([i32], ctypes.c_char_p),
            "qmd_last_error_detail": ([], ctypes.c_char_p),
            "qmd_get_device_error": ([vp], i32),
            "qmd_set_wait_limit_ns": ([u64], None),
            "qmd_qmatvec_launch_info": ([i32, i64, i64, i32, ip, ip, ip, ip, ip], i32),
            "qmd_qmatvec_launch_kernel": ([i32, i64, i64, i32], i32),
            "qmd_debug_qmatvec_dump": ([i32, vp, vp, Q8KPtrs, vp, i64, i64, i32, vp, vp, vp], i32),
            "qmd_debug_wait_timeout": ([u64, vp], i32),
            "qmd_measure_alu": ([ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)], i32),
            "qmd_measure_read_bw": ([vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_double)], i32),
            "qmd_debug_set_plan": ([i32, i32, i32, i32], None),
            "qmd_debug_set_launch_flags": ([ctypes.c_uint], None),
            "qmd_debug_set_dynamic_tiles": ([i32], None),
            "qmd_debug_set_split_k": ([i32], None),
            "qmd_version": ([], i32),
        }
        if hasattr(L, "qmd_debug_trace"):  # the traced build (include/qmd_trace.h)
            sigs["qmd_debug_trace"] = ([vp, i64], i32)
            sigs["qmd_debug_trace_launches"] = ([vp, vp, i64], i64)
        for name, (args, res) in sigs.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(st: int) -> None:
    if st != 0:
        detail = lib().qmd_last_error_detail()
        raise QmdError(st, detail.decode() if detail else "")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class Q8K:
    """q8_K-packed activations (torch tensors on one CUDA device): qs int8 [B, K], d f32 [B, nb],
    bsums int16 [B, nb, 8]."""
    qs: "object"
    d: "object"
    bsums: "object"

    @property
    def batch(self) -> int:
        return self.qs.shape[0]

    @property
    def K(self) -> int:
        return self.qs.shape[1]

    def ptrs(self) -> Q8KPtrs:
        return Q8KPtrs(_ptr(self.qs), _ptr(self.d), _ptr(self.bsums))

    @staticmethod
    def empty(batch: int, K: int, device="cuda") -> "Q8K":
        import torch
        nb = K // QMD_QK
        return Q8K(torch.empty((batch, K), dtype=torch.int8, device=device),
                   torch.empty((batch, nb), dtype=torch.float32, device=device),
                   torch.empty((batch, nb, 8), dtype=torch.int16, device=device))


def q8k_pack(x, out: Q8K | None = None, stream=None) -> Q8K:
    """qmd_q8k_pack: x f32 [batch, K] (CUDA, contiguous) -> Q8K."""
    batch, K = x.shape
    if out is None:
        out = Q8K.empty(batch, K, x.device)
    _check(lib().qmd_q8k_pack(_ptr(x), out.ptrs(), K, batch, _stream(stream)))
    return out


def rmsnorm_q8k_pack(x, r, g, eps: float, h_out=None, out: Q8K | None = None, stream=None) -> Q8K:
    """qmd_rmsnorm_q8k_pack: h = x + r (r may be None), n = RMSNorm(h) * g, packed to q8_K.
    x, r, h_out f32 [batch, K]; g f32 [K].  h_out (optional, may be x or r) receives h."""
    batch, K = x.shape
    if out is None:
        out = Q8K.empty(batch, K, x.device)
    _check(lib().qmd_rmsnorm_q8k_pack(_ptr(x), _ptr(r), _ptr(g), float(eps), _ptr(h_out), out.ptrs(), K, batch,
                                      _stream(stream)))
    return out


def workspace(device="cuda"):
    """A zeroed scheduling workspace for qmatvec / qmatvec_x (QMD_WORKSPACE_BYTES on `device`).
    Calls ordered in one stream may share it; concurrent calls need their own."""
    import torch
    return torch.zeros(QMD_WORKSPACE_BYTES // 4, dtype=torch.int32, device=device)


def qmatvec(fmt: int, W, W_aux, xq: Q8K, y=None, rows: int | None = None, stream=None, workspace=None):
    """qmd_qmatvec (qmd_qmatvec_ws with a workspace): y f32 [batch, rows] = W (fmt) x xq.  W is the
    uint8 weight tensor whose first dimension is rows; W_aux the Q6_K prefix (None for Q4_K)."""
    import torch
    rows = W.shape[0] if rows is None else rows
    if y is None:
        y = torch.empty((xq.batch, rows), dtype=torch.float32, device=xq.qs.device)
    if workspace is None:
        _check(lib().qmd_qmatvec(fmt, _ptr(W), _ptr(W_aux), xq.ptrs(), _ptr(y), rows, xq.K, xq.batch,
                                 _stream(stream)))
    else:
        _check(lib().qmd_qmatvec_ws(fmt, _ptr(W), _ptr(W_aux), xq.ptrs(), _ptr(y), rows, xq.K, xq.batch,
                                    _ptr(workspace), _stream(stream)))
    return y


def qmatvec_x(fmt: int, W, W_aux, x, y=None, rows: int | None = None, xq_out: Q8K | None = None,
              stream=None, workspace=None):
    """qmd_qmatvec_x (qmd_qmatvec_x_ws with a workspace): y f32 [batch, rows] = W (fmt) x
    q8k_pack(x), packing inside the kernel.  x: f32 [batch, K].  xq_out: optional Q8K that
    receives the packed activations."""
    import torch
    rows = W.shape[0] if rows is None else rows
    batch, K = x.shape
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    out = xq_out.ptrs() if xq_out is not None else Q8KPtrs(None, None, None)
    if workspace is None:
        _check(lib().qmd_qmatvec_x(fmt, _ptr(W), _ptr(W_aux), _ptr(x), out, _ptr(y), rows, K, batch,
                                   _stream(stream)))
    else:
        _check(lib().qmd_qmatvec_x_ws(fmt, _ptr(W), _ptr(W_aux), _ptr(x), out, _ptr(y), rows, K, batch,
                                      _ptr(workspace), _stream(stream)))
    return y


def qmatvec_x_static(fmt: int, W, W_aux, x, y=None, rows: int | None = None, xq_out: Q8K | None = None,
                     stream=None):
    """qmd_qmatvec_x_static: qmatvec_x scheduled through the library's own static workspace, for
    callers that cannot allocate; calls that overlap on the GPU race on that workspace."""
    import torch
    rows = W.shape[0] if rows is None else rows
    batch, K = x.shape
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    out = xq_out.ptrs() if xq_out is not None else Q8KPtrs(None, None, None)
    _check(lib().qmd_qmatvec_x_static(fmt, _ptr(W), _ptr(W_aux), _ptr(x), out, _ptr(y), rows, K, batch,
                                      _stream(stream)))
    return y


def qmatvec_rmsnorm_x(fmt: int, W, W_aux, x, r, g, eps: float, h_out=None, y=None, rows: int | None = None,
                      xq_out: Q8K | None = None, stream=None):
    """qmd_qmatvec_rmsnorm_x: y f32 [batch, rows] = W (fmt) x rmsnorm_q8k_pack(x, r, g, eps), in one
    launch.  x, r (may be None), h_out (optional; must not overlap x, r or g) f32 [batch, K];
    g f32 [K]."""
    import torch
    rows = W.shape[0] if rows is None else rows
    batch, K = x.shape
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    out = xq_out.ptrs() if xq_out is not None else Q8KPtrs(None, None, None)
    _check(lib().qmd_qmatvec_rmsnorm_x(fmt, _ptr(W), _ptr(W_aux), _ptr(x), _ptr(r), _ptr(g), float(eps),
                                       _ptr(h_out), out, _ptr(y), rows, K, batch, _stream(stream)))
    return y


def q6k_prefix_stride(K: int) -> int:
    return int(lib().qmd_q6k_prefix_stride(K))


def q6k_split_bytes(rows: int, K: int) -> tuple[int, int]:
    b, p = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().qmd_q6k_split_bytes(rows, K, ctypes.byref(b), ctypes.byref(p)))
    return b.value, p.value


def bind_q6k(gguf, rows: int, K: int, body=None, prefix=None, stream=None):
    """qmd_bind_q6k: canonical Q6_K bytes (uint8 CUDA tensor, rows*nb*210) -> (body u8
    [rows, nb*208], prefix int16-typed f16 bits [rows, prefix_stride])."""
    import torch
    nb = K // QMD_QK
    if body is None:
        body = torch.empty((rows, nb * 208), dtype=torch.uint8, device=gguf.device)
    if prefix is None:
        prefix = torch.empty((rows, q6k_prefix_stride(K)), dtype=torch.int16, device=gguf.device)
    _check(lib().qmd_bind_q6k(_ptr(gguf), _ptr(body), _ptr(prefix), rows, K, _stream(stream)))
    return body, prefix


def bind_q4k(gguf, rows: int, K: int):
    """qmd_bind_q4k: checks the slab can be read in place as 32-bit words; returns it unchanged."""
    _check(lib().qmd_bind_q4k(_ptr(gguf), rows, K))
    return gguf


def bind_q5k(gguf, rows: int, K: int):
    """qmd_bind_q5k: checks the slab can be read in place; returns it unchanged."""
    _check(lib().qmd_bind_q5k(_ptr(gguf), rows, K))
    return gguf


def get_device_error(stream=None) -> None:
    """qmd_get_device_error: synchronise and raise QmdError if a kernel's bounded wait gave up."""
    _check(lib().qmd_get_device_error(_stream(stream)))


def set_wait_limit_ns(ns: int) -> None:
    lib().qmd_set_wait_limit_ns(int(ns))


def status_str(st: int) -> str:
    return lib().qmd_status_str(st).decode()


def launch_info(fmt: int, rows: int, K: int, batch: int) -> dict:
    vals = [ctypes.c_int() for _ in range(5)]
    _check(lib().qmd_qmatvec_launch_info(fmt, rows, K, batch, *[ctypes.byref(v) for v in vals]))
    return dict(zip(("grid", "threads", "smem_bytes", "stages", "rows_per_stage"), (v.value for v in vals)))


KERNELS = {0: "qmv_kernel", 1: "qmv_tc_kernel", 2: "qmv_rl_kernel", 3: "qmv_sk_kernel"}


def launch_kernel(fmt: int, rows: int, K: int, batch: int) -> str:
    """qmd_qmatvec_launch_kernel: the name of the kernel qmatvec runs for these sizes."""
    k = int(lib().qmd_qmatvec_launch_kernel(fmt, rows, K, batch))
    if k < 0:
        _check(-k)
    return KERNELS[k]


def debug_qmatvec_dump(fmt: int, W, W_aux, xq: Q8K, rows: int | None = None, stream=None):
    """qmd_debug_qmatvec_dump -> (y [B, rows], dots int32 [B, rows, nb, 16], sm int32 [B, rows, nb, 2])."""
    import torch
    rows = W.shape[0] if rows is None else rows
    dev = xq.qs.device
    nb = xq.K // QMD_QK
    y = torch.empty((xq.batch, rows), dtype=torch.float32, device=dev)
    dots = torch.zeros((xq.batch, rows, nb, 16), dtype=torch.int32, device=dev)
    sm = torch.zeros((xq.batch, rows, nb, 2), dtype=torch.int32, device=dev)
    _check(lib().qmd_debug_qmatvec_dump(fmt, _ptr(W), _ptr(W_aux), xq.ptrs(), _ptr(y), rows, xq.K,
                                        xq.batch, _ptr(dots), _ptr(sm), _stream(stream)))
    return y, dots, sm


def measure_alu() -> tuple[float, float]:
    """qmd_measure_alu: (dp4a instructions/s, mma.sync f16 FLOP/s) measured on this device."""
    d, m = ctypes.c_double(), ctypes.c_double()
    _check(lib().qmd_measure_alu(ctypes.byref(d), ctypes.byref(m)))
    return d.value, m.value


def measure_read_bw(buf) -> float:
    """qmd_measure_read_bw: bytes/s of read-only bulk streaming of `buf` (a CUDA tensor whose
    byte size is a multiple of 16; make it several times the L2)."""
    r = ctypes.c_double()
    _check(lib().qmd_measure_read_bw(_ptr(buf), buf.numel() * buf.element_size(), ctypes.byref(r)))
    return r.value


def debug_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(lib().qmd_debug_wait_timeout(int(limit_ns), _stream(stream)))


def debug_set_plan(row_groups: int = 0, rows_per_stage: int = 0, max_stages: int = 0, ctas_per_sm: int = 0) -> None:
    lib().qmd_debug_set_plan(row_groups, rows_per_stage, max_stages, ctas_per_sm)


def debug_set_launch_flags(flags: int = 0) -> None:
    lib().qmd_debug_set_launch_flags(int(flags))


def debug_set_dynamic_tiles(per_mille: int = -1) -> None:
    lib().qmd_debug_set_dynamic_tiles(int(per_mille))


def debug_set_split_k(ctas: int = 0) -> None:
    """qmd_debug_set_split_k: split each row's blocks over `ctas` CTAs of a cluster (2..8); 0 restores the default."""
    lib().qmd_debug_set_split_k(int(ctas))


def version() -> int:
    return int(lib().qmd_version())
