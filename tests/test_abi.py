"""The C ABI on the host (no GPU needed): the library builds and loads, exports every function
include/qmd.h declares, and refuses bad arguments with named statuses before touching CUDA."""
import ctypes
import os
import re

import pytest

import quantised_decode_mat_gb300 as q
from quantised_decode_mat_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmd.h")


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return q.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(qmd_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("qmd_q8k_pack", "qmd_qmatvec", "qmd_bind_q6k", "qmd_bind_q4k", "qmd_q6k_split_bytes",
                     "qmd_status_str", "qmd_get_device_error"):
        assert required in names


def test_every_declared_function_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in qmd.h but not exported by libqmd.so"
        ctypes.cast(getattr(L, name), ctypes.c_void_p)


def test_status_strings(L):
    for code, name in q.STATUS.items():
        assert q.status_str(code) == name
    assert q.status_str(99) == "QMD_ERR_UNKNOWN"


def test_version(L):
    assert q.version() >= 100


def test_prefix_stride_and_split_bytes(L):
    assert q.q6k_prefix_stride(256) == 8
    assert q.q6k_prefix_stride(14336) == 56
    assert q.q6k_prefix_stride(2048) == 8
    assert q.q6k_prefix_stride(2304) == 16
    assert q.q6k_prefix_stride(100) == 0
    assert q.q6k_split_bytes(4096, 14336) == (4096 * 56 * 208, 4096 * 56 * 2)
    with pytest.raises(q.QmdError, match="QMD_ERR_K_NOT_MULTIPLE_OF_256"):
        q.q6k_split_bytes(4, 300)
    with pytest.raises(q.QmdError, match="QMD_ERR_SHAPE"):
        q.q6k_split_bytes(0, 256)


A = 0x10000  # aligned fake device addresses: validation must fail before any of them is used
YA = A + (1 << 24)  # an output buffer that overlaps none of the inputs


def _xq(qs=A, d=A, bs=A):
    return q.Q8KPtrs(qs, d, bs)


def st_qmatvec(L, fmt=q.Q4_K, W=A, Wa=A, xq=None, y=YA, rows=16, K=512, batch=1):
    return L.qmd_qmatvec(fmt, W, Wa, xq or _xq(), y, rows, K, batch, None)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=15), 2), (dict(fmt=11), 2),
    (dict(W=None), 1),
    (dict(y=None), 1),
    (dict(xq=_xq(qs=None)), 1),
    (dict(xq=_xq(d=None)), 1),
    (dict(xq=_xq(bs=None)), 1),                     # Q4_K needs the sub-block sums
    (dict(fmt=q.Q6_K_SPLIT, Wa=None), 1),           # Q6_K needs the scale prefix
    (dict(K=300), 3),
    (dict(K=128), 3),
    (dict(K=0), 6),
    (dict(K=-256), 6),
    (dict(batch=0), 4),
    (dict(batch=9), 4),
    (dict(rows=0), 6),
    (dict(W=A + 8), 5),
    (dict(fmt=q.Q6_K_SPLIT, Wa=A + 4), 5),
    (dict(xq=_xq(qs=A + 4)), 5),
    (dict(xq=_xq(bs=A + 2)), 5),
    (dict(xq=_xq(d=A + 2)), 5),
    (dict(y=YA + 2), 5),
    # y is written while other CTAs still read the packed input: no overlap allowed
    (dict(y=A), 10), (dict(y=A + 496), 10), (dict(y=A - 16 * 4 + 4), 10),
])
def test_qmatvec_refusals(L, kw, status):
    assert st_qmatvec(L, **kw) == status


def test_qmatvec_q6k_does_not_need_bsums_but_needs_a_device(L):
    # validation passes; with no GPU in this process the call is refused as QMD_ERR_DEVICE
    # (or runs, on a GPU machine) -- it never falls back to anything on the CPU
    st = st_qmatvec(L, fmt=q.Q6_K_SPLIT, xq=_xq(bs=None))
    assert st in (0, 9, 7)
    if st == 0:
        pytest.skip("a GPU is present; the refusal path is covered by the GPU tests")


@pytest.mark.parametrize("args,status", [
    (dict(x=None), 1),
    (dict(K=100), 3),
    (dict(K=0), 6),
    (dict(batch=0), 4),
    (dict(batch=9), 4),
    (dict(x=A + 4), 5),
    (dict(qs=A + 8), 5),
    (dict(bs=A + 2), 5),
    (dict(d=A + 1), 5),
])
def test_pack_refusals(L, args, status):
    x = args.get("x", A)
    xq = _xq(qs=args.get("qs", A), d=args.get("d", A), bs=args.get("bs", A))
    assert L.qmd_q8k_pack(x, xq, args.get("K", 512), args.get("batch", 1), None) == status


@pytest.mark.parametrize("args,status", [
    (dict(g=None), 1),
    (dict(K=200), 3),
    (dict(rows=0), 6),
    (dict(g=A + 1), 5),
    (dict(b=A + 8), 5),
    (dict(p=A + 4), 5),
])
def test_bind_refusals(L, args, status):
    st = L.qmd_bind_q6k(args.get("g", A), args.get("b", A), args.get("p", A), args.get("rows", 4),
                        args.get("K", 512), None)
    assert st == status


def test_bind_q4k_is_a_checked_view(L):
    assert L.qmd_bind_q4k(A, 4, 512) == 0
    assert L.qmd_bind_q4k(A + 8, 4, 512) == 5
    assert L.qmd_bind_q4k(None, 4, 512) == 1
    assert L.qmd_bind_q4k(A, 4, 500) == 3


def test_no_gpu_means_a_named_refusal_not_a_fallback(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    assert L.qmd_qmatvec_launch_info(q.Q4_K, 4096, 4096, 1, None, None, None, None, None) == 9
    assert st_qmatvec(L) == 9
    assert L.qmd_q8k_pack(A, _xq(), 512, 1, None) == 9


def test_bind_q5k_is_a_checked_view(L):
    assert L.qmd_bind_q5k(A, 4, 512) == 0
    assert L.qmd_bind_q5k(A + 8, 4, 512) == 5
    assert L.qmd_bind_q5k(None, 4, 512) == 1
    assert L.qmd_bind_q5k(A, 0, 512) == 6
    assert L.qmd_bind_q5k(A, 4, 500) == 3


def test_q5k_is_a_known_format_with_q4k_limits(L):
    # validation passes for Q5_K (no prefix needed), so without a GPU the call reaches the
    # device check; K above the limits is refused on the host either way
    st = st_qmatvec(L, fmt=q.Q5_K, Wa=None)
    assert st in (0, 9, 7)
    assert st_qmatvec(L, fmt=q.Q5_K, K=500) == 3
    assert st_qmatvec(L, fmt=q.Q5_K, W=A + 4) == 5


def st_rms(L, x=A, r=None, g=A, eps=1e-6, h=None, xq=None, K=512, batch=2):
    return L.qmd_rmsnorm_q8k_pack(x, r, g, ctypes.c_float(eps), h, xq or _xq(), K, batch, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1), (dict(g=None), 1), (dict(xq=_xq(qs=None)), 1), (dict(xq=_xq(bs=None)), 1),
    (dict(K=300), 3), (dict(K=0), 6), (dict(batch=0), 4), (dict(batch=9), 4),
    (dict(x=A + 4), 5), (dict(r=A + 8), 5), (dict(g=A + 12), 5), (dict(h=A + 4), 5),
    (dict(xq=_xq(d=A + 2)), 5), (dict(eps=-1e-3), 10), (dict(eps=float("nan")), 10),
    (dict(eps=float("inf")), 10),
])
def test_rmsnorm_pack_refusals(L, kw, status):
    assert st_rms(L, **kw) == status


def test_rmsnorm_pack_valid_arguments_reach_the_device_check(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    assert st_rms(L) == 9
    assert st_rms(L, r=A, h=A, eps=0.0) == 9


def test_fused_entry_point_reaches_the_device_check(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    none = q.Q8KPtrs(None, None, None)
    assert L.qmd_qmatvec_x(q.Q4_K, A, None, A, none, YA, 16, 512, 1, None) == 9
    assert L.qmd_qmatvec_x(q.Q5_K, A, None, A, none, YA, 16, 512, 8, None) == 9
    assert L.qmd_qmatvec(q.Q4_K, A, None, _xq(), A + 512, 16, 512, 1, None) == 9  # adjacent, not overlapping


def test_fused_outputs_must_not_overlap_the_input(L):
    """Every CTA of a fused launch reads x while others write y (and CTA 0 the packed copy), so
    an overlap is refused before anything is launched, with or without a workspace."""
    none = q.Q8KPtrs(None, None, None)
    assert L.qmd_qmatvec_x(q.Q4_K, A, None, A, none, A, 16, 512, 1, None) == 10
    assert L.qmd_qmatvec_x(q.Q4_K, A, None, A, none, A + 2048 - 4, 16, 512, 1, None) == 10
    assert L.qmd_qmatvec_x(q.Q4_K, A, None, A, q.Q8KPtrs(A + 1024, YA + 4096, YA + 8192), YA, 16, 512, 1,
                           None) == 10
    assert L.qmd_qmatvec_x(q.Q4_K, A, None, A, q.Q8KPtrs(YA + 4096, A, YA + 8192), YA, 16, 512, 1, None) == 10
    assert L.qmd_qmatvec_x_ws(q.Q4_K, A, None, A, none, A, 16, 512, 1, YA + 65536, None) == 10
    assert L.qmd_qmatvec_ws(q.Q4_K, A, None, _xq(), A, 16, 512, 1, YA + 65536, None) == 10


def test_measure_alu_refuses_null_pointers(L):
    import ctypes
    d = ctypes.c_double()
    assert L.qmd_measure_alu(None, ctypes.byref(d)) == 1
    assert L.qmd_measure_alu(ctypes.byref(d), None) == 1


def st_norm_mv(L, fmt=q.Q4_K, W=A, Wa=None, x=A, r=None, g=A, eps=1e-6, h=None, xq=None, y=YA, rows=16, K=512,
               batch=2):
    return L.qmd_qmatvec_rmsnorm_x(fmt, W, Wa, x, r, g, ctypes.c_float(eps), h, xq or q.Q8KPtrs(None, None, None),
                                   y, rows, K, batch, None)


FAR = A + (1 << 20)  # a buffer that overlaps none of the others (2 x 512 f32 = 4 KB each)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1), (dict(g=None), 1), (dict(W=None), 1), (dict(y=None), 1),
    (dict(fmt=q.Q6_K_SPLIT), 1), (dict(xq=q.Q8KPtrs(A, None, None)), 1), (dict(fmt=7), 2),
    (dict(K=300), 3), (dict(batch=0), 4), (dict(batch=9), 4), (dict(rows=0), 6),
    (dict(x=A + 4), 5), (dict(r=A + 8), 5), (dict(g=A + 12), 5), (dict(h=FAR + 4), 5),
    (dict(eps=-1e-3), 10), (dict(eps=float("nan")), 10), (dict(eps=float("inf")), 10),
    # h is written by one CTA while the others still read x and r: no overlap allowed
    (dict(h=A), 10), (dict(h=A + 4096 - 16), 10), (dict(r=FAR, h=FAR + 16), 10), (dict(h=A - 4096 + 16), 10),
    # nor may y or the packed copy overlap x or r
    (dict(y=A), 10), (dict(r=FAR, y=FAR + 64), 10), (dict(xq=q.Q8KPtrs(A, YA + 4096, YA + 8192)), 10),
])
def test_rmsnorm_matvec_refusals(L, kw, status):
    assert st_norm_mv(L, **kw) == status


def test_rmsnorm_matvec_valid_arguments_reach_the_device_check(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    assert st_norm_mv(L) == 9
    assert st_norm_mv(L, r=FAR, h=FAR + 4096, eps=0.0) == 9
    assert st_norm_mv(L, h=A + 4096) == 9  # adjacent, not overlapping
    assert st_norm_mv(L, fmt=q.Q6_K_SPLIT, Wa=A, batch=8) == 9
