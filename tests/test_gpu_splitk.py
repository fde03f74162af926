"""Split-K form of the mat-vec ("Language models on the device: the cajeta-llm kernels", §2.3:
partial sums along K, combined by a fixup): each row's groups of four blocks split over the CTAs
of a thread-block cluster, the slices' group sums added in the declared row order through
distributed shared memory.  Every output must have the bits of the same-order oracle (and of the
default plan), in the plain and the fused form, at one and two vectors, for every split count a
shape allows; the f64 brute force bounds it as everywhere else."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
import quantised_decode_mat_gb300 as q  # noqa: E402
from quantised_decode_mat_gb300 import synth  # noqa: E402
from tests.oracle_rows import oracle_rows_threaded  # noqa: E402

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

TOL_SAME_ORDER = 1e-5
TOL_F64 = 2e-3
GUARD = 64
DEV = "cuda"
OFMT = {"q4k": O.FMT_Q4_K, "q5k": O.FMT_Q5_K, "q6k": O.FMT_Q6_K}
QFMT = {"q4k": q.Q4_K, "q5k": q.Q5_K, "q6k": q.Q6_K_SPLIT}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from quantised_decode_mat_gb300 import build as qbuild
    qbuild.build()
    q.lib()
    q.debug_set_plan()
    q.debug_set_launch_flags(0)
    q.debug_set_split_k(0)
    yield
    q.debug_set_plan()
    q.debug_set_launch_flags(0)
    q.debug_set_split_k(0)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _weights(fmtname, Wg, rows, K):
    if fmtname in ("q4k", "q5k"):
        return QFMT[fmtname], _dev(Wg.reshape(rows, -1)), None
    body, prefix = q.bind_q6k(_dev(Wg.reshape(rows, -1)), rows, K)
    return q.Q6_K_SPLIT, body, prefix


def _poisoned(batch, rows):
    buf = torch.full((batch * rows + GUARD,), -1, dtype=torch.int32, device=DEV)
    buf[batch * rows:] = 0x5A5A5A5A
    return buf, buf[: batch * rows].view(torch.float32).view(batch, rows)


def _run(f, W, Wa, x, rows, fused, ks, plan=None):
    """y from one launch with split-K at ks CTAs a cluster (0: the default plan), into a poisoned
    buffer with guard words; also the packed activations of the fused form."""
    batch, K = x.shape
    q.debug_set_split_k(ks)
    if plan:
        q.debug_set_plan(*plan)
    try:
        kern = q.launch_kernel(f, rows, K, batch)
        buf, y = _poisoned(batch, rows)
        out = None
        if fused:
            out = q.Q8K.empty(batch, K, DEV)
            q.qmatvec_x(f, W, Wa, _dev(x), y, rows=rows, xq_out=out)
        else:
            q.qmatvec(f, W, Wa, q.q8k_pack(_dev(x)), y, rows)
        q.get_device_error()
    finally:
        q.debug_set_split_k(0)
        q.debug_set_plan()
    assert bool((buf[batch * rows:] == 0x5A5A5A5A).all()), "write past the end of y"
    return kern, y, out


def _check(fmtname, Wg, x, y, f64_rows=300):
    oqs, od, obs = O.q8k_pack(x)
    yg = y.cpu().numpy()
    assert np.isfinite(yg).all(), "unwritten (NaN) outputs"
    ref = oracle_rows_threaded(OFMT[fmtname], Wg, oqs, od, obs, O.ORDER_RUNS_OF_SIXTEEN)
    assert O.rel_err(yg, ref).max() <= TOL_SAME_ORDER
    diff = np.count_nonzero(yg.view(np.uint32) != ref.view(np.uint32))
    assert diff == 0, f"{diff} outputs differ in bits from the same-order oracle"
    rows = Wg.shape[0]
    idx = np.unique(np.linspace(0, rows - 1, min(rows, f64_rows)).astype(np.int64))
    ref64 = O.qmatvec_f64(OFMT[fmtname], Wg[idx], oqs, od)
    assert O.rel_err(yg[:, idx], ref64).max() <= TOL_F64


# config 0 (256 x 2048), config 1 and the step's o (4096 x 4096), the step's q|k|v (6144 x 4096)
SHAPES = [("cfg0", 0, 256, 2048), ("cfg1_o", 1, 4096, 4096), ("qkv", 3, 6144, 4096)]


@pytest.mark.parametrize("fused", [False, True], ids=["packed", "fused"])
@pytest.mark.parametrize("batch", [1, 2])
@pytest.mark.parametrize("name,seed,rows,K", SHAPES, ids=[s[0] for s in SHAPES])
def test_split_k_short_projections_every_row(name, seed, rows, K, batch, fused):
    """Every split count the shape allows (2..4 slices of its 2 or 4 groups) and the default plan:
    the same bits on every row."""
    Wg = synth.weights("q4k", seed, rows, K)
    x = synth.activations(seed + 100 * batch, batch, K)
    f, W, Wa = _weights("q4k", Wg, rows, K)
    gq = K // 1024
    _, y0, out0 = _run(f, W, Wa, x, rows, fused, 0)
    _check("q4k", Wg, x, y0)
    for ks in range(2, min(gq, 4) + 1):
        kern, y, out = _run(f, W, Wa, x, rows, fused, ks)
        assert kern == "qmv_sk_kernel"
        assert torch.equal(y.view(torch.int32), y0.view(torch.int32)), f"split {ks}"
        if fused:
            assert torch.equal(out.qs, out0.qs) and torch.equal(out.bsums, out0.bsums)
            assert torch.equal(out.d.view(torch.int32), out0.d.view(torch.int32))


RAGGED = [
    # fmt, rows, K, batch: ragged rows (not a multiple of 8), groups that do not divide evenly,
    # absent blocks in the last group, a last run of fewer than four groups, long rows
    ("q4k", 1000, 4352, 1), ("q4k", 1, 2048, 2), ("q4k", 9, 32768, 1), ("q4k", 3001, 1280, 2),
    ("q5k", 333, 1792, 1), ("q5k", 77, 4352, 2), ("q5k", 4096, 4096, 1),
    ("q6k", 77, 2304, 1), ("q6k", 300, 14336, 1), ("q6k", 40, 14336, 2), ("q6k", 9, 32768, 2),
    ("q6k", 4096, 14336, 1),
]


@pytest.mark.parametrize("fused", [False, True], ids=["packed", "fused"])
@pytest.mark.parametrize("fmtname,rows,K,batch", RAGGED)
def test_split_k_ragged_shapes(fmtname, rows, K, batch, fused):
    seed = 13 * rows + K + batch
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    f, W, Wa = _weights(fmtname, Wg, rows, K)
    gq = -(-K // 1024)
    for ks in sorted({2, 3, min(gq, 5), min(gq, 8)}):
        if ks < 2 or ks > gq:
            continue
        kern, y, _ = _run(f, W, Wa, x, rows, fused, ks)
        assert kern == "qmv_sk_kernel"
        _check(fmtname, Wg, x, y)


# (ring warps, pre-wait slots, ring slots, -): one-slot rings wrap at every step; one or two
# ring warps walk many tiles each
@pytest.mark.parametrize("plan", [(0, 1, 1, 0), (0, 2, 2, 0), (1, 1, 3, 0), (3, 4, 2, 0)])
@pytest.mark.parametrize("fmtname,rows,K,batch", [("q4k", 4096, 4096, 1), ("q6k", 600, 14336, 2),
                                                  ("q5k", 1500, 3072, 1)])
def test_split_k_forced_rings(plan, fmtname, rows, K, batch):
    Wg = synth.weights(fmtname, 7, rows, K)
    x = synth.activations(7, batch, K)
    f, W, Wa = _weights(fmtname, Wg, rows, K)
    kern, y, _ = _run(f, W, Wa, x, rows, True, 2, plan)
    assert kern == "qmv_sk_kernel"
    _check(fmtname, Wg, x, y)


def test_split_k_applies_only_where_it_can():
    """Three vectors and more, and rows with fewer groups than slices, keep their default kernels."""
    try:
        q.debug_set_split_k(4)
        assert q.launch_kernel(q.Q4_K, 4096, 4096, 1) == "qmv_sk_kernel"
        assert q.launch_kernel(q.Q4_K, 4096, 4096, 3) != "qmv_sk_kernel"
        assert q.launch_kernel(q.Q4_K, 256, 2048, 1) != "qmv_sk_kernel"  # two groups a row
        q.debug_set_split_k(9)  # out of range: the default plan
        assert q.launch_kernel(q.Q4_K, 4096, 4096, 1) != "qmv_sk_kernel"
    finally:
        q.debug_set_split_k(0)
