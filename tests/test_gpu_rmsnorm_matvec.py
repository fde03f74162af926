"""Residual add + RMSNorm + q8_K pack + mat-vec in one launch, through the C ABI (needs a GB300).

Bar: the same bits as the two-launch path (qmd_rmsnorm_q8k_pack, then qmd_qmatvec) -- y, the
packed codes and h -- and y bit-identical to the oracle's same-order epilogue applied to the
oracle's RMSNorm pack, within 2e-3 of its f64 brute force."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
import quantised_decode_mat_gb300 as q  # noqa: E402
from quantised_decode_mat_gb300 import synth  # noqa: E402

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]
DEV = "cuda"
GUARD = 64
OFMT = {"q4k": O.FMT_Q4_K, "q5k": O.FMT_Q5_K, "q6k": O.FMT_Q6_K}
QFMT = {"q4k": q.Q4_K, "q5k": q.Q5_K, "q6k": q.Q6_K_SPLIT}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from quantised_decode_mat_gb300 import build as qbuild
    qbuild.build()
    q.lib()
    q.debug_set_plan()
    q.debug_set_launch_flags(0)
    yield
    q.debug_set_plan()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def poisoned(batch, n):
    buf = torch.full((batch * n + GUARD,), -1, dtype=torch.int32, device=DEV)
    buf[batch * n:] = 0x5A5A5A5A
    return buf, buf[: batch * n].view(torch.float32).view(batch, n)


def intact(buf, batch, n):
    return bool((buf[batch * n:] == 0x5A5A5A5A).all())


def weights(fmtname, seed, rows, K):
    Wg = synth.weights(fmtname, seed, rows, K)
    if fmtname == "q6k":
        W, Wa = q.bind_q6k(dev(Wg.reshape(rows, -1)), rows, K)
    else:
        W, Wa = dev(Wg.reshape(rows, -1)), None
    return Wg, W, Wa


# (format, rows, K, batch, residual, eps): the decode step's shapes, one-row-group CTAs that the
# plan widens to 256 threads (K of one to three blocks of four), ragged row counts, batches 1..8
CASES = [("q4k", 4096, 4096, 1, True, 1e-5), ("q4k", 28672, 4096, 1, True, 1e-5),
         ("q6k", 512, 4096, 1, False, 1e-6), ("q5k", 300, 4096, 2, True, 1e-6),
         ("q4k", 77, 256, 1, True, 0.0), ("q6k", 45, 768, 3, True, 1e-6), ("q4k", 129, 2304, 5, False, 0.5),
         ("q5k", 64, 3328, 4, True, 1e-6), ("q4k", 500, 2048, 8, True, 1e-5), ("q6k", 17, 14336, 8, False, 1e-6),
         ("q4k", 9, 32768, 1, True, 1e-6), ("q6k", 33, 16384, 2, True, 1e-6), ("q4k", 1000, 1280, 2, False, 1e-6),
         ("q5k", 50, 14336, 6, True, 1e-5), ("q6k", 4096, 14336, 1, True, 1e-6)]


@pytest.mark.parametrize("fmtname,rows,K,batch,with_r,eps", CASES)
def test_rmsnorm_matvec_equals_two_launches_and_the_oracle(fmtname, rows, K, batch, with_r, eps):
    seed = 13 * rows + K + batch
    Wg, W, Wa = weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    r = synth.residual(seed, batch, K) if with_r else None
    g = synth.norm_gain(seed, K)
    xd, gd = dev(x), dev(g)
    rd = dev(r) if with_r else None
    f = QFMT[fmtname]

    xq2 = q.rmsnorm_q8k_pack(xd, rd, gd, eps)
    y2 = q.qmatvec(f, W, Wa, xq2, rows=rows)

    ybuf, y1 = poisoned(batch, rows)
    hbuf, h1 = poisoned(batch, K)
    out = q.Q8K.empty(batch, K, DEV)
    q.qmatvec_rmsnorm_x(f, W, Wa, xd, rd, gd, eps, h_out=h1, y=y1, rows=rows, xq_out=out)
    q.get_device_error()
    assert intact(ybuf, batch, rows) and intact(hbuf, batch, K)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert torch.equal(out.qs, xq2.qs) and torch.equal(out.bsums, xq2.bsums)
    assert torch.equal(out.d.view(torch.int32), xq2.d.view(torch.int32))

    oh, oqs, od, obs = O.rmsnorm_q8k_pack(x, r, g, eps)
    assert np.array_equal(h1.cpu().numpy().view(np.uint32), oh.view(np.uint32))
    idx = None if rows <= 600 else np.r_[0:64, rows // 2:rows // 2 + 64, rows - 64:rows]
    Wo = Wg if idx is None else Wg[idx]
    yg = y1.cpu().numpy() if idx is None else y1.cpu().numpy()[:, idx]
    ref = O.qmatvec(OFMT[fmtname], Wo, oqs, od, obs, O.ORDER_RUNS_OF_SIXTEEN)
    diff = np.count_nonzero(yg.view(np.uint32) != ref.view(np.uint32))
    assert diff == 0, f"{diff} outputs differ in bits from the same-order oracle"
    assert O.rel_err(yg, O.qmatvec_f64(OFMT[fmtname], Wo, oqs, od)).max() <= 2e-3


@pytest.mark.parametrize("flags", [0, 8], ids=["rowlane", "slice"])
@pytest.mark.parametrize("rg,cps", [(1, 1), (2, 3), (4, 2), (8, 1)])
def test_rmsnorm_matvec_under_forced_plans(rg, cps, flags):
    """Forced row groups (row-lane kernel: ring warps) and CTAs per SM (every CTA recomputes the
    norm; a CTA with fewer than 8 warps is widened to the 256 threads the sum of squares takes):
    the same bits, on the row-lane kernel (default at one vector) and the dp4a slice kernel."""
    q.debug_set_launch_flags(flags)
    rows, K, batch = 3000, 4096, 1
    Wg, W, Wa = weights("q4k", 5, rows, K)
    x, r, g = synth.activations(5, batch, K), synth.residual(5, batch, K), synth.norm_gain(5, K)
    xd, rd, gd = dev(x), dev(r), dev(g)
    y2 = q.qmatvec(q.Q4_K, W, Wa, q.rmsnorm_q8k_pack(xd, rd, gd, 1e-6), rows=rows)
    q.debug_set_plan(row_groups=rg, ctas_per_sm=cps)
    try:
        y1 = q.qmatvec_rmsnorm_x(q.Q4_K, W, Wa, xd, rd, gd, 1e-6, rows=rows)
        q.get_device_error()
    finally:
        q.debug_set_plan()
        q.debug_set_launch_flags(0)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_rmsnorm_matvec_refusals_write_nothing():
    rows, K, batch = 8, 512, 2
    W = torch.zeros(rows * 2 * 144, dtype=torch.uint8, device=DEV)
    x = torch.ones((batch, K), dtype=torch.float32, device=DEV)
    g = torch.ones(K, dtype=torch.float32, device=DEV)
    ybuf, y = poisoned(batch, rows)
    with pytest.raises(q.QmdError, match="QMD_ERR_VALUE"):  # h over x
        q.qmatvec_rmsnorm_x(q.Q4_K, W, None, x, None, g, 1e-6, h_out=x, y=y, rows=rows)
    with pytest.raises(q.QmdError, match="QMD_ERR_VALUE"):
        q.qmatvec_rmsnorm_x(q.Q4_K, W, None, x, None, g, -1.0, y=y, rows=rows)
    with pytest.raises(q.QmdError, match="QMD_ERR_SHAPE"):  # a row too long for every kernel's form
        Wl = torch.zeros(rows * 1024 * 144, dtype=torch.uint8, device=DEV)
        xl = torch.ones((1, 262144), dtype=torch.float32, device=DEV)
        gl = torch.ones(262144, dtype=torch.float32, device=DEV)
        q.qmatvec_rmsnorm_x(q.Q4_K, Wl, None, xl, None, gl, 1e-6, y=y[:1], rows=rows)
    torch.cuda.synchronize()
    assert torch.isnan(y).all() and intact(ybuf, batch, rows)
