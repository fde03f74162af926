"""GPU path vs the CPU oracle, through the C ABI (needs a GB300).

Bars (from the method's statement): q8_K packs and per-sub-block int32 dots bit-exact; f32
outputs within 1e-5 relative of the oracle's f32 epilogue in the same order (the kernel is
built to match it bit for bit, which is also checked), and within 2e-3 of the f64 brute force.
Relative error is per element, |d| / max(|ref|, 1e-3 * rms(ref over the output vector)).
Output buffers are poisoned with NaN (0xFF bytes) and followed by guard words, so a row that
is not written, or a write past the end, fails.
"""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from quantised_decode_mat_gb300 import build as qbuild
    qbuild.build()
    q.lib()
    q.debug_set_plan()
    q.debug_set_launch_flags(0)
    yield
    q.debug_set_plan()
    q.debug_set_launch_flags(0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def poisoned_y(batch, rows):
    """f32 [batch, rows] filled with NaN bits, followed by GUARD guard words."""
    buf = torch.full((batch * rows + GUARD,), -1, dtype=torch.int32, device=DEV)
    buf[batch * rows:] = 0x5A5A5A5A
    return buf, buf[: batch * rows].view(torch.float32).view(batch, rows)


def guard_intact(buf, batch, rows):
    return bool((buf[batch * rows:] == 0x5A5A5A5A).all())


def gpu_pack(x):
    xq = q.q8k_pack(dev(x))
    torch.cuda.synchronize()
    return xq


def run_matvec(fmtname, Wg, xq, rows, K, batch):
    """Upload canonical GGUF weights, bind (Q6_K), run the mat-vec into a poisoned buffer."""
    buf, y = poisoned_y(batch, rows)
    if fmtname in ("q4k", "q5k"):
        q.qmatvec(QFMT[fmtname], dev(Wg.reshape(rows, -1)), None, xq, y, rows)
    else:
        body, prefix = q.bind_q6k(dev(Wg.reshape(rows, -1)), rows, K)
        q.qmatvec(q.Q6_K_SPLIT, body, prefix, xq, y, rows)
    q.get_device_error()
    assert guard_intact(buf, batch, rows), "write past the end of y"
    return y.cpu().numpy()


OFMT = {"q4k": O.FMT_Q4_K, "q5k": O.FMT_Q5_K, "q6k": O.FMT_Q6_K}
QFMT = {"q4k": q.Q4_K, "q5k": q.Q5_K, "q6k": q.Q6_K_SPLIT}


def check_against_oracle(fmtname, Wg, x, y, rows_idx=None, exact=True, f64_idx=None):
    """y [B, R] from the GPU vs oracle on the same W (canonical) and x; rows_idx samples rows
    (default: every row); f64_idx limits the f64 brute force to a sample of those."""
    oqs, od, obs = O.q8k_pack(x)
    W = Wg if rows_idx is None else Wg[rows_idx]
    yg = y if rows_idx is None else y[:, rows_idx]
    ref = oracle_rows_threaded(OFMT[fmtname], W, oqs, od, obs, O.ORDER_RUNS_OF_SIXTEEN)
    assert np.isfinite(yg).all(), "unwritten (NaN) outputs"
    err = O.rel_err(yg, ref)
    assert err.max() <= TOL_SAME_ORDER, f"same-order rel err {err.max():.3g}"
    if exact:
        diff = np.count_nonzero(yg.view(np.uint32) != ref.view(np.uint32))
        assert diff == 0, f"{diff} outputs differ in bits from the same-order oracle"
    if f64_idx is not None:
        W, yg = W[f64_idx], yg[:, f64_idx]
    ref64 = O.qmatvec_f64(OFMT[fmtname], W, oqs, od)
    assert O.rel_err(yg, ref64).max() <= TOL_F64


# ---- q8_K pack --------------------------------------------------------------------------------------
def _pack_inputs():
    rng = np.random.default_rng(3)
    cases = [("n01_b1_k4096", synth.activations(1, 1, 4096)),
             ("n01_b8_k14336", synth.activations(2, 8, 14336)),
             ("n01_b3_k256", synth.activations(3, 3, 256))]
    x = synth.activations(4, 2, 1024)
    x[0, 256:512] = 0.0                         # all-zero block
    x[1, 0:256] = np.float32(1e-38)              # block whose 127/amax overflows to inf
    x[1, 3] = 0.0
    x[1, 512:768] = (np.arange(256) - 128).astype(np.float32) * np.float32(0.5)   # ties at .5 steps
    x[1, 768] = 1e30
    cases.append(("special", x))
    big = (rng.standard_normal((2, 2048)) * 1e4).astype(np.float32)
    cases.append(("large", big))
    return cases


@pytest.mark.parametrize("name,x", _pack_inputs(), ids=[c[0] for c in _pack_inputs()])
def test_pack_bit_exact(name, x):
    xq = gpu_pack(x)
    oqs, od, obs = O.q8k_pack(x)
    assert np.array_equal(xq.qs.cpu().numpy(), oqs)
    assert np.array_equal(xq.d.cpu().numpy().view(np.uint32), od.view(np.uint32))
    assert np.array_equal(xq.bsums.cpu().numpy(), obs)


# ---- integer dots, S and M, bit-exact (recording variant of the same kernel) -----------------------
@pytest.mark.parametrize("fmtname", ["q4k", "q5k", "q6k"])
@pytest.mark.parametrize("batch,rows,K", [(1, 37, 1024), (2, 19, 2304), (3, 11, 256), (5, 7, 3072), (8, 13, 4096),
                                          (1, 9, 14336), (2, 5, 5376)])
def test_subblock_dots_exact(fmtname, batch, rows, K):
    Wg = synth.weights(fmtname, 7, rows, K)
    x = synth.activations(7, batch, K)
    xq = gpu_pack(x)
    Wd = dev(Wg.reshape(rows, -1))
    if fmtname in ("q4k", "q5k"):
        y, dots, sm = q.debug_qmatvec_dump(QFMT[fmtname], Wd, None, xq)
    else:
        body, prefix = q.bind_q6k(Wd, rows, K)
        y, dots, sm = q.debug_qmatvec_dump(q.Q6_K_SPLIT, body, prefix, xq, rows)
    q.get_device_error()
    dots = dots.cpu().numpy()
    sm = sm.cpu().numpy()
    oqs, od, obs = O.q8k_pack(x)
    nb = K // 256
    for v in range(batch):
        for r in range(rows):
            od_ = O.subdots(OFMT[fmtname], Wg[r], oqs[v])
            if fmtname in ("q4k", "q5k"):
                got = dots[v, r][:, :8]  # entry j: sub-block j
                assert not dots[v, r][:, 8:].any()
            else:
                got = dots[v, r]
            assert np.array_equal(got, od_), (v, r)
            for b in range(nb):
                if fmtname in ("q4k", "q5k"):
                    _, _, sc, m, _ = (O.q4k_fields if fmtname == "q4k" else O.q5k_fields)(Wg[r, b])
                    S = int(np.dot(sc, od_[b]))
                    M = int(np.dot(m, obs[v, b].astype(np.int64)))
                else:
                    _, sc, _ = O.q6k_fields(Wg[r, b])
                    S, M = int(np.dot(sc, od_[b])), 0
                assert (sm[v, r, b, 0], sm[v, r, b, 1]) == (S, M), (v, r, b)
    check_against_oracle(fmtname, Wg, x, y.cpu().numpy())


# ---- outputs: the five workloads and a sweep of ragged shapes -----------------------------------------
@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_configs_full(cfg):
    c = synth.CONFIGS[cfg]
    for batch in c["batches"]:
        Wg = synth.weights(c["fmt"], c["seed"], c["rows"], c["K"])
        x = synth.activations(c["seed"], batch, c["K"])
        y = run_matvec(c["fmt"], Wg, gpu_pack(x), c["rows"], c["K"], batch)
        check_against_oracle(c["fmt"], Wg, x, y)


def _sample_rows(rows, n, seed):
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(rows, size=min(n, rows), replace=False).tolist())
    pick |= {0, 1, rows - 2, rows - 1}
    return np.array(sorted(pick))


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_config3_gate_up_every_row(batch):
    """The fused gate|up shape (28672 x 4096) at each of its batches, every output bit-identical to
    the same-order oracle (threaded over rows); the f64 brute force on a sample of rows."""
    c = synth.CONFIGS[3]
    Wg = synth.weights(c["fmt"], c["seed"], c["rows"], c["K"])
    x = synth.activations(c["seed"], batch, c["K"])
    y = run_matvec(c["fmt"], Wg, gpu_pack(x), c["rows"], c["K"], batch)
    assert np.isfinite(y).all()
    check_against_oracle(c["fmt"], Wg, x, y, f64_idx=_sample_rows(c["rows"], 400, batch))


SWEEP = [
    # fmt, rows, K, batch
    ("q4k", 1, 256, 1), ("q4k", 3, 512, 2), ("q4k", 129, 768, 3), ("q4k", 1000, 1280, 1),
    ("q4k", 333, 2048, 4), ("q4k", 77, 4352, 5), ("q4k", 250, 4096, 6), ("q4k", 61, 3840, 7),
    ("q4k", 500, 4096, 8), ("q4k", 5, 16384, 8), ("q4k", 9, 32768, 1), ("q4k", 6, 32768, 2),
    ("q4k", 1500, 5120, 2), ("q6k", 700, 4352, 1),
    ("q6k", 1, 256, 1), ("q6k", 5, 512, 2), ("q6k", 130, 1792, 1), ("q6k", 257, 2304, 3),
    ("q6k", 64, 3328, 4), ("q6k", 300, 14336, 1), ("q6k", 40, 14336, 2), ("q6k", 31, 14336, 4),
    ("q6k", 17, 14336, 8), ("q6k", 4, 32768, 1), ("q6k", 9, 16384, 7),
    ("q5k", 1, 256, 1), ("q5k", 4096, 4096, 1), ("q5k", 129, 768, 3), ("q5k", 333, 2048, 4),
    ("q5k", 77, 4352, 5), ("q5k", 500, 4096, 8), ("q5k", 9, 32768, 1), ("q5k", 6, 32768, 2),
    ("q5k", 40, 14336, 2), ("q5k", 5, 16384, 7), ("q5k", 1000, 1280, 2),
]


@pytest.mark.parametrize("fmtname,rows,K,batch", SWEEP)
def test_sweep_shapes(fmtname, rows, K, batch):
    seed = rows * 7 + K + batch
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    y = run_matvec(fmtname, Wg, gpu_pack(x), rows, K, batch)
    check_against_oracle(fmtname, Wg, x, y)


# (row groups per CTA, rows per group per stage, max stages, CTAs per SM)
@pytest.mark.parametrize("plan", [(1, 1, 1, 0), (2, 2, 2, 0), (1, 8, 1, 0), (3, 4, 2, 0), (4, 1, 3, 0),
                                  (2, 2, 8, 2), (5, 1, 2, 3)])
@pytest.mark.parametrize("fmtname,rows,K,batch", [("q4k", 2000, 4096, 1), ("q4k", 700, 2048, 3),
                                                  ("q6k", 600, 3584, 1), ("q6k", 150, 7168, 2),
                                                  ("q6k", 90, 14336, 1), ("q5k", 1500, 4096, 1),
                                                  ("q5k", 300, 3072, 4), ("q4k", 900, 4096, 6)])
@pytest.mark.parametrize("flags", [0, 8, 16, 4], ids=["default", "slice", "rowlane", "tensor"])
def test_pipeline_plans(plan, fmtname, rows, K, batch, flags):
    """Force small stage rings (many wrap-arounds per CTA) and other CTA shapes: same bits.  For
    the row-lane kernel (batches 1 and 2 by default, 3 and 4 with flag 16) the plan's row groups
    are its warps per CTA and its stages the slots of each warp's ring; flag 8 runs the dp4a
    slice kernel instead; flag 4 the tensor-core kernel from three vectors up (a ring cap of 2:
    its 32-row tiles, 3 or more: 16-row tiles in rings of at most that many)."""
    q.debug_set_plan(*plan)
    q.debug_set_launch_flags(flags)
    try:
        Wg = synth.weights(fmtname, 5, rows, K)
        x = synth.activations(5, batch, K)
        y = run_matvec(fmtname, Wg, gpu_pack(x), rows, K, batch)
    finally:
        q.debug_set_plan()
        q.debug_set_launch_flags(0)
    check_against_oracle(fmtname, Wg, x, y)


def test_degenerate_inputs():
    rows, K = 64, 1024
    # all-zero activations: every term is 0 * (...) = 0
    Wg = synth.q4k_weights(1, rows, K)
    x = np.zeros((2, K), np.float32)
    y = run_matvec("q4k", Wg, gpu_pack(x), rows, K, 2)
    assert np.all(y == 0.0)
    # zero codes: only the -dmin * min term remains (checked against the oracle bit for bit)
    Wz = Wg.copy()
    Wz[:, :, 16:] = 0
    x = synth.activations(2, 1, K)
    y = run_matvec("q4k", Wz, gpu_pack(x), rows, K, 1)
    check_against_oracle("q4k", Wz, x, y)
    # Q6_K codes all 32 give exactly zero
    W6 = synth.q6k_weights(1, rows, K).copy()
    W6[:, :, 0:128] = 0
    W6[:, :, 128:192] = 0xAA
    y = run_matvec("q6k", W6, gpu_pack(x), rows, K, 1)
    assert np.all(y == 0.0)
    # Q5_K with no fifth bits gives the Q4_K block's bits exactly
    W5 = synth.q5k_weights(1, rows, K).copy()
    W5[:, :, 16:48] = 0
    W4 = np.ascontiguousarray(np.concatenate([W5[:, :, 0:16], W5[:, :, 48:176]], axis=2))
    xq = gpu_pack(x)
    y5 = run_matvec("q5k", W5, xq, rows, K, 1)
    y4 = run_matvec("q4k", W4, xq, rows, K, 1)
    assert np.array_equal(y5.view(np.uint32), y4.view(np.uint32))
    # Q5_K with every fifth bit set and zero nibbles: codes all 16
    W5[:, :, 16:48] = 0xFF
    W5[:, :, 48:176] = 0
    y = run_matvec("q5k", W5, xq, rows, K, 1)
    check_against_oracle("q5k", W5, x, y)


def test_bind_q6k_matches_oracle_split():
    rows, K = 33, 2304
    g = synth.q6k_weights(9, rows, K)
    body, prefix = q.bind_q6k(dev(g.reshape(rows, -1)), rows, K)
    torch.cuda.synchronize()
    ob, op = O.q6k_split(g, q.q6k_prefix_stride(K))
    assert np.array_equal(body.cpu().numpy().reshape(ob.shape), ob)
    assert np.array_equal(prefix.cpu().numpy().view(np.uint16), op)


# ---- refusals launch nothing; bounded waits report instead of hanging ---------------------------------
def test_refused_calls_write_nothing():
    """Every buffer here is large enough for the largest shape passed, so a call that the host
    wrongly accepted could not read or write outside its buffers."""
    rows, Kmax, Bmax = 16, 1 << 20, 8
    W = torch.zeros(rows * (Kmax // 256) * 144, dtype=torch.uint8, device=DEV)
    xq = q.Q8K.empty(Bmax, Kmax, DEV)
    buf, y = poisoned_y(Bmax, rows)
    L = q.lib()
    assert L.qmd_qmatvec(q.Q4_K, W.data_ptr(), None, xq.ptrs(), y.data_ptr(), rows, 500, 1, None) == 3
    assert L.qmd_qmatvec(q.Q4_K, W.data_ptr() + 8, None, xq.ptrs(), y.data_ptr(), rows, 512, 1, None) == 5
    assert L.qmd_qmatvec(q.Q4_K, W.data_ptr(), None, xq.ptrs(), y.data_ptr(), rows, 512, 9, None) == 4
    # rows too long for either kernel: 4096 blocks (the tensor-core kernel's 255 earlier runs'
    # sums do not fit beside its rings), and past the 2^20-block limit
    for B in (1, 3, 8):
        assert L.qmd_qmatvec(q.Q4_K, W.data_ptr(), None, xq.ptrs(), y.data_ptr(), rows, Kmax, B, None) == 6
    assert L.qmd_qmatvec(q.Q4_K, W.data_ptr(), None, xq.ptrs(), y.data_ptr(), rows, 256 << 21, 1, None) == 6
    torch.cuda.synchronize()
    assert torch.isnan(y).all() and guard_intact(buf, Bmax, rows)
    q.get_device_error()


@pytest.mark.parametrize("fmtname", ["q4k", "q6k"])
@pytest.mark.parametrize("rows,K,batch", [(40, 65536, 1), (21, 32768, 3), (40, 20480, 4), (300, 36864, 2)])
def test_long_rows_beyond_the_dp4a_limit(fmtname, rows, K, batch):
    """Rows the dp4a slice kernel cannot take (more than 128 blocks at one or two vectors, 64
    above) run on the row-lane kernel, whose warps walk any row length step by step (the default
    at one or two vectors, flag 16 at three or four), or on the tensor-core kernel run by run
    (the default at three or four vectors, flag 8 below).  All bit-identical to the same-order
    oracle."""
    assert (q.launch_kernel(QFMT[fmtname], rows, K, batch) == "qmv_rl_kernel") == (batch <= 2)
    seed = rows + K + batch
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    xq = gpu_pack(x)
    y = run_matvec(fmtname, Wg, xq, rows, K, batch)
    check_against_oracle(fmtname, Wg, x, y)
    for flags, kern in ((SLICE, "qmv_tc_kernel"), (RL, "qmv_rl_kernel")):
        q.debug_set_launch_flags(flags)
        try:
            assert q.launch_kernel(QFMT[fmtname], rows, K, batch) == kern
            y2 = run_matvec(fmtname, Wg, xq, rows, K, batch)
        finally:
            q.debug_set_launch_flags(0)
        assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("cps", [1, 3, 8])
def test_long_rows_with_forced_ctas_per_sm(cps):
    """A forced CTAs-per-SM count can ask for more resident CTAs than fit; the run-by-run
    tensor-core kernel keeps its planned grid (its run sums are sized for it), and the CTAs that
    do not fit at once run later."""
    fmtname, rows, K, batch = "q4k", 700, 20480, 3
    seed = 91 + cps
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    q.debug_set_plan(0, 0, 0, cps)
    q.debug_set_launch_flags(SLICE)  # the tensor-core kernel, not the row-lane one
    try:
        assert q.launch_kernel(QFMT[fmtname], rows, K, batch) == "qmv_tc_kernel"
        y = run_matvec(fmtname, Wg, gpu_pack(x), rows, K, batch)
    finally:
        q.debug_set_plan()
        q.debug_set_launch_flags(0)
    check_against_oracle(fmtname, Wg, x, y)


def test_bounded_wait_reports_timeout_and_context_survives():
    q.debug_wait_timeout(2_000_000)  # 2 ms
    with pytest.raises(q.QmdError, match="QMD_ERR_DEVICE_TIMEOUT"):
        q.get_device_error()
    q.get_device_error()  # cleared
    # the context is still usable
    rows, K = 8, 256
    Wg = synth.q4k_weights(2, rows, K)
    x = synth.activations(2, 1, K)
    y = run_matvec("q4k", Wg, gpu_pack(x), rows, K, 1)
    check_against_oracle("q4k", Wg, x, y)


def test_launch_info_shapes():
    i1 = q.launch_info(q.Q4_K, 4096, 4096, 1)
    i2 = q.launch_info(q.Q6_K_SPLIT, 4096, 14336, 1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for i in (i1, i2):
        assert i["grid"] >= sms and i["stages"] >= 1 and i["threads"] % 32 == 0
        assert i["smem_bytes"] <= 232448


# ---- fused pack + mat-vec: the same bits as the two-call path -----------------------------------------
FUSED = [("q4k", 256, 2048, 1), ("q4k", 4096, 4096, 1), ("q6k", 4096, 14336, 1), ("q4k", 333, 2048, 4),
         ("q4k", 77, 4352, 5), ("q6k", 64, 3328, 4), ("q6k", 17, 14336, 8), ("q4k", 9, 32768, 1),
         ("q6k", 130, 1792, 3), ("q4k", 1000, 1280, 2), ("q5k", 4096, 4096, 1), ("q5k", 200, 2048, 3),
         ("q5k", 50, 14336, 8), ("q4k", 500, 2048, 8), ("q5k", 300, 4096, 6), ("q4k", 45, 3840, 5)]


@pytest.mark.parametrize("fmtname,rows,K,batch", FUSED)
def test_fused_equals_pack_then_matvec(fmtname, rows, K, batch):
    seed = 11 * rows + K + batch
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    xd = dev(x)
    if fmtname in ("q4k", "q5k"):
        W, Wa, f = dev(Wg.reshape(rows, -1)), None, QFMT[fmtname]
    else:
        W, Wa = q.bind_q6k(dev(Wg.reshape(rows, -1)), rows, K)
        f = q.Q6_K_SPLIT
    xq = q.q8k_pack(xd)
    y2 = q.qmatvec(f, W, Wa, xq, rows=rows)
    buf, y1 = poisoned_y(batch, rows)
    out = q.Q8K.empty(batch, K, DEV)
    q.qmatvec_x(f, W, Wa, xd, y1, rows=rows, xq_out=out)
    q.get_device_error()
    assert guard_intact(buf, batch, rows)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert torch.equal(out.qs, xq.qs) and torch.equal(out.bsums, xq.bsums)
    assert torch.equal(out.d.view(torch.int32), xq.d.view(torch.int32))
    check_against_oracle(fmtname, Wg, x, y1.cpu().numpy())


def test_fused_refusals():
    rows, K = 8, 512
    W = torch.zeros(rows * 2 * 144, dtype=torch.uint8, device=DEV)
    x = torch.zeros((1, K), dtype=torch.float32, device=DEV)
    buf, y = poisoned_y(1, rows)
    L = q.lib()
    none = q.Q8KPtrs(None, None, None)
    assert L.qmd_qmatvec_x(q.Q4_K, W.data_ptr(), None, None, none, y.data_ptr(), rows, K, 1, None) == 1
    assert L.qmd_qmatvec_x(q.Q4_K, W.data_ptr(), None, x.data_ptr() + 4, none, y.data_ptr(), rows, K, 1, None) == 5
    part = q.Q8KPtrs(x.data_ptr(), None, None)
    assert L.qmd_qmatvec_x(q.Q4_K, W.data_ptr(), None, x.data_ptr(), part, y.data_ptr(), rows, K, 1, None) == 1
    torch.cuda.synchronize()
    assert torch.isnan(y).all() and guard_intact(buf, 1, rows)


# ---- batches of 3..8 on the tensor cores: the same bits as the dp4a kernel -----------------------------
DP4A_ONLY = 2  # launch flag: keep batches of 5..8 on the dp4a kernel
TC_ALL = 4     # launch flag: every batch of 3..8 on the tensor-core kernel (long rows run by run)
SLICE = 8      # launch flag: the dp4a slice kernel instead of the row-lane one
RL = 16        # launch flag: the row-lane kernel for batches of 3 and 4 as well


# rows of one run of at most 16 blocks, and longer rows walked run by run: 17 blocks (a run of
# one block after a full one), one 16-row tile per CTA with 3 and 8 runs (the finishers of a
# tile's runs overlap), the 14336-wide down projection
TC_SHAPES = [(1000, 4096), (37, 256), (300, 2048), (17, 3840), (4099, 1280),
             (77, 4352), (16, 12288), (200, 14336), (33, 8192), (5, 32768)]


@pytest.mark.parametrize("fmtname", ["q4k", "q5k", "q6k"])
@pytest.mark.parametrize("batch", [5, 6, 7, 8])
@pytest.mark.parametrize("rows,K", TC_SHAPES)
def test_tensor_core_path_equals_dp4a_path(fmtname, batch, rows, K):
    seed = 3 * rows + K + batch
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    xq = gpu_pack(x)
    # the default plan: the tensor cores for Q4_K / Q5_K rows of at most 16 blocks and for rows
    # the dp4a kernel cannot take, the dp4a kernel otherwise
    default_tc = (fmtname != "q6k" and K <= 4096) or K > 16384
    assert (q.launch_kernel(QFMT[fmtname], rows, K, batch) == "qmv_tc_kernel") == default_tc
    q.debug_set_launch_flags(TC_ALL)
    try:
        info = q.launch_info(QFMT[fmtname], rows, K, batch)
        assert info["threads"] == 32 * min(K // 256, 16) and q.launch_kernel(QFMT[fmtname], rows, K, batch) == "qmv_tc_kernel"
        y_tc = run_matvec(fmtname, Wg, xq, rows, K, batch)
    finally:
        q.debug_set_launch_flags(0)
    if K <= 16384:  # the dp4a kernel's limit above two vectors
        q.debug_set_launch_flags(DP4A_ONLY)
        try:
            assert q.launch_kernel(QFMT[fmtname], rows, K, batch) == "qmv_kernel"
            y_dp = run_matvec(fmtname, Wg, xq, rows, K, batch)
        finally:
            q.debug_set_launch_flags(0)
        assert np.array_equal(y_tc.view(np.uint32), y_dp.view(np.uint32))
    idx = _sample_rows(rows, 96, seed)
    check_against_oracle(fmtname, Wg, x, y_tc, rows_idx=idx)


@pytest.mark.parametrize("batch", [3, 4])
@pytest.mark.parametrize("fmtname,rows,K", [("q4k", 9728, 4096), ("q4k", 28672, 4096), ("q5k", 19456, 2048),
                                            ("q4k", 10000, 4096), ("q4k", 6144, 4096)])
def test_tensor_cores_for_tall_tiles_at_three_and_four(fmtname, rows, K, batch):
    """Three and four vectors go to the tensor cores where 32-row tiles give every CTA at least
    64 rows and no more rows than 16-row tiles would (gate|up-like shapes), else to the dp4a
    kernel (q|k|v-like): the same bits either way."""
    seed = rows + K + batch
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    xq = gpu_pack(x)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas = sms * max(16 // min(K // 256, 16), 1)
    per_cta = lambda th: -(-(-(-rows // th)) // min(ctas, -(-rows // th))) * th  # whole tiles per CTA
    tall = per_cta(32) <= per_cta(16) and per_cta(32) >= 64
    kern = q.launch_kernel(QFMT[fmtname], rows, K, batch)
    assert kern == ("qmv_tc_kernel" if tall else "qmv_kernel")
    if tall and fmtname == "q4k":  # (Q5_K's two-slot rings of 32-row tiles do not fit: 16-row tiles)
        assert q.launch_info(QFMT[fmtname], rows, K, batch)["rows_per_stage"] == 32
    y = run_matvec(fmtname, Wg, xq, rows, K, batch)
    q.debug_set_launch_flags(DP4A_ONLY)
    try:
        assert q.launch_kernel(QFMT[fmtname], rows, K, batch) == "qmv_kernel"
        y_dp = run_matvec(fmtname, Wg, xq, rows, K, batch)
    finally:
        q.debug_set_launch_flags(0)
    assert np.array_equal(y.view(np.uint32), y_dp.view(np.uint32))
    check_against_oracle(fmtname, Wg, x, y, rows_idx=_sample_rows(rows, 64, seed))


@pytest.mark.parametrize("tile32", [False, True], ids=["tile16", "tile32"])
@pytest.mark.parametrize("fmtname,K", [("q4k", 4096), ("q5k", 4096), ("q5k", 2048), ("q4k", 8192),
                                       ("q6k", 4096), ("q6k", 14336)])
def test_tensor_core_extreme_magnitudes(fmtname, K, tile32):
    """The largest codes and scales against activations of +-127: the accumulator's partial
    sums reach their bound, and the integer dots must still be exact (Q6_K: scales -128 and
    127, codes 63 and 0, so a two-sub-block sum of scaled dots reaches 2 x 128 x 16 x 32 x 127).
    tile32: Q4_K / Q5_K rows of one run in 32-row tiles (a ring cap of 2), rows 0-31 in one tile
    (Q5_K's rings of 16 such tiles do not fit beside 16 warps' term slots: 8 blocks there)."""
    if tile32 and (fmtname == "q6k" or K > 4096 or (fmtname == "q5k" and K > 2048)):
        pytest.skip("16-row tiles only for this format and width")
    rows, batch = 48, 8
    Wg = synth.weights(fmtname, 77, rows, K).copy()
    if fmtname == "q6k":
        Wg[:, :, 0:192] = 0xFF             # ql, qh: every code 63 (q - 32 = 31)
        Wg[::2, :, 0:192] = 0x00           # even rows: every code 0 (q - 32 = -32)
        Wg[:, :, 192:208] = 0x80           # every scale -128
        Wg[1::4, :, 192:208] = 0x7F        # rows 1, 5, ...: every scale 127
    else:
        off = 48 if fmtname == "q5k" else 16
        Wg[:, :, 4:16] = 0xFF              # every scale and min 63
        Wg[:, :, off:] = 0xFF              # every nibble 15
        if fmtname == "q5k":
            Wg[:, :, 16:48] = 0xFF         # every fifth bit: codes 31
        Wg[::2, :, off:] = 0x00            # even rows: codes 0 (only the min term)
    x = np.ones((batch, K), np.float32)
    x[1::2] = -1.0                         # +-1 everywhere: codes +-127
    x[2, ::3] = -1.0                       # mixed signs
    x[4] = synth.activations(78, 1, K)[0]
    q.debug_set_launch_flags(TC_ALL)
    if tile32:
        q.debug_set_plan(0, 0, 2, 0)
    try:
        assert q.launch_kernel(QFMT[fmtname], rows, K, batch) == "qmv_tc_kernel"
        assert q.launch_info(QFMT[fmtname], rows, K, batch)["rows_per_stage"] == (32 if tile32 else 16)
        y = run_matvec(fmtname, Wg, gpu_pack(x), rows, K, batch)
        if fmtname == "q6k":
            body, prefix = q.bind_q6k(dev(Wg.reshape(rows, -1)), rows, K)
            yd, dots, sm = q.debug_qmatvec_dump(q.Q6_K_SPLIT, body, prefix, gpu_pack(x))
        else:
            yd, dots, sm = q.debug_qmatvec_dump(QFMT[fmtname], dev(Wg.reshape(rows, -1)), None, gpu_pack(x))
        q.get_device_error()
    finally:
        q.debug_set_launch_flags(0)
        q.debug_set_plan()
    check_against_oracle(fmtname, Wg, x, y)
    oqs, _, _ = O.q8k_pack(x)
    dots = dots.cpu().numpy()
    nsub = 16 if fmtname == "q6k" else 8
    for v in range(batch):
        for r in (0, 1, 2, 47):
            assert np.array_equal(dots[v, r][:, :nsub], O.subdots(OFMT[fmtname], Wg[r], oqs[v]))


# ---- several host threads, each with its own stream: the same bits as one thread ---------------------
def test_concurrent_host_threads():
    import threading
    shapes = [("q4k", 700, 4096, 1), ("q6k", 300, 14336, 1), ("q5k", 500, 2048, 6), ("q4k", 260, 1280, 3),
              ("q6k", 90, 3584, 2), ("q4k", 1000, 4096, 8)]
    jobs = []
    for i, (f, rows, K, batch) in enumerate(shapes):
        Wg = synth.weights(f, 60 + i, rows, K)
        if f == "q6k":
            W, Wa = q.bind_q6k(dev(Wg.reshape(rows, -1)), rows, K)
        else:
            W, Wa = dev(Wg.reshape(rows, -1)), None
        x = dev(synth.activations(60 + i, batch, K))
        ref = q.qmatvec_x(QFMT[f], W, Wa, x, rows=rows)
        jobs.append((QFMT[f], W, Wa, x, rows, ref))
    torch.cuda.synchronize()
    errors = []

    def work(job):
        f, W, Wa, x, rows, ref = job
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                outs = []
                for it in range(30):
                    if it % 2:
                        outs.append(q.qmatvec_x(f, W, Wa, x, rows=rows, stream=s))
                    else:
                        outs.append(q.qmatvec(f, W, Wa, q.q8k_pack(x, stream=s), rows=rows, stream=s))
            s.synchronize()
            for y in outs:
                if not torch.equal(y.view(torch.int32), ref.view(torch.int32)):
                    errors.append("differs")
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    q.get_device_error()
    assert not errors, errors[:3]


# ---- census: every kernel variant the library can launch, value-checked --------------------------------
CENSUS = [(f, b, fused, flags) for f in ("q4k", "q5k", "q6k") for b in range(1, 9) for fused in (False, True)
          for flags in ((0, DP4A_ONLY, TC_ALL) if b >= 5 else (0, TC_ALL, RL) if b >= 3 else (0, SLICE))]
_FLAG_ID = {0: "", DP4A_ONLY: "-dp4a", TC_ALL: "-tc", SLICE: "-slice", RL: "-rowlane"}


@pytest.mark.parametrize("fmtname,batch,fused,flags", CENSUS,
                         ids=[f"{f}-b{b}-{'fused' if fu else 'packed'}{_FLAG_ID[fl]}" for f, b, fu, fl in CENSUS])
def test_census_every_variant(fmtname, batch, fused, flags):
    """Each (format, batch, fused or packed input, kernel layout) the plan can choose, on a small
    ragged case, bit-identical to the same-order oracle; plus the recording variant's dots."""
    rows, K = 45, 1024
    seed = 1000 + 10 * batch + (3 if fused else 0)
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    xd = dev(x)
    if fmtname == "q6k":
        W, Wa = q.bind_q6k(dev(Wg.reshape(rows, -1)), rows, K)
    else:
        W, Wa = dev(Wg.reshape(rows, -1)), None
    q.debug_set_launch_flags(flags)
    try:
        buf, y = poisoned_y(batch, rows)
        if fused:
            q.qmatvec_x(QFMT[fmtname], W, Wa, xd, y, rows=rows)
        else:
            q.qmatvec(QFMT[fmtname], W, Wa, q.q8k_pack(xd), y, rows=rows)
        q.get_device_error()
        if not fused:
            _, dots, _ = q.debug_qmatvec_dump(QFMT[fmtname], W, Wa, q.q8k_pack(xd), rows)
            q.get_device_error()
    finally:
        q.debug_set_launch_flags(0)
    assert guard_intact(buf, batch, rows)
    check_against_oracle(fmtname, Wg, x, y.cpu().numpy())
    if not fused:
        oqs, _, _ = O.q8k_pack(x)
        d = dots.cpu().numpy()
        per = 16 if fmtname == "q6k" else 8
        for v in range(batch):
            assert np.array_equal(d[v, rows - 1][:, :per], O.subdots(OFMT[fmtname], Wg[rows - 1], oqs[v]))


# ---- a seeded random sweep of small shapes (stands in for a property-based sweep) -------------------------
def _random_cases(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        f = ("q4k", "q5k", "q6k")[i % 3]
        nb = int(rng.choice([1, 1, 2, 3, 5, 8, 13, 16, 17, 31, 40, 56]))
        rows = int(rng.integers(1, 300))
        batch = int(rng.integers(1, 9))
        out.append((f, rows, 256 * nb, batch, bool(rng.integers(0, 2)), int(rng.integers(0, 1 << 20))))
    return out


@pytest.mark.parametrize("fmtname,rows,K,batch,fused,seed", _random_cases())
def test_random_small_shapes(fmtname, rows, K, batch, fused, seed):
    if 2 < batch < 5 and K > 16384:
        pytest.skip("above the batch's K limit")
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    xd = dev(x)
    if fmtname == "q6k":
        W, Wa = q.bind_q6k(dev(Wg.reshape(rows, -1)), rows, K)
    else:
        W, Wa = dev(Wg.reshape(rows, -1)), None
    buf, y = poisoned_y(batch, rows)
    if fused:
        q.qmatvec_x(QFMT[fmtname], W, Wa, xd, y, rows=rows)
    else:
        q.qmatvec(QFMT[fmtname], W, Wa, q.q8k_pack(xd), y, rows=rows)
    q.get_device_error()
    assert guard_intact(buf, batch, rows)
    check_against_oracle(fmtname, Wg, x, y.cpu().numpy())


# ---- the scheduling workspace: the last tiles handed out by claims, the same bits -------------------
WS_SHAPES = [("q4k", 4096, 4096, 1, False), ("q4k", 28672, 4096, 1, True), ("q6k", 4096, 14336, 1, True),
             ("q6k", 333, 14336, 2, False), ("q5k", 1000, 2048, 2, True), ("q4k", 7, 256, 1, True),
             ("q4k", 150, 8192, 2, False), ("q6k", 9, 65536, 1, False)]


@pytest.mark.parametrize("fmtname,rows,K,batch,fused", WS_SHAPES)
@pytest.mark.parametrize("per_mille", [-1, 0, 500, 1000], ids=["default", "none", "half", "all"])
@pytest.mark.parametrize("warps", [0, 1, 3], ids=["plan", "w1", "w3"])
def test_workspace_same_bits(fmtname, rows, K, batch, fused, per_mille, warps):
    """qmd_qmatvec_ws / qmd_qmatvec_x_ws: bit-identical to the calls without a workspace and to the
    same-order oracle, three calls in a row on one workspace, which each call leaves zeroed.  Claims
    are used at one vector where every warp has two tiles of its own: the 28672-row shape on the
    default plan, and most one-vector shapes once the plan is forced to one or three warps per CTA."""
    seed = 7 * rows + K + batch
    Wg = synth.weights(fmtname, seed, rows, K)
    x = synth.activations(seed, batch, K)
    xd = dev(x)
    if fmtname == "q6k":
        W, Wa = q.bind_q6k(dev(Wg.reshape(rows, -1)), rows, K)
    else:
        W, Wa = dev(Wg.reshape(rows, -1)), None
    xq = q.q8k_pack(xd)
    ref = q.qmatvec(QFMT[fmtname], W, Wa, xq, rows=rows)
    ws = q.workspace(DEV)
    q.debug_set_dynamic_tiles(per_mille)
    q.debug_set_plan(warps, 0, 2 if warps else 0, 0)
    try:
        for _ in range(3):
            buf, y = poisoned_y(batch, rows)
            if fused:
                q.qmatvec_x(QFMT[fmtname], W, Wa, xd, y, rows=rows, workspace=ws)
            else:
                q.qmatvec(QFMT[fmtname], W, Wa, xq, y, rows=rows, workspace=ws)
            q.get_device_error()
            assert guard_intact(buf, batch, rows)
            assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
            assert int(ws.abs().sum()) == 0, "workspace not left zeroed"
    finally:
        q.debug_set_dynamic_tiles(-1)
        q.debug_set_plan()
    check_against_oracle(fmtname, Wg, x, ref.cpu().numpy(), f64_idx=_sample_rows(rows, min(rows, 200), seed))


def test_workspace_streams_in_parallel():
    """Two streams, each with its own workspace, chains of launches running at the same time: the
    same bits as one stream, and both workspaces left zeroed."""
    rows, K = 28672, 4096
    Wg = synth.q4k_weights(44, rows, K)
    W = dev(Wg.reshape(rows, -1))
    xs = [dev(synth.activations(45 + i, 1, K)) for i in range(2)]
    refs = [q.qmatvec_x(q.Q4_K, W, None, x, rows=rows) for x in xs]
    streams = [torch.cuda.Stream() for _ in range(2)]
    wss = [q.workspace(DEV) for _ in range(2)]
    ys = [[torch.empty((1, rows), dtype=torch.float32, device=DEV) for _ in range(6)] for _ in range(2)]
    torch.cuda.synchronize()
    for k in range(6):
        for i in range(2):
            q.qmatvec_x(q.Q4_K, W, None, xs[i], ys[i][k], rows=rows, stream=streams[i], workspace=wss[i])
    torch.cuda.synchronize()
    q.get_device_error()
    for i in range(2):
        assert int(wss[i].abs().sum()) == 0
        for k in range(6):
            assert torch.equal(ys[i][k].view(torch.int32), refs[i].view(torch.int32))


def test_workspace_refusals_write_nothing():
    L = q.lib()
    rows, K = 64, 1024
    W = dev(synth.q4k_weights(1, rows, K).reshape(rows, -1))
    xq = q.q8k_pack(dev(synth.activations(1, 1, K)))
    buf, y = poisoned_y(1, rows)
    ws = q.workspace(DEV)
    assert L.qmd_qmatvec_ws(q.Q4_K, W.data_ptr(), None, xq.ptrs(), y.data_ptr(), rows, K, 1, None, None) == 1
    assert L.qmd_qmatvec_ws(q.Q4_K, W.data_ptr(), None, xq.ptrs(), y.data_ptr(), rows, K, 1,
                            ws.data_ptr() + 4, None) == 5
    x = dev(synth.activations(1, 1, K))
    none = q.Q8KPtrs(None, None, None)
    assert L.qmd_qmatvec_x_ws(q.Q4_K, W.data_ptr(), None, x.data_ptr(), none, y.data_ptr(), rows, K, 1, None,
                              None) == 1
    torch.cuda.synchronize()
    assert torch.isnan(y).all() and guard_intact(buf, 1, rows) and int(ws.abs().sum()) == 0


def test_bind_then_matvec_in_one_stream_without_a_host_sync():
    """qmd_bind_q6k writes the split bodies and prefix with an ordinary launch; a mat-vec launched
    right after it in the same stream, as a programmatic dependent, starts reading weights before
    its dependency wait.  The bind kernel signals completion only by exiting, so the mat-vec must
    still see the final weights: checked with the destination buffers filled with other bytes
    first, the bind and the mat-vec back to back with no host synchronisation, three times."""
    rows, K = 4096, 14336
    nb = K // 256
    Wg = synth.q6k_weights(91, rows, K)
    g = dev(Wg.reshape(rows, -1))
    x = synth.activations(92, 1, K)
    xd = dev(x)
    s = torch.cuda.Stream()
    for fill in (0xA5, 0x00, 0xFF):
        body = torch.full((rows, nb * 208), fill, dtype=torch.uint8, device=DEV)
        prefix = torch.full((rows, q.q6k_prefix_stride(K)), -1 if fill == 0xFF else fill, dtype=torch.int16,
                            device=DEV)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            q.bind_q6k(g, rows, K, body=body, prefix=prefix, stream=s)
            y = q.qmatvec_x(q.Q6_K_SPLIT, body, prefix, xd, rows=rows, stream=s)
        torch.cuda.synchronize()
        q.get_device_error()
        check_against_oracle("q6k", Wg, x, y.cpu().numpy(), f64_idx=_sample_rows(rows, 200, fill))
