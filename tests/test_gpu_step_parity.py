"""The 7B-shaped decode step at full size, in the launch forms bench.py times (step.fuse_pack
decides, per projection and batch, between the pack fused into the mat-vec and a stand-alone
pack; batch 8 runs the 4096-wide projections on the tensor cores), against the oracle: layer 0's
four projections on every row (the oracle threaded over rows), layer 1's q|k|v and o on every
row and its gate|up and down on the rows at every CTA boundary of the plans the kernels may take
plus a random sample; the f64 brute force on sampled rows."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as O  # noqa: E402
import quantised_decode_mat_gb300 as q  # noqa: E402
from tests.oracle_rows import oracle_rows_threaded  # noqa: E402

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

TOL_SAME_ORDER = 1e-5
TOL_F64 = 2e-3
OFMT = {q.Q4_K: O.FMT_Q4_K, q.Q6_K_SPLIT: O.FMT_Q6_K}


@pytest.fixture(scope="module", params=[(1, 0), (4, 0), (8, 0), (1, 2), (1, 4)],
                ids=["b1", "b4", "b8", "b1-splitk2", "b1-splitk4"])
def step(request):
    """The 2-layer step at one batch; the split-K cases run every projection of it split over
    clusters of 2 or 4 CTAs (qmd_debug_set_split_k)."""
    from quantised_decode_mat_gb300 import build as qbuild
    from quantised_decode_mat_gb300 import step as qstep
    qbuild.build()
    q.lib()
    q.debug_set_plan()
    q.debug_set_launch_flags(0)
    batch, ks = request.param
    q.debug_set_split_k(ks)
    try:
        s = qstep.make_step(batch, layers=2, device="cuda", keep_host_layers=(0, 1))
        if ks:
            assert all(q.launch_kernel(p.fmt, p.rows, p.K, batch) == "qmv_sk_kernel" for p in s.projs)
        s.y_all.fill_(float("nan"))
        s.run()
        torch.cuda.synchronize()
        q.get_device_error()
    finally:
        q.debug_set_split_k(0)
    return s


def _rows_to_check(p, batch):
    if p.rows <= 6144 or p.layer == 0:
        return None
    rng = np.random.default_rng(p.rows + 7 * batch + p.layer)
    pick = set(rng.choice(p.rows, size=500, replace=False).tolist()) | {0, 1, p.rows - 2, p.rows - 1}
    G = q.launch_info(p.fmt, p.rows, p.K, batch)["grid"]
    tiles = (p.rows + 15) // 16
    for g in (G, 152, 304, 456, 608):  # the plan's grid and the grids the fused plans may take
        pick |= {(p.rows * b) // g for b in range(g)} | {(p.rows * b) // g - 1 for b in range(1, g)}
        # the tensor-core kernel splits whole 16-row tiles, the row-lane kernel whole 2-row tiles
        pick |= {16 * ((tiles * b) // g) for b in range(g)} | {16 * ((tiles * b) // g) - 1 for b in range(1, g)}
        t2 = (p.rows + 1) // 2
        pick |= {2 * ((t2 * b) // g) for b in range(g)} | {2 * ((t2 * b) // g) - 1 for b in range(1, g)}
    return np.array(sorted(r for r in pick if 0 <= r < p.rows))


def test_launch_forms_are_the_benched_ones(step):
    from quantised_decode_mat_gb300.step import fuse_pack
    for p in step.projs:
        assert p.fused == fuse_pack(step.batch, p.K)
    if step.batch == 1:
        assert [p.fused for p in step.projs[:4]] == [True, True, True, True]


@pytest.mark.parametrize("index", range(8), ids=[f"L{i // 4}-{n}" for i, n in
                                                  enumerate(["qkv", "o", "gate_up", "down"] * 2)])
def test_step_projection_matches_oracle(step, index):
    from quantised_decode_mat_gb300 import step as qstep
    p = step.projs[index]
    Wg = step.host_weights[(p.layer, p.name)]
    x = qstep.host_activation(step, p)
    y = p.y.cpu().numpy()
    idx = _rows_to_check(p, step.batch)
    oqs, od, obs = O.q8k_pack(x)
    W = Wg if idx is None else Wg[idx]
    yg = y if idx is None else y[:, idx]
    assert np.isfinite(yg).all(), "unwritten (NaN) outputs"
    ref = oracle_rows_threaded(OFMT[p.fmt], W, oqs, od, obs, O.ORDER_RUNS_OF_SIXTEEN)
    assert O.rel_err(yg, ref).max() <= TOL_SAME_ORDER
    assert np.count_nonzero(yg.view(np.uint32) != ref.view(np.uint32)) == 0
    s64 = np.random.default_rng(p.rows + p.layer).choice(W.shape[0], size=min(W.shape[0], 600), replace=False)
    assert O.rel_err(yg[:, s64], O.qmatvec_f64(OFMT[p.fmt], W[s64], oqs, od)).max() <= TOL_F64
    if not p.fused:  # the stand-alone pack's output, bit for bit
        assert np.array_equal(p.xq.qs.cpu().numpy().reshape(oqs.shape), oqs)
        assert np.array_equal(p.xq.d.cpu().numpy().reshape(od.shape).view(np.uint32), od.view(np.uint32))
        assert np.array_equal(p.xq.bsums.cpu().numpy().reshape(obs.shape), obs)
