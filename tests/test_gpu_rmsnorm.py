"""RMSNorm (+ residual add) fused into the q8_K pack: GPU vs the oracle, through the C ABI.

Bar: h, the packed codes, scales and sub-block sums bit-exact (the codes are integers decided
by f32 arithmetic, which both sides do in the same declared order)."""
import ctypes

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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from quantised_decode_mat_gb300 import build as qbuild
    qbuild.build()
    q.lib()
    yield


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def check_pack(xq, h_gpu, x, r, g, eps, h_written):
    oh, oqs, od, obs = O.rmsnorm_q8k_pack(x, r, g, eps)
    assert np.array_equal(xq.qs.cpu().numpy(), oqs)
    assert np.array_equal(xq.d.cpu().numpy().view(np.uint32), od.view(np.uint32))
    assert np.array_equal(xq.bsums.cpu().numpy(), obs)
    if h_written:
        assert np.array_equal(h_gpu.cpu().numpy().view(np.uint32), oh.view(np.uint32))


CASES = [(1, 256, True, 1e-6), (1, 4096, True, 1e-5), (2, 14336, True, 1e-6), (8, 4096, False, 1e-6),
         (3, 768, True, 0.0), (5, 2304, False, 0.5), (4, 16384, True, 1e-5), (1, 1280, False, 1e-6),
         # wider than 16384: h is not kept in shared memory, phase 2 re-reads or recomputes it
         (2, 16640, True, 1e-6), (3, 32768, False, 1e-6), (1, 65536, True, 1e-5)]


@pytest.mark.parametrize("batch,K,with_r,eps", CASES)
@pytest.mark.parametrize("h_mode", ["none", "separate", "in_place_r", "in_place_x"])
def test_rmsnorm_pack_bit_exact(batch, K, with_r, eps, h_mode):
    seed = 31 * K + batch
    x = synth.activations(seed, batch, K)
    r = synth.residual(seed, batch, K) if with_r else None
    g = synth.norm_gain(seed, K)
    xd, gd = dev(x), dev(g)
    rd = dev(r) if with_r else None
    if h_mode == "none":
        h = None
    elif h_mode == "separate":
        h = torch.full((batch, K), float("nan"), device=DEV)
    elif h_mode == "in_place_r":
        if not with_r:
            pytest.skip("no residual buffer")
        h = rd
    else:
        h = xd
    xq = q.rmsnorm_q8k_pack(xd, rd, gd, eps, h_out=h)
    q.get_device_error()
    check_pack(xq, h, x, r, g, eps, h is not None)


def test_rmsnorm_pack_special_values():
    K = 1024
    # one square of 2^24 among squares of 1: the declared order's total is 2^24 + 1020
    x = np.ones((1, K), np.float32)
    x[0, 0] = np.float32(4096.0)
    g = np.ones(K, np.float32)
    xq = q.rmsnorm_q8k_pack(dev(x), None, dev(g), 0.0)
    check_pack(xq, None, x, None, g, 0.0, False)
    # zero gain, all-zero input (eps keeps the norm finite), huge and tiny magnitudes
    x2 = synth.activations(7, 4, K)
    x2[1] = 0.0
    x2[2] *= np.float32(1e30)
    x2[3] *= np.float32(1e-30)
    g2 = synth.norm_gain(7, K)
    g2[:256] = 0.0
    xq2 = q.rmsnorm_q8k_pack(dev(x2), None, dev(g2), 1e-6)
    check_pack(xq2, None, x2, None, g2, 1e-6, False)
    assert not xq2.qs[:, :256].any() and not xq2.d[:, 0].any()


def test_rmsnorm_pack_refusals_write_nothing():
    K, B = 512, 2
    x = torch.zeros((B, K), device=DEV)
    g = torch.ones(K, device=DEV)
    xq = q.Q8K(torch.full((B, K), 7, dtype=torch.int8, device=DEV), torch.full((B, 2), 7.0, device=DEV),
               torch.full((B, 2, 8), 7, dtype=torch.int16, device=DEV))
    L = q.lib()
    f = L.qmd_rmsnorm_q8k_pack
    p = xq.ptrs()
    assert f(x.data_ptr(), None, g.data_ptr(), ctypes.c_float(-1.0), None, p, K, B, None) == 10
    assert f(x.data_ptr(), None, g.data_ptr(), ctypes.c_float(float("nan")), None, p, K, B, None) == 10
    assert f(x.data_ptr(), None, g.data_ptr(), ctypes.c_float(float("inf")), None, p, K, B, None) == 10
    assert f(None, None, g.data_ptr(), 1e-6, None, p, K, B, None) == 1
    assert f(x.data_ptr(), None, None, 1e-6, None, p, K, B, None) == 1
    assert f(x.data_ptr(), None, g.data_ptr(), 1e-6, None, p, 500, B, None) == 3
    assert f(x.data_ptr(), None, g.data_ptr(), 1e-6, None, p, K, 9, None) == 4
    assert f(x.data_ptr(), None, g.data_ptr() + 4, 1e-6, None, p, K, B, None) == 5
    assert f(x.data_ptr(), x.data_ptr() + 8, g.data_ptr(), 1e-6, None, p, K, B, None) == 5
    assert f(x.data_ptr(), None, g.data_ptr(), 1e-6, x.data_ptr() + 4, p, K, B, None) == 5
    torch.cuda.synchronize()
    assert (xq.qs == 7).all() and (xq.d == 7.0).all() and (xq.bsums == 7).all()
    assert q.status_str(10) == "QMD_ERR_VALUE"
