"""The decode step's host-buffer form (inputs copied in, outputs copied out, overlapped with the
mat-vecs on side streams) gives the same bits as the device-resident step."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import quantised_decode_mat_gb300 as q  # noqa: E402

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]


@pytest.fixture(scope="module")
def step():
    from quantised_decode_mat_gb300 import build as qbuild
    from quantised_decode_mat_gb300 import step as qstep
    qbuild.build()
    q.lib()
    return qstep.make_step(1, layers=3, device="cuda")


def _reference(step):
    step.run()
    torch.cuda.synchronize()
    return step.y_all.clone()


@pytest.mark.parametrize("chunks", [1, 2, 4])
def test_through_host_matches_device_step(step, chunks):
    ref = _reference(step)
    x_host = torch.empty(step.x_all.shape, dtype=torch.float32, pin_memory=True)
    x_host.copy_(step.x_all)
    x_keep = step.x_all.clone()
    y_host = torch.full(step.y_all.shape, float("nan"), dtype=torch.float32, pin_memory=True)
    step.x_all.fill_(float("nan"))
    step.y_all.fill_(float("nan"))
    step.run_through_host(x_host, y_host, chunks=chunks)
    torch.cuda.synchronize()
    q.get_device_error()
    assert torch.equal(step.x_all, x_keep)
    # every output row came back, bit for bit (padding between projections is not compared)
    for p in step.projs:
        off = p.y.data_ptr() - step.y_all.data_ptr()
        n = p.y.numel()
        got = y_host[off // 4: off // 4 + n].numpy().view(np.uint32)
        want = ref[off // 4: off // 4 + n].cpu().numpy().view(np.uint32)
        assert np.array_equal(got, want), p.name


def test_through_host_in_a_graph(step):
    ref = _reference(step)
    x_host = torch.empty(step.x_all.shape, dtype=torch.float32, pin_memory=True)
    x_host.copy_(step.x_all)
    y_host = torch.zeros(step.y_all.shape, dtype=torch.float32, pin_memory=True)
    g = step.capture(lambda: step.run_through_host(x_host, y_host))
    y_host.zero_()
    step.y_all.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for p in step.projs:
        off = (p.y.data_ptr() - step.y_all.data_ptr()) // 4
        assert torch.equal(y_host[off: off + p.y.numel()], ref[off: off + p.y.numel()].cpu()), p.name
