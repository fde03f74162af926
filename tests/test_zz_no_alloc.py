"""qmd_qmatvec_x_static: the mat-vec for callers that cannot allocate device memory (a plug-in
whose host framework hands it only its inputs and outputs), whose scheduling workspace is the
library's own static device array.  Checked through the C ABI against qmd_qmatvec_x, the
existing entry point, bit for bit (the tolerance every other GPU test uses here is exact
equality with the same-order result), on two calls in a row -- the array keeps what the first
call left, and the second must still give the same bits.  This file is collected last."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import quantised_decode_mat_gb300 as q  # noqa: E402
from quantised_decode_mat_gb300 import synth  # noqa: E402

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]

# (format, rows, K, batch): the fused gate|up shape, on which the workspace hands out tiles, and
# smaller shapes of every format on which it does not
CASES = [("q4k", 28672, 4096, 1), ("q6k", 4096, 14336, 1), ("q5k", 333, 2048, 2), ("q4k", 7, 256, 1)]


@pytest.mark.parametrize("fmtname,rows,K,batch", CASES)
def test_static_workspace_call_matches_qmatvec_x(fmtname, rows, K, batch):
    from quantised_decode_mat_gb300 import build as qbuild
    qbuild.build()
    L = q.lib()
    q.debug_set_plan()
    q.debug_set_launch_flags(0)
    dev = torch.device("cuda")
    fmt = {"q4k": q.Q4_K, "q5k": q.Q5_K, "q6k": q.Q6_K_SPLIT}[fmtname]
    seed = rows + K + batch
    Wg = synth.weights(fmtname, seed, rows, K)
    g = torch.from_numpy(np.ascontiguousarray(Wg.reshape(rows, -1))).to(dev)
    if fmtname == "q6k":
        W, Wa = q.bind_q6k(g, rows, K)
    else:
        W, Wa = g, None
    x = torch.from_numpy(synth.activations(seed, batch, K)).to(dev)
    none = q.Q8KPtrs(None, None, None)
    ref = torch.full((batch, rows), float("nan"), dtype=torch.float32, device=dev)
    st = L.qmd_qmatvec_x(fmt, W.data_ptr(), None if Wa is None else Wa.data_ptr(), x.data_ptr(), none,
                         ref.data_ptr(), rows, K, batch, None)
    assert st == 0, q.status_str(st)
    for _ in range(2):
        y = torch.full((batch, rows), float("nan"), dtype=torch.float32, device=dev)
        st = L.qmd_qmatvec_x_static(fmt, W.data_ptr(), None if Wa is None else Wa.data_ptr(), x.data_ptr(), none,
                                    y.data_ptr(), rows, K, batch, None)
        assert st == 0, q.status_str(st)
        torch.cuda.synchronize()
        assert torch.isfinite(y).all()
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
    q.get_device_error()
