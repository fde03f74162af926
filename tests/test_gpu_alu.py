"""qmd_measure_alu: the issue-rate microbenchmarks behind the ALU roofline give plausible rates."""
import pytest

torch = pytest.importorskip("torch")

import quantised_decode_mat_gb300 as q  # noqa: E402

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU"),
]


def test_measure_alu_rates_are_plausible():
    from quantised_decode_mat_gb300 import build as qbuild
    qbuild.build()
    dp4a, mma = q.measure_alu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # at least one dp4a per SM per microsecond and at most 512 per SM per clock at 3 GHz
    assert sms * 1e6 < dp4a < sms * 512 * 3e9
    # the f16 tensor path: above 10 TFLOP/s, below 10 PFLOP/s
    assert 1e13 < mma < 1e16
    d2, m2 = q.measure_alu()  # repeatable within a factor of two
    assert 0.5 < d2 / dp4a < 2 and 0.5 < m2 / mma < 2
