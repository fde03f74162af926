"""The build's spill gate: it reads ptxas -v logs and refuses a build in which a product kernel
instance spills registers to local memory; the test-only recording variant is the one exemption."""
import pytest

from quantised_decode_mat_gb300 import build as qbuild

LOG = """ptxas info    : Compiling entry function '_ZN3qmd10qmv_kernelILi12ELi1ELi8ELi2EEEvNS_10QmvKParamsE' for 'sm_103a'
ptxas info    : Function properties for _ZN3qmd10qmv_kernelILi12ELi1ELi8ELi2EEEvNS_10QmvKParamsE
    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads
ptxas info    : Used 56 registers, used 1 barriers, 1104 bytes cmem[0]
ptxas info    : Compiling entry function '_ZN3qmd10qmv_kernelILi14ELi7ELi2ELi1EEEvNS_10QmvKParamsE' for 'sm_103a'
ptxas info    : Function properties for _ZN3qmd10qmv_kernelILi14ELi7ELi2ELi1EEEvNS_10QmvKParamsE
    16 bytes stack frame, 16 bytes spill stores, 28 bytes spill loads
ptxas info    : Used 128 registers, used 1 barriers, 1104 bytes cmem[0]
"""

SPILL_PRODUCT = """ptxas info    : Compiling entry function '_ZN3qmd13qmv_rl_kernelILi12ELi1ELi2EEEvNS_8RlParamsE' for 'sm_103a'
ptxas info    : Function properties for _ZN3qmd13qmv_rl_kernelILi12ELi1ELi2EEEvNS_8RlParamsE
    8 bytes stack frame, 4 bytes spill stores, 4 bytes spill loads
ptxas info    : Used 120 registers, used 2 barriers, 1104 bytes cmem[0]
"""


def test_spills_are_read_per_entry_function():
    s = qbuild.spills(LOG)
    assert s == [("_ZN3qmd10qmv_kernelILi14ELi7ELi2ELi1EEEvNS_10QmvKParamsE", 16, 28)]


def test_only_the_recording_variant_is_exempt():
    # mode is template argument 3 of qmv_kernel, 1 of qmv_tc_kernel, 2 of qmv_rl_kernel; 1 records
    assert qbuild.spill_exempt("_ZN3qmd10qmv_kernelILi14ELi7ELi2ELi1EEEvNS_10QmvKParamsE")
    assert not qbuild.spill_exempt("_ZN3qmd10qmv_kernelILi14ELi7ELi2ELi2EEEvNS_10QmvKParamsE")
    assert qbuild.spill_exempt("_ZN3qmd13qmv_tc_kernelILi12ELi1ELi3ELb1EEEvNS_8TcParamsE")
    assert not qbuild.spill_exempt("_ZN3qmd13qmv_tc_kernelILi12ELi2ELi3ELb1EEEvNS_8TcParamsE")
    assert qbuild.spill_exempt("_ZN3qmd13qmv_rl_kernelILi14ELi2ELi1EEEvNS_8RlParamsE")
    assert not qbuild.spill_exempt("_ZN3qmd13qmv_rl_kernelILi12ELi1ELi2EEEvNS_8RlParamsE")
    assert not qbuild.spill_exempt("_ZN3qmd15q8k_pack_kernelEPKfPaPfPsl")


def test_gate_refuses_a_spilling_product_instance(tmp_path, monkeypatch):
    monkeypatch.setattr(qbuild, "UNITS", ("a", "b"))
    (tmp_path / "a.log").write_text(LOG)
    qbuild.check_spills(str(tmp_path))  # only the exempt recording variant spills
    (tmp_path / "b.log").write_text(SPILL_PRODUCT)
    with pytest.raises(RuntimeError, match="qmv_rl_kernel"):
        qbuild.check_spills(str(tmp_path))


def test_current_build_has_no_spilling_product_instance():
    """The logs of the library as built here (if it has been built) pass the gate."""
    import os
    if not os.path.isdir(qbuild.BUILD):
        pytest.skip("library not built")
    qbuild.check_spills(qbuild.BUILD)
