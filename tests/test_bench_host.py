"""Host-side pieces of bench.py and the decode step's byte accounting (no GPU needed)."""
import argparse

import bench
from quantised_decode_mat_gb300 import synth
from quantised_decode_mat_gb300.step import Projection, fuse_pack


def _args(**kw):
    base = dict(batch=1, fused=False, unfused=False, layers=32, gpus=1)
    base.update(kw)
    return argparse.Namespace(**base)


def test_pack_is_fused_for_one_vector_and_short_rows_unless_asked():
    assert bench.use_fused(_args(batch=1)) is None  # the per-projection default
    assert bench.use_fused(_args(batch=4, fused=True)) is True
    assert bench.use_fused(_args(batch=1, unfused=True)) is False
    assert fuse_pack(1, 4096) and fuse_pack(1, 14336) and fuse_pack(2, 4096) and fuse_pack(2, 14336)
    assert not fuse_pack(3, 4096) and not fuse_pack(4, 14336) and not fuse_pack(8, 256)


def test_workload_config_names_the_step():
    c = bench.workload_config(_args(batch=4))
    assert c["workload"] == "decode_step_7b_q4k_q6k_32layers_b4" and c["batch"] == 4 and c["layers"] == 32
    assert c["launch"] == "pack+mat-vec as two kernels"
    assert c["projections"] == ["qkv:q4k:6144x4096", "o:q4k:4096x4096", "gate_up:q4k:28672x4096",
                                "down:q6k:4096x14336"]
    assert bench.workload_config(_args(batch=1))["launch"] == (
        "pack fused into the mat-vec (one kernel per projection)")
    assert bench.workload_config(_args(batch=1, fused=True))["launch"] == (
        "pack fused into the mat-vec (one kernel per projection)")
    assert bench.workload_config(_args(batch=1, unfused=True))["launch"] == "pack+mat-vec as two kernels"


def test_step_bytes_match_the_workload_table():
    """Weights of one 7B-shaped layer (GGUF block sizes) and the algorithmic bytes per step at
    batch 1: 4,410,310,656 weight bytes and 4,419,223,552 algorithmic bytes over 32 layers."""
    layer_w = sum(rows * (K // 256) * (144 if f == "q4k" else 210) for (_, f, rows, K) in synth.STEP_PROJECTIONS)
    assert 32 * layer_w == 4_410_310_656
    alg = 0
    for (_, f, rows, K) in synth.STEP_PROJECTIONS:
        nb = K // 256
        w = rows * nb * 144 if f == "q4k" else rows * nb * 208 + rows * ((nb + 7) // 8 * 8) * 2
        alg += w + 4 * K + 4 * rows
    assert 32 * alg == 4_419_223_552


class _Q8:
    def __init__(self, batch):
        self.batch = batch


def test_projection_byte_accounting():
    p = Projection("o", 0, 12, 4096, 4096, None, None, None, _Q8(2), None, 4096 * 16 * 144)
    assert p.act_bytes() == 2 * 16 * 276
    assert p.matvec_bytes() == 4096 * 16 * 144 + 2 * 16 * 276 + 2 * 4096 * 4
    assert p.algorithmic_bytes() == 4096 * 16 * 144 + 2 * 4096 * 4 + 2 * 4096 * 4
    assert p.pack_bytes() == 2 * 4096 * 4 + 2 * (4096 + 16 * 4 + 16 * 16)


def test_traffic_figures_are_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    f = tmp_path / "traffic.txt"
    f.write_text(f"source_hash: {bench.kernel_source_hash()}\nqmv_q4k_dram_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(f))
    assert bench.profiled_traffic("qmv_q4k") == 123.0
    assert bench.profiled_traffic("qmv_q6k") is None
    f.write_text("source_hash: 0000\nqmv_q4k_dram_bytes_per_launch: 123\n")
    assert bench.profiled_traffic("qmv_q4k") is None


def test_cpu_model_is_a_name():
    m = bench.cpu_model()
    assert isinstance(m, str) and m.strip()
