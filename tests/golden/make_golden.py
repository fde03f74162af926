"""Writes tests/golden/oracle_regression.txt: oracle outputs on small seeded cases.

Calls only the oracle and the seeded input generator.  The stored values pin the oracle
against accidental change: a deliberate change to its arithmetic rewrites this file, and the
commit that does so names the passage (or reading of it) that justifies the change.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
from quantised_decode_mat_gb300 import synth  # noqa: E402


def _hex(a):
    return [format(int(v), "08x") for v in np.ascontiguousarray(a).view(np.uint32).reshape(-1)]


def compute():
    out = {}
    x = synth.activations(100, 2, 1024)
    qs, xd, bs = O.q8k_pack(x)
    out["q8k_d"] = _hex(xd)
    out["q8k_qs_sum_by_block"] = [format(int(s) & 0xFFFFFFFF, "08x") for s in qs.astype(np.int64).reshape(2, 4, 256).sum(-1).reshape(-1)]
    for name, fmt in (("q4k", O.FMT_Q4_K), ("q6k", O.FMT_Q6_K)):
        W = synth.weights(name, 100, 6, 1024)
        out[f"{name}_y_seq"] = _hex(O.qmatvec(fmt, W, qs, xd, bs, O.ORDER_SEQUENTIAL))
        out[f"{name}_y_grp4"] = _hex(O.qmatvec(fmt, W, qs, xd, bs, O.ORDER_GROUPS_OF_FOUR))
        out[f"{name}_dots_r0_v0"] = _hex(O.subdots(fmt, W[0], qs[0]).astype(np.int32))
    W5 = synth.weights("q5k", 100, 6, 1024)
    out["q5k_y_run16"] = _hex(O.qmatvec(O.FMT_Q5_K, W5, qs, xd, bs, O.ORDER_RUNS_OF_SIXTEEN))
    out["q5k_dots_r0_v0"] = _hex(O.subdots(O.FMT_Q5_K, W5[0], qs[0]).astype(np.int32))
    W6 = synth.weights("q6k", 101, 3, 5120)  # 20 blocks: two runs of sixteen
    x6 = synth.activations(101, 1, 5120)
    q6, d6, b6 = O.q8k_pack(x6)
    out["q6k_y_run16_nb20"] = _hex(O.qmatvec(O.FMT_Q6_K, W6, q6, d6, b6, O.ORDER_RUNS_OF_SIXTEEN))
    xr = synth.activations(102, 1, 512)
    rr = synth.residual(102, 1, 512)
    gr = synth.norm_gain(102, 512)
    h, n = O.rmsnorm(xr, rr, gr, 1e-6)
    out["rmsnorm_n_first16"] = _hex(n[0, :16])
    _, rq, rd, rb = O.rmsnorm_q8k_pack(xr, rr, gr, 1e-6)
    out["rmsnorm_pack_d"] = _hex(rd)
    out["rmsnorm_pack_bsums"] = [format(int(v) & 0xFFFF, "04x") for v in rb.reshape(-1)]
    return out


def main():
    path = os.path.join(HERE, "oracle_regression.txt")
    with open(path, "w") as f:
        f.write("# oracle outputs on seeded cases (f32/int32 bit patterns, hex); written by make_golden.py\n")
        for k, v in compute().items():
            f.write(f"{k}: {' '.join(v)}\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
