"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test below checks the oracle against something it does not compute itself: a library
routine (numpy's float16), values worked by hand from the block formats (tests/golden/),
bijections the formats imply, invariants of the q8_K pack, closed forms of special blocks,
and brute force in f64.  A plausible slip in the oracle (a swapped scale/min, a wrong shift,
an off-by-one sub-block, a dropped or sign-flipped min term) fails at least one of them.
"""
import os

import numpy as np
import pytest

import oracle as O
from quantised_decode_mat_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- f16 ----------------------------------------------------------------------------------------
def test_f16_decode_matches_numpy_on_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([O.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ---- hand-worked blocks ---------------------------------------------------------------------------
def _read_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_q4k_handworked_block():
    blk = np.zeros(144, np.uint8)
    want_w = {}
    for tok in _read_fixture("q4k_handworked.txt"):
        if tok[0] == "header":
            blk[:16] = [int(t, 16) for t in tok[1:]]
        elif tok[0] == "code":
            blk[16 + int(tok[1])] = int(tok[2], 16)
        elif tok[0] == "sc":
            want_sc = [int(t) for t in tok[1:]]
        elif tok[0] == "m":
            want_m = [int(t) for t in tok[1:]]
        elif tok[0] == "w":
            want_w[int(tok[1])] = float(tok[2])
    d, dmin, sc, m, q = O.q4k_fields(blk)
    assert (d, dmin) == (1.0, 0.5)
    assert list(sc) == want_sc
    assert list(m) == want_m
    w = O.dequant(O.FMT_Q4_K, blk)
    for e, v in want_w.items():
        assert w[e] == v, (e, w[e], v)


def test_q6k_handworked_block():
    blk = np.zeros(210, np.uint8)
    want_q, want_w = {}, {}
    for tok in _read_fixture("q6k_handworked.txt"):
        if tok[0] == "ql":
            blk[int(tok[1])] = int(tok[2], 16)
        elif tok[0] == "qh":
            blk[128 + int(tok[1])] = int(tok[2], 16)
        elif tok[0] == "scales":
            blk[192:208] = [int(t, 16) for t in tok[1:]]
        elif tok[0] == "d":
            blk[208:210] = [int(t, 16) for t in tok[1:]]
        elif tok[0] == "q":
            want_q[int(tok[1])] = int(tok[2])
        elif tok[0] == "w":
            want_w[int(tok[1])] = float(tok[2])
    d, sc, q = O.q6k_fields(blk)
    assert d == 0.5
    assert list(sc) == [-32, -1, 0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 31]
    for e, v in want_q.items():
        assert q[e] == v, (e, q[e], v)
    w = O.dequant(O.FMT_Q6_K, blk)
    for e, v in want_w.items():
        assert w[e] == v, (e, w[e], v)


# ---- bijections the formats imply -----------------------------------------------------------------
def test_q4k_scale_bits_are_a_bijection_onto_sixteen_6bit_fields():
    """The 12 scale bytes are 96 bits = 8 scales + 8 mins of 6 bits: every bit lands in exactly
    one field, at exactly one bit position, and no two bits land in the same place."""
    seen = set()
    for bit in range(96):
        blk = np.zeros(144, np.uint8)
        blk[4 + bit // 8] = 1 << (bit % 8)
        _, _, sc, m, _ = O.q4k_fields(blk)
        fields = np.concatenate([sc, m])
        nz = np.nonzero(fields)[0]
        assert len(nz) == 1, (bit, fields)
        val = int(fields[nz[0]])
        assert val & (val - 1) == 0 and val < 64
        seen.add((int(nz[0]), val.bit_length() - 1))
    assert len(seen) == 96


def _q4k_encode_scales(sc, m):
    """Inverse of the packing: low 6 bits of sc0..3 and m0..3 in bytes 0..7; for j >= 4 the low
    nibbles of sc_j / m_j share byte j+4 (scale low, min high) and the top two bits of sc_j / m_j
    ride in bits 6-7 of bytes j-4 / j."""
    s = np.zeros(12, np.uint8)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return s


def test_q4k_scale_min_round_trip_all_pairs():
    rng = np.random.default_rng(7)
    pairs = [(a, b) for a in range(64) for b in range(64)]
    for j in range(8):
        for a, b in pairs[:: 1 if j == 0 else 17]:
            sc = rng.integers(0, 64, 8)
            m = rng.integers(0, 64, 8)
            sc[j], m[j] = a, b
            blk = np.zeros(144, np.uint8)
            blk[4:16] = _q4k_encode_scales(sc, m)
            _, _, gsc, gm, _ = O.q4k_fields(blk)
            assert list(gsc) == list(sc) and list(gm) == list(m)


def test_q4k_code_nibbles_are_a_bijection_onto_elements():
    owner = {}
    for byte in range(128):
        for nib in range(2):
            blk = np.zeros(144, np.uint8)
            blk[16 + byte] = 1 << (4 * nib)
            _, _, _, _, q = O.q4k_fields(blk)
            nz = np.nonzero(q)[0]
            assert len(nz) == 1 and q[nz[0]] == 1
            owner[(byte, nib)] = int(nz[0])
    assert sorted(owner.values()) == list(range(256))
    # consecutive bytes feed consecutive elements of one 32-element sub-block
    for byte in range(127):
        if byte % 32 != 31:
            assert owner[(byte + 1, 0)] == owner[(byte, 0)] + 1
            assert owner[(byte + 1, 0)] // 32 == owner[(byte, 0)] // 32


def test_q6k_code_bits_are_a_bijection_onto_elements():
    low_owner, high_owner = {}, {}
    for byte in range(128):
        for nib in range(2):
            blk = np.zeros(210, np.uint8)
            blk[byte] = 1 << (4 * nib)
            _, _, q = O.q6k_fields(blk)
            nz = np.nonzero(q)[0]
            assert len(nz) == 1 and q[nz[0]] == 1
            low_owner[(byte, nib)] = int(nz[0])
    for byte in range(64):
        for pair in range(4):
            blk = np.zeros(210, np.uint8)
            blk[128 + byte] = 1 << (2 * pair)
            _, _, q = O.q6k_fields(blk)
            nz = np.nonzero(q)[0]
            assert len(nz) == 1 and q[nz[0]] == 16
            high_owner[(byte, pair)] = int(nz[0])
    assert sorted(low_owner.values()) == list(range(256))
    assert sorted(high_owner.values()) == list(range(256))


def test_q6k_scale_index_is_element_over_16():
    for s in range(16):
        blk = np.zeros(210, np.uint8)
        blk[208:210] = [0x00, 0x3C]  # d = 1
        blk[192 + s] = 1  # only scale s is 1; all codes 0 -> w = -32 exactly where e/16 == s
        w = O.dequant(O.FMT_Q6_K, blk)
        assert np.array_equal(np.nonzero(w)[0], np.arange(16 * s, 16 * s + 16))
        assert np.all(w[16 * s: 16 * s + 16] == -32.0)


# ---- q8_K invariants -------------------------------------------------------------------------------
def _pack_cases():
    rng = np.random.default_rng(11)
    xs = [synth.activations(0, 3, 2048)]
    xs.append((rng.standard_normal((2, 1024)) * 1e-3).astype(np.float32))
    xs.append((rng.standard_normal((1, 512)) * 1e4).astype(np.float32))
    spiky = rng.standard_normal((1, 768)).astype(np.float32)
    spiky[0, 5] = 80.0
    spiky[0, 300] = -40.0
    xs.append(spiky)
    return xs


@pytest.mark.parametrize("x", _pack_cases())
def test_q8k_invariants(x):
    qs, d, bs = O.q8k_pack(x)
    batch, K = x.shape
    nb = K // 256
    xb = x.reshape(batch, nb, 256).astype(np.float64)
    qb = qs.reshape(batch, nb, 256).astype(np.int64)
    # eight sums of 32 codes each
    assert np.array_equal(bs.astype(np.int64), qb.reshape(batch, nb, 8, 32).sum(-1))
    # codes in range, argmax maps to +-127 with the sign of x
    assert qb.min() >= -127 and qb.max() <= 127
    am = np.abs(xb).argmax(-1)
    top = np.take_along_axis(qb, am[..., None], -1)[..., 0]
    topx = np.take_along_axis(xb, am[..., None], -1)[..., 0]
    assert np.array_equal(top, np.where(topx > 0, 127, -127))
    # d = amax / 127 to f32 rounding, and reconstruction error at most half a step
    amax = np.abs(xb).max(-1)
    assert np.allclose(d.astype(np.float64), amax / 127.0, rtol=2 ** -23, atol=0)
    err = np.abs(xb - d[..., None].astype(np.float64) * qb)
    assert np.all(err <= d[..., None] * (0.5 + 2 ** -20))


def test_q8k_zero_block_and_exact_multiples():
    x = np.zeros((1, 512), np.float32)
    c = 2.0 ** -5
    k = np.arange(-127, 129, dtype=np.int64)[:256]
    k[-1] = 127
    x[0, 256:] = (k * c).astype(np.float32)
    qs, d, bs = O.q8k_pack(x)
    assert d[0, 0] == 0 and not qs[0, :256].any() and not bs[0, 0].any()
    assert d[0, 1] == np.float32(c)  # amax = 127c, d = 127c/127 exactly for a power-of-two c
    assert np.array_equal(qs[0, 256:].astype(np.int64), k)


def test_q8k_block_below_overflow_threshold():
    """amax = 1e-38 < 127/FLT_MAX: 127/amax is +inf in f32, so nonzero codes saturate to +-127 and a
    zero (0 * inf = NaN) gets code 0; d = amax/127 is subnormal but exact division."""
    x = np.zeros((1, 256), np.float32)
    x[0, :] = np.float32(1e-38)
    x[0, 1] = -np.float32(5e-39)
    x[0, 2] = 0.0
    qs, d, bs = O.q8k_pack(x)
    assert qs[0, 0] == 127 and qs[0, 1] == -127 and qs[0, 2] == 0
    assert d[0, 0] == np.float32(np.float32(1e-38) / np.float32(127.0))
    assert bs[0, 0, 0] == 127 * 29 and list(bs[0, 0, 1:]) == [127 * 32] * 7


def test_q8k_rounds_half_to_even():
    x = np.zeros((1, 256), np.float32)
    x[0, 0] = 127.0  # amax = 127 -> iscale = 1 exactly, so codes are rint(x)
    x[0, 1:7] = [2.5, 3.5, -2.5, -3.5, 0.5, 1.5]
    qs, d, _ = O.q8k_pack(x)
    assert d[0, 0] == 1.0
    assert list(qs[0, :7]) == [127, 2, 4, -2, -4, 0, 2]


# ---- integer dots: brute force and closed forms -----------------------------------------------------
def test_subdots_brute_force_tiny():
    x = synth.activations(5, 1, 512)
    qs, _, _ = O.q8k_pack(x)
    for fmt in (O.FMT_Q4_K, O.FMT_Q6_K):
        W = synth.weights("q4k" if fmt == O.FMT_Q4_K else "q6k", 5, 3, 512)
        for r in range(3):
            dots = O.subdots(fmt, W[r], qs[0])
            for b in range(2):
                if fmt == O.FMT_Q4_K:
                    _, _, _, _, q = O.q4k_fields(W[r, b])
                    ref = [int(np.dot(q[32 * j:32 * j + 32], qs[0, 256 * b + 32 * j: 256 * b + 32 * j + 32].astype(np.int64)))
                           for j in range(8)]
                else:
                    _, _, q = O.q6k_fields(W[r, b])
                    ref = [int(np.dot(q[16 * s:16 * s + 16] - 32, qs[0, 256 * b + 16 * s: 256 * b + 16 * s + 16].astype(np.int64)))
                           for s in range(16)]
                assert list(dots[b]) == ref


def _q4k_uniform_block(d_bits, dmin_bits, sc, m, code):
    blk = np.zeros(144, np.uint8)
    blk[0:2] = [d_bits & 255, d_bits >> 8]
    blk[2:4] = [dmin_bits & 255, dmin_bits >> 8]
    blk[4:16] = _q4k_encode_scales([sc] * 8, [m] * 8)
    blk[16:] = code | (code << 4)
    return blk


def test_q4k_unit_scales_reduce_to_a_plain_code_dot():
    """sc = 1, m = 0, every code c: y = sum_b dx_b * d * c * sum(q8 of block b)."""
    x = synth.activations(9, 1, 1024)
    qs, xd, bs = O.q8k_pack(x)
    for c in (0, 1, 7, 15):
        row = np.stack([_q4k_uniform_block(0x3C00, 0x3800, 1, 0, c)] * 4)[None]
        y = O.qmatvec(O.FMT_Q4_K, row, qs, xd, bs)
        ref = sum(float(xd[0, b]) * c * int(qs[0, 256 * b:256 * b + 256].astype(np.int64).sum()) for b in range(4))
        assert np.isclose(y[0, 0], ref, rtol=1e-6, atol=1e-6)


def test_q4k_zero_codes_reduce_to_minus_dmin_min_term():
    """All codes zero: y = -sum_b dx_b * dmin_b * sum_j m_j * bsum_j (the bsums carry it)."""
    x = synth.activations(3, 2, 2048)
    qs, xd, bs = O.q8k_pack(x)
    W = synth.q4k_weights(3, 5, 2048).copy()
    W[:, :, 16:] = 0
    y = O.qmatvec(O.FMT_Q4_K, W, qs, xd, bs)
    for v in range(2):
        for r in range(5):
            ref = 0.0
            for b in range(8):
                _, dmin, _, m, _ = O.q4k_fields(W[r, b])
                ref -= float(xd[v, b]) * dmin * int(np.dot(m, bs[v, b].astype(np.int64)))
            assert np.isclose(y[v, r], ref, rtol=1e-5, atol=0)


def test_q6k_special_blocks():
    x = synth.activations(4, 1, 768)
    qs, xd, bs = O.q8k_pack(x)
    nb = 3
    # every code 32 (ql nibbles 0, qh pairs 2): y = 0 exactly
    blk = np.zeros(210, np.uint8)
    blk[128:192] = 0xAA
    blk[192:208] = 5
    blk[208:210] = [0x00, 0x3C]
    y = O.qmatvec(O.FMT_Q6_K, np.stack([blk] * nb)[None], qs, xd, bs)
    assert y[0, 0] == 0.0
    # unit scales, d = 1, every code a + 16h: y = sum_b dx_b * (a + 16h - 32) * sum(q8 of block b)
    for a, h in ((0, 0), (15, 3), (7, 1)):
        blk = np.zeros(210, np.uint8)
        blk[0:128] = a | (a << 4)
        blk[128:192] = h * 0x55
        blk[192:208] = 1
        blk[208:210] = [0x00, 0x3C]
        y = O.qmatvec(O.FMT_Q6_K, np.stack([blk] * nb)[None], qs, xd, bs)
        ref = sum(float(xd[0, b]) * (a + 16 * h - 32) * int(qs[0, 256 * b:256 * b + 256].astype(np.int64).sum())
                  for b in range(nb))
        assert np.isclose(y[0, 0], ref, rtol=1e-6, atol=1e-6)


# ---- f32 epilogue against the f64 brute force and the closed-form bound ------------------------------
@pytest.mark.parametrize("fmt,K,rows,batch", [(O.FMT_Q4_K, 2048, 16, 2), (O.FMT_Q6_K, 1792, 12, 3)])
def test_epilogue_against_f64_brute_force(fmt, K, rows, batch):
    name = "q4k" if fmt == O.FMT_Q4_K else "q6k"
    W = synth.weights(name, 21, rows, K)
    x = synth.activations(21, batch, K)
    qs, xd, bs = O.q8k_pack(x)
    y64 = O.qmatvec_f64(fmt, W, qs, xd)
    for order in (O.ORDER_SEQUENTIAL, O.ORDER_GROUPS_OF_FOUR):
        y = O.qmatvec(fmt, W, qs, xd, bs, order)
        assert O.rel_err(y, y64).max() < 2e-3
        assert O.rel_err(y, y64).max() < 1e-5  # much tighter in practice: f32 rounding only
    # against raw x: |y64 - sum w x| <= sum |w| * dx / 2
    nb = K // 256
    for v in range(batch):
        for r in range(rows):
            w = np.concatenate([O.dequant(fmt, W[r, b]) for b in range(nb)])
            exact = float(np.dot(w, x[v].astype(np.float64)))
            bound = float(np.dot(np.abs(w), np.repeat(xd[v].astype(np.float64), 256))) * 0.5 * (1 + 2 ** -20)
            assert abs(y64[v, r] - exact) <= bound + 1e-12


def test_orders_differ_only_in_rounding():
    W = synth.weights("q4k", 8, 64, 4096)
    x = synth.activations(8, 1, 4096)
    qs, xd, bs = O.q8k_pack(x)
    y0 = O.qmatvec(O.FMT_Q4_K, W, qs, xd, bs, O.ORDER_SEQUENTIAL)
    y1 = O.qmatvec(O.FMT_Q4_K, W, qs, xd, bs, O.ORDER_GROUPS_OF_FOUR)
    # two f32 summation orders of n terms differ by at most 2 (n - 1) u sum|t| (u = 2^-24)
    for r in range(64):
        t = O.block_terms(O.FMT_Q4_K, W[r], qs[0], xd[0], bs[0]).astype(np.float64)
        assert abs(float(y1[0, r]) - float(y0[0, r])) <= 2 * 15 * 2.0 ** -24 * np.abs(t).sum()
    # the grouped order is the stated tree over the block terms
    for r in range(4):
        t = O.block_terms(O.FMT_Q4_K, W[r], qs[0], xd[0], bs[0]).astype(np.float32)
        groups = [(t[4 * g] + t[4 * g + 1]) + (t[4 * g + 2] + t[4 * g + 3]) for g in range(4)]
        acc = groups[0]
        for G in groups[1:]:
            acc = np.float32(acc + G)
        assert acc == y1[0, r]


def test_runs_of_sixteen_order_is_the_stated_tree():
    """Order 2: groups of four blocks, runs of four groups left to right (absent groups +0),
    runs left to right; identical to order 1 for rows of at most 16 blocks."""
    W = synth.weights("q6k", 6, 8, 14336)
    x = synth.activations(6, 1, 14336)
    qs, xd, bs = O.q8k_pack(x)
    y2 = O.qmatvec(O.FMT_Q6_K, W, qs, xd, bs, O.ORDER_RUNS_OF_SIXTEEN)
    for r in range(8):
        t = O.block_terms(O.FMT_Q6_K, W[r], qs[0], xd[0], bs[0]).astype(np.float32)
        t = np.concatenate([t, np.zeros(64 - len(t), np.float32)])  # 56 blocks, padded to 4 runs
        G = [np.float32((t[4 * g] + t[4 * g + 1]) + (t[4 * g + 2] + t[4 * g + 3])) for g in range(16)]
        runs = []
        for run in range(4):
            acc = G[4 * run]
            for g in range(1, 4):
                acc = np.float32(acc + G[4 * run + g])
            runs.append(acc)
        total = runs[0]
        for R in runs[1:]:
            total = np.float32(total + R)
        assert total == y2[0, r]
    W4 = synth.weights("q4k", 6, 8, 4096)
    x4 = synth.activations(6, 1, 4096)
    qs4, xd4, bs4 = O.q8k_pack(x4)
    assert np.array_equal(O.qmatvec(O.FMT_Q4_K, W4, qs4, xd4, bs4, O.ORDER_GROUPS_OF_FOUR).view(np.uint32),
                          O.qmatvec(O.FMT_Q4_K, W4, qs4, xd4, bs4, O.ORDER_RUNS_OF_SIXTEEN).view(np.uint32))


def test_q6k_split_round_trip():
    g = synth.q6k_weights(2, 6, 1792)
    body, prefix = O.q6k_split(g, prefix_stride=8)
    rebuilt = np.concatenate([body, prefix[:, :7].view(np.uint8).reshape(6, 7, 2)], axis=2)
    assert np.array_equal(rebuilt, g)
    assert not prefix[:, 7:].any()


def test_golden_regression():
    """Stored oracle outputs (written by tests/golden/make_golden.py, which calls only the oracle)."""
    path = os.path.join(GOLDEN, "oracle_regression.txt")
    from tests.golden.make_golden import compute
    stored = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, hexs = line.split(":", 1)
            stored[key.strip()] = hexs.split()
    now = compute()
    assert set(now) == set(stored)
    for k in now:
        assert now[k] == stored[k], k


# ---- RMSNorm (+ residual) before the pack --------------------------------------------------------
def test_rmsnorm_power_of_two_scaling_is_exact():
    """With eps = 0, scaling h by 2^k scales every square by 4^k exactly, so the norm's output
    is bit-identical; scaling g by 2 doubles n exactly."""
    x = synth.activations(21, 2, 1024)
    g = synth.norm_gain(21, 1024)
    _, n = O.rmsnorm(x, None, g, 0.0)
    for k in (-3, 1, 5):
        _, nk = O.rmsnorm(x * np.float32(2.0 ** k), None, g, 0.0)
        assert np.array_equal(nk.view(np.uint32), n.view(np.uint32))
    _, n2 = O.rmsnorm(x, None, g * np.float32(2.0), 0.0)
    assert np.array_equal(n2, n * np.float32(2.0))


def test_rmsnorm_constant_vector_closed_form():
    """h = a everywhere: every partial sum is exact, ms = a^2, n = a / sqrt(a^2 + eps) * g."""
    K = 768
    for a, eps in ((0.75, 0.0), (-1.5, 0.25), (3.0, 1e-5)):
        x = np.full((1, K), a, np.float32)
        g = np.linspace(0.5, 1.5, K).astype(np.float32)
        h, n = O.rmsnorm(x, None, g, eps)
        assert np.array_equal(h, x)
        inv = np.float32(1.0) / np.sqrt(np.float32(a * a) + np.float32(eps), dtype=np.float32)
        want = (np.float32(a) * inv) * g
        assert np.array_equal(n[0].view(np.uint32), want.view(np.uint32))


def test_rmsnorm_residual_is_the_f32_sum():
    x = synth.activations(22, 3, 512)
    r = synth.residual(22, 3, 512)
    g = synth.norm_gain(22, 512)
    h, n = O.rmsnorm(x, r, g, 1e-6)
    assert np.array_equal(h, x + r)
    h0, n0 = O.rmsnorm(x + r, None, g, 1e-6)
    assert np.array_equal(h0, h) and np.array_equal(n0.view(np.uint32), n.view(np.uint32))


def test_rmsnorm_matches_f64_within_the_rounding_bound():
    """f32 against the same formula in f64 from the same h: the sum of K squares in any order
    is within K*u relative, the rest adds a few u, so 1e-5 relative bounds K <= 16384."""
    for K, eps in ((256, 1e-6), (4096, 1e-5), (14336, 1e-6)):
        x = synth.activations(23, 2, K)
        r = synth.residual(23, 2, K)
        g = synth.norm_gain(23, K)
        h, n = O.rmsnorm(x, r, g, eps)
        h64 = h.astype(np.float64)
        n64 = h64 / np.sqrt(np.mean(h64 * h64, axis=1, keepdims=True) + eps) * g.astype(np.float64)
        assert np.max(np.abs(n - n64) / np.abs(n64)) < 1e-5


def test_rmsnorm_sum_of_squares_is_the_declared_tree():
    """The declared order: 256 lane sums (left to right over the lane's elements), a pairwise
    tree inside each group of 32 lanes, the eight group sums left to right.  Values spread over
    many orders of magnitude make other orders round differently."""
    K = 1024
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((1, K)) * np.exp2(rng.integers(-12, 12, size=(1, K)))).astype(np.float32)
    g = np.ones(K, np.float32)
    _, n = O.rmsnorm(x, None, g, 0.0)
    sq = (x[0] * x[0]).astype(np.float32)
    lane = np.zeros(256, np.float32)
    for i in range(K):
        lane[i % 256] = np.float32(lane[i % 256] + sq[i])
    total = None
    for w in range(8):
        v = lane[32 * w: 32 * w + 32].copy()
        s = 16
        while s >= 1:
            v[:s] = (v[:s] + v[s: 2 * s]).astype(np.float32)
            s //= 2
        total = v[0] if total is None else np.float32(total + v[0])
    ms = np.float32(total / np.float32(K))
    inv = np.float32(np.float32(1.0) / np.sqrt(ms, dtype=np.float32))
    want = (x[0] * inv).astype(np.float32) * g
    assert np.array_equal(n[0].view(np.uint32), want.view(np.uint32))
    # a sequential sum of the same squares gives other bits for some elements
    seq = np.float32(0.0)
    for v in sq:
        seq = np.float32(seq + v)
    assert seq != total


def test_rmsnorm_pack_is_pack_of_the_norm():
    x = synth.activations(24, 2, 2048)
    r = synth.residual(24, 2, 2048)
    g = synth.norm_gain(24, 2048)
    h, qs, d, bs = O.rmsnorm_q8k_pack(x, r, g, 1e-5)
    _, n = O.rmsnorm(x, r, g, 1e-5)
    qs2, d2, bs2 = O.q8k_pack(n)
    assert np.array_equal(qs, qs2) and np.array_equal(d.view(np.uint32), d2.view(np.uint32)) and np.array_equal(bs, bs2)
    # zero gain: a zero vector, packed as zeros with d = 0
    _, qz, dz, bz = O.rmsnorm_q8k_pack(x, r, np.zeros(2048, np.float32), 1e-5)
    assert not qz.any() and not dz.any() and not bz.any()


def test_rmsnorm_sum_order_by_absorption():
    """One square of 2^24 among squares of 1: adding a 1 to 2^24 rounds back to 2^24 (ties to
    even), so the total counts exactly the 1s that were summed before meeting the large value.
    Declared order, K = 1024: lane 0 holds 2^24 and absorbs its own three 1s; the other 255
    lanes hold 4 each and are added exactly, so the total is 2^24 + 1020.  A sequential sum
    gives 2^24, and lanes of stride 128 give 2^24 + 1016."""
    K = 1024
    x = np.ones((1, K), np.float32)
    x[0, 0] = np.float32(4096.0)
    g = np.ones(K, np.float32)
    _, n = O.rmsnorm(x, None, g, 0.0)
    total = np.float32(2.0 ** 24 + 1020)
    inv = np.float32(np.float32(1.0) / np.sqrt(np.float32(total / np.float32(K)), dtype=np.float32))
    assert np.array_equal(n[0].view(np.uint32), (x[0] * inv).view(np.uint32))
    for other in (2.0 ** 24, 2.0 ** 24 + 1016):
        inv_o = np.float32(np.float32(1.0) / np.sqrt(np.float32(np.float32(other) / np.float32(K)), dtype=np.float32))
        assert inv_o != inv


# ---- Q5_K: Q4_K's layout plus a plane of fifth bits --------------------------------------------------
def test_q5k_handworked_block():
    """d = 1, dmin = 0, every scale 1 and min 0, so w_e is the 5-bit code itself.  Worked by hand
    from the GGUF layout: element 64c + t takes the low nibble of qs[32c + t] (t < 32) or the
    high nibble of qs[32c + t - 32] (t >= 32), plus 16 x bit 2c of qh[t] (t < 32) or bit 2c+1
    of qh[t - 32] (t >= 32)."""
    blk = np.zeros(176, np.uint8)
    blk[0:2] = [0x00, 0x3C]            # d = 1.0
    blk[2:4] = [0x00, 0x00]            # dmin = 0
    blk[4:16] = _q4k_encode_scales([1] * 8, [0] * 8)
    qh, qs = blk[16:48], blk[48:176]
    qs[0] = 0x21                       # element 0: low nibble 1; element 32: high nibble 2
    qh[0] = 0b00000011                 # +16 on element 0 (bit 0) and element 32 (bit 1)
    qs[69] = 0x03                      # element 133 = 64*2 + 5: low nibble 3
    qh[5] = 0b00010000                 # bit 4 = 2c for c = 2: +16 on element 133
    qs[127] = 0xF0                     # element 255 = 64*3 + 32 + 31: high nibble 15
    qh[31] = 0b10000000                # bit 7 = 2c+1 for c = 3: +16 on element 255
    qs[40] = 0x50                      # element 64*1 + 32 + 8 = 104: high nibble 5, no fifth bit
    want = np.zeros(256)
    want[[0, 32, 133, 255, 104]] = [17, 18, 19, 31, 5]
    d, dmin, sc, m, q = O.q5k_fields(blk)
    assert (d, dmin) == (1.0, 0.0) and list(sc) == [1] * 8 and list(m) == [0] * 8
    assert np.array_equal(q, want.astype(np.int32))
    assert np.array_equal(O.dequant(O.FMT_Q5_K, blk), want)


def test_q5k_code_bits_are_a_bijection_onto_elements():
    """Each of the 160 code bytes' bits drives exactly one element's bit: nibble bits 0..3 and
    fifth bit 4, every (element, bit) pair exactly once."""
    seen = set()
    for byte in range(160):
        for bit in range(8):
            blk = np.zeros(176, np.uint8)
            blk[16 + byte] = 1 << bit
            _, _, _, _, q = O.q5k_fields(blk)
            nz = np.nonzero(q)[0]
            assert len(nz) == 1
            v = int(q[nz[0]])
            assert v in (1, 2, 4, 8, 16)
            seen.add((int(nz[0]), v))
    assert seen == {(e, 1 << b) for e in range(256) for b in range(5)}


def test_q5k_with_zero_fifth_bits_is_q4k():
    """qh = 0: a Q5_K block decodes, dots and sums exactly as the Q4_K block with the same d,
    dmin, scales and nibbles."""
    K, rows = 1536, 6
    W5 = synth.q5k_weights(12, rows, K).copy()
    W5[:, :, 16:48] = 0
    W4 = np.concatenate([W5[:, :, 0:16], W5[:, :, 48:176]], axis=2)
    x = synth.activations(12, 2, K)
    qs, xd, bs = O.q8k_pack(x)
    for r in range(rows):
        assert np.array_equal(O.subdots(O.FMT_Q5_K, W5[r], qs[0]), O.subdots(O.FMT_Q4_K, W4[r], qs[0]))
        assert np.array_equal(O.dequant(O.FMT_Q5_K, W5[r, 0]), O.dequant(O.FMT_Q4_K, W4[r, 0]))
    y5 = O.qmatvec(O.FMT_Q5_K, W5, qs, xd, bs, O.ORDER_RUNS_OF_SIXTEEN)
    y4 = O.qmatvec(O.FMT_Q4_K, W4, qs, xd, bs, O.ORDER_RUNS_OF_SIXTEEN)
    assert np.array_equal(y5.view(np.uint32), y4.view(np.uint32))


def test_q5k_fifth_bits_add_sixteen_times_the_block_sums():
    """All fifth bits set: every code is its nibble + 16, so each sub-block dot grows by exactly
    16 x the sub-block's q8 sum (the bsums)."""
    K = 1024
    W5 = synth.q5k_weights(13, 3, K).copy()
    x = synth.activations(13, 1, K)
    qs, xd, bs = O.q8k_pack(x)
    Wz = W5.copy()
    Wz[:, :, 16:48] = 0
    W5[:, :, 16:48] = 0xFF
    for r in range(3):
        d1 = O.subdots(O.FMT_Q5_K, W5[r], qs[0]).astype(np.int64)
        d0 = O.subdots(O.FMT_Q5_K, Wz[r], qs[0]).astype(np.int64)
        assert np.array_equal(d1 - d0, 16 * bs[0].astype(np.int64))


def test_q5k_subdots_and_epilogue_brute_force():
    K, rows, batch = 768, 5, 2
    W = synth.q5k_weights(14, rows, K)
    x = synth.activations(14, batch, K)
    qs, xd, bs = O.q8k_pack(x)
    for r in range(rows):
        dots = O.subdots(O.FMT_Q5_K, W[r], qs[1])
        for b in range(3):
            _, _, _, _, q = O.q5k_fields(W[r, b])
            ref = [int(np.dot(q[32 * j:32 * j + 32], qs[1, 256 * b + 32 * j: 256 * b + 32 * j + 32].astype(np.int64)))
                   for j in range(8)]
            assert list(dots[b]) == ref
    y64 = O.qmatvec_f64(O.FMT_Q5_K, W, qs, xd)
    y = O.qmatvec(O.FMT_Q5_K, W, qs, xd, bs, O.ORDER_RUNS_OF_SIXTEEN)
    assert O.rel_err(y, y64).max() < 1e-5
    # f64 brute force from the dequantised weights and the dequantised activations
    for v in range(batch):
        for r in range(rows):
            w = np.concatenate([O.dequant(O.FMT_Q5_K, W[r, b]) for b in range(3)])
            xh = np.repeat(xd[v].astype(np.float64), 256) * qs[v].astype(np.float64)
            assert np.isclose(y64[v, r], float(np.dot(w, xh)), rtol=1e-12, atol=1e-12)


def test_long_rows_are_computed_not_skipped():
    """Rows of more than 4096 blocks (K = 1,048,832 here) are computed like any other: the
    same-order result sits within the f32 summation bound of the f64 brute force, so the
    output cannot be the untouched zero buffer."""
    K = 4097 * 256
    W = synth.weights("q4k", 11, 2, K)
    x = synth.activations(11, 1, K)
    qs, xd, bs = O.q8k_pack(x)
    y = O.qmatvec(O.FMT_Q4_K, W, qs, xd, bs, O.ORDER_RUNS_OF_SIXTEEN)
    ref = O.qmatvec_f64(O.FMT_Q4_K, W, qs, xd)
    for r in range(2):
        t = O.block_terms(O.FMT_Q4_K, W[r], qs[0], xd[0], bs[0]).astype(np.float64)
        bound = 4 * 4097 * 2.0 ** -24 * np.abs(t).sum() + 64 * 2.0 ** -24 * abs(ref[0, r])
        assert y[0, r] != 0.0
        assert abs(float(y[0, r]) - ref[0, r]) <= bound


def test_refused_shape_raises():
    """A call the mat-vec is not defined on raises instead of returning a zero buffer."""
    W = np.zeros((1, 0), np.uint8)  # one row of K = 0
    qs = np.zeros((1, 0), np.int8)
    with pytest.raises(RuntimeError, match="refused"):
        O.qmatvec(O.FMT_Q4_K, W, qs, np.zeros((1, 0), np.float32), np.zeros((1, 0, 8), np.int16))
