"""Pins of the f64 oracle to facts outside the oracle itself.

Each definition comes from the S-MoE page "Metal Compute Kernels", section
"Fused FFN Kernels -- One Simdgroup Per Output Row" (w = (code - Z)(1/Z)s,
Z = 7.5 for Q4 and 1.5 for Q2; hidden = SiLU(gate.x) * (up.x);
out = down.hidden), section "Layout assumptions the kernels rely on" (codes
packed along a row, one scale per group of 64 columns) and section
"Coalesced Dense Matvec -- the Same Contract for bf16".  The pages print no
worked example, so the pins are:

* hand-derived values on tiny matrices whose bytes are written out literally
  (nibble / crumb order, group indexing, row/column orientation, Z),
* closed forms and invariants (all-zero and all-max codes, code flip,
  constant code, linearity, x = 0),
* the method's own fold s*((sum code*x)/Z - sum x), evaluated here with numpy
  from the unpacked codes, against the oracle's full dequantisation,
* SiLU against scipy's logistic function and its odd-part identity,
* bf16 widening of literal bit patterns.

A plausible slip in the oracle (swapped nibbles, wrong Z, a dropped sum-x
term, a wrong scale index, gate and up swapped, a transposed matrix) fails at
least one test below; the mutation tests at the end plant some of those slips
in a patched copy of the oracle's source and check that they are caught.
"""
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import smoe_inputs as inp


# ---------------------------------------------------------------- unpacking

def test_unpack_q4_literal_bytes():
    # byte j: column 2j in the low nibble, column 2j+1 in the high nibble
    packed = np.array([0x21, 0x43, 0xF0, 0x0F, 0xA5], dtype=np.uint8)
    assert oracle.unpack(packed, 4, 10).tolist() == [1, 2, 3, 4, 0, 15, 15, 0, 5, 10]


def test_unpack_q2_literal_bytes():
    # byte j: columns 4j..4j+3, the first column in the lowest two bits
    packed = np.array([0xE4, 0x1B, 0x80], dtype=np.uint8)  # 11 10 01 00 / 00 01 10 11 / 10 00 00 00
    assert oracle.unpack(packed, 2, 12).tolist() == [0, 1, 2, 3, 3, 2, 1, 0, 0, 0, 0, 2]


def test_unpack_every_byte_value_is_a_bijection():
    allb = np.arange(256, dtype=np.uint8)
    q4 = oracle.unpack(allb, 4, 512).reshape(256, 2)
    q2 = oracle.unpack(allb, 2, 1024).reshape(256, 4)
    assert len({tuple(r) for r in q4}) == 256 and q4.max() == 15
    assert len({tuple(r) for r in q2}) == 256 and q2.max() == 3
    # the integer a byte denotes is recovered from its codes (little end first)
    assert all(int(r[0]) + 16 * int(r[1]) == b for b, r in enumerate(q4))
    assert all(sum(int(c) << (2 * i) for i, c in enumerate(r)) == b for b, r in enumerate(q2))


# ------------------------------------------------- hand-derived tiny matrices

# One Q4 row of 64 columns whose code at column k is k % 16: bytes 0x10, 0x32,
# ..., 0xFE repeated four times (low nibble = even column).
Q4_RAMP_ROW = bytes([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE] * 4)


def _e(k, n):
    x = np.zeros(n)
    x[k] = 1.0
    return x


@pytest.mark.parametrize("k,expected", [
    (0, -0.5),            # code 0: 0.5 * (0 - 7.5) / 7.5
    (15, 0.5),            # code 15: 0.5 * 7.5 / 7.5
    (8, 1.0 / 30.0),      # code 8: 0.5 * 0.5 / 7.5
    (17, -13.0 / 30.0),   # code 1: 0.5 * (-6.5) / 7.5
    (62, 6.5 / 15.0),     # code 14: 0.5 * 6.5 / 7.5
])
def test_q4_single_row_one_hot(k, expected):
    codes = np.frombuffer(Q4_RAMP_ROW, dtype=np.uint8).reshape(1, 32)
    y, a = oracle.qgemv(4, codes, np.array([[0.5]], np.float32), 1, 64, 64, _e(k, 64))
    assert y[0] == pytest.approx(expected, rel=1e-15, abs=1e-15)
    assert a[0] == pytest.approx(abs(expected), rel=1e-15, abs=1e-15)


def test_q4_single_row_all_ones_sums_to_zero():
    # sum over four ramps of (c - 7.5) = 4 * (120 - 16*7.5) = 0
    codes = np.frombuffer(Q4_RAMP_ROW, dtype=np.uint8).reshape(1, 32)
    y, a = oracle.qgemv(4, codes, np.array([[0.5]], np.float32), 1, 64, 64, np.ones(64))
    assert abs(y[0]) < 1e-15
    # sum |c - 7.5| over one ramp = 2 * (0.5 + 1.5 + ... + 7.5) = 64
    assert a[0] == pytest.approx(0.5 / 7.5 * 4 * 64, rel=1e-15)


def test_q4_two_groups_uses_the_right_scale():
    # 1 x 128, two groups with scales 0.25 and 1.0.  Column 70 (group 1) has
    # code 70 % 16 = 6: y = 1.0 * (6 - 7.5) / 7.5 = -0.2.  A scale taken from
    # group 0 would give -0.05, swapped nibbles (code 7) would give -1/15.
    codes = np.frombuffer(Q4_RAMP_ROW * 2, dtype=np.uint8).reshape(1, 64)
    s = np.array([[0.25, 1.0]], np.float32)
    y, _ = oracle.qgemv(4, codes, s, 1, 128, 64, _e(70, 128))
    assert y[0] == pytest.approx(-0.2, rel=1e-15)
    y, _ = oracle.qgemv(4, codes, s, 1, 128, 64, _e(3, 128))  # code 3, group 0
    assert y[0] == pytest.approx(0.25 * (3 - 7.5) / 7.5, rel=1e-15)


def test_q4_two_rows_orientation():
    # 2 x 64: row 0 is the ramp, row 1 is all code 15 (bytes 0xFF).  y = W x is
    # a column of height 2, one value per row; a transposed reading of W would
    # not even have the right length.
    codes = np.frombuffer(Q4_RAMP_ROW + bytes([0xFF] * 32), dtype=np.uint8).reshape(2, 32)
    s = np.array([[0.5], [2.0]], np.float32)
    y, _ = oracle.qgemv(4, codes, s, 2, 64, 64, _e(1, 64))
    assert y.tolist() == pytest.approx([0.5 * (1 - 7.5) / 7.5, 2.0], rel=1e-15)
    y, _ = oracle.qgemv(4, codes, s, 2, 64, 64, np.full(64, 0.5))
    assert y.tolist() == pytest.approx([0.0, 2.0 * 32], abs=1e-13)


@pytest.mark.parametrize("k,expected", [(0, -0.3), (1, -0.1), (2, 0.1), (3, 0.3), (61, -0.1)])
def test_q2_single_row_one_hot(k, expected):
    # 1 x 64 Q2, code at column k = k % 4: every byte is 0b11100100 = 0xE4.
    # y = 0.3 * (code - 1.5) / 1.5
    codes = np.full((1, 16), 0xE4, dtype=np.uint8)
    y, _ = oracle.qgemv(2, codes, np.array([[0.3]], np.float32), 1, 64, 64, _e(k, 64))
    assert y[0] == pytest.approx(expected, rel=1e-7)   # 0.3 is not exact in f32


# --------------------------------------------- invariants and closed forms

def _random_q(bits, rows, cols, group, seed):
    codes = inp.packed_codes(rows, cols, bits, seed, 1)
    s = inp.scales(rows, cols // group, seed, 2)
    x = inp.activations(cols, seed, 3).astype(np.float64)
    return codes, s, x


def _group_sums(x, group):
    return x.reshape(-1, group).sum(axis=1)


@pytest.mark.parametrize("bits", [4, 2])
def test_all_zero_and_all_max_codes(bits):
    rows, cols, group = 8, 256, 64
    _, s, x = _random_q(bits, rows, cols, group, 11)
    sx = _group_sums(x, group)
    expect = (s.astype(np.float64) * sx).sum(axis=1)
    y0, _ = oracle.qgemv(bits, np.zeros((rows, cols * bits // 8), np.uint8), s, rows, cols, group, x)
    y1, _ = oracle.qgemv(bits, np.full((rows, cols * bits // 8), 0xFF, np.uint8), s, rows, cols,
                         group, x)
    np.testing.assert_allclose(y0, -expect, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(y1, expect, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("bits,code", [(4, 0), (4, 5), (4, 9), (4, 15), (2, 0), (2, 1), (2, 2)])
def test_constant_code(bits, code):
    rows, cols, group = 4, 192, 64
    _, s, x = _random_q(bits, rows, cols, group, 12)
    byte = code | (code << 4) if bits == 4 else code * 0x55
    z = 7.5 if bits == 4 else 1.5
    y, _ = oracle.qgemv(bits, np.full((rows, cols * bits // 8), byte, np.uint8), s, rows, cols,
                        group, x)
    expect = (code / z - 1.0) * (s.astype(np.float64) * _group_sums(x, group)).sum(axis=1)
    np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("bits", [4, 2])
def test_code_flip_negates(bits):
    # c -> 2Z - c maps every code of a byte at once: byte -> 255 - byte
    rows, cols, group = 16, 512, 64
    codes, s, x = _random_q(bits, rows, cols, group, 13)
    y, _ = oracle.qgemv(bits, codes, s, rows, cols, group, x)
    yf, _ = oracle.qgemv(bits, 255 - codes, s, rows, cols, group, x)
    np.testing.assert_allclose(yf, -y, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bits", [4, 2])
def test_linearity_in_x_and_s(bits):
    rows, cols, group = 16, 256, 64
    codes, s, x = _random_q(bits, rows, cols, group, 14)
    x2 = inp.activations(cols, 14, 9).astype(np.float64)
    y1, _ = oracle.qgemv(bits, codes, s, rows, cols, group, x)
    y2, _ = oracle.qgemv(bits, codes, s, rows, cols, group, x2)
    y12, _ = oracle.qgemv(bits, codes, s, rows, cols, group, 2.0 * x - 3.0 * x2)
    np.testing.assert_allclose(y12, 2.0 * y1 - 3.0 * y2, rtol=1e-11, atol=1e-11)
    ys, _ = oracle.qgemv(bits, codes, (2.0 * s).astype(np.float32), rows, cols, group, x)
    np.testing.assert_allclose(ys, 2.0 * y1, rtol=1e-13, atol=1e-14)
    yz, az = oracle.qgemv(bits, codes, s, rows, cols, group, np.zeros(cols))
    assert not yz.any() and not az.any()


@pytest.mark.parametrize("bits,cols,group", [(4, 4096, 64), (2, 4096, 64), (4, 1536, 64),
                                             (4, 256, 128), (2, 1536, 192)])
def test_matches_the_fold_identity(bits, cols, group):
    # sum_k w_k x_k = sum_g s_g * ((sum_{k in g} code_k x_k) / Z - sum_{k in g} x_k)
    rows = 12
    codes, s, x = _random_q(bits, rows, cols, group, 15)
    c = oracle.unpack(codes, bits, rows * cols).reshape(rows, cols).astype(np.float64)
    z = 7.5 if bits == 4 else 1.5
    cx = (c * x).reshape(rows, -1, group).sum(axis=2)
    fold = (s.astype(np.float64) * (cx / z - _group_sums(x, group)[None, :])).sum(axis=1)
    y, a = oracle.qgemv(bits, codes, s, rows, cols, group, x)
    np.testing.assert_allclose(y, fold, rtol=1e-12, atol=1e-12 * a.max())
    assert (a >= np.abs(y) - 1e-12).all()


def test_row_subset_equals_full():
    codes, s, x = _random_q(4, 40, 512, 64, 16)
    y, a = oracle.qgemv(4, codes, s, 40, 512, 64, x)
    ys, as_ = oracle.qgemv(4, codes, s, 40, 512, 64, x, row0=17, nrows=9)
    assert (ys == y[17:26]).all() and (as_ == a[17:26]).all()


def test_oracle_refuses_bad_shapes():
    codes, s, x = _random_q(4, 4, 256, 64, 17)
    with pytest.raises(ValueError):
        oracle.qgemv(4, codes, s, 4, 256, 48, x)       # group does not divide cols
    with pytest.raises(ValueError):
        oracle.qgemv(3, codes, s, 4, 256, 64, x)       # no such width
    with pytest.raises(ValueError):
        oracle.qgemv(4, codes, s, 4, 256, 64, x, row0=3, nrows=2)


# ------------------------------------------------------------------- SiLU

def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert oracle.silu(-800.0) == 0.0          # exp overflow gives -0, not NaN
    assert oracle.silu(800.0) == 800.0


@pytest.mark.parametrize("v", [0.1, 0.5, 1.0, 2.5, 7.0, 20.0, 35.5])
def test_silu_odd_part_and_logistic(v):
    special = pytest.importorskip("scipy.special")
    # silu(v) - silu(-v) = v (v*sigma(v) + v*sigma(v) - v ... = v)
    assert oracle.silu(v) - oracle.silu(-v) == pytest.approx(v, rel=1e-14)
    assert oracle.silu(v) == pytest.approx(v * special.expit(v), rel=1e-14)


def test_gate_up_applies_silu_to_gate_only():
    # gate: all code 15, up: the ramp row; x = v * e_k.
    # g = s_g * v; u = s_u * v * (k%16 - 7.5)/7.5; hidden = silu(g) * u.
    d_ff, d_model, group = 1, 64, 64
    gate = np.full((1, 32), 0xFF, np.uint8)
    up = np.frombuffer(Q4_RAMP_ROW, dtype=np.uint8).reshape(1, 32)
    for v, k in ((40.0, 3), (-40.0, 20), (0.0, 5), (1.0, 9)):
        x = v * _e(k, 64)
        r = oracle.gate_up(4, gate, np.array([[1.0]], np.float32), up,
                           np.array([[0.5]], np.float32), d_ff, d_model, group, x)
        g = v
        u = 0.5 * v * ((k % 16) - 7.5) / 7.5
        assert r["g"][0] == pytest.approx(g, abs=1e-14)
        assert r["u"][0] == pytest.approx(u, abs=1e-14)
        # SiLU(40) = 40 to 1e-16, SiLU(-40) = 0 to 1e-16, SiLU(0) = 0
        if v == 40.0:
            assert r["hidden"][0] == pytest.approx(40.0 * u, rel=1e-15)
        elif v == -40.0 or v == 0.0:
            assert abs(r["hidden"][0]) < 1e-14
        else:
            assert r["hidden"][0] == pytest.approx(u / (1.0 + math.exp(-1.0)), rel=1e-14)


def test_ffn_is_down_of_gate_up():
    e = inp.expert(4, 256, 256, 64, seed=18)
    x = inp.activations(256, 18).astype(np.float64)
    hidden, out, out_abs = oracle.ffn(4, e["gate_codes"], e["gate_scales"], e["up_codes"],
                                      e["up_scales"], e["down_codes"], e["down_scales"],
                                      256, 256, 64, x)
    r = oracle.gate_up(4, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
                       256, 256, 64, x)
    assert (r["hidden"] == hidden).all()
    y, a = oracle.qgemv(4, e["down_codes"], e["down_scales"], 256, 256, 64, hidden)
    assert (y == out).all() and (a == out_abs).all()


def test_ffn_with_known_hidden():
    # gate all code 15 with scale 1, x = 50 e_0: g = 50, SiLU(g) = 50 (to 1e-20).
    # up all code 15 with scale 0.02: u = 1.  So hidden = 50 in every row, and
    # down (all code 0, scale 0.1, one group per row) gives -0.1 * 50 * d_ff.
    d_model, d_ff, group = 64, 128, 64
    gate = np.full((d_ff, 32), 0xFF, np.uint8)
    up = np.full((d_ff, 32), 0xFF, np.uint8)
    down = np.zeros((d_model, d_ff // 2), np.uint8)
    x = 50.0 * _e(0, d_model)
    hidden, out, _ = oracle.ffn(4, gate, np.ones((d_ff, 1), np.float32), up,
                                np.full((d_ff, 1), 0.02, np.float32), down,
                                np.full((d_model, 2), 0.1, np.float32), d_model, d_ff, group, x)
    np.testing.assert_allclose(hidden, 50.0 * np.float64(np.float32(0.02)) * 50.0, rtol=1e-15)
    np.testing.assert_allclose(out, -np.float64(np.float32(0.1)) * hidden.sum(), rtol=1e-14)


def test_batch_rows_are_independent_tokens():
    e = inp.expert(4, 256, 256, 64, seed=19)
    X = inp.activations((5, 256), 19).astype(np.float64)
    args = (4, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
            e["down_codes"], e["down_scales"])
    hb, Yb, Ab = oracle.ffn_batch(*args, 5, 256, 256, 64, X)
    for t in range(5):
        h, y, a = oracle.ffn(*args, 256, 256, 64, X[t])
        assert (h == hb[t]).all() and (y == Yb[t]).all() and (a == Ab[t]).all()
    h2, Y2, _ = oracle.ffn_batch(*args, 5, 256, 256, 64, X, t0=2, nt=2)
    assert (Y2 == Yb[2:4]).all()
    _, Y0, _ = oracle.ffn_batch(*args, 0, 256, 256, 64, X[:0])
    assert Y0.shape == (0, 256)


# ------------------------------------------------------------------- bf16

@pytest.mark.parametrize("bits,value", [(0x3F80, 1.0), (0xC000, -2.0), (0x3E80, 0.25),
                                        (0x4049, 3.140625), (0x0001, 2.0 ** -133),
                                        (0x8000, -0.0), (0x7F80, math.inf)])
def test_bf16_widening(bits, value):
    assert oracle.bf16_value(bits) == value


def test_bf16_single_nonzero():
    rows, cols = 3, 16
    w = np.zeros((rows, cols), np.uint16)
    w[1, 5] = 0x4040                           # 3.0
    x = np.arange(cols, dtype=np.float64) - 4.0
    y, a = oracle.matvec_bf16(w, rows, cols, x)
    assert y.tolist() == [0.0, 3.0, 0.0] and a.tolist() == [0.0, 3.0, 0.0]


def test_bf16_generator_rounds_to_nearest_even():
    # inputs module: 1 + 2^-8 is a tie between bf16 1.0 and 1 + 2^-7 -> even (1.0);
    # 1 + 3*2^-8 is a tie -> even (1 + 2^-6)
    f = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5], np.float32)
    assert inp._f32_to_bf16_bits(f).tolist() == [0x3F80, 0x3F82, 0xC020]


# ------------------------------------------------------- threads and goldens

def test_threaded_rows_equal_serial():
    codes, s, x = _random_q(4, 97, 1024, 64, 20)
    old = oracle.get_threads()
    try:
        oracle.set_threads(1)
        y1, a1 = oracle.qgemv(4, codes, s, 97, 1024, 64, x)
        oracle.set_threads(7)
        y7, a7 = oracle.qgemv(4, codes, s, 97, 1024, 64, x)
    finally:
        oracle.set_threads(old)
    assert (y1 == y7).all() and (a1 == a7).all()


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4_ffn_256_seed0.txt")


def test_golden_q4_ffn_256_seed0_unchanged():
    """The stored oracle output of the 256/256 Q4 workload (written by
    tests/golden/make_golden.py, which calls only the oracle) still comes out."""
    from tests.golden import make_golden
    stored = make_golden.read(GOLDEN)
    now = make_golden.compute()
    for key in stored:
        np.testing.assert_allclose(now[key], stored[key], rtol=1e-15, atol=0)


# ------------------------------------------------------- routing / combine
# The pages leave selection and weighting open; these pin the readings in
# the oracle (largest logits first, ties to the lower index, NaN last,
# weights a softmax over the selected logits, combine in selection order).

def test_topk_order_and_ties():
    idx, w = oracle.topk(np.array([0.1, 3.0, -1.0, 3.0, 2.0]), 3)
    assert list(idx) == [1, 3, 4]            # 3 (index 1) before 3 (index 3), then 2
    assert w[0] == w[1] and w[2] < w[1]


def test_topk_nan_ranks_last_and_infinities():
    idx, w = oracle.topk(np.array([np.nan, -np.inf, 0.0, np.inf]), 3)
    assert list(idx) == [3, 2, 1]
    idx, _ = oracle.topk(np.array([np.nan, np.nan, 5.0]), 3)
    assert list(idx) == [2, 0, 1]            # two NaNs: lower index first


def test_topk_weights_are_a_distribution_invariant_to_shifts():
    rng = np.random.default_rng(3)
    l = rng.normal(size=128) * 3
    idx, w = oracle.topk(l, 8)
    assert abs(w.sum() - 1.0) < 1e-15 and (w > 0).all() and (np.diff(w) <= 0).all()
    idx2, w2 = oracle.topk(l + 1000.0, 8)
    assert list(idx2) == list(idx)
    np.testing.assert_allclose(w2, w, rtol=1e-12)


def test_topk_weight_ratio_of_logits_one_apart():
    # logits 1 apart: weight ratio e; equal logits: equal weights
    idx, w = oracle.topk(np.array([0.0, 1.0, 1.0, -5.0]), 3)
    assert list(idx) == [1, 2, 0]
    assert w[0] == w[1]
    assert abs(w[0] / w[2] - np.e) < 1e-14


def test_topk_all_experts_equal_logits_is_uniform():
    idx, w = oracle.topk(np.zeros(8), 8)
    assert list(idx) == list(range(8))
    np.testing.assert_allclose(w, np.full(8, 0.125), rtol=0, atol=1e-16)


def test_route_one_hot_gate_rows():
    # gate row e holds bf16 1.0 at column e: logit e = x[e]
    n, d = 6, 16
    g = np.zeros((n, d), np.uint16)
    for e in range(n):
        g[e, e] = 0x3F80
    x = np.array([0.5, -2.0, 4.0, 1.0, 4.0, -7.0] + [9.0] * (d - n))
    logits, a, idx, w = oracle.route(g, n, d, x, 2)
    np.testing.assert_array_equal(logits, x[:n])
    np.testing.assert_array_equal(a, np.abs(x[:n]))
    assert list(idx) == [2, 4] and w[0] == w[1] == 0.5


def test_combine_one_hot_and_linearity():
    rng = np.random.default_rng(4)
    eo = rng.normal(size=(3, 10))
    for i in range(3):
        w = np.zeros(3)
        w[i] = 1.0
        out, a = oracle.combine(eo, w)
        np.testing.assert_array_equal(out, eo[i])
        np.testing.assert_array_equal(a, np.abs(eo[i]))
    o1, _ = oracle.combine(eo, np.array([0.2, 0.3, 0.5]))
    o2, _ = oracle.combine(eo, np.array([0.4, 0.6, 1.0]))
    np.testing.assert_allclose(o2, 2 * o1, rtol=1e-15)


# -------------------------------------------------------------- mutations

MUTATIONS = [
    # (description, original text, planted slip); the first is the control
    ("control: no slip", "", ""),
    ("swapped nibbles", "(k % 2 == 0) ? (b & 0x0F) : (b >> 4)",
     "(k % 2 == 0) ? (b >> 4) : (b & 0x0F)"),
    ("wrong Z", "return bits == 4 ? 7.5 : 1.5;", "return bits == 4 ? 8.0 : 1.5;"),
    ("dropped offset", "return (code - z) / z * scale;", "return code / z * scale;"),
    ("scale of the wrong group", "(double)srow[k / c->group]", "(double)srow[k % c->group]"),
    ("SiLU on up", "hidden[i] = oracle_silu(gv[i]) * uv[i];",
     "hidden[i] = oracle_silu(uv[i]) * gv[i];"),
    ("crumb order reversed", "return (b >> (2 * (k % 4))) & 0x03;",
     "return (b >> (6 - 2 * (k % 4))) & 0x03;"),
    ("ties to the higher index", "return ia < ib;                   /* equal values",
     "return ia > ib;                   /* equal values"),
    ("NaN ranked first", "if (na != nb) return nb;", "if (na != nb) return na;"),
    ("weights not normalised", "for (long r = 0; r < k; ++r) w[r] /= sum;", "(void)sum;"),
    ("combine weight of the wrong row", "const double t = w[i] * eo[i * d_model + j];",
     "const double t = w[k - 1 - i] * eo[i * d_model + j];"),
]


@pytest.mark.parametrize("name,orig,slip", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_slips(name, orig, slip, tmp_path):
    """Builds a copy of the oracle with one slip planted and runs the pins
    above against it in a child process: at least one must fail."""
    if shutil.which(os.environ.get("CC", "gcc")) is None:
        pytest.skip("no C compiler")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "smoe_oracle.c")).read()
    if orig:
        assert src.count(orig) == 1, name
        src = src.replace(orig, slip)
    mdir = tmp_path / "oracle"
    mdir.mkdir()
    (mdir / "smoe_oracle.c").write_text(src)
    for f in ("__init__.py", "build.py"):
        shutil.copy(os.path.join(os.path.dirname(oracle.__file__), f), mdir / f)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=f"{tmp_path}{os.pathsep}{root}")
    r = subprocess.run(
        ["python", "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         "-k", "not pins_catch and not golden",
         os.path.join(root, "tests", "test_oracle_pins.py")],
        cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    if not orig:
        assert r.returncode == 0, f"the unmodified copy fails:\n{r.stdout[-2000:]}"
    else:
        assert r.returncode != 0, f"slip '{name}' went unnoticed:\n{r.stdout[-2000:]}"
        assert " failed" in r.stdout, r.stdout[-2000:]
