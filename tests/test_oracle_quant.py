"""Pins of the oracle's number formats (oracle/quant.py) and of its matvecs."""
import os

import numpy as np
import pytest

from oracle import quant as Q
from oracle.drafter import Matrix

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            out[key.strip()] = val.split()
    return out


def test_i8_rows_hand_cases():
    g = _golden("quant_cases.txt")
    x = np.array(g["i8_input"], dtype=np.float32)
    q, s = Q.quantize_rows_i8(x[None])
    assert q[0].tolist() == [int(v) for v in g["i8_codes"]]
    assert s[0] == np.float32(g["i8_scale"][0])


def test_q4_hand_cases():
    g = _golden("quant_cases.txt")
    w = np.array(g["q4_input"], dtype=np.float32)
    q, s = Q.quantize_q4g32(w[None])
    assert q[0].tolist() == [int(v) for v in g["q4_codes"]]
    assert float(s[0, 0]) == float(g["q4_scale"][0])
    wb = np.zeros(32, dtype=np.float32)
    vals = np.array(g["q4b_input"], dtype=np.float32)
    wb[:len(vals)] = vals
    q, s = Q.quantize_q4g32(wb[None])
    assert q[0, :len(vals)].tolist() == [int(v) for v in g["q4b_codes"]]
    assert float(s[0, 0]) == float(g["q4b_scale"][0])
    assert (q[0, len(vals):] == 0).all()


def test_zero_rows_and_groups():
    q, s = Q.quantize_rows_i8(np.zeros((2, 40), np.float32))
    assert (q == 0).all() and (s == 0).all()
    w = np.random.default_rng(0).standard_normal((3, 96)).astype(np.float32)
    w[1, 32:64] = 0
    q, s = Q.quantize_q4g32(w)
    assert s[1, 1] == 0 and (q[1, 32:64] == 0).all()


def test_q4_round_trip_bound():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    q, s = Q.quantize_q4g32(w)
    assert q.min() >= -8 and q.max() <= 7
    sf = s.astype(np.float32).astype(np.float64)
    err = np.abs(w.astype(np.float64) - Q.dequant_q4g32(q, s, np.float64))
    bound = np.repeat(sf, 32, axis=1) / 2
    assert (err <= bound * (1 + 1e-6)).all()
    # every group's largest magnitude lands on the top code (+-7 or -8)
    assert (np.abs(q).reshape(64, 8, 32).max(axis=-1) >= 7).all()


def test_i8_round_trip_bound():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((8, 300)).astype(np.float32)
    q, s = Q.quantize_rows_i8(x)
    assert (np.abs(q).max(axis=1) == 127).all()
    err = np.abs(x.astype(np.float64) - q.astype(np.float64) * s.astype(np.float64)[:, None])
    assert (err <= s.astype(np.float64)[:, None] / 2 * (1 + 1e-5)).all()


def test_group_sums_brute_force():
    """acc[t,n,g] against scalar integer loops (tiny shapes)."""
    rng = np.random.default_rng(3)
    qx = rng.integers(-127, 128, size=(3, 64), dtype=np.int64)
    qw = rng.integers(-8, 8, size=(5, 64), dtype=np.int64)
    acc = Q.q4_group_sums(qx, qw)
    for t in range(3):
        for n in range(5):
            for g in range(2):
                ref = 0
                for k in range(32 * g, 32 * g + 32):
                    ref += int(qx[t, k]) * int(qw[n, k])
                assert acc[t, n, g] == ref


def test_dequant_matvec_equals_definition():
    """The oracle applies 4-bit matrices as the dequantised product; that must
    equal the integer group-sum definition (up to float64 rounding)."""
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((48, 160)) * 0.02).astype(np.float32)
    x = rng.standard_normal((5, 160)).astype(np.float64)
    m = Matrix(w, "q4g32")
    y = m.apply(x)
    qx, sx = Q.quantize_rows_i8(x)
    ref = Q.q4_matvec_by_definition(qx, sx, m.q, m.s)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_head_matvec_equals_definition():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((37, 96)) * 0.02).astype(np.float32)
    x = rng.standard_normal((4, 96))
    m = Matrix(w, "i8row")
    qx, sx = Q.quantize_rows_i8(x)
    ref = Q.i8_matvec_by_definition(qx, sx, m.q, m.s)
    np.testing.assert_allclose(m.apply(x), ref, rtol=1e-13, atol=0)


def test_f32_matrix_is_plain_product():
    rng = np.random.default_rng(6)
    w = rng.standard_normal((7, 33)).astype(np.float32)
    x = rng.standard_normal((3, 33))
    y = Matrix(w, "f32").apply(x)
    for t in range(3):
        for n in range(7):
            assert y[t, n] == pytest.approx(sum(float(w[n, k]) * x[t, k] for k in range(33)), rel=1e-12)
