"""Pins of the oracle's context handling and block: incremental append equals
full recomputation, the page's position rules, and closed forms of the block."""
import dataclasses

import numpy as np
import pytest

import workloads as W
from oracle import OracleModel, OracleSeq, block, rms
from oracle import quant as Q


@pytest.fixture(scope="module", params=["tiny_f32", "small_q4_hd64"])
def model(request):
    wl = W.WORKLOADS[request.param]
    return OracleModel(wl.geom, W.make_weights(wl.geom)), wl


def _kv(seq):
    return [np.concatenate([k, v]) for k, v in zip(seq.k, seq.v)]


def test_incremental_append_equals_full(model):
    m, wl = model
    taps = W.make_taps(m.g, 70)
    full = OracleSeq(m)
    full.append(0, taps)
    for step in (1, 7, 64):
        s = OracleSeq(m)
        for r0 in range(0, 70, step):
            s.append(r0, taps[r0:r0 + step])
        assert s.len == 70 and s.first == 0
        for a, b in zip(_kv(s), _kv(full)):
            np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_truncate_then_reappend_equals_fresh(model):
    m, _ = model
    taps = W.make_taps(m.g, 30)
    other = W.make_taps(m.g, 30, call_id=9)
    s = OracleSeq(m)
    s.append(0, taps)
    s.truncate(12)
    assert s.next_position() == 12
    s.append(12, other[12:])
    fresh = OracleSeq(m)
    fresh.append(0, np.concatenate([taps[:12], other[12:]]))
    for a, b in zip(_kv(s), _kv(fresh)):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_position_rules(model):
    m, _ = model
    taps = W.make_taps(m.g, 10)
    s = OracleSeq(m)
    s.append(5, taps[:4])                   # empty context: starts at 5
    assert (s.first, s.len) == (5, 4)
    s.append(7, taps[4:6])                  # a held position replaces it and what follows
    assert (s.first, s.len) == (5, 4)
    s.append(20, taps[:2])                  # a gap starts the context over
    assert (s.first, s.len) == (20, 2)
    s.append(3, taps[:1])                   # before the first: over again
    assert (s.first, s.len) == (3, 1)
    s.reset()
    assert (s.first, s.len, s.next_position()) == (0, 0, 0)
    # a block reads [first, min(anchor, first + len))
    s.append(0, taps)
    assert s.ctx_range(0, 6) == (0, 6)
    assert s.ctx_range(0, 50) == (0, 10)


def test_window_covering_everything_equals_no_window(model):
    m, wl = model
    g2 = dataclasses.replace(m.g, window=10 ** 6)
    m2 = OracleModel(g2, W.make_weights(m.g))
    taps = W.make_taps(m.g, 20)
    s1, s2 = OracleSeq(m), OracleSeq(m2)
    s1.append(0, taps)
    s2.append(0, taps)
    l1, t1 = block(m, s1, 3, 20)
    l2, t2 = block(m2, s2, 3, 20)
    np.testing.assert_array_equal(l1, l2)


def test_zero_output_projections_closed_form(model):
    """With Wo = Wd = 0 in every layer the residual stream never changes, so
    every draft row's logits are head . Q(rms(embed[mask], norm)): one matvec."""
    m, wl = model
    g = m.g
    w = W.make_weights(g)
    for lw in w["layers"]:
        lw["o"][:] = 0
        lw["down"][:] = 0
    mz = OracleModel(g, w)
    s = OracleSeq(mz)
    s.append(0, W.make_taps(g, 9))
    logits, toks = block(mz, s, 11, 9)
    hn = rms(w["embed"][g.mask][None].astype(np.float64), w["norm"], g.eps)
    if g.quant:
        qh, sh = Q.quantize_rows_i8(w["head"])
        qx, sx = Q.quantize_rows_i8(hn)
        ref = Q.i8_matvec_by_definition(qx, sx, qh, sh)[0]
    else:
        ref = hn[0] @ w["head"].astype(np.float64).T
    for r in range(g.block - 1):
        np.testing.assert_allclose(logits[r], ref, rtol=1e-12, atol=1e-13)
    assert (toks == np.argmax(ref.astype(np.float32))).all()


def test_block_shapes_and_shorter_block(model):
    m, wl = model
    s = OracleSeq(m)
    s.append(0, W.make_taps(m.g, 12))
    logits, toks = block(m, s, 5, 12, block_len=3)
    assert logits.shape == (2, m.g.vocab) and toks.shape == (2,)
    with pytest.raises(ValueError):
        block(m, s, 5, 12, block_len=1)
    with pytest.raises(ValueError):
        block(m, s, 5, 12, block_len=m.g.block + 1)
