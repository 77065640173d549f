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


# ------------------------------------------------------------ attention variants
def _one_layer(m, **kw):
    g1 = dataclasses.replace(m.g, layers=1, **kw)
    return g1, W.make_weights(g1)


def test_window_row_equals_a_shorter_context(model):
    """With one layer a draft row's logits depend on its own attention only,
    so row r under a window w equals row r of an unwindowed block whose
    context holds only the positions that row may see (>= anchor + r + 1 - w):
    the row-dependent mask of page "cortiq-engine 0.8.71 — src/dflash.rs",
    `Drafter::block`, checked against plain truncation."""
    m, _ = model
    w_ = 5
    g1, wts = _one_layer(m)
    gw = dataclasses.replace(g1, window=w_)
    m_all, m_win = OracleModel(g1, wts), OracleModel(gw, wts)
    n = 20
    taps = W.make_taps(g1, n)
    sw = OracleSeq(m_win)
    sw.append(0, taps)
    lw, _ = block(m_win, sw, 7, n)
    for r in range(1, g1.block):
        start = n + r + 1 - w_
        s = OracleSeq(m_all)
        if start < n:
            s.append(start, taps[start:])
        lr, _ = block(m_all, s, 7, n)
        np.testing.assert_allclose(lw[r - 1], lr[r - 1], rtol=1e-12, atol=1e-13)


def test_windows_list_equals_one_window(model):
    """The per-layer list with every entry w is the one window w; entries
    that cover the whole context are no window."""
    m, _ = model
    g = m.g
    wts = W.make_weights(g)
    taps = W.make_taps(g, 24)
    outs = []
    for kw in ({"window": 6}, {"windows": (6,) * g.layers}, {"windows": (10 ** 6,) * g.layers}, {}):
        mm = OracleModel(dataclasses.replace(g, **kw), wts)
        s = OracleSeq(mm)
        s.append(0, taps)
        outs.append(block(mm, s, 5, 24)[0])
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[2], outs[3])
    assert not np.allclose(outs[0], outs[3])  # the window does cut something


def test_drop_keeps_what_the_window_sees(model):
    """Rows that fell out of every window are dropped as the context grows
    (`settle_rows`); appending in small chunks drops at other moments than
    one append does, and a block at the end reads the same rows either way."""
    m, _ = model
    g = dataclasses.replace(m.g, window=5)
    mm = OracleModel(g, W.make_weights(m.g))
    taps = W.make_taps(g, 60)
    one, chunked = OracleSeq(mm), OracleSeq(mm)
    one.append(0, taps)
    for r0 in range(0, 60, 7):
        chunked.append(r0, taps[r0:r0 + 7])
    assert one.dropped[0] == 55 and chunked.dropped[0] != one.dropped[0]
    assert all(one.len - d <= 2 * 5 for d in chunked.dropped)
    # (the projections of a row differ between the passes only in the order of the sums)
    np.testing.assert_allclose(block(mm, one, 9, 60)[0], block(mm, chunked, 9, 60)[0], rtol=1e-12, atol=1e-13)


def test_no_rope_layers_see_the_context_as_a_set(model):
    """Without the rotary position a layer's attention cannot tell the order
    of its context rows: reversing the context leaves every logit (up to the
    order of the sums); with it, reversing changes them."""
    m, _ = model
    g = m.g
    wts = W.make_weights(g)
    taps = W.make_taps(g, 16)
    res = {}
    for name, kw in (("plain", {}), ("no_rope", {"no_rope": tuple(range(g.layers))})):
        mm = OracleModel(dataclasses.replace(g, **kw), wts)
        a, b = OracleSeq(mm), OracleSeq(mm)
        a.append(0, taps)
        b.append(0, taps[::-1].copy())
        res[name] = (block(mm, a, 3, 16)[0], block(mm, b, 3, 16)[0])
    la, lb = res["no_rope"]
    np.testing.assert_allclose(la, lb, rtol=1e-9, atol=1e-10 * np.max(np.abs(la)))
    pa, pb = res["plain"]
    assert np.max(np.abs(pa - pb)) > 1e-6 * np.max(np.abs(pa))


@pytest.mark.parametrize("window", [0, 3, 5, 12, 40])
def test_zero_queries_average_the_visible_values(window):
    """With Wq = 0 every score is 0, so each query head's output is the plain
    mean of its KV head's values over exactly the keys its row sees: the
    context positions in the row's window plus every block row (the block is
    not causal).  With Wd = 0 as well, each layer adds Wo . mean to the rows,
    and the block reduces to sums and matrix products written out here,
    with no softmax, key ordering or position bookkeeping of the oracle's."""
    wl = W.WORKLOADS["tiny_f32"]
    g = dataclasses.replace(wl.geom, window=window)
    w = W.make_weights(g)
    for lw in w["layers"]:
        lw["q"][:] = 0
        lw["down"][:] = 0
    n, anchor, tok = 30, 30, 17
    taps = W.make_taps(g, n)
    mz = OracleModel(g, w)
    s = OracleSeq(mz)
    s.append(0, taps)
    logits, _ = block(mz, s, tok, anchor)

    f64 = lambda a: np.asarray(a, dtype=np.float64)

    def norm_rows(x, gain):
        return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + g.eps) * f64(gain)

    rows, kv, hd, rep = g.block, g.kv_heads, g.head_dim, g.rep
    t = norm_rows(f64(taps) @ f64(w["fc"]).T, w["hidden_norm"])
    h = f64(w["embed"][[tok] + [g.mask] * (rows - 1)])
    for lw in w["layers"]:
        vc = (t @ f64(lw["v"]).T).reshape(n, kv, hd)
        vb = (norm_rows(h, lw["in_norm"]) @ f64(lw["v"]).T).reshape(rows, kv, hd)
        y = np.empty((rows, g.heads, hd))
        for r in range(rows):
            # row r sits at position anchor + r and sees the context from
            # anchor + r + 1 - window on (none of it once that is past the end)
            lo = min(max(anchor + r + 1 - window, 0), n) if window else 0
            mean = (vc[lo:].sum(0) + vb.sum(0)) / (n - lo + rows)  # [kv, hd]
            y[r] = mean[np.arange(g.heads) // rep]
        h = h + y.reshape(rows, -1) @ f64(lw["o"]).T
    ref = norm_rows(h[1:], w["norm"]) @ f64(w["head"]).T
    np.testing.assert_allclose(logits, ref, rtol=1e-10, atol=1e-12 * np.max(np.abs(ref)))


def test_block_depends_only_on_relative_positions(model):
    """Rotary attention sees only position differences, so the same context
    held from position 0 or from position 64, with the block anchored the
    same distance after it, gives the same logits up to the rounding of the
    angles: each is one f32 product position x inv_freq, off by at most
    2^-24 of itself (under 1e-5 rad for positions below 110), which moves a
    logit by far less than the 1e-4 of max|logit| allowed here.  A block
    anchored one position later -- the off-by-one the test guards against --
    moves the logits by over a tenth of max|logit|."""
    m, _ = model
    taps = W.make_taps(m.g, 21)
    a, b = OracleSeq(m), OracleSeq(m)
    a.append(0, taps)
    b.append(64, taps)
    assert (b.first, b.len) == (64, 21)
    la, ta = block(m, a, 9, 21)
    lb, tb = block(m, b, 9, 85)
    top = np.max(np.abs(la))
    np.testing.assert_allclose(la, lb, rtol=0, atol=1e-4 * top)
    assert (ta == tb).all()
    lc, _ = block(m, a, 9, 22)
    assert np.max(np.abs(lc - la)) > 1e-2 * top


# ------------------------------------------------------------ row convolution
def test_row_conv_shift_closed_form():
    """Kernels of two rows with no dynamic part: output = (I + c S) x with S
    the one-row shift, as a matrix product."""
    from oracle import row_conv
    rng = np.random.default_rng(5)
    rows, hs, gs = 7, 12, 4
    x = rng.standard_normal((rows, hs))
    c = rng.standard_normal(hs)
    base = np.zeros((2, 2, hs))
    base[1, 0] = 1.0
    base[1, 1] = c
    d = np.zeros((rows, 2 * 2 * (hs // gs)))
    y = row_conv(base, d, x, 1, 2, gs)
    shift = np.eye(rows, k=-1)
    np.testing.assert_allclose(y, x + (shift @ x) * c, rtol=1e-14, atol=1e-15)
    # stage 0 of the same base is all zeros here
    np.testing.assert_array_equal(row_conv(base, d, x, 0, 2, gs), np.zeros_like(x))


def test_row_conv_dynamic_kernel_indexing():
    """A projection whose (stage 1, offset 0, group g) row picks column j_g of
    the row and a zero base: output column i = x[r, j_{g(i)}] * x[r, i],
    by fancy indexing -- the dynamic kernels' (stage, offset, group) order."""
    from oracle import row_conv
    rng = np.random.default_rng(6)
    rows, hs, gs, kn = 5, 16, 4, 3
    groups = hs // gs
    x = rng.standard_normal((rows, hs))
    pick = rng.integers(0, hs, size=groups)
    proj = np.zeros((2 * kn * groups, hs))
    for g_ in range(groups):
        proj[(1 * kn + 0) * groups + g_, pick[g_]] = 1.0
    d = x @ proj.T
    y = row_conv(np.zeros((2, kn, hs)), d, x, 1, kn, gs)
    ref = x * x[:, pick][:, np.arange(hs) // gs]
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-15)


def test_bypass_convolution_is_no_convolution(model):
    """kn = 1, base 1, projection 0: the convolution passes every row
    unchanged, so the block equals the unwrapped one exactly."""
    m, _ = model
    g = m.g
    gc = dataclasses.replace(g, conv_kernel=1, conv_group=g.hidden // 4)
    w = W.make_weights(gc)
    for lw in w["layers"]:
        for c in ("attn_conv", "mlp_conv"):
            lw[c + "_base"][:] = 1
            lw[c + "_proj"][:] = 0
    plain = {k: v for k, v in w.items() if k != "layers"}
    plain["layers"] = [{k: v for k, v in lw.items() if "conv" not in k} for lw in w["layers"]]
    mc, mp = OracleModel(gc, w), OracleModel(g, plain)
    taps = W.make_taps(g, 12)
    sc, sp = OracleSeq(mc), OracleSeq(mp)
    sc.append(0, taps)
    sp.append(0, taps)
    np.testing.assert_array_equal(block(mc, sc, 4, 12)[0], block(mp, sp, 4, 12)[0])


def test_single_row_kernel_folds_into_weights():
    """kn = 1 with no dynamic part scales columns: stage 0 of the attention
    convolution is a factor on in_norm's gains, its stage 1 one on O's output
    rows; the MLP's likewise on post_norm and on down's rows (all-f32 drafter,
    so the folded weights are exact)."""
    g = dataclasses.replace(W.WORKLOADS["tiny_f32"].geom, conv_kernel=1, conv_group=64)
    w = W.make_weights(g)
    rng = np.random.default_rng(8)
    for lw in w["layers"]:
        for c in ("attn_conv", "mlp_conv"):
            lw[c + "_proj"][:] = 0
            # powers of two: the folded float32 weights are exact
            lw[c + "_base"][:] = 2.0 ** rng.integers(-2, 3, size=lw[c + "_base"].shape)
    folded = {k: v for k, v in w.items() if k != "layers"}
    folded["layers"] = []
    for lw in w["layers"]:
        f = {k: v.copy() for k, v in lw.items() if "conv" not in k}
        f["in_norm"] = (lw["in_norm"].astype(np.float64) * lw["attn_conv_base"][0, 0]).astype(np.float64)
        f["o"] = lw["o"].astype(np.float64) * lw["attn_conv_base"][1, 0][:, None]
        f["post_norm"] = lw["post_norm"].astype(np.float64) * lw["mlp_conv_base"][0, 0]
        f["down"] = lw["down"].astype(np.float64) * lw["mlp_conv_base"][1, 0][:, None]
        folded["layers"].append(f)
    g0 = dataclasses.replace(g, conv_kernel=0, conv_group=0)
    mc, mf = OracleModel(g, w), OracleModel(g0, folded)
    taps = W.make_taps(g, 10)
    sc, sf = OracleSeq(mc), OracleSeq(mf)
    sc.append(0, taps)
    sf.append(0, taps)
    lc, lf = block(mc, sc, 2, 10)[0], block(mf, sf, 2, 10)[0]
    np.testing.assert_allclose(lc, lf, rtol=1e-10, atol=1e-12 * np.max(np.abs(lf)))


def test_convolution_is_causal_over_the_block_rows(model):
    """Row r's draft depends on rows <= r only: a longer block's first rows
    equal a shorter block's (a convolution looking ahead would change them
    through the later rows).  Attention mixes every block row, so it is taken
    out (Wo = 0) and the rows meet only in the convolutions."""
    m, _ = model
    g = dataclasses.replace(m.g, conv_kernel=3, conv_group=m.g.hidden // 4)
    w = W.make_weights(g)
    for lw in w["layers"]:
        lw["o"][:] = 0  # attention mixes all block rows; take it out
    mc = OracleModel(g, w)
    s = OracleSeq(mc)
    s.append(0, W.make_taps(g, 9))
    long_, _ = block(mc, s, 6, 9, block_len=g.block)
    short, _ = block(mc, s, 6, 9, block_len=4)
    np.testing.assert_allclose(long_[:3], short, rtol=1e-12, atol=1e-13 * np.max(np.abs(short)))


# ------------------------------------------------------------ candidate selector
def _sel_model(top, rank=2):
    g = dataclasses.replace(W.WORKLOADS["tiny_f32"].geom, selector_rank=rank, selector_top=top)
    return g, W.make_weights(g)


def test_selector_with_a_zero_codebook_keeps_each_rows_top():
    """C = 0: every candidate scores its own logit, so the selector returns
    each row's top token (the plain argmax, first of equals)."""
    g, w = _sel_model(top=8)
    w["successor_codebook"][:] = 0
    m = OracleModel(g, w)
    s = OracleSeq(m)
    s.append(0, W.make_taps(g, 12))
    logits, toks = block(m, s, 7, 12)
    np.testing.assert_array_equal(toks, np.argmax(logits.astype(np.float32), axis=1))


def test_selector_chains_the_previous_choice():
    """Codebooks built so that the anchor's predecessor row points every
    candidate score at token t1 and t1's at t2 (C rows one-hot, other P rows
    zero): the first two rows choose t1 then t2 over any logit, the rest keep
    their own top token -- the anchor feeds row 0 and each choice the next."""
    g_vocab = W.WORKLOADS["tiny_f32"].geom.vocab
    g, w = _sel_model(top=g_vocab)
    m0 = OracleModel(g, w)
    s0 = OracleSeq(m0)
    s0.append(0, W.make_taps(g, 12))
    anchor = 7
    logits, _, hn = block(m0, s0, anchor, 12, return_hidden=True)
    hp = hn[1:] @ w["selector_projection"].astype(np.float64).T
    plain = np.argmax(logits.astype(np.float32), axis=1)
    t1, t2 = [t for t in range(g_vocab) if t not in set(plain.tolist()) | {anchor}][:2]
    P = np.zeros((g.vocab, 2), dtype=np.float16)
    C = np.zeros((g.vocab, 2), dtype=np.float16)
    C[t1, 0] = C[t2, 1] = 1
    P[anchor, 0] = np.float16(1e4 * np.sign(hp[0, 0]))
    P[t1, 1] = np.float16(1e4 * np.sign(hp[1, 1]))
    w["predecessor_codebook"], w["successor_codebook"] = P, C
    m = OracleModel(g, w)
    s = OracleSeq(m)
    s.append(0, W.make_taps(g, 12))
    _, toks = block(m, s, anchor, 12)
    assert toks[0] == t1 and toks[1] == t2
    np.testing.assert_array_equal(toks[2:], plain[2:])


# ------------------------------------------------------------ context queue
def test_queue_then_settle_equals_append(model):
    """Rows queued in several calls and settled by the block read the same
    context as one append (page 1's queue_context / settle): the same keys
    and values, the same block."""
    m, _ = model
    taps = W.make_taps(m.g, 40)
    a, q = OracleSeq(m), OracleSeq(m)
    a.append(0, taps)
    for r0 in (0, 9, 23):
        q.queue(r0, taps[r0:r0 + (9 if r0 == 0 else 14 if r0 == 9 else 17)])
    assert q.len == 0 and q.next_position() == 40 and q.pending.shape[0] == 40
    la, _ = block(m, a, 3, 40)
    lq, _ = block(m, q, 3, 40)
    assert q.len == 40 and q.pending.shape[0] == 0
    for x, y in zip(_kv(a), _kv(q)):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(la, lq, rtol=1e-12, atol=1e-13)


def test_queue_limit_settles_the_oldest_in_chunks(model):
    """Past PENDING_ROWS waiting rows the oldest are settled, a multiple of 64
    of them; with every layer windowed the limit is the widest window plus
    the slack where that is larger."""
    m, _ = model
    s = OracleSeq(m)
    s.queue(0, W.make_taps(m.g, 500))
    assert (s.len, s.pending.shape[0]) == (0, 500)
    s.queue(500, W.make_taps(m.g, 100, call_id=2))      # 600 waiting: 88 over -> 128 settle
    assert (s.len, s.pending.shape[0], s.next_position()) == (128, 472, 600)
    gw = dataclasses.replace(m.g, window=700)
    mw = OracleModel(gw, W.make_weights(m.g))
    sw = OracleSeq(mw)
    sw.queue(0, W.make_taps(gw, 900))                     # limit 700 + 256 = 956: nothing settles
    assert (sw.len, sw.pending.shape[0]) == (0, 900)


def test_truncate_cuts_queued_rows_first(model):
    m, _ = model
    s = OracleSeq(m)
    taps = W.make_taps(m.g, 30)
    s.append(0, taps[:10])
    s.queue(10, taps[10:30])
    s.truncate(25)
    assert (s.len, s.pending.shape[0], s.next_position()) == (10, 15, 25)
    s.truncate(6)
    assert (s.len, s.pending.shape[0], s.next_position()) == (6, 0, 6)
    s.queue(4, taps[4:9])                                 # a held position: replaces from 4 on
    assert (s.len, s.pending.shape[0], s.next_position()) == (4, 5, 9)
    fresh = OracleSeq(m)
    fresh.append(0, taps[:9])
    np.testing.assert_allclose(block(m, s, 1, 9)[0], block(m, fresh, 1, 9)[0], rtol=1e-12, atol=1e-13)
