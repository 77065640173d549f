"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs, at sizes the oracle finishes in seconds (several
tiles, ragged vocabulary and context tails).

Bars: integer work bit-exact (4-bit and int8 codes, f16 and f32 scales, the
int32 group sums); f32 config logits within 1e-4 * max|logit|; quantised
logits within 2e-3 * max|logit|; draft tokens equal wherever the oracle's
top two logits are further apart than the logits' tolerance.
"""
import dataclasses

import numpy as np
import pytest

import workloads as W
from oracle import OracleModel, OracleSeq, block
from oracle import quant as Q

pytestmark = pytest.mark.gpu

TOL = {0: 1e-4, 1: 2e-3}  # relative to max|oracle logit|, by geometry.quant


def _dfl():
    import block_speculative_drafting_gb300 as dfl
    return dfl


class Pair:
    """A GPU model and an oracle model on the same weights."""

    def __init__(self, name, edit=None, **changes):
        wl = W.WORKLOADS[name]
        self.wl = wl
        self.g = dataclasses.replace(wl.geom, **changes) if changes else wl.geom
        self.w = W.make_weights(self.g)
        if edit is not None:
            edit(self.w)  # a special case's weights, changed in place before either side sees them
        self.gpu = _dfl().Model(self.g, self.w)
        self.ora = OracleModel(self.g, self.w)


_pairs = {}


def pair(name):
    if name not in _pairs:
        _pairs[name] = Pair(name)
    return _pairs[name]


def decision_noise(om, osq, anchor, anchor_pos, bl, ref, runs=2):
    """max |logits - ref| / max|ref| of the oracle against itself when the
    values it quantises carry f32-level noise (1e-7 relative): the spread
    that differing rounding-boundary decisions alone produce."""
    from oracle import quant as Q
    orig = Q.quantize_rows_i8
    rng = np.random.default_rng(123)
    devs = []
    try:
        Q.quantize_rows_i8 = lambda x: orig(np.asarray(x, np.float64) * (1 + 1e-7 * rng.standard_normal(np.shape(x))))
        for _ in range(runs):
            lp, _ = block(om, osq, anchor, anchor_pos, bl)
            devs.append(float(np.max(np.abs(lp - ref))) / float(np.max(np.abs(ref))))
    finally:
        Q.quantize_rows_i8 = orig
    return max(devs)


def check_logits(g, got, ref, tol_scale=1.0, noise=None):
    """f32 format: max |got - ref| <= 1e-4 * max|ref|.  Quantised format: the
    same with 2e-3, or, where the two sides' own quantisation decisions differ
    at rounding boundaries (free running), within three times the oracle's own
    decision-noise spread (`noise()` computes it when needed); the
    identical-decision tests hold the quantised path to 1e-5."""
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    tol = TOL[g.quant] * tol_scale * scale
    if err > tol and g.quant and noise is not None:
        tol = max(tol, 3 * noise() * scale + tol)
    assert err <= tol, f"max|dlogit| {err:.3e} > {tol:.3e}"
    return err / scale


def check_tokens(got_tok, ref_logits, tol_abs):
    ref32 = ref_logits.astype(np.float32)
    ref_tok = np.argmax(ref32, axis=-1)
    srt = np.sort(ref32, axis=-1)
    margin = srt[..., -1] - srt[..., -2]
    decided = margin > 2 * tol_abs
    got_tok = np.asarray(got_tok).reshape(ref_tok.shape)
    assert (got_tok[decided] == ref_tok[decided]).all()
    return float(np.mean(got_tok == ref_tok))


# ---------------------------------------------------------------- integer work
@pytest.mark.parametrize("name", ["small_q4", "small_q4_hd64"])
def test_q4_codes_and_scales_bit_exact(name):
    dfl = _dfl()
    p = pair(name)
    g = p.g
    mats = [(dfl.MAT_FC, p.w["fc"])]
    for l in range(g.layers):
        for which in dfl._abi.MAT_NAMES:
            mats.append((dfl.mat_layer(l, which), p.w["layers"][l][which]))
    for mid, w in mats:
        codes, scales = p.gpu.q4_codes(mid, *w.shape)
        rq, rs = Q.quantize_q4g32(w)
        np.testing.assert_array_equal(codes, rq)
        np.testing.assert_array_equal(scales.view(np.uint16), rs.view(np.uint16))


@pytest.mark.parametrize("name", ["small_q4", "small_q4_hd64"])
def test_head_codes_bit_exact(name):
    p = pair(name)
    codes, scales = p.gpu.head_codes()
    rq, rs = Q.quantize_rows_i8(p.w["head"])
    np.testing.assert_array_equal(codes, rq)
    np.testing.assert_array_equal(scales.view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("rows", [16, 5, 1])
def test_group_sums_bit_exact(rows):
    dfl = _dfl()
    p = pair("small_q4")
    rng = np.random.default_rng(rows)
    for mid, w in [(dfl.MAT_FC, p.w["fc"]), (dfl.mat_layer(1, "down"), p.w["layers"][1]["down"]),
                   (dfl.mat_layer(0, "k"), p.w["layers"][0]["k"])]:
        x = rng.integers(-127, 128, size=(rows, w.shape[1]), dtype=np.int8)
        x[0, :7] = 127
        x[-1, -9:] = -127
        got = p.gpu.q4_groupsums(mid, x, w.shape[0])
        rq, _ = Q.quantize_q4g32(w)
        np.testing.assert_array_equal(got, Q.q4_group_sums(x, rq).astype(np.int32))


@pytest.mark.parametrize("name,rows", [("small_q4", 300), ("small_q4", 17), ("small_q4", 128),
                                       ("small_q4_hd64", 200), ("small_q4", 9)])
def test_q4_matmul_matches_definition(name, rows):
    """The library's 4-bit matmul on given int8 rows (streaming kernel up to
    16 rows, tcgen05 kernel beyond: several 128-row tiles, ragged rows,
    sub-matrices at a row offset inside fused matrices, a ragged 256-row
    weight tile) against the quantised definition on the library's own codes:
    every product is exact on both paths, only the f32 accumulation rounds."""
    dfl = _dfl()
    p = pair(name)
    rng = np.random.default_rng(rows)
    mats = [(dfl.MAT_FC, p.w["fc"])]
    for which in ("q", "k", "up", "down"):
        mats.append((dfl.mat_layer(1, which), p.w["layers"][1][which]))
    for mid, w in mats:
        x = rng.integers(-127, 128, size=(rows, w.shape[1]), dtype=np.int8)
        x[0, :7] = 127
        x[-1, -9:] = -127
        xs = (rng.random(rows).astype(np.float32) + 0.5) / 127
        got = p.gpu.q4_matmul(mid, x, xs, w.shape[0])
        codes, scales = p.gpu.q4_codes(mid, *w.shape)
        ref = Q.q4_matvec_by_definition(x, xs, codes, scales.view(np.float16))
        err = float(np.max(np.abs(got - ref)))
        assert err <= 2e-5 * float(np.max(np.abs(ref))), (mid, err, float(np.max(np.abs(ref))))


def test_converter_path_matches():
    """With the "dense" option off the many-row matmuls and the head
    dequantise their weights in the tensor-core kernels instead of reading the
    dense f16 copies: the matmul against the quantised definition, and a
    batched block (matmuls and head) with identical decisions, to the same
    bounds as the default path."""
    dfl = _dfl()
    p = Pair("small_q4")
    p.gpu.option("dense", 0)
    rng = np.random.default_rng(11)
    for mid, w in [(dfl.MAT_FC, p.w["fc"]), (dfl.mat_layer(0, "up"), p.w["layers"][0]["up"])]:
        x = rng.integers(-127, 128, size=(300, w.shape[1]), dtype=np.int8)
        xs = (rng.random(300).astype(np.float32) + 0.5) / 127
        got = p.gpu.q4_matmul(mid, x, xs, w.shape[0])
        codes, scales = p.gpu.q4_codes(mid, *w.shape)
        ref = Q.q4_matvec_by_definition(x, xs, codes, scales.view(np.float16))
        assert float(np.max(np.abs(got - ref))) <= 2e-5 * float(np.max(np.abs(ref)))
    g = p.g
    lens = [7, 0, 33, 12]
    sc = Script(p, len(lens), 48)
    for i, n in enumerate(lens):
        sc.append(i, 0, W.make_taps(g, n, call_id=60 + i))
    sc.block(list(range(len(lens))), [11, 12, 13, 14], lens, g.block)
    sc.run(True).check(True)


def test_head_norm_guard_recompute_matches():
    """The dense head trusts its f32 tensor-memory sums only while the product
    of the two rows' code norms keeps every partial sum within 2^24 (Cauchy-
    Schwarz); past it an element is recomputed as an integer dot product.
    The "head_bound" option at 0 sends every element down that path: a
    batched block must still give the oracle's logits and identical decisions."""
    p = Pair("small_q4")
    p.gpu.option("head_bound", 0)
    lens = [5, 40, 0, 21]
    sc = Script(p, len(lens), 48)
    for i, n in enumerate(lens):
        sc.append(i, 0, W.make_taps(p.g, n, call_id=80 + i))
    sc.block(list(range(len(lens))), [21, 22, 23, 24], lens, p.g.block)
    sc.run(True).check(True)


# ---------------------------------------------------------------- context append
@pytest.mark.parametrize("name", ["tiny_f32", "small_q4", "small_q4_hd64"])
def test_kv_append_matches_oracle(name):
    p = pair(name)
    g, n = p.g, p.wl.ctx
    taps = W.make_taps(g, n, call_id=3)
    seq = p.gpu.new_sequence(n + 8)
    p.gpu.ctx_append(seq, 5, taps)
    assert seq.span() == (5, 5 + n)
    osq = OracleSeq(p.ora)
    osq.append(5, taps)
    tol = 1e-5 if g.quant == 0 else 2e-3
    for l in range(g.layers):
        k, v = p.gpu.read_kv(seq, l, 5, n)
        rk, rv = osq.k[l].transpose(1, 0, 2), osq.v[l].transpose(1, 0, 2)
        assert np.max(np.abs(k - rk)) <= tol * np.max(np.abs(rk))
        assert np.max(np.abs(v - rv)) <= tol * np.max(np.abs(rv))
    seq.close()


def test_append_in_chunks_equals_at_once():
    p = pair("small_q4")
    g = p.g
    taps = W.make_taps(g, 40, call_id=4)
    a = p.gpu.new_sequence(64)
    p.gpu.ctx_append(a, 0, taps)
    b = p.gpu.new_sequence(64)
    for r0, step in [(0, 1), (1, 7), (8, 13), (21, 19)]:
        p.gpu.ctx_append(b, r0, taps[r0:r0 + step])
    assert b.span() == (0, 40)
    for l in range(g.layers):
        ka, va = p.gpu.read_kv(a, l, 0, 40)
        kb, vb = p.gpu.read_kv(b, l, 0, 40)
        np.testing.assert_allclose(kb, ka, rtol=0, atol=2e-3 * np.max(np.abs(ka)))
        np.testing.assert_allclose(vb, va, rtol=0, atol=2e-3 * np.max(np.abs(va)))


# ---------------------------------------------------------------- the block
FLIP_SCALE = 0.1  # free running, quantised: gross-error bound (one flipped code moves logits by <= ~3 %)


class Script:
    """The same appends and blocks on the oracle (recording its quantisation
    decisions) and on the GPU (taking them, recording its own).  Returns per
    block the oracle's and the GPU's logits and tokens; check() compares every
    site and every block."""

    def __init__(self, p, n_seqs, cap):
        self.p = p
        self.n = n_seqs
        self.cap = cap
        self.actions = []

    def append(self, i, pos, taps):
        self.actions.append(("append", i, pos, taps))

    def queue(self, i, pos, taps):
        self.actions.append(("queue", i, pos, taps))

    def truncate(self, i, pos):
        self.actions.append(("truncate", i, pos))

    def block(self, seqs, anchors, positions, bl):
        self.actions.append(("block", list(seqs), list(anchors), list(positions), bl))

    def run(self, forced=True):
        import oracle.drafter as D
        p, g = self.p, self.p.g
        osq = [OracleSeq(p.ora) for _ in range(self.n)]
        D.TRACE = D.QuantTrace() if g.quant else None
        oracle_out, sites = [], []
        try:
            for a in self.actions:
                if a[0] in ("append", "queue"):
                    getattr(osq[a[1]], a[0])(a[2], a[3])
                    if D.TRACE is not None:
                        sites += D.TRACE.sites
                        D.TRACE.sites = []
                elif a[0] == "truncate":
                    osq[a[1]].truncate(a[2])
                else:
                    # a block settles its sequences' queued rows first, in sequence order
                    for i in a[1]:
                        osq[i].settle()
                        if D.TRACE is not None:
                            sites += D.TRACE.sites
                            D.TRACE.sites = []
                    _, ids, anchors, positions, bl = a
                    per_seq = []
                    res = []
                    for i, at, ap in zip(ids, anchors, positions):
                        res.append(block(p.ora, osq[i], at, ap, bl))
                        if D.TRACE is not None:
                            per_seq.append(D.TRACE.sites)
                            D.TRACE.sites = []
                    # the GPU runs the sequences' rows together: stack each site's rows
                    for k in range(len(per_seq[0]) if per_seq else 0):
                        sites.append(tuple(np.concatenate([ps[k][j] for ps in per_seq]) for j in range(3)))
                    oracle_out.append(res)
        finally:
            D.TRACE = None
        gseq = [p.gpu.new_sequence(self.cap) for _ in range(self.n)]
        gpu_out, own = [], []
        if g.quant and forced:
            p.gpu.trace(True)
            for x, q, s in sites:
                p.gpu.trace_force(q, s)
        try:
            for a in self.actions:
                if a[0] == "append":
                    p.gpu.ctx_append(gseq[a[1]], a[2], a[3])
                elif a[0] == "queue":
                    p.gpu.ctx_queue(gseq[a[1]], a[2], a[3])
                elif a[0] == "truncate":
                    gseq[a[1]].truncate(a[2])
                else:
                    _, ids, anchors, positions, bl = a
                    gpu_out.append(p.gpu.block([gseq[i] for i in ids], anchors, positions, bl))
            if g.quant and forced:
                own = p.gpu.trace_sites()
        finally:
            if g.quant and forced:
                p.gpu.trace(False)
        self.sites, self.own, self.oracle_out, self.gpu_out = sites, own, oracle_out, gpu_out
        self.osq, self.gseq = osq, gseq
        return self

    def check(self, forced=True):
        g = self.p.g
        if g.quant and forced:
            check_sites(self.sites, self.own, 1e-5)
        for res, (logits, toks) in zip(self.oracle_out, self.gpu_out):
            for i, (ref, ref_tok) in enumerate(res):
                scale = np.max(np.abs(ref))
                err = np.max(np.abs(logits[i].astype(np.float64) - ref))
                if g.quant == 0:
                    assert err <= 1e-4 * scale, f"block {i}: {err:.3e}"
                    check_tokens(toks[i], ref, 1e-4 * scale)
                elif forced:
                    assert err <= 1e-5 * scale, f"block {i}: {err:.3e}"
                    assert (toks[i] == ref_tok).all()
                else:
                    assert err <= FLIP_SCALE * scale, f"block {i}: {err:.3e}"
        for s in self.gseq:
            s.close()


@pytest.mark.parametrize("name", ["tiny_f32", "small_q4", "small_q4_hd64"])
@pytest.mark.parametrize("forced", [True, False])
def test_block_matches_oracle(name, forced):
    p = pair(name)
    g, n = p.g, p.wl.ctx
    sc = Script(p, 1, n + 16)
    sc.append(0, 0, W.make_taps(g, n))
    sc.block([0], [int(W.make_anchors(g, 1)[0])], [n], g.block)
    sc.run(forced).check(forced)


@pytest.mark.parametrize("name", ["tiny_f32", "small_q4"])
@pytest.mark.parametrize("forced", [True, False])
def test_windows_and_no_rope_match_oracle(name, forced):
    """Page 1's geometry variants: a windowed layer among whole-context ones,
    a layer without the rotary position, and the drop of context rows that
    fell out of every window (appends in chunks that cross it), in blocks of
    two sequences at the end of their contexts and one anchored inside the
    rows still held."""
    L = W.WORKLOADS[name].geom.layers
    p = Pair(name, windows=(9,) + (0,) * (L - 1), no_rope=(L - 1,))
    g = p.g
    sc = Script(p, 2, 64)
    taps = W.make_taps(g, 40)
    for r0 in range(0, 40, 13):
        sc.append(0, r0, taps[r0:r0 + 13])
    sc.append(1, 0, W.make_taps(g, 25, call_id=3))
    anchors = [int(a) for a in W.make_anchors(g, 2)]
    sc.block([0, 1], anchors, [40, 25], g.block)
    sc.block([0], [anchors[1]], [34], g.block)
    sc.run(forced).check(forced)


def _zero_queries_and_down(w):
    for lw in w["layers"]:
        lw["q"][:] = 0
        lw["down"][:] = 0


@pytest.mark.parametrize("name", ["tiny_f32", "small_q4"])
@pytest.mark.parametrize("forced", [True, False])
@pytest.mark.parametrize("window", [0, 3])
def test_equal_scores_match_oracle(name, forced, window):
    """Wq = 0 (and Wd = 0): every attention score is exactly 0, so each row's
    softmax is uniform over the keys it sees -- the degenerate case of the
    split-key online softmax, whose oracle side is pinned by a closed form.
    A window of 3 (shorter than the block) leaves the later rows no context
    key at all, only the block's rows."""
    p = Pair(name, edit=_zero_queries_and_down, window=window)
    g = p.g
    n = p.wl.ctx
    sc = Script(p, 1, n + 16)
    sc.append(0, 0, W.make_taps(g, n))
    anchor = int(W.make_anchors(g, 1)[0])
    sc.block([0], [anchor], [n], g.block)
    sc.block([0], [anchor], [n], 5)
    sc.run(forced).check(forced)


@pytest.mark.parametrize("name", ["tiny_f32", "small_q4"])
@pytest.mark.parametrize("forced", [True, False])
@pytest.mark.parametrize("variants", [False, True])
def test_row_convolution_matches_oracle(name, forced, variants):
    """The DFlash 2 row convolution around attention and the MLP (page 1's
    conv_in / conv_out), in a block of two sequences (the many-row matmuls
    at small_q4) and a shorter block of one (the streaming ones); with
    `variants` also a windowed layer and a layer without the rotary position."""
    L = W.WORKLOADS[name].geom.layers
    extra = dict(windows=(9,) + (0,) * (L - 1), no_rope=(L - 1,)) if variants else {}
    p = Pair(name, conv_kernel=4, conv_group=64, **extra)
    g = p.g
    sc = Script(p, 2, 64)
    sc.append(0, 0, W.make_taps(g, 30))
    sc.append(1, 0, W.make_taps(g, 17, call_id=5))
    anchors = [int(a) for a in W.make_anchors(g, 2)]
    sc.block([0, 1], anchors, [30, 17], g.block)
    sc.block([0], [anchors[1]], [30], 5)
    sc.run(forced).check(forced)


def test_selector_matches_oracle_forced():
    """The candidate selector after the head (page 1's select): with the
    oracle's quantisation decisions taken, the library's choices equal the
    oracle's, in a block of two sequences and a shorter block of one."""
    p = Pair("small_q4", selector_rank=16, selector_top=8)
    g = p.g
    sc = Script(p, 2, 64)
    sc.append(0, 0, W.make_taps(g, 30))
    sc.append(1, 0, W.make_taps(g, 17, call_id=5))
    anchors = [int(a) for a in W.make_anchors(g, 2)]
    sc.block([0, 1], anchors, [30, 17], g.block)
    sc.block([0], [anchors[1]], [30], 6)
    sc.run(True).check(True)


@pytest.mark.parametrize("top", [1, 8, 32])
def test_selector_choices_from_the_librarys_logits(top):
    """All-f32 drafter: the library's choices equal the oracle's selection run
    on the library's own logits and the oracle's normed rows (what remains
    is the f32 scoring against the oracle's f64: far from any tie here)."""
    from oracle import select
    p = Pair("tiny_f32", selector_rank=24, selector_top=top)
    g = p.g
    seq = p.gpu.new_sequence(64)
    taps = W.make_taps(g, 20)
    p.gpu.ctx_append(seq, 0, taps)
    osq = OracleSeq(p.ora)
    osq.append(0, taps)
    for anchor, bl in ((11, g.block), (3, 4)):
        logits, toks = p.gpu.block([seq], [anchor], [20], bl)
        ref_logits, _, hn = block(p.ora, osq, anchor, 20, bl, return_hidden=True)
        assert np.max(np.abs(logits[0] - ref_logits)) <= 1e-4 * np.max(np.abs(ref_logits))
        chosen, plain = select(p.ora, hn[1:], logits[0], anchor)
        np.testing.assert_array_equal(toks[0], chosen)
    seq.close()


@pytest.mark.parametrize("name", ["tiny_f32", "small_q4"])
@pytest.mark.parametrize("forced", [True, False])
def test_context_queue_matches_oracle(name, forced):
    """Page 1's context queue: rows queued over several calls and settled by
    the block that reads them; a truncation that cuts queued rows; a queue
    past its limit (the oldest settled in 64-row granules)."""
    p = Pair(name)
    g = p.g
    sc = Script(p, 2, 700)
    taps = W.make_taps(g, 40)
    sc.append(0, 0, taps[:10])
    sc.queue(0, 10, taps[10:25])
    sc.queue(0, 25, taps[25:40])
    sc.truncate(0, 33)
    sc.queue(0, 33, taps[33:40])
    sc.queue(1, 0, W.make_taps(g, 600, call_id=4))
    anchors = [int(a) for a in W.make_anchors(g, 2)]
    sc.block([0, 1], anchors, [40, 600], g.block)
    sc.queue(0, 40, W.make_taps(g, 16, call_id=6))
    sc.block([0], [anchors[1]], [56], g.block)
    sc.run(forced).check(forced)


def test_queue_span_and_settle():
    """The span counts queued rows; settle makes them context; the capacity
    counts them too."""
    dfl = _dfl()
    p = pair("tiny_f32")
    g = p.g
    seq = p.gpu.new_sequence(50)
    p.gpu.ctx_queue(seq, 0, W.make_taps(g, 30))
    assert seq.span() == (0, 30)
    with pytest.raises(dfl.DFlashError) as e:
        p.gpu.ctx_queue(seq, 30, W.make_taps(g, 21))
    assert e.value.code == dfl._abi.DFLASH_ECAPACITY
    assert seq.span() == (0, 30)
    p.gpu.settle(seq)
    assert seq.span() == (0, 30)
    seq.truncate(12)
    assert seq.span() == (0, 12)
    seq.close()


def test_geometry_lists_round_trip():
    """dflash_geometry_of gives back the per-layer windows and no-rope flags
    the model was made with."""
    dfl = _dfl()
    L = W.WORKLOADS["small_q4"].geom.layers
    p = Pair("small_q4", windows=(5,) + (0,) * (L - 1), no_rope=(0,))
    gs = dfl._abi.Geometry()
    assert dfl.lib().dflash_geometry_of(p.gpu.handle, dfl._abi.C.byref(gs)) == 0
    assert [gs.windows[i] for i in range(L)] == list(p.g.windows)
    assert [gs.no_rope[i] for i in range(L)] == [1 if i == 0 else 0 for i in range(L)]


@pytest.mark.parametrize("name", ["tiny_f32", "small_q4"])
def test_block_edge_cases(name):
    """Shorter blocks, an empty context, an anchor inside the held context, a
    block reading a context that starts past position 0."""
    p = pair(name)
    g = p.g
    taps = W.make_taps(g, 50, call_id=5)
    sc = Script(p, 1, 80)
    sc.append(0, 0, taps[:0])
    sc.block([0], [3], [0], 2)              # empty context, two rows
    sc.append(0, 0, taps[:33])
    sc.block([0], [17], [33], g.block)       # ragged context
    sc.append(0, 0, taps[:50])
    sc.block([0], [9], [20], 3)              # anchor inside the context: reads positions < 20 only
    sc.append(0, 100, taps[:50])
    sc.block([0], [0], [150], g.block)       # context starting at position 100
    sc.run().check()


@pytest.mark.parametrize("name", ["tiny_f32", "small_q4"])
def test_batched_sequences(name):
    """Several sequences in one call, each with its own context and anchor."""
    p = pair(name)
    g = p.g
    lens = [7, 0, 61]
    sc = Script(p, 3, 72)
    for i, n in enumerate(lens):
        sc.append(i, 0, W.make_taps(g, n, call_id=10 + i))
    sc.block([0, 1, 2], [11, 12, 13], lens, g.block)
    sc.block([2, 0], [14, 15], [61, 7], 5)
    sc.run().check()


@pytest.mark.parametrize("name", ["small_q4", "small_q4_hd64"])
@pytest.mark.parametrize("forced", [True, False])
def test_batched_many_sequences(name, forced):
    """Ten sequences in one call: every matmul and the head run on the
    tensor-core kernels with two 128-row tiles (the second ragged) and a
    ragged last vocabulary tile."""
    p = pair(name)
    g = p.g
    lens = [5, 0, 33, 44, 12, 1, 40, 27, 9, 44]
    sc = Script(p, len(lens), 64)
    for i, n in enumerate(lens):
        sc.append(i, 0, W.make_taps(g, n, call_id=40 + i))
    sc.block(list(range(len(lens))), [(37 * i + 5) % g.vocab for i in range(len(lens))], lens, g.block)
    sc.run(forced).check(forced)


def test_long_context_split_merge():
    """A context long enough that the attention splits its keys over plain
    CTAs (every SM busy) whose partial rows merge through global memory, not
    in a cluster: identical decisions, values and logits to 1e-5."""
    p = pair("small_q4")
    g = p.g
    n = 20000
    sc = Script(p, 1, n + 16)
    sc.append(0, 0, W.make_taps(g, n, call_id=90))
    sc.block([0], [123], [n], g.block)
    sc.run(True).check(True)


def test_truncate_and_reappend():
    p = pair("small_q4")
    g = p.g
    t1 = W.make_taps(g, 40, call_id=20)
    t2 = W.make_taps(g, 40, call_id=21)
    sc = Script(p, 1, 64)
    sc.append(0, 0, t1)
    sc.append(0, 25, t2[25:])       # replaces 25..
    sc.append(0, 30, t2[30:35])     # replaces 30.. : context ends at 35
    sc.block([0], [5], [35], g.block)
    sc.run().check()
    # truncate / reset on the GPU sequence directly
    seq = p.gpu.new_sequence(64)
    p.gpu.ctx_append(seq, 0, t1)
    seq.truncate(25)
    assert seq.span() == (0, 25)
    seq.reset()
    assert seq.span() == (0, 0)
    seq.close()


def test_device_io_matches_host_io():
    """Device-pointer and host-buffer calls compute the same block.  The GPU
    sums split-K partials with atomics, so two runs may round an activation
    code differently; the host run's decisions are recorded and forced on the
    device run, which must then agree to summation-order rounding."""
    import torch
    p = pair("small_q4")
    g = p.g
    taps = W.make_taps(g, 30, call_id=30)
    seq = p.gpu.new_sequence(40)
    p.gpu.ctx_append(seq, 0, torch.from_numpy(taps).cuda())

    def force(sites):
        p.gpu.trace(True)
        for _, q, s in sites:
            p.gpu.trace_force(q, s)

    p.gpu.trace(True)
    try:
        lh, th = p.gpu.block([seq], [7], [30], g.block)
        sites = p.gpu.trace_sites()
        ld = torch.empty((1, g.block - 1, g.vocab), dtype=torch.float32, device="cuda")
        td = torch.empty((1, g.block - 1), dtype=torch.int32, device="cuda")
        force(sites)
        p.gpu.block([seq], torch.tensor([7], dtype=torch.int32, device="cuda"), [30], g.block, logits=ld, tokens=td)
        torch.cuda.synchronize()
        assert len(p.gpu.trace_sites()) == len(sites)
        force(sites)
        _, t2 = p.gpu.block([seq], [7], [30], g.block, want_logits=False)  # tokens-only host call
    finally:
        p.gpu.trace(False)
    ref = lh.astype(np.float64)
    assert np.max(np.abs(ld.cpu().numpy() - ref)) <= 1e-5 * np.max(np.abs(ref))
    np.testing.assert_array_equal(td.cpu().numpy(), th)
    np.testing.assert_array_equal(t2, th)
    seq.close()


def test_bounded_wait_expiry_is_reported():
    """A kernel whose data never arrives gives up its bounded wait, raises the
    model's error flag and returns: the call reports ECUDA, the model stays
    poisoned, and the CUDA context still serves a fresh model."""
    dfl = _dfl()
    g = W.WORKLOADS["small_q4"].geom
    w = W.make_weights(g)
    m = dfl.Model(g, w)
    try:
        with pytest.raises(dfl.DFlashError) as ei:
            m.wait_expiry(50_000_000)  # 50 ms
        assert ei.value.code == dfl._abi.DFLASH_ECUDA
        assert "bounded wait" in str(ei.value)
        with pytest.raises(dfl.DFlashError):
            m.new_sequence(8)
    finally:
        m.close()
    m2 = dfl.Model(g, w)
    seq = m2.new_sequence(40)
    m2.ctx_append(seq, 0, W.make_taps(g, 20, call_id=5))
    logits, toks = m2.block([seq], [3], [20], g.block)
    assert np.isfinite(logits).all()
    seq.close()
    m2.close()


def test_error_codes():
    dfl = _dfl()
    p = pair("tiny_f32")
    g = p.g
    seq = p.gpu.new_sequence(10)
    with pytest.raises(dfl.DFlashError) as e:
        p.gpu.ctx_append(seq, 0, W.make_taps(g, 11))
    assert e.value.code == dfl._abi.DFLASH_ECAPACITY
    assert seq.span() == (0, 0)
    p.gpu.ctx_append(seq, 0, W.make_taps(g, 4))
    for bl in (1, g.block + 1):
        with pytest.raises(dfl.DFlashError) as e:
            p.gpu.block([seq], [1], [4], bl)
        assert e.value.code == dfl._abi.DFLASH_ERANGE
    with pytest.raises(dfl.DFlashError) as e:
        p.gpu.block([seq], [g.vocab], [4], 2)
    assert e.value.code == dfl._abi.DFLASH_EINVAL
    other = pair("small_q4")
    with pytest.raises(dfl.DFlashError) as e:
        other.gpu.block([seq], [1], [4], 2)
    assert e.value.code == dfl._abi.DFLASH_EINVAL
    # the model still works after rejected calls
    logits, _ = p.gpu.block([seq], [1], [4], 2)
    assert np.isfinite(logits).all()
    seq.close()


@pytest.mark.parametrize("name", ["tiny_f32", "small_q4", "small_q4_hd64"])
def test_attention_matches_oracle(name):
    """Row b4 alone: the block's attention over each sequence's context and
    its own rows, for seeded q/k/v block rows."""
    import math

    import torch
    from oracle import attention as oattn
    p = pair(name)
    g = p.g
    hd, nh, kv, B = g.head_dim, g.heads, g.kv_heads, g.block
    ctx = [p.wl.ctx, 3]
    seqs, oseqs = [], []
    for i, n in enumerate(ctx):
        s = p.gpu.new_sequence(n + 4)
        o = OracleSeq(p.ora)
        t = W.make_taps(g, n, call_id=40 + i)
        p.gpu.ctx_append(s, 0, t)
        o.append(0, t)
        seqs.append(s)
        oseqs.append(o)
    width = (nh + 2 * kv) * hd
    qkv = W.normal(7, 100, (len(ctx) * B, width))
    y = torch.empty((len(ctx) * B, nh * hd), dtype=torch.float32, device="cuda")
    layer = g.layers - 1
    p.gpu.attention(seqs, layer, ctx, torch.from_numpy(qkv).cuda(), y)
    got = y.cpu().numpy()
    tol = 1e-4 if g.quant == 0 else 2e-3
    for s in range(len(ctx)):
        rows = qkv[s * B:(s + 1) * B].astype(np.float64)
        q = rows[:, :nh * hd].reshape(B, nh, hd)
        kb = rows[:, nh * hd:(nh + kv) * hd].reshape(B, kv, hd)
        vb = rows[:, (nh + kv) * hd:].reshape(B, kv, hd)
        ref = oattn(q, kb, vb, oseqs[s].k[layer], oseqs[s].v[layer], g.rep, 1 / math.sqrt(hd))
        out = got[s * B:(s + 1) * B].reshape(B, nh, hd)
        assert np.max(np.abs(out - ref)) <= tol * np.max(np.abs(ref))
    for s in seqs:
        s.close()


# ---------------------------------------------------------------- identical decisions
def forced_run(p, ctx, anchor, taps, pos=0):
    """Run the oracle recording its quantisation decisions, then the GPU with
    every site's codes and scales replaced by the oracle's.  Returns the
    oracle's sites, the GPU's own sites, both logits and the GPU sequence."""
    import oracle.drafter as D
    g = p.g
    D.TRACE = D.QuantTrace()
    try:
        osq = OracleSeq(p.ora)
        osq.append(pos, taps)
        ref, ref_tok = block(p.ora, osq, anchor, pos + ctx, g.block)
        sites = D.TRACE.sites
    finally:
        D.TRACE = None
    seq = p.gpu.new_sequence(ctx + 8)
    p.gpu.trace(True)
    for x, q, s in sites:
        p.gpu.trace_force(q, s)
    try:
        p.gpu.ctx_append(seq, pos, taps)
        logits, toks = p.gpu.block([seq], [anchor], [pos + ctx], g.block)
        own = p.gpu.trace_sites()
    finally:
        p.gpu.trace(False)
    return sites, own, ref, ref_tok, logits[0], toks[0], seq, osq


def check_sites(sites, own, value_tol):
    """Per site: values agree to value_tol * max|x|, scales likewise, and the
    GPU's own codes equal the oracle's except where the oracle's value lies at
    a half-step boundary within the two sides' difference: within rounding of
    it, or with the GPU's own value (held to the bound above) on its other
    side -- a small element of a row carries the site's absolute error, which
    in code units can exceed its own relative rounding.  Returns the
    flipped-code count."""
    assert len(own) == len(sites), (len(own), len(sites))
    flips = 0
    for i, ((x, q, s), (v, qg, sg)) in enumerate(zip(sites, own)):
        assert v.shape == x.shape, (i, v.shape, x.shape)
        err = np.max(np.abs(v - x))
        assert err <= value_tol * np.max(np.abs(x)), f"site {i}: values differ by {err:.3e}"
        np.testing.assert_allclose(sg, s, rtol=value_tol, atol=0, err_msg=f"site {i} scales")
        diff = qg != q
        if diff.any():
            r = np.asarray(x, np.float32) / np.where(s > 0, s, 1)[:, None]
            rg = np.asarray(v, np.float64) / np.where(sg > 0, sg, 1)[:, None]
            dist = np.abs(np.abs(r - np.floor(r)) - 0.5)
            near = (dist <= value_tol * np.maximum(np.abs(r), 1.0) * 4) | \
                (dist <= np.abs(rg - r) + 1e-6 * np.maximum(np.abs(r), 1.0))
            assert (near[diff]).all(), f"site {i}: code differs away from a rounding boundary"
            assert (np.abs(qg.astype(int) - q)[diff] == 1).all()
            flips += int(diff.sum())
    return flips


@pytest.mark.parametrize("name", ["small_q4", "small_q4_hd64"])
def test_identical_decisions_parity(name):
    """With the oracle's quantisation decisions at every site, the GPU's
    continuous values at every site agree to f32 level (1e-5 relative), and so
    do the logits; its own decisions differ only at rounding boundaries."""
    p = pair(name)
    g, n = p.g, p.wl.ctx
    taps = W.make_taps(g, n, call_id=50)
    for anchor in (11, 4000 % g.vocab):
        sites, own, ref, ref_tok, logits, toks, seq, osq = forced_run(p, n, anchor, taps)
        assert len(sites) == 2 + 4 * g.layers + 1
        check_sites(sites, own, 1e-5)
        scale = np.max(np.abs(ref))
        assert np.max(np.abs(logits - ref)) <= 1e-5 * scale
        assert (toks == ref_tok).all()
        for l in range(g.layers):
            k, v = p.gpu.read_kv(seq, l, 0, n)
            assert np.max(np.abs(k - osq.k[l].transpose(1, 0, 2))) <= 1e-5 * np.max(np.abs(osq.k[l]))
            assert np.max(np.abs(v - osq.v[l].transpose(1, 0, 2))) <= 1e-5 * np.max(np.abs(osq.v[l]))
        seq.close()


# ---------------------------------------------------------------- argmax ties
def _duplicate_head_rows(w):
    """Head rows h.. are exact copies of rows 0.. (equal int8 codes and row
    scales, so equal logits): every draft row's maximum is tied with a copy."""
    V = w["head"].shape[0]
    h = (V + 1) // 2
    w["head"][h:] = w["head"][:V - h]


def _zero_head(w):
    w["head"][:] = 0.0


@pytest.mark.parametrize("edit", ["duplicate", "zero"])
@pytest.mark.parametrize("n_seqs", [1, 4])
def test_argmax_ties_keep_the_first_of_equals(edit, n_seqs):
    """Exactly tied logits (page "cortiq-engine 0.8.71 — src/dflash.rs",
    `top_k`: the first of equals is kept): with every head row duplicated
    further down, each draft token must be the lower copy's index; with a
    head of zeros (all logits 0), index 0.  One sequence runs the streaming
    head, four (60 rows) the tensor-core head; decisions identical to the
    oracle's, tokens equal to its lowest-index argmax."""
    p = Pair("small_q4", edit=_duplicate_head_rows if edit == "duplicate" else _zero_head)
    g = p.g
    lens = [77, 30, 0, 51][:n_seqs]
    sc = Script(p, n_seqs, 96)
    for i, n in enumerate(lens):
        sc.append(i, 0, W.make_taps(g, n, call_id=70 + i))
    sc.block(list(range(n_seqs)), [(53 * i + 9) % g.vocab for i in range(n_seqs)], lens, g.block)
    sc.run(True).check(True)
    V, h = g.vocab, (g.vocab + 1) // 2
    for (logits, toks), res in zip(sc.gpu_out, sc.oracle_out):
        toks = np.asarray(toks)
        if edit == "zero":
            assert (toks == 0).all()
            assert not np.asarray(logits).any()
        else:
            assert (toks < h).all(), "a later copy of a tied maximum was chosen"
            for i, (ref, ref_tok) in enumerate(res):
                lg = np.asarray(logits[i])
                # the tie is real: the chosen row's copy carries the same logit
                t = toks[i]
                keep = t < V - h
                assert (lg[np.arange(len(t))[keep], t[keep] + h] == lg[np.arange(len(t))[keep], t[keep]]).all()
                assert (t == ref_tok).all()


# ---------------------------------------------------------------- argmax agreement over many rows
MARGIN_BINS = [0.0, 1e-4, 1e-3, 1e-2, 3e-2, 1e-1, np.inf]


def agreement_table(records):
    """records: per block (oracle logits [rows][V], GPU tokens with the
    oracle's decisions, GPU tokens with its own).  Rows binned by the oracle's
    top-2 margin over max|logit| of the block; per bin the rows and the
    fraction of equal tokens under identical and under free-running decisions.
    Returns (table rows, overall forced, overall free)."""
    margins, eq_forced, eq_free = [], [], []
    for ref, tf, tr in records:
        ref32 = np.asarray(ref, np.float32)
        srt = np.sort(ref32, axis=-1)
        margins.append((srt[:, -1] - srt[:, -2]) / float(np.max(np.abs(ref32))))
        ref_tok = np.argmax(ref32, axis=-1)
        eq_forced.append(np.asarray(tf) == ref_tok)
        eq_free.append(np.asarray(tr) == ref_tok)
    m, ef, er = np.concatenate(margins), np.concatenate(eq_forced), np.concatenate(eq_free)
    table = []
    for lo, hi in zip(MARGIN_BINS[:-1], MARGIN_BINS[1:]):
        sel = (m >= lo) & (m < hi)
        if sel.any():
            table.append((lo, hi, int(sel.sum()), float(ef[sel].mean()), float(er[sel].mean())))
    return table, float(ef.mean()), float(er.mean()), m, er


def print_agreement(title, table, forced, free):
    print(f"{title}: identical decisions {forced:.4f}, free running {free:.4f}")
    print("  top-2 margin / max|logit|   rows   identical   free")
    for lo, hi, n, f, r in table:
        print(f"  [{lo:.0e}, {hi:.0e})  {n:6d}   {f:.4f}   {r:.4f}")


def test_argmax_agreement_over_3000_rows():
    """Draft tokens of 200 single-sequence blocks (3000 rows) against the
    oracle's: with identical quantisation decisions (context and block) every
    row's argmax must agree (the >= 99.9 % bar); free running, every row whose
    oracle top-2 margin exceeds a tenth of max|logit| (beyond what one flipped
    code can move) must agree, and the table reports the rest by margin."""
    import oracle.drafter as D
    p = pair("small_q4")
    g = p.g
    records = []
    for c, n in enumerate([77, 40, 120, 200]):
        taps = W.make_taps(g, n, call_id=300 + c)
        D.TRACE = D.QuantTrace()
        try:
            osq = OracleSeq(p.ora)
            osq.append(0, taps)
            ctx_sites = D.TRACE.sites
        finally:
            D.TRACE = None
        seq = p.gpu.new_sequence(n + 8)
        p.gpu.trace(True)
        for _, q, s in ctx_sites:
            p.gpu.trace_force(q, s)
        try:
            p.gpu.ctx_append(seq, 0, taps)
        finally:
            p.gpu.trace(False)
        anchors = W.make_anchors(g, 50, call_id=400 + c)
        for a in anchors:
            D.TRACE = D.QuantTrace()
            try:
                ref, _ = block(p.ora, osq, int(a), n, g.block)
                sites = D.TRACE.sites
            finally:
                D.TRACE = None
            p.gpu.trace(True)
            for _, q, s in sites:
                p.gpu.trace_force(q, s)
            try:
                _, tf = p.gpu.block([seq], [int(a)], [n], g.block)
            finally:
                p.gpu.trace(False)
            _, tr = p.gpu.block([seq], [int(a)], [n], g.block)
            records.append((ref, tf[0], tr[0]))
        seq.close()
    table, forced, free, m, er = agreement_table(records)
    print_agreement(f"small_q4, {len(records)} blocks, {sum(t[2] for t in table)} rows", table, forced, free)
    assert sum(t[2] for t in table) >= 1000
    assert forced == 1.0
    assert er[m >= 0.1].all()


# ---------------------------------------------------------------- the tcgen05 attention on small cases
def _tc_pair(name, **changes):
    """A fresh pair whose GPU model runs the block attention on the tcgen05
    kernel whatever the split length (the default keeps it for splits of at
    least 256 keys: long contexts and batches)."""
    p = Pair(name, **changes)
    p.gpu.option("attn_tc_min_keys", 0)
    return p


@pytest.mark.parametrize("name", ["small_q4", "small_q4_hd64"])
@pytest.mark.parametrize("forced", [True, False])
def test_tc_attention_block_matches_oracle(name, forced):
    """The block (and a context starting at position 100) with the tcgen05
    attention: a block step of the block's rows and tensor-copied context
    steps, the splits added into the accumulators."""
    p = _tc_pair(name)
    g, n = p.g, p.wl.ctx
    sc = Script(p, 1, n + 16)
    sc.append(0, 0, W.make_taps(g, n))
    sc.block([0], [int(W.make_anchors(g, 1)[0])], [n], g.block)
    sc.block([0], [0], [150], g.block)
    sc.run(forced).check(forced)


@pytest.mark.parametrize("name", ["small_q4", "small_q4_hd64"])
@pytest.mark.parametrize("forced", [True, False])
def test_tc_attention_windows_and_batches_match_oracle(name, forced):
    """Windowed layers (the row-dependent mask of the context steps), a layer
    without the rotary position, several sequences of different lengths (an
    empty one included) and a context longer than one 128-key step; head_dim
    128 and 64."""
    p = _tc_pair(name, windows=(3, 0), no_rope=(1,))
    g = p.g
    lens = [77, 0, 200, 9]
    sc = Script(p, len(lens), 224)
    for i, n in enumerate(lens):
        sc.append(i, 0, W.make_taps(g, n, call_id=110 + i))
    sc.block(list(range(len(lens))), [(29 * i + 3) % g.vocab for i in range(len(lens))], lens, g.block)
    sc.block([2], [17], [200], min(9, g.block - 1))
    sc.run(forced).check(forced)


@pytest.mark.parametrize("name,heads", [("small_q4", 12), ("small_q4", 16), ("small_q4_hd64", 27)])
@pytest.mark.parametrize("forced", [True, False])
def test_tc_attention_wide_query_tiles(name, heads, forced):
    """More than 64 query rows a kv head (q heads a kv head times the block's
    rows: 96, 128 and 72; the query tile reaches tensor memory in two staged
    passes of 64 rows, and at 128 the MMA's M is full), with a context of
    several 128-key steps and a second, shorter block."""
    p = _tc_pair(name, heads=heads)
    g, n = p.g, 300
    sc = Script(p, 1, n + 16)
    sc.append(0, 0, W.make_taps(g, n))
    sc.block([0], [int(W.make_anchors(g, 1)[0])], [n], g.block)
    sc.block([0], [9], [n], g.block - 5)
    sc.run(forced).check(forced)


@pytest.mark.parametrize("window", [0, 3])
def test_tc_attention_equal_scores(window):
    """All scores exactly 0 (Wq = Wd = 0): every row averages the values it
    sees, through the tcgen05 kernel's online softmax."""
    p = _tc_pair("small_q4", edit=_zero_queries_and_down, window=window)
    g, n = p.g, p.wl.ctx
    sc = Script(p, 1, n + 16)
    sc.append(0, 0, W.make_taps(g, n))
    sc.block([0], [5], [n], g.block)
    sc.run(True).check(True)
