"""Full-size parity of the other Qwen3-8B-shaped configurations (hidden 4096,
5 layers, 32/8 heads of 128, intermediate 12288, vocab 151936, 5 taps): the
8192-row context append, 32 batched sequences at context 4096, and one
sequence at context 32768.  The GPU runs every configuration whole, in the
launch configuration of its size; the oracle computes the outputs it can
afford one by one:

* append: context rows are independent, so the oracle projects sampled rows
  on their own (``OracleSeq.project``) and the GPU's stored K/V rows must
  match them;
* batched block: sequences are independent, so the oracle runs two of the
  32 sequences whole and the GPU's logits for those two must match;
* long context: the oracle runs the whole sequence.

Free running, each side takes its own quantisation decisions (an f32 value
within rounding of a half-step boundary can round either way), so a row or a
block is compared with the bound the identical-decision tests justify where
no decision differs, and with the spread that f32-level noise on the
oracle's own decisions produces where one does.  The blocks are then run
again with the oracle's decisions at every quantisation site of the block
and must agree at f32 level (the appended context keeps each side's own
decisions: a context row with a code at a boundary moves the attention by
about its 1/n weight times a code step).
"""
import numpy as np
import pytest

import workloads as W
from oracle import OracleModel, OracleSeq, block

pytestmark = pytest.mark.gpu

APPEND_CHUNK = 4096  # host rows of taps generated and appended at a time


@pytest.fixture(scope="module")
def qwen():
    import block_speculative_drafting_gb300 as dfl
    g = W.WORKLOADS["qwen3_8b_ctx2048"].geom
    w = W.make_weights(g)
    model = dfl.Model(g, w)
    om = OracleModel(g, w)
    yield g, model, om
    model.close()


def _noise_bound(om, osq, anchor, anchor_pos, B, ref, runs=2):
    """max |logit change| / max |logit| when the oracle's quantisers see
    f32-level noise on their inputs (its own decision sensitivity)."""
    from oracle import quant as Q
    orig = Q.quantize_rows_i8
    rng = np.random.default_rng(0)
    scale = float(np.max(np.abs(ref)))
    devs = []
    try:
        Q.quantize_rows_i8 = lambda x: orig(np.asarray(x, np.float64) * (1 + 1e-7 * rng.standard_normal(np.shape(x))))
        for _ in range(runs):
            lp, _ = block(om, osq, anchor, anchor_pos, B)
            devs.append(float(np.max(np.abs(lp - ref))) / scale)
    finally:
        Q.quantize_rows_i8 = orig
    return max(devs)


def _oracle_block_sites(om, osq, anchor, anchor_pos, B):
    """The oracle's block with its quantisation sites recorded."""
    import oracle.drafter as D
    D.TRACE = D.QuantTrace()
    try:
        ref, ref_tok = block(om, osq, anchor, anchor_pos, B)
        return ref, ref_tok, D.TRACE.sites
    finally:
        D.TRACE = None


def _forced_block(model, seqs, anchors, positions, B, sites):
    """The GPU block with every site's codes and scales replaced by `sites`."""
    model.trace(True)
    for _, q, sc in sites:
        model.trace_force(q, sc)
    try:
        out = model.block(seqs, anchors, positions, B)
        own = model.trace_sites()
    finally:
        model.trace(False)
    return out, own


def test_prefill_8192_rows_sampled(qwen):
    """One 8192-row append (the prefill configuration); sampled rows of the
    first and last layers against the oracle's projection of those rows."""
    g, model, om = qwen
    wl = W.WORKLOADS["qwen3_8b_prefill8192"]
    n = wl.prefill
    taps = W.make_taps(g, n, call_id=80)
    seq = model.new_sequence(n)
    model.ctx_append(seq, 0, taps)
    assert seq.span() == (0, n)
    rng = np.random.default_rng(5)
    rows = sorted(set([0, 1, 1023, 1024, 4095, 4096, n - 1] + list(rng.integers(0, n, 25))))
    osq = OracleSeq(om)
    close, flipped = 0, []
    for p in rows:
        ks, vs = osq.project(p, taps[p:p + 1])
        row_ok = True
        for l in (0, g.layers - 1):
            k, v = model.read_kv(seq, l, p, 1)
            for got, ref in ((k[0], ks[l][0]), (v[0], vs[l][0])):
                err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
                assert err <= 3e-2, f"row {p} layer {l}: {err:.2e}"  # at most a flipped code's worth
                row_ok &= err <= 5e-5
        close += row_ok
        if not row_ok:
            flipped.append(p)
    print(f"prefill 8192: {close}/{len(rows)} sampled rows at f32 level; others (a code at a boundary): {flipped}")
    assert close >= len(rows) - 2
    seq.close()


def test_prefill_8192_rows_identical_decisions(qwen):
    """The 8192-row append (the prefill configuration, the tcgen05 path) with
    the oracle's quantisation decisions at both of its sites (the taps, and
    the normed context rows feeding every layer's Wk/Wv): every stored K and
    V row of every layer agrees with the oracle's at f32 level (5e-5 of the
    largest value), and the GPU's own codes differ from the oracle's only at
    rounding boundaries.  Rows are independent, so the oracle projects all of
    them in one pass (float64, a few seconds of BLAS)."""
    import oracle.drafter as D
    from test_gpu_parity import check_sites
    g, model, om = qwen
    n = W.WORKLOADS["qwen3_8b_prefill8192"].prefill
    taps = W.make_taps(g, n, call_id=80)
    D.TRACE = D.QuantTrace()
    try:
        osq = OracleSeq(om)
        osq.append(0, taps)
        sites = D.TRACE.sites
    finally:
        D.TRACE = None
    assert len(sites) == 2
    seq = model.new_sequence(n)
    model.trace(True)
    for _, q, sc in sites:
        model.trace_force(q, sc)
    try:
        model.ctx_append(seq, 0, taps)
        own = model.trace_sites()
    finally:
        model.trace(False)
    flips = check_sites(sites, own, 5e-5)
    del sites, own
    worst = 0.0
    for l in range(g.layers):
        k, v = model.read_kv(seq, l, 0, n)
        rk, rv = osq.k[l].transpose(1, 0, 2), osq.v[l].transpose(1, 0, 2)
        ek = float(np.max(np.abs(k - rk))) / float(np.max(np.abs(rk)))
        ev = float(np.max(np.abs(v - rv))) / float(np.max(np.abs(rv)))
        worst = max(worst, ek, ev)
        assert ek <= 5e-5 and ev <= 5e-5, f"layer {l}: K {ek:.2e}, V {ev:.2e}"
    print(f"prefill 8192, identical decisions: every row of {g.layers} layers within {worst:.2e} "
          f"of max; {flips} own codes at boundaries")
    seq.close()


def test_batch32_ctx4096_sampled_sequences(qwen):
    """32 sequences of context 4096 in one batched block (the batched
    configuration); two of them against the oracle run whole."""
    g, model, om = qwen
    wl = W.WORKLOADS["qwen3_8b_batch32_ctx4096"]
    B, ctx, S = g.block, wl.ctx, wl.n_seqs
    anchors = W.make_anchors(g, S).astype(np.uint32)
    seqs = []
    for s in range(S):
        seq = model.new_sequence(ctx + B)
        for r0 in range(0, ctx, APPEND_CHUNK):
            model.ctx_append(seq, r0, W.make_taps(g, min(APPEND_CHUNK, ctx - r0), call_id=1000 + 64 * s + r0 // APPEND_CHUNK))
        seqs.append(seq)
    logits, toks = model.block(seqs, anchors, [ctx] * S, B)
    assert logits.shape == (S, B - 1, g.vocab) and toks.shape == (S, B - 1)
    # the GPU's own decisions of one more run, for the identical-decision pass
    model.trace(True)
    try:
        model.block(seqs, anchors, [ctx] * S, B)
        own = model.trace_sites()
    finally:
        model.trace(False)
    assert len(own) == 4 * g.layers + 1
    forced = [(None, q.copy(), sc.copy()) for _, q, sc in own]
    refs = {}
    for s in (0, S - 1):
        osq = OracleSeq(om)
        for r0 in range(0, ctx, APPEND_CHUNK):
            osq.append(r0, W.make_taps(g, min(APPEND_CHUNK, ctx - r0), call_id=1000 + 64 * s + r0 // APPEND_CHUNK))
        # free running: each side its own decisions
        ref, ref_tok, sites = _oracle_block_sites(om, osq, int(anchors[s]), ctx, B)
        scale = float(np.max(np.abs(ref)))
        dev = float(np.max(np.abs(logits[s] - ref))) / scale
        noise = _noise_bound(om, osq, int(anchors[s]), ctx, B, ref)
        agree = float(np.mean(toks[s] == ref_tok))
        print(f"batch32 sequence {s}: GPU vs oracle {dev:.2e} of max|logit|, oracle noise {noise:.2e}, "
              f"token agreement {agree:.3f}")
        assert dev <= 3 * noise + 2e-3
        # this sequence's rows of every site take the oracle's decisions; the
        # other sequences keep the GPU's own (sequences are independent: those
        # decisions move only their own sequences' outputs)
        assert len(sites) == len(own)
        for i, (_, q, sc) in enumerate(sites):
            rb = q.shape[0]  # B rows (layer sites) or B - 1 (the head's)
            forced[i][1][s * rb:(s + 1) * rb] = q
            forced[i][2][s * rb:(s + 1) * rb] = sc
        refs[s] = (ref, ref_tok)
    (logits_f, toks_f), _ = _forced_block(model, seqs, anchors, [ctx] * S, B, forced)
    for s, (ref, ref_tok) in refs.items():
        err = float(np.max(np.abs(logits_f[s] - ref))) / float(np.max(np.abs(ref)))
        print(f"batch32 sequence {s}, identical decisions: {err:.2e} of max|logit|")
        assert err <= 1e-4
        assert (toks_f[s] == ref_tok).all()
    for seq in seqs:
        seq.close()


def test_ctx32768_block(qwen):
    """One sequence at context 32768 (the long-context configuration)."""
    g, model, om = qwen
    wl = W.WORKLOADS["qwen3_8b_ctx32768"]
    B, ctx = g.block, wl.ctx
    seq = model.new_sequence(ctx + B)
    osq = OracleSeq(om)
    for r0 in range(0, ctx, APPEND_CHUNK):
        taps = W.make_taps(g, min(APPEND_CHUNK, ctx - r0), call_id=2000 + r0 // APPEND_CHUNK)
        model.ctx_append(seq, r0, taps)
        osq.append(r0, taps)
    assert seq.span() == (0, ctx)
    anchor = int(W.make_anchors(g, 1)[0])
    logits, toks = model.block([seq], [anchor], [ctx], B)
    ref, ref_tok = block(om, osq, anchor, ctx, B)
    scale = float(np.max(np.abs(ref)))
    dev = float(np.max(np.abs(logits[0] - ref))) / scale
    noise = _noise_bound(om, osq, anchor, ctx, B, ref)
    agree = float(np.mean(toks[0] == ref_tok))
    print(f"ctx 32768: GPU vs oracle {dev:.2e} of max|logit|, oracle noise {noise:.2e}, token agreement {agree:.3f}")
    assert dev <= 3 * noise + 2e-3
    # identical decisions in the block (the context's own decisions on each
    # side: a context row with a code at a boundary moves the attention by
    # about its 1/32768 weight times a code step)
    ref_f, ref_tok_f, sites = _oracle_block_sites(om, osq, anchor, ctx, B)
    (logits_f, toks_f), own = _forced_block(model, [seq], [anchor], [ctx], B, sites)
    err = float(np.max(np.abs(logits_f[0] - ref_f))) / float(np.max(np.abs(ref_f)))
    print(f"ctx 32768, identical decisions in the block: {err:.2e} of max|logit|")
    assert err <= 1e-4
    assert (toks_f[0] == ref_tok_f).all()
    # stored context rows near both ends and in the middle
    for p0 in (0, ctx // 2 + 7, ctx - B):
        k, v = model.read_kv(seq, g.layers - 1, p0, B)
        rk = osq.k[g.layers - 1][:, p0:p0 + B].transpose(1, 0, 2)
        rv = osq.v[g.layers - 1][:, p0:p0 + B].transpose(1, 0, 2)
        assert np.max(np.abs(k - rk)) <= 3e-2 * np.max(np.abs(rk))
        assert np.max(np.abs(v - rv)) <= 3e-2 * np.max(np.abs(rv))
    seq.close()
