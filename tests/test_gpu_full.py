"""Full-size parity on the Qwen3-8B-shaped drafter (hidden 4096, 5 layers,
32/8 heads of 128, intermediate 12288, vocab 151936, block 16, 5 taps) at
context 2048, in the launch configuration bench.py times.

* identical decisions: the oracle records every quantisation decision, the
  GPU takes the same ones; then every site's continuous values, the stored
  context K/V and the logits agree at f32 level, and the GPU's own codes
  differ from the oracle's only at rounding boundaries;
* free running: each side takes its own decisions; an f32 value within
  rounding of a half-step boundary then rounds the other way now and then,
  and every such code moves later values by a whole step, so the logits are
  compared against the spread that f32-level perturbations of the oracle's
  own decisions produce.
"""
import numpy as np
import pytest

import workloads as W
from oracle import OracleModel, OracleSeq, block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def full():
    import block_speculative_drafting_gb300 as dfl
    wl = W.WORKLOADS["qwen3_8b_ctx2048"]
    g = wl.geom
    w = W.make_weights(g)
    model = dfl.Model(g, w)
    om = OracleModel(g, w)
    yield wl, g, w, model, om
    model.close()


def _inputs(wl, g):
    B = g.block
    pre = wl.ctx - B
    return pre, W.make_taps(g, pre, call_id=0), W.make_taps(g, B, call_id=1), int(W.make_anchors(g, 1)[0])


def test_full_size_identical_decisions(full):
    import oracle.drafter as D
    from test_gpu_parity import check_sites
    wl, g, w, model, om = full
    B = g.block
    pre, taps0, taps1, anchor = _inputs(wl, g)
    D.TRACE = D.QuantTrace()
    try:
        osq = OracleSeq(om)
        osq.append(0, taps0)
        osq.append(pre, taps1)
        ref, ref_tok = block(om, osq, anchor, wl.ctx, B)
        sites = D.TRACE.sites
    finally:
        D.TRACE = None
    seq = model.new_sequence(wl.ctx + 2 * B)
    model.trace(True)
    for x, q, s in sites:
        model.trace_force(q, s)
    try:
        model.ctx_append(seq, 0, taps0)
        model.ctx_append(seq, pre, taps1)
        logits, toks = model.block([seq], [anchor], [wl.ctx], B)
        own = model.trace_sites()
    finally:
        model.trace(False)
    flips = check_sites(sites, own, 5e-5)
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(logits[0] - ref)))
    print(f"full-size, identical decisions: {len(sites)} sites, {flips} own codes at boundaries, "
          f"max|dlogit|/max|logit| = {err / scale:.2e}")
    assert err <= 1e-5 * scale
    assert (toks[0] == ref_tok).all()
    for l in (0, g.layers - 1):
        for p0 in (0, 1017, pre):
            k, v = model.read_kv(seq, l, p0, B)
            rk = osq.k[l][:, p0:p0 + B].transpose(1, 0, 2)
            rv = osq.v[l][:, p0:p0 + B].transpose(1, 0, 2)
            assert np.max(np.abs(k - rk)) <= 5e-5 * np.max(np.abs(rk))
            assert np.max(np.abs(v - rv)) <= 5e-5 * np.max(np.abs(rv))
    seq.close()


def test_full_size_free_running_within_decision_noise(full):
    import oracle.drafter as D
    from oracle import quant as Q
    wl, g, w, model, om = full
    B = g.block
    pre, taps0, taps1, anchor = _inputs(wl, g)
    seq = model.new_sequence(wl.ctx + 2 * B)
    model.ctx_append(seq, 0, taps0)
    model.ctx_append(seq, pre, taps1)
    logits, toks = model.block([seq], [anchor], [wl.ctx], B)
    osq = OracleSeq(om)
    osq.append(0, taps0)
    osq.append(pre, taps1)
    ref, ref_tok = block(om, osq, anchor, wl.ctx, B)
    scale = float(np.max(np.abs(ref)))
    gpu_dev = float(np.max(np.abs(logits[0] - ref))) / scale
    # the oracle against itself with f32-level noise on the values it quantises
    orig = Q.quantize_rows_i8
    rng = np.random.default_rng(0)
    devs = []
    try:
        Q.quantize_rows_i8 = lambda x: orig(np.asarray(x, np.float64) * (1 + 1e-7 * rng.standard_normal(np.shape(x))))
        for _ in range(2):
            lp, _ = block(om, osq, anchor, wl.ctx, B)
            devs.append(float(np.max(np.abs(lp - ref))) / scale)
    finally:
        Q.quantize_rows_i8 = orig
    agree = float(np.mean(toks[0] == ref_tok))
    print(f"full-size, free running: GPU vs oracle {gpu_dev:.2e} of max|logit| (token agreement {agree:.3f}); "
          f"oracle vs f32-perturbed oracle {devs}")
    assert gpu_dev <= 3 * max(devs) + 2e-3
    seq.close()


def test_full_size_argmax_agreement_over_1005_rows(full):
    """Draft tokens of 67 context-2048 blocks (1005 rows) against the
    oracle's, binned by the oracle's top-2 margin: with identical decisions
    (context and block) every row agrees; free running, every row whose
    margin exceeds a tenth of max|logit| agrees, and the table reports the
    rest."""
    import oracle.drafter as D
    from test_gpu_parity import agreement_table, print_agreement
    wl, g, w, model, om = full
    B, n = g.block, wl.ctx
    taps = W.make_taps(g, n, call_id=500)
    D.TRACE = D.QuantTrace()
    try:
        osq = OracleSeq(om)
        osq.append(0, taps)
        ctx_sites = D.TRACE.sites
    finally:
        D.TRACE = None
    seq = model.new_sequence(n + B)
    model.trace(True)
    for _, q, s in ctx_sites:
        model.trace_force(q, s)
    try:
        model.ctx_append(seq, 0, taps)
    finally:
        model.trace(False)
    records = []
    for a in W.make_anchors(g, 67, call_id=501):
        D.TRACE = D.QuantTrace()
        try:
            ref, _ = block(om, osq, int(a), n, B)
            sites = D.TRACE.sites
        finally:
            D.TRACE = None
        model.trace(True)
        for _, q, s in sites:
            model.trace_force(q, s)
        try:
            _, tf = model.block([seq], [int(a)], [n], B, want_logits=False)
        finally:
            model.trace(False)
        _, tr = model.block([seq], [int(a)], [n], B, want_logits=False)
        records.append((ref, tf[0], tr[0]))
    seq.close()
    table, forced, free, m, er = agreement_table(records)
    print_agreement(f"qwen3_8b_ctx2048, {len(records)} blocks, {sum(t[2] for t in table)} rows", table, forced, free)
    assert forced == 1.0
    assert er[m >= 0.1].all()
