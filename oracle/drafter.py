"""The DFlash 2 block drafter on the CPU, in float64 — TEST INFRASTRUCTURE.

Restated from the page "cortiq-engine 0.8.71 — src/dflash.rs" (module
documentation; ``rms``; ``Drafter::rotate``; ``Drafter::mlp``;
``Drafter::push_context`` / ``queue_context`` / ``truncate`` / ``reset``;
``Drafter::settle_rows``; ``Drafter::block``; ``top_k``), with:

* the DFlash 2 row convolution (``conv_in`` / ``conv`` / ``conv_out``:
  stage 0 on the normed rows before a sub-layer, stage 1 on its output before
  the residual add, both with the dynamic kernels projected from the normed
  rows) where the geometry has one (``conv_kernel > 0``); without one the
  sub-layers are unwrapped, the reading the workloads take since they fix no
  convolution geometry;
* rows queued for later settling not modelled: every append settles at once
  (the values are the same, only the time they are computed moves);
* in the quantised format (``quant=1``), every matrix input row quantised to
  int8 before its matvec (``oracle.quant``); the draft-layer matrices, ``fc``
  and the per-layer Wk/Wv 4-bit g32; the head int8 per row;
* the geometry's attention variants: per-layer windows (``window`` for
  every layer, or the ``windows`` list; 0 is the whole context) with the
  row-dependent mask of ``block`` and the drop of context rows no block row
  of a layer can see any more (``settle_rows``), and layers whose queries
  and keys carry no rotary position (``no_rope``);
* the candidate selector after the head where the geometry has one
  (``selector_rank > 0``): the draft tokens are then its choices;
* continuous arithmetic in float64; the decisions that pick an integer (the
  quantised codes, the draft token's argmax) taken in float32; the RoPE angle
  rounded to float32 before its cosine and sine, as the page's ``rotate``
  computes it (``inv_freq`` in f64 rounded to f32, times the f32 position).
"""
from __future__ import annotations

import math

import numpy as np

from . import quant as Q

F64 = np.float64


def rms(x, w, eps):
    """RMSNorm of each row: x / sqrt(mean(x^2) + eps) * w (float64)."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=F64)


def row_conv(base, d, x, stage, kn, gs):
    """One stage of the DFlash 2 row convolution over a block's rows (page
    "cortiq-engine 0.8.71 — src/dflash.rs", `conv`): output row r is the sum
    over row offsets o < min(kn, r + 1) of (base[stage][o] + the row's
    dynamic kernel value of its column group) times input row r - o.

    base: [2, kn, hidden]; d: [rows, 2 * kn * groups], row r's dynamic
    kernels in the order (stage, offset, group); x: [rows, hidden];
    gs: columns per group.  Returns [rows, hidden] (float64).
    """
    x = np.asarray(x, dtype=F64)
    rows, hs = x.shape
    groups = hs // gs
    dyn = np.asarray(d, dtype=F64).reshape(rows, 2, kn, groups)
    base = np.asarray(base, dtype=F64).reshape(2, kn, hs)
    y = np.zeros((rows, hs), dtype=F64)
    for r in range(rows):
        for o in range(min(kn, r + 1)):
            kernel = base[stage, o] + np.repeat(dyn[r, stage, o], gs)
            y[r] += kernel * x[r - o]
    return y


def silu(a):
    """a * sigmoid(a) = a / (1 + e^-a) (the page's ``mlp``)."""
    a = np.asarray(a, dtype=F64)
    return a / (1.0 + np.exp(-a))


def inv_freq(head_dim, theta):
    """inv_freq[i] = theta^(-2i/hd), computed in f64, kept as f32 (``Drafter::new``)."""
    half = head_dim // 2
    return np.array([theta ** (-(2.0 * i) / head_dim) for i in range(half)], dtype=np.float64).astype(np.float32)


def rope(x, pos, inv_f):
    """Rotate rows of heads by position, half-split pairs (``Drafter::rotate``).

    x: [rows, heads, hd] float64; pos: [rows] integer positions.
    The pair (lo[i], hi[i]) = (x[i], x[i + hd/2]) turns by the angle
    f32(f32(pos) * inv_freq[i]).
    """
    x = np.asarray(x, dtype=F64)
    hd = x.shape[-1]
    half = hd // 2
    p32 = np.asarray(pos, dtype=np.float32)
    ang = (p32[:, None] * inv_f[None, :]).astype(np.float32).astype(F64)  # one f32 multiply
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def top_k(x, k):
    """The k largest of x with their indices, largest first, the first of
    equal values kept ahead of later ones (the page's ``top_k``)."""
    x = np.asarray(x)
    order = np.argsort(-x, kind="stable")[:k]
    return [(x[i].item(), int(i)) for i in order]


def argmax_first(rows32):
    """Per row: the index of the largest value, the lowest index among equals
    (``top_k`` with k = 1), decided on float32 values."""
    return np.argmax(np.asarray(rows32, dtype=np.float32), axis=-1).astype(np.uint32)


def softmax(s):
    """Max-subtract, exp, divide by the sum (as ``Drafter::block``); -inf
    entries become 0."""
    top = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - top)
    return e / np.sum(e, axis=-1, keepdims=True)


class QuantTrace:
    """Records the oracle's quantisation decisions in call order: per site the
    input values (float64), the int8 codes and the f32 row scales.  A site whose
    input equals the previous site's (the same rows feeding Wq, Wk and Wv, or
    gate and up, or every layer's Wk/Wv of the context) is recorded once."""

    def __init__(self):
        self.sites = []

    def record(self, x, q, s):
        x = np.asarray(x, dtype=F64)
        if self.sites and self.sites[-1][0].shape == x.shape and np.array_equal(self.sites[-1][0], x):
            return
        self.sites.append((x.copy(), q.copy(), s.copy()))


TRACE = None  # a QuantTrace while the decisions are being recorded


class Matrix:
    """One weight matrix [out][in] as the oracle applies it.

    f32 format: the float32 weights.  4-bit format: codes q and f16 scales s
    (``oracle.quant.quantize_q4g32``), applied as the exact real values s*q.
    int8-row format (the head): codes and f32 row scales.
    """

    ROWS_PER_CHUNK = 8192

    def __init__(self, w, fmt):
        self.fmt = fmt
        self.rows, self.cols = w.shape
        if fmt == "f32":
            self.dq = np.ascontiguousarray(w, dtype=np.float32)
        elif fmt == "q4g32":
            self.q, self.s = Q.quantize_q4g32(w)
            self.dq = Q.dequant_q4g32(self.q, self.s, np.float32)  # s*q exact in f32
        elif fmt == "i8row":
            self.q, self.s = Q.quantize_rows_i8(w)
            self.dq = None  # applied as integer codes, scales after the sum
        else:
            raise ValueError(fmt)

    def apply(self, x):
        """y = W x for each row of x.  Quantised formats quantise each input
        row to int8 first (``oracle.quant.quantize_rows_i8``)."""
        x = np.asarray(x, dtype=F64)
        out = np.empty((x.shape[0], self.rows), dtype=F64)
        if self.fmt == "f32":
            xin = x
        else:
            qx, sx = Q.quantize_rows_i8(x)
            if TRACE is not None:
                TRACE.record(x, qx, sx)
            xin = qx.astype(F64)
        for r0 in range(0, self.rows, self.ROWS_PER_CHUNK):
            r1 = min(self.rows, r0 + self.ROWS_PER_CHUNK)
            w = (self.q if self.fmt == "i8row" else self.dq)[r0:r1].astype(F64)
            out[:, r0:r1] = xin @ w.T
        if self.fmt == "i8row":
            out *= self.s.astype(F64)[None, :]
        if self.fmt != "f32":
            out *= sx.astype(F64)[:, None]
        return out


class OracleModel:
    """A drafter's weights as the oracle holds them.

    ``weights`` is the dict of float32 arrays from ``workloads.make_weights``.
    """

    def __init__(self, geom, weights):
        g = self.g = geom
        if g.heads % g.kv_heads or g.head_dim % 2 or g.block < 2:
            raise ValueError(f"unsupported geometry {g}")
        mfmt = "q4g32" if g.quant else "f32"
        hfmt = "i8row" if g.quant else "f32"
        self.fc = Matrix(weights["fc"], mfmt)
        self.hidden_norm = np.asarray(weights["hidden_norm"], dtype=F64)
        self.norm = np.asarray(weights["norm"], dtype=F64)
        self.embed = weights["embed"]  # float32 [vocab][hidden], the target's
        self.head = Matrix(weights["head"], hfmt)
        if getattr(g, "selector_rank", 0):
            # the candidate selector: the rows' projection (f32 on the page)
            # and the predecessor / successor codebooks (f16 [vocab][rank])
            self.sel = np.asarray(weights["selector_projection"], dtype=F64)
            self.book_p = np.asarray(weights["predecessor_codebook"], dtype=np.float16).astype(F64)
            self.book_c = np.asarray(weights["successor_codebook"], dtype=np.float16).astype(F64)
        self.layers = []
        for lw in weights["layers"]:
            layer = {
                "in_norm": np.asarray(lw["in_norm"], dtype=F64),
                "post_norm": np.asarray(lw["post_norm"], dtype=F64),
                "q_norm": np.asarray(lw["q_norm"], dtype=F64),
                "k_norm": np.asarray(lw["k_norm"], dtype=F64),
                **{name: Matrix(lw[name], mfmt) for name in ("q", "k", "v", "o", "gate", "up", "down")},
            }
            if getattr(g, "conv_kernel", 0):
                # the row convolutions: base kernels and the f32 kernel projections
                for c in ("attn_conv", "mlp_conv"):
                    layer[c + "_base"] = np.asarray(lw[c + "_base"], dtype=F64)
                    layer[c + "_proj"] = np.asarray(lw[c + "_proj"], dtype=F64)
            self.layers.append(layer)
        self.inv_f = inv_freq(g.head_dim, g.rope_theta)

    def window_of(self, layer):
        """Positions a block row of layer `layer` sees back (0: all): the
        per-layer list where the geometry gives one, else the one window
        (page "cortiq-engine 0.8.71 — src/dflash.rs", `Geometry`: `window`,
        `windows`)."""
        g = self.g
        ws = getattr(g, "windows", ())
        return ws[layer] if ws else g.window

    def rotary(self, layer):
        """Whether layer `layer`'s queries and keys carry the rotary
        position (`Geometry::no_rope` lists the layers that do not)."""
        return layer not in getattr(self.g, "no_rope", ())


class OracleSeq:
    """One sequence's context: positions ``first .. first + len``; per layer,
    per KV head, the keys (normed, rotated) and values of the positions the
    layer still holds (``dropped`` rows left its window)."""

    # context rows projected at a time.  Rows are independent, so this only
    # groups the quantisation trace's records (one per pass and site); it is
    # the library's append pass, so that traced decisions line up one to one.
    ROWS_PER_PASS = 8192

    # rows that may wait in the queue before the oldest are settled, and the
    # granule they are settled in (page "cortiq-engine 0.8.71 —
    # src/dflash.rs": `PENDING_ROWS`, `CONTEXT_CHUNK`, `BLOCK_SLACK`)
    PENDING_ROWS = 512
    CONTEXT_CHUNK = 64
    BLOCK_SLACK = 256

    def __init__(self, model):
        self.m = model
        g = model.g
        self.first = 0
        self.len = 0
        self.k = [np.zeros((g.kv_heads, 0, g.head_dim)) for _ in range(g.layers)]
        self.v = [np.zeros((g.kv_heads, 0, g.head_dim)) for _ in range(g.layers)]
        self.dropped = [0] * g.layers
        self.pending = np.zeros((0, g.tap_width), dtype=np.float32)  # queued rows, not yet context

    # -- positions (``Drafter::next_position``, ``truncate``, ``reset``) --
    def next_position(self):
        return self.first + self.len + self.pending.shape[0]

    def truncate(self, pos):
        held = self.first + self.len
        self.pending = self.pending[:max(pos - held, 0)]
        keep = min(max(pos - self.first, 0), self.len)
        for li in range(self.m.g.layers):
            rows = max(keep - self.dropped[li], 0)
            self.k[li] = self.k[li][:, :rows]
            self.v[li] = self.v[li][:, :rows]
            self.dropped[li] = min(self.dropped[li], keep)
        self.len = keep

    def reset(self):
        self.truncate(0)
        self.first = 0

    # -- context (``push_context`` / ``queue_context`` then ``settle_rows``) --
    def append(self, pos, taps):
        """Add the target's rows of positions pos.. : rows at held positions
        replace them and what follows; a gap (or a position before the
        first) starts the context over at pos."""
        g = self.m.g
        taps = np.asarray(taps, dtype=np.float32).reshape(-1, g.tap_width)
        if pos > self.next_position() or pos < self.first:
            self.truncate(0)
            self.first = pos
        else:
            self.truncate(pos)
        # queued rows still held go first, all in one settle (`push_context`
        # is the queue then a settle; the queue's limit would only split the
        # same rows into two settles)
        rows, self.pending = np.concatenate([self.pending, taps]), self.pending[:0]
        self._settle(self.first + self.len, rows)

    def project(self, pos, taps):
        """The context rows' keys and values: t = rms(fc . taps, hidden_norm);
        per layer k = rot(rms_head(Wk t, k_norm), position), v = Wv t.
        Returns ([L] of [n, kv, hd] keys, [L] of [n, kv, hd] values)."""
        m, g = self.m, self.m.g
        n = taps.shape[0]
        t = rms(m.fc.apply(taps), m.hidden_norm, g.eps)
        ks, vs = [], []
        positions = np.arange(pos, pos + n)
        for li, L in enumerate(m.layers):
            k = L["k"].apply(t).reshape(n, g.kv_heads, g.head_dim)
            k = rms(k, L["k_norm"], g.eps)
            if m.rotary(li):
                k = rope(k, positions, m.inv_f)
            v = L["v"].apply(t).reshape(n, g.kv_heads, g.head_dim)
            ks.append(k)
            vs.append(v)
        return ks, vs

    def queue(self, pos, taps):
        """``append`` put off (`queue_context`): the rows wait until a block
        reads the context (``settle``); past the queue's limit the oldest go
        through at once, a multiple of the chunk granule.  The limit is the
        page's device one: with every layer windowed, the widest window plus
        a slack when that is more than PENDING_ROWS."""
        g = self.m.g
        taps = np.asarray(taps, dtype=np.float32).reshape(-1, g.tap_width)
        if pos > self.next_position() or pos < self.first:
            self.truncate(0)
            self.first = pos
        else:
            self.truncate(pos)
        self.pending = np.concatenate([self.pending, taps])
        wins = [self.m.window_of(li) for li in range(g.layers)]
        limit = self.PENDING_ROWS
        if all(w > 0 for w in wins):
            limit = max(self.PENDING_ROWS, max(wins) + self.BLOCK_SLACK)
        held = self.pending.shape[0]
        if held > limit:
            over = min(-(-(held - limit) // self.CONTEXT_CHUNK) * self.CONTEXT_CHUNK, held)
            rows, self.pending = self.pending[:over], self.pending[over:]
            self._settle(self.first + self.len, rows)

    def settle(self):
        """Make every queued row context (`settle`)."""
        if self.pending.shape[0]:
            rows, self.pending = self.pending, self.pending[:0]
            self._settle(self.first + self.len, rows)

    def _settle(self, pos, taps):
        g = self.m.g
        for r0 in range(0, taps.shape[0], self.ROWS_PER_PASS):
            chunk = taps[r0:r0 + self.ROWS_PER_PASS]
            ks, vs = self.project(pos + r0, chunk)
            for li in range(g.layers):
                self.k[li] = np.concatenate([self.k[li], ks[li].transpose(1, 0, 2)], axis=1)
                self.v[li] = np.concatenate([self.v[li], vs[li].transpose(1, 0, 2)], axis=1)
            self.len += chunk.shape[0]
        # no row of a layer sees further back than its window: drop what fell out
        for li in range(g.layers):
            w = self.m.window_of(li)
            held = self.len - self.dropped[li]
            if w > 0 and held > 2 * w:
                cut = held - w
                self.k[li] = self.k[li][:, cut:]
                self.v[li] = self.v[li][:, cut:]
                self.dropped[li] += cut

    def ctx_range(self, li, anchor_pos):
        """The context positions [lo, hi) a block anchored at anchor_pos reads
        in layer li."""
        base = self.first + self.dropped[li]
        hi = max(min(anchor_pos, self.first + self.len), base)
        w = self.m.window_of(li)
        lo = min(max(anchor_pos + 1 - w, base), hi) if w > 0 else base
        return lo, hi


def attention(q, kb, vb, kc, vc, rep, scale, row_from=None, ctx_lo=0):
    """Attention of a block's rows over the context plus the block (not causal).

    q: [rows, heads, hd]; kb, vb: [rows, kv, hd] (the block's own keys and
    values); kc, vc: [kv, n, hd] (context keys and values of positions
    ctx_lo .. ctx_lo + n).  Query head h reads KV head h // rep.
    row_from: optional [rows] first context position each row may see
    (a window); earlier positions are masked with -inf.
    Returns [rows, heads, hd].
    """
    rows, heads, hd = q.shape
    n = kc.shape[1]
    y = np.zeros(q.shape, dtype=F64)
    for h in range(heads):
        gi = h // rep
        keys = np.concatenate([kc[gi], kb[:, gi, :]], axis=0)  # [n + rows, hd]
        vals = np.concatenate([vc[gi], vb[:, gi, :]], axis=0)
        s = (q[:, h, :] @ keys.T) * scale  # [rows, n + rows]
        if row_from is not None:
            for r in range(rows):
                cut = min(max(row_from[r] - ctx_lo, 0), n)
                s[r, :cut] = -np.inf
        y[:, h, :] = softmax(s) @ vals
    return y


def block(model, seq, anchor_tok, anchor_pos, block_len=None, return_hidden=False):
    """One block: rows [anchor, MASK, ...] at positions anchor_pos.. through
    every draft layer, then the head over the rows after the anchor.

    Returns (logits float64 [block_len - 1, vocab], draft tokens uint32
    [block_len - 1]) and, with return_hidden, the final normed hidden rows.
    """
    m, g = model, model.g
    rows = g.block if block_len is None else block_len
    if not 2 <= rows <= g.block:
        raise ValueError(f"block_len {rows} outside [2, {g.block}]")
    seq.settle()  # the queued rows become context before a block reads it
    hd, nh, kv = g.head_dim, g.heads, g.kv_heads
    scale = 1.0 / math.sqrt(hd)
    toks = [int(anchor_tok)] + [g.mask] * (rows - 1)
    h = np.asarray(m.embed[toks], dtype=F64)
    positions = np.arange(anchor_pos, anchor_pos + rows)
    for li, L in enumerate(m.layers):
        lo, hi = seq.ctx_range(li, anchor_pos)
        base = seq.first + seq.dropped[li]
        kc = seq.k[li][:, lo - base:hi - base]
        vc = seq.v[li][:, lo - base:hi - base]
        conv = getattr(g, "conv_kernel", 0)
        kn, gs = conv, getattr(g, "conv_group", 0)
        x = rms(h, L["in_norm"], g.eps)
        if conv:
            # x, d = conv_in(x): the row's dynamic kernels from the normed rows, then stage 0
            da = x @ L["attn_conv_proj"].T
            x = row_conv(L["attn_conv_base"], da, x, 0, kn, gs)
        q = L["q"].apply(x).reshape(rows, nh, hd)
        k = L["k"].apply(x).reshape(rows, kv, hd)
        v = L["v"].apply(x).reshape(rows, kv, hd)
        q = rms(q, L["q_norm"], g.eps)
        k = rms(k, L["k_norm"], g.eps)
        if m.rotary(li):
            q = rope(q, positions, m.inv_f)
            k = rope(k, positions, m.inv_f)
        w = m.window_of(li)
        row_from = [max(anchor_pos + r + 1 - w, 0) for r in range(rows)] if w > 0 else None
        y = attention(q, k, v, kc, vc, g.rep, scale, row_from, lo)
        o = L["o"].apply(y.reshape(rows, nh * hd))
        if conv:
            o = row_conv(L["attn_conv_base"], da, o, 1, kn, gs)  # conv_out(O y, d)
        h = h + o
        x = rms(h, L["post_norm"], g.eps)
        if conv:
            dm = x @ L["mlp_conv_proj"].T
            x = row_conv(L["mlp_conv_base"], dm, x, 0, kn, gs)
        a = silu(L["gate"].apply(x)) * L["up"].apply(x)
        dn = L["down"].apply(a)
        if conv:
            dn = row_conv(L["mlp_conv_base"], dm, dn, 1, kn, gs)
        h = h + dn
    hn = rms(h, m.norm, g.eps)
    logits = m.head.apply(hn[1:])
    toks = argmax_first(logits)
    if getattr(g, "selector_rank", 0):
        toks, _ = select(m, hn[1:], logits, anchor_tok)
    if return_hidden:
        return logits, toks, hn
    return logits, toks


def select(model, hn, logits, anchor):
    """The candidate selector (page "cortiq-engine 0.8.71 — src/dflash.rs",
    `select` / `select_with`): row by row, its `selector_top` candidates by
    logit (``top_k`` on the float32 logits) re-scored as logit + (P[prev] ⊙
    S·h) · C[candidate], the best (the first of equals, in candidate order)
    taken and fed to the next row as prev; the anchor is the first row's prev.

    hn: [n, hidden] the rows after the last norm; logits: [n, vocab].
    Returns (chosen, plain) uint32 [n]: the selected tokens and each row's own
    top token.
    """
    g = model.g
    hp = np.asarray(hn, dtype=F64) @ model.sel.T  # S . h: [n, rank]
    prev, chosen, plain = int(anchor), [], []
    for j in range(hp.shape[0]):
        cand = top_k(np.asarray(logits[j], dtype=np.float32), g.selector_top)
        plain.append(cand[0][1])
        pc = model.book_p[prev] * hp[j]
        best_s, best_t = -math.inf, cand[0][1]
        for unary, tok in cand:
            s = unary + float(pc @ model.book_c[tok])
            if s > best_s:
                best_s, best_t = s, tok
        prev = best_t
        chosen.append(prev)
    return np.array(chosen, dtype=np.uint32), np.array(plain, dtype=np.uint32)
