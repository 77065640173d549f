"""Pins of the oracle's primitives: RMSNorm, RoPE, SiLU, softmax, attention,
top_k, against closed forms, invariants, library routines and the page's own
worked example."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention, inv_freq, rms, rope, silu, softmax, top_k
from oracle.drafter import argmax_first

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- RMSNorm
def test_rms_unit_rms_with_unit_gain():
    x = np.random.default_rng(0).standard_normal((4, 256)) * 3.0
    eps = 1e-6
    y = rms(x, np.ones(256), eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean(y * y, axis=1), ms / (ms + eps), rtol=1e-12)


def test_rms_against_torch_library():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 96))
    w = 1 + 0.1 * rng.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), eps=1e-5).numpy()
    np.testing.assert_allclose(rms(x, w, 1e-5), ref, rtol=1e-12, atol=1e-14)


def test_rms_constant_row_closed_form():
    # a row of constant c has mean square c^2: y = c / sqrt(c^2 + eps) * w
    c, eps = 0.5, 1e-3
    y = rms(np.full((1, 8), c), np.arange(1, 9, dtype=float), eps)
    np.testing.assert_allclose(y[0], c / math.sqrt(c * c + eps) * np.arange(1, 9), rtol=1e-14)


# ---------------------------------------------------------------- RoPE
def test_inv_freq_values():
    np.testing.assert_array_equal(inv_freq(4, 10000.0), np.array([1.0, 0.01], dtype=np.float32))
    f = inv_freq(128, 1e6)
    assert f.dtype == np.float32 and f[0] == 1.0
    assert f[-1] == np.float32(1e6 ** (-126 / 128))


def test_rope_is_complex_rotation_of_half_split_pairs():
    """Pair i = (x[i], x[i + hd/2]) as the complex number x[i] + j x[i+hd/2],
    multiplied by e^{j angle}, angle = f32(f32(p) * inv_freq[i])."""
    rng = np.random.default_rng(2)
    hd, heads = 16, 3
    f = inv_freq(hd, 1e4)
    pos = np.array([0, 1, 7, 1000, 32767])
    x = rng.standard_normal((len(pos), heads, hd))
    y = rope(x, pos, f)
    half = hd // 2
    for r, p in enumerate(pos):
        ang = (np.float32(p) * f).astype(np.float64)
        z = (x[r, :, :half] + 1j * x[r, :, half:]) * np.exp(1j * ang)[None, :]
        np.testing.assert_allclose(y[r, :, :half], z.real, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(y[r, :, half:], z.imag, rtol=1e-12, atol=1e-12)


def test_rope_identity_at_zero_and_pair_norms():
    rng = np.random.default_rng(3)
    hd = 64
    f = inv_freq(hd, 1e6)
    x = rng.standard_normal((2, 4, hd))
    np.testing.assert_array_equal(rope(x, np.array([0, 0]), f), x)
    y = rope(x, np.array([5, 12345]), f)
    half = hd // 2
    n_in = x[..., :half] ** 2 + x[..., half:] ** 2
    n_out = y[..., :half] ** 2 + y[..., half:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


def test_rope_dot_depends_on_position_difference():
    # with exactly representable angles (p * 2^-k), <rot(q,p), rot(k,p')> depends on p - p' only
    hd = 8
    f = np.array([1.0, 0.5, 0.25, 0.125], dtype=np.float32)
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 1, hd))
    k = rng.standard_normal((1, 1, hd))
    d = [float(np.sum(rope(q, np.array([p + 3]), f) * rope(k, np.array([p]), f))) for p in (0, 1, 10, 100)]
    np.testing.assert_allclose(d, d[0], rtol=1e-10)


# ---------------------------------------------------------------- SiLU
def test_silu_identities_and_library():
    x = np.linspace(-30, 30, 601)
    s = silu(x)
    np.testing.assert_allclose(s - silu(-x), x, atol=1e-12)  # x*sig(x) - (-x)*sig(-x) = x
    assert silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(s, torch.nn.functional.silu(torch.from_numpy(x)).numpy(), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- softmax / attention
def test_softmax_against_library_and_masked():
    from scipy.special import softmax as sp_softmax
    s = np.random.default_rng(5).standard_normal((4, 9)) * 5
    np.testing.assert_allclose(softmax(s), sp_softmax(s, axis=-1), rtol=1e-13)
    s[:, :3] = -np.inf
    p = softmax(s)
    assert (p[:, :3] == 0).all()
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=1e-14)


def _sdpa(q, kb, vb, kc, vc, rep, scale, mask=None):
    """torch's library attention over [context ++ block] keys, KV heads
    repeated rep times (query head h reads KV head h // rep)."""
    keys = np.concatenate([kc.transpose(1, 0, 2), kb], axis=0)  # [n+rows, kv, hd]
    vals = np.concatenate([vc.transpose(1, 0, 2), vb], axis=0)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]  # [1, heads, rows, hd]
    tk = torch.from_numpy(keys).permute(1, 0, 2).repeat_interleave(rep, dim=0)[None]
    tv = torch.from_numpy(vals).permute(1, 0, 2).repeat_interleave(rep, dim=0)[None]
    m = None if mask is None else torch.from_numpy(mask)
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, scale=scale)
    return out[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("rows,heads,kv,n", [(4, 4, 2, 9), (3, 6, 6, 5), (8, 8, 1, 0), (2, 2, 1, 1)])
def test_attention_against_library(rows, heads, kv, n):
    rng = np.random.default_rng(rows * 100 + heads + n)
    hd = 16
    q = rng.standard_normal((rows, heads, hd))
    kb, vb = rng.standard_normal((2, rows, kv, hd))
    kc, vc = rng.standard_normal((2, kv, n, hd))
    scale = 1 / math.sqrt(hd)
    y = attention(q, kb, vb, kc, vc, heads // kv, scale)
    np.testing.assert_allclose(y, _sdpa(q, kb, vb, kc, vc, heads // kv, scale), rtol=1e-10, atol=1e-12)


def test_attention_brute_force_scalar_loops():
    rng = np.random.default_rng(7)
    rows, heads, kv, n, hd = 3, 2, 1, 4, 4
    q = rng.standard_normal((rows, heads, hd))
    kb, vb = rng.standard_normal((2, rows, kv, hd))
    kc, vc = rng.standard_normal((2, kv, n, hd))
    y = attention(q, kb, vb, kc, vc, 2, 0.5)
    for r in range(rows):
        for h in range(heads):
            keys = [kc[0, j] for j in range(n)] + [kb[j, 0] for j in range(rows)]
            vals = [vc[0, j] for j in range(n)] + [vb[j, 0] for j in range(rows)]
            sc = [0.5 * sum(q[r, h, d] * kk[d] for d in range(hd)) for kk in keys]
            mx = max(sc)
            e = [math.exp(v - mx) for v in sc]
            tot = sum(e)
            for d in range(hd):
                assert y[r, h, d] == pytest.approx(sum(e[j] * vals[j][d] for j in range(len(e))) / tot, rel=1e-12)


def test_attention_constant_values_and_window_cases():
    rng = np.random.default_rng(8)
    rows, heads, kv, n, hd = 4, 4, 2, 6, 8
    q = rng.standard_normal((rows, heads, hd))
    kb = rng.standard_normal((rows, kv, hd))
    kc = rng.standard_normal((kv, n, hd))
    c = rng.standard_normal(hd)
    vb = np.broadcast_to(c, (rows, kv, hd)).copy()
    vc = np.broadcast_to(c, (kv, n, hd)).copy()
    y = attention(q, kb, vb, kc, vc, 2, 0.3)
    np.testing.assert_allclose(y, np.broadcast_to(c, y.shape), rtol=1e-12)
    # window reaching past the whole context equals no window
    vb, vc = rng.standard_normal((rows, kv, hd)), rng.standard_normal((kv, n, hd))
    a, lo = 100, 94  # context positions 94..99, anchor 100
    full = attention(q, kb, vb, kc, vc, 2, 0.3)
    wide = attention(q, kb, vb, kc, vc, 2, 0.3, row_from=[max(a + r + 1 - 1000, 0) for r in range(rows)], ctx_lo=lo)
    np.testing.assert_allclose(wide, full, rtol=1e-14)
    # window 1: a row sees no context position at all, only the block's rows
    one = attention(q, kb, vb, kc, vc, 2, 0.3, row_from=[a + r for r in range(rows)], ctx_lo=lo)
    blk = attention(q, kb, vb, kc[:, :0], vc[:, :0], 2, 0.3)
    np.testing.assert_allclose(one, blk, rtol=1e-14)
    # window 3 against the library with an explicit boolean mask
    w = 3
    mask = np.ones((rows, n + rows), dtype=bool)
    for r in range(rows):
        for j in range(n):
            mask[r, j] = lo + j >= a + r + 1 - w
    got = attention(q, kb, vb, kc, vc, 2, 0.3, row_from=[a + r + 1 - w for r in range(rows)], ctx_lo=lo)
    np.testing.assert_allclose(got, _sdpa(q, kb, vb, kc, vc, 2, 0.3, mask), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- top_k
def test_top_k_page_example():
    with open(os.path.join(GOLDEN, "top_k_page_example.txt")) as fh:
        lines = [l.strip() for l in fh if l.strip() and not l.startswith("#")]
    x = [float(v) for v in lines[0].split(":", 1)[1].split()]
    for line in lines[1:]:
        k, rest = line.split(":", 1)
        want = [(float(p.split(",")[0]), int(p.split(",")[1])) for p in rest.split()]
        assert top_k(x, int(k)) == want


# ---------------------------------------------------------------- argmax_first
def _page_example_row():
    with open(os.path.join(GOLDEN, "top_k_page_example.txt")) as fh:
        lines = [l.strip() for l in fh if l.strip() and not l.startswith("#")]
    return [float(v) for v in lines[0].split(":", 1)[1].split()]


def test_argmax_first_keeps_the_first_of_equals_page_example():
    # The page's `top_k` test (page "cortiq-engine 0.8.71 — src/dflash.rs",
    # `top_k_orders_and_keeps_first_of_equals`) ranks the value 2.0 at index 1
    # ahead of the equal 2.0 at index 3.  With the unique maximum 3.5 taken
    # out of that row, the draft token's argmax must therefore be index 1.
    x = np.array(_page_example_row())
    assert argmax_first(x[None, :])[0] == 4
    y = x.copy()
    y[4] = -np.inf
    assert argmax_first(y[None, :])[0] == 1
    # the same row with the equal pair moved: the first of them wins wherever it sits
    for a, b in [(0, 5), (2, 3), (1, 2), (0, 1)]:
        z = np.full(6, -1.0)
        z[a] = z[b] = 7.0
        assert argmax_first(z[None, :])[0] == min(a, b)


def test_argmax_first_ties_at_several_positions():
    rng = np.random.default_rng(5)
    rows, width = 64, 997
    x = rng.uniform(-1.0, 1.0, size=(rows, width)).astype(np.float32)
    want = np.empty(rows, dtype=np.uint32)
    for r in range(rows):
        pos = np.sort(rng.choice(width, size=1 + r % 5, replace=False))
        x[r, pos] = 2.0
        want[r] = pos[0]
    assert np.array_equal(argmax_first(x), want)
    # an all-equal row (a head of zeros gives one): index 0
    assert argmax_first(np.zeros((3, 17), dtype=np.float32)).tolist() == [0, 0, 0]


def test_argmax_first_decides_in_float32():
    # two values distinct in float64 but the same float32 are equals: the first wins
    a = 1.0 + 2.0 ** -30
    x = np.array([[0.0, 1.0, a, 0.5]])
    assert np.float32(a) == np.float32(1.0)
    assert argmax_first(x)[0] == 1
    # distinct in float32: the larger wins, wherever it sits
    x = np.array([[0.0, 1.0, 1.0 + 2.0 ** -20, 0.5]])
    assert argmax_first(x)[0] == 2
