"""dflash_attention_noalloc: the block's attention for callers that cannot
allocate device memory when they run it (a host framework that owns every
device byte through its own pool allocator, a latency-critical loop that must
not block in the allocator or synchronise the device).  Its scratch is a
fixed array inside the library, so it must give the same result as the
allocating entry point (dflash_debug_attention), call after call, without
leaking anything from one call into the next -- in the cluster-merge plan
(short contexts: only the array's view area is used) and in the split plan
(a long context: the key splits' partial rows go through the array).

This file is collected last on purpose: a run that stops at the first failure
has run every other test before it.
"""
import math

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

REL_TOL = 1e-4  # the f32 tolerance of the parity tests


def _setup(ctx):
    import torch

    import block_speculative_drafting_gb300 as dfl
    wl = W.WORKLOADS["small_q4"]
    g = wl.geom
    w = W.make_weights(g)
    model = dfl.Model(g, w)
    seqs = []
    for i, n in enumerate(ctx):
        s = model.new_sequence(n + 4)
        model.ctx_append(s, 0, W.make_taps(g, n, call_id=60 + i))
        seqs.append(s)
    width = (g.heads + 2 * g.kv_heads) * g.head_dim
    rows = len(ctx) * g.block
    return torch, dfl, g, w, model, seqs, width, rows


def _two_calls(torch, g, model, seqs, ctx, width, rows, layer, seed):
    """Two calls in a row with different q/k/v: the no-alloc result against the
    allocating entry point's.  Returns the inputs and outputs of each call."""
    out = []
    for call in range(2):
        qkv = torch.from_numpy(W.normal(seed, 200 + call, (rows, width))).cuda()
        y_ref = torch.empty((rows, g.heads * g.head_dim), dtype=torch.float32, device="cuda")
        y_na = torch.full_like(y_ref, float("nan"))
        model.attention(seqs, layer, ctx, qkv, y_ref)
        model.attention_noalloc(seqs, layer, ctx, qkv, y_na)
        torch.cuda.synchronize()
        ref, got = y_ref.cpu().numpy(), y_na.cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}"
        assert np.max(np.abs(got - ref)) <= REL_TOL * np.max(np.abs(ref)), f"call {call}"
        out.append((qkv.cpu().numpy(), got))
    return out


def test_noalloc_attention_matches_allocating_entry_point_twice():
    ctx = [77, 9, 0]
    torch, dfl, g, w, model, seqs, width, rows = _setup(ctx)
    _two_calls(torch, g, model, seqs, ctx, width, rows, layer=1, seed=11)
    for s in seqs:
        s.close()
    model.close()


def test_noalloc_attention_split_plan_through_the_array():
    """A 20000-row context: the keys split over plain CTAs whose partial rows
    go through the fixed array and merge in a second kernel.  Compared with
    the allocating entry point and with the oracle's attention, twice; the
    call launches the view kernel and the two attention kernels."""
    from oracle import OracleModel, OracleSeq
    from oracle import attention as oattn
    n = 20000
    ctx = [n]
    torch, dfl, g, w, model, seqs, width, rows = _setup(ctx)
    om = OracleModel(g, w)
    osq = OracleSeq(om)
    osq.append(0, W.make_taps(g, n, call_id=60))
    layer = g.layers - 1
    before = model.launch_count()
    model.attention_noalloc(seqs, layer, ctx, torch.zeros((rows, width), device="cuda"),
                            torch.empty((rows, g.heads * g.head_dim), device="cuda"))
    torch.cuda.synchronize()
    assert model.launch_count() - before == 3  # views, split attention, merge
    B, nh, kv, hd = g.block, g.heads, g.kv_heads, g.head_dim
    for qkv, got in _two_calls(torch, g, model, seqs, ctx, width, rows, layer, seed=12):
        r = qkv.astype(np.float64)
        q = r[:, :nh * hd].reshape(B, nh, hd)
        kb = r[:, nh * hd:(nh + kv) * hd].reshape(B, kv, hd)
        vb = r[:, (nh + kv) * hd:].reshape(B, kv, hd)
        ref = oattn(q, kb, vb, osq.k[layer], osq.v[layer], g.rep, 1 / math.sqrt(hd))
        out = got.reshape(B, nh, hd)
        # the context's K/V are the library's own projection (its own decisions), so
        # the bar is the parity tests' bound for the quantised format's attention
        assert np.max(np.abs(out - ref)) <= 2e-3 * np.max(np.abs(ref))
    for s in seqs:
        s.close()
    model.close()


def test_noalloc_attention_rejects_more_than_its_array_holds():
    ctx = [77, 9, 0]
    torch, dfl, g, w, model, seqs, width, rows = _setup(ctx)
    many = [seqs[0]] * 257
    qkv = torch.zeros((257 * g.block, width), dtype=torch.float32, device="cuda")
    y = torch.zeros((257 * g.block, g.heads * g.head_dim), dtype=torch.float32, device="cuda")
    before = model.launch_count()
    with pytest.raises(dfl.DFlashError) as e:
        model.attention_noalloc(many, 0, [ctx[0]] * 257, qkv, y)
    assert e.value.code == dfl._abi.DFLASH_ERANGE
    assert "at most 256" in str(e.value)
    assert model.launch_count() == before  # nothing launched
    for s in seqs:
        s.close()
    model.close()
