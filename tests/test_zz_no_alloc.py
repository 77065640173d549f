"""dflash_attention_noalloc: the block's attention for callers that cannot
allocate device memory (another component capturing a CUDA graph, a framework
that owns every device byte through its own pool, a loop that must not block
in the allocator).  Its scratch is a fixed array inside the library, so it
must give the same result as the allocating entry point
(dflash_debug_attention), call after call, without leaking anything from one
call into the next.

This file is collected last on purpose: a run that stops at the first failure
has run every other test before it.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

REL_TOL = 1e-4  # the f32 tolerance of the parity tests


def _setup():
    import torch

    import block_speculative_drafting_gb300 as dfl
    wl = W.WORKLOADS["small_q4"]
    g = wl.geom
    model = dfl.Model(g, W.make_weights(g))
    ctx = [wl.ctx, 9, 0]
    seqs = []
    for i, n in enumerate(ctx):
        s = model.new_sequence(n + 4)
        model.ctx_append(s, 0, W.make_taps(g, n, call_id=60 + i))
        seqs.append(s)
    width = (g.heads + 2 * g.kv_heads) * g.head_dim
    rows = len(ctx) * g.block
    return torch, dfl, g, model, seqs, ctx, width, rows


def test_noalloc_attention_matches_allocating_entry_point_twice():
    torch, dfl, g, model, seqs, ctx, width, rows = _setup()
    layer = 1
    for call in range(2):  # two calls in a row with different inputs
        qkv = torch.from_numpy(W.normal(11, 200 + call, (rows, width))).cuda()
        y_ref = torch.empty((rows, g.heads * g.head_dim), dtype=torch.float32, device="cuda")
        y_na = torch.full_like(y_ref, float("nan"))
        model.attention(seqs, layer, ctx, qkv, y_ref)
        model.attention_noalloc(seqs, layer, ctx, qkv, y_na)
        torch.cuda.synchronize()
        ref, got = y_ref.cpu().numpy(), y_na.cpu().numpy()
        assert np.isfinite(got).all()
        assert np.max(np.abs(got - ref)) <= REL_TOL * np.max(np.abs(ref)), f"call {call}"
    for s in seqs:
        s.close()
    model.close()


def test_noalloc_attention_rejects_more_than_its_array_holds():
    torch, dfl, g, model, seqs, ctx, width, rows = _setup()
    many = [seqs[0]] * 257
    qkv = torch.zeros((257 * g.block, width), dtype=torch.float32, device="cuda")
    y = torch.zeros((257 * g.block, g.heads * g.head_dim), dtype=torch.float32, device="cuda")
    with pytest.raises(dfl.DFlashError) as e:
        model.attention_noalloc(many, 0, [ctx[0]] * 257, qkv, y)
    assert e.value.code == dfl._abi.DFLASH_ERANGE
    assert "at most 256" in str(e.value)
    for s in seqs:
        s.close()
    model.close()
