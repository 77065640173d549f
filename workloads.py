"""Seeded synthetic workloads for the DFlash 2 block drafter.

This module holds only geometry records and seeded random draws: no step of
the drafter's arithmetic lives here.  It is the one module shared by the CPU
oracle (``oracle/``) and the CUDA path's tests and benchmark, so that both
sides see the same input values.

Recipe (all draws float32, all seeded, no dataset):

* every weight matrix and the embedding: N(0, 0.02);
* every norm gain (hidden_norm, norm, in_norm, post_norm, q_norm, k_norm):
  1 + N(0, 0.02), so the gain multiply is exercised;
* a row convolution's base kernels (when the geometry has one): N(0, 0.02),
  plus 1 at row offset 0; its kernel projections N(0, 0.02);
* the candidate selector (when the geometry has one): its projection
  N(0, 0.02), its two codebooks N(0, 1) stored as float16;
* context taps: N(0, 1);
* anchor tokens: uniform over the vocabulary.

Each tensor has its own stream ``default_rng([seed, tensor_id, chunk])``;
tensors are cut into fixed chunks of ``CHUNK`` values so that large tensors
can be filled by several threads while the values stay independent of the
thread count.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 22

WEIGHT_SEED = 0
TAPS_SEED = 1
ANCHOR_SEED = 2

# tensor ids of the model-wide tensors; layer l's tensors are
# LAYER_BASE + LAYER_STRIDE * l + (offset in LAYER_TENSORS)
TID_FC, TID_HIDDEN_NORM, TID_NORM, TID_EMBED, TID_HEAD = 0, 1, 2, 3, 4
TID_SELECTOR, TID_BOOK_P, TID_BOOK_C = 5, 6, 7
LAYER_BASE, LAYER_STRIDE = 16, 16
LAYER_TENSORS = ("in_norm", "post_norm", "q_norm", "k_norm", "q", "k", "v", "o", "gate", "up", "down",
                 "attn_conv_base", "attn_conv_proj", "mlp_conv_base", "mlp_conv_proj")
CONV_TENSORS = LAYER_TENSORS[11:]  # drawn only for a geometry with a row convolution
GAINS = {"in_norm", "post_norm", "q_norm", "k_norm", "hidden_norm", "norm"}


@dataclasses.dataclass(frozen=True)
class Geometry:
    """The drafter's hyper-parameters (the fields a DFlash 2 checkpoint fixes,
    minus the convolution and selector ones that this path does not use)."""

    hidden: int
    intermediate: int
    layers: int
    heads: int
    kv_heads: int
    head_dim: int
    vocab: int
    block: int
    n_taps: int
    eps: float = 1e-6
    rope_theta: float = 1e6
    quant: int = 0  # 0: all f32; 1: 4-bit g32 matrices, int8 head, int8 activations
    mask_token: int | None = None  # None: vocab - 1
    window: int = 0  # positions a block row sees back; 0 = all
    selector_rank: int = 0  # the candidate selector's rank; 0: none (each row's own top token)
    selector_top: int = 0  # candidates a row's selector re-scores
    conv_kernel: int = 0  # rows of the DFlash 2 row convolution; 0: none (the sub-layers unwrapped)
    conv_group: int = 0  # hidden columns that share one dynamic kernel value
    windows: tuple = ()  # the same per layer where layers differ (0: all); empty: `window` for every layer
    no_rope: tuple = ()  # layers whose queries and keys carry no rotary position

    def window_of(self, layer: int) -> int:
        return self.windows[layer] if self.windows else self.window

    def rotary(self, layer: int) -> bool:
        return layer not in self.no_rope

    @property
    def mask(self) -> int:
        return self.vocab - 1 if self.mask_token is None else self.mask_token

    @property
    def tap_width(self) -> int:
        return self.n_taps * self.hidden

    @property
    def rep(self) -> int:
        return self.heads // self.kv_heads


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    geom: Geometry
    ctx: int  # context rows per sequence before the block
    n_seqs: int = 1
    prefill: int = 0  # rows pushed in one append (the prefill workload)


QWEN3_8B_DRAFT = dict(hidden=4096, intermediate=12288, layers=5, heads=32, kv_heads=8, head_dim=128,
                      vocab=151936, block=16, n_taps=5, eps=1e-6, rope_theta=1e6, quant=1)

WORKLOADS = {
    # tiny all-f32 drafter
    "tiny_f32": Workload("tiny_f32", Geometry(hidden=256, intermediate=768, layers=2, heads=4, kv_heads=2,
                                              head_dim=64, vocab=4096, block=8, n_taps=2), ctx=64),
    # Qwen3-8B-shaped single-sequence decode block, context 2048
    "qwen3_8b_ctx2048": Workload("qwen3_8b_ctx2048", Geometry(**QWEN3_8B_DRAFT), ctx=2048),
    # the same at long context
    "qwen3_8b_ctx32768": Workload("qwen3_8b_ctx32768", Geometry(**QWEN3_8B_DRAFT), ctx=32768),
    # 32 independent sequences, context 4096 each
    "qwen3_8b_batch32_ctx4096": Workload("qwen3_8b_batch32_ctx4096", Geometry(**QWEN3_8B_DRAFT), ctx=4096, n_seqs=32),
    # the single-sequence block with the DFlash 2 pieces no config fixes: a
    # row convolution around every sub-layer (4 rows, 32 groups of 128
    # columns) and the candidate selector (rank 64, 8 candidates) -- sizes of
    # this build's choosing
    "qwen3_8b_ctx2048_dflash2": Workload("qwen3_8b_ctx2048_dflash2",
                                         Geometry(**QWEN3_8B_DRAFT, conv_kernel=4, conv_group=128, selector_rank=64,
                                                  selector_top=8), ctx=2048),
    # one append of 8192 target rows
    "qwen3_8b_prefill8192": Workload("qwen3_8b_prefill8192", Geometry(**QWEN3_8B_DRAFT), ctx=0, prefill=8192),
    # the same kernels on 1024 rows: the small case for profiler captures
    "qwen3_8b_prefill1024": Workload("qwen3_8b_prefill1024", Geometry(**QWEN3_8B_DRAFT), ctx=0, prefill=1024),
    # the batched block's matmul and head shapes (32 blocks of 16 rows) with one
    # layer and a 64-row context: a few GB on the device, for profiler captures
    "qwen3_8b_l1_batch32_ctx64": Workload("qwen3_8b_l1_batch32_ctx64", Geometry(**dict(QWEN3_8B_DRAFT, layers=1)),
                                          ctx=64, n_seqs=32),
    # the 1024-row prefill's FC (the same matrix at any layer count) with one
    # layer: a few GB on the device, for profiler captures
    "qwen3_8b_l1_prefill1024": Workload("qwen3_8b_l1_prefill1024", Geometry(**dict(QWEN3_8B_DRAFT, layers=1)),
                                        ctx=0, prefill=1024),
    # small quantised shapes the oracle finishes in seconds: several tiles and
    # ragged tails (vocab and context not multiples of any tile)
    "small_q4": Workload("small_q4", Geometry(hidden=512, intermediate=1536, layers=2, heads=8, kv_heads=2,
                                              head_dim=128, vocab=5003, block=16, n_taps=3, quant=1), ctx=77),
    "small_q4_hd64": Workload("small_q4_hd64", Geometry(hidden=384, intermediate=1024, layers=2, heads=6, kv_heads=3,
                                                       head_dim=64, vocab=3001, block=8, n_taps=2, quant=1), ctx=45),
}


def layer_tid(layer: int, name: str) -> int:
    return LAYER_BASE + LAYER_STRIDE * layer + LAYER_TENSORS.index(name)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal(seed: int, tensor_id: int, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """float32 N(mean, std) of `shape` from the streams (seed, tensor_id, chunk)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    std32, mean32 = np.float32(std), np.float32(mean)

    def fill(c: int) -> None:
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        part = out[lo:hi]
        np.random.default_rng([seed, tensor_id, c]).standard_normal(hi - lo, dtype=np.float32, out=part)
        if std32 != 1:
            part *= std32
        if mean32 != 0:
            part += mean32

    chunks = (n + CHUNK - 1) // CHUNK
    if chunks <= 1:
        for c in range(chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(chunks)))
    return out.reshape(shape)


def weight_shapes(g: Geometry) -> dict:
    hs, ffn, qd, kd = g.hidden, g.intermediate, g.heads * g.head_dim, g.kv_heads * g.head_dim
    shapes = {
        "in_norm": (hs,), "post_norm": (hs,), "q_norm": (g.head_dim,), "k_norm": (g.head_dim,),
        "q": (qd, hs), "k": (kd, hs), "v": (kd, hs), "o": (hs, qd),
        "gate": (ffn, hs), "up": (ffn, hs), "down": (hs, ffn),
    }
    if g.conv_kernel:
        kn, groups = g.conv_kernel, hs // g.conv_group
        for c in ("attn_conv", "mlp_conv"):
            shapes[c + "_base"] = (2, kn, hs)  # [stage][row offset][column]
            shapes[c + "_proj"] = (2 * kn * groups, hs)  # the dynamic kernels [stage][offset][group] of a row
    return shapes


def make_weights(g: Geometry, seed: int = WEIGHT_SEED, std: float = 0.02) -> dict:
    """All weights of a drafter as float32 host arrays, row-major [out][in].

    Returns {"fc", "hidden_norm", "norm", "embed", "head", "layers": [dict]}.
    """
    hs = g.hidden

    def draw(tid, name, shape):
        if name in GAINS:
            return normal(seed, tid, shape, std=std, mean=1.0)
        return normal(seed, tid, shape, std=std)

    w = {
        "fc": draw(TID_FC, "fc", (hs, g.tap_width)),
        "hidden_norm": draw(TID_HIDDEN_NORM, "hidden_norm", (hs,)),
        "norm": draw(TID_NORM, "norm", (hs,)),
        "embed": draw(TID_EMBED, "embed", (g.vocab, hs)),
        "head": draw(TID_HEAD, "head", (g.vocab, hs)),
    }
    if g.selector_rank:
        w["selector_projection"] = draw(TID_SELECTOR, "selector_projection", (g.selector_rank, hs))
        # the codebooks as the page stores them: f16 [vocab][rank], N(0, 1)
        for tid, name in ((TID_BOOK_P, "predecessor_codebook"), (TID_BOOK_C, "successor_codebook")):
            w[name] = normal(seed, tid, (g.vocab, g.selector_rank)).astype(np.float16)
    shapes = weight_shapes(g)
    w["layers"] = [{name: draw(layer_tid(l, name), name, shapes[name]) for name in LAYER_TENSORS if name in shapes}
                   for l in range(g.layers)]
    for lw in w["layers"]:
        # a convolution's base kernel: 1 + N(0, 0.02) at row offset 0, N(0, 0.02) further back
        for c in ("attn_conv_base", "mlp_conv_base"):
            if c in lw:
                lw[c][:, 0, :] += np.float32(1.0)
    return w


def make_taps(g: Geometry, n_rows: int, call_id: int = 0, seed: int = TAPS_SEED) -> np.ndarray:
    """`n_rows` context rows of joined tapped-layer outputs, float32 [n_rows][n_taps*hidden]."""
    return normal(seed, call_id, (n_rows, g.tap_width))


def make_anchors(g: Geometry, n: int, call_id: int = 0, seed: int = ANCHOR_SEED) -> np.ndarray:
    """`n` anchor tokens drawn uniformly over the vocabulary (uint32)."""
    return np.random.default_rng([seed, call_id]).integers(0, g.vocab, size=n, dtype=np.uint32)
