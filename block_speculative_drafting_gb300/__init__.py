"""DFlash 2 block drafter on GB300 (sm_103a): Python binding of libdflash.so.

Argument marshalling only -- every step of the drafter runs in the library's
CUDA kernels; there is no Python or CPU fallback.  PyTorch provides device
memory and streams: device inputs and outputs are torch CUDA tensors, host
ones numpy arrays; calls run on torch's current stream unless given one.

    model = Model(geom, weights)          # weights: dict of float32 arrays
    seq = model.new_sequence(max_ctx_rows)
    model.ctx_append(seq, pos, taps)      # taps [n][n_taps*hidden] float32
    logits, tokens = model.block([seq], [anchor_tok], [anchor_pos], block_len)
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import _abi
from ._abi import QUANT_F32, QUANT_Q4G32, MAT_FC, MAT_HEAD, mat_layer  # noqa: F401

_lib = None

GEOM_FIELDS = ("hidden", "intermediate", "layers", "heads", "kv_heads", "head_dim", "vocab", "block", "n_taps")
LAYER_TENSORS = ("in_norm", "post_norm", "q_norm", "k_norm", "q", "k", "v", "o", "gate", "up", "down")
CONV_TENSORS = ("attn_conv_base", "attn_conv_proj", "mlp_conv_base", "mlp_conv_proj")  # with a row convolution


def lib():
    """The loaded library (raises ImportError when it is not built)."""
    global _lib
    if _lib is None:
        _lib = _abi.load()
    return _lib


class DFlashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_abi.CODES.get(code, code)}: {msg}")
        self.code = code


def _torch():
    import torch
    return torch


def _stream(stream):
    if stream is not None:
        return C.c_void_p(int(stream))
    torch = _torch()
    if torch.cuda.is_available():
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return C.c_void_p(0)


def _is_torch(x) -> bool:
    return type(x).__module__.startswith("torch")


def _ptr(x):
    """Data pointer of a numpy array or a torch tensor (None -> NULL)."""
    if x is None:
        return None
    if _is_torch(x):
        return x.data_ptr()
    return x.ctypes.data


def geometry_struct(g) -> _abi.Geometry:
    """Build the C geometry from any object with the geometry's attributes."""
    s = _abi.Geometry()
    for f in GEOM_FIELDS:
        setattr(s, f, int(getattr(g, f)))
    mask = getattr(g, "mask_token", None)
    s.mask_token = int(g.vocab - 1 if mask is None else mask)
    s.window = int(getattr(g, "window", 0))
    s.quant = int(getattr(g, "quant", 0))
    s.eps = float(getattr(g, "eps", 1e-6))
    s.rope_theta = float(getattr(g, "rope_theta", 1e6))
    s.selector_rank = int(getattr(g, "selector_rank", 0))
    s.selector_top = int(getattr(g, "selector_top", 0))
    s.conv_kernel = int(getattr(g, "conv_kernel", 0))
    s.conv_group = int(getattr(g, "conv_group", 0))
    # per-layer lists: arrays kept alive on the struct until dflash_init has copied them
    L = int(g.layers)
    wins = tuple(getattr(g, "windows", ()) or ())
    if wins:
        if len(wins) != L:
            raise ValueError(f"windows has {len(wins)} entries for {L} layers")
        s._windows = (C.c_int32 * L)(*[int(w) for w in wins])
        s.windows = C.cast(s._windows, C.POINTER(C.c_int32))
    nr = tuple(getattr(g, "no_rope", ()) or ())
    if nr:
        if any(not 0 <= int(l) < L for l in nr):
            raise ValueError(f"no_rope lists a layer outside [0, {L})")
        s._no_rope = (C.c_int32 * L)(*[1 if l in nr else 0 for l in range(L)])
        s.no_rope = C.cast(s._no_rope, C.POINTER(C.c_int32))
    return s


class Sequence:
    """One sequence's context (device K/V storage owned by the library)."""

    def __init__(self, model: "Model", max_ctx_rows: int):
        self.model = model
        h = C.c_void_p()
        model._check(lib().dflash_seq_new(model.handle, int(max_ctx_rows), C.byref(h)))
        self.handle = h
        self.max_ctx_rows = int(max_ctx_rows)

    def span(self):
        a, b = C.c_int64(), C.c_int64()
        self.model._check(lib().dflash_seq_span(self.handle, C.byref(a), C.byref(b)))
        return a.value, b.value

    def truncate(self, pos: int):
        self.model._check(lib().dflash_truncate(self.handle, int(pos)))

    def reset(self):
        self.model._check(lib().dflash_reset(self.handle))

    def close(self):
        if getattr(self, "handle", None):
            lib().dflash_seq_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Model:
    """A drafter's weights on the current CUDA device."""

    def __init__(self, geom, weights: dict, stream=None):
        self.geom = geom
        self.gs = geometry_struct(geom)
        L = self.gs.layers
        on_device = _is_torch(weights["fc"])
        if not on_device:
            weights = {**weights, "layers": [{k: np.ascontiguousarray(v, dtype=np.float32) for k, v in lw.items()}
                                             for lw in weights["layers"]]}
            for k in ("fc", "hidden_norm", "norm", "embed", "head", "selector_projection"):
                if k in weights:
                    weights[k] = np.ascontiguousarray(weights[k], dtype=np.float32)
            for k in ("predecessor_codebook", "successor_codebook"):
                if k in weights:
                    weights[k] = np.ascontiguousarray(weights[k], dtype=np.float16)
        self._keep = weights  # alive during init
        w = _abi.Weights()
        FP = C.POINTER(C.c_float)
        for k in ("fc", "hidden_norm", "norm", "embed", "head"):
            setattr(w, k, C.cast(C.c_void_p(_ptr(weights[k])), FP))
        if self.gs.selector_rank > 0:
            if "selector_projection" in weights:
                w.selector_projection = C.cast(C.c_void_p(_ptr(weights["selector_projection"])), FP)
            for k in ("predecessor_codebook", "successor_codebook"):
                if k in weights:
                    setattr(w, k, _ptr(weights[k]))
        arrays = []
        names = LAYER_TENSORS + (CONV_TENSORS if self.gs.conv_kernel > 0 else ())
        for name in names:
            if any(name not in lw for lw in weights["layers"]):
                continue  # left NULL: the library names what is missing
            arr = (FP * L)(*[C.cast(C.c_void_p(_ptr(weights["layers"][l][name])), FP) for l in range(L)])
            arrays.append(arr)
            setattr(w, name, C.cast(arr, C.POINTER(FP)))
        h = C.c_void_p()
        rc = lib().dflash_init(C.byref(self.gs), C.byref(w), 1 if on_device else 0, _stream(stream), C.byref(h))
        self._keep = None
        if rc != 0:
            raise DFlashError(rc, lib().dflash_last_error(None).decode())
        self.handle = h

    def _check(self, rc: int):
        if rc != 0:
            raise DFlashError(rc, lib().dflash_last_error(self.handle).decode())

    def close(self):
        if getattr(self, "handle", None):
            lib().dflash_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_sequence(self, max_ctx_rows: int) -> Sequence:
        return Sequence(self, max_ctx_rows)

    # ---------------------------------------------------------------- the path
    def ctx_append(self, seq: Sequence, pos: int, taps, stream=None):
        """Add rows of taps at positions pos.. (numpy: host, torch CUDA tensor: device)."""
        n = 0 if taps is None else int(taps.shape[0])
        on_dev = taps is not None and _is_torch(taps)
        if taps is not None and not on_dev:
            taps = np.ascontiguousarray(taps, dtype=np.float32)
        self._check(lib().dflash_ctx_append(self.handle, seq.handle, int(pos), _ptr(taps), n, 1 if on_dev else 0,
                                            _stream(stream)))

    def ctx_queue(self, seq: Sequence, pos: int, taps, stream=None):
        """ctx_append put off: the rows wait until a block (or settle) reads them."""
        n = 0 if taps is None else int(taps.shape[0])
        on_dev = taps is not None and _is_torch(taps)
        if taps is not None and not on_dev:
            taps = np.ascontiguousarray(taps, dtype=np.float32)
        self._check(lib().dflash_ctx_queue(self.handle, seq.handle, int(pos), _ptr(taps), n, 1 if on_dev else 0,
                                           _stream(stream)))

    def settle(self, seq: Sequence, stream=None):
        """Make every queued row of `seq` context."""
        self._check(lib().dflash_settle(self.handle, seq.handle, _stream(stream)))

    def block(self, seqs, anchor_tok, anchor_pos, block_len=None, logits=None, tokens=None, want_logits=True,
              stream=None):
        """One block per sequence.  Host mode (numpy or lists): returns
        (logits [n][block_len-1][vocab] float32 or None, tokens [n][block_len-1]
        uint32).  Device mode (anchor_tok a torch CUDA tensor): fills the given
        torch tensors `logits` / `tokens` and returns them."""
        n = len(seqs)
        bl = int(self.gs.block if block_len is None else block_len)
        handles = (C.c_void_p * n)(*[s.handle for s in seqs])
        pos = (C.c_int64 * n)(*[int(p) for p in anchor_pos])
        if _is_torch(anchor_tok):
            self._check(lib().dflash_block(self.handle, handles, n, _ptr(anchor_tok), pos, bl, _ptr(logits),
                                           _ptr(tokens), 1, _stream(stream)))
            return logits, tokens
        at = np.ascontiguousarray(np.asarray(anchor_tok, dtype=np.uint32))
        if logits is None and want_logits:
            logits = np.empty((n, bl - 1, self.gs.vocab), dtype=np.float32)
        if tokens is None:
            tokens = np.empty((n, bl - 1), dtype=np.uint32)
        self._check(lib().dflash_block(self.handle, handles, n, _ptr(at), pos, bl, _ptr(logits), _ptr(tokens), 0,
                                       _stream(stream)))
        return logits, tokens

    # ---------------------------------------------------------------- tracing
    def profile_start(self):
        self._check(lib().dflash_profile_start(self.handle))

    def profile_stop(self) -> dict:
        """{kernel name: (launches, total device ms, total algorithmic bytes)}."""
        self._check(lib().dflash_profile_stop(self.handle))
        out, i = {}, 0
        name, n, ms, by = C.c_char_p(), C.c_int64(), C.c_double(), C.c_double()
        while lib().dflash_profile_entry(self.handle, i, C.byref(name), C.byref(n), C.byref(ms), C.byref(by)) == 0:
            out[name.value.decode()] = (n.value, ms.value, by.value)
            i += 1
        return out

    def launch_count(self) -> int:
        return int(lib().dflash_launch_count(self.handle))

    def option(self, name: str, value: int):
        """Switch one of the model's kernel choices (test hook): "tc", "dense",
        "head_bound" (include/dflash.h, dflash_debug_option)."""
        self._check(lib().dflash_debug_option(self.handle, name.encode(), int(value)))

    # ---------------------------------------------------------------- test hooks
    def q4_codes(self, matrix_id: int, rows: int, cols: int, stream=None):
        codes = np.empty((rows, cols), dtype=np.int8)
        scales = np.empty((rows, cols // 32), dtype=np.uint16)
        self._check(lib().dflash_debug_q4_codes(self.handle, matrix_id, _ptr(codes), _ptr(scales), _stream(stream)))
        return codes, scales.view(np.float16)

    def head_codes(self, stream=None):
        codes = np.empty((self.gs.vocab, self.gs.hidden), dtype=np.int8)
        scales = np.empty(self.gs.vocab, dtype=np.float32)
        self._check(lib().dflash_debug_head_codes(self.handle, _ptr(codes), _ptr(scales), _stream(stream)))
        return codes, scales

    def q4_groupsums(self, matrix_id: int, x_codes, n_rows_out: int, stream=None):
        x = np.ascontiguousarray(x_codes, dtype=np.int8)
        out = np.empty((x.shape[0], n_rows_out, x.shape[1] // 32), dtype=np.int32)
        self._check(lib().dflash_debug_q4_groupsums(self.handle, matrix_id, _ptr(x), x.shape[0], _ptr(out),
                                                    _stream(stream)))
        return out

    def q4_matmul(self, matrix_id: int, x_codes, x_scales, n_rows_out: int, stream=None):
        """y[r][n] = xs[r] * sum_g s[n][g] sum_k q[n][k] x[r][k] by the library's kernels (the
        streaming kernel for up to 16 rows, the tensor-core kernel beyond)."""
        x = np.ascontiguousarray(x_codes, dtype=np.int8)
        xs = np.ascontiguousarray(x_scales, dtype=np.float32)
        out = np.empty((x.shape[0], n_rows_out), dtype=np.float32)
        self._check(lib().dflash_debug_q4_matmul(self.handle, matrix_id, _ptr(x), _ptr(xs), x.shape[0], _ptr(out),
                                                 _stream(stream)))
        return out

    def wait_expiry(self, limit_ns: int, stream=None):
        """Run the library's bounded wait on an mbarrier that nothing arrives on
        (raises DFlashError ECUDA when the wait gives up, as it must)."""
        self._check(lib().dflash_debug_wait_expiry(self.handle, int(limit_ns), _stream(stream)))

    def trace(self, enable: bool = True):
        self._check(lib().dflash_debug_trace(self.handle, 1 if enable else 0))

    def trace_force(self, codes, scales):
        codes = np.ascontiguousarray(codes, dtype=np.int8)
        scales = np.ascontiguousarray(scales, dtype=np.float32)
        self._check(lib().dflash_debug_trace_force(self.handle, codes.shape[0], codes.shape[1], _ptr(codes),
                                                   _ptr(scales)))

    def trace_sites(self):
        """[(values f32 [rows][cols], codes int8, scales f32)] in execution order."""
        out, i = [], 0
        r, c = C.c_int32(), C.c_int32()
        while lib().dflash_debug_trace_site(self.handle, i, C.byref(r), C.byref(c), None, None, None) == 0:
            v = np.empty((r.value, c.value), dtype=np.float32)
            q = np.empty((r.value, c.value), dtype=np.int8)
            s = np.empty(r.value, dtype=np.float32)
            lib().dflash_debug_trace_site(self.handle, i, None, None, _ptr(v), _ptr(q), _ptr(s))
            out.append((v, q, s))
            i += 1
        return out

    def read_kv(self, seq: Sequence, layer: int, pos: int, n: int, stream=None):
        k = np.empty((n, self.gs.kv_heads, self.gs.head_dim), dtype=np.float32)
        v = np.empty_like(k)
        self._check(lib().dflash_debug_read_kv(self.handle, seq.handle, layer, int(pos), int(n), _ptr(k), _ptr(v),
                                               _stream(stream)))
        return k, v

    def attention(self, seqs, layer: int, anchor_pos, qkv, y, stream=None):
        """The block's attention alone (torch CUDA tensors): qkv [rows][(heads+2kv)*hd]
        with q, k normed and rotated; writes y [rows][heads*hd]."""
        n = len(seqs)
        handles = (C.c_void_p * n)(*[s.handle for s in seqs])
        pos = (C.c_int64 * n)(*[int(p) for p in anchor_pos])
        bl = int(qkv.shape[0]) // n
        self._check(lib().dflash_debug_attention(self.handle, handles, n, int(layer), pos, bl, _ptr(qkv), _ptr(y),
                                                 _stream(stream)))
        return y

    def attention_noalloc(self, seqs, layer: int, anchor_pos, qkv, y, stream=None):
        """`attention` for callers that cannot allocate device memory: its
        scratch is a fixed array inside the library (see include/dflash.h,
        dflash_attention_noalloc); calls on one GPU must not overlap."""
        n = len(seqs)
        handles = (C.c_void_p * n)(*[s.handle for s in seqs])
        pos = (C.c_int64 * n)(*[int(p) for p in anchor_pos])
        bl = int(qkv.shape[0]) // n
        self._check(lib().dflash_attention_noalloc(self.handle, handles, n, int(layer), pos, bl, _ptr(qkv), _ptr(y),
                                                   _stream(stream)))
        return y

