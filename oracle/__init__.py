"""CPU oracle of the continuous-batching decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg and
reference arm of ``bench.py`` may import this package.  It shares no code with the CUDA path
(``continuous_batching_transformer_gb300``); the two meet only in the seeded
input generator ``synth``.

The arithmetic lives in ``cbt_oracle.c`` (plain C, double accumulation, no
fused multiply-add); this module builds it, lays the synthetic weights out in
the oracle's own format and marshals calls through ctypes.

What it computes follows the gnosis page "Continuous Decode Batching -- the
transformer capture" (sections on forward_batch_segmented and
decode_step_batch) and the mlx-bun batching design (greedy argmax, lowest id
on ties).  Pins: ``tests/test_oracle_pins.py`` -- every component (RMSNorm,
RoPE, attention, SwiGLU, the projections, the quantisers, argmax) against closed
forms, hand examples and library routines, and the whole model against an fp64
composition of library routines and the pages' invariants.  The pages print no
worked example with values, so the end-to-end logits of the full model are
parity unpinned beyond those pins and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

import synth
from synth.recipes import ModelShape

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libcbt_oracle.so")
_lib = None

c_int = ctypes.c_int
c_void = ctypes.c_void_p


def build() -> str:
    srcs = [os.path.join(_HERE, "cbt_oracle.c"), os.path.join(_HERE, "cbt_oracle.h")]
    if os.path.exists(_SO) and all(os.path.getmtime(s) <= os.path.getmtime(_SO) for s in srcs):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-o", tmp, srcs[0], "-lm"])
    os.replace(tmp, _SO)
    return _SO


class Config(ctypes.Structure):
    _fields_ = [("n_layers", c_int), ("d_model", c_int), ("n_heads", c_int),
                ("n_kv_heads", c_int), ("head_dim", c_int), ("d_ff", c_int), ("vocab", c_int),
                ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
                ("weight_format", c_int), ("group_size", c_int)]


class Linear(ctypes.Structure):
    _fields_ = [("w", c_void), ("packed", c_void), ("scales", c_void), ("biases", c_void)]


class Layer(ctypes.Structure):
    _fields_ = [("wq", Linear), ("wk", Linear), ("wv", Linear), ("wo", Linear), ("wg", Linear),
                ("wu", Linear), ("wd", Linear), ("attn_norm", c_void), ("ffn_norm", c_void)]


class Model(ctypes.Structure):
    _fields_ = [("cfg", Config), ("embed", c_void), ("lm_head", Linear), ("final_norm", c_void),
                ("layers", ctypes.POINTER(Layer))]


class KV(ctypes.Structure):
    _fields_ = [("capacity", c_int), ("len", c_int), ("k", c_void), ("v", c_void),
                ("kq", c_void), ("vq", c_void), ("ks", c_void), ("kb", c_void), ("vs", c_void),
                ("vb", c_void), ("qlen", c_int), ("bits", c_int)]


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.POINTER
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_rmsnorm.argtypes = [c_void, c_void, c_int, ctypes.c_double, c_void]
        L.orc_rope.argtypes = [c_void, c_int, c_int, ctypes.c_double]
        L.orc_attention.argtypes = [c_void, c_void, c_void, c_int, c_int, c_void]
        L.orc_silu.argtypes = [ctypes.c_double]
        L.orc_silu.restype = ctypes.c_double
        L.orc_linear_apply.argtypes = [P(Config), P(Linear), c_int, c_int, c_void, c_int, c_void]
        L.orc_argmax.argtypes = [c_void, c_int]
        L.orc_quantize_affine4.argtypes = [c_void, c_int, c_int, c_int, c_void, c_void, c_void]
        L.orc_dequantize_affine4.argtypes = [c_void, c_void, c_void, c_int, c_int, c_int, c_void]
        L.orc_quantize_kv8.argtypes = [c_void, c_int, c_int, c_void, c_void, c_void]
        L.orc_quantize_kv.argtypes = [c_void, c_int, c_int, c_int, c_void, c_void, c_void]
        L.orc_attention_kv8.argtypes = [c_void, c_void, c_void, c_void, c_void, c_void, c_void,
                                        c_int, c_int, c_void]
        L.orc_attention_kvq.argtypes = [c_void, c_void, c_void, c_void, c_void, c_void, c_void,
                                        c_int, c_int, c_int, c_void]
        L.orc_kv_convert.argtypes = [P(Config), P(KV)]
        L.orc_kvq_export_value.argtypes = [ctypes.c_uint16, ctypes.c_uint16, c_int]
        L.orc_kvq_export_value.restype = ctypes.c_uint16
        L.orc_forward.argtypes = [P(Model), P(KV), c_int, c_int, c_void, c_void, c_void, c_void,
                                  c_void]
        L.orc_decode_step_batch.argtypes = [P(Model), P(KV), c_int, c_void, c_void]
        L.orc_prefill_segmented.argtypes = [P(Model), P(KV), c_int, c_void, c_void, c_void]
        L.orc_prefill_sequence.argtypes = [P(Model), P(KV), c_int, c_void, c_void]
        L.orc_num_threads.restype = c_int
        L.orc_set_num_threads.argtypes = [c_int]
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags.c_contiguous
    return a.ctypes.data


# ---- building blocks ------------------------------------------------------------------
def rmsnorm(x: np.ndarray, gain_bf16: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    g = np.ascontiguousarray(gain_bf16, dtype=np.uint16)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_ptr(x), _ptr(g), x.size, eps, _ptr(out))
    return out


def rope(vec: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = np.array(vec, dtype=np.float32, copy=True)
    lib().orc_rope(_ptr(v), v.size, pos, theta)
    return v


def attention(q: np.ndarray, k_bf16: np.ndarray, v_bf16: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
    v = np.ascontiguousarray(v_bf16, dtype=np.uint16)
    out = np.empty(q.size, dtype=np.float32)
    lib().orc_attention(_ptr(q), _ptr(k), _ptr(v), k.shape[0], q.size, _ptr(out))
    return out


def silu(z: float) -> float:
    return lib().orc_silu(z)


def argmax(logits: np.ndarray) -> int:
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    return lib().orc_argmax(_ptr(lg), lg.size)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """The oracle's own fp32 -> bf16 rounding (round to nearest even), as bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32).ravel()
    L = lib()
    return np.array([L.orc_f32_to_bf16(float(t)) for t in f], dtype=np.uint16).reshape(np.shape(x))


def quantize_affine4(w_bf16: np.ndarray, group: int = 64):
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    rows, cols = w.shape
    packed = np.empty((rows, cols // 8), dtype=np.uint32)
    scales = np.empty((rows, cols // group), dtype=np.uint16)
    biases = np.empty((rows, cols // group), dtype=np.uint16)
    rc = lib().orc_quantize_affine4(_ptr(w), rows, cols, group, _ptr(packed), _ptr(scales),
                                    _ptr(biases))
    if rc != 0:
        raise ValueError("bad quantisation shape")
    return packed, scales, biases


def dequantize_affine4(packed, scales, biases, group: int = 64) -> np.ndarray:
    rows = packed.shape[0]
    cols = packed.shape[1] * 8
    out = np.empty((rows, cols), dtype=np.float64)
    lib().orc_dequantize_affine4(_ptr(packed), _ptr(scales), _ptr(biases), rows, cols, group,
                                 _ptr(out))
    return out


def quantize_kv(x_bf16: np.ndarray, bits: int):
    """Affine rows of 8 or 4 bits (groups of 64 along the last axis): codes (cols * bits / 8
    bytes a row; 4 bits: element 2i in the low nibble of byte i), bf16 scales, bf16 biases."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    codes = np.empty((rows, cols * bits // 8), dtype=np.uint8)
    scales = np.empty((rows, cols // 64), dtype=np.uint16)
    biases = np.empty((rows, cols // 64), dtype=np.uint16)
    if lib().orc_quantize_kv(_ptr(x), rows, cols, bits, _ptr(codes), _ptr(scales),
                             _ptr(biases)) != 0:
        raise ValueError("bad quantisation shape")
    return codes, scales, biases


def quantize_kv8(x_bf16: np.ndarray):
    """8-bit affine rows (groups of 64 along the last axis): codes, bf16 scales, bf16 biases."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    codes = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty((rows, cols // 64), dtype=np.uint16)
    biases = np.empty((rows, cols // 64), dtype=np.uint16)
    if lib().orc_quantize_kv8(_ptr(x), rows, cols, _ptr(codes), _ptr(scales), _ptr(biases)) != 0:
        raise ValueError("bad quantisation shape")
    return codes, scales, biases


def attention_kvq(q: np.ndarray, kq, vq, bits: int) -> np.ndarray:
    """Attention of one query over quantised K/V rows: kq and vq are (codes, scales, biases)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    parts = [np.ascontiguousarray(a) for a in (*kq, *vq)]
    out = np.empty(q.size, dtype=np.float32)
    lib().orc_attention_kvq(_ptr(q), *[_ptr(a) for a in parts], parts[1].shape[0], q.size, bits,
                            _ptr(out))
    return out


def attention_kv8(q: np.ndarray, k8, v8) -> np.ndarray:
    """Attention of one query over 8-bit K/V rows: k8 and v8 are (codes, scales, biases)."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    parts = [np.ascontiguousarray(a) for a in (*k8, *v8)]
    out = np.empty(q.size, dtype=np.float32)
    lib().orc_attention_kv8(_ptr(q), *[_ptr(a) for a in parts], parts[0].shape[0], q.size,
                            _ptr(out))
    return out


def kvq_export_values(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray,
                      bits: int) -> np.ndarray:
    """bf16 bits of quantised rows as an export gives them (scale * code + bias in double,
    rounded to fp32, then to bf16); codes [rows][cols * bits / 8], scales/biases
    [rows][cols / 64]."""
    rows, ng = scales.shape
    cols = ng * 64
    L = lib()
    out = np.empty((rows, cols), dtype=np.uint16)
    for r in range(rows):
        for i in range(cols):
            if bits == 8:
                q = int(codes[r, i])
            else:
                byte = int(codes[r, i // 2])
                q = (byte >> 4) if (i & 1) else (byte & 0xF)
            out[r, i] = L.orc_kvq_export_value(int(scales[r, i // 64]), int(biases[r, i // 64]), q)
    return out


# ---- the model ----------------------------------------------------------------------
class LinearW:
    """One projection in the oracle's format: bf16 [out, in], or 4-bit affine triple."""

    def __init__(self, w_bf16: np.ndarray, fmt: str, group: int):
        self.out_dim, self.in_dim = w_bf16.shape
        if fmt == "bf16":
            self.w, self.packed, self.scales, self.biases = w_bf16, None, None, None
        else:
            self.w = None
            self.packed, self.scales, self.biases = quantize_affine4(w_bf16, group)

    def struct(self) -> Linear:
        return Linear(_ptr(self.w), _ptr(self.packed), _ptr(self.scales), _ptr(self.biases))


def project(lin: LinearW, x: np.ndarray, group: int = 64) -> np.ndarray:
    """y = x W^T for one stand-alone projection (bf16 or 4-bit affine, as `lin` holds it)."""
    fmt = 0 if lin.w is not None else 1
    cfg = Config(1, lin.in_dim, 1, 1, 2, 1, lin.out_dim, 0.0, 1.0, fmt, group)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, lin.in_dim)
    y = np.empty((x.shape[0], lin.out_dim), dtype=np.float32)
    st = lin.struct()
    lib().orc_linear_apply(ctypes.byref(cfg), ctypes.byref(st), lin.out_dim, lin.in_dim, _ptr(x),
                           x.shape[0], _ptr(y))
    return y


class OracleModel:
    """Synthetic weights of a ModelShape, drawn from ``synth`` in the oracle's own layout
    (separate Wq, Wk, Wv, Wg, Wu matrices, each [out, in])."""

    def __init__(self, shape: ModelShape):
        self.shape = s = shape
        fmt, G = s.weight_format, s.group_size
        seed, sig = s.weight_seed, s.weight_sigma

        def mat(layer, kind, rows, cols):
            w = synth.normal_bf16(rows * cols, seed, synth.stream_weight(layer, kind), sigma=sig)
            return LinearW(w.reshape(rows, cols), fmt, G)

        def gain(layer, kind):
            return synth.normal_bf16(s.d_model, seed, synth.stream_weight(layer, kind),
                                     mean=1.0, sigma=s.gain_sigma)

        d, qd, kvd, F = s.d_model, s.q_dim, s.kv_dim, s.d_ff
        self.embed = synth.normal_bf16(s.vocab * d, seed, synth.stream_weight(-1, synth.EMBED),
                                       sigma=sig).reshape(s.vocab, d)
        self.lm_head = mat(-1, synth.LM_HEAD, s.vocab, d)
        self.final_norm = gain(-1, synth.FINAL_NORM)
        self.layers = []
        for l in range(s.n_layers):
            self.layers.append(dict(
                wq=mat(l, synth.WQ, qd, d), wk=mat(l, synth.WK, kvd, d), wv=mat(l, synth.WV, kvd, d),
                wo=mat(l, synth.WO, d, qd), wg=mat(l, synth.WG, F, d), wu=mat(l, synth.WU, F, d),
                wd=mat(l, synth.WD, d, F), attn_norm=gain(l, synth.ATTN_NORM),
                ffn_norm=gain(l, synth.FFN_NORM)))
        self._build_struct()

    def _build_struct(self):
        s = self.shape
        self.cfg = Config(s.n_layers, s.d_model, s.n_heads, s.n_kv_heads, s.head_dim, s.d_ff,
                          s.vocab, s.rms_eps, s.rope_theta, 0 if s.weight_format == "bf16" else 1,
                          s.group_size)
        arr = (Layer * s.n_layers)()
        for l, L in enumerate(self.layers):
            arr[l] = Layer(L["wq"].struct(), L["wk"].struct(), L["wv"].struct(), L["wo"].struct(),
                           L["wg"].struct(), L["wu"].struct(), L["wd"].struct(),
                           _ptr(L["attn_norm"]), _ptr(L["ffn_norm"]))
        self._layers_arr = arr
        self.model = Model(self.cfg, _ptr(self.embed), self.lm_head.struct(), _ptr(self.final_norm),
                           ctypes.cast(arr, ctypes.POINTER(Layer)))

    def linear(self, lin: LinearW, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, lin.in_dim)
        y = np.empty((x.shape[0], lin.out_dim), dtype=np.float32)
        st = lin.struct()
        lib().orc_linear_apply(ctypes.byref(self.cfg), ctypes.byref(st), lin.out_dim, lin.in_dim,
                               _ptr(x), x.shape[0], _ptr(y))
        return y


class KVCache:
    """One sequence's cache, bf16 bits [n_layers, n_kv_heads, capacity, head_dim] for K and V;
    with kv_bits = 8 or 4 also their affine codes (groups of 64 along head_dim; head_dim *
    kv_bits / 8 bytes a position) and bf16 scales/biases, which attention reads once the
    cache's first call has converted it."""

    def __init__(self, shape: ModelShape, capacity: int, kv_bits: int = 16):
        if kv_bits not in (4, 8, 16):
            raise ValueError("kv_bits is 16 (bf16), 8 or 4 (affine)")
        self.shape = shape
        dims = (shape.n_layers, shape.n_kv_heads, capacity, shape.head_dim)
        self.k = np.zeros(dims, dtype=np.uint16)
        self.v = np.zeros(dims, dtype=np.uint16)
        self.capacity = capacity
        self.len = 0
        self.kv_bits = kv_bits
        self.qlen = 0
        self.q8 = None
        if kv_bits in (4, 8):
            gdims = dims[:-1] + (shape.head_dim // 64,)
            cdims = dims[:-1] + (shape.head_dim * kv_bits // 8,)
            self.q8 = {"kq": np.zeros(cdims, np.uint8), "vq": np.zeros(cdims, np.uint8),
                       "ks": np.zeros(gdims, np.uint16), "kb": np.zeros(gdims, np.uint16),
                       "vs": np.zeros(gdims, np.uint16), "vb": np.zeros(gdims, np.uint16)}

    def struct(self) -> KV:
        q = self.q8 or {}
        return KV(self.capacity, self.len, _ptr(self.k), _ptr(self.v),
                  *[_ptr(q.get(n)) for n in ("kq", "vq", "ks", "kb", "vs", "vb")], self.qlen,
                  self.kv_bits if self.q8 else 0)

    def convert(self) -> None:
        """Quantise positions [qlen, len) (a quantised cache filled with bf16 K/V directly)."""
        st = self.struct()
        s = self.shape
        m = Config(s.n_layers, s.d_model, s.n_heads, s.n_kv_heads, s.head_dim, s.d_ff, s.vocab,
                   s.rms_eps, s.rope_theta, 0, s.group_size)
        if lib().orc_kv_convert(ctypes.byref(m), ctypes.byref(st)) != 0:
            raise ValueError("not a quantised cache")
        self.qlen = st.qlen

    def fill_synthetic(self, row: int, n_tok: int, seed: int) -> None:
        """Positions [0, n_tok) from the seeded KV draws of synthetic row `row`."""
        s = self.shape
        assert n_tok <= self.capacity
        for kv_sel, dst in ((0, self.k), (1, self.v)):
            src = synth.kv(row, kv_sel, s.n_layers, s.n_kv_heads, n_tok, s.head_dim, seed,
                           s.kv_sigma)
            dst[:, :, :n_tok, :] = src
        self.len = n_tok
        if self.kv_bits in (4, 8):
            self.qlen = 0
            self.convert()


def _kv_array(caches):
    arr = (KV * max(1, len(caches)))()
    for i, c in enumerate(caches):
        arr[i] = c.struct()
    return arr


def _sync_back(arr, caches):
    for i, c in enumerate(caches):
        c.len = arr[i].len
        c.qlen = arr[i].qlen


def forward(m: OracleModel, caches, seq, pos, tok, want) -> np.ndarray:
    n = len(tok)
    seq = np.ascontiguousarray(seq, dtype=np.int32)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    want = np.ascontiguousarray(want, dtype=np.int32)
    logits = np.empty((int(want.sum()), m.shape.vocab), dtype=np.float32)
    arr = _kv_array(caches)
    rc = lib().orc_forward(ctypes.byref(m.model), arr, len(caches), n, _ptr(seq), _ptr(pos),
                           _ptr(tok), _ptr(want), _ptr(logits) if logits.size else None)
    if rc != 0:
        raise ValueError("oracle rejected the token list")
    _sync_back(arr, caches)
    return logits


def decode_step_batch(m: OracleModel, caches, last_tokens) -> np.ndarray:
    B = len(caches)
    toks = np.ascontiguousarray(last_tokens, dtype=np.int32)
    logits = np.empty((B, m.shape.vocab), dtype=np.float32)
    arr = _kv_array(caches)
    rc = lib().orc_decode_step_batch(ctypes.byref(m.model), arr, B, _ptr(toks), _ptr(logits))
    if rc != 0:
        raise ValueError("oracle rejected the decode step")
    _sync_back(arr, caches)
    return logits


def prefill_segmented(m: OracleModel, caches, seg_lens, tokens) -> np.ndarray:
    K = len(caches)
    lens = np.ascontiguousarray(seg_lens, dtype=np.int32)
    toks = np.ascontiguousarray(tokens, dtype=np.int32)
    logits = np.empty((K, m.shape.vocab), dtype=np.float32)
    arr = _kv_array(caches)
    rc = lib().orc_prefill_segmented(ctypes.byref(m.model), arr, K, _ptr(lens), _ptr(toks),
                                     _ptr(logits))
    if rc != 0:
        raise ValueError("oracle rejected the segmented prefill")
    _sync_back(arr, caches)
    return logits


def prefill_continue(m: OracleModel, caches, seg_lens, tokens) -> np.ndarray:
    """Segmented prefill where segment s continues cache s at its current length (a prompt
    admitted in chunks: the mlx-bun batching design, section 4.2 "Joiner prefill", one chunk
    per scheduler iteration).  Token j of segment s sits at position caches[s].len + j and
    attends to [0, that position] of its own cache; returns each segment's last logits.  With
    empty caches this is prefill_segmented."""
    lens = [int(n) for n in seg_lens]
    if any(n <= 0 for n in lens) or sum(lens) != len(tokens):
        raise ValueError("segment lengths do not cover the tokens")
    seq = np.repeat(np.arange(len(lens), dtype=np.int32), lens)
    pos = np.concatenate([np.arange(c.len, c.len + n, dtype=np.int32) for c, n in zip(caches, lens)])
    want = np.zeros(len(tokens), dtype=np.int32)
    want[np.cumsum(lens) - 1] = 1
    return forward(m, caches, seq, pos, tokens, want)


def prefill_sequence(m: OracleModel, cache: KVCache, tokens) -> np.ndarray:
    toks = np.ascontiguousarray(tokens, dtype=np.int32)
    logits = np.empty(m.shape.vocab, dtype=np.float32)
    arr = _kv_array([cache])
    rc = lib().orc_prefill_sequence(ctypes.byref(m.model), arr, len(toks), _ptr(toks),
                                    _ptr(logits))
    if rc != 0:
        raise ValueError("oracle rejected the prefill")
    _sync_back(arr, [cache])
    return logits


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(n)
