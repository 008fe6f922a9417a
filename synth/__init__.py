"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Only input generation lives here (weights, token ids, lengths, KV contents):
no step of the transformer's arithmetic.  The generator is counter based
(``synth.h``), so the host fill (``synth_host.c``) and the device fill
(``synth_dev.cu``) give identical bits for the same (seed, stream, index).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_HOST_SO = os.path.join(_BUILD, "libsynth_host.so")
_DEV_SO = os.path.join(_BUILD, "libsynth_dev.so")
_host = None
_dev = None

U64 = ctypes.c_uint64


def _newer(target, sources):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(s) <= t for s in sources)


def _build_host():
    srcs = [os.path.join(_HERE, "synth_host.c"), os.path.join(_HERE, "synth.h")]
    if _newer(_HOST_SO, srcs):
        return
    os.makedirs(_BUILD, exist_ok=True)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-o", _HOST_SO, srcs[0]])


def _build_dev():
    srcs = [os.path.join(_HERE, "synth_dev.cu"), os.path.join(_HERE, "synth.h")]
    if _newer(_DEV_SO, srcs):
        return
    os.makedirs(_BUILD, exist_ok=True)
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                           "-Xcompiler", "-fPIC", "-shared", "-o", _DEV_SO, srcs[0]])


def build(device: bool = True) -> None:
    with ThreadPoolExecutor(2) as ex:
        futs = [ex.submit(_build_host)]
        if device:
            futs.append(ex.submit(_build_dev))
        for f in futs:
            f.result()


def host():
    global _host
    if _host is None:
        _build_host()
        lib = ctypes.CDLL(_HOST_SO)
        lib.syn_fill_normal_bf16.argtypes = [ctypes.c_void_p, U64, U64, U64, U64,
                                             ctypes.c_double, ctypes.c_double]
        lib.syn_fill_kv.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 6 + [U64, ctypes.c_double]
        lib.syn_fill_tokens.argtypes = [ctypes.c_void_p, U64, U64, U64, U64, ctypes.c_uint32]
        lib.syn_fill_uniform_int.argtypes = [ctypes.c_void_p, U64, U64, U64, ctypes.c_int32,
                                             ctypes.c_int32]
        lib.syn_fill_u64.argtypes = [ctypes.c_void_p, U64, U64, U64]
        _host = lib
    return _host


def dev():
    global _dev
    if _dev is None:
        _build_dev()
        lib = ctypes.CDLL(_DEV_SO)
        lib.syn_dev_fill_normal_bf16.argtypes = [ctypes.c_void_p, U64, U64, U64, U64,
                                                 ctypes.c_double, ctypes.c_double, ctypes.c_void_p]
        lib.syn_dev_fill_kv.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 6 + [
            U64, ctypes.c_double, ctypes.c_void_p]
        lib.syn_dev_fill_tokens.argtypes = [ctypes.c_void_p, U64, U64, U64, U64, ctypes.c_uint32,
                                            ctypes.c_void_p]
        _dev = lib
    return _dev


# ---- stream ids (mirror of the enum in synth.h) -------------------------------------------
EMBED, LM_HEAD, FINAL_NORM = 1, 2, 3
WQ, WK, WV, WO, WG, WU, WD, ATTN_NORM, FFN_NORM = range(16, 25)


def stream_weight(layer: int, kind: int) -> int:
    return kind if layer < 0 else ((layer + 1) << 8) | kind


def stream_tokens(row: int) -> int:
    return (2 << 48) | row


def stream_misc(what: int) -> int:
    return (3 << 48) | what


# ---- host (numpy) fills -----------------------------------------------------------------
def normal_bf16(n: int, seed: int, stream: int, first: int = 0, mean: float = 0.0,
                sigma: float = 0.02, out: np.ndarray | None = None) -> np.ndarray:
    """uint16 bf16 bit patterns of mean + sigma * N(0,1) draws."""
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    host().syn_fill_normal_bf16(out.ctypes.data, n, seed, stream, first, mean, sigma)
    return out


def kv(row: int, kv_sel: int, L: int, Hkv: int, n_tok: int, hd: int, seed: int,
       sigma: float) -> np.ndarray:
    """Synthetic K (kv_sel=0) or V (kv_sel=1) of one sequence, uint16 [L, Hkv, n_tok, hd]."""
    out = np.empty((L, Hkv, n_tok, hd), dtype=np.uint16)
    host().syn_fill_kv(out.ctypes.data, row, kv_sel, L, Hkv, n_tok, hd, seed, sigma)
    return out


def tokens(n: int, seed: int, stream: int, vocab: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    host().syn_fill_tokens(out.ctypes.data, n, seed, stream, first, vocab)
    return out


def uniform_ints(n: int, seed: int, stream: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    host().syn_fill_uniform_int(out.ctypes.data, n, seed, stream, lo, hi)
    return out


def words(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    host().syn_fill_u64(out.ctypes.data, n, seed, stream)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ---- device (torch) fills ---------------------------------------------------------------
def _check(rc):
    if rc != 0:
        raise RuntimeError(f"synthetic device fill failed: cudaError {rc}")


def dev_normal_bf16(ptr: int, n: int, seed: int, stream: int, first: int = 0, mean: float = 0.0,
                    sigma: float = 0.02, cuda_stream: int = 0) -> None:
    _check(dev().syn_dev_fill_normal_bf16(ptr, n, seed, stream, first, mean, sigma, cuda_stream))


def dev_kv(ptr: int, row: int, kv_sel: int, L: int, Hkv: int, n_tok: int, hd: int, seed: int,
           sigma: float, cuda_stream: int = 0) -> None:
    _check(dev().syn_dev_fill_kv(ptr, row, kv_sel, L, Hkv, n_tok, hd, seed, sigma, cuda_stream))


def dev_tokens(ptr: int, n: int, seed: int, stream: int, vocab: int, first: int = 0,
               cuda_stream: int = 0) -> None:
    _check(dev().syn_dev_fill_tokens(ptr, n, seed, stream, first, vocab, cuda_stream))
