"""Thin ctypes binding of libcbt.so: the C ABI of include/cbt.h under the same names.

Argument marshalling only -- every step of the decode path runs in the library's CUDA
kernels.  Device buffers are passed as raw pointers (``tensor.data_ptr()``); PyTorch only
provides device memory and streams.  If the library has not been built, ``lib()`` raises:
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

c_int32 = ctypes.c_int32
c_void = ctypes.c_void_p
P = ctypes.POINTER

OK = 0
STATUS = {0: "CBT_OK", -1: "CBT_ERR_INVALID", -2: "CBT_ERR_NULL", -3: "CBT_ERR_BAD_SLAB",
          -4: "CBT_ERR_DUP_SLAB", -5: "CBT_ERR_BATCH", -6: "CBT_ERR_CAPACITY",
          -7: "CBT_ERR_POOL_EXHAUSTED", -8: "CBT_ERR_TOKENS", -9: "CBT_ERR_CUDA",
          -10: "CBT_ERR_DEVICE", -11: "CBT_ERR_UNSUPPORTED", -12: "CBT_ERR_LIMIT"}
NOALLOC_MAX_ROWS = 32
NOALLOC_SCRATCH_BYTES = 20 << 20
WEIGHTS_BF16, WEIGHTS_AFFINE4 = 0, 1
DEV_OK, DEV_TOKEN_RANGE = 0, 1

# every entry point include/cbt.h declares
EXPORTS = ["cbt_status_str", "cbt_engine_create", "cbt_engine_destroy", "cbt_slab_bytes",
           "cbt_kv_slab_alloc", "cbt_kv_slab_free", "cbt_retire", "cbt_kv_slab_position",
           "cbt_kv_slab_import", "cbt_kv_slab_export", "cbt_prefill_segmented",
           "cbt_decode_step_batch", "cbt_last_device_error", "cbt_engine_stats",
           "cbt_kernel_launches", "cbt_quantize_affine4", "cbt_engine_set_timing",
           "cbt_engine_timing", "cbt_greedy_head_noalloc", "cbt_kv_slab_copy_prefix",
           "cbt_kv_slab_share_prefix", "cbt_slab_bytes_kv8", "cbt_quantize_kv8",
           "cbt_slab_bytes_kvq", "cbt_quantize_kv", "cbt_engine_set_stamps", "cbt_engine_stamps",
           "cbt_engine_test_stall"]
KCLASS_PROJ, KCLASS_ATTN, KCLASS_OTHER = 0, 1, 2


class CbtError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class ModelConfig(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("d_model", c_int32), ("n_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32), ("d_ff", c_int32),
                ("vocab", c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_double),
                ("weight_format", c_int32), ("group_size", c_int32)]


class Linear(ctypes.Structure):
    _fields_ = [("w", c_void), ("scales", c_void), ("biases", c_void)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("wqkv", Linear), ("wo", Linear), ("wgu", Linear), ("wd", Linear),
                ("attn_norm", c_void), ("ffn_norm", c_void)]


class Weights(ctypes.Structure):
    _fields_ = [("embed", c_void), ("lm_head", Linear), ("final_norm", c_void),
                ("layers", P(LayerWeights))]


class EngineParams(ctypes.Structure):
    _fields_ = [("kv_arena", c_void), ("kv_arena_bytes", ctypes.c_size_t),
                ("max_batch", c_int32), ("max_prefill_tokens", c_int32), ("stream", c_void),
                ("kv_page_tokens", c_int32), ("kv_bits", c_int32)]


class Stats(ctypes.Structure):
    _fields_ = [("live_slabs", c_int32), ("max_batch", c_int32),
                ("slab_bytes_in_use", ctypes.c_int64), ("arena_bytes", ctypes.c_int64),
                ("largest_free_bytes", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64),
                ("decode_steps", ctypes.c_int64), ("prefill_tokens", ctypes.c_int64)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded libcbt.so.  Raises if it has not been built (no fallback path exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libcbt.so is not built: call __graft_entry__.build() "
                               "(or continuous_batching_transformer_gb300._build.build())")
        L = ctypes.CDLL(_build.LIB)
        L.cbt_status_str.argtypes = [c_int32]
        L.cbt_status_str.restype = ctypes.c_char_p
        L.cbt_engine_create.argtypes = [P(ModelConfig), P(Weights), P(EngineParams), P(c_void)]
        L.cbt_engine_destroy.argtypes = [c_void]
        L.cbt_slab_bytes.argtypes = [P(ModelConfig), c_int32]
        L.cbt_slab_bytes.restype = ctypes.c_size_t
        L.cbt_slab_bytes_kv8.argtypes = [P(ModelConfig), c_int32]
        L.cbt_slab_bytes_kv8.restype = ctypes.c_size_t
        L.cbt_quantize_kv8.argtypes = [c_void, c_int32, c_int32, c_void, c_void, c_void, c_void]
        L.cbt_slab_bytes_kvq.argtypes = [P(ModelConfig), c_int32, c_int32]
        L.cbt_slab_bytes_kvq.restype = ctypes.c_size_t
        L.cbt_quantize_kv.argtypes = [c_void, c_int32, c_int32, c_int32, c_void, c_void, c_void,
                                      c_void]
        L.cbt_kv_slab_alloc.argtypes = [c_void, c_int32, P(c_int32)]
        L.cbt_kv_slab_free.argtypes = [c_void, c_int32]
        L.cbt_retire.argtypes = [c_void, c_void, c_int32]
        L.cbt_kv_slab_position.argtypes = [c_void, c_int32, P(c_int32)]
        L.cbt_kv_slab_import.argtypes = [c_void, c_int32, c_void, c_void, c_int32, c_int32]
        L.cbt_kv_slab_export.argtypes = [c_void, c_int32, c_void, c_void, c_int32, c_int32]
        L.cbt_kv_slab_copy_prefix.argtypes = [c_void, c_int32, c_int32, c_int32]
        L.cbt_kv_slab_share_prefix.argtypes = [c_void, c_int32, c_int32, c_int32]
        L.cbt_prefill_segmented.argtypes = [c_void, c_void, c_void, c_int32, c_void, c_void,
                                            c_void]
        L.cbt_decode_step_batch.argtypes = [c_void, c_void, c_int32, c_void, c_void, c_void]
        L.cbt_last_device_error.argtypes = [c_void, P(c_int32), P(c_int32)]
        L.cbt_engine_stats.argtypes = [c_void, P(Stats)]
        L.cbt_kernel_launches.argtypes = [c_void]
        L.cbt_kernel_launches.restype = ctypes.c_int64
        L.cbt_quantize_affine4.argtypes = [c_void, c_int32, c_int32, c_int32, c_void, c_void,
                                           c_void, c_void]
        L.cbt_greedy_head_noalloc.argtypes = [P(ModelConfig), c_void, c_int32, c_void, P(Linear),
                                              c_void, c_void, c_void]
        L.cbt_engine_set_timing.argtypes = [c_void, c_int32]
        L.cbt_engine_set_stamps.argtypes = [c_void, c_int32]
        L.cbt_engine_test_stall.argtypes = [c_void, c_int32]
        L.cbt_engine_stamps.argtypes = [c_void, c_int32, P(c_int32), c_void, c_void]
        L.cbt_engine_timing.argtypes = [c_void, c_int32, P(ctypes.c_double), P(ctypes.c_int64),
                                        P(ctypes.c_double)]
        for name in EXPORTS:
            if name not in ("cbt_status_str", "cbt_slab_bytes", "cbt_slab_bytes_kv8",
                            "cbt_slab_bytes_kvq", "cbt_kernel_launches"):
                getattr(L, name).restype = c_int32
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise CbtError(rc, what)


def _i32_array(vals):
    arr = (c_int32 * max(1, len(vals)))(*[int(v) for v in vals])
    return arr


# ---- the C ABI, one function per entry point ------------------------------------------
def status_str(s: int) -> str:
    return lib().cbt_status_str(s).decode()


def engine_create(cfg: ModelConfig, weights: Weights, params: EngineParams) -> int:
    h = c_void()
    _check(lib().cbt_engine_create(ctypes.byref(cfg), ctypes.byref(weights),
                                   ctypes.byref(params), ctypes.byref(h)), "cbt_engine_create")
    return h.value


def engine_destroy(e: int) -> None:
    _check(lib().cbt_engine_destroy(e), "cbt_engine_destroy")


def slab_bytes(cfg: ModelConfig, capacity: int) -> int:
    return lib().cbt_slab_bytes(ctypes.byref(cfg), capacity)


def slab_bytes_kv8(cfg: ModelConfig, capacity: int) -> int:
    return lib().cbt_slab_bytes_kv8(ctypes.byref(cfg), capacity)


def slab_bytes_kvq(cfg: ModelConfig, capacity: int, bits: int) -> int:
    return lib().cbt_slab_bytes_kvq(ctypes.byref(cfg), capacity, bits)


def quantize_kv(x_ptr: int, rows: int, cols: int, bits: int, codes_ptr: int, scales_ptr: int,
                biases_ptr: int, stream: int = 0) -> None:
    _check(lib().cbt_quantize_kv(x_ptr, rows, cols, bits, codes_ptr, scales_ptr, biases_ptr,
                                 stream), "cbt_quantize_kv")


def quantize_kv8(x_ptr: int, rows: int, cols: int, codes_ptr: int, scales_ptr: int,
                 biases_ptr: int, stream: int = 0) -> None:
    _check(lib().cbt_quantize_kv8(x_ptr, rows, cols, codes_ptr, scales_ptr, biases_ptr, stream),
           "cbt_quantize_kv8")


def kv_slab_alloc(e: int, capacity: int) -> int:
    sid = c_int32()
    _check(lib().cbt_kv_slab_alloc(e, capacity, ctypes.byref(sid)), "cbt_kv_slab_alloc")
    return sid.value


def kv_slab_free(e: int, slab_id: int) -> None:
    _check(lib().cbt_kv_slab_free(e, slab_id), "cbt_kv_slab_free")


def retire(e: int, slab_ids) -> None:
    arr = _i32_array(slab_ids)
    _check(lib().cbt_retire(e, ctypes.cast(arr, c_void), len(slab_ids)), "cbt_retire")


def kv_slab_position(e: int, slab_id: int) -> int:
    p = c_int32()
    _check(lib().cbt_kv_slab_position(e, slab_id, ctypes.byref(p)), "cbt_kv_slab_position")
    return p.value


def kv_slab_import(e: int, slab_id: int, k_ptr: int, v_ptr: int, n_tokens: int,
                   on_host: bool) -> None:
    _check(lib().cbt_kv_slab_import(e, slab_id, k_ptr, v_ptr, n_tokens, int(on_host)),
           "cbt_kv_slab_import")


def kv_slab_copy_prefix(e: int, src: int, dst: int, n_tokens: int) -> None:
    _check(lib().cbt_kv_slab_copy_prefix(e, src, dst, n_tokens), "cbt_kv_slab_copy_prefix")


def kv_slab_share_prefix(e: int, src: int, dst: int, n_tokens: int) -> None:
    _check(lib().cbt_kv_slab_share_prefix(e, src, dst, n_tokens), "cbt_kv_slab_share_prefix")


def kv_slab_export(e: int, slab_id: int, k_ptr: int, v_ptr: int, n_tokens: int,
                   on_host: bool) -> None:
    _check(lib().cbt_kv_slab_export(e, slab_id, k_ptr, v_ptr, n_tokens, int(on_host)),
           "cbt_kv_slab_export")


def prefill_segmented(e: int, slab_ids, seg_lens, tokens_ptr: int, logits_ptr: int | None,
                      next_ptr: int | None) -> None:
    ids = _i32_array(slab_ids)
    lens = _i32_array(seg_lens)
    _check(lib().cbt_prefill_segmented(e, ctypes.cast(ids, c_void), ctypes.cast(lens, c_void),
                                       len(slab_ids), tokens_ptr, logits_ptr, next_ptr),
           "cbt_prefill_segmented")


def decode_step_batch(e: int, slab_ids, last_tokens_ptr: int, logits_ptr: int | None,
                      next_ptr: int | None) -> None:
    ids = _i32_array(slab_ids)
    _check(lib().cbt_decode_step_batch(e, ctypes.cast(ids, c_void), len(slab_ids),
                                       last_tokens_ptr, logits_ptr, next_ptr),
           "cbt_decode_step_batch")


def last_device_error(e: int):
    code, info = c_int32(), c_int32()
    _check(lib().cbt_last_device_error(e, ctypes.byref(code), ctypes.byref(info)),
           "cbt_last_device_error")
    return code.value, info.value


def engine_stats(e: int) -> Stats:
    st = Stats()
    _check(lib().cbt_engine_stats(e, ctypes.byref(st)), "cbt_engine_stats")
    return st


def kernel_launches(e: int | None = None) -> int:
    return lib().cbt_kernel_launches(e)


def greedy_head_noalloc(cfg: ModelConfig, hidden_ptr: int, n: int, final_norm_ptr: int,
                        lm_head: Linear, logits_ptr: int, next_ptr: int | None,
                        stream: int = 0) -> None:
    """Final RMSNorm + lm_head + greedy argmax on caller-owned hidden states, using only the
    library's fixed device scratch (no allocation; see include/cbt.h)."""
    _check(lib().cbt_greedy_head_noalloc(ctypes.byref(cfg), hidden_ptr, n, final_norm_ptr,
                                         ctypes.byref(lm_head), logits_ptr, next_ptr, stream),
           "cbt_greedy_head_noalloc")


def engine_set_timing(e: int, class_mask: int) -> None:
    _check(lib().cbt_engine_set_timing(e, class_mask), "cbt_engine_set_timing")


def engine_timing(e: int, kclass: int):
    """(total device ms, intervals, algorithmic bytes) of one kernel class."""
    ms, n, by = ctypes.c_double(), ctypes.c_int64(), ctypes.c_double()
    _check(lib().cbt_engine_timing(e, kclass, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(by)),
           "cbt_engine_timing")
    return ms.value, n.value, by.value


def quantize_affine4(w_ptr: int, rows: int, cols: int, group: int, packed_ptr: int,
                     scales_ptr: int, biases_ptr: int, stream: int = 0) -> None:
    _check(lib().cbt_quantize_affine4(w_ptr, rows, cols, group, packed_ptr, scales_ptr,
                                      biases_ptr, stream), "cbt_quantize_affine4")


def engine_set_stamps(e: int, enable: bool) -> None:
    _check(lib().cbt_engine_set_stamps(e, 1 if enable else 0), "cbt_engine_set_stamps")


def engine_stamps(e: int, cap: int = 1024):
    """The last decode step's stamps: a list of (class, begin_ns, end_ns)."""
    import numpy as np
    n = c_int32()
    cls = np.zeros(cap, dtype=np.int32)
    t = np.zeros(2 * cap, dtype=np.uint64)
    _check(lib().cbt_engine_stamps(e, cap, ctypes.byref(n), cls.ctypes.data, t.ctypes.data),
           "cbt_engine_stamps")
    k = min(cap, n.value)
    return [(int(cls[i]), int(t[2 * i]), int(t[2 * i + 1])) for i in range(k)]


def engine_test_stall(e: int, spin_limit: int) -> None:
    _check(lib().cbt_engine_test_stall(e, spin_limit), "cbt_engine_test_stall")
