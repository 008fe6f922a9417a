"""CPU checks of the C ABI library: it builds for sm_103a, loads without a GPU, exports every
entry point include/cbt.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import continuous_batching_transformer_gb300 as cbt
from continuous_batching_transformer_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(cbt_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    cbt.build()
    return B.lib()


def test_exports_every_declared_entry_point(lib):
    names = declared_entry_points()
    assert "cbt_decode_step_batch" in names and "cbt_prefill_segmented" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding covers the same set
    assert set(names) <= set(B.EXPORTS) | {n for n in names if n in B.EXPORTS}
    assert sorted(set(B.EXPORTS)) == names


def test_status_strings(lib):
    for code in B.STATUS:
        assert B.status_str(code)
    assert "arena" in B.status_str(-7)


def test_create_rejects_null_and_bad_config(lib):
    cfg = B.ModelConfig(2, 256, 4, 4, 64, 1024, 1024, 1e-6, 1e4, 0, 64)
    h = ctypes.c_void_p()
    assert lib.cbt_engine_create(None, None, None, ctypes.byref(h)) == -2
    assert lib.cbt_engine_create(ctypes.byref(cfg), None, None, None) == -2
    lw = (B.LayerWeights * 2)()
    fake = 0x1000
    for l in range(2):
        lin = B.Linear(fake, None, None)
        lw[l] = B.LayerWeights(lin, lin, lin, lin, fake, fake)
    w = B.Weights(fake, B.Linear(fake, None, None), fake, ctypes.cast(lw, ctypes.POINTER(B.LayerWeights)))
    p = B.EngineParams(fake, 1 << 20, 4, 64, None)
    bad = B.ModelConfig(2, 256, 4, 3, 64, 1024, 1024, 1e-6, 1e4, 0, 64)   # heads % kv_heads != 0
    assert lib.cbt_engine_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(p), ctypes.byref(h)) == -1
    bad = B.ModelConfig(2, 256, 4, 4, 96, 1024, 1024, 1e-6, 1e4, 0, 64)   # head_dim 96
    assert lib.cbt_engine_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(p), ctypes.byref(h)) == -11
    bad = B.ModelConfig(2, 256, 4, 4, 64, 1024, 1024, 1e-6, 1e4, 1, 32)   # affine4 group 32
    assert lib.cbt_engine_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(p), ctypes.byref(h)) == -11
    p0 = B.EngineParams(fake, 1 << 20, 0, 64, None)                        # max_batch 0
    assert lib.cbt_engine_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(p0), ctypes.byref(h)) == -1
    for pages in (100, -128):                                              # page size: k * 128
        pp = B.EngineParams(fake, 1 << 20, 4, 64, None, pages)
        assert lib.cbt_engine_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(pp),
                                     ctypes.byref(h)) == -1
    lw[1] = B.LayerWeights(B.Linear(None, None, None), lw[0].wo, lw[0].wgu, lw[0].wd, fake, fake)
    assert lib.cbt_engine_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(p), ctypes.byref(h)) == -2
    assert not h.value


def test_slab_bytes(lib):
    cfg = B.ModelConfig(32, 4096, 32, 8, 128, 14336, 32000, 1e-5, 1e6, 0, 64)
    # 32 layers x (K, V) x 8 heads x 128 dims x 2 bytes = 131072 bytes per position, and a
    # slab holds whole groups of 64 positions (V is stored as transposed 64-key groups)
    assert B.slab_bytes(cfg, 64) == 64 * 131072
    assert B.slab_bytes(cfg, 1) == 64 * 131072
    assert B.slab_bytes(cfg, 2048) == 2048 * 131072
    assert B.slab_bytes(cfg, 2049) == 2112 * 131072
    tiny = B.ModelConfig(2, 256, 4, 4, 64, 1024, 1024, 1e-6, 1e4, 0, 64)
    assert B.slab_bytes(tiny, 2) == 64 * 2048  # 2048 bytes per position
    assert B.slab_bytes(tiny, 65) == 128 * 2048
    assert B.slab_bytes(tiny, 0) == 0
    # 8-bit KV: per position and (layer, K|V, kv head) head_dim codes + a bf16 scale and bias per
    # 64 dims: 32 x 2 x 8 x (128 + 4 + 4) = 69632 bytes per position
    assert B.slab_bytes_kv8(cfg, 2048) == 2048 * 69632
    assert B.slab_bytes_kv8(cfg, 1) == 64 * 69632
    assert B.slab_bytes_kv8(tiny, 100) == -(-(128 * 2 * 2 * 4 * (64 + 2 + 2)) // 4096) * 4096
    assert B.slab_bytes_kv8(tiny, 0) == 0
    odd = B.ModelConfig(2, 256, 4, 4, 96, 1024, 1024, 1e-6, 1e4, 0, 64)
    assert B.slab_bytes_kv8(odd, 64) == 0          # head_dim not a multiple of 64


def test_quantize_kv8_argument_checks(lib):
    """Rejected before anything is queued (no GPU needed): NULL buffers, a row length that is
    not a multiple of 64, misaligned buffers."""
    fake = ctypes.c_void_p(0x1000)
    assert lib.cbt_quantize_kv8(None, 4, 64, fake, fake, fake, None) == -2
    assert lib.cbt_quantize_kv8(fake, 4, 96, fake, fake, fake, None) == -1
    assert lib.cbt_quantize_kv8(ctypes.c_void_p(0x1002), 4, 64, fake, fake, fake, None) == -1
    assert lib.cbt_quantize_kv8(fake, 4, 64, ctypes.c_void_p(0x1001), fake, fake, None) == -1
    assert lib.cbt_quantize_kv8(fake, -1, 64, fake, fake, fake, None) == -1


def test_calls_reject_null_engine(lib):
    i = ctypes.c_int32()
    assert lib.cbt_kv_slab_alloc(None, 16, ctypes.byref(i)) == -2
    assert lib.cbt_kv_slab_free(None, 1) == -2
    assert lib.cbt_decode_step_batch(None, None, 1, None, None, None) == -2
    assert lib.cbt_prefill_segmented(None, None, None, 1, None, None, None) == -2
    assert lib.cbt_retire(None, None, 0) == -2
    assert lib.cbt_kv_slab_copy_prefix(None, 1, 2, 3) == -2
    assert lib.cbt_kv_slab_share_prefix(None, 1, 2, 3) == -2
    assert lib.cbt_quantize_affine4(None, 1, 64, 64, None, None, None, None) == -2
    fake = ctypes.c_void_p(0x1000)
    assert lib.cbt_quantize_affine4(fake, 4, 96, 64, fake, fake, fake, None) == -1  # cols % group


def test_kv8_engine_rejects_unsupported_head_groups(lib):
    """8-bit KV decode attention is built for 1, 2, 4 or 8 q heads per kv head: any other ratio
    is refused by cbt_engine_create before anything reaches the device."""
    fake = 0x1000
    h = ctypes.c_void_p()

    def create(n_heads, n_kv_heads, kv_bits):
        cfg = B.ModelConfig(2, 256, n_heads, n_kv_heads, 64, 1024, 1024, 1e-6, 1e4, 0, 64)
        lw = (B.LayerWeights * 2)()
        for l in range(2):
            lin = B.Linear(fake, None, None)
            lw[l] = B.LayerWeights(lin, lin, lin, lin, fake, fake)
        w = B.Weights(fake, B.Linear(fake, None, None), fake,
                      ctypes.cast(lw, ctypes.POINTER(B.LayerWeights)))
        p = B.EngineParams(fake, 1 << 30, 4, 64, None, 0, kv_bits)
        return lib.cbt_engine_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(p),
                                     ctypes.byref(h))

    for heads, kv in ((12, 4), (20, 4), (24, 4), (28, 4), (16, 1)):  # 3, 5, 6, 7, 16 per kv head
        assert create(heads, kv, 8) == -11, (heads, kv)
        assert not h.value
    # a supported ratio gets past the check (here it then fails on the missing device)
    assert create(16, 4, 8) != -11
    assert not h.value
