"""8-bit affine KV (engine kv_bits = 8) against the oracle's 8-bit cache.  The quantiser agrees
with the oracle's byte for byte; a prompt is prefilled in bf16 and then converted, so prefill
logits equal the bf16 engine's bit for bit; decode steps (each appending quantised K/V and
attending over every position's codes) follow the oracle within the logit tolerance, over
contexts spanning several 128-key work items, with imported KV too; the calls an 8-bit engine
does not offer fail before queuing anything."""
import numpy as np
import pytest
import torch

import oracle
import synth
from continuous_batching_transformer_gb300 import binding as B
from continuous_batching_transformer_gb300.model import DeviceWeights, Engine
from synth.recipes import TINY, ModelShape
from tests.gpu_harness import TOL, check_logits, ensure_built, to_dev

pytestmark = pytest.mark.gpu

GQA = ModelShape("kv8-gqa", 2, 512, 4, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1)


def seeded(n, seed, vocab):
    return np.asarray(np.random.default_rng(seed).integers(0, vocab, n), np.int32)


def status_of(fn, *a):
    try:
        fn(*a)
    except B.CbtError as e:
        return e.status
    return 0


def test_kv8_quantizer_matches_oracle_bytes():
    ensure_built()
    dev = torch.device("cuda:0")
    rows, cols = 200, 128
    x = synth.normal_bf16(rows * cols, 5, 4321, sigma=1.3).reshape(rows, cols)
    x[3, :] = x[3, 0]                                   # a constant row: scale 0
    q = np.random.default_rng(9).integers(0, 256, (cols,))
    q[0], q[1] = 0, 255
    x[4] = (((q - 128) / 64.0).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    xt = torch.from_numpy(x.view(np.int16)).to(dev)
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    sc = torch.empty((rows, cols // 64), dtype=torch.int16, device=dev)
    bi = torch.empty_like(sc)
    B.quantize_kv8(xt.data_ptr(), rows, cols, codes.data_ptr(), sc.data_ptr(), bi.data_ptr(), 0)
    torch.cuda.synchronize()
    c, s, b = oracle.quantize_kv8(x)
    assert np.array_equal(codes.cpu().numpy(), c)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), s)
    assert np.array_equal(bi.cpu().numpy().view(np.uint16), b)


def run(w, shape, kv_bits, lens, feeds):
    dev = torch.device("cuda:0")
    caps = [n + len(feeds) + 4 for n in lens]
    per = B.slab_bytes_kv8 if kv_bits == 8 else B.slab_bytes
    arena = sum(per(w.cfg, c) + B.slab_bytes(w.cfg, c) for c in caps) + 8 * B.slab_bytes(w.cfg, 128)
    eng = Engine(w, arena_bytes=arena, max_batch=8, max_prefill_tokens=sum(lens), kv_bits=kv_bits)
    slabs = [eng.kv_slab_alloc(c) for c in caps]
    toks = np.concatenate([seeded(n, 700 + r, shape.vocab) for r, n in enumerate(lens)])
    lg = torch.empty((len(lens), shape.vocab), dtype=torch.float32, device=dev)
    eng.prefill_segmented(slabs, lens, to_dev(toks, dev), lg)
    out = [lg.cpu().numpy().copy()]
    for f in feeds:
        eng.decode_step_batch(slabs, to_dev(f, dev), lg)
        out.append(lg.cpu().numpy().copy())
    assert eng.device_error() == (0, 0)
    eng.close()
    return out, toks


@pytest.mark.parametrize("shape", [TINY, GQA], ids=["tiny-hd64", "gqa-hd128"])
def test_kv8_engine_matches_oracle(shape):
    """Segments of 5, 130 and 300 positions (one to three 128-key items per head), prefill then
    four decode steps on the oracle's tokens."""
    ensure_built()
    w = DeviceWeights(shape, torch.device("cuda:0"))
    om = oracle.OracleModel(shape)
    lens = [5, 130, 300]
    caches = [oracle.KVCache(shape, n + 8, kv_bits=8) for n in lens]
    toks = np.concatenate([seeded(n, 700 + r, shape.vocab) for r, n in enumerate(lens)])
    refs = [oracle.prefill_segmented(om, caches, lens, toks)]
    feeds = []
    for _ in range(4):
        feeds.append(np.array([oracle.argmax(x) for x in refs[-1]], np.int32))
        refs.append(oracle.decode_step_batch(om, caches, feeds[-1]))
    got, _ = run(w, shape, 8, lens, feeds)
    flat, _ = run(w, shape, 16, lens, feeds[:0])
    np.testing.assert_array_equal(got[0], flat[0])   # prefill runs in bf16
    for k, (g, r) in enumerate(zip(got, refs)):
        check_logits(g, r, TOL["bf16"], f"kv8 {shape.name} call {k}")


def test_kv8_imported_context_matches_oracle():
    """Synthetic KV imported into two slabs (450 and 700 positions), then three decode steps."""
    ensure_built()
    dev = torch.device("cuda:0")
    w = DeviceWeights(GQA, dev)
    om = oracle.OracleModel(GQA)
    ctx = [450, 700]
    arena = sum(B.slab_bytes_kv8(w.cfg, c + 8) + B.slab_bytes(w.cfg, c) for c in ctx) \
        + 4 * B.slab_bytes(w.cfg, 128)
    eng = Engine(w, arena_bytes=arena, max_batch=4, max_prefill_tokens=64, kv_bits=8)
    slabs = [eng.kv_slab_alloc(c + 8) for c in ctx]
    caches = [oracle.KVCache(GQA, c + 8, kv_bits=8) for c in ctx]
    for r, (sl, c) in enumerate(zip(slabs, ctx)):
        eng.fill_synthetic_kv(sl, r, c, seed=3)
        caches[r].fill_synthetic(r, c, 3)
        assert eng.position(sl) == c
    lg = torch.empty((2, GQA.vocab), dtype=torch.float32, device=dev)
    feed = seeded(2, 71, GQA.vocab)
    for step in range(3):
        eng.decode_step_batch(slabs, to_dev(feed, dev), lg)
        ref = oracle.decode_step_batch(om, caches, feed)
        check_logits(lg.cpu().numpy(), ref, TOL["bf16"], f"kv8 imported step {step}")
        feed = np.array([oracle.argmax(x) for x in ref], np.int32)
    assert eng.device_error() == (0, 0)
    eng.close()


def test_kv8_sizes_and_unsupported_calls():
    ensure_built()
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    c = TINY
    assert B.slab_bytes_kv8(w.cfg, 100) == -(-(c.n_layers * 2 * c.n_kv_heads * 128
                                              * (c.head_dim + c.head_dim // 16)) // 4096) * 4096
    stage = 2 * B.slab_bytes(w.cfg, 128)
    with pytest.raises(B.CbtError):          # no room for the decode rows' staging
        Engine(w, arena_bytes=stage - 4096, max_batch=2, max_prefill_tokens=64, kv_bits=8)
    with pytest.raises(B.CbtError):          # 8-bit KV needs contiguous slabs
        Engine(w, arena_bytes=8 << 20, max_batch=2, max_prefill_tokens=64, kv_bits=8,
               page_tokens=128)
    eng = Engine(w, arena_bytes=stage + 4 * B.slab_bytes(w.cfg, 64), max_batch=2,
                 max_prefill_tokens=64, kv_bits=8)
    assert eng.stats().slab_bytes_in_use == stage
    a, b = eng.kv_slab_alloc(64), eng.kv_slab_alloc(64)
    eng.prefill_segmented([a], [10], to_dev(seeded(10, 1, c.vocab), dev))
    assert eng.position(a) == 10
    # the bf16 intermediate of a prefill is returned
    assert eng.stats().slab_bytes_in_use == stage + 2 * B.slab_bytes_kv8(w.cfg, 64)
    assert status_of(eng.prefill_segmented, [a], [5], to_dev(seeded(5, 2, c.vocab), dev)) == -11
    k = torch.zeros((c.n_layers, c.n_kv_heads, 10, c.head_dim), dtype=torch.bfloat16)
    assert status_of(eng.export_kv, a, k, k.clone(), 10) == -11
    assert status_of(eng.copy_prefix, a, b, 5) == -11
    assert status_of(eng.share_prefix, a, b, 5) == -11
    assert eng.position(a) == 10 and eng.position(b) == 0
    assert eng.device_error() == (0, 0)
    eng.close()


G4 = ModelShape("kv8-g4", 2, 512, 8, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1)
G8 = ModelShape("kv8-g8", 2, 512, 16, 2, 64, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1)
GQA_Q4 = ModelShape("kv8-gqa-affine4", 2, 512, 4, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1,
                    weight_format="affine4")


@pytest.mark.parametrize("shape", [G4, G8, GQA_Q4], ids=["g4-hd128", "g8-hd64", "affine4-g2"])
def test_kv8_head_groups_and_staging_page_change(shape):
    """4 and 8 q heads per kv head (the 7B shape's ratio and the widest), and 4-bit affine
    weights with 8-bit KV; prompts of 126 and 127 positions so that the decode steps write
    positions 126..130, crossing from the decode rows' first 128-position staging page into the
    next, plus a short and a 300-position prompt."""
    ensure_built()
    w = DeviceWeights(shape, torch.device("cuda:0"))
    om = oracle.OracleModel(shape)
    lens = [126, 127, 7, 300]
    caches = [oracle.KVCache(shape, n + 8, kv_bits=8) for n in lens]
    toks = np.concatenate([seeded(n, 700 + r, shape.vocab) for r, n in enumerate(lens)])
    refs = [oracle.prefill_segmented(om, caches, lens, toks)]
    feeds = []
    for _ in range(4):
        feeds.append(np.array([oracle.argmax(x) for x in refs[-1]], np.int32))
        refs.append(oracle.decode_step_batch(om, caches, feeds[-1]))
    got, _ = run(w, shape, 8, lens, feeds)
    tol = TOL["affine4" if shape.weight_format == "affine4" else "bf16"]
    for k, (g, r) in enumerate(zip(got, refs)):
        check_logits(g, r, tol, f"kv8 {shape.name} call {k}")
