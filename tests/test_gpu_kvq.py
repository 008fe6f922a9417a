"""Affine KV of 8 and 4 bits (engine kv_bits = 8 / 4) against the oracle's quantised cache.

- The quantiser agrees with the oracle's byte for byte.
- A prompt that starts a sequence is prefilled in bf16 and then converted, so its logits equal
  the bf16 engine's bit for bit; decode steps (each quantising what it appends and attending over
  every position's codes on the tensor cores) follow the oracle within the logit tolerance, over
  contexts spanning several 128-key work items and both 128-position staging pages.
- Paged quantised KV equals contiguous quantised KV bit for bit.
- A prompt admitted in chunks: later chunks continue the slab and attend over codes, as in the
  oracle (prefill_continue on a quantised cache).
- Export gives each value as bf16(fp32(scale * code + bias)) -- the oracle's values for the same
  codes, bit for bit; copy and share of a prefix carry codes, scales and biases.
"""
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

GQA = ModelShape("kvq-gqa", 2, 512, 4, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1)
G4 = ModelShape("kvq-g4", 2, 512, 8, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1)
G8 = ModelShape("kvq-g8", 2, 512, 16, 2, 64, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1)
GQA_Q4 = ModelShape("kvq-gqa-affine4", 2, 512, 4, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1,
                    weight_format="affine4")
BITS = [8, 4]

_weights = {}


def weights(shape):
    if shape.name not in _weights:
        _weights[shape.name] = DeviceWeights(shape, torch.device("cuda:0"))
    return _weights[shape.name]


def seeded(n, seed, vocab):
    return np.asarray(np.random.default_rng(seed).integers(0, vocab, n), np.int32)


def tol_of(shape):
    return TOL["affine4" if shape.weight_format == "affine4" else "bf16"]


def arena_for(w, bits, caps, page=0):
    """Room for the slabs (or their pages), one bf16 intermediate per slab and the staging."""
    if page:
        q = sum(B.slab_bytes_kvq(w.cfg, page, bits) * (-(-c // page)) for c in caps)
    else:
        q = sum(B.slab_bytes_kvq(w.cfg, c, bits) for c in caps)
    return q + sum(B.slab_bytes(w.cfg, c) for c in caps) + 8 * B.slab_bytes(w.cfg, 128)


@pytest.mark.parametrize("bits", BITS)
def test_kvq_quantizer_matches_oracle_bytes(bits):
    ensure_built()
    dev = torch.device("cuda:0")
    rows, cols = 200, 128
    x = synth.normal_bf16(rows * cols, 5, 4321, sigma=1.3).reshape(rows, cols)
    x[3, :] = x[3, 0]                                   # a constant row: scale 0
    L = (1 << bits) - 1
    q = np.random.default_rng(9).integers(0, L + 1, (cols,))
    q[0], q[1] = 0, L
    x[4] = ((((q - L // 2) / 64.0).astype(np.float32).view(np.uint32)) >> 16).astype(np.uint16)
    xt = torch.from_numpy(x.view(np.int16)).to(dev)
    codes = torch.empty((rows, cols * bits // 8), dtype=torch.uint8, device=dev)
    sc = torch.empty((rows, cols // 64), dtype=torch.int16, device=dev)
    bi = torch.empty_like(sc)
    B.quantize_kv(xt.data_ptr(), rows, cols, bits, codes.data_ptr(), sc.data_ptr(), bi.data_ptr(), 0)
    torch.cuda.synchronize()
    c, s, b = oracle.quantize_kv(x, bits)
    assert np.array_equal(codes.cpu().numpy(), c)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), s)
    assert np.array_equal(bi.cpu().numpy().view(np.uint16), b)


def run(shape, kv_bits, lens, feeds, page=0, chunk=None):
    """Prefill the prompts (whole, or in chunks of `chunk` tokens, every prompt advancing one
    chunk per call), then one decode step per feed.  Returns the prefill logits (of each prompt's
    last chunk) and each step's logits."""
    dev = torch.device("cuda:0")
    w = weights(shape)
    caps = [n + len(feeds) + 4 for n in lens]
    assert kv_bits != 16 or not page
    arena = arena_for(w, kv_bits, caps, page) if kv_bits != 16 else \
        sum(B.slab_bytes(w.cfg, c) for c in caps)
    eng = Engine(w, arena_bytes=arena, max_batch=8, max_prefill_tokens=sum(lens),
                 kv_bits=kv_bits, page_tokens=page)
    slabs = [eng.kv_slab_alloc(c) for c in caps]
    toks = [seeded(n, 700 + r, shape.vocab) for r, n in enumerate(lens)]
    lg = torch.empty((len(lens), shape.vocab), dtype=torch.float32, device=dev)
    if chunk is None:
        eng.prefill_segmented(slabs, lens, to_dev(np.concatenate(toks), dev), lg)
        pre = lg.cpu().numpy().copy()
    else:
        done = [0] * len(lens)
        pre = np.zeros((len(lens), shape.vocab), np.float32)
        while min(d - n for d, n in zip(done, lens)) < 0:
            idx = [r for r in range(len(lens)) if done[r] < lens[r]]
            part = [min(chunk, lens[r] - done[r]) for r in idx]
            t = np.concatenate([toks[r][done[r]:done[r] + m] for r, m in zip(idx, part)])
            out = torch.empty((len(idx), shape.vocab), dtype=torch.float32, device=dev)
            eng.prefill_segmented([slabs[r] for r in idx], part, to_dev(t, dev), out)
            got = out.cpu().numpy()
            for j, (r, m) in enumerate(zip(idx, part)):
                done[r] += m
                if done[r] == lens[r]:
                    pre[r] = got[j]
    outs = [pre]
    for f in feeds:
        eng.decode_step_batch(slabs, to_dev(f, dev), lg)
        outs.append(lg.cpu().numpy().copy())
    assert eng.device_error() == (0, 0)
    assert [eng.position(s) for s in slabs] == [n + len(feeds) for n in lens]
    eng.close()
    return outs


def oracle_run(shape, kv_bits, lens, steps, chunk=None):
    om = oracle.OracleModel(shape)
    caches = [oracle.KVCache(shape, n + steps + 8, kv_bits=kv_bits) for n in lens]
    toks = [seeded(n, 700 + r, shape.vocab) for r, n in enumerate(lens)]
    if chunk is None:
        pre = oracle.prefill_segmented(om, caches, lens, np.concatenate(toks))
    else:
        done = [0] * len(lens)
        pre = np.zeros((len(lens), shape.vocab), np.float32)
        while min(d - n for d, n in zip(done, lens)) < 0:
            idx = [r for r in range(len(lens)) if done[r] < lens[r]]
            part = [min(chunk, lens[r] - done[r]) for r in idx]
            t = np.concatenate([toks[r][done[r]:done[r] + m] for r, m in zip(idx, part)])
            got = oracle.prefill_continue(om, [caches[r] for r in idx], part, t)
            for j, (r, m) in enumerate(zip(idx, part)):
                done[r] += m
                if done[r] == lens[r]:
                    pre[r] = got[j]
    refs, feeds = [pre], []
    for _ in range(steps):
        feeds.append(np.array([oracle.argmax(x) for x in refs[-1]], np.int32))
        refs.append(oracle.decode_step_batch(om, caches, feeds[-1]))
    return refs, feeds


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("shape", [TINY, GQA], ids=["tiny-hd64", "gqa-hd128"])
def test_kvq_engine_matches_oracle(shape, bits):
    """Segments of 5, 130 and 300 positions (one to three 128-key items per head), prefill then
    four decode steps on the oracle's tokens; prefill logits equal the bf16 engine's."""
    ensure_built()
    lens = [5, 130, 300]
    refs, feeds = oracle_run(shape, bits, lens, 4)
    got = run(shape, bits, lens, feeds)
    flat = run(shape, 16, lens, feeds[:0])
    np.testing.assert_array_equal(got[0], flat[0])   # a fresh prompt runs in bf16
    for k, (g, r) in enumerate(zip(got, refs)):
        check_logits(g, r, tol_of(shape), f"kv{bits} {shape.name} call {k}")


@pytest.mark.parametrize("shape,bits", [(G4, 8), (G8, 8), (GQA_Q4, 8), (G4, 4), (GQA_Q4, 4)],
                         ids=["g4-8", "g8-8", "affine4-8", "g4-4", "affine4-4"])
def test_kvq_head_groups_and_staging_page_change(shape, bits):
    """4 and 8 q heads per kv head, and 4-bit affine weights; prompts of 126 and 127 positions so
    the decode steps write positions 126..130, crossing from the decode rows' first 128-position
    staging page into the next, plus a short and a 300-position prompt."""
    ensure_built()
    lens = [126, 127, 7, 300]
    refs, feeds = oracle_run(shape, bits, lens, 4)
    got = run(shape, bits, lens, feeds)
    for k, (g, r) in enumerate(zip(got, refs)):
        check_logits(g, r, tol_of(shape), f"kv{bits} {shape.name} call {k}")


@pytest.mark.parametrize("bits", BITS)
def test_kvq_paged_equals_contiguous(bits):
    """Pages of 128 positions: prompts of 5, 200 and 300 positions (items in the second and third
    page) give the contiguous engine's logits bit for bit, at prefill and four decode steps."""
    ensure_built()
    lens = [5, 200, 300]
    refs, feeds = oracle_run(GQA, bits, lens, 4)
    paged = run(GQA, bits, lens, feeds, page=128)
    flat = run(GQA, bits, lens, feeds)
    for k, (p, f, r) in enumerate(zip(paged, flat, refs)):
        np.testing.assert_array_equal(p, f)
        check_logits(p, r, TOL["bf16"], f"paged kv{bits} call {k}")


@pytest.mark.parametrize("bits,page", [(8, 0), (4, 0), (8, 128), (4, 128)])
def test_kvq_chunked_prefill_matches_oracle(bits, page):
    """Prompts of 70, 200 and 33 tokens admitted 64 tokens per call: the first chunk of each
    starts its sequence (bf16, then converted), later chunks continue the slab and attend over
    codes; a call mixes starting and continuing segments.  Then three decode steps."""
    ensure_built()
    lens = [70, 200, 33]
    refs, feeds = oracle_run(GQA, bits, lens, 3, chunk=64)
    got = run(GQA, bits, lens, feeds, page=page, chunk=64)
    for k, (g, r) in enumerate(zip(got, refs)):
        check_logits(g, r, TOL["bf16"], f"chunked kv{bits} page {page} call {k}")


def synthetic_quant_slab(eng, shape, row, n, seed=3):
    sl = eng.kv_slab_alloc(n + 8)
    eng.fill_synthetic_kv(sl, row, n, seed)
    return sl


def export(eng, shape, slab, n):
    dims = (shape.n_layers, shape.n_kv_heads, n, shape.head_dim)
    k = torch.empty(dims, dtype=torch.bfloat16)
    v = torch.empty(dims, dtype=torch.bfloat16)
    eng.export_kv(slab, k, v, n)
    return k.view(torch.int16).numpy().view(np.uint16), v.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("bits,page", [(8, 0), (4, 0), (8, 128), (4, 128)])
def test_kvq_export_and_prefix_reuse(bits, page):
    """Synthetic KV imported (quantised on the device) into a slab of 450 positions: its export
    equals the oracle's export values for the oracle's codes of the same KV, bit for bit.  A
    prefix of 300 positions copied (and, on the paged engine, shared) into other slabs exports
    the same values; decode steps on the copies follow the oracle's cache."""
    ensure_built()
    dev = torch.device("cuda:0")
    shape = GQA
    w = weights(shape)
    n, pre = 450, 300
    eng = Engine(w, arena_bytes=arena_for(w, bits, [n + 8] * 4, page), max_batch=4,
                 max_prefill_tokens=64, kv_bits=bits, page_tokens=page)
    src = synthetic_quant_slab(eng, shape, 0, n)
    c = oracle.KVCache(shape, n + 8, kv_bits=bits)
    c.fill_synthetic(0, n, 3)
    k, v = export(eng, shape, src, n)
    hd = shape.head_dim
    for name, got in (("k", k), ("v", v)):
        q = c.q8
        want = oracle.kvq_export_values(q[name + "q"][:, :, :n].reshape(-1, hd * bits // 8),
                                        q[name + "s"][:, :, :n].reshape(-1, hd // 64),
                                        q[name + "b"][:, :, :n].reshape(-1, hd // 64), bits)
        np.testing.assert_array_equal(got.reshape(-1, hd), want, err_msg=f"export {name}")
    dst = [eng.kv_slab_alloc(pre + 8) for _ in range(2)]
    eng.copy_prefix(src, dst[0], pre)
    eng.share_prefix(src, dst[1], pre)   # a contiguous engine copies
    for d in dst:
        assert eng.position(d) == pre
        dk, dv = export(eng, shape, d, pre)
        assert np.array_equal(dk, k[:, :, :pre]) and np.array_equal(dv, v[:, :, :pre])
    # decode on both copies: the oracle's cache holds the same prefix
    om = oracle.OracleModel(shape)
    caches = []
    for _ in dst:
        cc = oracle.KVCache(shape, pre + 8, kv_bits=bits)
        cc.k[:, :, :pre], cc.v[:, :, :pre] = c.k[:, :, :pre], c.v[:, :, :pre]
        for key in cc.q8:
            cc.q8[key][:, :, :pre] = c.q8[key][:, :, :pre]
        cc.len = cc.qlen = pre
        caches.append(cc)
    feed = seeded(2, 71, shape.vocab)
    lg = torch.empty((2, shape.vocab), dtype=torch.float32, device=dev)
    for step in range(3):
        eng.decode_step_batch(dst, to_dev(feed, dev), lg)
        ref = oracle.decode_step_batch(om, caches, feed)
        check_logits(lg.cpu().numpy(), ref, TOL["bf16"], f"kv{bits} prefix copy step {step}")
        feed = np.array([oracle.argmax(x) for x in ref], np.int32)
    # the source is unchanged by the copies' writes
    k2, v2 = export(eng, shape, src, n)
    assert np.array_equal(k2, k) and np.array_equal(v2, v)
    assert eng.device_error() == (0, 0)
    eng.close()


def test_kvq_imported_context_matches_oracle():
    """Synthetic KV imported into two slabs (450 and 700 positions), then three decode steps, at
    8 and 4 bits."""
    ensure_built()
    dev = torch.device("cuda:0")
    w = weights(GQA)
    om = oracle.OracleModel(GQA)
    ctx = [450, 700]
    for bits in BITS:
        eng = Engine(w, arena_bytes=arena_for(w, bits, [c + 8 for c in ctx]), max_batch=4,
                     max_prefill_tokens=64, kv_bits=bits)
        slabs = [synthetic_quant_slab(eng, GQA, r, c) for r, c in enumerate(ctx)]
        caches = [oracle.KVCache(GQA, c + 8, kv_bits=bits) for c in ctx]
        for r, c in enumerate(ctx):
            caches[r].fill_synthetic(r, c, 3)
        lg = torch.empty((2, GQA.vocab), dtype=torch.float32, device=dev)
        feed = seeded(2, 71, GQA.vocab)
        for step in range(3):
            eng.decode_step_batch(slabs, to_dev(feed, dev), lg)
            ref = oracle.decode_step_batch(om, caches, feed)
            check_logits(lg.cpu().numpy(), ref, TOL["bf16"], f"kv{bits} imported step {step}")
            feed = np.array([oracle.argmax(x) for x in ref], np.int32)
        assert eng.device_error() == (0, 0)
        eng.close()


def test_kvq_sizes_and_staging():
    ensure_built()
    w = weights(TINY)
    c = TINY
    for bits in BITS:
        per = c.n_layers * 2 * c.n_kv_heads * (c.head_dim * bits // 8 + c.head_dim // 16)
        assert B.slab_bytes_kvq(w.cfg, 100, bits) == -(-(per * 128) // 4096) * 4096
    assert B.slab_bytes_kv8(w.cfg, 100) == B.slab_bytes_kvq(w.cfg, 100, 8)
    stage = 2 * B.slab_bytes(w.cfg, 128)
    with pytest.raises(B.CbtError):          # no room for the decode rows' staging
        Engine(w, arena_bytes=stage - 4096, max_batch=2, max_prefill_tokens=64, kv_bits=4)
    eng = Engine(w, arena_bytes=stage + 4 * B.slab_bytes(w.cfg, 64), max_batch=2,
                 max_prefill_tokens=64, kv_bits=4)
    assert eng.stats().slab_bytes_in_use == stage
    a = eng.kv_slab_alloc(64)
    eng.prefill_segmented([a], [10], to_dev(seeded(10, 1, c.vocab), torch.device("cuda:0")))
    assert eng.position(a) == 10
    # the bf16 intermediate of the prefill was returned
    assert eng.stats().slab_bytes_in_use == stage + B.slab_bytes_kvq(w.cfg, 64, 4)
    assert eng.device_error() == (0, 0)
    eng.close()
