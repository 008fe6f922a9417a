"""Paged KV (engine kv_page_tokens = 128): a slab takes pages of 128 positions from the arena
as its positions are first written.  The same computation as contiguous slabs, so logits must
match the oracle and, bit for bit, the contiguous engine; pages are taken lazily (prefill,
decode at a page boundary, import, prefix copy), a call the arena cannot serve fails before
queuing anything and keeps nothing, and retiring returns pages."""
import numpy as np
import pytest
import torch

import oracle
from continuous_batching_transformer_gb300 import binding as B
from continuous_batching_transformer_gb300.model import DeviceWeights, Engine
from synth.recipes import TINY, ModelShape
from tests.gpu_harness import TOL, check_logits, ensure_built, to_dev

pytestmark = pytest.mark.gpu
PAGE = 128


def seeded(n, seed, vocab):
    return np.asarray(np.random.default_rng(seed).integers(0, vocab, n), np.int32)


def status_of(fn, *a):
    try:
        fn(*a)
    except B.CbtError as e:
        return e.status
    return 0


def run_engine(w, shape, page, lens, steps, feeds=None):
    """Prefill `lens` in one call, then `steps` decode steps fed the oracle's tokens (or
    `feeds`); every call's logits."""
    dev = torch.device("cuda:0")
    caps = [n + steps + 4 for n in lens]
    arena = sum(B.slab_bytes(w.cfg, (c + PAGE - 1) // PAGE * PAGE) for c in caps)
    eng = Engine(w, arena_bytes=arena, max_batch=8, max_prefill_tokens=sum(lens), page_tokens=page)
    slabs = [eng.kv_slab_alloc(c) for c in caps]
    toks = np.concatenate([seeded(n, 500 + r, shape.vocab) for r, n in enumerate(lens)])
    lg = torch.empty((len(lens), shape.vocab), dtype=torch.float32, device=dev)
    eng.prefill_segmented(slabs, lens, to_dev(toks, dev), lg)
    out = [lg.cpu().numpy().copy()]
    for s in range(steps):
        eng.decode_step_batch(slabs, to_dev(feeds[s], dev), lg)
        out.append(lg.cpu().numpy().copy())
    assert eng.device_error() == (0, 0)
    eng.close()
    return out, toks


@pytest.mark.parametrize("fmt", ["bf16", "affine4"])
def test_paged_matches_oracle_and_contiguous(fmt):
    """Segments of 5, 130 and 300 positions (one, two and three pages; prefill keys across
    page boundaries), then three decode steps; 4-bit prefill above 32 tokens takes the CUDA-core
    attention, which reads pages through the page table too."""
    ensure_built()
    shape = ModelShape("paged-check", 2, 512, 4, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1,
                       weight_format=fmt)
    w = DeviceWeights(shape, torch.device("cuda:0"))
    om = oracle.OracleModel(shape)
    lens = [5, 130, 300]
    caches = [oracle.KVCache(shape, n + 8) for n in lens]
    toks = np.concatenate([seeded(n, 500 + r, shape.vocab) for r, n in enumerate(lens)])
    refs = [oracle.prefill_segmented(om, caches, lens, toks)]
    feeds = []
    for s in range(3):
        feeds.append(np.array([oracle.argmax(x) for x in refs[-1]], np.int32))
        refs.append(oracle.decode_step_batch(om, caches, feeds[-1]))
    paged, _ = run_engine(w, shape, PAGE, lens, 3, feeds)
    flat, _ = run_engine(w, shape, 0, lens, 3, feeds)
    for k, (p, f, r) in enumerate(zip(paged, flat, refs)):
        check_logits(p, r, TOL[fmt], f"{fmt} paged call {k}")
        np.testing.assert_array_equal(p, f)


def test_paged_allocation_errors_and_state():
    ensure_built()
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    om = oracle.OracleModel(TINY)
    page_bytes = B.slab_bytes(w.cfg, PAGE)
    eng = Engine(w, arena_bytes=4 * page_bytes, max_batch=4, max_prefill_tokens=512,
                 page_tokens=PAGE)
    assert eng.stats().slab_bytes_in_use == 0
    a, b = eng.kv_slab_alloc(400), eng.kv_slab_alloc(200)      # no pages yet
    assert eng.stats().slab_bytes_in_use == 0
    ta, tb = seeded(400, 11, TINY.vocab), seeded(120, 12, TINY.vocab)
    ca, cb = oracle.KVCache(TINY, 400), oracle.KVCache(TINY, 200)
    lg = torch.empty((1, TINY.vocab), dtype=torch.float32, device=dev)
    eng.prefill_segmented([a], [255], to_dev(ta[:255], dev), lg)   # 2 pages
    check_logits(lg.cpu().numpy(), oracle.prefill_segmented(om, [ca], [255], ta[:255]),
                 TOL["bf16"], "prefill 255")
    eng.prefill_segmented([b], [120], to_dev(tb, dev), lg)          # 1 page
    oracle.prefill_segmented(om, [cb], [120], tb)
    assert eng.stats().slab_bytes_in_use == 3 * page_bytes
    # two more pages for a's positions [255, 400): only one is free -- nothing changes
    assert status_of(eng.prefill_segmented, [a], [145], to_dev(ta[255:], dev)) == -7
    assert eng.position(a) == 255 and eng.stats().slab_bytes_in_use == 3 * page_bytes
    # decode: position 255 is still in page 1, position 256 takes page 2 (the last free one)
    lg2 = torch.empty((2, TINY.vocab), dtype=torch.float32, device=dev)
    feed = np.array([ta[255], 7], np.int32)
    for step in range(2):
        eng.decode_step_batch([a, b], to_dev(feed, dev), lg2)
        ref = oracle.decode_step_batch(om, [ca, cb], feed)
        check_logits(lg2.cpu().numpy(), ref, TOL["bf16"], f"decode across a page boundary {step}")
        feed = np.array([ta[256 + step], 9 + step], np.int32)
    assert eng.stats().slab_bytes_in_use == 4 * page_bytes
    # the arena is full: a new slab gets no page until one is returned
    c = eng.kv_slab_alloc(64)
    assert status_of(eng.prefill_segmented, [c], [3], to_dev(tb[:3], dev)) == -7
    eng.retire([b])                                                  # its page comes back
    assert eng.stats().slab_bytes_in_use == 3 * page_bytes
    eng.prefill_segmented([c], [3], to_dev(tb[:3], dev), lg)
    assert eng.stats().slab_bytes_in_use == 4 * page_bytes
    # export a (257 positions over three pages) and import it into a fresh slab after freeing c
    n = eng.position(a)
    k = torch.empty((TINY.n_layers, TINY.n_kv_heads, n, TINY.head_dim), dtype=torch.bfloat16)
    v = torch.empty_like(k)
    eng.export_kv(a, k, v, n)
    assert n == 257
    eng.retire([c])
    d = eng.kv_slab_alloc(300)
    assert status_of(eng.import_kv, d, k, v, n) == -7                # needs 3 pages, 1 free
    eng.retire([a])
    eng.import_kv(d, k, v, n)
    k2, v2 = torch.empty_like(k), torch.empty_like(v)
    eng.export_kv(d, k2, v2, n)
    assert torch.equal(k, k2) and torch.equal(v, v2)
    # prefix copy into a paged slab: 130 positions would need two pages (one is free)
    e2 = eng.kv_slab_alloc(200)
    assert status_of(eng.copy_prefix, d, e2, 130) == -7 and eng.position(e2) == 0
    eng.copy_prefix(d, e2, 100)
    assert eng.position(e2) == 100
    k3 = torch.empty((TINY.n_layers, TINY.n_kv_heads, 100, TINY.head_dim), dtype=torch.bfloat16)
    v3 = torch.empty_like(k3)
    eng.export_kv(e2, k3, v3, 100)
    assert torch.equal(k3, k[:, :, :100]) and torch.equal(v3, v[:, :, :100])
    assert eng.device_error() == (0, 0)
    eng.close()


def shared_prefix_run(w, mode):
    """A 200-token prompt prefilled into s; d1 starts from its 200 positions and d2 from its
    first 150 (shared pages, or copies), each prefills tokens of its own (both land in the
    prompt's second page, which s still holds), all three decode a step, s retires, d1 and d2
    decode again.  Every call's logits, and the arena bytes held after each stage."""
    dev = torch.device("cuda:0")
    pb = B.slab_bytes(w.cfg, PAGE)
    eng = Engine(w, arena_bytes=8 * pb, max_batch=4, max_prefill_tokens=512, page_tokens=PAGE)
    pre = seeded(200, 21, TINY.vocab)
    own = np.concatenate([seeded(30, 22, TINY.vocab), seeded(20, 23, TINY.vocab)])
    lg = torch.empty((3, TINY.vocab), dtype=torch.float32, device=dev)
    out, used = [], []
    s = eng.kv_slab_alloc(400)
    eng.prefill_segmented([s], [200], to_dev(pre, dev), lg[:1])
    out.append(lg[:1].cpu().numpy().copy())
    d1, d2 = eng.kv_slab_alloc(400), eng.kv_slab_alloc(400)
    reuse = eng.share_prefix if mode == "share" else eng.copy_prefix
    reuse(s, d1, 200)
    reuse(s, d2, 150)
    used.append(eng.stats().slab_bytes_in_use // pb)
    eng.prefill_segmented([d1, d2], [30, 20], to_dev(own, dev), lg[:2])
    out.append(lg[:2].cpu().numpy().copy())
    used.append(eng.stats().slab_bytes_in_use // pb)
    eng.decode_step_batch([s, d1, d2], to_dev(np.array([7, 8, 9], np.int32), dev), lg)
    out.append(lg.cpu().numpy().copy())
    used.append(eng.stats().slab_bytes_in_use // pb)
    eng.retire([s])
    used.append(eng.stats().slab_bytes_in_use // pb)
    eng.decode_step_batch([d1, d2], to_dev(np.array([10, 11], np.int32), dev), lg[:2])
    out.append(lg[:2].cpu().numpy().copy())
    assert eng.device_error() == (0, 0)
    eng.close()
    return out, used, pre, own


def test_shared_prefix_pages_match_oracle_and_copy():
    """Prefix sharing: the shared run's logits follow the oracle (each sequence computed from
    its whole prompt in one pass) and equal, bit for bit, the same run with prefix copies; the
    shared run holds one copy of the prompt's pages and copies only the page both sequences
    write into."""
    ensure_built()
    w = DeviceWeights(TINY, torch.device("cuda:0"))
    om = oracle.OracleModel(TINY)
    shared, used_s, pre, own = shared_prefix_run(w, "share")
    copied, used_c, _, _ = shared_prefix_run(w, "copy")
    cs, c1, c2 = (oracle.KVCache(TINY, 400) for _ in range(3))
    refs = [oracle.prefill_segmented(om, [cs], [200], pre),
            oracle.prefill_segmented(om, [c1, c2], [230, 170],
                                     np.concatenate([pre, own[:30], pre[:150], own[30:]])),
            oracle.decode_step_batch(om, [cs, c1, c2], np.array([7, 8, 9], np.int32)),
            oracle.decode_step_batch(om, [c1, c2], np.array([10, 11], np.int32))]
    for k, (a, b, r) in enumerate(zip(shared, copied, refs)):
        check_logits(a, r, TOL["bf16"], f"shared prefix call {k}")
        np.testing.assert_array_equal(a, b)
    # shared: 2 pages after sharing; d1 and d2 each copy the second page when they write into
    # it; s's retirement returns only its second page (the first is still held by d1 and d2)
    assert used_s == [2, 4, 4, 3]
    assert used_c == [6, 6, 6, 4]


def test_shared_pages_copy_on_write_under_a_full_arena():
    """A write into a shared page needs a free page for its copy: with none free the call fails
    before queuing anything and changes nothing; once a page is returned it goes through, and
    the other holders keep their contents."""
    ensure_built()
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    om = oracle.OracleModel(TINY)
    pb = B.slab_bytes(w.cfg, PAGE)
    eng = Engine(w, arena_bytes=3 * pb, max_batch=4, max_prefill_tokens=512, page_tokens=PAGE)
    pre, o1, o2 = seeded(200, 31, TINY.vocab), seeded(30, 32, TINY.vocab), seeded(20, 33, TINY.vocab)
    lg = torch.empty((1, TINY.vocab), dtype=torch.float32, device=dev)
    s, d1 = eng.kv_slab_alloc(400), eng.kv_slab_alloc(400)
    eng.prefill_segmented([s], [200], to_dev(pre, dev), lg)
    # errors: a non-empty destination, the same slab, more positions than the source holds
    assert status_of(eng.share_prefix, s, s, 10) == -1
    assert status_of(eng.share_prefix, s, d1, 201) == -6
    assert status_of(eng.share_prefix, s, 12345, 10) == -3
    eng.share_prefix(s, d1, 200)
    assert status_of(eng.share_prefix, s, d1, 100) == -1 and eng.position(d1) == 200
    eng.prefill_segmented([d1], [30], to_dev(o1, dev), lg)      # copies page 1: arena full
    assert eng.stats().slab_bytes_in_use == 3 * pb
    d2 = eng.kv_slab_alloc(400)
    eng.share_prefix(s, d2, 200)
    assert status_of(eng.prefill_segmented, [d2], [20], to_dev(o2, dev)) == -7
    assert eng.position(d2) == 200 and eng.stats().slab_bytes_in_use == 3 * pb
    k1 = torch.empty((TINY.n_layers, TINY.n_kv_heads, 230, TINY.head_dim), dtype=torch.bfloat16)
    v1 = torch.empty_like(k1)
    eng.export_kv(d1, k1, v1, 230)
    eng.retire([d1])                                            # returns d1's copy of page 1
    assert eng.stats().slab_bytes_in_use == 2 * pb
    eng.prefill_segmented([d2], [20], to_dev(o2, dev), lg)      # copies page 1 again
    c2 = oracle.KVCache(TINY, 400)
    ref = oracle.prefill_segmented(om, [c2], [220], np.concatenate([pre, o2]))
    check_logits(lg.cpu().numpy(), ref, TOL["bf16"], "prefill after a copy on write")
    assert eng.stats().slab_bytes_in_use == 3 * pb
    # an import over a shared first page: no page for the copy until s retires
    d3 = eng.kv_slab_alloc(400)
    eng.share_prefix(s, d3, 100)
    g = torch.Generator().manual_seed(5)
    k = torch.randn((TINY.n_layers, TINY.n_kv_heads, 100, TINY.head_dim), generator=g).to(torch.bfloat16)
    v = torch.randn(k.shape, generator=g).to(torch.bfloat16)
    assert status_of(eng.import_kv, d3, k, v, 100) == -7 and eng.position(d3) == 100
    eng.retire([s])
    eng.import_kv(d3, k, v, 100)
    k3, v3 = torch.empty_like(k), torch.empty_like(v)
    eng.export_kv(d3, k3, v3, 100)
    assert torch.equal(k3, k) and torch.equal(v3, v)
    # d2 still reads the prompt it shared (positions [0, 200) as d1 saw them)
    k2 = torch.empty((TINY.n_layers, TINY.n_kv_heads, 200, TINY.head_dim), dtype=torch.bfloat16)
    v2 = torch.empty_like(k2)
    eng.export_kv(d2, k2, v2, 200)
    assert torch.equal(k2, k1[:, :, :200]) and torch.equal(v2, v1[:, :, :200])
    assert eng.device_error() == (0, 0)
    eng.close()


def test_share_on_a_contiguous_engine_copies():
    ensure_built()
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    eng = Engine(w, arena_bytes=2 * B.slab_bytes(w.cfg, 128), max_batch=2, max_prefill_tokens=128)
    s, d = eng.kv_slab_alloc(128), eng.kv_slab_alloc(128)
    eng.prefill_segmented([s], [50], to_dev(seeded(50, 41, TINY.vocab), dev))
    eng.share_prefix(s, d, 50)
    assert eng.position(d) == 50
    shape = (TINY.n_layers, TINY.n_kv_heads, 50, TINY.head_dim)
    ks, vs, kd, vd = (torch.empty(shape, dtype=torch.bfloat16) for _ in range(4))
    eng.export_kv(s, ks, vs, 50)
    eng.export_kv(d, kd, vd, 50)
    assert torch.equal(ks, kd) and torch.equal(vs, vd)
    eng.close()
