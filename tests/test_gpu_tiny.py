"""GPU parity on the tiny decoder (2 layers, d_model 256, 4 heads, vocab 1024), through the C
ABI, against the CPU oracle: segmented prefill of prompts {5, 17, 32, 9}, then 16 greedy
decode steps, logits element by element (bf16 tolerance 2e-2) and greedy tokens."""
import numpy as np
import pytest
import torch

import oracle
from continuous_batching_transformer_gb300.model import DeviceWeights, Engine
from synth.recipes import TINY, TINY_RUN, ModelShape
from tests.gpu_harness import TOL, check_logits, ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    ensure_built()
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    om = oracle.OracleModel(TINY)
    return dev, w, om


def run_tiny(dev, w, om, use_register: bool):
    lens = [int(n) for n in TINY_RUN.context_lengths()]
    toks = np.concatenate([TINY_RUN.row_tokens(r, n) for r, n in enumerate(lens)])
    eng = Engine(w, arena_bytes=32 << 20, max_batch=8, max_prefill_tokens=128)
    cap = 64
    slabs = [eng.kv_slab_alloc(cap) for _ in lens]
    B = len(lens)
    logits = torch.empty((B, TINY.vocab), dtype=torch.float32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    eng.prefill_segmented(slabs, lens, to_dev(toks, dev), logits, nxt)
    caches = [oracle.KVCache(TINY, cap) for _ in lens]
    ref = oracle.prefill_segmented(om, caches, lens, toks)
    errs = [check_logits(logits.cpu().numpy(), ref, TOL["bf16"], "prefill")]
    assert [eng.position(s) for s in slabs] == lens
    feed = np.array([oracle.argmax(r) for r in ref], dtype=np.int32)
    gpu_tokens, ref_tokens = [nxt.cpu().numpy().copy()], [feed.copy()]
    for step in range(TINY_RUN.steps):
        if use_register:
            last = nxt.clone()  # device-side feed, no host round trip
        else:
            last = to_dev(feed, dev)  # teacher-forced on the oracle's tokens
        eng.decode_step_batch(slabs, last, logits, nxt)
        if use_register:  # the device-side tokens are the oracle's greedy tokens
            assert np.array_equal(last.cpu().numpy(), feed), f"step {step}: device tokens"
        ref = oracle.decode_step_batch(om, caches, feed)
        errs.append(check_logits(logits.cpu().numpy(), ref, TOL["bf16"], f"decode step {step}"))
        feed = np.array([oracle.argmax(r) for r in ref], dtype=np.int32)
        gpu_tokens.append(nxt.cpu().numpy().copy())
        ref_tokens.append(feed.copy())
    assert [eng.position(s) for s in slabs] == [n + TINY_RUN.steps for n in lens]
    # the slabs hold the K/V the oracle cached.  Prefill projections take bf16 operands
    # (8 significant bits), so a cached value carries a relative error of order 2^-8 of the
    # spread of its dot product's terms: with K/V spread 0.32 here, 1e-2 absolute bounds it.
    for r, sl in enumerate(slabs):
        n = lens[r] + TINY_RUN.steps
        k = torch.empty((TINY.n_layers, TINY.n_kv_heads, n, TINY.head_dim), dtype=torch.bfloat16)
        v = torch.empty_like(k)
        eng.export_kv(sl, k, v, n)
        ck = torch.from_numpy(caches[r].k[:, :, :n].view(np.int16)).view(torch.bfloat16)
        cv = torch.from_numpy(caches[r].v[:, :, :n].view(np.int16)).view(torch.bfloat16)
        torch.testing.assert_close(k.float(), ck.float(), atol=1e-2, rtol=1e-2)
        torch.testing.assert_close(v.float(), cv.float(), atol=1e-2, rtol=1e-2)
    assert eng.device_error() == (0, 0)
    eng.close()
    return errs, np.array(gpu_tokens), np.array(ref_tokens)


def test_tiny_teacher_forced(setup):
    dev, w, om = setup
    errs, g, r = run_tiny(dev, w, om, use_register=False)
    print(f"tiny: max |logit - oracle| over prefill + 16 steps = {max(errs):.3e}")


def test_tiny_device_register_feed(setup):
    """Greedy decode fed from the device next-token buffer: every token the GPU feeds itself
    must be the oracle's own greedy token (the oracle runs on its own tokens)."""
    dev, w, om = setup
    errs, g, r = run_tiny(dev, w, om, use_register=True)
    assert max(errs) <= TOL["bf16"]


@pytest.mark.parametrize("fmt", ["bf16", "affine4"])
def test_gqa_shape_parity(fmt):
    """Grouped-query heads (4 q heads over 2 kv heads), non-unit norm gains, head_dim 128 and
    both weight formats; prompts straddle several GEMM tiles (tiled and skinny paths)."""
    ensure_built()
    from dataclasses import replace
    shape = ModelShape("gqa-check", 2, 512, 4, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1,
                       weight_format=fmt)
    dev = torch.device("cuda:0")
    w = DeviceWeights(shape, dev)
    om = oracle.OracleModel(shape)
    lens = [40, 1, 77, 33, 9]
    toks = np.concatenate([np.asarray(np.random.default_rng(r).integers(0, shape.vocab, n), np.int32)
                           for r, n in enumerate(lens)])
    eng = Engine(w, arena_bytes=64 << 20, max_batch=8, max_prefill_tokens=256)
    slabs = [eng.kv_slab_alloc(96) for _ in lens]
    caches = [oracle.KVCache(shape, 96) for _ in lens]
    logits = torch.empty((len(lens), shape.vocab), dtype=torch.float32, device=dev)
    nxt = torch.empty(len(lens), dtype=torch.int32, device=dev)
    eng.prefill_segmented(slabs, lens, to_dev(toks, dev), logits, nxt)
    ref = oracle.prefill_segmented(om, caches, lens, toks)
    check_logits(logits.cpu().numpy(), ref, TOL[fmt], f"{fmt} prefill")
    feed = np.array([oracle.argmax(r) for r in ref], dtype=np.int32)
    for step in range(3):
        eng.decode_step_batch(slabs, to_dev(feed, dev), logits, nxt)
        ref = oracle.decode_step_batch(om, caches, feed)
        check_logits(logits.cpu().numpy(), ref, TOL[fmt], f"{fmt} decode {step}")
        feed = np.array([oracle.argmax(r) for r in ref], dtype=np.int32)
    eng.close()


@pytest.mark.parametrize("B", [1, 5, 12, 24])
def test_affine4_decode_operand_widths(B):
    """4-bit affine weights through the tensor-core projections at every operand width (N
    tiles of 16, 32 and 64 operand rows): B rows with ragged prompts (each prefilled by its own
    call, so every call is a skinny one), two greedy steps against the oracle, and the last
    row's logits equal, bit for bit, to those of the row decoded alone."""
    ensure_built()
    shape = ModelShape("gqa-check-affine4", 2, 512, 4, 2, 128, 1024, 2048, 1e-5, 1e6,
                       gain_sigma=0.1, weight_format="affine4")
    dev = torch.device("cuda:0")
    w = DeviceWeights(shape, dev)
    om = oracle.OracleModel(shape)
    lens = [1 + (7 * r) % 23 for r in range(B)]
    toks = [np.asarray(np.random.default_rng(50 + r).integers(0, shape.vocab, n), np.int32)
            for r, n in enumerate(lens)]

    def engine_with(rows):
        eng = Engine(w, arena_bytes=64 << 20, max_batch=32, max_prefill_tokens=64)
        slabs, firsts = [], []
        lg = torch.empty((1, shape.vocab), dtype=torch.float32, device=dev)
        for r in rows:
            slabs.append(eng.kv_slab_alloc(64))
            eng.prefill_segmented([slabs[-1]], [lens[r]], to_dev(toks[r], dev), lg)
            firsts.append(lg.cpu().numpy()[0].copy())
        return eng, slabs, np.stack(firsts)

    eng, slabs, first = engine_with(range(B))
    caches = [oracle.KVCache(shape, 64) for _ in lens]
    ref = oracle.prefill_segmented(om, caches, lens, np.concatenate(toks))
    check_logits(first, ref, TOL["affine4"], "affine4 prefill")
    feeds, outs = [], []
    feed = np.array([oracle.argmax(r) for r in ref], dtype=np.int32)
    logits = torch.empty((B, shape.vocab), dtype=torch.float32, device=dev)
    for step in range(2):
        eng.decode_step_batch(slabs, to_dev(feed, dev), logits)
        got = logits.cpu().numpy().copy()
        ref = oracle.decode_step_batch(om, caches, feed)
        check_logits(got, ref, TOL["affine4"], f"affine4 B={B} decode {step}")
        feeds.append(feed)
        outs.append(got)
        feed = np.array([oracle.argmax(r) for r in ref], dtype=np.int32)
    assert eng.device_error() == (0, 0)
    eng.close()
    solo, s1, _ = engine_with([B - 1])
    lg1 = torch.empty((1, shape.vocab), dtype=torch.float32, device=dev)
    for step in range(2):
        solo.decode_step_batch(s1, to_dev(feeds[step][B - 1:], dev), lg1)
        np.testing.assert_array_equal(lg1.cpu().numpy()[0], outs[step][B - 1])
    solo.close()


def test_long_rows_take_two_subchunk_items():
    """Rows whose context reaches 8192 keys are split into attention items of two 128-key
    sub-chunks (the others into items of one): rows of 8300 (an odd count of sub-chunks, so its
    last item has one), 8191 and 300 positions of seeded synthetic KV, two decode steps fed the
    oracle's own greedy tokens, against the oracle, and the long row's logits equal, bit for
    bit, to those of the row decoded alone (the item split depends on the row's own length)."""
    ensure_built()
    shape = ModelShape("long-items", 2, 512, 4, 2, 128, 1024, 2048, 1e-5, 1e6, gain_sigma=0.1)
    dev = torch.device("cuda:0")
    ctx = [8300, 8191, 300]
    seed = 5
    om = oracle.OracleModel(shape)
    caches = []
    for r, n in enumerate(ctx):
        c = oracle.KVCache(shape, n + 8)
        c.fill_synthetic(r, n, seed)
        caches.append(c)
    feeds = [np.asarray(np.random.default_rng(9).integers(0, shape.vocab, len(ctx)), np.int32)]
    refs = []
    for step in range(2):
        refs.append(oracle.decode_step_batch(om, caches, feeds[-1]))
        feeds.append(np.array([oracle.argmax(o) for o in refs[-1]], dtype=np.int32))
    w = DeviceWeights(shape, dev)

    def run(rows):
        eng = Engine(w, arena_bytes=96 << 20, max_batch=4, max_prefill_tokens=64)
        slabs = []
        for r in rows:
            slabs.append(eng.kv_slab_alloc(ctx[r] + 8))
            eng.fill_synthetic_kv(slabs[-1], r, ctx[r], seed)
        logits = torch.empty((len(rows), shape.vocab), dtype=torch.float32, device=dev)
        outs = []
        for step in range(2):
            eng.decode_step_batch(slabs, to_dev(feeds[step][rows], dev), logits)
            outs.append(logits.cpu().numpy().copy())
        assert eng.device_error() == (0, 0)
        eng.close()
        return outs

    batched = run([0, 1, 2])
    for step in range(2):
        check_logits(batched[step], refs[step], TOL["bf16"], f"long rows step {step}")
    solo = run([0])
    for step in range(2):
        assert np.array_equal(solo[step][0], batched[step][0]), f"step {step}: batched != solo"
