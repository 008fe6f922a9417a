"""Engine host logic through the C ABI on a GPU: the slab allocator, host-detected errors
(reported before any work is queued, engine unchanged), the device error word, state
save/restore, and the batching invariants of the pages on the GPU path itself."""
import numpy as np
import pytest
import torch

from continuous_batching_transformer_gb300 import binding as B
from continuous_batching_transformer_gb300.model import DeviceWeights, Engine
from synth.recipes import TINY
from tests.gpu_harness import ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def weights():
    ensure_built()
    return DeviceWeights(TINY, torch.device("cuda:0"))


def small_engine(weights, arena_positions=512, max_batch=4):
    return Engine(weights, arena_bytes=B.slab_bytes(weights.cfg, arena_positions), max_batch=max_batch,
                  max_prefill_tokens=64)


def status_of(fn, *a):
    try:
        fn(*a)
    except B.CbtError as e:
        return e.status
    return 0


def test_allocator_first_fit_and_coalescing(weights):
    """First fit with coalescing; capacities are whole 64-position groups."""
    eng = small_engine(weights, arena_positions=256)
    arena = eng.stats().arena_bytes
    assert arena == B.slab_bytes(weights.cfg, 256)
    a = eng.kv_slab_alloc(64)
    b = eng.kv_slab_alloc(40)  # rounds up to 64 positions
    c = eng.kv_slab_alloc(64)
    st = eng.stats()
    assert st.live_slabs == 3 and st.slab_bytes_in_use == 3 * B.slab_bytes(weights.cfg, 64)
    eng.kv_slab_free(b)
    d = eng.kv_slab_alloc(64)  # first fit: reuses b's extent
    assert status_of(eng.kv_slab_alloc, 128) == -7  # only 64 positions left at the end
    eng.kv_slab_free(a)
    eng.kv_slab_free(c)
    eng.kv_slab_free(d)
    st = eng.stats()
    assert st.live_slabs == 0 and st.slab_bytes_in_use == 0 and st.largest_free_bytes == arena
    big = eng.kv_slab_alloc(250)  # after coalescing the whole arena is one extent again
    assert status_of(eng.kv_slab_alloc, 1) == -7  # pool exhausted
    eng.kv_slab_free(big)
    eng.close()


def test_host_errors_leave_engine_unchanged(weights):
    eng = small_engine(weights)
    dev = torch.device("cuda:0")
    s1, s2 = eng.kv_slab_alloc(8), eng.kv_slab_alloc(2)
    tok = to_dev(np.array([1, 2, 3, 4, 5], np.int32), dev)
    assert status_of(eng.kv_slab_free, 999) == -3                       # unknown id
    assert status_of(eng.decode_step_batch, [s1, s1], tok) == -4        # duplicate id
    assert status_of(eng.decode_step_batch, [s1, 12345], tok) == -3     # bad id
    assert status_of(eng.decode_step_batch, [s1] * 5, tok) in (-5, -4)  # over max_batch
    assert status_of(eng.prefill_segmented, [s2], [3], tok) == -6       # capacity
    assert status_of(eng.prefill_segmented, [s1], [0], tok) == -1       # empty segment
    assert status_of(eng.prefill_segmented, [s1, s2], [70, 1], tok) in (-6, -8)
    assert eng.position(s1) == 0 and eng.position(s2) == 0
    eng.decode_step_batch([], tok)  # B == 0 is a no-op
    eng.prefill_segmented([s2], [2], tok)
    assert eng.position(s2) == 2
    assert status_of(eng.decode_step_batch, [s2], tok) == -6             # slab full
    assert eng.position(s2) == 2
    eng.retire([s1, s2])
    assert status_of(eng.retire, [s1]) == -3                             # double free
    assert eng.stats().live_slabs == 0
    assert eng.device_error() == (0, 0)
    eng.close()


def test_device_error_word_on_bad_token(weights):
    eng = small_engine(weights)
    dev = torch.device("cuda:0")
    s = [eng.kv_slab_alloc(8), eng.kv_slab_alloc(8)]
    eng.decode_step_batch(s, to_dev(np.array([3, TINY.vocab + 7], np.int32), dev))
    code, info = eng.device_error()
    assert code == B.DEV_TOKEN_RANGE and info == 1
    assert eng.device_error() == (0, 0)  # read clears it
    # the engine stays usable
    eng.decode_step_batch(s, to_dev(np.array([3, 4], np.int32), dev))
    assert eng.device_error() == (0, 0)
    eng.close()


def test_import_export_round_trip(weights):
    eng = small_engine(weights)
    s = eng.kv_slab_alloc(20)
    dims = (TINY.n_layers, TINY.n_kv_heads, 13, TINY.head_dim)
    k = torch.randn(dims).to(torch.bfloat16)
    v = torch.randn(dims).to(torch.bfloat16)
    eng.import_kv(s, k, v, 13)
    assert eng.position(s) == 13
    k2, v2 = torch.empty_like(k), torch.empty_like(v)
    eng.export_kv(s, k2, v2, 13)
    assert torch.equal(k, k2) and torch.equal(v, v2)
    kd, vd = torch.empty_like(k).cuda(), torch.empty_like(v).cuda()
    eng.export_kv(s, kd, vd, 13)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), k)
    eng.close()


def _decode(eng, slabs, toks, dev):
    lg = torch.empty((len(slabs), TINY.vocab), dtype=torch.float32, device=dev)
    eng.decode_step_batch(slabs, to_dev(np.asarray(toks, np.int32), dev), lg)
    return lg.cpu().numpy()


def test_batched_equals_solo_and_no_leakage_on_gpu(weights):
    """decode_step_batch of K rows == K solo steps, and a perturbed slab changes only its
    own row (the gnosis page's parity gate and its no-cross-segment-leakage property)."""
    dev = torch.device("cuda:0")
    lens = [5, 12, 30]
    toks = [np.arange(n, dtype=np.int32) * 7 % TINY.vocab for n in lens]

    def fresh():
        eng = small_engine(weights)
        slabs = [eng.kv_slab_alloc(40) for _ in lens]
        eng.prefill_segmented(slabs, lens, to_dev(np.concatenate(toks), dev))
        return eng, slabs

    eng, slabs = fresh()
    batched = _decode(eng, slabs, [11, 22, 33], dev)
    for r in range(3):
        e2, s2 = fresh()
        solo = _decode(e2, [s2[r]], [[11, 22, 33][r]], dev)
        np.testing.assert_array_equal(batched[r], solo[0])
        e2.close()
    # perturb row 1's cached keys: rows 0 and 2 are bit-identical
    e3, s3 = fresh()
    n = lens[1]
    k = torch.empty((TINY.n_layers, TINY.n_kv_heads, n, TINY.head_dim), dtype=torch.bfloat16)
    v = torch.empty_like(k)
    e3.export_kv(s3[1], k, v, n)
    e3.import_kv(s3[1], (k.float() * 1.5).to(torch.bfloat16), v, n)
    other = _decode(e3, s3, [11, 22, 33], dev)
    np.testing.assert_array_equal(other[0], batched[0])
    np.testing.assert_array_equal(other[2], batched[2])
    assert not np.array_equal(other[1], batched[1])
    eng.close()
    e3.close()


def test_quantizer_matches_oracle_bytes(weights):
    """The engine's 4-bit quantiser and the oracle's (written separately) agree byte for byte."""
    import oracle
    import synth
    rows, cols = 96, 512
    wb = synth.normal_bf16(rows * cols, 3, 1234, sigma=0.02).reshape(rows, cols)
    dev = torch.device("cuda:0")
    wt = torch.from_numpy(wb.view(np.int16)).to(dev)
    packed = torch.empty((rows, cols // 8), dtype=torch.int32, device=dev)
    sc = torch.empty((rows, cols // 64), dtype=torch.int16, device=dev)
    bi = torch.empty_like(sc)
    B.quantize_affine4(wt.data_ptr(), rows, cols, 64, packed.data_ptr(), sc.data_ptr(),
                       bi.data_ptr(), 0)
    torch.cuda.synchronize()
    p, s, b = oracle.quantize_affine4(wb, 64)
    assert np.array_equal(packed.cpu().numpy().view(np.uint32), p)
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), s)
    assert np.array_equal(bi.cpu().numpy().view(np.uint16), b)


def test_prefix_copy_then_continue(weights):
    """Prefix reuse: one row prefills a 100-token system prompt plus its own 30 tokens; a second
    row takes the first 100 positions by copy and prefills only its own 20 tokens.  Its logits
    (and two decode steps of both rows) match the oracle's full computation; host errors queue
    nothing and change nothing."""
    import oracle
    from tests.gpu_harness import TOL, check_logits
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(77)
    system = rng.integers(0, TINY.vocab, 100).astype(np.int32)
    own = [rng.integers(0, TINY.vocab, n).astype(np.int32) for n in (30, 20)]
    eng = Engine(weights, arena_bytes=B.slab_bytes(weights.cfg, 1024), max_batch=4,
                 max_prefill_tokens=160)
    a, b, c = eng.kv_slab_alloc(192), eng.kv_slab_alloc(160), eng.kv_slab_alloc(64)
    lg = torch.empty((1, TINY.vocab), dtype=torch.float32, device=dev)
    eng.prefill_segmented([a], [130], to_dev(np.concatenate([system, own[0]]), dev), lg)
    la = lg.cpu().numpy().copy()
    assert status_of(eng.copy_prefix, a, a, 10) == -1        # same slab
    assert status_of(eng.copy_prefix, a, b, 131) == -6       # beyond the source's position
    assert status_of(eng.copy_prefix, a, c, 100) == -6       # beyond the target's capacity
    assert status_of(eng.copy_prefix, a, 999, 10) == -3      # unknown slab
    assert eng.position(b) == 0 and eng.position(c) == 0
    eng.copy_prefix(a, b, 100)
    assert eng.position(b) == 100
    eng.prefill_segmented([b], [20], to_dev(own[1], dev), lg)
    lb = lg.cpu().numpy().copy()

    om = oracle.OracleModel(TINY)
    ca, cb = oracle.KVCache(TINY, 192), oracle.KVCache(TINY, 160)
    ra = oracle.prefill_segmented(om, [ca], [130], np.concatenate([system, own[0]]))
    rb = oracle.prefill_segmented(om, [cb], [120], np.concatenate([system, own[1]]))
    check_logits(la, ra, TOL["bf16"], "row a prefill")
    check_logits(lb, rb, TOL["bf16"], "row b after the copied prefix")
    feed = np.array([oracle.argmax(ra[0]), oracle.argmax(rb[0])], np.int32)
    lg2 = torch.empty((2, TINY.vocab), dtype=torch.float32, device=dev)
    for step in range(2):
        eng.decode_step_batch([a, b], to_dev(feed, dev), lg2)
        ref = oracle.decode_step_batch(om, [ca, cb], feed)
        check_logits(lg2.cpu().numpy(), ref, TOL["bf16"], f"decode {step}")
        feed = np.array([oracle.argmax(x) for x in ref], np.int32)
    assert eng.device_error() == (0, 0)
    eng.close()


def test_decode_stamps_cover_every_projection_and_attention_launch():
    """cbt_engine_set_stamps: a replayed decode step records a [begin, end] interval for each
    projection (4 per layer and the lm_head) and each attention launch (attention and merge per
    layer); stamps change no result."""
    ensure_built()
    from continuous_batching_transformer_gb300 import binding as B
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    eng = Engine(w, arena_bytes=32 << 20, max_batch=4, max_prefill_tokens=64)
    slabs = [eng.kv_slab_alloc(64) for _ in range(3)]
    eng.prefill_segmented(slabs, [5, 9, 3], torch.arange(17, dtype=torch.int32, device=dev))
    tok = torch.tensor([1, 2, 3], dtype=torch.int32, device=dev)
    lg0 = torch.empty((3, TINY.vocab), dtype=torch.float32, device=dev)
    lg1 = torch.empty_like(lg0)
    eng.decode_step_batch(slabs, tok, lg0)
    B.engine_set_stamps(eng.handle, True)
    for _ in range(2):
        eng.decode_step_batch(slabs, tok, lg1)
    recs = B.engine_stamps(eng.handle)
    B.engine_set_stamps(eng.handle, False)
    n_proj = sum(1 for c, _, _ in recs if c == B.KCLASS_PROJ)
    n_attn = sum(1 for c, _, _ in recs if c == B.KCLASS_ATTN)
    assert n_proj == 4 * TINY.n_layers + 1 and n_attn == 2 * TINY.n_layers
    assert all(0 < b <= e for _, b, e in recs)
    span = max(e for _, _, e in recs) - min(b for _, b, _ in recs)
    assert span < 1e9  # one step, in nanoseconds
    assert eng.device_error() == (0, 0)
    eng.close()


def test_bounded_wait_reports_timeout_and_engine_stays_usable():
    """Failure detection without a fault: the armed step's lm_head projection requests none of
    its weight tiles, so its waits run out after a short limit; the step reports
    CBT_DEV_TIMEOUT through the device error word, and the next step (fed the oracle's tokens)
    matches the oracle -- the K/V the stalled step appended are intact."""
    ensure_built()
    import oracle
    from continuous_batching_transformer_gb300 import binding as B
    from tests.gpu_harness import TOL, check_logits
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    om = oracle.OracleModel(TINY)
    eng = Engine(w, arena_bytes=32 << 20, max_batch=4, max_prefill_tokens=64)
    lens = [5, 9, 3]
    slabs = [eng.kv_slab_alloc(64) for _ in lens]
    caches = [oracle.KVCache(TINY, 64) for _ in lens]
    toks = np.arange(sum(lens), dtype=np.int32) * 37 % TINY.vocab
    lg = torch.empty((3, TINY.vocab), dtype=torch.float32, device=dev)
    eng.prefill_segmented(slabs, lens, to_dev(toks, dev), lg)
    ref = oracle.prefill_segmented(om, caches, lens, toks)
    feed = np.array([oracle.argmax(r) for r in ref], np.int32)
    B.engine_test_stall(eng.handle, 1 << 12)
    eng.decode_step_batch(slabs, to_dev(feed, dev), lg)
    ref = oracle.decode_step_batch(om, caches, feed)
    code, info = eng.device_error()
    assert code == 2 and 200 <= info < 300, (code, info)  # CBT_DEV_TIMEOUT from a projection role
    assert [eng.position(s) for s in slabs] == [n + 1 for n in lens]
    feed = np.array([oracle.argmax(r) for r in ref], np.int32)
    for step in range(2):
        eng.decode_step_batch(slabs, to_dev(feed, dev), lg)
        ref = oracle.decode_step_batch(om, caches, feed)
        check_logits(lg.cpu().numpy(), ref, TOL["bf16"], f"after the stall, step {step}")
        feed = np.array([oracle.argmax(r) for r in ref], np.int32)
    assert eng.device_error() == (0, 0)
    with pytest.raises(B.CbtError):
        B.engine_test_stall(eng.handle, 0)
    eng.close()
