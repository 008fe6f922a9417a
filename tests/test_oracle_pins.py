"""Pins of the CPU oracle against things other than itself.

Each building block is checked against a library routine (PyTorch / NumPy in
fp64), a closed form, or a worked example derived by hand
(tests/golden/hand_examples.json); the composed model is checked against an
fp64 PyTorch composition of library routines (rms_norm,
scaled_dot_product_attention with grouped-query heads, silu, matmul) with
RoPE written as complex multiplication; and the batching semantics are
checked by the invariants the pages state for the path (batched == solo,
segmented == per-sequence, no cross-segment leakage).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from synth.recipes import ModelShape, TINY

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))


def bf16_bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32(bits):
    return synth.bf16_to_f32(np.asarray(bits, dtype=np.uint16))


# ---- bf16 rounding -------------------------------------------------------------------
def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 3,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 1e-40, -2.5e-39],
                                 dtype=np.float32)])
    # exact ties: 1 + 2^-8 (tie, even -> 1.0) and 1 + 3*2^-8 (tie, odd -> up)
    ours = oracle.bf16_round(x)
    assert np.array_equal(ours, bf16_bits(x))


# ---- RMSNorm ----------------------------------------------------------------------------
def test_rmsnorm_matches_library():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(257).astype(np.float32) * 2
    g = bf16_bits(1 + 0.1 * rng.standard_normal(257))
    got = oracle.rmsnorm(x, g, 1e-6)
    ref = F.rms_norm(torch.tensor(x, dtype=torch.float64), (257,),
                     weight=torch.tensor(f32(g), dtype=torch.float64), eps=1e-6).numpy()
    np.testing.assert_allclose(got, ref, rtol=2e-7, atol=1e-7)


def test_rmsnorm_hand_example_and_constant_input():
    ex = GOLD["rmsnorm_3_4"]
    got = oracle.rmsnorm(np.array(ex["x"], np.float32), bf16_bits(ex["gain"]), ex["eps"])
    np.testing.assert_allclose(got, ex["out"], rtol=1e-7)
    # constant input c gives sign(c) * g * |c| / sqrt(c^2 + eps)
    c, eps = -0.75, 1e-5
    got = oracle.rmsnorm(np.full(64, c, np.float32), bf16_bits(np.full(64, 1.5)), eps)
    np.testing.assert_allclose(got, np.full(64, -1.5 * 0.75 / math.sqrt(0.5625 + eps)), rtol=1e-7)


# ---- RoPE -------------------------------------------------------------------------------
def rope_complex(v, pos, theta):
    """RoPE as complex multiplication: z_i = v[i] + 1j*v[i+hd/2] times exp(1j*pos*theta^(-2i/hd))."""
    hd = v.size
    half = hd // 2
    z = v[:half].astype(np.float64) + 1j * v[half:].astype(np.float64)
    w = np.exp(1j * pos * theta ** (-2.0 * np.arange(half) / hd))
    r = z * w
    return np.concatenate([r.real, r.imag])


def test_rope_hand_example():
    ex = GOLD["rope_quarter_turn"]
    got = oracle.rope(np.array(ex["x"], np.float32), ex["pos"], ex["theta"])
    np.testing.assert_allclose(got, ex["out"], atol=1e-7)


@pytest.mark.parametrize("hd,theta", [(64, 1e4), (128, 1e6)])
def test_rope_properties(hd, theta):
    rng = np.random.default_rng(hd)
    q = rng.standard_normal(hd).astype(np.float32)
    k = rng.standard_normal(hd).astype(np.float32)
    # identity at position 0
    assert np.array_equal(oracle.rope(q, 0, theta), q)
    for pos in (1, 7, 511, 16383):
        r = oracle.rope(q, pos, theta)
        # complex-multiplication form (pairs i, i+hd/2; positive rotation)
        np.testing.assert_allclose(r, rope_complex(q, pos, theta), atol=3e-6)
        # each pair keeps its norm
        half = hd // 2
        np.testing.assert_allclose(np.hypot(r[:half], r[half:]), np.hypot(q[:half], q[half:]),
                                   rtol=1e-6)
    # q(p) . k(p') depends only on p - p'
    d1 = float(np.dot(oracle.rope(q, 100, theta).astype(np.float64), oracle.rope(k, 90, theta)))
    d2 = float(np.dot(oracle.rope(q, 1010, theta).astype(np.float64), oracle.rope(k, 1000, theta)))
    assert abs(d1 - d2) < 1e-4 * max(1.0, abs(d1))


# ---- attention ----------------------------------------------------------------------------
def test_attention_hand_example():
    ex = GOLD["attention_two_keys"]
    got = oracle.attention(np.array(ex["q"], np.float32), bf16_bits(ex["k"]), bf16_bits(ex["v"]))
    np.testing.assert_allclose(got, ex["out"], rtol=1e-6)


@pytest.mark.parametrize("hd,n", [(4, 1), (4, 5), (8, 3), (64, 37), (128, 300)])
def test_attention_matches_library(hd, n):
    rng = np.random.default_rng(hd * 1000 + n)
    q = (rng.standard_normal(hd) * 1.3).astype(np.float32)
    kb = bf16_bits(rng.standard_normal((n, hd)) * 1.3)
    vb = bf16_bits(rng.standard_normal((n, hd)))
    got = oracle.attention(q, kb, vb)
    t = lambda a: torch.tensor(a, dtype=torch.float64)[None, None]
    ref = F.scaled_dot_product_attention(t(q[None]), t(f32(kb)), t(f32(vb)))[0, 0, 0].numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-7)


def test_attention_special_cases():
    rng = np.random.default_rng(3)
    vb = bf16_bits(rng.standard_normal((6, 8)))
    kb = bf16_bits(rng.standard_normal((6, 8)))
    # a single key returns its value exactly
    np.testing.assert_array_equal(oracle.attention(rng.standard_normal(8).astype(np.float32), kb[:1], vb[:1]), f32(vb[0]))
    # q = 0 gives the mean of the values
    np.testing.assert_allclose(oracle.attention(np.zeros(8, np.float32), kb, vb),
                               f32(vb).astype(np.float64).mean(0), rtol=1e-6, atol=1e-7)


# ---- SiLU, argmax ----------------------------------------------------------------------------
def test_silu_matches_library():
    for z in (-30.0, -2.5, -1e-3, 0.0, 0.7, 4.0, 30.0):
        assert abs(oracle.silu(z) - F.silu(torch.tensor(z, dtype=torch.float64)).item()) < 1e-15


def test_argmax_lowest_index_on_ties():
    lg = np.array([0.1, 0.7, -3, 0.7, 0.2, 0.7], np.float32)
    assert oracle.argmax(lg) == 1
    rng = np.random.default_rng(5)
    for _ in range(20):
        lg = np.round(rng.standard_normal(1000), 1).astype(np.float32)  # many ties
        assert oracle.argmax(lg) == int(np.argmax(lg))  # numpy returns the first maximum


# ---- projections --------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["bf16", "affine4"])
def test_linear_matches_matmul(fmt):
    s = ModelShape("lin", 1, 128, 2, 2, 64, 192, 10, 1e-6, 1e4, weight_format=fmt)
    rng = np.random.default_rng(7)
    wb = bf16_bits(rng.standard_normal((96, 192)) * 0.02)
    lin = oracle.LinearW(wb, fmt, 64)
    m = oracle.OracleModel.__new__(oracle.OracleModel)
    m.shape = s
    m.cfg = oracle.Config(1, 128, 2, 2, 64, 192, 10, 1e-6, 1e4, 0 if fmt == "bf16" else 1, 64)
    x = rng.standard_normal((5, 192)).astype(np.float32)
    y = m.linear(lin, x)
    W = f32(wb).astype(np.float64) if fmt == "bf16" else oracle.dequantize_affine4(
        lin.packed, lin.scales, lin.biases, 64)
    np.testing.assert_allclose(y, x.astype(np.float64) @ W.T, rtol=1e-6, atol=1e-6)


# ---- 4-bit affine quantiser ---------------------------------------------------------------------
def test_affine4_hand_example():
    ex = GOLD["affine4_group"]
    w = np.array([-0.5 + i / 64 if i < 16 else 0.25 for i in range(64)], np.float32)
    wb = bf16_bits(w)[None, :]
    packed, scales, biases = oracle.quantize_affine4(wb, 64)
    assert f32(scales)[0, 0] == ex["scale_bf16_value"]
    assert f32(biases)[0, 0] == ex["bias_value"]
    codes = [(int(packed[0, i // 8]) >> (4 * (i % 8))) & 0xF for i in range(64)]
    assert codes[0] == ex["code_0"] and codes[8] == ex["code_8"] and codes[16] == ex["code_16"]
    assert int(packed[0, 2]) == ex["word_2"]


def test_affine4_round_trip_bound():
    rng = np.random.default_rng(11)
    wb = bf16_bits(rng.standard_normal((64, 256)) * 0.02)
    packed, scales, biases = oracle.quantize_affine4(wb, 64)
    deq = oracle.dequantize_affine4(packed, scales, biases, 64)
    w = f32(wb).astype(np.float64)
    sc = np.repeat(f32(scales).astype(np.float64), 64, axis=1)
    # |dequant - w| <= scale/2, plus the slack from rounding scale to bf16 (<= 15 * 2^-9 * scale)
    assert np.all(np.abs(deq - w) <= sc * (0.5 + 15 * 2.0 ** -9) + 1e-12)
    codes = np.stack([(packed >> np.uint32(4 * k)) & np.uint32(0xF) for k in range(8)], -1).reshape(64, 256)
    g = w.reshape(64, 4, 64)
    cg = codes.reshape(64, 4, 64)
    # each group's minimum maps to 0 and its maximum to 15
    assert np.all(cg[np.arange(64)[:, None], np.arange(4)[None], g.argmin(-1)] == 0)
    assert np.all(cg[np.arange(64)[:, None], np.arange(4)[None], g.argmax(-1)] == 15)


# ---- the composed model against an fp64 PyTorch composition of library routines -------------
PIN_SHAPE = ModelShape("pin-gqa", 2, 128, 4, 2, 32, 256, 300, 1e-6, 1e4, gain_sigma=0.1)


def torch_reference_logits(m: oracle.OracleModel, tokens):
    """fp64 PyTorch forward of one sequence, all positions; K/V rounded to bf16 as cached."""
    s = m.shape
    dt = torch.float64

    def W(lin):
        if lin.w is not None:
            return torch.tensor(f32(lin.w), dtype=dt)
        return torch.tensor(oracle.dequantize_affine4(lin.packed, lin.scales, lin.biases, s.group_size), dtype=dt)

    def g(bits):
        return torch.tensor(f32(bits), dtype=dt)

    def rope(t, pos):  # t: [T, H, hd]
        half = s.head_dim // 2
        z = torch.complex(t[..., :half], t[..., half:])
        ang = pos[:, None, None] * s.rope_theta ** (-2.0 * torch.arange(half, dtype=dt) / s.head_dim)
        r = z * torch.polar(torch.ones_like(ang), ang)
        return torch.cat([r.real, r.imag], -1)

    T = len(tokens)
    pos = torch.arange(T, dtype=dt)
    x = torch.tensor(f32(m.embed[np.asarray(tokens)]), dtype=dt)
    for L in m.layers:
        h = F.rms_norm(x, (s.d_model,), weight=g(L["attn_norm"]), eps=s.rms_eps)
        q = rope((h @ W(L["wq"]).T).view(T, s.n_heads, s.head_dim), pos)
        k = rope((h @ W(L["wk"]).T).view(T, s.n_kv_heads, s.head_dim), pos)
        v = (h @ W(L["wv"]).T).view(T, s.n_kv_heads, s.head_dim)
        k = k.float().to(torch.bfloat16).to(dt)
        v = v.float().to(torch.bfloat16).to(dt)
        o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                           v.transpose(0, 1)[None], is_causal=True,
                                           enable_gqa=True)[0].transpose(0, 1).reshape(T, -1)
        x = x + o @ W(L["wo"]).T
        h = F.rms_norm(x, (s.d_model,), weight=g(L["ffn_norm"]), eps=s.rms_eps)
        x = x + (F.silu(h @ W(L["wg"]).T) * (h @ W(L["wu"]).T)) @ W(L["wd"]).T
    h = F.rms_norm(x, (s.d_model,), weight=g(m.final_norm), eps=s.rms_eps)
    return (h @ W(m.lm_head).T).numpy()


@pytest.mark.parametrize("fmt", ["bf16", "affine4"])
def test_model_matches_torch_composition(fmt):
    from dataclasses import replace
    m = oracle.OracleModel(replace(PIN_SHAPE, weight_format=fmt))
    toks = synth.tokens(23, 9, synth.stream_tokens(0), PIN_SHAPE.vocab)
    ref = torch_reference_logits(m, toks)
    # every position's logits: prefill of the first p+1 tokens, last logits
    cache = oracle.KVCache(m.shape, 32)
    got_last = oracle.prefill_sequence(m, cache, toks)
    np.testing.assert_allclose(got_last, ref[-1], atol=2e-5)
    # token by token through decode steps
    c2 = oracle.KVCache(m.shape, 32)
    for p, t in enumerate(toks):
        lg = oracle.decode_step_batch(m, [c2], [t])[0]
        np.testing.assert_allclose(lg, ref[p], atol=2e-5)


# ---- batching invariants (the pages' parity gates) ----------------------------------------------
@pytest.fixture(scope="module")
def pin_model():
    return oracle.OracleModel(PIN_SHAPE)


def _prefilled(m, lens, cap=48, seed=4):
    caches, toks = [], []
    for r, n in enumerate(lens):
        t = synth.tokens(n, seed, synth.stream_tokens(r), m.shape.vocab)
        c = oracle.KVCache(m.shape, cap)
        oracle.prefill_sequence(m, c, t)
        caches.append(c)
        toks.append(t)
    return caches, toks


def _clone(c):
    d = oracle.KVCache(c.shape, c.capacity)
    d.k[...] = c.k
    d.v[...] = c.v
    d.len = c.len
    return d


def test_batched_decode_equals_solo(pin_model):
    caches, _ = _prefilled(pin_model, [3, 11, 7])
    solo = [_clone(c) for c in caches]
    last = [5, 17, 250]
    lg = oracle.decode_step_batch(pin_model, caches, last)
    for b in range(3):
        lb = oracle.decode_step_batch(pin_model, [solo[b]], [last[b]])[0]
        assert np.array_equal(lg[b], lb)
        assert np.array_equal(caches[b].k, solo[b].k) and np.array_equal(caches[b].v, solo[b].v)
        assert caches[b].len == solo[b].len


def test_segmented_equals_per_sequence(pin_model):
    lens = [5, 17, 1, 9]
    toks = [synth.tokens(n, 6, synth.stream_tokens(r), PIN_SHAPE.vocab) for r, n in enumerate(lens)]
    seg = [oracle.KVCache(PIN_SHAPE, 32) for _ in lens]
    lg = oracle.prefill_segmented(pin_model, seg, lens, np.concatenate(toks))
    for r, n in enumerate(lens):
        c = oracle.KVCache(PIN_SHAPE, 32)
        ls = oracle.prefill_sequence(pin_model, c, toks[r])
        assert np.array_equal(lg[r], ls)
        assert np.array_equal(seg[r].k, c.k) and np.array_equal(seg[r].v, c.v) and seg[r].len == n


def test_chunked_prefill_equals_one_pass(pin_model):
    """A prompt admitted in chunks (each continuing its cache, other rows' chunks and new rows
    sharing the calls) ends with the logits and K/V of one segmented prefill of the prompt."""
    lens = [13, 5, 9]
    toks = [synth.tokens(n, 9, synth.stream_tokens(r), PIN_SHAPE.vocab) for r, n in enumerate(lens)]
    one = [oracle.KVCache(PIN_SHAPE, 16) for _ in lens]
    ref = oracle.prefill_segmented(pin_model, one, lens, np.concatenate(toks))
    ch = [oracle.KVCache(PIN_SHAPE, 16) for _ in lens]
    # call 1: rows 0 and 1 start (4 and 5 tokens: row 1 completes); call 2: row 0 continues
    # (7 more), row 2 starts (3); call 3: both finish
    calls = [[(0, 0, 4), (1, 0, 5)], [(0, 4, 11), (2, 0, 3)], [(0, 11, 13), (2, 3, 9)]]
    last = {}
    for call in calls:
        caches = [ch[r] for r, _, _ in call]
        lg = oracle.prefill_continue(pin_model, caches, [b - a for _, a, b in call],
                                     np.concatenate([toks[r][a:b] for r, a, b in call]))
        for k, (r, _, b) in enumerate(call):
            if b == lens[r]:
                last[r] = lg[k]
    for r, n in enumerate(lens):
        assert np.array_equal(last[r], ref[r])
        assert ch[r].len == n
        assert np.array_equal(ch[r].k, one[r].k) and np.array_equal(ch[r].v, one[r].v)
    with pytest.raises(ValueError):
        oracle.prefill_continue(pin_model, [ch[0]], [2], np.zeros(3, np.int32))


def test_no_cross_row_leakage(pin_model):
    caches, _ = _prefilled(pin_model, [6, 6, 6])
    other = [_clone(c) for c in caches]
    other[1].k[:, :, :6] ^= np.uint16(0x0040)  # perturb every cached K value of row 1
    last = [1, 2, 3]
    a = oracle.decode_step_batch(pin_model, caches, last)
    b = oracle.decode_step_batch(pin_model, other, last)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])
    assert not np.array_equal(a[1], b[1])
    # segmented prefill: a different token in segment 1 changes no other segment
    lens = [4, 4, 4]
    t = synth.tokens(12, 8, synth.stream_tokens(0), PIN_SHAPE.vocab)
    t2 = t.copy()
    t2[5] = (t2[5] + 1) % PIN_SHAPE.vocab
    l1 = oracle.prefill_segmented(pin_model, [oracle.KVCache(PIN_SHAPE, 8) for _ in lens], lens, t)
    l2 = oracle.prefill_segmented(pin_model, [oracle.KVCache(PIN_SHAPE, 8) for _ in lens], lens, t2)
    assert np.array_equal(l1[0], l2[0]) and np.array_equal(l1[2], l2[2])
    assert not np.array_equal(l1[1], l2[1])


def test_prefill_then_decode_equals_longer_prefill(pin_model):
    t = synth.tokens(13, 12, synth.stream_tokens(0), PIN_SHAPE.vocab)
    c = oracle.KVCache(PIN_SHAPE, 16)
    oracle.prefill_sequence(pin_model, c, t[:12])
    lg = oracle.decode_step_batch(pin_model, [c], [t[12]])[0]
    c2 = oracle.KVCache(PIN_SHAPE, 16)
    ref = oracle.prefill_sequence(pin_model, c2, t)
    np.testing.assert_allclose(lg, ref, atol=1e-6)


def test_row_permutation(pin_model):
    caches, _ = _prefilled(pin_model, [2, 9, 4, 7])
    perm = [2, 0, 3, 1]
    last = np.array([10, 20, 30, 40])
    pc = [_clone(caches[i]) for i in perm]
    a = oracle.decode_step_batch(pin_model, caches, last)
    b = oracle.decode_step_batch(pin_model, pc, last[perm])
    assert np.array_equal(a[perm], b)


def test_rejects_bad_token_lists(pin_model):
    c = oracle.KVCache(PIN_SHAPE, 4)
    with pytest.raises(ValueError):  # token id out of range
        oracle.decode_step_batch(pin_model, [c], [PIN_SHAPE.vocab])
    with pytest.raises(ValueError):  # capacity exceeded
        oracle.prefill_sequence(pin_model, c, np.zeros(5, np.int32))


# ---- the seeded generator -------------------------------------------------------------------------
def test_synth_deterministic_and_normal():
    a = synth.normal_bf16(200000, 0, 77, sigma=1.0)
    b = synth.normal_bf16(200000, 0, 77, sigma=1.0)
    assert np.array_equal(a, b)
    x = f32(a).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    # sub-range fills agree with the whole (counter based)
    c = synth.normal_bf16(1000, 0, 77, first=5000, sigma=1.0)
    assert np.array_equal(c, a[5000:6000])
    t = synth.tokens(100000, 0, 3, 1024)
    assert t.min() >= 0 and t.max() < 1024 and abs(t.mean() - 511.5) < 5
    k1 = synth.kv(0, 0, 2, 4, 9, 64, 0, 0.32)
    k2 = synth.kv(0, 0, 2, 4, 5, 64, 0, 0.32)
    assert np.array_equal(k1[:, :, :5], k2)  # KV draws do not depend on the context length


# ---- 8-bit affine KV -------------------------------------------------------------------
def _bf16_bits(x):
    """Exact bf16 bit patterns of values that bf16 holds exactly (checked)."""
    f = np.asarray(x, dtype=np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), f)
    return bits


def test_kv8_hand_example():
    """Groups whose values lie on an exact grid quantise losslessly: a group spanning
    [0, 255/8] has scale 1/8 and bias 0, one spanning [-4, -4 + 255/32] scale 1/32 and bias -4,
    and every code is the grid index.  A value halfway between two steps rounds to the even
    code; a constant group has scale 0, bias equal to the value and all codes 0."""
    rng = np.random.default_rng(3)
    qa = rng.integers(0, 256, 64)
    qa[5], qa[40] = 0, 255
    qb = rng.integers(0, 256, 64)
    qb[0], qb[63] = 255, 0
    row0 = np.concatenate([qa / 8.0, -4.0 + qb / 32.0])
    ties = np.zeros(64)
    ties[1], ties[2], ties[3] = 255 / 8.0, 1.5 / 8.0, 2.5 / 8.0    # steps 1.5 -> 2, 2.5 -> 2
    row1 = np.concatenate([ties, np.full(64, 1.5)])
    codes, scales, biases = oracle.quantize_kv8(_bf16_bits(np.stack([row0, row1])))
    assert list(codes[0, :64]) == list(qa) and list(codes[0, 64:]) == list(qb)
    assert list(scales[0]) == list(_bf16_bits([1 / 8.0, 1 / 32.0]))
    assert list(biases[0]) == list(_bf16_bits([0.0, -4.0]))
    assert codes[1, 1] == 255 and codes[1, 2] == 2 and codes[1, 3] == 2 and codes[1, 0] == 0
    assert scales[1, 1] == 0 and biases[1, 1] == _bf16_bits([1.5])[0]
    assert not codes[1, 64:].any()


def test_kv8_round_trip_bound():
    """Random rows: every value read back is within half a step of the original, plus what
    the bf16 rounding of the scale and bias can add over 255 steps."""
    rng = np.random.default_rng(4)
    x = _bf16_bits(oracle_f32_from_bits(oracle.bf16_round(rng.normal(0, 1.3, (40, 128)))))
    codes, scales, biases = oracle.quantize_kv8(x)
    xf = oracle_f32_from_bits(x).astype(np.float64).reshape(40, 2, 64)
    sc = oracle_f32_from_bits(scales).astype(np.float64)[..., None]
    bi = oracle_f32_from_bits(biases).astype(np.float64)[..., None]
    back = sc * codes.reshape(40, 2, 64) + bi
    mn, mx = xf.min(-1, keepdims=True), xf.max(-1, keepdims=True)
    slack = np.abs(bi - mn) + 255 * np.abs(sc - (mx - mn) / 255)
    assert np.all(np.abs(back - xf) <= sc / 2 + slack + 1e-12)
    assert codes.min() == 0 and codes.max() == 255


def oracle_f32_from_bits(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def _grid_kv(rng, n, hd):
    """bf16 rows whose groups of 64 are exact grids (lossless under 8-bit quantisation)."""
    q = rng.integers(0, 256, (n, hd // 64, 64))
    q[:, :, 0], q[:, :, 1] = 0, 255
    step = 2.0 ** rng.integers(-9, -5, (n, hd // 64, 1))
    return _bf16_bits(((q - 128) * step).reshape(n, hd))


def test_kv8_attention_over_lossless_codes_equals_bf16():
    rng = np.random.default_rng(5)
    for n, hd in ((1, 64), (37, 128)):
        k, v = _grid_kv(rng, n, hd), _grid_kv(rng, n, hd)
        q = rng.normal(0, 1, hd).astype(np.float32)
        got = oracle.attention_kv8(q, oracle.quantize_kv8(k), oracle.quantize_kv8(v))
        np.testing.assert_array_equal(got, oracle.attention(q, k, v))


KV8_SHAPE = ModelShape("kv8-pin", 2, 256, 4, 2, 128, 512, 512, 1e-5, 1e4, gain_sigma=0.1)


def test_kv8_cache_conversion_points():
    """An 8-bit cache's first call (the prompt) runs on bf16 K/V -- its logits equal the bf16
    cache's bit for bit -- and is then converted; a decode step quantises the position it
    appends and reads every position through its codes, so its logits move off the bf16
    cache's by no more than the quantisation error allows, and each position's codes are the
    quantiser's output for that position's bf16 row."""
    m = oracle.OracleModel(KV8_SHAPE)
    rng = np.random.default_rng(6)
    toks = rng.integers(0, KV8_SHAPE.vocab, 21).astype(np.int32)
    c8, c16 = oracle.KVCache(KV8_SHAPE, 32, kv_bits=8), oracle.KVCache(KV8_SHAPE, 32)
    l8 = oracle.prefill_segmented(m, [c8], [20], toks[:20])
    l16 = oracle.prefill_segmented(m, [c16], [20], toks[:20])
    np.testing.assert_array_equal(l8, l16)
    assert c8.qlen == 20 and np.array_equal(c8.k, c16.k) and np.array_equal(c8.v, c16.v)
    d8 = oracle.decode_step_batch(m, [c8], toks[20:21])
    d16 = oracle.decode_step_batch(m, [c16], toks[20:21])
    assert c8.qlen == 21
    assert 0 < np.abs(d8 - d16).max() < 5e-2
    hd = KV8_SHAPE.head_dim
    for name, src in (("k", c8.k), ("v", c8.v)):
        rows = src[:, :, :21, :].reshape(-1, hd)
        codes, scales, biases = oracle.quantize_kv8(rows)
        np.testing.assert_array_equal(c8.q8[name + "q"][:, :, :21, :].reshape(-1, hd), codes)
        np.testing.assert_array_equal(c8.q8[name + "s"][:, :, :21, :].reshape(-1, hd // 64), scales)
        np.testing.assert_array_equal(c8.q8[name + "b"][:, :, :21, :].reshape(-1, hd // 64), biases)


def test_kv8_decode_over_a_lossless_prefix():
    """A cache whose prompt K/V are exact grids loses nothing in its conversion; a decode step
    over it differs from the bf16 cache's only through the appended position's rounding, and
    planting a different code at one prompt position changes the result."""
    m = oracle.OracleModel(KV8_SHAPE)
    rng = np.random.default_rng(7)
    s = KV8_SHAPE
    c8, c16 = oracle.KVCache(s, 16, kv_bits=8), oracle.KVCache(s, 16)
    for c in (c8, c16):
        r = np.random.default_rng(8)
        for arr in (c.k, c.v):
            arr[:, :, :12, :] = _grid_kv(r, s.n_layers * s.n_kv_heads * 12, s.head_dim).reshape(
                s.n_layers, s.n_kv_heads, 12, s.head_dim)
        c.len = 12
    c8.convert()
    tok = rng.integers(0, s.vocab, 1).astype(np.int32)
    d8 = oracle.decode_step_batch(m, [c8], tok)
    d16 = oracle.decode_step_batch(m, [c16], tok)
    assert np.abs(d8 - d16).max() < 5e-2
    c8b = oracle.KVCache(s, 16, kv_bits=8)
    c8b.k[:], c8b.v[:] = c8.k, c8.v
    c8b.len = 12
    c8b.convert()
    c8b.q8["kq"][1, 0, 3, 7] ^= 0x40
    c8b.len, c8b.qlen = 12, 12
    assert not np.array_equal(oracle.decode_step_batch(m, [c8b], tok), d8)


# ---- 4-bit affine KV (the batching design's "--kv-quant 4|8": groups of 64 along head_dim) ------
def test_kv4_hand_example_and_nibble_order():
    """Groups on exact 16-level grids quantise losslessly: [0, 15/4] has scale 1/4 and bias 0,
    [-2, -2 + 15/8] scale 1/8 and bias -2, every code the grid index.  Element 2i sits in the
    low nibble of byte i, 2i + 1 in its high nibble.  A value halfway between steps rounds to
    the even code (1.5 -> 2, 2.5 -> 2); a constant group has scale 0 and all codes 0."""
    rng = np.random.default_rng(13)
    qa = rng.integers(0, 16, 64)
    qa[3], qa[50] = 0, 15
    qb = rng.integers(0, 16, 64)
    qb[0], qb[63] = 15, 0
    row0 = np.concatenate([qa / 4.0, -2.0 + qb / 8.0])
    ties = np.zeros(64)
    ties[1], ties[2], ties[3] = 15 / 4.0, 1.5 / 4.0, 2.5 / 4.0
    row1 = np.concatenate([ties, np.full(64, -0.75)])
    codes, scales, biases = oracle.quantize_kv(_bf16_bits(np.stack([row0, row1])), 4)
    assert codes.shape == (2, 64)
    q0 = np.concatenate([qa, qb])
    assert list(codes[0]) == [int(q0[2 * i]) | (int(q0[2 * i + 1]) << 4) for i in range(64)]
    assert list(scales[0]) == list(_bf16_bits([1 / 4.0, 1 / 8.0]))
    assert list(biases[0]) == list(_bf16_bits([0.0, -2.0]))
    # codes of row 1, group 0: element 1 -> 15, 2 -> 2, 3 -> 2 (bytes 0 and 1)
    assert codes[1, 0] == (0 | (15 << 4)) and codes[1, 1] == (2 | (2 << 4))
    assert scales[1, 1] == 0 and biases[1, 1] == _bf16_bits([-0.75])[0]
    assert not codes[1, 32:].any()


def test_kv4_round_trip_bound():
    rng = np.random.default_rng(14)
    x = _bf16_bits(oracle_f32_from_bits(oracle.bf16_round(rng.normal(0, 1.3, (40, 128)))))
    codes, scales, biases = oracle.quantize_kv(x, 4)
    q = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(40, 128).astype(np.float64)
    xf = oracle_f32_from_bits(x).astype(np.float64).reshape(40, 2, 64)
    sc = oracle_f32_from_bits(scales).astype(np.float64)[..., None]
    bi = oracle_f32_from_bits(biases).astype(np.float64)[..., None]
    back = sc * q.reshape(40, 2, 64) + bi
    mn, mx = xf.min(-1, keepdims=True), xf.max(-1, keepdims=True)
    slack = np.abs(bi - mn) + 15 * np.abs(sc - (mx - mn) / 15)
    assert np.all(np.abs(back - xf) <= sc / 2 + slack + 1e-12)
    assert q.min() == 0 and q.max() == 15
    # the 8-bit quantiser on the same rows is the kv8 format, unchanged
    c8 = oracle.quantize_kv(x, 8)
    for a, b in zip(c8, oracle.quantize_kv8(x)):
        assert np.array_equal(a, b)


def _grid_kv4(rng, n, hd):
    """bf16 rows whose groups of 64 are exact 16-level grids (lossless at 4 bits)."""
    q = rng.integers(0, 16, (n, hd // 64, 64))
    q[:, :, 0], q[:, :, 1] = 0, 15
    step = 2.0 ** rng.integers(-5, -1, (n, hd // 64, 1))
    return _bf16_bits(((q - 8) * step).reshape(n, hd))


def test_kv4_attention_over_lossless_codes_equals_bf16():
    rng = np.random.default_rng(15)
    for n, hd in ((1, 64), (29, 128)):
        k, v = _grid_kv4(rng, n, hd), _grid_kv4(rng, n, hd)
        q = rng.normal(0, 1, hd).astype(np.float32)
        got = oracle.attention_kvq(q, oracle.quantize_kv(k, 4), oracle.quantize_kv(v, 4), 4)
        np.testing.assert_array_equal(got, oracle.attention(q, k, v))


def test_kv4_cache_conversion_points():
    """As for 8 bits: the prompt runs on bf16 K/V (logits equal the bf16 cache's bit for bit),
    the cache is then converted, a decode step quantises what it appends, and the codes of
    every position are the 4-bit quantiser's output for its bf16 row; over a lossless prefix a
    decode step differs from the bf16 cache's only through the appended position."""
    m = oracle.OracleModel(KV8_SHAPE)
    rng = np.random.default_rng(16)
    toks = rng.integers(0, KV8_SHAPE.vocab, 21).astype(np.int32)
    c4, c16 = oracle.KVCache(KV8_SHAPE, 32, kv_bits=4), oracle.KVCache(KV8_SHAPE, 32)
    np.testing.assert_array_equal(oracle.prefill_segmented(m, [c4], [20], toks[:20]),
                                  oracle.prefill_segmented(m, [c16], [20], toks[:20]))
    assert c4.qlen == 20
    d4 = oracle.decode_step_batch(m, [c4], toks[20:21])
    d16 = oracle.decode_step_batch(m, [c16], toks[20:21])
    assert c4.qlen == 21 and np.abs(d4 - d16).max() > 0
    hd = KV8_SHAPE.head_dim
    for name, src in (("k", c4.k), ("v", c4.v)):
        codes, scales, biases = oracle.quantize_kv(src[:, :, :21, :].reshape(-1, hd), 4)
        np.testing.assert_array_equal(c4.q8[name + "q"][:, :, :21, :].reshape(-1, hd // 2), codes)
        np.testing.assert_array_equal(c4.q8[name + "s"][:, :, :21, :].reshape(-1, hd // 64), scales)
        np.testing.assert_array_equal(c4.q8[name + "b"][:, :, :21, :].reshape(-1, hd // 64), biases)
    s = KV8_SHAPE
    g4, g16 = oracle.KVCache(s, 16, kv_bits=4), oracle.KVCache(s, 16)
    for c in (g4, g16):
        r = np.random.default_rng(17)
        for arr in (c.k, c.v):
            arr[:, :, :12, :] = _grid_kv4(r, s.n_layers * s.n_kv_heads * 12, s.head_dim).reshape(
                s.n_layers, s.n_kv_heads, 12, s.head_dim)
        c.len = 12
    g4.convert()
    tok = toks[:1]
    assert np.abs(oracle.decode_step_batch(m, [g4], tok) - oracle.decode_step_batch(m, [g16], tok)).max() < 0.25


def test_kvq_export_value_hand_example():
    """Export of a quantised position: scale * code + bias in double, to fp32, to bf16.
    scale 1/8, bias -4, code 37: -4 + 37/8 = 0.625 exactly.  scale 1.5 * 2^-7, bias 1, code
    255: 1 + 255 * 0.01171875 = 3.98828125; bf16 steps are 2^-6 in [2, 4), and 3.98828125 is
    255.25 steps, so it rounds to 255 steps = 3.984375."""
    L = oracle.lib()
    b = lambda v: int(_bf16_bits([v])[0])
    assert L.orc_kvq_export_value(b(1 / 8.0), b(-4.0), 37) == b(0.625)
    assert L.orc_kvq_export_value(b(1.5 * 2 ** -7), b(1.0), 255) == b(3.984375)
    # the Python helper unpacks 4-bit codes in the stated nibble order
    codes = np.array([[0x21] + [0] * 31], dtype=np.uint8)
    sc = np.array([[b(1.0)]], dtype=np.uint16)
    bi = np.array([[b(0.0)]], dtype=np.uint16)
    vals = oracle.kvq_export_values(codes, sc, bi, 4)
    assert vals[0, 0] == b(1.0) and vals[0, 1] == b(2.0) and not vals[0, 2:].any()
