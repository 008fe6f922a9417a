"""cbt_greedy_head_noalloc: the decode step's final RMSNorm + lm_head + greedy argmax for
callers that cannot allocate device memory (code that runs inside another allocator, or
that may only use buffers planned in advance).  Its scratch is a fixed array inside the
library, so it must give what decode_step_batch gives for the same hidden states.

To know the hidden states decode_step_batch ends with, the model here has all-zero layer
weights: attention and the FFN then add exactly zero, so the residual stream after the last
layer is the embedding row of each token.  Kept in its own file, collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from continuous_batching_transformer_gb300 import binding as B
from continuous_batching_transformer_gb300.model import config_struct
from synth.recipes import TINY
from tests.gpu_harness import TOL, ensure_built

pytestmark = pytest.mark.gpu


def zero_layer_model(dev):
    s = TINY
    d, V = s.d_model, s.vocab
    keep = []

    def t(shape, dtype=torch.bfloat16, fill=None):
        x = torch.zeros(shape, dtype=dtype, device=dev) if fill is None else torch.full(shape, fill, dtype=dtype, device=dev)
        keep.append(x)
        return x

    embed = t((V, d))
    synth.dev_normal_bf16(embed.data_ptr(), V * d, 11, synth.stream_weight(-1, synth.EMBED))
    lm = t((V, d))
    synth.dev_normal_bf16(lm.data_ptr(), V * d, 11, synth.stream_weight(-1, synth.LM_HEAD))
    fnorm = t((d,))
    synth.dev_normal_bf16(fnorm.data_ptr(), d, 11, synth.stream_weight(-1, synth.FINAL_NORM),
                          mean=1.0, sigma=0.1)
    layers = (B.LayerWeights * s.n_layers)()
    for l in range(s.n_layers):
        z = lambda r, c: B.Linear(t((r, c)).data_ptr(), None, None)
        layers[l] = B.LayerWeights(z(s.q_dim + 2 * s.kv_dim, d), z(d, s.q_dim), z(2 * s.d_ff, d),
                                   z(d, s.d_ff), t((d,), fill=1.0).data_ptr(), t((d,), fill=1.0).data_ptr())
    lm_lin = B.Linear(lm.data_ptr(), None, None)
    w = B.Weights(embed.data_ptr(), lm_lin, fnorm.data_ptr(),
                  ctypes.cast(layers, ctypes.POINTER(B.LayerWeights)))
    torch.cuda.synchronize()
    return w, layers, embed, fnorm, lm_lin, keep


def test_noalloc_head_matches_decode_step():
    ensure_built()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    cfg = config_struct(TINY)
    w, layers, embed, fnorm, lm_lin, keep = zero_layer_model(dev)
    arena = torch.empty(B.slab_bytes(cfg, 64) * 8, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    eng = B.engine_create(cfg, w, B.EngineParams(arena.data_ptr(), arena.numel(), 8, 64,
                                                 stream.cuda_stream))
    slabs = [B.kv_slab_alloc(eng, 64) for _ in range(5)]
    toks = torch.tensor([3, 1000, 17, 512, 3], dtype=torch.int32, device=dev)
    ref_logits = torch.empty((5, TINY.vocab), dtype=torch.float32, device=dev)
    ref_next = torch.empty(5, dtype=torch.int32, device=dev)
    B.decode_step_batch(eng, slabs, toks.data_ptr(), ref_logits.data_ptr(), ref_next.data_ptr())
    assert B.last_device_error(eng) == (0, 0)

    hidden = embed[toks.long()].float().contiguous()
    outs = []
    for call in range(2):  # two calls in a row share (and overwrite) the fixed scratch
        lg = torch.full((5, TINY.vocab), float("nan"), dtype=torch.float32, device=dev)
        nx = torch.full((5,), -1, dtype=torch.int32, device=dev)
        B.greedy_head_noalloc(cfg, hidden.data_ptr(), 5, fnorm.data_ptr(), lm_lin, lg.data_ptr(),
                              nx.data_ptr(), stream.cuda_stream)
        stream.synchronize()
        err = (lg - ref_logits).abs().max().item()
        assert err <= TOL["bf16"], f"call {call}: max |noalloc - decode_step_batch| = {err}"
        assert torch.equal(nx, ref_next), (nx, ref_next)
        outs.append(lg.clone())
    assert torch.equal(outs[0], outs[1])
    B.engine_destroy(eng)


def oracle_head(hidden, fnorm, lm_bf16, fmt):
    """The oracle's final RMSNorm, lm_head projection and greedy argmax of each row."""
    g = fnorm.view(torch.int16).cpu().numpy().view(np.uint16)
    w = lm_bf16.view(torch.int16).cpu().numpy().view(np.uint16)
    h = np.stack([oracle.rmsnorm(r, g, TINY.rms_eps) for r in hidden.cpu().numpy()])
    logits = oracle.project(oracle.LinearW(w, fmt, 64), h)
    return logits, np.array([oracle.argmax(r) for r in logits], dtype=np.int32)


@pytest.mark.parametrize("fmt", ["bf16", "affine4"])
def test_noalloc_head_matches_oracle(fmt):
    """The head on its own against the oracle's RMSNorm + lm_head + argmax, bf16 weights and
    4-bit affine weights (quantised on the device by cbt_quantize_affine4; the oracle quantises
    the same bf16 values with its own quantiser), two calls in a row."""
    ensure_built()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    cfg = config_struct(TINY)
    d, V, n = TINY.d_model, TINY.vocab, 7
    lm = torch.empty((V, d), dtype=torch.bfloat16, device=dev)
    synth.dev_normal_bf16(lm.data_ptr(), V * d, 13, synth.stream_weight(-1, synth.LM_HEAD))
    fnorm = torch.empty(d, dtype=torch.bfloat16, device=dev)
    synth.dev_normal_bf16(fnorm.data_ptr(), d, 13, synth.stream_weight(-1, synth.FINAL_NORM),
                          mean=1.0, sigma=0.1)
    hid = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
    synth.dev_normal_bf16(hid.data_ptr(), n * d, 13, synth.stream_weight(-1, synth.EMBED), sigma=1.0)
    hidden = hid.float().contiguous()
    keep = []
    if fmt == "bf16":
        lin = B.Linear(lm.data_ptr(), None, None)
    else:
        cfg.weight_format = B.WEIGHTS_AFFINE4
        packed = torch.empty((V, d // 8), dtype=torch.int32, device=dev)
        sc = torch.empty((V, d // 64), dtype=torch.bfloat16, device=dev)
        bi = torch.empty_like(sc)
        B.quantize_affine4(lm.data_ptr(), V, d, 64, packed.data_ptr(), sc.data_ptr(),
                           bi.data_ptr(), stream.cuda_stream)
        keep += [packed, sc, bi]
        lin = B.Linear(packed.data_ptr(), sc.data_ptr(), bi.data_ptr())
    torch.cuda.synchronize()
    ref_logits, ref_next = oracle_head(hidden, fnorm, lm, fmt)
    for call in range(2):
        lg = torch.full((n, V), float("nan"), dtype=torch.float32, device=dev)
        nx = torch.full((n,), -1, dtype=torch.int32, device=dev)
        B.greedy_head_noalloc(cfg, hidden.data_ptr(), n, fnorm.data_ptr(), lin, lg.data_ptr(),
                              nx.data_ptr(), stream.cuda_stream)
        stream.synchronize()
        got = lg.cpu().numpy()
        err = float(np.abs(got - ref_logits).max())
        assert err <= TOL[fmt], f"{fmt} call {call}: max |noalloc - oracle| = {err}"
        for r in range(n):  # greedy tokens equal, except at a near-tie within the tolerance
            g, o = int(nx[r]), int(ref_next[r])
            if g != o:
                assert ref_logits[r][o] - ref_logits[r][g] < TOL[fmt], (fmt, call, r, g, o)


def test_noalloc_head_rejects_sizes_above_its_scratch():
    ensure_built()
    dev = torch.device("cuda:0")
    cfg = config_struct(TINY)
    dummy = torch.zeros(16, device=dev)
    lin = B.Linear(dummy.data_ptr(), None, None)
    p = dummy.data_ptr()
    with pytest.raises(B.CbtError) as e:
        B.greedy_head_noalloc(cfg, p, B.NOALLOC_MAX_ROWS + 1, p, lin, p, p)
    assert e.value.status == -12
    big = config_struct(TINY)
    big.vocab = 1 << 20  # 32 rows x 1M logits of partial sums do not fit
    with pytest.raises(B.CbtError) as e:
        B.greedy_head_noalloc(big, p, 32, p, lin, p, p)
    assert e.value.status == -12
    B.greedy_head_noalloc(cfg, p, 0, p, lin, p, p)  # n == 0: nothing to do
