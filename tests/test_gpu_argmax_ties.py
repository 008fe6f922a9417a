"""Greedy sampling with exact ties on the GPU: the lowest vocabulary id wins (mlx-bun batching
design, its campaign note on tied candidate scores).

Exact ties are planted by construction: the layers' weights are all zero (attention and the
FFN then add exactly zero, so the hidden state after the last layer is the token's embedding
row) and the lm_head repeats seven distinct rows in a scrambled order, row r being pattern
(3 r + 5) mod 7.  Rows with the same pattern get bit-identical logits, so the maximum of a
logits row is shared by every id of its pattern and the greedy token must be the smallest of
them.  Checked through decode_step_batch (tensor-core projection + argmax kernel), segmented
prefill, and the no-allocation head (CUDA-core projection + the same argmax kernel)."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from continuous_batching_transformer_gb300 import binding as B
from continuous_batching_transformer_gb300.model import config_struct
from synth.recipes import TINY
from tests.gpu_harness import ensure_built

pytestmark = pytest.mark.gpu

N_PATTERNS = 7


def pattern(r):
    return (3 * r + 5) % N_PATTERNS


def tied_model(dev):
    s = TINY
    d, V = s.d_model, s.vocab
    keep = []

    def t(shape, fill=None):
        x = torch.zeros(shape, dtype=torch.bfloat16, device=dev) if fill is None \
            else torch.full(shape, fill, dtype=torch.bfloat16, device=dev)
        keep.append(x)
        return x

    embed = t((V, d))
    synth.dev_normal_bf16(embed.data_ptr(), V * d, 21, synth.stream_weight(-1, synth.EMBED))
    base = t((N_PATTERNS, d))
    synth.dev_normal_bf16(base.data_ptr(), N_PATTERNS * d, 21, synth.stream_weight(-1, synth.LM_HEAD))
    idx = torch.tensor([pattern(r) for r in range(V)], dtype=torch.long, device=dev)
    lm = base[idx].contiguous()
    keep.append(lm)
    fnorm = t((d,))
    synth.dev_normal_bf16(fnorm.data_ptr(), d, 21, synth.stream_weight(-1, synth.FINAL_NORM),
                          mean=1.0, sigma=0.1)
    layers = (B.LayerWeights * s.n_layers)()
    for l in range(s.n_layers):
        z = lambda r, c: B.Linear(t((r, c)).data_ptr(), None, None)
        layers[l] = B.LayerWeights(z(s.q_dim + 2 * s.kv_dim, d), z(d, s.q_dim), z(2 * s.d_ff, d),
                                   z(d, s.d_ff), t((d,), fill=1.0).data_ptr(),
                                   t((d,), fill=1.0).data_ptr())
    lm_lin = B.Linear(lm.data_ptr(), None, None)
    w = B.Weights(embed.data_ptr(), lm_lin, fnorm.data_ptr(),
                  ctypes.cast(layers, ctypes.POINTER(B.LayerWeights)))
    torch.cuda.synchronize()
    return w, layers, embed, fnorm, lm_lin, keep


def check_ties(logits: np.ndarray, nxt: np.ndarray, what: str):
    pats = np.array([pattern(r) for r in range(logits.shape[1])])
    for b in range(logits.shape[0]):
        row = logits[b]
        for p in range(N_PATTERNS):  # the construction gives bit-identical ties
            vals = row[pats == p]
            assert np.all(vals.view(np.uint32) == vals[0].view(np.uint32)), f"{what}: pattern {p}"
        top = row.max()
        tied = np.flatnonzero(row == top)
        assert len(tied) > 1, f"{what}: row {b} has no tie at its maximum"
        assert int(nxt[b]) == int(tied[0]), f"{what}: row {b} chose {int(nxt[b])}, not {tied[0]}"


def test_greedy_ties_take_the_lowest_id():
    ensure_built()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    cfg = config_struct(TINY)
    w, layers, embed, fnorm, lm_lin, keep = tied_model(dev)
    arena = torch.empty(B.slab_bytes(cfg, 64) * 16, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    eng = B.engine_create(cfg, w, B.EngineParams(arena.data_ptr(), arena.numel(), 12, 64,
                                                 stream.cuda_stream))
    toks = torch.tensor([3, 1000, 17, 512, 3, 77, 640, 999, 0, 5, 250], dtype=torch.int32, device=dev)
    n = toks.numel()
    slabs = [B.kv_slab_alloc(eng, 64) for _ in range(n)]
    lg = torch.empty((n, TINY.vocab), dtype=torch.float32, device=dev)
    nx = torch.full((n,), -1, dtype=torch.int32, device=dev)
    # decode: the tensor-core projection and the argmax kernel
    B.decode_step_batch(eng, slabs, toks.data_ptr(), lg.data_ptr(), nx.data_ptr())
    stream.synchronize()
    check_ties(lg.cpu().numpy(), nx.cpu().numpy(), "decode_step_batch")
    # segmented prefill of one-token segments into fresh slabs
    fresh = [B.kv_slab_alloc(eng, 64) for _ in range(4)]
    nx4 = torch.full((4,), -1, dtype=torch.int32, device=dev)
    lg4 = torch.empty((4, TINY.vocab), dtype=torch.float32, device=dev)
    B.prefill_segmented(eng, fresh, [1, 1, 1, 1], toks[:4].data_ptr(), lg4.data_ptr(), nx4.data_ptr())
    stream.synchronize()
    check_ties(lg4.cpu().numpy(), nx4.cpu().numpy(), "prefill_segmented")
    assert B.last_device_error(eng) == (0, 0)
    B.engine_destroy(eng)
    # the no-allocation head on the same hidden states (the embedding rows)
    hidden = embed[toks.long()].float().contiguous()
    lg2 = torch.empty((n, TINY.vocab), dtype=torch.float32, device=dev)
    nx2 = torch.full((n,), -1, dtype=torch.int32, device=dev)
    B.greedy_head_noalloc(cfg, hidden.data_ptr(), n, fnorm.data_ptr(), lm_lin, lg2.data_ptr(),
                          nx2.data_ptr(), stream.cuda_stream)
    stream.synchronize()
    check_ties(lg2.cpu().numpy(), nx2.cpu().numpy(), "greedy_head_noalloc")
