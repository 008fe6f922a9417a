"""Full-size parity: the 7B-shaped decoder (32 layers, d_model 4096, 32/8 heads, SwiGLU 14336,
vocab 32000) in the launch configuration bench.py times (bench.setup_decode).  The GPU runs
the whole batch; the oracle recomputes sampled rows one by one (its per-row arithmetic does
not depend on the other rows), over two greedy steps so the K/V appended at t_s is read back."""
import gc

import numpy as np
import pytest
import torch

import bench
import oracle
from synth.recipes import DECODE_7B_B8, LONG_7B_B32, decode_7b_fixed
from tests.gpu_harness import TOL, check_logits, ensure_built, to_dev

pytestmark = pytest.mark.gpu


def run_sampled(wl, rows, tol, page_tokens=0):
    ensure_built()
    dev = torch.device("cuda:0")
    w, eng, slabs, ctx, tok = bench.setup_decode(wl, dev, extra_positions=8,
                                                 page_tokens=page_tokens)
    Bsz, V = len(slabs), wl.shape.vocab
    logits = torch.empty((Bsz, V), dtype=torch.float32, device=dev)
    nxt = torch.empty(Bsz, dtype=torch.int32, device=dev)
    m = oracle.OracleModel(wl.shape)
    caches = []
    for r in rows:
        kc = oracle.KVCache(wl.shape, ctx[r] + 4)
        kc.fill_synthetic(r, ctx[r], wl.seed)
        caches.append(kc)
    feed = tok.cpu().numpy()
    errs = []
    for step in range(2):
        eng.decode_step_batch(slabs, to_dev(feed, dev), logits, nxt)
        ref = oracle.decode_step_batch(m, caches, feed[rows])
        got = logits.cpu().numpy()[rows]
        errs.append(check_logits(got, ref, tol, f"{wl.name} step {step}"))
        feed = nxt.cpu().numpy().copy()
        feed[rows] = [oracle.argmax(r) for r in ref]  # sampled rows follow the oracle
    assert eng.device_error() == (0, 0)
    assert [eng.position(s) for s in slabs] == [c + 2 for c in ctx]
    eng.close()
    del w, m, caches
    gc.collect()
    torch.cuda.empty_cache()
    print(f"{wl.name}: max |logit - oracle| = {max(errs):.3e}")


def test_7b_bf16_b8_ragged_contexts():
    run_sampled(DECODE_7B_B8, [0, 5], TOL["bf16"])


def test_7b_affine4_b4_ctx2048():
    run_sampled(decode_7b_fixed(4, 2048, "affine4"), [0, 3], TOL["affine4"])


def test_7b_bf16_b32_long_contexts():
    """The long-context workload (32 rows of 8k-16k tokens, about 64 GB of KV): the rows
    with the longest and the shortest context, where the split-K attention has the most and
    the fewest partials to merge."""
    ctx = [int(c) for c in LONG_7B_B32.context_lengths()]
    run_sampled(LONG_7B_B32, [int(np.argmax(ctx)), int(np.argmin(ctx))], TOL["bf16"])


def test_7b_affine4_b16_one_pass():
    """4-bit weights at B = 16: the projections take all 16 rows (32 operand columns) in one
    pass over the weights; rows from both halves of the operand."""
    run_sampled(decode_7b_fixed(16, 2048, "affine4"), [0, 9, 15], TOL["affine4"])


def test_7b_affine4_b32_two_passes():
    """4-bit weights at B = 32: two passes of 16 rows over the same weights; rows from both
    passes."""
    run_sampled(decode_7b_fixed(32, 2048, "affine4"), [0, 17, 31], TOL["affine4"])


def test_7b_bf16_b8_paged_kv():
    """The headline workload on a paged engine (pages of 128 positions; the synthetic KV is
    imported page by page)."""
    run_sampled(DECODE_7B_B8, [0, 5], TOL["bf16"], page_tokens=128)
