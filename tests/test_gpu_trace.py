"""Continuous batching over a small request trace on the tiny decoder: requests are admitted
by segmented prefill at step boundaries, share decode steps with whatever else is live, and
leave when done.  Each request's greedy tokens must equal the oracle's for that request alone
(prefill of its prompt, then greedy decode); where they differ, the oracle's top two logits
must be within the bf16 tolerance (a near-tie), after which the trajectories may part."""
import numpy as np
import pytest
import torch

import oracle
from continuous_batching_transformer_gb300.model import DeviceWeights, Engine
from continuous_batching_transformer_gb300.trace import prompt_tokens, run_trace
from synth.recipes import TINY, Request, agent_requests
from tests.gpu_harness import TOL, ensure_built

pytestmark = pytest.mark.gpu

# (arrival, prompt length, output length, token stream): more requests than batch slots, so
# rows join and leave mid-trace; one request ends on its prefill token
REQS = [Request(0.0, 5, 4, 11), Request(0.0, 17, 7, 12), Request(0.0, 32, 2, 13),
        Request(0.0, 9, 9, 14), Request(0.0, 24, 5, 15), Request(0.0, 3, 1, 16),
        Request(0.0, 12, 6, 17)]


def oracle_greedy(om, req, seed):
    toks = prompt_tokens(req, seed, TINY.vocab)
    cache = oracle.KVCache(TINY, req.prompt_len + req.output_len + 2)
    ref = oracle.prefill_segmented(om, [cache], [req.prompt_len], toks)
    logits = [ref[0]]
    out = [oracle.argmax(ref[0])]
    while len(out) < req.output_len:
        r = oracle.decode_step_batch(om, [cache], np.array([out[-1]], dtype=np.int32))
        logits.append(r[0])
        out.append(oracle.argmax(r[0]))
    return out, logits


@pytest.mark.parametrize("chunk", [None, 16])
def test_trace_rows_match_oracle(chunk):
    """chunk None: whole prompts per admission; 16: prompts admitted 16 tokens per call, one
    decode step between chunks (the 17- to 32-token prompts take two or three calls)."""
    ensure_built()
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    om = oracle.OracleModel(TINY)
    eng = Engine(w, arena_bytes=32 << 20, max_batch=3, max_prefill_tokens=64)
    res = run_trace(eng, REQS, seed=0, live_cap=3, record_tokens=True, chunk_tokens=chunk)
    assert eng.device_error() == (0, 0)
    assert res.generated == sum(r.output_len for r in REQS)
    assert eng.stats().live_slabs == 0  # every request's slab was retired
    assert max(res.step_rows) == 3 and min(res.step_rows) >= 1
    for i, req in enumerate(REQS):
        got = res.tokens[i]
        assert len(got) == req.output_len
        want, logits = oracle_greedy(om, req, 0)
        for t, (g, wv) in enumerate(zip(got, want)):
            if g != wv:
                top2 = np.sort(logits[t])[-2:]
                assert top2[1] - top2[0] < TOL["bf16"], f"request {i} token {t}: {g} != {wv}"
                break
    eng.close()


@pytest.mark.parametrize("chunk,mode", [(None, True), (8, True), (None, "share"), (8, "share")])
def test_shared_prefix_trace_matches_oracle(chunk, mode):
    """Sub-agents sharing a 20-token system prompt, with prefix reuse: the prompt is prefilled
    once and copied into each request's slab (or, on a paged engine, its page shared), so a
    request prefills only its own tokens.  Each request's greedy tokens against the oracle's
    for its whole prompt."""
    ensure_built()
    dev = torch.device("cuda:0")
    w = DeviceWeights(TINY, dev)
    om = oracle.OracleModel(TINY)
    reqs = agent_requests(5, 20, 3, 12, 4.0, 7, seed=3)
    eng = Engine(w, arena_bytes=32 << 20, max_batch=3, max_prefill_tokens=64,
                 page_tokens=128 if mode == "share" else 0)
    res = run_trace(eng, reqs, seed=0, live_cap=3, record_tokens=True, chunk_tokens=chunk,
                    reuse_prefix=mode)
    assert eng.device_error() == (0, 0)
    assert res.prefill_tokens == 20 + sum(r.prompt_len - 20 for r in reqs)
    assert eng.stats().live_slabs == 0
    for i, req in enumerate(reqs):
        got = res.tokens[i]
        assert len(got) == req.output_len
        want, logits = oracle_greedy(om, req, 0)
        for t, (g, wv) in enumerate(zip(got, want)):
            if g != wv:
                top2 = np.sort(logits[t])[-2:]
                assert top2[1] - top2[0] < TOL["bf16"], f"request {i} token {t}: {g} != {wv}"
                break
    eng.close()
