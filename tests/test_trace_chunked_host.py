"""Host logic of the chunked-admission trace driver, against a fake engine on the CPU: every
prefill call stays within the chunk budget, each segment continues its slab exactly where the
previous chunk stopped, a decode step follows every chunk while rows are live, the live cap
holds, and every request gets exactly its output length."""
from types import SimpleNamespace

import torch

from continuous_batching_transformer_gb300.trace import run_trace
import pytest

from synth.recipes import Request, agent_requests


class FakeEngine:
    def __init__(self, max_batch=3, max_prefill_tokens=64):
        self.weights = SimpleNamespace(device=torch.device("cpu"))
        self.shape = SimpleNamespace(vocab=1000)
        self.stream = SimpleNamespace(synchronize=lambda: None)
        self.max_batch = max_batch
        self.max_prefill_tokens = max_prefill_tokens
        self.pos, self.cap, self.live = {}, {}, set()
        self.calls = []  # ("prefill", [(slab, start, n)]) or ("decode", [slabs])
        self.next_id = 0

    def kv_slab_alloc(self, cap):
        s = self.next_id
        self.next_id += 1
        self.pos[s], self.cap[s] = 0, cap
        self.live.add(s)
        return s

    def retire(self, slabs):
        for s in slabs:
            self.live.remove(s)

    def prefill_segmented(self, slabs, lens, tokens, logits=None, next_tokens=None):
        assert len(set(slabs)) == len(slabs) and sum(lens) == tokens.numel()
        self.calls.append(("prefill", [(s, self.pos[s], n) for s, n in zip(slabs, lens)]))
        for k, (s, n) in enumerate(zip(slabs, lens)):
            assert s in self.live and self.pos[s] + n <= self.cap[s]
            self.pos[s] += n
            if next_tokens is not None:
                next_tokens[k] = s

    def copy_prefix(self, src, dst, n):
        assert src in self.live and dst in self.live and self.pos[src] >= n
        self.calls.append(("copy", (src, dst, n)))
        self.pos[dst] = n

    def share_prefix(self, src, dst, n):
        assert src in self.live and dst in self.live and self.pos[src] >= n and self.pos[dst] == 0
        self.calls.append(("share", (src, dst, n)))
        self.pos[dst] = n

    def decode_step_batch(self, slabs, last_tokens, logits=None, next_tokens=None):
        assert len(slabs) <= self.max_batch and all(s in self.live for s in slabs)
        self.calls.append(("decode", list(slabs)))
        for k, s in enumerate(slabs):
            self.pos[s] += 1
            next_tokens[k] = s


def test_chunked_admission_policy():
    reqs = [Request(0.0, 40, 3, 1), Request(0.0, 7, 1, 2), Request(0.0, 25, 5, 3),
            Request(0.0, 16, 2, 4), Request(0.0, 33, 4, 5)]
    eng = FakeEngine(max_batch=3, max_prefill_tokens=64)
    chunk = 16
    res = run_trace(eng, reqs, seed=0, live_cap=3, chunk_tokens=chunk)
    assert res.generated == sum(r.output_len for r in reqs)
    assert res.prefill_tokens == sum(r.prompt_len for r in reqs)
    assert not eng.live  # every slab retired
    prefilled = {}
    for kind, what in eng.calls:
        if kind == "prefill":
            assert sum(n for _, _, n in what) <= chunk
            for s, start, n in what:
                assert start == prefilled.get(s, 0)  # continues where the last chunk stopped
                prefilled[s] = start + n
    # once rows are decoding, a decode step separates every two chunks (in this trace some row
    # stays live from the first decode step to the last chunk)
    kinds = [k for k, _ in eng.calls]
    first_decode = kinds.index("decode")
    for a, b in zip(kinds[first_decode:], kinds[first_decode + 1:]):
        assert not (a == "prefill" and b == "prefill")
    assert max(res.step_rows) <= 3
    # each request's slab saw exactly its whole prompt
    assert sorted(prefilled.values()) == sorted(r.prompt_len for r in reqs)


@pytest.mark.parametrize("chunk", [None, 16])
@pytest.mark.parametrize("mode", [True, "share"])
def test_shared_prefix_reuse(chunk, mode):
    """Requests sharing a 40-token prefix: with reuse the prefix is prefilled once, every
    request's slab starts from it (a copy, or its pages shared), and only the requests' own
    tokens are prefilled."""
    reqs = agent_requests(6, 40, 3, 20, 3.0, 6, seed=5)
    eng = FakeEngine(max_batch=3, max_prefill_tokens=64)
    res = run_trace(eng, reqs, seed=0, live_cap=3, chunk_tokens=chunk, reuse_prefix=mode)
    own = sum(r.prompt_len - r.prefix_len for r in reqs)
    assert res.prefill_tokens == own + 40
    assert res.generated == sum(r.output_len for r in reqs)
    kind_used = "share" if mode == "share" else "copy"
    assert not any(kind == ("copy" if mode == "share" else "share") for kind, _ in eng.calls)
    copies = [what for kind, what in eng.calls if kind == kind_used]
    assert len(copies) == len(reqs) and all(n == 40 for _, _, n in copies)
    assert len({src for src, _, _ in copies}) == 1     # one prefix slab
    assert not eng.live                                 # it is retired at the end too
    # every prefill of a request's slab starts at or after its copied prefix
    copied = {dst for _, dst, _ in copies}
    for kind, what in eng.calls:
        if kind == "prefill":
            for s, start, n in what:
                assert s not in copied or start >= 40
    plain = FakeEngine(max_batch=3, max_prefill_tokens=64)
    res2 = run_trace(plain, reqs, seed=0, live_cap=3, chunk_tokens=chunk)
    assert res2.prefill_tokens == sum(r.prompt_len for r in reqs)


def test_reuse_mode_checked():
    with pytest.raises(ValueError):
        run_trace(FakeEngine(), agent_requests(2, 40, 3, 20, 3.0, 6, seed=5), seed=0,
                  reuse_prefix="pages")
