"""Continuous batching over a request trace, on the engine's public calls only.

Requests arrive over time (``synth.recipes.trace_requests``: Poisson arrivals, ragged prompts,
geometric output lengths).  At every step boundary the driver

1. retires the rows that have produced all their tokens (``retire`` frees their slabs),
2. admits the requests that have arrived, up to ``live_cap`` live rows and the engine's
   prefill token budget, in one ``prefill_segmented`` call (each prompt in its own slab,
   positions restarting at 0; the argmax of each segment's last logits is the request's
   first token),
3. runs one ``decode_step_batch`` over every live row (the previous step's tokens stay on the
   device: the step reads them from and writes the next ones to a device token buffer).

A row that has produced ``output_len`` tokens (the first one from the prefill) leaves at the
next boundary.  Time to first token is measured from the request's arrival to the end of the
prefill that produced it; time per output token is the mean gap between a request's later
tokens.  ``realtime=False`` replays the trace with every request arriving at t = 0 (a
throughput measurement); ``realtime=True`` waits for the arrival times.
"""
from __future__ import annotations

import time
from collections import deque
from dataclasses import dataclass, field

import numpy as np
import torch

import synth


@dataclass
class TraceResult:
    generated: int = 0                                  # tokens produced by every request
    wall_s: float = 0.0
    steps: int = 0                                      # decode steps
    step_rows: list = field(default_factory=list)       # live rows of each decode step
    step_s: list = field(default_factory=list)          # duration of each decode step
    step_start: list = field(default_factory=list)      # its start, seconds from the trace start
    step_reqs: list = field(default_factory=list)       # the request indices it decoded
    step_kv_tokens: list = field(default_factory=list)  # live positions the step's attention read
    prefill_tokens: int = 0
    prefill_s: float = 0.0
    ttft_s: dict = field(default_factory=dict)          # request index -> time to first token
    tpot_s: dict = field(default_factory=dict)          # request index -> time per output token
    tokens: dict = field(default_factory=dict)          # request index -> generated tokens
    kv_bytes_peak: int = 0                              # most KV arena bytes held after a call

    def note_kv(self, eng):
        if hasattr(eng, "stats"):
            self.kv_bytes_peak = max(self.kv_bytes_peak, int(eng.stats().slab_bytes_in_use))


def prompt_tokens(req, seed: int, vocab: int) -> np.ndarray:
    """The request's prompt: its shared prefix (if any), then its own seeded token stream."""
    own = synth.tokens(req.prompt_len - req.prefix_len, seed, synth.stream_tokens(req.row), vocab)
    if not req.prefix_len:
        return own
    pre = synth.tokens(req.prefix_len, seed, synth.stream_tokens(req.prefix_row), vocab)
    return np.concatenate([pre, own])


class SharedPrefixes:
    """Prefix reuse (the batching design: sub-agents share long system prompts and reuse one
    prefill): each shared prefix is prefilled once into a slab of its own, and a request's
    slab starts from it, so only the request's own tokens are prefilled.  `reuse` True or
    "copy": the slab starts as a copy of the prefix (``copy_prefix``); "share": it holds the
    prefix's pages by reference (``share_prefix``: a paged engine copies a page only when a
    slab writes into it, so N requests hold one copy of the prompt).  Without reuse every
    prompt is prefilled whole."""

    def __init__(self, eng, seed: int, res: TraceResult, reuse):
        if reuse not in (False, True, "copy", "share"):
            raise ValueError(f"reuse must be False, True, 'copy' or 'share', not {reuse!r}")
        self.eng, self.seed, self.res, self.reuse = eng, seed, res, reuse
        self.slabs = {}

    def start(self, req, slab) -> int:
        """Prompt tokens already in `slab` (its shared prefix) -- 0 without reuse."""
        if not (self.reuse and req.prefix_len):
            return 0
        if req.prompt_len <= req.prefix_len:
            raise ValueError("a request needs at least one token of its own after the prefix")
        key = (req.prefix_row, req.prefix_len)
        if key not in self.slabs:
            src = self.eng.kv_slab_alloc(req.prefix_len)
            toks = synth.tokens(req.prefix_len, self.seed, synth.stream_tokens(req.prefix_row),
                                self.eng.shape.vocab)
            ta = time.perf_counter()
            self.eng.prefill_segmented([src], [req.prefix_len],
                                       torch.from_numpy(toks).to(self.eng.weights.device))
            self.eng.stream.synchronize()
            self.res.prefill_s += time.perf_counter() - ta
            self.res.prefill_tokens += req.prefix_len
            self.slabs[key] = src
        if self.reuse == "share":
            self.eng.share_prefix(self.slabs[key], slab, req.prefix_len)
        else:
            self.eng.copy_prefix(self.slabs[key], slab, req.prefix_len)
        return req.prefix_len

    def close(self):
        if self.slabs:
            self.eng.retire(list(self.slabs.values()))
        self.slabs = {}


def run_trace(eng, reqs, seed: int, live_cap: int = 8, realtime: bool = False,
              record_tokens: bool = False, max_prefill_tokens: int | None = None,
              slab_margin: int = 8, chunk_tokens: int | None = None,
              reuse_prefix: bool | str = False) -> TraceResult:
    """Serve `reqs` on `eng` (an ``Engine``) with continuous batching; see the module text.
    With `chunk_tokens`, prompts are admitted in chunks instead (``run_trace_chunked``); with
    `reuse_prefix` (True or "copy", or "share"), shared prompt prefixes are prefilled once
    (``SharedPrefixes``)."""
    if chunk_tokens:
        return run_trace_chunked(eng, reqs, seed, chunk_tokens, live_cap, realtime,
                                 record_tokens, slab_margin, reuse_prefix)
    dev = eng.weights.device
    vocab = eng.shape.vocab
    stream = eng.stream
    live_cap = min(live_cap, eng.max_batch)
    budget = max_prefill_tokens or eng.max_prefill_tokens
    order = sorted(range(len(reqs)), key=lambda i: (0.0 if not realtime else reqs[i].arrival_s, i))
    pending = deque(order)
    live = []  # per row: [request index, slab, tokens produced, time of last token]
    res = TraceResult()
    shared = SharedPrefixes(eng, seed, res, reuse_prefix)
    tok = torch.zeros(eng.max_batch, dtype=torch.int32, device=dev)  # the live rows' last tokens
    nxt = torch.zeros(eng.max_batch, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()

    def now() -> float:
        return time.perf_counter() - t0

    def arrived(i) -> bool:
        return not realtime or reqs[i].arrival_s <= now()

    while pending or live:
        # 1. retire finished rows; the others keep their order and their last tokens
        keep = [k for k, r in enumerate(live) if r[2] < reqs[r[0]].output_len]
        if len(keep) < len(live):
            eng.retire([r[1] for k, r in enumerate(live) if r[2] >= reqs[r[0]].output_len])
            if keep:
                tok[:len(keep)] = tok[torch.tensor(keep, dtype=torch.long, device=dev)]
            live = [live[k] for k in keep]
        # 2. admit arrivals
        if realtime and not live and pending and not arrived(pending[0]):
            time.sleep(max(0.0, reqs[pending[0]].arrival_s - now()))
        admit = []
        total = 0

        def to_fill(i):  # prompt tokens a request's admission prefills
            return reqs[i].prompt_len - (reqs[i].prefix_len if reuse_prefix else 0)

        while (pending and len(live) + len(admit) < live_cap and arrived(pending[0])
               and total + to_fill(pending[0]) <= budget):
            i = pending.popleft()
            admit.append(i)
            total += to_fill(i)
        if admit:
            slabs = [eng.kv_slab_alloc(reqs[i].prompt_len + reqs[i].output_len + slab_margin)
                     for i in admit]
            done = [shared.start(reqs[i], s) for i, s in zip(admit, slabs)]
            host = np.concatenate([prompt_tokens(reqs[i], seed, vocab)[d:]
                                   for i, d in zip(admit, done)])
            dtok = torch.from_numpy(host.astype(np.int32)).to(dev, non_blocking=False)
            first = torch.empty(len(admit), dtype=torch.int32, device=dev)
            ta = time.perf_counter()
            eng.prefill_segmented(slabs, [reqs[i].prompt_len - d for i, d in zip(admit, done)],
                                  dtok, None, first)
            stream.synchronize()
            tb = time.perf_counter()
            res.prefill_tokens += total
            res.prefill_s += tb - ta
            res.note_kv(eng)
            firsts = first.cpu().tolist() if record_tokens else None
            # the new rows join the live set; their first token is the next step's input
            rows_before = len(live)
            for k, i in enumerate(admit):
                live.append([i, slabs[k], 1, tb - t0])
                res.ttft_s[i] = (tb - t0) - (reqs[i].arrival_s if realtime else 0.0)
                res.generated += 1
                if record_tokens:
                    res.tokens[i] = [firsts[k]]
            tok[rows_before:rows_before + len(admit)] = first
            continue  # a boundary again: new rows may already be complete (output_len 1)
        if not live:
            continue
        # 3. one decode step over the live rows
        B = len(live)
        ta = time.perf_counter()
        eng.decode_step_batch([r[1] for r in live], tok[:B], None, nxt[:B])
        stream.synchronize()
        tb = time.perf_counter()
        res.steps += 1
        res.note_kv(eng)
        res.step_rows.append(B)
        res.step_s.append(tb - ta)
        res.step_start.append(ta - t0)
        res.step_reqs.append(tuple(r[0] for r in live))
        # row r reads positions [0, prompt + produced] (the new token is appended first)
        res.step_kv_tokens.append(sum(reqs[r[0]].prompt_len + r[2] for r in live))
        step_tokens = nxt[:B].cpu().tolist() if record_tokens else None
        for k, r in enumerate(live):
            r[2] += 1
            res.generated += 1
            if record_tokens:
                res.tokens[r[0]].append(step_tokens[k])
            if r[2] >= reqs[r[0]].output_len:
                n = reqs[r[0]].output_len
                first_t = res.ttft_s[r[0]] + (reqs[r[0]].arrival_s if realtime else 0.0)
                res.tpot_s[r[0]] = ((tb - t0) - first_t) / max(1, n - 1)
        # the next step's inputs are this step's outputs, row for row (finished rows leave at
        # the boundary)
        tok[:B] = nxt[:B]
    shared.close()
    res.wall_s = now()
    return res


def run_trace_chunked(eng, reqs, seed: int, chunk_tokens: int, live_cap: int = 8,
                      realtime: bool = False, record_tokens: bool = False,
                      slab_margin: int = 8, reuse_prefix: bool | str = False) -> TraceResult:
    """Continuous batching with chunked admission (the batching design's joiner prefill: one
    chunk per scheduler iteration, one decode step between chunks, so a running row waits at
    most one chunk for each joiner).  At every boundary the driver

    1. retires finished rows,
    2. opens a slab for each arrived request while live + joining rows stay within
       ``live_cap``,
    3. prefills one chunk of at most ``chunk_tokens`` prompt tokens in one
       ``prefill_segmented`` call, taken from the joining rows in arrival order (each segment
       continues its slab where the previous chunk stopped); a row whose prompt is complete
       takes the argmax of its last logits as its first token and joins the live rows,
    4. runs one ``decode_step_batch`` over the live rows.

    Time to first token ends with the chunk that completes the prompt."""
    dev = eng.weights.device
    vocab = eng.shape.vocab
    stream = eng.stream
    live_cap = min(live_cap, eng.max_batch)
    chunk_tokens = min(chunk_tokens, eng.max_prefill_tokens)
    order = sorted(range(len(reqs)), key=lambda i: (0.0 if not realtime else reqs[i].arrival_s, i))
    pending = deque(order)
    joining = []  # per row: [request index, slab, prompt tokens prefilled]
    live = []     # per row: [request index, slab, tokens produced, time of last token]
    prompts = {}
    res = TraceResult()
    shared = SharedPrefixes(eng, seed, res, reuse_prefix)
    tok = torch.zeros(eng.max_batch, dtype=torch.int32, device=dev)
    nxt = torch.zeros(eng.max_batch, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()

    def now() -> float:
        return time.perf_counter() - t0

    def arrived(i) -> bool:
        return not realtime or reqs[i].arrival_s <= now()

    def retire_done():
        nonlocal live
        keep = [k for k, r in enumerate(live) if r[2] < reqs[r[0]].output_len]
        if len(keep) < len(live):
            eng.retire([r[1] for k, r in enumerate(live) if r[2] >= reqs[r[0]].output_len])
            if keep:
                tok[:len(keep)] = tok[torch.tensor(keep, dtype=torch.long, device=dev)]
            live = [live[k] for k in keep]

    while pending or live or joining:
        retire_done()
        if realtime and not live and not joining and pending and not arrived(pending[0]):
            time.sleep(max(0.0, reqs[pending[0]].arrival_s - now()))
        while pending and len(live) + len(joining) < live_cap and arrived(pending[0]):
            i = pending.popleft()
            slab = eng.kv_slab_alloc(reqs[i].prompt_len + reqs[i].output_len + slab_margin)
            joining.append([i, slab, shared.start(reqs[i], slab)])
            prompts[i] = prompt_tokens(reqs[i], seed, vocab)
        if joining:
            segs, left = [], chunk_tokens
            for row in joining:
                if left == 0:
                    break
                n = min(reqs[row[0]].prompt_len - row[2], left)
                segs.append((row, row[2], row[2] + n))
                left -= n
            host = np.concatenate([prompts[row[0]][a:b] for row, a, b in segs])
            dtok = torch.from_numpy(host.astype(np.int32)).to(dev, non_blocking=False)
            first = torch.empty(len(segs), dtype=torch.int32, device=dev)
            ta = time.perf_counter()
            eng.prefill_segmented([row[1] for row, _, _ in segs], [b - a for _, a, b in segs],
                                  dtok, None, first)
            stream.synchronize()
            tb = time.perf_counter()
            res.prefill_tokens += len(host)
            res.prefill_s += tb - ta
            res.note_kv(eng)
            done = [k for k, (row, _, b) in enumerate(segs) if b == reqs[row[0]].prompt_len]
            firsts = first.cpu().tolist() if (record_tokens and done) else None
            rows_before = len(live)
            for row, _, b in segs:
                row[2] = b
            for k in done:
                i, slab = segs[k][0][0], segs[k][0][1]
                live.append([i, slab, 1, tb - t0])
                res.ttft_s[i] = (tb - t0) - (reqs[i].arrival_s if realtime else 0.0)
                res.generated += 1
                if record_tokens:
                    res.tokens[i] = [firsts[k]]
            if done:
                idx = torch.tensor(done, dtype=torch.long, device=dev)
                tok[rows_before:rows_before + len(done)] = first[idx]
            joining = [row for row in joining if row[2] < reqs[row[0]].prompt_len]
            retire_done()  # rows complete on their first token leave before the step
        if not live:
            continue
        B = len(live)
        ta = time.perf_counter()
        eng.decode_step_batch([r[1] for r in live], tok[:B], None, nxt[:B])
        stream.synchronize()
        tb = time.perf_counter()
        res.steps += 1
        res.note_kv(eng)
        res.step_rows.append(B)
        res.step_s.append(tb - ta)
        res.step_start.append(ta - t0)
        res.step_reqs.append(tuple(r[0] for r in live))
        res.step_kv_tokens.append(sum(reqs[r[0]].prompt_len + r[2] for r in live))
        step_tokens = nxt[:B].cpu().tolist() if record_tokens else None
        for k, r in enumerate(live):
            r[2] += 1
            res.generated += 1
            if record_tokens:
                res.tokens[r[0]].append(step_tokens[k])
            if r[2] >= reqs[r[0]].output_len:
                n = reqs[r[0]].output_len
                first_t = res.ttft_s[r[0]] + (reqs[r[0]].arrival_s if realtime else 0.0)
                res.tpot_s[r[0]] = ((tb - t0) - first_t) / max(1, n - 1)
        tok[:B] = nxt[:B]
    shared.close()
    res.wall_s = now()
    return res


def decode_gaps(res: TraceResult):
    """Time between the end of one decode step and the start of the next, for consecutive
    steps that share a row: the admission work a running row waits for between two of its
    tokens (idle time with no row running is not a stall)."""
    out = []
    for i in range(len(res.step_s) - 1):
        if set(res.step_reqs[i]) & set(res.step_reqs[i + 1]):
            out.append(res.step_start[i + 1] - (res.step_start[i] + res.step_s[i]))
    return out


def percentiles(values, qs=(50, 95)):
    v = np.asarray(list(values), dtype=np.float64)
    if v.size == 0:
        return {f"p{q}": None for q in qs}
    return {f"p{q}": float(np.percentile(v, q)) for q in qs}
