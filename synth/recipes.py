"""The synthetic workloads: model shapes, seeds and draw recipes.

Shapes are the five workloads the decode step is specified on: a tiny
2-layer decoder checked in full against the CPU oracle, and a 7B-shaped
(Mistral-like) decoder in bf16 or 4-bit affine weights.  All values come
from ``synth`` draws; nothing here computes any part of the transformer.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

from . import uniform_ints, tokens, stream_misc, stream_tokens, words


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    rms_eps: float
    rope_theta: float
    weight_sigma: float = 0.02
    weight_seed: int = 0
    # norm gains: 1.0 exactly unless gain_sigma > 0 (then 1 + gain_sigma * N(0,1), used by
    # tests so that a misplaced gain cannot hide behind g == 1)
    gain_sigma: float = 0.0
    weight_format: str = "bf16"       # "bf16" or "affine4"
    group_size: int = 64

    @property
    def q_dim(self):
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim

    @property
    def kv_sigma(self) -> float:
        """Spread of synthetic KV values: that of a projection of a unit-RMS vector through
        N(0, weight_sigma^2) weights, i.e. weight_sigma * sqrt(d_model)."""
        return self.weight_sigma * math.sqrt(self.d_model)

    def linear_params(self) -> int:
        per_layer = (self.q_dim + 2 * self.kv_dim) * self.d_model + self.q_dim * self.d_model \
            + 3 * self.d_ff * self.d_model
        return self.n_layers * per_layer + self.vocab * self.d_model

    def kv_bytes_per_token(self) -> int:
        return self.n_layers * 2 * self.kv_dim * 2

    def weight_bytes_per_step(self) -> int:
        """Bytes of linear weights one decode step streams (embedding rows excluded)."""
        n = self.linear_params()
        if self.weight_format == "bf16":
            return 2 * n
        return n // 2 + (n // self.group_size) * 4


TINY = ModelShape("tiny-2L-d256", 2, 256, 4, 4, 64, 1024, 1024, 1e-6, 1e4)
MISTRAL_7B = ModelShape("mistral-7b-shape", 32, 4096, 32, 8, 128, 14336, 32000, 1e-5, 1e6)
MISTRAL_7B_Q4 = replace(MISTRAL_7B, name="mistral-7b-shape-affine4", weight_format="affine4")


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    seed: int
    batch: int
    ctx_lo: int          # context lengths uniform in [ctx_lo, ctx_hi] (inclusive)
    ctx_hi: int
    steps: int
    prompt_lens: tuple = field(default=())   # explicit prompt lengths (tiny workload)

    def context_lengths(self) -> np.ndarray:
        if self.prompt_lens:
            return np.asarray(self.prompt_lens, dtype=np.int32)
        if self.ctx_lo == self.ctx_hi:
            return np.full(self.batch, self.ctx_lo, dtype=np.int32)
        return uniform_ints(self.batch, self.seed, stream_misc(1), self.ctx_lo, self.ctx_hi)

    def row_tokens(self, row: int, n: int) -> np.ndarray:
        """Token ids of row `row` (prompt, then the decode step's last token at index n-1)."""
        return tokens(n, self.seed, stream_tokens(row), self.shape.vocab)


# tiny decoder: segmented prefill of 4 prompts, then 16 greedy decode steps
TINY_RUN = Workload("tiny-prefill+16-decode", TINY, 0, 4, 0, 0, 16, prompt_lens=(5, 17, 32, 9))
# 7B bf16: 8 persistent slabs, contexts uniform in [512, 4096], 128 greedy decode steps
DECODE_7B_B8 = Workload("7b-bf16-B8-ctx512..4096", MISTRAL_7B, 2, 8, 512, 4096, 128)


def decode_7b_fixed(batch: int, ctx: int = 2048, fmt: str = "bf16", steps: int = 64) -> Workload:
    shape = MISTRAL_7B if fmt == "bf16" else MISTRAL_7B_Q4
    return Workload(f"7b-{fmt}-B{batch}-ctx{ctx}", shape, 3, batch, ctx, ctx, steps)


# long-context GQA decode: 32 slabs of 8k-16k tokens, 32 steps
LONG_7B_B32 = Workload("7b-bf16-B32-ctx8192..16384", MISTRAL_7B, 5, 32, 8192, 16384, 32)


@dataclass(frozen=True)
class Request:
    arrival_s: float
    prompt_len: int
    output_len: int
    row: int             # synthetic token stream id
    prefix_len: int = 0  # the prompt starts with this many tokens of a shared prefix ...
    prefix_row: int = 0  # ... drawn from this token stream (the same for every request)


def trace_requests(n: int = 64, rate_per_s: float = 2.0, prompt_lo: int = 256,
                   prompt_hi: int = 4096, mean_out: float = 256.0, out_cap: int = 4096,
                   seed: int = 1) -> list:
    """Continuous-batching trace: Poisson arrivals (exponential gaps by inversion of a
    uniform word), prompt lengths uniform, output lengths geometric with the given mean
    (P(n) = p(1-p)^(n-1), n >= 1) capped at out_cap."""
    u_gap = (words(n, seed, stream_misc(10)) >> np.uint64(11)).astype(np.float64) / float(1 << 53)
    u_out = (words(n, seed, stream_misc(11)) >> np.uint64(11)).astype(np.float64) / float(1 << 53)
    plen = uniform_ints(n, seed, stream_misc(12), prompt_lo, prompt_hi)
    p = 1.0 / mean_out
    t = 0.0
    reqs = []
    for i in range(n):
        t += -math.log1p(-u_gap[i]) / rate_per_s
        k = 1 + int(math.floor(math.log1p(-u_out[i]) / math.log1p(-p)))
        reqs.append(Request(t, int(plen[i]), min(k, out_cap), 1000 + i))
    return reqs


def agent_requests(n: int = 32, prefix_len: int = 2048, own_lo: int = 64, own_hi: int = 512,
                   mean_out: float = 128.0, out_cap: int = 1024, seed: int = 2) -> list:
    """Sub-agents of one harness: n requests at t = 0 whose prompts are one shared system
    prompt of prefix_len tokens followed by an own part of U[own_lo, own_hi] tokens; outputs
    geometric with the given mean, capped."""
    u_out = (words(n, seed, stream_misc(21)) >> np.uint64(11)).astype(np.float64) / float(1 << 53)
    own = uniform_ints(n, seed, stream_misc(22), own_lo, own_hi)
    p = 1.0 / mean_out
    reqs = []
    for i in range(n):
        k = 1 + int(math.floor(math.log1p(-u_out[i]) / math.log1p(-p)))
        reqs.append(Request(0.0, prefix_len + int(own[i]), min(k, out_cap), 3000 + i,
                            prefix_len, 2999))
    return reqs
