"""Shared set-up for the GPU parity tests: the engine (through the C ABI) and the CPU oracle
on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from continuous_batching_transformer_gb300.model import DeviceWeights, Engine

# max-abs logit tolerance against the oracle: bf16 weights, 4-bit affine weights
TOL = {"bf16": 2e-2, "affine4": 5e-2}

_built = False


def ensure_built():
    global _built
    if not _built:
        import __graft_entry__
        __graft_entry__.build()
        _built = True


def top2_margin(row: np.ndarray) -> float:
    p = np.partition(row, -2)
    return float(p[-1] - p[-2])


def check_logits(gpu: np.ndarray, ref: np.ndarray, tol: float, what: str):
    """Element-wise logit parity plus greedy-token parity.  Where the oracle's top-2 margin
    is below the tolerance, either of the tied tokens passes (the comparison is then made
    on the oracle's token, which both sides are fed next)."""
    err = np.abs(gpu - ref)
    assert np.isfinite(gpu).all(), f"{what}: non-finite logits"
    assert err.max() <= tol, f"{what}: max |gpu - oracle| = {err.max():.3e} > {tol}"
    for r in range(ref.shape[0]):
        g, o = int(np.argmax(gpu[r])), oracle.argmax(ref[r])
        if g != o:
            assert top2_margin(ref[r]) < tol and ref[r][g] >= ref[r][o] - tol, \
                f"{what}: row {r} greedy token {g} != oracle {o} with margin {top2_margin(ref[r]):.3e}"
    return float(err.max())


def to_dev(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
