"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This module holds none of the training step's arithmetic: it only draws the
inputs that both sides consume, so that a parity test feeds the same bytes to
each.  Neither side's parameter initialisation lives here (each side draws its
own initial weights from the seed with its own copy of the generator).

Inputs stand in for the token streams the llm.c pages train on (FineWeb /
Tiny Shakespeare shards, "What Is karpathy/llm.c?" §Hands-On, and the pyshine
tour's install section): there is no dataset here, so tokens are drawn i.i.d.
from a Zipf(s) law over the GPT-2 vocabulary, a heavy-tailed frequency profile
like natural text.  The dataloader reads B*T+1 tokens and shifts the targets
left by one; so do we.
"""
from __future__ import annotations

import numpy as np

__all__ = ["zipf_tokens", "normal_array", "uniform_array"]


def zipf_tokens(B: int, T: int, V: int, seed: int = 1234, s: float = 1.1):
    """Draw B*(T+1) i.i.d. Zipf(s) token ids over [0, V) and split them.

    P(k) is proportional to (k+1)^-s.  Sampling is by inverse CDF on a
    float64 cumulative table with numpy's PCG64 stream seeded by `seed`.
    Returns (tokens, targets), each int32 [B, T], targets = tokens shifted
    left by one position within each row.
    """
    if B <= 0 or T <= 0 or V <= 0:
        raise ValueError("B, T, V must be positive")
    rng = np.random.default_rng(seed)
    k = np.arange(V, dtype=np.float64)
    cdf = np.cumsum((k + 1.0) ** (-s))
    cdf /= cdf[-1]
    u = rng.random(B * (T + 1))
    idx = np.searchsorted(cdf, u, side="right")
    np.minimum(idx, V - 1, out=idx)
    seq = idx.astype(np.int32).reshape(B, T + 1)
    return np.ascontiguousarray(seq[:, :T]), np.ascontiguousarray(seq[:, 1:])


def normal_array(shape, seed: int, std: float = 1.0, dtype=np.float32):
    """N(0, std^2) values from numpy's PCG64 stream (for kernel-level tests)."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(size=shape) * std).astype(dtype)


def uniform_array(shape, seed: int, lo: float = -1.0, hi: float = 1.0, dtype=np.float32):
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=shape).astype(dtype)
