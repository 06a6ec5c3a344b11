"""Scalar pure-Python restatement of single-query attention, for tiny inputs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Used only as a cross-check of the vectorised numpy code in
:mod:`oracle.attention` on inputs of a few tokens: it walks the definition
("The Reasoning Engine Meltdown", §2.1 attention equation) one scalar at a
time with ``math.exp`` and Python floats (IEEE binary64), with no matrix
products, so an operand transposed or an axis confused in the numpy code
shows up as a mismatch.
"""

from __future__ import annotations

import math


def single_query(q, keys, values, scale):
    """q: list of d floats; keys/values: lists of L rows; returns list of dv."""
    scores = []
    for k in keys:
        acc = 0.0
        for a, b in zip(q, k):
            acc += a * b
        scores.append(acc * scale)
    top = max(scores)
    weights = [math.exp(s - top) for s in scores]
    total = sum(weights)
    out = [0.0] * len(values[0])
    for w, v in zip(weights, values):
        for j, x in enumerate(v):
            out[j] += (w / total) * x
    return out
