"""Plain fp64 CPU oracle for the VAE group-norm + SiLU step.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU legs use this module; the product path never imports it.  It shares no
code with the CUDA library.

What it computes.  "fused qknorm rope Flux 2.0" (TensorRT-Model-Connect PR
#239, section "Not in this PR — follow-ups") lists ``group_norm_silu`` for
the VAE, which runs once per generation.  Read plainly: a group
normalisation of an NCHW activation followed by the SiLU activation.  For
sample n and group g of G (channels g*C/G .. (g+1)*C/G - 1), over all
(C/G)*H*W elements of that group:

    mu    = mean(x),  var = mean((x - mu)^2)
    y     = (x - mu) / sqrt(var + eps) * gamma[c] + beta[c]
    out   = y * sigmoid(y) = y / (1 + exp(-y))

returned unrounded in fp64.
"""
from __future__ import annotations

import numpy as np

from .qknr_oracle import decode


def group_norm_silu(x: np.ndarray, dtype: str, groups: int, gamma: np.ndarray, beta: np.ndarray,
                    eps: float) -> np.ndarray:
    """x: [N, C, H, W] uint16 bits of ``dtype``; gamma, beta: fp32 [C].
    Returns fp64 [N, C, H, W]."""
    N, C, H, W = x.shape
    if C % groups:
        raise ValueError("channels must divide into groups")
    e = float(np.float32(eps))
    xd = decode(x, dtype).reshape(N, groups, -1)
    mu = xd.mean(axis=-1, keepdims=True)
    d = xd - mu
    var = (d * d).mean(axis=-1, keepdims=True)
    y = (d / np.sqrt(var + e)).reshape(N, C, H, W)
    y = y * decode(gamma, "fp32")[None, :, None, None] + decode(beta, "fp32")[None, :, None, None]
    return y / (1.0 + np.exp(-y))


def group_norm_silu_at(x: np.ndarray, dtype: str, groups: int, gamma: np.ndarray, beta: np.ndarray, eps: float,
                       index: tuple) -> np.ndarray:
    """The same values as ``group_norm_silu`` at the elements ``x[index]``
    (a tuple of four integer arrays n, c, h, w), computing the statistics of
    only the groups those elements belong to."""
    N, C, H, W = x.shape
    n, c, h, w = (np.asarray(i) for i in index)
    gsize = C // groups
    e = float(np.float32(eps))
    g = c // gsize
    stats = {}
    for key in set(zip(n.tolist(), g.tolist())):
        ni, gi = key
        xd = decode(x[ni, gi * gsize:(gi + 1) * gsize], dtype)
        mu = xd.mean()
        var = ((xd - mu) ** 2).mean()
        stats[key] = (mu, var)
    mu = np.array([stats[(a, b)][0] for a, b in zip(n.tolist(), g.tolist())])
    var = np.array([stats[(a, b)][1] for a, b in zip(n.tolist(), g.tolist())])
    xv = decode(x[n, c, h, w], dtype)
    y = (xv - mu) / np.sqrt(var + e) * decode(gamma, "fp32")[c] + decode(beta, "fp32")[c]
    return y / (1.0 + np.exp(-y))
