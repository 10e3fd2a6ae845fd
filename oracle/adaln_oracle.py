"""Plain fp64 CPU oracle for the AdaLN scale/shift step.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU legs use this module; the product path never imports it.  It shares no
code with the CUDA library.

What it computes.  "fused qknorm rope Flux 2.0" (TensorRT-Model-Connect PR
#239, section "Not in this PR — follow-ups") names the next fusion target
as AdaLN's ``fuse_scale_shift``, 81 calls per FLUX.2 step.  The plain
reading is adaptive layer normalisation: each token row of the hidden
state is layer-normalised without a learned affine, then modulated by a
per-sample scale and shift computed from the conditioning:

    mu   = (1/C) sum_c x[c]
    var  = (1/C) sum_c (x[c] - mu)^2
    out[c] = (x[c] - mu) / sqrt(var + eps) * (1 + scale[b, c]) + shift[b, c]

where ``b`` is the sample (batch entry) that token row ``t`` belongs to:
``b = t // rows_per_batch``.  The result is returned unrounded in fp64.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .qknr_oracle import decode


def layer_norm_rows(x: np.ndarray, eps: float) -> np.ndarray:
    """(x - mean) / sqrt(biased variance + eps) along the last axis, fp64."""
    C = x.shape[-1]
    mu = np.sum(x, axis=-1, keepdims=True) / C
    d = x - mu
    var = np.sum(d * d, axis=-1, keepdims=True) / C
    return d / np.sqrt(var + eps)


def adaln_modulate(
    x: np.ndarray,
    dtype: str,
    scale: np.ndarray,
    shift: np.ndarray,
    mod_dtype: str,
    eps: float,
    rows_per_batch: int,
    rows: Optional[np.ndarray] = None,
    chunk: int = 2048,
) -> np.ndarray:
    """Oracle over token rows of ``x`` [T, C] (uint16 bits of ``dtype``).

    ``scale`` and ``shift`` are [B, C] in ``mod_dtype`` (fp32 arrays, or
    uint16 bits of bf16/fp16).  ``rows`` selects token rows (default all);
    the result has one row per selected token.  eps is taken as the fp32
    value the kernel receives.
    """
    tok = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    sc = decode(scale, mod_dtype)
    sh = decode(shift, mod_dtype)
    e = float(np.float32(eps))
    out = []
    for i in range(0, len(tok), chunk):
        t = tok[i:i + chunk]
        b = t // rows_per_batch
        xn = layer_norm_rows(decode(x[t], dtype), e)
        out.append(xn * (1.0 + sc[b]) + sh[b])
    return np.concatenate(out) if out else np.zeros((0, x.shape[1]))
