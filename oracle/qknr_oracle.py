"""Plain, slow fp64 CPU oracle for the fused DiT QK-RMSNorm + RoPE step.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg use this module; the product path never imports it.  It
shares no code with the CUDA library: it has its own decoders, its own pair
tables and its own rounding, and it takes every input as a plain array.

What it computes (the plain reading of the two pages):

"fused qknorm rope Flux 2.0" (TensorRT-Model-Connect PR #239, title
section) replaces, per block, a chain of per-head RMSNorms followed by RoPEs
with one fused call.  "VisualGen Wan: deduplicate shared RoPE SMEM staging"
(TensorRT-LLM PR #18036, Description) stages one cos/sin row per token and
indexes it by dimension for every head, and its Test Coverage section
requires the shared and per-head expanded tables to agree exactly and the V
slice to stay unchanged.  For every token t, every head h of Q (gain
gamma_q) and of K (gain gamma_k):

    ms      = (1/D) * sum_d x[d]^2
    r       = 1 / sqrt(ms + eps)
    y[d]    = x[d] * r * gamma[d]
    o[d]    = y[d] * cos[t, d] + s(d) * y[p(d)] * sin[t, d]

where p(d) is the rotation partner of d (interleaved: d xor 1; rotate-half:
d +/- D/2) and s(d) = -1 for the first member of each pair, +1 for the
second.  cos/sin come from row ``t % cos_rows`` of a shared [rows, D]
table, or from ``[t % cos_rows, h]`` of the per-head expanded table.  V is
passed through bit for bit.

The fused kernel reaches this definition up to rounding: it keeps every
intermediate in fp32 and rounds once at the output.  The oracle keeps every
intermediate in fp64 and does not round; ``round_rne`` gives the correctly
rounded 16-bit value of its result for bit-level comparisons.

Parity pins (tests/test_oracle_pins.py) tie this code to things other than
itself: the textbook RMSNorm in torch, RoPE as a complex multiplication,
hand-worked D=4 cases, norm preservation, the relative-position property,
and torch/numpy casts for the decoders and the rounding.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

__all__ = [
    "decode", "round_rne", "pair_table", "rms_norm_heads", "rope_rotate",
    "qk_norm_rope", "forward_packed", "forward_separate",
]


# --------------------------------------------------------------------------
# exact decoding of the storage formats

def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored values to fp64 exactly.

    ``bf16`` and ``fp16`` arrays hold uint16 bit patterns.  A bf16 value is
    the upper half of an IEEE binary32 word, so shifting its bits up by 16
    gives the fp32 word with the same value.
    """
    if dtype == "fp32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "fp64":
        return np.asarray(a, dtype=np.float64)
    bits = np.asarray(a)
    if bits.dtype != np.uint16:
        raise TypeError("16-bit storage must be passed as uint16 bit patterns")
    if dtype == "bf16":
        word = bits.astype(np.uint32) << np.uint32(16)
        return word.view(np.float32).astype(np.float64)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------
# correctly rounded encoding (round to nearest, ties to even)

_FORMATS = {
    # significand bits incl. the implicit one, min normal exponent, max finite
    "bf16": (8, -126, float.fromhex("0x1.fep127")),
    "fp16": (11, -14, 65504.0),
}


def round_rne(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values directly (no intermediate fp32) to bf16 or fp16,
    round-half-to-even, and return uint16 bit patterns.

    A finite x is m * 2**e with 0.5 <= |m| < 1.  A format with p significand
    bits keeps m * 2**p rounded to an integer, except below the normal range
    where the quantum stays at the subnormal step.  ``np.rint`` rounds
    halves to even.
    """
    p, emin, vmax = _FORMATS[dtype]
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2**e
    # exponent of the quantum: e - p for normals; fixed below normal range
    qexp = np.maximum(e - p, emin - (p - 1))
    q = np.ldexp(np.rint(np.ldexp(x, -qexp)), qexp)
    q = np.where(np.abs(q) > vmax, np.copysign(np.inf, x), q)
    q = np.where(np.isnan(x), np.nan, q)
    if dtype == "fp16":
        return q.astype(np.float16).view(np.uint16)   # q is exact in fp16
    word = q.astype(np.float32).view(np.uint32)       # q is exact in fp32
    return (word >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# the method

def pair_table(D: int, rope_style: str):
    """Partner index p(d) and sign s(d) for every dimension of a head.

    Interleaved pairing rotates (2i, 2i+1); rotate-half pairing rotates
    (i, i + D/2).  The first member of a pair gets -partner*sin, the second
    +partner*sin (page 1, Test Coverage: interleaved and rotate-half RoPE).
    """
    if D % 2:
        raise ValueError("head_dim must be even")
    d = np.arange(D)
    if rope_style == "interleaved":
        partner = d ^ 1
        first = (d % 2) == 0
    elif rope_style == "rotate_half":
        h = D // 2
        partner = np.where(d < h, d + h, d - h)
        first = d < h
    else:
        raise ValueError(f"unknown rope_style {rope_style!r}")
    sign = np.where(first, -1.0, 1.0)
    return partner, sign


def rms_norm_heads(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Per-head RMSNorm of x [..., D] with gain gamma [D], all in fp64:
    y = x / sqrt(mean(x^2) + eps) * gamma."""
    D = x.shape[-1]
    ms = np.sum(x * x, axis=-1, keepdims=True) / D
    r = 1.0 / np.sqrt(ms + eps)
    return x * r * np.asarray(gamma, dtype=np.float64)


def rope_rotate(y: np.ndarray, c: np.ndarray, s: np.ndarray, rope_style: str) -> np.ndarray:
    """o[d] = y[d]*c[d] + s(d)*y[p(d)]*s[d]; c and s broadcast against y
    [T, H, D] (shared rows arrive as [T, 1, D], expanded as [T, H, D])."""
    partner, sign = pair_table(y.shape[-1], rope_style)
    return y * c + sign * y[..., partner] * s


def qk_norm_rope(
    x: np.ndarray,
    gamma: np.ndarray,
    eps: float,
    cos: np.ndarray,
    sin: np.ndarray,
    rope_style: str,
    cos_layout: str = "shared_row",
    rows: Optional[np.ndarray] = None,
) -> np.ndarray:
    """Normalise then rotate one tensor of heads.

    x: [T, H, D] fp64 values.  cos/sin: fp64, [cos_rows, D] (shared_row) or
    [cos_rows, H, D] (per_head_expanded).  ``rows`` gives each of the T rows
    its token index (default 0..T-1); the table row used is
    ``token % cos_rows``.  Returns [T, H, D] fp64, unrounded.
    """
    T = x.shape[0]
    tok = np.arange(T) if rows is None else np.asarray(rows)
    trow = tok % cos.shape[0]
    if cos_layout == "shared_row":
        c = cos[trow][:, None, :]
        s = sin[trow][:, None, :]
    elif cos_layout == "per_head_expanded":
        if cos.shape[1] != x.shape[1]:
            raise ValueError("expanded table must have one row per head")
        c = cos[trow]
        s = sin[trow]
    else:
        raise ValueError(f"unknown cos_layout {cos_layout!r}")
    y = rms_norm_heads(x, gamma, eps)
    return rope_rotate(y, c, s, rope_style)


def _eps64(eps: float) -> float:
    # the kernel receives eps as an fp32 argument; use that exact value
    return float(np.float32(eps))


def forward_packed(
    qkv: np.ndarray,
    dtype: str,
    n_heads_q: int,
    n_heads_k: int,
    n_heads_v: int,
    head_dim: int,
    gamma_q: np.ndarray,
    gamma_k: np.ndarray,
    eps: float,
    cos: np.ndarray,
    sin: np.ndarray,
    cos_dtype: str,
    rope_style: str,
    cos_layout: str = "shared_row",
    rows: Optional[np.ndarray] = None,
    chunk: int = 4096,
) -> Dict[str, np.ndarray]:
    """Oracle over a packed QKV activation [T, (Hq+Hk+Hv)*D] of uint16 bits.

    ``rows``, when given, selects token rows of ``qkv`` to evaluate (the
    result then has one row per selected token).  Returns ``q`` [n, Hq, D]
    and ``k`` [n, Hk, D] in fp64 and ``v`` — the V column slice of the input
    bits, unchanged.
    """
    D = head_dim
    tok = np.arange(qkv.shape[0]) if rows is None else np.asarray(rows)
    c = decode(cos, cos_dtype)
    s = decode(sin, cos_dtype)
    gq = decode(gamma_q, "fp32")
    gk = decode(gamma_k, "fp32")
    e = _eps64(eps)
    oq, ok = [], []
    for i in range(0, len(tok), chunk):
        t = tok[i:i + chunk]
        x = decode(qkv[t], dtype)
        xq = x[:, : n_heads_q * D].reshape(len(t), n_heads_q, D)
        xk = x[:, n_heads_q * D:(n_heads_q + n_heads_k) * D].reshape(len(t), n_heads_k, D)
        oq.append(qk_norm_rope(xq, gq, e, c, s, rope_style, cos_layout, t))
        ok.append(qk_norm_rope(xk, gk, e, c, s, rope_style, cos_layout, t))
    q0 = (n_heads_q + n_heads_k) * D
    return {
        "q": np.concatenate(oq) if oq else np.zeros((0, n_heads_q, D)),
        "k": np.concatenate(ok) if ok else np.zeros((0, n_heads_k, D)),
        "v": qkv[tok][:, q0:q0 + n_heads_v * D].copy(),
    }


def forward_separate(
    x: np.ndarray,
    dtype: str,
    n_heads: int,
    head_dim: int,
    gamma: np.ndarray,
    eps: float,
    cos: np.ndarray,
    sin: np.ndarray,
    cos_dtype: str,
    rope_style: str,
    cos_layout: str = "shared_row",
    rows: Optional[np.ndarray] = None,
    chunk: int = 4096,
) -> np.ndarray:
    """Oracle for one separate tensor [T, H*D] (the per-tensor launch of
    page 2: one fused call per tensor).  Returns [n, H, D] fp64."""
    D = head_dim
    tok = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    c = decode(cos, cos_dtype)
    s = decode(sin, cos_dtype)
    g = decode(gamma, "fp32")
    e = _eps64(eps)
    out = []
    for i in range(0, len(tok), chunk):
        t = tok[i:i + chunk]
        xt = decode(x[t], dtype).reshape(len(t), n_heads, D)
        out.append(qk_norm_rope(xt, g, e, c, s, rope_style, cos_layout, t))
    return np.concatenate(out) if out else np.zeros((0, n_heads, D))
