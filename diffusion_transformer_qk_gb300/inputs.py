"""Seeded synthetic inputs for the fused DiT QK-RMSNorm + RoPE step.

This module builds the inputs that both the CUDA path and the CPU oracle
consume: activations, RMSNorm gains and finished RoPE cos/sin tables.  It
holds none of the normalisation or rotation arithmetic; it only draws random
numbers, rounds them to the storage dtype and tabulates rotary angles.

Storage conventions shared by every consumer:

* 16-bit activations (bf16 or fp16) are ``numpy.uint16`` arrays holding the
  raw bit patterns, because numpy has no bfloat16 type.
* gamma is fp32 ``[D]``.
* cos/sin are ``[cos_rows, D]`` (one row per sequence position, indexed by
  dimension for every head) in fp32, or the bf16 bit patterns of the same
  values.  Token ``t`` uses row ``t % cos_rows``, which broadcasts one table
  over a batch.

Workload shapes follow the two pages this project implements: the Wan-A14B
dispatch of "VisualGen Wan: deduplicate shared RoPE SMEM staging"
(TensorRT-LLM PR #18036, Description: one head_dim=128 row shared by 40
heads) and the FLUX.2 per-tensor launch of "fused qknorm rope Flux 2.0"
(TensorRT-Model-Connect PR #239, title section).  The RoPE axis splits and
positions are this project's reading where the pages are silent.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

DTYPES = ("bf16", "fp16")
COS_DTYPES = ("fp32", "bf16")
ROPE_STYLES = ("interleaved", "rotate_half")
COS_LAYOUTS = ("shared_row", "per_head_expanded")


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtypes, RoPE style and seed."""

    name: str
    batch: int
    seq: int                       # tokens per sequence; cos/sin has seq rows
    n_heads_q: int
    n_heads_k: int
    n_heads_v: int
    head_dim: int
    dtype: str = "bf16"            # activation storage
    packed: bool = True            # packed [T, (Hq+Hk+Hv)*D] or separate tensors
    rope_style: str = "interleaved"
    cos_dtype: str = "fp32"
    cos_layout: str = "shared_row"
    positions: str = "1d"          # "1d" | "wan3d" | "flux2d1d"
    grid: Tuple[int, ...] = ()     # wan3d: (F, H, W); flux2d1d: (text, img_h, img_w)
    axes_dim: Tuple[int, ...] = () # head_dim split per RoPE axis
    theta: float = 10000.0
    scale: float = 1.0             # activations are scale * N(0,1)
    eps: float = 1e-6
    seed: int = 0
    single_launch: bool = False    # separate tensors: Q and K in one launch
    out_of_place: bool = False     # write Q/K (and copy V) to a second buffer

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the pages' kernels are quoted on, with synthetic values.
WORKLOADS: Dict[str, Workload] = {
    # 256 tokens, packed bf16 [256, 3*24*64], 1-D positions, interleaved.
    "tiny_256x24x64": Workload(
        "tiny_256x24x64", 1, 256, 24, 24, 24, 64, "bf16", True,
        "interleaved", "fp32", "shared_row", "1d", (), (64,)),
    # 4096 tokens, packed [4096, 3*24*128], N(0,1)*2, rotate-half, 1-D.
    "dense_4096x24x128": Workload(
        "dense_4096x24x128", 1, 4096, 24, 24, 24, 128, "bf16", True,
        "rotate_half", "fp32", "shared_row", "1d", (), (128,), scale=2.0),
    # Wan-A14B: 21x30x52 latent grid = 32760 tokens, 40 heads x 128,
    # 3-axis RoPE with head_dim split 44/42/42 (frame, height, width).
    "wan_32760x40x128": Workload(
        "wan_32760x40x128", 1, 32760, 40, 40, 40, 128, "bf16", True,
        "interleaved", "fp32", "shared_row", "wan3d", (21, 30, 52), (44, 42, 42)),
    # Same Wan shape with the per-head expanded fp32 table [T, 40, 128].
    "wan_32760x40x128_expanded": Workload(
        "wan_32760x40x128_expanded", 1, 32760, 40, 40, 40, 128, "bf16", True,
        "interleaved", "fp32", "per_head_expanded", "wan3d", (21, 30, 52),
        (44, 42, 42)),
    # FLUX.2: batch 2 x (512 text + 64x64 image) tokens, separate Q, K, V
    # [2*4608, 48*128], rotate-half, 1-D text + 2-D image positions over
    # three axes split 32/48/48 (text index, image row, image column).
    "flux2_2x4608x48x128": Workload(
        "flux2_2x4608x48x128", 2, 4608, 48, 48, 48, 128, "bf16", False,
        "rotate_half", "fp32", "shared_row", "flux2d1d", (512, 64, 64),
        (32, 48, 48)),
}

# Variants of the same workloads for the staging and launch-form comparisons:
# bf16 tables (shared and expanded), out-of-place with V copied once, and
# FLUX.2's Q and K in one launch instead of one launch per tensor.
WORKLOADS.update({
    "wan_32760x40x128_bf16cos": WORKLOADS["wan_32760x40x128"].with_(
        name="wan_32760x40x128_bf16cos", cos_dtype="bf16"),
    "wan_32760x40x128_expanded_bf16cos": WORKLOADS["wan_32760x40x128_expanded"].with_(
        name="wan_32760x40x128_expanded_bf16cos", cos_dtype="bf16"),
    "wan_32760x40x128_out_of_place": WORKLOADS["wan_32760x40x128"].with_(
        name="wan_32760x40x128_out_of_place", out_of_place=True),
    "flux2_2x4608x48x128_single_launch": WORKLOADS["flux2_2x4608x48x128"].with_(
        name="flux2_2x4608x48x128_single_launch", single_launch=True),
})


# --------------------------------------------------------------------------
# storage helpers (bit patterns only; no method arithmetic)

def to_storage_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32/fp64 values to bf16 or fp16 (round-to-nearest-even) and
    return the bit patterns as uint16.  Uses torch's CPU casts."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    return t.to(tdt).view(torch.int16).numpy().view(np.uint16)


def storage_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of bf16/fp16 bit patterns to fp32 (for generators and
    reporting; the oracle decodes with its own routine)."""
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float32)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# rotary tables

def positions_for(w: Workload) -> np.ndarray:
    """Integer positions [seq, n_axes] for each sequence index."""
    s = np.arange(w.seq, dtype=np.int64)
    if w.positions == "1d":
        return s[:, None]
    if w.positions == "wan3d":
        F, H, W = w.grid
        if F * H * W != w.seq:
            raise ValueError("wan3d grid does not match seq")
        # raster order: frame-major, then height, then width
        return np.stack([s // (H * W), (s // W) % H, s % W], axis=1)
    if w.positions == "flux2d1d":
        n_text, ih, iw = w.grid
        if n_text + ih * iw != w.seq:
            raise ValueError("flux2d1d grid does not match seq")
        pos = np.zeros((w.seq, 3), dtype=np.int64)
        pos[:n_text, 0] = s[:n_text]                 # text: (i, 0, 0)
        img = s[n_text:] - n_text
        pos[n_text:, 1] = img // iw                  # image: (0, row, col)
        pos[n_text:, 2] = img % iw
        return pos
    raise ValueError(w.positions)


def rope_half_angles(pos: np.ndarray, axes_dim: Sequence[int], theta: float) -> np.ndarray:
    """Per-pair rotation angles [seq, D/2] in fp64.

    Axis ``a`` owns ``axes_dim[a]`` dimensions, i.e. ``axes_dim[a]/2`` pairs;
    its pair ``j`` turns at frequency ``theta ** (-2j / axes_dim[a])`` times
    the token's position on that axis.  Axes are concatenated in order.
    """
    if pos.shape[1] != len(axes_dim):
        raise ValueError("one axis size per position column")
    cols = []
    for a, da in enumerate(axes_dim):
        if da % 2:
            raise ValueError("each axis needs an even number of dimensions")
        j = np.arange(da // 2, dtype=np.float64)
        freq = theta ** (-2.0 * j / da)
        cols.append(pos[:, a:a + 1].astype(np.float64) * freq[None, :])
    return np.concatenate(cols, axis=1)


def rope_table(w: Workload) -> Tuple[np.ndarray, np.ndarray]:
    """Shared cos/sin rows [seq, D] (fp32, or bf16 bits when cos_dtype is bf16).

    Both members of a rotation pair get the pair's angle: for interleaved
    pairing pair k sits at dims (2k, 2k+1); for rotate-half at (k, k + D/2).
    """
    D = w.head_dim
    if sum(w.axes_dim) != D:
        raise ValueError("axes_dim must sum to head_dim")
    ang = rope_half_angles(positions_for(w), w.axes_dim, w.theta)  # [seq, D/2]
    if w.rope_style == "interleaved":
        full = np.repeat(ang, 2, axis=1)
    elif w.rope_style == "rotate_half":
        full = np.concatenate([ang, ang], axis=1)
    else:
        raise ValueError(w.rope_style)
    c = np.cos(full).astype(np.float32)
    s = np.sin(full).astype(np.float32)
    if w.cos_dtype == "bf16":
        return to_storage_bits(c, "bf16"), to_storage_bits(s, "bf16")
    if w.cos_dtype != "fp32":
        raise ValueError(w.cos_dtype)
    return np.ascontiguousarray(c), np.ascontiguousarray(s)


def expand_per_head(table: np.ndarray, n_heads: int) -> np.ndarray:
    """Materialise a shared [rows, D] table as the per-head layout
    [rows, H, D] (every head gets an identical copy)."""
    return np.ascontiguousarray(
        np.broadcast_to(table[:, None, :], (table.shape[0], n_heads, table.shape[1])))


def per_head_tables(rows: int, n_heads: int, head_dim: int, rope_style: str, cos_dtype: str, seed: int,
                    per_dim: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Per-head expanded cos/sin tables [rows, H, D] whose rows differ from
    head to head: every (row, head, pair) gets its own angle, uniform in
    [-pi, pi), drawn from numpy PCG64(seed) in fp32.  Both members of a pair
    hold the pair's angle (interleaved: dims 2k, 2k+1; rotate-half: k,
    k + D/2).  With ``per_dim`` every (row, head, dimension) gets an angle
    of its own instead, so the two members of a pair differ too.

    Returns fp32 arrays, or bf16 bit patterns when ``cos_dtype`` is bf16.
    """
    g = np.random.Generator(np.random.PCG64(seed))
    D = head_dim
    if per_dim:
        full = g.uniform(-np.pi, np.pi, size=(rows, n_heads, D)).astype(np.float32)
    else:
        ang = g.uniform(-np.pi, np.pi, size=(rows, n_heads, D // 2)).astype(np.float32)
        if rope_style == "interleaved":
            full = np.repeat(ang, 2, axis=2)
        elif rope_style == "rotate_half":
            full = np.concatenate([ang, ang], axis=2)
        else:
            raise ValueError(rope_style)
        del ang
    c = np.cos(full)
    s = np.sin(full)
    del full
    if cos_dtype == "bf16":
        return to_storage_bits(c, "bf16"), to_storage_bits(s, "bf16")
    if cos_dtype != "fp32":
        raise ValueError(cos_dtype)
    return np.ascontiguousarray(c), np.ascontiguousarray(s)


# --------------------------------------------------------------------------
# activations

def _normal(g: np.random.Generator, shape, scale: float) -> np.ndarray:
    x = g.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def make_inputs(w: Workload, tokens: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Draw one seeded instance of ``w``.

    Draw order (numpy PCG64 seeded with ``w.seed``): activations (packed
    QKV, or Q then K then V), then gamma_q, then gamma_k.  Activations are
    ``scale * N(0,1)`` rounded to the storage dtype; gamma = 1 + 0.1*N(0,1)
    in fp32.  ``tokens`` overrides the row count (for reduced test sizes);
    the rotary table keeps ``w.seq`` rows and is indexed modulo its length.

    Returned keys: ``qkv`` (packed) or ``q``, ``k``, ``v``; ``gamma_q``,
    ``gamma_k``; ``cos``, ``sin`` (shared rows).
    """
    T = w.tokens if tokens is None else int(tokens)
    D = w.head_dim
    g = np.random.Generator(np.random.PCG64(w.seed))
    out: Dict[str, np.ndarray] = {}
    if w.packed:
        width = (w.n_heads_q + w.n_heads_k + w.n_heads_v) * D
        out["qkv"] = to_storage_bits(_normal(g, (T, width), w.scale), w.dtype)
    else:
        for name, h in (("q", w.n_heads_q), ("k", w.n_heads_k), ("v", w.n_heads_v)):
            out[name] = to_storage_bits(_normal(g, (T, h * D), w.scale), w.dtype)
    out["gamma_q"] = (1.0 + 0.1 * g.standard_normal(D)).astype(np.float32)
    out["gamma_k"] = (1.0 + 0.1 * g.standard_normal(D)).astype(np.float32)
    out["cos"], out["sin"] = rope_table(w)
    return out


def split_packed(qkv: np.ndarray, hq: int, hk: int, hv: int, d: int):
    """Views of the Q, K and V column slices of a packed [T, (Hq+Hk+Hv)*D] array."""
    return (qkv[:, : hq * d], qkv[:, hq * d:(hq + hk) * d], qkv[:, (hq + hk) * d:(hq + hk + hv) * d])


def algorithmic_bytes(w: Workload, v_copied: bool = False, launches: str = "all",
                      tokens: Optional[int] = None) -> int:
    """Bytes one call must move at minimum: Q and K read once and written
    once, the cos/sin table rows it uses read once (the expanded layout is
    charged its full [T, H, D] table), V read and written once when copied,
    plus gamma.

    ``launches="q"`` counts one per-tensor launch over Q only (FLUX.2 style).
    ``tokens`` overrides the row count (a reduced case of the workload).
    """
    es = 2
    T, D = (w.tokens if tokens is None else int(tokens)), w.head_dim
    hq, hk = w.n_heads_q, w.n_heads_k
    if launches == "q":
        hk = 0
    v_copied = v_copied or w.out_of_place
    cos_es = 4 if w.cos_dtype == "fp32" else 2
    if w.cos_layout == "shared_row":
        cos_bytes = 2 * min(w.seq, T) * D * cos_es
    else:
        cos_bytes = 2 * T * w.n_heads_q * D * cos_es
    qk = 2 * T * (hq + hk) * D * es
    v = 2 * T * w.n_heads_v * D * es if v_copied else 0
    gam = (2 if hk else 1) * D * 4
    return qk + cos_bytes + v + gam


# --------------------------------------------------------------------------
# AdaLN scale/shift workloads (the next fused step named by "fused qknorm
# rope Flux 2.0", section "Not in this PR — follow-ups": fuse_scale_shift,
# 81 calls per FLUX.2 step)

@dataclass(frozen=True)
class AdaLNWorkload:
    """Token rows [batch*seq, hidden] with one modulation row per sample."""

    name: str
    batch: int
    seq: int                       # rows per sample (one scale/shift row each)
    hidden: int
    dtype: str = "bf16"            # activations
    mod_dtype: str = "bf16"        # scale / shift storage: "fp32" or the activation dtype
    scale: float = 1.0             # activations are scale * N(0,1)
    mod_scale: float = 0.1         # scale and shift are mod_scale * N(0,1)
    eps: float = 1e-6
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def with_(self, **kw) -> "AdaLNWorkload":
        return replace(self, **kw)


ADALN_WORKLOADS: Dict[str, AdaLNWorkload] = {
    # FLUX.2 single-stream block: 2 x (512 text + 4096 image) tokens, hidden 48*128
    "adaln_flux2_2x4608x6144": AdaLNWorkload("adaln_flux2_2x4608x6144", 2, 4608, 6144),
    # Wan-A14B: 32760 latent tokens, hidden 40*128
    "adaln_wan_32760x5120": AdaLNWorkload("adaln_wan_32760x5120", 1, 32760, 5120),
}


def make_adaln_inputs(w: AdaLNWorkload, tokens: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Seeded instance: draw order x, scale, shift (numpy PCG64(w.seed)).
    ``x`` is [T, C] uint16 bits; ``scale``/``shift`` are [B, C] fp32 or
    uint16 bits of the activation dtype.  ``tokens`` overrides T."""
    T = w.tokens if tokens is None else int(tokens)
    B = max(1, -(-T // w.seq))
    g = np.random.Generator(np.random.PCG64(w.seed))
    out = {"x": to_storage_bits(_normal(g, (T, w.hidden), w.scale), w.dtype)}
    for k in ("scale", "shift"):
        m = _normal(g, (B, w.hidden), w.mod_scale)
        out[k] = m if w.mod_dtype == "fp32" else to_storage_bits(m, w.mod_dtype)
    return out


def adaln_algorithmic_bytes(w: AdaLNWorkload, tokens: Optional[int] = None) -> int:
    """x read once and written once, plus every sample's scale and shift rows."""
    T = w.tokens if tokens is None else int(tokens)
    B = max(1, -(-T // w.seq))
    mes = 4 if w.mod_dtype == "fp32" else 2
    return 2 * T * w.hidden * 2 + 2 * B * w.hidden * mes


# --------------------------------------------------------------------------
# VAE group-norm + SiLU workloads ("fused qknorm rope Flux 2.0", section
# "Not in this PR — follow-ups": group_norm_silu for the VAE).  Decoder
# feature maps of a 1024 x 1024 image: 512 channels at 128^2 and 256^2,
# 256 at 512^2, 128 at 1024^2; 32 groups.

@dataclass(frozen=True)
class GroupNormWorkload:
    name: str
    n: int
    c: int
    h: int
    w: int
    groups: int = 32
    dtype: str = "bf16"
    scale: float = 1.0             # x = scale * N(0,1) + offset
    offset: float = 0.0
    eps: float = 1e-6
    seed: int = 0

    @property
    def elements(self) -> int:
        return self.n * self.c * self.h * self.w

    def with_(self, **kw) -> "GroupNormWorkload":
        return replace(self, **kw)


GN_WORKLOADS: Dict[str, GroupNormWorkload] = {
    "gn_vae_1x512x128x128": GroupNormWorkload("gn_vae_1x512x128x128", 1, 512, 128, 128),
    "gn_vae_1x512x256x256": GroupNormWorkload("gn_vae_1x512x256x256", 1, 512, 256, 256),
    "gn_vae_1x256x512x512": GroupNormWorkload("gn_vae_1x256x512x512", 1, 256, 512, 512),
    "gn_vae_1x128x1024x1024": GroupNormWorkload("gn_vae_1x128x1024x1024", 1, 128, 1024, 1024),
}


def make_gn_inputs(w: GroupNormWorkload) -> Dict[str, np.ndarray]:
    """Seeded instance: draw order x, gamma, beta.  x is [N, C, H, W] uint16
    bits; gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1), fp32 [C]."""
    g = np.random.Generator(np.random.PCG64(w.seed))
    x = _normal(g, (w.n, w.c, w.h, w.w), w.scale)
    if w.offset:
        x += np.float32(w.offset)
    return {
        "x": to_storage_bits(x, w.dtype),
        "gamma": (1.0 + 0.1 * g.standard_normal(w.c)).astype(np.float32),
        "beta": (0.1 * g.standard_normal(w.c)).astype(np.float32),
    }


def gn_algorithmic_bytes(w: GroupNormWorkload) -> int:
    """x read once and written once, plus gamma and beta."""
    return 2 * w.elements * 2 + 2 * w.c * 4
