"""Seeded stress cases for the three kernels against the fp64 oracles:
values with spikes at random positions and first, means far from zero
against the spread, tiny and mixed-scale values, zero heads, gains of
either sign, eps up to 1e-2.  Every output must be within 1 ulp of the
correctly rounded oracle value (compare_ulps), in bf16 and fp16."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import adaln_oracle as A
from oracle import groupnorm_oracle as G
from oracle import qknr_oracle as O
from tests.gpu_util import compare_ulps, to_bits, to_dev

pytestmark = pytest.mark.gpu
BOUND = {"bf16": 1, "fp16": 1}


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield
    assert Q.read_status() == 0


def values(g, shape, dtype):
    """Seeded test values of one of five kinds, as storage bits."""
    kind = g.choice(["normal", "mean", "spikes", "tiny", "mixed"])
    scale = float(g.choice([1.0, 0.05, 20.0]))
    x = g.standard_normal(shape) * scale
    if kind == "mean":
        x += float(g.choice([-30.0, 8.0, 200.0])) * scale      # a mean of 8 to 200 spreads
    elif kind == "spikes":
        n = max(1, x.size // 5000)
        idx = g.integers(0, x.size, n)
        x.reshape(-1)[idx] = g.choice([-1, 1], n) * scale * float(g.choice([30.0, 300.0]))
        if g.random() < 0.5:
            x.reshape(-1)[0] = scale * 300.0
    elif kind == "tiny":
        x *= 1e-3
    elif kind == "mixed":
        x[..., : x.shape[-1] // 2] *= 50.0
    lim = 6e4 if dtype == "fp16" else 1e30
    return I.to_storage_bits(np.clip(x, -lim, lim).astype(np.float32), dtype), kind


@pytest.mark.parametrize("seed", range(100))
def test_gn_stress(seed):
    g = np.random.Generator(np.random.PCG64(90000 + seed))
    dtype = str(g.choice(["bf16", "fp16"]))
    groups = int(g.choice([1, 4, 32])); cpg = int(g.integers(1, 9)); n = int(g.integers(1, 3))
    c = groups * cpg
    hw = int(g.integers(1, max(2, 400_000 // (n * c * 8)))) * 8
    w_ = int(g.choice([d for d in (8, 16, 40, 64) if hw % d == 0] or [8])); h = hw // w_
    xb, kind = values(g, (n, c, h, w_), dtype)
    gamma = (float(g.choice([1.0, -2.0, 0.3])) * (1 + 0.1 * g.standard_normal(c))).astype(np.float32)
    beta = (float(g.choice([0.0, 0.5, -3.0])) + 0.1 * g.standard_normal(c)).astype(np.float32)
    eps = float(g.choice([1e-6, 1e-3]))
    g.choice(["fused", "two_pass"])                  # (kept so the seeds draw what they always drew)
    ref = G.group_norm_silu(xb, dtype, groups, gamma, beta, eps)
    for mode in ("fused", "two_pass", "cluster"):
        res = Q.group_norm_silu(to_dev(xb, dtype), groups, torch.from_numpy(gamma).cuda(),
                                torch.from_numpy(beta).cuda(), eps=eps, mode=mode)
        torch.cuda.synchronize()
        compare_ulps(to_bits(res), ref, dtype, BOUND[dtype], f"gn {dtype} {kind} {mode} {(n, c, h, w_)} G{groups}")


@pytest.mark.parametrize("seed", range(100))
def test_adaln_stress(seed):
    g = np.random.Generator(np.random.PCG64(91000 + seed))
    dtype = str(g.choice(["bf16", "fp16"]))
    C = int(g.choice([64, 1000, 3072, 5120, 6144, 12288]))
    T = int(g.integers(1, 200)); rpb = int(g.choice([T, max(1, T // 3)]))
    B = -(-T // rpb)
    xb, kind = values(g, (T, C), dtype)
    ms = float(g.choice([0.1, 1.0]))
    sc = (ms * g.standard_normal((B, C))).astype(np.float32)
    sh = (ms * g.standard_normal((B, C))).astype(np.float32)
    eps = float(g.choice([1e-6, 1e-3]))
    res = Q.adaln_modulate(to_dev(xb, dtype), torch.from_numpy(sc).cuda(), torch.from_numpy(sh).cuda(),
                           rows_per_batch=rpb, eps=eps)
    torch.cuda.synchronize()
    ref = A.adaln_modulate(xb, dtype, sc, sh, "fp32", eps, rpb)
    compare_ulps(to_bits(res), ref, dtype, BOUND[dtype], f"adaln {dtype} {kind} C{C} T{T}")


@pytest.mark.parametrize("seed", range(100))
def test_qk_stress(seed):
    g = np.random.Generator(np.random.PCG64(92000 + seed))
    dtype = str(g.choice(["bf16", "fp16"]))
    D = int(g.choice([64, 128])); hq = int(g.integers(1, 9)); hk = int(g.integers(0, 9)); hv = int(g.integers(0, 3))
    T = int(g.integers(1, 500))
    xb, kind = values(g, (T, (hq + hk + hv) * D), dtype)
    if g.random() < 0.2:                                # a zero head
        xb[:, :D] = 0
    style = str(g.choice(["interleaved", "rotate_half"]))
    ang = g.uniform(-np.pi, np.pi, size=(T, D // 2))
    full = np.repeat(ang, 2, axis=1) if style == "interleaved" else np.concatenate([ang, ang], axis=1)
    cos, sin = np.cos(full).astype(np.float32), np.sin(full).astype(np.float32)
    gs = float(g.choice([1.0, 3.0, 0.2]))
    gq = (gs * (1 + 0.1 * g.standard_normal(D))).astype(np.float32)
    gk = (gs * (1 + 0.1 * g.standard_normal(D))).astype(np.float32)
    eps = float(g.choice([1e-6, 1e-2]))
    x = to_dev(xb, dtype)
    Q.qk_norm_rope_packed(x, hq, hk, hv, D, torch.from_numpy(gq).cuda(), torch.from_numpy(gk).cuda(),
                          torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(), rope_style=style, eps=eps)
    torch.cuda.synchronize()
    got = to_bits(x)
    ref = O.forward_packed(xb, dtype, hq, hk, hv, D, gq, gk, eps, cos, sin, "fp32", style)
    compare_ulps(got[:, :hq * D], ref["q"], dtype, BOUND[dtype], f"qk Q {dtype} {kind}")
    if hk:
        compare_ulps(got[:, hq * D:(hq + hk) * D], ref["k"], dtype, BOUND[dtype], f"qk K {dtype} {kind}")
