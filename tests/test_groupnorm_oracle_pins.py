"""Pins of the group-norm + SiLU oracle against torch's group_norm and silu,
closed forms and invariants (no GPU)."""
import numpy as np
import torch

from oracle import groupnorm_oracle as G
from oracle import qknr_oracle as O


def _bits(x, dtype="bf16"):
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(tdt).view(torch.int16).numpy().view(
        np.uint16)


def test_matches_torch_group_norm_then_silu():
    g = np.random.Generator(np.random.PCG64(1))
    N, C, H, W, groups = 2, 64, 5, 7, 8
    x = _bits(g.standard_normal((N, C, H, W)) * 2 + 0.5)
    gamma = (1 + 0.2 * g.standard_normal(C)).astype(np.float32)
    beta = (0.2 * g.standard_normal(C)).astype(np.float32)
    got = G.group_norm_silu(x, "bf16", groups, gamma, beta, 1e-6)
    xt = torch.from_numpy(O.decode(x, "bf16"))
    y = torch.nn.functional.group_norm(xt, groups, torch.from_numpy(gamma.astype(np.float64)),
                                       torch.from_numpy(beta.astype(np.float64)), eps=float(np.float32(1e-6)))
    ref = torch.nn.functional.silu(y).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_constant_group_gives_silu_of_beta():
    N, C, H, W = 1, 4, 3, 3
    x = np.full((N, C, H, W), 0x4040, np.uint16)          # bf16 3.0
    gamma = np.full(C, 5.0, np.float32)
    beta = np.array([0.0, 1.0, -2.0, 30.0], np.float32)
    got = G.group_norm_silu(x, "bf16", 2, gamma, beta, 1e-6)
    b = beta.astype(np.float64)
    expect = b / (1 + np.exp(-b))
    np.testing.assert_allclose(got[0, :, 1, 1], expect, rtol=1e-15)
    assert got[0, 0].max() == 0.0                          # silu(0) = 0


def test_silu_closed_forms():
    # unit gain, zero bias: y = normalised x; silu(y) = y * sigmoid(y)
    x = _bits(np.array([[[[1.0, -1.0], [1.0, -1.0]]]]))    # mean 0, var 1
    got = G.group_norm_silu(x, "bf16", 1, np.ones(1, np.float32), np.zeros(1, np.float32), 0.0)
    s = 1.0 / (1.0 + np.exp(-1.0))
    np.testing.assert_allclose(got[0, 0], [[s, -(1 - s)], [s, -(1 - s)]], rtol=1e-15)


def test_normalisation_invariant_to_affine_input_change():
    g = np.random.Generator(np.random.PCG64(2))
    x = g.standard_normal((1, 8, 4, 4))
    gamma, beta = np.ones(8, np.float32), np.zeros(8, np.float32)
    a = G.group_norm_silu(_bits(x, "fp16"), "fp16", 4, gamma, beta, 0.0)
    # the fp16 values of 4*x + 3 are not exactly 4*(fp16 x) + 3, so compare on
    # values built from the same stored numbers
    xs = O.decode(_bits(x, "fp16"), "fp16")
    b = G.group_norm_silu(_bits(xs * 4.0, "fp16"), "fp16", 4, gamma, beta, 0.0)   # power-of-two scale is exact
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_groups_are_independent():
    g = np.random.Generator(np.random.PCG64(3))
    x = g.standard_normal((2, 6, 3, 3)).astype(np.float32)
    gamma = np.ones(6, np.float32); beta = np.zeros(6, np.float32)
    full = G.group_norm_silu(_bits(x), "bf16", 3, gamma, beta, 1e-6)
    x2 = x.copy(); x2[1, 2:4] *= 100.0                      # change sample 1, group 1 only
    part = G.group_norm_silu(_bits(x2), "bf16", 3, gamma, beta, 1e-6)
    mask = np.ones_like(full, bool); mask[1, 2:4] = False
    np.testing.assert_array_equal(full[mask], part[mask])


def test_sampled_values_equal_the_full_oracle():
    g = np.random.Generator(np.random.PCG64(4))
    N, C, H, W, groups = 2, 16, 6, 5, 4
    x = _bits(g.standard_normal((N, C, H, W)))
    gamma = (1 + 0.1 * g.standard_normal(C)).astype(np.float32)
    beta = (0.1 * g.standard_normal(C)).astype(np.float32)
    full = G.group_norm_silu(x, "bf16", groups, gamma, beta, 1e-6)
    idx = tuple(g.integers(0, s, 40) for s in (N, C, H, W))
    np.testing.assert_allclose(G.group_norm_silu_at(x, "bf16", groups, gamma, beta, 1e-6, idx), full[idx],
                               rtol=1e-13, atol=1e-15)
