"""Pins of the AdaLN oracle against torch's layer_norm, closed forms and
invariants (no GPU)."""
import numpy as np
import pytest
import torch

from oracle import adaln_oracle as A
from oracle import qknr_oracle as O


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _f32_bits(x):
    return x.astype(np.float32)


def test_zero_modulation_is_torch_layer_norm():
    g = _rng(1)
    x = (g.standard_normal((9, 512)) * 3 + 1.5).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xd = O.decode(bits, "bf16")
    zero = np.zeros((1, 512), np.float32)
    got = A.adaln_modulate(bits, "bf16", zero, zero, "fp32", 1e-6, 9)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(xd), (512,), eps=float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_modulation_is_layer_norm_affine_per_batch():
    # torch's affine layer norm with weight = 1 + scale[b], bias = shift[b]
    g = _rng(2)
    B, S, C = 3, 5, 256
    x = g.standard_normal((B * S, C)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    scale = (0.3 * g.standard_normal((B, C))).astype(np.float32)
    shift = (0.3 * g.standard_normal((B, C))).astype(np.float32)
    got = A.adaln_modulate(bits, "fp16", scale, shift, "fp32", 1e-5, S)
    xd = torch.from_numpy(O.decode(bits, "fp16"))
    for b in range(B):
        ref = torch.nn.functional.layer_norm(xd[b * S:(b + 1) * S], (C,),
                                             weight=torch.from_numpy(1.0 + scale[b].astype(np.float64)),
                                             bias=torch.from_numpy(shift[b].astype(np.float64)),
                                             eps=float(np.float32(1e-5))).numpy()
        np.testing.assert_allclose(got[b * S:(b + 1) * S], ref, rtol=1e-12, atol=1e-12)


def test_constant_row_gives_shift():
    C = 64
    x = np.full((2, C), 0x3FC0, np.uint16)      # bf16 1.5
    scale = np.full((1, C), 7.0, np.float32)
    shift = np.arange(C, dtype=np.float32)[None, :]
    got = A.adaln_modulate(x, "bf16", scale, shift, "fp32", 1e-6, 2)
    np.testing.assert_array_equal(got, np.broadcast_to(shift.astype(np.float64), (2, C)))


def test_alternating_row_closed_form():
    # x = [a, -a, a, -a, ...]: mean 0, variance a^2 -> +-a / sqrt(a^2 + eps)
    C, a, eps = 128, 2.0, 0.25
    row = np.where(np.arange(C) % 2 == 0, a, -a).astype(np.float32)
    bits = torch.from_numpy(row[None]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    zero = np.zeros((1, C), np.float32)
    got = A.adaln_modulate(bits, "bf16", zero, zero, "fp32", eps, 1)
    expect = np.where(np.arange(C) % 2 == 0, 1.0, -1.0) * a / np.sqrt(a * a + eps)
    np.testing.assert_allclose(got[0], expect, rtol=1e-15)


def test_shift_and_scale_invariance_of_the_normalisation():
    # with eps = 0, LN(alpha x + beta) = LN(x) for alpha > 0
    g = _rng(3)
    x = g.standard_normal((4, 256))
    np.testing.assert_allclose(A.layer_norm_rows(3.0 * x - 7.0, 0.0), A.layer_norm_rows(x, 0.0),
                               rtol=1e-10, atol=1e-12)
    y = A.layer_norm_rows(x, 0.0)
    np.testing.assert_allclose(y.mean(axis=-1), 0.0, atol=1e-14)
    np.testing.assert_allclose((y ** 2).mean(axis=-1), 1.0, rtol=1e-13)


def test_rows_select_batches():
    g = _rng(4)
    S, C = 4, 32
    x = torch.from_numpy(g.standard_normal((3 * S, C)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    scale = (0.5 * g.standard_normal((3, C))).astype(np.float32)
    shift = (0.5 * g.standard_normal((3, C))).astype(np.float32)
    full = A.adaln_modulate(bits, "bf16", scale, shift, "fp32", 1e-6, S)
    rows = np.array([11, 0, 5, 4])
    np.testing.assert_array_equal(A.adaln_modulate(bits, "bf16", scale, shift, "fp32", 1e-6, S, rows=rows),
                                  full[rows])
    # a row of batch 2 moved to batch 0 changes only through the modulation
    moved = A.adaln_modulate(bits[[9]], "bf16", scale, shift, "fp32", 1e-6, S)
    xn = A.layer_norm_rows(O.decode(bits[[9]], "bf16"), float(np.float32(1e-6)))
    np.testing.assert_allclose(moved, xn * (1 + scale[0].astype(np.float64)) + shift[0], rtol=1e-15)


def test_bf16_modulation_is_decoded_exactly():
    g = _rng(5)
    C = 64
    x = torch.from_numpy(g.standard_normal((2, C)).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    sc = torch.from_numpy((0.2 * g.standard_normal((1, C))).astype(np.float32)).to(torch.bfloat16)
    sh = torch.from_numpy((0.2 * g.standard_normal((1, C))).astype(np.float32)).to(torch.bfloat16)
    a = A.adaln_modulate(xb, "bf16", sc.view(torch.int16).numpy().view(np.uint16),
                         sh.view(torch.int16).numpy().view(np.uint16), "bf16", 1e-6, 2)
    b = A.adaln_modulate(xb, "bf16", sc.float().numpy(), sh.float().numpy(), "fp32", 1e-6, 2)
    np.testing.assert_array_equal(a, b)
