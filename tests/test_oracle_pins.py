"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a library routine (torch RMSNorm, numpy
complex multiplication, torch/numpy casts), a hand-worked closed form, or an
invariant the method must keep.  Together they catch a dropped eps, eps in
the wrong place, a wrong rotation sign or partner, gamma at the wrong index,
a transposed table, a wrong batch broadcast and wrong decoding/rounding.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import qknr_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_d4.json")


def _rng(seed=0):
    return np.random.Generator(np.random.PCG64(seed))


# --------------------------------------------------------------------------
# decoding and rounding vs library casts

def test_decode_bf16_matches_torch():
    g = _rng(1)
    bits = g.integers(0, 1 << 16, size=200_000, dtype=np.uint16)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]                       # drop inf/nan patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.decode(bits, "bf16"), ref)


def test_decode_fp16_matches_torch():
    g = _rng(2)
    bits = g.integers(0, 1 << 16, size=200_000, dtype=np.uint16)
    exp = (bits >> 10) & 0x1F
    bits = bits[exp != 0x1F]
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.decode(bits, "fp16"), ref)


def _fp32_probe_values(n, seed):
    g = _rng(seed)
    parts = [
        g.standard_normal(n).astype(np.float32),
        (g.standard_normal(n) * 1e3).astype(np.float32),
        (g.standard_normal(n) * 1e-3).astype(np.float32),
        (g.standard_normal(n) * 1e-6).astype(np.float32),      # fp16 subnormal range
        g.integers(0, 1 << 31, size=n, dtype=np.uint32).view(np.float32),  # arbitrary patterns
    ]
    v = np.concatenate(parts)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_round_rne_matches_torch_cast_on_fp32_values(dtype):
    v = _fp32_probe_values(2_000_000, 3)
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    ref = torch.from_numpy(v).to(tdt).view(torch.int16).numpy().view(np.uint16)
    got = O.round_rne(v.astype(np.float64), dtype)
    np.testing.assert_array_equal(got, ref)


def test_round_rne_fp16_matches_numpy_on_fp64_values():
    g = _rng(4)
    v = np.concatenate([g.standard_normal(2_000_000), g.standard_normal(500_000) * 2e4,
                        g.standard_normal(500_000) * 1e-5, [65504.0, 65519.99, 65520.0, 1e6, -1e6]])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(O.round_rne(v, "fp16"), ref)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_round_rne_ties_go_to_even(dtype):
    # exact midpoints between neighbouring finite positive values k and k+1
    g = _rng(5)
    top = 0x7F7F if dtype == "bf16" else 0x7BFF
    k = g.integers(1, top, size=100_000).astype(np.uint16)
    lo = O.decode(k, dtype)
    hi = O.decode((k + 1).astype(np.uint16), dtype)
    mid = (lo + hi) / 2                                 # exact in fp64
    expect = np.where(k % 2 == 0, k, k + 1).astype(np.uint16)
    np.testing.assert_array_equal(O.round_rne(mid, dtype), expect)
    np.testing.assert_array_equal(O.round_rne(-mid, dtype), expect | np.uint16(0x8000))
    # just off the midpoint rounds to the nearer neighbour
    up = np.nextafter(mid, np.inf)
    np.testing.assert_array_equal(O.round_rne(up, dtype), (k + 1).astype(np.uint16))


# --------------------------------------------------------------------------
# hand-worked closed forms at head_dim 4

def _golden_cases():
    with open(GOLDEN) as f:
        data = json.load(f)
    for case in data["cases"]:
        for style, expected in case["expected"].items():
            yield pytest.param(case, style, expected, id=f"{case['name']}-{style}")


@pytest.mark.parametrize("case,style,expected", list(_golden_cases()))
def test_hand_worked_d4(case, style, expected):
    x = np.array(case["x"], dtype=np.float64).reshape(1, 1, 4)
    cos = np.array(case["cos"], dtype=np.float64).reshape(1, 4)
    sin = np.array(case["sin"], dtype=np.float64).reshape(1, 4)
    o = O.qk_norm_rope(x, np.array(case["gamma"], float), case["eps"], cos, sin, style)
    np.testing.assert_allclose(o.reshape(4), expected, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# library routines: torch RMSNorm and complex multiplication

def _torch_rmsnorm(x, gamma, eps):
    t = torch.from_numpy(x)
    return torch.nn.functional.rms_norm(t, (x.shape[-1],), weight=torch.from_numpy(gamma), eps=eps).numpy()


@pytest.mark.parametrize("D", [4, 64, 128])
def test_no_rotation_is_torch_rms_norm(D):
    g = _rng(6)
    x = g.standard_normal((7, 3, D)) * 3
    gamma = 1 + 0.1 * g.standard_normal(D)
    eps = 1e-6
    ones, zeros = np.ones((7, D)), np.zeros((7, D))
    for style in ("interleaved", "rotate_half"):
        o = O.qk_norm_rope(x, gamma, eps, ones, zeros, style)
        np.testing.assert_allclose(o, _torch_rmsnorm(x, gamma, eps), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("D", [4, 64, 128])
@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
def test_rotation_is_complex_multiplication(D, style):
    g = _rng(7)
    T, H = 5, 3
    x = g.standard_normal((T, H, D))
    gamma = 1 + 0.3 * g.standard_normal(D)          # distinct per dim: pins the gain index
    eps = 1e-3
    theta = g.uniform(-math.pi, math.pi, size=(T, D // 2))  # distinct per token: pins row indexing
    y = _torch_rmsnorm(x, gamma, eps)
    if style == "interleaved":
        a, b = y[..., 0::2], y[..., 1::2]
        cos = np.repeat(np.cos(theta), 2, axis=1)
        sin = np.repeat(np.sin(theta), 2, axis=1)
    else:
        a, b = y[..., : D // 2], y[..., D // 2:]
        cos = np.concatenate([np.cos(theta)] * 2, axis=1)
        sin = np.concatenate([np.sin(theta)] * 2, axis=1)
    z = (a + 1j * b) * np.exp(1j * theta)[:, None, :]
    o = O.qk_norm_rope(x, gamma, eps, cos, sin, style)
    if style == "interleaved":
        oa, ob = o[..., 0::2], o[..., 1::2]
    else:
        oa, ob = o[..., : D // 2], o[..., D // 2:]
    np.testing.assert_allclose(oa, z.real, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ob, z.imag, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# invariants

def _fp64_tables(theta, style):
    if style == "interleaved":
        return np.repeat(np.cos(theta), 2, axis=1), np.repeat(np.sin(theta), 2, axis=1)
    return np.concatenate([np.cos(theta)] * 2, axis=1), np.concatenate([np.sin(theta)] * 2, axis=1)


@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
def test_rotation_preserves_pair_norms(style):
    g = _rng(8)
    T, H, D = 9, 4, 128
    x = g.standard_normal((T, H, D))
    gamma = 1 + 0.1 * g.standard_normal(D)
    theta = g.uniform(0, 100, size=(T, D // 2))
    cos, sin = _fp64_tables(theta, style)
    y = O.rms_norm_heads(x, gamma, 1e-6)
    o = O.qk_norm_rope(x, gamma, 1e-6, cos, sin, style)
    p, _ = O.pair_table(D, style)
    np.testing.assert_allclose(o ** 2 + o[..., p] ** 2, y ** 2 + y[..., p] ** 2, rtol=1e-12)


@pytest.mark.parametrize("eps", [1e-6, 0.25, 4.0])
def test_unit_gain_head_rms_closed_form(eps):
    # gamma = 1: rms(y) = sqrt(ms / (ms + eps)); a rotation keeps it.
    g = _rng(9)
    T, H, D = 6, 5, 64
    x = g.standard_normal((T, H, D)) * g.uniform(0.1, 3, size=(T, H, 1))
    ms = np.mean(x ** 2, axis=-1)
    theta = g.uniform(0, 10, size=(T, D // 2))
    cos, sin = _fp64_tables(theta, "rotate_half")
    o = O.qk_norm_rope(x, np.ones(D), eps, cos, sin, "rotate_half")
    rms = np.sqrt(np.mean(o ** 2, axis=-1))
    np.testing.assert_allclose(rms, np.sqrt(ms / (ms + eps)), rtol=1e-12)


@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
def test_relative_position_property(style):
    # <o_q(p), o_k(p')> depends only on p - p' for 1-D RoPE tables.
    g = _rng(10)
    D = 64
    xq = g.standard_normal((1, 1, D))
    xk = g.standard_normal((1, 1, D))
    gq, gk = 1 + 0.1 * g.standard_normal(D), 1 + 0.1 * g.standard_normal(D)
    freq = 10000.0 ** (-2.0 * np.arange(D // 2) / D)

    def at(x, gm, p):
        cos, sin = _fp64_tables(np.array([[p]]) * freq[None, :], style)
        return O.qk_norm_rope(x, gm, 1e-6, cos, sin, style).reshape(D)

    for delta in (0, 3, -17, 250):
        dots = [at(xq, gq, p) @ at(xk, gk, p - delta) for p in (0, 5, 41, 1000)]
        np.testing.assert_allclose(dots, dots[0], rtol=1e-9, atol=1e-12)
    # and it does change with the offset (the rotation is not a no-op)
    assert abs(at(xq, gq, 10) @ at(xk, gk, 0) - at(xq, gq, 10) @ at(xk, gk, 10)) > 1e-6


def test_interleaved_is_permuted_rotate_half():
    g = _rng(11)
    T, H, D = 4, 3, 64
    x = g.standard_normal((T, H, D))
    gamma = 1 + 0.2 * g.standard_normal(D)
    theta = g.uniform(0, 7, size=(T, D // 2))
    cos_il, sin_il = _fp64_tables(theta, "interleaved")
    P = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])  # rh index i <- il index P[i]
    o_il = O.qk_norm_rope(x, gamma, 1e-6, cos_il, sin_il, "interleaved")
    o_rh = O.qk_norm_rope(x[..., P], gamma[P], 1e-6, cos_il[:, P], sin_il[:, P], "rotate_half")
    # equal up to the order of the sum of squares
    np.testing.assert_allclose(o_rh, o_il[..., P], rtol=1e-14, atol=1e-15)


def test_shared_row_equals_expanded_exactly():
    g = _rng(12)
    T, H, D = 6, 5, 128
    x = g.standard_normal((T, H, D))
    gamma = 1 + 0.1 * g.standard_normal(D)
    cos = g.uniform(-1, 1, size=(T, D))
    sin = g.uniform(-1, 1, size=(T, D))
    ce = np.broadcast_to(cos[:, None, :], (T, H, D)).copy()
    se = np.broadcast_to(sin[:, None, :], (T, H, D)).copy()
    for style in ("interleaved", "rotate_half"):
        a = O.qk_norm_rope(x, gamma, 1e-6, cos, sin, style, "shared_row")
        b = O.qk_norm_rope(x, gamma, 1e-6, ce, se, style, "per_head_expanded")
        np.testing.assert_array_equal(a, b)


def test_expanded_table_is_read_per_head():
    # a per-head table that differs between heads must change those heads only
    g = _rng(13)
    T, H, D = 3, 4, 64
    x = g.standard_normal((T, H, D))
    gamma = np.ones(D)
    cos = np.ones((T, H, D)); sin = np.zeros((T, H, D))
    cos[:, 2], sin[:, 2] = 0.0, 1.0                      # quarter turn on head 2 only
    o = O.qk_norm_rope(x, gamma, 0.0, cos, sin, "interleaved", "per_head_expanded")
    y = O.rms_norm_heads(x, gamma, 0.0)
    np.testing.assert_array_equal(o[:, [0, 1, 3]], y[:, [0, 1, 3]])
    np.testing.assert_array_equal(o[:, 2, 0::2], -y[:, 2, 1::2])
    np.testing.assert_array_equal(o[:, 2, 1::2], y[:, 2, 0::2])


def test_table_row_is_token_mod_rows():
    # a batch of two identical sequences against one table: both halves agree,
    # and row t uses table row t % rows
    g = _rng(14)
    S, H, D = 5, 2, 64
    xs = g.standard_normal((S, H, D))
    x = np.concatenate([xs, xs])
    cos = g.uniform(-1, 1, (S, D)); sin = g.uniform(-1, 1, (S, D))
    o = O.qk_norm_rope(x, np.ones(D), 1e-6, cos, sin, "rotate_half")
    np.testing.assert_array_equal(o[:S], o[S:])
    # evaluating selected rows gives the same rows
    rows = np.array([7, 2, 9])
    sub = O.qk_norm_rope(x[rows], np.ones(D), 1e-6, cos, sin, "rotate_half", rows=rows)
    np.testing.assert_array_equal(sub, o[rows])


def test_forward_packed_splits_heads_and_keeps_v():
    g = _rng(15)
    T, hq, hk, hv, D = 10, 3, 2, 4, 64
    bits = g.integers(0, 1 << 16, size=(T, (hq + hk + hv) * D), dtype=np.uint16)
    bits &= np.uint16(0xBFFF)                   # keep exponents finite and moderate
    gq = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)
    gk = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)
    cos = g.uniform(-1, 1, (T, D)).astype(np.float32)
    sin = g.uniform(-1, 1, (T, D)).astype(np.float32)
    r = O.forward_packed(bits, "bf16", hq, hk, hv, D, gq, gk, 1e-6, cos, sin, "fp32", "interleaved")
    x = O.decode(bits, "bf16")
    eps = float(np.float32(1e-6))
    c, s = cos.astype(np.float64), sin.astype(np.float64)
    np.testing.assert_array_equal(
        r["q"], O.qk_norm_rope(x[:, : hq * D].reshape(T, hq, D), gq.astype(float), eps, c, s, "interleaved"))
    np.testing.assert_array_equal(
        r["k"], O.qk_norm_rope(x[:, hq * D:(hq + hk) * D].reshape(T, hk, D), gk.astype(float), eps, c, s,
                               "interleaved"))
    np.testing.assert_array_equal(r["v"], bits[:, (hq + hk) * D:])
    # Q uses gamma_q and K uses gamma_k: swapping them changes the result
    r2 = O.forward_packed(bits, "bf16", hq, hk, hv, D, gk, gq, 1e-6, cos, sin, "fp32", "interleaved")
    assert not np.array_equal(r["q"], r2["q"])
