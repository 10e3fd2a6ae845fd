"""Checks of the seeded input generator (shapes, determinism, RoPE tables)."""
import numpy as np
import pytest

from diffusion_transformer_qk_gb300 import inputs as I


def test_workload_shapes():
    w = I.WORKLOADS["wan_32760x40x128"]
    assert w.tokens == 21 * 30 * 52 == 32760
    assert sum(w.axes_dim) == 128
    f = I.WORKLOADS["flux2_2x4608x48x128"]
    assert f.tokens == 2 * 4608 and f.seq == 512 + 64 * 64
    assert not f.packed


def test_make_inputs_deterministic_and_rounded():
    w = I.WORKLOADS["tiny_256x24x64"]
    a = I.make_inputs(w)
    b = I.make_inputs(w)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])
    assert a["qkv"].shape == (256, 3 * 24 * 64) and a["qkv"].dtype == np.uint16
    assert a["cos"].shape == (256, 64) and a["cos"].dtype == np.float32
    x = I.storage_to_f32(a["qkv"], "bf16")
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1) < 0.02
    assert a["gamma_q"].dtype == np.float32 and not np.array_equal(a["gamma_q"], a["gamma_k"])


def test_scale_and_fp16():
    w = I.WORKLOADS["dense_4096x24x128"].with_(dtype="fp16")
    a = I.make_inputs(w, tokens=512)
    x = I.storage_to_f32(a["qkv"], "fp16")
    assert abs(float(x.std()) - 2.0) < 0.05


def test_separate_tensors():
    w = I.WORKLOADS["flux2_2x4608x48x128"]
    a = I.make_inputs(w, tokens=64)
    assert a["q"].shape == a["k"].shape == a["v"].shape == (64, 48 * 128)
    assert a["cos"].shape == (4608, 128)


@pytest.mark.parametrize("name", list(I.WORKLOADS))
def test_position_zero_has_no_turn(name):
    w = I.WORKLOADS[name]
    cos, sin = I.rope_table(w)
    if w.cos_dtype == "bf16":
        cos, sin = I.storage_to_f32(cos, "bf16"), I.storage_to_f32(sin, "bf16")
    # 1-D and Wan tables start at position 0 on every axis; FLUX text token 0 too
    np.testing.assert_array_equal(cos[0], 1.0)
    np.testing.assert_array_equal(sin[0], 0.0)


@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
def test_pair_members_share_an_angle(style):
    w = I.WORKLOADS["wan_32760x40x128"].with_(rope_style=style)
    cos, sin = I.rope_table(w)
    D = 128
    if style == "interleaved":
        a, b = cos[:, 0::2], cos[:, 1::2]
    else:
        a, b = cos[:, : D // 2], cos[:, D // 2:]
    np.testing.assert_array_equal(a, b)


def test_wan_axes_follow_raster_positions():
    w = I.WORKLOADS["wan_32760x40x128"]
    pos = I.positions_for(w)
    assert pos.shape == (32760, 3)
    t = 2 * 30 * 52 + 7 * 52 + 11
    assert tuple(pos[t]) == (2, 7, 11)
    ang = I.rope_half_angles(pos, w.axes_dim, w.theta)
    # pair 0 of each axis turns at frequency 1 by that axis' position
    assert ang[t, 0] == 2 and ang[t, 22] == 7 and ang[t, 43] == 11
    # the last pair of the frame axis: theta ** (-2*21/44)
    np.testing.assert_allclose(ang[t, 21], 2 * 10000.0 ** (-42 / 44), rtol=1e-15)


def test_flux_text_then_image_positions():
    w = I.WORKLOADS["flux2_2x4608x48x128"]
    pos = I.positions_for(w)
    assert tuple(pos[5]) == (5, 0, 0)
    assert tuple(pos[512]) == (0, 0, 0)
    assert tuple(pos[512 + 64 * 3 + 9]) == (0, 3, 9)


def test_expand_per_head():
    c = np.arange(12, dtype=np.float32).reshape(3, 4)
    e = I.expand_per_head(c, 5)
    assert e.shape == (3, 5, 4) and e.flags.c_contiguous
    for h in range(5):
        np.testing.assert_array_equal(e[:, h], c)


def test_algorithmic_bytes_wan():
    w = I.WORKLOADS["wan_32760x40x128"]
    # Q+K read and written once (bf16) + fp32 cos/sin rows + two fp32 gains
    assert I.algorithmic_bytes(w) == 1_341_849_600 + 33_546_240 + 1024
    assert I.algorithmic_bytes(w, v_copied=True) == 1_341_849_600 + 33_546_240 + 1024 + 670_924_800
    f = I.WORKLOADS["flux2_2x4608x48x128"]
    assert I.algorithmic_bytes(f, launches="q") == 226_492_416 + 4_718_592 + 512
