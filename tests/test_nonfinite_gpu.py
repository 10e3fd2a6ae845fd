"""Non-finite inputs stay where they are: a NaN or Inf in one head of one
token row makes that head's output non-finite and leaves every other head
and row exactly as without it; the same for a row of the AdaLN call and a
group of the group norm (on both group-norm paths, whose statistics of
different groups pass through shared workspace records)."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from tests.gpu_util import table_to_dev, to_bits, to_dev

pytestmark = pytest.mark.gpu

BF16_NAN, BF16_INF = 0x7FC0, 0x7F80


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()


def finite(bits):
    return (bits & 0x7F80) != 0x7F80                 # bf16: exponent not all ones


@pytest.mark.parametrize("bad", [BF16_NAN, BF16_INF])
def test_qk_nonfinite_stays_in_its_head(bad):
    w = I.WORKLOADS["wan_32760x40x128"].with_(n_heads_q=6, n_heads_k=6, n_heads_v=2)
    T, D = 500, 128
    inp = I.make_inputs(w, tokens=T)
    gq, gk = torch.from_numpy(inp["gamma_q"]).cuda(), torch.from_numpy(inp["gamma_k"]).cuda()
    cos, sin = table_to_dev(inp["cos"], "fp32"), table_to_dev(inp["sin"], "fp32")

    def run(bits):
        x = to_dev(bits, "bf16")
        Q.qk_norm_rope_packed(x, 6, 6, 2, D, gq, gk, cos, sin, rope_style=w.rope_style)
        torch.cuda.synchronize()
        return to_bits(x)

    clean = run(inp["qkv"])
    dirty_in = inp["qkv"].copy()
    t, h = 137, 8                                     # K head 2 of row 137
    dirty_in[t, h * D + 5] = bad
    dirty = run(dirty_in)
    head = np.zeros_like(clean, dtype=bool)
    head[t, h * D:(h + 1) * D] = True
    assert not np.any(finite(dirty[head]) & (dirty[head] == clean[head]))   # the head is poisoned
    np.testing.assert_array_equal(dirty[~head], clean[~head])                 # nothing else moved


def test_adaln_nonfinite_stays_in_its_row():
    w = I.AdaLNWorkload("n", 2, 300, 3072, mod_dtype="fp32", seed=61)
    inp = I.make_adaln_inputs(w)
    sc, sh = torch.from_numpy(inp["scale"]).cuda(), torch.from_numpy(inp["shift"]).cuda()

    def run(bits):
        x = to_dev(bits, "bf16")
        Q.adaln_modulate(x, sc, sh, rows_per_batch=w.seq, eps=w.eps)
        torch.cuda.synchronize()
        return to_bits(x)

    clean = run(inp["x"])
    dirty_in = inp["x"].copy()
    dirty_in[299, 17] = BF16_NAN                      # the last row of sample 0
    dirty = run(dirty_in)
    assert not np.any(finite(dirty[299]))
    others = np.arange(w.tokens) != 299
    np.testing.assert_array_equal(dirty[others], clean[others])


@pytest.mark.parametrize("mode", ["fused", "two_pass", "cluster"])
def test_group_norm_nonfinite_stays_in_its_group(mode):
    w = I.GroupNormWorkload("n", 2, 64, 96, 96, groups=32, seed=62)
    inp = I.make_gn_inputs(w)
    gm, bt = torch.from_numpy(inp["gamma"]).cuda(), torch.from_numpy(inp["beta"]).cuda()

    def run(bits):
        x = to_dev(bits, "bf16")
        Q.group_norm_silu(x, w.groups, gm, bt, eps=w.eps, mode=mode)
        torch.cuda.synchronize()
        return to_bits(x)

    clean = run(inp["x"])
    dirty_in = inp["x"].copy()
    dirty_in[1, 10, 40, 40] = BF16_NAN                # sample 1, group 5 (channels 10-11)
    dirty = run(dirty_in)
    group = np.zeros(clean.shape, dtype=bool)
    group[1, 10:12] = True
    assert not np.any(finite(dirty[group]))
    np.testing.assert_array_equal(dirty[~group], clean[~group])
