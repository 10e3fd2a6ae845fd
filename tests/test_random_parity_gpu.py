"""Seeded random configurations of the fused QK-norm + RoPE call vs the fp64
oracle: shapes, dtypes, pairing, table dtype and layout, batch-broadcast
tables, padded row strides, in place / out of place and launch knobs.
Per-head expanded tables hold a different angle for every head."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import qknr_oracle as O
from tests.gpu_util import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield
    assert Q.read_status() == 0


def random_case(seed):
    g = np.random.Generator(np.random.PCG64(1000 + seed))
    D = int(g.choice([64, 128]))
    hq = int(g.integers(0, 9))
    hk = int(g.integers(0 if hq else 1, 9))
    layout = "per_head_expanded" if (g.random() < 0.3 and hq and hk) else "shared_row"
    if layout == "per_head_expanded":
        hk = hq
    hv = int(g.integers(0, 5))
    T = int(g.integers(1, 700))
    return dict(
        D=D, hq=hq, hk=hk, hv=hv, T=T, layout=layout,
        dtype=str(g.choice(["bf16", "fp16"])), cos_dtype=str(g.choice(["fp32", "bf16"])),
        style=str(g.choice(["interleaved", "rotate_half"])),
        rows=int(g.choice([T, max(1, T // 3), T + 5])), pad=int(g.choice([0, 8, 64])),
        out=bool(g.random() < 0.4), scale=float(g.choice([1.0, 0.01, 30.0])),
        tune=dict(consumer_warps=int(g.choice([0, 1, 4, 12, 16])), stages=int(g.choice([0, 2, 3])),
                  ctas_per_sm=int(g.choice([0, 1, 2]))),
        seed=seed)


@pytest.mark.parametrize("seed", range(40))
def test_random_configuration(seed):
    c = random_case(seed)
    D, hq, hk, hv, T = c["D"], c["hq"], c["hk"], c["hv"], c["T"]
    g = np.random.Generator(np.random.PCG64(c["seed"]))
    width = (hq + hk + hv) * D
    x = (g.standard_normal((T, width)) * c["scale"]).astype(np.float32)
    bits = I.to_storage_bits(x, c["dtype"])
    if c["layout"] == "per_head_expanded":
        # [rows, H, D] with an angle of its own per (row, head, pair)
        cos, sin = I.per_head_tables(c["rows"], hq, D, c["style"], c["cos_dtype"], seed=5000 + seed)
    else:
        ang = g.uniform(-np.pi, np.pi, size=(c["rows"], D // 2))
        full = np.repeat(ang, 2, axis=1) if c["style"] == "interleaved" else np.concatenate([ang, ang], axis=1)
        cos, sin = np.cos(full).astype(np.float32), np.sin(full).astype(np.float32)
        if c["cos_dtype"] == "bf16":
            cos, sin = I.to_storage_bits(cos, "bf16"), I.to_storage_bits(sin, "bf16")
    gq = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)
    gk = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)

    def dev_tab(t):
        if c["cos_dtype"] == "fp32":
            return torch.from_numpy(t).cuda()
        return to_dev(t, "bf16")

    buf = torch.zeros((T, width + c["pad"]), dtype=torch.bfloat16 if c["dtype"] == "bf16" else torch.float16,
                      device="cuda")
    buf[:, :width] = to_dev(bits, c["dtype"])
    qkv = buf[:, :width]
    out = torch.zeros_like(buf)[:, :width] if c["out"] else None
    def call(tune):
        Q.qk_norm_rope_packed(qkv, hq, hk, hv, D, torch.from_numpy(gq).cuda(), torch.from_numpy(gk).cuda(),
                              dev_tab(cos), dev_tab(sin), out=out, rope_style=c["style"], cos_layout=c["layout"],
                              cos_rows=c["rows"], **tune)

    # launch knobs may be refused for the shape (rows too wide for the
    # ring): then the case runs with the default launch shape
    try:
        call(c["tune"])
    except Q.QknrError as e:
        assert e.status in (2, 4), e
        call({})
    torch.cuda.synchronize()
    got = to_bits(out if out is not None else qkv)
    ref = O.forward_packed(bits, c["dtype"], hq, hk, hv, D, gq, gk, 1e-6, cos, sin, c["cos_dtype"], c["style"],
                           c["layout"])
    if hq:
        compare(got[:, : hq * D], ref["q"], c["dtype"], f"Q {c}")
    if hk:
        compare(got[:, hq * D:(hq + hk) * D], ref["k"], c["dtype"], f"K {c}")
    if out is None:
        np.testing.assert_array_equal(got[:, (hq + hk) * D:], bits[:, (hq + hk) * D:])
    else:
        # V copied when out of place; padding untouched
        np.testing.assert_array_equal(got[:, (hq + hk) * D:], bits[:, (hq + hk) * D:])
        np.testing.assert_array_equal(to_bits(qkv), bits)
