"""Group-norm + SiLU CUDA path vs the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import groupnorm_oracle as G
from tests.gpu_util import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()


def run(w, inp, out=False, **kw):
    x = to_dev(inp["x"], w.dtype)
    o = torch.empty_like(x) if out else None
    res = Q.group_norm_silu(x, w.groups, torch.from_numpy(inp["gamma"]).cuda(), torch.from_numpy(inp["beta"]).cuda(),
                            out=o, eps=w.eps, **kw)
    torch.cuda.synchronize()
    return res, x


@pytest.mark.parametrize("shape,groups", [((2, 64, 16, 16), 32), ((1, 32, 8, 8), 8), ((3, 12, 4, 6), 3),
                                          ((1, 512, 64, 64), 32), ((2, 4, 2, 4), 1)])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_small_shapes_full(shape, groups, dtype):
    w = I.GroupNormWorkload("s", *shape, groups=groups, dtype=dtype, scale=1.5, offset=0.3, seed=sum(shape))
    inp = I.make_gn_inputs(w)
    res, _ = run(w, inp)
    ref = G.group_norm_silu(inp["x"], dtype, groups, inp["gamma"], inp["beta"], w.eps)
    compare(to_bits(res), ref, dtype, "gn")


@pytest.mark.parametrize("name", list(I.GN_WORKLOADS))
def test_vae_shapes_sampled(name):
    w = I.GN_WORKLOADS[name]
    inp = I.make_gn_inputs(w)
    res, _ = run(w, inp)
    got = to_bits(res)
    g = np.random.Generator(np.random.PCG64(7))
    idx = tuple(g.integers(0, s, 4000) for s in (w.n, w.c, w.h, w.w))
    ref = G.group_norm_silu_at(inp["x"], w.dtype, w.groups, inp["gamma"], inp["beta"], w.eps, idx)
    compare(got[idx], ref, w.dtype, name)


def test_batches_and_in_place_give_the_same_bits():
    w = I.GroupNormWorkload("b", 2, 64, 32, 32, groups=32, seed=9)
    inp = I.make_gn_inputs(w)
    a, _ = run(w, inp)
    for kw in (dict(l2_batch_bytes=-1), dict(l2_batch_bytes=1), dict(l2_batch_bytes=100000)):
        b, src = run(w, inp, out=True, **kw)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), kw
        np.testing.assert_array_equal(to_bits(src), inp["x"])


@pytest.mark.parametrize("piece", [8, 1024, 8192, 32768, 1 << 20])
def test_piece_sizes_match_the_oracle(piece):
    # the piece size changes the order of the fp32 sums: each is checked
    w = I.GroupNormWorkload("p", 1, 64, 64, 64, groups=32, scale=3.0, offset=-2.0, seed=11)
    inp = I.make_gn_inputs(w)
    res, _ = run(w, inp, piece_elems=piece)
    ref = G.group_norm_silu(inp["x"], w.dtype, w.groups, inp["gamma"], inp["beta"], w.eps)
    compare(to_bits(res), ref, w.dtype, f"piece {piece}")


def test_degenerate_groups():
    w = I.GroupNormWorkload("d", 1, 8, 4, 4, groups=4, seed=12)
    inp = I.make_gn_inputs(w)
    x = I.storage_to_f32(inp["x"], "bf16").copy()
    x[0, 0:2] = 2.5                                 # constant group: silu(beta)
    x[0, 2:4] *= 1e-20                              # eps dominates
    x[0, 4:6] += 500.0                              # large mean
    inp["x"] = I.to_storage_bits(x, "bf16")
    res, _ = run(w, inp)
    ref = G.group_norm_silu(inp["x"], "bf16", 4, inp["gamma"], inp["beta"], w.eps)
    compare(to_bits(res), ref, "bf16", "degenerate")


def test_workspace_checks():
    x = torch.zeros((1, 32, 8, 8), dtype=torch.bfloat16, device="cuda")
    gm = torch.ones(32, device="cuda")
    a = Q.gn_args(x, 8, gm, gm)
    need = Q.gn_workspace_bytes(a)
    assert need == 8 * (1 + 1) * 16               # 8 spans, 1 piece each, plus the shift record
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(Q.QknrError) as e:
        Q.group_norm_silu(x, 8, gm, gm, workspace=small)
    assert e.value.status == 2
