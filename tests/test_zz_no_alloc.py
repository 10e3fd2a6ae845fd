"""The group-norm + SiLU entry point for callers that cannot allocate device
memory — a plugin or runtime with no allocator on its execution path, a
fixed device-memory budget, or a workspace size fixed before the shapes
were known.  Its statistics scratch is a fixed array inside the library, so
it is checked against the entry point that takes a caller workspace and
against the fp64 oracle, on calls in a row that each run on the scratch the
previous one left behind: the fused path, then the two-pass path on another
shape."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import groupnorm_oracle as G
from tests.gpu_util import TOL, compare, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()


def test_no_alloc_entry_point_matches_the_workspace_one_twice_in_a_row():
    # (workload, launch options): two fused calls, then a two-pass call of
    # another shape, each on the scratch the call before it left behind
    cases = [(I.GroupNormWorkload("a", 2, 128, 64, 64, groups=32, scale=2.0, offset=0.5, seed=31), {}),
             (I.GroupNormWorkload("b", 1, 64, 32, 48, groups=16, dtype="fp16", seed=32), {}),
             (I.GroupNormWorkload("c", 2, 96, 40, 40, groups=24, dtype="fp16", scale=1.5, offset=-0.25, seed=33),
              dict(mode="two_pass", piece_elems=4096))]
    for w, opts in cases:
        inp = I.make_gn_inputs(w)
        x = to_dev(inp["x"], w.dtype)
        gamma = torch.from_numpy(inp["gamma"]).cuda()
        beta = torch.from_numpy(inp["beta"]).cuda()
        ref = torch.empty_like(x)
        Q.group_norm_silu(x, w.groups, gamma, beta, out=ref, eps=w.eps, **opts)
        out = torch.empty_like(x)
        a = Q.gn_args(x, w.groups, gamma, beta, out=out, eps=w.eps, **opts)
        assert Q.gn_workspace_bytes(a) <= Q.GN_NOALLOC_SCRATCH_BYTES
        if opts:
            assert Q.gn_query(a)["kernel"].startswith("gn_stats")
        Q.gn_launch_noalloc(a)
        torch.cuda.synchronize()
        got = to_bits(out).astype(np.int32)
        exp = to_bits(ref).astype(np.int32)
        diff = np.abs(I.storage_to_f32(to_bits(out), w.dtype) - I.storage_to_f32(to_bits(ref), w.dtype))
        assert float(diff.max()) <= TOL[w.dtype]
        np.testing.assert_array_equal(got, exp)       # the same kernels on the same pieces
        np.testing.assert_array_equal(to_bits(x), inp["x"])
        oracle = G.group_norm_silu(inp["x"], w.dtype, w.groups, inp["gamma"], inp["beta"], w.eps)
        compare(to_bits(out), oracle, w.dtype, f"no-alloc {w.name}")


def test_no_alloc_entry_point_rejects_shapes_beyond_its_scratch():
    # 8-element pieces of a 1 x 32 x 256 x 256 tensor need 32 * (8192 + 1) * 16
    # bytes of statistics: more than the fixed scratch holds
    x = torch.zeros((1, 32, 256, 256), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(32, device="cuda")
    a = Q.gn_args(x, 32, g, g, piece_elems=8)
    assert Q.gn_workspace_bytes(a) > Q.GN_NOALLOC_SCRATCH_BYTES
    with pytest.raises(Q.QknrError) as e:
        Q.gn_launch_noalloc(a)
    assert e.value.status == 4
