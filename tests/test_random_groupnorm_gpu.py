"""Seeded random configurations of the group-norm + SiLU call vs the fp64
oracle: batch, groups, channels per group (past the 1280 channels that the
fused kernel stages in shared memory), ragged H*W, dtypes, value scale and
offset, in place / out of place; the fused path is also checked bit for bit
against the two-pass path with pieces of the same size, and groups that fit a
cluster also go through the cluster path (the automatic choice for them)."""
import re

import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import groupnorm_oracle as G
from tests.gpu_util import compare, to_bits, to_dev

pytestmark = pytest.mark.gpu

FUSED_PIECE = 12288          # elements per piece of the fused path


def cluster_part_bytes(L, c=16):
    return ((L + c - 1) // c + 7) // 8 * 8 * 2


def cluster_auto(L):
    """Whether the automatic choice takes the cluster path for groups of L
    elements: parts of at most 32 KB over at most 16 CTAs."""
    return cluster_part_bytes(L) <= 32 * 1024


def cluster_any(L):
    """Whether the cluster path can run: parts of at most 200 KB."""
    return cluster_part_bytes(L) <= 200 * 1024


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield
    assert Q.read_status() == 0


def random_case(seed):
    g = np.random.Generator(np.random.PCG64(5000 + seed))
    groups = int(g.choice([1, 2, 4, 8, 16, 32]))
    cpg = int(g.integers(1, 25))
    if seed % 6 == 0:
        groups, cpg = 32, int(g.integers(65, 90))          # C > 1280: gamma / beta from global memory
    n = int(g.integers(1, 4))
    c = groups * cpg
    # H*W a multiple of 8, sized so a case holds at most about 2 M elements
    budget = max(8, (2_000_000 // (n * c)) // 8 * 8)
    hw = int(g.integers(1, max(2, budget // 8) + 1)) * 8
    w = int(g.choice([d for d in (8, 16, 24, 40, 64, 104, 128) if hw % d == 0] or [8]))
    h = hw // w
    return I.GroupNormWorkload(f"r{seed}", n, c, h, w, groups=groups, dtype=str(g.choice(["bf16", "fp16"])),
                               scale=float(g.choice([1.0, 0.05, 8.0])), offset=float(g.choice([0.0, 0.5, -30.0])),
                               seed=seed), bool(g.random() < 0.4)


def call(x, w, inp, **kw):
    return Q.group_norm_silu(x, w.groups, torch.from_numpy(inp["gamma"]).cuda(),
                             torch.from_numpy(inp["beta"]).cuda(), eps=w.eps, **kw)


@pytest.mark.parametrize("seed", range(30))
def test_random_group_norm(seed):
    w, out_of_place = random_case(seed)
    inp = I.make_gn_inputs(w)
    x = to_dev(inp["x"], w.dtype)
    out = torch.empty_like(x) if out_of_place else None
    L = (w.c // w.groups) * w.h * w.w
    ones = torch.ones(w.c, device="cuda")
    info = Q.gn_query(Q.gn_args(x, w.groups, ones, ones))
    # the automatic choice: the cluster path for small groups whose clusters
    # all fit on the GPU at once (the query reports how many fit)
    auto_cluster = False
    if cluster_auto(L):
        resident = int(re.search(r"(\d+) resident", Q.gn_query(Q.gn_args(x, w.groups, ones, ones,
                                                                          mode="cluster"))["kernel"]).group(1))
        auto_cluster = w.n * w.groups <= resident
    assert info["kernel"].startswith("gn_cluster" if auto_cluster else "gn_fused"), info
    res = call(x, w, inp, out=out, mode="fused")
    two = call(to_dev(inp["x"], w.dtype), w, inp, mode="two_pass", piece_elems=FUSED_PIECE)
    torch.cuda.synchronize()
    assert torch.equal(res.view(torch.int16), two.view(torch.int16)), w
    if out_of_place:
        np.testing.assert_array_equal(to_bits(x), inp["x"])
    ref = G.group_norm_silu(inp["x"], w.dtype, w.groups, inp["gamma"], inp["beta"], w.eps)
    compare(to_bits(res), ref, w.dtype, w.name)
    if cluster_any(L):
        xc = to_dev(inp["x"], w.dtype)
        cl = call(xc, w, inp, out=torch.empty_like(xc) if out_of_place else None, mode="cluster")
        auto = call(to_dev(inp["x"], w.dtype), w, inp)
        torch.cuda.synchronize()
        if auto_cluster:
            assert torch.equal(cl.view(torch.int16), auto.view(torch.int16)), w
        if out_of_place:
            np.testing.assert_array_equal(to_bits(xc), inp["x"])
        compare(to_bits(cl), ref, w.dtype, w.name + " cluster")
