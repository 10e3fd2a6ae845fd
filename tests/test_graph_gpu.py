"""The fused calls inside a captured CUDA graph: a replay on new data in the
same buffers gives the bits an eager call gives.  For the fused group norm,
whose statistics records carry a tag that a replay cannot change, several
replays in a row on changing data each match an eager call."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()


def test_qk_norm_rope_replays_in_a_cuda_graph():
    w = I.WORKLOADS["wan_32760x40x128"]
    T = 4000
    a = I.make_inputs(w, tokens=T)
    b = I.make_inputs(w.with_(seed=5), tokens=T)
    gq, gk = torch.from_numpy(a["gamma_q"]).cuda(), torch.from_numpy(a["gamma_k"]).cuda()
    cos, sin = torch.from_numpy(a["cos"]).cuda(), torch.from_numpy(a["sin"]).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qkv = to_dev(a["qkv"], "bf16")
    # eager reference on the second input
    ref = to_dev(b["qkv"], "bf16")
    Q.qk_norm_rope_packed(ref, 40, 40, 40, 128, gq, gk, cos, sin, dev_status=status)
    # warm-up call (configures the kernel), then capture
    Q.qk_norm_rope_packed(qkv.clone(), 40, 40, 40, 128, gq, gk, cos, sin, dev_status=status)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Q.qk_norm_rope_packed(qkv, 40, 40, 40, 128, gq, gk, cos, sin, dev_status=status)
    torch.cuda.synchronize()
    qkv.copy_(to_dev(b["qkv"], "bf16"))
    g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(qkv.view(torch.int16), ref.view(torch.int16))


def test_chain_of_calls_with_the_prefetch_replays_in_a_cuda_graph():
    # three in-place calls in a row, each reading the previous output, after a
    # copy kernel that writes the input: captured, the calls keep their
    # programmatic dependent launch (graph edges) and the L2 prefetch before
    # each wait (64 rows per CTA), and a replay gives the eager bits
    w = I.WORKLOADS["wan_32760x40x128"]
    T = 9728
    a = I.make_inputs(w, tokens=T)
    gq, gk = torch.from_numpy(a["gamma_q"]).cuda(), torch.from_numpy(a["gamma_k"]).cuda()
    cos, sin = torch.from_numpy(a["cos"]).cuda(), torch.from_numpy(a["sin"]).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    src = to_dev(a["qkv"], "bf16")
    assert Q.query(Q.packed_args(src, 40, 40, 40, 128, gq, gk, cos, sin))["prefetch_rows"] > 0
    ref = src.clone()
    for _ in range(3):
        Q.qk_norm_rope_packed(ref, 40, 40, 40, 128, gq, gk, cos, sin, flags=Q.FLAG_NO_OVERLAP)
    qkv = torch.zeros_like(src)
    Q.qk_norm_rope_packed(qkv.clone(), 40, 40, 40, 128, gq, gk, cos, sin, dev_status=status)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            torch.bitwise_or(src.view(torch.int16), 0, out=qkv.view(torch.int16))
            for _ in range(3):
                Q.qk_norm_rope_packed(qkv, 40, 40, 40, 128, gq, gk, cos, sin, dev_status=status)
    for _ in range(2):
        qkv.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(qkv.view(torch.int16), ref.view(torch.int16))


def test_adaln_replays_in_a_cuda_graph():
    w = I.ADALN_WORKLOADS["adaln_flux2_2x4608x6144"]
    a = I.make_adaln_inputs(w, tokens=3000)
    b = I.make_adaln_inputs(w.with_(seed=9), tokens=3000)
    sc = to_dev(a["scale"], "bf16")
    sh = to_dev(a["shift"], "bf16")
    ref = to_dev(b["x"], "bf16")
    Q.adaln_modulate(ref, sc, sh, rows_per_batch=w.seq)
    x = to_dev(a["x"], "bf16")
    Q.adaln_modulate(x.clone(), sc, sh, rows_per_batch=w.seq)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Q.adaln_modulate(x, sc, sh, rows_per_batch=w.seq)
    x.copy_(to_dev(b["x"], "bf16"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))


def test_fused_group_norm_replays_in_a_cuda_graph():
    w = I.GroupNormWorkload("g", 1, 128, 96, 96, groups=32, scale=1.5, offset=0.2, seed=21)
    base = I.make_gn_inputs(w)
    gamma, beta = torch.from_numpy(base["gamma"]).cuda(), torch.from_numpy(base["beta"]).cuda()
    # eager references on three inputs
    refs = []
    for sd in (22, 23, 24):
        bits = I.make_gn_inputs(w.with_(seed=sd))["x"]
        r = to_dev(bits, "bf16")
        Q.group_norm_silu(r, w.groups, gamma, beta, eps=w.eps, mode="fused")
        refs.append((bits, r))
    x = to_dev(base["x"], "bf16")
    a = Q.gn_args(x, w.groups, gamma, beta, eps=w.eps, mode="fused")
    assert Q.gn_query(a)["kernel"].startswith("gn_fused")
    ws = torch.empty(Q.gn_workspace_bytes(a), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.group_norm_silu(x.clone(), w.groups, gamma, beta, eps=w.eps, mode="fused", workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Q.group_norm_silu(x, w.groups, gamma, beta, eps=w.eps, mode="fused", workspace=ws, dev_status=status)
    # replays in a row on changing data: each must match its eager call
    for bits, ref in refs:
        x.copy_(to_dev(bits, "bf16"))
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(x.view(torch.int16), ref.view(torch.int16))


def test_cluster_group_norm_replays_in_a_cuda_graph():
    # clusters of 4 CTAs per group; a graph keeps the launch's cluster shape
    w = I.GroupNormWorkload("gc", 3, 256, 128, 64, groups=32, scale=1.5, offset=0.2, seed=25)
    base = I.make_gn_inputs(w)
    gamma, beta = torch.from_numpy(base["gamma"]).cuda(), torch.from_numpy(base["beta"]).cuda()
    refs = []
    for sd in (26, 27):
        bits = I.make_gn_inputs(w.with_(seed=sd))["x"]
        r = to_dev(bits, "bf16")
        Q.group_norm_silu(r, w.groups, gamma, beta, eps=w.eps, mode="cluster")
        refs.append((bits, r))
    x = to_dev(base["x"], "bf16")
    a = Q.gn_args(x, w.groups, gamma, beta, eps=w.eps, mode="cluster")
    assert Q.gn_query(a)["kernel"].startswith("gn_cluster<bf16>, clusters of 4 CTAs")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Q.group_norm_silu(x, w.groups, gamma, beta, eps=w.eps, mode="cluster", dev_status=status)
    for bits, ref in refs:
        x.copy_(to_dev(bits, "bf16"))
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(x.view(torch.int16), ref.view(torch.int16))
