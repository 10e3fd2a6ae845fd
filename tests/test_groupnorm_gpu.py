"""Group-norm + SiLU CUDA path vs the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import groupnorm_oracle as G
from tests.gpu_util import compare, compare_ulps, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield
    assert Q.read_status() == 0, "a kernel reported a wait timeout"


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
    # 8 spans, 1 piece each, plus the shift record; the fused path adds 16
    # bytes (its abort word)
    assert need == 8 * (1 + 1) * 16 + 16
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(Q.QknrError) as e:
        Q.group_norm_silu(x, 8, gm, gm, workspace=small)
    assert e.value.status == 2


# ---------------------------------------------------------------------------
# the fused one-launch path

def gn_call(x, w, inp, **kw):
    return Q.group_norm_silu(x, w.groups, torch.from_numpy(inp["gamma"]).cuda(),
                             torch.from_numpy(inp["beta"]).cuda(), eps=w.eps, **kw)


def query(w, **kw):
    x = torch.empty((w.n, w.c, w.h, w.w), dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float16,
                    device="cuda")
    g = torch.ones(w.c, device="cuda")
    return Q.gn_query(Q.gn_args(x, w.groups, g, g, **kw))


# groups of up to 512 KB (16 parts of at most 32 KB) take the cluster path,
# larger ones the fused one
VAE_PATHS = {"gn_vae_1x128x1024x1024": "gn_fused", "gn_vae_1x256x512x512": "gn_fused",
             "gn_vae_1x512x256x256": "gn_fused", "gn_vae_1x512x128x128": "gn_cluster"}


@pytest.mark.parametrize("name", list(I.GN_WORKLOADS))
def test_vae_shapes_take_the_expected_path(name):
    info = query(I.GN_WORKLOADS[name])
    assert info["kernel"].startswith(VAE_PATHS[name] + "<bf16>"), info
    fused = query(I.GN_WORKLOADS[name], mode="fused")
    assert fused["kernel"].startswith("gn_fused<bf16>"), fused
    assert fused["grid"] == fused["num_sms"] and fused["block"] == 800 and fused["stages"] == 9
    two = query(I.GN_WORKLOADS[name], mode="two_pass")
    assert two["kernel"].startswith("gn_stats+gn_apply"), two


@pytest.mark.parametrize("shape,groups", [((2, 64, 16, 16), 32), ((1, 32, 8, 8), 8), ((3, 12, 4, 6), 3),
                                          ((2, 4, 2, 4), 1), ((1, 512, 64, 64), 32), ((2, 96, 40, 72), 32),
                                          ((1, 8, 100, 104), 2), ((1, 128, 256, 256), 32)])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fused_equals_two_pass_with_the_same_pieces(shape, groups, dtype):
    # same per-thread order, same CTA reduction, same combine: the same bits
    w = I.GroupNormWorkload("f", *shape, groups=groups, dtype=dtype, scale=1.7, offset=-0.4, seed=sum(shape) + 1)
    inp = I.make_gn_inputs(w)
    a = gn_call(to_dev(inp["x"], dtype), w, inp, mode="fused")
    b = gn_call(to_dev(inp["x"], dtype), w, inp, mode="two_pass", piece_elems=12288)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    if w.elements <= 1 << 20:
        ref = G.group_norm_silu(inp["x"], dtype, groups, inp["gamma"], inp["beta"], w.eps)
        compare(to_bits(a), ref, dtype, "fused")


@pytest.mark.parametrize("dtype,spread,mean", [("fp16", 0.05, -30.0), ("fp16", 0.01, -8.0), ("bf16", 0.05, -30.0),
                                               ("bf16", 0.02, 60.0)])
@pytest.mark.parametrize("mode", ["fused", "two_pass", "cluster"])
def test_large_mean_small_spread(dtype, spread, mean, mode):
    # groups whose mean is hundreds of times their spread: the small
    # differences must not be lost to the rounding of the mean (every output
    # of magnitude >= 2^-6 within 1 ulp of the rounded oracle)
    w = I.GroupNormWorkload("m", 2, 64, 48, 40, groups=32, dtype=dtype, scale=spread, offset=mean, seed=65)
    inp = I.make_gn_inputs(w)
    res = gn_call(to_dev(inp["x"], dtype), w, inp, mode=mode)
    torch.cuda.synchronize()
    ref = G.group_norm_silu(inp["x"], dtype, w.groups, inp["gamma"], inp["beta"], w.eps)
    compare(to_bits(res), ref, dtype, f"mean {mean}, spread {spread}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("spike", [300.0, 3000.0])
@pytest.mark.parametrize("mode", ["fused", "two_pass", "cluster"])
def test_outlier_at_the_first_element(dtype, spike, mode):
    # the group's first element is an outlier that carries most of the
    # variance: neither the statistics nor the shift may let it cancel the
    # rest away (every output within 1 ulp of the rounded oracle)
    w = I.GroupNormWorkload("o", 1, 64, 128, 128, groups=4, dtype=dtype, seed=5)    # 262144 per group
    inp = I.make_gn_inputs(w)
    x = inp["x"].copy()
    x[0, 0, 0, 0] = I.to_storage_bits(np.array([spike], np.float32), dtype)[0]
    res = gn_call(to_dev(x, dtype), w, inp, mode=mode)
    torch.cuda.synchronize()
    ref = G.group_norm_silu(x, dtype, w.groups, inp["gamma"], inp["beta"], w.eps)
    compare_ulps(to_bits(res), ref, dtype, 1, f"spike {spike}")


@pytest.mark.parametrize("mode,piece", [("fused", 0), ("two_pass", 0), ("two_pass", 12288), ("cluster", 0)])
def test_spikes_scattered_through_large_groups(mode, piece):
    # fp16 groups of 110k values with 30-sigma spikes scattered through them
    # and a 300-sigma one first, gamma near -2 and beta near -3 (outputs
    # that are small differences of large terms); the two-pass path's default
    # pieces give each thread hundreds of values, summed per batch
    g = np.random.Generator(np.random.PCG64(1900))
    n, c, h, w_ = 2, 1, 13734, 8
    x = 0.05 * g.standard_normal((n, c, h, w_))
    idx = g.integers(0, x.size, x.size // 5000)
    x.reshape(-1)[idx] = g.choice([-1, 1], idx.size) * 1.5
    x.reshape(-1)[0] = 15.0
    xb = I.to_storage_bits(x.astype(np.float32), "fp16")
    gamma = (-2.0 * (1 + 0.1 * g.standard_normal(c))).astype(np.float32)
    beta = (-3.0 + 0.1 * g.standard_normal(c)).astype(np.float32)
    kw = {"piece_elems": piece} if piece else {}
    res = Q.group_norm_silu(to_dev(xb, "fp16"), 1, torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda(),
                            eps=1e-3, mode=mode, **kw)
    torch.cuda.synchronize()
    ref = G.group_norm_silu(xb, "fp16", 1, gamma, beta, 1e-3)
    compare_ulps(to_bits(res), ref, "fp16", 1, f"{mode} {piece}")


def test_fused_in_place_equals_out_of_place_and_repeats():
    w = I.GroupNormWorkload("ip", 2, 64, 96, 96, groups=32, scale=2.0, seed=41)
    inp = I.make_gn_inputs(w)
    src = to_dev(inp["x"], "bf16")
    out = torch.empty_like(src)
    gn_call(src, w, inp, out=out, mode="fused")
    for _ in range(3):                                  # earlier calls' records carry other tags
        x = to_dev(inp["x"], "bf16")
        gn_call(x, w, inp, mode="fused")
        torch.cuda.synchronize()
        assert torch.equal(x.view(torch.int16), out.view(torch.int16))
    np.testing.assert_array_equal(to_bits(src), inp["x"])


@pytest.mark.parametrize("shape,per_cta", [((1, 1, 2880, 2800), 5), ((1, 3, 2048, 2000), 7),
                                           ((1, 2, 2720, 2700), 8), ((1, 1, 4096, 4096), 9)])
def test_fused_large_groups(shape, per_cta):
    # 657, 1000, 1196 and 1366 pieces of 12288 elements per group over 152
    # CTAs; at most 9 per CTA
    w = I.GroupNormWorkload("big", *shape, groups=1, scale=1.2, offset=0.7, seed=43)
    info = query(w)
    assert info["kernel"].startswith("gn_fused") and info["kernel"].endswith(f" {per_cta} per CTA"), info
    inp = I.make_gn_inputs(w)
    res = gn_call(to_dev(inp["x"], "bf16"), w, inp)
    torch.cuda.synchronize()
    got = to_bits(res)
    g = np.random.Generator(np.random.PCG64(8))
    idx = tuple(g.integers(0, s, 3000) for s in (w.n, w.c, w.h, w.w))
    ref = G.group_norm_silu_at(inp["x"], w.dtype, w.groups, inp["gamma"], inp["beta"], w.eps, idx)
    compare(got[idx], ref, w.dtype, "large group")


def test_groups_beyond_the_fused_limit_fall_back_to_two_pass():
    # 1400 pieces per group: 10 per CTA, more than the 9 ring slots
    w = I.GroupNormWorkload("huge", 1, 1, 4200, 4096, groups=1, seed=44)
    assert query(w)["kernel"].startswith("gn_stats+gn_apply")
    x = torch.zeros((1, 1, 4200, 4096), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(1, device="cuda")
    with pytest.raises(Q.QknrError) as e:
        Q.group_norm_silu(x, 1, g, g, mode="fused")
    assert e.value.status == 4 and "per CTA" in str(e.value)


@pytest.mark.parametrize("flag", [Q.FLAG_TEST_STALL, Q.GN_FLAG_TEST_NO_RECORDS])
def test_fused_bounded_waits_report_timeout(flag):
    w = I.GroupNormWorkload("s", 1, 64, 64, 64, groups=32, seed=45)
    inp = I.make_gn_inputs(w)
    x = to_dev(inp["x"], "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gn_call(x, w, inp, mode="fused", dev_status=status, flags=flag, wait_limit_ns=2_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == Q.ERR_TIMEOUT
    np.testing.assert_array_equal(to_bits(x), inp["x"])   # nothing was written
    # the context stays usable and the next call starts clean
    status.zero_()
    res = gn_call(x, w, inp, mode="fused", dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = G.group_norm_silu(inp["x"], "bf16", w.groups, inp["gamma"], inp["beta"], w.eps)
    compare(to_bits(res), ref, "bf16", "after timeout")


@pytest.mark.parametrize("name", list(I.GN_WORKLOADS))
def test_vae_shapes_fused_equals_two_pass(name):
    # the full VAE shapes: hundreds of pieces per group over all CTAs
    w = I.GN_WORKLOADS[name]
    inp = I.make_gn_inputs(w)
    a = gn_call(to_dev(inp["x"], w.dtype), w, inp, mode="fused")
    b = gn_call(to_dev(inp["x"], w.dtype), w, inp, mode="two_pass", piece_elems=12288)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------------------
# the cluster path: one cluster of CTAs per group (of one sample), each CTA
# holding an equal part in shared memory, the parts' statistics merged over
# distributed shared memory

# (shape, groups, CTAs per cluster on 152 SMs): the fewest CTAs whose parts
# take at most 32 KB (200 KB when no cluster of 16 holds the group so), then
# twice as many while the grid has fewer than 2 CTAs per SM and parts stay at
# 4 KB or more; ragged last parts at 40040 and 1040040 elements per group
CLUSTER_CASES = [((2, 64, 16, 16), 32, 1), ((3, 12, 4, 6), 3, 1), ((6, 256, 64, 64), 32, 2),
                 ((3, 256, 128, 64), 32, 4), ((4, 128, 64, 64), 32, 4), ((2, 256, 128, 128), 32, 8),
                 ((20, 10, 88, 91), 2, 8), ((1, 512, 128, 128), 32, 16), ((1, 10, 88, 91), 2, 16),
                 ((1, 10, 24, 8667), 2, 16), ((1, 512, 256, 256), 32, 16)]


@pytest.mark.parametrize("shape,groups,cluster", CLUSTER_CASES)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_cluster_path_matches_the_oracle(shape, groups, cluster, dtype):
    w = I.GroupNormWorkload("c", *shape, groups=groups, dtype=dtype, scale=1.5, offset=0.3, seed=sum(shape) + 5)
    info = query(w, mode="cluster")
    assert info["kernel"].startswith(f"gn_cluster<{dtype}>, clusters of {cluster} CTAs"), info
    inp = I.make_gn_inputs(w)
    res, src = run(w, inp, out=True, mode="cluster")
    np.testing.assert_array_equal(to_bits(src), inp["x"])              # out of place: x unchanged
    got = to_bits(res)
    if inp["x"].size <= 1 << 22:
        ref = G.group_norm_silu(inp["x"], dtype, groups, inp["gamma"], inp["beta"], w.eps)
        compare(got, ref, dtype, f"cluster {shape}")
    else:
        g = np.random.Generator(np.random.PCG64(17))
        idx = tuple(g.integers(0, s_, 6000) for s_ in shape)
        ref = G.group_norm_silu_at(inp["x"], dtype, groups, inp["gamma"], inp["beta"], w.eps, idx)
        compare(got[idx], ref, dtype, f"cluster {shape}")
    # in place gives the same bits
    ip, _ = run(w, inp, mode="cluster")
    assert torch.equal(ip.view(torch.int16), res.view(torch.int16))


def test_cluster_path_with_one_cta_equals_the_one_piece_paths():
    # a group held by one CTA is one part: the same sums in the same order as
    # one piece of the fused and two-pass paths
    w = I.GroupNormWorkload("one", 2, 64, 32, 32, groups=32, scale=2.0, offset=-1.0, seed=46)
    inp = I.make_gn_inputs(w)
    assert query(w, mode="cluster")["kernel"].startswith("gn_cluster<bf16>, clusters of 1 CTAs")
    a = gn_call(to_dev(inp["x"], "bf16"), w, inp, mode="cluster")
    b = gn_call(to_dev(inp["x"], "bf16"), w, inp, mode="fused")
    c = gn_call(to_dev(inp["x"], "bf16"), w, inp, mode="two_pass")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_cluster_path_needs_no_workspace():
    w = I.GroupNormWorkload("nw", 1, 64, 64, 64, groups=32, seed=47)
    inp = I.make_gn_inputs(w)
    x = to_dev(inp["x"], "bf16")
    g, b = torch.from_numpy(inp["gamma"]).cuda(), torch.from_numpy(inp["beta"]).cuda()
    a = Q.gn_args(x, w.groups, g, b, eps=w.eps, mode="cluster", dev_status=Q.status_buffer())
    assert Q.gn_workspace_bytes(a) == 0
    Q.gn_launch(a)                                      # a.workspace is NULL
    torch.cuda.synchronize()
    ref = G.group_norm_silu(inp["x"], "bf16", w.groups, inp["gamma"], inp["beta"], w.eps)
    compare(to_bits(x), ref, "bf16", "no workspace")


def test_many_groups_take_the_fused_path():
    # 256 groups of 512 KB: their clusters of 16 do not all fit at once, so
    # the automatic choice is the fused path; the cluster path still runs
    # when asked for
    w = I.GroupNormWorkload("many", 8, 512, 128, 128, groups=32, seed=49)
    assert query(w)["kernel"].startswith("gn_fused<bf16>")
    cl = query(w, mode="cluster")
    assert cl["kernel"].startswith("gn_cluster<bf16>, clusters of 16 CTAs"), cl
    inp = I.make_gn_inputs(w)
    res, _ = run(w, inp, mode="cluster")
    g = np.random.Generator(np.random.PCG64(19))
    idx = tuple(g.integers(0, s_, 4000) for s_ in (w.n, w.c, w.h, w.w))
    ref = G.group_norm_silu_at(inp["x"], w.dtype, w.groups, inp["gamma"], inp["beta"], w.eps, idx)
    compare(to_bits(res)[idx], ref, w.dtype, "many groups, cluster path")


def test_cluster_path_rejects_groups_too_large():
    w = I.GN_WORKLOADS["gn_vae_1x256x512x512"]             # 4 MB groups: 256 KB parts at 16 CTAs
    with pytest.raises(Q.QknrError) as e:
        query(w, mode="cluster")
    assert e.value.status == 4


@pytest.mark.parametrize("cluster_shape", [(1, 64, 64, 64), (1, 512, 128, 128), (1, 10, 24, 8667)])
def test_cluster_bounded_wait_reports_timeout(cluster_shape):
    # no copy is issued: every CTA's wait runs out, every CTA of every
    # cluster still passes both cluster barriers, nothing is written
    groups = 2 if cluster_shape[1] == 10 else 32
    w = I.GroupNormWorkload("t", *cluster_shape, groups=groups, seed=48)
    inp = I.make_gn_inputs(w)
    x = to_dev(inp["x"], "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gn_call(x, w, inp, mode="cluster", dev_status=status, flags=Q.FLAG_TEST_STALL, wait_limit_ns=2_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == Q.ERR_TIMEOUT
    np.testing.assert_array_equal(to_bits(x), inp["x"])
    status.zero_()
    res = gn_call(x, w, inp, mode="cluster", dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = np.random.Generator(np.random.PCG64(18))
    idx = tuple(g.integers(0, s_, 3000) for s_ in cluster_shape)
    ref = G.group_norm_silu_at(inp["x"], "bf16", groups, inp["gamma"], inp["beta"], w.eps, idx)
    compare(to_bits(res)[idx], ref, "bf16", "after timeout")
