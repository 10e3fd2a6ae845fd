"""AdaLN scale/shift CUDA path vs the fp64 oracle, through the C ABI.

Full-size FLUX.2 and Wan shapes are compared on sampled rows, smaller ones
element by element; plus bitwise launch-shape independence, in place vs
out of place, degenerate rows, the bounded wait and host-side errors."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import adaln_oracle as A
from tests.gpu_util import TORCH, compare, compare_ulps, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield
    assert Q.read_status() == 0, "a kernel reported a wait timeout"


def mod_to_dev(m, w):
    if w.mod_dtype == "fp32":
        return torch.from_numpy(m).cuda()
    return to_dev(m, w.mod_dtype)


def run(w, inp, out=False, **kw):
    x = to_dev(inp["x"], w.dtype)
    o = torch.empty_like(x) if out else None
    res = Q.adaln_modulate(x, mod_to_dev(inp["scale"], w), mod_to_dev(inp["shift"], w), rows_per_batch=w.seq,
                           out=o, eps=w.eps, **kw)
    torch.cuda.synchronize()
    return res, x


def check(w, got_bits, inp, rows=None):
    ref = A.adaln_modulate(inp["x"], w.dtype, inp["scale"], inp["shift"], w.mod_dtype, w.eps, w.seq, rows=rows)
    g = got_bits if rows is None else got_bits[rows]
    return compare(g, ref, w.dtype, w.name)


def sample_rows(T, n, seed=0):
    g = np.random.Generator(np.random.PCG64(seed))
    return np.unique(np.concatenate([[0, 1, T // 2, T - 1], g.choice(T, size=min(n, T), replace=False)]))


@pytest.mark.parametrize("name", list(I.ADALN_WORKLOADS))
@pytest.mark.parametrize("mod_dtype", ["bf16", "fp32"])
def test_full_size_sampled(name, mod_dtype):
    w = I.ADALN_WORKLOADS[name].with_(mod_dtype=mod_dtype)
    inp = I.make_adaln_inputs(w)
    res, _ = run(w, inp)
    bits = to_bits(res)
    rows = sample_rows(w.tokens, 96)
    if w.batch > 1:
        rows = np.unique(np.concatenate([rows, [w.seq - 1, w.seq]]))
    check(w, bits, inp, rows)


def test_in_place_equals_out_of_place():
    w = I.ADALN_WORKLOADS["adaln_flux2_2x4608x6144"]
    inp = I.make_adaln_inputs(w)
    a, _ = run(w, inp)
    b, src = run(w, inp, out=True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    np.testing.assert_array_equal(to_bits(src), inp["x"])


@pytest.mark.parametrize("C", [8, 64, 1000, 4096, 5120, 6144, 12288, 32768])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_hidden_sizes_full(C, dtype):
    w = I.AdaLNWorkload("c", 3, 101, C, dtype=dtype, mod_dtype="fp32", seed=C)
    inp = I.make_adaln_inputs(w)
    res, _ = run(w, inp)
    check(w, to_bits(res), inp)


@pytest.mark.parametrize("dtype,spread,mean", [("fp16", 0.05, -30.0), ("fp16", 0.01, -8.0), ("bf16", 0.05, -30.0),
                                               ("fp16", 1.0, -200.0), ("bf16", 0.02, 60.0)])
def test_large_mean_small_spread(dtype, spread, mean):
    # rows whose mean is hundreds of times their spread: the small
    # differences must not be lost to the rounding of the mean (every output
    # of magnitude >= 2^-6 within 1 ulp of the rounded oracle)
    g = np.random.Generator(np.random.PCG64(64))
    T, C, rpb = 300, 3072, 150
    xb = I.to_storage_bits((g.standard_normal((T, C)) * spread + mean).astype(np.float32), dtype)
    sc = (0.1 * g.standard_normal((2, C))).astype(np.float32)
    sh = (0.1 * g.standard_normal((2, C))).astype(np.float32)
    res = Q.adaln_modulate(to_dev(xb, dtype), torch.from_numpy(sc).cuda(), torch.from_numpy(sh).cuda(),
                           rows_per_batch=rpb, eps=1e-6)
    torch.cuda.synchronize()
    ref = A.adaln_modulate(xb, dtype, sc, sh, "fp32", 1e-6, rpb)
    compare(to_bits(res), ref, dtype, f"mean {mean}, spread {spread}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("C", [6144, 32768])
def test_outlier_channel_at_the_first_element(dtype, C):
    # channel 0, the shift of every row's sums, carries a massive activation
    # (10 sqrt(C) against unit noise) that dominates the row's variance
    g = np.random.Generator(np.random.PCG64(9))
    T = 64
    xf = g.standard_normal((T, C)).astype(np.float32)
    xf[:, 0] = 10.0 * np.sqrt(C)
    xb = I.to_storage_bits(xf, dtype)
    sc = (0.1 * g.standard_normal((1, C))).astype(np.float32)
    sh = (0.1 * g.standard_normal((1, C))).astype(np.float32)
    res = Q.adaln_modulate(to_dev(xb, dtype), torch.from_numpy(sc).cuda(), torch.from_numpy(sh).cuda(),
                           rows_per_batch=T, eps=1e-6)
    torch.cuda.synchronize()
    ref = A.adaln_modulate(xb, dtype, sc, sh, "fp32", 1e-6, T)
    compare_ulps(to_bits(res), ref, dtype, 1, f"C {C}")


@pytest.mark.parametrize("T,rpb", [(1, 1), (2, 1), (151, 7), (152, 152), (1000, 1), (4099, 4099), (4099, 100)])
def test_ragged_rows_and_batches(T, rpb):
    w = I.AdaLNWorkload("r", 1, rpb, 512, mod_dtype="bf16", seed=T)
    inp = I.make_adaln_inputs(w, tokens=T)
    assert inp["scale"].shape[0] == -(-T // rpb)
    res, _ = run(w, inp)
    check(w, to_bits(res), inp)


def test_degenerate_rows():
    C = 256
    w = I.AdaLNWorkload("d", 1, 6, C, mod_dtype="fp32", seed=3)
    inp = I.make_adaln_inputs(w)
    x = I.storage_to_f32(inp["x"], "bf16").copy()
    x[0] = 1.5                                      # constant: output is exactly shift
    x[1] = 0.0
    x[2] *= 1e-20                                   # eps dominates
    x[3] *= 1e15                                    # large, squares still in fp32 range
    x[4] += 1000.0                                  # large mean, small spread
    inp["x"] = I.to_storage_bits(x, "bf16")
    res, _ = run(w, inp)
    got = to_bits(res)
    shift_bits = I.to_storage_bits(inp["shift"][0], "bf16")
    np.testing.assert_array_equal(got[0], shift_bits)
    np.testing.assert_array_equal(got[1], shift_bits)
    check(w, got, inp)


@pytest.mark.parametrize("tune", [dict(consumer_warps=16, group_warps=2), dict(consumer_warps=8, group_warps=2),
                                  dict(consumer_warps=4, group_warps=2, stages=4),
                                  dict(consumer_warps=4, group_warps=2, ctas_per_sm=2),
                                  dict(consumer_warps=2, group_warps=2, stages=6)])
def test_same_group_size_gives_the_same_bits(tune):
    # the fp32 sums' order is fixed by the warps per row (2 here by default),
    # not by the number of groups, the ring depth or the grid
    w = I.AdaLNWorkload("t", 2, 700, 6144, mod_dtype="bf16", seed=4)
    inp = I.make_adaln_inputs(w)
    a, _ = run(w, inp)
    b, _ = run(w, inp, **tune)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("tune", [dict(consumer_warps=16, group_warps=16), dict(consumer_warps=12, group_warps=12),
                                  dict(consumer_warps=4, group_warps=4), dict(consumer_warps=16, group_warps=8),
                                  dict(consumer_warps=8, group_warps=1)])
def test_other_group_sizes_match_the_oracle(tune):
    # another warps-per-row sums in another order: a different, equally
    # valid rounding, held to the same tolerance
    w = I.AdaLNWorkload("t", 2, 700, 6144, mod_dtype="bf16", seed=4)
    inp = I.make_adaln_inputs(w)
    b, _ = run(w, inp, **tune)
    check(w, to_bits(b), inp)


def test_query_reports_the_launch():
    w = I.ADALN_WORKLOADS["adaln_flux2_2x4608x6144"]
    x = torch.zeros((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    m = torch.zeros((2, w.hidden), dtype=torch.bfloat16, device="cuda")
    info = Q.adaln_query(Q.adaln_args(x, m, m, rows_per_batch=w.seq))
    assert info["consumer_warps"] % info["group_warps"] == 0
    assert info["stage_bytes"] == w.hidden * 2 and info["registers"] > 0
    assert info["kernel"].startswith("adaln<bf16,act,cpl")


def test_bounded_wait_reports_timeout():
    w = I.AdaLNWorkload("s", 1, 500, 1024, mod_dtype="fp32", seed=5)
    inp = I.make_adaln_inputs(w)
    x = to_dev(inp["x"], "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Q.adaln_modulate(x, torch.from_numpy(inp["scale"]).cuda(), torch.from_numpy(inp["shift"]).cuda(),
                     dev_status=status, flags=Q.FLAG_TEST_STALL, wait_limit_ns=1_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == Q.ERR_TIMEOUT
    np.testing.assert_array_equal(to_bits(x), inp["x"])
    status.zero_()
    res, _ = run(w, inp, dev_status=status)
    assert int(status.item()) == 0
    check(w, to_bits(res), inp)


def test_errors_on_device_pointers():
    x = torch.zeros((8, 520), dtype=torch.bfloat16, device="cuda")
    m = torch.zeros((1, 512), dtype=torch.float32, device="cuda")
    with pytest.raises(Q.QknrError) as e:
        Q.adaln_modulate(x[:, 1:513], m, m)                      # 2-byte misaligned base
    assert e.value.status == 3
    with pytest.raises(ValueError):
        Q.adaln_modulate(x[:, :512], m.to(torch.float16), m.to(torch.float16))
