"""Edge cases of the CUDA path: empty and ragged inputs, mixed head counts,
one-tensor launches, V-only copies, strided rows, degenerate heads, the
largest row the stage ring holds, launch-shape independence, the bounded
wait and host-side errors on real device pointers."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import qknr_oracle as O
from tests.gpu_util import compare, table_to_dev, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def make_case(T, hq, hk, hv, D, dtype="bf16", style="interleaved", cos_dtype="fp32", seed=0, scale=1.0,
              cos_rows=None):
    g = _rng(seed)
    x = (g.standard_normal((T, (hq + hk + hv) * D)) * scale).astype(np.float32)
    rows = cos_rows or max(T, 1)
    ang = g.uniform(-np.pi, np.pi, size=(rows, D // 2))
    full = np.repeat(ang, 2, axis=1) if style == "interleaved" else np.concatenate([ang, ang], axis=1)
    cos, sin = np.cos(full).astype(np.float32), np.sin(full).astype(np.float32)
    if cos_dtype == "bf16":
        cos, sin = I.to_storage_bits(cos, "bf16"), I.to_storage_bits(sin, "bf16")
    return dict(qkv=I.to_storage_bits(x, dtype), gamma_q=(1 + 0.1 * g.standard_normal(D)).astype(np.float32),
                gamma_k=(1 + 0.1 * g.standard_normal(D)).astype(np.float32), cos=cos, sin=sin)


def run_case(c, hq, hk, hv, D, dtype="bf16", style="interleaved", cos_dtype="fp32", out=False, **kw):
    qkv = to_dev(c["qkv"], dtype)
    o = torch.empty_like(qkv) if out else None
    Q.qk_norm_rope_packed(qkv, hq, hk, hv, D, torch.from_numpy(c["gamma_q"]).cuda(),
                          torch.from_numpy(c["gamma_k"]).cuda(), table_to_dev(c["cos"], cos_dtype),
                          table_to_dev(c["sin"], cos_dtype), out=o, rope_style=style, **kw)
    torch.cuda.synchronize()
    return to_bits(qkv if o is None else o)


def check_case(c, got, hq, hk, hv, D, dtype="bf16", style="interleaved", cos_dtype="fp32"):
    ref = O.forward_packed(c["qkv"], dtype, hq, hk, hv, D, c["gamma_q"], c["gamma_k"], 1e-6, c["cos"], c["sin"],
                           cos_dtype, style)
    if hq:
        compare(got[:, : hq * D], ref["q"], dtype, "Q")
    if hk:
        compare(got[:, hq * D:(hq + hk) * D], ref["k"], dtype, "K")
    np.testing.assert_array_equal(got[:, (hq + hk) * D:], ref["v"])


def test_zero_tokens_is_a_no_op():
    qkv = torch.empty((0, 12 * 128), dtype=torch.bfloat16, device="cuda")
    Q.qk_norm_rope_packed(qkv, 4, 4, 4, 128, torch.ones(128, device="cuda"), torch.ones(128, device="cuda"),
                          torch.ones((1, 128), device="cuda"), torch.zeros((1, 128), device="cuda"))
    torch.cuda.synchronize()


@pytest.mark.parametrize("T", [1, 2, 151, 152, 153, 4099])
def test_ragged_token_counts(T):
    c = make_case(T, 5, 5, 3, 128, seed=T)
    check_case(c, run_case(c, 5, 5, 3, 128), 5, 5, 3, 128)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("cos_dtype", ["fp32", "bf16"])
def test_all_instances(D, style, dtype, cos_dtype):
    c = make_case(777, 3, 5, 2, D, dtype, style, cos_dtype, seed=D)
    got = run_case(c, 3, 5, 2, D, dtype, style, cos_dtype)
    check_case(c, got, 3, 5, 2, D, dtype, style, cos_dtype)


@pytest.mark.parametrize("hq,hk,hv", [(1, 0, 0), (0, 1, 0), (7, 0, 3), (0, 9, 1), (1, 1, 1), (13, 2, 0)])
def test_head_count_mixes(hq, hk, hv):
    D = 64
    c = make_case(300, hq, hk, hv, D, seed=hq * 10 + hk)
    qkv = to_dev(c["qkv"], "bf16")
    views = dict(q=qkv[:, : hq * D] if hq else None, k=qkv[:, hq * D:(hq + hk) * D] if hk else None)
    a = Q.make_args(**views, n_heads_q=hq, n_heads_k=hk, head_dim=D,
                    gamma_q=torch.from_numpy(c["gamma_q"]).cuda() if hq else None,
                    gamma_k=torch.from_numpy(c["gamma_k"]).cuda() if hk else None,
                    cos=torch.from_numpy(c["cos"]).cuda(), sin=torch.from_numpy(c["sin"]).cuda(), tokens=300,
                    dev_status=Q.status_buffer())
    Q.launch(a)
    torch.cuda.synchronize()
    check_case(c, to_bits(qkv), hq, hk, hv, D)


def test_v_copy_only():
    D, hv = 128, 6
    c = make_case(500, 0, 0, hv, D)
    v = to_dev(c["qkv"], "bf16")
    v_out = torch.zeros_like(v)
    Q.launch(Q.make_args(v=v, v_out=v_out, n_heads_v=hv, head_dim=D, dev_status=Q.status_buffer()))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(v_out), c["qkv"])


def test_strided_rows_and_out_of_place():
    # rows padded to a wider stride, outputs to a third buffer with its own stride
    T, hq, hk, D = 333, 4, 4, 128
    c = make_case(T, hq, hk, 0, D, seed=3)
    pad = 64
    big = torch.zeros((T, (hq + hk) * D + pad), dtype=torch.bfloat16, device="cuda")
    big[:, : (hq + hk) * D] = to_dev(c["qkv"], "bf16")
    out = torch.zeros((T, (hq + hk) * D + 2 * pad), dtype=torch.bfloat16, device="cuda")
    a = Q.make_args(q=big[:, : hq * D], k=big[:, hq * D:(hq + hk) * D], q_out=out[:, pad:pad + hq * D],
                    k_out=out[:, pad + hq * D:pad + (hq + hk) * D], n_heads_q=hq, n_heads_k=hk, head_dim=D,
                    gamma_q=torch.from_numpy(c["gamma_q"]).cuda(), gamma_k=torch.from_numpy(c["gamma_k"]).cuda(),
                    cos=torch.from_numpy(c["cos"]).cuda(), sin=torch.from_numpy(c["sin"]).cuda(),
                    dev_status=Q.status_buffer())
    Q.launch(a)
    torch.cuda.synchronize()
    ob = to_bits(out)
    assert not ob[:, :pad].any() and not ob[:, pad + (hq + hk) * D:].any()     # padding untouched
    check_case(c, ob[:, pad:pad + (hq + hk) * D], hq, hk, 0, D)
    np.testing.assert_array_equal(to_bits(big)[:, : (hq + hk) * D], c["qkv"])   # input untouched


def test_degenerate_heads():
    # zero heads stay zero; constant heads give gamma*cos-style values; tiny and large scales
    T, H, D = 64, 4, 128
    c = make_case(T, H, H, 0, D, seed=5)
    x = I.storage_to_f32(c["qkv"], "bf16").copy()
    x[:, 0:D] = 0.0                                   # head 0 of Q is all zero
    x[:, D:2 * D] = 0.75                              # head 1 constant
    x[:, 2 * D:3 * D] *= 1e-20                        # tiny: eps dominates
    x[:, 3 * D:4 * D] *= 1e15                         # huge, while D*x^2 still fits in fp32
    c["qkv"] = I.to_storage_bits(x, "bf16")
    got = run_case(c, H, H, 0, D)
    assert not got[:, 0:D].any() or np.all(np.abs(I.storage_to_f32(got[:, 0:D], "bf16")) == 0)
    check_case(c, got, H, H, 0, D)


def test_fp16_extremes():
    T, H, D = 64, 2, 64
    c = make_case(T, H, H, 0, D, "fp16", "rotate_half", seed=6)
    x = I.storage_to_f32(c["qkv"], "fp16").copy()
    x[:, :D] *= 1e4                                   # near fp16 max: the fp32 sum of squares does not overflow
    x[:, D:2 * D] *= 1e-4                             # near fp16 subnormals
    c["qkv"] = I.to_storage_bits(x, "fp16")
    got = run_case(c, H, H, 0, D, "fp16", "rotate_half")
    check_case(c, got, H, H, 0, D, "fp16", "rotate_half")


def test_batch_broadcast_of_table_rows():
    T, S, H, D = 600, 200, 3, 128
    c = make_case(T, H, H, 0, D, style="rotate_half", seed=8, cos_rows=S)
    got = run_case(c, H, H, 0, D, style="rotate_half")
    check_case(c, got, H, H, 0, D, style="rotate_half")


def test_largest_row_that_fits_two_stages():
    # shared fp32 table, D=128: a row of (Hq+Hk)*256 B + 1 KB of cos/sin; two
    # stages must fit in the opt-in shared memory of one CTA
    T, H, D = 40, 220, 128
    c = make_case(T, H, H, 0, D, seed=9)
    check_case(c, run_case(c, H, H, 0, D), H, H, 0, D)
    qkv = to_dev(make_case(4, 260, 260, 0, D)["qkv"], "bf16")
    with pytest.raises(Q.QknrError) as e:
        Q.qk_norm_rope_packed(qkv, 260, 260, 0, D, torch.ones(D, device="cuda"), torch.ones(D, device="cuda"),
                              torch.ones((4, D), device="cuda"), torch.zeros((4, D), device="cuda"))
    assert e.value.status == 4


@pytest.mark.parametrize("tune", [dict(stages=2), dict(stages=8, group_warps=16),
                                  dict(consumer_warps=12, group_warps=6, stages=8),
                                  dict(ctas_per_sm=2), dict(ctas_per_sm=4),
                                  dict(consumer_warps=8, group_warps=1), dict(group_warps=2), dict(group_warps=4),
                                  dict(consumer_warps=1), dict(consumer_warps=3), dict(consumer_warps=16),
                                  dict(consumer_warps=8, group_warps=1, stages=2)])
def test_result_does_not_depend_on_launch_shape(tune):
    T, H, D = 2000, 12, 128
    c = make_case(T, H, H, H, D, style="rotate_half", seed=10)
    base = run_case(c, H, H, H, D, style="rotate_half")
    other = run_case(c, H, H, H, D, style="rotate_half", **tune)
    np.testing.assert_array_equal(base, other)


def test_query_reports_the_launch():
    c = make_case(1000, 40, 40, 40, 128)
    qkv = to_dev(c["qkv"], "bf16")
    a = Q.packed_args(qkv, 40, 40, 40, 128, torch.ones(128, device="cuda"), torch.ones(128, device="cuda"),
                      torch.from_numpy(c["cos"]).cuda(), torch.from_numpy(c["sin"]).cuda())
    info = Q.query(a)
    assert info["num_sms"] > 0 and 0 < info["grid"] <= 1000
    assert info["block"] == 32 * (info["consumer_warps"] + 1)
    assert info["consumer_warps"] % info["group_warps"] == 0
    groups = info["consumer_warps"] // info["group_warps"]
    assert info["stage_bytes"] == 80 * 256 + 1024
    assert info["dyn_smem"] >= 2 * groups * info["stage_bytes"] and info["registers"] > 0
    assert info["stages"] * groups <= 32


def test_bounded_wait_reports_timeout_and_leaves_context_usable():
    T, H, D = 1000, 4, 128
    c = make_case(T, H, H, 0, D, seed=11)
    qkv = to_dev(c["qkv"], "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gq, gk = torch.from_numpy(c["gamma_q"]).cuda(), torch.from_numpy(c["gamma_k"]).cuda()
    cos, sin = torch.from_numpy(c["cos"]).cuda(), torch.from_numpy(c["sin"]).cuda()
    # the producer issues no loads, so every consumer wait runs out (1 ms)
    Q.qk_norm_rope_packed(qkv, H, H, 0, D, gq, gk, cos, sin, dev_status=status, flags=Q.FLAG_TEST_STALL,
                          wait_limit_ns=1_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == Q.ERR_TIMEOUT
    np.testing.assert_array_equal(to_bits(qkv), c["qkv"])           # nothing written
    # the context still works
    status.zero_()
    Q.qk_norm_rope_packed(qkv, H, H, 0, D, gq, gk, cos, sin, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_case(c, to_bits(qkv), H, H, 0, D)


def test_misaligned_device_pointer_is_rejected():
    qkv = torch.zeros((8, 3 * 4 * 128 + 8), dtype=torch.bfloat16, device="cuda")
    view = qkv[:, 1:1 + 3 * 4 * 128]                                  # 2-byte offset
    with pytest.raises(Q.QknrError) as e:
        Q.qk_norm_rope_packed(view, 4, 4, 4, 128, torch.ones(128, device="cuda"), torch.ones(128, device="cuda"),
                              torch.ones((8, 128), device="cuda"), torch.zeros((8, 128), device="cuda"))
    assert e.value.status == 3
