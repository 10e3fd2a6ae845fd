"""Programmatic dependent launch: the QK and AdaLN kernels may launch while
the kernel before them in the stream finishes, and must still see that
kernel's writes and must not overwrite what it still reads.  Checked with
chains of calls that read each other's outputs, a torch kernel that reads
the activation just before an in-place call, and one that writes it just
before; every result is compared bit for bit with plain launches
(QKNR_FLAG_NO_OVERLAP) and, for the first call, with the oracle."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import adaln_oracle as A
from oracle import qknr_oracle as O
from tests.gpu_util import compare, table_to_dev, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield
    assert Q.read_status() == 0, "a kernel reported a wait timeout"


def _dense(tokens=4096):
    w = I.WORKLOADS["dense_4096x24x128"]
    inp = I.make_inputs(w, tokens=tokens)
    dev = dict(gq=torch.from_numpy(inp["gamma_q"]).cuda(), gk=torch.from_numpy(inp["gamma_k"]).cuda(),
               cos=table_to_dev(inp["cos"], "fp32"), sin=table_to_dev(inp["sin"], "fp32"))
    return w, inp, dev


def _call(w, qkv, dev, flags):
    Q.qk_norm_rope_packed(qkv, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim, dev["gq"], dev["gk"],
                          dev["cos"], dev["sin"], rope_style=w.rope_style, eps=w.eps, flags=flags)


def _prefetch_rows(w, qkv, dev):
    a = Q.packed_args(qkv, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim, dev["gq"], dev["gk"], dev["cos"],
                      dev["sin"], rope_style=w.rope_style, eps=w.eps)
    return Q.query(a)["prefetch_rows"]


# 4096 rows: 27 per CTA, no L2 prefetch before the dependency wait; 9728
# rows: 64 per CTA, each CTA prefetches its second ring fill before it
PREFETCH_CASES = [(4096, False), (9728, True)]


@pytest.mark.parametrize("tokens,prefetch", PREFETCH_CASES)
def test_chain_of_dependent_calls_matches_plain_launches(tokens, prefetch):
    # every call reads the previous call's output in place
    w, inp, dev = _dense(tokens)
    assert (_prefetch_rows(w, to_dev(inp["qkv"], w.dtype), dev) > 0) == prefetch
    outs = []
    for flags in (0, Q.FLAG_NO_OVERLAP):
        qkv = to_dev(inp["qkv"], w.dtype)
        steps = []
        for _ in range(6):
            _call(w, qkv, dev, flags)
            steps.append(qkv.clone())
        torch.cuda.synchronize()
        outs.append([to_bits(s) for s in steps])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
    ref = O.forward_packed(inp["qkv"], w.dtype, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim,
                           inp["gamma_q"], inp["gamma_k"], w.eps, inp["cos"], inp["sin"], w.cos_dtype,
                           w.rope_style)
    D, h = w.head_dim, w.n_heads_q
    compare(outs[0][0][:, : h * D], ref["q"], w.dtype, "Q")
    compare(outs[0][0][:, h * D:2 * h * D], ref["k"], w.dtype, "K")


def test_in_place_call_waits_for_a_kernel_still_reading_its_input():
    # a torch kernel reads the 1 GB Wan activation; the in-place call right
    # after it must not overwrite rows that kernel has not read yet
    w = I.WORKLOADS["wan_32760x40x128"]
    inp = I.make_inputs(w)
    qkv = to_dev(inp["qkv"], w.dtype)
    gq, gk = torch.from_numpy(inp["gamma_q"]).cuda(), torch.from_numpy(inp["gamma_k"]).cuda()
    cos, sin = table_to_dev(inp["cos"], "fp32"), table_to_dev(inp["sin"], "fp32")
    seen = torch.empty_like(qkv)
    for _ in range(3):
        qkv.copy_(to_dev(inp["qkv"], w.dtype))
        torch.cuda.synchronize()
        # an elementwise kernel that reads every element of qkv (exact on bits)
        torch.bitwise_or(qkv.view(torch.int16), 0, out=seen.view(torch.int16))
        Q.qk_norm_rope_packed(qkv, 40, 40, 40, 128, gq, gk, cos, sin, rope_style=w.rope_style, eps=w.eps)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_bits(seen), inp["qkv"])


def test_no_prefetch_flag_gives_the_same_bits():
    w, inp, dev = _dense(9728)
    ref = to_dev(inp["qkv"], w.dtype)
    a = Q.packed_args(ref, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim, dev["gq"], dev["gk"], dev["cos"],
                      dev["sin"], rope_style=w.rope_style, eps=w.eps, flags=Q.FLAG_NO_PREFETCH)
    assert Q.query(a)["prefetch_rows"] == 0
    got = to_dev(inp["qkv"], w.dtype)
    for _ in range(3):
        _call(w, ref, dev, 0)
        _call(w, got, dev, Q.FLAG_NO_PREFETCH)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("tokens,prefetch", PREFETCH_CASES)
def test_call_sees_the_writes_of_the_kernel_before_it(tokens, prefetch):
    # a torch kernel writes the activation; the call right after it reads it
    # (with the prefetch, L2 may be asked for rows before that kernel wrote
    # them: the loads after the wait must still see the new bits)
    w, inp, dev = _dense(tokens)
    src = to_dev(inp["qkv"], w.dtype)
    assert (_prefetch_rows(w, src, dev) > 0) == prefetch
    plain = to_dev(inp["qkv"], w.dtype)
    _call(w, plain, dev, Q.FLAG_NO_OVERLAP)
    for _ in range(3):
        qkv = torch.full_like(src, 7.0)
        torch.cuda.synchronize()
        # an elementwise kernel that writes every element of qkv (exact on bits)
        torch.bitwise_or(src.view(torch.int16), 0, out=qkv.view(torch.int16))
        _call(w, qkv, dev, 0)
        torch.cuda.synchronize()
        assert torch.equal(qkv.view(torch.int16), plain.view(torch.int16))


def test_per_tensor_pair_matches_plain_launches():
    # page 2's form: Q then K, one launch per tensor, back to back
    w = I.WORKLOADS["flux2_2x4608x48x128"]
    inp = I.make_inputs(w)
    H, D = w.n_heads_q, w.head_dim
    gq, gk = torch.from_numpy(inp["gamma_q"]).cuda(), torch.from_numpy(inp["gamma_k"]).cuda()
    cos, sin = table_to_dev(inp["cos"], "fp32"), table_to_dev(inp["sin"], "fp32")
    res = []
    for flags in (0, Q.FLAG_NO_OVERLAP):
        q, k = to_dev(inp["q"], w.dtype), to_dev(inp["k"], w.dtype)
        for _ in range(3):                                 # each pair normalises the last one's output
            Q.qk_norm_rope_tensor(q, H, D, gq, cos, sin, rope_style=w.rope_style, flags=flags)
            Q.qk_norm_rope_tensor(k, H, D, gk, cos, sin, rope_style=w.rope_style, flags=flags)
        torch.cuda.synchronize()
        res.append((to_bits(q), to_bits(k)))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])


def test_adaln_chain_matches_plain_launches():
    w = I.ADALN_WORKLOADS["adaln_flux2_2x4608x6144"]
    inp = I.make_adaln_inputs(w, tokens=2000)
    sc = to_dev(inp["scale"], w.mod_dtype) if w.mod_dtype != "fp32" else torch.from_numpy(inp["scale"]).cuda()
    sh = to_dev(inp["shift"], w.mod_dtype) if w.mod_dtype != "fp32" else torch.from_numpy(inp["shift"]).cuda()
    outs = []
    for flags in (0, Q.FLAG_NO_OVERLAP):
        x = to_dev(inp["x"], w.dtype)
        steps = []
        for _ in range(4):
            Q.adaln_modulate(x, sc, sh, rows_per_batch=w.seq, eps=w.eps, flags=flags)
            steps.append(x.clone())
        torch.cuda.synchronize()
        outs.append([to_bits(s) for s in steps])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
    ref = A.adaln_modulate(inp["x"], w.dtype, inp["scale"], inp["shift"], w.mod_dtype, w.eps, w.seq)
    compare(outs[0][0], ref, w.dtype, "AdaLN")


def test_adaln_call_sees_the_writes_of_the_kernel_before_it():
    # a torch kernel writes x; the in-place AdaLN call right after it, which
    # asks L2 for its first rows before its dependency wait, must read the
    # new bits; and QKNR_FLAG_NO_PREFETCH gives the same bits
    w = I.ADALN_WORKLOADS["adaln_flux2_2x4608x6144"]
    inp = I.make_adaln_inputs(w, tokens=3000)
    sc, sh = to_dev(inp["scale"], w.mod_dtype), to_dev(inp["shift"], w.mod_dtype)
    src = to_dev(inp["x"], w.dtype)
    info = Q.adaln_query(Q.adaln_args(src, sc, sh, rows_per_batch=w.seq, eps=w.eps))
    assert info["prefetch_rows"] > 0
    assert Q.adaln_query(Q.adaln_args(src, sc, sh, rows_per_batch=w.seq, eps=w.eps,
                                      flags=Q.FLAG_NO_PREFETCH))["prefetch_rows"] == 0
    plain = src.clone()
    Q.adaln_modulate(plain, sc, sh, rows_per_batch=w.seq, eps=w.eps, flags=Q.FLAG_NO_OVERLAP)
    for flags in (0, Q.FLAG_NO_PREFETCH):
        for _ in range(3):
            x = torch.full_like(src, 3.0)
            torch.cuda.synchronize()
            torch.bitwise_or(src.view(torch.int16), 0, out=x.view(torch.int16))
            Q.adaln_modulate(x, sc, sh, rows_per_batch=w.seq, eps=w.eps, flags=flags)
            torch.cuda.synchronize()
            assert torch.equal(x.view(torch.int16), plain.view(torch.int16))


def test_calls_right_after_a_cooperative_group_norm_launch():
    # the fused group norm is a cooperative launch; the QK and AdaLN calls
    # launched right after it (programmatic dependent launch) read what it
    # wrote and must give the bits of plain launches
    wg = I.GroupNormWorkload("g", 1, 64, 96, 96, groups=32, seed=41)
    ig = I.make_gn_inputs(wg)
    gam, bet = torch.from_numpy(ig["gamma"]).cuda(), torch.from_numpy(ig["beta"]).cuda()
    w, inp, dev = _dense(tokens=2304)
    res = []
    for flags in (0, Q.FLAG_NO_OVERLAP):
        x = to_dev(ig["x"], wg.dtype)
        qkv = to_dev(inp["qkv"], w.dtype)
        torch.cuda.synchronize()
        # the group norm writes x; the QK call then takes x's bits as its Q|K
        # columns' source: copy x into them with a kernel, then normalise
        Q.group_norm_silu(x, wg.groups, gam, bet, eps=wg.eps, mode="fused")
        rows = x.numel() // (48 * 128)                      # 96 rows of Q|K columns
        qk = qkv.view(torch.int16)[:rows, : 48 * 128]
        torch.bitwise_or(x.view(torch.int16).reshape(rows, 48 * 128), 0, out=qk)
        _call(w, qkv, dev, flags)
        Q.group_norm_silu(x, wg.groups, gam, bet, eps=wg.eps, mode="fused")
        _call(w, qkv, dev, flags)
        torch.cuda.synchronize()
        res.append((to_bits(x), to_bits(qkv)))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])
