"""CUDA path vs the fp64 oracle on the seeded workloads, through the C ABI.

Small workloads are compared element by element; the full-size Wan and
FLUX.2 workloads (in the launch configuration the benchmark times) are
compared on sampled token rows, and every output is checked for the
properties that hold at any size: V bit-exact, shared vs expanded tables
bitwise equal, in place vs out of place bitwise equal.
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import qknr_oracle as O
from tests.gpu_util import TOL, compare, table_to_dev, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield
    assert Q.read_status() == 0, "a kernel reported a wait timeout"


def sample_rows(T, n, seed=0):
    g = np.random.Generator(np.random.PCG64(seed))
    fixed = [0, 1, T // 2, T - 2, T - 1]
    rows = np.unique(np.concatenate([[r for r in fixed if 0 <= r < T], g.choice(T, size=min(n, T), replace=False)]))
    return rows


def run_packed(w, inp, *, out=False, cos_layout=None, dev_tabs=None, **kw):
    """Launch on a device copy of inp['qkv']; returns (result tensor, input tensor)."""
    qkv = to_dev(inp["qkv"], w.dtype)
    gq = torch.from_numpy(inp["gamma_q"]).cuda()
    gk = torch.from_numpy(inp["gamma_k"]).cuda()
    if dev_tabs is None:
        cos = table_to_dev(inp["cos"], w.cos_dtype)
        sin = table_to_dev(inp["sin"], w.cos_dtype)
    else:
        cos, sin = dev_tabs
    layout = cos_layout or w.cos_layout
    o = torch.empty_like(qkv) if out else None
    res = Q.qk_norm_rope_packed(qkv, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim, gq, gk, cos, sin,
                                out=o, rope_style=w.rope_style, cos_layout=layout, eps=w.eps, **kw)
    torch.cuda.synchronize()
    return res, qkv


def oracle_packed(w, inp, rows=None, cos_layout="shared_row", tables=None):
    cos, sin = (inp["cos"], inp["sin"]) if tables is None else tables
    return O.forward_packed(inp["qkv"], w.dtype, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim,
                            inp["gamma_q"], inp["gamma_k"], w.eps, cos, sin, w.cos_dtype, w.rope_style,
                            cos_layout, rows=rows)


def check_packed(w, got_bits, inp, rows=None):
    """Compare Q/K of a packed result with the oracle; V bitwise."""
    ref = oracle_packed(w, inp, rows)
    D, hq, hk = w.head_dim, w.n_heads_q, w.n_heads_k
    g = got_bits if rows is None else got_bits[rows]
    mq, fq = compare(g[:, : hq * D], ref["q"], w.dtype, "Q")
    mk, fk = compare(g[:, hq * D:(hq + hk) * D], ref["k"], w.dtype, "K")
    np.testing.assert_array_equal(g[:, (hq + hk) * D:], ref["v"])
    return max(mq, mk), max(fq, fk)


# ---------------------------------------------------------------------------
# the tiny and 4096-token workloads, element by element

def test_tiny_workload_full():
    w = I.WORKLOADS["tiny_256x24x64"]
    inp = I.make_inputs(w)
    res, _ = run_packed(w, inp)
    m, f = check_packed(w, to_bits(res), inp)
    assert m <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_dense_4096_full(dtype):
    w = I.WORKLOADS["dense_4096x24x128"].with_(dtype=dtype)
    inp = I.make_inputs(w)
    res, _ = run_packed(w, inp)
    m, f = check_packed(w, to_bits(res), inp)
    assert m <= TOL[dtype] and f < 0.02


# ---------------------------------------------------------------------------
# full-size Wan: sampled rows vs oracle, plus bitwise properties

@pytest.fixture(scope="module")
def wan():
    w = I.WORKLOADS["wan_32760x40x128"]
    return w, I.make_inputs(w)


def test_wan_shared_fp32_sampled(wan):
    w, inp = wan
    res, _ = run_packed(w, inp)
    bits = to_bits(res)
    rows = sample_rows(w.tokens, 160)
    m, f = check_packed(w, bits, inp, rows)
    # V is untouched everywhere
    D3 = 2 * w.n_heads_q * w.head_dim
    np.testing.assert_array_equal(bits[:, D3:], inp["qkv"][:, D3:])


@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
@pytest.mark.parametrize("cos_dtype", ["fp32", "bf16"])
def test_wan_expanded_bitwise_equals_shared(wan, style, cos_dtype):
    w0, inp0 = wan
    w = w0.with_(rope_style=style, cos_dtype=cos_dtype)
    inp = dict(inp0)
    inp["cos"], inp["sin"] = I.rope_table(w)
    shared, _ = run_packed(w, inp)
    cos = table_to_dev(inp["cos"], cos_dtype)
    sin = table_to_dev(inp["sin"], cos_dtype)
    H = w.n_heads_q
    ce = cos[:, None, :].expand(cos.shape[0], H, w.head_dim).contiguous()
    se = sin[:, None, :].expand(sin.shape[0], H, w.head_dim).contiguous()
    expanded, _ = run_packed(w, inp, cos_layout="per_head_expanded", dev_tabs=(ce, se))
    assert torch.equal(shared.view(torch.int16), expanded.view(torch.int16))
    del ce, se, expanded
    rows = sample_rows(w.tokens, 48, seed=1)
    check_packed(w, to_bits(shared), inp, rows)


def test_wan_out_of_place_equals_in_place_and_copies_v(wan):
    w, inp = wan
    inplace, _ = run_packed(w, inp)
    outp, src = run_packed(w, inp, out=True)
    assert torch.equal(inplace.view(torch.int16), outp.view(torch.int16))
    # the input buffer is untouched when writing elsewhere
    np.testing.assert_array_equal(to_bits(src), inp["qkv"])


# ---------------------------------------------------------------------------
# FLUX.2: separate Q, K, V, per-tensor launches, batch-broadcast table

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_flux_per_tensor_sampled(dtype):
    w = I.WORKLOADS["flux2_2x4608x48x128"].with_(dtype=dtype)
    inp = I.make_inputs(w)
    D, H = w.head_dim, w.n_heads_q
    q, k, v = (to_dev(inp[n], dtype) for n in ("q", "k", "v"))
    gq = torch.from_numpy(inp["gamma_q"]).cuda()
    gk = torch.from_numpy(inp["gamma_k"]).cuda()
    cos = table_to_dev(inp["cos"], "fp32")
    sin = table_to_dev(inp["sin"], "fp32")
    Q.qk_norm_rope_tensor(q, H, D, gq, cos, sin, rope_style=w.rope_style)
    Q.qk_norm_rope_tensor(k, H, D, gk, cos, sin, rope_style=w.rope_style)
    torch.cuda.synchronize()
    rows = sample_rows(w.tokens, 128, seed=2)
    rows = np.unique(np.concatenate([rows, [511, 512, 4607, 4608, 4608 + 511, 4608 + 512]]))
    for name, t, g in (("q", q, inp["gamma_q"]), ("k", k, inp["gamma_k"])):
        ref = O.forward_separate(inp[name], dtype, H, D, g, w.eps, inp["cos"], inp["sin"], "fp32",
                                 w.rope_style, rows=rows)
        compare(to_bits(t)[rows], ref, dtype, name)
    np.testing.assert_array_equal(to_bits(v), inp["v"])
    # the single-launch Q+K form gives the same bits as two per-tensor launches
    q2, k2 = to_dev(inp["q"], dtype), to_dev(inp["k"], dtype)
    v_out = torch.empty_like(v)
    Q.qk_norm_rope_separate(q2, k2, H, D, gq, gk, cos, sin, v=v, v_out=v_out, rope_style=w.rope_style)
    torch.cuda.synchronize()
    assert torch.equal(q2.view(torch.int16), q.view(torch.int16))
    assert torch.equal(k2.view(torch.int16), k.view(torch.int16))
    assert torch.equal(v_out.view(torch.int16), v.view(torch.int16))


# ---------------------------------------------------------------------------
# page 1's layout-parity matrix: 2 styles x (24,64), (24,128), (40,128),
# rtol = atol = 0, with an unchanged V slice

@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
@pytest.mark.parametrize("H,D", [(24, 64), (24, 128), (40, 128)])
def test_shared_fp32_matches_expanded_matrix(style, H, D):
    w = I.Workload("parity", 1, 301, H, H, H, D, "bf16", True, style, "fp32", "shared_row", "1d", (), (D,),
                   seed=7)
    inp = I.make_inputs(w)
    shared, _ = run_packed(w, inp)
    ce = I.expand_per_head(inp["cos"], H)
    se = I.expand_per_head(inp["sin"], H)
    expanded, _ = run_packed(w, inp, cos_layout="per_head_expanded",
                             dev_tabs=(torch.from_numpy(ce).cuda(), torch.from_numpy(se).cuda()))
    sb, eb = to_bits(shared), to_bits(expanded)
    np.testing.assert_array_equal(sb, eb)
    np.testing.assert_array_equal(sb[:, 2 * H * D:], inp["qkv"][:, 2 * H * D:])
    check_packed(w, sb, inp)


# ---------------------------------------------------------------------------
# host-resident activations through the chunked pipeline

@pytest.mark.parametrize("T,chunk", [(10000, 4096), (4096, 4096), (777, 256), (20000, 2048)])
def test_host_pipeline_matches_device_path(T, chunk):
    w = I.WORKLOADS["wan_32760x40x128"].with_(n_heads_q=8, n_heads_k=8, n_heads_v=8)
    inp = I.make_inputs(w, tokens=T)
    ref, _ = run_packed(w, inp)
    host = torch.from_numpy(inp["qkv"].view(np.int16)).view(torch.bfloat16).pin_memory()
    cos = torch.from_numpy(inp["cos"]).pin_memory()
    sin = torch.from_numpy(inp["sin"]).pin_memory()
    gq = torch.from_numpy(inp["gamma_q"]).pin_memory()
    gk = torch.from_numpy(inp["gamma_k"]).pin_memory()
    pipe = Q.HostPipeline(host.shape[1], torch.bfloat16, chunk_rows=chunk)
    out = torch.empty_like(host).pin_memory()
    pipe(host, 8, 8, 8, 128, gq, gk, cos, sin, out_host=out, rope_style=w.rope_style)
    torch.cuda.synchronize()
    assert pipe.read_status() == 0
    assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16))
    np.testing.assert_array_equal(host.view(torch.int16).numpy().view(np.uint16), inp["qkv"])   # input kept
    # in place, twice in a row through the same staging ring
    for _ in range(2):
        h2 = torch.from_numpy(inp["qkv"].view(np.int16)).view(torch.bfloat16).pin_memory()
        pipe(h2, 8, 8, 8, 128, gq, gk, cos, sin, rope_style=w.rope_style)
        torch.cuda.synchronize()
        assert torch.equal(h2.view(torch.int16), out.view(torch.int16))


def test_host_pipeline_in_place_moves_only_q_and_k():
    # a host activation with padded rows: in place, only the Q|K columns
    # travel; V and the padding are never written
    w = I.WORKLOADS["wan_32760x40x128"].with_(n_heads_q=4, n_heads_k=4, n_heads_v=4)
    T = 3000
    inp = I.make_inputs(w, tokens=T)
    ref, _ = run_packed(w, inp)
    width = 12 * 128
    padded = np.full((T, width + 64), 0x7F7F, dtype=np.uint16)
    padded[:, :width] = inp["qkv"]
    host_full = torch.from_numpy(padded.view(np.int16)).view(torch.bfloat16).pin_memory()
    host = host_full[:, :width]
    pipe = Q.HostPipeline(width, torch.bfloat16, chunk_rows=1024)
    pipe(host, 4, 4, 4, 128, torch.from_numpy(inp["gamma_q"]), torch.from_numpy(inp["gamma_k"]),
         torch.from_numpy(inp["cos"]), torch.from_numpy(inp["sin"]), rope_style=w.rope_style)
    torch.cuda.synchronize()
    assert pipe.read_status() == 0
    got = host_full.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got[:, :width], ref.cpu().view(torch.int16).numpy().view(np.uint16))
    assert np.all(got[:, width:] == 0x7F7F)
    assert pipe.last_d2h_bytes == T * 8 * 128 * 2


def test_host_pipeline_batch_broadcast_table():
    w = I.WORKLOADS["dense_4096x24x128"].with_(seq=500, batch=4, positions="1d")
    T = w.tokens
    inp = I.make_inputs(w)
    ref, _ = run_packed(w, inp)
    host = torch.from_numpy(inp["qkv"].view(np.int16)).view(torch.bfloat16).pin_memory()
    pipe = Q.HostPipeline(host.shape[1], torch.bfloat16, chunk_rows=1000)
    pipe(host, 24, 24, 24, 128, torch.from_numpy(inp["gamma_q"]), torch.from_numpy(inp["gamma_k"]),
         torch.from_numpy(inp["cos"]), torch.from_numpy(inp["sin"]), rope_style=w.rope_style)
    torch.cuda.synchronize()
    assert torch.equal(host.view(torch.int16), ref.cpu().view(torch.int16))
    # chunks must start on a multiple of the batch-broadcast table's rows
    with pytest.raises(Q.QknrError) as e:
        Q.HostPipeline(host.shape[1], torch.bfloat16, chunk_rows=700)(
            host, 24, 24, 24, 128, torch.from_numpy(inp["gamma_q"]), torch.from_numpy(inp["gamma_k"]),
            torch.from_numpy(inp["cos"]), torch.from_numpy(inp["sin"]))
    assert e.value.status == 2


# ---------------------------------------------------------------------------
# per-head expanded tables whose rows differ from head to head: head h of Q
# and head h of K must read table row [t, h] ("VisualGen Wan: deduplicate
# shared RoPE SMEM staging", Description: materialised per-head embeddings;
# Test Coverage: shared and per-head tables).  Tables that repeat one row
# for every head cannot tell a wrong head index from the right one; these
# can.

def _dev_table(t, cos_dtype):
    return table_to_dev(t, cos_dtype)


@pytest.mark.parametrize("out", [False, True], ids=["in_place", "out_of_place"])
@pytest.mark.parametrize("cos_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
@pytest.mark.parametrize("H,D", [(24, 64), (24, 128), (40, 128)])
def test_expanded_distinct_heads_packed(H, D, style, cos_dtype, out):
    w = I.Workload("expanded_distinct", 1, 613, H, H, H, D, "bf16", True, style, cos_dtype, "per_head_expanded",
                   "1d", (), (D,), seed=11)
    inp = I.make_inputs(w)
    ce, se = I.per_head_tables(w.seq, H, D, style, cos_dtype, seed=100 + H + D)
    res, src = run_packed(w, inp, out=out, dev_tabs=(_dev_table(ce, cos_dtype), _dev_table(se, cos_dtype)))
    ref = oracle_packed(w, inp, cos_layout="per_head_expanded", tables=(ce, se))
    bits = to_bits(res)
    compare(bits[:, : H * D], ref["q"], "bf16", "Q")
    compare(bits[:, H * D:2 * H * D], ref["k"], "bf16", "K")
    np.testing.assert_array_equal(bits[:, 2 * H * D:], ref["v"])
    if out:
        np.testing.assert_array_equal(to_bits(src), inp["qkv"])


@pytest.mark.parametrize("style", ["interleaved", "rotate_half"])
def test_expanded_distinct_per_dimension_angles(style):
    # every dimension of every head has its own angle, so the two members of
    # a pair read different table entries: the entry used for output d must
    # be entry d of head h
    H, D = 24, 128
    w = I.Workload("expanded_per_dim", 1, 300, H, H, 0, D, "fp16", True, style, "fp32", "per_head_expanded",
                   "1d", (), (D,), seed=12)
    inp = I.make_inputs(w)
    ce, se = I.per_head_tables(w.seq, H, D, style, "fp32", seed=5, per_dim=True)
    res, _ = run_packed(w, inp, dev_tabs=(_dev_table(ce, "fp32"), _dev_table(se, "fp32")))
    ref = oracle_packed(w, inp, cos_layout="per_head_expanded", tables=(ce, se))
    bits = to_bits(res)
    compare(bits[:, : H * D], ref["q"], "fp16", "Q")
    compare(bits[:, H * D:], ref["k"], "fp16", "K")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("cos_dtype", ["fp32", "bf16"])
def test_expanded_distinct_heads_separate_tensors(dtype, cos_dtype):
    # the per-tensor launch (k = NULL: one tensor's heads against the table)
    # and the single-launch Q+K form (with a V copy), batch-broadcast table
    H, D, S, B = 48, 128, 250, 2
    T = B * S
    g = np.random.Generator(np.random.PCG64(21))
    xs = {n: I.to_storage_bits(g.standard_normal((T, H * D)).astype(np.float32), dtype) for n in "qkv"}
    gq = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)
    gk = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)
    ce, se = I.per_head_tables(S, H, D, "rotate_half", cos_dtype, seed=22)
    cos, sin = _dev_table(ce, cos_dtype), _dev_table(se, cos_dtype)
    kw = dict(rope_style="rotate_half", cos_layout="per_head_expanded")
    refs = {n: O.forward_separate(xs[n], dtype, H, D, gam, 1e-6, ce, se, cos_dtype, "rotate_half",
                                  "per_head_expanded") for n, gam in (("q", gq), ("k", gk))}
    # one launch per tensor
    q, k = to_dev(xs["q"], dtype), to_dev(xs["k"], dtype)
    Q.qk_norm_rope_tensor(q, H, D, torch.from_numpy(gq).cuda(), cos, sin, **kw)
    Q.qk_norm_rope_tensor(k, H, D, torch.from_numpy(gk).cuda(), cos, sin, **kw)
    torch.cuda.synchronize()
    compare(to_bits(q), refs["q"], dtype, "Q per tensor")
    compare(to_bits(k), refs["k"], dtype, "K per tensor")
    # Q and K in one launch, out of place, V copied
    q2, k2, v2 = (to_dev(xs[n], dtype) for n in "qkv")
    qo, ko, vo = torch.empty_like(q2), torch.empty_like(k2), torch.empty_like(v2)
    Q.qk_norm_rope_separate(q2, k2, H, D, torch.from_numpy(gq).cuda(), torch.from_numpy(gk).cuda(), cos, sin,
                            v=v2, q_out=qo, k_out=ko, v_out=vo, **kw)
    torch.cuda.synchronize()
    compare(to_bits(qo), refs["q"], dtype, "Q single launch")
    compare(to_bits(ko), refs["k"], dtype, "K single launch")
    np.testing.assert_array_equal(to_bits(vo), xs["v"])
    assert torch.equal(qo.view(torch.int16), q.view(torch.int16))
    assert torch.equal(ko.view(torch.int16), k.view(torch.int16))
    for n, t in (("q", q2), ("k", k2), ("v", v2)):
        np.testing.assert_array_equal(to_bits(t), xs[n])


@pytest.mark.parametrize("style,cos_dtype", [("interleaved", "fp32"), ("rotate_half", "fp32"),
                                             ("interleaved", "bf16"), ("rotate_half", "bf16")])
def test_wan_expanded_distinct_heads_sampled(wan, style, cos_dtype):
    # the full Wan shape in the launch the benchmark times, with a table
    # [32760, 40, 128] that differs per head; sampled rows vs the oracle
    w0, inp = wan
    w = w0.with_(rope_style=style, cos_dtype=cos_dtype, cos_layout="per_head_expanded")
    H, D = w.n_heads_q, w.head_dim
    ce, se = I.per_head_tables(w.tokens, H, D, style, cos_dtype, seed=31)
    res, _ = run_packed(w, inp, dev_tabs=(_dev_table(ce, cos_dtype), _dev_table(se, cos_dtype)))
    bits = to_bits(res)
    rows = sample_rows(w.tokens, 96, seed=3)
    sub = dict(inp, qkv=inp["qkv"][rows])
    ref = oracle_packed(w, sub, cos_layout="per_head_expanded", tables=(ce[rows], se[rows]))
    compare(bits[rows][:, : H * D], ref["q"], "bf16", "Q")
    compare(bits[rows][:, H * D:2 * H * D], ref["k"], "bf16", "K")
    np.testing.assert_array_equal(bits[:, 2 * H * D:], inp["qkv"][:, 2 * H * D:])


@pytest.mark.parametrize("cos_dtype", ["fp32", "bf16"])
def test_expanded_distinct_heads_separate_tensors_with_the_prefetch(cos_dtype):
    # as above at 68 rows per CTA, where both launch forms prefetch their
    # second ring fill into L2 before the dependency wait (Q/K/V segments
    # and the per-head table rows of a batch-broadcast table)
    H, D, S, B, dtype = 16, 128, 5120, 2, "bf16"
    T = B * S
    g = np.random.Generator(np.random.PCG64(23))
    xs = {n: I.to_storage_bits(g.standard_normal((T, H * D)).astype(np.float32), dtype) for n in "qkv"}
    gq = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)
    gk = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)
    ce, se = I.per_head_tables(S, H, D, "interleaved", cos_dtype, seed=24)
    cos, sin = _dev_table(ce, cos_dtype), _dev_table(se, cos_dtype)
    dgq, dgk = torch.from_numpy(gq).cuda(), torch.from_numpy(gk).cuda()
    kw = dict(rope_style="interleaved", cos_layout="per_head_expanded")
    refs = {n: O.forward_separate(xs[n], dtype, H, D, gam, 1e-6, ce, se, cos_dtype, "interleaved",
                                  "per_head_expanded") for n, gam in (("q", gq), ("k", gk))}
    q, k = to_dev(xs["q"], dtype), to_dev(xs["k"], dtype)
    assert Q.query(Q.make_args(q=q, n_heads_q=H, head_dim=D, gamma_q=dgq, cos=cos, sin=sin, cos_rows=S,
                               **kw))["prefetch_rows"] > 0
    Q.qk_norm_rope_tensor(q, H, D, dgq, cos, sin, **kw)
    Q.qk_norm_rope_tensor(k, H, D, dgk, cos, sin, **kw)
    torch.cuda.synchronize()
    compare(to_bits(q), refs["q"], dtype, "Q per tensor")
    compare(to_bits(k), refs["k"], dtype, "K per tensor")
    q2, k2, v2 = (to_dev(xs[n], dtype) for n in "qkv")
    qo, ko, vo = torch.empty_like(q2), torch.empty_like(k2), torch.empty_like(v2)
    a = Q.make_args(q=q2, k=k2, v=v2, q_out=qo, k_out=ko, v_out=vo, n_heads_q=H, n_heads_k=H, n_heads_v=H,
                    head_dim=D, gamma_q=dgq, gamma_k=dgk, cos=cos, sin=sin, cos_rows=S, **kw)
    assert Q.query(a)["prefetch_rows"] > 0
    Q.qk_norm_rope_separate(q2, k2, H, D, dgq, dgk, cos, sin, v=v2, q_out=qo, k_out=ko, v_out=vo, **kw)
    torch.cuda.synchronize()
    compare(to_bits(qo), refs["q"], dtype, "Q single launch")
    compare(to_bits(ko), refs["k"], dtype, "K single launch")
    np.testing.assert_array_equal(to_bits(vo), xs["v"])
