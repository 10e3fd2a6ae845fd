"""Buffers past 2 GiB: byte offsets that do not fit 32 bits, for the QK,
AdaLN and group-norm calls.  The QK and AdaLN cases place narrow rows at a
wide row stride, so the buffer is large while the generated data stays
small; the group norm's NCHW activation is 2.3 GB of data.  Results are
checked against the oracle on rows and groups near the start, across the
2^31-byte boundary and at the end; padding columns must come back
untouched."""
import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from oracle import adaln_oracle as A
from oracle import groupnorm_oracle as G
from oracle import qknr_oracle as O
from tests.gpu_util import compare, to_bits, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SENTINEL = 0x7F7F          # a bf16 bit pattern no kernel here writes to padding


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()
    Q.status_buffer().zero_()
    yield
    assert Q.read_status() == 0


def boundary_rows(T, row_bytes):
    """Rows at the start, either side of the 2^31-byte offset, and the end."""
    b = (1 << 31) // row_bytes
    return np.unique(np.array([0, 1, b - 1, b, b + 1, T // 2, T - 2, T - 1]))


def wide_buffer(T, stride, used_bits):
    """Device bf16 [T, stride] with the first columns set to used_bits and
    the rest to SENTINEL."""
    buf = torch.full((T, stride), 0, dtype=torch.int16, device="cuda")
    buf.fill_(SENTINEL)
    buf[:, :used_bits.shape[1]].copy_(torch.from_numpy(used_bits.view(np.int16)))
    return buf.view(torch.bfloat16)


def test_qk_tensor_past_2gib():
    T, H, D, stride = 70000, 4, 128, 16384          # 32 KB rows: 2.29 GB
    g = np.random.Generator(np.random.PCG64(81))
    xb = I.to_storage_bits(g.standard_normal((T, H * D)).astype(np.float32), "bf16")
    gamma = (1 + 0.1 * g.standard_normal(D)).astype(np.float32)
    ang = g.uniform(-np.pi, np.pi, size=(4096, D // 2))
    full = np.concatenate([ang, ang], axis=1)
    cos, sin = np.cos(full).astype(np.float32), np.sin(full).astype(np.float32)
    buf = wide_buffer(T, stride, xb)
    assert buf.numel() * 2 > (1 << 31)
    x = buf[:, :H * D]
    Q.qk_norm_rope_tensor(x, H, D, torch.from_numpy(gamma).cuda(), torch.from_numpy(cos).cuda(),
                          torch.from_numpy(sin).cuda(), rope_style="rotate_half")
    torch.cuda.synchronize()
    rows = boundary_rows(T, stride * 2)
    got = to_bits(buf[torch.from_numpy(rows).cuda()])
    ref = O.forward_separate(xb, "bf16", H, D, gamma, 1e-6, cos, sin, "fp32", "rotate_half", rows=rows)
    compare(got[:, :H * D], ref, "bf16", "qk past 2 GiB")
    assert np.all(got[:, H * D:] == SENTINEL)


def test_adaln_past_2gib():
    T, C, stride, rpb = 40000, 1024, 32768, 9999     # 64 KB rows: 2.62 GB; 5 samples
    g = np.random.Generator(np.random.PCG64(82))
    xb = I.to_storage_bits((3 * g.standard_normal((T, C)) + 1.0).astype(np.float32), "bf16")
    B = -(-T // rpb)
    sc = (0.1 * g.standard_normal((B, C))).astype(np.float32)
    sh = (0.1 * g.standard_normal((B, C))).astype(np.float32)
    buf = wide_buffer(T, stride, xb)
    assert buf.numel() * 2 > (1 << 31)
    x = buf[:, :C]
    Q.adaln_modulate(x, torch.from_numpy(sc).cuda(), torch.from_numpy(sh).cuda(), rows_per_batch=rpb, eps=1e-6)
    torch.cuda.synchronize()
    rows = boundary_rows(T, stride * 2)
    got = to_bits(buf[torch.from_numpy(rows).cuda()])
    ref = A.adaln_modulate(xb, "bf16", sc, sh, "fp32", 1e-6, rpb, rows=rows)
    compare(got[:, :C], ref, "bf16", "adaln past 2 GiB")
    assert np.all(got[:, C:] == SENTINEL)


def bf16_bits(g, n):
    """n random bf16 bit patterns of magnitude in [2^-8, 2), either sign
    (made as bits directly: 2.3 GB of normals would take minutes)."""
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 26
    for i in range(0, n, step):
        r = g.integers(0, 1 << 32, size=min(step, n - i), dtype=np.uint32)
        sign = (r >> 31).astype(np.uint16) << 15
        exp = (119 + ((r >> 7) & 7)).astype(np.uint16) << 7
        out[i:i + len(r)] = sign | exp | (r & 0x7F).astype(np.uint16)
    return out


def test_group_norm_past_2gib():
    N, C, H, W, groups = 17, 64, 1024, 1024, 32      # 1.14 G elements: 2.28 GB
    g = np.random.Generator(np.random.PCG64(83))
    xb = bf16_bits(g, N * C * H * W).reshape(N, C, H, W)
    gamma = (1 + 0.1 * g.standard_normal(C)).astype(np.float32)
    beta = (0.1 * g.standard_normal(C)).astype(np.float32)
    x = to_dev(xb, "bf16")
    assert x.numel() * 2 > (1 << 31)
    gm, bt = torch.from_numpy(gamma).cuda(), torch.from_numpy(beta).cuda()
    out = torch.empty_like(x)
    Q.group_norm_silu(x, groups, gm, bt, out=out, eps=1e-6)          # fused
    torch.cuda.synchronize()
    two = torch.empty_like(x)
    Q.group_norm_silu(x, groups, gm, bt, out=two, eps=1e-6, mode="two_pass", piece_elems=12288)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), two.view(torch.int16))
    del two
    # elements of the first and last samples and of the sample crossing 2^31 bytes
    n_cross = (1 << 31) // (C * H * W * 2)
    rng = np.random.Generator(np.random.PCG64(84))
    k = 600
    idx = (np.repeat([0, n_cross, N - 1], k // 3), rng.integers(0, C, k), rng.integers(0, H, k),
           rng.integers(0, W, k))
    got = to_bits(out[tuple(torch.from_numpy(np.ascontiguousarray(i)).cuda() for i in idx)])
    ref = G.group_norm_silu_at(xb, "bf16", groups, gamma, beta, 1e-6, idx)
    compare(got, ref, "bf16", "group norm past 2 GiB")
