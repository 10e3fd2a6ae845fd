"""Host threads calling the library at once, each on its own CUDA stream.

The entry points are documented as thread-safe: the per-device attribute
cache, the one-time kernel configuration and the per-thread error text are
shared or per-thread state that concurrent first calls must not corrupt.
Eight threads run the QK, AdaLN and group-norm calls concurrently (ctypes
drops the GIL for each call), and every result must equal, bit for bit,
the same call made alone on one thread."""
import threading

import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from tests.gpu_util import table_to_dev, to_dev

pytestmark = pytest.mark.gpu

THREADS = 8
REPEATS = 5


@pytest.fixture(scope="module", autouse=True)
def _lib(built_lib, cuda_device):
    Q.load()


def qk_packed_case():
    w = I.WORKLOADS["dense_4096x24x128"]
    inp = I.make_inputs(w, tokens=1500)
    qkv = to_dev(inp["qkv"], w.dtype)
    gq, gk = torch.from_numpy(inp["gamma_q"]).cuda(), torch.from_numpy(inp["gamma_k"]).cuda()
    cos, sin = table_to_dev(inp["cos"], w.cos_dtype), table_to_dev(inp["sin"], w.cos_dtype)

    def call(status):
        x = qkv.clone()
        Q.qk_norm_rope_packed(x, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim, gq, gk, cos, sin,
                              rope_style=w.rope_style, dev_status=status)
        return x
    return call


def qk_tensor_case():
    w = I.WORKLOADS["flux2_2x4608x48x128"]
    inp = I.make_inputs(w, tokens=700)
    q = to_dev(inp["q"], w.dtype)
    g = torch.from_numpy(inp["gamma_q"]).cuda()
    cos, sin = table_to_dev(inp["cos"], w.cos_dtype), table_to_dev(inp["sin"], w.cos_dtype)

    def call(status):
        out = torch.empty_like(q)
        Q.qk_norm_rope_tensor(q, w.n_heads_q, w.head_dim, g, cos, sin, out=out, rope_style=w.rope_style,
                              dev_status=status)
        return out
    return call


def adaln_case():
    w = I.AdaLNWorkload("t", 2, 333, 3072, mod_dtype="fp32", seed=11)
    inp = I.make_adaln_inputs(w)
    x = to_dev(inp["x"], w.dtype)
    sc, sh = torch.from_numpy(inp["scale"]).cuda(), torch.from_numpy(inp["shift"]).cuda()

    def call(status):
        out = torch.empty_like(x)
        Q.adaln_modulate(x, sc, sh, rows_per_batch=w.seq, out=out, eps=w.eps, dev_status=status)
        return out
    return call


def gn_case():
    w = I.GroupNormWorkload("t", 2, 64, 40, 48, groups=32, seed=12)
    inp = I.make_gn_inputs(w)
    x = to_dev(inp["x"], w.dtype)
    g, b = torch.from_numpy(inp["gamma"]).cuda(), torch.from_numpy(inp["beta"]).cuda()

    def call(status):
        # each call has its own workspace: calls sharing one must not overlap
        out = torch.empty_like(x)
        Q.group_norm_silu(x, w.groups, g, b, out=out, eps=w.eps)
        return out
    return call


def test_concurrent_threads_match_single_thread():
    cases = [qk_packed_case(), qk_tensor_case(), adaln_case(), gn_case()]
    status = torch.zeros(THREADS, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()

    results = [[None] * REPEATS for _ in range(THREADS)]
    errors = []
    start = threading.Barrier(THREADS)

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            call = cases[i % len(cases)]
            start.wait(timeout=60)
            with torch.cuda.stream(stream):
                for r in range(REPEATS):
                    results[i][r] = call(status[i:i + 1])
            stream.synchronize()
        except BaseException as e:                      # reported on the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    assert status.cpu().numpy().tolist() == [0] * THREADS, "a kernel reported a wait timeout"

    # the same calls, one at a time on the main thread
    refs = [c(None).view(torch.int16).cpu().numpy() for c in cases]
    for i in range(THREADS):
        for r in range(REPEATS):
            got = results[i][r].view(torch.int16).cpu().numpy()
            np.testing.assert_array_equal(got, refs[i % len(cases)], err_msg=f"thread {i} call {r}")


def test_last_error_is_per_thread():
    # a worker fails, the main thread then fails differently, and the
    # worker still reads its own message
    x = torch.zeros((8, 3 * 128), dtype=torch.bfloat16, device="cuda")
    x96 = torch.zeros((8, 3 * 96), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(128, dtype=torch.float32, device="cuda")
    cos = torch.ones((8, 128), dtype=torch.float32, device="cuda")
    cos96 = torch.ones((8, 96), dtype=torch.float32, device="cuda")
    failed, main_failed = threading.Event(), threading.Event()
    seen = {}

    def worker():
        try:
            Q.qk_norm_rope_packed(x96, 1, 1, 1, 96, g, g, cos96, cos96)
        except Q.QknrError as e:
            seen["status"] = e.status
        failed.set()
        main_failed.wait(timeout=60)
        seen["msg"] = Q.last_error()

    t = threading.Thread(target=worker)
    t.start()
    assert failed.wait(timeout=60)
    with pytest.raises(Q.QknrError):
        Q.qk_norm_rope_packed(x, 1, 1, 1, 128, g, g, cos, cos, eps=-1.0)
    main_failed.set()
    t.join(timeout=60)
    assert seen.get("status") == 4                         # QKNR_ERR_UNSUPPORTED
    assert "head_dim 96" in seen["msg"]
    assert "eps" in Q.last_error()
