"""The C-ABI library builds, loads and exports every declared symbol, and its
host-side validation rejects bad arguments before any CUDA call.  Runs
without a GPU: the pointers here are plain integers that are never touched
because every call returns during validation."""
import ctypes
import os
import re

import pytest
import torch

from diffusion_transformer_qk_gb300 import qknr as Q

# These tests hand the library fake device addresses and rely on it
# rejecting every call before a launch; they never run where a GPU is
# visible, so a call that validation let through cannot touch a device.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="host-only tests with fake device addresses")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib(built_lib):
    return Q.load()


def declared_functions():
    names = set()
    for f in sorted(os.listdir(INCLUDE)):
        if f.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, f)).read(), flags=re.S)
            names.update(re.findall(r"\b(qknr_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_exports():
    assert sorted(Q.EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_struct_layouts_match(lib):
    assert lib.qknr_gn_sizeof_args() == ctypes.sizeof(Q.QknrGnArgs)
    assert lib.qknr_adaln_sizeof_args() == ctypes.sizeof(Q.QknrAdaLNArgs)
    assert lib.qknr_sizeof_args() == ctypes.sizeof(Q.QknrArgs)
    assert lib.qknr_sizeof_launch_info() == ctypes.sizeof(Q.QknrLaunchInfo)
    assert lib.qknr_abi_version() == Q.ABI_VERSION


def test_args_init_defaults(lib):
    a = Q.QknrArgs()
    ctypes.memset(ctypes.byref(a), 0xFF, ctypes.sizeof(a))
    lib.qknr_args_init(ctypes.byref(a))
    assert a.abi_version == Q.ABI_VERSION
    assert a.dtype == Q.BF16 and a.cos_dtype == Q.FP32
    assert abs(a.eps - 1e-6) < 1e-12
    assert a.q is None and a.tokens == 0 and a.stages == 0 and a.wait_limit_ns == 0


def test_status_strings(lib):
    for code, name in Q.STATUS.items():
        s = lib.qknr_status_string(code).decode()
        assert s and s != "unknown status", name
    assert lib.qknr_status_string(99).decode() == "unknown status"


FAKE = 1 << 40        # 16-byte aligned addresses that are never dereferenced


def valid_packed(T=64, H=4, D=128):
    """Args for an in-place packed call with fake device pointers."""
    a = Q.QknrArgs()
    Q.load().qknr_args_init(ctypes.byref(a))
    row = 3 * H * D
    a.q, a.k, a.v = FAKE, FAKE + H * D * 2, FAKE + 2 * H * D * 2
    a.q_stride = a.k_stride = a.v_stride = row
    a.tokens = T
    a.n_heads_q = a.n_heads_k = a.n_heads_v = H
    a.head_dim = D
    a.gamma_q, a.gamma_k = FAKE + (1 << 30), FAKE + (1 << 30) + 4096
    a.cos, a.sin = FAKE + (2 << 30), FAKE + (3 << 30)
    return a


def call(lib, a):
    st = lib.qknr_forward(ctypes.byref(a), None)
    return st, lib.qknr_last_error().decode()


def test_null_args(lib):
    assert lib.qknr_forward(None, None) == 1


@pytest.mark.parametrize("mutate,expect", [
    (lambda a: setattr(a, "abi_version", 7), 8),
    (lambda a: setattr(a, "head_dim", 96), 4),
    (lambda a: setattr(a, "dtype", 2), 4),
    (lambda a: setattr(a, "cos_dtype", 1), 4),
    (lambda a: setattr(a, "rope_style", 5), 4),
    (lambda a: setattr(a, "cos_layout", 3), 4),
    (lambda a: setattr(a, "tokens", -1), 2),
    (lambda a: setattr(a, "n_heads_k", -2), 2),
    (lambda a: setattr(a, "stages", 1), 2),
    (lambda a: setattr(a, "stages", 17), 2),
    (lambda a: setattr(a, "consumer_warps", 17), 2),
    (lambda a: setattr(a, "ctas_per_sm", 5), 2),
    (lambda a: (setattr(a, "consumer_warps", 12), setattr(a, "group_warps", 5)), 2),
    (lambda a: setattr(a, "group_warps", 17), 2),
    (lambda a: setattr(a, "eps", -1.0), 2),
    (lambda a: setattr(a, "gamma_q", None), 1),
    (lambda a: setattr(a, "k", None), 1),
    (lambda a: setattr(a, "cos", None), 1),
    (lambda a: setattr(a, "q_stride", 100), 2),            # < heads * D
    (lambda a: setattr(a, "q", FAKE + 8), 3),              # not 16-byte aligned
    (lambda a: setattr(a, "q_stride", 3 * 4 * 128 + 4), 3),  # 8-byte row stride
    (lambda a: setattr(a, "sin", FAKE + (3 << 30) + 4), 3),
    (lambda a: setattr(a, "gamma_k", FAKE + (1 << 30) + 2), 3),
    (lambda a: setattr(a, "cos_rows", -3), 2),
])
def test_validation_rejects(lib, mutate, expect):
    a = valid_packed()
    mutate(a)
    st, msg = call(lib, a)
    assert st == expect, (st, msg)
    assert msg


def test_expanded_layout_needs_equal_head_counts(lib):
    a = valid_packed()
    a.cos_layout = 1
    a.n_heads_k = 2
    assert call(lib, a)[0] == 2


def test_out_of_place_output_overlapping_an_input_is_rejected(lib):
    a = valid_packed()
    a.q_out = FAKE + 4 * 128 * 2          # lands on K
    assert call(lib, a)[0] == 7
    b = valid_packed()
    b.q_out = FAKE
    b.q_out_stride = 4 * 128              # same base, different stride
    assert call(lib, b)[0] == 7
    c = valid_packed()
    c.v_out = c.cos                        # V copied onto the cos table
    assert call(lib, c)[0] == 7


def test_nothing_to_do_returns_ok_without_cuda(lib):
    # zero tokens, or no heads and no V copy: OK before any device query
    a = valid_packed(T=0)
    assert call(lib, a)[0] == 0
    b = valid_packed()
    b.n_heads_q = b.n_heads_k = 0
    b.gamma_q = b.gamma_k = None
    assert call(lib, b)[0] == 0          # V untouched (v_out NULL): no work


def test_query_validates_too(lib):
    info = Q.QknrLaunchInfo()
    a = valid_packed()
    a.head_dim = 32
    assert lib.qknr_query(ctypes.byref(a), ctypes.byref(info)) == 4
    b = valid_packed(T=0)
    assert lib.qknr_query(ctypes.byref(b), ctypes.byref(info)) == 0
    assert info.grid == 0 and "qknr_fused<bf16,fp32,D128,interleaved,shared>" == info.kernel.decode()


def test_product_path_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        Q.load(str(tmp_path / "libqknr.so"))


# ---------------------------------------------------------------------------
# AdaLN scale/shift host validation

def valid_adaln(T=64, C=6144):
    a = Q.QknrAdaLNArgs()
    Q.load().qknr_adaln_args_init(ctypes.byref(a))
    a.x, a.tokens, a.hidden = FAKE, T, C
    a.scale, a.shift = FAKE + (1 << 30), FAKE + (2 << 30)
    return a


def adaln_call(lib, a):
    return lib.qknr_adaln_forward(ctypes.byref(a), None), lib.qknr_last_error().decode()


def test_adaln_args_init_defaults(lib):
    a = Q.QknrAdaLNArgs()
    ctypes.memset(ctypes.byref(a), 0xFF, ctypes.sizeof(a))
    lib.qknr_adaln_args_init(ctypes.byref(a))
    assert a.abi_version == Q.ABI_VERSION and a.dtype == Q.BF16 and a.mod_dtype == Q.BF16
    assert abs(a.eps - 1e-6) < 1e-12 and a.x is None and a.tokens == 0


@pytest.mark.parametrize("mutate,expect", [
    (lambda a: setattr(a, "abi_version", Q.ABI_VERSION + 1), 8),
    (lambda a: setattr(a, "dtype", 2), 4),
    (lambda a: setattr(a, "mod_dtype", 1), 4),            # fp16 modulation for bf16 activations
    (lambda a: setattr(a, "hidden", 100), 4),             # not a multiple of 8
    (lambda a: setattr(a, "hidden", 32776), 4),
    (lambda a: setattr(a, "tokens", -1), 2),
    (lambda a: setattr(a, "rows_per_batch", -5), 2),
    (lambda a: setattr(a, "eps", -0.5), 2),
    (lambda a: setattr(a, "x", None), 1),
    (lambda a: setattr(a, "shift", None), 1),
    (lambda a: setattr(a, "x_stride", 6000), 2),
    (lambda a: setattr(a, "x", FAKE + 8), 3),
    (lambda a: setattr(a, "x_stride", 6148), 3),          # 8-byte row stride
    (lambda a: setattr(a, "scale", FAKE + (1 << 30) + 4), 3),
    (lambda a: setattr(a, "out", FAKE + 2 * 6144 * 2), 7),  # out lands inside x
    (lambda a: setattr(a, "out", FAKE + (2 << 30)), 7),   # out on shift
    (lambda a: setattr(a, "stages", 1), 2),
    (lambda a: (setattr(a, "consumer_warps", 16), setattr(a, "group_warps", 3)), 2),
])
def test_adaln_validation_rejects(lib, mutate, expect):
    a = valid_adaln()
    mutate(a)
    st, msg = adaln_call(lib, a)
    assert st == expect, (st, msg)
    assert msg


def test_adaln_zero_tokens_is_ok_without_cuda(lib):
    a = valid_adaln(T=0)
    a.x = a.scale = a.shift = None
    assert adaln_call(lib, a)[0] == 0


# ---------------------------------------------------------------------------
# group norm + SiLU host validation

def valid_gn():
    a = Q.QknrGnArgs()
    Q.load().qknr_gn_args_init(ctypes.byref(a))
    a.x = FAKE
    a.n, a.c, a.h, a.w, a.groups = 1, 64, 16, 16, 32
    a.gamma, a.beta = FAKE + (1 << 30), FAKE + (1 << 30) + 4096
    a.workspace, a.workspace_bytes = FAKE + (2 << 30), 1 << 20
    return a


def gn_ws(lib, a):
    n = ctypes.c_size_t(0)
    assert lib.qknr_gn_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 0, lib.qknr_last_error()
    return n.value


def test_gn_workspace_bytes(lib):
    a = valid_gn()
    # 32 spans of 2*16*16 = 512 elements: one piece each on both paths
    # (two-pass pieces are at least 65536 elements, fused ones 12288), plus
    # the shift record; the fused path adds 16 bytes (its abort word)
    a.mode = Q.GN_MODE["two_pass"]
    assert gn_ws(lib, a) == 32 * 2 * 16
    a.mode = Q.GN_MODE["fused"]
    assert gn_ws(lib, a) == 32 * 2 * 16 + 16
    a.mode = Q.GN_MODE["auto"]                     # the larger of the two
    assert gn_ws(lib, a) == 32 * 2 * 16 + 16
    a.piece_elems = 64                             # two-pass tuning: two-pass only
    assert gn_ws(lib, a) == 32 * (8 + 1) * 16
    # a group of 2 x 128 x 128 = 32768 elements: 3 fused pieces of 12288
    a = valid_gn()
    a.h = a.w = 128
    a.mode = Q.GN_MODE["fused"]
    assert gn_ws(lib, a) == 32 * (3 + 1) * 16 + 16


def test_gn_cluster_mode_needs_no_workspace_and_takes_groups_up_to_a_cluster(lib):
    a = valid_gn()
    a.mode = Q.GN_MODE["cluster"]
    assert gn_ws(lib, a) == 0
    # 16 CTAs of at most 200 KB each: a group of 1,638,400 elements fits,
    # one of 1,703,936 does not (checked before any CUDA call)
    a.c, a.groups, a.h, a.w = 25, 1, 256, 256
    assert gn_ws(lib, a) == 0
    a.c = 26
    n = ctypes.c_size_t(0)
    assert lib.qknr_gn_workspace_bytes(ctypes.byref(a), ctypes.byref(n)) == 4


def test_gn_workspace_does_not_depend_on_the_device(lib):
    # no CUDA call is made: the size comes from the arguments alone
    a = valid_gn()
    a.x = a.gamma = a.beta = a.workspace = None
    assert gn_ws(lib, a) > 0


@pytest.mark.parametrize("mutate,expect", [
    (lambda a: setattr(a, "abi_version", 0), 8),
    (lambda a: setattr(a, "dtype", 2), 4),
    (lambda a: setattr(a, "groups", 5), 2),                 # does not divide 64
    (lambda a: (setattr(a, "w", 3), setattr(a, "h", 3)), 4),  # H*W = 9, not a multiple of 8
    (lambda a: setattr(a, "n", 0), 2),
    (lambda a: setattr(a, "eps", -1.0), 2),
    (lambda a: setattr(a, "piece_elems", 12), 2),
    (lambda a: setattr(a, "l2_batch_bytes", -7), 2),
    (lambda a: setattr(a, "x", None), 1),
    (lambda a: setattr(a, "workspace", None), 1),
    (lambda a: setattr(a, "workspace_bytes", 100), 2),
    (lambda a: setattr(a, "x", FAKE + 8), 3),
    (lambda a: setattr(a, "workspace", FAKE + (2 << 30) + 8), 3),
    (lambda a: setattr(a, "gamma", FAKE + (1 << 30) + 2), 3),
    (lambda a: setattr(a, "out", FAKE + 1024), 7),          # out inside x
    (lambda a: setattr(a, "workspace", FAKE + 4096), 7),    # workspace inside x
    (lambda a: setattr(a, "mode", 4), 4),
    (lambda a: setattr(a, "dev_status", FAKE + 3 * (1 << 30) + 2), 3),
])
def test_gn_validation_rejects(lib, mutate, expect):
    a = valid_gn()
    mutate(a)
    st = lib.qknr_gn_silu_forward(ctypes.byref(a), None)
    assert st == expect, (st, lib.qknr_last_error().decode())


# ---------------------------------------------------------------------------
# qknr_forward_host: plan validation returns before any CUDA call

def valid_host_plan(n=3, chunk=16):
    p = Q.QknrHostPlan()
    Q.load().qknr_host_plan_init(ctypes.byref(p))
    assert p.abi_version == Q.ABI_VERSION and p.n_buffers == 3 and p.chunk_rows == 2048
    p.n_buffers, p.chunk_rows = n, chunk
    for i in range(n):
        p.dev_buffers[i] = FAKE + (4 << 30) + i * (1 << 24)
    for i in range(3 * n + 2):
        p.events[i] = 0x1000 + 16 * i
    return p


def call_host(lib, a, p):
    st = lib.qknr_forward_host(ctypes.byref(a) if a is not None else None,
                               ctypes.byref(p) if p is not None else None, None)
    return st, lib.qknr_last_error().decode()


@pytest.mark.parametrize("mutate,expect", [
    (lambda a, p: setattr(p, "n_buffers", 0), 2),
    (lambda a, p: setattr(p, "n_buffers", 5), 2),
    (lambda a, p: setattr(p, "chunk_rows", 0), 2),
    (lambda a, p: setattr(p, "abi_version", 1), 8),
    (lambda a, p: p.dev_buffers.__setitem__(2, None), 1),
    (lambda a, p: p.dev_buffers.__setitem__(1, FAKE + 8), 3),
    (lambda a, p: p.events.__setitem__(10, None), 1),
    (lambda a, p: setattr(a, "head_dim", 96), 4),
    (lambda a, p: setattr(a, "q", None), 1),
    (lambda a, p: setattr(a, "q_stride", 100), 2),
    # a batch-broadcast table of 12 rows with 16-row chunks
    (lambda a, p: setattr(a, "cos_rows", 12), 2),
    # a separate output that overlaps the K input rows
    (lambda a, p: setattr(a, "q_out", FAKE + 4 * 128 * 2 + 64), 7),
])
def test_host_call_validation_rejects(lib, mutate, expect):
    a, p = valid_packed(), valid_host_plan()
    mutate(a, p)
    st, msg = call_host(lib, a, p)
    assert st == expect, (st, msg)
    assert msg


def test_host_call_null_arguments(lib):
    assert call_host(lib, None, valid_host_plan())[0] == 1
    assert call_host(lib, valid_packed(), None)[0] == 1


def test_host_buffer_bytes(lib):
    a, p = valid_packed(T=100, H=4, D=128), valid_host_plan(chunk=16)
    n = ctypes.c_size_t(0)
    # in place: Q and K columns only
    assert lib.qknr_host_buffer_bytes(ctypes.byref(a), ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value == 16 * 8 * 128 * 2
    # V copied to a separate output: Q, K and V columns
    a.v_out = FAKE + (5 << 30)
    assert lib.qknr_host_buffer_bytes(ctypes.byref(a), ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value == 16 * 12 * 128 * 2
    p.chunk_rows = 0
    assert lib.qknr_host_buffer_bytes(ctypes.byref(a), ctypes.byref(p), ctypes.byref(n)) == 2


def test_host_call_with_no_rows_is_a_no_op(lib):
    a, p = valid_packed(T=0), valid_host_plan()
    assert call_host(lib, a, p)[0] == 0
