"""Python binding of libqknr.so (ctypes).

Argument marshalling only: tensors are turned into device pointers, row
strides and the current CUDA stream, and every step of the operation runs
in the library's kernels.  The binding has no fallback: if the library is
missing or cannot be loaded, every call raises.

The operation (per-head RMSNorm of Q and K followed by RoPE, V passed
through) is described in ``include/qknr.h``.
"""
from __future__ import annotations

import ctypes
import glob
import os
import threading
from ctypes import c_char, c_float, c_int32, c_int64, c_size_t, c_uint32, c_uint64, c_void_p
from typing import Optional

import torch

from . import build as _build

# enum values of include/qknr.h
BF16, FP16, FP32 = 0, 1, 2
ROPE = {"interleaved": 0, "rotate_half": 1}
COS_LAYOUT = {"shared_row": 0, "per_head_expanded": 1}
STATUS = {
    0: "QKNR_OK", 1: "QKNR_ERR_NULL", 2: "QKNR_ERR_SHAPE", 3: "QKNR_ERR_ALIGN",
    4: "QKNR_ERR_UNSUPPORTED", 5: "QKNR_ERR_CUDA", 6: "QKNR_ERR_TIMEOUT",
    7: "QKNR_ERR_OVERLAP", 8: "QKNR_ERR_ABI", 9: "QKNR_ERR_BOUNDS",
}
STATUS_BY_NAME = {v: k for k, v in STATUS.items()}
OK, ERR_TIMEOUT = 0, 6
FLAG_TEST_STALL = 0x1
FLAG_NO_OVERLAP = 0x2
FLAG_TEST_SHORT_OUT = 0x4
FLAG_NO_PREFETCH = 0x8
ABI_VERSION = 3

EXPORTS = (
    "qknr_args_init", "qknr_forward", "qknr_query", "qknr_status_string",
    "qknr_last_error", "qknr_abi_version", "qknr_sizeof_args", "qknr_sizeof_launch_info",
    "qknr_adaln_args_init", "qknr_adaln_forward", "qknr_adaln_query", "qknr_adaln_sizeof_args",
    "qknr_gn_args_init", "qknr_gn_workspace_bytes", "qknr_gn_silu_forward", "qknr_gn_sizeof_args",
    "qknr_gn_silu_forward_noalloc", "qknr_gn_query",
    "qknr_host_plan_init", "qknr_host_buffer_bytes", "qknr_forward_host", "qknr_sizeof_host_plan",
)
GN_MODE = {"auto": 0, "fused": 1, "two_pass": 2, "cluster": 3}
GN_FLAG_TEST_NO_RECORDS = 0x2
GN_NOALLOC_SCRATCH_BYTES = 1 << 20
HOST_MAX_BUFFERS = 4


class QknrArgs(ctypes.Structure):
    """Mirror of ``qknr_args``."""

    _fields_ = [
        ("abi_version", c_uint32), ("dtype", c_int32),
        ("q", c_void_p), ("k", c_void_p), ("v", c_void_p),
        ("q_out", c_void_p), ("k_out", c_void_p), ("v_out", c_void_p),
        ("q_stride", c_int64), ("k_stride", c_int64), ("v_stride", c_int64),
        ("q_out_stride", c_int64), ("k_out_stride", c_int64), ("v_out_stride", c_int64),
        ("tokens", c_int64),
        ("n_heads_q", c_int32), ("n_heads_k", c_int32), ("n_heads_v", c_int32),
        ("head_dim", c_int32),
        ("gamma_q", c_void_p), ("gamma_k", c_void_p), ("eps", c_float),
        ("cos", c_void_p), ("sin", c_void_p),
        ("cos_dtype", c_int32), ("cos_layout", c_int32), ("cos_rows", c_int64),
        ("rope_style", c_int32),
        ("dev_status", c_void_p),
        ("ctas_per_sm", c_int32), ("stages", c_int32), ("consumer_warps", c_int32),
        ("group_warps", c_int32), ("flags", c_uint32), ("wait_limit_ns", c_uint64),
    ]


class QknrLaunchInfo(ctypes.Structure):
    """Mirror of ``qknr_launch_info``."""

    _fields_ = [
        ("grid", c_int32), ("block", c_int32), ("dyn_smem", c_int32), ("stages", c_int32),
        ("ctas_per_sm", c_int32), ("consumer_warps", c_int32), ("group_warps", c_int32),
        ("stage_bytes", c_int32),
        ("registers", c_int32), ("num_sms", c_int32), ("prefetch_rows", c_int32), ("kernel", c_char * 96),
    ]

    def as_dict(self):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["kernel"] = self.kernel.decode()
        return d


class QknrAdaLNArgs(ctypes.Structure):
    """Mirror of ``qknr_adaln_args``."""

    _fields_ = [
        ("abi_version", c_uint32), ("dtype", c_int32),
        ("x", c_void_p), ("out", c_void_p),
        ("x_stride", c_int64), ("out_stride", c_int64),
        ("tokens", c_int64), ("hidden", c_int32), ("rows_per_batch", c_int64),
        ("scale", c_void_p), ("shift", c_void_p), ("mod_dtype", c_int32), ("mod_stride", c_int64),
        ("eps", c_float), ("dev_status", c_void_p),
        ("ctas_per_sm", c_int32), ("stages", c_int32), ("consumer_warps", c_int32), ("group_warps", c_int32),
        ("flags", c_uint32), ("wait_limit_ns", c_uint64),
    ]


class QknrGnArgs(ctypes.Structure):
    """Mirror of ``qknr_gn_args``."""

    _fields_ = [
        ("abi_version", c_uint32), ("dtype", c_int32),
        ("x", c_void_p), ("out", c_void_p),
        ("n", c_int32), ("c", c_int32), ("h", c_int32), ("w", c_int32), ("groups", c_int32),
        ("gamma", c_void_p), ("beta", c_void_p), ("eps", c_float),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("piece_elems", c_int32), ("l2_batch_bytes", c_int64),
        ("dev_status", c_void_p), ("mode", c_int32), ("flags", c_uint32), ("wait_limit_ns", c_uint64),
    ]


class QknrHostPlan(ctypes.Structure):
    """Mirror of ``qknr_host_plan``."""

    _fields_ = [
        ("abi_version", c_uint32), ("n_buffers", c_int32), ("chunk_rows", c_int64),
        ("dev_buffers", c_void_p * HOST_MAX_BUFFERS), ("h2d_stream", c_void_p), ("d2h_stream", c_void_p),
        ("events", c_void_p * (3 * HOST_MAX_BUFFERS + 2)),
        ("host_gamma_q", c_void_p), ("host_gamma_k", c_void_p), ("host_cos", c_void_p), ("host_sin", c_void_p),
    ]


class QknrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path(checked: bool = False) -> str:
    return _build.library_path(checked)


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libqknr.so (once).  Raises if it is missing or malformed."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is not built; build it with diffusion_transformer_qk_gb300.build.build_library()")
        lib = ctypes.CDLL(p)
        lib.qknr_args_init.argtypes = [ctypes.POINTER(QknrArgs)]
        lib.qknr_args_init.restype = None
        lib.qknr_forward.argtypes = [ctypes.POINTER(QknrArgs), c_void_p]
        lib.qknr_forward.restype = c_int32
        lib.qknr_query.argtypes = [ctypes.POINTER(QknrArgs), ctypes.POINTER(QknrLaunchInfo)]
        lib.qknr_query.restype = c_int32
        lib.qknr_status_string.argtypes = [c_int32]
        lib.qknr_status_string.restype = ctypes.c_char_p
        lib.qknr_last_error.argtypes = []
        lib.qknr_last_error.restype = ctypes.c_char_p
        lib.qknr_abi_version.argtypes = []
        lib.qknr_abi_version.restype = c_int32
        lib.qknr_sizeof_args.restype = c_size_t
        lib.qknr_sizeof_launch_info.restype = c_size_t
        lib.qknr_adaln_args_init.argtypes = [ctypes.POINTER(QknrAdaLNArgs)]
        lib.qknr_adaln_args_init.restype = None
        lib.qknr_adaln_forward.argtypes = [ctypes.POINTER(QknrAdaLNArgs), c_void_p]
        lib.qknr_adaln_forward.restype = c_int32
        lib.qknr_adaln_query.argtypes = [ctypes.POINTER(QknrAdaLNArgs), ctypes.POINTER(QknrLaunchInfo)]
        lib.qknr_adaln_query.restype = c_int32
        lib.qknr_adaln_sizeof_args.restype = c_size_t
        lib.qknr_gn_args_init.argtypes = [ctypes.POINTER(QknrGnArgs)]
        lib.qknr_gn_args_init.restype = None
        lib.qknr_gn_workspace_bytes.argtypes = [ctypes.POINTER(QknrGnArgs), ctypes.POINTER(c_size_t)]
        lib.qknr_gn_workspace_bytes.restype = c_int32
        lib.qknr_gn_silu_forward.argtypes = [ctypes.POINTER(QknrGnArgs), c_void_p]
        lib.qknr_gn_silu_forward.restype = c_int32
        lib.qknr_gn_sizeof_args.restype = c_size_t
        lib.qknr_gn_silu_forward_noalloc.argtypes = [ctypes.POINTER(QknrGnArgs), c_void_p]
        lib.qknr_gn_silu_forward_noalloc.restype = c_int32
        lib.qknr_gn_query.argtypes = [ctypes.POINTER(QknrGnArgs), ctypes.POINTER(QknrLaunchInfo)]
        lib.qknr_gn_query.restype = c_int32
        lib.qknr_host_plan_init.argtypes = [ctypes.POINTER(QknrHostPlan)]
        lib.qknr_host_plan_init.restype = None
        lib.qknr_host_buffer_bytes.argtypes = [ctypes.POINTER(QknrArgs), ctypes.POINTER(QknrHostPlan),
                                               ctypes.POINTER(c_size_t)]
        lib.qknr_host_buffer_bytes.restype = c_int32
        lib.qknr_forward_host.argtypes = [ctypes.POINTER(QknrArgs), ctypes.POINTER(QknrHostPlan), c_void_p]
        lib.qknr_forward_host.restype = c_int32
        lib.qknr_sizeof_host_plan.restype = c_size_t
        if lib.qknr_abi_version() != ABI_VERSION:
            raise RuntimeError("libqknr.so ABI version mismatch")
        if lib.qknr_sizeof_args() != ctypes.sizeof(QknrArgs) or \
                lib.qknr_sizeof_launch_info() != ctypes.sizeof(QknrLaunchInfo) or \
                lib.qknr_adaln_sizeof_args() != ctypes.sizeof(QknrAdaLNArgs) or \
                lib.qknr_gn_sizeof_args() != ctypes.sizeof(QknrGnArgs) or \
                lib.qknr_sizeof_host_plan() != ctypes.sizeof(QknrHostPlan):
            raise RuntimeError("libqknr.so struct layout differs from the binding")
        if path is None:
            _lib = lib
        return lib


def last_error() -> str:
    return load().qknr_last_error().decode()


# ---------------------------------------------------------------------------
# marshalling helpers

_ACT = {torch.bfloat16: BF16, torch.float16: FP16}
_TAB = {torch.float32: FP32, torch.bfloat16: BF16}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _rows(t: Optional[torch.Tensor], name: str) -> int:
    """Row stride (elements) of a 2-D activation view with unit inner stride."""
    if t is None:
        return 0
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D [tokens, heads*head_dim]")
    if t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.stride(0)


_status_bufs = {}


def status_buffer(device=None) -> torch.Tensor:
    """The per-device int32 status word the binding passes by default."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    buf = _status_bufs.get(dev.index)
    if buf is None:
        buf = torch.zeros(1, dtype=torch.int32, device=dev)
        _status_bufs[dev.index] = buf
    return buf


def read_status(device=None, reset: bool = True) -> int:
    """Synchronise and return the kernel-side status word (0 = no timeout)."""
    buf = status_buffer(device)
    v = int(buf.item())
    if reset and v:
        buf.zero_()
    return v


def make_args(
    *,
    q: Optional[torch.Tensor] = None,
    k: Optional[torch.Tensor] = None,
    v: Optional[torch.Tensor] = None,
    q_out: Optional[torch.Tensor] = None,
    k_out: Optional[torch.Tensor] = None,
    v_out: Optional[torch.Tensor] = None,
    n_heads_q: int = 0,
    n_heads_k: int = 0,
    n_heads_v: int = 0,
    head_dim: int,
    gamma_q: Optional[torch.Tensor] = None,
    gamma_k: Optional[torch.Tensor] = None,
    cos: Optional[torch.Tensor] = None,
    sin: Optional[torch.Tensor] = None,
    rope_style: str = "interleaved",
    cos_layout: str = "shared_row",
    cos_rows: Optional[int] = None,
    eps: float = 1e-6,
    tokens: Optional[int] = None,
    dev_status: Optional[torch.Tensor] = None,
    ctas_per_sm: int = 0,
    stages: int = 0,
    consumer_warps: int = 0,
    group_warps: int = 0,
    flags: int = 0,
    wait_limit_ns: int = 0,
) -> QknrArgs:
    """Build a ``QknrArgs`` from tensors (no checks beyond marshalling; the
    library validates)."""
    a = QknrArgs()
    load().qknr_args_init(ctypes.byref(a))
    acts = [t for t in (q, k, v) if t is not None]
    if acts:
        dt = acts[0].dtype
        if dt not in _ACT or any(t.dtype != dt for t in acts):
            raise ValueError("q, k, v must share one dtype: bfloat16 or float16")
        a.dtype = _ACT[dt]
    for out, inp, name in ((q_out, q, "q_out"), (k_out, k, "k_out"), (v_out, v, "v_out")):
        if out is not None and inp is not None and out.dtype != inp.dtype:
            raise ValueError(f"{name} dtype differs from its input")
    a.q, a.k, a.v = _ptr(q), _ptr(k), _ptr(v)
    a.q_out, a.k_out, a.v_out = _ptr(q_out), _ptr(k_out), _ptr(v_out)
    a.q_stride, a.k_stride, a.v_stride = _rows(q, "q"), _rows(k, "k"), _rows(v, "v")
    a.q_out_stride = _rows(q_out, "q_out")
    a.k_out_stride = _rows(k_out, "k_out")
    a.v_out_stride = _rows(v_out, "v_out")
    if tokens is None:
        tokens = acts[0].shape[0] if acts else 0
    a.tokens = tokens
    a.n_heads_q, a.n_heads_k, a.n_heads_v, a.head_dim = n_heads_q, n_heads_k, n_heads_v, head_dim
    for g, name in ((gamma_q, "gamma_q"), (gamma_k, "gamma_k")):
        if g is not None and (g.dtype != torch.float32 or not g.is_cuda or not g.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    a.gamma_q, a.gamma_k = _ptr(gamma_q), _ptr(gamma_k)
    a.eps = eps
    if cos is not None:
        if cos.dtype not in _TAB or sin is None or sin.dtype != cos.dtype:
            raise ValueError("cos and sin must both be float32 or both bfloat16")
        if not (cos.is_contiguous() and sin.is_contiguous() and cos.is_cuda and sin.is_cuda):
            raise ValueError("cos and sin must be contiguous CUDA tensors")
        if cos.shape != sin.shape:
            raise ValueError("cos and sin shapes differ")
        a.cos_dtype = _TAB[cos.dtype]
        if cos_rows is None:
            cos_rows = cos.shape[0]
    a.cos, a.sin = _ptr(cos), _ptr(sin)
    a.cos_layout = COS_LAYOUT[cos_layout]
    a.cos_rows = cos_rows or 0
    a.rope_style = ROPE[rope_style]
    a.dev_status = _ptr(dev_status)
    a.ctas_per_sm, a.stages, a.consumer_warps, a.group_warps = ctas_per_sm, stages, consumer_warps, group_warps
    a.flags, a.wait_limit_ns = flags, wait_limit_ns
    return a


def launch(a: QknrArgs, stream: Optional[torch.cuda.Stream] = None) -> None:
    """qknr_forward on ``stream`` (default: the current stream)."""
    lib = load()
    s = torch.cuda.current_stream() if stream is None else stream
    st = lib.qknr_forward(ctypes.byref(a), c_void_p(s.cuda_stream))
    if st != OK:
        raise QknrError(st, lib.qknr_last_error().decode())


def query(a: QknrArgs) -> dict:
    """qknr_query: the launch qknr_forward would make, as a dict."""
    lib = load()
    info = QknrLaunchInfo()
    st = lib.qknr_query(ctypes.byref(a), ctypes.byref(info))
    if st != OK:
        raise QknrError(st, lib.qknr_last_error().decode())
    return info.as_dict()


# ---------------------------------------------------------------------------
# convenience forms

def _check_table(cos, head_dim, cos_layout, heads):
    if cos_layout == "shared_row":
        if cos.dim() != 2 or cos.shape[1] != head_dim:
            raise ValueError("shared cos/sin must be [rows, head_dim]")
    else:
        if cos.dim() != 3 or cos.shape[1] != heads or cos.shape[2] != head_dim:
            raise ValueError("expanded cos/sin must be [rows, heads, head_dim]")


def packed_args(qkv, n_heads_q, n_heads_k, n_heads_v, head_dim, gamma_q, gamma_k, cos, sin, *,
                out=None, **kw) -> QknrArgs:
    """Arguments for a packed [T, (Hq+Hk+Hv)*D] activation.  ``out=None``
    normalises Q and K in place and leaves V alone; otherwise ``out`` (same
    shape) receives Q, K and a copy of V."""
    D = head_dim
    width = (n_heads_q + n_heads_k + n_heads_v) * D
    if qkv.dim() != 2 or qkv.shape[1] != width:
        raise ValueError(f"qkv must be [tokens, {width}]")
    _check_table(cos, D, kw.get("cos_layout", "shared_row"), n_heads_q)
    q0, k0, v0, v1 = 0, n_heads_q * D, (n_heads_q + n_heads_k) * D, width
    views = dict(q=qkv[:, q0:k0] if n_heads_q else None,
                 k=qkv[:, k0:v0] if n_heads_k else None,
                 v=qkv[:, v0:v1] if n_heads_v else None)
    if out is not None:
        if out.shape != qkv.shape or out.dtype != qkv.dtype:
            raise ValueError("out must match qkv's shape and dtype")
        views.update(q_out=out[:, q0:k0] if n_heads_q else None,
                     k_out=out[:, k0:v0] if n_heads_k else None,
                     v_out=out[:, v0:v1] if n_heads_v else None)
    return make_args(**views, n_heads_q=n_heads_q, n_heads_k=n_heads_k, n_heads_v=n_heads_v,
                     head_dim=D, gamma_q=gamma_q if n_heads_q else None,
                     gamma_k=gamma_k if n_heads_k else None, cos=cos, sin=sin,
                     tokens=qkv.shape[0], **kw)


def qk_norm_rope_packed(qkv, n_heads_q, n_heads_k, n_heads_v, head_dim, gamma_q, gamma_k, cos, sin, *,
                        out=None, stream=None, status=True, **kw):
    """Fused QK-RMSNorm + RoPE on a packed QKV activation; returns the
    tensor holding the result (``qkv`` itself when in place)."""
    if status and "dev_status" not in kw:
        kw["dev_status"] = status_buffer(qkv.device)
    launch(packed_args(qkv, n_heads_q, n_heads_k, n_heads_v, head_dim, gamma_q, gamma_k, cos, sin,
                       out=out, **kw), stream)
    return qkv if out is None else out


def qk_norm_rope_tensor(x, n_heads, head_dim, gamma, cos, sin, *, out=None, stream=None, status=True,
                        **kw):
    """Per-tensor launch (one separate Q or K tensor [T, H*D]), the form
    of page 2's FLUX.2 integration.  In place unless ``out`` is given."""
    if x.dim() != 2 or x.shape[1] != n_heads * head_dim:
        raise ValueError("x must be [tokens, n_heads*head_dim]")
    _check_table(cos, head_dim, kw.get("cos_layout", "shared_row"), n_heads)
    if status and "dev_status" not in kw:
        kw["dev_status"] = status_buffer(x.device)
    launch(make_args(q=x, q_out=out, n_heads_q=n_heads, head_dim=head_dim, gamma_q=gamma, cos=cos, sin=sin,
                     **kw), stream)
    return x if out is None else out


def qk_norm_rope_separate(q, k, n_heads, head_dim, gamma_q, gamma_k, cos, sin, *, v=None, q_out=None,
                          k_out=None, v_out=None, n_heads_v=None, stream=None, status=True, **kw):
    """Q and K as separate [T, H*D] tensors in one launch (and V copied into
    ``v_out`` when both are given)."""
    _check_table(cos, head_dim, kw.get("cos_layout", "shared_row"), n_heads)
    if status and "dev_status" not in kw:
        kw["dev_status"] = status_buffer(q.device)
    hv = (n_heads if n_heads_v is None else n_heads_v) if (v is not None and v_out is not None) else 0
    launch(make_args(q=q, k=k, v=v if hv else None, q_out=q_out, k_out=k_out, v_out=v_out if hv else None,
                     n_heads_q=n_heads, n_heads_k=n_heads, n_heads_v=hv, head_dim=head_dim,
                     gamma_q=gamma_q, gamma_k=gamma_k, cos=cos, sin=sin, **kw), stream)


# ---------------------------------------------------------------------------
# host-resident activations: qknr_forward_host (include/qknr.h)

_cudart = None


def _cudart_lib() -> ctypes.CDLL:
    """The CUDA runtime libqknr.so links (already loaded with it), for the
    events the host pipeline hands the library."""
    global _cudart
    if _cudart is None:
        load()
        cands = sorted(glob.glob(os.path.join(_build.cuda_lib_dir(), "libcudart.so*")))
        if not cands:
            raise RuntimeError("libcudart.so not found next to the CUDA toolkit")
        lib = ctypes.CDLL(cands[-1])
        lib.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(c_void_p), c_uint32]
        lib.cudaEventCreateWithFlags.restype = c_int32
        lib.cudaEventDestroy.argtypes = [c_void_p]
        lib.cudaEventDestroy.restype = c_int32
        _cudart = lib
    return _cudart


def host_args(*, q=None, k=None, v=None, q_out=None, k_out=None, v_out=None, n_heads_q=0, n_heads_k=0,
              n_heads_v=0, head_dim, tokens, gamma_q=None, gamma_k=None, cos=None, sin=None, cos_rows=0,
              rope_style="interleaved", cos_layout="shared_row", eps=1e-6, dtype=torch.bfloat16, cos_dtype=FP32,
              dev_status=None, ctas_per_sm=0, stages=0, consumer_warps=0, group_warps=0, flags=0,
              wait_limit_ns=0) -> QknrArgs:
    """``qknr_args`` for qknr_forward_host: q, k, v and the outputs are host
    tensor views ([T, heads*D] rows with unit inner stride) or None; gamma,
    cos and sin are device tensors."""
    a = QknrArgs()
    load().qknr_args_init(ctypes.byref(a))
    a.dtype = _ACT[dtype]
    for name, t in (("q", q), ("k", k), ("v", v), ("q_out", q_out), ("k_out", k_out), ("v_out", v_out)):
        if t is None:
            continue
        if t.is_cuda or t.dim() != 2 or t.stride(1) != 1 or t.dtype != dtype:
            raise ValueError(f"{name} must be a 2-D host tensor of {dtype} with contiguous rows")
        setattr(a, name, t.data_ptr())
        setattr(a, name + "_stride", t.stride(0))
    a.tokens = tokens
    a.n_heads_q, a.n_heads_k, a.n_heads_v, a.head_dim = n_heads_q, n_heads_k, n_heads_v, head_dim
    a.gamma_q, a.gamma_k = _ptr(gamma_q), _ptr(gamma_k)
    a.eps = eps
    a.cos, a.sin = _ptr(cos), _ptr(sin)
    a.cos_dtype = cos_dtype
    a.cos_layout = COS_LAYOUT[cos_layout]
    a.cos_rows = cos_rows
    a.rope_style = ROPE[rope_style]
    a.dev_status = _ptr(dev_status)
    a.ctas_per_sm, a.stages, a.consumer_warps, a.group_warps = ctas_per_sm, stages, consumer_warps, group_warps
    a.flags, a.wait_limit_ns = flags, wait_limit_ns
    return a


class HostPipeline:
    """The fused QK-RMSNorm + RoPE on a packed QKV activation that lives in
    (pinned) host memory, through qknr_forward_host: token rows go through
    device staging buffers in chunks, with the host-to-device copy of one
    chunk, the kernel on the previous one and the device-to-host copy of the
    one before that on three streams.  All of that runs inside the library;
    this class only owns what the library does not allocate (the staging
    buffers and the device copies of the gains and tables, made by torch;
    two copy streams; the events) and marshals the call.

    In place on the host (``out_host`` None or the input) only the Q and K
    columns of each row cross the host link: V is neither read nor written
    by the operation, so it stays where it is.  With a separate ``out_host``
    the Q, K and V columns go both ways and V is copied through unchanged.
    The gains and tables are copied from the host to the device every call.
    Results are bitwise those of ``qk_norm_rope_packed`` on the whole
    activation.
    """

    def __init__(self, width: int, dtype: torch.dtype, chunk_rows: int = 2048, n_buffers: int = 3,
                 device=None):
        lib = load()
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index)
        if not 1 <= n_buffers <= 4:
            raise ValueError("n_buffers must be 1..4")
        self.chunk_rows = int(chunk_rows)
        self.width = int(width)
        self.dtype = dtype
        self.bufs = [torch.empty(self.chunk_rows * self.width, dtype=dtype, device=self.device)
                     for _ in range(n_buffers)]
        self.h2d = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.tables = {}
        rt = _cudart_lib()
        self.events = []
        with torch.cuda.device(self.device):
            for _ in range(3 * n_buffers + 2):
                e = c_void_p()
                err = rt.cudaEventCreateWithFlags(ctypes.byref(e), 2)   # cudaEventDisableTiming
                if err != 0:
                    raise RuntimeError(f"cudaEventCreateWithFlags failed with error {err}")
                self.events.append(e.value)
        self.plan = QknrHostPlan()
        lib.qknr_host_plan_init(ctypes.byref(self.plan))
        self.plan.n_buffers = n_buffers
        self.plan.chunk_rows = self.chunk_rows
        for i, b in enumerate(self.bufs):
            self.plan.dev_buffers[i] = b.data_ptr()
        self.plan.h2d_stream = self.h2d.cuda_stream
        self.plan.d2h_stream = self.d2h.cuda_stream
        for i, e in enumerate(self.events):
            self.plan.events[i] = e
        self.last_h2d_bytes = self.last_d2h_bytes = 0

    def __del__(self):
        rt = _cudart
        if rt is not None:
            for e in getattr(self, "events", []):
                rt.cudaEventDestroy(c_void_p(e))

    def _device_table(self, name, t):
        """The device buffer the host table ``t`` is copied into (kept across calls)."""
        d = self.tables.get(name)
        if d is None or d.shape != t.shape or d.dtype != t.dtype:
            d = torch.empty(t.shape, dtype=t.dtype, device=self.device)
            self.tables[name] = d
        return d

    def read_status(self) -> int:
        """Synchronise and return (then clear) the kernels' status word."""
        v = int(self.status.item())
        if v:
            self.status.zero_()
        return v

    def __call__(self, qkv_host, n_heads_q, n_heads_k, n_heads_v, head_dim, gamma_q, gamma_k, cos, sin, *,
                 out_host=None, rope_style="interleaved", cos_layout="shared_row", eps=1e-6, **tune):
        if qkv_host.is_cuda or qkv_host.dim() != 2 or qkv_host.shape[1] != self.width or qkv_host.stride(1) != 1:
            raise ValueError("qkv_host must be a 2-D host tensor of the pipeline's width with contiguous rows")
        if qkv_host.dtype != self.dtype:
            raise ValueError("qkv_host dtype differs from the pipeline's")
        if (n_heads_q + n_heads_k + n_heads_v) * head_dim != self.width:
            raise ValueError("head counts do not match the pipeline's width")
        in_place = out_host is None or out_host.data_ptr() == qkv_host.data_ptr()
        if out_host is not None and (out_host.shape != qkv_host.shape or out_host.dtype != qkv_host.dtype or
                                     out_host.stride(1) != 1):
            raise ValueError("out_host must match qkv_host")
        T, D = qkv_host.shape[0], head_dim
        q0, k0, v0 = 0, n_heads_q * D, (n_heads_q + n_heads_k) * D

        def cols(t, a, b):
            return None if t is None or a == b else t[:, a:b]

        dev = {n: self._device_table(n, t) for n, t in (("gamma_q", gamma_q), ("gamma_k", gamma_k), ("cos", cos),
                                                       ("sin", sin))}
        cos_dtype = _TAB[cos.dtype]
        a = host_args(q=cols(qkv_host, q0, k0), k=cols(qkv_host, k0, v0), v=cols(qkv_host, v0, self.width),
                      q_out=None if in_place else cols(out_host, q0, k0),
                      k_out=None if in_place else cols(out_host, k0, v0),
                      v_out=None if in_place else cols(out_host, v0, self.width),
                      n_heads_q=n_heads_q, n_heads_k=n_heads_k, n_heads_v=n_heads_v, head_dim=D, tokens=T,
                      gamma_q=dev["gamma_q"], gamma_k=dev["gamma_k"], cos=dev["cos"], sin=dev["sin"],
                      cos_rows=cos.shape[0], rope_style=rope_style, cos_layout=cos_layout, eps=eps,
                      dtype=qkv_host.dtype, cos_dtype=cos_dtype, dev_status=self.status, **tune)
        self.plan.host_gamma_q, self.plan.host_gamma_k = gamma_q.data_ptr(), gamma_k.data_ptr()
        self.plan.host_cos, self.plan.host_sin = cos.data_ptr(), sin.data_ptr()
        lib = load()
        stream = torch.cuda.current_stream(self.device)
        st = lib.qknr_forward_host(ctypes.byref(a), ctypes.byref(self.plan), c_void_p(stream.cuda_stream))
        if st != OK:
            raise QknrError(st, lib.qknr_last_error().decode())
        # the host tables and device buffers are in use until the stream's
        # work is done
        for t in list(dev.values()) + self.bufs:
            t.record_stream(stream)
        es = qkv_host.element_size()
        moved = (n_heads_q + n_heads_k + (0 if in_place else n_heads_v)) * D * es * T
        tables = sum(t.numel() * t.element_size() for t in (gamma_q, gamma_k, cos, sin))
        self.last_h2d_bytes = moved + tables
        self.last_d2h_bytes = moved
        return qkv_host if in_place else out_host


# ---------------------------------------------------------------------------
# AdaLN scale/shift (include/qknr_adaln.h)

def adaln_args(x, scale, shift, *, rows_per_batch=None, out=None, eps=1e-6, dev_status=None, ctas_per_sm=0,
               stages=0, consumer_warps=0, group_warps=0, flags=0, wait_limit_ns=0) -> QknrAdaLNArgs:
    """Arguments for ``out = LN(x) * (1 + scale[b]) + shift[b]`` over token
    rows ``x`` [T, C]; ``scale``/``shift`` are [B, C] (fp32 or x's dtype);
    row t belongs to sample t // rows_per_batch (default: one sample)."""
    a = QknrAdaLNArgs()
    load().qknr_adaln_args_init(ctypes.byref(a))
    if x.dtype not in _ACT:
        raise ValueError("x must be bfloat16 or float16")
    a.dtype = _ACT[x.dtype]
    a.x, a.x_stride = x.data_ptr(), _rows(x, "x")
    if out is not None:
        if out.dtype != x.dtype or out.shape != x.shape:
            raise ValueError("out must match x's shape and dtype")
        a.out, a.out_stride = out.data_ptr(), _rows(out, "out")
    a.tokens, a.hidden = x.shape[0], x.shape[1]
    a.rows_per_batch = rows_per_batch or 0
    for m, name in ((scale, "scale"), (shift, "shift")):
        if m.dim() != 2 or m.shape[1] != x.shape[1] or m.dtype != scale.dtype:
            raise ValueError(f"{name} must be [B, C] like scale")
    if scale.dtype == torch.float32:
        a.mod_dtype = FP32
    elif scale.dtype == x.dtype:
        a.mod_dtype = a.dtype
    else:
        raise ValueError("scale/shift must be float32 or x's dtype")
    a.scale, a.shift = scale.data_ptr(), shift.data_ptr()
    if _rows(scale, "scale") != _rows(shift, "shift"):
        raise ValueError("scale and shift need the same row stride")
    a.mod_stride = _rows(scale, "scale")
    a.eps = eps
    a.dev_status = _ptr(dev_status)
    a.ctas_per_sm, a.stages, a.consumer_warps, a.group_warps = ctas_per_sm, stages, consumer_warps, group_warps
    a.flags, a.wait_limit_ns = flags, wait_limit_ns
    return a


def adaln_launch(a: QknrAdaLNArgs, stream: Optional[torch.cuda.Stream] = None) -> None:
    lib = load()
    s = torch.cuda.current_stream() if stream is None else stream
    st = lib.qknr_adaln_forward(ctypes.byref(a), c_void_p(s.cuda_stream))
    if st != OK:
        raise QknrError(st, lib.qknr_last_error().decode())


def adaln_query(a: QknrAdaLNArgs) -> dict:
    lib = load()
    info = QknrLaunchInfo()
    st = lib.qknr_adaln_query(ctypes.byref(a), ctypes.byref(info))
    if st != OK:
        raise QknrError(st, lib.qknr_last_error().decode())
    return info.as_dict()


def adaln_modulate(x, scale, shift, *, rows_per_batch=None, out=None, stream=None, status=True, **kw):
    """AdaLN scale/shift on token rows ``x``; in place unless ``out`` is given."""
    if status and "dev_status" not in kw:
        kw["dev_status"] = status_buffer(x.device)
    adaln_launch(adaln_args(x, scale, shift, rows_per_batch=rows_per_batch, out=out, **kw), stream)
    return x if out is None else out


# ---------------------------------------------------------------------------
# group norm + SiLU (include/qknr_gn.h)

def gn_args(x, groups, gamma, beta, *, out=None, eps=1e-6, workspace=None, piece_elems=0,
            l2_batch_bytes=0, mode="auto", dev_status=None, flags=0, wait_limit_ns=0) -> QknrGnArgs:
    """Arguments for ``silu(group_norm(x))`` on an NCHW tensor ``x``."""
    if x.dim() != 4 or not x.is_contiguous() or not x.is_cuda or x.dtype not in _ACT:
        raise ValueError("x must be a contiguous 4-D (NCHW) bfloat16/float16 CUDA tensor")
    a = QknrGnArgs()
    load().qknr_gn_args_init(ctypes.byref(a))
    a.dtype = _ACT[x.dtype]
    a.x = x.data_ptr()
    if out is not None:
        if out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
            raise ValueError("out must be contiguous and match x")
        a.out = out.data_ptr()
    a.n, a.c, a.h, a.w = x.shape
    a.groups = groups
    for t, name in ((gamma, "gamma"), (beta, "beta")):
        if t.dtype != torch.float32 or not t.is_cuda or t.numel() != x.shape[1] or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of C values")
    a.gamma, a.beta = gamma.data_ptr(), beta.data_ptr()
    a.eps = eps
    a.piece_elems, a.l2_batch_bytes = piece_elems, l2_batch_bytes
    a.mode = GN_MODE[mode]
    a.dev_status = _ptr(dev_status)
    a.flags, a.wait_limit_ns = flags, wait_limit_ns
    if workspace is not None:
        a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    return a


def gn_query(a: QknrGnArgs) -> dict:
    """qknr_gn_query: the path and launch qknr_gn_silu_forward would take."""
    lib = load()
    info = QknrLaunchInfo()
    st = lib.qknr_gn_query(ctypes.byref(a), ctypes.byref(info))
    if st != OK:
        raise QknrError(st, lib.qknr_last_error().decode())
    return info.as_dict()


def gn_workspace_bytes(a: QknrGnArgs) -> int:
    lib = load()
    n = c_size_t(0)
    st = lib.qknr_gn_workspace_bytes(ctypes.byref(a), ctypes.byref(n))
    if st != OK:
        raise QknrError(st, lib.qknr_last_error().decode())
    return n.value


def gn_launch(a: QknrGnArgs, stream: Optional[torch.cuda.Stream] = None) -> None:
    lib = load()
    s = torch.cuda.current_stream() if stream is None else stream
    st = lib.qknr_gn_silu_forward(ctypes.byref(a), c_void_p(s.cuda_stream))
    if st != OK:
        raise QknrError(st, lib.qknr_last_error().decode())


def group_norm_silu(x, groups, gamma, beta, *, out=None, workspace=None, stream=None, status=True, **kw):
    """silu(group_norm(x)) on NCHW ``x``; in place unless ``out`` is given.
    ``workspace`` (a CUDA tensor of at least gn_workspace_bytes) is created
    by this binding when not given."""
    if status and "dev_status" not in kw:
        kw["dev_status"] = status_buffer(x.device)
    a = gn_args(x, groups, gamma, beta, out=out, **kw)
    if workspace is None:
        workspace = torch.empty(gn_workspace_bytes(a), dtype=torch.uint8, device=x.device)
    a.workspace, a.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    gn_launch(a, stream)
    return x if out is None else out


def gn_launch_noalloc(a: QknrGnArgs, stream: Optional[torch.cuda.Stream] = None) -> None:
    """qknr_gn_silu_forward_noalloc: the group-norm + SiLU call for callers
    that cannot allocate device memory; its statistics scratch is a fixed
    array inside the library (GN_NOALLOC_SCRATCH_BYTES), shared by every
    call on the device, and a.workspace is ignored."""
    lib = load()
    s = torch.cuda.current_stream() if stream is None else stream
    st = lib.qknr_gn_silu_forward_noalloc(ctypes.byref(a), c_void_p(s.cuda_stream))
    if st != OK:
        raise QknrError(st, lib.qknr_last_error().decode())
