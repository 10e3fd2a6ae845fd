"""qknr_forward_host from a C caller that holds its activation in host
memory: a C99 program (CUDA runtime only, no Python in the path) reads a
packed QKV activation and the tables from files, makes its staging buffers,
streams and events, runs the call in place and out of place, and writes the
results back; they must be bitwise those of qknr_forward on a device copy of
the whole activation, with V unchanged (in place) or copied (out of place)."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from diffusion_transformer_qk_gb300 import build as B
from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from tests.gpu_util import table_to_dev, to_bits, to_dev

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "qknr.h"

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
  fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 2; } } while (0)
#define QK(x) do { qknr_status s_ = (x); if (s_ != QKNR_OK) { \
  fprintf(stderr, "%s: %s (%s)\n", #x, qknr_status_string(s_), qknr_last_error()); return 3; } } while (0)

static int read_file(const char *path, void *dst, size_t n) {
  FILE *f = fopen(path, "rb");
  if (!f || fread(dst, 1, n, f) != n) { fprintf(stderr, "read %s\n", path); return 1; }
  fclose(f);
  return 0;
}

static int write_file(const char *path, const void *src, size_t n) {
  FILE *f = fopen(path, "wb");
  if (!f || fwrite(src, 1, n, f) != n) { fprintf(stderr, "write %s\n", path); return 1; }
  fclose(f);
  return 0;
}

int main(int argc, char **argv) {
  /* argv: dir T H D cos_rows chunk_rows n_buffers */
  char path[1024];
  const char *dir = argv[1];
  const long long T = atoll(argv[2]), cos_rows = atoll(argv[5]), chunk = atoll(argv[6]);
  const int H = atoi(argv[3]), D = atoi(argv[4]), nb = atoi(argv[7]);
  const size_t row = (size_t)3 * H * D, qkv_bytes = (size_t)T * row * 2;
  const size_t tab_bytes = (size_t)cos_rows * D * 4;
  unsigned short *qkv, *out;
  float *gq, *gk, *cs, *sn;
  void *d_gq, *d_gk, *d_cos, *d_sin, *bufs[QKNR_HOST_MAX_BUFFERS] = {0};
  int *d_status, status = 0, i;
  cudaStream_t stream, h2d, d2h;
  qknr_args a;
  qknr_host_plan plan;
  size_t need = 0;

  (void)argc;
  CK(cudaMallocHost((void **)&qkv, qkv_bytes));
  CK(cudaMallocHost((void **)&out, qkv_bytes));
  CK(cudaMallocHost((void **)&gq, D * 4));
  CK(cudaMallocHost((void **)&gk, D * 4));
  CK(cudaMallocHost((void **)&cs, tab_bytes));
  CK(cudaMallocHost((void **)&sn, tab_bytes));
  snprintf(path, sizeof path, "%s/qkv.bin", dir); if (read_file(path, qkv, qkv_bytes)) return 1;
  snprintf(path, sizeof path, "%s/gq.bin", dir); if (read_file(path, gq, D * 4)) return 1;
  snprintf(path, sizeof path, "%s/gk.bin", dir); if (read_file(path, gk, D * 4)) return 1;
  snprintf(path, sizeof path, "%s/cos.bin", dir); if (read_file(path, cs, tab_bytes)) return 1;
  snprintf(path, sizeof path, "%s/sin.bin", dir); if (read_file(path, sn, tab_bytes)) return 1;
  CK(cudaMalloc(&d_gq, D * 4));
  CK(cudaMalloc(&d_gk, D * 4));
  CK(cudaMalloc(&d_cos, tab_bytes));
  CK(cudaMalloc(&d_sin, tab_bytes));
  CK(cudaMalloc((void **)&d_status, 4));
  CK(cudaMemset(d_status, 0, 4));
  CK(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
  CK(cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking));
  CK(cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking));

  /* in place on the host activation: Q and K columns only */
  qknr_args_init(&a);
  a.dtype = QKNR_BF16;
  a.q = qkv;
  a.k = qkv + (size_t)H * D;
  a.v = qkv + (size_t)2 * H * D;
  a.q_stride = a.k_stride = a.v_stride = (int64_t)row;
  a.tokens = T;
  a.n_heads_q = a.n_heads_k = a.n_heads_v = H;
  a.head_dim = D;
  a.gamma_q = (const float *)d_gq;
  a.gamma_k = (const float *)d_gk;
  a.cos = d_cos;
  a.sin = d_sin;
  a.cos_rows = cos_rows;
  a.rope_style = QKNR_ROPE_ROTATE_HALF;
  a.dev_status = d_status;
  qknr_host_plan_init(&plan);
  plan.n_buffers = nb;
  plan.chunk_rows = chunk;
  plan.h2d_stream = (qknr_stream_t)h2d;
  plan.d2h_stream = (qknr_stream_t)d2h;
  plan.host_gamma_q = gq;
  plan.host_gamma_k = gk;
  plan.host_cos = cs;
  plan.host_sin = sn;
  /* room for the out-of-place call below too (V columns carried) */
  a.v_out = out;
  QK(qknr_host_buffer_bytes(&a, &plan, &need));
  a.v_out = NULL;
  for (i = 0; i < nb; ++i) CK(cudaMalloc(&bufs[i], need));
  for (i = 0; i < nb; ++i) plan.dev_buffers[i] = bufs[i];
  for (i = 0; i < QKNR_HOST_EVENTS(nb); ++i) {
    cudaEvent_t e;
    CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    plan.events[i] = (qknr_event_t)e;
  }
  /* out of place first (input kept), then in place twice in a row: the
     second in-place call normalises the first one's output */
  a.q_out = out;
  a.k_out = out + (size_t)H * D;
  a.v_out = out + (size_t)2 * H * D;
  QK(qknr_forward_host(&a, &plan, (qknr_stream_t)stream));
  CK(cudaStreamSynchronize(stream));
  snprintf(path, sizeof path, "%s/out_of_place.bin", dir); if (write_file(path, out, qkv_bytes)) return 1;
  a.q_out = a.k_out = a.v_out = NULL;
  QK(qknr_forward_host(&a, &plan, (qknr_stream_t)stream));
  CK(cudaStreamSynchronize(stream));
  snprintf(path, sizeof path, "%s/in_place.bin", dir); if (write_file(path, qkv, qkv_bytes)) return 1;
  QK(qknr_forward_host(&a, &plan, (qknr_stream_t)stream));
  CK(cudaStreamSynchronize(stream));
  snprintf(path, sizeof path, "%s/in_place_twice.bin", dir); if (write_file(path, qkv, qkv_bytes)) return 1;
  CK(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));
  printf("ok %d\n", status);
  return status != 0;
}
"""


@pytest.fixture(scope="module")
def program(tmp_path_factory, built_lib, cuda_device):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    d = tmp_path_factory.mktemp("hostc")
    src, exe = d / "host.c", d / "host"
    src.write_text(PROGRAM)
    libdir, cudalib = os.path.dirname(built_lib), B.cuda_lib_dir()
    cudainc = os.path.join(os.path.dirname(cudalib), "include")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I" + os.path.join(ROOT, "include"),
                        "-I" + cudainc, str(src), "-o", str(exe), "-L" + libdir, "-L" + cudalib, "-lqknr",
                        "-lcudart", "-Wl,-rpath," + libdir, "-Wl,-rpath," + cudalib],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def device_reference(w, inp, times=1):
    """qknr_forward on a device copy of the whole activation, `times` in a row."""
    qkv = to_dev(inp["qkv"], w.dtype)
    gq, gk = torch.from_numpy(inp["gamma_q"]).cuda(), torch.from_numpy(inp["gamma_k"]).cuda()
    cos, sin = table_to_dev(inp["cos"], "fp32"), table_to_dev(inp["sin"], "fp32")
    outs = []
    for _ in range(times):
        Q.qk_norm_rope_packed(qkv, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim, gq, gk, cos, sin,
                              rope_style=w.rope_style, eps=w.eps)
        outs.append(to_bits(qkv))
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("T,seq,chunk,nb", [(9000, 9000, 2048, 3), (6000, 1500, 3000, 2), (777, 777, 256, 1),
                                            (3000, 3000, 4096, 4)])
def test_c_program_host_call_matches_the_device_path(program, tmp_path, T, seq, chunk, nb):
    H, D = 8, 128
    w = I.WORKLOADS["dense_4096x24x128"].with_(seq=seq, batch=T // seq, n_heads_q=H, n_heads_k=H, n_heads_v=H)
    inp = I.make_inputs(w)
    assert inp["qkv"].shape == (T, 3 * H * D) and inp["cos"].shape[0] == seq
    for name, arr in (("qkv", inp["qkv"]), ("gq", inp["gamma_q"]), ("gk", inp["gamma_k"]), ("cos", inp["cos"]),
                      ("sin", inp["sin"])):
        np.ascontiguousarray(arr).tofile(tmp_path / f"{name}.bin")
    r = subprocess.run([str(program), str(tmp_path), str(T), str(H), str(D), str(seq), str(chunk), str(nb)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.stdout, r.stderr)
    assert r.stdout.strip() == "ok 0"
    once, twice = device_reference(w, inp, times=2)

    def load(name):
        return np.fromfile(tmp_path / name, dtype=np.uint16).reshape(T, 3 * H * D)

    oop, ip, ip2 = load("out_of_place.bin"), load("in_place.bin"), load("in_place_twice.bin")
    np.testing.assert_array_equal(oop, once)                          # V copied through unchanged
    np.testing.assert_array_equal(ip, once)                           # V never left the host
    np.testing.assert_array_equal(ip2, twice)
    np.testing.assert_array_equal(ip[:, 2 * H * D:], inp["qkv"][:, 2 * H * D:])


# ---------------------------------------------------------------------------
# qknr_forward_host through the binding: per-head expanded tables, separate
# host tensors, fp16

def _pinned_bits(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.pin_memory()


@pytest.mark.parametrize("dtype,cos_dtype", [("bf16", "fp32"), ("fp16", "bf16")])
def test_host_pipeline_with_expanded_tables_that_differ_per_head(built_lib, cuda_device, dtype, cos_dtype):
    H, D, T, chunk = 8, 128, 9000, 1024           # T >= 4 chunks: the chunk sizes ramp up and down
    w = I.WORKLOADS["wan_32760x40x128"].with_(n_heads_q=H, n_heads_k=H, n_heads_v=H, dtype=dtype, seq=T,
                                              positions="1d", grid=(), axes_dim=(D,), rope_style="rotate_half",
                                              cos_dtype=cos_dtype, cos_layout="per_head_expanded")
    inp = I.make_inputs(w)
    ce, se = I.per_head_tables(T, H, D, "rotate_half", cos_dtype, seed=71)
    dev_tab = (lambda t: table_to_dev(t, cos_dtype))
    ref = to_dev(inp["qkv"], dtype)
    Q.qk_norm_rope_packed(ref, H, H, H, D, torch.from_numpy(inp["gamma_q"]).cuda(),
                          torch.from_numpy(inp["gamma_k"]).cuda(), dev_tab(ce), dev_tab(se), rope_style="rotate_half",
                          cos_layout="per_head_expanded", eps=w.eps)
    host = _pinned_bits(inp["qkv"], dtype)
    host_tab = (lambda t: torch.from_numpy(t).pin_memory() if cos_dtype == "fp32" else _pinned_bits(t, "bf16"))
    pipe = Q.HostPipeline(host.shape[1], host.dtype, chunk_rows=chunk)
    pipe(host, H, H, H, D, torch.from_numpy(inp["gamma_q"]).pin_memory(), torch.from_numpy(inp["gamma_k"]).pin_memory(),
         host_tab(ce), host_tab(se), rope_style="rotate_half", cos_layout="per_head_expanded", eps=w.eps)
    torch.cuda.synchronize()
    assert pipe.read_status() == 0
    np.testing.assert_array_equal(host.view(torch.int16).numpy().view(np.uint16), to_bits(ref))


def test_host_call_on_separate_host_tensors_with_a_v_copy(built_lib, cuda_device):
    # FLUX.2-style separate Q, K, V in host memory, written to separate host
    # outputs with V copied through, in one qknr_forward_host call
    H, D, S, B = 16, 128, 1000, 3                 # a batch-broadcast table: chunks are whole samples
    T = B * S
    w = I.WORKLOADS["flux2_2x4608x48x128"].with_(n_heads_q=H, n_heads_k=H, n_heads_v=H, seq=S, batch=B,
                                                 positions="1d", grid=(), axes_dim=(D,))
    inp = I.make_inputs(w)
    cos, sin = table_to_dev(inp["cos"], "fp32"), table_to_dev(inp["sin"], "fp32")
    gq, gk = torch.from_numpy(inp["gamma_q"]).cuda(), torch.from_numpy(inp["gamma_k"]).cuda()
    dq, dk = to_dev(inp["q"], "bf16"), to_dev(inp["k"], "bf16")
    Q.qk_norm_rope_separate(dq, dk, H, D, gq, gk, cos, sin, rope_style=w.rope_style)
    hq, hk, hv = (_pinned_bits(inp[n], "bf16") for n in ("q", "k", "v"))
    oq, ok, ov = (torch.empty_like(t).pin_memory() for t in (hq, hk, hv))
    pipe = Q.HostPipeline(3 * H * D, torch.bfloat16, chunk_rows=2000)      # staging rows hold Q | K | V
    a = Q.host_args(q=hq, k=hk, v=hv, q_out=oq, k_out=ok, v_out=ov, n_heads_q=H, n_heads_k=H, n_heads_v=H,
                    head_dim=D, tokens=T, gamma_q=gq, gamma_k=gk, cos=cos, sin=sin, cos_rows=S,
                    rope_style=w.rope_style, eps=w.eps, dev_status=pipe.status)
    need = ctypes.c_size_t(0)
    lib = Q.load()
    assert lib.qknr_host_buffer_bytes(ctypes.byref(a), ctypes.byref(pipe.plan), ctypes.byref(need)) == 0
    assert need.value == 2000 * 3 * H * D * 2                          # chunks of 2000 and 1000 rows
    pipe.plan.host_gamma_q = pipe.plan.host_gamma_k = pipe.plan.host_cos = pipe.plan.host_sin = None
    st = lib.qknr_forward_host(ctypes.byref(a), ctypes.byref(pipe.plan), ctypes.c_void_p(
        torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.qknr_last_error()
    torch.cuda.synchronize()
    assert pipe.read_status() == 0
    np.testing.assert_array_equal(oq.view(torch.int16).numpy().view(np.uint16), to_bits(dq))
    np.testing.assert_array_equal(ok.view(torch.int16).numpy().view(np.uint16), to_bits(dk))
    np.testing.assert_array_equal(ov.view(torch.int16).numpy().view(np.uint16), inp["v"])
    for t, n in ((hq, "q"), (hk, "k"), (hv, "v")):                         # inputs untouched
        np.testing.assert_array_equal(t.view(torch.int16).numpy().view(np.uint16), inp[n])
