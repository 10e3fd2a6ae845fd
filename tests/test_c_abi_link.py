"""The public headers are plain C99 and a C program links against
libqknr.so and uses it with no Python or C++ in between.

The program only makes calls that return during host-side validation (or
that have nothing to launch), so it runs with or without a GPU."""
import os
import shutil
import subprocess

import pytest

from diffusion_transformer_qk_gb300 import build as B
from diffusion_transformer_qk_gb300 import qknr as Q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "qknr.h"
#include "qknr_adaln.h"
#include "qknr_gn.h"

#define CHECK(cond, code) do { if (!(cond)) { fprintf(stderr, "failed: %s\n", #cond); return code; } } while (0)

int main(void) {
  qknr_args a;
  qknr_launch_info info;
  qknr_adaln_args ad;
  qknr_gn_args g;
  size_t ws = 0;

  CHECK(qknr_abi_version() == QKNR_ABI_VERSION, 10);
  CHECK(qknr_sizeof_args() == sizeof(qknr_args), 11);
  CHECK(qknr_sizeof_launch_info() == sizeof(qknr_launch_info), 12);
  CHECK(qknr_adaln_sizeof_args() == sizeof(qknr_adaln_args), 13);
  CHECK(qknr_gn_sizeof_args() == sizeof(qknr_gn_args), 14);

  qknr_args_init(&a);
  CHECK(a.abi_version == QKNR_ABI_VERSION && a.dtype == QKNR_BF16 && a.cos_dtype == QKNR_FP32, 20);
  /* head_dim 0 is unsupported: rejected before any CUDA call */
  CHECK(qknr_forward(&a, NULL) == QKNR_ERR_UNSUPPORTED, 21);
  CHECK(strlen(qknr_last_error()) > 0, 22);
  CHECK(qknr_forward(NULL, NULL) == QKNR_ERR_NULL, 23);
  CHECK(qknr_query(&a, NULL) == QKNR_ERR_NULL, 24);
  a.abi_version = QKNR_ABI_VERSION + 1;
  CHECK(qknr_forward(&a, NULL) == QKNR_ERR_ABI, 25);
  /* zero tokens: valid, nothing to launch, pointers may be NULL */
  qknr_args_init(&a);
  a.head_dim = 128;
  a.n_heads_q = a.n_heads_k = 24;
  CHECK(qknr_forward(&a, NULL) == QKNR_OK, 26);
  CHECK(qknr_query(&a, &info) == QKNR_OK && info.grid == 0 && strncmp(info.kernel, "qknr_fused<", 11) == 0, 27);
  CHECK(strcmp(qknr_status_string(QKNR_ERR_TIMEOUT), "in-kernel wait timed out") == 0, 28);
  CHECK(strcmp(qknr_status_string(99), "unknown status") == 0, 29);

  qknr_adaln_args_init(&ad);
  CHECK(ad.abi_version == QKNR_ABI_VERSION, 30);
  CHECK(qknr_adaln_forward(&ad, NULL) != QKNR_OK, 31);           /* hidden 0 */
  CHECK(qknr_adaln_query(NULL, &info) == QKNR_ERR_NULL, 32);

  qknr_gn_args_init(&g);
  g.n = 1; g.c = 64; g.h = 16; g.w = 16; g.groups = 32;
  g.mode = QKNR_GN_TWO_PASS;
  CHECK(qknr_gn_workspace_bytes(&g, &ws) == QKNR_OK && ws == 32 * 2 * 2 * sizeof(double), 40);
  g.mode = QKNR_GN_AUTO;
  CHECK(qknr_gn_workspace_bytes(&g, &ws) == QKNR_OK && ws >= 32 * 2 * 2 * sizeof(double), 44);
  g.groups = 3;                                                 /* does not divide C */
  CHECK(qknr_gn_workspace_bytes(&g, &ws) == QKNR_ERR_SHAPE, 41);
  g.groups = 32;
  CHECK(qknr_gn_silu_forward(&g, NULL) == QKNR_ERR_NULL, 42);   /* no x / gamma / beta */
  CHECK(qknr_gn_silu_forward_noalloc(&g, NULL) == QKNR_ERR_NULL, 43);
  CHECK(qknr_gn_query(&g, NULL) == QKNR_ERR_NULL, 45);
  g.mode = 7;
  CHECK(qknr_gn_workspace_bytes(&g, &ws) == QKNR_ERR_UNSUPPORTED, 46);
  {
    qknr_host_plan hp;
    qknr_args_init(&a);
    qknr_host_plan_init(&hp);
    CHECK(qknr_sizeof_host_plan() == sizeof(qknr_host_plan), 50);
    CHECK(hp.abi_version == QKNR_ABI_VERSION && hp.n_buffers == 3 && hp.chunk_rows == 2048, 51);
    CHECK(qknr_forward_host(NULL, &hp, NULL) == QKNR_ERR_NULL, 52);
    CHECK(qknr_forward_host(&a, NULL, NULL) == QKNR_ERR_NULL, 53);
    a.head_dim = 128;
    a.n_heads_q = a.n_heads_k = 24;
    a.tokens = 1000;
    hp.chunk_rows = 256;
    CHECK(qknr_host_buffer_bytes(&a, &hp, &ws) == QKNR_OK && ws == (size_t)256 * 48 * 128 * 2, 54);
    hp.n_buffers = 0;
    CHECK(qknr_forward_host(&a, &hp, NULL) == QKNR_ERR_SHAPE, 55);
  }
  printf("ok %d\n", QKNR_GN_NOALLOC_SCRATCH_BYTES);
  return 0;
}
"""


def test_c99_program_links_and_runs(tmp_path, built_lib):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(built_lib)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I" + INCLUDE, str(src),
                        "-o", str(exe), "-L" + libdir, "-lqknr", "-Wl,-rpath," + libdir,
                        "-Wl,-rpath," + B.cuda_lib_dir()],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    # the binding's copy of the no-allocation scratch size is the header's
    assert run.stdout.strip() == f"ok {Q.GN_NOALLOC_SCRATCH_BYTES}"
