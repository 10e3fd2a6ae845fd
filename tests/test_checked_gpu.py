"""The checked build (libqknr_checked.so, the same sources compiled with
QKNR_CHECKED): every kernel tests each global access against the span of
the buffer it belongs to and each shared-memory stage read against its
stage, skips an access that misses and reports QKNR_ERR_BOUNDS in the
status word.  The seeded random sweeps of the three kernels (ragged sizes,
padded strides, all instances, both group-norm paths, launch knobs) run
through it with the status word required to stay 0, and a few cases are
compared bit for bit with the regular build.  A test-only flag shortens the
Q output span the kernel checks against, to show a refused store is
reported and skipped."""
import numpy as np
import pytest
import torch

import tests.test_random_adaln_gpu as RA
import tests.test_random_groupnorm_gpu as RG
import tests.test_random_parity_gpu as RQ
from diffusion_transformer_qk_gb300 import build as B
from diffusion_transformer_qk_gb300 import inputs as I
from diffusion_transformer_qk_gb300 import qknr as Q
from tests.gpu_util import table_to_dev, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs(built_lib, cuda_device):
    return Q.load(), Q.load(B.ensure_built(checked=True))


@pytest.fixture
def checked(libs, monkeypatch):
    """The binding's calls go to the checked library for one test."""
    monkeypatch.setattr(Q, "_lib", libs[1])
    Q.status_buffer().zero_()
    yield
    torch.cuda.synchronize()
    assert Q.read_status() == 0, "the checked build found an access outside a buffer"


@pytest.mark.parametrize("seed", range(40))
def test_qk_random_configurations_stay_in_bounds(checked, seed):
    RQ.test_random_configuration(seed)


@pytest.mark.parametrize("seed", range(30))
def test_adaln_random_configurations_stay_in_bounds(checked, seed):
    RA.test_random_adaln(seed)


@pytest.mark.parametrize("seed", range(30))
def test_group_norm_random_configurations_stay_in_bounds(checked, seed):
    RG.test_random_group_norm(seed)


def _dense_call(w, inp, **kw):
    qkv = to_dev(inp["qkv"], w.dtype)
    Q.qk_norm_rope_packed(qkv, w.n_heads_q, w.n_heads_k, w.n_heads_v, w.head_dim,
                          torch.from_numpy(inp["gamma_q"]).cuda(), torch.from_numpy(inp["gamma_k"]).cuda(),
                          table_to_dev(inp["cos"], "fp32"), table_to_dev(inp["sin"], "fp32"),
                          rope_style=w.rope_style, eps=w.eps, **kw)
    torch.cuda.synchronize()
    return to_bits(qkv)


@pytest.mark.parametrize("tokens", [4096, 1003])
def test_checked_build_gives_the_regular_bits(libs, monkeypatch, tokens):
    w = I.WORKLOADS["dense_4096x24x128"]
    inp = I.make_inputs(w, tokens=tokens)
    regular = _dense_call(w, inp)
    monkeypatch.setattr(Q, "_lib", libs[1])
    Q.status_buffer().zero_()
    got = _dense_call(w, inp)
    assert Q.read_status() == 0
    np.testing.assert_array_equal(got, regular)


def test_a_refused_store_is_reported_and_skipped(libs, monkeypatch):
    w = I.WORKLOADS["dense_4096x24x128"]
    T = 777
    inp = I.make_inputs(w, tokens=T)
    regular = _dense_call(w, inp)
    # the regular build ignores the flag
    np.testing.assert_array_equal(_dense_call(w, inp, flags=Q.FLAG_TEST_SHORT_OUT), regular)
    assert Q.read_status() == 0
    monkeypatch.setattr(Q, "_lib", libs[1])
    Q.status_buffer().zero_()
    got = _dense_call(w, inp, flags=Q.FLAG_TEST_SHORT_OUT)
    assert Q.read_status() == Q.STATUS_BY_NAME["QKNR_ERR_BOUNDS"]
    hq = w.n_heads_q * w.head_dim
    np.testing.assert_array_equal(got[:-1], regular[:-1])                    # every other row as usual
    np.testing.assert_array_equal(got[-1, :hq], inp["qkv"][-1, :hq])        # last Q row not written
    np.testing.assert_array_equal(got[-1, hq:], regular[-1, hq:])           # its K as usual
    # the library still works normally afterwards
    Q.status_buffer().zero_()
    np.testing.assert_array_equal(_dense_call(w, inp), regular)
    assert Q.read_status() == 0
