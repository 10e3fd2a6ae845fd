"""Shared helpers of the GPU tests: moving uint16 bit arrays to and from the
device and comparing kernel outputs with the fp64 oracle."""
import numpy as np
import torch

from oracle import qknr_oracle as O

# max |gpu - oracle| allowed, from "fused qknorm rope Flux 2.0" (Numbers:
# kernel correctness vs a PyTorch reference, bf16 limit 3e-2, fp16 limit 5e-3)
TOL = {"bf16": 3e-2, "fp16": 5e-3}
TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16}


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH[dtype]).to(device)


def table_to_dev(tab: np.ndarray, cos_dtype: str, device="cuda") -> torch.Tensor:
    if cos_dtype == "fp32":
        return torch.from_numpy(np.ascontiguousarray(tab)).to(device)
    return to_dev(tab, "bf16", device)


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def ordered(bits: np.ndarray) -> np.ndarray:
    """Map 16-bit float patterns to integers whose order is the value order."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def compare(got_bits: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    """Assert the GPU result is within the pages' max_abs limit of the fp64
    oracle and at most one unit in the last place from the correctly
    rounded oracle value.  Returns (max_abs, fraction off by one ulp)."""
    got_bits = got_bits.reshape(ref.shape)
    got = O.decode(got_bits, dtype)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    assert max_abs <= TOL[dtype], f"{what}: max_abs {max_abs} > {TOL[dtype]}"
    rn = O.round_rne(ref, dtype)
    ulp = np.abs(ordered(got_bits) - ordered(rn))
    # Near zero a result can be a cancellation whose fp32 rounding error
    # (~1e-6 absolute) spans several ulps; those elements are held to the
    # max_abs limit only.
    big = np.abs(ref) >= 2.0 ** -6
    worst = int(ulp[big].max(initial=0))
    assert worst <= 1, f"{what}: {worst} ulp from the rounded oracle"
    frac = float((ulp != 0).mean()) if ulp.size else 0.0
    return max_abs, frac

def ulp_of(v: np.ndarray, dtype: str) -> np.ndarray:
    """The spacing of the 16-bit float format at magnitude |v| (normal range)."""
    mant = {"bf16": 7, "fp16": 10}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -14)))
    return 2.0 ** (e - mant)


def compare_ulps(got_bits: np.ndarray, ref: np.ndarray, dtype: str, ulps: int, what: str = ""):
    """Assert every output is at most `ulps` units in the last place from the
    correctly rounded fp64 oracle: |got - ref| <= (ulps + 1/2) spacings of
    the format at max(|ref|, |got|, 2^-6).  A relative bound for outputs far
    above 1 (where the pages' absolute limit is below one ulp) and the bound
    at 2^-6 for smaller ones."""
    got_bits = got_bits.reshape(ref.shape)
    got = O.decode(got_bits, dtype)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = ulp_of(np.maximum(np.maximum(np.abs(ref), np.abs(got)), 2.0 ** -6), dtype)
    worst = float((np.abs(got - ref) / scale).max()) - 0.5
    assert worst <= ulps, f"{what}: {worst:.2f} ulps from the rounded oracle (bound {ulps})"
    return worst
