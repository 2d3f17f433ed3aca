"""Shared helpers for the GPU parity tests (marshalling and error metrics only)."""
import numpy as np
import torch

import synth

# Linear tolerance: the task's bar on bf16 outputs, against the oracle's bf16
# output (both sides rounded once to bf16).
MAX_REL = 2e-2
MAE = 1e-3


def dev():
    return torch.device("cuda", 0)


def bf16_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(torch.bfloat16)


def canon_to_dev(qw: np.ndarray, sc: np.ndarray):
    return (torch.from_numpy(np.ascontiguousarray(qw).view(np.int32)).to(dev()),
            torch.from_numpy(np.ascontiguousarray(sc).view(np.float16)).to(dev()))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def linear_errors(got_bits: np.ndarray, ref_bits: np.ndarray):
    """(mae, max_rel, exact_fraction). max_rel uses a floor of 1e-3 * rms(ref)
    in the denominator so that outputs near zero do not dominate."""
    g = synth.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = synth.bf16_bits_to_f32(ref_bits).astype(np.float64)
    err = np.abs(g - r)
    mae = float(err.mean()) if err.size else 0.0
    floor = 1e-3 * float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    denom = np.maximum(np.abs(r), max(floor, 1e-30))
    max_rel = float((err / denom).max()) if err.size else 0.0
    exact = float(np.mean(got_bits == ref_bits)) if err.size else 1.0
    return mae, max_rel, exact


def assert_linear_close(got_bits, ref_bits, what=""):
    mae, max_rel, exact = linear_errors(got_bits, ref_bits)
    assert np.all(np.isfinite(synth.bf16_bits_to_f32(got_bits))), f"{what}: non-finite output"
    assert mae <= MAE and max_rel <= MAX_REL, f"{what}: mae={mae:.3e} max_rel={max_rel:.3e} exact={exact:.4f}"
    return mae, max_rel, exact
