"""Writes chain_floors.json: how far two correct evaluations of the H3 block
drift apart end to end when one sums in fp64 and the other in fp32.

Both sides are CPU oracles (oracle/h3_oracle.py in fp64, oracle/h3_oracle_fp32.py
in fp32) evaluating the same definition with the same bf16 cast points on the
same seeded inputs; nothing here runs or reads the CUDA path.  The distance
is measured with the tests' error metric,
    e_i = |a_i - ref_i| / max(RMS(ref), |ref_i|),
and stored as the max and the mean of e.  The end-to-end tests of the CUDA
path take twice these floors as their bounds (tests/h3_testutil.py).

Cases:
  block505     one full-width block (D 5376, 56 heads, F 14336, C 2688) over
               505 packed rows (17 text + 360 video on 6x6x10 + 128 audio),
               12 timestep rows, seed 0, block 0 weights;
  refiner256   the two-block token refiner and its final RMSNorm at full
               width over 256 rows (the refiner workload's inputs);
  tiny72x50    50 blocks of the tiny H3-shaped block (D 512, 4 heads) over
               72 packed rows, each block with its own weights (block ids
               0..49), one evaluation chained end to end.

Run from the repository root:  python tests/golden/make_chain_floors.py
"""
from __future__ import annotations

import json
import os
import platform
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import h3_inputs as hi  # noqa: E402
from oracle import h3_oracle as O  # noqa: E402
from oracle import h3_oracle_fp32 as O32  # noqa: E402

OUT = os.path.join(HERE, "chain_floors.json")


def metric(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    e = np.abs(a - ref) / np.maximum(rms, np.abs(ref))
    return float(e.max()), float(e.mean())


def _f64(t):
    return None if t is None else t.detach().to(torch.float64).numpy()


def _f32(t):
    return None if t is None else t.detach().to(torch.float32).numpy()


def floor_block505(seed: int = 0):
    w = hi.WORKLOADS["block505"]
    meta, acts, wts = hi.workload_inputs(w, seed=seed)
    args = (meta["token_tag"].numpy(), meta["timestep_index"].numpy(), meta["pos_thw"].numpy())
    ref = O.block_forward(_f64(acts["x"]), *args, acts["t_cond"].numpy().astype(np.float64),
                          {k: _f64(v) for k, v in wts.items()})["y"]
    got = O32.block_forward(_f32(acts["x"]), *args, acts["t_cond"].numpy(), {k: _f32(v) for k, v in wts.items()})
    return metric(got, ref)


def refiner_inputs(seed: int = 0):
    """The full-width refiner test's inputs: blocks with ids 7 and 8, the final
    gain and the rows with tensor ids 90 and 91."""
    shape = hi.H3_SHAPE
    wts = [hi.block_weights(shape, seed, b) for b in (7, 8)]
    gfin = hi.normal((shape.dim,), 0.1, 1.0, seed, 90)
    x = hi.normal((256, shape.dim), 1.0, 0.0, seed, 91)
    return wts, gfin, x


def floor_refiner256(seed: int = 0):
    wts, gfin, x = refiner_inputs(seed)
    ref = O.refiner_forward(_f64(x), [{k: _f64(v) for k, v in w.items()} for w in wts], _f64(gfin))
    got = O32.refiner_forward(_f32(x), [{k: _f32(v) for k, v in w.items()} for w in wts], _f32(gfin))
    return metric(got, ref)


def tiny_chain_inputs(n_blocks: int = 50, seed: int = 0):
    w = hi.WORKLOADS["tiny72"]
    meta = hi.packed_metadata(w.layout, w.n_timesteps, seed)
    acts = hi.activations(w.shape, w.layout.n_rows, w.n_timesteps, seed)
    wts = [hi.block_weights(w.shape, seed, b) for b in range(n_blocks)]
    return w, meta, acts, wts


def floor_tiny_chain(n_blocks: int = 50, seed: int = 0):
    w, meta, acts, wts = tiny_chain_inputs(n_blocks, seed)
    args = (meta["token_tag"].numpy(), meta["timestep_index"].numpy(), meta["pos_thw"].numpy())
    ref = O.blocks_forward(_f64(acts["x"]), *args, acts["t_cond"].numpy().astype(np.float64),
                           [{k: _f64(v) for k, v in ww.items()} for ww in wts])
    got = O32.blocks_forward(_f32(acts["x"]), *args, acts["t_cond"].numpy(),
                             [{k: _f32(v) for k, v in ww.items()} for ww in wts])
    return metric(got, ref)


CASES = {"block505": floor_block505, "refiner256": floor_refiner256, "tiny72x50": floor_tiny_chain}


def main():
    out = {"metric": "e_i = |a_i - ref_i| / max(RMS(ref), |ref_i|); fp32 evaluation vs fp64 oracle",
           "numpy": np.__version__, "machine": platform.machine(), "floors": {}}
    for name, fn in CASES.items():
        t0 = time.perf_counter()
        mx, mn = fn()
        out["floors"][name] = {"max_e": round(mx, 6), "mean_e": round(mn, 7)}
        print(f"{name}: max_e={mx:.5f} mean_e={mn:.6f} ({time.perf_counter() - t0:.1f} s)", flush=True)
    with open(OUT, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
