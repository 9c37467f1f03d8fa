"""The end-to-end bounds come from committed evidence: the stored
fp32-vs-fp64 floors reproduce when the script that wrote them is re-run on
the CPU, and every end-to-end bound is twice its floor.

The floors are recomputed in full: the 505-row block and the 256-row refiner
at full width (about a minute and a half of CPU time together) and the
50-block tiny chain.  A different BLAS may sum the fp32 products in another
order, which moves individual bf16 flips; the stored values are required to
reproduce within a few per cent."""
import json
import os
import sys

import pytest

import h3_testutil as U

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
import make_chain_floors as M  # noqa: E402

pytestmark = pytest.mark.slow


def stored():
    with open(os.path.join(HERE, "golden", "chain_floors.json")) as f:
        return json.load(f)["floors"]


def test_bounds_are_twice_the_floors():
    fl = stored()
    pairs = [("block505", U.CHAIN_MAX_E, U.CHAIN_MEAN_E),
             ("refiner256", U.REFINER_CHAIN_MAX_E, U.REFINER_CHAIN_MEAN_E),
             ("tiny72x50", U.TINY50_CHAIN_MAX_E, U.TINY50_CHAIN_MEAN_E)]
    for name, bmax, bmean in pairs:
        for bound, floor in ((bmax, fl[name]["max_e"]), (bmean, fl[name]["mean_e"])):
            assert 2.0 * floor <= bound <= 2.0 * floor * 1.1, (name, bound, floor)
    # the per-operator bound stays the stated one
    assert (U.MAX_E, U.MEAN_E) == (2e-2, 2e-3)


@pytest.mark.parametrize("case", sorted(M.CASES))
def test_stored_floor_reproduces(case):
    mx, mn = M.CASES[case]()
    fl = stored()[case]
    print(f"{case}: max_e={mx:.5f} (stored {fl['max_e']}) mean_e={mn:.6f} (stored {fl['mean_e']})")
    assert mx == pytest.approx(fl["max_e"], rel=0.15)
    assert mn == pytest.approx(fl["mean_e"], rel=0.05)
