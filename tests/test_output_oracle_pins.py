"""Pins of the output-side and sampler oracle against what the pages and the
mathematics fix: closed forms of the sigma transform, hand-computed grids,
identities of the Euler update and the noise mix, brute-force loops for the
final AdaLN and the heads, and the RFC's mismatch probes H9-H14, each of
which must move the result."""
import numpy as np
import pytest

from oracle import h3_output_oracle as OO

f32 = np.float32


# ---------------------------------------------------------------- sigma grid

def test_shift_closed_forms():
    assert OO.shift_sigma(1.0, 12.0) == f32(1.0)
    assert OO.shift_sigma(0.0, 12.0) == f32(0.0)
    # s * 0.5 / (1 + (s-1) * 0.5) = s / (s + 1)
    assert OO.shift_sigma(0.5, 12.0) == f32(f32(6.0) / f32(6.5))
    assert OO.shift_sigma(0.5, 3.0) == f32(0.75)
    sg = np.linspace(0.0, 1.0, 101).astype(f32)
    np.testing.assert_array_equal(OO.shift_sigma(sg, 1.0), sg)       # shift 1 is the identity
    for s in (3.0, 12.0):
        y = OO.shift_sigma(sg, s)
        assert np.all(np.diff(y.astype(np.float64)) > 0)              # monotone
        assert np.all(y[1:-1] > sg[1:-1])                             # s > 1 pushes sigma up


def test_sigma_grid_hand_values():
    # base 1, .75, .5, .25, 0 with shift 3: 3x / (1 + 2x) = 1, .9, .75, .5, 0
    g = OO.sigma_grid(5, 3.0)
    np.testing.assert_array_equal(g, np.array([1.0, f32(f32(2.25) / f32(2.5)), 0.75, 0.5, 0.0], dtype=f32))
    np.testing.assert_array_equal(OO.sigma_grid(3, 12.0), np.array([1.0, f32(6.0) / f32(6.5), 0.0], dtype=f32))
    # the appended terminal zero collapses with the linspace's own zero
    np.testing.assert_array_equal(OO.sigma_grid(2, 12.0), np.array([1.0, 0.0], dtype=f32))


@pytest.mark.parametrize("n,s", [(13, 12.0), (13, 3.0), (50, 12.0), (1000, 3.0)])
def test_sigma_grid_structure(n, s):
    g = OO.sigma_grid(n, s)
    assert g.dtype == f32 and g[0] == 1.0 and g[-1] == 0.0
    assert g.size == n                                     # n - 1 model evaluations
    assert np.all(np.diff(g.astype(np.float64)) < 0)        # strictly decreasing, no duplicate left


def test_probes_h11_h12_h10():
    video, audio = OO.sigma_grid(13, OO.VIDEO_SHIFT), OO.sigma_grid(13, OO.AUDIO_SHIFT)
    generic = np.linspace(1, 0, 13).astype(f32)
    assert not np.array_equal(video, generic)             # H11: unshifted grid differs
    assert not np.array_equal(video, audio)               # H12: the two schedulers differ
    t = OO.timesteps(video)
    np.testing.assert_array_equal(t, (f32(1) - video).astype(f32))
    assert t[0] == 0.0 and t[-1] == 1.0                    # t = 1 clean
    assert not np.array_equal(t, video)                    # H10: t = sigma differs


# ---------------------------------------------------------------- Euler step

def _rand(n, seed):
    return np.random.default_rng(seed).standard_normal(n).astype(f32)


def test_ode_step_end_and_identity_cases():
    xt, v = _rand(1000, 1), _rand(1000, 2)
    sg = f32(0.7)
    x0 = (xt + (sg * v).astype(f32)).astype(f32)
    np.testing.assert_array_equal(OO.ode_step(xt, v, sg, 0.0), x0)     # last step lands on x0
    np.testing.assert_array_equal(OO.ode_step(xt, v, sg, sg), xt)      # r = 1 keeps xt


def test_ode_step_follows_the_straight_path():
    # data-ward velocity towards a fixed x_data: v = (x_data - xt) / sigma
    xt, xd = _rand(4096, 3), _rand(4096, 4)
    sg, sn = 0.8, 0.35
    v = ((xd.astype(np.float64) - xt) / sg).astype(f32)
    got = OO.ode_step(xt, v, sg, sn).astype(np.float64)
    want = (sn / sg) * xt + (1 - sn / sg) * xd.astype(np.float64)
    np.testing.assert_allclose(got, want, atol=2e-6)


def test_probes_h9_h13():
    xt, v = _rand(4096, 5), _rand(4096, 6)
    sg, sn = f32(0.6), f32(0.45)
    good = OO.ode_step(xt, v, sg, sn)
    bad_sign = OO.ode_step(xt, -v, sg, sn)                   # H9: subtract the velocity
    assert np.abs(good - bad_sign).max() > 0.1
    r = f32(sn / sg)
    x0 = (xt + (sg * v).astype(f32)).astype(f32)
    reordered = (xt + ((f32(1) - r) * (x0 - xt).astype(f32)).astype(f32)).astype(f32)   # H13
    assert not np.array_equal(good, reordered)               # same value mathematically, not bitwise
    np.testing.assert_allclose(good, reordered, atol=1e-5)


def test_noise_mix_ends_and_linearity():
    x0, nz = _rand(512, 7), _rand(512, 8)
    np.testing.assert_array_equal(OO.noise_mix(x0, nz, 1.0), x0)
    np.testing.assert_array_equal(OO.noise_mix(x0, nz, 0.0), nz)
    got = OO.noise_mix(x0, nz, 0.25).astype(np.float64)
    np.testing.assert_allclose(got, 0.25 * x0 + 0.75 * nz.astype(np.float64), atol=1e-6)
    assert not np.array_equal(OO.noise_mix(x0, nz, 0.25), OO.noise_mix(nz, x0, 0.25))   # H15 order


# ---------------------------------------------------------------- output side

def test_select_rows_and_probe_h14():
    tag = np.random.default_rng(9).integers(0, 3, 257).astype(np.int32)
    for m in range(3):
        np.testing.assert_array_equal(OO.select_rows(tag, m), np.flatnonzero(tag == m).astype(np.int32))
    stale = OO.select_rows(np.roll(tag, 1), OO.TAG_VIDEO)        # H14: stale indices
    assert not np.array_equal(stale, OO.select_rows(tag, OO.TAG_VIDEO))


def test_final_adaln_table_against_loops():
    rng = np.random.default_rng(10)
    T, C, D = 3, 7, 5
    tc = rng.standard_normal((T, C))
    w = rng.standard_normal((2 * D, C)) * 0.1
    b = rng.standard_normal(2 * D) * 0.1
    tab = OO.final_adaln_table(tc, w, b)
    assert tab.shape == (T, 2, D) and tab.dtype == f32
    for t in range(T):
        for j in range(2 * D):
            acc = b[j]
            for k in range(C):
                x = tc[t, k]
                acc += (x / (1.0 + np.exp(-x))) * w[j, k]
            assert tab[t, j // D, j % D] == f32(acc)
    z = OO.final_adaln_table(tc, np.zeros((2 * D, C)), b)       # zero weights: the bias alone
    np.testing.assert_array_equal(z.reshape(T, 2 * D), np.broadcast_to(b.astype(f32), (T, 2 * D)))


def test_final_norm_and_head_against_loops():
    rng = np.random.default_rng(11)
    S, D, P, T = 9, 16, 4, 2
    x = rng.standard_normal((S, D))
    tag = np.array([1, 0, 0, 2, 0, 1, 2, 0, 2], dtype=np.int32)
    tidx = np.array([0, 1, 0, 1, 1, 0, 0, 0, 1], dtype=np.int32)
    table = rng.standard_normal((T, 2, D)).astype(f32) * 0.1
    w = rng.standard_normal((P, D)) * 0.2
    b = rng.standard_normal(P) * 0.1
    got = OO.output_head(x, tag, tidx, OO.TAG_VIDEO, table, w, b)
    rows = [1, 2, 4, 7]
    assert got.shape == (len(rows), P)
    for i, r in enumerate(rows):
        rms = np.sqrt(sum(x[r, k] ** 2 for k in range(D)) / D + OO.EPS)
        for p in range(P):
            acc = b[p]
            for k in range(D):
                m = x[r, k] / rms * (1.0 + float(table[tidx[r], 1, k])) + float(table[tidx[r], 0, k])
                acc += m * w[p, k]
            assert abs(got[i, p] - acc) < 1e-12
    # shift = scale = 0 and identity head: the normalised row, unit RMS
    ident = np.eye(D)
    n = OO.output_head(x, tag, tidx, OO.TAG_AUDIO, np.zeros((T, 2, D), f32), ident, None)
    np.testing.assert_allclose(np.sqrt(np.mean(n * n, axis=1)), 1.0, rtol=1e-4)
    # the timestep index selects the table row
    t2 = table.copy()
    t2[1] += 1.0
    assert np.abs(OO.output_head(x, tag, tidx, OO.TAG_VIDEO, t2, w, b) - got).max() > 1e-3
