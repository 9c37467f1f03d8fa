"""Pins of the input-side oracle: the patch permutation against explicit
loops and its exact inverse, the projections and the MLP against loops, the
sinusoid's closed forms, the scatter's zero rows, and probes H7 and H10."""
import numpy as np

from oracle import h3_input_oracle as IO
from oracle import h3_oracle as O

f32 = np.float32


def test_patch_pack_against_loops_and_inverse():
    rng = np.random.default_rng(1)
    C, T, H, W = 3, 2, 4, 6
    lat = rng.standard_normal((C, T, H, W)).astype(f32)
    rows = IO.patch_pack(lat)
    assert rows.shape == (T * (H // 2) * (W // 2), C * 4)
    r = 0
    for t in range(T):
        for h in range(H // 2):
            for w in range(W // 2):
                feat = [lat[c, t, 2 * h + a, 2 * w + b] for c in range(C) for a in range(2) for b in range(2)]
                np.testing.assert_array_equal(rows[r], np.array(feat, dtype=f32))
                r += 1
    np.testing.assert_array_equal(IO.patch_unpack(rows, C, T, H, W), lat)     # exact inverse
    assert IO.VIDEO_CHANNELS * 4 == 96                                          # RFC s2 flattened width


def test_input_projection_against_loops_and_probe_h7():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 7)).astype(f32)
    w = (0.3 * rng.standard_normal((4, 7))).astype(f32)
    b = (0.1 * rng.standard_normal(4)).astype(f32)
    y = IO.input_projection(x, w, b)
    for i in range(5):
        for j in range(4):
            acc = float(b[j]) + sum(float(x[i, k]) * float(w[j, k]) for k in range(7))
            assert y[i, j] == O.bf16_round(acc)
    early = IO.input_projection(O.bf16_round(x), w, b)           # H7: input cast to bf16 early
    assert not np.array_equal(early, y)


def test_packed_index_copy_scatter_and_zero_rows():
    a = np.arange(6.0).reshape(2, 3)
    b = -np.arange(3.0).reshape(1, 3) - 1
    out = IO.packed_index_copy(5, 3, [(a, [4, 1]), (b, [2])])
    np.testing.assert_array_equal(out[4], a[0])
    np.testing.assert_array_equal(out[1], a[1])
    np.testing.assert_array_equal(out[2], b[0])
    assert not out[0].any() and not out[3].any()
    swapped = IO.packed_index_copy(5, 3, [(a, [1, 4]), (b, [2])])   # H1: permuted index, unpermuted rows
    assert not np.array_equal(swapped, out)


def test_sinusoid_closed_forms_and_probe_h10():
    e = IO.timestep_sinusoid(np.array([0.0, 1.0, 0.25]))
    assert e.shape == (3, 256) and e.dtype == f32
    np.testing.assert_array_equal(e[0, :128], 1.0)              # cos(0)
    np.testing.assert_array_equal(e[0, 128:], 0.0)              # sin(0)
    assert e[1, 0] == f32(np.cos(1.0)) and e[1, 128] == f32(np.sin(1.0))    # f_0 = 1
    f127 = np.exp(-np.log(10000.0) * 127 / 128)
    assert e[2, 127] == f32(np.cos(0.25 * f127))
    np.testing.assert_allclose(e[:, :128] ** 2 + e[:, 128:] ** 2, 1.0, rtol=1e-6)
    assert not np.allclose(IO.timestep_sinusoid(np.array([250.0])), e[2:3])   # H10: scaled 0..1000


def test_timestep_mlp_against_loops():
    rng = np.random.default_rng(3)
    e = rng.standard_normal((2, 6))
    w1, b1 = rng.standard_normal((5, 6)), rng.standard_normal(5)
    w2, b2 = rng.standard_normal((3, 5)), rng.standard_normal(3)
    y = IO.timestep_mlp(e, w1, b1, w2, b2)
    for t in range(2):
        h = [b1[j] + sum(e[t, k] * w1[j, k] for k in range(6)) for j in range(5)]
        h = [v / (1 + np.exp(-v)) for v in h]
        for i in range(3):
            assert abs(float(y[t, i]) - (b2[i] + sum(h[j] * w2[i, j] for j in range(5)))) < 1e-5 * (1 + abs(y[t, i]))
