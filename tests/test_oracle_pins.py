"""Pins of the CPU oracle against facts that do not come from the oracle itself:
closed forms, library routines, brute-force loops on tiny inputs, invariants of
the method, the dimension table printed by the MiniMax-H3 RFC, and mismatch
probes H1-H8 of the RFC's ablation matrix (section 6.2), each of which must move
the result well beyond tolerance.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import h3_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_torch(x):
    """Library routine: torch's fp32 -> bf16 conversion (round to nearest even)."""
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def rand_bf16(rng, shape, std=1.0):
    return O.bf16_round(rng.standard_normal(shape) * std)


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def test_bf16_round_matches_torch_on_fp32_values(rng):
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 10.0,
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),     # fp32 subnormals
        np.array([3.0e38, -3.39e38, 1e-45, 0.0, -0.0], np.float32),
        # exact ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -126 * (1 + 2 ** -8)],
                 np.float32),
    ])
    np.testing.assert_array_equal(O.bf16_round(x.astype(np.float64)), bf16_torch(x))


def test_bf16_round_rounds_float64_directly():
    # 1 + 2^-8 + 2^-40 is above the midpoint: a direct round goes up.
    # (Rounding to fp32 first would land exactly on the tie and go down.)
    assert O.bf16_round(1 + 2 ** -8 + 2 ** -40) == 1 + 2 ** -7
    assert O.bf16_round(1 + 2 ** -8) == 1.0            # tie to even
    assert O.bf16_round(1 + 3 * 2 ** -8) == 1 + 2 ** -6  # tie to even (up)
    assert O.bf16_round(2.0 ** 128) == np.inf
    assert O.bf16_round(-2.0 ** 200) == -np.inf
    assert O.bf16_round(2.0 ** -140) == 0.0            # below half the subnormal step


# ---------------------------------------------------------------------------
# fingerprint printed by the RFC
# ---------------------------------------------------------------------------

def test_fingerprint_table():
    fp = json.load(open(os.path.join(GOLDEN, "h3_fingerprint.json")))
    v = {k: d["value"] for k, d in fp.items() if not k.startswith("_")}
    assert v["attention_heads"] * v["head_dim"] == v["attention_inner_dim"]
    assert 6 * 3 * v["residual_hidden_size"] == v["adaln_out_width"]
    assert 3 * v["rope_freqs_per_axis"] * 2 == v["rotary_channels"]
    assert v["modality_tags"] == {"video": 0, "text": 1, "audio": 2}
    assert O.EPS == v["block_norm_eps"] == v["qk_norm_eps"]
    assert O.ROPE_THETA == v["rope_theta"] and O.ROPE_FREQS_PER_AXIS == v["rope_freqs_per_axis"]
    assert O.ROPE_CHANNELS == v["rotary_channels"] and O.HEAD_DIM == v["head_dim"]
    # the oracle's table at full width has the printed width
    D, C = v["residual_hidden_size"], 2
    w = np.zeros((v["adaln_out_width"], C))
    tab = O.adaln_table(np.zeros((1, C)), w, None, D)
    assert tab.shape == (3, 6, D) and tab.size == v["adaln_out_width"]
    import h3_inputs as hi
    s = hi.H3_SHAPE
    assert (s.dim, s.n_heads, s.head_dim, s.ffn_dim, s.cond_dim) == (
        v["residual_hidden_size"], v["attention_heads"], v["head_dim"], v["ffn_hidden_size"],
        v["adaln_cond_width"])


# ---------------------------------------------------------------------------
# AdaLN projection, row rule and modulation
# ---------------------------------------------------------------------------

def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(O.silu(-2.0) - (-2.0 / (1.0 + math.exp(2.0)))) < 1e-15
    assert abs(O.silu(40.0) - 40.0) < 1e-12


def test_adaln_table_brute_force(rng):
    T, C, D = 2, 5, 3
    t_cond = rng.standard_normal((T, C))
    w = rand_bf16(rng, (18 * D, C), 0.3)
    b = rand_bf16(rng, (18 * D,), 0.1)
    tab = O.adaln_table(t_cond, w, b, D)
    for t in range(T):
        u = [float(O.bf16_round(t_cond[t, k] / (1.0 + math.exp(-t_cond[t, k])))) for k in range(C)]
        for m in range(3):
            for c in range(6):
                for d in range(D):
                    n = m * 6 * D + c * D + d              # [modality][chunk][D] per timestep
                    acc = sum(u[k] * w[n, k] for k in range(C)) + b[n]
                    assert tab[t * 3 + m, c, d] == O.bf16_round(acc)


def test_adaln_identity_slice(rng):
    T, C, D = 3, 4, 2
    t_cond = rng.standard_normal((T, C))
    w = np.zeros((18 * D, C))
    for n in range(18 * D):
        w[n, n % C] = 1.0
    tab = O.adaln_table(t_cond, w, None, D).reshape(T, 18 * D)
    for n in range(18 * D):
        np.testing.assert_array_equal(tab[:, n], O.bf16_round(O.silu(t_cond[:, n % C])))


def test_adaln_row_rule():
    tags = np.array([0, 1, 2, 0, 2, 1])
    tidx = np.array([0, 0, 0, 1, 3, 5])
    np.testing.assert_array_equal(O.adaln_rows(tags, tidx), [0, 1, 2, 3, 11, 16])


def _row_valued_table(T, D):
    """Table whose shift_msa row rho is the constant rho and scale_msa = -1, so
    the modulated output of a packed row equals its table row index."""
    tab = np.zeros((3 * T, 6, D))
    for rho in range(3 * T):
        tab[rho, O.CHUNK_SHIFT_MSA, :] = rho
        tab[rho, O.CHUNK_SCALE_MSA, :] = -1.0
    return tab


def test_adaln_gather_shows_row_index(rng):
    T, D, S = 5, 8, 40
    tags = rng.integers(0, 3, S)
    tidx = rng.integers(0, T, S)
    tab = _row_valued_table(T, D)
    mod = tab[O.adaln_rows(tags, tidx)]
    h = O.rmsnorm_modulate(rng.standard_normal((S, D)), np.ones(D), mod[:, 0], mod[:, 1])
    np.testing.assert_array_equal(h, np.repeat((tidx * 3 + tags)[:, None], D, axis=1))
    # probe H2: one flipped tag changes that row's modulation
    tags2 = tags.copy()
    tags2[7] = (tags2[7] + 1) % 3
    h2 = O.rmsnorm_modulate(rng.standard_normal((S, D)), np.ones(D),
                            tab[O.adaln_rows(tags2, tidx)][:, 0], tab[O.adaln_rows(tags2, tidx)][:, 1])
    assert np.all(h2[7] != h[7]) and np.array_equal(np.delete(h2, 7, 0), np.delete(h, 7, 0))
    # probe H3: offset timestep index
    tidx3 = tidx.copy()
    tidx3[3] = (tidx3[3] + 1) % T
    assert O.adaln_rows(tags, tidx3)[3] != O.adaln_rows(tags, tidx)[3]


def test_adaln_layout_probe_h4(rng):
    """Probe H4: a six-chunk-major layout [6][3][D] reads different rows."""
    T, C, D = 2, 6, 4
    t_cond = rng.standard_normal((T, C))
    w = rand_bf16(rng, (18 * D, C), 0.3)
    tab = O.adaln_table(t_cond, w, None, D)
    flat = tab.reshape(T, 18 * D)
    chunk_major = flat.reshape(T, 6, 3, D).transpose(0, 2, 1, 3).reshape(3 * T, 6, D)
    assert np.abs(chunk_major - tab).max() > 0.1


def test_rmsnorm_closed_forms(rng):
    D = 64
    for c in [0.5, 3.0, -7.25, 1e-3]:
        x = np.full((1, D), c)
        h = O.rmsnorm_modulate(x, np.ones(D), np.zeros((1, D)), np.zeros((1, D)))
        np.testing.assert_array_equal(h, O.bf16_round(np.full((1, D), c / math.sqrt(c * c + 1e-5))))
    # per-channel gain, then (1 + scale), then + shift
    x = np.full((1, 4), 2.0)
    g = np.array([1.0, 2.0, 0.5, -1.0])
    sc = np.array([[0.0, 1.0, -0.5, 0.25]])
    sh = np.array([[0.0, 0.0, 1.0, -2.0]])
    n = 2.0 / math.sqrt(4.0 + 1e-5)
    want = O.bf16_round(np.array([[n, n * 2 * 2, n * 0.5 * 0.5 + 1.0, -n * 1.25 - 2.0]]))
    np.testing.assert_array_equal(O.rmsnorm_modulate(x, g, sh, sc), want)


def test_rmsnorm_unit_rms_and_scale_invariance(rng):
    S, D = 16, 512
    x = rng.standard_normal((S, D)) * 3.0
    z = np.zeros((S, D))
    h = O.rmsnorm_modulate(x, np.ones(D), z, z)
    rms = np.sqrt(np.mean(h * h, axis=1))
    want = np.sqrt(np.mean(x * x, 1) / (np.mean(x * x, 1) + 1e-5))
    assert np.max(np.abs(rms - want)) < 2 ** -8
    # with eps = 0 the norm is invariant to a power-of-two scale, bit for bit
    np.testing.assert_array_equal(O.rmsnorm_modulate(8.0 * x, np.ones(D), z, z, eps=0.0),
                                  O.rmsnorm_modulate(x, np.ones(D), z, z, eps=0.0))


# ---------------------------------------------------------------------------
# projections
# ---------------------------------------------------------------------------

def test_linear_brute_force(rng):
    x = rand_bf16(rng, (3, 5))
    w = rand_bf16(rng, (4, 5))
    b = rand_bf16(rng, (4,))
    y = O.linear(x, w, b)
    for i in range(3):
        for j in range(4):
            assert y[i, j] == O.bf16_round(sum(x[i, k] * w[j, k] for k in range(5)) + b[j])


def test_linear_identity_weights(rng):
    x = rand_bf16(rng, (6, 8))
    np.testing.assert_array_equal(O.linear(x, np.eye(8)), x)


# ---------------------------------------------------------------------------
# Q/K norm and MM-RoPE
# ---------------------------------------------------------------------------

def test_head_rmsnorm_unit_rms_and_brute_force(rng):
    v = rng.standard_normal((10, 3, 128)) * 5
    h = O.head_rmsnorm(v, np.ones(128))
    assert np.max(np.abs(np.sqrt(np.mean(h * h, -1)) - 1.0)) < 2 ** -7
    g = rand_bf16(rng, (128,), 0.1) + 1.0
    h = O.head_rmsnorm(v, g)
    vv = v[2, 1]
    inv = 1.0 / math.sqrt(sum(t * t for t in vv) / 128 + 1e-5)
    for j in range(128):
        assert abs(h[2, 1, j] - O.bf16_round(vv[j] * inv * g[j])) == 0


def test_rope_frequencies_closed_form():
    om = O.rope_frequencies()
    assert om.dtype == np.float32 and om.shape == (16,)
    for i, want in [(0, 1.0), (4, 0.1), (8, 0.01), (12, 0.001)]:
        assert om[i] == np.float32(want)
    assert om[1] == np.float32(10000.0 ** (-1.0 / 16.0))


def test_rope_identity_at_zero_position(rng):
    x = rand_bf16(rng, (5, 4, 128))
    np.testing.assert_array_equal(O.mm_rope(x, np.zeros((5, 3), np.int32)), x)


def test_rope_passthrough_channels_and_pair_norm(rng):
    S = 30
    x = rand_bf16(rng, (S, 4, 128))
    pos = rng.integers(0, 40, (S, 3))
    y = O.mm_rope(x, pos)
    np.testing.assert_array_equal(y[..., 96:], x[..., 96:])
    n_in = x[..., :48] ** 2 + x[..., 48:96] ** 2
    n_out = y[..., :48] ** 2 + y[..., 48:96] ** 2
    assert np.max(np.abs(n_out - n_in) / np.maximum(n_in, 1e-3)) < 2 * 2 ** -7


def test_rope_hand_values():
    # one unit vector per band; positions (t,h,w) = (1, 2, 3)
    x = np.zeros((1, 1, 128))
    x[0, 0, 0] = 1.0      # band t, frequency 0 -> angle 1 * 1
    x[0, 0, 17] = 1.0     # band h, frequency 1 -> angle 2 * 10000^(-1/16)
    x[0, 0, 40] = 1.0     # band w, frequency 8 -> angle 3 * 0.01
    y = O.mm_rope(x, np.array([[1, 2, 3]]))
    a_h = float(np.float32(2.0) * np.float32(10000.0 ** (-1 / 16)))
    a_w = float(np.float32(3.0) * np.float32(0.01))
    assert y[0, 0, 0] == O.bf16_round(math.cos(1.0)) and y[0, 0, 48] == O.bf16_round(math.sin(1.0))
    assert y[0, 0, 17] == O.bf16_round(math.cos(a_h)) and y[0, 0, 65] == O.bf16_round(math.sin(a_h))
    assert y[0, 0, 40] == O.bf16_round(math.cos(a_w)) and y[0, 0, 88] == O.bf16_round(math.sin(a_w))
    # the partner channel rotates the other way: x_{j+48} = 1 -> (-sin, cos)
    x = np.zeros((1, 1, 128))
    x[0, 0, 48] = 1.0
    y = O.mm_rope(x, np.array([[1, 0, 0]]))
    assert y[0, 0, 0] == O.bf16_round(-math.sin(1.0)) and y[0, 0, 48] == O.bf16_round(math.cos(1.0))


def _rope_attention(q, k, v, pos):
    return O.attention(O.mm_rope(q, pos), O.mm_rope(k, pos), v)


def test_rope_relative_position_property(rng):
    S, H = 24, 2
    q, k, v = (rand_bf16(rng, (S, H, 128)) for _ in range(3))
    pos = rng.integers(0, 8, (S, 3))
    o1 = _rope_attention(q, k, v, pos)
    o2 = _rope_attention(q, k, v, pos + np.array([3, 5, 7]))
    rms = np.sqrt(np.mean(o1 ** 2))
    assert np.max(np.abs(o1 - o2)) / rms < 0.05 and np.mean(np.abs(o1 - o2)) / rms < 5e-3


def test_rope_probe_h5_full_rotation(rng):
    """Probe H5: rotating all 128 channels (standard full-head RoPE) or concatenating
    the axes in another order changes the result."""
    S = 16
    x = rand_bf16(rng, (S, 2, 128))
    pos = rng.integers(1, 10, (S, 3))
    good = O.mm_rope(x, pos)
    # full-head split-half with a 64-frequency ladder
    om = O.fp32(10000.0 ** (-np.arange(64) / 64))
    ang = (O.fp32(pos[:, 0])[:, None] * om[None, :]).astype(np.float64)[:, None, :]
    full = np.concatenate([x[..., :64] * np.cos(ang) - x[..., 64:] * np.sin(ang),
                           x[..., 64:] * np.cos(ang) + x[..., :64] * np.sin(ang)], -1)
    assert np.abs(full - good).max() > 0.5
    swapped = O.mm_rope(x, pos[:, [2, 1, 0]])       # (w, h, t) axis order
    assert np.abs(swapped - good).max() > 0.5


def test_rope_probe_h6_order(rng):
    """Probe H6: RoPE then Q/K norm differs from Q/K norm then RoPE (non-uniform gain)."""
    S = 16
    x = rand_bf16(rng, (S, 2, 128), 2.0)
    g = rand_bf16(rng, (128,), 0.3) + 1.0
    pos = rng.integers(1, 10, (S, 3))
    good = O.mm_rope(O.head_rmsnorm(x, g), pos)
    bad = O.head_rmsnorm(O.mm_rope(x, pos), g)
    assert np.abs(good - bad).max() > 0.1


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def test_attention_brute_force(rng):
    S = 7
    q, k, v = (rng.standard_normal((S, 128)) for _ in range(3))
    got = O.attention_head(q, k, v)
    for i in range(S):
        sc = [sum(q[i, c] * k[j, c] for c in range(128)) / math.sqrt(128) for j in range(S)]
        m = max(sc)
        e = [math.exp(s - m) for s in sc]
        z = sum(e)
        for c in range(0, 128, 17):
            want = sum(e[j] / z * v[j, c] for j in range(S))
            assert abs(got[i, c] - want) < 1e-12


def test_attention_special_cases(rng):
    S = 9
    k, v = rng.standard_normal((S, 128)), rng.standard_normal((S, 128))
    np.testing.assert_allclose(O.attention_head(np.zeros((3, 128)), k, v),
                               np.repeat(v.mean(0, keepdims=True), 3, 0), rtol=0, atol=1e-14)
    one = rng.standard_normal((1, 128))
    np.testing.assert_allclose(O.attention_head(one, one, v[:1]), v[:1], atol=1e-15)
    p = O.attention_probs(rng.standard_normal((4, 128)), k)
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-14)


def test_attention_permutation_equivariance(rng):
    S, H = 20, 3
    q, k, v = (rand_bf16(rng, (S, H, 128)) for _ in range(3))
    perm = rng.permutation(S)
    o = O.attention(q, k, v)
    op = O.attention(q[perm], k[perm], v[perm])
    np.testing.assert_array_equal(op, o[perm])


def test_attention_probe_h8_causal_mask(rng):
    S = 16
    q, k, v = (rng.standard_normal((S, 128)) for _ in range(3))
    good = O.attention_head(q, k, v)
    s = q @ k.T / math.sqrt(128)
    s[np.triu_indices(S, 1)] = -np.inf
    p = np.exp(s - s.max(1, keepdims=True))
    causal = (p / p.sum(1, keepdims=True)) @ v
    assert np.abs(causal - good).max() > 0.1


# ---------------------------------------------------------------------------
# gated residual and SwiGLU
# ---------------------------------------------------------------------------

def test_gated_residual(rng):
    x = rand_bf16(rng, (4, 8))
    y = rand_bf16(rng, (4, 8))
    np.testing.assert_array_equal(O.gated_residual(x, np.zeros((4, 8)), y), x)
    assert O.gated_residual(np.array([1.0]), np.array([0.5]), np.array([2.0]))[0] == 2.0
    assert O.gated_residual(np.array([1.0]), np.array([-0.25]), np.array([8.0]))[0] == -1.0


def test_swiglu_order_and_values():
    assert O.swiglu(np.array([0.0]), np.array([5.0]))[0] == 0.0
    a = O.swiglu(np.array([2.0]), np.array([3.0]))[0]
    assert a == O.bf16_round(3.0 * 2.0 / (1.0 + math.exp(-2.0)))
    assert a != O.swiglu(np.array([3.0]), np.array([2.0]))[0]


# ---------------------------------------------------------------------------
# the whole block
# ---------------------------------------------------------------------------

def _tiny_block(seed=0, S=None):
    import h3_inputs as hi
    wl = hi.WORKLOADS["tiny72"]
    meta, acts, wts = hi.workload_inputs(wl, seed=seed)
    to = lambda t: None if t is None else (t.to(torch.float64).numpy())
    w = {k: to(v) for k, v in wts.items()}
    m = {k: v.numpy() for k, v in meta.items()}
    return to(acts["x"]), m, to(acts["t_cond"]), w


def test_block_permutation_equivariance_and_probe_h1(rng):
    x, m, tc, w = _tiny_block()
    S = x.shape[0]
    ref = O.block_forward(x, m["token_tag"], m["timestep_index"], m["pos_thw"], tc, w)["y"]
    perm = rng.permutation(S)
    out = O.block_forward(x[perm], m["token_tag"][perm], m["timestep_index"][perm],
                          m["pos_thw"][perm], tc, w)["y"]
    np.testing.assert_array_equal(out, ref[perm])
    # probe H1: one metadata tensor left unpermuted.  The first drift is at the
    # first MM-RoPE use (positions) or AdaLN use (tags): check q after RoPE and h1.
    full = O.block_forward(x, m["token_tag"], m["timestep_index"], m["pos_thw"], tc, w)
    bad = O.block_forward(x[perm], m["token_tag"][perm], m["timestep_index"][perm],
                          m["pos_thw"], tc, w)
    q_ref = full["q"][perm]
    assert np.mean(np.abs(bad["q"] - q_ref)) / np.sqrt(np.mean(q_ref ** 2)) > 0.1
    bad = O.block_forward(x[perm], m["token_tag"], m["timestep_index"][perm],
                          m["pos_thw"][perm], tc, w)
    h_ref = full["h1"][perm]
    assert np.mean(np.abs(bad["h1"] - h_ref)) / np.sqrt(np.mean(h_ref ** 2)) > 0.1


def test_block_zero_gates_is_identity():
    x, m, tc, w = _tiny_block()
    D = x.shape[1]
    w = dict(w)
    w_ada = w["w_ada"].copy().reshape(3, 6, D, -1)
    b_ada = w["b_ada"].copy().reshape(3, 6, D)
    for c in (O.CHUNK_GATE_MSA, O.CHUNK_GATE_MLP):
        w_ada[:, c] = 0.0
        b_ada[:, c] = 0.0
    w["w_ada"], w["b_ada"] = w_ada.reshape(18 * D, -1), b_ada.reshape(-1)
    out = O.block_forward(x, m["token_tag"], m["timestep_index"], m["pos_thw"], tc, w)
    np.testing.assert_array_equal(out["y"], x)


def test_block_rows_subset_and_determinism(rng):
    x, m, tc, w = _tiny_block()
    args = (x, m["token_tag"], m["timestep_index"], m["pos_thw"], tc, w)
    full = O.block_forward(*args)
    again = O.block_forward(*args)
    np.testing.assert_array_equal(full["y"], again["y"])       # control H-C0
    rows = np.array([0, 5, 8, 31, 71])
    part = O.block_forward(*args, rows=rows)
    np.testing.assert_array_equal(part["y"], full["y"][rows])


def test_block_chain_two_blocks():
    x, m, tc, w = _tiny_block()
    y1 = O.block_forward(x, m["token_tag"], m["timestep_index"], m["pos_thw"], tc, w)["y"]
    y2 = O.block_forward(y1, m["token_tag"], m["timestep_index"], m["pos_thw"], tc, w)["y"]
    np.testing.assert_array_equal(
        O.blocks_forward(x, m["token_tag"], m["timestep_index"], m["pos_thw"], tc, [w, w]), y2)


def test_qk_norm_rope_composition(rng):
    S, H = 6, 2
    qkv = rand_bf16(rng, (S, H, 3, 128), 2.0)
    pos = rng.integers(0, 9, (S, 3))
    gq, gk = rand_bf16(rng, (128,), 0.1) + 1, rand_bf16(rng, (128,), 0.1) + 1
    q, k, v = O.qk_norm_rope(qkv, pos, gq, gk)
    np.testing.assert_array_equal(q, O.mm_rope(O.head_rmsnorm(qkv[:, :, 0], gq), pos))
    np.testing.assert_array_equal(k, O.mm_rope(O.head_rmsnorm(qkv[:, :, 1], gk), pos))
    np.testing.assert_array_equal(v, qkv[:, :, 2])


def test_attention_probs_brute_force(rng):
    S = 5
    q, k = rng.standard_normal((2, 128)), rng.standard_normal((S, 128))
    p = O.attention_probs(q, k)
    for i in range(2):
        e = [math.exp(sum(q[i, c] * k[j, c] for c in range(128)) / math.sqrt(128)) for j in range(S)]
        for j in range(S):
            assert abs(p[i, j] - e[j] / sum(e)) < 1e-14


# ---------------------------------------------------------------- token refiner

def _refiner_case(S=11, D=64, H=2, F=96, seed=21):
    rng = np.random.default_rng(seed)
    b = lambda a: O.bf16_round(a)
    w = {"norm1_g": b(1 + 0.1 * rng.standard_normal(D)), "norm2_g": b(1 + 0.1 * rng.standard_normal(D)),
         "w_qkv": b(0.1 * rng.standard_normal((3 * H * 128, D))), "q_norm_g": b(1 + 0.1 * rng.standard_normal(128)),
         "k_norm_g": b(1 + 0.1 * rng.standard_normal(128)), "w_o": b(0.05 * rng.standard_normal((D, H * 128))),
         "w_fc1": b(0.1 * rng.standard_normal((2 * F, D))), "w_fc2": b(0.1 * rng.standard_normal((D, F)))}
    x = b(rng.standard_normal((S, D)))
    return x, w


def test_refiner_equals_block_with_identity_modulation_and_zero_positions():
    # the same arithmetic as the block: shift = scale = 0, gates = 1, RoPE at position 0
    x, w = _refiner_case()
    S, D = x.shape
    C = 8
    wb = dict(w, w_ada=np.zeros((18 * D, C)),
              b_ada=np.tile(np.repeat(np.array([0, 0, 1, 0, 0, 1], float), D), 3))
    ref = O.block_forward(x, np.ones(S, np.int32), np.zeros(S, np.int32), np.zeros((S, 3), np.int32),
                          np.zeros((1, C)), wb)["y"]
    np.testing.assert_array_equal(O.refiner_block_forward(x, w)["y"], ref)


def test_refiner_permutation_equivariant_and_residual_identity():
    x, w = _refiner_case()
    y = O.refiner_forward(x, [w, w], w["norm2_g"])
    perm = np.random.default_rng(2).permutation(x.shape[0])
    np.testing.assert_allclose(O.refiner_forward(x[perm], [w, w], w["norm2_g"]), y[perm], rtol=0, atol=1e-12)
    w0 = dict(w, w_o=np.zeros_like(w["w_o"]), w_fc2=np.zeros_like(w["w_fc2"]))
    np.testing.assert_array_equal(O.refiner_block_forward(x, w0)["y"], x)      # zero sublayers: y = x
    ones = O.refiner_forward(x, [], np.ones(x.shape[1]))
    np.testing.assert_allclose(np.sqrt(np.mean(ones ** 2, axis=1)), 1.0, rtol=1e-2)   # final norm: unit RMS
