"""Pins of the single-precision evaluation (oracle/h3_oracle_fp32.py), which
sets the floor of the end-to-end bounds.  It is checked against things other
than itself: torch's fp32 -> bf16 conversion (a library routine), closed
forms, and the fp64 oracle stage by stage on the tiny block (two independent
codings of one definition must agree to within the per-operator bound; a
transposed operand, a wrong chunk, a sign or a dropped term in either would
not)."""
import numpy as np
import pytest
import torch

import h3_inputs as hi
from oracle import h3_oracle as O
from oracle import h3_oracle_fp32 as O32
from h3_testutil import MAX_E, MEAN_E, assert_close

f32 = np.float32


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000).astype(f32) * f32(3.0),
        (rng.standard_normal(2000) * 1e-39).astype(f32),            # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38, 1.0 + 2.0 ** -8,
                  1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20], dtype=f32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = O32.bf16(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.isnan(O32.bf16(np.array([np.nan], f32)))[0]


def test_closed_forms():
    c = f32(3.0)
    row = np.full((1, 64), c, f32)
    assert O32.inv_rms(row)[0, 0] == pytest.approx(1.0 / np.sqrt(9.0 + 1e-5), rel=1e-6)
    assert O32.silu(np.zeros(4, f32)).tolist() == [0.0] * 4
    # RoPE is the identity at position zero and leaves channels 96..127 alone
    x = O32.bf16(np.random.default_rng(1).standard_normal((5, 2, 128)).astype(f32))
    out = O32.rope(x, np.zeros((5, 3), np.int32))
    assert np.array_equal(out, x)
    out = O32.rope(x, np.array([[1, 2, 3]] * 5, np.int32))
    assert np.array_equal(out[..., 96:], x[..., 96:])
    # pair j=0 (t band, frequency 1) turns by exactly 1 rad at t = 1
    x1 = np.zeros((1, 1, 128), f32)
    x1[0, 0, 0] = 1.0
    r = O32.rope(x1, np.array([[1, 0, 0]], np.int32))
    assert r[0, 0, 0] == O32.bf16(np.cos(f32(1)))[()] and r[0, 0, 48] == O32.bf16(np.sin(f32(1)))[()]
    # attention over one key returns its value row
    q = np.random.default_rng(2).standard_normal((1, 1, 128)).astype(f32)
    v = O32.bf16(np.random.default_rng(3).standard_normal((1, 1, 128)).astype(f32))
    assert np.array_equal(O32.attention(q, q, v, np.arange(1)), v.reshape(1, 128))


def _tiny():
    w = hi.WORKLOADS["tiny72"]
    meta, acts, wts = hi.workload_inputs(w)
    f64 = lambda t: None if t is None else t.to(torch.float64).numpy()
    return (w, meta, f64(acts["x"]), acts["t_cond"].numpy(), {k: f64(v) for k, v in wts.items()})


def test_stages_agree_with_fp64_oracle_on_tiny_block():
    w, meta, x, tc, wts = _tiny()
    tag, tidx, pos = meta["token_tag"].numpy(), meta["timestep_index"].numpy(), meta["pos_thw"].numpy()
    w32 = {k: (v.astype(f32) if v is not None else None) for k, v in wts.items()}
    D = w.shape.dim
    ref = O.block_forward(x, tag, tidx, pos, tc.astype(np.float64), wts)
    # each stage fed the fp64 oracle's own input of that stage
    tab = O32.adaln_table(tc, w32["w_ada"], w32["b_ada"], D)
    assert_close(tab, ref["table"], "fp32 AdaLN table")
    mod = ref["table"][ref["rows"]].astype(f32)
    assert_close(O32.norm_mod(x.astype(f32), w32["norm1_g"], mod[:, 0], mod[:, 1]), ref["h1"], "fp32 norm1")
    qkv = ref["qkv"].astype(f32)
    q = O32.rope(O32.head_norm(qkv[:, :, 0], w32["q_norm_g"]), pos)
    k = O32.rope(O32.head_norm(qkv[:, :, 1], w32["k_norm_g"]), pos)
    assert_close(q, ref["q"], "fp32 q")
    assert_close(k, ref["k"], "fp32 k")
    o = O32.attention(ref["q"].astype(f32), ref["k"].astype(f32), ref["v"].astype(f32), np.arange(x.shape[0]))
    assert_close(o, ref["o"], "fp32 attention")
    assert_close(O32.bf16(O32.mm(ref["o"], w32["w_o"])), ref["attn"], "fp32 O projection")
    y = O32.block_forward(x, tag, tidx, pos, tc, w32)
    assert_close(y, ref["y"], "fp32 block output", MAX_E, MEAN_E)
    # the sampled-rows path is the same block
    rows = np.array([0, 7, 8, 40, 71])
    assert np.array_equal(O32.block_forward(x, tag, tidx, pos, tc, w32, rows=rows), y[rows])


def test_zero_gates_give_the_input_back():
    w, meta, x, tc, wts = _tiny()
    w32 = {k: (v.astype(f32) if v is not None else None) for k, v in wts.items()}
    D = w.shape.dim
    w32["w_ada"] = w32["w_ada"].copy()
    w32["b_ada"] = w32["b_ada"].copy()
    for m in range(3):
        for chunk in (2, 5):
            lo = (m * 6 + chunk) * D
            w32["w_ada"][lo:lo + D] = 0.0
            w32["b_ada"][lo:lo + D] = 0.0
    y = O32.block_forward(x, meta["token_tag"].numpy(), meta["timestep_index"].numpy(), meta["pos_thw"].numpy(),
                          tc, w32)
    assert np.array_equal(y, x.astype(f32))


def test_refiner_agrees_with_fp64_oracle_on_tiny_shape():
    shape = hi.TINY_SHAPE
    wts = [hi.block_weights(shape, 0, b) for b in (7, 8)]
    g = hi.normal((shape.dim,), 0.1, 1.0, 0, 90).to(torch.float64).numpy()
    x = hi.normal((37, shape.dim), 1.0, 0.0, 0, 91).to(torch.float64).numpy()
    w64 = [{k: (v.to(torch.float64).numpy() if v is not None else None) for k, v in w.items()} for w in wts]
    ref = O.refiner_forward(x, w64, g)
    got = O32.refiner_forward(x.astype(f32), [{k: (v.astype(f32) if v is not None else None)
                                               for k, v in w.items()} for w in w64], g.astype(f32))
    assert_close(got, ref, "fp32 refiner", MAX_E, MEAN_E)
