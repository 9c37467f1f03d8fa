"""Single-precision evaluation of the MiniMax-H3 block, for the end-to-end floor.

TEST INFRASTRUCTURE.  Only the tests and the script that writes the stored
floors (tests/golden/make_chain_floors.py) may import this module.  The CUDA
product path never calls it and shares no code with it.

What it is for.  The fp64 oracle (h3_oracle.py) defines the block: bf16
rounding at each declared cast point, every sum in double precision.  A
correct implementation that accumulates in fp32 (as any tensor-core kernel
does) rounds some elements to the neighbouring bf16 value at those cast
points, and the block carries those flips forward (the SwiGLU FFN amplifies
them).  How far two correct evaluations drift apart end to end is therefore
a property of the definition and the inputs, not of a kernel.  This module
is a second, independent evaluation of the same definition with every
product and sum in fp32; its distance from the fp64 oracle is the floor the
end-to-end tests scale their bounds from.

It is written from the same passages as the fp64 oracle, without importing
it:
  [RFC] RL-Kernel RFC "[MiniMax-H3][CUDA/ROCm] WS1/WS2 kernel roadmap,
        ablation matrix and integration plan": section 2 (Omni-Transformer
        fingerprint and mixed-precision tables), section 4 (H3-specific
        arithmetic rules), section 5 (work items adaln_projection_3mod ..
        h3_ffn_down_gemm, token_refiner_block).
and takes the same readings where the pages are silent: AdaLN table rows
t*3+m with chunks shift/scale/gate for attention then MLP; modulation
n*(1+scale)+shift; per-channel norm gains; one [128] gain each for Q and K;
split-half MM-RoPE on channels 0..95 with bands t, h, w of 16 frequencies
10000^(-i/16); two bf16 casts on Q/K (after the norm, after the rotation);
softmax scale 1/sqrt(128) without a mask; FC1 gate rows first; the token
refiner is the block without modulation, RoPE or residual gates, followed by
a final RMSNorm.

Every array here is numpy float32.  Matrix products are numpy's float32
matmul (a library primitive; it accumulates in fp32).  Reductions use
numpy's float32 sums.  bf16 rounding is done on the fp32 bit pattern.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

f32 = np.float32
EPS = 1e-5
HEAD_DIM = 128
ROPE_FREQS = 16          # per axis
ROPE_HALF = 48           # 3 axes x 16 frequencies: channel j pairs with j + 48


def bf16(x) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) and return them as
    fp32: add 0x7FFF plus the lowest kept bit to the bit pattern and clear the
    16 dropped bits.  NaN stays NaN; values beyond the bf16 range become inf."""
    x = np.ascontiguousarray(x, dtype=f32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return np.where(np.isnan(x), x, r.view(f32))


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x) = x / (1 + e^-x), in fp32."""
    x = np.asarray(x, f32)
    return x / (f32(1) + np.exp(-x))


def inv_rms(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    """1 / sqrt(mean(x^2) + eps) over the last axis, fp32 sums ([RFC] s2,
    row "Block norm")."""
    x = np.asarray(x, f32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=f32)
    return (f32(1) / np.sqrt(ms + f32(eps))).astype(f32)


def mm(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """a @ w^T in fp32 (weights are [out][in])."""
    return np.asarray(a, f32) @ np.asarray(w, f32).T


def adaln_table(t_cond: np.ndarray, w_ada: np.ndarray, b_ada: Optional[np.ndarray], dim: int) -> np.ndarray:
    """[3T][6][D] table: bf16(bf16(SiLU(t_cond)) W_ada^T + b_ada) ([RFC] s2
    "AdaLN projection", s4: only the SiLU result is cast before the
    projection)."""
    u = bf16(silu(t_cond))
    m = mm(u, w_ada)
    if b_ada is not None:
        m = m + np.asarray(b_ada, f32)[None, :]
    return bf16(m).reshape(-1, 6, dim)


def norm_mod(x: np.ndarray, g: np.ndarray, shift: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """bf16(x * inv_rms(x) * g * (1 + scale) + shift)."""
    n = np.asarray(x, f32) * inv_rms(x) * np.asarray(g, f32)[None, :]
    return bf16(n * (f32(1) + scale) + shift)


def head_norm(v: np.ndarray, g: np.ndarray) -> np.ndarray:
    """Per-head RMSNorm over the last 128 channels, one shared gain, then
    bf16 ([RFC] s2 "Q/K preprocessing")."""
    return bf16(np.asarray(v, f32) * inv_rms(v) * np.asarray(g, f32))


def rope(xh: np.ndarray, pos_thw: np.ndarray) -> np.ndarray:
    """Split-half rotation of channels 0..95 of [S][H][128]; angle of band a,
    frequency i: fp32(pos[a]) * fp32(10000^(-i/16)), all in fp32 ([RFC] s2
    "Position encoding", "RoPE frequencies", "Rotary channels")."""
    om = (10000.0 ** (-np.arange(ROPE_FREQS, dtype=np.float64) / ROPE_FREQS)).astype(f32)
    p = np.asarray(pos_thw).astype(f32)
    ang = (p[:, :, None] * om[None, None, :]).reshape(p.shape[0], ROPE_HALF)
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    out = np.array(xh, dtype=f32, copy=True)
    a = out[..., :ROPE_HALF].copy()
    b = out[..., ROPE_HALF:2 * ROPE_HALF].copy()
    out[..., :ROPE_HALF] = bf16(a * c - b * s)
    out[..., ROPE_HALF:2 * ROPE_HALF] = bf16(b * c + a * s)
    return out


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Unmasked softmax attention per head in fp32 for query rows `rows`;
    bf16 output [R][H*128] ([RFC] s2 "Attention", s4)."""
    R, H = len(rows), q.shape[1]
    out = np.empty((R, H, HEAD_DIM), f32)
    sc = f32(1.0 / np.sqrt(HEAD_DIM))
    for h in range(H):
        s = (q[rows, h] @ k[:, h].T) * sc
        s = s - s.max(axis=-1, keepdims=True)
        e = np.exp(s)
        out[:, h] = (e / e.sum(axis=-1, keepdims=True, dtype=f32)) @ v[:, h]
    return bf16(out.reshape(R, H * HEAD_DIM))


def block_forward(x, token_tag, timestep_index, pos_thw, t_cond, w: Dict[str, Optional[np.ndarray]],
                  rows: Optional[np.ndarray] = None) -> np.ndarray:
    """One block in fp32 ([RFC] s5 work items in order); returns y for
    `rows` (all rows by default; keys and values always use every row)."""
    x = np.asarray(x, f32)
    S, D = x.shape
    tab = adaln_table(np.asarray(t_cond, f32), w["w_ada"], w.get("b_ada"), D)
    mod = tab[np.asarray(timestep_index, np.int64) * 3 + np.asarray(token_tag, np.int64)]
    h1 = norm_mod(x, w["norm1_g"], mod[:, 0], mod[:, 1])
    qkv = bf16(mm(h1, w["w_qkv"]) + (0 if w.get("b_qkv") is None else np.asarray(w["b_qkv"], f32)))
    H = qkv.shape[1] // (3 * HEAD_DIM)
    qkv = qkv.reshape(S, H, 3, HEAD_DIM)
    q = rope(head_norm(qkv[:, :, 0], w["q_norm_g"]), pos_thw)
    k = rope(head_norm(qkv[:, :, 1], w["k_norm_g"]), pos_thw)
    v = qkv[:, :, 2]
    sel = np.arange(S) if rows is None else np.asarray(rows)
    o = attention(q, k, v, sel)
    m = mod[sel]
    x1 = bf16(x[sel] + m[:, 2] * bf16(mm(o, w["w_o"])))
    h2 = norm_mod(x1, w["norm2_g"], m[:, 3], m[:, 4])
    gu = bf16(mm(h2, w["w_fc1"]))
    F = gu.shape[1] // 2
    a = bf16(silu(gu[:, :F]) * gu[:, F:])
    return bf16(x1 + m[:, 5] * bf16(mm(a, w["w_fc2"])))


def blocks_forward(x, token_tag, timestep_index, pos_thw, t_cond, weights_list) -> np.ndarray:
    """Blocks in order, each block's output the next one's input."""
    x = np.asarray(x, f32)
    for w in weights_list:
        x = block_forward(x, token_tag, timestep_index, pos_thw, t_cond, w)
    return x


def refiner_block_forward(x: np.ndarray, w: Dict[str, Optional[np.ndarray]]) -> np.ndarray:
    """Token-refiner block: pre-norm attention and SwiGLU FFN without
    modulation, RoPE or gates ([RFC] s5 token_refiner_block)."""
    x = np.asarray(x, f32)
    S = x.shape[0]
    h1 = bf16(x * inv_rms(x) * np.asarray(w["norm1_g"], f32)[None, :])
    qkv = bf16(mm(h1, w["w_qkv"])).reshape(S, -1, 3, HEAD_DIM)
    q = head_norm(qkv[:, :, 0], w["q_norm_g"])
    k = head_norm(qkv[:, :, 1], w["k_norm_g"])
    o = attention(q, k, qkv[:, :, 2], np.arange(S))
    x1 = bf16(x + bf16(mm(o, w["w_o"])))
    h2 = bf16(x1 * inv_rms(x1) * np.asarray(w["norm2_g"], f32)[None, :])
    gu = bf16(mm(h2, w["w_fc1"]))
    F = gu.shape[1] // 2
    return bf16(x1 + bf16(mm(bf16(silu(gu[:, :F]) * gu[:, F:]), w["w_fc2"])))


def refiner_forward(x: np.ndarray, weights_list, final_norm_g: np.ndarray) -> np.ndarray:
    """Refiner blocks in order, then RMSNorm with the final gain."""
    x = np.asarray(x, f32)
    for w in weights_list:
        x = refiner_block_forward(x, w)
    return bf16(x * inv_rms(x) * np.asarray(final_norm_g, f32)[None, :])
