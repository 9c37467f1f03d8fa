"""CPU oracle for one MiniMax-H3 Omni-Transformer block forward.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  The CUDA product path never calls it
and shares no code with it.

Plain numpy, float64 arithmetic, with a round-to-nearest-even cast to bf16 at
each declared cast point of the block.  Matrix products use numpy's float64
matmul as a library primitive; nothing is blocked, fused or reordered beyond
the definitions below.

Sources (web pages; each function names the passage it follows):
  [RFC]  RL-Kernel RFC "[MiniMax-H3][CUDA/ROCm] WS1/WS2 kernel roadmap, ablation
         matrix and integration plan": section 2 (Omni-Transformer and
         mixed-precision fingerprint tables), section 4 ("H3-specific
         arithmetic rules"), section 5 (work-item table), section 6 (ablation
         matrix, probes H1-H8, controls H-C0..H-C3).
  [METAL] "h3-metal" README: "Checkpoint layout and media pipeline" (QKV rows
         interleaved per head), "Metal 4 and TensorOps paths" (paired FC1
         gate/up tiles feeding SwiGLU).
  [LEDGER] "H3 Parity Evidence Ledger": "Current Runtime Scope" (fused Q/K
         RMSNorm followed by split-half RoPE).
  [DIST] "Distributed H3 Execution": "Partition Contract" (FC1 gate and value
         halves).

Readings taken where the pages are silent (each is one argument or constant
below):
  R1 AdaLN projection output per timestep is [3 modality][6 chunk][D], so table
     row t*3+m is a plain reshape; chunk order shift_msa, scale_msa, gate_msa,
     shift_mlp, scale_mlp, gate_mlp.
  R3 modulation is norm * (1 + scale) + shift.
  R4 block RMSNorm has a per-channel gain; eps inside the square root.
  R5 one Q gain and one K gain vector of 128, shared by all heads.
  R6 MM-RoPE: channels 0..95 rotate, 96..127 pass through; channel j pairs with
     j+48 (split half); bands j in [0,16) t, [16,32) h, [32,48) w;
     omega_i = 10000^(-i/16) rounded once to fp32; angle = fp32(pos) * omega_i
     in fp32.
  R7 two bf16 casts on Q/K: after the per-head norm and after RoPE.
  R8 softmax scale 1/sqrt(128), no mask, exact exp.
  R9 FC1 rows 0..F-1 are the gate (SiLU'd), rows F..2F-1 the value.
  R10 QKV weight rows interleaved per head as [H][q,k,v][128].
  R11 token refiner: the block without AdaLN modulation or RoPE (norm gains,
      per-head Q/K RMSNorm, SwiGLU kept), residuals without a gate, and a
      final RMSNorm with its own gain after the last refiner block.
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np

EPS = 1e-5
ROPE_THETA = 10000.0
ROPE_FREQS_PER_AXIS = 16
ROPE_CHANNELS = 96
HEAD_DIM = 128
N_CHUNKS = 6          # shift/scale/gate for the attention and MLP branches
N_MODALITIES = 3      # video=0, text=1, audio=2

CHUNK_SHIFT_MSA, CHUNK_SCALE_MSA, CHUNK_GATE_MSA = 0, 1, 2
CHUNK_SHIFT_MLP, CHUNK_SCALE_MLP, CHUNK_GATE_MLP = 3, 4, 5


# ---------------------------------------------------------------------------
# rounding
# ---------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits and fp32's exponent range: normal quantum is
    2^(e-8) for |x| in [2^(e-1), 2^e); below 2^-126 the quantum is the fixed
    subnormal step 2^-133.  Results at or beyond 2^128 overflow to infinity.
    Returned as float64 holding exactly representable bf16 values.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # |x| in [2^(e-1), 2^e)
    q_exp = np.maximum(e - 8, -133)
    scaled = np.ldexp(x, -q_exp)             # exact (power-of-two scale)
    r = np.ldexp(np.rint(scaled), q_exp)     # np.rint: round half to even
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


def fp32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32)


# ---------------------------------------------------------------------------
# AdaLN: projection and row selection
# ---------------------------------------------------------------------------

def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def adaln_table(t_cond: np.ndarray, w_ada: np.ndarray, b_ada: Optional[np.ndarray],
                dim: int) -> np.ndarray:
    """AdaLN modulation table of one block, shape [3T][6][D].

    [RFC] s2 fingerprint table, row "AdaLN projection" (2688 inputs to
    6*3*5376 outputs per block); s4 arithmetic rules: the SiLU is evaluated at
    the precision of the timestep embedding and only its result is cast to
    bf16 for the projection, so u = bf16(SiLU(t_cond)).  The projection itself
    is listed among the BF16 modules (s2 mixed-precision table), so its output
    is cast to bf16.
    Layout per timestep is [modality][chunk][D] (reading R1), i.e. table row
    t*3 + m, the "[t0m0, t0m1, t0m2, ...]" order of probe H4 (s6.2).
    """
    T = t_cond.shape[0]
    u = bf16_round(silu(t_cond))
    m = u @ np.asarray(w_ada, np.float64).T
    if b_ada is not None:
        m = m + np.asarray(b_ada, np.float64)[None, :]
    m = bf16_round(m)
    return m.reshape(T * N_MODALITIES, N_CHUNKS, dim)


def adaln_rows(token_tag: np.ndarray, timestep_index: np.ndarray) -> np.ndarray:
    """Modulation row of each packed row.

    [RFC] s2 fingerprint table, rows "AdaLN conditioning" (the row index is
    three times the timestep index plus the tag) and "AdaLN modalities" (tags
    0 video, 1 text, 2 audio); work item adaln_row_gather (s5).
    """
    return np.asarray(timestep_index, np.int64) * N_MODALITIES + np.asarray(token_tag, np.int64)


# ---------------------------------------------------------------------------
# norms and modulation
# ---------------------------------------------------------------------------

def rms_inv(x: np.ndarray, eps: float = EPS) -> np.ndarray:
    """1/sqrt(mean(x^2) + eps) over the last axis ([RFC] s2 fingerprint
    table, row "Block norm": an RMSNorm with eps 1e-5)."""
    x = np.asarray(x, np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rmsnorm_modulate(x: np.ndarray, gain: np.ndarray, shift: np.ndarray,
                     scale: np.ndarray, eps: float = EPS) -> np.ndarray:
    """h = bf16( rms(x) * g * (1 + scale) + shift ), one cast at the end.

    [RFC] s2 fingerprint table, row "Block norm"; work items h3_rmsnorm and
    adaln_row_gather (s5).  Modulation form norm*(1+scale)+shift is reading R3;
    the per-channel gain is reading R4.  shift/scale are per-row [S][D].
    """
    x = np.asarray(x, np.float64)
    n = x * rms_inv(x, eps) * np.asarray(gain, np.float64)[None, :]
    return bf16_round(n * (1.0 + np.asarray(scale, np.float64)) + np.asarray(shift, np.float64))


def head_rmsnorm(v: np.ndarray, gain: np.ndarray, eps: float = EPS) -> np.ndarray:
    """Per-head RMSNorm over the 128 head channels, cast to bf16.

    [RFC] s2 fingerprint table, row "Q/K preprocessing" (an RMSNorm per head,
    eps 1e-5); the s2 mixed-precision table puts the norm outputs on the BF16
    side, after their cast (reading R7).  v has shape [..., 128]; one gain shared across heads (R5).
    """
    v = np.asarray(v, np.float64)
    return bf16_round(v * rms_inv(v, eps) * np.asarray(gain, np.float64))


# ---------------------------------------------------------------------------
# MM-RoPE
# ---------------------------------------------------------------------------

def rope_frequencies(n_freq: int = ROPE_FREQS_PER_AXIS, theta: float = ROPE_THETA) -> np.ndarray:
    """omega_i = theta^(-i/n_freq), i = 0..n_freq-1, rounded once to fp32.

    [RFC] s2 fingerprint table, row "RoPE frequencies" (16 per axis, base
    10000); the s2 mixed-precision table lists the frequency construction as
    an FP32 path.
    """
    i = np.arange(n_freq, dtype=np.float64)
    return fp32(theta ** (-i / n_freq))


def rope_angles(pos_thw: np.ndarray, n_freq: int = ROPE_FREQS_PER_AXIS,
                theta: float = ROPE_THETA) -> np.ndarray:
    """fp32 angles [S][3*n_freq]: band a (t, h, w in that order) holds
    fp32(pos[:, a]) * omega_i computed in fp32.

    [RFC] s2 fingerprint table, row "Position encoding" (three axes, t then h
    then w); s4 arithmetic rules: the frequencies are built in FP32.
    """
    om = rope_frequencies(n_freq, theta)
    p = fp32(np.asarray(pos_thw))                                   # [S][3]
    ang = p[:, :, None] * om[None, None, :]                         # fp32 products
    return fp32(ang.reshape(p.shape[0], 3 * n_freq))


def mm_rope(xhat: np.ndarray, pos_thw: np.ndarray, n_freq: int = ROPE_FREQS_PER_AXIS,
            theta: float = ROPE_THETA) -> np.ndarray:
    """Partial three-axis rotary embedding on [S][H][128] (bf16 values in).

    [RFC] s2 fingerprint table, row "Rotary channels" (96 of the 128 head
    channels rotate, the other 32 are left as they are); s5 work item
    h3_mm_rope_3axis_partial (a rotate-half rotation); [LEDGER] names the
    pairing split-half.  Reading R6: with half = 48, channel j < 48
    pairs with j + 48 and uses angle column j:
        out_j      = x_j cos - x_{j+48} sin
        out_{j+48} = x_{j+48} cos + x_j sin
    then a bf16 cast (R7).  Channels 96..127 are returned unchanged.
    """
    xhat = np.asarray(xhat, np.float64)
    half = 3 * n_freq
    ang = rope_angles(pos_thw, n_freq, theta).astype(np.float64)    # [S][48]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    out = xhat.copy()
    x1 = xhat[..., :half]
    x2 = xhat[..., half:2 * half]
    out[..., :half] = bf16_round(x1 * c - x2 * s)
    out[..., half:2 * half] = bf16_round(x2 * c + x1 * s)
    return out


# ---------------------------------------------------------------------------
# projections, attention, residuals
# ---------------------------------------------------------------------------

def linear(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray] = None) -> np.ndarray:
    """bf16(x @ w^T + b): a BF16 projection with its declared output cast
    ([RFC] s2 mixed-precision table, BF16 column: the Q/K/V/O and FFN
    projections)."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + np.asarray(b, np.float64)[None, :]
    return bf16_round(y)


def qk_norm_rope(qkv: np.ndarray, pos_thw: np.ndarray, q_gain: np.ndarray,
                 k_gain: np.ndarray, eps: float = EPS):
    """From the projected [S][H][3][128] buffer, return (q_hat, k_hat, v).

    [RFC] s4 arithmetic rules: the Q/K norm comes first, RoPE second; v is
    not touched.
    """
    q = head_rmsnorm(qkv[:, :, 0, :], q_gain, eps)
    k = head_rmsnorm(qkv[:, :, 1, :], k_gain, eps)
    return mm_rope(q, pos_thw), mm_rope(k, pos_thw), np.asarray(qkv[:, :, 2, :], np.float64)


def attention_head(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(128)) v for one head, exact exp, no mask.

    [RFC] s2 fingerprint table, row "Attention" (bidirectional
    self-attention); s4 arithmetic rules: every packed row attends to every
    row of the document, with no causal or padding mask.  q: [R][128] query rows
    (any subset), k, v: [S][128].  Returns float64 (uncast) [R][128].
    """
    s = (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T) / math.sqrt(q.shape[-1])
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ np.asarray(v, np.float64)


def attention_probs(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """The softmax matrix of one head for the given query rows ([R][S])."""
    s = (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T) / math.sqrt(q.shape[-1])
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    return p / p.sum(axis=-1, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
              rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Multi-head attention over [S][H][128] inputs; returns bf16 o [R][H*128]
    for query rows `rows` (all rows by default)."""
    S, H, d = q.shape
    rows = np.arange(S) if rows is None else np.asarray(rows)
    out = np.empty((rows.shape[0], H, d), np.float64)
    for h in range(H):
        out[:, h, :] = attention_head(q[rows, h, :], k[:, h, :], v[:, h, :])
    return bf16_round(out.reshape(rows.shape[0], H * d))


def gated_residual(x: np.ndarray, gate: np.ndarray, y: np.ndarray) -> np.ndarray:
    """bf16(x + gate * y), in that order ([RFC] s4 arithmetic rules: the
    residual plus the row's gate times the sublayer output; s5
    adaln_gate_residual)."""
    return bf16_round(np.asarray(x, np.float64) + np.asarray(gate, np.float64) * np.asarray(y, np.float64))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """a = bf16(SiLU(g) * u) ([RFC] s2 fingerprint table, row "FFN
    activation"; s5 work item h3_swiglu, computed in FP32; gate/value order is
    reading R9)."""
    return bf16_round(silu(g) * np.asarray(u, np.float64))


# ---------------------------------------------------------------------------
# the block
# ---------------------------------------------------------------------------

def block_forward(x: np.ndarray, token_tag: np.ndarray, timestep_index: np.ndarray,
                  pos_thw: np.ndarray, t_cond: np.ndarray, w: Dict[str, Optional[np.ndarray]],
                  eps: float = EPS, rows: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """One Omni-Transformer block ([RFC] s3 figure 2, s5
    work items adaln_projection_3mod .. h3_ffn_down_gemm in that order).

    All inputs are float arrays holding bf16 values (t_cond: fp32 values),
    weights keyed as in the input generator.  Returns every intermediate so a
    comparison can localise the first drift ([RFC] s4, comparison hierarchy).  With `rows` given, every row-wise stage after attention is
    evaluated for those query rows only (keys and values still use all rows).
    """
    S, D = x.shape
    x = np.asarray(x, np.float64)
    table = adaln_table(t_cond, w["w_ada"], w.get("b_ada"), D)       # [3T][6][D]
    r = adaln_rows(token_tag, timestep_index)
    mod = table[r]                                                     # [S][6][D]

    h1 = rmsnorm_modulate(x, w["norm1_g"], mod[:, CHUNK_SHIFT_MSA], mod[:, CHUNK_SCALE_MSA], eps)
    qkv = linear(h1, w["w_qkv"], w.get("b_qkv"))                       # [S][H*3*128]
    H = qkv.shape[1] // (3 * HEAD_DIM)
    qkv = qkv.reshape(S, H, 3, HEAD_DIM)
    q, k, v = qk_norm_rope(qkv, pos_thw, w["q_norm_g"], w["k_norm_g"], eps)

    sel = np.arange(S) if rows is None else np.asarray(rows)
    o = attention(q, k, v, sel)                                        # [R][H*128]
    attn = linear(o, w["w_o"], w.get("b_o"))
    x1 = gated_residual(x[sel], mod[sel, CHUNK_GATE_MSA], attn)
    h2 = rmsnorm_modulate(x1, w["norm2_g"], mod[sel, CHUNK_SHIFT_MLP], mod[sel, CHUNK_SCALE_MLP], eps)
    gu = linear(h2, w["w_fc1"], w.get("b_fc1"))
    F = gu.shape[1] // 2
    a = swiglu(gu[:, :F], gu[:, F:])
    ffn = linear(a, w["w_fc2"], w.get("b_fc2"))
    y = gated_residual(x1, mod[sel, CHUNK_GATE_MLP], ffn)
    return {"table": table, "rows": r, "h1": h1, "qkv": qkv, "q": q, "k": k, "v": v,
            "o": o, "attn": attn, "x1": x1, "h2": h2, "gu": gu, "a": a, "ffn": ffn, "y": y}


def blocks_forward(x, token_tag, timestep_index, pos_thw, t_cond, weights_list, eps: float = EPS):
    """A chain of blocks, each with its own weights ([RFC] s2 fingerprint
    table, row "Transformer layers": 50); the output of block b is the input
    of block b+1."""
    for w in weights_list:
        x = block_forward(x, token_tag, timestep_index, pos_thw, t_cond, w, eps)["y"]
    return x


# ---------------------------------------------------------------------------
# token refiner ([RFC] s2 fingerprint rows "Text-refiner layers" 2 and "Text
# projection" 5120 -> 5376 then the 2-layer token refiner; s5 work item
# token_refiner_block: two pre-norm attention/FFN blocks without AdaLN or
# RoPE; [LEDGER] "Current Runtime Scope": the refiner ends with a final
# RMSNorm).  Reading R11: everything else is the block above - per-channel
# norm gains, per-head Q/K RMSNorm, full unmasked attention over the refined
# rows, SwiGLU - and the residuals carry no gate.
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, gain: np.ndarray, eps: float = EPS) -> np.ndarray:
    """h = bf16(rms(x) * g): the block norm without modulation."""
    x = np.asarray(x, np.float64)
    return bf16_round(x * rms_inv(x, eps) * np.asarray(gain, np.float64)[None, :])


def refiner_block_forward(x: np.ndarray, w: Dict[str, Optional[np.ndarray]], eps: float = EPS) -> Dict[str, np.ndarray]:
    """One token-refiner block: pre-norm attention then pre-norm SwiGLU FFN,
    each added back to the residual stream with one bf16 cast."""
    S = x.shape[0]
    x = np.asarray(x, np.float64)
    h1 = rmsnorm(x, w["norm1_g"], eps)
    qkv = linear(h1, w["w_qkv"], w.get("b_qkv"))
    H = qkv.shape[1] // (3 * HEAD_DIM)
    qkv = qkv.reshape(S, H, 3, HEAD_DIM)
    q = head_rmsnorm(qkv[:, :, 0, :], w["q_norm_g"], eps)
    k = head_rmsnorm(qkv[:, :, 1, :], w["k_norm_g"], eps)
    v = np.asarray(qkv[:, :, 2, :], np.float64)
    o = attention(q, k, v, np.arange(S))
    x1 = bf16_round(x + linear(o, w["w_o"], w.get("b_o")))
    h2 = rmsnorm(x1, w["norm2_g"], eps)
    gu = linear(h2, w["w_fc1"], w.get("b_fc1"))
    F = gu.shape[1] // 2
    a = swiglu(gu[:, :F], gu[:, F:])
    y = bf16_round(x1 + linear(a, w["w_fc2"], w.get("b_fc2")))
    return {"h1": h1, "q": q, "k": k, "v": v, "o": o, "x1": x1, "h2": h2, "a": a, "y": y}


def refiner_forward(x: np.ndarray, weights_list, final_norm_g: Optional[np.ndarray],
                    eps: float = EPS) -> np.ndarray:
    """The refiner blocks in order, then the final RMSNorm (skipped when no
    gain is given)."""
    for w in weights_list:
        x = refiner_block_forward(x, w, eps)["y"]
    return rmsnorm(x, final_norm_g, eps) if final_norm_g is not None else x
