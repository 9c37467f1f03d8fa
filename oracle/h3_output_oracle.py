"""CPU oracle for the H3 output side and sampler arithmetic.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  The CUDA product path never calls it
and shares no code with it.

What it covers, after the 50-block stack: the final AdaLN of the video and
audio rows, the FP32 output heads with row selection, the two shifted sigma
grids, the data-ward Euler update, and the conditioning noise mix.

Sources (web pages; each function names the passage it follows):
  [RFC]  RL-Kernel RFC "[MiniMax-H3][CUDA/ROCm] WS1/WS2 kernel roadmap, ablation
         matrix and integration plan": section 2 ("Mixed-precision
         fingerprint" and "Scheduler fingerprint" tables), section 4
         ("H3-specific arithmetic rules"), section 5 (work items
         final_adaln_out, video/audio_output_projection_fp32,
         packed_index_select, h3_sigma_schedule, h3_ode_step,
         conditioning_noise_mix), section 6.2 (probes H9-H15).
  [LEDGER] "H3 Parity Evidence Ledger": "Current Runtime Scope" (the H3 final
         layer row: final AdaLN, target-row modulation, video/audio patch rows).
  [METAL] "h3-metal" README: "Sampler and DiT controls" (terminal zero after
         the last pass); the final-head paragraphs (per-modality final AdaLN
         over the modality's rows of the residual stream, FP32 heads as the
         close reference).

Precision.  The pages fix the scheduler arithmetic as FP32, so the sampler
functions compute in numpy float32 with one rounding per written operation,
in the written order (no fused multiply-add).  The FP32 modules of the final
layer (SiLU/projection, RMSNorm, heads) are evaluated in float64 and rounded
to float32 once where the module hands a tensor on.

Readings taken where the pages are silent (each is one argument or constant):
  O1 sigma grid: n_points values of linspace(1, 0, n_points), each the float64
     value 1 - i/(n_points-1) rounded once to float32; the shift
     s*sigma / (1 + (s-1)*sigma) in float32 with num = s*sigma,
     den = 1 + (s-1)*sigma, sigma' = num/den; a terminal zero appended;
     consecutive equal float32 values collapsed.  The linspace ends at zero,
     so the terminal zero collapses with it: n_points sigmas, n_points - 1
     model evaluations.
  O2 Euler update as written: x0 = xt + sigma*v, r = sigma_next/sigma,
     x_next = r*xt + (1-r)*x0, each operation rounded to float32 in turn.
  O3 final layer per modality m in {video, audio}: a table fp32(SiLU(t_cond)
     W_m^T + b_m) of rows [shift | scale] (2*D wide, the block AdaLN's
     shift-before-scale order); a row of modality m at timestep index t uses
     row t of table m; plain RMSNorm without a gain (eps 1e-5) of the bf16
     residual row, then norm*(1 + scale) + shift, then the FP32 head
     (P = 96 video, 32 audio) with bias, on the modality's rows in packed order.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

EPS = 1e-5
VIDEO_SHIFT = 12.0     # RFC s2 scheduler fingerprint, default video shift
AUDIO_SHIFT = 3.0      # RFC s2 scheduler fingerprint, default audio shift
TAG_VIDEO, TAG_TEXT, TAG_AUDIO = 0, 1, 2
VIDEO_PATCH = 96       # RFC s5 video_output_projection_fp32: 5376 -> 96
AUDIO_PATCH = 32       # RFC s5 audio_output_projection_fp32: 5376 -> 32

f32 = np.float32


# ---------------------------------------------------------------------------
# sampler (RFC s2 scheduler fingerprint; s5 h3_sigma_schedule, h3_ode_step,
# conditioning_noise_mix; probes H9-H13, H15)
# ---------------------------------------------------------------------------

def shift_sigma(sigma, shift: float) -> np.ndarray:
    """The sigma transform of the scheduler table, s*sigma / (1 + (s-1)*sigma),
    in float32 with one rounding per operation (reading O1)."""
    sg = np.asarray(sigma, dtype=f32)
    s = f32(shift)
    num = (s * sg).astype(f32)
    den = (f32(1.0) + ((s - f32(1.0)).astype(f32) * sg).astype(f32)).astype(f32)
    return (num / den).astype(f32)


def sigma_grid(n_points: int, shift: float) -> np.ndarray:
    """Shifted linspace(1, 0, n_points) with a terminal zero and consecutive
    float32 duplicates collapsed (scheduler table rows "Sigma transform" and
    "Grid"; work item h3_sigma_schedule; reading O1)."""
    if n_points < 2:
        raise ValueError("the grid needs at least its two end points")
    base = np.array([1.0 - i / (n_points - 1) for i in range(n_points)], dtype=np.float64).astype(f32)
    shifted = np.concatenate([shift_sigma(base, shift), np.zeros(1, dtype=f32)])
    keep = [0]
    for i in range(1, shifted.size):
        if shifted[i] != shifted[keep[-1]]:
            keep.append(i)
    return shifted[keep]


def timesteps(sigmas) -> np.ndarray:
    """Timestep convention t = 1 - sigma (t = 1 clean), float32 (scheduler
    table row "Timestep convention"; probe H10)."""
    return (f32(1.0) - np.asarray(sigmas, dtype=f32)).astype(f32)


def ode_step(xt: np.ndarray, v: np.ndarray, sigma: float, sigma_next: float) -> np.ndarray:
    """Data-ward denoised estimate x0 = xt + sigma*v, then the Euler blend
    x_next = r*xt + (1-r)*x0 with r = sigma_next/sigma, all in float32 in the
    written order (scheduler table rows "Velocity convention", "Euler update";
    work item h3_ode_step; probes H9, H13; reading O2)."""
    xt = np.asarray(xt, dtype=f32)
    v = np.asarray(v, dtype=f32)
    sg, sn = f32(sigma), f32(sigma_next)
    x0 = (xt + (sg * v).astype(f32)).astype(f32)
    r = (sn / sg).astype(f32)
    one_m_r = (f32(1.0) - r).astype(f32)
    return ((r * xt).astype(f32) + (one_m_r * x0).astype(f32)).astype(f32)


def noise_mix(x0: np.ndarray, noise: np.ndarray, t: float) -> np.ndarray:
    """Conditioning-anchor augmentation t*x0 + (1-t)*noise in float32 as
    written (work item conditioning_noise_mix; probe H15)."""
    x0 = np.asarray(x0, dtype=f32)
    noise = np.asarray(noise, dtype=f32)
    tt = f32(t)
    one_m_t = (f32(1.0) - tt).astype(f32)
    return ((tt * x0).astype(f32) + (one_m_t * noise).astype(f32)).astype(f32)


# ---------------------------------------------------------------------------
# output side (RFC s5 packed_index_select, final_adaln_out,
# video/audio_output_projection_fp32; ledger "H3 final layer"; probe H14)
# ---------------------------------------------------------------------------

def select_rows(token_tag: np.ndarray, tag: int) -> np.ndarray:
    """Packed-row indices of one modality in packed order (work item
    packed_index_select: deterministic video/audio row selection)."""
    return np.array([i for i, g in enumerate(np.asarray(token_tag)) if int(g) == tag], dtype=np.int32)


def silu64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def final_adaln_table(t_cond: np.ndarray, w_fin: np.ndarray, b_fin: Optional[np.ndarray]) -> np.ndarray:
    """FP32 SiLU/projection shift-scale table of one modality's final AdaLN:
    [T][2][D] float32, chunk 0 shift, chunk 1 scale (work item
    final_adaln_out; mixed-precision table: output path FP32; reading O3)."""
    u = silu64(t_cond)                                       # [T][C]
    m = u @ np.asarray(w_fin, dtype=np.float64).T            # [T][2D]
    if b_fin is not None:
        m = m + np.asarray(b_fin, dtype=np.float64)[None, :]
    T, D2 = m.shape
    return m.reshape(T, 2, D2 // 2).astype(f32)


def final_norm_modulate(x_rows: np.ndarray, shift: np.ndarray, scale: np.ndarray,
                        eps: float = EPS) -> np.ndarray:
    """Plain RMSNorm of each residual row (no gain, eps inside the root) then
    norm*(1 + scale) + shift, float64 (ledger "H3 final layer": final AdaLN
    and target-row modulation; RFC s5 h3_rmsnorm; reading O3)."""
    x = np.asarray(x_rows, dtype=np.float64)
    inv = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    n = x * inv
    return n * (1.0 + np.asarray(scale, dtype=np.float64)) + np.asarray(shift, dtype=np.float64)


def output_head(x: np.ndarray, token_tag: np.ndarray, timestep_index: np.ndarray, tag: int,
                table: np.ndarray, w_head: np.ndarray, b_head: Optional[np.ndarray],
                rows: Optional[np.ndarray] = None, eps: float = EPS) -> np.ndarray:
    """Velocity rows of one modality: select the modality's rows in packed
    order, final AdaLN with the row's timestep entry of the modality table,
    then the FP32 head [P][D] with bias; float64 (work items
    video/audio_output_projection_fp32, packed_index_select; reading O3).
    `rows` restricts the result to positions of the selected list."""
    sel = select_rows(token_tag, tag)
    if rows is not None:
        sel = sel[np.asarray(rows)]
    ti = np.asarray(timestep_index)[sel]
    tab = np.asarray(table, dtype=np.float64)
    m = final_norm_modulate(np.asarray(x)[sel], tab[ti, 0], tab[ti, 1], eps)
    y = m @ np.asarray(w_head, dtype=np.float64).T
    if b_head is not None:
        y = y + np.asarray(b_head, dtype=np.float64)[None, :]
    return y
