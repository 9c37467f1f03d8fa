"""CPU oracle for the H3 input side.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  The CUDA product path never calls it
and shares no code with it.

What it covers, before the 50-block stack: packing the video latent into
patch rows and back, the FP32 video/audio input projections scattered into
the packed bf16 residual stream, the row scatter of already-projected rows,
the 256-channel timestep sinusoid and the FP32 timestep MLP that produces
the conditioning rows t_cond.

Sources (web pages; each function names the passage it follows):
  [RFC]  RL-Kernel RFC "[MiniMax-H3][CUDA/ROCm] WS1/WS2 kernel roadmap, ablation
         matrix and integration plan": section 2 ("Input, output and
         conditioning fingerprint": visual VAE latent 24 channels, video
         patch (1, 2, 2) with flattened width 96, audio latent 32 channels,
         heads 96 -> 5376 and 32 -> 5376, sinusoid width 256, timestep MLP
         256 -> 5376 -> 2688, packed layout scattered by index tensors;
         "Mixed-precision fingerprint": input projections and the timestep
         MLP are FP32 modules), section 5 (work items video_patch_pack_unpack,
         video/audio_input_projection_fp32, packed_index_copy,
         timestep_sinusoid_h3, timestep_mlp_fp32), section 6.2 (probes H1,
         H7, H10).
  [METAL] "h3-metal" README, the patch-projection paragraph: FP32 weights,
         inputs and accumulation, the tile result rounded directly to BF16
         into the packed hidden stream.

Readings taken where the pages are silent (each is one argument or constant):
  I1 patch flattening: latent [C][T][H][W] -> rows ordered (t, h/2, w/2) with t
     slowest (the order of the video positions), features ordered (c, ph, pw)
     with c slowest (the latent's own axis order, then the patch offsets).
  I2 sinusoid: 128 frequencies f_i = exp(-ln(10000) * i / 128), features
     [cos(t f_i) | sin(t f_i)], with t = 1 - sigma used as is (probe H10:
     no 0..1000 scaling).
  I3 timestep MLP: Linear(256 -> 5376), SiLU, Linear(5376 -> 2688), with
     biases, all FP32; its output is the conditioning row t_cond.
  I4 rows of the packed stream that no modality writes are zero.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from oracle.h3_oracle import bf16_round

PATCH = (1, 2, 2)         # RFC s2: transformer video patch
VIDEO_CHANNELS = 24       # RFC s2: visual VAE latent channels
SINUSOID = 256            # RFC s2: timestep sinusoid width
f32 = np.float32


def patch_pack(latent: np.ndarray) -> np.ndarray:
    """[C][T][H][W] -> [T*(H/2)*(W/2)][C*4] (work item video_patch_pack_unpack;
    reading I1)."""
    C, T, H, W = latent.shape
    pt, ph, pw = PATCH
    x = np.asarray(latent).reshape(C, T // pt, pt, H // ph, ph, W // pw, pw)
    x = x.transpose(1, 3, 5, 0, 2, 4, 6)                  # t, h, w | c, pt, ph, pw
    return x.reshape((T // pt) * (H // ph) * (W // pw), C * pt * ph * pw)


def patch_unpack(rows: np.ndarray, C: int, T: int, H: int, W: int) -> np.ndarray:
    """The exact inverse of patch_pack."""
    pt, ph, pw = PATCH
    x = np.asarray(rows).reshape(T // pt, H // ph, W // pw, C, pt, ph, pw)
    return x.transpose(3, 0, 4, 1, 5, 2, 6).reshape(C, T, H, W)


def input_projection(rows: np.ndarray, w: np.ndarray, b: Optional[np.ndarray]) -> np.ndarray:
    """FP32 module x W^T + b evaluated in float64, rounded once to bf16 (work
    items video/audio_input_projection_fp32; [METAL] patch projection)."""
    y = np.asarray(rows, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + np.asarray(b, np.float64)[None, :]
    return bf16_round(y)


def packed_index_copy(n_rows: int, width: int, parts) -> np.ndarray:
    """Zero-initialised packed stream [n_rows][width] with each part's rows
    written at its destination indices (work item packed_index_copy; RFC s2
    "Packed layout"; reading I4).  parts: iterable of (rows, dst_index)."""
    out = np.zeros((n_rows, width), np.float64)
    for rows, idx in parts:
        out[np.asarray(idx)] = rows
    return out


def timestep_sinusoid(t) -> np.ndarray:
    """[T] -> [T][256] float32 features [cos(t f) | sin(t f)] (work item
    timestep_sinusoid_h3; reading I2)."""
    t = np.asarray(t, np.float64)
    half = SINUSOID // 2
    f = np.exp(-np.log(10000.0) * np.arange(half, dtype=np.float64) / half)
    a = t[:, None] * f[None, :]
    return np.concatenate([np.cos(a), np.sin(a)], axis=1).astype(f32)


def timestep_mlp(e: np.ndarray, w1: np.ndarray, b1: Optional[np.ndarray], w2: np.ndarray,
                 b2: Optional[np.ndarray]) -> np.ndarray:
    """FP32 MLP 256 -> 5376 -> 2688 with SiLU in between, evaluated in float64
    and rounded to float32 at its output (work item timestep_mlp_fp32;
    reading I3)."""
    h = np.asarray(e, np.float64) @ np.asarray(w1, np.float64).T
    if b1 is not None:
        h = h + np.asarray(b1, np.float64)[None, :]
    h = h / (1.0 + np.exp(-h))
    y = h @ np.asarray(w2, np.float64).T
    if b2 is not None:
        y = y + np.asarray(b2, np.float64)[None, :]
    return y.astype(f32)
