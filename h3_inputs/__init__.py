"""Seeded synthetic inputs for the MiniMax-H3 Omni-Transformer block.

This module only *draws* inputs: shapes, packed-row structure and random
values.  It holds none of the block's arithmetic, and both the CUDA path and
the CPU oracle consume what it produces, so neither side depends on the other.

Workload shapes follow the block fingerprint of the MiniMax-H3 model (RL-Kernel
RFC "MiniMax-H3 WS1/WS2 kernel roadmap", section 2, "Omni-Transformer
fingerprint" table): residual width 5376, 56 heads of 128, FFN 14336, AdaLN
conditioning width 2688.  The packed layout is text, video and audio rows with
explicit tags (video=0, text=1, audio=2) and per-row timestep indices (same
table, rows "AdaLN modalities" and "AdaLN conditioning").  The pages give no
positions for the synthetic shapes; the rule used here is: text rows at
(0,0,0), video rows enumerate their latent (t,h,w) grid t-major then h then w,
audio rows at (i,0,0).

Random values (all seeded, one generator per tensor):
  * weights ~ N(0, 0.02) rounded to bf16, no projection biases except the
    AdaLN one, b_ada ~ N(0, 0.02) in bf16;
  * RMSNorm gains 1 + N(0, 0.1) in bf16 (block norms and the Q/K norms);
  * activations x ~ N(0, 1) in bf16;
  * timestep conditioning t_cond ~ N(0, 1) in fp32 (pre-SiLU);
  * timestep indices uniform in [0, T).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import torch

TAG_VIDEO, TAG_TEXT, TAG_AUDIO = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class BlockShape:
    """Model widths of one Omni-Transformer block."""
    dim: int          # residual width D
    n_heads: int      # H
    head_dim: int     # d (128 for H3)
    ffn_dim: int      # F (SwiGLU hidden width)
    cond_dim: int     # C (timestep embedding width fed to the AdaLN projection)

    @property
    def inner(self) -> int:
        return self.n_heads * self.head_dim


@dataclasses.dataclass(frozen=True)
class PackedLayout:
    """One packed document: contiguous text, video and audio segments."""
    n_text: int
    video_grid: Tuple[int, int, int]   # latent (t, h, w) grid of the video rows
    n_audio: int

    @property
    def n_video(self) -> int:
        t, h, w = self.video_grid
        return t * h * w

    @property
    def n_rows(self) -> int:
        return self.n_text + self.n_video + self.n_audio


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: BlockShape
    layout: PackedLayout
    n_timesteps: int
    n_blocks: int = 1
    description: str = ""


H3_SHAPE = BlockShape(dim=5376, n_heads=56, head_dim=128, ffn_dim=14336, cond_dim=2688)
TINY_SHAPE = BlockShape(dim=512, n_heads=4, head_dim=128, ffn_dim=1536, cond_dim=256)

WORKLOADS: Dict[str, Workload] = {
    "tiny72": Workload(
        "tiny72", TINY_SHAPE, PackedLayout(8, (3, 4, 4), 16), n_timesteps=4,
        description="H3-shaped tiny block, D=512, 4 heads, 72 packed rows"),
    "block505": Workload(
        "block505", H3_SHAPE, PackedLayout(17, (6, 6, 10), 128), n_timesteps=12,
        description="one full-width H3 block, 505 packed rows, 12 timestep rows"),
    "block1824": Workload(
        "block1824", H3_SHAPE, PackedLayout(32, (6, 16, 16), 256), n_timesteps=12,
        description="one full-width H3 block at the 512x512 22-frame shape, 1824 rows"),
    "denoiser15860": Workload(
        "denoiser15860", H3_SHAPE, PackedLayout(256, (36, 15, 27), 1024), n_timesteps=1,
        n_blocks=50,
        description="50-block denoiser forward at the 864x480 141-frame shape, 15860 rows"),
    "input15860": Workload(
        "input15860", H3_SHAPE, PackedLayout(256, (36, 15, 27), 1024), n_timesteps=1, n_blocks=0,
        description="input side of one evaluation at the 15860-row shape: video patch packing "
                    "(24 x 36 x 30 x 54 latent), FP32 video/audio input projections into the packed "
                    "stream, BF16 text projection 5120 -> 5376, timestep sinusoid and FP32 MLP"),
    "refiner256": Workload(
        "refiner256", H3_SHAPE, PackedLayout(256, (0, 0, 0), 0), n_timesteps=1, n_blocks=2,
        description="2-layer token refiner plus final RMSNorm over 256 projected text rows"),
    "output15860": Workload(
        "output15860", H3_SHAPE, PackedLayout(256, (36, 15, 27), 1024), n_timesteps=1, n_blocks=0,
        description="output side of one evaluation at the 15860-row shape: row selection, FP32 final "
                    "AdaLN of both modalities, FP32 heads (14580 x 96, 1024 x 32), both Euler steps"),
    "attn4096": Workload(
        "attn4096", H3_SHAPE, PackedLayout(86, (9, 20, 20), 410), n_timesteps=1,
        description="attention core alone, 4096 packed rows"),
    "attn16384": Workload(
        "attn16384", H3_SHAPE, PackedLayout(346, (16, 30, 30), 1638), n_timesteps=1,
        description="attention core alone, 16384 packed rows"),
    "attn32768": Workload(
        "attn32768", H3_SHAPE, PackedLayout(691, (32, 30, 30), 3277), n_timesteps=1,
        description="attention core alone, 32768 packed rows"),
}


def custom_workload(shape: BlockShape, n_text: int, video_grid: Tuple[int, int, int],
                    n_audio: int, n_timesteps: int, name: str = "custom") -> Workload:
    return Workload(name, shape, PackedLayout(n_text, tuple(video_grid), n_audio), n_timesteps)


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

def _generator(seed: int, tensor_id: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tensor_id * 7919 + 12345) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal(shape: Sequence[int], std: float, mean: float, seed: int, tensor_id: int,
           device: str = "cpu", dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """N(mean, std^2) drawn in fp32, then rounded once to `dtype`."""
    g = _generator(seed, tensor_id, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def packed_metadata(layout: PackedLayout, n_timesteps: int, seed: int = 0,
                    device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Row tags, timestep indices and (t,h,w) positions for one packed document."""
    tags: List[int] = [TAG_TEXT] * layout.n_text + [TAG_VIDEO] * layout.n_video + \
        [TAG_AUDIO] * layout.n_audio
    pos: List[Tuple[int, int, int]] = [(0, 0, 0)] * layout.n_text
    gt, gh, gw = layout.video_grid
    for t in range(gt):
        for h in range(gh):
            for w in range(gw):
                pos.append((t, h, w))
    pos += [(i, 0, 0) for i in range(layout.n_audio)]
    g = _generator(seed, 3, "cpu")
    tidx = torch.randint(0, n_timesteps, (layout.n_rows,), generator=g, dtype=torch.int64)
    return {
        "token_tag": torch.tensor(tags, dtype=torch.int32, device=device),
        "timestep_index": tidx.to(torch.int32).to(device),
        "pos_thw": torch.tensor(pos, dtype=torch.int32, device=device).reshape(-1, 3),
    }


def block_weights(shape: BlockShape, seed: int = 0, block: int = 0,
                  device: str = "cpu") -> Dict[str, Optional[torch.Tensor]]:
    """Random-init bf16 weights of one block.

    Layouts (row-major, weights are [out][in]):
      w_ada  [18*D][C]      b_ada [18*D]
      norm1_g, norm2_g [D]
      w_qkv  [H*3*128][D]   per-head interleaved rows: head h owns rows
                            h*384 .. h*384+383 as q(128), k(128), v(128)
      q_norm_g, k_norm_g [128]
      w_o    [D][H*128]
      w_fc1  [2F][D]        gate rows first, then the value ("up") rows
      w_fc2  [D][F]
    """
    D, C, F, I = shape.dim, shape.cond_dim, shape.ffn_dim, shape.inner
    base = 100 + 32 * block
    n = lambda shp, std, mean, k: normal(shp, std, mean, seed, base + k, device)
    return {
        "w_ada": n((18 * D, C), 0.02, 0.0, 0),
        "b_ada": n((18 * D,), 0.02, 0.0, 1),
        "norm1_g": n((D,), 0.1, 1.0, 2),
        "norm2_g": n((D,), 0.1, 1.0, 3),
        "w_qkv": n((3 * I, D), 0.02, 0.0, 4),
        "b_qkv": None,
        "q_norm_g": n((shape.head_dim,), 0.1, 1.0, 5),
        "k_norm_g": n((shape.head_dim,), 0.1, 1.0, 6),
        "w_o": n((D, I), 0.02, 0.0, 7),
        "b_o": None,
        "w_fc1": n((2 * F, D), 0.02, 0.0, 8),
        "b_fc1": None,
        "w_fc2": n((D, F), 0.02, 0.0, 9),
        "b_fc2": None,
    }


def activations(shape: BlockShape, n_rows: int, n_timesteps: int, seed: int = 0,
                device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Packed residual rows x [S][D] bf16 and the timestep conditioning [T][C] fp32."""
    return {
        "x": normal((n_rows, shape.dim), 1.0, 0.0, seed, 1, device),
        "t_cond": normal((n_timesteps, shape.cond_dim), 1.0, 0.0, seed, 2, device,
                         dtype=torch.float32),
    }


def attention_inputs(shape: BlockShape, n_rows: int, seed: int = 0,
                     device: str = "cpu") -> Dict[str, torch.Tensor]:
    """q, k, v ~ N(0,1) in bf16 packed as one [S][H][3][128] buffer (per-head q|k|v),
    plus the Q/K norm gains, for the attention-core workloads."""
    H, d = shape.n_heads, shape.head_dim
    return {
        "qkv": normal((n_rows, H, 3, d), 1.0, 0.0, seed, 20, device),
        "q_norm_g": normal((d,), 0.1, 1.0, seed, 21, device),
        "k_norm_g": normal((d,), 0.1, 1.0, seed, 22, device),
    }


VIDEO_PATCH, AUDIO_PATCH = 96, 32   # latent channels per video / audio row


def output_weights(shape: BlockShape, seed: int = 0, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Random-init FP32 weights of the final layer: per modality (video, audio)
    a final AdaLN projection w_fin [2*D][C] (shift rows, then scale rows) with
    bias b_fin [2*D], and a head w_head [P][D] with bias b_head [P]
    (P = 96 video, 32 audio); all ~N(0, 0.02) in fp32."""
    D, C = shape.dim, shape.cond_dim
    n = lambda shp, k: normal(shp, 0.02, 0.0, seed, 60 + k, device, dtype=torch.float32)
    return {
        "w_fin_video": n((2 * D, C), 0), "b_fin_video": n((2 * D,), 1),
        "w_fin_audio": n((2 * D, C), 2), "b_fin_audio": n((2 * D,), 3),
        "w_head_video": n((VIDEO_PATCH, D), 4), "b_head_video": n((VIDEO_PATCH,), 5),
        "w_head_audio": n((AUDIO_PATCH, D), 6), "b_head_audio": n((AUDIO_PATCH,), 7),
    }


def input_weights(shape: BlockShape, seed: int = 0, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Random-init FP32 weights of the input side, all ~N(0, 0.02): the video
    and audio input projections w_in_video [D][96], w_in_audio [D][32] with
    biases [D], and the timestep MLP w_t1 [D][256], b_t1 [D], w_t2 [C][D],
    b_t2 [C]."""
    D, C = shape.dim, shape.cond_dim
    n = lambda shp, k: normal(shp, 0.02, 0.0, seed, 80 + k, device, dtype=torch.float32)
    return {
        "w_in_video": n((D, VIDEO_PATCH), 0), "b_in_video": n((D,), 1),
        "w_in_audio": n((D, AUDIO_PATCH), 2), "b_in_audio": n((D,), 3),
        "w_t1": n((D, 256), 4), "b_t1": n((D,), 5),
        "w_t2": n((C, D), 6), "b_t2": n((C,), 7),
    }


def latents(n_rows: int, width: int, seed: int = 0, tensor_id: int = 70,
            device: str = "cpu") -> torch.Tensor:
    """Patch-packed fp32 latent rows [n_rows][width] ~N(0, 1) (noisy latents,
    velocities or noise for the sampler)."""
    return normal((n_rows, width), 1.0, 0.0, seed, tensor_id, device, dtype=torch.float32)


def workload_inputs(w: Workload, seed: int = 0, device: str = "cpu", block: int = 0):
    """Everything one block forward of workload `w` consumes."""
    meta = packed_metadata(w.layout, w.n_timesteps, seed, device)
    acts = activations(w.shape, w.layout.n_rows, w.n_timesteps, seed, device)
    wts = block_weights(w.shape, seed, block, device)
    return meta, acts, wts
