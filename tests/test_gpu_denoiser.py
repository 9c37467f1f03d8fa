"""Full-size block workloads: the denoiser (15,860 packed rows: 256 text +
14,580 video on a 36x15x27 grid + 1,024 audio; one timestep row) and the
1824-row block.

* Block 0 at full size against the oracle on sampled rows: the oracle computes
  the AdaLN table, norm1 and q/k/v for every row (keys and values of the
  whole document), then attention and the rest of the block for the sampled
  query rows only.
* The 50-block chain (about 64.5 GB of bf16 weights generated on the device):
  bitwise repeatable (control H-C0), finite, bounded.
"""
import numpy as np
import pytest
import torch

import h3_inputs as hi
from oracle import h3_oracle as O
from h3_testutil import CHAIN_MAX_E, CHAIN_MEAN_E, assert_close, errors, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

W = hi.WORKLOADS["denoiser15860"]


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available()
    import audio_video_flow_gb300 as m
    m.lib()
    return m


def _meta(h3, meta_d, tc):
    return h3.make_meta(meta_d["token_tag"], meta_d["timestep_index"], meta_d["pos_thw"], tc, W.n_timesteps)


def test_denoiser_block0_sampled_rows(h3):
    meta, acts, wts = hi.workload_inputs(W)          # CPU, block 0
    S = W.layout.n_rows
    lay = W.layout
    rows = np.unique(np.concatenate([
        [0, 1, lay.n_text - 1, lay.n_text, lay.n_text + 1],
        np.linspace(lay.n_text, lay.n_text + lay.n_video - 1, 40).astype(int),
        [S - lay.n_audio, S - lay.n_audio + 1, S - 2, S - 1],
        np.random.default_rng(7).integers(0, S, 16)]))
    f64 = lambda t: to_np(t)
    ref = O.block_forward(f64(acts["x"]), meta["token_tag"].numpy(), meta["timestep_index"].numpy(),
                          meta["pos_thw"].numpy(), acts["t_cond"].numpy().astype(np.float64),
                          {k: (f64(v) if v is not None else None) for k, v in wts.items()}, rows=rows)
    shape = W.shape
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    d_w = {k: (v.cuda() if v is not None else None) for k, v in wts.items()}
    meta_d = {k: v.cuda() for k, v in meta.items()}
    x = acts["x"].cuda()
    tc = acts["t_cond"].cuda()
    ws = torch.empty(h3.h3_block_workspace_bytes(cfg, S, W.n_timesteps), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    h3.h3_block_forward(cfg, h3.make_weights(d_w), _meta(h3, meta_d, tc), x, y, ws)
    assert h3.h3_sync_check(timeout_ms=60000) == 0
    got = to_np(y)[rows]
    mx, mn = errors(got, ref["y"])
    print(f"denoiser block 0, {rows.size} sampled rows: max_e={mx:.4f} mean_e={mn:.5f}")
    assert_close(got, ref["y"], "denoiser block 0 (sampled rows)", CHAIN_MAX_E, CHAIN_MEAN_E)


def test_block1824_sampled_rows(h3):
    """The 1824-row block (32 text + 1536 video on a 6x16x16 grid + 256 audio,
    12 timestep rows) at full size, the bench's launch configuration (stream-K
    O and FC2), against the oracle on sampled rows."""
    w = hi.WORKLOADS["block1824"]
    meta, acts, wts = hi.workload_inputs(w)
    S, lay = w.layout.n_rows, w.layout
    rows = np.unique(np.concatenate([
        [0, lay.n_text - 1, lay.n_text, S - lay.n_audio, S - 1],
        np.linspace(lay.n_text, lay.n_text + lay.n_video - 1, 24).astype(int),
        np.random.default_rng(8).integers(0, S, 16)]))
    f64 = lambda t: to_np(t)
    ref = O.block_forward(f64(acts["x"]), meta["token_tag"].numpy(), meta["timestep_index"].numpy(),
                          meta["pos_thw"].numpy(), acts["t_cond"].numpy().astype(np.float64),
                          {k: (f64(v) if v is not None else None) for k, v in wts.items()}, rows=rows)
    shape = w.shape
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    d_w = {k: (v.cuda() if v is not None else None) for k, v in wts.items()}
    meta_d = {k: v.cuda() for k, v in meta.items()}
    x, tc = acts["x"].cuda(), acts["t_cond"].cuda()
    ws = torch.empty(h3.h3_block_workspace_bytes(cfg, S, w.n_timesteps), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    m = h3.make_meta(meta_d["token_tag"], meta_d["timestep_index"], meta_d["pos_thw"], tc, w.n_timesteps)
    h3.h3_block_forward(cfg, h3.make_weights(d_w), m, x, y, ws)
    assert h3.h3_sync_check(timeout_ms=60000) == 0
    assert "stream-k=0" not in h3.h3_last_kernel_info()
    got = to_np(y)[rows]
    mx, mn = errors(got, ref["y"])
    print(f"block1824, {rows.size} sampled rows: max_e={mx:.4f} mean_e={mn:.5f}")
    assert_close(got, ref["y"], "block1824 (sampled rows)", CHAIN_MAX_E, CHAIN_MEAN_E)


def test_denoiser_chain_repeatable(h3):
    shape, S, T = W.shape, W.layout.n_rows, W.n_timesteps
    meta = hi.packed_metadata(W.layout, T, 0, device="cuda")
    acts = hi.activations(shape, S, T, 0, device="cuda")
    wts = [hi.block_weights(shape, 0, b, device="cuda") for b in range(W.n_blocks)]
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    ws = torch.empty(h3.h3_block_workspace_bytes(cfg, S, T), dtype=torch.uint8, device="cuda")
    cw = [h3.make_weights(w) for w in wts]
    m = _meta(h3, meta, acts["t_cond"])
    y1 = torch.empty_like(acts["x"])
    y2 = torch.empty_like(acts["x"])
    h3.h3_blocks_forward(cfg, cw, m, acts["x"], y1, ws)
    assert h3.h3_sync_check(timeout_ms=120000) == 0
    h3.h3_blocks_forward(cfg, cw, m, acts["x"], y2, ws)
    assert h3.h3_sync_check(timeout_ms=120000) == 0
    assert torch.equal(y1, y2)
    yf = y1.float()
    assert torch.isfinite(yf).all()
    rms = yf.pow(2).mean().sqrt().item()
    print(f"50-block chain output RMS {rms:.3f}")
    assert 0.1 < rms < 1e4
