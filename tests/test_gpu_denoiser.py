"""Full-size block workloads: the denoiser (15,860 packed rows: 256 text +
14,580 video on a 36x15x27 grid + 1,024 audio; one timestep row) and the
1824-row block.

* Block 0 at full size against the oracle on sampled rows: the oracle computes
  the AdaLN table, norm1 and q/k/v for every row (keys and values of the
  whole document), then attention and the rest of the block for the sampled
  query rows only.
* The 50-block chain (about 64.5 GB of bf16 weights generated on the device):
  bitwise repeatable (control H-C0), finite, bounded; run piecewise it equals
  the one-call chain bit for bit; blocks 25 and 49, each fed the GPU's own
  input to it, against the oracle on sampled rows.
* A 50-block chain of tiny blocks with distinct weights against the oracle's
  chain end to end, and block by block on the GPU's own inputs.
"""
import os
import sys

import numpy as np
import pytest
import torch

import h3_inputs as hi
from oracle import h3_oracle as O
from h3_testutil import (CHAIN_MAX_E, CHAIN_MEAN_E, TINY50_CHAIN_MAX_E, TINY50_CHAIN_MEAN_E, assert_close,
                         errors, to_np)

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
import make_chain_floors  # noqa: E402

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
    # at this length the residual GEMMs run whole tiles and share the k-blocks
    # of their last waves out over every pair (the sampled rows include rows
    # of those tiles: the last row tiles, all columns)
    info = h3.h3_last_kernel_info()
    assert "stream-k=0" not in info and "sk-whole-tiles=-1" not in info, info
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


@pytest.fixture(scope="module")
def denoiser(h3):
    """The 50-block evaluation's inputs on the device (about 64.5 GB of bf16
    weights, generated there)."""
    shape, S, T = W.shape, W.layout.n_rows, W.n_timesteps
    meta = hi.packed_metadata(W.layout, T, 0, device="cuda")
    acts = hi.activations(shape, S, T, 0, device="cuda")
    wts = [hi.block_weights(shape, 0, b, device="cuda") for b in range(W.n_blocks)]
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    ws = torch.empty(h3.h3_blocks_workspace_bytes(cfg, W.n_blocks, S, T), dtype=torch.uint8, device="cuda")
    cw = [h3.make_weights(w) for w in wts]
    m = _meta(h3, meta, acts["t_cond"])
    yield {"meta": meta, "acts": acts, "wts": wts, "cfg": cfg, "ws": ws, "cw": cw, "m": m}
    del wts, cw
    torch.cuda.empty_cache()


def test_denoiser_chain_repeatable(h3, denoiser):
    d = denoiser
    y1 = torch.empty_like(d["acts"]["x"])
    y2 = torch.empty_like(d["acts"]["x"])
    h3.h3_blocks_forward(d["cfg"], d["cw"], d["m"], d["acts"]["x"], y1, d["ws"])
    assert h3.h3_sync_check(timeout_ms=120000) == 0
    h3.h3_blocks_forward(d["cfg"], d["cw"], d["m"], d["acts"]["x"], y2, d["ws"])
    assert h3.h3_sync_check(timeout_ms=120000) == 0
    assert torch.equal(y1, y2)
    yf = y1.float()
    assert torch.isfinite(yf).all()
    rms = yf.pow(2).mean().sqrt().item()
    print(f"50-block chain output RMS {rms:.3f}")
    assert 0.1 < rms < 1e4
    d["y50"] = y1


def _sampled_rows(seed):
    S, lay = W.layout.n_rows, W.layout
    return np.unique(np.concatenate([
        [0, lay.n_text - 1, lay.n_text, S - lay.n_audio, S - 1],
        np.linspace(lay.n_text, lay.n_text + lay.n_video - 1, 24).astype(int),
        np.random.default_rng(seed).integers(0, S, 16)]))


def test_denoiser_blocks_25_and_49_on_gpu_inputs(h3, denoiser):
    """Blocks 25 and 49 of the 50-block evaluation, each fed the GPU's own bf16
    input to that block (the output of the blocks before it), against the
    oracle on sampled rows (keys and values over all 15,860 rows).  The chain
    is also run piecewise (blocks 0-24, 25, 26-48, 49) and must equal the
    one-call 50-block evaluation bit for bit: no block is skipped, repeated or
    given another block's weights."""
    d = denoiser
    cfg, ws, cw, m, x = d["cfg"], d["ws"], d["cw"], d["m"], d["acts"]["x"]
    x25, y25 = torch.empty_like(x), torch.empty_like(x)
    x49, y49 = torch.empty_like(x), torch.empty_like(x)
    h3.h3_blocks_forward(cfg, cw[:25], m, x, x25, ws)
    h3.h3_block_forward(cfg, cw[25], m, x25, y25, ws)
    h3.h3_blocks_forward(cfg, cw[26:49], m, y25, x49, ws)
    h3.h3_block_forward(cfg, cw[49], m, x49, y49, ws)
    assert h3.h3_sync_check(timeout_ms=120000) == 0
    y50 = d.get("y50")
    if y50 is None:
        y50 = torch.empty_like(x)
        h3.h3_blocks_forward(cfg, cw, m, x, y50, ws)
        assert h3.h3_sync_check(timeout_ms=120000) == 0
    assert torch.equal(y49, y50)
    meta = {k: v.cpu().numpy() for k, v in d["meta"].items()}
    tc = d["acts"]["t_cond"].cpu().numpy().astype(np.float64)
    for b, xin, yout, seed in ((25, x25, y25, 11), (49, x49, y49, 12)):
        rows = _sampled_rows(seed)
        w64 = {k: (to_np(v) if v is not None else None) for k, v in d["wts"][b].items()}
        ref = O.block_forward(to_np(xin), meta["token_tag"], meta["timestep_index"], meta["pos_thw"], tc, w64,
                              rows=rows)
        got = to_np(yout)[rows]
        mx, mn = errors(got, ref["y"])
        print(f"denoiser block {b} on the GPU's input, {rows.size} sampled rows: max_e={mx:.4f} mean_e={mn:.5f}")
        assert_close(got, ref["y"], f"denoiser block {b} (sampled rows)", CHAIN_MAX_E, CHAIN_MEAN_E)
        del w64, ref


def test_tiny_chain_50_blocks(h3):
    """50 tiny H3-shaped blocks (D 512, 4 heads, 72 packed rows), each with its
    own weights, through h3_blocks_forward: the output against the oracle's
    50-block chain (bound: twice the stored fp32-vs-fp64 floor of this chain),
    and every block, fed the GPU's own input to it, against the oracle block at
    the per-operator bound."""
    w, meta, acts, wts = make_chain_floors.tiny_chain_inputs(50)
    shape, S, T = w.shape, w.layout.n_rows, w.n_timesteps
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    d_w = [{k: (v.cuda() if v is not None else None) for k, v in ww.items()} for ww in wts]
    cw = [h3.make_weights(dw) for dw in d_w]
    meta_d = {k: v.cuda() for k, v in meta.items()}
    tc = acts["t_cond"].cuda()
    m = h3.make_meta(meta_d["token_tag"], meta_d["timestep_index"], meta_d["pos_thw"], tc, T)
    ws = torch.empty(h3.h3_blocks_workspace_bytes(cfg, 50, S, T), dtype=torch.uint8, device="cuda")
    x = acts["x"].cuda()
    y = torch.empty_like(x)
    h3.h3_blocks_forward(cfg, cw, m, x, y, ws)
    assert h3.h3_sync_check() == 0
    xs = [x]
    for b in range(50):
        yb = torch.empty_like(x)
        h3.h3_block_forward(cfg, cw[b], m, xs[-1], yb, ws)
        xs.append(yb)
    assert h3.h3_sync_check() == 0
    assert torch.equal(xs[-1], y)
    args = (meta["token_tag"].numpy(), meta["timestep_index"].numpy(), meta["pos_thw"].numpy(),
            acts["t_cond"].numpy().astype(np.float64))
    w64 = [{k: (to_np(v) if v is not None else None) for k, v in ww.items()} for ww in wts]
    ref = O.blocks_forward(to_np(acts["x"]), *args, w64)
    mx, mn = errors(to_np(y), ref)
    print(f"tiny 50-block chain end to end: max_e={mx:.4f} mean_e={mn:.5f}")
    assert_close(to_np(y), ref, "tiny 50-block chain", TINY50_CHAIN_MAX_E, TINY50_CHAIN_MEAN_E)
    worst = (0.0, 0.0)
    for b in range(50):
        rb = O.block_forward(to_np(xs[b]), *args, w64[b])["y"]
        e = assert_close(to_np(xs[b + 1]), rb, f"tiny chain block {b} on the GPU's input")
        worst = (max(worst[0], e[0]), max(worst[1], e[1]))
    print(f"tiny chain, worst block on its GPU input: max_e={worst[0]:.4f} mean_e={worst[1]:.6f}")
