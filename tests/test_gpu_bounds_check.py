"""The bounds-checked build on the GPU (the stand-in for a memory checker,
which is not available on the test machines): libh3_bounds.so is compiled
with H3_BOUNDS_CHECK=1, so every checked global access of the kernels first
tests that it lies inside the buffer its call's arguments describe and
reports H3_ERR_BOUNDS instead of touching memory outside it.

A child process loads that build (H3_LIBRARY=bounds; one CUDA runtime per
process) and runs the small and odd shapes: blocks of 1, 7, 72, 129 and 205
packed rows, the full-width 505-row block (stream-K residual GEMMs, the
side-stream AdaLN table), a three-block chain with its tables computed up
front, the standalone Q/K norm + RoPE, attention with its LSE, and a plain
projection.  Every call must end with H3_OK, and every output must equal
the normal build's bit for bit (the checks change no arithmetic).

Run as a script (`python tests/test_gpu_bounds_check.py --cases OUT.npz`)
it is that child: it runs the cases with whichever library H3_LIBRARY
selects and saves the outputs.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import h3_inputs as hi  # noqa: E402

pytestmark = pytest.mark.gpu

TINY = hi.TINY_SHAPE
RAGGED = hi.BlockShape(dim=640, n_heads=3, head_dim=128, ffn_dim=1024, cond_dim=192)
D576 = hi.BlockShape(dim=576, n_heads=2, head_dim=128, ffn_dim=512, cond_dim=128)
BLOCKS = {
    "S1": hi.custom_workload(TINY, 1, (0, 0, 0), 0, 1),
    "S7": hi.custom_workload(TINY, 2, (1, 1, 3), 2, 3),
    "S72": hi.WORKLOADS["tiny72"],
    "S129": hi.custom_workload(TINY, 5, (2, 4, 8), 60, 3),
    "S205": hi.custom_workload(RAGGED, 13, (2, 5, 9), 102, 7),
    "S505": hi.WORKLOADS["block505"],
}


def _block(h3, w, nb=1):
    shape, S, T = w.shape, w.layout.n_rows, w.n_timesteps
    meta = {k: v.cuda() for k, v in hi.packed_metadata(w.layout, T, 0).items()}
    acts = hi.activations(shape, S, T, 0)
    wts = [{k: (v.cuda() if v is not None else None) for k, v in hi.block_weights(shape, 0, b).items()}
           for b in range(nb)]
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    m = h3.make_meta(meta["token_tag"], meta["timestep_index"], meta["pos_thw"], acts["t_cond"].cuda(), T)
    ws = torch.empty(h3.h3_blocks_workspace_bytes(cfg, nb, S, T), dtype=torch.uint8, device="cuda")
    x = acts["x"].cuda()
    y = torch.empty_like(x)
    cw = [h3.make_weights(d) for d in wts]
    if nb == 1:
        h3.h3_block_forward(cfg, cw[0], m, x, y, ws)
    else:
        h3.h3_blocks_forward(cfg, cw, m, x, y, ws)
    return y


def run_cases(h3):
    """Outputs of every case, with the status after each call."""
    out, status = {}, {}

    def done(name, t):
        torch.cuda.synchronize()
        status[name] = h3.h3_sync_check(timeout_ms=60000)
        out[name] = t.detach().float().cpu().numpy()

    for name, w in BLOCKS.items():
        done(name, _block(h3, w))
    chain = hi.custom_workload(D576, 5, (2, 3, 4), 11, 3)
    done("chain3_d576", _block(h3, chain, nb=3))
    # standalone Q/K norm + RoPE and attention (with LSE) on the ragged shape
    S, H = 205, 3
    g = torch.Generator().manual_seed(11)
    qkv = torch.randn(S, H, 3, 128, generator=g).to(torch.bfloat16).cuda()
    pos = hi.packed_metadata(BLOCKS["S205"].layout, 1, 0)["pos_thw"].cuda()
    qg = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16).cuda()
    kg = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16).cuda()
    cfg = h3.make_config(RAGGED.dim, H, RAGGED.ffn_dim, RAGGED.cond_dim)
    h3.h3_rope_qknorm(cfg, S, pos, qkv[:, :, 0], qkv[:, :, 1], H * 384, 384, qg, kg)
    done("rope205", qkv)
    o = torch.empty(S, H * 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(H, S, dtype=torch.float32, device="cuda")
    h3.h3_attention(S, H, qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2], H * 384, 384, o, lse)
    done("attention205", o)
    out["lse205"] = lse.cpu().numpy()
    x = torch.randn(200, 320, generator=g).to(torch.bfloat16).cuda()
    wl = (0.05 * torch.randn(264, 320, generator=g)).to(torch.bfloat16).cuda()
    bl = (0.1 * torch.randn(264, generator=g)).to(torch.bfloat16).cuda()
    y = torch.empty(200, 264, dtype=torch.bfloat16, device="cuda")
    h3.h3_linear(200, 264, 320, x, wl, bl, y)
    done("linear200", y)
    return out, status


def test_bounds_checked_build_matches_and_reports_nothing(tmp_path):
    assert torch.cuda.is_available()
    from audio_video_flow_gb300 import _build
    _build.build(bounds=True)
    dst = tmp_path / "bounds.npz"
    env = dict(os.environ, H3_LIBRARY="bounds")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cases", str(dst)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    got = dict(np.load(dst))
    import audio_video_flow_gb300 as h3
    assert os.path.basename(h3.LIB_PATH) == "libh3.so"
    h3.lib()
    ref, status = run_cases(h3)
    assert all(s == 0 for s in status.values()), status
    for k, v in ref.items():
        assert k in got, k
        assert np.array_equal(got[k], v, equal_nan=True), f"{k}: bounds-checked build differs"


def _child(dst):
    import audio_video_flow_gb300 as h3
    assert os.path.basename(h3.LIB_PATH) == "libh3_bounds.so"
    h3.lib()
    out, status = run_cases(h3)
    bad = {k: (v, h3.status_string(v)) for k, v in status.items() if v != 0}
    if bad:
        print("bounds-checked build reported:", bad, h3.h3_last_error_site())
        sys.exit(3)
    np.savez(dst, **out)


if __name__ == "__main__":
    if len(sys.argv) == 3 and sys.argv[1] == "--cases":
        _child(sys.argv[2])
