"""GPU parity: every stage of the CUDA path, called through the C ABI, against
the CPU oracle on the same seeded inputs.

Per-stage tests feed each kernel the oracle's own input of that stage, so each
comparison measures one operator.  The block tests run h3_block_forward end to
end.  Sizes: the tiny H3-shaped block (72 rows: several tiles of every kernel
but one M tile), a ragged small block (205 rows, odd head count: two M tiles, a
ragged tail, a half-empty v tile), and the full-width 505-row block.
"""
import time

import numpy as np
import pytest
import torch

import h3_inputs as hi
from oracle import h3_oracle as O
from h3_testutil import (CHAIN_MAX_E, CHAIN_MEAN_E, MAX_E, MEAN_E, REFINER_CHAIN_MAX_E, REFINER_CHAIN_MEAN_E,
                         assert_close, errors, to_bf16, to_np)

pytestmark = pytest.mark.gpu

# D not a multiple of 128: the block computes the AdaLN table in one launch
# (its 128-row weight tiles straddle two chunks)
D576 = hi.custom_workload(hi.BlockShape(dim=576, n_heads=2, head_dim=128, ffn_dim=512, cond_dim=128),
                          n_text=5, video_grid=(2, 3, 4), n_audio=11, n_timesteps=3, name="d576")
RAGGED = hi.custom_workload(hi.BlockShape(dim=640, n_heads=3, head_dim=128, ffn_dim=1024, cond_dim=192),
                            n_text=13, video_grid=(2, 5, 9), n_audio=102, n_timesteps=7, name="ragged205")


@pytest.fixture(scope="session")
def h3():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import audio_video_flow_gb300 as m
    m.lib()   # raises if libh3.so is missing: no fallback path exists
    return m


class Case:
    """Inputs of one workload on the CPU (numpy, for the oracle) and on the GPU."""

    def __init__(self, w: hi.Workload, seed: int = 0, rows=None):
        self.w = w
        meta, acts, wts = hi.workload_inputs(w, seed=seed)
        self.S = w.layout.n_rows
        self.T = w.n_timesteps
        self.np_w = {k: (to_np(v) if v is not None else None) for k, v in wts.items()}
        self.np_x = to_np(acts["x"])
        self.np_tc = acts["t_cond"].numpy().astype(np.float64)
        self.np_meta = {k: v.numpy() for k, v in meta.items()}
        self.ref = O.block_forward(self.np_x, self.np_meta["token_tag"], self.np_meta["timestep_index"],
                                   self.np_meta["pos_thw"], self.np_tc, self.np_w, rows=rows)
        self.d_w = {k: (v.cuda() if v is not None else None) for k, v in wts.items()}
        self.d_x = acts["x"].cuda()
        self.d_tc = acts["t_cond"].cuda()
        self.d_meta = {k: v.cuda() for k, v in meta.items()}

    def cfg(self, h3):
        s = self.w.shape
        return h3.make_config(s.dim, s.n_heads, s.ffn_dim, s.cond_dim)

    def meta(self, h3):
        m = self.d_meta
        return h3.make_meta(m["token_tag"], m["timestep_index"], m["pos_thw"], self.d_tc, self.T)


_CASES = {}


def get_case(name):
    if name not in _CASES:
        w = {"ragged205": RAGGED, "d576": D576}.get(name) or hi.WORKLOADS[name]
        _CASES[name] = Case(w)
    return _CASES[name]


CASE_NAMES = ["tiny72", "ragged205", "block505"]


def table_tensor(case):
    return to_bf16(case.ref["table"].reshape(case.T, -1))


# ---------------------------------------------------------------------------
# stages
# ---------------------------------------------------------------------------

def test_linear_plain(h3, gemm_bn):
    g = torch.Generator().manual_seed(5)
    M, N, K = 200, 264, 320
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    b = (torch.randn(N, generator=g) * 0.1).to(torch.bfloat16)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    h3.h3_linear(M, N, K, x.cuda(), w.cuda(), b.cuda(), y)
    torch.cuda.synchronize()
    assert_close(to_np(y), O.linear(to_np(x), to_np(w), to_np(b)), "linear")


@pytest.mark.parametrize("M,N,K", [(505, 2928, 320), (505, 2560, 192), (200, 4864, 128)])
def test_linear_balanced_column_tiles(h3, M, N, K):
    """Few row tiles and many columns: the columns are split into tiles of two
    widths so every CTA pair gets one tile."""
    g = torch.Generator().manual_seed(6)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    b = (torch.randn(N, generator=g) * 0.1).to(torch.bfloat16)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    h3.h3_linear(M, N, K, x.cuda(), w.cuda(), b.cuda(), y)
    torch.cuda.synchronize()
    info = h3.h3_last_kernel_info()
    assert "balanced:" in info, info
    assert_close(to_np(y), O.linear(to_np(x), to_np(w), to_np(b)), f"linear {M}x{N}x{K}")


@pytest.mark.parametrize("name", CASE_NAMES)
def test_adaln_table(h3, name):
    c = get_case(name)
    out = torch.empty(c.T, 18 * c.w.shape.dim, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(h3.h3_adaln_table_workspace_bytes(c.cfg(h3)), dtype=torch.uint8, device="cuda")
    h3.h3_adaln_table(c.cfg(h3), c.d_w["w_ada"], c.d_w["b_ada"], c.d_tc, out, ws)
    assert h3.h3_sync_check() == 0
    assert_close(to_np(out), c.ref["table"].reshape(c.T, -1), f"adaln_table[{name}]")


@pytest.mark.parametrize("name", CASE_NAMES)
@pytest.mark.parametrize("branch", [0, 1])
def test_adaln_modulate(h3, name, branch):
    c = get_case(name)
    x_np = c.np_x if branch == 0 else c.ref["x1"]
    g_key = "norm1_g" if branch == 0 else "norm2_g"
    mod = c.ref["table"][c.ref["rows"]]
    ref = O.rmsnorm_modulate(x_np, c.np_w[g_key], mod[:, 3 * branch], mod[:, 3 * branch + 1])
    h = torch.empty(c.S, c.w.shape.dim, dtype=torch.bfloat16, device="cuda")
    h3.h3_adaln_modulate(c.cfg(h3), c.meta(h3), table_tensor(c), branch, to_bf16(x_np), c.d_w[g_key], h)
    assert h3.h3_sync_check() == 0
    assert_close(to_np(h), ref, f"modulate[{name},{branch}]")


@pytest.fixture(params=["auto", "256", "192", "128"])
def gemm_bn(request, monkeypatch):
    """Every GEMM tile width: the library picks one per launch; H3_GEMM_BN forces it."""
    if request.param == "auto":
        monkeypatch.delenv("H3_GEMM_BN", raising=False)
    else:
        monkeypatch.setenv("H3_GEMM_BN", request.param)
    return request.param


@pytest.mark.parametrize("D", [512, 5376])
def test_modulate_same_bits_for_long_and_short_documents(h3, D):
    """Documents of 4096 rows and more run the norm + modulate kernel with
    128-thread CTAs (two virtual threads each), shorter ones with 256; both
    follow the same reduction tree, so a row gives the same bits in either."""
    S_long, S_short, T = 4096, 505, 3
    g = torch.Generator().manual_seed(D)
    x = torch.randn(S_long, D, generator=g).to(torch.bfloat16).cuda()
    gain = (1 + 0.1 * torch.randn(D, generator=g)).to(torch.bfloat16).cuda()
    table = (0.3 * torch.randn(3 * T, 6, D, generator=g)).to(torch.bfloat16).cuda()
    tag = torch.randint(0, 3, (S_long,), generator=g, dtype=torch.int32).cuda()
    tidx = torch.randint(0, T, (S_long,), generator=g, dtype=torch.int32).cuda()
    pos = torch.zeros(S_long, 3, dtype=torch.int32, device="cuda")
    tc = torch.zeros(T, 256, dtype=torch.float32, device="cuda")
    cfg = h3.make_config(D, 4, 1536, 256)
    outs = []
    for S in (S_long, S_short):
        m = h3.make_meta(tag[:S], tidx[:S], pos[:S], tc, T)
        h = torch.empty(S, D, dtype=torch.bfloat16, device="cuda")
        h3.h3_adaln_modulate(cfg, m, table.reshape(T, -1), 1, x[:S], gain, h)
        assert h3.h3_sync_check() == 0
        outs.append(h)
    assert torch.equal(outs[0][:S_short], outs[1])
    mod = to_np(table)[(to_np(tidx) * 3 + to_np(tag)).astype(int)]
    ref = O.rmsnorm_modulate(to_np(x), to_np(gain), mod[:, 3], mod[:, 4])
    assert_close(to_np(outs[0]), ref, f"modulate D={D} S={S_long}")


@pytest.mark.parametrize("name", CASE_NAMES)
def test_qkv_projection(h3, name, gemm_bn):
    c = get_case(name)
    H = c.w.shape.n_heads
    out = torch.zeros(c.S, H, 3, 128, dtype=torch.bfloat16, device="cuda")
    h3.h3_qkv_projection(c.cfg(h3), c.meta(h3), to_bf16(c.ref["h1"]), c.d_w["w_qkv"], None,
                         c.d_w["q_norm_g"], c.d_w["k_norm_g"], out)
    assert h3.h3_sync_check() == 0
    o = to_np(out)
    assert_close(o[:, :, 2], c.ref["v"], f"qkv.v[{name}]")
    assert_close(o[:, :, 0], c.ref["q"], f"qkv.q[{name}]")
    assert_close(o[:, :, 1], c.ref["k"], f"qkv.k[{name}]")


@pytest.mark.parametrize("name", CASE_NAMES)
def test_rope_qknorm_standalone(h3, name):
    c = get_case(name)
    H = c.w.shape.n_heads
    buf = to_bf16(c.ref["qkv"].reshape(c.S, H, 3, 128))
    h3.h3_rope_qknorm(c.cfg(h3), c.S, c.d_meta["pos_thw"], buf[:, :, 0], buf[:, :, 1], H * 384, 384,
                      c.d_w["q_norm_g"], c.d_w["k_norm_g"])
    assert h3.h3_sync_check() == 0
    o = to_np(buf)
    assert_close(o[:, :, 0], c.ref["q"], f"rope.q[{name}]")
    assert_close(o[:, :, 1], c.ref["k"], f"rope.k[{name}]")
    np.testing.assert_array_equal(o[:, :, 2], c.ref["v"])   # v untouched


@pytest.fixture(params=["auto", "1", "2"])
def attn_qtiles(request, monkeypatch):
    """Both attention kernels (one or two query tiles per CTA); H3_ATTN_QTILES forces one."""
    if request.param == "auto":
        monkeypatch.delenv("H3_ATTN_QTILES", raising=False)
    else:
        monkeypatch.setenv("H3_ATTN_QTILES", request.param)
    return request.param


@pytest.mark.parametrize("name", CASE_NAMES)
def test_attention(h3, name, attn_qtiles):
    c = get_case(name)
    H, S = c.w.shape.n_heads, c.S
    buf = torch.stack([to_bf16(c.ref["q"]), to_bf16(c.ref["k"]), to_bf16(c.ref["v"])], dim=2).contiguous()
    o = torch.empty(S, H * 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(H, S, dtype=torch.float32, device="cuda")
    h3.h3_attention(S, H, buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], H * 384, 384, o, lse)
    assert h3.h3_sync_check() == 0
    assert_close(to_np(o), c.ref["o"], f"attention[{name}]")
    # probabilities within 1e-3: P from the exported LSE vs the oracle's P
    lse_np = lse.cpu().numpy().astype(np.float64)
    rows = np.unique(np.linspace(0, S - 1, 24).astype(int))
    for h in range(H):
        q, k = c.ref["q"][rows, h], c.ref["k"][:, h]
        p_gpu = np.exp(q @ k.T / np.sqrt(128.0) - lse_np[h, rows][:, None])
        p_ref = O.attention_probs(q, k)
        assert np.abs(p_gpu - p_ref).max() <= 1e-3, f"probabilities head {h}"


@pytest.mark.parametrize("S,qtiles", [(256, "2"), (505, "2"), (505, "1"), (1824, "2")])
def test_attention_start_mode_follows_wave_count(h3, S, qtiles, monkeypatch):
    """A grid of at most one wave (CTAs <= SMs) starts in plain stream order,
    since CTAs that start early beside the kernel before them measured slower.
    A longer grid may start early.  The provenance string says which, and the
    output is bitwise repeatable either way."""
    monkeypatch.setenv("H3_ATTN_QTILES", qtiles)
    H = 56
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas = -(-S // (128 * int(qtiles))) * H
    g = torch.Generator().manual_seed(S)
    buf = torch.randn(S, H, 3, 128, generator=g).to(torch.bfloat16).cuda()
    outs = []
    for _ in range(2):
        o = torch.empty(S, H * 128, dtype=torch.bfloat16, device="cuda")
        h3.h3_attention(S, H, buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], H * 384, 384, o, None)
        assert h3.h3_sync_check() == 0
        outs.append(o)
    info = h3.h3_last_kernel_info()
    assert f"early-start={1 if ctas > sms else 0}" in info, info
    assert torch.equal(outs[0], outs[1])
    assert torch.isfinite(outs[0].float()).all()


@pytest.mark.parametrize("name", CASE_NAMES)
def test_out_projection(h3, name, gemm_bn):
    c = get_case(name)
    D = c.w.shape.dim
    x1 = torch.empty(c.S, D, dtype=torch.bfloat16, device="cuda")
    h3.h3_out_projection(c.cfg(h3), c.meta(h3), table_tensor(c), to_bf16(c.ref["o"]), c.d_w["w_o"], None,
                         c.d_x, x1)
    assert h3.h3_sync_check() == 0
    assert_close(to_np(x1), c.ref["x1"], f"out_projection[{name}]")


@pytest.mark.parametrize("name", ["ragged205", "block505"])
def test_residual_epilogue_skips_rows_with_bad_metadata(h3, name, gemm_bn):
    """The gated-residual epilogue leaves a row whose tag or timestep index is
    out of range unwritten and reports it; every other row is the one the
    good metadata give, bit for bit (256-wide tiles pass each warp's rows
    through shared memory, and the rows of a warp there are written by other
    lanes than the ones that checked them)."""
    c = get_case(name)
    D = c.w.shape.dim
    o = to_bf16(c.ref["o"])
    good = torch.empty(c.S, D, dtype=torch.bfloat16, device="cuda")
    h3.h3_out_projection(c.cfg(h3), c.meta(h3), table_tensor(c), o, c.d_w["w_o"], None, c.d_x, good)
    assert h3.h3_sync_check() == 0
    tag = c.d_meta["token_tag"].clone()
    tidx = c.d_meta["timestep_index"].clone()
    bad_rows = [3, 37, c.S - 1]
    tag[bad_rows[0]] = 7
    tidx[bad_rows[1]] = c.T
    tag[bad_rows[2]] = -1
    meta = h3.make_meta(tag, tidx, c.d_meta["pos_thw"], c.d_tc, c.T)
    y = torch.full((c.S, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    h3.h3_out_projection(c.cfg(h3), meta, table_tensor(c), o, c.d_w["w_o"], None, c.d_x, y)
    assert h3.h3_sync_check() == h3.H3_ERR_INDEX
    keep = torch.ones(c.S, dtype=torch.bool)
    keep[bad_rows] = False
    yc, gc = y.cpu(), good.cpu()
    assert torch.isnan(yc[~keep].float()).all(), "a row with bad metadata was written"
    assert torch.equal(yc[keep].view(torch.int16), gc[keep].view(torch.int16))


@pytest.mark.parametrize("name", CASE_NAMES)
def test_ffn_up_swiglu(h3, name):
    c = get_case(name)
    a = torch.empty(c.S, c.w.shape.ffn_dim, dtype=torch.bfloat16, device="cuda")
    h3.h3_ffn_up_swiglu(c.cfg(h3), c.S, to_bf16(c.ref["h2"]), c.d_w["w_fc1"], None, a)
    assert h3.h3_sync_check() == 0
    assert_close(to_np(a), c.ref["a"], f"ffn_up_swiglu[{name}]")


@pytest.mark.parametrize("name", CASE_NAMES)
def test_ffn_down_residual(h3, name, gemm_bn):
    c = get_case(name)
    y = torch.empty(c.S, c.w.shape.dim, dtype=torch.bfloat16, device="cuda")
    h3.h3_ffn_down_residual(c.cfg(h3), c.meta(h3), table_tensor(c), to_bf16(c.ref["a"]), c.d_w["w_fc2"], None,
                            to_bf16(c.ref["x1"]), y)
    assert h3.h3_sync_check() == 0
    assert_close(to_np(y), c.ref["y"], f"ffn_down_residual[{name}]")


# ---------------------------------------------------------------------------
# the block
# ---------------------------------------------------------------------------

def run_block(h3, c, x=None, meta=None, ws=None):
    cfg = c.cfg(h3)
    nbytes = h3.h3_block_workspace_bytes(cfg, c.S, c.T)
    assert nbytes > 0
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    y = torch.empty(c.S, c.w.shape.dim, dtype=torch.bfloat16, device="cuda")
    h3.h3_block_forward(cfg, h3.make_weights(c.d_w), meta or c.meta(h3), c.d_x if x is None else x, y, ws)
    assert h3.h3_sync_check() == 0
    return y


@pytest.mark.parametrize("name", ["tiny72", "ragged205", "d576"])
def test_block_forward_small(h3, name):
    c = get_case(name)
    y = run_block(h3, c)
    assert_close(to_np(y), c.ref["y"], f"block[{name}]")


def test_block_forward_505(h3):
    c = get_case("block505")
    y = run_block(h3, c)
    mx, mn = errors(to_np(y), c.ref["y"])
    print(f"block505 end-to-end: max_e={mx:.4f} mean_e={mn:.5f}")
    assert_close(to_np(y), c.ref["y"], "block505 end to end", CHAIN_MAX_E, CHAIN_MEAN_E)


@pytest.mark.parametrize("name,units", [("ragged205", 2), ("ragged205", 7), ("d576", 5), ("d576", 76),
                                        ("block505", 4), ("block505", 76), ("block505", 0)])
def test_block_forward_stream_k(h3, name, units, monkeypatch):
    """The residual GEMMs of the block with their k-blocks shared out over
    `units` CTA pairs (stream-K, units / row tiles pairs per 256-row tile):
    runs that start inside a tile hand partial accumulators to the pair
    holding the tile's first k-block, which adds them in k order.  Against
    the oracle, and bitwise repeatable.  units = 0: stream-K off (the strict
    reduction order), whole tiles only."""
    if units:
        monkeypatch.setenv("H3_GEMM_SK_UNITS", str(units))
    else:
        monkeypatch.setenv("H3_GEMM_SK", "0")
    c = get_case(name)
    y = run_block(h3, c)
    info = h3.h3_last_kernel_info()
    assert ("stream-k=0" in info) == (units == 0), info
    if name == "block505":
        assert_close(to_np(y), c.ref["y"], f"block[{name}] stream-k {units}", CHAIN_MAX_E, CHAIN_MEAN_E)
    else:
        assert_close(to_np(y), c.ref["y"], f"block[{name}] stream-k {units}")
    assert torch.equal(y, run_block(h3, c))


@pytest.mark.parametrize("name,units", [("ragged205", 2), ("d576", 2), ("block505", 5), ("block505", 10),
                                        ("block505", 76)])
def test_block_forward_stream_k_tail(h3, name, units, monkeypatch):
    """The residual GEMMs with whole tiles first and the rest shared out as
    one stream-K lane over `units` pairs (the form long documents take when
    their last wave is short, forced here on small shapes): every full wave
    but the last runs whole tiles, and the remaining tiles' k-blocks are cut
    into `units` runs whose partials are added in k order by the pair that
    holds each tile's first k-block.  Against the oracle, and bitwise
    repeatable."""
    monkeypatch.setenv("H3_GEMM_SK_TAIL", str(units))
    c = get_case(name)
    y = run_block(h3, c)
    info = h3.h3_last_kernel_info()
    D = c.w.shape.dim
    tiles = -(-c.S // 256) * -(-D // 256)
    full = tiles // units
    dp = (full - 1) * units if full > 0 else 0
    assert f"stream-k={units} " in info and f"sk-whole-tiles={dp} " in info, info
    if name == "block505":
        assert_close(to_np(y), c.ref["y"], f"block[{name}] stream-k tail {units}", CHAIN_MAX_E, CHAIN_MEAN_E)
    else:
        assert_close(to_np(y), c.ref["y"], f"block[{name}] stream-k tail {units}")
    assert torch.equal(y, run_block(h3, c))


@pytest.mark.parametrize("name,units", [("block505", None), ("d576", "12"), ("ragged205", "6")])
def test_norm2_fused_into_out_projection(h3, name, units, monkeypatch):
    """With H3_NORM_FUSE=1, where the O projection runs stream-K (every SM
    pair resident), its epilogue also emits norm2 + modulation: each owner
    warp stores per-row partial sums of squares of the bf16 residual, counts
    itself for the row tile, and after its tiles normalises and modulates the
    columns it owns; the separate norm2 kernel is not launched.  Against the
    oracle, equal to the default (separate norm2) block within the bound,
    bitwise repeatable, and one kernel fewer per block."""
    if units:   # small blocks: stream-K forced over `units` pairs (one k-block or a few per run)
        monkeypatch.setenv("H3_GEMM_SK_UNITS", units)
    c = get_case(name)
    cfg = c.cfg(h3)
    sep_count = h3.h3_blocks_kernel_count(cfg, 1, c.S)
    y_sep = run_block(h3, c)
    monkeypatch.setenv("H3_NORM_FUSE", "1")     # off by default: measured slower
    assert h3.h3_blocks_kernel_count(cfg, 1, c.S) == sep_count - 1
    y = run_block(h3, c)
    assert torch.equal(y, run_block(h3, c))
    monkeypatch.delenv("H3_NORM_FUSE")
    lim = (CHAIN_MAX_E, CHAIN_MEAN_E) if name == "block505" else (MAX_E, MEAN_E)
    assert_close(to_np(y), c.ref["y"], f"block[{name}] norm2 fused", *lim)
    assert_close(to_np(y), to_np(y_sep), f"block[{name}] fused vs separate norm2", *lim)


def test_block_forward_host_matches_device(h3):
    """h3_block_forward_host (pinned host input, metadata and output, copies
    ordered on the stream inside the call) gives the device call's output bit
    for bit, also in place on the host buffer."""
    c = get_case("ragged205")
    y_dev = run_block(h3, c)
    cfg = c.cfg(h3)
    ws = torch.empty(h3.h3_block_host_workspace_bytes(cfg, c.S, c.T), dtype=torch.uint8, device="cuda")
    assert ws.numel() > h3.h3_block_workspace_bytes(cfg, c.S, c.T)
    md = {k: v.cpu().pin_memory() for k, v in c.d_meta.items()}
    tc = c.d_tc.cpu().pin_memory()
    meta_h = h3.make_meta(md["token_tag"], md["timestep_index"], md["pos_thw"], tc, c.T)
    x_h = c.d_x.cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory()
    h3.h3_block_forward_host(cfg, h3.make_weights(c.d_w), meta_h, x_h, y_h, ws)
    torch.cuda.synchronize()
    assert h3.h3_sync_check() == 0
    assert torch.equal(y_h, y_dev.cpu())
    h3.h3_block_forward_host(cfg, h3.make_weights(c.d_w), meta_h, x_h, x_h, ws)   # in place
    torch.cuda.synchronize()
    assert torch.equal(x_h, y_dev.cpu())
    small = torch.empty(h3.h3_block_workspace_bytes(cfg, c.S, c.T), dtype=torch.uint8, device="cuda")
    with pytest.raises(h3.H3Error):
        h3.h3_block_forward_host(cfg, h3.make_weights(c.d_w), meta_h, x_h, y_h, small)


def _chain_case(name, nb, seed=0):
    w = {"d576": D576}.get(name) or hi.WORKLOADS[name]
    shape, S, T = w.shape, w.layout.n_rows, w.n_timesteps
    meta = {k: v.cuda() for k, v in hi.packed_metadata(w.layout, T, seed).items()}
    acts = hi.activations(shape, S, T, seed, device="cuda")
    wts = [{k: (v.cuda() if v is not None else None) for k, v in hi.block_weights(shape, seed, b).items()}
           for b in range(nb)]
    return w, meta, acts, wts


@pytest.mark.parametrize("name,nb", [("d576", 3), ("d576", 70), ("block1824", 2)])
def test_chain_batched_tables_match_block_calls(h3, name, nb):
    """Chains whose blocks get no side-stream overlap compute every block's
    AdaLN table up front (one SiLU launch, one table launch per 64 blocks:
    70 blocks take two), and at 1824 rows run stream-K residual GEMMs whose
    flag epochs continue across the chain.  The chain must equal the blocks
    called one by one bit for bit, through h3_blocks_forward, its CUDA graph
    and the host-buffer call; a workspace without room for the tables is
    refused."""
    w, meta, acts, wts = _chain_case(name, nb)
    shape, S, T = w.shape, w.layout.n_rows, w.n_timesteps
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    assert h3.h3_block_adaln_side_ctas(cfg, S) == 0
    cw = [h3.make_weights(x) for x in wts]
    m = h3.make_meta(meta["token_tag"], meta["timestep_index"], meta["pos_thw"], acts["t_cond"], T)
    nbytes = h3.h3_blocks_workspace_bytes(cfg, nb, S, T)
    assert nbytes > h3.h3_block_workspace_bytes(cfg, S, T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    x = acts["x"]
    y_ref = x.clone()
    for b in range(nb):
        h3.h3_block_forward(cfg, cw[b], m, y_ref, y_ref, ws)
    y = torch.empty_like(x)
    h3.h3_blocks_forward(cfg, cw, m, x, y, ws)
    assert h3.h3_sync_check() == 0
    if name == "block1824":
        assert "stream-k=0" not in h3.h3_last_kernel_info()
    assert torch.equal(y, y_ref)
    g = h3.BlocksGraph(cfg, cw, m, x, y, ws)
    y.zero_()
    g.launch()
    assert h3.h3_sync_check() == 0
    assert torch.equal(y, y_ref)
    g.close()
    wsh = torch.empty(h3.h3_blocks_host_workspace_bytes(cfg, nb, S, T), dtype=torch.uint8, device="cuda")
    md = {k: v.cpu().pin_memory() for k, v in meta.items()}
    tc = acts["t_cond"].cpu().pin_memory()
    meta_h = h3.make_meta(md["token_tag"], md["timestep_index"], md["pos_thw"], tc, T)
    x_h = x.cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory()
    h3.h3_blocks_forward_host(cfg, cw, meta_h, x_h, y_h, wsh)
    torch.cuda.synchronize()
    assert h3.h3_sync_check() == 0
    assert torch.equal(y_h, y_ref.cpu())
    small = torch.empty(h3.h3_block_workspace_bytes(cfg, S, T), dtype=torch.uint8, device="cuda")
    with pytest.raises(h3.H3Error) as e:
        h3.h3_blocks_forward(cfg, cw, m, x, y, small)
    assert e.value.status == h3.H3_ERR_WORKSPACE


def test_stream_k_lost_flags_time_out(h3, monkeypatch):
    """The stream-K hand-off's failure path, without a GPU fault: with
    H3_SK_FLAG_TEST=1 the owners wait for a flag value that nothing sets, so
    their bounded waits (2 s) run out; the launch records a device timeout
    that h3_sync_check reports as H3_ERR_TIMEOUT, and the next call on the
    same context works and gives the normal result bit for bit."""
    c = get_case("block505")          # O and FC2 run stream-K at 505 rows
    y_ref = run_block(h3, c)
    assert "stream-k=0" not in h3.h3_last_kernel_info()
    monkeypatch.setenv("H3_SK_FLAG_TEST", "1")
    cfg = c.cfg(h3)
    ws = torch.empty(h3.h3_block_workspace_bytes(cfg, c.S, c.T), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(y_ref)
    h3.h3_block_forward(cfg, h3.make_weights(c.d_w), c.meta(h3), c.d_x, y, ws)
    assert h3.h3_sync_check(timeout_ms=60000) == h3.H3_ERR_TIMEOUT
    assert h3.h3_last_error_site() == "gemm: stream-K partial-sum flag"
    # The timeout bit is sticky until h3_sync_check: once the first launch with
    # lost flags has given up (its waits run out after 2 s, some one after
    # another), every later kernel of the queue reads the bit at entry and
    # skips its work.  Without that, each of the eight stream-K launches of
    # four blocks pays its own limits (26 s were measured before the entry
    # check existed).
    cw = [h3.make_weights(c.d_w)] * 4
    ws = torch.empty(h3.h3_blocks_workspace_bytes(cfg, 4, c.S, c.T), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    h3.h3_blocks_forward(cfg, cw, c.meta(h3), c.d_x, y, ws)
    assert h3.h3_sync_check(timeout_ms=60000) == h3.H3_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    print(f"four blocks with lost stream-K flags: {elapsed:.1f} s until the timeout is reported")
    assert elapsed < 10.0, f"four blocks with lost flags took {elapsed:.1f} s"
    monkeypatch.delenv("H3_SK_FLAG_TEST")
    assert torch.equal(run_block(h3, c, ws=ws), y_ref)
    assert h3.h3_sync_check() == 0


def test_block_repeatable_and_inplace(h3):
    """Control H-C0 (repeated call: bitwise equal), a fresh workspace, and
    x_out aliasing x_in."""
    c = get_case("ragged205")
    y1 = run_block(h3, c)
    y2 = run_block(h3, c)
    assert torch.equal(y1, y2)
    x = c.d_x.clone()
    cfg = c.cfg(h3)
    ws = torch.empty(h3.h3_block_workspace_bytes(cfg, c.S, c.T), dtype=torch.uint8, device="cuda")
    h3.h3_block_forward(cfg, h3.make_weights(c.d_w), c.meta(h3), x, x, ws)
    assert h3.h3_sync_check() == 0
    assert torch.equal(x, y1)


def test_block_permutation_equivariance(h3):
    """Control H-C3: a consistent permutation of rows and metadata permutes the
    output (keys are summed in another order, so equal within tolerance)."""
    c = get_case("ragged205")
    y = to_np(run_block(h3, c))
    perm = torch.randperm(c.S, generator=torch.Generator().manual_seed(3))
    pd = perm.cuda()
    m = c.d_meta
    tag, tidx, pos = (m[k][pd].contiguous() for k in ("token_tag", "timestep_index", "pos_thw"))
    meta = h3.make_meta(tag, tidx, pos, c.d_tc, c.T)
    x_p = c.d_x[pd].contiguous()
    yp = to_np(run_block(h3, c, x=x_p, meta=meta))
    assert_close(yp, y[perm.numpy()], "permuted block")


def test_chain_two_blocks(h3):
    c = get_case("tiny72")
    cfg = c.cfg(h3)
    ws = torch.empty(h3.h3_blocks_workspace_bytes(cfg, 2, c.S, c.T), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(c.d_x)
    wts = h3.make_weights(c.d_w)
    h3.h3_blocks_forward(cfg, [wts, wts], c.meta(h3), c.d_x, y, ws)
    assert h3.h3_sync_check() == 0
    y1 = run_block(h3, c)
    y2 = run_block(h3, c, x=y1)
    assert torch.equal(y, y2)
    ref = O.block_forward(c.ref["y"], c.np_meta["token_tag"], c.np_meta["timestep_index"], c.np_meta["pos_thw"],
                          c.np_tc, c.np_w)["y"]
    assert_close(to_np(y), ref, "two-block chain")


@pytest.mark.parametrize("cond", [128, 2816])
def test_block_maximum_table_sizes(h3, cond):
    """The largest AdaLN table the kernels take: 16 timestep rows, and a
    conditioning width of 2816 (the most the table kernel keeps resident in
    shared memory), on a small block with every timestep row used."""
    shape = hi.BlockShape(dim=512, n_heads=4, head_dim=128, ffn_dim=1536, cond_dim=cond)
    w = hi.custom_workload(shape, n_text=9, video_grid=(2, 4, 5), n_audio=23, n_timesteps=16,
                           name=f"maxtable{cond}")
    c = Case(w)
    assert set(np.unique(c.np_meta["timestep_index"])) <= set(range(16))
    y = run_block(h3, c)
    assert_close(to_np(y), c.ref["y"], f"block T=16 cond={cond}")


@pytest.mark.parametrize("layout", [(2, (1, 1, 3), 2), (5, (2, 4, 8), 60)], ids=["S7", "S129"])
def test_block_odd_row_counts(h3, layout):
    """Odd packed-row counts: 7 rows (one partial tile of every kernel, two
    rows of each modality's segment) and 129 rows (one row past a 128-row
    tile: a second, one-row tile in the GEMMs' A operand and in attention)."""
    n_text, grid, n_audio = layout
    w = hi.custom_workload(hi.TINY_SHAPE, n_text=n_text, video_grid=grid, n_audio=n_audio, n_timesteps=3,
                           name=f"odd{n_text + grid[0] * grid[1] * grid[2] + n_audio}")
    c = Case(w)
    y = run_block(h3, c)
    assert_close(to_np(y), c.ref["y"], f"block S={c.S}")


def test_block_maximum_width(h3):
    """The widest residual the library takes (D = 8192: the norm kernels' 16-byte
    chunks at their limit, 32 column tiles per GEMM row) on a short ragged
    document with two heads."""
    shape = hi.BlockShape(dim=8192, n_heads=2, head_dim=128, ffn_dim=256, cond_dim=128)
    w = hi.custom_workload(shape, n_text=3, video_grid=(2, 2, 5), n_audio=14, n_timesteps=2, name="wide8192")
    c = Case(w)
    y = run_block(h3, c)
    assert_close(to_np(y), c.ref["y"], "block D=8192")


def _large_positions(S, seed):
    """Positions up to the largest the kernels accept (2^24 - 1 on every
    axis): the extremes, values just below them, and random ones."""
    rng = np.random.default_rng(seed)
    top = (1 << 24) - 1
    pos = rng.integers(0, 1 << 24, size=(S, 3)).astype(np.int32)
    pos[:8] = [[top, top, top], [top - 1, 0, 5], [0, top, top - 2], [1 << 23, (1 << 23) + 1, top],
               [top, 1, 2], [12345678, 7654321, 16000000], [0, 0, 0], [1, 1, 1]]
    return pos


@pytest.mark.parametrize("name", ["tiny72", "ragged205"])
def test_rope_at_large_positions(h3, name):
    """MM-RoPE at positions near the accepted maximum, where the fp32 angle is
    large (up to 1.7e7 rad) and the sine and cosine depend on a full-range
    argument reduction: the QKV epilogue and the standalone kernel against
    the oracle's cosine and sine (fp64) of the same fp32 angle."""
    c = get_case(name)
    H = c.w.shape.n_heads
    pos = _large_positions(c.S, 21)
    d_pos = torch.from_numpy(pos).cuda()
    m = c.d_meta
    meta = h3.make_meta(m["token_tag"], m["timestep_index"], d_pos, c.d_tc, c.T)
    q_ref, k_ref, _ = O.qk_norm_rope(c.ref["qkv"], pos, c.np_w["q_norm_g"], c.np_w["k_norm_g"])
    out = torch.zeros(c.S, H, 3, 128, dtype=torch.bfloat16, device="cuda")
    h3.h3_qkv_projection(c.cfg(h3), meta, to_bf16(c.ref["h1"]), c.d_w["w_qkv"], None,
                         c.d_w["q_norm_g"], c.d_w["k_norm_g"], out)
    assert h3.h3_sync_check() == 0
    o = to_np(out)
    assert_close(o[:, :, 0], q_ref, f"qkv epilogue q, large positions [{name}]")
    assert_close(o[:, :, 1], k_ref, f"qkv epilogue k, large positions [{name}]")
    buf = to_bf16(c.ref["qkv"].reshape(c.S, H, 3, 128))
    h3.h3_rope_qknorm(c.cfg(h3), c.S, d_pos, buf[:, :, 0], buf[:, :, 1], H * 384, 384,
                      c.d_w["q_norm_g"], c.d_w["k_norm_g"])
    assert h3.h3_sync_check() == 0
    o = to_np(buf)
    assert_close(o[:, :, 0], q_ref, f"standalone q, large positions [{name}]")
    assert_close(o[:, :, 1], k_ref, f"standalone k, large positions [{name}]")


def test_single_row_block(h3):
    w = hi.custom_workload(hi.TINY_SHAPE, n_text=1, video_grid=(0, 0, 0), n_audio=0, n_timesteps=1)
    c = Case(w)
    y = run_block(h3, c)
    assert_close(to_np(y), c.ref["y"], "block S=1")


# ---------------------------------------------------------------------------
# the chain as one CUDA graph: replays equal direct calls bit for bit
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,nb", [("tiny72", 3), ("block505", 2)])
def test_blocks_graph_replay_matches_direct(h3, name, nb):
    w = hi.WORKLOADS[name]
    shape, S, T = w.shape, w.layout.n_rows, w.n_timesteps
    meta = {k: v.cuda() for k, v in hi.packed_metadata(w.layout, T, 0).items()}
    acts = hi.activations(shape, S, T, 0, device="cuda")
    wts = [{k: (v.cuda() if v is not None else None) for k, v in hi.block_weights(shape, 0, b).items()}
           for b in range(nb)]
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    cw = [h3.make_weights(x) for x in wts]
    m = h3.make_meta(meta["token_tag"], meta["timestep_index"], meta["pos_thw"], acts["t_cond"], T)
    ws = torch.empty(h3.h3_blocks_workspace_bytes(cfg, nb, S, T), dtype=torch.uint8, device="cuda")
    x = acts["x"].clone()
    y_direct = torch.empty_like(x)
    h3.h3_blocks_forward(cfg, cw, m, x, y_direct, ws)
    y_graph = torch.zeros_like(x)
    g = h3.BlocksGraph(cfg, cw, m, x, y_graph, ws)
    g.launch()
    assert h3.h3_sync_check() == 0
    assert torch.equal(y_graph, y_direct)
    # a replay reads the buffers' current contents
    x.copy_(hi.normal((S, shape.dim), 1.0, 0.0, 5, 1, device="cuda"))
    h3.h3_blocks_forward(cfg, cw, m, x, y_direct, ws)
    g.launch()
    assert h3.h3_sync_check() == 0
    assert torch.equal(y_graph, y_direct)
    g.close()


# ---------------------------------------------------------------------------
# token refiner: two pre-norm blocks without AdaLN or RoPE, then a final norm
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape_name,S", [("tiny", 37), ("h3", 256)])
def test_refiner_forward(h3, shape_name, S):
    shape = hi.WORKLOADS["tiny72" if shape_name == "tiny" else "block505"].shape
    wts = [hi.block_weights(shape, 0, b) for b in (7, 8)]
    gfin = hi.normal((shape.dim,), 0.1, 1.0, 0, 90)
    x = hi.normal((S, shape.dim), 1.0, 0.0, 0, 91)
    ref = O.refiner_forward(to_np(x), [{k: (to_np(v) if v is not None else None) for k, v in w.items()} for w in wts],
                            to_np(gfin))
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    d_w = [{k: (v.cuda() if v is not None else None) for k, v in w.items()} for w in wts]
    ws = torch.empty(h3.h3_refiner_workspace_bytes(cfg, S), dtype=torch.uint8, device="cuda")
    d_x = x.cuda()
    y = torch.empty_like(d_x)
    h3.h3_refiner_forward(cfg, [h3.make_weights(w) for w in d_w], gfin.cuda(), S, d_x, y, ws)
    assert h3.h3_sync_check() == 0
    lim = (MAX_E, MEAN_E) if shape_name == "tiny" else (REFINER_CHAIN_MAX_E, REFINER_CHAIN_MEAN_E)
    mx, mn = assert_close(to_np(y), ref, f"refiner {shape_name} S={S}", *lim)
    print(f"refiner {shape_name} S={S}: max_e={mx:.4f} mean_e={mn:.5f}")
    # in place, and repeatable bit for bit
    h3.h3_refiner_forward(cfg, [h3.make_weights(w) for w in d_w], gfin.cuda(), S, d_x, d_x, ws)
    assert h3.h3_sync_check() == 0
    assert torch.equal(d_x, y)


# ---------------------------------------------------------------------------
# failure handling (host-detected and device-detected; nothing faults)
# ---------------------------------------------------------------------------

def test_bad_metadata_is_reported_not_faulted(h3):
    c = get_case("tiny72")
    bad = c.d_meta["token_tag"].clone()
    bad[5] = 7
    meta = h3.make_meta(bad, c.d_meta["timestep_index"], c.d_meta["pos_thw"], c.d_tc, c.T)
    cfg = c.cfg(h3)
    ws = torch.empty(h3.h3_block_workspace_bytes(cfg, c.S, c.T), dtype=torch.uint8, device="cuda")
    y = torch.zeros_like(c.d_x)
    h3.h3_block_forward(cfg, h3.make_weights(c.d_w), meta, c.d_x, y, ws)
    assert h3.h3_sync_check() == h3.H3_ERR_INDEX
    assert h3.h3_sync_check() == 0          # the word was cleared
    run_block(h3, c)                        # the context is still usable


def test_host_validation_launches_nothing(h3):
    c = get_case("tiny72")
    cfg = c.cfg(h3)
    bad_cfg = h3.make_config(c.w.shape.dim, c.w.shape.n_heads, c.w.shape.ffn_dim, c.w.shape.cond_dim,
                             head_dim=64)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(c.d_x)
    with pytest.raises(h3.H3Error) as e:
        h3.h3_block_forward(bad_cfg, h3.make_weights(c.d_w), c.meta(h3), c.d_x, y, ws)
    assert e.value.status == h3.H3_ERR_UNSUPPORTED
    with pytest.raises(h3.H3Error) as e:
        h3.h3_block_forward(cfg, h3.make_weights(c.d_w), c.meta(h3), c.d_x, y, ws)
    assert e.value.status == h3.H3_ERR_WORKSPACE
    with pytest.raises(h3.H3Error) as e:
        h3.h3_attention(c.S, 4, c.d_x, c.d_x, c.d_x, 1540, 384, y)
    assert e.value.status == h3.H3_ERR_ALIGN
    assert "tcgen05" in h3.h3_last_kernel_info() or h3.h3_last_kernel_info() != ""


# ---------------------------------------------------------------------------
# attention core at 4096 packed rows (56 heads): QK-norm + RoPE prologue on the
# GPU against the oracle, then attention on sampled query rows
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def attn4096():
    w = hi.WORKLOADS["attn4096"]
    meta = hi.packed_metadata(w.layout, 1, 0)
    ins = hi.attention_inputs(w.shape, w.layout.n_rows, 0)
    qkv = to_np(ins["qkv"])
    gq, gk = to_np(ins["q_norm_g"]), to_np(ins["k_norm_g"])
    pos = meta["pos_thw"].numpy()
    q, k, v = O.qk_norm_rope(qkv, pos, gq, gk)
    return {"w": w, "ins": ins, "pos": meta["pos_thw"], "q": q, "k": k, "v": v}


def test_rope_qknorm_4096(h3, attn4096):
    d = attn4096
    w = d["w"]
    S, H = w.layout.n_rows, w.shape.n_heads
    cfg = h3.make_config(w.shape.dim, H, w.shape.ffn_dim, w.shape.cond_dim)
    buf = d["ins"]["qkv"].cuda()
    h3.h3_rope_qknorm(cfg, S, d["pos"].cuda(), buf[:, :, 0], buf[:, :, 1], H * 384, 384,
                      d["ins"]["q_norm_g"].cuda(), d["ins"]["k_norm_g"].cuda())
    assert h3.h3_sync_check() == 0
    o = to_np(buf)
    assert_close(o[:, :, 0], d["q"], "rope4096.q")
    assert_close(o[:, :, 1], d["k"], "rope4096.k")


def test_rope_qknorm_separate_buffers_two_head_blocks(h3):
    """q and k in separate, row-padded buffers (head stride 128, row stride
    H*128 + 64) and 70 heads, more than one shared-memory unit holds: the
    heads of a row are split into two units of 35."""
    S, H = 301, 70
    pos = hi.packed_metadata(hi.PackedLayout(9, (4, 6, 11), 28), 1, 3)["pos_thw"]
    assert pos.shape[0] == S
    g = torch.Generator().manual_seed(11)
    q = torch.randn(S, H, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(S, H, 128, generator=g).to(torch.bfloat16)
    gq = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16)
    gk = (1 + 0.1 * torch.randn(128, generator=g)).to(torch.bfloat16)
    qkv = np.stack([to_np(q), to_np(k), np.zeros((S, H, 128))], axis=2)
    ref_q, ref_k, _ = O.qk_norm_rope(qkv, pos.numpy(), to_np(gq), to_np(gk))
    rs = H * 128 + 64
    dq = torch.zeros(S, rs, dtype=torch.bfloat16, device="cuda")
    dk = torch.zeros(S, rs, dtype=torch.bfloat16, device="cuda")
    dq[:, :H * 128] = q.reshape(S, -1).cuda()
    dk[:, :H * 128] = k.reshape(S, -1).cuda()
    cfg = h3.make_config(512, H, 1536, 256)
    h3.h3_rope_qknorm(cfg, S, pos.cuda(), dq, dk, rs, 128, gq.cuda(), gk.cuda())
    assert h3.h3_sync_check() == 0
    assert "heads/unit=35" in h3.h3_last_kernel_info()
    assert_close(to_np(dq[:, :H * 128]).reshape(S, H, 128), ref_q, "rope70.q")
    assert_close(to_np(dk[:, :H * 128]).reshape(S, H, 128), ref_k, "rope70.k")
    assert not dq[:, H * 128:].any() and not dk[:, H * 128:].any()   # padding untouched
    # a position out of range is reported and its row is left as it was
    bad = pos.clone()
    bad[17, 1] = 1 << 24
    dq2 = dq.clone()
    h3.h3_rope_qknorm(cfg, S, bad.cuda(), dq2, dk.clone(), rs, 128, gq.cuda(), gk.cuda())
    assert h3.h3_sync_check() == h3.H3_ERR_INDEX
    assert torch.equal(dq2[17], dq[17])


def test_attention_4096_sampled_rows(h3, attn4096, attn_qtiles):
    d = attn4096
    S, H = d["w"].layout.n_rows, d["w"].shape.n_heads
    buf = torch.stack([to_bf16(d["q"]), to_bf16(d["k"]), to_bf16(d["v"])], dim=2).contiguous()
    o = torch.empty(S, H * 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(H, S, dtype=torch.float32, device="cuda")
    h3.h3_attention(S, H, buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], H * 384, 384, o, lse)
    assert h3.h3_sync_check() == 0
    rows = np.unique(np.concatenate([np.arange(0, 3), np.linspace(0, S - 1, 93).astype(int), [S - 1]]))
    ref = O.attention(d["q"], d["k"], d["v"], rows)
    assert_close(to_np(o)[rows], ref, f"attention4096[{attn_qtiles}]")
    lse_np = lse.cpu().numpy().astype(np.float64)
    for h in range(0, H, 5):
        q, k = d["q"][rows[:16], h], d["k"][:, h]
        p_gpu = np.exp(q @ k.T / np.sqrt(128.0) - lse_np[h, rows[:16]][:, None])
        assert np.abs(p_gpu - O.attention_probs(q, k)).max() <= 1e-3


# ---------------------------------------------------------------------------
# attention core at 16,384 and 32,768 packed rows: the QK-norm + RoPE prologue
# and attention exactly as the benchmark launches them, checked on every row
# of the prologue and on sampled query rows of attention
# ---------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("wl", ["attn16384", "attn32768"])
def test_attention_core_full_size_sampled_rows(h3, wl):
    w = hi.WORKLOADS[wl]
    S, H = w.layout.n_rows, w.shape.n_heads
    meta = hi.packed_metadata(w.layout, 1, 0)
    ins = hi.attention_inputs(w.shape, S, 0)
    q, k, v = O.qk_norm_rope(to_np(ins["qkv"]), meta["pos_thw"].numpy(), to_np(ins["q_norm_g"]),
                             to_np(ins["k_norm_g"]))
    cfg = h3.make_config(w.shape.dim, H, w.shape.ffn_dim, w.shape.cond_dim)
    buf = ins["qkv"].cuda()
    h3.h3_rope_qknorm(cfg, S, meta["pos_thw"].cuda(), buf[:, :, 0], buf[:, :, 1], H * 384, 384,
                      ins["q_norm_g"].cuda(), ins["k_norm_g"].cuda())
    o = torch.empty(S, H * 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(H, S, dtype=torch.float32, device="cuda")
    h3.h3_attention(S, H, buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], H * 384, 384, o, lse)
    assert h3.h3_sync_check(timeout_ms=60000) == 0
    got = to_np(buf)
    assert_close(got[:, :, 0], q, f"{wl} rope.q")
    assert_close(got[:, :, 1], k, f"{wl} rope.k")
    # attention from the GPU's own q, k, v (bf16 after the prologue): the
    # oracle's rounding of the prologue differs by at most an ulp in a few
    # elements, which the prologue check above bounds
    qg, kg, vg = got[:, :, 0], got[:, :, 1], got[:, :, 2]
    rows = np.unique(np.concatenate([[0, 1, w.layout.n_text, S - w.layout.n_audio, S - 1],
                                     np.random.default_rng(12).integers(0, S, 27)]))
    ref = O.attention(qg, kg, vg, rows)
    assert_close(to_np(o)[rows], ref, f"{wl} attention (sampled rows)")
    lse_np = lse.cpu().numpy().astype(np.float64)
    for h in range(0, H, 11):
        qh, kh = qg[rows[:8], h], kg[:, h]
        p_gpu = np.exp(qh @ kh.T / np.sqrt(128.0) - lse_np[h, rows[:8]][:, None])
        assert np.abs(p_gpu - O.attention_probs(qh, kh)).max() <= 1e-3
