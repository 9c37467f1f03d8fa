"""GPU parity of the output side and the sampler against the CPU oracle.

The sampler arithmetic (sigma grid, Euler step, noise mix) and row selection
are defined in fp32 / integers, so they are compared bit for bit.  The FP32
final AdaLN and heads accumulate in fp32 against an fp64 oracle and are held
to 1e-4 (max) / 1e-5 (mean) of the error metric used for the block.
"""
import numpy as np
import pytest
import torch

import h3_inputs as hi
from oracle import h3_output_oracle as OO
from h3_testutil import assert_close, to_np

pytestmark = pytest.mark.gpu

F32_MAX_E, F32_MEAN_E = 1e-4, 1e-5


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available()
    import audio_video_flow_gb300 as m
    m.lib()
    return m


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


# ---------------------------------------------------------------- sampler

@pytest.mark.parametrize("n,s", [(2, 12.0), (5, 3.0), (13, 12.0), (13, 3.0), (50, 12.0), (1000, 3.0),
                                 (4097, 12.0), (7, 1.0)])
def test_sigma_schedule_bit_exact(h3, n, s):
    sig = torch.full((n + 1,), float("nan"), dtype=torch.float32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    h3.h3_sigma_schedule(n, s, sig, cnt)
    assert h3.h3_sync_check() == 0
    ref = OO.sigma_grid(n, s)
    k = int(cnt.item())
    assert k == ref.size
    np.testing.assert_array_equal(sig[:k].cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dual_schedules_and_timesteps(h3):
    out = {}
    for name, s in [("video", OO.VIDEO_SHIFT), ("audio", OO.AUDIO_SHIFT)]:
        sig = torch.empty(14, dtype=torch.float32, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
        h3.h3_sigma_schedule(13, s, sig, cnt)
        out[name] = sig[: int(cnt.item())].cpu().numpy()
    assert not np.array_equal(out["video"], out["audio"])        # probe H12 on the device path
    np.testing.assert_array_equal(OO.timesteps(out["video"]), (np.float32(1) - out["video"]).astype(np.float32))


@pytest.mark.parametrize("n", [14580 * 96 + 3, 1024 * 32, 5, 0])
def test_ode_step_bit_exact(h3, n):
    xt = hi.latents(max(n, 1), 1, 0, 70).reshape(-1)[:n].contiguous()
    v = hi.latents(max(n, 1), 1, 0, 71).reshape(-1)[:n].contiguous()
    grid = OO.sigma_grid(13, OO.VIDEO_SHIFT)
    for a, b in [(0, 1), (5, 6), (11, 12)]:          # the last step lands on sigma = 0
        sg, sn = float(grid[a]), float(grid[b])
        d_xt, d_v = xt.cuda(), v.cuda()
        out = torch.empty_like(d_xt)
        h3.h3_ode_step(n, d_xt, d_v, sg, sn, out)
        h3.h3_ode_step(n, d_xt, d_v, sg, sn, d_xt)    # in place
        assert h3.h3_sync_check() == 0
        ref = OO.ode_step(xt.numpy(), v.numpy(), sg, sn)
        np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
        np.testing.assert_array_equal(d_xt.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("t", [0.0, 0.25, 0.7, 1.0])
def test_noise_mix_bit_exact(h3, t):
    n = 1024 * 32 + 1
    x0 = hi.latents(n, 1, 0, 72).reshape(-1)
    nz = hi.latents(n, 1, 0, 73).reshape(-1)
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    h3.h3_noise_mix(n, x0.cuda(), nz.cuda(), t, out)
    assert h3.h3_sync_check() == 0
    ref = OO.noise_mix(x0.numpy(), nz.numpy(), t)
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_sampler_host_validation(h3):
    buf = torch.empty(8, dtype=torch.float32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    for n, s in [(1, 12.0), (5, 0.0), (5, float("nan"))]:
        with pytest.raises(h3.H3Error) as e:
            h3.h3_sigma_schedule(n, s, buf, cnt)
        assert e.value.status == h3.H3_ERR_SHAPE
    with pytest.raises(h3.H3Error) as e:
        h3.h3_ode_step(8, buf, buf, 0.0, 0.0, buf)          # sigma must be > 0
    assert e.value.status == h3.H3_ERR_SHAPE
    with pytest.raises(h3.H3Error) as e:
        h3.h3_ode_step(4, buf[1:], buf, 0.5, 0.1, buf)      # misaligned
    assert e.value.status == h3.H3_ERR_ALIGN


# ---------------------------------------------------------------- output side

def test_select_rows_bit_exact(h3):
    tags = torch.from_numpy(np.random.default_rng(3).integers(0, 3, 20011).astype(np.int32))
    d_tags = tags.cuda()
    for m in range(3):
        rows = torch.full((tags.numel(),), -7, dtype=torch.int32, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
        h3.h3_select_rows(tags.numel(), d_tags, m, rows, cnt)
        assert h3.h3_sync_check() == 0
        ref = OO.select_rows(tags.numpy(), m)
        k = int(cnt.item())
        assert k == ref.size
        np.testing.assert_array_equal(rows[:k].cpu().numpy(), ref)
        assert bool((rows[k:] == -7).all())


def _cfg(h3, shape):
    return h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)


@pytest.mark.parametrize("wl,T", [("tiny72", 4), ("block505", 12), ("denoiser15860", 1)])
def test_final_adaln_table(h3, wl, T):
    shape = hi.WORKLOADS[wl].shape
    ow = hi.output_weights(shape, 0)
    tc = hi.activations(shape, 1, T, 0)["t_cond"]
    for m in ("video", "audio"):
        tab = torch.empty(T, 2, shape.dim, dtype=torch.float32, device="cuda")
        h3.h3_final_adaln_table(_cfg(h3, shape), ow[f"w_fin_{m}"].cuda(), ow[f"b_fin_{m}"].cuda(), tc.cuda(), T,
                                tab)
        assert h3.h3_sync_check() == 0
        ref = OO.final_adaln_table(tc.numpy(), ow[f"w_fin_{m}"].numpy(), ow[f"b_fin_{m}"].numpy())
        assert_close(tab.cpu().numpy(), ref, f"final adaln {m} {wl}", F32_MAX_E, F32_MEAN_E)


@pytest.mark.parametrize("wl,T", [("tiny72", 4), ("denoiser15860", 1), ("denoiser15860", 11)])
def test_final_adaln_tables_in_one_launch(h3, wl, T):
    """Both modalities' tables from one launch equal the per-modality calls
    bit for bit (the same per-row sums), with and without biases; a single
    table through the batched call is the single call."""
    shape = hi.WORKLOADS[wl].shape
    ow = hi.output_weights(shape, 0)
    tc = hi.activations(shape, 1, T, 0)["t_cond"].cuda()
    cfg = _cfg(h3, shape)
    ws = [ow["w_fin_video"].cuda(), ow["w_fin_audio"].cuda()]
    for bs in ([ow["b_fin_video"].cuda(), ow["b_fin_audio"].cuda()], None):
        one = []
        for m in range(2):
            t = torch.empty(T, 2, shape.dim, dtype=torch.float32, device="cuda")
            h3.h3_final_adaln_table(cfg, ws[m], None if bs is None else bs[m], tc, T, t)
            one.append(t)
        both = [torch.full((T, 2, shape.dim), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
        h3.h3_final_adaln_tables(cfg, ws, bs, tc, T, both)
        assert h3.h3_sync_check() == 0
        assert "tables=2" in h3.h3_last_kernel_info()
        for m in range(2):
            assert torch.equal(both[m].view(torch.int32), one[m].view(torch.int32)), f"table {m}, bias {bs is not None}"
    single = torch.empty(T, 2, shape.dim, dtype=torch.float32, device="cuda")
    h3.h3_final_adaln_tables(cfg, ws[:1], None, tc, T, [single])
    assert h3.h3_sync_check() == 0
    assert torch.equal(single.view(torch.int32), one[0].view(torch.int32))


@pytest.mark.parametrize("wl", ["tiny72", "ragged", "denoiser15860"])
def test_output_heads(h3, wl):
    if wl == "ragged":
        w = hi.custom_workload(hi.BlockShape(dim=640, n_heads=3, head_dim=128, ffn_dim=1024, cond_dim=192),
                               n_text=13, video_grid=(2, 5, 9), n_audio=102, n_timesteps=7)
    else:
        w = hi.WORKLOADS[wl]
    shape, S, T = w.shape, w.layout.n_rows, w.n_timesteps
    meta = hi.packed_metadata(w.layout, T, 0)
    x = hi.activations(shape, S, T, 0)["x"]
    tc = hi.activations(shape, S, T, 0)["t_cond"]
    ow = hi.output_weights(shape, 0)
    cfg = _cfg(h3, shape)
    d_tag, d_tidx, d_x = meta["token_tag"].cuda(), meta["timestep_index"].cuda(), x.cuda()
    for m, tag, P in [("video", OO.TAG_VIDEO, hi.VIDEO_PATCH), ("audio", OO.TAG_AUDIO, hi.AUDIO_PATCH)]:
        tab_ref = OO.final_adaln_table(tc.numpy(), ow[f"w_fin_{m}"].numpy(), ow[f"b_fin_{m}"].numpy())
        rows = torch.empty(S, dtype=torch.int32, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
        h3.h3_select_rows(S, d_tag, tag, rows, cnt)
        n_sel = int(cnt.item())
        v = torch.full((n_sel, P), float("nan"), dtype=torch.float32, device="cuda")
        h3.h3_output_head(cfg, S, n_sel, rows, d_tidx, T, d_x, _f32(tab_ref), ow[f"w_head_{m}"].cuda(),
                          ow[f"b_head_{m}"].cuda(), P, v)
        assert h3.h3_sync_check() == 0
        ref = OO.output_head(to_np(x), meta["token_tag"].numpy(), meta["timestep_index"].numpy(), tag, tab_ref,
                             ow[f"w_head_{m}"].numpy(), ow[f"b_head_{m}"].numpy())
        assert_close(v.cpu().numpy(), ref, f"head {m} {wl}", F32_MAX_E, F32_MEAN_E)


@pytest.mark.parametrize("D,P,n_rows", [(512, 48, 300), (512, 128, 129), (640, 7, 77), (192, 96, 140)])
def test_output_head_widths(h3, D, P, n_rows):
    """Head widths of every register-tile variant (P up to 32, 64, 96, 128),
    a residual width whose 32-column chunks do not split evenly over the eight
    CTAs of a cluster (640: 20 chunks) or leave some of them without chunks
    (192: 6 chunks), and row counts that end inside a 96-row tile."""
    shape = hi.BlockShape(dim=D, n_heads=1, head_dim=128, ffn_dim=256, cond_dim=128)
    T = 3
    g = torch.Generator().manual_seed(D + P)
    x = (torch.randn(n_rows, D, generator=g)).to(torch.bfloat16)
    tidx = torch.randint(0, T, (n_rows,), generator=g, dtype=torch.int32)
    tab = (torch.randn(T, 2, D, generator=g) * 0.3).to(torch.float32)
    w = (torch.randn(P, D, generator=g) * 0.02).to(torch.float32)
    b = (torch.randn(P, generator=g) * 0.02).to(torch.float32)
    sel = torch.sort(torch.randperm(n_rows, generator=g)[: (2 * n_rows) // 3]).values.to(torch.int32)
    tags = torch.ones(n_rows, dtype=torch.int32)
    tags[sel.long()] = OO.TAG_VIDEO
    v = torch.full((sel.numel(), P), float("nan"), dtype=torch.float32, device="cuda")
    h3.h3_output_head(_cfg(h3, shape), n_rows, sel.numel(), sel.cuda(), tidx.cuda(), T, x.cuda(), tab.cuda(),
                      w.cuda(), b.cuda(), P, v)
    assert h3.h3_sync_check() == 0
    ref = OO.output_head(to_np(x), tags.numpy(), tidx.numpy(), OO.TAG_VIDEO, tab.numpy().astype(np.float64),
                         w.numpy(), b.numpy())
    assert_close(v.cpu().numpy(), ref, f"head D={D} P={P}", F32_MAX_E, F32_MEAN_E)


@pytest.mark.parametrize("fill", [0.1, 0.25, 0.6, 1.01, 2.02])
def test_output_head_every_k_split(h3, fill):
    """The k-split follows the row count (the fewest CTAs per 96-row tile
    that give two per SM): selections from a tenth of that target up to
    twice it take every split, 16, 8, 4, 2 and 1 (16 in a cluster beyond the
    portable size, 1 without a cluster), each within the fp32 bound of the
    oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_sel = int(fill * sms * 96) - 5
    tiles = (n_sel + 95) // 96
    want = next((k for k in (1, 2, 4, 8) if tiles * k >= 2 * sms), 16)
    D, P, T, n_rows = 320, 96, 2, n_sel + 37
    g = torch.Generator().manual_seed(n_sel)
    x = (torch.randn(n_rows, D, generator=g)).to(torch.bfloat16)
    tidx = torch.randint(0, T, (n_rows,), generator=g, dtype=torch.int32)
    tab = (torch.randn(T, 2, D, generator=g) * 0.3).to(torch.float32)
    w = (torch.randn(P, D, generator=g) * 0.02).to(torch.float32)
    b = (torch.randn(P, generator=g) * 0.02).to(torch.float32)
    sel = torch.sort(torch.randperm(n_rows, generator=g)[:n_sel]).values.to(torch.int32)
    tags = torch.ones(n_rows, dtype=torch.int32)
    tags[sel.long()] = OO.TAG_VIDEO
    shape = hi.BlockShape(dim=D, n_heads=1, head_dim=128, ffn_dim=256, cond_dim=128)
    v = torch.full((n_sel, P), float("nan"), dtype=torch.float32, device="cuda")
    h3.h3_output_head(_cfg(h3, shape), n_rows, n_sel, sel.cuda(), tidx.cuda(), T, x.cuda(), tab.cuda(), w.cuda(),
                      b.cuda(), P, v)
    assert h3.h3_sync_check() == 0
    assert f"k-split={want} " in h3.h3_last_kernel_info()
    ref = OO.output_head(to_np(x), tags.numpy(), tidx.numpy(), OO.TAG_VIDEO, tab.numpy().astype(np.float64),
                         w.numpy(), b.numpy())
    assert_close(v.cpu().numpy(), ref, f"head k-split {want}", F32_MAX_E, F32_MEAN_E)


def test_output_head_bad_timestep_is_reported(h3):
    w = hi.WORKLOADS["tiny72"]
    shape, S, T = w.shape, w.layout.n_rows, w.n_timesteps
    meta = hi.packed_metadata(w.layout, T, 0)
    x = hi.activations(shape, S, T, 0)["x"].cuda()
    ow = hi.output_weights(shape, 0)
    tidx = meta["timestep_index"].clone()
    vid = OO.select_rows(meta["token_tag"].numpy(), OO.TAG_VIDEO)
    tidx[int(vid[3])] = T                       # out of range
    rows = torch.from_numpy(vid).cuda()
    tab = torch.zeros(T, 2, shape.dim, dtype=torch.float32, device="cuda")
    v = torch.full((vid.size, 96), float("nan"), dtype=torch.float32, device="cuda")
    h3.h3_output_head(_cfg(h3, shape), S, vid.size, rows, tidx.cuda(), T, x, tab, ow["w_head_video"].cuda(), None,
                      96, v)
    assert h3.h3_sync_check() == h3.H3_ERR_INDEX
    assert bool(torch.isnan(v[3]).all()) and bool(torch.isfinite(v[4]).all())


def test_one_sampler_step_end_to_end(h3):
    """Velocity of the video rows from a residual stream, then the Euler step
    on the video latents: v within the fp32 tolerance, and x_next bit-exact
    against the oracle's step applied to the device's own v."""
    w = hi.WORKLOADS["block505"]
    shape, S, T = w.shape, w.layout.n_rows, w.n_timesteps
    meta = hi.packed_metadata(w.layout, T, 0)
    x = hi.activations(shape, S, T, 0)["x"]
    tc = hi.activations(shape, S, T, 0)["t_cond"]
    ow = hi.output_weights(shape, 0)
    cfg = _cfg(h3, shape)
    tab = torch.empty(T, 2, shape.dim, dtype=torch.float32, device="cuda")
    h3.h3_final_adaln_table(cfg, ow["w_fin_video"].cuda(), ow["b_fin_video"].cuda(), tc.cuda(), T, tab)
    rows = torch.empty(S, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    h3.h3_select_rows(S, meta["token_tag"].cuda(), OO.TAG_VIDEO, rows, cnt)
    n_sel = int(cnt.item())
    v = torch.empty(n_sel, 96, dtype=torch.float32, device="cuda")
    h3.h3_output_head(cfg, S, n_sel, rows, meta["timestep_index"].cuda(), T, x.cuda(), tab,
                      ow["w_head_video"].cuda(), ow["b_head_video"].cuda(), 96, v)
    xt = hi.latents(n_sel, 96, 0, 74)
    grid = OO.sigma_grid(13, OO.VIDEO_SHIFT)
    d_xt = xt.cuda()
    h3.h3_ode_step(xt.numel(), d_xt, v, float(grid[3]), float(grid[4]), d_xt)
    assert h3.h3_sync_check() == 0
    tab_ref = OO.final_adaln_table(tc.numpy(), ow["w_fin_video"].numpy(), ow["b_fin_video"].numpy())
    v_ref = OO.output_head(to_np(x), meta["token_tag"].numpy(), meta["timestep_index"].numpy(), OO.TAG_VIDEO,
                           tab_ref, ow["w_head_video"].numpy(), ow["b_head_video"].numpy())
    assert_close(v.cpu().numpy(), v_ref, "velocity", F32_MAX_E, F32_MEAN_E)
    x_ref = OO.ode_step(xt.numpy(), v.cpu().numpy(), grid[3], grid[4])
    np.testing.assert_array_equal(d_xt.cpu().numpy().view(np.uint32), x_ref.view(np.uint32))
