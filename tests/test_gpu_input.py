"""GPU parity of the input side against the CPU oracle: the patch permutation
and the row scatter bit for bit, the FP32 input projections (one bf16
rounding) within the operator bound, the FP32 timestep features and MLP
within 1e-4 / 1e-5 of the error metric."""
import numpy as np
import pytest
import torch

import h3_inputs as hi
from oracle import h3_input_oracle as IO
from oracle import h3_output_oracle as OO
from h3_testutil import MAX_E, MEAN_E, assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h3():
    assert torch.cuda.is_available()
    import audio_video_flow_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("C,T,H,W", [(24, 36, 30, 54), (3, 2, 4, 6), (24, 1, 2, 2)])
def test_patch_pack_unpack_bit_exact(h3, C, T, H, W):
    lat = hi.normal((C, T, H, W), 1.0, 0.0, 0, 95, dtype=torch.float32)
    rows = torch.full((T * (H // 2) * (W // 2), 4 * C), float("nan"), dtype=torch.float32, device="cuda")
    h3.h3_patch_pack(C, T, H, W, lat.cuda(), rows)
    back = torch.full_like(lat.cuda(), float("nan"))
    h3.h3_patch_unpack(C, T, H, W, rows, back)
    assert h3.h3_sync_check() == 0
    np.testing.assert_array_equal(rows.cpu().numpy(), IO.patch_pack(lat.numpy()))
    assert torch.equal(back.cpu(), lat)


def test_patch_pack_rejects_odd_sizes(h3):
    buf = torch.empty(64, dtype=torch.float32, device="cuda")
    with pytest.raises(h3.H3Error) as e:
        h3.h3_patch_pack(2, 2, 3, 4, buf, buf)
    assert e.value.status == h3.H3_ERR_SHAPE


@pytest.mark.parametrize("wl", ["tiny72", "denoiser15860"])
def test_input_projections_into_packed_stream(h3, wl):
    w = hi.WORKLOADS[wl]
    shape, S = w.shape, w.layout.n_rows
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    meta = hi.packed_metadata(w.layout, 1, 0)
    iw = hi.input_weights(shape, 0)
    tags = meta["token_tag"].numpy()
    x = torch.zeros(S, shape.dim, dtype=torch.bfloat16, device="cuda")
    parts = []
    for tag, P, m, tid in [(OO.TAG_VIDEO, 96, "video", 96), (OO.TAG_AUDIO, 32, "audio", 97)]:
        idx = OO.select_rows(tags, tag)
        src = hi.latents(idx.size, P, 0, tid)
        h3.h3_input_projection(cfg, idx.size, P, src.cuda(), iw[f"w_in_{m}"].cuda(), iw[f"b_in_{m}"].cuda(),
                               torch.from_numpy(idx).cuda(), S, x)
        parts.append((IO.input_projection(src.numpy(), iw[f"w_in_{m}"].numpy(), iw[f"b_in_{m}"].numpy()), idx))
    assert h3.h3_sync_check() == 0
    ref = IO.packed_index_copy(S, shape.dim, parts)
    got = to_np(x)
    text = OO.select_rows(tags, OO.TAG_TEXT)
    assert not got[text].any()                                   # rows no modality writes stay zero
    mod = np.setdiff1d(np.arange(S), text)
    assert_close(got[mod], ref[mod], f"input projections {wl}", MAX_E, MEAN_E)


def test_packed_index_copy_bit_exact_and_bad_index(h3):
    D, S = 512, 300
    cfg = h3.make_config(D, 4, 1536, 256)
    src = hi.normal((40, D), 1.0, 0.0, 0, 98).cuda()
    dst = torch.from_numpy(np.random.default_rng(4).permutation(S)[:40].astype(np.int32)).cuda()
    x = torch.zeros(S, D, dtype=torch.bfloat16, device="cuda")
    h3.h3_packed_index_copy(cfg, 40, src, dst, S, x)
    assert h3.h3_sync_check() == 0
    ref = IO.packed_index_copy(S, D, [(to_np(src), dst.cpu().numpy())])
    np.testing.assert_array_equal(to_np(x), ref)
    dst[5] = S + 3
    h3.h3_packed_index_copy(cfg, 40, src, dst, S, x)
    assert h3.h3_sync_check() == h3.H3_ERR_INDEX


@pytest.mark.parametrize("wl,T", [("tiny72", 4), ("block505", 12), ("denoiser15860", 1)])
def test_timestep_embedding(h3, wl, T):
    shape = hi.WORKLOADS[wl].shape
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    iw = hi.input_weights(shape, 0)
    sig = OO.sigma_grid(13, OO.VIDEO_SHIFT)
    t = torch.from_numpy(OO.timesteps(sig)[:T].copy()) if T <= 13 else None
    scratch = torch.empty(T * (256 + shape.dim), dtype=torch.float32, device="cuda")
    tc = torch.empty(T, shape.cond_dim, dtype=torch.float32, device="cuda")
    h3.h3_timestep_embedding(cfg, T, t.cuda(), iw["w_t1"].cuda(), iw["b_t1"].cuda(), iw["w_t2"].cuda(),
                             iw["b_t2"].cuda(), scratch, tc)
    assert h3.h3_sync_check() == 0
    e_ref = IO.timestep_sinusoid(t.numpy())
    assert_close(scratch[:T * 256].reshape(T, 256).cpu().numpy(), e_ref, f"sinusoid {wl}", 1e-5, 1e-6)
    ref = IO.timestep_mlp(e_ref, iw["w_t1"].numpy(), iw["b_t1"].numpy(), iw["w_t2"].numpy(), iw["b_t2"].numpy())
    assert_close(tc.cpu().numpy(), ref, f"timestep mlp {wl}", 1e-4, 1e-5)
