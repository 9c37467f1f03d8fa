"""h3_adaln_table_noalloc: the AdaLN table for callers that cannot allocate
device memory (its scratch is a static array inside the library).  Called
through the C ABI twice in a row with different inputs; each result must
match the workspace entry point h3_adaln_table within the suite's tolerance.
Collected last on purpose, and self-contained so it also passes alone in a
fresh process."""
import numpy as np
import pytest
import torch

import h3_inputs as hi
from h3_testutil import assert_close, to_np

pytestmark = pytest.mark.gpu


def _case(shape, T, seed):
    w = hi.block_weights(shape, seed=seed)
    t_cond = hi.normal((T, shape.cond_dim), 1.0, 0.0, seed, 2, dtype=torch.float32)
    return w["w_ada"].cuda(), w["b_ada"].cuda(), t_cond.cuda()


def test_noalloc_matches_workspace_entry_point_twice():
    assert torch.cuda.is_available()
    import audio_video_flow_gb300 as h3
    h3.lib()
    for shape, calls in [(hi.TINY_SHAPE, [(4, 11), (1, 12)]), (hi.H3_SHAPE, [(12, 13), (5, 14)])]:
        cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
        ws = torch.empty(h3.h3_adaln_table_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
        for T, seed in calls:          # two calls in a row; the second has fewer timestep rows
            w_ada, b_ada, t_cond = _case(shape, T, seed)
            ref = torch.empty(T, 18 * shape.dim, dtype=torch.bfloat16, device="cuda")
            out = torch.full_like(ref, float("nan"))
            h3.h3_adaln_table(cfg, w_ada, b_ada, t_cond, ref, ws)
            h3.h3_adaln_table_noalloc(cfg, w_ada, b_ada, t_cond, out)
            assert h3.h3_sync_check() == 0
            assert_close(to_np(out), to_np(ref), f"noalloc D={shape.dim} T={T}")


def test_noalloc_rejects_oversize_without_launching():
    import audio_video_flow_gb300 as h3
    big = h3.make_config(512, 4, 1536, 2816 + 64)
    x = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(h3.H3Error) as e:
        h3.h3_adaln_table_noalloc(big, x, None, x.reshape(1, -1), x)
    assert e.value.status == h3.H3_ERR_UNSUPPORTED
    ok = h3.make_config(512, 4, 1536, 256)
    with pytest.raises(h3.H3Error) as e:
        h3.h3_adaln_table_noalloc(ok, x, None, torch.zeros(17, 256, device="cuda"), x)
    assert e.value.status == h3.H3_ERR_UNSUPPORTED
