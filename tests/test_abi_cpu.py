"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/h3.h declares, and rejects bad arguments on the host before
anything would be launched (fail closed)."""
import ctypes

import pytest

import audio_video_flow_gb300 as h3
from audio_video_flow_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()      # no-op when up to date
    return h3.lib()


def test_exports_every_declared_symbol(lib):
    names = h3.declared_symbols()
    assert len(names) >= 17
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    for n in ["h3_block_forward", "h3_attention", "h3_rope_qknorm", "h3_adaln_modulate"]:
        assert n in names


def test_status_strings(lib):
    for s in range(10):
        assert h3.status_string(s)
    assert "closed" in h3.status_string(h3.H3_ERR_UNSUPPORTED)
    assert h3.h3_version().startswith("libh3")


def test_workspace_bytes_and_config_validation(lib):
    cfg = h3.make_config(5376, 56, 14336, 2688)
    n = h3.h3_block_workspace_bytes(cfg, 505, 12)
    D, I, F, S, T = 5376, 7168, 14336, 505, 12
    at_least = 2 * (16 * 2688 + T * 18 * D + S * D + S * max(3 * I, F) + S * I + S * D)
    # plus the stream-K scratch of the residual GEMMs: per resident CTA pair one
    # 2 x 128 x 256 fp32 partial slot and 16 flags (none without a GPU)
    sk_per_pair = 2 * 128 * 256 * 4 + 16 * 4
    assert at_least <= n < at_least + 8 * 256 + 256 * sk_per_pair
    assert h3.h3_block_workspace_bytes(cfg, 0, 12) == 0
    assert h3.h3_block_workspace_bytes(cfg, 10, 17) == 0
    # a chain needs at least one block's workspace, at most that plus every
    # block's table; its host variant adds the staging
    nb = h3.h3_blocks_workspace_bytes(cfg, 50, 505, 12)
    assert n <= nb <= n + 50 * (12 * 18 * D * 2 + 256)
    assert h3.h3_blocks_workspace_bytes(cfg, 1, 505, 12) == n
    assert h3.h3_blocks_host_workspace_bytes(cfg, 50, 505, 12) > nb
    assert h3.h3_blocks_workspace_bytes(cfg, 0, 505, 12) == 0
    assert h3.h3_blocks_host_workspace_bytes(cfg, 3, 505, 17) == 0
    for bad in [h3.make_config(5376, 56, 14336, 2688, head_dim=64),
                h3.make_config(5376 + 32, 56, 14336, 2688),
                h3.make_config(5376, 56, 14336 + 64, 2688),
                h3.make_config(5376, 56, 14336, 2688 + 32),
                h3.make_config(5376, 0, 14336, 2688)]:
        assert h3.h3_block_workspace_bytes(bad, 10, 1) == 0


def test_host_rejections_return_before_any_launch(lib):
    cfg = h3.make_config(512, 4, 1536, 256)
    bad = h3.make_config(512, 4, 1536, 256, head_dim=96)
    meta = h3.PackedMeta(0, 1, None, None, None, None)
    w = h3.BlockWeights()
    nul = ctypes.c_void_p(None)
    L = lib
    assert L.h3_block_forward(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(meta), None, None, None, 0,
                              None) == h3.H3_ERR_UNSUPPORTED
    assert L.h3_block_forward(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(meta), None, None, None, 0,
                              None) == h3.H3_ERR_SHAPE
    meta = h3.PackedMeta(8, 1, 16, 32, 48, 64)
    assert L.h3_block_forward(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(meta), 16, 32, 256, 1 << 30,
                              None) == h3.H3_ERR_NULL
    meta17 = h3.PackedMeta(8, 17, 16, 32, 48, 64)
    assert L.h3_block_forward(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(meta17), 16, 32, 256, 1 << 30,
                              None) == h3.H3_ERR_UNSUPPORTED
    assert L.h3_attention(0, 4, 16, 16, 16, 1536, 384, 16, None, None) == h3.H3_ERR_SHAPE
    assert L.h3_attention(8, 4, None, 16, 16, 1536, 384, 16, None, None) == h3.H3_ERR_NULL
    assert L.h3_attention(8, 4, 16, 16, 16, 1537, 384, 16, None, None) == h3.H3_ERR_ALIGN
    assert L.h3_attention(8, 4, 24, 16, 16, 1536, 384, 16, None, None) == h3.H3_ERR_ALIGN
    assert L.h3_rope_qknorm(ctypes.byref(cfg), 8, 16, 16, 16, 1540, 384, 16, 16, None) == h3.H3_ERR_ALIGN
    assert L.h3_linear(0, 8, 64, 16, 16, None, 16, None) == h3.H3_ERR_SHAPE
    assert L.h3_linear(8, 8, 96, 16, 16, None, 16, None) == h3.H3_ERR_UNSUPPORTED
    assert L.h3_adaln_modulate(ctypes.byref(cfg), ctypes.byref(meta), 16, 2, 16, 16, 16, None) == h3.H3_ERR_SHAPE
    assert L.h3_adaln_table(ctypes.byref(cfg), 16, None, 16, 17, 16, 256, 1 << 20, None) == h3.H3_ERR_UNSUPPORTED
    assert L.h3_adaln_table(ctypes.byref(cfg), 16, None, 16, 4, 16, 256, 16, None) == h3.H3_ERR_WORKSPACE
    assert L.h3_adaln_table_workspace_bytes(ctypes.byref(cfg)) == 16 * 256 * 2
    ptrs = (ctypes.c_void_p * 5)(16, 32, 48, 64, 80)
    ptrs_null = (ctypes.c_void_p * 2)(16, None)
    assert L.h3_final_adaln_tables(ctypes.byref(cfg), 0, ptrs, None, 16, 1, ptrs, None) == h3.H3_ERR_UNSUPPORTED
    assert L.h3_final_adaln_tables(ctypes.byref(cfg), 5, ptrs, None, 16, 1, ptrs, None) == h3.H3_ERR_UNSUPPORTED
    assert L.h3_final_adaln_tables(ctypes.byref(cfg), 2, ptrs, None, 16, 17, ptrs, None) == h3.H3_ERR_UNSUPPORTED
    assert L.h3_final_adaln_tables(ctypes.byref(cfg), 2, None, None, 16, 1, ptrs, None) == h3.H3_ERR_NULL
    assert L.h3_final_adaln_tables(ctypes.byref(cfg), 2, ptrs, None, 16, 1, ptrs_null, None) == h3.H3_ERR_NULL
    assert L.h3_final_adaln_tables(ctypes.byref(cfg), 2, ptrs_null, None, 16, 1, ptrs, None) == h3.H3_ERR_NULL
    ptrs_odd = (ctypes.c_void_p * 2)(16, 40)
    assert L.h3_final_adaln_tables(ctypes.byref(cfg), 2, ptrs_odd, None, 16, 1, ptrs, None) == h3.H3_ERR_ALIGN
    buf = ctypes.create_string_buffer(64)
    assert L.h3_last_kernel_info(None, 0) == h3.H3_ERR_NULL
    assert L.h3_last_kernel_info(buf, 64) == h3.H3_OK
    assert L.h3_last_error_site(None, 0) == h3.H3_ERR_NULL
    assert L.h3_last_error_site(buf, 64) == h3.H3_OK and buf.value == b"none"


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(h3, "_lib", None)
    monkeypatch.setattr(h3, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        h3.lib()
