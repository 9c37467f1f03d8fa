"""Python binding of libh3, the GB300 (sm_103a) MiniMax-H3 block forward.

Argument marshalling only: every function here passes device pointers, sizes
and the current CUDA stream to the C ABI declared in include/h3.h and raises
H3Error on a non-OK status.  All arithmetic runs in the library's CUDA
kernels; there is no other code path.  PyTorch supplies device memory and
streams.
"""
from __future__ import annotations

import ctypes
import os
import re
from ctypes import c_float, c_int32, c_int64, c_size_t, c_void_p, c_char_p
from typing import Dict, Optional, Sequence

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
# H3_LIBRARY=bounds in the environment loads the bounds-checked build
# (libh3_bounds.so: every checked global access first tests that it lies in
# the buffer its call's arguments describe); otherwise the normal build.
LIB_PATH = os.path.join(PKG_DIR, "libh3_bounds.so" if os.environ.get("H3_LIBRARY") == "bounds" else "libh3.so")
HEADER = os.path.join(os.path.dirname(PKG_DIR), "include", "h3.h")

H3_OK, H3_ERR_NULL, H3_ERR_SHAPE, H3_ERR_ALIGN, H3_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
H3_ERR_INDEX, H3_ERR_CUDA, H3_ERR_TIMEOUT, H3_ERR_WORKSPACE, H3_ERR_BOUNDS = 5, 6, 7, 8, 9
N_STAGES = 8
STAGE_NAMES = ("adaln_table", "norm1_modulate", "qkv_qknorm_rope", "attention", "out_proj_residual",
               "norm2_modulate", "fc1_swiglu", "fc2_residual")


class H3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class BlockConfig(ctypes.Structure):
    _fields_ = [("dim", c_int32), ("n_heads", c_int32), ("head_dim", c_int32), ("ffn_dim", c_int32),
                ("cond_dim", c_int32), ("rope_freqs_per_axis", c_int32), ("rope_channels", c_int32),
                ("eps", c_float), ("rope_theta", c_float)]


_W_FIELDS = ("w_ada", "b_ada", "norm1_g", "norm2_g", "w_qkv", "b_qkv", "q_norm_g", "k_norm_g",
             "w_o", "b_o", "w_fc1", "b_fc1", "w_fc2", "b_fc2")


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in _W_FIELDS]


class PackedMeta(ctypes.Structure):
    _fields_ = [("n_rows", c_int32), ("n_timesteps", c_int32), ("token_tag", c_void_p),
                ("timestep_index", c_void_p), ("pos_thw", c_void_p), ("t_cond", c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libh3.so.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        i32, sz, vp = c_int32, c_size_t, c_void_p
        cfgp, wp, mp = ctypes.POINTER(BlockConfig), ctypes.POINTER(BlockWeights), ctypes.POINTER(PackedMeta)
        sig = {
            "h3_block_workspace_bytes": (sz, [cfgp, i32, i32]),
            "h3_block_adaln_side_ctas": (i32, [cfgp, i32]),
            "h3_block_forward": (i32, [cfgp, wp, mp, vp, vp, vp, sz, vp]),
            "h3_block_host_workspace_bytes": (sz, [cfgp, i32, i32]),
            "h3_blocks_host_workspace_bytes": (sz, [cfgp, i32, i32, i32]),
            "h3_blocks_workspace_bytes": (sz, [cfgp, i32, i32, i32]),
            "h3_blocks_kernel_count": (i32, [cfgp, i32, i32]),
            "h3_block_forward_host": (i32, [cfgp, wp, mp, vp, vp, vp, sz, vp]),
            "h3_blocks_forward_host": (i32, [cfgp, i32, wp, mp, vp, vp, vp, sz, vp]),
            "h3_block_forward_profiled": (i32, [cfgp, wp, mp, vp, vp, vp, sz, vp, vp, i32]),
            "h3_blocks_forward": (i32, [cfgp, i32, wp, mp, vp, vp, vp, sz, vp]),
            "h3_adaln_table_workspace_bytes": (sz, [cfgp]),
            "h3_adaln_table": (i32, [cfgp, vp, vp, vp, i32, vp, vp, sz, vp]),
            "h3_adaln_table_noalloc": (i32, [cfgp, vp, vp, vp, i32, vp, vp]),
            "h3_adaln_modulate": (i32, [cfgp, mp, vp, i32, vp, vp, vp, vp]),
            "h3_qkv_projection": (i32, [cfgp, mp, vp, vp, vp, vp, vp, vp, vp]),
            "h3_rope_qknorm": (i32, [cfgp, i32, vp, vp, vp, c_int64, c_int64, vp, vp, vp]),
            "h3_attention": (i32, [i32, i32, vp, vp, vp, c_int64, c_int64, vp, vp, vp]),
            "h3_out_projection": (i32, [cfgp, mp, vp, vp, vp, vp, vp, vp, vp]),
            "h3_ffn_up_swiglu": (i32, [cfgp, i32, vp, vp, vp, vp, vp]),
            "h3_ffn_down_residual": (i32, [cfgp, mp, vp, vp, vp, vp, vp, vp, vp]),
            "h3_linear": (i32, [i32, i32, i32, vp, vp, vp, vp, vp]),
            "h3_blocks_graph_create": (i32, [cfgp, i32, wp, mp, vp, vp, vp, sz, ctypes.POINTER(vp)]),
            "h3_graph_launch": (i32, [vp, vp]),
            "h3_graph_destroy": (i32, [vp]),
            "h3_patch_pack": (i32, [i32, i32, i32, i32, vp, vp, vp]),
            "h3_patch_unpack": (i32, [i32, i32, i32, i32, vp, vp, vp]),
            "h3_input_projection": (i32, [cfgp, i32, i32, vp, vp, vp, vp, i32, vp, vp]),
            "h3_packed_index_copy": (i32, [cfgp, i32, vp, vp, i32, vp, vp]),
            "h3_timestep_embedding": (i32, [cfgp, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
            "h3_refiner_workspace_bytes": (sz, [cfgp, i32]),
            "h3_refiner_forward": (i32, [cfgp, i32, wp, vp, i32, vp, vp, vp, sz, vp]),
            "h3_sigma_schedule": (i32, [i32, ctypes.c_float, vp, vp, vp]),
            "h3_ode_step": (i32, [c_int64, vp, vp, ctypes.c_float, ctypes.c_float, vp, vp]),
            "h3_noise_mix": (i32, [c_int64, vp, vp, ctypes.c_float, vp, vp]),
            "h3_select_rows": (i32, [i32, vp, i32, vp, vp, vp]),
            "h3_final_adaln_table": (i32, [cfgp, vp, vp, vp, i32, vp, vp]),
            "h3_final_adaln_tables": (i32, [cfgp, i32, vp, vp, vp, i32, vp, vp]),
            "h3_output_head": (i32, [cfgp, i32, i32, vp, vp, i32, vp, vp, vp, vp, i32, vp, vp]),
            "h3_sync_check": (i32, [vp, i32]),
            "h3_status_string": (c_char_p, [i32]),
            "h3_last_kernel_info": (i32, [ctypes.c_char_p, sz]),
            "h3_last_error_site": (i32, [ctypes.c_char_p, sz]),
            "h3_version": (c_char_p, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def declared_symbols() -> Sequence[str]:
    """Function names declared in include/h3.h."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|h3_status|size_t)\s*\**\s*(h3_\w+)\s*\(",
                                 txt, flags=re.M)))


def status_string(status: int) -> str:
    try:
        return lib().h3_status_string(status).decode()
    except Exception:  # library missing: still give a readable message
        return f"status {status}"


def _check(status: int, where: str) -> None:
    if status != H3_OK:
        raise H3Error(status, where)


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(dim: int, n_heads: int, ffn_dim: int, cond_dim: int, head_dim: int = 128,
                eps: float = 1e-5, rope_theta: float = 10000.0) -> BlockConfig:
    return BlockConfig(dim, n_heads, head_dim, ffn_dim, cond_dim, 16, 96, eps, rope_theta)


def make_weights(w: Dict[str, object]) -> BlockWeights:
    """Struct of device pointers; it keeps the tensors alive while it lives."""
    s = BlockWeights(*[_ptr(w.get(n)) for n in _W_FIELDS])
    s._tensors = [w.get(n) for n in _W_FIELDS]
    return s


def make_meta(token_tag, timestep_index, pos_thw, t_cond=None, n_timesteps: int = 0) -> PackedMeta:
    """Struct of the tensors' pointers (device ones, or host ones for
    h3_block_forward_host); it keeps the tensors alive while it lives."""
    s = PackedMeta(int(token_tag.shape[0]), int(n_timesteps), _ptr(token_tag), _ptr(timestep_index),
                   _ptr(pos_thw), _ptr(t_cond))
    s._tensors = (token_tag, timestep_index, pos_thw, t_cond)
    return s


# ---------------------------------------------------------------------------
# the C ABI, one Python function per entry point
# ---------------------------------------------------------------------------

def h3_block_workspace_bytes(cfg: BlockConfig, n_rows: int, n_timesteps: int) -> int:
    return int(lib().h3_block_workspace_bytes(ctypes.byref(cfg), n_rows, n_timesteps))


def h3_blocks_kernel_count(cfg: BlockConfig, n_blocks: int, n_rows: int) -> int:
    return int(lib().h3_blocks_kernel_count(ctypes.byref(cfg), n_blocks, n_rows))


def h3_block_adaln_side_ctas(cfg: BlockConfig, n_rows: int) -> int:
    return int(lib().h3_block_adaln_side_ctas(ctypes.byref(cfg), n_rows))


def h3_block_forward(cfg, weights, meta, x_in, x_out, workspace, stream=None) -> None:
    _check(lib().h3_block_forward(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(meta), _ptr(x_in),
                                  _ptr(x_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)), "h3_block_forward")


def h3_block_host_workspace_bytes(cfg: BlockConfig, n_rows: int, n_timesteps: int) -> int:
    return int(lib().h3_block_host_workspace_bytes(ctypes.byref(cfg), n_rows, n_timesteps))


def h3_blocks_workspace_bytes(cfg: BlockConfig, n_blocks: int, n_rows: int, n_timesteps: int) -> int:
    return int(lib().h3_blocks_workspace_bytes(ctypes.byref(cfg), n_blocks, n_rows, n_timesteps))


def h3_blocks_host_workspace_bytes(cfg: BlockConfig, n_blocks: int, n_rows: int, n_timesteps: int) -> int:
    return int(lib().h3_blocks_host_workspace_bytes(ctypes.byref(cfg), n_blocks, n_rows, n_timesteps))


def h3_block_forward_host(cfg, weights, meta_host, x_host, y_host, workspace, stream=None) -> None:
    """meta_host: make_meta() of host (preferably pinned) tensors; x_host,
    y_host: host bf16 [S][D]; weights and workspace on the device."""
    _check(lib().h3_block_forward_host(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(meta_host),
                                       _ptr(x_host), _ptr(y_host), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "h3_block_forward_host")


def h3_blocks_forward_host(cfg, weights_list, meta_host, x_host, y_host, workspace, stream=None) -> None:
    arr = (BlockWeights * len(weights_list))(*weights_list)
    _check(lib().h3_blocks_forward_host(ctypes.byref(cfg), len(weights_list), arr, ctypes.byref(meta_host),
                                        _ptr(x_host), _ptr(y_host), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)),
           "h3_blocks_forward_host")


def h3_block_forward_profiled(cfg, weights, meta, x_in, x_out, workspace, events, stream=None) -> None:
    arr = (c_void_p * len(events))(*[e.cuda_event if hasattr(e, "cuda_event") else e for e in events])
    _check(lib().h3_block_forward_profiled(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(meta),
                                           _ptr(x_in), _ptr(x_out), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream),
                                           arr, len(events)), "h3_block_forward_profiled")


def h3_blocks_forward(cfg, weights_list: Sequence[BlockWeights], meta, x_in, x_out, workspace,
                      stream=None) -> None:
    arr = (BlockWeights * len(weights_list))(*weights_list)
    _check(lib().h3_blocks_forward(ctypes.byref(cfg), len(weights_list), arr, ctypes.byref(meta), _ptr(x_in),
                                   _ptr(x_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "h3_blocks_forward")


class BlocksGraph:
    """A captured chain of blocks (h3_blocks_graph_create); launch() replays it.
    Keeps the weight structs and tensors it was captured with alive."""

    def __init__(self, cfg, weights_list: Sequence[BlockWeights], meta, x_in, x_out, workspace):
        self._keep = (cfg, list(weights_list), meta, x_in, x_out, workspace)
        arr = (BlockWeights * len(weights_list))(*weights_list)
        self._arr = arr
        h = c_void_p()
        _check(lib().h3_blocks_graph_create(ctypes.byref(cfg), len(weights_list), arr, ctypes.byref(meta),
                                            _ptr(x_in), _ptr(x_out), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), ctypes.byref(h)),
               "h3_blocks_graph_create")
        self._h = h

    def launch(self, stream=None) -> None:
        _check(lib().h3_graph_launch(self._h, _stream(stream)), "h3_graph_launch")

    def close(self) -> None:
        if self._h is not None and self._h.value:
            lib().h3_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def h3_adaln_table_workspace_bytes(cfg: BlockConfig) -> int:
    return int(lib().h3_adaln_table_workspace_bytes(ctypes.byref(cfg)))


def h3_adaln_table(cfg, w_ada, b_ada, t_cond, table_out, workspace, stream=None) -> None:
    _check(lib().h3_adaln_table(ctypes.byref(cfg), _ptr(w_ada), _ptr(b_ada), _ptr(t_cond), int(t_cond.shape[0]),
                                _ptr(table_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream)), "h3_adaln_table")


def h3_adaln_table_noalloc(cfg, w_ada, b_ada, t_cond, table_out, stream=None) -> None:
    """h3_adaln_table for callers that cannot allocate device memory: the
    library's own static scratch replaces the workspace (serialise calls)."""
    _check(lib().h3_adaln_table_noalloc(ctypes.byref(cfg), _ptr(w_ada), _ptr(b_ada), _ptr(t_cond),
                                        int(t_cond.shape[0]), _ptr(table_out), _stream(stream)),
           "h3_adaln_table_noalloc")


def h3_adaln_modulate(cfg, meta, table, branch: int, x, norm_g, h_out, stream=None) -> None:
    _check(lib().h3_adaln_modulate(ctypes.byref(cfg), ctypes.byref(meta), _ptr(table), branch, _ptr(x),
                                   _ptr(norm_g), _ptr(h_out), _stream(stream)), "h3_adaln_modulate")


def h3_qkv_projection(cfg, meta, h, w_qkv, b_qkv, q_norm_g, k_norm_g, qkv_out, stream=None) -> None:
    _check(lib().h3_qkv_projection(ctypes.byref(cfg), ctypes.byref(meta), _ptr(h), _ptr(w_qkv), _ptr(b_qkv),
                                   _ptr(q_norm_g), _ptr(k_norm_g), _ptr(qkv_out), _stream(stream)),
           "h3_qkv_projection")


def h3_rope_qknorm(cfg, n_rows: int, pos_thw, q, k, row_stride: int, head_stride: int, q_norm_g, k_norm_g,
                   stream=None) -> None:
    _check(lib().h3_rope_qknorm(ctypes.byref(cfg), n_rows, _ptr(pos_thw), _ptr(q), _ptr(k), row_stride,
                                head_stride, _ptr(q_norm_g), _ptr(k_norm_g), _stream(stream)), "h3_rope_qknorm")


def h3_attention(n_rows: int, n_heads: int, q, k, v, row_stride: int, head_stride: int, o, lse=None,
                 stream=None) -> None:
    _check(lib().h3_attention(n_rows, n_heads, _ptr(q), _ptr(k), _ptr(v), row_stride, head_stride, _ptr(o),
                              _ptr(lse), _stream(stream)), "h3_attention")


def h3_out_projection(cfg, meta, table, o, w_o, b_o, x, x_out, stream=None) -> None:
    _check(lib().h3_out_projection(ctypes.byref(cfg), ctypes.byref(meta), _ptr(table), _ptr(o), _ptr(w_o),
                                   _ptr(b_o), _ptr(x), _ptr(x_out), _stream(stream)), "h3_out_projection")


def h3_ffn_up_swiglu(cfg, n_rows: int, h, w_fc1, b_fc1, a_out, stream=None) -> None:
    _check(lib().h3_ffn_up_swiglu(ctypes.byref(cfg), n_rows, _ptr(h), _ptr(w_fc1), _ptr(b_fc1), _ptr(a_out),
                                  _stream(stream)), "h3_ffn_up_swiglu")


def h3_ffn_down_residual(cfg, meta, table, a, w_fc2, b_fc2, x1, y_out, stream=None) -> None:
    _check(lib().h3_ffn_down_residual(ctypes.byref(cfg), ctypes.byref(meta), _ptr(table), _ptr(a), _ptr(w_fc2),
                                      _ptr(b_fc2), _ptr(x1), _ptr(y_out), _stream(stream)), "h3_ffn_down_residual")


def h3_linear(M: int, N: int, K: int, x, w, b, y, stream=None) -> None:
    _check(lib().h3_linear(M, N, K, _ptr(x), _ptr(w), _ptr(b), _ptr(y), _stream(stream)), "h3_linear")


def h3_patch_pack(C: int, T: int, H: int, W: int, latent, rows, stream=None) -> None:
    _check(lib().h3_patch_pack(C, T, H, W, _ptr(latent), _ptr(rows), _stream(stream)), "h3_patch_pack")


def h3_patch_unpack(C: int, T: int, H: int, W: int, rows, latent, stream=None) -> None:
    _check(lib().h3_patch_unpack(C, T, H, W, _ptr(rows), _ptr(latent), _stream(stream)), "h3_patch_unpack")


def h3_input_projection(cfg, n: int, K: int, src, w, b, dst_rows, n_rows: int, x_out, stream=None) -> None:
    _check(lib().h3_input_projection(ctypes.byref(cfg), n, K, _ptr(src), _ptr(w), _ptr(b), _ptr(dst_rows), n_rows,
                                     _ptr(x_out), _stream(stream)), "h3_input_projection")


def h3_packed_index_copy(cfg, n: int, src, dst_rows, n_rows: int, x_out, stream=None) -> None:
    _check(lib().h3_packed_index_copy(ctypes.byref(cfg), n, _ptr(src), _ptr(dst_rows), n_rows, _ptr(x_out),
                                      _stream(stream)), "h3_packed_index_copy")


def h3_timestep_embedding(cfg, n_timesteps: int, t, w1, b1, w2, b2, scratch, t_cond, stream=None) -> None:
    _check(lib().h3_timestep_embedding(ctypes.byref(cfg), n_timesteps, _ptr(t), _ptr(w1), _ptr(b1), _ptr(w2),
                                       _ptr(b2), _ptr(scratch), _ptr(t_cond), _stream(stream)),
           "h3_timestep_embedding")


def h3_refiner_workspace_bytes(cfg: BlockConfig, n_rows: int) -> int:
    return int(lib().h3_refiner_workspace_bytes(ctypes.byref(cfg), n_rows))


def h3_refiner_forward(cfg, weights_list: Sequence[BlockWeights], final_norm_g, n_rows: int, x_in, x_out,
                       workspace, stream=None) -> None:
    arr = (BlockWeights * max(len(weights_list), 1))(*weights_list)
    _check(lib().h3_refiner_forward(ctypes.byref(cfg), len(weights_list), arr, _ptr(final_norm_g), n_rows,
                                    _ptr(x_in), _ptr(x_out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "h3_refiner_forward")


def h3_sigma_schedule(n_points: int, shift: float, sigmas, n_sigmas, stream=None) -> None:
    _check(lib().h3_sigma_schedule(n_points, shift, _ptr(sigmas), _ptr(n_sigmas), _stream(stream)),
           "h3_sigma_schedule")


def h3_ode_step(n: int, xt, v, sigma: float, sigma_next: float, x_next, stream=None) -> None:
    _check(lib().h3_ode_step(n, _ptr(xt), _ptr(v), sigma, sigma_next, _ptr(x_next), _stream(stream)), "h3_ode_step")


def h3_noise_mix(n: int, x0, noise, t: float, out, stream=None) -> None:
    _check(lib().h3_noise_mix(n, _ptr(x0), _ptr(noise), t, _ptr(out), _stream(stream)), "h3_noise_mix")


def h3_select_rows(n_rows: int, token_tag, tag: int, rows, n_selected, stream=None) -> None:
    _check(lib().h3_select_rows(n_rows, _ptr(token_tag), tag, _ptr(rows), _ptr(n_selected), _stream(stream)),
           "h3_select_rows")


def h3_final_adaln_table(cfg, w_fin, b_fin, t_cond, n_timesteps: int, table, stream=None) -> None:
    _check(lib().h3_final_adaln_table(ctypes.byref(cfg), _ptr(w_fin), _ptr(b_fin), _ptr(t_cond), n_timesteps,
                                      _ptr(table), _stream(stream)), "h3_final_adaln_table")


def h3_final_adaln_tables(cfg, w_fin, b_fin, t_cond, n_timesteps: int, tables, stream=None) -> None:
    """w_fin, b_fin (or None) and tables: sequences of the same length (the
    modalities), passed as host arrays of device pointers."""
    n = len(w_fin)
    arr = ctypes.c_void_p * max(n, 1)
    w_a = arr(*[_ptr(w) for w in w_fin])
    b_a = None if b_fin is None else arr(*[_ptr(b) for b in b_fin])
    t_a = arr(*[_ptr(t) for t in tables])
    _check(lib().h3_final_adaln_tables(ctypes.byref(cfg), n, ctypes.cast(w_a, ctypes.c_void_p),
                                       None if b_a is None else ctypes.cast(b_a, ctypes.c_void_p), _ptr(t_cond),
                                       n_timesteps, ctypes.cast(t_a, ctypes.c_void_p), _stream(stream)),
           "h3_final_adaln_tables")


def h3_output_head(cfg, n_rows: int, n_sel: int, rows, timestep_index, n_timesteps: int, x, table, w_head, b_head,
                   P: int, v_out, stream=None) -> None:
    _check(lib().h3_output_head(ctypes.byref(cfg), n_rows, n_sel, _ptr(rows), _ptr(timestep_index), n_timesteps,
                                _ptr(x), _ptr(table), _ptr(w_head), _ptr(b_head), P, _ptr(v_out),
                                _stream(stream)), "h3_output_head")


def h3_sync_check(stream=None, timeout_ms: int = 10000) -> int:
    """Returns the status (does not raise): H3_OK, H3_ERR_INDEX, H3_ERR_TIMEOUT or H3_ERR_CUDA."""
    return int(lib().h3_sync_check(_stream(stream), timeout_ms))


def h3_last_kernel_info() -> str:
    buf = ctypes.create_string_buffer(512)
    lib().h3_last_kernel_info(buf, 512)
    return buf.value.decode()


def h3_last_error_site() -> str:
    """Where the first device wait that ran out was (read by the last
    h3_sync_check that returned H3_ERR_TIMEOUT), or "none"."""
    buf = ctypes.create_string_buffer(128)
    lib().h3_last_error_site(buf, 128)
    return buf.value.decode()


def h3_version() -> str:
    return lib().h3_version().decode()
