"""Benchmark of the H3 block forward on GB300.

One step = one pass of the whole hot path over one packed document: the AdaLN
table, norm1/modulate, QKV + QK-norm + MM-RoPE, attention, O projection +
gated residual, norm2/modulate, FC1 + SwiGLU, FC2 + gated residual, for every
block of the workload.  Default workload: one velocity evaluation of the
denoiser, 50 full-width blocks over 15,860 packed rows (256 text + 14,580
video on a 36x15x27 latent grid + 1,024 audio, one timestep row), about
64.5 GB of bf16 weights resident on the GPU.  `--workload block505` (and the
others in h3_inputs.WORKLOADS) selects another shape.

Prints ONE JSON line (rank 0).  `value` is whole-job TFLOP/s of algorithmic
work (dense GEMMs, full attention, AdaLN projection) measured with CUDA events
on the launching stream, max over ranks; `e2e` is the same metric with the
inputs copied host->device and the output device->host inside the timed
region.  `--impl reference` times the CPU oracle on the host cores instead.
Multi-GPU (torchrun): every rank runs an independent replica (the batch axis
is pure replication), so scaling is weak and no data-path collective exists.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "H3 block fwd TFLOP/s & packed tokens/s (bf16, 1 GB300); % of tensor/HBM roofline"
def launches_per_step(shape, S: int, n_blocks: int) -> int:
    """Kernels one h3_blocks_forward call launches (the library's own count)."""
    import audio_video_flow_gb300 as h3
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    return h3.h3_blocks_kernel_count(cfg, n_blocks, S)


STAGES = ("adaln_table", "norm1_modulate", "qkv_qknorm_rope", "attention", "out_proj_residual",
          "norm2_modulate", "fc1_swiglu", "fc2_residual")
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# kernel, from ncu captures of the current kernel build, keyed
# "stage@workload"; absent when not captured.  At 505 rows QKV and FC1 take
# turns as the longest stage, so both are here.  Attention's DRAM traffic is
# reading q, k, v and writing o once (K/V re-reads hit L2), so the 32,768-
# and 15,860-row values are the 16,384-row capture scaled by the row count.
TRAFFIC = {
    "qkv_qknorm_rope@block505": 252525312,
    "fc1_swiglu@block505": 332613888,
    "qkv_qknorm_rope@block1824": 328294144,
    "fc1_swiglu@block1824": 378740736,
    "attention@attn4096": 214936064,
    "attention@attn16384": 921477120,
    "attention@attn32768": 1842954240,
    "attention@denoiser15860": 892006050,
}


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def adaln_split(shape, S: int) -> bool:
    """True when the library computes AdaLN chunks 3-5 on its side stream."""
    import audio_video_flow_gb300 as h3
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    return h3.h3_block_adaln_side_ctas(cfg, S) > 0


def stage_work(shape, S: int, T: int, split: bool = False):
    """(flops, bytes) per stage of one block: the method's own dense work and
    the bytes each kernel must move at least once.  With the AdaLN split, the
    critical-path stage covers chunks 0-2 and adaln_table_side chunks 3-5."""
    D, I, F, C = shape.dim, shape.n_heads * shape.head_dim, shape.ffn_dim, shape.cond_dim
    b = 2  # bf16
    ada = (2.0 * T * C * 18 * D, 18 * D * C * b + T * C * 4 + T * 18 * D * b)
    frac = 3.0 / 6.0 if split else 1.0
    return {
        "adaln_table": (ada[0] * frac, ada[1] * frac),
        "adaln_table_side": (ada[0] * (1 - frac), ada[1] * (1 - frac)),
        "norm1_modulate": (0.0, 2.0 * S * D * b),
        "qkv_qknorm_rope": (2.0 * S * D * 3 * I, 3 * I * D * b + S * D * b + S * 3 * I * b),
        "attention": (4.0 * S * S * I, 4.0 * S * I * b),
        "out_proj_residual": (2.0 * S * I * D, D * I * b + S * I * b + 2 * S * D * b),
        "norm2_modulate": (0.0, 2.0 * S * D * b),
        "fc1_swiglu": (2.0 * S * D * 2 * F, 2 * F * D * b + S * D * b + S * F * b),
        "fc2_residual": (2.0 * S * F * D, D * F * b + S * F * b + 2 * S * D * b),
    }


def weight_bytes(shape):
    D, I, F, C = shape.dim, shape.n_heads * shape.head_dim, shape.ffn_dim, shape.cond_dim
    return 2 * (18 * D * C + 3 * I * D + D * I + 2 * F * D + D * F)


BOUND = {"adaln_table": "hbm", "adaln_table_side": "hbm", "norm1_modulate": "hbm", "norm2_modulate": "hbm", "qkv_qknorm_rope": "tensor",
         "attention": "tensor", "out_proj_residual": "tensor", "fc1_swiglu": "tensor", "fc2_residual": "tensor"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def tensor_peak(peaks, timed_ms: float):
    """bf16 denominator: the burst figure for a timed region shorter than a
    second, the sustained (power-capped) one for a region of a second or more."""
    if timed_ms >= 1000.0:
        return peaks["bf16_tflops_sustained"], peaks["source"] + " bf16 sustained"
    return peaks["bf16_tflops"], peaks["source"] + " bf16 burst"


# ---------------------------------------------------------------------------
# ranks (replicas): timing aggregation is the only cross-rank step
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(elapsed_ms: float, units: float, world_size: int):
    """Max elapsed time and summed work over ranks (host-side timing reduction)."""
    if world_size <= 1:
        return elapsed_ms, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world_size: int):
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[2]))
            except ValueError:
                pass
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
               "samples": len(sm)}
        # median board power, where the region held enough samples (2 s) for
        # the median to be taken under load rather than around it
        if len(pw) >= 20:
            out["power_w"] = round(statistics.median(pw), 1)
        return out


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_attention_core(args, ws_n: int, rank: int, local: int):
    """Attention core alone: per-head Q/K RMSNorm + MM-RoPE prologue (in place)
    and full non-causal attention over S packed rows, 56 heads."""
    import torch
    import audio_video_flow_gb300 as h3
    import h3_inputs as hi

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    wl = hi.WORKLOADS[args.workload]
    shape, S = wl.shape, wl.layout.n_rows
    H = shape.n_heads
    cfg = h3.make_config(shape.dim, H, shape.ffn_dim, shape.cond_dim)
    meta = hi.packed_metadata(wl.layout, 1, args.seed)
    ins = hi.attention_inputs(shape, S, args.seed, device=dev)
    qkv, qg, kg = ins["qkv"], ins["q_norm_g"], ins["k_norm_g"]
    pos = meta["pos_thw"].to(dev)
    o = torch.empty(S, H * 128, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    rs, hs = H * 384, 384
    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]

    def step(i=None):
        if i is not None:
            ev[i][0].record(stream)
        h3.h3_rope_qknorm(cfg, S, pos, q, k, rs, hs, qg, kg)
        if i is not None:
            ev[i][1].record(stream)
        h3.h3_attention(S, H, q, k, v, rs, hs, o)
        if i is not None:
            ev[i][2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flops = 4.0 * S * S * H * 128
    rope_bytes = 2.0 * 2 * S * H * 128 * 2
    with ClockSampler(local) as clk:
        barrier(ws_n)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(n):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_n)
    status = h3.h3_sync_check(timeout_ms=60000)
    if status != 0:
        raise RuntimeError(f"device error: {h3.status_string(status)}")
    elapsed_ms, units = aggregate(t0.elapsed_time(t1), n * flops, ws_n)
    rope_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    peaks = load_peaks()
    t_peak, t_src = tensor_peak(peaks, elapsed_ms)
    achieved = flops / (attn_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": round(units / (elapsed_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
        "n_gpus": ws_n, "steps": n, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / n, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": round(ws_n * S * n / (elapsed_ms * 1e-3), 1),
        "config": {"workload": wl.name, "description": wl.description, "rows": S, "heads": H,
                   "l2": "inputs larger than L2" if S * H * 384 * 2 > 129e6 else "inputs L2-resident",
                   "parallelism": f"replicas x{ws_n}"},
        "e2e": None, "gpu_launches": 2 * n,
        "roofline": {"kernel": "attention", "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": t_peak, "unit": "TFLOP/s",
                     "frac": round(achieved / t_peak, 4), "peak_source": t_src,
                     "traffic": TRAFFIC.get(f"attention@{wl.name}")},
        "stages": {"rope_qknorm": {"us": round(rope_ms * 1e3, 2),
                                   "gbs": round(rope_bytes / (rope_ms * 1e-3) / 1e9, 1),
                                   "hbm_frac": round(rope_bytes / (rope_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
                   "attention": {"us": round(attn_ms * 1e3, 2), "tflops": round(achieved, 1)}},
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline and ws_n == 1:
        try:
            st = OracleAttnStepper(wl, args.seed)
            n_st, dt, _ = time_stepper(st, args.cpu_seconds)
            line["cpu_baseline"] = {
                "value": round(n_st * st.step_flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_cores(),
                "kind": "oracle", "tokens_per_s": round(n_st * st.rows / dt, 2),
                "sample": f"{n_st * st.rows} query rows of {wl.name}, {st.rows} per step: Q norm + RoPE and attention "
                          f"over all {S} keys for {H} heads in fp64 numpy (every row's k and v computed before "
                          f"timing), {dt:.1f} s"}
        except Exception as e:   # the GPU line stands without the oracle's timing
            line["cpu_baseline"] = {"unavailable": f"{type(e).__name__}: {e}"}
    return line


FP32_LANES_PER_SM = 128   # fp32 FMA lanes per SM (4 sub-partitions x 32)


def alu_fp32_peak_tflops(sm_mhz: float, n_sms: int) -> float:
    """FP32 FMA peak: SMs x 128 lanes x 2 FLOP x clock."""
    return n_sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def run_output_side(args, ws_n: int, rank: int, local: int):
    """One evaluation's output side at the 15,860-row shape: row selection,
    FP32 final AdaLN table of both modalities, the FP32 velocity heads and the
    two Euler steps on the patch-packed fp32 latents."""
    import torch
    import audio_video_flow_gb300 as h3
    import h3_inputs as hi

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    wl = hi.WORKLOADS[args.workload]
    shape, S, T = wl.shape, wl.layout.n_rows, wl.n_timesteps
    D, C = shape.dim, shape.cond_dim
    cfg = h3.make_config(D, shape.n_heads, shape.ffn_dim, C)
    meta = {k: v.to(dev) for k, v in hi.packed_metadata(wl.layout, T, args.seed).items()}
    acts = hi.activations(shape, S, T, args.seed, device=dev)
    ow = hi.output_weights(shape, args.seed, device=dev)
    mods = [("video", 0, hi.VIDEO_PATCH, wl.layout.n_video), ("audio", 2, hi.AUDIO_PATCH, wl.layout.n_audio)]
    rows = {m: torch.empty(S, dtype=torch.int32, device=dev) for m, *_ in mods}
    cnt = {m: torch.zeros(1, dtype=torch.int32, device=dev) for m, *_ in mods}
    tab = {m: torch.empty(T, 2, D, dtype=torch.float32, device=dev) for m, *_ in mods}
    vel = {m: torch.empty(n, P, dtype=torch.float32, device=dev) for m, _, P, n in mods}
    lat = {m: hi.latents(n, P, args.seed, 74 + i, device=dev) for i, (m, _, P, n) in enumerate(mods)}
    sig = {"video": (0.9, 0.8), "audio": (0.75, 0.6)}
    stream = torch.cuda.current_stream()
    n = args.steps
    names = ["select_rows", "final_adaln_table", "output_head", "ode_step"]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(n)]

    def step(i=None):
        rec = (lambda k: ev[i][k].record(stream)) if i is not None else (lambda k: None)
        rec(0)
        for m, tag, P, nr in mods:
            h3.h3_select_rows(S, meta["token_tag"], tag, rows[m], cnt[m])
        rec(1)
        h3.h3_final_adaln_tables(cfg, [ow[f"w_fin_{m}"] for m, *_ in mods], [ow[f"b_fin_{m}"] for m, *_ in mods],
                                 acts["t_cond"], T, [tab[m] for m, *_ in mods])   # both modalities, one launch
        rec(2)
        for m, tag, P, nr in mods:
            h3.h3_output_head(cfg, S, nr, rows[m], meta["timestep_index"], T, acts["x"], tab[m],
                              ow[f"w_head_{m}"], ow[f"b_head_{m}"], P, vel[m])
        rec(3)
        for m, tag, P, nr in mods:
            h3.h3_ode_step(lat[m].numel(), lat[m], vel[m], sig[m][0], sig[m][1], lat[m])
        rec(4)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for e3 in ev:
        for e in e3:
            e.record(stream)
    head_flops = sum(2.0 * nr * P * D for _, _, P, nr in mods)
    table_bytes = 2 * (2 * D * C * 4)
    ode_bytes = sum(3 * 4 * nr * P for _, _, P, nr in mods)
    with ClockSampler(local) as clk:
        barrier(ws_n)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(n):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_n)
    status = h3.h3_sync_check(timeout_ms=60000)
    if status != 0:
        raise RuntimeError(f"device error: {h3.status_string(status)}")
    elapsed_ms, units = aggregate(t0.elapsed_time(t1), n * head_flops, ws_n)
    st = {nm: statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev) for k, nm in enumerate(names)}
    clocks = clk.summary()
    peak = alu_fp32_peak_tflops(clocks.get("sm_max_mhz") or 2070.0, torch.cuda.get_device_properties(dev).multi_processor_count)
    head_tf = head_flops / (st["output_head"] * 1e-3) / 1e12
    peaks = load_peaks()
    return {
        "metric": METRIC, "value": round(units / (elapsed_ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
        "n_gpus": ws_n, "steps": n, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / n, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "tokens_per_s": round(ws_n * S * n / (elapsed_ms * 1e-3), 1),
        "config": {"workload": wl.name, "description": wl.description, "rows": S,
                   "video_rows": wl.layout.n_video, "audio_rows": wl.layout.n_audio, "dim": D, "cond": C,
                   "flop_per_step": head_flops, "l2": "inputs larger than L2: 231 MB of fp32 final-AdaLN "
                   "weights re-read every step", "parallelism": f"replicas x{ws_n}"},
        "e2e": None, "gpu_launches": 7 * n,
        "roofline": {"kernel": "output_head", "bound": "alu", "achieved": round(head_tf, 2),
                     "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(head_tf / peak, 4),
                     "peak_source": "fp32 FMA lanes x 2 x max SM clock", "traffic": None},
        "stages": {
            "select_rows": {"us": round(st["select_rows"] * 1e3, 2)},
            "final_adaln_table": {"us": round(st["final_adaln_table"] * 1e3, 2),
                                  "gbs": round(table_bytes / (st["final_adaln_table"] * 1e-3) / 1e9, 1),
                                  "hbm_frac": round(table_bytes / (st["final_adaln_table"] * 1e-3) / 1e9
                                                    / peaks["hbm_gbs"], 4)},
            "output_head": {"us": round(st["output_head"] * 1e3, 2), "tflops": round(head_tf, 2)},
            "ode_step": {"us": round(st["ode_step"] * 1e3, 2),
                         "gbs": round(ode_bytes / (st["ode_step"] * 1e-3) / 1e9, 1)},
        },
        "clocks": clocks,
    }


def run_input_side(args, ws_n: int, rank: int, local: int):
    """One evaluation's input side at the 15,860-row shape: the video patch
    permutation, the FP32 video and audio input projections scattered into
    the packed stream, the BF16 text projection of the text rows and its
    scatter, and the timestep conditioning row."""
    import torch
    import audio_video_flow_gb300 as h3
    import h3_inputs as hi

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    wl = hi.WORKLOADS[args.workload]
    shape, S, T = wl.shape, wl.layout.n_rows, wl.n_timesteps
    D, C = shape.dim, shape.cond_dim
    cfg = h3.make_config(D, shape.n_heads, shape.ffn_dim, C)
    lay = wl.layout
    gt, gh, gw = lay.video_grid
    lat = hi.normal((24, gt, 2 * gh, 2 * gw), 1.0, 0.0, args.seed, 95, device=dev, dtype=torch.float32)
    vrows = torch.empty(lay.n_video, 96, dtype=torch.float32, device=dev)
    arows = hi.latents(lay.n_audio, 32, args.seed, 97, device=dev)
    text = hi.normal((lay.n_text, 5120), 1.0, 0.0, args.seed, 99, device=dev)
    w_text = hi.normal((D, 5120), 0.02, 0.0, args.seed, 100, device=dev)
    iw = hi.input_weights(shape, args.seed, device=dev)
    idx = torch.arange(S, dtype=torch.int32, device=dev)
    i_text, i_vid, i_aud = idx[:lay.n_text], idx[lay.n_text:lay.n_text + lay.n_video], idx[lay.n_text + lay.n_video:]
    t = torch.full((T,), 0.5, dtype=torch.float32, device=dev)
    x = torch.zeros(S, D, dtype=torch.bfloat16, device=dev)
    tproj = torch.empty(lay.n_text, D, dtype=torch.bfloat16, device=dev)
    scratch = torch.empty(T * (256 + D), dtype=torch.float32, device=dev)
    tc = torch.empty(T, C, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    names = ["patch_pack", "input_projection", "text_projection", "timestep_embedding"]
    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(n)]

    def step(i=None):
        rec = (lambda k: ev[i][k].record(stream)) if i is not None else (lambda k: None)
        rec(0)
        h3.h3_patch_pack(24, gt, 2 * gh, 2 * gw, lat, vrows)
        rec(1)
        h3.h3_input_projection(cfg, lay.n_video, 96, vrows, iw["w_in_video"], iw["b_in_video"], i_vid, S, x)
        h3.h3_input_projection(cfg, lay.n_audio, 32, arows, iw["w_in_audio"], iw["b_in_audio"], i_aud, S, x)
        rec(2)
        h3.h3_linear(lay.n_text, D, 5120, text, w_text, None, tproj)
        h3.h3_packed_index_copy(cfg, lay.n_text, tproj, i_text, S, x)
        rec(3)
        h3.h3_timestep_embedding(cfg, T, t, iw["w_t1"], iw["b_t1"], iw["w_t2"], iw["b_t2"], scratch, tc)
        rec(4)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for e3 in ev:
        for e in e3:
            e.record(stream)
    proj_flops = 2.0 * D * (lay.n_video * 96 + lay.n_audio * 32)
    text_flops = 2.0 * lay.n_text * 5120 * D
    mlp_bytes = 4 * (D * 256 + C * D)
    with ClockSampler(local) as clk:
        barrier(ws_n)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(n):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_n)
    status = h3.h3_sync_check(timeout_ms=60000)
    if status != 0:
        raise RuntimeError(f"device error: {h3.status_string(status)}")
    elapsed_ms, units = aggregate(t0.elapsed_time(t1), n * (proj_flops + text_flops), ws_n)
    st = {nm: statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev) for k, nm in enumerate(names)}
    clocks = clk.summary()
    peak = alu_fp32_peak_tflops(clocks.get("sm_max_mhz") or 2070.0,
                                torch.cuda.get_device_properties(dev).multi_processor_count)
    proj_tf = proj_flops / (st["input_projection"] * 1e-3) / 1e12
    peaks = load_peaks()
    return {
        "metric": METRIC, "value": round(units / (elapsed_ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
        "n_gpus": ws_n, "steps": n, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / n, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "tokens_per_s": round(ws_n * S * n / (elapsed_ms * 1e-3), 1),
        "config": {"workload": wl.name, "description": wl.description, "rows": S, "dim": D,
                   "flop_per_step": proj_flops + text_flops, "l2": "video latent and projections written "
                   "every step (157 MB of bf16 rows)", "parallelism": f"replicas x{ws_n}"},
        "e2e": None, "gpu_launches": 7 * n,
        "roofline": {"kernel": "input_projection", "bound": "alu", "achieved": round(proj_tf, 2),
                     "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(proj_tf / peak, 4),
                     "peak_source": "fp32 FMA lanes x 2 x max SM clock", "traffic": None},
        "stages": {
            "patch_pack": {"us": round(st["patch_pack"] * 1e3, 2),
                           "gbs": round(2 * 4 * lat.numel() / (st["patch_pack"] * 1e-3) / 1e9, 1)},
            "input_projection": {"us": round(st["input_projection"] * 1e3, 2), "tflops": round(proj_tf, 2)},
            "text_projection": {"us": round(st["text_projection"] * 1e3, 2),
                                "tflops": round(text_flops / (st["text_projection"] * 1e-3) / 1e12, 1)},
            "timestep_embedding": {"us": round(st["timestep_embedding"] * 1e3, 2),
                                   "gbs": round(mlp_bytes / (st["timestep_embedding"] * 1e-3) / 1e9, 1),
                                   "hbm_frac": round(mlp_bytes / (st["timestep_embedding"] * 1e-3) / 1e9
                                                     / peaks["hbm_gbs"], 4)},
        },
        "clocks": clocks,
    }


def run_refiner(args, ws_n: int, rank: int, local: int):
    """The 2-layer token refiner and its final RMSNorm over the text rows."""
    import torch
    import audio_video_flow_gb300 as h3
    import h3_inputs as hi

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    wl = hi.WORKLOADS[args.workload]
    shape, S, NB = wl.shape, wl.layout.n_rows, wl.n_blocks
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    wts = [hi.block_weights(shape, args.seed, 60 + b, device=dev) for b in range(NB)]
    for w in wts:
        w["w_ada"] = w["b_ada"] = None          # the refiner has no AdaLN
    cw = [h3.make_weights(w) for w in wts]
    gfin = hi.normal((shape.dim,), 0.1, 1.0, args.seed, 90, device=dev)
    x = hi.normal((S, shape.dim), 1.0, 0.0, args.seed, 91, device=dev)
    y = torch.empty_like(x)
    ws = torch.empty(h3.h3_refiner_workspace_bytes(cfg, S), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    work = stage_work(shape, S, 1)
    flops_step = NB * sum(f for k, (f, _) in work.items() if k != "adaln_table")
    for _ in range(args.warmup):
        h3.h3_refiner_forward(cfg, cw, gfin, S, x, y, ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        barrier(ws_n)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            h3.h3_refiner_forward(cfg, cw, gfin, S, x, y, ws)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_n)
    status = h3.h3_sync_check(timeout_ms=60000)
    if status != 0:
        raise RuntimeError(f"device error: {h3.status_string(status)}")
    elapsed_ms, units = aggregate(t0.elapsed_time(t1), args.steps * flops_step, ws_n)
    peaks = load_peaks()
    t_peak, t_src = tensor_peak(peaks, elapsed_ms)
    achieved = units / (elapsed_ms * 1e-3) / 1e12
    return {
        "metric": METRIC, "value": round(achieved, 3), "unit": "TFLOP/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": round(ws_n * S * args.steps / (elapsed_ms * 1e-3), 1),
        "config": {"workload": wl.name, "description": wl.description, "rows": S, "blocks": NB,
                   "dim": shape.dim, "heads": shape.n_heads, "ffn": shape.ffn_dim, "flop_per_step": flops_step,
                   "l2": "inputs larger than L2: %.2f GB of refiner weights re-read every step" %
                         (NB * (weight_bytes(shape) - 2 * 18 * shape.dim * shape.cond_dim) / 1e9),
                   "parallelism": f"replicas x{ws_n}"},
        "e2e": None, "gpu_launches": args.steps * (1 + 7 * NB + 1),
        "roofline": {"kernel": "refiner_step", "bound": "tensor", "achieved": round(achieved, 1), "peak": t_peak,
                     "unit": "TFLOP/s", "frac": round(achieved / t_peak, 4), "peak_source": t_src,
                     "traffic": None, "note": "whole step (all launches), not one kernel"},
        "clocks": clk.summary(),
    }


def run_ours(args, ws_n: int, rank: int, local: int):
    import torch
    import audio_video_flow_gb300 as h3
    import h3_inputs as hi

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    wl = hi.WORKLOADS[args.workload]
    if wl.name.startswith("attn"):
        return run_attention_core(args, ws_n, rank, local)
    if wl.name.startswith("output"):
        return run_output_side(args, ws_n, rank, local)
    if wl.name.startswith("refiner"):
        return run_refiner(args, ws_n, rank, local)
    if wl.name.startswith("input"):
        return run_input_side(args, ws_n, rank, local)
    shape, S, T, NB = wl.shape, wl.layout.n_rows, wl.n_timesteps, wl.n_blocks
    cfg = h3.make_config(shape.dim, shape.n_heads, shape.ffn_dim, shape.cond_dim)
    meta_c, acts_c, _ = hi.workload_inputs(wl, seed=args.seed, device="cpu", block=0) if NB == 1 else \
        (hi.packed_metadata(wl.layout, T, args.seed), hi.activations(shape, S, T, args.seed), None)
    if NB == 1:
        wts = [hi.block_weights(shape, args.seed, 0, device=dev)]
    else:   # 50 blocks: generated on the device (about 1.3 GB each)
        wts = [hi.block_weights(shape, args.seed, b, device=dev) for b in range(NB)]
    cw = [h3.make_weights(w) for w in wts]
    meta_d = {k: v.to(dev) for k, v in meta_c.items()}
    x = acts_c["x"].to(dev)
    tc = acts_c["t_cond"].to(dev)
    y = torch.empty_like(x)
    meta = h3.make_meta(meta_d["token_tag"], meta_d["timestep_index"], meta_d["pos_thw"], tc, T)
    wsp = torch.empty(h3.h3_blocks_workspace_bytes(cfg, NB, S, T), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # one set of stage events per timed step and block: the per-kernel launch
    # durations are read from the timed region itself
    # per step and block: start, 8 stage ends, side-stream start and end
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 3)] for _ in range(NB)]
          for _ in range(args.steps)]
    # torch only reports elapsed time between events it has recorded itself:
    # record each once here; inside the timed region the library re-records
    # the stage events after each launch (the latest record is what counts).
    for e3 in ev:
        for e2 in e3:
            for e in e2:
                e.record(stream)

    def step(i=None):
        if i is None:     # the evaluation as a user runs it: one chain call
            h3.h3_blocks_forward(cfg, cw, meta, x, y, wsp)
            return
        for b in range(NB):   # per-block calls with an event after every launch
            ev[i][b][0].record(stream)
            h3.h3_block_forward_profiled(cfg, cw[b], meta, x if b == 0 else y, y, wsp, ev[i][b][1:])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if h3.h3_sync_check(timeout_ms=60000) != 0:
        raise RuntimeError("device error during warm-up")

    split = adaln_split(shape, S)
    work = stage_work(shape, S, T, split)
    flops_step = NB * sum(f for f, _ in work.values())

    # ---- timed region (device time on the launching stream).  The headline
    # value comes from K plain steps: an event recorded between two launches
    # would cut the programmatic overlap of consecutive kernels.  A second
    # timed pass of K steps records an event after every launch and gives the
    # per-kernel times (and the dominant kernel's roofline).
    with ClockSampler(local) as clk:
        barrier(ws_n)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        host0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        host1 = time.perf_counter()
        barrier(ws_n)
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for i in range(args.steps):
            step(i)
        s1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_n)
    elapsed_ms = t0.elapsed_time(t1)
    instrumented_ms = s0.elapsed_time(s1)
    status = h3.h3_sync_check(timeout_ms=60000)
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {h3.status_string(status)}")
    stage_ms = {}
    for k, s in enumerate(STAGES):
        stage_ms[s] = statistics.mean(ev[i][b][k].elapsed_time(ev[i][b][k + 1])
                                      for i in range(args.steps) for b in range(NB))
    side_ms = None
    if split:
        side_ms = statistics.mean(ev[i][b][9].elapsed_time(ev[i][b][10])
                                  for i in range(args.steps) for b in range(NB))

    elapsed_ms, units = aggregate(elapsed_ms, float(args.steps) * flops_step, ws_n)
    ms_per_step = elapsed_ms / args.steps
    tflops = units / (elapsed_ms * 1e-3) / 1e12
    tokens_per_s = ws_n * S * args.steps / (elapsed_ms * 1e-3)

    # ---- end to end through the host-buffer entry point: pinned host input
    # and metadata copied in, the block(s), the output copied back, all inside
    # one h3_blocks_forward_host call per step
    e2e = None
    if not args.no_e2e:
        h_x = acts_c["x"].pin_memory()
        h_meta = {k: v.pin_memory() for k, v in meta_c.items()}
        h_tc = acts_c["t_cond"].pin_memory()
        h_y = torch.empty_like(acts_c["x"]).pin_memory()
        meta_h = h3.make_meta(h_meta["token_tag"], h_meta["timestep_index"], h_meta["pos_thw"], h_tc, T)
        ws_h = torch.empty(h3.h3_blocks_host_workspace_bytes(cfg, NB, S, T), dtype=torch.uint8, device=dev)
        bi = h_x.numel() * 2 + h_tc.numel() * 4 + sum(v.numel() * 4 for v in h_meta.values())
        bo = h_y.numel() * 2
        n_e2e = max(3, min(args.steps, 200))

        def e2e_step():
            h3.h3_blocks_forward_host(cfg, cw, meta_h, h_x, h_y, ws_h)

        for _ in range(3):
            e2e_step()
        with ClockSampler(local) as clk_e2e:   # the e2e pass runs later, on a warmer GPU
            barrier(ws_n)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n_e2e):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize()
            barrier(ws_n)
        e_ms, e_units = aggregate(e0.elapsed_time(e1), float(n_e2e) * flops_step, ws_n)
        ce = clk_e2e.summary()
        e2e = {"value": round(e_units / (e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
               "ms_per_step": round(e_ms / n_e2e, 4), "steps": n_e2e,
               "clocks": {"sm_mhz": ce["sm_mhz"], "reasons": ce["reasons"]}}

    # ---- roofline of the dominant kernel
    peaks = load_peaks()
    dom = max(STAGES, key=lambda s: stage_ms[s])
    fl, by = work[dom]
    d_ms = stage_ms[dom]
    t_peak, t_src = tensor_peak(peaks, elapsed_ms)
    if BOUND[dom] == "tensor":
        achieved, peak, unit, src = fl / (d_ms * 1e-3) / 1e12, t_peak, "TFLOP/s", t_src
    else:
        achieved, peak, unit, src = by / (d_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s", peaks["source"] + " hbm copy"
    stages_out = {}
    for s in STAGES:
        f, bts = work[s]
        ms = stage_ms[s]
        stages_out[s] = {"us": round(ms * 1e3, 2), "share": round(ms / sum(stage_ms.values()), 4),
                         "tflops": round(f / (ms * 1e-3) / 1e12, 1) if f else None,
                         "gbs": round(bts / (ms * 1e-3) / 1e9, 1)}
    if side_ms is not None:
        f, bts = work["adaln_table_side"]
        stages_out["adaln_table_side"] = {"us": round(side_ms * 1e3, 2), "overlapped": True,
                                          "gbs": round(bts / (side_ms * 1e-3) / 1e9, 1)}
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": round(tokens_per_s, 1),
        "config": {"workload": wl.name, "description": wl.description, "rows": S, "timestep_rows": T,
                   "blocks": NB, "dim": shape.dim, "heads": shape.n_heads, "ffn": shape.ffn_dim,
                   "cond": shape.cond_dim, "flop_per_step": flops_step,
                   "l2": "inputs larger than L2: %.2f GB of block weights re-read every step" %
                         (NB * weight_bytes(shape) / 1e9),
                   "parallelism": f"replicas x{ws_n}",
                   "timing": "value from K plain steps (one h3_blocks_forward call each); stage times from K "
                             "more steps of per-block calls with an event after every launch (those events cut "
                             "the overlap of consecutive launches, and each block computes its own AdaLN table)"},
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step(shape, S, NB),
        "roofline": {"kernel": dom, "bound": BOUND[dom], "achieved": round(achieved, 1), "peak": peak,
                     "unit": unit, "frac": round(achieved / peak, 4),
                     "peak_source": src,
                     "traffic": TRAFFIC.get(f"{dom}@{wl.name}")},
        "stages": stages_out,
        "instrumented_ms_per_step": round(instrumented_ms / args.steps, 5),
        "clocks": clocks,
        "host_ms_per_step": round((host1 - host0) * 1e3 / args.steps, 4),
    }
    if args.graph:
        # the same steps replayed from one captured CUDA graph (no stage events)
        g = h3.BlocksGraph(cfg, cw, meta, x, y, wsp)
        for _ in range(args.warmup):
            g.launch()
        torch.cuda.synchronize()
        barrier(ws_n)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.launch()
        g1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_n)
        if h3.h3_sync_check(timeout_ms=60000) != 0:
            raise RuntimeError("device error in the graph replays")
        g_ms, g_units = aggregate(g0.elapsed_time(g1), float(args.steps) * flops_step, ws_n)
        line["graph"] = {"ms_per_step": round(g_ms / args.steps, 5),
                         "value": round(g_units / (g_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s"}
        g.close()
    if rank == 0 and not args.no_cpu_baseline and ws_n == 1:
        try:
            if NB == 1:
                line["cpu_baseline"] = cpu_baseline(wl, args.seed, args.cpu_seconds)
            else:
                line["cpu_baseline"] = cpu_baseline_chain(h3, wl, args.seed, args.cpu_seconds, cfg, cw, wts, meta,
                                                          x, wsp)
        except Exception as e:   # the GPU line stands without the oracle's timing
            line["cpu_baseline"] = {"unavailable": f"{type(e).__name__}: {e}"}
    return line


# ---------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------

class OracleRowStepper:
    """Times the CPU oracle on one block a few packed rows at a time.  Before
    timing: the AdaLN table and every row's q/k/v (the keys and values all
    rows attend to).  Each step then evaluates the block's work for `rows`
    packed rows: their QKV projection and QK-norm/RoPE, attention over all
    keys, the O projection and residual, norm2, FC1/SwiGLU and FC2/residual.

    x, t_cond and the weights are the block's own inputs (float64 numpy
    holding the bf16 / fp32 values); meta holds int32 numpy tags, timestep
    indices and positions."""

    def __init__(self, shape, meta, x, t_cond, w, rows: int = 8):
        import numpy as np
        from oracle import h3_oracle as O
        self.O, self.np = O, np
        self.w = w
        self.x = x
        S = x.shape[0]
        self.tag, self.tidx, self.pos = meta["token_tag"], meta["timestep_index"], meta["pos_thw"]
        self.table = O.adaln_table(t_cond, self.w["w_ada"], self.w["b_ada"], shape.dim)
        self.r = O.adaln_rows(self.tag, self.tidx)
        # every row's k and v, a few hundred rows at a time (the oracle's
        # functions are row-wise; chunks only bound the temporaries)
        H = shape.n_heads
        self.k = np.empty((S, H, 128))
        self.v = np.empty((S, H, 128))
        for c0 in range(0, S, 512):
            sl = slice(c0, min(S, c0 + 512))
            mod = self.table[self.r[sl]]
            h1 = O.rmsnorm_modulate(self.x[sl], self.w["norm1_g"], mod[:, 0], mod[:, 1])
            qkv = O.linear(h1, self.w["w_qkv"]).reshape(-1, H, 3, 128)
            _, self.k[sl], self.v[sl] = O.qk_norm_rope(qkv, self.pos[sl], self.w["q_norm_g"], self.w["k_norm_g"])
        self.S, self.shape = S, shape
        self.rows = rows
        self.row_flops = sum(f for f, _ in stage_work(shape, S, t_cond.shape[0]).values()) / S
        self.step_flops = rows * self.row_flops
        self.i = 0
        self.last_rows = None

    def step(self):
        O, np = self.O, self.np
        r = (np.arange(self.rows) + self.i) % self.S
        self.i += self.rows
        self.last_rows = r
        mod = self.table[self.r[r]]
        h1 = O.rmsnorm_modulate(self.x[r], self.w["norm1_g"], mod[:, 0], mod[:, 1])
        qkv = O.linear(h1, self.w["w_qkv"]).reshape(self.rows, self.shape.n_heads, 3, 128)
        q, _, _ = O.qk_norm_rope(qkv, self.pos[r], self.w["q_norm_g"], self.w["k_norm_g"])
        o = np.empty((self.rows, self.shape.n_heads * 128))
        for h in range(self.shape.n_heads):
            o[:, h * 128:(h + 1) * 128] = O.attention_head(q[:, h], self.k[:, h], self.v[:, h])
        o = O.bf16_round(o)
        x1 = O.gated_residual(self.x[r], mod[:, 2], O.linear(o, self.w["w_o"]))
        h2 = O.rmsnorm_modulate(x1, self.w["norm2_g"], mod[:, 3], mod[:, 4])
        gu = O.linear(h2, self.w["w_fc1"])
        F = gu.shape[1] // 2
        return O.gated_residual(x1, mod[:, 5], O.linear(O.swiglu(gu[:, :F], gu[:, F:]), self.w["w_fc2"]))


class OracleAttnStepper:
    """Times the CPU oracle on the attention core a few query rows at a time.
    Before timing: every row's normed and rotated k and v.  Each step then
    evaluates `rows` query rows: their Q norm + RoPE and unmasked softmax
    attention over all keys, for every head."""

    def __init__(self, wl, seed, rows: int = 8):
        import numpy as np
        import h3_inputs as hi
        from oracle import h3_oracle as O
        self.O, self.np = O, np
        S, H = wl.layout.n_rows, wl.shape.n_heads
        ins = hi.attention_inputs(wl.shape, S, seed)
        self.pos = hi.packed_metadata(wl.layout, 1, seed)["pos_thw"].numpy()
        self.qg, self.kg = _f64(ins["q_norm_g"]), _f64(ins["k_norm_g"])
        qkv = ins["qkv"]
        self.qkv = qkv
        self.k = np.empty((S, H, 128))
        self.v = np.empty((S, H, 128))
        for c0 in range(0, S, 1024):
            sl = slice(c0, min(S, c0 + 1024))
            _, self.k[sl], self.v[sl] = O.qk_norm_rope(_f64(qkv[sl]), self.pos[sl], self.qg, self.kg)
        self.S, self.H, self.rows = S, H, rows
        self.step_flops = rows * 4.0 * S * H * 128
        self.i = 0

    def step(self):
        O, np = self.O, self.np
        r = (np.arange(self.rows) + self.i) % self.S
        self.i += self.rows
        q, _, _ = O.qk_norm_rope(_f64(self.qkv[r]), self.pos[r], self.qg, self.kg)
        o = np.empty((self.rows, self.H, 128))
        for h in range(self.H):
            o[:, h] = O.attention_head(q[:, h], self.k[:, h], self.v[:, h])
        return O.bf16_round(o)


def _f64(t):
    import torch
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def oracle_stepper(wl, seed, block: int = 0, x=None, weights=None, rows: int = 8):
    """The stepper for block `block` of workload `wl`: its inputs drawn on the
    host (x defaults to the workload's x, weights to the block's own), or the
    given device/host tensors (the GPU's input to that block, the weights the
    GPU used)."""
    import numpy as np
    import h3_inputs as hi
    meta = {k: v.numpy() for k, v in hi.packed_metadata(wl.layout, wl.n_timesteps, seed).items()}
    acts = hi.activations(wl.shape, wl.layout.n_rows, wl.n_timesteps, seed)
    xs = _f64(acts["x"] if x is None else x)
    w = weights if weights is not None else hi.block_weights(wl.shape, seed, block)
    w64 = {k: _f64(v) for k, v in w.items()}
    return OracleRowStepper(wl.shape, meta, xs, acts["t_cond"].numpy().astype(np.float64), w64, rows)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_stepper(st, seconds: float, y_gpu=None):
    """Steps for about `seconds` (after one untimed step); returns (steps,
    seconds, parity): parity is the error of the timed rows against the
    GPU's output rows of the same block when y_gpu (float64 numpy) is given."""
    import numpy as np
    st.step()
    n, t0 = 0, time.perf_counter()
    got, ref = [], []
    while time.perf_counter() - t0 < seconds:
        y = st.step()
        n += 1
        if y_gpu is not None:
            ref.append(y)
            got.append(y_gpu[st.last_rows])
    dt = time.perf_counter() - t0
    par = None
    if got:
        g, r = np.concatenate(got), np.concatenate(ref)
        rms = float(np.sqrt(np.mean(r * r)))
        e = np.abs(g - r) / np.maximum(rms, np.abs(r))
        par = [round(float(e.max()), 5), round(float(e.mean()), 6)]
    return n, dt, par


def cpu_baseline(wl, seed, seconds: float):
    st = oracle_stepper(wl, seed)
    n, dt, _ = time_stepper(st, seconds)
    tflops = n * st.step_flops / dt / 1e12
    return {"value": round(tflops, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "tokens_per_s": round(n * st.rows / dt, 2),
            "sample": f"{n * st.rows} packed rows of {wl.name}, {st.rows} rows' block work per step in fp64 "
                      f"numpy (AdaLN table and all rows' K/V computed before timing), {dt:.1f} s"}


# blocks of the 50-block evaluation whose oracle work is timed
CPU_BLOCKS = (0, 25, 49)


def cpu_baseline_chain(h3, wl, seed, seconds: float, cfg, cw, wts, meta, x, ws):
    """The oracle on blocks 0, 25 and 49 of the evaluation, each fed the GPU's
    own bf16 input to that block and the weights the GPU used, a few sampled
    rows per step (keys and values over all rows, computed before timing);
    the evaluation's rate is extrapolated as 50 times one block.  The timed
    rows are also compared with the GPU's output of that block."""
    import torch
    xin = {0: x}
    cur = x
    done = 0
    outs = {}
    for b in CPU_BLOCKS:
        if b > done:
            nxt = torch.empty_like(x)
            h3.h3_blocks_forward(cfg, cw[done:b], meta, cur, nxt, ws)
            cur = nxt
        xin[b] = cur
        yb = torch.empty_like(x)
        h3.h3_block_forward(cfg, cw[b], meta, cur, yb, ws)
        outs[b] = yb
        cur, done = yb, b + 1
    if h3.h3_sync_check(timeout_ms=120000) != 0:
        raise RuntimeError("device error while running the blocks before the sampled ones")
    total_n, total_dt, total_fl, parity = 0, 0.0, 0.0, {}
    rows = 8
    for b in CPU_BLOCKS:
        st = oracle_stepper(wl, seed, b, x=xin[b], weights=wts[b], rows=rows)
        n, dt, par = time_stepper(st, seconds / len(CPU_BLOCKS), _f64(outs[b]))
        total_n += n
        total_dt += dt
        total_fl += n * st.step_flops
        parity[f"block{b}"] = par
        del st
    nb = wl.n_blocks
    return {"value": round(total_fl / total_dt / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_cores(),
            "kind": "oracle", "extrapolated": True,
            "tokens_per_s": round(total_n * rows / total_dt / nb, 3),
            "sample": f"{total_n * rows} packed rows' block work in fp64 numpy, {rows} rows per step, on blocks "
                      f"{', '.join(str(b) for b in CPU_BLOCKS)} of the {nb}-block evaluation, each fed the GPU's "
                      f"bf16 input to that block (AdaLN table and all {wl.layout.n_rows} rows' K/V computed "
                      f"before timing), {total_dt:.1f} s; tokens/s = rows/s of one block / {nb} (extrapolated)",
            "parity_vs_gpu": parity}


def run_reference(args, ws_n: int, rank: int):
    import h3_inputs as hi
    wl = hi.WORKLOADS[args.workload]
    if rank != 0:
        return None
    if wl.n_blocks < 1 or wl.name.startswith(("refiner", "input", "output")):
        return {"impl": "reference", "unavailable": f"no oracle timing for the {wl.name} workload"}
    st = OracleAttnStepper(wl, args.seed) if wl.name.startswith("attn") else oracle_stepper(wl, args.seed)
    for _ in range(args.warmup):
        st.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st.step()
    dt = time.perf_counter() - t0
    flops_step = st.step_flops
    value = args.steps * flops_step / dt / 1e12
    nb = wl.n_blocks
    sample = f"{st.rows} packed rows' block work per step (AdaLN table and all rows' K/V computed before timing)"
    if isinstance(st, OracleAttnStepper):
        sample = f"{st.rows} query rows per step: Q norm + RoPE and attention over all keys (all k, v computed before timing)"
    if nb > 1:
        sample += f"; block 0 of the {nb}-block evaluation, the evaluation extrapolated as {nb} x this block"
    return {"metric": METRIC, "impl": "reference", "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "tokens_per_s": round(args.steps * st.rows / dt / nb, 3),
            "config": {"workload": wl.name, "rows": wl.layout.n_rows, "blocks": nb,
                       "sample": f"{st.rows} packed rows per step"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "extrapolated": nb > 1, "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 10 for the 50-block evaluation, 300 for one block)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default: 3 / 10)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="denoiser15860")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--graph", action="store_true", help="also time the block chain replayed from one CUDA graph")
    args = ap.parse_args(argv)
    import h3_inputs as hi
    if args.workload not in hi.WORKLOADS:
        ap.error(f"unknown workload {args.workload}; one of {', '.join(hi.WORKLOADS)}")
    long_step = hi.WORKLOADS[args.workload].n_blocks > 2
    if args.steps is None:
        args.steps = 10 if long_step else 300
    if args.warmup is None:
        args.warmup = 3 if long_step else 10
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws_n, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, ws_n, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if ws_n > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    line = run_ours(args, ws_n, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
