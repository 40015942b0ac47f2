"""Throughput bench: committed tokens/s of block-cached threshold decoding.

One step = one whole generation (Algorithm 1: prefill refresh, every block's
denoise steps, the block-boundary refreshes) of the workload's batch on one
GPU.  Default workload: the 8B-shaped random-init dLLM, prompt 512, gen 256,
block 32, tau 0.9, DualCache, batch 1.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 8b] [--mode dual] [--tau 0.9] [--batch B]
                    [--precision split|bf16]

Prints one JSON line (rank 0).  Under torchrun each rank decodes its own
replica (different prompts): no collective touches the data path; the barrier
and a max-reduction of the timed interval are the only communication.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from cached_masked_decoding_gb300 import configs, replicas, roofline, synth  # noqa: E402

METRIC = "committed tokens/s per GB300 (8B dLLM, blk32, DualCache, τ=0.9); % HBM roofline"
UNIT = "tokens/s"


# DRAM traffic (ncu dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernel, keyed by (kernel class, workload), with the SHA-256 prefix of
# the device sources it was measured on and how the figure was obtained.  A
# figure whose sources have changed since is reported as null.
STEP_SOURCES = ("attention.cuh", "gemm.cuh", "ptx.cuh", "small_kernels.cuh", "step_kernel.cuh",
                "step_hd64.cu", "step_hd128.cu")
MEASURED_TRAFFIC = {
    ("persistent_step", "8b"): (15892279296 + 112541440, "19a7cd3aa89b8ce4",
                                "ncu one-pass capture of dram__bytes_read.sum + dram__bytes_write.sum, one launch"),
}


def sources_sha() -> str:
    import hashlib

    h = hashlib.sha256()
    for f in STEP_SOURCES:
        with open(os.path.join(ROOT, "cached_masked_decoding_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    rec = MEASURED_TRAFFIC.get((kernel, workload))
    if rec is None or rec[1] != sources_sha():
        return None, None
    return rec[0], rec[2]


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- CPU oracle sample
def oracle_sample(wl: configs.Workload, steps: int, refreshes: int, refresh_frac: int = 1) -> dict:
    """Time the CPU oracle on a bounded sample of the workload and extrapolate.

    Sample: one transformer layer of the model at the workload's shapes - a
    DualCache denoise step over the block rows (batch*block rows attending to a
    T-long K/V context) and a refresh forward over the T rows (or over T /
    refresh_frac of them against all T keys, scaled up by refresh_frac: every
    cost of a forward is linear in its query rows at fixed T) - plus the final
    norm and LM head over the block rows.  A generation's time is then
    steps*(L*layer_step + head) + refreshes*(L*layer_refresh), with the step and
    refresh counts the GPU path takes on the same workload.
    """
    from oracle import model as OM

    cfg = wl.model
    t_setup = time.perf_counter()
    lw = OM.LayerWeights(**{n: synth.bf16_to_f64(synth.tensor_bf16(cfg, wl.seed, n, 0))
                            for n in synth.LAYER_TENSORS})
    lm = synth.bf16_to_f64(synth.tensor_bf16(cfg, wl.seed, "lm_head"))
    fnorm = synth.bf16_to_f64(synth.tensor_bf16(cfg, wl.seed, "final_norm"))
    setup_s = time.perf_counter() - t_setup
    rng = np.random.default_rng(0)
    T, H, hd, d = wl.T, cfg.n_heads, cfg.head_dim, cfg.d_model
    b, B = wl.batch, wl.block
    ctx_k = rng.standard_normal((T, H, hd))
    ctx_v = rng.standard_normal((T, H, hd))
    rows = np.arange(wl.prompt_len, wl.prompt_len + B)

    def layer(h, pos):
        q, k, v = OM.qkv(cfg, lw, h, pos)
        kk = ctx_k.copy()
        vv = ctx_v.copy()
        kk[pos] = k
        vv[pos] = v
        return OM.attn_ffn(cfg, lw, h, q, kk, vv)

    h_step = rng.standard_normal((B, d)) * 0.5
    n_ref = max(1, T // refresh_frac)
    h_ref = rng.standard_normal((n_ref, d)) * 0.5
    t0 = time.perf_counter()
    reps = 0
    while True:
        for _ in range(b):
            layer(h_step, rows)
        reps += 1
        if time.perf_counter() - t0 > 0.5 or reps >= 5:
            break
    t_layer_step = (time.perf_counter() - t0) / reps
    t0 = time.perf_counter()
    for _ in range(b):
        x = OM.rms_norm(h_step, fnorm, cfg.norm_eps)
        lg = x @ lm.T
        lg.max(axis=-1)
    t_head = time.perf_counter() - t0
    t0 = time.perf_counter()
    for _ in range(b):
        layer(h_ref, np.arange(n_ref))
    t_ref_part = time.perf_counter() - t0
    t_layer_refresh = t_ref_part * (T / n_ref)
    step_s = cfg.n_layers * t_layer_step + t_head
    refresh_s = cfg.n_layers * t_layer_refresh
    gen_s = steps * step_s + refreshes * refresh_s
    return {"gen_s": gen_s, "step_s": step_s, "refresh_s": refresh_s, "setup_s": setup_s,
            "sample_s": t_layer_step * reps + t_head + t_ref_part,
            "tokens_per_gen": wl.batch * wl.gen_len}


def blas_threads() -> int | None:
    """Threads of numpy's BLAS (threadpoolctl where installed, else the
    OPENBLAS_NUM_THREADS / OMP_NUM_THREADS setting, else None)."""
    try:
        from threadpoolctl import threadpool_info

        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return None


def oracle_sample_one_thread(workload: str, steps: int, refreshes: int, batch: int, tau: float) -> dict | None:
    """The same sample in a fresh interpreter whose BLAS runs one thread; the
    refresh part over an eighth of the rows (scaled up), to stay within tens
    of seconds."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", workload,
           "--batch", str(batch), "--tau", str(tau), "--ref-steps-per-gen", str(steps),
           "--ref-refreshes-per-gen", str(refreshes)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    except (OSError, subprocess.TimeoutExpired):
        return None
    if r.returncode != 0:
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def generation_counts(wl: configs.Workload, mode: str) -> tuple:
    """(steps, refreshes, source) per generation for the oracle's extrapolation."""
    rec = configs.STEPS_PER_GENERATION.get(wl.name)
    base = configs.WORKLOADS.get(wl.name)
    if rec and mode == "dual" and base is not None and wl.tau == base.tau and wl.batch == base.batch:
        return rec[0], rec[1], "the GPU path's measured steps and refreshes on this workload"
    return max(1, int(round(wl.gen_len / 3.0))), wl.gen_len // wl.block, "assumed tau-bar 3 (no measured count)"


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- GPU arm
def run_ours(args, wl: configs.Workload, rank: int, world: int, local_rank: int) -> dict | None:
    import torch

    from cached_masked_decoding_gb300 import binding

    torch.cuda.set_device(local_rank)
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    peaks = load_peaks()
    cfg = wl.model
    model = binding.Model.from_synth(cfg, seed=wl.seed)
    stream = torch.cuda.current_stream()
    b, P, gen, B = wl.batch, wl.prompt_len, wl.gen_len, wl.block
    sh = replicas.shard(rank, world, b)
    prompts_dev = torch.empty(b * max(P, 1), dtype=torch.int32, device="cuda")
    synth.device_fill_prompts(prompts_dev.data_ptr(), cfg, wl.seed, b, P, first_seq=sh.first_seq,
                              stream=stream.cuda_stream)
    state = binding.State(model, None, b, P, gen, B, stream=stream.cuda_stream)
    state.set_precision(args.precision)
    state.set_persistent(args.persistent)
    state.set_fused_refresh(args.fused_refresh)
    state.set_run_ahead(args.run_ahead)
    state.set_mask(args.mask)
    if args.rule == "fixed":
        sel = binding.make_select(binding.SEL_FIXED_K, wl.tau, args.k)
    else:
        sel = binding.make_select(binding.SEL_THRESHOLD, wl.tau)
    mode = args.mode

    def one_generation():
        state.set_prompts_device(prompts_dev.data_ptr())
        return state.run(sel, mode, refresh_interval=args.refresh_interval)

    for _ in range(args.warmup):
        one_generation()
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    stats = [one_generation() for _ in range(args.steps)]
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    elapsed_ms = ev0.elapsed_time(ev1)
    elapsed_ms, tokens = replicas.reduce_timing(elapsed_ms, sum(s["committed"] for s in stats),
                                                device=torch.device("cuda", local_rank))
    value = tokens / (elapsed_ms / 1e3)
    launches = sum(s["kernel_launches"] for s in stats) + args.steps   # + one canvas reset each
    steps = sum(s["steps"] for s in stats)
    refreshes = sum(s["refreshes"] for s in stats)
    # a step fused with the refresh before it is timed with the refreshes
    fused = sum(s["fused_steps"] for s in stats)
    step_ms = sum(s["step_ms"] for s in stats) / max(steps - fused, 1)
    refresh_ms = sum(s["refresh_ms"] for s in stats) / max(refreshes, 1)

    # ---------------------------------------------------------------- per-kernel timing pass
    state.set_kernel_timing(True)
    one_generation()
    torch.cuda.synchronize()
    kt = state.kernel_times()
    state.set_kernel_timing(False)
    step_classes = ("embed", "qkv_gemm", "attention", "o_gemm", "gateup_gemm", "down_gemm", "lm_head_gemm",
                    "merge_select", "persistent_step")
    gemm_classes = ("qkv_gemm", "o_gemm", "gateup_gemm", "down_gemm", "lm_head_gemm")
    dom = max(step_classes, key=lambda k: kt[k]["ms"])
    per_launch_ms = kt[dom]["ms"] / max(kt[dom]["launches"], 1)
    per_launch_bytes = kt[dom]["bytes"] / max(kt[dom]["launches"], 1)
    achieved = per_launch_bytes / (per_launch_ms / 1e3) / 1e9
    # algorithmic flops of a DualCache step (counted once, whatever the MMA
    # width of the precision) and per launch of each step kernel class
    dm, Fm, Lm, Vm = cfg.d_model, cfg.d_ffn, cfg.n_layers, cfg.vocab
    n_blk = b * B
    attn_flops_layer = 4.0 * b * cfg.n_heads * B * wl.T * cfg.head_dim
    class_flops = {"qkv_gemm": 2.0 * n_blk * dm * 3 * dm, "o_gemm": 2.0 * n_blk * dm * dm,
                   "gateup_gemm": 2.0 * n_blk * dm * 2 * Fm, "down_gemm": 2.0 * n_blk * Fm * dm,
                   "lm_head_gemm": 2.0 * n_blk * dm * Vm, "attention": attn_flops_layer}
    step_flops = Lm * (class_flops["qkv_gemm"] + class_flops["o_gemm"] + class_flops["gateup_gemm"] +
                       class_flops["down_gemm"] + attn_flops_layer) + class_flops["lm_head_gemm"]
    class_flops["persistent_step"] = step_flops
    gemm_ms = sum(kt[c]["ms"] for c in gemm_classes)
    gemm_bytes = sum(kt[c]["bytes"] for c in gemm_classes)
    # refresh: n = b*T rows through every layer's projections; a refresh on its
    # own stops after the last layer's QKV, one fused with its step finishes
    # the last layer (counted from the O-projection launches)
    d, F = cfg.d_model, cfg.d_ffn
    n_ref = b * wl.T
    n_refresh_timed = max(kt["refresh_qkv_gemm"]["launches"] // cfg.n_layers, 1)
    full_layers = kt["refresh_o_gemm"]["launches"] / n_refresh_timed
    refresh_flops = 2.0 * n_ref * (full_layers * (d * d + 3 * d * F) + cfg.n_layers * 3 * d * d)
    refresh_gemm_ms = sum(kt["refresh_" + c]["ms"] for c in ("qkv_gemm", "o_gemm", "gateup_gemm", "down_gemm"))

    # ---------------------------------------------------------------- end to end (host buffers)
    host_prompts = synth.prompts(cfg, wl.seed, b, P, first_seq=sh.first_seq)
    toks = np.zeros((b, wl.T), dtype=np.int32)
    e2e_state = state
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    e2e_tokens = 0
    e2e_steps = 0
    for _ in range(args.steps if args.e2e else 0):
        e2e_state.reset(host_prompts)                   # H2D: canvas b*T int32
        st = e2e_state.run(sel, mode, refresh_interval=args.refresh_interval)
        toks[:] = e2e_state.tokens()                    # D2H: canvas b*T int32
        e2e_tokens += st["committed"]
        e2e_steps += st["steps"]
    e2e_ms, e2e_tokens = replicas.reduce_timing((time.perf_counter() - t0) * 1e3, e2e_tokens,
                                                device=torch.device("cuda", local_rank))
    e2e_s = e2e_ms / 1e3
    h2d = b * wl.T * 4
    d2h = b * wl.T * 4 + (e2e_steps // max(args.steps, 1)) * (b + 1) * 4

    traffic, traffic_src = measured_traffic(dom, wl.name) if mode == "dual" and b == wl.batch else (None, None)
    # algorithmic bytes count every weight and the bf16 K/V cache once; split
    # precision also reads the K/V low halves, an implementation cost reported
    # on its own
    step_bytes = roofline.dual_step_bytes(cfg.weight_bytes_step(), cfg.kv_bytes(wl.T, b))
    split_extra = cfg.kv_bytes(wl.T, b) if args.precision == "split" else 0
    # The roofline that bounds the work: the HBM time of its algorithmic bytes
    # against the tensor time of its algorithmic flops (the sustained bf16
    # figure: the kernels run inside a long step).  A DualCache step of b*B
    # rows is HBM-bound up to a few hundred rows, tensor-bound above.
    tf_peak = peaks["bf16_tflops_sustained"]
    dual = mode == "dual"
    step_tensor = dual and step_flops / (tf_peak * 1e12) > step_bytes / (peaks["hbm_gbs"] * 1e9)
    step_roofline = {
        "what": "one denoise step (all kernels, launch gaps included)", "ms": step_ms,
        "algorithmic_bytes": step_bytes, "algorithmic_flops": step_flops if dual else None,
        "hbm_frac": step_bytes / (step_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
        "tensor_frac": step_flops / (step_ms / 1e3) / 1e12 / tf_peak if dual else None,
    }
    if step_tensor:
        step_roofline.update({"bound": "tensor", "achieved": step_flops / (step_ms / 1e3) / 1e12, "peak": tf_peak,
                              "unit": "TFLOP/s", "frac": step_roofline["tensor_frac"],
                              "peak_source": f"{peaks['source']} bf16 GEMM rate, sustained"})
    else:
        step_roofline.update({"bound": "hbm", "achieved": step_bytes / (step_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                              "unit": "GB/s", "frac": step_roofline["hbm_frac"]})
    kernel_roofline = {
        "kernel": dom, "traffic": traffic, "traffic_source": traffic_src,
        "timing": "per-launch CUDA events around each kernel, one extra generation after the timed region",
        "bytes_per_launch": per_launch_bytes, "ms_per_launch": per_launch_ms,
        "split_kv_extra_bytes": split_extra if dom == "persistent_step" else None,
        "traffic_over_algorithmic": traffic / per_launch_bytes if traffic else None,
    }
    if step_tensor and dom in class_flops:
        kf = class_flops[dom]
        kernel_roofline.update({"bound": "tensor", "flops_per_launch": kf,
                                "achieved": kf / (per_launch_ms / 1e3) / 1e12, "peak": tf_peak, "unit": "TFLOP/s",
                                "frac": kf / (per_launch_ms / 1e3) / 1e12 / tf_peak,
                                "peak_source": f"{peaks['source']} bf16 GEMM rate, sustained"})
    else:
        kernel_roofline.update({"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": achieved / peaks["hbm_gbs"],
                                "peak_source": f"{peaks['source']} HBM copy bandwidth"})
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"{wl.name}: {cfg.name}-shaped random-init dLLM, batch {b}, prompt {P}, gen {gen}, "
                        f"block {B}, tau {wl.tau}, {mode} cache",
            "model": f"{cfg.n_layers}L d{cfg.d_model} H{cfg.n_heads} F{cfg.d_ffn} V{cfg.vocab} (random init)",
            "global_batch": sh.global_batch, "seq_len": wl.T, "block": B, "tau": wl.tau, "cache_mode": mode,
            "rule": "threshold" if args.rule == "threshold" else f"fixed k={args.k}",
            "refresh_interval": args.refresh_interval,
            "precision": f"{args.precision} activations, bf16 weights and K/V, f32 accumulate",
            "mask": "bidirectional" if args.mask == "full" else "block-causal (refresh = one block forward)",
            "step_launch": "persistent (one cooperative launch per denoise step)" if args.persistent
            else "one launch per kernel",
            "refresh": "fused with the step after it (one forward)" if args.fused_refresh
            else "separate forward, then the step",
            "host_loop": "a block's next step enqueued before the current step's commits are read" if args.run_ahead
            else "every step's commits read before the next launch",
            "l2": "inputs larger than L2 (every step streams all weights)",
            "parallelism": f"replicas x{world} (no data-path collective)",
        },
        "e2e": {"value": e2e_tokens / e2e_s if args.e2e else None, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "api": "dllm_state_reset(host prompts) + dllm_run + dllm_read_state(host tokens)"},
        "roofline": kernel_roofline,
        "step_roofline": step_roofline,
        "gemm_roofline": {"achieved": gemm_bytes / (gemm_ms / 1e3) / 1e9 if gemm_ms else None,
                          "frac": (gemm_bytes / (gemm_ms / 1e3) / 1e9 / peaks["hbm_gbs"]) if gemm_ms else None},
        "refresh_roofline": {
            "bound": "tensor", "what": "projection GEMMs of one refresh (per-launch events)",
            "flops": refresh_flops, "ms": refresh_gemm_ms / n_refresh_timed,
            "achieved": refresh_flops / (refresh_gemm_ms / n_refresh_timed / 1e3) / 1e12 if refresh_gemm_ms else None,
            "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
            "frac": (refresh_flops / (refresh_gemm_ms / n_refresh_timed / 1e3) / 1e12 / peaks["bf16_tflops_sustained"])
            if refresh_gemm_ms else None,
            "note": "split activations double the MMA work; flops counted once",
        },
        "kernel_times": {k: v for k, v in kt.items() if v["launches"]},
        "tau_bar": sum(s["committed"] for s in stats) / max(sum(s["steps"] for s in stats) * b, 1),
        "denoise_steps_per_s": (steps - fused) / (sum(s["step_ms"] for s in stats) / 1e3),
        "steps_per_generation": steps / args.steps, "refreshes_per_generation": refreshes / args.steps,
        "fused_steps_per_generation": fused / args.steps,
        "steps_per_block": steps / args.steps / max(gen // B, 1),
        "max_steps_per_block": max(s["max_steps_per_block"] for s in stats),
        "eq15": {"S": steps / args.steps, "C_active_ms": step_ms, "R_ms": refresh_ms * refreshes / args.steps,
                 "note": "C_active over the cached steps; R includes the fused refresh-and-step forwards"},
        "clocks": clk, "gpu_launches": launches,
    }
    if args.cpu_baseline and rank == 0 and world == 1:
        g_steps, g_refreshes = steps // args.steps, refreshes // args.steps
        samp = oracle_sample(wl, g_steps, g_refreshes)
        one = oracle_sample_one_thread(wl.name, g_steps, g_refreshes, b, wl.tau)
        out["cpu_baseline"] = {
            "value": samp["tokens_per_gen"] / samp["gen_s"], "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "blas_threads": blas_threads(),
            "sample": (f"one layer of the {cfg.name} model at the workload's shapes (a DualCache step over "
                       f"{b}x{B} block rows against a {wl.T}-key context, a refresh over {wl.T} rows) plus "
                       f"the LM head; extrapolated to {cfg.n_layers} layers and to this run's "
                       f"{g_steps} steps and {g_refreshes} refreshes per generation"),
            "extrapolated": True,
            "sample_seconds": samp["sample_s"], "extrapolated_generation_s": samp["gen_s"],
            "one_thread": ({"value": one["tokens_per_gen"] / one["gen_s"], "cores": 1, "blas_threads": 1,
                            "sample_seconds": one["sample_s"],
                            "sample": "the same, refresh over T/8 query rows scaled by 8"} if one else None),
        }
    state.free()
    model.free()
    return out if rank == 0 else None


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, wl: configs.Workload, rank: int) -> dict | None:
    if rank != 0:
        return None
    cfg = wl.model
    steps, refreshes, count_src = generation_counts(wl, args.mode)
    if args.ref_steps_per_gen:
        steps, count_src = args.ref_steps_per_gen, "given on the command line"
    samples = []
    wall = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        s = oracle_sample(wl, steps, refreshes)
        if i >= args.warmup:
            samples.append(s)
            wall.append(time.perf_counter() - t0)
    gen_s = statistics.mean(s["gen_s"] for s in samples)
    value = wl.batch * wl.gen_len / gen_s
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": gen_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "ms_per_step_kind": "extrapolated: one generation's time from a timed one-layer sample",
        "sample_wall_ms_per_step": statistics.mean(wall) * 1e3,
        "config": {"workload": f"{wl.name}: {cfg.name}-shaped dLLM, batch {wl.batch}, prompt {wl.prompt_len}, "
                               f"gen {wl.gen_len}, block {wl.block}, tau {wl.tau}, {args.mode} cache",
                   "global_batch": wl.batch, "seq_len": wl.T, "parallelism": "CPU oracle",
                   "steps_per_generation": steps, "refreshes_per_generation": refreshes,
                   "counts_source": count_src},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "blas_threads": blas_threads(), "extrapolated": True,
                         "sample": "one layer step + one layer refresh + LM head per bench step, extrapolated to "
                                   f"{cfg.n_layers} layers, {steps} steps and {refreshes} refreshes per generation"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="8b", choices=sorted(configs.WORKLOADS))
    ap.add_argument("--mode", default="dual", choices=("dual", "prefix", "none"))
    ap.add_argument("--tau", type=float, default=None)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--precision", default="split", choices=("split", "bf16"))
    ap.add_argument("--rule", default="threshold", choices=("threshold", "fixed"),
                    help="selection rule: the threshold rule (Algorithm 2) or a fixed k tokens per step")
    ap.add_argument("--k", type=int, default=1, help="tokens per step of the fixed rule")
    ap.add_argument("--refresh-interval", type=int, default=0,
                    help="also refresh the cache every this many steps inside a block (0: block boundaries only)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--ref-steps-per-gen", type=int, default=0)
    ap.add_argument("--ref-refreshes-per-gen", type=int, default=0)
    ap.add_argument("--oracle-sample", action="store_true",
                    help="print one timed oracle sample as JSON (the bench runs this with a one-thread BLAS)")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (profiling captures of a small case)")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--mask", default="full", choices=("full", "block_causal"),
                    help="attention mask: bidirectional (the method's) or block-causal (exact cache)")
    ap.add_argument("--no-persistent", dest="persistent", action="store_false",
                    help="one launch per kernel instead of the persistent DualCache step")
    ap.add_argument("--no-fused-refresh", dest="fused_refresh", action="store_false",
                    help="run every refresh (and block-causal commit forward) apart from the step after it")
    ap.add_argument("--no-run-ahead", dest="run_ahead", action="store_false",
                    help="read every step's commits back before launching the next step")
    args = ap.parse_args()
    wl = configs.WORKLOADS[args.workload]
    import dataclasses
    if args.tau is not None or args.batch is not None:
        wl = dataclasses.replace(wl, tau=args.tau if args.tau is not None else wl.tau,
                                 batch=args.batch if args.batch is not None else wl.batch)
    if args.layers:
        wl = dataclasses.replace(wl, model=dataclasses.replace(wl.model, n_layers=args.layers,
                                                               name=f"{wl.model.name}-{args.layers}L"))
    rank, world, local_rank = dist_env()
    if args.oracle_sample:
        print(json.dumps(oracle_sample(wl, args.ref_steps_per_gen, args.ref_refreshes_per_gen, refresh_frac=8)))
        return
    if args.impl == "reference":
        out = run_reference(args, wl, rank)
    else:
        out = run_ours(args, wl, rank, world, local_rank)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
