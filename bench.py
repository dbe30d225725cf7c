#!/usr/bin/env python3
"""Benchmark of the tensor/sequence-parallel MLP block on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--mode fused|partials]

One step = forward + backward of the block (every hot-path kernel: dim-0
all-gather of X, fc1 + GeLU/SwiGLU, fc2 + shard sum / reduce-scatter, dZ
all-gather and X re-gather, fc2 input gradient + act', both weight gradients,
fc1 input gradient + reduce-scatter) through the C ABI on one synthetic batch.
Default workload: the 22B-width TP+SP MLP, [s,b,h] = [4096,1,6144], f = 24576,
tp = 8 logical shards, SP on, bf16.  Prints ONE JSON line (rank 0).

With --gpus N > 1 (launched by torch.distributed.run) every rank runs an
independent replica of the block on its own GPU (the tensor shards are logical
partitions inside one GPU, so there is no cross-GPU exchange): weak scaling,
value = all ranks' FLOPs / max-over-ranks time.

--impl reference times the CPU oracle (NumPy fp64) on a bounded token sample of
the same workload, on the host cores, with the same metric and unit.

--block attention times the tensor-parallel self-attention block instead
(QKV projection, per-head attention core, output projection, and the
backward) on the Llama-70B width ([4096,1,8192], 64 heads of 128, tp = 8, SP,
causal, bf16) or another --config from synthetic.ATTN_CONFIGS.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TP/SP MLP fwd+bwd TFLOP/s on 1 GB300 and % of dense BF16 peak"
ATTN_METRIC = "TP/SP attention block fwd+bwd TFLOP/s on 1 GB300 and % of dense BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="w22b_tpsp8_bf16")
    ap.add_argument("--mode", choices=["fused", "partials"], default="fused")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-dim0", action="store_true", help="skip the stand-alone dim-0 kernel measurement")
    ap.add_argument("--main-grad", action="store_true",
                    help="weight gradients accumulated into float32 main_grad (gradient-accumulation fusion)")
    ap.add_argument("--block", choices=["mlp", "attention"], default="mlp")
    ap.add_argument("--sp-region", action="store_true",
                    help="time the whole SP sublayer: LayerNorm on the chunks -> block -> dropout + residual, "
                         "and its backward (FLOPs counted are the block's)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- helpers


L2_BYTES = 129e6  # GB300 L2


def l2_note(tensors: dict) -> str:
    """How the timed steps stand to the L2 cache (no flush between steps): the
    main tensors one step reads and writes, with their sizes, together are or
    are not larger than L2."""
    sizes = ", ".join(f"{k} {v / 1e6:.0f} MB" for k, v in tensors.items())
    if sum(tensors.values()) > L2_BYTES:
        return f"inputs larger than L2 ({sizes} per step), no flush"
    return f"L2-resident ({sizes} per step), no flush: a small-case figure"


def attn_workload_desc(cfg) -> dict:
    """The attention block's config entry (the same in both arms)."""
    kv = f" ({cfg.groups} key/value heads)" if cfg.groups != cfg.heads else ""
    return {"workload": f"TP self-attention [s,b,h]=[{cfg.s},{cfg.b},{cfg.h}] {cfg.heads} heads of {cfg.d}{kv} "
                        f"tp={cfg.tp} SP {'on' if cfg.sp else 'off'} {'causal' if cfg.causal else 'unmasked'} "
                        f"{cfg.dtype}, fwd+bwd",
            "name": cfg.name, "kv_heads": cfg.groups, "flops_per_step": float(cfg.flops_fwd_bwd()),
            "flops_note": "12·M·h·(h + h_kv) projections + 12·b·h·(visible query-key pairs) core, "
                          "no recomputation",
            "l2": l2_note({"Wqkv": cfg.qkv_rows * cfg.h * 2, "QKV": cfg.qkv_rows * cfg.s * cfg.b * 2})}


def workload_desc(cfg) -> dict:
    names = {
        "tiny_tp2_f32": "tiny TP MLP",
        "tpsp4_bf16": "TP+SP MLP",
        "w8p3b_tp8_f16": "8.3B-width TP MLP",
        "w22b_tpsp8_bf16": "22B-width TP+SP MLP",
        "llama70b_swiglu_tpsp8_bf16": "Llama-70B-like SwiGLU TP+SP MLP",
    }
    return {
        "workload": f"{names.get(cfg.name, cfg.name)} [s,b,h]=[{cfg.s},{cfg.b},{cfg.h}] "
                    f"{'F' if cfg.act == 'swiglu' else 'f'}={cfg.f} tp={cfg.tp} SP {'on' if cfg.sp else 'off'} "
                    f"{cfg.dtype} {cfg.act}, fwd+bwd",
        "name": cfg.name,
        "s": cfg.s, "b": cfg.b, "h": cfg.h, "f": cfg.f, "tp": cfg.tp, "sp": cfg.sp, "act": cfg.act,
    }


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sp_partitioned_transformer_gb300", "csrc")
    for f in ("gemm_tc.cu", "common.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(config_name: str, mode: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "gemm_dram_traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    ent = d.get("per_step", {}).get(f"{config_name}/{mode}")
    return ent


def attn_kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sp_partitioned_transformer_gb300", "csrc")
    for f in ("attn.cu", "common.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def attn_ncu_traffic(config_name: str):
    """DRAM bytes of one fwd+bwd pass of the attention core (its four kernels) from
    the committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "attn_dram_traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256_16") != attn_kernel_source_hash():
        return None
    return d.get("per_step", {}).get(config_name)


# A timed region shorter than this runs at burst clocks: the GPU reaches its power
# cap and settles its clock only over seconds of load.
BURST_REGION_S = 1.0


def choose_peak(peaks: dict, region_s: float, key_burst: str = "bf16_tflops",
                key_sustained: str = "bf16_tflops_sustained"):
    """The tensor peak that applies to a kernel timed over a region of region_s
    seconds: the burst figure for a short region, the sustained (power-capped)
    one for a long one.  Returns (peak, regime, key)."""
    if region_s < BURST_REGION_S:
        return (peaks.get(key_burst) or FALLBACK_PEAKS[key_burst]), "burst", key_burst
    return (peaks.get(key_sustained) or FALLBACK_PEAKS[key_sustained]), "sustained", key_sustained


def e2e_guard(ms_device: float, ms_e2e: float):
    """End to end contains the device-only step's work plus its copies, so a
    shorter e2e step time can only be a clock difference between the two
    windows.  Such a figure is not reported as measured: the e2e time is raised
    to the device-only time and a flag says so.  Returns (ms, flag or None)."""
    if ms_e2e < ms_device:
        return ms_device, (f"measured e2e {ms_e2e:.4f} ms/step < device-only {ms_device:.4f} ms/step "
                           f"(clock difference between the windows): reported at the device-only time")
    return ms_e2e, None


def parse_smi_time(text: str):
    """nvidia-smi's timestamp ('YYYY/MM/DD HH:MM:SS.mmm', local time) in epoch seconds."""
    try:
        base, _, frac = text.strip().partition(".")
        t = time.mktime(time.strptime(base, "%Y/%m/%d %H:%M:%S"))
        return t + (float("0." + frac) if frac.isdigit() else 0.0)
    except ValueError:
        return None


def summarize_clocks(rows, windows=(), util_min: float = 50.0):
    """Clock record of nvidia-smi samples (dicts with the ClockSampler fields).

    A sample counts as under load when the GPU was busy (utilization.gpu ≥
    util_min) — not by its clock, which sits near its maximum when idle too.
    `windows` are (t0, t1) host epoch intervals of the timed regions; samples
    inside them are summarised separately.  The throttle reasons are those seen
    in loaded samples."""
    def num(x):
        try:
            return float(x)
        except (TypeError, ValueError):
            return None

    loaded = [r for r in rows if (num(r.get("utilization.gpu")) or 0.0) >= util_min]
    timed = [r for r in loaded
             if r.get("t") is not None and any(a <= r["t"] <= b for a, b in windows)]
    sm = [num(r["clocks.sm"]) for r in loaded if num(r.get("clocks.sm")) is not None]
    sm_t = [num(r["clocks.sm"]) for r in timed if num(r.get("clocks.sm")) is not None]
    mx = [num(r["clocks.max.sm"]) for r in rows if num(r.get("clocks.max.sm")) is not None]
    power = [num(r["power.draw"]) for r in loaded if num(r.get("power.draw")) is not None]
    reasons = set()
    for r in loaded:
        for name in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"):
            if str(r.get("clocks_event_reasons." + name, "")).lower().startswith("active"):
                reasons.add(name)
    return {
        "sm_mhz": statistics.median(sm) if sm else None,
        "sm_max_mhz": max(mx) if mx else None,
        "reasons": sorted(reasons),
        "samples": len(rows),
        "samples_loaded": len(loaded),
        "samples_in_timed_regions": len(timed),
        "sm_mhz_timed_regions": statistics.median(sm_t) if sm_t else None,
        "power_w_max": max(power) if power else None,
        "load_rule": f"utilization.gpu >= {util_min:g}%",
    }


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of the SM clock, utilisation, power and
    throttle reasons while the benchmark runs; stop() keeps the loaded ones."""

    FIELDS = ["timestamp", "utilization.gpu", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.proc = None
        self.path = None
        self.windows = []
        try:
            import tempfile

            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", gpu_id], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def mark(self, t0: float, t1: float) -> None:
        """Host epoch interval of a timed region."""
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    r = dict(zip(self.FIELDS, parts))
                    r["t"] = parse_smi_time(r["timestamp"])
                    rows.append(r)
        os.unlink(self.path)
        if not rows:
            return None
        return summarize_clocks(rows, self.windows)


def profiled_region(tpmlp, step, steps, stream, barrier, clocks):
    """K more steps with launch accounting on; returns (ms per step, profile)."""
    import torch

    tpmlp.profile_start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    barrier()
    if clocks is not None:
        clocks.mark(t_host0, time.time())
    prof = tpmlp.profile_stop()
    return e0.elapsed_time(e1) / steps, prof


def gpu_uuid(dev) -> str:
    import torch

    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else f"GPU-{s}"
    except Exception:  # noqa: BLE001
        return str(dev)


# ---------------------------------------------------------------- CPU oracle timing


def oracle_sample(cfg, inputs, target_s: float, max_tokens: int | None = None):
    """Time the fp64 oracle's fwd+bwd on the first M' tokens (full weights); M' is
    sized so one run takes about target_s.  Returns (flops/s, seconds, tokens, setup)."""
    import numpy as np

    import oracle as O

    W1 = inputs["W1"].double().numpy()
    W2 = inputs["W2"].double().numpy()
    X = O.flatten_sbh(inputs["X"].double().numpy())
    dZ = O.flatten_sbh(inputs["dZ"].double().numpy())
    M = X.shape[0]
    cap = min(M, max_tokens or M)

    def run(mt):
        t0 = time.perf_counter()
        O.mlp_backward(X[:mt], W1, W2, dZ[:mt], cfg.act)
        return time.perf_counter() - t0

    probe = min(32, cap)
    t_probe = run(probe)
    mt = probe
    if t_probe < target_s:
        mt = int(min(cap, max(probe, probe * target_s / max(t_probe, 1e-3))))
        mt = max(probe, (mt // 32) * 32) if mt >= 32 else mt
    per = {"tokens": mt}
    del np
    return run, mt, per


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def flops_for_tokens(cfg, tokens: int) -> float:
    return float(cfg.with_(s=tokens, b=1).flops_fwd_bwd())


# ---------------------------------------------------------------- dim-0 kernels alone


def measure_dim0(tpmlp, cfg, dev, stream, iters: int = 50) -> dict:
    """GB/s of the stand-alone SP all-gather, split and reduce-scatter kernels at
    this workload's sizes (tpmlp_gather_dim0 / split_dim0 / reduce_scatter_dim0).
    Buffer sets rotate so that more than 4x the 129 MB L2 is touched between
    reuses: each launch streams from HBM."""
    import torch

    l2 = 129e6
    dt = cfg.torch_dtype
    s, b, h, tp = cfg.s, cfg.b, cfg.h, cfg.tp
    if s % tp != 0:
        return {}
    e = torch.finfo(dt).bits // 8
    act_bytes = s * b * h * e
    nsets = max(2, int(4 * l2 // (2 * act_bytes)) + 1)
    fulls = [torch.randn(s, b, h, device=dev).to(dt) for _ in range(nsets)]
    shards = [[torch.empty(s // tp, b, h, device=dev, dtype=dt) for _ in range(tp)] for _ in range(nsets)]
    out = {}

    def timed(fn, nbytes):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(iters):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / iters
        return {"GB/s": nbytes / (ms / 1e3) / 1e9, "us": ms * 1e3, "bytes": nbytes}

    out["gather"] = timed(lambda i: tpmlp.gather_dim0(shards[i % nsets], fulls[(i + 1) % nsets], s=s, b=b, h=h,
                                                      tp=tp, stream=stream), 2 * act_bytes)
    out["split"] = timed(lambda i: tpmlp.split_dim0(fulls[i % nsets], shards[(i + 1) % nsets], s=s, b=b, h=h,
                                                    tp=tp, stream=stream), 2 * act_bytes)
    del fulls
    p_bytes = tp * s * b * h * 4
    psets = max(2, int(4 * l2 // p_bytes) + 1)
    parts = [torch.randn(tp, s * b * h, device=dev) for _ in range(psets)]
    outs = [[torch.empty(s // tp, b, h, device=dev, dtype=dt) for _ in range(tp)] for _ in range(psets)]
    out["reduce_scatter"] = timed(lambda i: tpmlp.reduce_scatter_dim0(parts[i % psets], outs[i % psets], s=s, b=b,
                                                                      h=h, tp=tp, scatter=1, stream=stream),
                                  p_bytes + act_bytes)
    for v in out.values():
        v["frac_of_hbm"] = None
    return out


# ---------------------------------------------------------------- reference arm


def run_reference_attention(args, world: int) -> int:
    """The reference arm of --block attention: the fp64 attention oracle, timed
    on a bounded sample of the attention workload, under the attention arm's
    metric and config."""
    from synthetic import ATTN_CONFIGS, attn_inputs

    name = args.config if args.config in ATTN_CONFIGS else "llama70b_attn_tpsp8_bf16"
    cfg = ATTN_CONFIGS[name]
    per_step_s = max(0.2, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    run, sp_, fl = attn_oracle_sample(cfg, attn_inputs(cfg), per_step_s)
    for _ in range(args.warmup):
        run(sp_)
    times = [run(sp_) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = fl / t / 1e12
    sample = (f"first {sp_} of {cfg.s} tokens of each of {cfg.b} sequence(s), full weights; fp64 NumPy attention "
              f"block fwd+bwd")
    line = {
        "impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": attn_workload_desc(cfg),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args) -> int:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    if args.block == "attention":
        return run_reference_attention(args, world)
    from synthetic import CONFIGS, block_inputs

    cfg = CONFIGS[args.config]
    inputs = block_inputs(cfg)
    # each step a bounded sample so that the whole run stays within a few minutes
    per_step_s = max(0.2, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    run, mt, _ = oracle_sample(cfg, inputs, per_step_s)
    for _ in range(args.warmup):
        run(mt)
    times = [run(mt) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = flops_for_tokens(cfg, mt) / t / 1e12
    sample = (f"first {mt} of {cfg.M} tokens of the workload, full weights; fp64 NumPy oracle fwd+bwd "
              f"(12·M'·h·f FLOPs)" if cfg.act != "swiglu" else
              f"first {mt} of {cfg.M} tokens of the workload, full weights; fp64 NumPy oracle fwd+bwd (18·M'·h·F FLOPs)")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": workload_desc(cfg),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- ranks
# With --gpus N > 1 every rank runs an independent replica of the block on its
# own GPU (the tensor shards are partitions inside one GPU): the ranks only meet
# at the barriers around the timed region and in the max over their times.


def rank_barrier(world: int, sync=None) -> None:
    """Device synchronisation, then (N > 1) a process-group barrier, then again."""
    import torch.distributed as dist

    if sync is not None:
        sync()
    if world > 1:
        dist.barrier()
    if sync is not None:
        sync()


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest of the ranks' values (the job's time is its slowest replica's)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_replica: float, world: int, ms_max: float) -> float:
    """Whole-job TFLOP/s: every replica's FLOPs over the slowest replica's time."""
    return world * flops_per_replica / (ms_max / 1e3) / 1e12


# ---------------------------------------------------------------- our arm


def run_ours(args) -> int:
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and args.gpus != 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))

    from sp_partitioned_transformer_gb300 import build as _build

    _build.build()
    import sp_partitioned_transformer_gb300 as tpmlp
    from synthetic import CONFIGS, ELEM_BYTES, block_inputs

    tpmlp.load()
    cfg = CONFIGS[args.config]
    dt = cfg.torch_dtype
    inputs = block_inputs(cfg)
    dev = torch.device("cuda", local_rank)
    W1 = inputs["W1"].to(dev)
    W2 = inputs["W2"].to(dev)
    X = inputs["X"].to(dev)
    dZ = inputs["dZ"].to(dev)
    x = [c.contiguous() for c in X.chunk(cfg.tp)] if cfg.sp else X
    dz = [c.contiguous() for c in dZ.chunk(cfg.tp)] if cfg.sp else dZ
    blk = tpmlp.MLPBlock(cfg.s, cfg.b, cfg.h, cfg.f, cfg.tp, cfg.sp, dt, cfg.act, args.mode, device=dev)
    fw = blk.alloc_forward()
    bw = blk.alloc_backward()
    stream = torch.cuda.current_stream(dev)

    mg1 = mg2 = None
    if args.main_grad:
        mg1 = torch.zeros(cfg.fc1_rows, cfg.h, dtype=torch.float32, device=dev)
        mg2 = torch.zeros(cfg.h, cfg.f, dtype=torch.float32, device=dev)

    def block_step(xin, dzin):
        blk.forward(xin, W1, W2, out=fw, stream=stream)
        if args.main_grad:
            blk.backward_main_grad(xin, W1, W2, fw, dzin, mg1, mg2, out=bw, stream=stream)
        else:
            blk.backward(xin, W1, W2, fw, dzin, out=bw, stream=stream)

    if args.sp_region:
        if not cfg.sp:
            raise SystemExit("--sp-region needs an SP workload")
        from synthetic import sp_region_inputs

        reg = sp_region_inputs(cfg.s, cfg.b, cfg.h, 0.1, seed=cfg.seed + 1, dtype=cfg.dtype)
        R = [c.contiguous() for c in reg["R"].to(dev).chunk(cfg.tp)]
        keep = [c.contiguous() for c in reg["keep"].to(dev).chunk(cfg.tp)]
        dOut = [c.contiguous() for c in reg["dOut"].to(dev).chunk(cfg.tp)]
        gamma, beta = reg["gamma"].to(dev), reg["beta"].to(dev)
        ln_out = [torch.empty_like(c) for c in R]
        mean = torch.empty(cfg.M, device=dev)
        rstd = torch.empty(cfg.M, device=dev)
        out = [torch.empty_like(c) for c in R]
        dZs = [torch.empty_like(c) for c in R]
        dgam = torch.empty(cfg.h, device=dev)
        dbet = torch.empty(cfg.h, device=dev)
        ln_ws = torch.empty(max(16, tpmlp.sp_layernorm_backward_workspace(cfg.s, cfg.b, cfg.h)), dtype=torch.uint8,
                            device=dev)
        kw = dict(s=cfg.s, b=cfg.b, h=cfg.h, tp=cfg.tp, stream=stream)

        def step():
            tpmlp.sp_layernorm_forward(R, gamma, beta, 1e-5, ln_out, mean, rstd, **kw)
            blk.forward(ln_out, W1, W2, out=fw, stream=stream)
            tpmlp.sp_residual_dropout_forward(R, fw["z"], keep, 0.1, out, **kw)
            tpmlp.sp_residual_dropout_backward(dOut, keep, 0.1, dZs, **kw)
            if args.main_grad:
                blk.backward_main_grad(ln_out, W1, W2, fw, dZs, mg1, mg2, out=bw, stream=stream)
            else:
                blk.backward(ln_out, W1, W2, fw, dZs, out=bw, stream=stream)
            # dR = dOut (residual branch) + LayerNorm backward, accumulated in place into
            # the incoming-gradient chunks as a training step would (their values drift
            # from step to step; timing does not depend on values)
            tpmlp.sp_layernorm_backward(R, gamma, mean, rstd, bw["dx"], dOut, dgam, dbet, accumulate=True,
                                        workspace=ln_ws, **kw)
    else:
        def step():
            block_step(x, dz)

    def barrier():
        rank_barrier(world, lambda: torch.cuda.synchronize(dev))

    clocks = ClockSampler(gpu_uuid(local_rank)) if rank == 0 else None
    for _ in range(max(3, args.warmup)):
        step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    if clocks is not None:
        clocks.mark(t_host0, time.time())
    ms = e0.elapsed_time(e1) / args.steps
    # The same K steps again with a CUDA-event pair around every kernel launch
    # (tpmlp_profile_start/stop): the per-kernel durations of the roofline.
    # Kept out of the first region, whose step time they would lengthen.
    ms_prof, prof = profiled_region(tpmlp, step, args.steps, stream, barrier, clocks)
    status = tpmlp.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}: {tpmlp.last_error()}")
    ms_max = max_over_ranks(ms, world, dev)
    flops = float(cfg.flops_fwd_bwd())
    value = job_throughput(flops, world, ms_max)

    # ------------------------------------------------ end to end through the public API
    # Every step copies its input chunks (X, dZ) from pinned host memory and reads
    # its results (Z, dX) back, as a training loop feeding the layer would.  Two
    # device buffer sets and two copy streams double-buffer the traffic: the
    # inputs of step i+1 are uploaded and the results of step i-1 downloaded
    # while step i computes.  Weights and weight gradients are layer state that
    # stays on the device.
    e2e = None
    if not args.no_e2e and not args.sp_region:
        as_list = lambda t: list(t) if isinstance(t, (list, tuple)) else [t]  # noqa: E731
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        nset = 2
        xin = [[c.clone() for c in as_list(x)] for _ in range(nset)]
        dzin = [[c.clone() for c in as_list(dz)] for _ in range(nset)]
        fws = [blk.alloc_forward() for _ in range(nset)]
        bws = [blk.alloc_backward() for _ in range(nset)]
        xh = [pin(c) for c in as_list(x)]
        dzh = [pin(c) for c in as_list(dz)]
        zh = [[torch.empty_like(t, device="cpu").pin_memory() for t in as_list(fws[0]["z"])] for _ in range(nset)]
        dxh = [[torch.empty_like(t, device="cpu").pin_memory() for t in as_list(bws[0]["dx"])] for _ in range(nset)]
        h2d = sum(t.numel() * t.element_size() for t in xh + dzh)
        d2h = sum(t.numel() * t.element_size() for t in zh[0] + dxh[0])
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready = [ev() for _ in range(nset)]
        done = [ev() for _ in range(nset)]
        out_done = [ev() for _ in range(nset)]

        def upload(k):
            with torch.cuda.stream(s_in):
                s_in.wait_event(done[k])  # the set's previous step has consumed its inputs
                for d_, h_ in zip(xin[k], xh):
                    d_.copy_(h_, non_blocking=True)
                for d_, h_ in zip(dzin[k], dzh):
                    d_.copy_(h_, non_blocking=True)
                in_ready[k].record(s_in)

        def run_e2e(n):
            for k in range(nset):
                done[k].record(stream)
                out_done[k].record(stream)
            upload(0)
            for i in range(n):
                k = i % nset
                if i + 1 < n:
                    upload((i + 1) % nset)
                stream.wait_event(in_ready[k])
                stream.wait_event(out_done[k])  # the set's previous results have been downloaded
                xk = xin[k] if cfg.sp else xin[k][0]
                dzk = dzin[k] if cfg.sp else dzin[k][0]
                blk.forward(xk, W1, W2, out=fws[k], stream=stream)
                if args.main_grad:
                    blk.backward_main_grad(xk, W1, W2, fws[k], dzk, mg1, mg2, out=bws[k], stream=stream)
                else:
                    blk.backward(xk, W1, W2, fws[k], dzk, out=bws[k], stream=stream)
                done[k].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[k])
                    for h_, d_ in zip(zh[k], as_list(fws[k]["z"])):
                        h_.copy_(d_, non_blocking=True)
                    for h_, d_ in zip(dxh[k], as_list(bws[k]["dx"])):
                        h_.copy_(d_, non_blocking=True)
                    out_done[k].record(s_out)
            stream.wait_stream(s_out)

        run_e2e(max(3, args.warmup))
        barrier()
        n_e2e = args.steps  # the same number of steps as the device-only region, right after it
        t_host0 = time.time()
        e0.record(stream)
        run_e2e(n_e2e)
        e1.record(stream)
        barrier()
        if clocks is not None:
            clocks.mark(t_host0, time.time())
        ms_e2e_meas = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
        ms_e2e, flag = e2e_guard(ms_max, ms_e2e_meas)
        e2e = {"value": job_throughput(flops, world, ms_e2e), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
               "ms_per_step_measured": ms_e2e_meas, "steps": n_e2e,
               "note": "pinned-host chunks in, results out every step; copies double-buffered on two "
                       "copy streams against the compute stream; timed right after the device-only region "
                       "over as many steps"}
        if flag:
            e2e["flag"] = flag

    clock_info = clocks.stop() if clocks is not None else None
    dim0 = measure_dim0(tpmlp, cfg, dev, stream) if rank == 0 and not args.no_dim0 else {}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    # ------------------------------------------------ roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    g = prof["gemm_tc"] if prof["gemm_tc"]["launches"] else prof["gemm_f32"]
    launches_total = sum(v["launches"] for v in prof.values())
    per_kernel = {}
    for k, v in prof.items():
        if v["launches"]:
            unit = "TFLOP/s" if k.startswith("gemm") or k == "attn_core" else "GB/s"
            rate = v["work"] / (v["ms"] / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
            per_kernel[k] = {"launches_per_step": v["launches"] / args.steps, "ms_per_step": v["ms"] / args.steps,
                             "achieved": rate, "unit": unit,
                             "share_of_step": v["ms"] / args.steps / ms_prof}
    region_s = ms_max * args.steps / 1e3
    peak, regime, peak_key = choose_peak(peaks, region_s)
    # When every launch of the step is this kernel (the fused block), the timed
    # region is nothing but its launches back to back: their average duration is
    # the region's time over the launches, in the same window as `value`.  Else
    # (shard sums, SP-region kernels) the event pairs of the second region split
    # the step by kernel.
    only_kernel = launches_total == g["launches"]
    if only_kernel and g["launches"]:
        kernel_ms = ms_max * args.steps
        timing_note = (f"the timed region itself: the step runs only this kernel ({g['launches'] // args.steps} "
                       f"launches a step), so its launch durations are the region's {ms_max:.4f} ms/step "
                       f"(gaps between launches included)")
    else:
        kernel_ms = g["ms"]
        timing_note = (f"event pairs around every launch over a second region of the same {args.steps} steps "
                       f"({ms_prof:.4f} ms/step with the events; the line's ms_per_step is the region without them)")
    achieved = g["work"] / (kernel_ms / 1e3) / 1e12 if kernel_ms > 0 else None
    traffic = ncu_traffic(cfg.name, args.mode)
    roofline = {
        "bound": "tensor",
        "kernel": "tpmlp::tc::gemm_pair_kernel / gemm_kernel (tcgen05, all six GEMMs of the step)",
        "achieved": achieved,
        "peak": peak,
        "peak_source": f"{peak_src} {peak_key} (dense BF16; fp16 has the same tensor rate)",
        "peak_regime": f"{regime}: timed region {region_s:.3f} s "
                       f"({'<' if regime == 'burst' else '>='} {BURST_REGION_S:g} s)",
        "unit": "TFLOP/s",
        "frac": (achieved / peak) if achieved else None,
        "traffic": traffic.get("dram_bytes_per_launch") if traffic else None,
        "flops_per_launch": g["work"] / max(1, g["launches"]),
        "avg_launch_ms": kernel_ms / max(1, g["launches"]),
        "timing": timing_note,
        "frac_of_burst_peak": (achieved / peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) if achieved else None,
        "frac_of_sustained_peak": (achieved / (peaks.get("bf16_tflops_sustained")
                                               or FALLBACK_PEAKS["bf16_tflops_sustained"])) if achieved else None,
        "per_kernel": per_kernel,
    }
    hbm_peak = peaks.get("hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
    for v in dim0.values():
        v["frac_of_hbm"] = v["GB/s"] / hbm_peak
    if "copy_dim0" in per_kernel:
        hbm = peaks.get("hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
        roofline["per_kernel"]["copy_dim0"]["frac_of_hbm"] = per_kernel["copy_dim0"]["achieved"] / hbm
    if "shard_sum" in per_kernel:
        hbm = peaks.get("hbm_gbs") or FALLBACK_PEAKS["hbm_gbs"]
        roofline["per_kernel"]["shard_sum"]["frac_of_hbm"] = per_kernel["shard_sum"]["achieved"] / hbm

    # ------------------------------------------------ CPU oracle baseline (rank 0, N = 1)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        run, mt, _ = oracle_sample(cfg, inputs, args.cpu_seconds)
        t_cpu = run(mt)
        cpu = {"value": flops_for_tokens(cfg, mt) / t_cpu / 1e12, "unit": UNIT, "cores": cpu_cores(),
               "kind": "oracle",
               "sample": f"first {mt} of {cfg.M} tokens, full weights, fp64 NumPy fwd+bwd, one run of {t_cpu:.1f} s"}

    ebytes = ELEM_BYTES[cfg.dtype]
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic",
        "config": {**workload_desc(cfg), "reduce": args.mode,
                   "variant": ("sp-sublayer " if args.sp_region else "") + ("main_grad" if args.main_grad else "block"),
                   "l2": l2_note({"W1": cfg.fc1_rows * cfg.h * ebytes, "W2": cfg.h * cfg.f * ebytes,
                                  "U": cfg.M * cfg.fc1_rows * ebytes, "Y": cfg.M * cfg.f * ebytes}),
                   "flops_per_step": flops,
                   "replicas": world},
        "frac_of_dense_bf16_peak": {
            "applies": regime,
            "frac": value / world / peak,
            "sustained": value / world / (peaks.get("bf16_tflops_sustained") or FALLBACK_PEAKS["bf16_tflops_sustained"]),
            "burst": value / world / (peaks.get("bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"]),
            "peak_source": peak_src},
        "roofline": roofline,
        "dim0_kernels": {"note": "stand-alone launches at this workload's sizes, buffers rotating through >4x L2; "
                                 "in the step itself the all-gathers are fused into the GEMM loads when every "
                                 "sequence chunk is a whole number of 128-row blocks",
                         "hbm_peak_gbs": hbm_peak, **dim0},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_total,
        "clocks": clock_info,
        "kernel_source_sha256_16": kernel_source_hash(),
        "device": {"name": torch.cuda.get_device_name(dev),
                   "sms": torch.cuda.get_device_properties(dev).multi_processor_count},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_attention(args) -> int:
    """Forward + backward of the tensor-parallel attention block through the C ABI."""
    import torch

    from sp_partitioned_transformer_gb300 import build as _build

    _build.build()
    import sp_partitioned_transformer_gb300 as tpmlp
    from synthetic import ATTN_CONFIGS, attn_inputs

    tpmlp.load()
    name = args.config if args.config in ATTN_CONFIGS else "llama70b_attn_tpsp8_bf16"
    cfg = ATTN_CONFIGS[name]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    t = attn_inputs(cfg)
    X, Wqkv, Wo, dZ = (t[k].to(dev) for k in ("X", "Wqkv", "Wo", "dZ"))
    x = [c.contiguous() for c in X.chunk(cfg.tp)] if cfg.sp else X
    dz = [c.contiguous() for c in dZ.chunk(cfg.tp)] if cfg.sp else dZ
    blk = tpmlp.AttnBlock(cfg.s, cfg.b, cfg.h, cfg.heads, cfg.tp, cfg.sp, cfg.torch_dtype, cfg.causal, device=dev,
                          kv_heads=cfg.groups)
    stream = torch.cuda.current_stream(dev)
    fw = blk.forward(x, Wqkv, Wo, stream=stream)
    bw = blk.backward(x, Wqkv, Wo, fw, dz, stream=stream)
    kw = dict(s=cfg.s, b=cfg.b, h=cfg.h, heads=cfg.heads, tp=cfg.tp, sp=cfg.sp, causal=cfg.causal,
              kv_heads=cfg.groups, workspace=blk.ws, stream=stream)

    def step():
        tpmlp.attn_forward(x, Wqkv, Wo, fw["qkv"], fw["o"], fw["lse"], fw["z"], **kw)
        tpmlp.attn_backward(x, Wqkv, Wo, fw["qkv"], fw["o"], fw["lse"], dz, bw["dx"], bw["dwqkv"], bw["dwo"],
                            bw["dqkv"], bw["dout"], **kw)

    clocks = ClockSampler(gpu_uuid(0))
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(t_host0, time.time())
    ms = e0.elapsed_time(e1) / args.steps
    ms_prof, prof = profiled_region(tpmlp, step, args.steps, stream, lambda: torch.cuda.synchronize(dev), clocks)
    if tpmlp.device_status() != 0:
        raise RuntimeError(f"device status {tpmlp.device_status()}: {tpmlp.last_error()}")
    flops = float(cfg.flops_fwd_bwd())
    peaks, peak_src = load_peaks()
    region_s = ms * args.steps / 1e3
    peak, regime, peak_key = choose_peak(peaks, region_s)
    per_kernel = {}
    for k, v in prof.items():
        if v["launches"]:
            tf = k.startswith("gemm") or k == "attn_core"
            rate = v["work"] / (v["ms"] / 1e3) / (1e12 if tf else 1e9)
            per_kernel[k] = {"launches_per_step": v["launches"] / args.steps, "ms_per_step": v["ms"] / args.steps,
                             "achieved": rate, "unit": "TFLOP/s" if tf else "GB/s",
                             "share_of_step": v["ms"] / args.steps / ms_prof}
    a = prof["attn_core"]
    achieved = a["work"] / (a["ms"] / 1e3) / 1e12
    traffic = attn_ncu_traffic(cfg.name)

    # ------------------------------------------------ end to end through the C ABI
    # Every step uploads the X and dZ chunks from pinned host memory and
    # downloads Z and dX, double-buffered on two copy streams against the compute
    # stream (weights and weight gradients stay on the device), as for the MLP.
    e2e = None
    if not args.no_e2e:
        as_list = lambda v: list(v) if isinstance(v, (list, tuple)) else [v]  # noqa: E731
        pin = lambda v: v.cpu().pin_memory()  # noqa: E731
        nset = 2
        xin = [[c.clone() for c in as_list(x)] for _ in range(nset)]
        dzin = [[c.clone() for c in as_list(dz)] for _ in range(nset)]
        fws = [blk.forward(x, Wqkv, Wo, stream=stream) for _ in range(nset)]
        bws = [blk.backward(x, Wqkv, Wo, fws[k], dz, stream=stream) for k in range(nset)]
        xh = [pin(c) for c in as_list(x)]
        dzh = [pin(c) for c in as_list(dz)]
        zh = [[torch.empty_like(v, device="cpu").pin_memory() for v in as_list(fws[0]["z"])] for _ in range(nset)]
        dxh = [[torch.empty_like(v, device="cpu").pin_memory() for v in as_list(bws[0]["dx"])] for _ in range(nset)]
        h2d = sum(v.numel() * v.element_size() for v in xh + dzh)
        d2h = sum(v.numel() * v.element_size() for v in zh[0] + dxh[0])
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(nset)]
        done = [torch.cuda.Event() for _ in range(nset)]
        out_done = [torch.cuda.Event() for _ in range(nset)]

        def upload(k):
            with torch.cuda.stream(s_in):
                s_in.wait_event(done[k])  # the set's previous step has consumed its inputs
                for d_, h_ in zip(xin[k] + dzin[k], xh + dzh):
                    d_.copy_(h_, non_blocking=True)
                in_ready[k].record(s_in)

        def run_e2e(n):
            for k in range(nset):
                done[k].record(stream)
                out_done[k].record(stream)
            upload(0)
            for i in range(n):
                k = i % nset
                if i + 1 < n:
                    upload((i + 1) % nset)
                stream.wait_event(in_ready[k])
                stream.wait_event(out_done[k])  # the set's previous results have been downloaded
                xk = xin[k] if cfg.sp else xin[k][0]
                dzk = dzin[k] if cfg.sp else dzin[k][0]
                f_, b_ = fws[k], bws[k]
                tpmlp.attn_forward(xk, Wqkv, Wo, f_["qkv"], f_["o"], f_["lse"], f_["z"], **kw)
                tpmlp.attn_backward(xk, Wqkv, Wo, f_["qkv"], f_["o"], f_["lse"], dzk, b_["dx"], b_["dwqkv"],
                                    b_["dwo"], b_["dqkv"], b_["dout"], **kw)
                done[k].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[k])
                    for h_, d_ in zip(zh[k] + dxh[k], as_list(f_["z"]) + as_list(b_["dx"])):
                        h_.copy_(d_, non_blocking=True)
                    out_done[k].record(s_out)
            stream.wait_stream(s_out)

        run_e2e(max(3, args.warmup))
        n_e2e = args.steps  # the same number of steps as the device-only region
        torch.cuda.synchronize(dev)
        t_host0 = time.time()
        e0.record(stream)
        run_e2e(n_e2e)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(t_host0, time.time())
        if tpmlp.device_status() != 0:
            raise RuntimeError(f"device status {tpmlp.device_status()}: {tpmlp.last_error()}")
        ms_e2e_meas = e0.elapsed_time(e1) / n_e2e
        ms_e2e, flag = e2e_guard(ms, ms_e2e_meas)
        e2e = {"value": flops / (ms_e2e / 1e3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e, "ms_per_step_measured": ms_e2e_meas,
               "steps": n_e2e,
               "note": "pinned-host chunks in, results out every step; copies double-buffered on two "
                       "copy streams against the compute stream; timed right after the device-only region "
                       "over as many steps"}
        if flag:
            e2e["flag"] = flag
    clock_info = clocks.stop()

    # ------------------------------------------------ CPU oracle baseline
    cpu = None
    if not args.no_cpu_baseline:
        cpu = attn_oracle_baseline(cfg, t, args.cpu_seconds)

    line = {
        "metric": ATTN_METRIC,
        "value": flops / (ms / 1e3) / 1e12,
        "unit": UNIT,
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic",
        "config": attn_workload_desc(cfg),
        "frac_of_dense_bf16_peak": {"applies": regime, "frac": flops / (ms / 1e3) / 1e12 / peak,
                                    "peak_source": peak_src},
        "roofline": {"bound": "tensor", "kernel": "tpmlp::attn core (attn_fwd_kernel, attn_bwd_dkdv_kernel, "
                                                  "attn_bwd_dq_kernel, attn_bwd_delta_kernel)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} {peak_key}",
                     "peak_regime": f"{regime}: timed region {region_s:.3f} s "
                                    f"({'<' if regime == 'burst' else '>='} {BURST_REGION_S:g} s)",
                     "traffic": traffic.get("dram_bytes_per_pass") if traffic else None,
                     "traffic_note": "DRAM bytes of one fwd+bwd pass of the four core kernels (ncu, "
                                     "profiles/attn_dram_traffic.json, matched to the built source)",
                     "timing": f"event pairs around every launch over a second region of the same {args.steps} "
                               f"steps ({ms_prof:.4f} ms/step with the events)",
                     "per_kernel": per_kernel},
        "gpu_launches": sum(v["launches"] for v in prof.values()),
        "clocks": clock_info,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "device": {"name": torch.cuda.get_device_name(dev),
                   "sms": torch.cuda.get_device_properties(dev).multi_processor_count},
    }
    print(json.dumps(line), flush=True)
    return 0


def attn_oracle_sample(cfg, inputs, target_s: float):
    """The fp64 oracle's attention block fwd+bwd (its backward runs the forward
    too) on the first s' tokens of every sequence with full weights, s' sized so
    one run takes about target_s and at most 1024 (the oracle holds several
    [b, heads, s', s'] fp64 matrices); FLOPs counted as on the GPU (12·M'·h·(h + h_kv) for
    the projections, 12·b·h per visible query-key pair).  Returns (run, s',
    flops): run(s') times one pass in seconds."""
    import oracle as O

    X = inputs["X"].double().numpy()
    dZ = inputs["dZ"].double().numpy()
    Wqkv = inputs["Wqkv"].double().numpy()
    Wo = inputs["Wo"].double().numpy()

    def flops(sp_):
        pairs = sp_ * (sp_ + 1) / 2 if cfg.causal else float(sp_) * sp_
        return 12.0 * sp_ * cfg.b * cfg.h * (cfg.h + cfg.h_kv) + 12.0 * cfg.b * cfg.h * pairs

    def run(sp_):
        t0 = time.perf_counter()
        O.attn_backward(X[:sp_].reshape(sp_ * cfg.b, cfg.h), Wqkv, Wo, dZ[:sp_].reshape(sp_ * cfg.b, cfg.h), sp_,
                        cfg.b, cfg.heads, cfg.causal, cfg.groups)
        return time.perf_counter() - t0

    probe = min(32, cfg.s)
    t_probe = run(probe)
    sp_ = probe
    if t_probe < target_s:
        sp_ = int(min(cfg.s, 1024, max(probe, probe * target_s / max(t_probe, 1e-3))))
        sp_ = max(probe, sp_ // 32 * 32)
    return run, sp_, flops(sp_)


def attn_oracle_baseline(cfg, inputs, target_s: float):
    """One timed oracle run of attn_oracle_sample's size, as a cpu_baseline entry."""
    run, sp_, fl = attn_oracle_sample(cfg, inputs, target_s)
    t_run = run(sp_)
    return {"value": fl / t_run / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"first {sp_} of {cfg.s} tokens of each of {cfg.b} sequence(s), full weights, fp64 NumPy "
                      f"attention block fwd+bwd, one run of {t_run:.1f} s"}


def main(argv=None) -> int:
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.block == "attention":
        return run_attention(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
