"""Decode-step benchmark: tokens/s of the 27B-class 64-layer INT4 stack at batch 1.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--batch B] [--weights int4|bf16] [--mode 0|1]

A step is one decode step of the whole stack (every layer's fused QKV+RoPE+
append, GQA attention, Wo, gate/up+SwiGLU, down) for one batch of synthetic
input, with weights and KV history resident in HBM.  The stack streams
18.7 GB per step, far more than the 129 MB L2, so no flush is needed
between steps.  Under torchrun (N > 1) every rank runs an independent
replica of the step (the path has no exchange step); value = tokens of all
ranks / the slowest rank's time.  Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tokens/s (27B-shape INT4, 64 layers); achieved HBM GB/s vs 8 TB/s"


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=None)
    p.add_argument("--batch", type=int, default=None)
    p.add_argument("--weights", default=None, choices=[None, "int4", "bf16"])
    p.add_argument("--layers", type=int, default=None)
    p.add_argument("--mode", type=int, default=0, help="0 persistent kernel, 1 launch per stage")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-token-step", action="store_true",
                   help="skip the token step (embedding + stack + LM head + greedy id)")
    return p.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _slowest(ms: float, world: int, device: str) -> float:
    """The slowest rank's time (max over ranks); every rank gets it."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _job_rate(world: int, batch: int, ms: float) -> float:
    """Whole-job tokens/s: each rank decodes `batch` tokens a step and the
    job's step takes the slowest rank's time."""
    return world * batch / (ms * 1e-3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The sources the batch-1 decode kernel is compiled from.
_DECODE_SOURCES = ("ddl_decode.cu", "ddl_device.cuh", "ddl_plan.h")


def _source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "memory_bound_transformer_decode_gb300", "csrc")
    for f in _DECODE_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def _traffic(workload: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")
    try:
        d = json.load(open(path))
        e = d.get(workload)
        if e and e.get("source_hash") == _source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class Clocks:
    """nvidia-smi samples (every 50 ms) kept for the timed region: the sampler
    is started before the warm-up and each line is stamped on arrival, so a
    short timed region still has its own samples (the nearest one on each
    side when it is shorter than the sampling period)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []  # (monotonic seconds at arrival, line)
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.monotonic() + 5.0
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def begin(self):
        self.t0 = time.monotonic()

    def end(self):
        self.t1 = time.monotonic()
        if self.proc:  # one more period, so that a sample after the region exists
            time.sleep(1.5 * self.period_ms / 1000)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.t0 is None or self.t1 is None:
            return None
        inside = [ln for t, ln in self.lines if self.t0 <= t <= self.t1]
        if not inside:  # a region shorter than the period: the samples around it
            before = [ln for t, ln in self.lines if t < self.t0][-1:]
            after = [ln for t, ln in self.lines if t > self.t1][:1]
            inside = before + after
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in inside:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "period_ms": self.period_ms,
                "region_s": round(self.t1 - self.t0, 4)}


def _oracle_layer(cfg):
    """Layer 0 of the workload for the oracle: quantized weights, its K/V
    cache and the step's input, on the host."""
    import torch

    import oracle
    from memory_bound_transformer_decode_gb300 import synth

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = {k: synth.bits(v) for k, v in synth.layer_weights(cfg, 0, device=dev).items()}
    lw = oracle.quantized_layer(w)
    del w
    kc, vc = synth.kv_cache(cfg, 0, cfg.kv_len + 1, device=dev, batch=cfg.batch)
    kc, vc = synth.bits(kc).copy(), synth.bits(vc).copy()
    x = oracle.bf16_to_f64(synth.bits(synth.input_x(cfg, device=dev, batch=cfg.batch)))
    return lw, kc, vc, x


def _cpu_baseline(cfg, target_s: float = 12.0):
    """The oracle as it stands, on the host cores, over whole layers of the
    workload; tokens/s = 1 / (seconds per layer * layers)."""
    import oracle

    lw, kc, vc, x = _oracle_layer(cfg)
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle.layer_decode(cfg, lw, kc, vc, cfg.pos, x)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > target_s or len(times) >= 50:
            break
    per_layer = statistics.median(times)
    return {
        "value": cfg.batch / (per_layer * cfg.layers),
        "unit": "tokens/s",
        "cores": oracle.num_threads(),
        "kind": "oracle",
        "sample": f"{len(times)} decode steps of one layer (layer 0) of the {cfg.layers}-layer "
                  f"stack, fp64 C oracle, median {per_layer:.3f} s/layer, scaled x{cfg.layers} layers",
    }, per_layer


def _config_json(cfg, B, wname, L):
    return {"workload": cfg.name, "layers": L, "batch": B, "kv_len": cfg.kv_len, "D": cfg.D,
            "H_q": cfg.H_q, "H_kv": cfg.H_kv, "head_dim": cfg.head_dim, "d_ff": cfg.d_ff,
            "weights": "int4-g64-bf16-scale" if wname == "int4" else "bf16",
            "l2": "inputs larger than L2 (no flush needed)", "parallelism": "replicas"}


def run_reference(args):
    from memory_bound_transformer_decode_gb300 import configs

    rank, world, _ = _dist()
    if rank != 0:
        return
    cfg = configs.BY_NAME.get(args.workload) if args.workload else configs.STACK27B
    B = args.batch or cfg.batch
    cfg = cfg.with_(batch=B)
    import oracle

    lw, kc, vc, x0 = _oracle_layer(cfg)
    cores = oracle.num_threads()
    # A step is the stack's layers in turn, each on layer 0's weights and
    # cache with the previous layer's output as input: the whole step's
    # arithmetic and bytes.  Only if K + W such steps would take longer than
    # about 150 s does a step run fewer layers (then scaled to the stack).
    t0 = time.perf_counter()
    oracle.layer_decode(cfg, lw, kc, vc, cfg.pos, x0)
    t_layer = time.perf_counter() - t0
    budget = 150.0 / max(1, args.warmup + args.steps)
    n = max(1, min(cfg.layers, int(budget / max(t_layer, 1e-6))))
    per = []
    for i in range(args.warmup + args.steps):
        x = x0
        t0 = time.perf_counter()
        for _ in range(n):
            x = oracle.layer_decode(cfg, lw, kc, vc, cfg.pos, x)
        if i >= args.warmup:
            per.append(time.perf_counter() - t0)
    step_s = statistics.median(per) * cfg.layers / n
    value = B / step_s
    sample = (f"each step: {n} of the {cfg.layers} layers in turn through the fp64 C oracle, each on "
              f"layer 0's weights and K/V cache with the previous layer's output as input"
              + (f", scaled x{cfg.layers}/{n}" if n < cfg.layers else " (measured, not scaled)")
              + f"; median of {args.steps} timed steps")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config_json(cfg, B, cfg.weights, cfg.layers),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }))


def _token_step(args, cfg, st, wname, world, barrier, stream):
    """The whole token step on the device: embedding rows of the previous
    step's ids -> the layer stack -> the LM head over the vocabulary (the tied
    table, with a final RMSNorm) -> greedy ids, fed back to the next step."""
    import torch

    from memory_bound_transformer_decode_gb300 import configs, ddl, synth

    B, D, V = cfg.batch, cfg.D, configs.VOCAB
    wt = ddl.INT4 if wname == "int4" else ddl.BF16
    hw = synth.head_weights(cfg, V, device="cuda")
    if wt == ddl.INT4:
        q, s = ddl.ddl_quantize_int4(hw["embed"])
        packed = ddl.ddl_pack_head((q, s), D, V, wt)
        del q, s
    else:
        packed = ddl.ddl_pack_head(hw["embed"], D, V, wt)
    table, norm_f = hw["embed"], hw["norm_f"]
    ws = torch.empty(ddl.ddl_head_workspace_bytes(D, V, B), dtype=torch.uint8, device="cuda")
    tok = torch.zeros(B, dtype=torch.int32, device="cuda")
    x = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((B, D), dtype=torch.float32, device="cuda")

    def step(ev=None):
        ddl.ddl_embed(table, tok, out=x)
        st.decode(resid_out=res, x=x)
        if ev:
            ev[0].record(stream)
        ddl.ddl_lm_head(D, V, wt, packed, res, norm_f=norm_f, eps=cfg.eps, tokens=tok, workspace=ws)
        if ev:
            ev[1].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    barrier()
    hev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(hev[i])
    e1.record(stream)
    barrier()
    status = ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max)
    if status != 0:
        raise RuntimeError(f"device status {status} in the token step")
    ms = _slowest(e0.elapsed_time(e1) / args.steps, world, "cuda")
    head_ms = statistics.mean(a.elapsed_time(b) for a, b in hev)
    head_bytes = ddl.ddl_packed_head_bytes(D, V, wt)
    return {"value": _job_rate(world, B, ms), "unit": "tokens/s", "ms_per_step": ms, "vocab": V,
            "sampling": "greedy", "head_ms": head_ms,
            "head_roofline": {"bound": "hbm", "achieved": head_bytes / (head_ms * 1e-3) / 1e9,
                              "unit": "GB/s", "traffic": None,
                              "kernel": "head_prep + head_gemv + head_select (one step's LM head)"}}


def run_ours(args):
    import torch

    from memory_bound_transformer_decode_gb300 import configs, ddl, roofline, workload

    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    ddl.load(build_if_missing=True)
    ddl.ddl_set_launch_mode(args.mode)
    cfg = configs.BY_NAME.get(args.workload) if args.workload else configs.STACK27B
    B = args.batch or cfg.batch
    wname = args.weights or cfg.weights
    L = args.layers or cfg.layers
    cfg = cfg.with_(batch=B, weights=wname, layers=L)
    st = workload.build_stack(cfg)
    stream = torch.cuda.current_stream()
    out = torch.empty((B, cfg.D), dtype=torch.bfloat16, device="cuda")

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    clk = Clocks(local).start()
    for _ in range(max(3, args.warmup)):
        st.decode(out_bf16=out)
    barrier()
    status = ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max)
    if status != 0:
        clk.stop()
        raise RuntimeError(f"device status {status} after warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    try:
        barrier()
        clk.begin()
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            st.decode(out_bf16=out)
            ev[i][1].record(stream)
        t_all1.record(stream)
        barrier()
        clk.end()
    finally:
        clk.stop()
    total_ms = t_all0.elapsed_time(t_all1)
    per_ms = [a.elapsed_time(b) for a, b in ev]
    ms = _slowest(total_ms / args.steps, world, "cuda")
    status = ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max)
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")

    # end to end through the public API: pinned host x in, bf16 out back, every step
    x_host = st.x.cpu().pin_memory()
    out_host = torch.empty((B, cfg.D), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(st.x)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        x_dev.copy_(x_host, non_blocking=True)
        st.decode(out_bf16=out, x=x_dev)
        out_host.copy_(out, non_blocking=True)
    e1.record(stream)
    barrier()
    e2e_ms = _slowest(e0.elapsed_time(e1) / args.steps, world, "cuda")

    token = None if args.no_token_step else _token_step(args, cfg, st, wname, world, barrier, stream)

    nbytes = roofline.step_bytes(cfg)
    peak, peak_kind = _peaks()
    kernel_ms = statistics.mean(per_ms)
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    tc = (wname == "int4" and B >= 16) or (wname == "bf16" and B > 4)
    if tc:  # per layer: 4 tensor-core GEMMs, 4 epilogues, the attention operands, the attention stage
        launches_per_step = L * 10 + (L + 95) // 96
        kernel = ("tc_gemm_kernel + tc_epi_kernel per weight stage, decode_kernel for attention "
                  "(step-level roofline over all launches)")
    else:
        launches_per_step = (L + 95) // 96 if args.mode == 0 else L * 5
        kernel = "decode_kernel (one persistent launch per step)"
    line = {
        "metric": METRIC,
        "value": _job_rate(world, B, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,0.02) weights quantized to INT4, N(0,1) KV and x)",
        "config": _config_json(cfg, B, wname, L),
        "us_per_layer": ms * 1e3 / L,
        "hbm_gbs": nbytes / (ms * 1e-3) / 1e9,
        "bytes_per_step": nbytes,
        "p10_p50_p90_ms": [float(np.percentile(per_ms, q)) for q in (10, 50, 90)],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"hbm_gbs of {peak_kind}",
                     "traffic": _traffic(cfg.name),
                     "kernel": kernel},
        "e2e": {"value": _job_rate(world, B, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": B * cfg.D * 2, "d2h_bytes_per_step": B * cfg.D * 2},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if token is not None:
        token["head_roofline"]["frac"] = token["head_roofline"]["achieved"] / peak
        token["head_roofline"]["peak"] = peak
        line["token_step"] = token
    if rank == 0 and not args.no_cpu_baseline:
        cb, _ = _cpu_baseline(cfg)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
