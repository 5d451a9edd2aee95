#!/usr/bin/env python
"""Benchmark of the MoE layer forward pass on B300: layer tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = one moe_forward over a resident batch of the Mixtral-shaped
prefill layer (T=4096 tokens, d_model=4096, d_ff=14336, 8 experts, top-2,
dropless): gate, TopK-then-softmax routing, dispatch, both grouped expert
GEMMs, combine and the balance loss. Synthetic inputs on the 1/64 grid, random
bf16 expert weights. The expert weights alone (1.88 GB) exceed L2, so every
step streams them from HBM; no explicit flush is added.

Prints ONE JSON line on rank 0. Under torchrun (N > 1) every rank runs an
independent replica on its own GPU and batch (no collective on the data path;
"scaling": "weak"); a barrier and a max-reduction of the elapsed time are the
only cross-rank traffic.

--impl reference times the CPU oracle (plain C, fp64, OpenMP) on the host
cores instead: each step runs the oracle's full layer on a bounded sub-batch
of the same workload's tokens (dropless, so tokens are independent).
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

METRIC = "MoE-layer tokens/s"
UNIT = "tokens/s"


def gemm_traffic(kernel_source: str):
    """DRAM bytes per step of the grouped GEMM from the committed ncu summary,
    or None when the kernel source changed since those counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "grouped_gemm_mixtral_prefill.json")) as fh:
            prof = json.load(fh)
        with open(os.path.join(ROOT, kernel_source), "rb") as fh:
            h = hashlib.sha256(fh.read()).hexdigest()
    except (OSError, ValueError):
        return None
    return prof["dram_bytes_per_step"] if prof.get("source_sha256") == h else None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 100 ms) while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid: str | None):
        self.uuid = device_uuid
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.25)

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [s for s, p in zip(sm, power) if p > 200.0] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample(cfg, inp_cpu, n_tokens: int, seed: int = 0):
    """Run the oracle's whole layer on a sub-batch of n_tokens of the workload;
    returns (seconds, n_tokens)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    sel = np.sort(rng.choice(cfg.T, size=n_tokens, replace=False))
    xs = inp_cpu.x[sel].contiguous()
    t0 = time.perf_counter()
    oracle.default().forward(xs, inp_cpu.Wg, inp_cpu.W1, inp_cpu.b1, inp_cpu.W2, inp_cpu.b2, cfg.K,
                             cfg.capacity_factor, cfg.aux_alpha, inp_cpu.sel_bias, inp_cpu.Ws1, inp_cpu.bs1,
                             inp_cpu.Ws2, inp_cpu.bs2)
    return time.perf_counter() - t0, n_tokens


def cpu_cores() -> int:
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def sample_desc(cfg, n):
    return (f"oracle full layer (fp64 gate, TopK, softmax, dispatch, expert FFNs, combine, aux) on a "
            f"sub-batch of {n} of the {cfg.T} tokens of {cfg.name}; dropless, so each token's work is "
            f"identical to the full batch's")


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(dist, value: float, device) -> float:
    """The slowest rank's time: every rank's number, reduced with MAX (the
    only cross-rank traffic besides barriers; replicas exchange no data)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, tokens_per_rank: int, steps: int, elapsed_ms: float) -> float:
    """Tokens per second summed over all ranks (weak scaling: each rank runs
    its own batch of tokens_per_rank every step)."""
    return world * tokens_per_rank * steps / (elapsed_ms * 1e-3)


def workload_config(cfg, extra=None):
    c = {"workload": f"{cfg.name}: T={cfg.T} d_model={cfg.d_model} d_ff={cfg.d_ff} N={cfg.N} K={cfg.K} "
                     f"capacity_factor={'dropless' if cfg.capacity_factor <= 0 else cfg.capacity_factor}"
                     f"{' +shared' if cfg.has_shared else ''}{' +sel_bias' if cfg.sel_bias else ''}"
                     f"{' expert_weights=fp8_e4m3 (per-output-channel scales)' if cfg.weights == 'fp8_e4m3' else ''}",
         "tokens_per_step_per_gpu": cfg.T,
         "l2": "inputs larger than L2: the expert weights read every step exceed the 126 MB L2; no flush"}
    if extra:
        c.update(extra)
    return c


def run_reference(args, cfg):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from top_routing_expert_then_b300.inputs import make_inputs
    import oracle
    oracle.build()
    inp = make_inputs(cfg, args.seed, device="cpu")
    # calibrate the sub-batch so the whole run stays within a few minutes
    t1, _ = oracle_sample(cfg, inp, 2, seed=99)
    per_tok = max(t1 / 2, 1e-4)
    budget = 150.0 / max(args.steps + args.warmup, 1)
    n = int(max(1, min(cfg.T, budget / per_tok)))
    for i in range(args.warmup):
        oracle_sample(cfg, inp, n, seed=1000 + i)
    tot_t, tot_n = 0.0, 0
    for i in range(args.steps):
        dt, k = oracle_sample(cfg, inp, n, seed=i)
        tot_t += dt
        tot_n += k
    value = tot_n / tot_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(cfg, {"tokens_per_step_per_gpu": n}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample_desc(cfg, n)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="mixtral_prefill")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-sample", type=int, default=1024, help="tokens in the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--backward-steps", type=int, default=10,
                    help="also time moe_backward (forward recompute + backward) for this many steps; 0 = off")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from top_routing_expert_then_b300.inputs import CONFIGS
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)

    import torch
    from top_routing_expert_then_b300 import lib
    from top_routing_expert_then_b300.inputs import make_dy, make_inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    inp = make_inputs(cfg, args.seed + rank, device=dev)
    layer = lib.MoELayer.from_inputs(inp)
    ro = layer.route_outputs()
    y = torch.empty_like(inp.x)
    stream = torch.cuda.current_stream()
    P = peaks()

    # warm-up (also yields the kept-row count for the FLOP figure)
    for _ in range(args.warmup):
        layer.forward(inp.x, inp.sel_bias, y=y, route_out=ro)
    torch.cuda.synchronize()
    if lib.device_error() != 0:
        raise RuntimeError("device error during warm-up")
    R = int(ro.expert_offsets[-1].item())
    hit = int((ro.kept > 0).sum().item())
    T, d, f = cfg.T, cfg.d_model, cfg.d_ff
    ffn_flops = 4.0 * R * d * f + (4.0 * T * d * f if cfg.has_shared else 0.0)
    # algorithmic bytes of the two grouped GEMMs: weights of every expert that
    # received rows (+ shared), x_perm in, H out and back in, y_perm out
    rows_all = R + (T if cfg.has_shared else 0)
    fp8 = cfg.weights == "fp8_e4m3"
    w_elem = 1 if fp8 else 2  # bytes per expert weight (+ one fp32 scale per output channel with FP8)
    w_bytes = 2.0 * d * f * w_elem + ((d + f) * 4 if fp8 else 0)
    ffn_bytes = (hit + (1 if cfg.has_shared else 0)) * w_bytes + rows_all * (2 * d + 4 * f + 2 * d)

    # ---- timed region: K steps, per-stage marks on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for row in ev:  # torch creates the CUDA event on its first record
        for e in row:
            e.record(stream)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    launches0 = lib.launch_count()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        layer.forward_marked(inp.x, ev[i], inp.sel_bias, y=y, route_out=ro)
    stop.record(stream)
    torch.cuda.synchronize()
    launches = lib.launch_count() - launches0
    if pg:
        pg.barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(pg, start.elapsed_time(stop), dev)
    if lib.device_error() != 0:
        raise RuntimeError("device error during the timed region")

    stage_names = ["route_aux", "dispatch", "ffn_gemm1", "ffn_gemm2", "combine"]
    stage_ms = [sum(e[j].elapsed_time(e[j + 1]) for e in ev) / args.steps for j in range(5)]
    gemm_ms = stage_ms[2] + stage_ms[3]
    achieved_tflops = ffn_flops / (gemm_ms * 1e-3) / 1e12
    peak_t = P["bf16_tflops_sustained"]
    achieved_gbs = ffn_bytes / (gemm_ms * 1e-3) / 1e9
    # the binding roof: tensor when the GEMMs' FLOP per byte exceeds the
    # machine balance (sustained bf16 / HBM), else HBM
    tensor_bound = ffn_flops / ffn_bytes > peak_t * 1e12 / (P["hbm_gbs"] * 1e9)

    # HBM-bound stages: algorithmic bytes per step
    K, N = cfg.K, cfg.N
    route_bytes = T * d * 2 + N * d * 2 + T * K * 8 + N * 8
    dispatch_bytes = T * K * 4 * 4 + T * d * 2 + R * d * 2
    combine_bytes = R * d * 2 + T * d * 2 + (T * d * 2 if cfg.has_shared else 0) + T * K * 8

    value = whole_job_rate(world, T, args.steps, elapsed_ms)

    # ---- end to end through the public API with host buffers
    # (moe_forward_hostio_batches: every step copies its input from pinned host
    # memory and its output back, double-buffered on the library's copy
    # streams so the copies of steps i+1 and i-1 overlap step i's forward)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    xd = torch.empty((2,) + tuple(inp.x.shape), dtype=inp.x.dtype, device=dev)
    yd = torch.empty_like(xd)
    layer.forward_hostio_batches(x_host, y_host, 3, xd, yd, inp.sel_bias, same_host=True, stream=stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer.forward_hostio_batches(x_host, y_host, args.e2e_steps, xd, yd, inp.sel_bias, same_host=True,
                                 stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(pg, e0.elapsed_time(e1), dev)
    e2e_value = whole_job_rate(world, T, args.e2e_steps, e2e_ms)

    # ---- training step: moe_backward (recomputes the forward, then every gradient)
    train = None
    if args.backward_steps > 0 and cfg.weights == "bf16":
        dy = make_dy(cfg, args.seed, device=dev)
        bws = lib.workspace(layer.shape, lib.MOE_WS_BACKWARD, dev)
        for _ in range(2):
            layer.backward(inp.x, dy, inp.sel_bias, ws=bws)
        torch.cuda.synchronize()
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(args.backward_steps):
            layer.backward(inp.x, dy, inp.sel_bias, ws=bws)
        b1.record(stream)
        torch.cuda.synchronize()
        bwd_ms = max_over_ranks(pg, b0.elapsed_time(b1), dev) / args.backward_steps
        train = {"ms_per_step": bwd_ms, "tokens_per_s": whole_job_rate(world, T, 1, bwd_ms),
                 "steps": args.backward_steps, "what": "moe_backward: forward recompute + all gradients (fp32)"}
        del bws

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        inp_cpu = inp.to("cpu")
        dt, n = oracle_sample(cfg, inp_cpu, args.cpu_sample, seed=7)
        cpu = {"value": n / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": sample_desc(cfg, n), "seconds": round(dt, 2)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg, {"kept_rows": R, "parallelism": f"replicas{world}"}),
        "roofline": {"kernel": ("grouped_gemm_fp8t_kernel (both expert Linears, FP8 weights widened into tensor "
                                "memory, channel-major tcgen05)") if fp8 else
                               "grouped_gemm_kernel (both expert Linears, tcgen05)",
                     "bound": "tensor" if tensor_bound else "hbm",
                     "achieved": achieved_tflops if tensor_bound else achieved_gbs,
                     "peak": peak_t if tensor_bound else P["hbm_gbs"],
                     "unit": "TFLOP/s" if tensor_bound else "GB/s",
                     "frac": achieved_tflops / peak_t if tensor_bound else achieved_gbs / P["hbm_gbs"],
                     "tflops": achieved_tflops, "gbs": achieved_gbs, "bytes_per_step": ffn_bytes,
                     "traffic": gemm_traffic("top_routing_expert_then_b300/csrc/grouped_gemm.cuh")
                     if cfg.name == "mixtral_prefill" else None,
                     "traffic_unit": "DRAM bytes per step (both launches), ncu",
                     "peak_kind": f"{P['source']} sustained bf16" if tensor_bound else f"{P['source']} HBM copy",
                     "frac_of_burst": achieved_tflops / P["bf16_tflops"],
                     "flops_per_step": ffn_flops, "ms_per_step": gemm_ms},
        "stages_us": {n: round(1e3 * m, 2) for n, m in zip(stage_names, stage_ms)},
        "hbm_stages": {
            "route_aux": {"bytes": route_bytes, "gbs": route_bytes / (stage_ms[0] * 1e-3) / 1e9},
            "dispatch": {"bytes": dispatch_bytes, "gbs": dispatch_bytes / (stage_ms[1] * 1e-3) / 1e9},
            "combine": {"bytes": combine_bytes, "gbs": combine_bytes / (stage_ms[4] * 1e-3) / 1e9},
            "peak_gbs": P["hbm_gbs"]},
        "cpu_baseline": cpu,
        "train_step": train,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * d * 2,
                "api": "moe_forward_hostio_batches (pinned host in/out every step, copies overlapped)",
                "steps": args.e2e_steps},
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
