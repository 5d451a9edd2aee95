#!/usr/bin/env python
"""Benchmark of the MoE layer forward pass on B300: layer tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = one moe_forward over a resident batch of the DeepSeek-V3-shaped
layer (T=4096 tokens, d_model=7168, d_ff=2048, 256 routed experts + 1 shared,
top-8, per-expert selection bias, dropless), the largest of the pages'
workloads that fits one GPU: gate, TopK-then-softmax routing, dispatch, the
grouped expert GEMMs, combine and the balance loss. Synthetic inputs on the
1/64 grid, random bf16 expert weights. The expert weights read every step
(15 GB) exceed L2, so every step streams them from HBM; no explicit flush is
added. The same run times further workloads (the Mixtral-shaped prefill layer,
the tensor-core target, and the 16-token decode layer with bf16 and FP8
expert weights, the weight-streaming targets) and reports them under
"workloads".

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


def gemm_traffic(workload: str):
    """DRAM bytes per step of the grouped GEMM launches of `workload` from the
    committed ncu summary (profiles/grouped_gemm_<workload>.json), or None
    when there is none or the kernel source changed since the counters were
    taken (the summary records the source's sha256)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", f"grouped_gemm_{workload}.json")) as fh:
            prof = json.load(fh)
        with open(os.path.join(ROOT, prof["source"]), "rb") as fh:
            h = hashlib.sha256(fh.read()).hexdigest()
    except (OSError, ValueError, KeyError):
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


def choose_peak(P, clk, region_ms: float):
    """The bf16 peak that matches the timed region's conditions: the burst
    figure (a short run at full clocks) when the region lasted under a second
    or the median sampled SM clock was at least 95% of the maximum; the
    sustained, power-capped figure otherwise."""
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    burst = region_ms < 1000.0 or (sm is not None and smax and sm >= 0.95 * smax)
    return ("burst", P["bf16_tflops"]) if burst else ("sustained", P["bf16_tflops_sustained"])


def ffn_work(cfg, R: int, hit: int):
    """Algorithmic FLOPs and bytes of one step's expert GEMMs: 4 d f FLOPs per
    kept row (two Linears) plus the shared expert's per token. Bytes: the
    weights of every expert that received rows (+ the shared expert's, + one
    fp32 scale per output channel with FP8); x once (the bf16 path gathers the
    kept rows of x inside the first GEMM; the FP8 path reads the regrouped
    copy, one row per kept row, and the shared expert reads x); the hidden
    rows written and read back; the output rows written (and z)."""
    T, d, f = cfg.T, cfg.d_model, cfg.d_ff
    flops = 4.0 * R * d * f + (4.0 * T * d * f if cfg.has_shared else 0.0)
    rows_all = R + (T if cfg.has_shared else 0)
    if cfg.weights == "fp8_e4m3":      # one byte a weight + an fp32 scale per output channel
        w_bytes = 2.0 * d * f + (d + f) * 4
    elif cfg.weights == "int4_g128":   # half a byte a weight + a bf16 scale per channel and 128 columns
        w_bytes = 1.0 * d * f + 2.0 * (d * f / 128) * 2
    else:
        w_bytes = 4.0 * d * f
    quant = cfg.weights != "bf16"
    x_bytes = (R * 2 * d + (T * 2 * d if cfg.has_shared else 0)) if quant else T * 2 * d
    nbytes = ((hit + (1 if cfg.has_shared else 0)) * w_bytes + x_bytes + rows_all * 4 * f
              + R * 2 * d + (T * 2 * d if cfg.has_shared else 0))
    return flops, nbytes


def time_forward(cfg, dev, pg, seed: int, steps: int, warmup: int):
    """Warm-up, then `steps` timed forwards with per-stage CUDA-event marks on
    the launching stream, barrier + synchronize on both sides and nvidia-smi
    clock samples during the timed region. Returns the inputs, the layer and
    the measurements."""
    import torch
    from top_routing_expert_then_b300 import lib
    from top_routing_expert_then_b300.inputs import make_inputs

    inp = make_inputs(cfg, seed, device=dev)
    layer = lib.MoELayer.from_inputs(inp)
    ro = layer.route_outputs()
    y = torch.empty_like(inp.x)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        layer.forward(inp.x, inp.sel_bias, y=y, route_out=ro)
    torch.cuda.synchronize()
    if lib.device_error() != 0:
        raise RuntimeError(f"{cfg.name}: device error during warm-up")
    R = int(ro.expert_offsets[-1].item())
    hit = int((ro.kept > 0).sum().item())

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
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
    for i in range(steps):
        layer.forward_marked(inp.x, ev[i], inp.sel_bias, y=y, route_out=ro)
    stop.record(stream)
    torch.cuda.synchronize()
    launches = lib.launch_count() - launches0
    if pg:
        pg.barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(pg, start.elapsed_time(stop), dev)
    if lib.device_error() != 0:
        raise RuntimeError(f"{cfg.name}: device error during the timed region")
    stage_ms = [sum(e[j].elapsed_time(e[j + 1]) for e in ev) / steps for j in range(5)]
    return {"inp": inp, "layer": layer, "R": R, "hit": hit, "elapsed_ms": elapsed_ms, "stage_ms": stage_ms,
            "launches": launches, "clocks": clk, "stream": stream}


STAGES = ["route_aux", "dispatch", "ffn_gemm1", "ffn_gemm2", "combine"]


def gemm_roofline(cfg, m, P, peak_kind, peak_t):
    """Roofline of the grouped expert GEMM (the dominant kernel) for one timed
    workload: its launches' time per step from the stage marks, algorithmic
    FLOPs and bytes per step, the binding roof chosen by FLOPs per byte
    against the machine balance at the chosen bf16 peak."""
    flops, nbytes = ffn_work(cfg, m["R"], m["hit"])
    gemm_ms = m["stage_ms"][2] + m["stage_ms"][3]
    tflops = flops / (gemm_ms * 1e-3) / 1e12
    gbs = nbytes / (gemm_ms * 1e-3) / 1e9
    tensor_bound = cfg.weights == "bf16" and flops / nbytes > peak_t * 1e12 / (P["hbm_gbs"] * 1e9)
    kernel = {"fp8_e4m3": "grouped_gemm_quant_kernel<FP8> (expert Linears, E4M3 codes widened into tensor "
                          "memory, channel-major tcgen05)",
              "int4_g128": "grouped_gemm_quant_kernel<INT4> (expert Linears, 4-bit codes and group scales "
                           "widened into tensor memory, channel-major tcgen05)"}.get(
        cfg.weights, "grouped_gemm_kernel (expert Linears, tcgen05)")
    return {"kernel": kernel,
            "bound": "tensor" if tensor_bound else "hbm",
            "achieved": tflops if tensor_bound else gbs,
            "peak": peak_t if tensor_bound else P["hbm_gbs"],
            "unit": "TFLOP/s" if tensor_bound else "GB/s",
            "frac": tflops / peak_t if tensor_bound else gbs / P["hbm_gbs"],
            "peak_kind": (f"{P['source']} {peak_kind} bf16" if tensor_bound else f"{P['source']} HBM copy"),
            "tflops": tflops, "gbs": gbs,
            "frac_of_burst_bf16": tflops / P["bf16_tflops"],
            "frac_of_sustained_bf16": tflops / P["bf16_tflops_sustained"],
            "frac_of_hbm": gbs / P["hbm_gbs"],
            "flops_per_step": flops, "bytes_per_step": nbytes, "ms_per_step": gemm_ms,
            "traffic": gemm_traffic(cfg.name),
            "traffic_unit": "DRAM bytes per step (all grouped-GEMM launches), ncu"}


def hbm_stages(cfg, m, P):
    """GB/s of the HBM-bound stages from their algorithmic bytes per step."""
    T, d, K, N, R = cfg.T, cfg.d_model, cfg.K, cfg.N, m["R"]
    route_bytes = T * d * 2 + N * d * 2 + T * K * 8 + N * 8
    # token placement: topk_idx read, slot_of / row_token written, bases read;
    # the x-row permute runs here only for FP8 experts (the bf16 path gathers
    # the rows inside the first expert GEMM)
    dispatch_bytes = T * K * 4 * 4 + ((T * d * 2 + R * d * 2) if cfg.weights != "bf16" else 0)
    combine_bytes = R * d * 2 + T * d * 2 + (T * d * 2 if cfg.has_shared else 0) + T * K * 8
    sm = m["stage_ms"]
    return {"route_aux": {"bytes": route_bytes, "gbs": route_bytes / (sm[0] * 1e-3) / 1e9},
            "dispatch": {"bytes": dispatch_bytes, "gbs": dispatch_bytes / (sm[1] * 1e-3) / 1e9},
            "combine": {"bytes": combine_bytes, "gbs": combine_bytes / (sm[4] * 1e-3) / 1e9},
            "peak_gbs": P["hbm_gbs"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="dsv3",
                    help="headline workload (default: the DeepSeek-V3-shaped layer, the largest that fits one GPU)")
    ap.add_argument("--extras", default="mixtral_prefill,mixtral_decode16,mixtral_decode16_fp8,mixtral_decode16_int4",
                    help="further workloads timed in the same run and reported under 'workloads' "
                         "(comma-separated names, or 'none')")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-sample", type=int, default=512, help="tokens in the CPU-oracle sample")
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
    from top_routing_expert_then_b300.inputs import make_dy

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    P = peaks()

    # ---- headline workload
    m = time_forward(cfg, dev, pg, args.seed + rank, args.steps, args.warmup)
    inp, layer, stream = m["inp"], m["layer"], m["stream"]
    T, d = cfg.T, cfg.d_model
    value = whole_job_rate(world, T, args.steps, m["elapsed_ms"])
    peak_kind, peak_t = choose_peak(P, m["clocks"], m["elapsed_ms"])
    roof = gemm_roofline(cfg, m, P, peak_kind, peak_t)

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
    del xd, yd

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
        del bws, dy
        if lib.device_error() != 0:
            raise RuntimeError("device error during the backward")

    inp_cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_cpu = inp.to("cpu")
    del layer, inp, m["layer"], m["inp"]
    torch.cuda.empty_cache()

    # ---- further workloads: the prefill tensor-core target and the decode
    # weight-streaming targets, each timed like the headline
    workloads = {}
    extras = [] if args.extras.strip().lower() == "none" else [w for w in args.extras.split(",") if w]
    for name in extras:
        if name == cfg.name:
            continue
        xc = CONFIGS[name]
        mx = time_forward(xc, dev, pg, args.seed + rank, args.steps, args.warmup)
        pk, pt = choose_peak(P, mx["clocks"], mx["elapsed_ms"])
        workloads[name] = {
            "value": whole_job_rate(world, xc.T, args.steps, mx["elapsed_ms"]), "unit": UNIT,
            "ms_per_step": mx["elapsed_ms"] / args.steps,
            "roofline": gemm_roofline(xc, mx, P, pk, pt),
            "stages_us": {n: round(1e3 * v, 2) for n, v in zip(STAGES, mx["stage_ms"])},
            "hbm_stages": hbm_stages(xc, mx, P),
            "kept_rows": mx["R"], "gpu_launches": mx["launches"], "clocks": mx["clocks"]}
        del mx
        torch.cuda.empty_cache()

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0

    cpu = None
    if inp_cpu is not None:
        import oracle
        oracle.build()
        dt, n = oracle_sample(cfg, inp_cpu, min(args.cpu_sample, cfg.T), seed=7)
        cpu = {"value": n / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": sample_desc(cfg, n), "seconds": round(dt, 2)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": m["elapsed_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg, {"kept_rows": m["R"], "parallelism": f"replicas{world}"}),
        "roofline": roof,
        "stages_us": {n: round(1e3 * v, 2) for n, v in zip(STAGES, m["stage_ms"])},
        "hbm_stages": hbm_stages(cfg, m, P),
        "cpu_baseline": cpu,
        "train_step": train,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * d * 2,
                "api": "moe_forward_hostio_batches (pinned host in/out every step, copies overlapped)",
                "steps": args.e2e_steps},
        "gpu_launches": m["launches"],
        "clocks": m["clocks"],
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
