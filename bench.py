"""Prefill throughput of the GB300 library on the Qwen2-0.5B-shaped workload.

One step = one whole prefill forward (every layer, every prompt token, the
last-row tail and lm_head) over a 512-token synthetic prompt at positions
0..511 into n_ctx-4096 KV regions, through the C ABI.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (test infrastructure, plain C++) on the
box's host cores on the same workload.  Multi-GPU runs are independent
replicas (one prompt and one model per GPU, no collective).
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
sys.path.insert(0, ROOT)

import numpy as np

import synth

WORKLOAD = "qwen2-0.5b-512"
METRIC = "prefill tokens/sec on 1 GB300"
UNIT = "tokens/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def gemm_flops(cfg, nt):
    """Algorithmic FLOPs per launch of each GEMM class (2 per MAC)."""
    H, q = cfg.n_embd, cfg.n_head * cfg.head_dim
    kv = cfg.n_head_kv * cfg.head_dim
    F = cfg.n_ff
    return {"gemm_qkv": 2.0 * nt * H * (q + 2 * kv), "gemm_o": 2.0 * nt * q * H,
            "gemm_gate_up_swiglu": 2.0 * nt * H * 2 * F, "gemm_down": 2.0 * nt * F * H}


def forward_macs(cfg, nt, p0=0, n_out=1):
    """Matmul, lm_head and causal-attention MACs of one forward whose last
    layer carries the n_out tail rows past its K/V projections."""
    H, q = cfg.n_embd, cfg.n_head * cfg.head_dim
    kv = cfg.n_head_kv * cfg.head_dim
    F, L, V = cfg.n_ff, cfg.n_layer, cfg.n_vocab
    per_tok = H * (q + 2 * kv) + q * H + 3 * H * F
    mm = (L - 1) * nt * per_tok + nt * H * (q + 2 * kv) + n_out * (q * H + 3 * H * F)
    keys = sum(p0 + t + 1 for t in range(nt))
    tail_keys = sum(p0 + t + 1 for t in range(nt - n_out, nt))
    attn = (L - 1) * keys * 2 * q + tail_keys * 2 * q
    return mm, n_out * H * V, attn


_PROFILE_OF = {"gemm_gate_up_swiglu": "gemm_gate_up", "attention": "attention",
               "rmsnorm_quant": "row_quant"}


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) of `kernel` on `workload` from the
    committed ncu summary under profiles/, or None when there is none."""
    name = _PROFILE_OF.get(kernel)
    if not name:
        return None
    path = os.path.join(ROOT, "profiles", f"{name}_{workload}.md")
    try:
        with open(path) as f:
            for line in f:
                if line.startswith("traffic_bytes_per_launch:"):
                    return int(line.split(":")[1])
    except OSError:
        pass
    return None


def oracle_model(cfg):
    import oracle
    m = oracle.Model(cfg)
    for spec in synth.tensor_specs(cfg):
        m.set_f32(spec.name, synth.tensor_data(spec))
    return m


def cpu_baseline(w, reps: int = 2):
    """The oracle, as it stands, on the host cores: full prefills of the
    bench workload (bounded: `reps` forwards)."""
    import oracle
    oracle.build()
    cfg = w.model
    m = oracle_model(cfg)
    ids, pos = w.ids(), w.positions()
    times = []
    for _ in range(reps):
        kv = m.kv(w.n_ctx)
        t = time.perf_counter()
        rc, _, _ = m.prefill(kv, ids, pos)
        times.append(time.perf_counter() - t)
        assert rc == 0
    dt = min(times)
    return {"value": w.n_tokens / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} full {w.n_tokens}-token prefills of {w.name} (best taken)",
            "seconds_per_forward": dt}


def reference_arm(args, w, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = w.model
    m = oracle_model(cfg)
    ids, pos = w.ids(), w.positions()
    for _ in range(args.warmup):
        m.prefill(m.kv(w.n_ctx), ids, pos)
    times = []
    for _ in range(args.steps):
        kv = m.kv(w.n_ctx)
        t = time.perf_counter()
        rc, _, _ = m.prefill(kv, ids, pos)
        times.append(time.perf_counter() - t)
        assert rc == 0
    total = sum(times)
    value = w.n_tokens * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64",
            "data": "synthetic", "config": {"workload": w.name, "n_tokens": w.n_tokens,
                                            "n_ctx": w.n_ctx, "positions": "0..511"},
            "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                             "cores": os.cpu_count(),
                             "sample": f"{args.steps} full prefills of {w.name}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def ours(args, w, rank, world, dist):
    import torch
    import quantized_transformer_prefill_gb300 as qp

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    cfg = w.model
    model = qp.Model(qp.hparams_of(cfg))
    for spec in synth.tensor_specs(cfg):
        model.set_tensor(spec.name, synth.tensor_data(spec), spec.ne0, spec.ne1, qp.MINFER_F32)
    model.finalize()
    kv = model.kv(w.n_ctx)
    if w.prefill_tokens:  # the cached turn an append attends over (untimed)
        model.prefill(kv, w.prefill_ids(), np.arange(w.prefill_tokens, dtype=np.int32))
    ids, pos = w.ids(), w.positions()
    nt = w.n_tokens
    d_ids = torch.from_numpy(ids).cuda()
    d_pos = torch.from_numpy(pos).cuda()
    n_out = w.n_out
    d_logits = torch.empty((n_out, cfg.n_vocab), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream

    def step():
        rc = model.prefill_device_n(kv, d_ids.data_ptr(), d_pos.data_ptr(), nt, n_out,
                                    d_logits.data_ptr(), sp)
        if rc != 0:
            raise RuntimeError(f"prefill_device rc={rc}")

    for _ in range(max(3, args.warmup)):
        step()
    qp.check(model.sync_status(sp), "warmup")

    def barrier():
        if dist is not None:
            dist.barrier()

    # ---- timed region: K graph replays, device-resident inputs
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                step()
            e1.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.25)
    barrier()
    qp.check(model.sync_status(sp), "timed region")
    ms = e0.elapsed_time(e1)
    if dist is not None:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_per_step = ms / args.steps
    value = world * nt * args.steps / (ms / 1e3)

    # ---- per-kernel times: same replays with CUDA events around every launch
    model.profile_enable(True)
    for _ in range(2):
        step()
    qp.check(model.sync_status(sp), "profile warmup")
    model.profile_enable(True)  # reset the totals
    torch.cuda.synchronize()
    for _ in range(args.steps):
        step()
    qp.check(model.sync_status(sp), "profiled region")
    prof = model.profile_read()  # the last replay's launches and times
    model.profile_enable(False)
    launches_per_step = sum(n for n, _ in prof.values())

    # ---- end-to-end through the host-buffer call (H2D inputs, D2H logits inside)
    h_ids = torch.from_numpy(ids).pin_memory().numpy()
    h_pos = torch.from_numpy(pos).pin_memory().numpy()
    h_logits = torch.empty((n_out, cfg.n_vocab), dtype=torch.float32).pin_memory().numpy()
    for _ in range(3):
        model.prefill_n(kv, h_ids, h_pos, n_out, h_logits)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        model.prefill_n(kv, h_ids, h_pos, n_out, h_logits)
    e2e_s = time.perf_counter() - t0
    if dist is not None:
        t = torch.tensor([e2e_s], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_value = world * nt * args.steps / e2e_s

    if rank != 0:
        return
    hbm, bf16, peak_src = _peaks()
    flops = gemm_flops(cfg, nt)
    # dominant kernel by device time
    dom = max(prof.items(), key=lambda kv_: kv_[1][1])[0]
    gemm_stats = {}
    for k, f in flops.items():
        n, tot = prof.get(k, (0, 0.0))
        if n:
            avg_ms = tot / n
            gemm_stats[k] = {"avg_us": 1e3 * avg_ms, "tflops": f / (avg_ms / 1e3) / 1e12,
                             "frac_of_bf16_peak": f / (avg_ms / 1e3) / 1e12 / bf16}
    if dom in flops:
        n, tot = prof[dom]
        avg_ms = tot / n
        achieved = flops[dom] / (avg_ms / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": bf16,
                "unit": "TFLOP/s", "frac": achieved / bf16,
                "traffic": profiled_traffic(dom, w.name),
                "peak_source": f"{peak_src} bf16 burst (fp16 operands run at the bf16 rate)",
                "per_launch_flops": flops[dom], "avg_launch_us": 1e3 * avg_ms}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": None, "peak": hbm, "unit": "GB/s",
                "frac": None, "traffic": profiled_traffic(dom, w.name)}
    mm, lm, attn = forward_macs(cfg, nt, w.p0, n_out)
    # forward roofline: GEMM + attention flops at the tensor peak, lm_head and
    # the hidden-state traffic at HBM bandwidth
    # lm_head: its weights read once (Q8_0 bytes) or its flops, whichever is longer
    lm_bytes = cfg.n_vocab * cfg.n_embd * 34 / 32
    t_star = (2 * mm / (bf16 * 1e12) + 2 * attn / (bf16 * 1e12)
              + max(lm_bytes / (hbm * 1e9), 2 * lm / (bf16 * 1e12)))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "q8_0 (fp16-held int8 codes, f32 acc)",
        "data": "synthetic (seeded N(0,0.02) weights, uniform ids)",
        "config": {"workload": w.name, "n_tokens": nt, "n_out": n_out,
                   "positions": f"{w.p0}..{w.p0 + nt - 1}", "n_ctx": w.n_ctx,
                   "layers": cfg.n_layer, "hidden": cfg.n_embd, "vocab": cfg.n_vocab,
                   "l2": "weights (>= 0.9 GB) larger than L2 stream through it every step",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "gemm": gemm_stats,
        "forward_roofline": {"t_star_ms": 1e3 * t_star, "frac": 1e3 * t_star / ms_per_step,
                             "matmul_macs": mm, "attn_macs": attn, "lm_head_macs": lm},
        "kernels_last_step": {k: {"launches": n, "ms": t} for k, (n, t) in prof.items() if n},
        "gpu_launches": int(launches_per_step * args.steps),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 2 * nt * 4,
                "d2h_bytes_per_step": n_out * cfg.n_vocab * 4},
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and world >= 1 and rank == 0:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", 1))
    rank = int(os.environ.get("RANK", 0))
    dist = None
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist_mod
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    if args.impl == "reference":
        reference_arm(args, w, rank, world)
    else:
        ours(args, w, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
