"""Decode-step benchmark: tok/s and fraction of the HBM Speed-of-Light.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload a3b_8k]
                    [--impl ours|reference] [--layers L] [--no-cpu-baseline]

One step = one decode step of the whole batch through the persistent kernel
(all layers, attention + MoE + LM head).  Prints one JSON line (rank 0).

value     : B * K / device time of K steps (CUDA events on the launching
            stream, inputs resident in HBM; every step reads > L2 bytes).
e2e       : the same metric through the C ABI with host buffers: each step
            uploads its tokens / page tables / lengths from host memory and
            reads the logits back, the next token chosen on the host.
roofline  : algorithmic bytes per step (dense weights, distinct routed
            experts, attended K/V, LM head) / average kernel duration,
            against the measured HBM copy bandwidth.
cpu_baseline : the CPU oracle timed on a bounded sample of the same step.
Multi-GPU: replicas only (independent sequences per GPU, no collective in the
data path); value is the sum over ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode tok/s at 1 GB300 (batch 1 & 16) and % of HBM Speed-of-Light"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_traffic(workload: str):
    """dram bytes per step from a committed ncu summary, if one matches this build."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        ent = t.get(workload)
        if ent and ent.get("kernel_sha") == kernel_sha():
            return float(ent["bytes_per_step"])
    except Exception:
        pass
    return None


def kernel_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "persistent_moe_decode_gb300", "csrc")
    for fn in sorted(os.listdir(cs)):
        if fn.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(cs, fn), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling during the timed region (SM clock, throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.dev = dev_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def step_bytes(dims, routing_idx, keys_per_seq):
    from persistent_moe_decode_gb300.configs import algorithmic_bytes
    distinct = [len(set(routing_idx[l].reshape(-1).tolist())) for l in range(dims.n_layers)]
    return algorithmic_bytes(dims, distinct, keys_per_seq)


class CpuSample:
    """The CPU oracle on a bounded sample of one step: layers [0, n) at the full
    shapes and 1/lm_frac of the LM-head rows, extrapolated to a whole token."""

    def __init__(self, model, k_pool, v_pool, batch, n_layers_sample: int, lm_frac: int = 8):
        import dataclasses

        import oracle
        from persistent_moe_decode_gb300.synth import SynthModel, bf16_bits
        d = model.dims
        n = n_layers_sample
        w = {}
        for name in SynthModel.NAMES:
            t = getattr(model, name)
            t = t if name in ("embed", "lm_head", "final_norm") else t[:n]
            w[name] = bf16_bits(t.cpu().contiguous())
        kp = bf16_bits(k_pool[:n].cpu().contiguous()).copy()
        vp = bf16_bits(v_pool[:n].cpu().contiguous()).copy()
        self.oracle = oracle
        self.orc = oracle.Oracle({**dataclasses.asdict(d), "n_layers": n}, w, kp, vp)
        self.d, self.n, self.lm_frac, self.batch = d, n, lm_frac, batch
        B = batch.wl.batch
        self.h0 = oracle.bf16_to_f64(w["embed"][batch.tokens[:B]])
        self.lm = w["lm_head"][:d.vocab // lm_frac]

    def time_token(self) -> float:
        """Seconds the oracle needs per decode step of the whole batch."""
        B = self.batch.wl.batch
        t0 = time.perf_counter()
        self.orc.run_layers(0, self.n, self.h0, self.batch.seq_lens[:B], self.batch.page_tables[:B])
        t1 = time.perf_counter()
        self.oracle.matvec(self.lm, self.h0)
        t2 = time.perf_counter()
        return (t1 - t0) * (self.d.n_layers / self.n) + (t2 - t1) * self.lm_frac

    def describe(self, reps: int) -> str:
        return (f"layers 0..{self.n - 1} of one decode step at the full shapes (context "
                f"{int(self.batch.seq_lens[0])}, batch {self.batch.wl.batch}) plus 1/{self.lm_frac} of "
                f"the LM-head rows, {reps} repetitions, extrapolated to {self.d.n_layers} layers and "
                f"the whole LM head")

    def measure(self, min_seconds: float) -> dict:
        B = self.batch.wl.batch
        ts, t_start = [], time.perf_counter()
        while not ts or time.perf_counter() - t_start < min_seconds:
            ts.append(self.time_token())
        return {"value": B / float(np.median(ts)), "unit": "tok/s", "cores": self.oracle.get_threads(),
                "kind": "oracle", "sample": self.describe(len(ts)),
                "seconds": round(time.perf_counter() - t_start, 2)}


def run_reference(args, wl):
    """Reference arm: the CPU oracle as it stands, one bounded sample per step."""
    from persistent_moe_decode_gb300.synth import DecodeBatch, make_kv_pools, make_model
    d = wl.dims
    n = min(args.ref_layers, d.n_layers)
    small = type(d)(**{**d.__dict__, "n_layers": n})
    model = make_model(small, wl.seed, "cpu")
    batch = DecodeBatch(wl)
    kp, vp = make_kv_pools(small, batch.num_pages, wl.kv_std, wl.seed, "cpu")
    model.dims = d
    cs = CpuSample(model, kp, vp, batch, n)
    for _ in range(args.warmup):
        cs.time_token()
    t_all = time.perf_counter()
    secs = [cs.time_token() for _ in range(args.steps)]
    wall = time.perf_counter() - t_all
    v = wl.batch * args.steps / float(np.sum(secs))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * float(np.mean(secs)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "context": int(batch.seq_lens[0]),
                       "layers": d.n_layers, "l2": "inputs larger than L2"},
            "cpu_baseline": {"value": v, "unit": "tok/s", "kind": "oracle",
                             "cores": cs.oracle.get_threads(), "sample": cs.describe(args.steps)},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 2)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="a3b_8k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="profiling: run only the first L layers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-layers", type=int, default=2)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    assert args.warmup >= 3 or args.layers, "at least 3 warm-up steps"

    from persistent_moe_decode_gb300.configs import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.layers:
        wl = wl.with_(dims=type(wl.dims)(**{**wl.dims.__dict__, "n_layers": args.layers}))

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl)
        return

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from persistent_moe_decode_gb300 import build
    build.build()
    from persistent_moe_decode_gb300 import mk
    from persistent_moe_decode_gb300.runner import StepRunner

    dims = wl.dims
    run = StepRunner(wl.with_(seed=wl.seed + rank), device=f"cuda:{local}")
    stream = torch.cuda.current_stream()
    B = wl.batch
    rng = np.random.default_rng(1234 + rank)
    total = args.warmup + args.steps
    tok_seq = rng.integers(0, dims.vocab, size=(total, B)).astype(np.int32)

    # ---- device-timed loop: inputs resident, tokens drawn ahead of time
    def one_step(i):
        run.schedule(stream)
        run.launch(stream)

    for i in range(args.warmup):
        one_step(i)
        run.advance(tok_seq[i])
    torch.cuda.synchronize()
    run.check_status()
    keys0 = (run.batch.seq_lens + 1).copy()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    keys = []
    for i in range(args.steps):
        run.schedule(stream)
        ev[i][0].record(stream)
        run.launch(stream)
        ev[i][1].record(stream)
        keys.append((run.batch.seq_lens + 1).copy())
        run.advance(tok_seq[args.warmup + i])
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    run.check_status()
    elapsed_ms = t0.elapsed_time(t1)
    kern_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    if dist:
        tt = torch.tensor([elapsed_ms], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        elapsed_ms = float(tt.item())
    tok_s = B * args.steps * world / (elapsed_ms / 1000.0)

    # bytes: routing of the last step (B = 1: always top_k distinct experts per layer)
    idx, _ = run.dec.routing()
    bytes_step = step_bytes(dims, idx, keys[-1])
    peak, peak_kind = load_peaks()
    achieved = bytes_step / (kern_ms / 1000.0) / 1e9

    # ---- end-to-end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        host_logits = torch.empty(B, dims.vocab, dtype=torch.float32, pin_memory=True)
        for i in range(3):
            run.step(stream)
            host_logits.copy_(run.logits, non_blocking=True)
            torch.cuda.synchronize()
            run.advance(host_logits.numpy().argmax(1).astype(np.int32))
        torch.cuda.synchronize()
        h2d = d2h = 0
        ts = time.perf_counter()
        for i in range(args.steps):
            run.step(stream)
            h2d += mk.mk_step_upload_bytes(run.dec.h, B)
            host_logits.copy_(run.logits, non_blocking=True)
            torch.cuda.synchronize()
            d2h += host_logits.numel() * 4
            run.advance(host_logits.numpy().argmax(1).astype(np.int32))
        te = time.perf_counter()
        run.check_status()
        e2e = {"value": B * args.steps * world / (te - ts), "unit": "tok/s",
               "h2d_bytes_per_step": int(h2d // args.steps), "d2h_bytes_per_step": int(d2h // args.steps)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = CpuSample(run.model, run.k_pool, run.v_pool, run.batch,
                            min(4, dims.n_layers)).measure(args.cpu_seconds)
        except Exception as e:  # report, do not hide
            cpu = {"value": None, "error": repr(e)}

    traffic = load_traffic(wl.name if not args.layers else f"{wl.name}:L{args.layers}")
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name + (f" (first {args.layers} layers)" if args.layers else ""),
                   "batch": B, "context": int(keys0[0] - 1) if B == 1 else "ragged",
                   "layers": dims.n_layers,
                   "l2": f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB read per step)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "sol_frac": {"of_measured_hbm": achieved / peak, "of_nominal_8tbs": achieved / 8000.0},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic,
                     "algorithmic_bytes_per_step": bytes_step, "kernel_ms": kern_ms,
                     "kernel": "mk_step_kernel (persistent, one block per SM)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    run.close()
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
