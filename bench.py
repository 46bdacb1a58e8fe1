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
    """dram bytes per step from a committed ncu summary measured with the current kernel code."""
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


def kernel_code(text: str) -> str:
    """A CUDA / C++ source without its comments, trailing blanks and blank
    lines: what the compiler turns into code."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_sha() -> str:
    """Key of the traffic record: a hash of the kernel sources' code (comments
    excluded, so an edit to the documentation keeps the record)."""
    import hashlib
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "persistent_moe_decode_gb300", "csrc")
    for fn in sorted(os.listdir(cs)):
        if fn.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(cs, fn), encoding="utf-8") as f:
                h.update(fn.encode() + b"\0" + kernel_code(f.read()).encode() + b"\0")
    return h.hexdigest()[:16]


def slowest(seconds: float, dist=None) -> float:
    """The slowest rank's time, on every rank (one rank: its own time).  The
    whole-job rate divides all ranks' units by it."""
    if dist is None:
        return seconds
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world: int, seconds: float) -> float:
    """Units all ranks processed per second of the slowest rank's time."""
    return units_per_rank * world / seconds


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


def step_bytes(dims, routing_idx, keys_per_seq, expert_format="bf16"):
    from persistent_moe_decode_gb300.configs import algorithmic_bytes
    distinct = [len(set(routing_idx[l].reshape(-1).tolist())) for l in range(dims.n_layers)]
    return algorithmic_bytes(dims, distinct, keys_per_seq, expert_format)


class CpuSample:
    """The CPU oracle on a bounded sample of one step: layers [0, n) at the full
    shapes and 1/lm_frac of the LM-head rows, extrapolated to a whole step.

    ``state`` = (tokens, seq_lens, page_tables) of a step that was scheduled
    (every sequence owns the page its new token lands in)."""

    def __init__(self, model, k_pool, v_pool, state, wl, n_layers_sample: int, lm_frac: int = 8):
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
        fp8 = None if model.fp8 is None else \
            {name: t[:n].cpu().contiguous().numpy() for name, t in model.fp8.items()}
        self.oracle = oracle
        self.orc = oracle.Oracle({**dataclasses.asdict(d), "n_layers": n}, w, kp, vp, fp8=fp8)
        self.d, self.n, self.lm_frac, self.wl = d, n, lm_frac, wl
        tokens, lens, pt = state
        self.B = len(tokens)
        self.lens = np.ascontiguousarray(lens, dtype=np.int32).copy()
        self.pt = np.ascontiguousarray(pt, dtype=np.int32).copy()
        self.h0 = oracle.bf16_to_f64(w["embed"][np.asarray(tokens)])
        self.lm = w["lm_head"][:d.vocab // lm_frac]

    def time_token(self) -> float:
        """Seconds the oracle needs per decode step of the whole batch."""
        t0 = time.perf_counter()
        self.orc.run_layers(0, self.n, self.h0, self.lens, self.pt)
        t1 = time.perf_counter()
        self.oracle.matvec(self.lm, self.h0)
        t2 = time.perf_counter()
        return (t1 - t0) * (self.d.n_layers / self.n) + (t2 - t1) * self.lm_frac

    def describe(self, reps: int) -> str:
        ctx = f"context {int(self.lens[0])}" if self.B == 1 else \
            f"contexts {int(self.lens.min())}..{int(self.lens.max())}"
        return (f"layers 0..{self.n - 1} of one decode step of {self.wl.name} at the full shapes "
                f"({ctx}, batch {self.B}) plus 1/{self.lm_frac} of the LM-head rows, {reps} "
                f"repetitions, extrapolated to {self.d.n_layers} layers and the whole LM head")

    def measure(self, min_seconds: float) -> dict:
        ts, t_start = [], time.perf_counter()
        while not ts or time.perf_counter() - t_start < min_seconds:
            ts.append(self.time_token())
        return {"value": self.B / float(np.median(ts)), "unit": "tok/s", "cores": self.oracle.get_threads(),
                "kind": "oracle", "sample": self.describe(len(ts)),
                "seconds": round(time.perf_counter() - t_start, 2)}


def snapshot(batch):
    """(tokens, seq_lens, page_tables) of the batch's next step, pages present."""
    batch.prepare_step()
    B = batch.wl.batch
    return batch.tokens[:B].copy(), batch.seq_lens[:B].copy(), batch.page_tables[:B].copy()


def context_of(lens) -> int | str:
    return int(lens[0]) if len(lens) == 1 else "ragged"


def run_reference(args, wl):
    """Reference arm: the CPU oracle as it stands, one bounded sample per step.

    The batch goes through the same warm-up steps as the GPU arm (bookkeeping
    only: tokens, lengths, pages, churn), so the timed steps start at the same
    context."""
    from persistent_moe_decode_gb300.synth import DecodeBatch, make_kv_pools, make_model
    d = wl.dims
    n = min(args.ref_layers, d.n_layers)
    small = type(d)(**{**d.__dict__, "n_layers": n})
    model = make_model(small, wl.seed, "cpu", wl.expert_format)
    batch = DecodeBatch(wl)
    kp, vp = make_kv_pools(small, batch.num_pages, wl.kv_std, wl.seed, "cpu")
    model.dims = d
    rng = np.random.default_rng(1234)
    B = wl.batch

    def advance():
        batch.advance(rng.integers(0, d.vocab, size=B).astype(np.int32))
        if wl.churn:
            batch.churn()

    for _ in range(args.warmup):
        advance()
    state = snapshot(batch)
    cs = CpuSample(model, kp, vp, state, wl, n)
    cs.time_token()                       # untimed: first touch of the host arrays
    t_all = time.perf_counter()
    secs = [cs.time_token() for _ in range(args.steps)]
    wall = time.perf_counter() - t_all
    v = B * args.steps / float(np.sum(secs))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * float(np.mean(secs)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "batch": B, "context": context_of(state[1]),
                       "layers": d.n_layers, "l2": "inputs larger than L2"},
            "cpu_baseline": {"value": v, "unit": "tok/s", "kind": "oracle",
                             "cores": cs.oracle.get_threads(), "sample": cs.describe(args.steps)},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 2)}
    print(json.dumps(line), flush=True)


def device_timed(run, wl, args, stream, tok_seq, dist=None, clocks=None):
    """Warm-up, then K steps timed with CUDA events on the launching stream.

    Returns (elapsed ms over the K steps, mean kernel ms, the state of the first
    timed step, the keys attended per sequence in the last timed step, the
    clocks sampled during the timed steps).  The
    churn bookkeeping between steps stays in the loop; the joining sequences'
    pages keep the random K/V they hold (no random-number kernels in the loop)."""
    import torch
    for i in range(args.warmup):
        run.schedule(stream)
        run.launch(stream)
        run.advance(tok_seq[i], refill=False)
    torch.cuda.synchronize()
    run.check_status()
    state = snapshot(run.batch)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if clocks:
        clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    keys = None
    for i in range(args.steps):
        run.schedule(stream)
        ev[i][0].record(stream)
        run.launch(stream)
        ev[i][1].record(stream)
        keys = (run.batch.seq_lens + 1).copy()
        run.advance(tok_seq[args.warmup + i], refill=False)
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    run.check_status()
    elapsed_ms = t0.elapsed_time(t1)
    kern_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    return elapsed_ms, kern_ms, state, keys, clk


def roofline_of(run, wl, kern_ms, keys, traffic_key):
    idx, _ = run.dec.routing()
    bytes_step = step_bytes(wl.dims, idx, keys, wl.expert_format)
    peak, peak_kind = load_peaks()
    achieved = bytes_step / (kern_ms / 1000.0) / 1e9
    return bytes_step, {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                        "frac": achieved / peak, "peak_kind": peak_kind,
                        "traffic": load_traffic(traffic_key),
                        "algorithmic_bytes_per_step": bytes_step, "kernel_ms": kern_ms,
                        "kernel": "mk_step_kernel (persistent, one block per SM)"}


def e2e_timed(run, wl, args, stream, world, dist=None):
    """The same metric end to end through the C ABI: per step the host arrays
    go up (schedule), the step runs, the logits come back to pinned host
    memory and the host picks the next tokens (greedy)."""
    import torch
    from persistent_moe_decode_gb300 import mk
    B = wl.batch
    host_logits = torch.empty(B, wl.dims.vocab, dtype=torch.float32, pin_memory=True)
    for i in range(3):
        run.step(stream)
        host_logits.copy_(run.logits, non_blocking=True)
        torch.cuda.synchronize()
        run.advance(host_logits.numpy().argmax(1).astype(np.int32), refill=False)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    h2d = d2h = 0
    ts = time.perf_counter()
    for i in range(args.steps):
        run.step(stream)
        h2d += mk.mk_step_upload_bytes(run.dec.h, B)
        host_logits.copy_(run.logits, non_blocking=True)
        torch.cuda.synchronize()
        d2h += host_logits.numel() * 4
        run.advance(host_logits.numpy().argmax(1).astype(np.int32), refill=False)
    te = time.perf_counter()
    run.check_status()
    return {"value": job_rate(B * args.steps, world, slowest(te - ts, dist)), "unit": "tok/s",
            "h2d_bytes_per_step": int(h2d // args.steps), "d2h_bytes_per_step": int(d2h // args.steps)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="a3b_8k",
                    help="a3b_8k (default), a3b_b16, a3b_256k, mid_8k, tiny")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="profiling: run only the first L layers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-b16", action="store_true",
                    help="a3b_8k: skip the batch-16 line measured on the same model")
    ap.add_argument("--waves", default=None, choices=["default", "attn_first", "interleaved"],
                    help="schedule ablation: every SM runs every phase in this wave order (no roles)")
    ap.add_argument("--attn-sms", type=int, default=0,
                    help="schedule ablation: SMs on the attention branch (0 = chosen per step)")
    ap.add_argument("--kv-split", type=int, default=0,
                    help="schedule ablation: split-KV chunk in tokens (0 = one run per attention SM)")
    ap.add_argument("--moe-depth", type=int, default=0,
                    help="schedule ablation: stages an expert-branch SM keeps in flight (0 = per step)")
    ap.add_argument("--claim-rows", type=int, default=0,
                    help="several tokens: rows per expert tile claimed from per-layer counters "
                         "(0 = the default, 128; -1 = static equal shares)")
    ap.add_argument("--ref-layers", type=int, default=2)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    assert args.warmup >= 3 or args.layers, "at least 3 warm-up steps"

    from persistent_moe_decode_gb300.configs import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.layers:
        wl = wl.with_(dims=type(wl.dims)(**{**wl.dims.__dict__, "n_layers": args.layers}))
    # the page pool covers every step this run takes: warm-up, the device-timed
    # steps, and the end-to-end leg (3 warm-up steps and K timed ones)
    wl = wl.with_(steps=max(wl.steps, args.warmup + 2 * args.steps + 3))

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
    from persistent_moe_decode_gb300.runner import StepRunner

    dims = wl.dims
    sched = {}
    if args.waves:
        from persistent_moe_decode_gb300 import mk
        sched["n_attn_claimers"] = 1 << 20
        sched["wave_order"] = {"default": mk.MK_WAVES_DEFAULT, "attn_first": mk.MK_WAVES_ATTN_FIRST,
                               "interleaved": mk.MK_WAVES_INTERLEAVED}[args.waves]
    elif args.attn_sms:
        sched["n_attn_claimers"] = args.attn_sms
    if args.kv_split:
        sched["kv_split_tokens"] = args.kv_split
    if args.moe_depth:
        sched["moe_stage_depth"] = args.moe_depth
    if args.claim_rows:
        sched["moe_claim_rows"] = args.claim_rows
    run = StepRunner(wl.with_(seed=wl.seed + rank), device=f"cuda:{local}", **sched)
    stream = torch.cuda.current_stream()
    B = wl.batch
    rng = np.random.default_rng(1234 + rank)
    tok_seq = rng.integers(0, dims.vocab, size=(args.warmup + args.steps, B)).astype(np.int32)

    elapsed_ms, kern_ms, state, keys, clk = device_timed(run, wl, args, stream, tok_seq, dist,
                                                         ClockSampler(local))
    elapsed_ms = slowest(elapsed_ms, dist)
    tok_s = job_rate(B * args.steps, world, elapsed_ms / 1000.0)
    traffic_key = wl.name if not args.layers else f"{wl.name}:L{args.layers}"
    bytes_step, roof = roofline_of(run, wl, kern_ms, keys, traffic_key)

    e2e = None if args.no_e2e else e2e_timed(run, wl, args, stream, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = CpuSample(run.model, run.k_pool, run.v_pool, state, wl,
                            min(4 if B == 1 else 2, dims.n_layers)).measure(args.cpu_seconds)
        except Exception as e:  # report, do not hide
            cpu = {"value": None, "error": repr(e)}

    # the metric names batch 1 and batch 16: with the 30B/3.3B model at batch 1,
    # the batch-16 continuous-batching workload runs on the same weights
    b16 = None
    if wl.name == "a3b_8k" and not args.layers and not args.no_b16 and not sched:
        wl16 = WORKLOADS["a3b_b16"]
        run16 = StepRunner(wl16.with_(seed=wl16.seed + rank), device=f"cuda:{local}", model=run.model)
        tok16 = rng.integers(0, dims.vocab, size=(args.warmup + args.steps, 16)).astype(np.int32)
        a16 = argparse.Namespace(**{**vars(args), "steps": min(args.steps, 20)})
        el16, kern16, st16, keys16, clk16 = device_timed(run16, wl16, a16, stream, tok16, dist,
                                                         ClockSampler(local))
        bytes16, roof16 = roofline_of(run16, wl16, kern16, keys16, wl16.name)
        el16 = slowest(el16, dist)
        b16 = {"workload": wl16.name, "batch": 16, "steps": a16.steps,
               "value": job_rate(16 * a16.steps, world, el16 / 1000.0), "unit": "tok/s",
               "ms_per_step": el16 / a16.steps,
               "contexts": f"{int(st16[1].min())}..{int(st16[1].max())} at the first timed step",
               "roofline": roof16, "clocks": clk16}
        run16.close()

    line = {
        "metric": METRIC, "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.expert_format == "bf16" else "bf16 (routed experts e4m3 + fp32 row scales)",
        "data": "synthetic",
        "config": {"workload": wl.name + (f" (first {args.layers} layers)" if args.layers else ""),
                   "batch": B, "context": context_of(state[1]),
                   "context_note": "cached tokens at the first timed step",
                   "layers": dims.n_layers,
                   "l2": f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB read per step)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "schedule": ({"waves": args.waves} if args.waves else
                                {"attention_sms": args.attn_sms or "per step"})
                               | ({"kv_split_tokens": args.kv_split} if args.kv_split else {})
                               | ({"moe_stage_depth": args.moe_depth} if args.moe_depth else {})
                               | ({"moe_claim_rows": args.claim_rows} if args.claim_rows else {})},
        "sol_frac": {"of_measured_hbm": roof["frac"], "of_nominal_8tbs": roof["achieved"] / 8000.0},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if b16 is not None:
        line["batch16"] = b16
    if rank == 0:
        print(json.dumps(line), flush=True)
    run.close()
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
