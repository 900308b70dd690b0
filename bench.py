"""Benchmark: goinfer's turn-9 suffix prefill on one GB300 (or N replicas).

Workload (default): Qwen2.5-7B-shaped 28-layer stack, random int4 g32 weights,
4 slots of 16384 bf16 KV.  Slot 0 holds a conversation whose first 1668 tokens
match every timed prompt; slots 1-3 hold conversations that share only the
7-token chat-template start.  One step = kvr_slot_match(1922-token prompt)
-> slot 0, reused 1668 -> kvr_prefill_suffix(254 rows).  Each step's prompt
has a fresh 254-token tail, so every step is a complete turn-9 (match,
cut back, prefill) and no state is reset between steps.

value       = suffix rows/s over the timed steps (device time, inputs resident).
e2e         = the same through the public API with pinned host buffers: the
              step's hidden rows copied in, the output copied back.
roofline    = the projection kernels (the dominant class, each launch timed by
              its own event pair) against the measured burst bf16 tensor peak;
              attended-KV GB/s of the attention kernels is reported beside it,
              and the whole step's causal flops against the same peak.
verify      = the m <= 16 half of the metric in the same run: a speculative
              verify of m = 1 and m = 8 rows on the dense 9B-class shape over a
              4096-token slot, ms per call and the fraction of measured HBM
              bandwidth its algorithmic bytes reach.
cpu_baseline= the oracle (float64 numpy) on a bounded sample of the same
              workload: one layer, the 254 suffix rows, over a 1668-row prefix,
              extrapolated to the 28-layer stack.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvr|reference]
For N > 1, launch under torch.distributed.run: each rank runs an independent
replica (slots shard by conversation; no collective on the data path).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

P_CACHED, M_ROWS, PROMPT = 1668, 254, 1922
# DRAM bytes (read + write) of the four projection GEMMs of one layer of this workload, from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum, cold L2): 11.17 + 9.11 + 80.23 + 48.35 MB.
# Re-take the capture whenever gemm_int4_tc_kernel changes.
PROJ_TRAFFIC_PER_LAYER = 148.85e6


def peaks():
    try:
        with open(PEAKS_PATH) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def dist_setup(n_gpus):
    """One process per GPU under torch.distributed.run (RANK / WORLD_SIZE /
    LOCAL_RANK / MASTER_* from the environment): NCCL with a GPU, gloo without."""
    rank, world = 0, 1
    if n_gpus > 1 or "RANK" in os.environ:
        import torch.distributed as dist
        rank = int(os.environ.get("RANK", 0))
        world = int(os.environ.get("WORLD_SIZE", 1))
        local = int(os.environ.get("LOCAL_RANK", 0))
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float) -> float:
    """The slowest rank's time: every rank's clock brackets the same barrier-aligned region."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        on_gpu = dist.get_backend() == "nccl"
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return x


def whole_job_rate(world: int, rows_per_rank: int, steps: int, ms_max: float) -> float:
    """Rows/s of the whole job: every rank's rows over the slowest rank's time."""
    return world * rows_per_rank * steps / (ms_max / 1e3)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        out_dir = os.environ.get("KVR_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1])); mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

FORMAT_LABEL = {"int4": "int4-g32", "q4k": "K-quant 4-bit superblocks"}


def turn9_config(world, fmt="int4"):
    return {"workload": f"turn-9 suffix prefill: Qwen2.5-7B-shaped 28-layer {FORMAT_LABEL[fmt]} "
                        "stack, 1922-token prompt, 1668 cached, 254 suffix rows, 4 slots x 16384",
            "global_batch": M_ROWS * world, "seq_len": PROMPT, "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2: 3.67 GB of 4-bit weights streamed per step"}


def build_turn9(device, steps_total, layers=None, fmt="int4"):
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    shape = workloads.SHAPES["qwen7b" if fmt == "int4" else "qwen7b_q4k"]
    if layers:
        shape = dataclasses.replace(shape, n_layers=layers)
    seed = workloads.config_seed(2)
    tk = workloads.turn9_tokens(seed)
    t0 = time.time()
    lws = workloads.stack_weights(shape, seed, device=device)
    kv = Kvr(config_for_shape(shape, 4, 16384, 256), device=device)
    w = kv.weights(lws)
    for s in (1, 2, 3):
        kv.kvr_slot_assign(s, tk[f"slot{s}"])   # their K/V are never read by the timed steps
    slot0 = tk["slot0"]
    assert kv.kvr_slot_match(slot0[:1]) == (0, 0)
    for a in range(0, len(slot0), 256):
        chunk = slot0[a:a + 256]
        kv.kvr_prefill_suffix(0, chunk, workloads.hidden_for_tokens(chunk, shape.hidden, seed).to(device), w)
    kv.kvr_sync_status()
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    common = tk["prompt"][:P_CACHED]
    tails, xs = [], []
    for _ in range(steps_total):
        tail = rng.integers(0, workloads.VOCAB, size=M_ROWS).tolist()
        if tail[0] == slot0[P_CACHED]:
            tail[0] = (tail[0] + 1) % workloads.VOCAB
        tails.append(common + tail)
        xs.append(workloads.hidden_for_tokens(tail, shape.hidden, seed))
    setup_s = time.time() - t0
    return shape, kv, w, tails, xs, setup_s


def run_gpu(args, rank, world):
    device = torch.device("cuda", torch.cuda.current_device())
    pk, pk_kind = peaks()
    total = args.warmup + args.steps
    shape, kv, w, prompts, xs_host, setup_s = build_turn9(device, 3 * total + 2, args.layers, args.format)
    xs_dev = [x.to(device) for x in xs_host[:2 * total]]
    out = torch.empty((M_ROWS, shape.hidden), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream()

    def step(i):
        slot, reused = kv.kvr_slot_match(prompts[i])
        assert (slot, reused) == (0, P_CACHED), (slot, reused)
        kv.kvr_prefill_suffix(0, prompts[i][P_CACHED:], xs_dev[i], w, out=out)

    for i in range(args.warmup):
        step(i)
    kv.kvr_sync_status()
    kv.kvr_profile_read()  # reset counters
    # ---------------- timed region (device time)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.warmup, total):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    kv.kvr_sync_status()
    _, launches = kv.kvr_profile_read()
    ms = max_over_ranks(ms)
    ms_step = ms / args.steps
    value = whole_job_rate(world, M_ROWS, args.steps, ms)

    # ---------------- the same steps with per-kernel-class events (roofline)
    kv.kvr_profile_enable(True)
    for i in range(total + args.warmup, 2 * total):
        step(i)
    torch.cuda.synchronize()
    cls_ms, cls_n = kv.kvr_profile_read()
    kv.kvr_profile_enable(False)

    # ---------------- end to end through the public API with host buffers
    pinned_in = [x.pin_memory() for x in xs_host[2 * total:3 * total]]
    pinned_out = torch.empty((M_ROWS, shape.hidden), dtype=torch.bfloat16).pin_memory()
    dev_in = torch.empty((M_ROWS, shape.hidden), dtype=torch.bfloat16, device=device)

    def e2e_step(j):
        p = prompts[2 * total + j]
        slot, reused = kv.kvr_slot_match(p)
        dev_in.copy_(pinned_in[j], non_blocking=True)
        kv.kvr_prefill_suffix(slot, p[reused:], dev_in, w, out=out)
        pinned_out.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for j in range(min(args.warmup, total)):
        e2e_step(j)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for j in range(args.warmup, total):
        e2e_step(j)
    torch.cuda.synchronize()
    barrier()
    e2e_s = max_over_ranks(time.perf_counter() - t0)
    kv.kvr_sync_status()
    bytes_io = M_ROWS * shape.hidden * 2

    # ---------------- roofline of the dominant class (projections)
    L = shape.n_layers
    proj_flops = 2.0 * M_ROWS * shape.params_per_layer() * L          # per step
    proj_ms = cls_ms[0] / args.steps
    n_proj = cls_n[0] / args.steps
    achieved_tf = proj_flops / (proj_ms / 1e3) / 1e12
    attn_bytes = (P_CACHED + M_ROWS) * shape.n_kv_heads * shape.head_dim * 2 * 2 * L
    attn_ms = cls_ms[1] / args.steps
    attn_gbs = attn_bytes / (attn_ms / 1e3) / 1e9
    attn_flops = 4.0 * shape.head_dim * shape.n_q_heads * sum(P_CACHED + i + 1 for i in range(M_ROWS)) * L
    # each projection launch is timed alone, inside ~0.1 s of steps at full clock: the burst peak
    peak_tf = pk.get("bf16_tflops", FALLBACK["bf16_tflops"])
    weight_bytes = shape.params_per_layer() * L * 0.5625
    line = {
        "metric": "suffix-prefill rows/s",
        "value": round(value, 1),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": turn9_config(world, args.format),
        "attended_kv_gbs": round(attn_gbs, 1),
        "attended_kv_frac_hbm": round(attn_gbs / pk["hbm_gbs"], 4),
        "attention_causal_tflops": round(attn_flops / (attn_ms / 1e3) / 1e12, 1),
        "attention_frac_tensor": round(attn_flops / (attn_ms / 1e3) / 1e12 / peak_tf, 4),
        "roofline": {"bound": "tensor", "achieved": round(achieved_tf, 2),
                     "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": round(achieved_tf / peak_tf, 4),
                     # DRAM bytes from an ncu capture of the int4 kernels
                     "traffic": None if args.layers or args.format != "int4" else round(PROJ_TRAFFIC_PER_LAYER * L),
                     "traffic_per": "step (the class's 112 launches)",
                     "peak_kind": f"bf16 burst ({pk_kind})",
                     "kernel": "projections (gemv_int4 / gemm_int4)",
                     "launches_per_step": n_proj, "ms_per_step": round(proj_ms, 4),
                     "weight_gbs": round(weight_bytes / (proj_ms / 1e3) / 1e9, 1)},
        # the whole step (every launch, PDL overlap included): projection and causal attention flops
        "step_tensor": {"tflops": round((proj_flops + attn_flops) / (ms_step / 1e3) / 1e12, 1),
                        "frac": round((proj_flops + attn_flops) / (ms_step / 1e3) / 1e12 / peak_tf, 4),
                        "peak": peak_tf, "peak_kind": f"bf16 burst ({pk_kind})"},
        "kernel_ms_per_step": {"projections": round(cls_ms[0] / args.steps, 4),
                               "attention": round(cls_ms[1] / args.steps, 4),
                               "epilogues": round(cls_ms[2] / args.steps, 4),
                               "prefix_match": round(cls_ms[3] / args.steps, 4)},
        "e2e": {"value": round(world * M_ROWS * args.steps / e2e_s, 1), "unit": "rows/s",
                "h2d_bytes_per_step": bytes_io + PROMPT * 4, "d2h_bytes_per_step": bytes_io + 4 * 4 * 4},
        "gpu_launches": int(sum(launches)),
        "clocks": clk,
        "setup_s": round(setup_s, 1),
    }
    if args.layers:
        line["config"]["workload"] += f" (REDUCED to {args.layers} layers: profiling case, not the bench line)"
    del kv, w, xs_dev
    torch.cuda.empty_cache()
    if not args.no_verify and not args.layers:
        line["verify"] = verify_summary(args, pk, pk_kind)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(args.cpu_rows)
    return line, rank


def verify_summary(args, pk, pk_kind, ms_rows=(1, 8)):
    """The m <= 16 half of the metric in the bench run itself: kvr_verify of
    m rows on the dense 9B-class shape (36 x (H 4096, 32/8 heads, F 12288),
    4096 cached tokens), median of CUDA-event times per call with the slot cut
    back after each (outside the timed call), clocks sampled meanwhile.
    Algorithmic bytes per call: the weights once (0.5625 B per int4 weight),
    the slot's K/V once per KV head, the appended rows."""
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    device = torch.device("cuda", torch.cuda.current_device())
    shape = workloads.SHAPES["dense9b" if args.format == "int4" else "dense9b_q4k"]
    seed = workloads.config_seed(3)
    tk = workloads.verify_tokens(seed)
    P = len(tk["state"])
    lws = workloads.stack_weights(shape, seed, device=device)
    kv = Kvr(config_for_shape(shape, 1, P + 256, 256), device=device)
    w = kv.weights(lws)
    assert kv.kvr_slot_match(tk["state"][:1]) == (0, 0)
    _prefill_state(kv, 0, tk["state"], shape, seed, w, device)
    L = shape.n_layers
    reps = max(args.steps, 20)
    out = {}
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    for m in ms_rows:
        draft = tk["draft"][:m]
        x = workloads.hidden_for_tokens(draft, shape.hidden, seed).to(device)
        o = torch.empty((m, shape.hidden), dtype=torch.bfloat16, device=device)
        ms = _event_ms(lambda: kv.kvr_verify(0, draft, x, w, out=o), reps, args.warmup,
                       after=lambda: kv.kvr_slot_truncate(0, P))
        nbytes = (shape.params_per_layer() * 0.5625 * L
                  + (P + m) * shape.n_kv_heads * shape.head_dim * 2 * 2 * L
                  + m * shape.n_kv_heads * shape.head_dim * 4 * L)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[f"m{m}"] = {"ms": round(ms, 4), "algorithmic_gb": round(nbytes / 1e9, 4), "gbs": round(gbs, 1),
                        "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}
    kv.kvr_sync_status()
    kv.close()
    if args.format == "int4":
        # the same calls through the opt-in persistent pass (one launch per call)
        prev = os.environ.get("KVR_PASS")
        os.environ["KVR_PASS"] = "1"
        try:
            kvp = Kvr(config_for_shape(shape, 1, P + 256, 256), device=device)
        finally:
            if prev is None:
                del os.environ["KVR_PASS"]
            else:
                os.environ["KVR_PASS"] = prev
        wp = kvp.weights(lws)
        assert kvp.kvr_slot_match(tk["state"][:1]) == (0, 0)
        _prefill_state(kvp, 0, tk["state"], shape, seed, wp, device)
        out["pass"] = {"what": "KVR_PASS=1: the whole stack as one persistent launch per call (opt-in)"}
        for m in ms_rows:
            draft = tk["draft"][:m]
            x = workloads.hidden_for_tokens(draft, shape.hidden, seed).to(device)
            o = torch.empty((m, shape.hidden), dtype=torch.bfloat16, device=device)
            ms = _event_ms(lambda: kvp.kvr_verify(0, draft, x, wp, out=o), reps, args.warmup,
                           after=lambda: kvp.kvr_slot_truncate(0, P))
            nbytes = out[f"m{m}"]["algorithmic_gb"] * 1e9
            out["pass"][f"m{m}"] = {"ms": round(ms, 4), "frac_hbm": round(nbytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}
        kvp.kvr_sync_status()
        kvp.close()
    out["clocks"] = clocks.stop()
    out.update({"workload": f"speculative verify: 36 x (H 4096, 32/8 heads, F 12288) {FORMAT_LABEL[args.format]}, "
                            "4096 cached tokens, m = k+1 rows",
                "peak_hbm_gbs": pk["hbm_gbs"], "peak_kind": pk_kind, "reps": reps,
                "l2": "inputs larger than L2 (3.9 GB of weights and 0.6 GB of K/V per call)"})
    return out


# ---------------------------------------------------------------------------
# the other measured workloads (verify sweep, priming, attention crossover)
# ---------------------------------------------------------------------------

def _event_ms(call, reps, warm, before=None, after=None):
    """Median device time of `call` over `reps` runs (CUDA events on the
    launching stream); `before`/`after` run outside the timed region."""
    stream = torch.cuda.current_stream()
    for _ in range(warm):
        if before: before()
        call()
        if after: after()
    ts = []
    for _ in range(reps):
        if before: before()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
        if after: after()
    return statistics.median(ts)


def _prefill_state(kv, slot, toks, shape, seed, w, device, chunk=256):
    for a in range(0, len(toks), chunk):
        c = toks[a:a + chunk]
        kv.kvr_prefill_suffix(slot, c, workloads.hidden_for_tokens(c, shape.hidden, seed).to(device), w)
    kv.kvr_sync_status()


def run_verify(args):
    """Speculative verify: 36 layers (H 4096, 32/8 heads, F 12288), one slot
    holding 4096 tokens, m = k+1 in {1,2,3,4,6,8}; the slot is cut back to
    4096 after each call (outside the timed region).  Reports t(m) and the
    least-squares fit a + b m, and the HBM fraction of each m against the
    bytes one call must move (weights once, K/V once per KV head, the append)."""
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    device = torch.device("cuda", torch.cuda.current_device())
    pk, pk_kind = peaks()
    shape = workloads.SHAPES["dense9b" if args.format == "int4" else "dense9b_q4k"]
    if args.layers:   # profiling aid: a reduced stack
        shape = dataclasses.replace(shape, n_layers=args.layers)
    seed = workloads.config_seed(3)
    tk = workloads.verify_tokens(seed)
    P = len(tk["state"])
    lws = workloads.stack_weights(shape, seed, device=device)
    kv = Kvr(config_for_shape(shape, 1, P + 256, 256, vocab=workloads.VOCAB), device=device)
    w = kv.weights(lws)
    head = workloads.head_weights(shape, seed, device=device)
    assert kv.kvr_slot_match(tk["state"][:1]) == (0, 0)
    _prefill_state(kv, 0, tk["state"], shape, seed, w, device)
    L = shape.n_layers
    table = []
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    for m in (1, 2, 3, 4, 6, 8):
        draft = tk["draft"][:m]
        x = workloads.hidden_for_tokens(draft, shape.hidden, seed).to(device)
        out = torch.empty((m, shape.hidden), dtype=torch.bfloat16, device=device)
        ms = _event_ms(lambda: kv.kvr_verify(0, draft, x, w, out=out), args.steps, args.warmup,
                       after=lambda: kv.kvr_slot_truncate(0, P))
        kv.kvr_sync_status()
        # the same rows, then the output head, the argmax and the acceptance count
        # (one device-to-host read of m token ids and a stream synchronisation inside)
        ms_acc = _event_ms(lambda: kv.kvr_verify_accept(0, draft, x, w, head, out=out), args.steps,
                           args.warmup, after=lambda: kv.kvr_slot_truncate(0, P))
        # one speculative step as a caller sees it: the rows' hidden states from
        # pinned host memory, the call, the decision back on the host (wall clock,
        # the host's launch work included)
        x_host = x.cpu().pin_memory()
        x_dev = torch.empty_like(x)
        walls = []
        for i in range(args.warmup + args.steps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            x_dev.copy_(x_host, non_blocking=True)
            kv.kvr_verify_accept(0, draft, x_dev, w, head, out=out)
            walls.append((time.perf_counter() - t0) * 1e3)
            kv.kvr_slot_truncate(0, P)
        step_ms = statistics.median(walls[args.warmup:])
        kv.kvr_profile_read()
        kv.kvr_profile_enable(True)
        for _ in range(3):
            kv.kvr_verify(0, draft, x, w, out=out)
            kv.kvr_slot_truncate(0, P)
        cls_ms, cls_n = kv.kvr_profile_read()
        kv.kvr_profile_enable(False)
        nbytes = (shape.params_per_layer() * 0.5625 * L
                  + (P + m) * shape.n_kv_heads * shape.head_dim * 2 * 2 * L
                  + m * shape.n_kv_heads * shape.head_dim * 4 * L)
        gbs = nbytes / (ms / 1e3) / 1e9
        table.append({"m": m, "ms": round(ms, 4), "accept_ms": round(ms_acc, 4), "step_e2e_ms": round(step_ms, 4),
                      "rows_per_s": round(m / (ms / 1e3), 1),
                      "algorithmic_gb": round(nbytes / 1e9, 4), "gbs": round(gbs, 1),
                      "frac_hbm": round(gbs / pk["hbm_gbs"], 4),
                      "class_ms_serialised": {k: round(v / 3, 4) for k, v in
                                              zip(("projections", "attention", "epilogues"), cls_ms)},
                      "launches": cls_n[0] // 3 + cls_n[1] // 3 + cls_n[2] // 3})
    clk = clocks.stop()
    ms_ = np.array([r["m"] for r in table], dtype=np.float64)
    ts = np.array([r["ms"] for r in table])
    b, a = np.polyfit(ms_, ts, 1)
    kv.close()
    reduced = f" (REDUCED to {args.layers} layers: profiling case)" if args.layers else ""
    return {"metric": "verify ms per call", "workload": "speculative verify: 36 x (H 4096, 32/8 heads, F 12288) "
            f"{FORMAT_LABEL[args.format]}, 4096 cached tokens, m = k+1 rows" + reduced, "unit": "ms", "higher_is_better": False,
            "fit_ms": {"a": round(float(a), 4), "b_per_row": round(float(b), 4)},
            "accept": {"vocab": workloads.VOCAB, "what": "accept_ms: kvr_verify_accept (verify + final "
                       "RMSNorm + int4 LM head + argmax + acceptance, read back to the host), device events; "
                       "step_e2e_ms: the same call as one speculative step on the host's wall clock, hidden "
                       "rows copied from pinned host memory, host launch work included"},
            "page_fit_ms": {"a": 9.0, "b_per_row": 5.5, "hardware": "the page's own (not a GB300)"},
            "per_m": table, "peak_hbm_gbs": pk["hbm_gbs"], "peak_kind": pk_kind,
            "l2": "inputs larger than L2 (3.9 GB of weights and 0.6 GB of K/V per call)",
            "reps": args.steps, "warmup": args.warmup, "clocks": clk, "dtype": "bf16", "data": "synthetic"}


def run_priming(args):
    """Multi-branch priming: 36 layers (H 2560, 16/8 heads, F 9728), a 1200-token
    state, 4 questions of 40 tokens in one kvr_prefill_branches call, against the
    same 4 questions as 4 separate kvr_prefill_suffix calls (each followed by a
    cut back to 1200, a host-only step)."""
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    device = torch.device("cuda", torch.cuda.current_device())
    shape = workloads.SHAPES["dense4b"]
    seed = workloads.config_seed(4)
    tk = workloads.priming_tokens(seed)
    P = len(tk["state"])
    lws = workloads.stack_weights(shape, seed, device=device)
    kv = Kvr(config_for_shape(shape, 1, P + 272, 256), device=device)
    w = kv.weights(lws)
    assert kv.kvr_slot_match(tk["state"][:1]) == (0, 0)
    _prefill_state(kv, 0, tk["state"], shape, seed, w, device)
    qs = tk["questions"]
    lens = [len(q) for q in qs]
    allq = sum(qs, [])
    xq = workloads.hidden_for_tokens(allq, shape.hidden, seed).to(device)
    xs = [xq[sum(lens[:b]):sum(lens[:b + 1])].contiguous() for b in range(len(qs))]
    out = torch.empty((sum(lens), shape.hidden), dtype=torch.bfloat16, device=device)
    outs = [torch.empty((n, shape.hidden), dtype=torch.bfloat16, device=device) for n in lens]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    ms_batched = _event_ms(lambda: kv.kvr_prefill_branches(0, lens, allq, xq, w, out=out),
                           args.steps, args.warmup)

    def separate():
        for b in range(len(qs)):
            kv.kvr_prefill_suffix(0, qs[b], xs[b], w, out=outs[b])
            kv.kvr_slot_truncate(0, P)
    ms_sep = _event_ms(separate, args.steps, args.warmup)
    clk = clocks.stop()
    kv.kvr_sync_status()
    assert kv.kvr_slot_len(0) == P
    kv.close()
    rows = sum(lens)
    return {"metric": "priming rows/s", "workload": "multi-branch priming: 36 x (H 2560, 16/8 heads, F 9728) "
            "int4-g32, 1200-token state, 4 questions x 40 tokens", "unit": "rows/s", "higher_is_better": True,
            "value": round(rows / (ms_batched / 1e3), 1), "ms_batched": round(ms_batched, 4),
            "ms_separate_4_calls": round(ms_sep, 4), "speedup": round(ms_sep / ms_batched, 3),
            "l2": "inputs larger than L2 (1.83 GB of weights per call)",
            "reps": args.steps, "warmup": args.warmup, "clocks": clk, "dtype": "bf16", "data": "synthetic"}


def run_batch(args):
    """Continuous batching across conversations: the verify shape (36 layers,
    H 4096, 32/8 heads, F 12288, int4-g32), 4 slots each holding its own
    4096-token conversation; m rows per conversation (m in {1, 4}) verified in
    one kvr_prefill_batch call against 4 separate kvr_verify calls (the slots
    are cut back outside the timed region).  Reports both times and the HBM
    fraction of the batched call against its algorithmic bytes (weights once,
    every conversation's K/V once per KV head, the appends)."""
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    device = torch.device("cuda", torch.cuda.current_device())
    pk, pk_kind = peaks()
    shape = workloads.SHAPES["dense9b"]
    n = 4
    seed = workloads.config_seed(3)
    tks = [workloads.verify_tokens(seed + 17 * j) for j in range(n)]
    P = len(tks[0]["state"])
    lws = workloads.stack_weights(shape, seed, device=device)
    kv = Kvr(config_for_shape(shape, n, P + 256, 256, vocab=workloads.VOCAB), device=device)
    w = kv.weights(lws)
    head = workloads.head_weights(shape, seed, device=device)
    for j in range(n):
        _prefill_state(kv, j, tks[j]["state"], shape, seed + j, w, device)
    L = shape.n_layers
    table = []
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()

    def cut():
        for j in range(n):
            kv.kvr_slot_truncate(j, P)
    for m in (1, 4):
        drafts = [tks[j]["draft"][:m] for j in range(n)]
        xs = [workloads.hidden_for_tokens(d, shape.hidden, seed + j).to(device) for j, d in enumerate(drafts)]
        xall = torch.cat(xs).contiguous()
        out = torch.empty((n * m, shape.hidden), dtype=torch.bfloat16, device=device)
        outs = [torch.empty((m, shape.hidden), dtype=torch.bfloat16, device=device) for _ in range(n)]
        ms_b = _event_ms(lambda: kv.kvr_prefill_batch(list(range(n)), drafts, xall, w, out=out),
                         args.steps, args.warmup, after=cut)

        def separate():
            for j in range(n):
                kv.kvr_verify(j, drafts[j], xs[j], w, out=outs[j])
        ms_s = _event_ms(separate, args.steps, args.warmup, after=cut)
        # the same rows with the greedy decision for every conversation (one call,
        # read back to the host)
        ms_acc = _event_ms(lambda: kv.kvr_verify_accept_batch(list(range(n)), drafts, xall, w, head, out=out),
                           args.steps, args.warmup, after=cut)
        kv.kvr_sync_status()
        nbytes = (shape.params_per_layer() * 0.5625 * L
                  + n * (P + m) * shape.n_kv_heads * shape.head_dim * 2 * 2 * L
                  + n * m * shape.n_kv_heads * shape.head_dim * 4 * L)
        gbs = nbytes / (ms_b / 1e3) / 1e9
        table.append({"m_per_conversation": m, "rows": n * m, "ms_batched": round(ms_b, 4),
                      "ms_separate_4_calls": round(ms_s, 4), "speedup": round(ms_s / ms_b, 3),
                      "accept_batch_ms": round(ms_acc, 4),
                      "rows_per_s_batched": round(n * m / (ms_b / 1e3), 1),
                      "algorithmic_gb": round(nbytes / 1e9, 4), "gbs": round(gbs, 1),
                      "frac_hbm": round(gbs / pk["hbm_gbs"], 4)})
    clk = clocks.stop()
    kv.close()
    return {"metric": "batched verify rows/s", "workload": "4 conversations x 4096 cached tokens, 36 x (H 4096, "
            "32/8 heads, F 12288) int4-g32, m rows each in one call", "unit": "rows/s", "higher_is_better": True,
            "per_m": table, "peak_hbm_gbs": pk["hbm_gbs"], "peak_kind": pk_kind,
            "l2": "inputs larger than L2 (3.9 GB of weights and 2.4 GB of K/V per call)",
            "reps": args.steps, "warmup": args.warmup, "clocks": clk, "dtype": "bf16", "data": "synthetic"}


def run_crossover(args):
    """Attention crossover: one 7B-shaped attention + QKV/O layer, 4 slots of
    16384; the target slot holds P cached tokens (K/V drawn N(0,1)); m rows are
    prefilled after them.  L2 is flushed (a 2 x L2 write) before every timed
    call.  Reports the call time, the attention kernels' time (per-class
    events) and the attended-KV GB/s for each (P, m)."""
    from prefix_reused_prefill_gb300 import Kvr, config_for_shape
    device = torch.device("cuda", torch.cuda.current_device())
    pk, pk_kind = peaks()
    shape = workloads.SHAPES["qwen7b_attn"]
    seed = workloads.config_seed(5)
    lw = workloads.layer_weights(shape, seed, 0, device=device)
    kv = Kvr(config_for_shape(shape, 4, 16384, 1024), device=device)
    w = kv.weights([lw])
    flush_buf = torch.empty(2 * 129 * 2 ** 20 // 4, dtype=torch.float32, device=device)  # 2 x L2
    Hkv, d, Hq = shape.n_kv_heads, shape.head_dim, shape.n_q_heads
    table = []
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    Ps = [int(v) for v in args.crossover_p.split(",")] if args.crossover_p else (512, 2048, 8192, 15360)
    ms_list = [int(v) for v in args.crossover_m.split(",")] if args.crossover_m else (1, 4, 16, 64, 256, 1024)
    for P in Ps:
        kk, vv = workloads.random_kv(Hkv, P, d, seed + P)
        k, v = kv.kvr_slot_kv(3, 0)
        k[:, :P] = kk.to(device)
        v[:, :, :P] = vv.transpose(1, 2).to(device)
        kv.kvr_slot_assign(3, list(range(P)))
        for m in ms_list:
            new = list(range(40000, 40000 + m))
            x = workloads.hidden_for_tokens(new, shape.hidden, seed).to(device)
            out = torch.empty((m, shape.hidden), dtype=torch.bfloat16, device=device)
            call = lambda: kv.kvr_prefill_suffix(3, new, x, w, out=out)  # noqa: E731
            flush = lambda: flush_buf.fill_(1.0)  # noqa: E731
            cut = lambda: kv.kvr_slot_truncate(3, P)  # noqa: E731
            ms = _event_ms(call, args.steps, args.warmup, before=flush, after=cut)
            kv.kvr_profile_read()
            kv.kvr_profile_enable(True)
            for _ in range(args.steps):
                flush()
                call()
                cut()
            torch.cuda.synchronize()
            cls_ms, _ = kv.kvr_profile_read()
            kv.kvr_profile_enable(False)
            attn_ms = cls_ms[1] / args.steps
            kv_bytes = (P + m) * Hkv * d * 2 * 2
            flops = 4.0 * d * Hq * sum(P + i + 1 for i in range(m))
            table.append({"P": P, "m": m, "ms": round(ms, 4), "attn_ms": round(attn_ms, 4),
                          "proj_ms": round(cls_ms[0] / args.steps, 4),
                          "attended_kv_gbs": round(kv_bytes / (attn_ms / 1e3) / 1e9, 1),
                          "attn_tflops": round(flops / (attn_ms / 1e3) / 1e12, 2)})
        kv.kvr_sync_status()
    clk = clocks.stop()
    kv.close()
    return {"metric": "attention crossover", "workload": "one 7B-shaped attention + QKV/O layer (H 3584, 28/4 "
            "heads, int4-g32), 4 slots x 16384, P cached x m new rows", "unit": "ms",
            "higher_is_better": False, "per_case": table, "peak_hbm_gbs": pk["hbm_gbs"],
            "peak_bf16_tflops": pk.get("bf16_tflops"), "peak_kind": pk_kind,
            "l2": "flushed before every timed call (2 x L2 write)",
            "reps": args.steps, "warmup": args.warmup, "clocks": clk, "dtype": "bf16", "data": "synthetic"}


# ---------------------------------------------------------------------------
# the oracle, timed on the host cores
# ---------------------------------------------------------------------------

_ORACLE_SETUP = {}


def _oracle_turn9_layer(rows: int):
    """Decoded layer-0 weights, the cached prefix and the suffix rows (built once)."""
    if rows in _ORACLE_SETUP:
        return _ORACLE_SETUP[rows]
    from oracle import model as om
    from oracle import formats
    shape = workloads.SHAPES["qwen7b"]
    seed = workloads.config_seed(2)
    lw = workloads.layer_weights(shape, seed, 0, device="cpu")
    W = {}
    for k, v in lw.items():
        if hasattr(v, "packed"):
            W[k] = formats.dequant_int4(v.packed.numpy(), v.scales.numpy())
        else:
            W[k] = v.to(torch.float64).numpy()
    dims = om.Dims(shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn, False,
                   shape.rope_theta, shape.rms_eps)
    cache = om.SlotKV(1, shape.n_kv_heads, P_CACHED + rows, shape.head_dim)
    k, v = workloads.random_kv(shape.n_kv_heads, P_CACHED, shape.head_dim, seed)
    cache.K[0][:, :P_CACHED] = workloads.bf16_to_f64(k)
    cache.V[0][:, :P_CACHED] = workloads.bf16_to_f64(v)
    x = workloads.bf16_to_f64(workloads.hidden_for_tokens(list(range(rows)), shape.hidden, seed))
    _ORACLE_SETUP[rows] = (shape, dims, W, cache, x)
    return _ORACLE_SETUP[rows]


def cpu_baseline(rows: int, min_seconds: float = 10.0):
    """Oracle (float64 numpy, as it stands) on the turn-9 workload: the layer
    evaluated for `rows` suffix rows over a 1668-row cached prefix (K/V drawn
    N(0,1)), repeated until at least `min_seconds` of CPU work, scaled to rows/s
    of the full 28-layer stack.  Weight decoding happens before timing."""
    from oracle import model as om
    shape, dims, W, cache, x = _oracle_turn9_layer(rows)
    n_eval = 0
    t0 = time.perf_counter()
    while True:
        om.layer(dims, W, x, cache.K[0], cache.V[0], om.plain_rows(P_CACHED, rows))
        n_eval += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    per_row_stack = dt / (n_eval * rows) * shape.n_layers
    cores = int(os.environ.get("OMP_NUM_THREADS", 0)) or os.cpu_count()
    return {"value": round(1.0 / per_row_stack, 3), "unit": "rows/s", "cores": cores,
            "kind": "oracle", "extrapolated": f"one layer timed, scaled x{shape.n_layers} to the stack",
            "layer_s": round(dt / n_eval, 3),
            "sample": f"{n_eval} layer evaluation(s) of {rows} suffix rows over 1668 cached rows "
                      f"(float64 numpy, {dt:.1f} s), extrapolated to the 28-layer stack"}


def run_reference(args, rank, world):
    """--impl reference: the oracle as the reference arm (host cores).  A timed
    step is one layer of the turn-9 workload (254 suffix rows over the
    1668-row prefix): ms_per_step is that measured time, and value is the
    rate of the whole 28-layer stack extrapolated from it (named beside it)."""
    if rank != 0:
        return None, rank
    vals = []
    for _ in range(args.warmup):
        cpu_baseline(args.cpu_rows, min_seconds=0.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(args.cpu_rows, min_seconds=0.0))
    dt = time.perf_counter() - t0
    v = statistics.median(x["value"] for x in vals)
    layer_ms = 1000.0 * statistics.median(x["layer_s"] for x in vals)
    n_layers = workloads.SHAPES["qwen7b"].n_layers
    cb = dict(vals[0]); cb["value"] = v; cb["layer_s"] = round(layer_ms / 1e3, 3)
    line = {"impl": "reference", "metric": "suffix-prefill rows/s", "value": v, "unit": "rows/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(layer_ms, 1),
            "step": "one layer of the stack (the timed unit); value extrapolates it to all layers",
            "stack_ms_extrapolated": round(layer_ms * n_layers, 1),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": turn9_config(world),
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0},
            "wall_s": round(dt, 1)}
    return line, rank


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kvr", choices=["kvr", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=M_ROWS)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-verify", action="store_true", help="turn9: skip the verify object")
    ap.add_argument("--workload", default="turn9", choices=["turn9", "verify", "priming", "crossover", "batch"],
                    help="turn9 is the bench line; the others print their own measurement line")
    ap.add_argument("--format", default="int4", choices=["int4", "q4k"],
                    help="weight format of the turn9 and verify workloads")
    ap.add_argument("--crossover-p", default="", help="crossover: cached lengths to run (comma-separated)")
    ap.add_argument("--crossover-m", default="", help="crossover: row counts to run (comma-separated)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: run a reduced stack of this many layers")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "kvr" else max(args.warmup, 0)
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        line, rank = run_reference(args, rank, world)
    elif args.workload != "turn9":
        runner = {"verify": run_verify, "priming": run_priming, "crossover": run_crossover,
                  "batch": run_batch}[args.workload]
        line = runner(args) if rank == 0 else None
    else:
        line, rank = run_gpu(args, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
