#!/usr/bin/env python
"""Benchmark of the mixed prefill+decode step on GB300.

Default workload (the largest single-GPU configuration): the 40-layer
Qwen3-14B-shaped stack (random-init weights, seeded synthetic data) over a
whole 32,768-token prompt fed as 2,048-token chunks, prefix 0 .. 30,720, beside
96 running decodes with contexts log-uniform in [1024, 8192], KV fully paged in
HBM.  One step = one mb_stack_step: 2,144 tokens (the decodes and one chunk)
through all 40 layers (RMSNorm, QKV GEMM, q/k-norm + RoPE + KV append,
prefill-chunk attention tiles, split-KV decode rows + merge, O GEMM +
residual, RMSNorm, gate/up GEMM + SwiGLU, down GEMM + residual, per layer);
step i takes chunk i mod 16 of the prompt.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the reference arm: a plain float64 restatement of the method).
``--workload`` selects a single-layer workload instead of the stack.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]
                    [--workload qwen3_14b_stack40_prompt32768|llama3_8b_T576|qwen3_14b_P0|
                                qwen3_14b_P1024|qwen3_14b_P2200|tiny_T68]
"""

from __future__ import annotations

import argparse
import json
import math
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

from mixed_prefill_decode_gb300 import workload as W  # noqa: E402

METRIC = "mixed prefill+decode step tokens/s; decode-attn HBM GB/s; GEMM TFLOP/s % peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Empties L2 between timed steps: writes a 256 MiB buffer (twice L2),
    then reads another one, so that the lines left in L2 are clean.  After the
    write alone, up to the whole L2 (129 MB) is dirty, and writing it back to
    HBM costs the next timed kernel ~18 us (measured on GB300: a 356 MB
    read-only TMA stream took 73 us after a write-only flush, 59 us after this
    one)."""

    def __init__(self, torch):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device="cuda")

    def __call__(self, i: int = 0) -> None:
        self.w.fill_(i & 0xFF)
        self.r.sum()


HEADLINE = "qwen3_14b_stack40_prompt32768"


def workload_by_name(name: str) -> W.Workload:
    if name == "llama3_8b_T576":
        return W.llama3_8b_mixed()
    if name.startswith("qwen3_14b_P"):
        return W.qwen3_14b_mixed(int(name.split("P")[1]))
    if name == "tiny_T68":
        return W.tiny_mixed()
    raise SystemExit(f"unknown workload {name}")


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture, keyed by kernel; each is valid only for the sources it was captured on
# and reads as null once any of them changes.
NCU_TRAFFIC = {
    "gemm_gate_up": {"bytes": 283.620864e6, "sha256_16": "4ac6531ba35ed8ed",
                     "sources": ("csrc/mb_gemm.cu", "csrc/mb_ptx.cuh", "csrc/mb_kernels.h"),
                     "capture": "ncu DRAM bytes of bench.py --case llama_T576, the third GEMM of the fourth step"},
    # mean over the 16 chunk-alone launches of the prompt sweep (one capture
    # of each: bench.py --case chunk_all), as the roofline's time is
    "attention_chunk": {"bytes": 174.216528e6, "sha256_16": "fbd573b13e2c7b6f",
                        "sources": ("csrc/mb_attn.cu", "csrc/mb_ptx.cuh", "csrc/mb_kernels.h", "csrc/mb_api.cpp"),
                        "capture": "ncu DRAM bytes of bench.py --case chunk_all, the 16 launches of the second pass"},
}


def ncu_traffic(kernel: str):
    import hashlib
    rec = NCU_TRAFFIC.get(kernel)
    if rec is None:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        with open(os.path.join(ROOT, "mixed_prefill_decode_gb300", f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["sha256_16"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- accounting
def algorithmic(shape: W.LayerShape, batch: W.Batch) -> dict:
    """Per-launch algorithmic work of each kernel (what the method must do)."""
    T = batch.num_tokens
    d, hd, F = shape.d_model, shape.head_dim, shape.d_ff
    Hq, Hkv = shape.n_q_heads, shape.n_kv_heads
    qo = batch.qo_len()
    c = batch.cached()
    dec = qo == 1
    pairs = float(np.sum(qo[~dec] * c[~dec] + qo[~dec] * (qo[~dec] + 1) / 2))
    return {
        "rmsnorm_attn": ("hbm", 2.0 * T * d * 2),
        "gemm_qkv": ("tensor", 2.0 * T * shape.qkv_dim * d),
        "rope_append": ("hbm", 2.0 * T * shape.qkv_dim * 2),
        # one grid: chunk tiles (tensor FLOPs) and decode rows (KV bytes)
        "attention": ("mixed", (4.0 * hd * Hq * pairs, float(np.sum(batch.kv_len[dec])) * Hkv * hd * 2 * 2)),
        "attn_merge": ("hbm", 0.0),
        "gemm_o": ("tensor", 2.0 * T * d * Hq * hd),
        "rmsnorm_ffn": ("hbm", 2.0 * T * d * 2),
        "gemm_gate_up": ("tensor", 2.0 * T * 2 * F * d),
        "gemm_down": ("tensor", 2.0 * T * d * F),
    }


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms while running (read-only queries)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, world, local, pg


def reduce_max(pg, v: float) -> float:
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg):
    if pg is not None:
        pg.barrier()


def replica_throughput(pg, world: int, tokens_per_step: int, ms_local: float):
    """Replicas only: every rank runs the same step on its own GPU.  The job's
    step time is the slowest rank's; the value counts the tokens of all ranks."""
    ms = reduce_max(pg, ms_local)
    return ms, world * tokens_per_step / (ms / 1e3)


# ----------------------------------------------------------- CPU oracle
def oracle_inputs(wl: W.Workload):
    from oracle import layer as OL
    wb, x, batch, pool = W.materialize(wl, unit_gains=True)
    return OL, OL.weights_to_f64(wb), OL.bf16_bits_to_f64(x), batch, OL.bf16_bits_to_f64(pool)


def sub_batch(batch: W.Batch, x: np.ndarray, n_dec: int, n_chunk: int):
    """First n_dec decode rows and the first n_chunk rows of the chunk (same
    prefix), as a batch of their own: a bounded sample of the workload."""
    qo = batch.qo_len()
    rows, xs = [], []
    kept_dec = 0
    for r in range(batch.num_reqs):
        t0 = batch.qo_indptr[r]
        table = batch.bt[batch.bt_indptr[r]:batch.bt_indptr[r + 1]]
        c = int(batch.kv_len[r] - qo[r])
        if qo[r] == 1 and kept_dec < n_dec:
            rows.append((1, c + 1, table))
            xs.append(x[t0:t0 + 1])
            kept_dec += 1
        elif qo[r] > 1 and n_chunk > 0:
            n = min(n_chunk, int(qo[r]))
            rows.append((n, c + n, table[:W.pages_for(c + n)]))
            xs.append(x[t0:t0 + n])
    qo_indptr = np.cumsum([0] + [r[0] for r in rows])
    kv = np.array([r[1] for r in rows])
    bti = np.cumsum([0] + [len(r[2]) for r in rows])
    bt = np.concatenate([r[2] for r in rows])
    return qo_indptr, kv, bti, bt, np.concatenate(xs)


def time_oracle_step(OL, shape, w, pool, qo_indptr, kv, bti, bt, x) -> float:
    p = pool.copy() if pool.size < (1 << 27) else pool   # appends rewrite the same slots each step
    t = time.perf_counter()
    OL.layer_step(shape.as_dict(), w, p, qo_indptr, kv, bti, bt, x)
    return time.perf_counter() - t


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def calibrate_sample(OL, wl, w, x, batch, pool, target_s: float):
    """Pick (n_dec, n_chunk), a fixed fraction of the workload's decode and
    chunk rows, so that one oracle step takes about target_s."""
    n_dec_all = int(np.sum(batch.qo_len() == 1))
    n_chunk_all = int(np.max(batch.qo_len())) if np.any(batch.qo_len() > 1) else 0
    frac = 1.0 / 64
    while True:
        nd = max(1, int(round(n_dec_all * frac)))
        nc = int(round(n_chunk_all * frac))
        dt = time_oracle_step(OL, wl.shape, w, pool, *sub_batch(batch, x, nd, nc))
        if dt >= 0.5 * target_s or frac >= 1.0:
            return nd, nc
        frac = min(1.0, frac * min(4.0, max(1.5, target_s / max(dt, 1e-6))))


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    if args.workload == HEADLINE:
        sw = W.qwen3_14b_prompt_sweep()
        per_step = 150.0 / max(1, args.steps + args.warmup)
        tokens, t, desc = stack_cpu_sample(sw, per_step, steps=args.steps, warmup=args.warmup)
        value = tokens / (sw.n_layers * t)
        desc = "each step: " + desc
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": sw.n_layers * t * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded)",
                "config": {"workload": sw.name, "tokens_per_step": tokens, "sample": desc},
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    wl = workload_by_name(args.workload)
    OL, w, x, batch, pool = oracle_inputs(wl)
    budget_s = 150.0
    per_step = budget_s / max(1, args.steps + args.warmup)
    nd, nc = calibrate_sample(OL, wl, w, x, batch, pool, per_step)
    sample = sub_batch(batch, x, nd, nc)
    tokens = int(sample[0][-1])
    for _ in range(args.warmup):
        time_oracle_step(OL, wl.shape, w, pool, *sample)
    times = [time_oracle_step(OL, wl.shape, w, pool, *sample) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = tokens / t
    desc = (f"each step: oracle layer step over {nd} of the decode rows and the first {nc} rows of the "
            f"chunk ({tokens} tokens) of workload {wl.name}, float64 NumPy")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": wl.name, "tokens_per_step": tokens, "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU arm
def decode_only_attention(mb, torch, peaks, steps: int = 30) -> dict:
    """Attention of a decode-only step (Qwen3-14B-shaped layer, 16 decodes at
    8,192-token contexts: 537 MB of KV), timed with the layer's own events:
    the decode rows' HBM rate with no chunk tiles in the grid."""
    wl = W.qwen3_14b_mixed(0)
    wb, x, batch, pool = W.materialize(wl, unit_gains=True)
    dw = {k: to_dev(v, torch) for k, v in wb.items()}
    dpool = to_dev(pool.reshape(-1), torch)
    layer = mb.Layer(wl.shape.as_dict(), dw, batch.num_tokens, pool.shape[0], kv_buf=dpool)
    cb = mb.Batch.of(batch)
    dx = to_dev(x, torch)
    dy = torch.empty_like(dx)
    s = torch.cuda.current_stream().cuda_stream
    flush = L2Flush(torch)
    for _ in range(3):
        layer.step(cb, dx, dy, s)
    mb.mb_layer_set_timing(layer.handle, True)
    for i in range(steps):
        flush(i & 0xFF)
        layer.step(cb, dx, dy, s)
    km, n = mb.mb_layer_timing(layer.handle)
    mb.mb_device_status(layer.handle, s)
    layer.close()
    ms = (km["attention"] + km["attn_merge"]) / max(1, n)
    by = float(np.sum(batch.kv_len)) * wl.shape.n_kv_heads * wl.shape.head_dim * 4
    gbs = by / (ms / 1e3) / 1e9
    return {"workload": wl.name, "ms": round(ms, 5), "kv_bytes": by, "gbs": round(gbs, 1),
            "frac": round(gbs / peaks["hbm_gbs"], 4), "includes": "attention launch + merge"}


def stack_step_time(mb, torch, wl, n_layers, steps: int = 10, warmup: int = 3, share_pool_bytes: float = 0.0,
                    weights=None) -> dict:
    """Device time of one step of an n_layers stack (one descriptor, CUDA
    graph replay), L2 flushed between steps.  Weights and KV are drawn on the
    device.  If the layers' KV would exceed `share_pool_bytes` (> 0), all
    layers use one physical pool: timing-equivalent, since every layer's KV is
    far larger than L2 and layers run one after another."""
    sh = wl.shape
    batch, num_pages = W.make_batch(wl.reqs, wl.seed + 1, spare_pages=4)
    x = W.make_embeddings(batch.num_tokens, sh.d_model, wl.seed + 2)
    pool_bytes = num_pages * 2 * sh.n_kv_heads * 16 * sh.head_dim * 2
    shared = share_pool_bytes > 0 and pool_bytes * n_layers > share_pool_bytes
    layers, keep = [], []
    shared_pool = W.device_kv_pool(sh, num_pages, wl.seed + 200) if shared else None
    for l in range(n_layers):
        dw = weights[l] if weights is not None else W.device_weights(sh, wl.seed + 100 + l)
        dpool = shared_pool if shared else W.device_kv_pool(sh, num_pages, wl.seed + 200 + l)
        layers.append(mb.Layer(sh.as_dict(), dw, batch.num_tokens, num_pages, kv_buf=dpool))
        keep.append((dw, dpool))
    stack = mb.mb_stack_create([L.handle for L in layers], True)
    cb = mb.Batch.of(batch)
    dx = to_dev(x, torch)
    dy = torch.empty_like(dx)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    flush = L2Flush(torch)
    kvs = [L.kv for L in layers]
    for _ in range(warmup):
        mb.mb_stack_step(stack, kvs, cb, dx, dy, s)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush(i & 0xFF)
        e0[i].record(stream)
        mb.mb_stack_step(stack, kvs, cb, dx, dy, s)
        e1[i].record(stream)
    torch.cuda.synchronize()
    mb.mb_device_status(layers[0].handle, s)
    ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / steps
    launches = mb.mb_stack_last_launches(stack)
    mb.mb_stack_destroy(stack)
    for L in layers:
        L.close()
    del keep, shared_pool
    torch.cuda.empty_cache()
    T = batch.num_tokens
    return {"workload": wl.name, "layers": n_layers, "tokens_per_step": T, "ms_per_step": round(ms, 4),
            "tokens_per_s": round(T / (ms / 1e3), 1), "launches_per_step": launches,
            "kv_pool": "one physical pool shared by all layers" if shared else "one pool per layer"}


def qwen3_14b_piggyback(mb, torch, prefill_tokens=(0, 1024, 2200), timer=None) -> dict:
    """Qwen3-14B shape, 16 decodes at 8,192-token contexts plus P piggybacked
    prompt tokens (prefix 0), P in {0, 1024, 2200}: the single layer's step
    and the 40-layer stack's step, whose time is the decodes' time between
    tokens (ConfluxServe's setting: how many prompt tokens ride along within a
    TBT target).  Weights and KV drawn on the device, graph-replayed, L2
    flushed between steps.  A point that fails records its error instead, so
    the rest of the line still prints."""
    timer = timer or stack_step_time
    out = {}
    for P in prefill_tokens:
        wl = W.qwen3_14b_mixed(P)
        try:
            one = timer(mb, torch, wl, 1, steps=20)
            full = timer(mb, torch, wl, 40)
            out[f"P{P}"] = {"tokens_per_step": one["tokens_per_step"],
                            "layer_ms": one["ms_per_step"], "layer_tokens_per_s": one["tokens_per_s"],
                            "stack40_ms": full["ms_per_step"], "stack40_tokens_per_s": full["tokens_per_s"],
                            "stack40_launches": full["launches_per_step"]}
        except Exception as e:   # recorded, not raised: the headline line must still print
            out[f"P{P}"] = {"error": f"{type(e).__name__}: {e}"[:300]}
    return {"workload": "qwen3_14b_mixed_P{0,1024,2200}", "decodes": 16, "decode_context": 8192,
            "points": out}


def generation_step_time(mb, torch, peaks, n_decodes: int = 64, vocab: int = 128256, steps: int = 8,
                         warmup: int = 3) -> dict:
    """Token generation on the 32-layer Llama-3-8B-shaped stack (pofe.ai
    "Chunked prefill", step 5: the pass samples its next tokens): per step,
    the stack over n_decodes decode rows, the final RMSNorm + LM head (vocab x
    d, bf16) + greedy argmax of every row, and the embedding of the sampled ids
    as the next step's input.  Weights, KV and the LM head are drawn on the
    device; L2 flushed between steps.  Reports output tokens/s and the LM
    head's share (its time also alone, against HBM: the weights are read once
    per step)."""
    sh = W.LLAMA3_8B
    wl, nl = W.llama3_8b_stack(n_decodes, n_decodes)   # a budget of b: decodes only
    batch, num_pages = W.make_batch(wl.reqs, wl.seed + 1, spare_pages=4 * n_decodes)
    d = sh.d_model
    free_budget = torch.cuda.mem_get_info()[0] - (24 << 30)
    pool_bytes = num_pages * 2 * sh.n_kv_heads * 16 * sh.head_dim * 2
    shared = pool_bytes * nl > free_budget
    shared_pool = W.device_kv_pool(sh, num_pages, wl.seed + 200) if shared else None
    layers, keep = [], []
    for l in range(nl):
        dw = W.device_weights(sh, 5100 + l)
        dpool = shared_pool if shared else W.device_kv_pool(sh, num_pages, wl.seed + 200 + l)
        layers.append(mb.Layer(sh.as_dict(), dw, batch.num_tokens, num_pages, kv_buf=dpool))
        keep.append((dw, dpool))
    stack = mb.mb_stack_create([L.handle for L in layers], True)
    g = torch.Generator(device="cuda").manual_seed(wl.seed + 7)
    w_lm = (torch.randn((vocab, d), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    table = torch.randn((vocab, d), generator=g, device="cuda").to(torch.bfloat16)
    g_final = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    T = batch.num_tokens
    x = torch.randn((T, d), generator=g, device="cuda").to(torch.bfloat16)
    y = torch.empty_like(x)
    rows = torch.arange(T, dtype=torch.int32, device="cuda")
    yw = torch.empty_like(x)
    logits = torch.empty((T, vocab), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((T,), dtype=torch.int32, device="cuda")
    kvs = [L.kv for L in layers]
    cb = mb.Batch.of(batch)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    flush = L2Flush(torch)

    def one_step():
        mb.mb_stack_step(stack, kvs, cb, x, y, s)
        mb.mb_sample_greedy(y, T, rows, T, d, sh.rms_eps, g_final, w_lm, vocab, yw, logits, ids, s)
        mb.mb_embed(table, vocab, d, ids, T, x, s)

    for _ in range(warmup):
        one_step()
    torch.cuda.synchronize()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush(i & 0xFF)
        e0[i].record(stream)
        one_step()
        e1[i].record(stream)
    torch.cuda.synchronize()
    mb.mb_device_status(layers[0].handle, s)
    mb.mb_device_status(None, s)
    ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / steps
    # the sampling part alone (final norm + LM head + argmax), L2 flushed
    h0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    h1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush(i & 0xFF)
        h0[i].record(stream)
        mb.mb_sample_greedy(y, T, rows, T, d, sh.rms_eps, g_final, w_lm, vocab, yw, logits, ids, s)
        h1[i].record(stream)
    torch.cuda.synchronize()
    mb.mb_device_status(None, s)
    head_ms = sum(a.elapsed_time(b) for a, b in zip(h0, h1)) / steps
    head_bytes = vocab * d * 2 + T * vocab * 2
    mb.mb_stack_destroy(stack)
    for L in layers:
        L.close()
    del keep, shared_pool
    torch.cuda.empty_cache()
    return {"workload": f"llama3_8b_stack32_generate_b{n_decodes}", "layers": nl, "vocab": vocab,
            "decodes": T, "ms_per_step": round(ms, 4), "output_tokens_per_s": round(T / (ms / 1e3), 1),
            "sample_ms": round(head_ms, 4), "sample_share": round(head_ms / ms, 4),
            "sample_gbs": round(head_bytes / (head_ms / 1e3) / 1e9, 1),
            "sample_frac_hbm": round(head_bytes / (head_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "batch": "the same decode rows every step (positions held: timing-equivalent)",
            "kv_pool": "one physical pool shared by all layers" if shared else "one pool per layer"}


def to_dev(bits, torch):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).cuda()


def kernel_table(alg: dict, kern_ms: dict, ksteps: int, peaks: dict) -> dict:
    """Per-kernel time and achieved rate against its roofline (mean per launch)."""
    kernels = {}
    for name, total in kern_ms.items():
        ms = total / max(1, ksteps)
        bound, work = alg[name]
        if bound == "mixed":
            fl, by = work
            serial = fl / (peaks["bf16_tflops"] * 1e12) + by / (peaks["hbm_gbs"] * 1e9)
            overlap = max(fl / (peaks["bf16_tflops"] * 1e12), by / (peaks["hbm_gbs"] * 1e9))
            kernels[name] = {"ms": round(ms, 5), "chunk_tflops_over_launch": round(fl / (ms / 1e3) / 1e12, 1),
                             "decode_gbs_over_launch": round(by / (ms / 1e3) / 1e9, 1),
                             "roofline_ms_serial": round(serial * 1e3, 5),
                             "roofline_ms_overlapped": round(overlap * 1e3, 5),
                             "frac": round(serial * 1e3 / ms, 4) if ms > 0 else None}
            continue
        if ms <= 0 or work <= 0:
            kernels[name] = {"ms": round(ms, 5)}
            continue
        if bound == "tensor":
            ach = work / (ms / 1e3) / 1e12
            kernels[name] = {"ms": round(ms, 5), "tflops": round(ach, 1),
                             "frac_burst": round(ach / peaks["bf16_tflops"], 4),
                             "frac_sustained": round(ach / peaks["bf16_tflops_sustained"], 4)}
        else:
            ach = work / (ms / 1e3) / 1e9
            kernels[name] = {"ms": round(ms, 5), "gbs": round(ach, 1), "frac": round(ach / peaks["hbm_gbs"], 4)}
    return kernels


def roofline_obj(kernel: str, bound: str, work: float, ms: float, peaks: dict, peak_kind: str, traffic_key: str,
                 peak_which: str = "bf16_tflops") -> dict:
    if bound == "tensor":
        ach = work / (ms / 1e3) / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": round(ach, 2), "peak": peaks[peak_which],
                "unit": "TFLOP/s", "frac": round(ach / peaks[peak_which], 4), "traffic": ncu_traffic(traffic_key),
                "algorithmic_per_launch": work, "launch_ms": round(ms, 5),
                "peak_kind": f"{peak_kind} bf16 {'burst' if peak_which == 'bf16_tflops' else 'sustained'}"}
    ach = work / (ms / 1e3) / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": round(ach, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": ncu_traffic(traffic_key),
            "algorithmic_per_launch": work, "launch_ms": round(ms, 5), "peak_kind": f"{peak_kind} HBM copy"}


GEMM_NAMES = ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down")


def layer_measurements(mb, torch, wl, steps: int, warmup: int, peaks: dict, peak_kind: str, pg=None, world: int = 1,
                       local: int = 0, clocks: bool = False) -> dict:
    """One layer's mb_step over one batch: the step time (per-step events,
    L2 flushed between steps), per-kernel times from a second pass with events
    around every launch, rooflines, and the end-to-end figure with host
    buffers."""
    wb, x, batch, pool = W.materialize(wl, unit_gains=True)
    T = batch.num_tokens
    dw = {k: to_dev(v, torch) for k, v in wb.items()}
    dpool = to_dev(pool.reshape(-1), torch)
    layer = mb.Layer(wl.shape.as_dict(), dw, T, pool.shape[0], kv_buf=dpool)
    cb = mb.Batch.of(batch)
    dx = to_dev(x, torch)
    dy = torch.empty_like(dx)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    flush = L2Flush(torch)
    for _ in range(warmup):
        flush(1)
        layer.step(cb, dx, dy, s)
    mb.mb_device_status(layer.handle, s)
    launches_per_step = mb.mb_layer_last_launches(layer.handle)
    # timed: no per-kernel events here, since an event between two kernels
    # would stop the next one from starting its set-up early (PDL)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(pg)
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if clocks else None
    wall0 = time.perf_counter()
    for i in range(steps):
        flush(i & 0xFF)
        ev0[i].record(stream)
        layer.step(cb, dx, dy, s)
        ev1[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(pg)
    clk = sampler.stop() if sampler else None
    mb.mb_device_status(layer.handle, s)
    step_ms_local = sum(a.elapsed_time(b) for a, b in zip(ev0, ev1)) / steps
    step_ms, value = replica_throughput(pg, world, T, step_ms_local)
    # per-kernel times: a second pass with events around every launch
    n_kt = max(1, min(steps, 200))
    mb.mb_layer_set_timing(layer.handle, True)
    for i in range(n_kt):
        flush(i & 0xFF)
        layer.step(cb, dx, dy, s)
    torch.cuda.synchronize()
    mb.mb_device_status(layer.handle, s)
    kern_ms, ksteps = mb.mb_layer_timing(layer.handle)
    mb.mb_layer_set_timing(layer.handle, False)
    alg = algorithmic(wl.shape, batch)
    kernels = kernel_table(alg, kern_ms, ksteps, peaks)
    dom = max((k for k in kern_ms if alg[k][0] != "mixed"), key=lambda k: kern_ms[k])
    roofline = roofline_obj(dom, alg[dom][0], alg[dom][1], kern_ms[dom] / max(1, ksteps), peaks, peak_kind, dom)
    gemm_flops = sum(alg[n][1] for n in GEMM_NAMES)
    gemm_ms = sum(kern_ms[n] for n in GEMM_NAMES) / max(1, ksteps)
    roof_ms = 0.0
    for name, (bnd, wk) in alg.items():
        if bnd == "mixed":
            roof_ms += (wk[0] / (peaks["bf16_tflops"] * 1e12) + wk[1] / (peaks["hbm_gbs"] * 1e9)) * 1e3
        elif bnd == "tensor":
            roof_ms += wk / (peaks["bf16_tflops"] * 1e12) * 1e3
        else:
            roof_ms += wk / (peaks["hbm_gbs"] * 1e9) * 1e3
    weight_bytes = 2.0 * sum(int(np.prod(v.shape)) for v in wb.values())
    roof_ms = max(roof_ms, weight_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3)
    # end to end through the public API with host buffers
    n_e2e = max(1, min(steps, 200))
    xh = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    torch.cuda.synchronize()
    for i in range(n_e2e):
        flush(i & 0xFF)
        e0[i].record(stream)
        dx.copy_(xh, non_blocking=True)
        layer.step(cb, dx, dy, s)
        yh.copy_(dy, non_blocking=True)
        e1[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms, e2e_value = replica_throughput(pg, world, T, sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / n_e2e)
    upload = mb.mb_layer_last_upload_bytes(layer.handle)
    # pofe.ai's step-time model with GB300 peaks, as an analytic comparator
    from mixed_prefill_decode_gb300 import step_model as SM
    sh = wl.shape
    n_params = sum(int(np.prod(v.shape)) for k, v in wb.items() if k.startswith("w_"))
    gb300 = SM.Machine(flops=peaks["bf16_tflops_sustained"] * 1e12, bandwidth=peaks["hbm_gbs"] * 1e9, t_iter=0.0)
    model = SM.Model(n_params=n_params, kappa=sh.kv_bytes_per_token, d_model=sh.d_model, n_layers=1)
    qo = batch.qo_len()
    c = batch.cached()
    chunks = [(int(qo[r]), int(c[r])) for r in range(batch.num_reqs) if qo[r] > 1]
    decs = [int(c[r]) for r in range(batch.num_reqs) if qo[r] == 1]
    model_ms = SM.iteration_time(gb300, model, chunks, decs) * 1e3
    layer.close()
    del dw, dpool
    return {"workload": wl.name, "tokens_per_step": T, "ms_per_step": round(step_ms, 5),
            "tokens_per_s": round(value, 1), "value": value, "step_ms": step_ms,
            "requests": batch.num_reqs, "decodes": int(np.sum(qo == 1)),
            "chunk_rows": int(np.sum(qo[qo > 1])), "chunk_prefix": [int(v) for v in c[qo > 1]],
            "roofline": roofline, "kernels": kernels,
            "gemm": {"tflops": round(gemm_flops / (gemm_ms / 1e3) / 1e12, 1),
                     "frac_burst": round(gemm_flops / (gemm_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                     "frac_sustained": round(gemm_flops / (gemm_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"],
                                             4)},
            "roofline_step_ms": round(roof_ms, 5), "step_model_ms": round(model_ms, 5),
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(x.nbytes + upload),
                    "d2h_bytes_per_step": int(x.nbytes), "ms_per_step": round(e2e_ms, 5)},
            "gpu_launches": int(launches_per_step * steps), "clocks": clk, "wall_s_timed_region": round(wall, 4),
            "x_bits": x, "oracle_wl": wl}


def layer_cpu_baseline(wl, target_s: float = 15.0, layers: int = 1) -> dict:
    """The oracle timed on a bounded sample of a layer workload (rank 0)."""
    OL, w64, x64, b2, pool64 = oracle_inputs(wl)
    nd, nc = calibrate_sample(OL, wl, w64, x64, b2, pool64, target_s)
    smp = sub_batch(b2, x64, nd, nc)
    tok = int(smp[0][-1])
    dt = time_oracle_step(OL, wl.shape, w64, pool64, *smp)
    return {"value": tok / (dt * layers), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"one oracle layer step over {nd} decode rows and {nc} chunk rows ({tok} tokens) of "
                      f"{wl.name}, float64 NumPy, {dt:.1f} s"}


# ------------------------------------------------------ stack over a prompt
def stack_cpu_sample(sw: "W.PromptSweep", target_s: float, steps: int = 1, warmup: int = 0):
    """The oracle on a bounded sample of one prompt-sweep step: the first nd
    decode rows (their whole contexts) and the first nc rows of the chunk at
    the middle of the prompt (prefix 16,384), one layer, float64 NumPy.  The
    sample grows until one layer step takes about target_s.  Returns the
    tokens of the sample, the mean step time over `steps` timed layer steps,
    and a description; the stack's rate is tokens / (n_layers x time),
    extrapolated from one layer."""
    from oracle import layer as OL
    sh = sw.shape
    wb = W.make_weights(sh, sw.seed + 5, unit_gains=True)
    w64 = OL.weights_to_f64(wb)
    del wb
    prefix = sw.prompt // 2

    def sample(nd, nc):
        reqs = [(c, 1) for c in sw.decodes[:nd]] + ([(prefix, nc)] if nc else [])
        batch, num_pages = W.make_batch(reqs, sw.seed + 6, spare_pages=0)
        x = OL.bf16_bits_to_f64(W.make_embeddings(batch.num_tokens, sh.d_model, sw.seed + 7))
        pool = OL.bf16_bits_to_f64(W.make_kv_pool(sh, num_pages, batch, sw.seed + 8))
        return batch, x, pool

    def run(batch, x, pool):
        t = time.perf_counter()
        OL.layer_step(sh.as_dict(), w64, pool, batch.qo_indptr, batch.kv_len, batch.bt_indptr, batch.bt, x)
        return time.perf_counter() - t

    nd_all, nc_all = len(sw.decodes), sw.chunk
    frac = 1.0 / 64
    while True:
        nd, nc = max(1, int(round(nd_all * frac))), int(round(nc_all * frac))
        b, x, pool = sample(nd, nc)
        dt = run(b, x, pool)
        if dt >= 0.5 * target_s or frac >= 1.0:
            break
        frac = min(1.0, frac * min(4.0, max(1.5, target_s / max(dt, 1e-6))))
    for _ in range(warmup):
        run(b, x, pool)
    times = [run(b, x, pool) for _ in range(steps)] if steps > 1 or warmup else [dt]
    t = sum(times) / len(times)
    desc = (f"oracle layer step over {nd} of the {nd_all} decode rows (whole contexts) and the first {nc} rows of "
            f"the chunk at prefix {prefix} ({b.num_tokens} tokens) of {sw.name}, float64 NumPy, {t:.2f} s per "
            f"layer; the {sw.n_layers}-layer rate is extrapolated from one layer")
    return b.num_tokens, t, desc


def stack_layers(mb, torch, sh, n_layers: int, num_pages: int, max_tokens: int, wseed: int, pseed: int):
    layers, keep = [], []
    for l in range(n_layers):
        dw = W.device_weights(sh, wseed + l)
        dpool = W.device_kv_pool(sh, num_pages, pseed + l)
        layers.append(mb.Layer(sh.as_dict(), dw, max_tokens, num_pages, kv_buf=dpool))
        keep.append((dw, dpool))
    return layers, keep


def prompt_sweep_kernels(mb, torch, sw, full, layer, peaks, peak_kind, reps: int = 3) -> dict:
    """Per-kernel times of one layer (mb_step with events around every launch,
    L2 flushed) at every chunk position of the sweep: the mixed step, the same
    chunk alone and the decodes alone.  The roofline goes to the kernel with
    the most time over the whole prompt; for the attention launch, the chunk
    tiles' rate is taken from the chunk-alone launches (where no decode rows
    share the grid)."""
    sh = sw.shape
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    flush = L2Flush(torch)

    def timed(batch):
        cb = mb.Batch.of(batch)
        T = batch.num_tokens
        x = torch.randn((T, sh.d_model), device="cuda").to(torch.bfloat16)
        y = torch.empty_like(x)
        layer.step(cb, x, y, s)
        mb.mb_layer_set_timing(layer.handle, True)
        for i in range(reps):
            flush(i & 0xFF)
            layer.step(cb, x, y, s)
        torch.cuda.synchronize()
        km, n = mb.mb_layer_timing(layer.handle)
        mb.mb_layer_set_timing(layer.handle, False)
        mb.mb_device_status(layer.handle, s)
        return {k: v / max(1, n) for k, v in km.items()}

    tot = {}
    work = {}
    chunk_flops = chunk_ms = 0.0
    per_pos = []
    for k in range(sw.steps):
        b = sw.batch_at(k, full)
        km = timed(b)
        alg = algorithmic(sh, b)
        for name, ms in km.items():
            tot[name] = tot.get(name, 0.0) + ms
            bound, wk = alg[name]
            if bound == "mixed":
                f0, b0 = work.get(name, (0.0, 0.0))
                work[name] = (f0 + wk[0], b0 + wk[1])
            else:
                work[name] = work.get(name, 0.0) + wk
        bc = sw.batch_at(k, full, with_decodes=False)
        kc = timed(bc)
        fl = algorithmic(sh, bc)["attention"][1][0]
        chunk_flops += fl
        chunk_ms += kc["attention"]
        per_pos.append({"prefix": k * sw.chunk, "layer_ms": round(sum(km.values()), 4),
                        "attention_ms": round(km["attention"], 4), "chunk_alone_attention_ms": round(kc["attention"], 4),
                        "chunk_tflops": round(fl / (kc["attention"] / 1e3) / 1e12, 1)})
    bd = sw.batch_at(0, full, with_chunk=False)
    kd = timed(bd)
    dec_bytes = float(np.sum(bd.kv_len)) * sh.n_kv_heads * sh.head_dim * 4
    n = sw.steps
    alg_mean = {}
    for name, wk in work.items():
        bound = "mixed" if isinstance(wk, tuple) else algorithmic(sh, sw.batch_at(0, full))[name][0]
        alg_mean[name] = (bound, (wk[0] / n, wk[1] / n) if bound == "mixed" else wk / n)
    kernels = kernel_table(alg_mean, {k: v / n for k, v in tot.items()}, 1, peaks)
    dom = max(tot, key=lambda k: tot[k])
    if dom == "attention":
        roofline = roofline_obj("attention_kernel chunk tiles (chunk alone, mean over the 16 prefixes)", "tensor",
                                chunk_flops / n, chunk_ms / n, peaks, peak_kind, "attention_chunk")
    else:
        bound, wk = alg_mean[dom]
        roofline = roofline_obj(dom, bound, wk, tot[dom] / n, peaks, peak_kind, dom)
    gemm_flops = sum(alg_mean[g][1] for g in GEMM_NAMES)
    gemm_ms = sum(tot[g] for g in GEMM_NAMES) / n
    share = {k: round(v / sum(tot.values()), 4) for k, v in sorted(tot.items(), key=lambda kv: -kv[1])}
    return {"roofline": roofline, "kernels": kernels, "share_of_layer_time": share, "dominant": dom,
            "gemm": {"tflops": round(gemm_flops / (gemm_ms / 1e3) / 1e12, 1),
                     "frac_burst": round(gemm_flops / (gemm_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                     "frac_sustained": round(gemm_flops / (gemm_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"],
                                             4)},
            "chunk_attention": {"tflops": round(chunk_flops / (chunk_ms / 1e3) / 1e12, 1),
                                "frac_burst": round(chunk_flops / (chunk_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                                "per_prefix": per_pos},
            "decode_attention_alone": {"decodes": len(sw.decodes), "kv_bytes": dec_bytes,
                                       "ms": round(kd["attention"], 5),
                                       "gbs": round(dec_bytes / (kd["attention"] / 1e3) / 1e9, 1),
                                       "frac": round(dec_bytes / (kd["attention"] / 1e3) / 1e9 / peaks["hbm_gbs"], 4)},
            "per_layer": "layer 0 alone (mb_step), events around every launch, L2 flushed, "
                         f"{reps} steps per position"}


def run_stack_headline(args, rank: int, world: int, local: int, pg, mb, torch, peaks, peak_kind):
    sw = W.qwen3_14b_prompt_sweep()
    sh = sw.shape
    full, num_pages = sw.layout()
    batches = [sw.batch_at(k, full) for k in range(sw.steps)]
    cbs = [mb.Batch.of(b) for b in batches]
    T = batches[0].num_tokens
    assert all(b.num_tokens == T for b in batches)
    layers, keep = stack_layers(mb, torch, sh, sw.n_layers, num_pages, T, sw.seed + 100, sw.seed + 200)
    stack = mb.mb_stack_create([L.handle for L in layers], True)
    kvs = [L.kv for L in layers]
    x = W.make_embeddings(T, sh.d_model, sw.seed + 2)
    dx = to_dev(x, torch)
    dy = torch.empty_like(dx)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    flush = L2Flush(torch)

    def step(i):
        mb.mb_stack_step(stack, kvs, cbs[i % sw.steps], dx, dy, s)

    # set-up: one pass over every chunk position (graph capture, descriptor
    # buffers), then the warm-up steps; step i takes chunk i mod 16
    for k in range(sw.steps):
        step(k)
    mb.mb_device_status(layers[0].handle, s)
    for i in range(args.warmup):
        flush(i & 0xFF)
        step(i)
    mb.mb_device_status(layers[0].handle, s)
    launches_per_step = mb.mb_stack_last_launches(stack)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(pg)
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    wall0 = time.perf_counter()
    for j in range(args.steps):
        flush(j & 0xFF)
        ev0[j].record(stream)
        step(args.warmup + j)
        ev1[j].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(pg)
    clk = clocks.stop() if clocks else None
    mb.mb_device_status(layers[0].handle, s)
    times = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    step_ms_local = sum(times) / args.steps
    step_ms, value = replica_throughput(pg, world, T, step_ms_local)
    positions = [(args.warmup + j) % sw.steps for j in range(args.steps)]

    # the whole prompt once more, one step per chunk position (untimed for
    # the headline): its prefill time beside the 96 decodes is the prompt's
    # time to first token
    p0 = [torch.cuda.Event(enable_timing=True) for _ in range(sw.steps)]
    p1 = [torch.cuda.Event(enable_timing=True) for _ in range(sw.steps)]
    torch.cuda.synchronize()
    for k in range(sw.steps):
        flush(k & 0xFF)
        p0[k].record(stream)
        step(k)
        p1[k].record(stream)
    torch.cuda.synchronize()
    mb.mb_device_status(layers[0].handle, s)
    pos_ms = [a.elapsed_time(b) for a, b in zip(p0, p1)]

    # end to end through the public API with host buffers: per step the H2D
    # of the step's inputs (and the library's descriptor upload), the stack,
    # the D2H of its output
    n_e2e = max(1, min(args.steps, 32))
    xh = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    torch.cuda.synchronize()
    for i in range(n_e2e):
        flush(i & 0xFF)
        e0[i].record(stream)
        dx.copy_(xh, non_blocking=True)
        step(args.warmup + i)
        yh.copy_(dy, non_blocking=True)
        e1[i].record(stream)
    torch.cuda.synchronize()
    mb.mb_device_status(layers[0].handle, s)
    e2e_ms, e2e_value = replica_throughput(pg, world, T, sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / n_e2e)
    upload = mb.mb_layer_last_upload_bytes(layers[0].handle)
    mb.mb_stack_destroy(stack)

    # per-kernel times and the roofline: layer 0 alone at every position
    kern = prompt_sweep_kernels(mb, torch, sw, full, layers[0], peaks, peak_kind) if rank == 0 else None
    for L in layers:
        L.close()
    del keep, layers
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok, t, desc = stack_cpu_sample(sw, 15.0)
        cpu = {"value": tok / (sw.n_layers * t), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": desc}

    aux = {}
    if rank == 0 and not args.no_aux:
        aux = run_aux(mb, torch, peaks, peak_kind)
    if rank != 0:
        return
    prefill_ms = sum(pos_ms)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) embeddings and KV, "
                                                      "N(0,0.02) random-init weights, generated on the device)",
        "config": {"workload": sw.name, "layers": sw.n_layers, "tokens_per_step": T, "decodes": len(sw.decodes),
                   "decode_context": "log-uniform in [1024, 8192] (positions held)", "prompt": sw.prompt,
                   "chunk": sw.chunk, "step_i_chunk_prefix": "2048 * (i mod 16)",
                   "timed_chunk_prefixes": sorted(set(p * sw.chunk for p in positions)),
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                   "kv_pool": "one paged pool per layer in HBM", "cuda_graph": "one graph for the 40 layers",
                   "l2": "flushed between timed steps (256 MiB written, then 256 MiB read, leaving L2 clean); inputs larger than L2 (26 GB of weights, "
                         "up to 1.9 GB of KV read per layer)",
                   "wall_s_timed_region": round(wall, 4)},
        "prompt": {"prefill_ms_beside_decodes": round(prefill_ms, 3),
                   "tokens_per_s": round(sw.steps * T / (prefill_ms / 1e3), 1),
                   "prompt_tokens_per_s": round(sw.prompt / (prefill_ms / 1e3), 1),
                   "step_ms_by_prefix": {str(k * sw.chunk): round(v, 3) for k, v in enumerate(pos_ms)},
                   "note": "one pass of the 16 chunk positions after the timed region; its sum is the prompt's "
                           "time to first token beside 96 decodes"},
        "roofline": kern["roofline"] if kern else None,
        "kernels": kern["kernels"] if kern else None,
        "gemm": kern["gemm"] if kern else None,
        "decode_attn_sweep": kern["decode_attention_alone"] if kern else None,
        "prompt_sweep_per_layer": {k: v for k, v in kern.items() if k not in ("roofline", "kernels")} if kern else None,
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT,
                "h2d_bytes_per_step": int(x.nbytes + upload), "d2h_bytes_per_step": int(x.nbytes),
                "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clk,
        "peaks": {"kind": peak_kind, **peaks},
        **aux,
    }
    print(json.dumps(line), flush=True)


def run_aux(mb, torch, peaks, peak_kind) -> dict:
    """Auxiliary lines: the Llama-3-8B-shaped layer at 576 tokens with its
    per-kernel rooflines, decode attention alone, token generation through
    the 32-layer stack, and the Qwen3-14B piggyback points.  A part that
    fails records its error; the headline still prints."""
    out = {}

    def guard(key, fn):
        try:
            out[key] = fn()
        except Exception as e:   # recorded, not raised
            out[key] = {"error": f"{type(e).__name__}: {e}"[:300]}
        torch.cuda.empty_cache()

    def llama_layer():
        r = layer_measurements(mb, torch, W.llama3_8b_mixed(), 200, 10, peaks, peak_kind)
        r.pop("x_bits")
        r.pop("oracle_wl")
        r.pop("value")
        r.pop("step_ms")
        return r

    guard("llama3_8b_T576", llama_layer)
    guard("decode_attn", lambda: decode_only_attention(mb, torch, peaks))
    guard("generate_llama3_8b_32", lambda: generation_step_time(mb, torch, peaks))
    guard("qwen3_14b_piggyback", lambda: qwen3_14b_piggyback(mb, torch))
    return out


def run_mine(args, rank: int, world: int, local: int, pg):
    import torch
    from mixed_prefill_decode_gb300 import build as B
    from mixed_prefill_decode_gb300 import binding as mb

    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        B.build()
    barrier(pg)
    B.build()
    peaks, peak_kind = load_peaks()
    if args.workload == HEADLINE:
        return run_stack_headline(args, rank, world, local, pg, mb, torch, peaks, peak_kind)
    wl = workload_by_name(args.workload)
    r = layer_measurements(mb, torch, wl, args.steps, args.warmup, peaks, peak_kind, pg, world, local,
                           clocks=rank == 0)
    cpu = layer_cpu_baseline(wl) if rank == 0 and world == 1 and not args.no_cpu_baseline else None
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(r["value"], 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["step_ms"], 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) embeddings and KV prefix, "
                                                      "N(0,0.02) random-init weights)",
        "config": {"workload": wl.name, "tokens_per_step": r["tokens_per_step"], "requests": r["requests"],
                   "decodes": r["decodes"], "chunk_rows": r["chunk_rows"], "chunk_prefix": r["chunk_prefix"],
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                   "l2": "flushed between timed steps (256 MiB written, then 256 MiB read, leaving L2 clean); step time = per-step CUDA events",
                   "wall_s_timed_region": r["wall_s_timed_region"]},
        "roofline": r["roofline"], "kernels": r["kernels"], "gemm": r["gemm"],
        "roofline_step_ms": r["roofline_step_ms"], "step_model_ms": r["step_model_ms"],
        "cpu_baseline": cpu, "e2e": r["e2e"], "gpu_launches": r["gpu_launches"], "clocks": r["clocks"],
        "peaks": {"kind": peak_kind, **peaks},
    }
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """Token budget C x decode batch b on the 32-layer Llama-3-8B-shaped stack
    (compute/bandwidth crossover): tokens/s per point, with the pofe.ai step
    model (GB300 peaks) beside each."""
    import torch
    from mixed_prefill_decode_gb300 import build as B
    from mixed_prefill_decode_gb300 import binding as mb
    from mixed_prefill_decode_gb300 import step_model as SM
    B.build()
    peaks, _ = load_peaks()
    sh = W.LLAMA3_8B
    weights = [W.device_weights(sh, 5100 + l) for l in range(32)]
    n_params = 32 * (sh.qkv_dim * sh.d_model + sh.d_model * sh.n_q_heads * sh.head_dim + 3 * sh.d_ff * sh.d_model)
    gb300 = SM.Machine(flops=peaks["bf16_tflops_sustained"] * 1e12, bandwidth=peaks["hbm_gbs"] * 1e9, t_iter=0.0)
    model = SM.Model(n_params=n_params, kappa=32 * sh.kv_bytes_per_token, d_model=sh.d_model, n_layers=32)
    free_budget = torch.cuda.mem_get_info()[0] - (24 << 30)
    for C in (256, 512, 1024, 2048, 4096, 8192):
        for b in (1, 16, 64, 256):
            if C <= b:
                continue
            wl, nl = W.llama3_8b_stack(C, b)
            r = stack_step_time(mb, torch, wl, nl, steps=5, warmup=2, share_pool_bytes=free_budget,
                                weights=weights)
            qo = np.array([q for _, q in wl.reqs])
            cs = np.array([c for c, _ in wl.reqs])
            chunks = [(int(q), int(c)) for c, q in wl.reqs if q > 1]
            decs = [int(c) for c, q in wl.reqs if q == 1]
            r.update({"budget": C, "decodes": b,
                      "step_model_ms": round(SM.iteration_time(gb300, model, chunks, decs) * 1e3, 4)})
            print(json.dumps(r), flush=True)


def run_partition(args):
    """SM partition for decode attention (row f1: ConfluxServe gives decode
    "just enough SMs" for most of its bandwidth).  (1) Decode-only attention
    (Qwen3-14B-shaped, 16 x 8,192 tokens) against the cap on decode-worker
    CTAs; (2) the Llama-3-8B-shaped step (T = 576) with each cap against the
    one-grid default, where workers take every SM the chunk tiles leave;
    (3) the decode and chunk rows as two micro-batches on two streams with
    SM caps (decode attention beside the other micro-batch's GEMMs), on the
    Llama-3-8B step and the Qwen3-14B step with 2,200 piggybacked tokens.  One
    JSON line per point."""
    import torch
    from mixed_prefill_decode_gb300 import build as B
    from mixed_prefill_decode_gb300 import binding as mb
    B.build()
    peaks, _ = load_peaks()
    s = torch.cuda.current_stream()
    flush = L2Flush(torch)

    def make(wl):
        wb, x, batch, pool = W.materialize(wl, unit_gains=True)
        dw = {k: to_dev(v, torch) for k, v in wb.items()}
        dpool = to_dev(pool.reshape(-1), torch)
        layer = mb.Layer(wl.shape.as_dict(), dw, batch.num_tokens, pool.shape[0], kv_buf=dpool)
        dx = to_dev(x, torch)
        return layer, mb.Batch.of(batch), dx, torch.empty_like(dx), batch

    def kernel_ms(layer, cb, dx, dy, n=20):
        for _ in range(3):
            layer.step(cb, dx, dy, s.cuda_stream)
        mb.mb_layer_set_timing(layer.handle, True)
        for i in range(n):
            flush(i & 0xFF)
            layer.step(cb, dx, dy, s.cuda_stream)
        km, k = mb.mb_layer_timing(layer.handle)
        mb.mb_layer_set_timing(layer.handle, False)
        mb.mb_device_status(layer.handle, s.cuda_stream)
        return {name: v / max(1, k) for name, v in km.items()}

    wl = W.qwen3_14b_mixed(0)
    layer, cb, dx, dy, batch = make(wl)
    by = float(np.sum(batch.kv_len)) * wl.shape.n_kv_heads * wl.shape.head_dim * 4
    for cap in (8, 16, 24, 32, 48, 64, 96, 128, 0):
        mb.mb_layer_set_decode_sms(layer.handle, cap)
        km = kernel_ms(layer, cb, dx, dy)
        ms = km["attention"] + km["attn_merge"]
        print(json.dumps({"kind": "decode_only", "workload": wl.name, "decode_sms": cap or "all",
                          "ms": round(ms, 5), "gbs": round(by / (ms / 1e3) / 1e9, 1),
                          "frac": round(by / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)}), flush=True)
    layer.close()

    wl = W.llama3_8b_mixed()
    layer, cb, dx, dy, batch = make(wl)
    T = batch.num_tokens
    for cap in (16, 24, 32, 48, 64, 88, 0):
        mb.mb_layer_set_decode_sms(layer.handle, cap)
        km = kernel_ms(layer, cb, dx, dy)
        for _ in range(3):
            layer.step(cb, dx, dy, s.cuda_stream)
        n = 200
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        torch.cuda.synchronize()
        for i in range(n):
            flush(i & 0xFF)
            e0[i].record(s)
            layer.step(cb, dx, dy, s.cuda_stream)
            e1[i].record(s)
        torch.cuda.synchronize()
        mb.mb_device_status(layer.handle, s.cuda_stream)
        ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / n
        print(json.dumps({"kind": "mixed_step", "workload": wl.name, "decode_sms": cap or "all (one grid)",
                          "ms_per_step": round(ms, 5), "tokens_per_s": round(T / (ms / 1e3), 1),
                          "attention_ms": round(km["attention"] + km["attn_merge"], 5)}), flush=True)
    layer.close()
    # decode attention beside the GEMMs of another micro-batch, on two streams
    for wl in (W.llama3_8b_mixed(), W.qwen3_14b_mixed(2200)):
        for line in two_stream_micro_batches(mb, torch, wl):
            print(json.dumps(line), flush=True)


def two_stream_micro_batches(mb, torch, wl, shares=(6, 4, 3), steps: int = 50) -> list:
    """Row f1's other half: the decode rows and the chunk rows of one batch as
    two micro-batches, stepped by two layers (same weights and KV pool, GEMM
    workspaces of their own) on two streams at once, the decode micro-batch
    on sms/share SMs (its GEMMs and decode workers) beside the chunk
    micro-batch's GEMMs on the rest, so that decode attention runs beside the
    other micro-batch's GEMMs (ConfluxServe's overlap).  Against the one-grid
    mixed step and the two micro-batches one after the other.  L2 flushed
    between steps; per-step events on the launching stream."""
    wb, x, batch, pool = W.materialize(wl, unit_gains=True)
    sh = wl.shape
    qo = batch.qo_len()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count

    def sub(rs):
        rows = np.concatenate([np.arange(batch.qo_indptr[r], batch.qo_indptr[r + 1]) for r in rs])
        q = np.cumsum([0] + [int(qo[r]) for r in rs]).astype(np.int32)
        tabs = [batch.bt[batch.bt_indptr[r]:batch.bt_indptr[r + 1]] for r in rs]
        bti = np.cumsum([0] + [len(t) for t in tabs]).astype(np.int32)
        return rows, W.Batch(q, batch.kv_len[rs].astype(np.int32), bti, np.concatenate(tabs).astype(np.int32))

    parts = {"decode": sub([r for r in range(batch.num_reqs) if qo[r] == 1]),
             "chunk": sub([r for r in range(batch.num_reqs) if qo[r] > 1])}
    dw = {k: to_dev(v, torch) for k, v in wb.items()}
    dpool = to_dev(pool.reshape(-1), torch)
    main = torch.cuda.current_stream()
    flush = L2Flush(torch)
    full = mb.Layer(sh.as_dict(), dw, batch.num_tokens, pool.shape[0], kv_buf=dpool)
    L = {n: mb.Layer(sh.as_dict(), dw, b.num_tokens, pool.shape[0], kv_buf=dpool) for n, (r, b) in parts.items()}
    ws = {n: torch.zeros(mb.mb_gemm_workspace_bytes(), dtype=torch.uint8, device="cuda") for n in parts}
    for n in parts:
        mb.mb_layer_set_gemm_workspace(L[n].handle, ws[n])
    cb = {n: mb.Batch.of(b) for n, (r, b) in parts.items()}
    xs = {n: to_dev(x[r], torch) for n, (r, b) in parts.items()}
    ys = {n: torch.empty_like(xs[n]) for n in parts}
    st = {n: torch.cuda.Stream() for n in parts}
    xf, yf, cbf = to_dev(x, torch), None, mb.Batch.of(batch)
    yf = torch.empty_like(xf)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush(i & 0xFF)
            e0[i].record(main)
            fn()
            e1[i].record(main)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / steps

    def one_grid():
        full.step(cbf, xf, yf, main.cuda_stream)

    def serial():
        for n in parts:
            L[n].step(cb[n], xs[n], ys[n], main.cuda_stream)

    def overlapped():
        start = torch.cuda.Event()
        start.record(main)
        ends = []
        for n in ("decode", "chunk"):
            st[n].wait_event(start)
            L[n].step(cb[n], xs[n], ys[n], st[n].cuda_stream)
            e = torch.cuda.Event()
            e.record(st[n])
            ends.append(e)
        for e in ends:
            main.wait_event(e)

    out = []
    T = batch.num_tokens
    ms = timed(one_grid)
    out.append({"kind": "micro_batches", "workload": wl.name, "schedule": "one grid (mixed step)", "ms": round(ms, 5),
                "tokens_per_s": round(T / (ms / 1e3), 1)})
    for n in parts:
        mb.mb_layer_set_gemm_sms(L[n].handle, 0)
        mb.mb_layer_set_decode_sms(L[n].handle, 0)
    ms = timed(serial)
    out.append({"kind": "micro_batches", "workload": wl.name, "schedule": "decode then chunk micro-batch, one stream",
                "ms": round(ms, 5), "tokens_per_s": round(T / (ms / 1e3), 1)})
    for share in shares:
        d = sms // share
        mb.mb_layer_set_gemm_sms(L["decode"].handle, d)
        mb.mb_layer_set_decode_sms(L["decode"].handle, d)
        mb.mb_layer_set_gemm_sms(L["chunk"].handle, sms - d)
        ms = timed(overlapped)
        out.append({"kind": "micro_batches", "workload": wl.name,
                    "schedule": f"two streams: decode micro-batch on {d} SMs, chunk micro-batch GEMMs on {sms - d}",
                    "ms": round(ms, 5), "tokens_per_s": round(T / (ms / 1e3), 1)})
    for n in parts:
        mb.mb_device_status(L[n].handle, st[n].cuda_stream)
    mb.mb_device_status(full.handle, main.cuda_stream)
    full.close()
    for n in parts:
        L[n].close()
    return out


def run_budget(args):
    """Budget selection on GB300 (pofe.ai "Chunked prefill", "Tuning knobs"):
    time the 32-layer Llama-3-8B-shaped stack over token budgets and decode
    counts, fit the step-time model t = t0 + a T + b KVd + c pairs, take the
    largest budget within each TBT target, and replay seeded load through the
    packer on the fitted model (p99 TBT / TTFT, goodput at p99 TBT <= 50 ms and
    TTFT <= 1 s).  One JSON line per profiled point, then the fit, the choices
    and the load tests."""
    import torch
    from mixed_prefill_decode_gb300 import build as B
    from mixed_prefill_decode_gb300 import binding as mb
    from mixed_prefill_decode_gb300 import budget as BU
    B.build()
    sh = W.LLAMA3_8B
    weights = [W.device_weights(sh, 5100 + l) for l in range(32)]
    free_budget = torch.cuda.mem_get_info()[0] - (24 << 30)
    batches, secs, curve = [], [], {}
    for C in (256, 512, 1024, 2048, 4096, 8192):
        for b in (16, 64, 256):
            if C <= b:
                continue
            wl, nl = W.llama3_8b_stack(C, b)
            r = stack_step_time(mb, torch, wl, nl, steps=5, warmup=2, share_pool_bytes=free_budget, weights=weights)
            rows = [(i, q, c + q) for i, (c, q) in enumerate(wl.reqs)]
            batches.append(rows)
            secs.append(r["ms_per_step"] / 1e3)
            if b == 64:
                curve[C] = r["ms_per_step"] / 1e3
            r.update({"kind": "profile", "budget": C, "decodes": b})
            print(json.dumps(r), flush=True)
    fit = BU.StepTimeFit.fit(batches, secs)
    resid = [abs(fit(rw) - t) / t for rw, t in zip(batches, secs)]
    print(json.dumps({"kind": "fit", "t0_ms": round(fit.t0 * 1e3, 4), "a_us_per_token": round(fit.a * 1e6, 5),
                      "b_ns_per_decode_key": round(fit.b * 1e9, 5), "c_ps_per_pair": round(fit.c * 1e12, 5),
                      "max_rel_residual": round(max(resid), 4), "points": len(secs)}), flush=True)
    choices = {}
    for tbt in (0.025, 0.050, 0.100):
        choices[tbt] = BU.select_budget(curve, tbt)
        print(json.dumps({"kind": "select", "tbt_target_ms": tbt * 1e3, "decodes": 64,
                          "curve_ms": {str(k): round(v * 1e3, 3) for k, v in sorted(curve.items())},
                          "budget": choices[tbt]}), flush=True)
    rates = [5, 10, 15, 20, 25, 30, 40, 50, 60, 80]
    for C in sorted({256, 512, 1024, 2048, 4096, 8192} | {c for c in choices.values() if c}):
        g, pts = BU.goodput(C, rates, fit, n_requests=1000, seed=7)
        print(json.dumps({"kind": "load_test", "budget": C, "step_time": "GB300 fit", "goodput_rps": g,
                          "points": pts}), flush=True)
    # the chosen budget with a fixed per-request cap (head-of-line blocking)
    # and with the adaptive per-step chunk size (min 128, base 512, max 4,096,
    # pressure 16: the llm-stack-book defaults)
    C50 = choices.get(0.050) or 2048
    for label, kw in (("chunk_cap 512", {"chunk_cap": 512}), ("adaptive 128/512/4096/16", {"adaptive": (128, 512, 4096, 16)})):
        g, pts = BU.goodput(C50, rates, fit, n_requests=1000, seed=7, **kw)
        print(json.dumps({"kind": "load_test", "budget": C50, "policy": label, "step_time": "GB300 fit",
                          "goodput_rps": g, "points": pts}), flush=True)


PROFILE_CASES = {
    # one layer of the headline stack: the last chunk position (2,048 rows
    # after 30,720 cached tokens) beside the 96 decodes, the chunk alone, and
    # the decodes alone
    "sweep_P30720": dict(k=15, decodes=True, chunk=True),
    "chunk_P30720": dict(k=15, decodes=False, chunk=True),
    "chunk_P14336": dict(k=7, decodes=False, chunk=True),
    "sweep_decodes": dict(k=0, decodes=True, chunk=False),
    # every position once per step (16 mb_step calls): one layer's share of
    # each kernel over the whole prompt
    "sweep_all": dict(k=None, decodes=True, chunk=True),
    # the chunk alone at every position (the roofline's launches)
    "chunk_all": dict(k=None, decodes=False, chunk=True),
    # one Llama-3-8B-shaped layer on the 576-token mixed batch (64 decodes +
    # a 512-token chunk), the auxiliary layer line's batch
    "llama_T576": dict(workload="llama3_8b_mixed"),
}


def run_case(args):
    """One layer of the headline workload on one fixed batch, for profiling
    (ncu) and quick timing: `--warmup` untimed steps, then `--steps` steps
    with events around every launch (L2 flushed between steps); prints the
    per-kernel mean times.  Under ncu, `-s <warmup * launches per step>`
    skips the warm-up launches."""
    import torch
    from mixed_prefill_decode_gb300 import build as B
    from mixed_prefill_decode_gb300 import binding as mb
    B.build()
    peaks, peak_kind = load_peaks()
    spec = PROFILE_CASES[args.case]
    if "workload" in spec:   # a fixed batch of a named workload
        wl = getattr(W, spec["workload"])()
        sh = wl.shape
        batch, num_pages = W.make_batch(wl.reqs, wl.seed + 2)   # the layout materialize() gives it
        batches = [batch]
        dw = W.device_weights(sh, wl.seed + 100)
        dpool = W.device_kv_pool(sh, num_pages, wl.seed + 200)
    else:                    # positions of the prompt sweep
        sw = W.qwen3_14b_prompt_sweep()
        sh = sw.shape
        full, num_pages = sw.layout()
        ks = range(sw.steps) if spec["k"] is None else [spec["k"]]
        batches = [sw.batch_at(k, full, with_decodes=spec["decodes"], with_chunk=spec["chunk"]) for k in ks]
        dw = W.device_weights(sh, sw.seed + 100)
        dpool = W.device_kv_pool(sh, num_pages, sw.seed + 200)
    T = max(b.num_tokens for b in batches)
    layer = mb.Layer(sh.as_dict(), dw, T, num_pages, kv_buf=dpool)
    cbs = [mb.Batch.of(b) for b in batches]
    x = torch.randn((T, sh.d_model), device="cuda").to(torch.bfloat16)
    y = torch.empty_like(x)
    s = torch.cuda.current_stream().cuda_stream
    flush = L2Flush(torch)

    def one(i):
        for cb in cbs:
            flush(i & 0xFF)
            layer.step(cb, x, y, s)

    for i in range(args.warmup):
        one(i)
    mb.mb_device_status(layer.handle, s)
    mb.mb_layer_set_timing(layer.handle, True)
    for i in range(args.steps):
        one(i)
    torch.cuda.synchronize()
    km, n = mb.mb_layer_timing(layer.handle)
    mb.mb_device_status(layer.handle, s)
    alg = {}
    for b in batches:   # algorithmic work summed over the positions of one step
        for name, (bound, wk) in algorithmic(sh, b).items():
            if name not in alg:
                alg[name] = (bound, wk)
            elif bound == "mixed":
                alg[name] = (bound, (alg[name][1][0] + wk[0], alg[name][1][1] + wk[1]))
            else:
                alg[name] = (bound, alg[name][1] + wk)
    km_step = {k: v * len(batches) for k, v in km.items()}   # per pass over the positions
    out = {"case": args.case, "tokens": sum(b.num_tokens for b in batches), "positions": len(batches),
           "launches_per_step": mb.mb_layer_last_launches(layer.handle) * len(batches),
           "kernels": kernel_table(alg, km_step, n, peaks)}
    if not spec.get("decodes", True) and spec.get("chunk", True):
        fl = alg["attention"][1][0]
        out["chunk_attention"] = {"flop": fl, "tflops": round(fl / (km_step["attention"] / n / 1e3) / 1e12, 1)}
    print(json.dumps(out), flush=True)
    layer.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-aux", action="store_true",
                    help="skip the auxiliary lines (Llama-3-8B layer, decode-only, generation, piggyback)")
    ap.add_argument("--sweep", action="store_true",
                    help="token-budget sweep on the 32-layer Llama-3-8B stack: one JSON line per point")
    ap.add_argument("--partition", action="store_true",
                    help="decode SM partition: decode-only bandwidth and the mixed step against the decode-SM cap")
    ap.add_argument("--budget", action="store_true",
                    help="budget selection: profile the stack, fit the step time, choose budgets, load-test them")
    ap.add_argument("--case", choices=sorted(PROFILE_CASES),
                    help="one layer of the headline workload on one fixed batch (profiling): per-kernel times")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, world, local, pg = dist_setup()
    if args.sweep:
        run_sweep(args)
        return
    if args.budget:
        run_budget(args)
        return
    if args.partition:
        run_partition(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_mine(args, rank, world, local, pg)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
