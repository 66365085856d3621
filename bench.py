#!/usr/bin/env python
"""Benchmark of the mixed prefill+decode layer step on GB300.

One step = one mb_step call: the whole hot path (RMSNorm, QKV GEMM, q/k-norm +
RoPE + KV append, prefill-chunk attention tiles, split-KV decode rows + merge,
O GEMM + residual, RMSNorm, gate/up GEMM + SwiGLU, down GEMM + residual) over
one mixed batch.  Default workload: the Llama-3-8B-shaped layer with 64
decodes at 1,125-token contexts plus one 512-token chunk on a U[0, 4096]
prefix (T = 576 tokens), synthetic seeded data, random-init weights.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the reference arm: a plain float64 restatement of the method).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]
                    [--workload llama3_8b_T576|qwen3_14b_P0|qwen3_14b_P1024|qwen3_14b_P2200|tiny_T68]
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
    "gemm_gate_up": {"bytes": 253.111296e6, "sha256_16": "0b09e0cf7d698eff",
                     "sources": ("csrc/mb_gemm.cu", "csrc/mb_ptx.cuh", "csrc/mb_kernels.h"),
                     "capture": "profiles/launches_llama3_8b_T576.md (llama3_8b_T576, second warm-up step)"},
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
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        layer.step(cb, dx, dy, s)
    mb.mb_layer_set_timing(layer.handle, True)
    for i in range(steps):
        flush.fill_(i & 0xFF)
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
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    kvs = [L.kv for L in layers]
    for _ in range(warmup):
        mb.mb_stack_step(stack, kvs, cb, dx, dy, s)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i & 0xFF)
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
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

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
        flush.fill_(i & 0xFF)
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
        flush.fill_(i & 0xFF)
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
    wl = workload_by_name(args.workload)
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
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    for _ in range(args.warmup):
        flush.fill_(1)
        layer.step(cb, dx, dy, s)
    mb.mb_device_status(layer.handle, s)
    launches_per_step = mb.mb_layer_last_launches(layer.handle)

    # ---- timed region: K steps, L2 flushed between steps, per-step events.
    # No per-kernel events here: an event between two kernels would stop the
    # next one from starting its set-up early (programmatic dependent launch).
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(pg)
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev0[i].record(stream)
        layer.step(cb, dx, dy, s)
        ev1[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(pg)
    clk = clocks.stop() if clocks else None
    mb.mb_device_status(layer.handle, s)
    step_ms_local = sum(a.elapsed_time(b) for a, b in zip(ev0, ev1)) / args.steps
    # ---- per-kernel times: a second pass of the same steps with events
    # around every launch (kernels then run back to back, not overlapped)
    n_kt = max(1, min(args.steps, 200))
    mb.mb_layer_set_timing(layer.handle, True)
    for i in range(n_kt):
        flush.fill_(i & 0xFF)
        layer.step(cb, dx, dy, s)
    torch.cuda.synchronize()
    mb.mb_device_status(layer.handle, s)
    kern_ms, ksteps = mb.mb_layer_timing(layer.handle)
    mb.mb_layer_set_timing(layer.handle, False)
    step_ms, value = replica_throughput(pg, world, T, step_ms_local)

    # ---- per-kernel rooflines from the live events of the second pass
    alg = algorithmic(wl.shape, batch)
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
    dom = max((k for k in kern_ms if alg[k][0] != "mixed"), key=lambda k: kern_ms[k])
    bound, work = alg[dom]
    dom_ms = kern_ms[dom] / max(1, ksteps)
    if bound == "tensor":
        achieved = work / (dom_ms / 1e3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 2),
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": ncu_traffic(dom),
                    "algorithmic_per_launch": work, "peak_kind": f"{peak_kind} bf16 burst"}
    else:
        achieved = work / (dom_ms / 1e3) / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": ncu_traffic(dom),
                    "algorithmic_per_launch": work, "peak_kind": f"{peak_kind} HBM copy"}
    gemm_names = ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down")
    gemm_flops = sum(alg[n][1] for n in gemm_names)
    gemm_ms = sum(kern_ms[n] for n in gemm_names) / max(1, ksteps)
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

    # ---- end to end through the public API with host buffers
    n_e2e = max(1, min(args.steps, 200))
    xh = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    torch.cuda.synchronize()
    for i in range(n_e2e):
        flush.fill_(i & 0xFF)
        e0[i].record(stream)
        dx.copy_(xh, non_blocking=True)
        layer.step(cb, dx, dy, s)
        yh.copy_(dy, non_blocking=True)
        e1[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms, e2e_value = replica_throughput(pg, world, T, sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / n_e2e)
    upload = mb.mb_layer_last_upload_bytes(layer.handle)

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        OL, w64, x64, b2, pool64 = oracle_inputs(wl)
        nd, nc = calibrate_sample(OL, wl, w64, x64, b2, pool64, 15.0)
        smp = sub_batch(b2, x64, nd, nc)
        tok = int(smp[0][-1])
        dt = time_oracle_step(OL, wl.shape, w64, pool64, *smp)
        cpu = {"value": tok / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"one oracle layer step over {nd} decode rows and {nc} chunk rows ({tok} tokens) of "
                         f"{wl.name}, float64 NumPy, {dt:.1f} s"}

    # ---- decode rows alone (no chunk tiles in the grid), and the 40-layer stack
    dec_only = decode_only_attention(mb, torch, peaks) if rank == 0 and not args.no_aux else None
    stack40 = gen = None
    if rank == 0 and not args.no_aux:
        swl, nl = W.qwen3_14b_stack(prefix=30720)
        stack40 = stack_step_time(mb, torch, swl, nl)
        gen = generation_step_time(mb, torch, peaks)

    # ---- P3 step-time model with GB300 peaks, as an analytic comparator
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
    # last GPU work of the run: nothing after it touches the device
    piggy = qwen3_14b_piggyback(mb, torch) if rank == 0 and not args.no_aux else None
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) embeddings and KV prefix, "
                                                      "N(0,0.02) random-init weights)",
        "config": {"workload": wl.name, "tokens_per_step": T, "requests": batch.num_reqs,
                   "decodes": int(np.sum(batch.qo_len() == 1)),
                   "chunk_rows": int(np.sum(batch.qo_len()[batch.qo_len() > 1])),
                   "chunk_prefix": [int(v) for v in batch.cached()[batch.qo_len() > 1]],
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU",
                   "l2": "flushed between timed steps (256 MiB write); step time = per-step CUDA events",
                   "wall_s_timed_region": round(wall, 4)},
        "roofline": roofline,
        "kernels": kernels,
        "gemm": {"tflops": round(gemm_flops / (gemm_ms / 1e3) / 1e12, 1),
                 "frac_burst": round(gemm_flops / (gemm_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                 "frac_sustained": round(gemm_flops / (gemm_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"], 4)},
        "decode_attn": dec_only,
        "stack_qwen3_14b_40": stack40,
        "generate_llama3_8b_32": gen,
        "qwen3_14b_piggyback": piggy,
        "roofline_step_ms": round(roof_ms, 5),
        "step_model_ms": round(model_ms, 5),
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT,
                "h2d_bytes_per_step": int(x.nbytes + upload), "d2h_bytes_per_step": int(x.nbytes),
                "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clk,
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
    one-grid default, where workers take every SM the chunk tiles leave.  One
    JSON line per point."""
    import torch
    from mixed_prefill_decode_gb300 import build as B
    from mixed_prefill_decode_gb300 import binding as mb
    B.build()
    peaks, _ = load_peaks()
    s = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

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
            flush.fill_(i & 0xFF)
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
            flush.fill_(i & 0xFF)
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--workload", default="llama3_8b_T576")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-aux", action="store_true", help="skip the decode-only and 40-layer stack measurements")
    ap.add_argument("--sweep", action="store_true",
                    help="token-budget sweep on the 32-layer Llama-3-8B stack: one JSON line per point")
    ap.add_argument("--partition", action="store_true",
                    help="decode SM partition: decode-only bandwidth and the mixed step against the decode-SM cap")
    ap.add_argument("--budget", action="store_true",
                    help="budget selection: profile the stack, fit the step time, choose budgets, load-test them")
    args = ap.parse_args()
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
