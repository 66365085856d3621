"""GPU parity at the token-budget sweep's lengths (Llama-3-8B-shaped layer):
decode contexts up to 32,768 keys, up to 256 decodes, chunks of up to 8,176
rows after prefixes up to 16,384 (pofe.ai "Chunked prefill", "Simulated
numbers: choosing the budget"; llm-stack-book 7.8, "Attention on Partial KV
Caches").

Long decodes are split along their keys into up to 32 pieces whose partial
softmax states are merged by log-sum-exp, one split per lane of a warp.
These cases reach a single decode at 32,768 keys (32 splits: every lane of the
merge), split counts spread over 4..31, and the sweep's own batches.

Each case runs one mb_step through the C ABI and checks:
* KV placement bit-exact on the device: only this step's (page, slot) pairs
  change in the whole pool;
* sampled rows (every kind: shortest and longest decodes, chunk rows at tile
  boundaries and the chunk's last row) against the oracle, stage by stage
  (tests/sampled.py), within max|d| <= 2e-2 max|ref| per tensor."""

import math

import numpy as np
import pytest
import torch

from oracle import layer as OL
from mixed_prefill_decode_gb300 import workload as W
from gpu_util import to_dev, from_dev
from sampled import changed_slots_within_written, check_rows, layer_bits

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


def decode_splits(batch: W.Batch, n_kv_heads: int, sms: int, items_per_sm: int = 4):
    """Split count of every decode request, by the library's rule (restated
    here only to report and assert which counts a case reaches): about
    items_per_sm work items per SM; a request's 128-key blocks are spread
    over round(blocks / blocks-per-item) splits, at least 1, at most 32."""
    qo = batch.qo_len()
    dec = [r for r in range(batch.num_reqs) if qo[r] == 1]
    dec_pages = sum(W.pages_for(int(batch.kv_len[r])) for r in dec)
    dec_blocks = (dec_pages + 7) // 8
    target = sms * items_per_sm
    bps = max(1, -(-(dec_blocks * n_kv_heads) // target))
    out = {}
    for r in dec:
        nblk = (W.pages_for(int(batch.kv_len[r])) + 7) // 8
        out[r] = max(1, min(nblk, (nblk + bps // 2) // bps, 32))
    return out


def _sample_tokens(batch: W.Batch, splits: dict, n_dec: int = 16):
    qo = batch.qo_len()
    toks = []
    dec = sorted(splits, key=lambda r: int(batch.kv_len[r]))
    if dec:
        picks = set(np.linspace(0, len(dec) - 1, min(n_dec, len(dec))).round().astype(int).tolist())
        # every distinct split count at least once
        seen = set()
        for i, r in enumerate(dec):
            if splits[r] not in seen:
                seen.add(splits[r])
                picks.add(i)
        toks += [int(batch.qo_indptr[dec[i]]) for i in sorted(picks)]
    for r in range(batch.num_reqs):
        if qo[r] > 1:
            n = int(qo[r])
            rows = {0, 1, 127, 128, 129, 255, 256, n // 2, n - 2, n - 1}
            toks += [int(batch.qo_indptr[r]) + i for i in sorted(rows) if 0 <= i < n]
    return toks


CASES = {
    # one decode at 32,768 keys: 256 blocks in 32 splits
    "b1_kv32768": [(32767, 1)],
    # decodes at 16,385 / 24,000 / 6,001 / 3,001 keys beside a 1,024-row chunk:
    # split counts spread between 4 and 31
    "splits_4_31_chunk1024": [(16384, 1), (23999, 1), (6000, 1), (3000, 1), (0, 1024)],
    # the sweep's own batches (one layer): 256 decodes with contexts
    # log-uniform in [512, 32768] plus a 256-token chunk; 64 decodes plus a
    # 1,984-token chunk; 16 decodes plus an 8,176-token chunk
    "sweep_C512_b256": "C512_b256",
    "sweep_C2048_b64": "C2048_b64",
    "sweep_C8192_b16": "C8192_b16",
}


def _reqs(spec):
    if isinstance(spec, str):
        C, b = spec[1:].split("_b")
        wl, _ = W.llama3_8b_stack(int(C), int(b))
        return wl.reqs, wl.seed
    return spec, 9100 + len(spec)


@pytest.mark.parametrize("name", list(CASES))
def test_sweep_lengths_sampled_parity(mb, name):
    sh = W.LLAMA3_8B
    reqs, seed = _reqs(CASES[name])
    batch, num_pages = W.make_batch(reqs, seed + 1, spare_pages=16)
    T = batch.num_tokens
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    splits = decode_splits(batch, sh.n_kv_heads, sms)
    counts = sorted(set(splits.values()))
    print(f"{name}: T={T}, decodes={len(splits)}, max kv={int(batch.kv_len.max())}, split counts {counts}")
    if name == "b1_kv32768":
        assert counts == [32]
    if name == "splits_4_31_chunk1024":
        assert any(6 <= c <= 31 for c in counts) and min(counts) >= 2

    wb = W.make_weights(sh, seed + 2, unit_gains=True)
    dw = {k: to_dev(v) for k, v in wb.items()}
    x = W.make_embeddings(T, sh.d_model, seed + 3)
    dpool = W.device_kv_pool(sh, num_pages, seed + 4)
    before = dpool.clone()
    layer = mb.Layer(sh.as_dict(), dw, T, num_pages, kv_buf=dpool)
    try:
        dx = to_dev(x)
        dy = torch.empty_like(dx)
        layer.step(mb.Batch.of(batch), dx, dy, _stream())
        mb.mb_device_status(layer.handle, _stream())
        changed, written = changed_slots_within_written(before, dpool, batch)
        del before
        hq = sh.n_q_heads * sh.head_dim
        q_bits = layer_bits(layer, 2, T, hq)
        o_bits = layer_bits(layer, 3, T, hq)
        y_bits = from_dev(dy)
        toks = _sample_tokens(batch, splits)
        errs = check_rows(sh, OL.weights_to_f64(wb), batch, x, y_bits, q_bits, o_bits, dpool, toks, name)
        print(name, f"{len(toks)} rows, {changed}/{written} slots changed/written",
              {k: f"{v:.2e}" for k, v in errs.items()})
    finally:
        layer.close()
