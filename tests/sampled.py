"""Row-sampled oracle checks for full-size steps whose whole oracle run would
not fit in host memory or time (decode contexts up to 32,768 keys, 256
decodes, 8,192-token chunks).

A row's output depends on the other rows only through the keys and values
they append (a mixed batch's rows equal each request run alone, and a decode
step equals the last row of a prefill over the same tokens: both are pinned
in the oracle's own tests).  So the oracle reproduces token t of request r,
at position p = c_r + i, as a one-token request at that position whose
earlier keys and values are the GPU's own (from the pool after the step),
read through a compact copy of the request's pages.  That checks every stage
of the row (norm, QKV, q/k-norm, RoPE, its appended K/V, attention over p + 1
keys, O, FFN) at the full context length, with each stage's error measured
against the acceptance tolerance over all sampled rows together.

The attention alone is also checked per row on the GPU's q and pool, which
isolates the attention kernels (decode splits and their merge, chunk tiles)
from upstream rounding."""

from __future__ import annotations

import numpy as np
import torch

from oracle import layer as OL
from mixed_prefill_decode_gb300 import workload as W
from gpu_util import assert_close, f64, dev_buffer_bits

PAGE = W.PAGE_TOKENS


def row_positions(batch: W.Batch):
    """(request, position) of every token of the batch, in token order."""
    qo = batch.qo_len()
    c = batch.cached()
    req = np.repeat(np.arange(batch.num_reqs), qo)
    pos = np.concatenate([c[r] + np.arange(qo[r]) for r in range(batch.num_reqs)])
    return req, pos


def changed_slots_within_written(dpool_before: torch.Tensor, dpool_after: torch.Tensor, batch: W.Batch):
    """KV placement, bit-exact, on the device: the (page, slot) pairs whose
    bits changed must all be slots this step appends (token p of request r
    goes to page bt_r[p // 16], slot p % 16).  Returns (changed, written)."""
    P = dpool_before.shape[0]
    diff = (dpool_before.view(torch.int16) != dpool_after.view(torch.int16))   # [P, 2, Hkv, 16, hd]
    changed = diff.any(dim=4).any(dim=2).any(dim=1)                            # [P, 16]
    req, pos = row_positions(batch)
    written = torch.zeros((P, PAGE), dtype=torch.bool, device=dpool_before.device)
    pages = np.array([batch.bt[batch.bt_indptr[r] + p // PAGE] for r, p in zip(req, pos)], dtype=np.int64)
    slots = (pos % PAGE).astype(np.int64)
    written[torch.from_numpy(pages).to(written.device), torch.from_numpy(slots).to(written.device)] = True
    stray = changed & ~written
    assert not bool(stray.any()), f"{int(stray.sum())} KV slots outside this step's appends changed"
    return int(changed.sum()), int(written.sum())


def check_rows(shape: W.LayerShape, w64: dict, batch: W.Batch, x_bits: np.ndarray, y_bits: np.ndarray,
               q_bits: np.ndarray, o_bits: np.ndarray, dpool_after: torch.Tensor, tokens, label: str):
    """Oracle check of the sampled tokens (indices into the batch's rows).
    q_bits / o_bits: the GPU's rotated q [T, Hq, hd] and attention output
    [T, Hq hd] (bf16 bits)."""
    sh = shape.as_dict()
    Hq, Hkv, hd = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    req, pos = row_positions(batch)
    pool5 = dpool_after.view(-1, 2, Hkv, PAGE, hd)
    got = {k: [] for k in ("y", "k", "v", "o_iso", "q")}
    ref = {k: [] for k in got}
    for t in tokens:
        r, p = int(req[t]), int(pos[t])
        table = batch.bt[batch.bt_indptr[r]:batch.bt_indptr[r + 1]]
        n_pages = W.pages_for(p + 1)
        pages = torch.from_numpy(table[:n_pages].astype(np.int64)).to(dpool_after.device)
        compact = pool5.index_select(0, pages).contiguous()
        cbits = compact.cpu().view(torch.int16).numpy().view(np.uint16)
        cpool = f64(cbits)                                   # [n_pages, 2, Hkv, 16, hd]
        # the GPU's appended K/V of this row and its attention on its own q / pool
        got["k"].append(cpool[p // PAGE, 0, :, p % PAGE, :].copy())
        got["v"].append(cpool[p // PAGE, 1, :, p % PAGE, :].copy())
        K, V = OL.gather_kv(cpool, np.arange(n_pages), p + 1)
        qrow = f64(q_bits[t]).reshape(1, Hq, hd)
        ref["o_iso"].append(OL.attention_request(qrow, K, V, p)[0].reshape(-1))
        got["o_iso"].append(f64(o_bits[t]).reshape(-1))
        # the whole row as a one-token request at position p
        out = OL.layer_step(sh, w64, cpool, [0, 1], [p + 1], [0, n_pages], np.arange(n_pages, dtype=np.int32),
                            f64(x_bits[t:t + 1]))
        ref["y"].append(out["y"][0])
        ref["k"].append(out["k"][0])
        ref["v"].append(out["v"][0])
        ref["q"].append(out["q"][0].reshape(-1))
        got["q"].append(f64(q_bits[t]).reshape(-1))
        got["y"].append(f64(y_bits[t]))
    errs = {}
    for k in ("q", "k", "v", "o_iso", "y"):
        errs[k] = assert_close(f"{label} sampled {k}", np.stack(got[k]), np.stack(ref[k]))
    return errs


def layer_bits(layer, which: int, T: int, width: int) -> np.ndarray:
    ptr, nbytes = layer.buffer(which)
    return dev_buffer_bits(ptr, nbytes).reshape(T, width)
