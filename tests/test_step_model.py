"""Pins for the roofline step-time model: every number the pofe.ai "Chunked
prefill" page prints from it (tests/golden/pofe_step_model.json)."""

import json
import os

from mixed_prefill_decode_gb300 import step_model as S

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pofe_step_model.json")))
M, MOD = S.H100_CLASS, S.LLAMA_8B


def _close(v, key):
    g = G[key]
    assert abs(v - g["value"]) <= g["abs_tol"], (key, v, g["value"])


def test_ridge():
    _close(S.ridge_tokens(M), "ridge_tokens")


def test_decode_and_prefill_iterations():
    _close(S.iteration_time(M, MOD, [], [1125] * 64) * 1e3, "decode_64_at_1125_ms")
    _close(S.iteration_time(M, MOD, [(4096, 0)], []) * 1e3, "prefill_4096_ms")
    _close(S.iteration_time(M, MOD, [(8192, 0)], []) * 1e3, "prefill_8192_one_shot_ms")
    _close(S.chunked_prompt_time(M, MOD, 8192, 128) * 1e3, "prefill_8192_chunk128_ms")
    gap = (S.iteration_time(M, MOD, [(4096, 0)], []) + S.iteration_time(M, MOD, [], [1125] * 64)) * 1e3
    _close(gap, "worked_example_no_chunk_gap_ms")


def test_chunk_overheads():
    one = S.iteration_time(M, MOD, [(8192, 0)], [])
    g = G["chunk_overhead_pct"]
    for c in ("128", "256", "512", "2048"):
        pct = (S.chunked_prompt_time(M, MOD, 8192, int(c)) / one - 1) * 100
        assert abs(pct - g[c]) <= g["abs_tol_pct"][c], (c, pct)


def test_worked_example_mixed_iterations():
    its = [S.iteration_time(M, MOD, [(512, 512 * k)], [1125] * 64) * 1e3 for k in range(8)]
    _close(its[0], "worked_example_first_iter_ms")
    _close(its[-1], "worked_example_last_iter_ms")
    _close(sum(its), "worked_example_total_ms")
    assert all(b > a for a, b in zip(its, its[1:]))


def test_repeated_kv_reads_and_kappa():
    assert S.kv_bytes_per_token(32, 8, 128) == 131072
    b = S.repeated_kv_bytes(MOD, 4096, 512)
    assert b == 131072 * 512 * 28
    _close(b / 1e9, "repeated_kv_gb")
    _close(b / M.bandwidth * 1e3, "repeated_kv_ms_at_2p68")
