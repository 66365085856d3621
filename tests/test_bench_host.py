"""Host logic of bench.py that needs no GPU: the Qwen3-14B piggyback entry of
the JSON line (one layer and the 40-layer stack for 0, 1,024 and 2,200
piggybacked tokens), driven by a stand-in timer."""

import bench


def _fake_timer(calls, fail_on=None):
    def timer(mb, torch, wl, n_layers, steps=10):
        calls.append((wl.name, n_layers))
        T = sum(q for _, q in wl.reqs)
        if fail_on is not None and T == fail_on:
            raise RuntimeError("stand-in failure")
        ms = 0.1 * n_layers + 1e-4 * T
        return {"tokens_per_step": T, "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3),
                "launches_per_step": 8 * n_layers}
    return timer


def test_piggyback_points_time_one_layer_and_the_40_layer_stack():
    calls = []
    r = bench.qwen3_14b_piggyback(None, None, timer=_fake_timer(calls))
    assert sorted(r["points"]) == ["P0", "P1024", "P2200"]
    assert [c[1] for c in calls] == [1, 40] * 3
    assert {c[0] for c in calls} == {"qwen3_14b_mixed_P0", "qwen3_14b_mixed_P1024", "qwen3_14b_mixed_P2200"}
    for P, pt in r["points"].items():
        assert pt["tokens_per_step"] == 16 + int(P[1:])          # 16 decodes + the piggybacked tokens
        assert pt["stack40_launches"] == 320
        assert abs(pt["stack40_ms"] - (4.0 + 1e-4 * pt["tokens_per_step"])) < 1e-12


def test_a_failing_point_records_its_error_and_the_rest_still_report():
    calls = []
    r = bench.qwen3_14b_piggyback(None, None, timer=_fake_timer(calls, fail_on=1040))
    assert "error" in r["points"]["P1024"] and "stand-in failure" in r["points"]["P1024"]["error"]
    assert "layer_ms" in r["points"]["P0"] and "layer_ms" in r["points"]["P2200"]


def test_prompt_sweep_batches_cover_the_prompt_chunk_by_chunk(mb):
    """The headline workload's 16 step descriptors: 96 decodes plus chunk k
    of the 32,768-token prompt (qo 2,048, kv 2,048 (k + 1)), whose table is
    the first pages of the prompt's; every descriptor passes the library's
    rules, and the chunks' appended positions tile the prompt exactly once."""
    import numpy as np
    from mixed_prefill_decode_gb300 import workload as W

    sw = W.qwen3_14b_prompt_sweep()
    full, num_pages = sw.layout()
    assert sw.steps == 16 and len(sw.decodes) == 96
    assert all(1024 <= c <= 8192 for c in sw.decodes)
    prompt_table = full.bt[full.bt_indptr[96]:full.bt_indptr[97]]
    covered = []
    for k in range(sw.steps):
        b = sw.batch_at(k, full)
        assert b.num_reqs == 97 and b.num_tokens == 96 + 2048
        assert list(b.qo_len()[:96]) == [1] * 96 and b.qo_len()[96] == 2048
        assert b.kv_len[96] == 2048 * (k + 1) and b.cached()[96] == 2048 * k
        assert np.array_equal(b.bt[b.bt_indptr[96]:], prompt_table[:W.pages_for(2048 * (k + 1))])
        assert list(b.kv_len[:96]) == [c + 1 for c in sw.decodes]
        mb.mb_batch_validate(mb.Batch.of(b), num_pages, b.num_tokens)
        covered += list(range(b.cached()[96], b.kv_len[96]))
        only_chunk = sw.batch_at(k, full, with_decodes=False)
        assert only_chunk.num_reqs == 1 and np.array_equal(only_chunk.bt, b.bt[b.bt_indptr[96]:])
    assert covered == list(range(32768))
    dec = sw.batch_at(3, full, with_chunk=False)
    assert dec.num_reqs == 96 and dec.num_tokens == 96
