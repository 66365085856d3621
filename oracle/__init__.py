"""CPU oracle for the mixed prefill+decode layer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library; both are fed from the seeded generator in
``mixed_prefill_decode_gb300.workload``.

Modules
  layer       the layer step in float64 NumPy, KV read through the block table
  packer      the token-budget packer

Parity status (what pins each part, tests in ``tests/test_oracle_*.py``):
  attention   torch SDPA (float64, explicit mask) on gathered KV; kv = 1 gives
              o = v; identical keys give mean(v); chunked == unchunked prefill;
              decode == last row of prefill; page permutation invariance
  rope        complex-multiplication form; position 0 is the identity; norm
              preservation; relative-position invariance
  rms_norm    torch.nn.functional.rms_norm; scale invariance; constant rows
  linear      one-hot weights select the expected input column
  swiglu      silu closed form at 0 and large |x|; gate/up half order
  layer       all-zero weights give y = x; one key gives h = x + v W_o^T; the
              FFN half reads only h (two inputs with the same h give the same
              y); q/k-norm per head before RoPE (closed form at a one-hot
              row); chunked == unchunked and decode == last prefill row.  The
              pages print no worked layer output, so no printed value pins it;
              instead, 28 plausible mistakes planted in a copy of layer.py
              each fail at least one of these pins
              (tests/test_oracle_mutations.py)
  packer      the worked example of the pofe.ai page (8 x (64 + 512) at budget
              576), hand traces of the sequence limit, page exhaustion, the
              free-list order and the adaptive size, and brute-force
              invariants; 19 planted mistakes each fail one of them
              (tests/test_oracle_mutations.py)
"""
