"""The oracle's pins have power: each plausible mistake planted in a copy of
oracle/layer.py or oracle/packer.py makes at least one CPU pin fail.

Every case writes a scratch tree (the oracle with one edit, the oracle tests,
a link to the package) under pytest's tmp_path and runs the pins there in a
fresh interpreter.  The unedited copy must pass, so a failure is the planted
mistake's doing.  Nothing here touches the CUDA path."""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = {"layer": ["test_oracle_attention.py", "test_oracle_parts.py"], "packer": ["test_oracle_packer.py"]}

# (mistake, text in oracle/layer.py, replacement)
MUTATIONS = [
    ("scale 1/hd instead of 1/sqrt(hd)", "scale = 1.0 / math.sqrt(hd)", "scale = 1.0 / hd"),
    ("causal mask hides the diagonal", "allowed = k_pos[None, :] <= q_pos[:, None]",
     "allowed = (k_pos[None, :] < q_pos[:, None]) | (k_pos[None, :] == 0)"),
    ("causal mask shows the next key", "allowed = k_pos[None, :] <= q_pos[:, None]",
     "allowed = k_pos[None, :] <= q_pos[:, None] + 1"),
    ("GQA head h % Hkv", "hk = h // group", "hk = h % Hkv"),
    ("gather reads V as K", "K = pool[pages, 0, :, slots, :]", "K = pool[pages, 1, :, slots, :]"),
    ("gather ignores later table entries", "pages = block_table[p // PAGE_TOKENS]",
     "pages = block_table[(p // PAGE_TOKENS) % 2]"),
    ("append one slot late", "return int(block_table[p // PAGE_TOKENS]), p % PAGE_TOKENS",
     "return int(block_table[p // PAGE_TOKENS]), (p + 1) % PAGE_TOKENS"),
    ("RoPE rotates the wrong way", "x1 * c - x2 * s, x2 * c + x1 * s", "x1 * c + x2 * s, x2 * c - x1 * s"),
    ("RoPE frequency theta^(-i/hd)", "inv_freq = theta ** (-2.0 * i / hd)", "inv_freq = theta ** (-1.0 * i / hd)"),
    ("RoPE pairs adjacent elements", "x1, x2 = x[..., :half], x[..., half:]", "x1, x2 = x[..., 0::2], x[..., 1::2]"),
    ("positions start at c + 1", "pos[t0:t1] = c + np.arange(t1 - t0)", "pos[t0:t1] = c + 1 + np.arange(t1 - t0)"),
    ("RMSNorm eps outside the root", "return x / np.sqrt(ms + eps) * g", "return x / (np.sqrt(ms) + eps) * g"),
    ("RMSNorm of mean |x|", "ms = np.mean(x * x, axis=-1, keepdims=True)",
     "ms = np.mean(np.abs(x), axis=-1, keepdims=True) ** 2"),
    ("RMSNorm gain dropped", "return x / np.sqrt(ms + eps) * g", "return x / np.sqrt(ms + eps)"),
    ("sigmoid for SiLU", "return x / (1.0 + np.exp(-x))", "return 1.0 / (1.0 + np.exp(-x))"),
    ("gate and up halves swapped", "a = silu(gu[:, :F]) * gu[:, F:]", "a = silu(gu[:, F:]) * gu[:, :F]"),
    ("attention residual dropped", 'h = x + linear(o, w["w_o"])', 'h = linear(o, w["w_o"])'),
    ("FFN normalises x, not h", 'hn = rms_norm(h, w["g_ffn"], eps)', 'hn = rms_norm(x, w["g_ffn"], eps)'),
    ("FFN residual is x, not h", 'y = h + linear(a, w["w_down"])', 'y = x + linear(a, w["w_down"])'),
    ("V taken from the K columns", "v = qkv[:, (Hq + Hkv) * hd:].reshape(T, Hkv, hd)",
     "v = qkv[:, Hq * hd: (Hq + Hkv) * hd].reshape(T, Hkv, hd)"),
    ("q-norm with the k gains", 'q = rms_norm(q, w["g_q"], eps)', 'q = rms_norm(q, w["g_k"], eps)'),
    ("k not rotated", 'k = rope(k, pos[:, None], shape["rope_theta"])', "pass"),
    ("q not rotated", 'q = rope(q, pos[:, None], shape["rope_theta"])', "pass"),
    ("decode rows treated as uncached", "o[t0:t1] = attention_request(q[t0:t1], K, V, n - (t1 - t0))",
     "o[t0:t1] = attention_request(q[t0:t1], K, V, 0)"),
    ("greedy sampler takes the minimum", "return logits, np.argmax(logits, axis=1)",
     "return logits, np.argmax(-logits, axis=1)"),
    ("greedy ties go to the highest id", "return logits, np.argmax(logits, axis=1)",
     "return logits, logits.shape[1] - 1 - np.argmax(logits[:, ::-1], axis=1)"),
]

# Two mistakes need a second edit: the norm moved after RoPE, and attention
# that reads the pool as it was before this step's append.
_NORM = ('    if shape["qk_norm"]:\n        q = rms_norm(q, w["g_q"], eps)\n'
         '        k = rms_norm(k, w["g_k"], eps)\n')
_ROPE_K = '    k = rope(k, pos[:, None], shape["rope_theta"])\n'
_APPEND = "    # append this step's keys and values, then attend\n"
PAIRED = [
    ("q/k-norm after RoPE", [(_NORM, ""), (_ROPE_K, _ROPE_K + _NORM)]),
    ("attention before the append", [(_APPEND, "    pool0 = pool.copy()\n" + _APPEND),
                                     ("K, V = gather_kv(pool, table, n)", "K, V = gather_kv(pool0, table, n)")]),
]
CASES = [("layer", name, [(a, b)]) for name, a, b in MUTATIONS] + [("layer", n, e) for n, e in PAIRED]

# Packer mistakes.  Not listed: ">" for ">=" at the pressure threshold of the
# adaptive size, which is no mistake (the line already reaches the minimum
# there, so both give the same size).
_DEC_SKIP = "            if need > len(self.free):\n                continue\n            self._take(r, need)\n"
PACKER = [
    ("decodes ignore the budget", "            if left < 1:\n                break\n            need = pages_for",
     "            need = pages_for"),
    ("decode takes no page at a boundary", "need = pages_for(r.computed + 1) - len(r.pages)",
     "need = pages_for(r.computed) - len(r.pages)"),
    ("a decode without a page stops the others", _DEC_SKIP, _DEC_SKIP.replace("continue", "break")),
    ("partial prefills last in, first out", "for r in list(self.partial):", "for r in reversed(list(self.partial)):"),
    ("partial prefills ignore the cap",
     "            n = min(left, r.prompt_len - r.computed)\n            if cap:\n                n = min(n, cap)",
     "            n = min(left, r.prompt_len - r.computed)"),
    ("partial prefills ignore their page room", "            n = min(n, room)\n", ""),
    ("admission ignores the sequence limit",
     "            if len(self.running) + len(self.partial) >= self.max_seqs:\n                break\n", ""),
    ("sequence limit off by one", "if len(self.running) + len(self.partial) >= self.max_seqs:",
     "if len(self.running) + len(self.partial) > self.max_seqs:"),
    ("admission ignores the cap", "            n = min(left, r.prompt_len)\n            if cap:\n                n = min(n, cap)",
     "            n = min(left, r.prompt_len)"),
    ("admission page check off by one", "if pages_for(n) > len(self.free):\n                break",
     "if pages_for(n) > len(self.free) + 1:\n                break"),
    ("admission takes an extra page", "self._take(r, pages_for(n))", "self._take(r, pages_for(n + 1))"),
    ("admission ignores the budget left", "n = min(left, r.prompt_len)", "n = r.prompt_len"),
    ("adaptive size rounded, not truncated",
     "chunk = int(base_chunk - (decodes / pressure) * (base_chunk - min_chunk))",
     "chunk = round(base_chunk - (decodes / pressure) * (base_chunk - min_chunk))"),
    ("adaptive size and cap combined by max", "cap = min(cap, eff) if cap else eff",
     "cap = max(cap, eff) if cap else eff"),
    ("adaptive size idle value is the base", "if decodes == 0:\n        return max_chunk",
     "if decodes == 0:\n        return base_chunk"),
    ("freed pages go to the head", "self.free.extend(r.pages)", "self.free.extendleft(reversed(r.pages))"),
    ("freed pages reversed", "self.free.extend(r.pages)", "self.free.extend(reversed(r.pages))"),
    ("prompt becomes a decode one step late", "if is_prefill and r.computed >= r.prompt_len:",
     "if is_prefill and r.computed > r.prompt_len:"),
    ("free list last in, first out", "r.pages.append(self.free.popleft())", "r.pages.append(self.free.pop())"),
]
CASES += [("packer", name, [(a, b)]) for name, a, b in PACKER]


def _run_pins(tmp_path, module, edits):
    src = open(os.path.join(ROOT, "oracle", module + ".py")).read()
    for a, b in edits:
        assert src.count(a) == 1, f"edit site not unique or gone: {a!r}"
        src = src.replace(a, b)
    tree = tmp_path / "tree"
    shutil.copytree(os.path.join(ROOT, "oracle"), tree / "oracle", ignore=shutil.ignore_patterns("__pycache__"))
    (tree / "oracle" / (module + ".py")).write_text(src)
    (tree / "tests").mkdir()
    for f in ["conftest.py"] + PINS[module]:
        shutil.copy(os.path.join(ROOT, "tests", f), tree / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tree / "tests" / "golden",
                    ignore=shutil.ignore_patterns("__pycache__"))
    os.symlink(os.path.join(ROOT, "mixed_prefill_decode_gb300"), tree / "mixed_prefill_decode_gb300")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        *[os.path.join("tests", f) for f in PINS[module]]], cwd=tree, capture_output=True, text=True,
                       timeout=600)
    return r


@pytest.mark.parametrize("module", list(PINS))
def test_unedited_copy_passes(tmp_path, module):
    r = _run_pins(tmp_path, module, [])
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("module,name,edits", CASES, ids=[f"{c[0]}: {c[1]}" for c in CASES])
def test_planted_mistake_fails_a_pin(tmp_path, module, name, edits):
    r = _run_pins(tmp_path, module, edits)
    tail = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else r.stderr[-500:]
    assert r.returncode == 1 and " failed" in tail, f"{name}: no pin failed ({tail})"
