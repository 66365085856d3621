"""Oracle token-budget packer (the scheduler that builds a mixed batch).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the fixed priority order of the pofe.ai "Chunked prefill" page, "How it
works, step by step" (steps 1-3 and its ``schedule()`` sketch):

  1. one token for every running decode;
  2. the next chunk of each partially processed prompt, min(C_left, p - p_done)
     tokens from offset p_done;
  3. admit waiting prompts in arrival order while budget, sequence slots and KV
     blocks remain, each taking as many prompt tokens as fit.

Readings where the pages are silent or disagree:

  * decodes never drive the budget negative: a decode is scheduled only while
    at least one unit is left (llm-stack-book 7.8 ``ChunkedPrefillScheduler``
    checks ``budget >= 1``; the pofe.ai sketch would let ``left`` go negative);
  * an admission takes as many tokens as fit (pofe.ai), not only when a whole
    ``chunk_size`` fits (llm-stack-book);
  * an optional per-request cap ``chunk_cap`` (0 = none) bounds every prefill
    chunk (pofe.ai "Head-of-line blocking among prefills"; ``chunk_size`` in the
    llm-stack-book scheduler);
  * admission stops at the first waiting prompt that fails the sequence limit
    or cannot get pages for its chunk (the ``break`` in the pofe.ai sketch);
  * pages are 16 tokens, handed out FIFO from a free list whose initial order
    the caller gives; a request holds exactly ceil(kv_len / 16) pages, and
    pages are taken at pack time in the order rows are scheduled;
  * a running decode that needs a new page when none is free is skipped for
    this step; a partial prefill's chunk is shortened to what its pages plus
    the free pages can hold, and skipped if that is nothing;
  * finishing a request returns its pages to the tail of the free list in
    block-table order;
  * adaptive chunk size (optional; llm-stack-book 7.8, "Priority and
    Preemption Policies", ``adaptive_chunk_size``, applied per step as in its
    exercise 4): the step's chunk cap follows the number of running decodes d
    at the start of the step: max with d = 0, min from d >= pressure on, else
    the base-to-min line at d / pressure, truncated, kept in [min, base]; it
    combines with ``chunk_cap`` by taking the smaller.

Each scheduled row is (req_id, qo_len, kv_len, block_table); a row with
qo_len = 1 is a decode row whatever the request's phase.  ``pack`` advances the
state as if the forward pass ran: prefilled counts grow by the chunk, and a
prompt whose last chunk was scheduled becomes a running decode from the next
step on (pofe.ai step 5).
"""

from __future__ import annotations

from collections import deque
from typing import Dict, List, Optional, Sequence, Tuple

PAGE_TOKENS = 16


def pages_for(n: int) -> int:
    return (n + PAGE_TOKENS - 1) // PAGE_TOKENS


class NoSpace(Exception):
    pass


class _Req:
    __slots__ = ("rid", "prompt_len", "computed", "pages")

    def __init__(self, rid: int, prompt_len: int, computed: int):
        self.rid = rid
        self.prompt_len = prompt_len
        self.computed = computed
        self.pages: List[int] = []


def adaptive_chunk(decodes: int, min_chunk: int, base_chunk: int, max_chunk: int, pressure: int) -> int:
    """The step's chunk size from the number of running decodes
    (llm-stack-book 7.8, ``adaptive_chunk_size``)."""
    if decodes == 0:
        return max_chunk
    if decodes >= pressure:
        return min_chunk
    chunk = int(base_chunk - (decodes / pressure) * (base_chunk - min_chunk))
    return max(min_chunk, min(chunk, base_chunk))


class Packer:
    def __init__(self, budget: int, max_seqs: int, chunk_cap: int, free_order: Sequence[int],
                 adaptive: Optional[Tuple[int, int, int, int]] = None):
        if budget < 1 or max_seqs < 1 or chunk_cap < 0:
            raise ValueError("bad packer config")
        self.budget = budget
        self.max_seqs = max_seqs
        self.chunk_cap = chunk_cap
        self.adaptive = adaptive        # (min, base, max, pressure) or None
        self.free = deque(int(p) for p in free_order)
        self.reqs: Dict[int, _Req] = {}
        self.running: List[_Req] = []
        self.partial: List[_Req] = []
        self.waiting: deque = deque()

    # -- request lifecycle --------------------------------------------------
    def add(self, rid: int, prompt_len: int, computed: int = 0) -> None:
        """A new request.  ``computed`` tokens of it are already in the KV
        cache (0 for a fresh prompt; >= prompt_len for a running decode)."""
        if rid in self.reqs or prompt_len < 1 or computed < 0:
            raise ValueError("bad request")
        r = _Req(rid, prompt_len, computed)
        need = pages_for(computed)
        if need > len(self.free):
            raise NoSpace()
        self._take(r, need)
        self.reqs[rid] = r
        if computed == 0:
            self.waiting.append(r)
        elif computed < prompt_len:
            self.partial.append(r)
        else:
            self.running.append(r)

    def finish(self, rid: int) -> None:
        r = self.reqs.pop(rid)
        for q in (self.running, self.partial):
            if r in q:
                q.remove(r)
        if r in self.waiting:
            self.waiting.remove(r)
        self.free.extend(r.pages)
        r.pages = []

    def _take(self, r: _Req, n: int) -> None:
        for _ in range(n):
            r.pages.append(self.free.popleft())

    # -- one step -----------------------------------------------------------
    def pack(self) -> List[Tuple[int, int, int, List[int]]]:
        left = self.budget
        sched: List[Tuple[_Req, int, bool]] = []   # (req, n, is_prefill)
        cap = self.chunk_cap
        if self.adaptive:
            eff = adaptive_chunk(len(self.running), *self.adaptive)
            cap = min(cap, eff) if cap else eff

        # 1. decodes first
        for r in self.running:
            if left < 1:
                break
            need = pages_for(r.computed + 1) - len(r.pages)
            if need > len(self.free):
                continue
            self._take(r, need)
            sched.append((r, 1, False))
            left -= 1

        # 2. continue partial prefills, FIFO
        for r in list(self.partial):
            if left <= 0:
                break
            n = min(left, r.prompt_len - r.computed)
            if cap:
                n = min(n, cap)
            room = (len(r.pages) + len(self.free)) * PAGE_TOKENS - r.computed
            n = min(n, room)
            if n <= 0:
                continue
            self._take(r, pages_for(r.computed + n) - len(r.pages))
            sched.append((r, n, True))
            left -= n

        # 3. admissions in arrival order
        while self.waiting and left > 0:
            r = self.waiting[0]
            if len(self.running) + len(self.partial) >= self.max_seqs:
                break
            n = min(left, r.prompt_len)
            if cap:
                n = min(n, cap)
            if pages_for(n) > len(self.free):
                break
            self.waiting.popleft()
            self.partial.append(r)
            self._take(r, pages_for(n))
            sched.append((r, n, True))
            left -= n

        rows = []
        for r, n, is_prefill in sched:
            rows.append((r.rid, n, r.computed + n, list(r.pages)))
            r.computed += n
            if is_prefill and r.computed >= r.prompt_len:
                self.partial.remove(r)
                self.running.append(r)
        return rows


STATE_MAGIC = 0x4D4253434844
STATE_VERSION = 1


def state_words(pk: Packer) -> List[int]:
    """The packer's state in the checkpoint layout of the C ABI: what the
    later batches depend on, per request its id, prompt length, prefilled
    count and block table (pofe.ai "How it works, step by step": the only new
    state is the prefilled count; llm-stack-book 7.8's SequenceState keeps
    num_computed), in queue order, and the free list in hand-out order."""
    ad = pk.adaptive or (0, 0, 0, 0)
    w = [STATE_MAGIC, STATE_VERSION, pk.budget, pk.max_seqs, pk.chunk_cap,
         len(pk.free) + sum(len(r.pages) for r in pk.reqs.values()), *ad, len(pk.free), *pk.free]
    for queue in (pk.running, pk.partial, list(pk.waiting)):
        w.append(len(queue))
        for r in queue:
            w += [r.rid, r.prompt_len, r.computed, len(r.pages), *r.pages]
    return [int(v) for v in w]


def from_state_words(words: Sequence[int]) -> Packer:
    """Inverse of state_words (trusted input: the checks live in the C ABI)."""
    it = iter(int(v) for v in words)
    assert next(it) == STATE_MAGIC and next(it) == STATE_VERSION
    budget, max_seqs, chunk_cap, num_pages = next(it), next(it), next(it), next(it)
    ad = tuple(next(it) for _ in range(4))
    free = [next(it) for _ in range(next(it))]
    pk = Packer(budget, max_seqs, chunk_cap, free, adaptive=None if ad == (0, 0, 0, 0) else ad)
    for queue in (pk.running, pk.partial, pk.waiting):
        for _ in range(next(it)):
            rid, prompt_len, computed, n = next(it), next(it), next(it), next(it)
            r = _Req(rid, prompt_len, computed)
            r.pages = [next(it) for _ in range(n)]
            pk.reqs[rid] = r
            queue.append(r)
    assert next(it, None) is None
    return pk


def rows_to_csr(rows):
    """(req_id, qo, kv, table) rows -> qo_indptr, kv_len, bt_indptr, bt, req_ids."""
    qo_indptr = [0]
    bt_indptr = [0]
    kv_len, bt, ids = [], [], []
    for rid, qo, kv, table in rows:
        qo_indptr.append(qo_indptr[-1] + qo)
        kv_len.append(kv)
        bt.extend(table)
        bt_indptr.append(len(bt))
        ids.append(rid)
    return qo_indptr, kv_len, bt_indptr, bt, ids
