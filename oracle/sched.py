"""Oracle stall-free scheduler and page allocator (test infrastructure only).

Restates Algorithm 3 of the *Sarathi-Serve digest* (§2 Q2 item 2 and the
§3 flowchart; "implementation details" item 1 in §7): every iteration

1. starts with an empty budget count ``n_t = 0``;
2. adds one decode token for every running request whose prefill is done;
3. if a request's prefill is unfinished, adds its next chunk,
   ``c = get_next_chunk_size(R, tau, n_t)``, ``n_t += c``;
4. admits new requests while ``can_allocate`` and ``n_t < tau``, each with
   its first chunk ``c = get_next_chunk_size(R_new, tau, n_t)``, ``n_t += c``
   (the flowchart's admission loop), so one batch may carry several chunks;
5. processes the hybrid batch, then drops finished requests.

Every admitted request but the last fits whole in the budget left to it, and
an ongoing chunk that stops short of its prompt's end fills the budget, so
at most one prompt is unfinished after any iteration -- the "at most one
ongoing prefill chunk" of the digest's §2 Q2 item 2.

Readings where the pages are silent (the CUDA-side scheduler follows the same):

* the token budget is rounded down to a multiple of the GEMM tile (the
  "batch token count must be a multiple of the tile size" rule,
  *Sarathi-Serve digest* §2 Q2 item 3; *SARATHI reading notes* part 3 §3);
* ``get_next_chunk_size = min(remaining prompt, tau - n_t)``;
* ``max_chunks`` caps the chunks of one batch (0 = no cap: the admission
  loop above).  ``max_chunks = 1`` is the one-chunk reading of *SARATHI
  technique write-up* §3.2 ("one prefill chunk per batch"): a new request is
  then admitted only when no prompt is unfinished, and leftover budget stays
  unused;
* admission is first-come-first-served with head-of-line blocking: the loop
  stops at the first ready request that cannot be allocated;
* waiting requests are served first-come-first-served by (arrival, id) and
  only once ``arrival <= now``;
* ``can_allocate``: free pages >= ceil(prompt_len / page_size) + 1 and fewer
  than ``max_batch`` requests hold pages (the bound B of *SARATHI technique
  write-up* §4.1); the prompt's pages are taken at admission;
* a decode at context ``ctx`` writes slot ``ctx`` and takes a new page when
  ``ctx % page_size == 0``; no preemption -- an empty pool is an error;
* pages are handed out lowest id first and returned on completion;
* the first output token comes from the chunk that completes the prompt; a
  request with ``output_len`` outputs then runs ``output_len - 1`` decodes.

Parity pins: ordering and budget invariants (``tests/test_oracle_sched.py``)
and bit-exact agreement with a brute-force replay of small traces.
"""

from __future__ import annotations

import dataclasses
import heapq


class NoPages(RuntimeError):
    pass


class PagePool:
    """Free list handing out the lowest-numbered page first."""

    def __init__(self, num_pages: int):
        self.free = list(range(num_pages))
        heapq.heapify(self.free)

    def n_free(self) -> int:
        return len(self.free)

    def alloc(self) -> int:
        if not self.free:
            raise NoPages("page pool exhausted")
        return heapq.heappop(self.free)

    def release(self, pages) -> None:
        for p in pages:
            heapq.heappush(self.free, p)


@dataclasses.dataclass
class Req:
    req: int
    arrival: float
    prompt_len: int
    output_len: int
    prompt_tokens: list | None = None
    prefill_done: int = 0
    generated: int = 0
    pages: list = dataclasses.field(default_factory=list)
    tokens: list = dataclasses.field(default_factory=list)


@dataclasses.dataclass
class Batch:
    """One iteration's decision: the prefill chunks, then the decodes.

    ``prefills``: list of ``(req, start_pos, len, block_table)`` (the ongoing
    prompt's chunk first, then newly admitted requests in admission order);
    ``decodes``: list of ``(req, ctx_len, block_table)``; ``tokens``: input
    token id per batch row (chunk rows first) when prompt tokens are known.
    """

    prefills: list
    decodes: list
    tokens: list | None

    @property
    def prefill(self) -> tuple | None:
        """The first chunk, or None."""
        return self.prefills[0] if self.prefills else None

    @property
    def n_tokens(self) -> int:
        return sum(p[2] for p in self.prefills) + len(self.decodes)

    @property
    def logit_rows(self) -> int:
        """Rows sampled: the last row of every chunk, then every decode."""
        return len(self.prefills) + len(self.decodes)


def round_budget(tau: int, tile: int) -> int:
    """Token budget rounded down to a whole number of GEMM row tiles."""
    if tile <= 0 or tau < tile:
        raise ValueError("token budget smaller than one tile")
    return (tau // tile) * tile


class StallFreeScheduler:
    def __init__(self, tau: int, tile: int, page_size: int, num_pages: int, max_batch: int,
                 max_chunks: int = 0):
        if max_chunks < 0:
            raise ValueError("negative chunk cap")
        self.max_chunks = max_chunks
        self.tau = round_budget(tau, tile)
        self.page_size = page_size
        self.max_batch = max_batch
        self.pool = PagePool(num_pages)
        self.waiting: list[Req] = []
        self.running: list[Req] = []
        self.finished: list[Req] = []
        self._last: Batch | None = None

    def add(self, req: int, arrival: float, prompt_len: int, output_len: int,
            prompt_tokens=None) -> None:
        if prompt_len <= 0 or output_len <= 0:
            raise ValueError("empty prompt or output")
        self.waiting.append(Req(req, arrival, prompt_len, output_len,
                                list(prompt_tokens) if prompt_tokens is not None else None))

    def _can_allocate(self, r: Req) -> bool:
        need = -(-r.prompt_len // self.page_size) + 1
        return self.pool.n_free() >= need and len(self.running) < self.max_batch

    def next(self, now: float) -> Batch:
        n_t = 0
        decodes = []
        for r in self.running:
            if r.prefill_done == r.prompt_len and r.generated < r.output_len:
                ctx = r.prompt_len + r.generated - 1
                if ctx % self.page_size == 0:
                    r.pages.append(self.pool.alloc())
                decodes.append(r)
                n_t += 1
        chunks = []
        ongoing = next((r for r in self.running if r.prefill_done < r.prompt_len), None)
        if ongoing is not None:
            c = min(ongoing.prompt_len - ongoing.prefill_done, self.tau - n_t)
            if c > 0:
                chunks.append((ongoing, ongoing.prefill_done, c))
                n_t += c
        if ongoing is None or self.max_chunks != 1:
            ready = sorted((r for r in self.waiting if r.arrival <= now),
                           key=lambda r: (r.arrival, r.req))
            for r in ready:
                if self.max_chunks and len(chunks) >= self.max_chunks:
                    break
                if not (n_t < self.tau and self._can_allocate(r)):
                    break
                self.waiting.remove(r)
                for _ in range(-(-r.prompt_len // self.page_size)):
                    r.pages.append(self.pool.alloc())
                self.running.append(r)
                c = min(r.prompt_len, self.tau - n_t)
                chunks.append((r, 0, c))
                n_t += c
        tokens = None
        if all(r.prompt_tokens is not None for r in self.running):
            tokens = []
            for r, s, c in chunks:
                tokens += r.prompt_tokens[s:s + c]
            for r in decodes:
                tokens.append(r.tokens[-1] if r.tokens else 0)
        b = Batch(
            prefills=[(r.req, s, c, list(r.pages)) for r, s, c in chunks],
            decodes=[(r.req, r.prompt_len + r.generated - 1, list(r.pages)) for r in decodes],
            tokens=tokens,
        )
        self._last = b
        self._last_objs = (chunks, decodes)
        return b

    def commit(self, sampled) -> list[int]:
        """Advance state with one sampled token per logits row (each chunk's last
        row first, in batch order, then each decode).  Returns the ids of
        finished requests."""
        chunks, decodes = self._last_objs
        i = 0
        for r, s, c in chunks:
            r.prefill_done += c
            if r.prefill_done == r.prompt_len:
                r.generated = 1
                r.tokens.append(int(sampled[i]))
            i += 1
        for r in decodes:
            r.generated += 1
            r.tokens.append(int(sampled[i]))
            i += 1
        done = [r for r in self.running if r.generated >= r.output_len]
        for r in done:
            self.pool.release(r.pages)
            r.pages = []
            self.running.remove(r)
            self.finished.append(r)
        self._last_objs = ([], [])
        return [r.req for r in done]

    def idle(self) -> bool:
        return not self.running and not self.waiting
