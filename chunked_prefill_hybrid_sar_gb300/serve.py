"""Trace driver: the stall-free scheduler feeding hybrid steps of a model with
token inputs and greedy sampling, at wall-clock (or replayed) times.

Each iteration asks the scheduler for the next batch at time ``now``, runs one
``sar_step`` on its token ids, samples the logits rows greedily on the device
and commits the sampled ids (*Sarathi-Serve digest*, Algorithm 3: build the
hybrid batch, process it, drop finished requests).  The ``now`` of every
iteration is logged so that another scheduler can replay the exact decisions.
"""

from __future__ import annotations

import dataclasses
import time

import torch

from . import Batch, Scheduler, SAR_IN_TOKENS


@dataclasses.dataclass
class TraceResult:
    steps: int = 0
    rows: int = 0
    busy_s: float = 0.0
    wall_s: float = 0.0
    now_log: list = dataclasses.field(default_factory=list)
    batches: list = dataclasses.field(default_factory=list)     # (chunks, decodes) per step
    sampled: list = dataclasses.field(default_factory=list)     # token ids per step
    step_ms: list = dataclasses.field(default_factory=list)
    ttft: dict = dataclasses.field(default_factory=dict)        # req -> seconds
    tbt: list = dataclasses.field(default_factory=list)         # seconds between tokens

    def percentile(self, xs, q):
        if not xs:
            return None
        s = sorted(xs)
        return s[min(len(s) - 1, int(round(q / 100.0 * (len(s) - 1))))]

    def summary(self) -> dict:
        tt = list(self.ttft.values())
        return {"steps": self.steps, "rows": self.rows, "busy_s": self.busy_s, "wall_s": self.wall_s,
                "tokens_per_s_busy": self.rows / self.busy_s if self.busy_s else None,
                "ttft_p50_s": self.percentile(tt, 50), "ttft_p99_s": self.percentile(tt, 99),
                "tbt_p50_s": self.percentile(self.tbt, 50), "tbt_p99_s": self.percentile(self.tbt, 99)}


def run_trace(model, kv, trace, prompt_tokens: dict, tau: int, tile: int = 128, max_batch: int = 256,
              now_log=None, max_steps: int | None = None, keep_batches: bool = True,
              on_step=None, max_chunks: int = 0) -> TraceResult:
    """Runs every request of ``trace`` to completion.

    ``now_log``: replay these times instead of the wall clock (one per step).
    ``on_step(i, batch, x, hidden, logits)`` is called after each step's launch.
    ``max_chunks``: the scheduler's cap on prefill chunks per batch (0 = none).
    """
    dims = model.dims
    sched = Scheduler(tau, tile, kv.page_size, kv.num_pages, max_batch, max_chunks=max_chunks)
    for r in trace:
        sched.add(r.req, r.arrival, r.prompt_len, r.output_len, prompt_tokens[r.req])
    res = TraceResult()
    max_rows = max_batch + tau  # every chunk's last row and every decode row
    logits = torch.empty(max_rows, dims.vocab, dtype=torch.float32, device="cuda")
    tok_dev = torch.empty(tau, dtype=torch.int32, device="cuda")
    sampled_dev = torch.empty(max_rows, dtype=torch.int32, device="cuda")
    sampled_host = torch.empty(max_rows, dtype=torch.int32).pin_memory()
    tok_host = torch.empty(tau, dtype=torch.int32).pin_memory()
    last_emit = {}
    by_req = {r.req: r for r in trace}
    t0 = time.perf_counter()
    i = 0
    while True:
        waiting, running, finished, _ = sched.stats()
        if waiting == 0 and running == 0:
            break
        if max_steps is not None and i >= max_steps:
            break
        now = now_log[i] if now_log is not None else time.perf_counter() - t0
        chunks, decs, tokens, _ = sched.next(now)
        m = sum(c[2] for c in chunks) + len(decs)
        if m == 0:
            if now_log is None:
                nxt = min((r.arrival for r in trace if r.arrival > now), default=now)
                time.sleep(max(0.0, min(nxt - now, 0.05)))
            sched.commit([])
            res.now_log.append(now)
            res.batches.append(([], []))
            res.sampled.append([])
            i += 1
            continue
        ts = time.perf_counter()
        tok_host[:m] = torch.tensor(tokens, dtype=torch.int32)
        tok_dev[:m].copy_(tok_host[:m], non_blocking=True)
        b = Batch(chunks, decs, in_kind=SAR_IN_TOKENS)
        rows = b.logit_rows
        model.step(kv, b, tok_dev[:m], logits_out=logits[:rows])
        model.sample_greedy(logits[:rows], rows, sampled_dev[:rows])
        sampled_host[:rows].copy_(sampled_dev[:rows], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        te = time.perf_counter()
        if on_step is not None:
            on_step(i, b, tok_dev[:m], logits[:rows])
        sampled = sampled_host[:rows].tolist()
        sched.commit(sampled)
        wall = te - t0
        res.step_ms.append((te - ts) * 1e3)
        res.busy_s += te - ts
        res.rows += m
        res.now_log.append(now)
        if keep_batches:
            res.batches.append((chunks, decs))
            res.sampled.append(sampled)
        # latency bookkeeping: the chunk that completes a prompt emits its first token
        for req, start, n, _ in chunks:
            if start + n == by_req[req].prompt_len:
                res.ttft[req] = wall - by_req[req].arrival
                last_emit[req] = wall
        for (req, _, _) in decs:
            if req in last_emit:
                res.tbt.append(wall - last_emit[req])
            last_emit[req] = wall
        i += 1
    res.steps = i
    res.wall_s = time.perf_counter() - t0
    return res
