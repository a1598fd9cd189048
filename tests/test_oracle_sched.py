"""Pins of the oracle scheduler (Algorithm 3 restated) against the pages' Figure 4
timeline and against the ordering/budget invariants the pages state."""

import json
import os
import random

import pytest

import synth
from oracle import sched as osch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_figure4_timeline():
    # the one-chunk reading: D waits until C's prefill is complete
    with open(os.path.join(GOLDEN, "figure4_schedule.json")) as f:
        g = json.load(f)
    s = osch.StallFreeScheduler(g["tau"], g["tile"], g["page_size"], g["num_pages"], g["max_batch"],
                                max_chunks=1)
    for r in g["requests"]:
        s.add(r["req"], r["arrival"], r["prompt_len"], r["output_len"])
    for it in g["iterations"]:
        b = s.next(it["now"])
        pre = list(b.prefill[:3]) if b.prefill else None
        assert pre == it["prefill"], it
        assert [d[0] for d in b.decodes] == it["decodes"], it
        s.commit([7] * ((1 if b.prefill else 0) + len(b.decodes)))
    assert [r.req for r in s.running] == [1]  # B started one iteration after A


def test_figure4_timeline_admission_loop():
    # the full admission loop: A and B share a batch; C's two chunks fill the budget, D follows
    with open(os.path.join(GOLDEN, "figure4_schedule_algorithm3.json")) as f:
        g = json.load(f)
    s = osch.StallFreeScheduler(g["tau"], g["tile"], g["page_size"], g["num_pages"], g["max_batch"],
                                max_chunks=g["max_chunks"])
    for r in g["requests"]:
        s.add(r["req"], r["arrival"], r["prompt_len"], r["output_len"])
    for it in g["iterations"]:
        b = s.next(it["now"])
        assert [list(p[:3]) for p in b.prefills] == it["prefills"], it
        assert [d[0] for d in b.decodes] == it["decodes"], it
        s.commit([7] * b.logit_rows)
    assert not s.running and sorted(r.req for r in s.finished) == [0, 1, 2, 3]


def test_budget_rounds_down_to_tile():
    assert osch.round_budget(512, 128) == 512
    assert osch.round_budget(600, 128) == 512
    with pytest.raises(ValueError):
        osch.round_budget(100, 128)


def run_trace(trace, tau=256, tile=128, page_size=16, num_pages=4000, max_batch=64, dt=0.01,
              check=True, max_chunks=0):
    s = osch.StallFreeScheduler(tau, tile, page_size, num_pages, max_batch, max_chunks=max_chunks)
    for r in trace:
        s.add(r.req, r.arrival, r.prompt_len, r.output_len)
    now, steps = 0.0, []
    total_pages = num_pages
    while not s.idle():
        before = {r.req: (r.prefill_done, r.generated) for r in s.running}
        waiting_before = list(s.waiting)
        b = s.next(now)
        steps.append((now, b))
        if check:
            check_batch(s, b, before, page_size, total_pages)
            check_admission(s, b, now, before, waiting_before)
        s.commit([1] * b.logit_rows)
        # at most one prompt is unfinished after any iteration
        assert sum(1 for r in s.running if r.prefill_done < r.prompt_len) <= 1
        now += dt if b.n_tokens else 0.5
        assert len(steps) < 200000
    return s, steps


def check_batch(s, b, before, page_size, total_pages):
    # every prefill-complete running request decodes in every batch (decodes never stall)
    expect = [r for r, (p, g) in before.items()
              if any(x.req == r and p == x.prompt_len for x in s.running)]
    assert sorted(d[0] for d in b.decodes) == sorted(expect)
    # total within budget whenever the decodes alone fit; chunks of distinct requests
    if len(b.decodes) <= s.tau:
        assert b.n_tokens <= s.tau
    assert len({p[0] for p in b.prefills}) == len(b.prefills)
    if s.max_chunks:
        assert len(b.prefills) <= s.max_chunks
    for req, start, n, bt in b.prefills:
        assert n > 0 and start + n <= [r for r in s.running if r.req == req][0].prompt_len
        assert len(bt) * page_size >= start + n
    # only the last chunk of a batch may stop short of its prompt's end
    for req, start, n, bt in b.prefills[:-1]:
        assert start + n == [r for r in s.running if r.req == req][0].prompt_len
    # block tables: pages distinct across requests, slot ctx covered
    seen = set()
    for r in s.running:
        assert not (set(r.pages) & seen)
        seen |= set(r.pages)
    for req, ctx, bt in b.decodes:
        assert len(bt) * page_size > ctx
    assert len(seen) + s.pool.n_free() == total_pages


def check_admission(s, b, now, before, waiting_before):
    """Admissions follow the flowchart: the ongoing prompt's chunk comes first,
    new requests are taken first-come-first-served, and the batch stops
    admitting only when the budget is spent, the chunk cap is reached or the
    next ready request cannot be allocated."""
    new = [p for p in b.prefills if p[1] == 0 and p[0] not in before]
    cont = [p for p in b.prefills if p not in new]
    assert b.prefills == cont + new and len(cont) <= 1
    ready = sorted((r for r in waiting_before if r.arrival <= now), key=lambda r: (r.arrival, r.req))
    assert [p[0] for p in new] == [r.req for r in ready[:len(new)]]
    if s.max_chunks == 1 and cont:
        assert not new
        return
    rest = [r for r in ready[len(new):]]
    if rest and b.n_tokens < s.tau and not (s.max_chunks and len(b.prefills) >= s.max_chunks):
        head = rest[0]
        need = -(-head.prompt_len // s.page_size) + 1
        assert s.pool.n_free() < need or len(s.running) >= s.max_batch


@pytest.mark.parametrize("max_chunks", [0, 1, 2])
@pytest.mark.parametrize("tau", [128, 256, 512, 1024])
def test_invariants_on_lognormal_trace(tau, max_chunks):
    trace = synth.request_trace(3, 48, rate=40.0, prompt_median=300, prompt_clip=(8, 2000),
                                out_median=20, out_clip=(1, 80))
    s, steps = run_trace(trace, tau=tau, max_chunks=max_chunks)
    assert len(s.finished) == len(trace)
    # first-come-first-served: admission order follows (arrival, id)
    admitted = []
    for _, b in steps:
        for p in b.prefills:
            if p[1] == 0:
                admitted.append(p[0])
    order = [r.req for r in sorted(trace, key=lambda r: (r.arrival, r.req))]
    assert admitted == order
    # every request produced exactly output_len tokens
    for r in s.finished:
        assert len(r.tokens) == r.output_len


def test_pages_lowest_first_and_returned():
    s = osch.StallFreeScheduler(128, 128, 16, 10, 4)
    s.add(0, 0.0, 40, 2)
    b = s.next(0.0)
    assert b.prefill[3] == [0, 1, 2]
    s.commit([5])
    b = s.next(0.0)  # decode at ctx 40 fits page 2 (slots 32..47)
    assert b.decodes == [(0, 40, [0, 1, 2])]
    s.commit([5])
    assert s.pool.n_free() == 10 and s.idle()


def test_decode_takes_page_on_boundary_and_pool_exhaustion_errors():
    s = osch.StallFreeScheduler(128, 128, 16, 3, 4)
    s.add(0, 0.0, 32, 5)
    s.next(0.0)
    s.commit([1])
    b = s.next(0.0)  # ctx 32 needs a third page
    assert b.decodes[0][2] == [0, 1, 2]
    s.commit([1])
    for _ in range(14):
        s.next(0.0)
        s.commit([1]) if not s.idle() else None
    # a prompt that needs more pages than exist is never admitted
    s2 = osch.StallFreeScheduler(128, 128, 16, 2, 4)
    s2.add(0, 0.0, 32, 2)
    assert s2.next(0.0).prefill is None


def test_exhaustion_during_decode_raises():
    s = osch.StallFreeScheduler(128, 128, 16, 3, 4)
    s.add(0, 0.0, 16, 40)
    s.next(0.0)
    s.commit([1])
    with pytest.raises(osch.NoPages):
        for _ in range(40):
            s.next(0.0)
            s.commit([1])


def test_max_batch_caps_running_set():
    trace = [synth.TraceRequest(i, 0.0, 20, 50) for i in range(10)]
    s, steps = run_trace(trace, tau=128, max_batch=3)
    assert max(len(b.decodes) for _, b in steps) <= 3
    assert len(steps[0][1].prefills) == 3  # three 20-token prompts share the first batch


def test_admission_loop_fills_leftover_budget():
    s = osch.StallFreeScheduler(256, 128, 16, 1000, 16)
    for i, n in enumerate((100, 60, 50, 200)):
        s.add(i, 0.0, n, 3)
    b = s.next(0.0)
    # 100 + 60 + 50 fit whole, the fourth gets the 46 tokens left and stays unfinished
    assert [p[:3] for p in b.prefills] == [(0, 0, 100), (1, 0, 60), (2, 0, 50), (3, 0, 46)]
    assert b.n_tokens == 256 and b.logit_rows == 4
    s.commit([9, 9, 9, 9])
    b = s.next(0.0)
    # three decodes, then the unfinished prompt's next chunk (its remaining 154)
    assert [d[0] for d in b.decodes] == [0, 1, 2]
    assert [p[:3] for p in b.prefills] == [(3, 46, 154)]
    # the one-chunk reading leaves the budget unused instead
    s1 = osch.StallFreeScheduler(256, 128, 16, 1000, 16, max_chunks=1)
    for i, n in enumerate((100, 60, 50, 200)):
        s1.add(i, 0.0, n, 3)
    assert [p[:3] for p in s1.next(0.0).prefills] == [(0, 0, 100)]


def test_admission_stops_at_first_request_that_cannot_allocate():
    # first come, first served: a small later request does not overtake a big one
    s = osch.StallFreeScheduler(512, 128, 16, 12, 16)
    s.add(0, 0.0, 64, 4)     # 4 pages + 1
    s.add(1, 0.0, 200, 4)    # 13 pages + 1: never fits the 8 pages left
    s.add(2, 0.0, 16, 4)     # would fit
    b = s.next(0.0)
    assert [p[0] for p in b.prefills] == [0]


def test_tokens_follow_rows():
    s = osch.StallFreeScheduler(128, 128, 16, 100, 4)
    s.add(0, 0.0, 5, 3, prompt_tokens=[10, 11, 12, 13, 14])
    b = s.next(0.0)
    assert b.tokens == [10, 11, 12, 13, 14]
    s.commit([99])
    s.add(1, 0.0, 2, 2, prompt_tokens=[20, 21])
    b = s.next(0.0)
    assert b.tokens == [20, 21, 99]
