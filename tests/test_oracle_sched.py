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
    with open(os.path.join(GOLDEN, "figure4_schedule.json")) as f:
        g = json.load(f)
    s = osch.StallFreeScheduler(g["tau"], g["tile"], g["page_size"], g["num_pages"], g["max_batch"])
    for r in g["requests"]:
        s.add(r["req"], r["arrival"], r["prompt_len"], r["output_len"])
    for it in g["iterations"]:
        b = s.next(it["now"])
        pre = list(b.prefill[:3]) if b.prefill else None
        assert pre == it["prefill"], it
        assert [d[0] for d in b.decodes] == it["decodes"], it
        s.commit([7] * ((1 if b.prefill else 0) + len(b.decodes)))
    assert [r.req for r in s.running] == [1]  # B started one iteration after A


def test_budget_rounds_down_to_tile():
    assert osch.round_budget(512, 128) == 512
    assert osch.round_budget(600, 128) == 512
    with pytest.raises(ValueError):
        osch.round_budget(100, 128)


def run_trace(trace, tau=256, tile=128, page_size=16, num_pages=4000, max_batch=64, dt=0.01,
              check=True):
    s = osch.StallFreeScheduler(tau, tile, page_size, num_pages, max_batch)
    for r in trace:
        s.add(r.req, r.arrival, r.prompt_len, r.output_len)
    now, steps = 0.0, []
    total_pages = num_pages
    while not s.idle():
        before = {r.req: (r.prefill_done, r.generated) for r in s.running}
        b = s.next(now)
        steps.append((now, b))
        if check:
            check_batch(s, b, before, page_size, total_pages)
        s.commit([1] * ((1 if b.prefill else 0) + len(b.decodes)))
        now += dt if b.n_tokens else 0.5
        assert len(steps) < 200000
    return s, steps


def check_batch(s, b, before, page_size, total_pages):
    # every prefill-complete running request decodes in every batch (decodes never stall)
    expect = [r for r, (p, g) in before.items()
              if any(x.req == r and p == x.prompt_len for x in s.running)]
    assert sorted(d[0] for d in b.decodes) == sorted(expect)
    # at most one chunk; total within budget whenever the decodes alone fit
    if len(b.decodes) <= s.tau:
        assert b.n_tokens <= s.tau
    if b.prefill:
        req, start, n, bt = b.prefill
        assert n > 0 and start + n <= [r for r in s.running if r.req == req][0].prompt_len
        assert len(bt) * page_size >= start + n
    # block tables: pages distinct across requests, slot ctx covered
    seen = set()
    for r in s.running:
        assert not (set(r.pages) & seen)
        seen |= set(r.pages)
    for req, ctx, bt in b.decodes:
        assert len(bt) * page_size > ctx
    assert len(seen) + s.pool.n_free() == total_pages


@pytest.mark.parametrize("tau", [128, 256, 512, 1024])
def test_invariants_on_lognormal_trace(tau):
    trace = synth.request_trace(3, 48, rate=40.0, prompt_median=300, prompt_clip=(8, 2000),
                                out_median=20, out_clip=(1, 80))
    s, steps = run_trace(trace, tau=tau)
    assert len(s.finished) == len(trace)
    # first-come-first-served: admission order follows (arrival, id)
    admitted = []
    for _, b in steps:
        if b.prefill and b.prefill[1] == 0:
            admitted.append(b.prefill[0])
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


def test_tokens_follow_rows():
    s = osch.StallFreeScheduler(128, 128, 16, 100, 4)
    s.add(0, 0.0, 5, 3, prompt_tokens=[10, 11, 12, 13, 14])
    b = s.next(0.0)
    assert b.tokens == [10, 11, 12, 13, 14]
    s.commit([99])
    s.add(1, 0.0, 2, 2, prompt_tokens=[20, 21])
    b = s.next(0.0)
    assert b.tokens == [20, 21, 99]
