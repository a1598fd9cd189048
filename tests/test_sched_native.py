"""The library's C++ stall-free scheduler agrees bit for bit with the oracle's
restatement of Algorithm 3: same batches, same block tables, same input ids."""

import json
import os

import pytest

import chunked_prefill_hybrid_sar_gb300 as sar
import synth
from oracle import sched as osch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def replay(trace, tau, tile=128, page_size=16, num_pages=4000, max_batch=64, dt=0.013,
           with_tokens=False, max_steps=100000, max_chunks=0):
    """Drive both schedulers with the same `now` sequence and sampled tokens."""
    o = osch.StallFreeScheduler(tau, tile, page_size, num_pages, max_batch, max_chunks=max_chunks)
    c = sar.Scheduler(tau, tile, page_size, num_pages, max_batch, max_chunks=max_chunks)
    toks = synth.prompt_tokens(5, trace, 1000) if with_tokens else {}
    for r in trace:
        pt = toks.get(r.req)
        o.add(r.req, r.arrival, r.prompt_len, r.output_len, pt)
        c.add(r.req, r.arrival, r.prompt_len, r.output_len, pt)
    now, steps, multi = 0.0, 0, 0
    while not o.idle():
        ob = o.next(now)
        chunks, decs, tokens, _ = c.next(now)
        assert [tuple(p) for p in chunks] == [tuple(p) for p in ob.prefills], (steps, chunks, ob.prefills)
        assert decs == ob.decodes, steps
        if with_tokens:
            assert tokens == ob.tokens, steps
        multi += len(chunks) > 1
        n = ob.logit_rows
        sampled = [(steps * 7 + i) % 1000 for i in range(n)]
        o.commit(sampled)
        c.commit(sampled)
        now += dt if n else 0.25
        steps += 1
        assert steps < max_steps
    assert c.stats()[:3] == (0, 0, len(trace))
    return steps, multi


def test_figure4_timeline_native():
    with open(os.path.join(GOLDEN, "figure4_schedule.json")) as f:
        g = json.load(f)
    c = sar.Scheduler(g["tau"], g["tile"], g["page_size"], g["num_pages"], g["max_batch"], max_chunks=1)
    for r in g["requests"]:
        c.add(r["req"], r["arrival"], r["prompt_len"], r["output_len"])
    for it in g["iterations"]:
        chunks, decs, _, _ = c.next(it["now"])
        assert (list(chunks[0][:3]) if chunks else None) == it["prefill"]
        assert len(chunks) <= 1
        assert [d[0] for d in decs] == it["decodes"]
        c.commit([7] * (len(chunks) + len(decs)))


def test_figure4_timeline_admission_loop_native():
    with open(os.path.join(GOLDEN, "figure4_schedule_algorithm3.json")) as f:
        g = json.load(f)
    c = sar.Scheduler(g["tau"], g["tile"], g["page_size"], g["num_pages"], g["max_batch"],
                      max_chunks=g["max_chunks"])
    for r in g["requests"]:
        c.add(r["req"], r["arrival"], r["prompt_len"], r["output_len"])
    for it in g["iterations"]:
        chunks, decs, _, _ = c.next(it["now"])
        assert [list(p[:3]) for p in chunks] == it["prefills"]
        assert [d[0] for d in decs] == it["decodes"]
        c.commit([7] * (len(chunks) + len(decs)))


@pytest.mark.parametrize("max_chunks", [0, 1])
@pytest.mark.parametrize("tau", [256, 512, 1024])
def test_native_matches_oracle_on_serving_trace(tau, max_chunks):
    # the serving workload's shape (Poisson arrivals, lognormal lengths), scaled down
    trace = synth.request_trace(0, 64, rate=4.0, prompt_median=1024, prompt_clip=(64, 8192),
                                out_median=64, out_clip=(16, 256))
    replay(trace, tau, dt=0.02, max_chunks=max_chunks)


@pytest.mark.parametrize("max_chunks", [0, 1, 3])
def test_native_matches_oracle_with_prompt_tokens_and_small_pool(max_chunks):
    trace = synth.request_trace(1, 40, rate=50.0, prompt_median=200, prompt_clip=(1, 900),
                                out_median=12, out_clip=(1, 60))
    _, multi = replay(trace, 256, num_pages=120, max_batch=6, with_tokens=True, max_chunks=max_chunks)
    assert (multi > 0) == (max_chunks != 1)  # the admission loop did batch several chunks


def test_native_reports_pool_exhaustion():
    c = sar.Scheduler(128, 128, 16, 3, 4)
    c.add(0, 0.0, 16, 40)
    c.next(0.0)
    c.commit([1])
    with pytest.raises(sar.SarError) as e:
        for _ in range(40):
            c.next(0.0)
            c.commit([1])
    assert e.value.code == 2


def test_commit_needs_one_token_per_row():
    c = sar.Scheduler(128, 128, 16, 8, 4)
    c.add(0, 0.0, 10, 2)
    c.next(0.0)
    with pytest.raises(sar.SarError):
        c.commit([1, 2])
