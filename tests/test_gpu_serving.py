"""The 32-layer Mistral-7B-shaped model driven by the stall-free scheduler:
token inputs, greedy sampling, wall-clock arrivals from a Poisson/lognormal
trace.  Checks: the first chunk's per-layer hidden states against the oracle
(layers 0 and 1), the scheduler decisions of the GPU run replayed bit for bit
by the oracle scheduler from the logged times, and every request completing
with its output length."""

import numpy as np
import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth
from chunked_prefill_hybrid_sar_gb300 import harness, serve
from oracle import model as om
from oracle import sched as osch

pytestmark = pytest.mark.gpu


def serving_trace():
    return synth.request_trace(0, 256, rate=4.0, prompt_median=1024, prompt_clip=(64, 8192),
                               out_median=256, out_clip=(16, 1024))


@pytest.fixture(scope="module")
def mistral32():
    dims = synth.MISTRAL_7B
    m, kept = harness.load_synthetic_model(0, dims, max_tokens=1024, max_decodes=256,
                                           keep_layers=(0, 1, "head"))
    kv = sar.KVCache(m, 16, 6000)
    return dims, m, kv, kept


def test_first_chunk_layers_match_oracle(mistral32):
    dims, m, kv, kept = mistral32
    toks = synth.prompt_tokens(1, serving_trace()[:1], dims.vocab)[0][:512]
    n = len(toks)
    bt = list(range(5900, 5900 + (n + 15) // 16))
    x = torch.tensor(toks, dtype=torch.int32, device="cuda")
    lo = torch.empty(dims.n_layers, n, dims.hidden, dtype=torch.float32, device="cuda")
    logits = torch.empty(1, dims.vocab, dtype=torch.float32, device="cuda")
    m.step(kv, sar.Batch((0, 0, n, bt), [], in_kind=sar.SAR_IN_TOKENS), x, layer_out=lo, logits_out=logits)
    m.sync_status()
    torch.cuda.synchronize()
    x0 = om.to_np(kept["head"]["embed"][torch.tensor(toks)])
    layers = [om.layer_weights_np(kept[0]), om.layer_weights_np(kept[1])]
    outs, _ = om.forward(layers, dims, x0)
    for l in range(2):
        got = lo[l].cpu().numpy().astype(np.float64)
        err = np.abs(got - outs[l]).max()
        rel = np.linalg.norm(got - outs[l]) / np.linalg.norm(outs[l])
        assert err <= 3e-2 and rel <= 1e-2, (l, err, rel)
    assert torch.isfinite(logits).all()


def test_trace_runs_and_replays_bit_exactly(mistral32):
    dims, m, kv, _ = mistral32
    # the first 12 requests, arrivals compressed 50x and outputs capped so the test takes seconds
    trace = [synth.TraceRequest(r.req, r.arrival / 50.0, min(r.prompt_len, 1500), min(r.output_len, 24))
             for r in serving_trace()[:12]]
    toks = synth.prompt_tokens(1, trace, dims.vocab)
    res = serve.run_trace(m, kv, trace, toks, tau=512)
    m.sync_status()
    assert res.steps > 0
    # replay: the oracle scheduler, same times, same sampled tokens -> same batches
    o = osch.StallFreeScheduler(512, 128, kv.page_size, kv.num_pages, 256)
    for r in trace:
        o.add(r.req, r.arrival, r.prompt_len, r.output_len, toks[r.req])
    for i, now in enumerate(res.now_log):
        ob = o.next(now)
        chunks, decs = res.batches[i]
        assert [tuple(c) for c in chunks] == [tuple(c) for c in ob.prefills], i
        assert decs == ob.decodes, i
        o.commit(res.sampled[i])
    assert o.idle()
    assert sorted(len(r.tokens) for r in o.finished) == sorted(r.output_len for r in trace)
    summary = res.summary()
    assert summary["ttft_p50_s"] is not None and summary["tbt_p50_s"] is not None
