"""One step captured as a CUDA graph (sar_graph_*) against the same step
launched kernel by kernel and against the oracle.

The graph keeps its own copy of the step's metadata; ``update`` swaps in the
metadata of another batch with the same plan shape (here: the decodes one
token further, within the same pages).  Bars: the oracle's (per-layer hidden
max-abs <= 3e-2, relative L2 <= 1e-2); graph vs kernel-by-kernel relative L2
<= 1e-3 (the split-K projections add their K ranges atomically, in an order
that differs from run to run; in small steps that includes the QKV
projection, whose k and v are then rounded to 16 bits, so a last-bit
difference can flip a stored key).
"""

import numpy as np
import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth
from chunked_prefill_hybrid_sar_gb300 import harness
from oracle import model as om

pytestmark = pytest.mark.gpu

RUN_TO_RUN = 1e-3


def rel(a, b):
    a, b = a.double(), b.double()
    return ((a - b).norm() / b.norm()).item()


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref).max()
    r = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= 3e-2 and r <= 1e-2, f"{what}: max-abs {err:.3e}, rel-L2 {r:.3e}"


def mistral_kv(case, m, ps=16):
    dims = case["dims"]
    need = sum((c + 2 + ps - 1) // ps for c in case["ctxs"]) + 2048 // ps + 8
    kv = sar.KVCache(m, ps, need)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(7), need))
    dec_bt = []
    for i, c in enumerate(case["ctxs"]):
        bt = alloc.take((c + 2 + ps - 1) // ps)
        k, v = case["histories"][i]
        harness.write_history(kv, dims, 0, k, v, bt)
        dec_bt.append(bt)
    return kv, dec_bt, alloc.take(2048 // ps)


@pytest.fixture(scope="module")
def mistral():
    case = synth.mistral_layer_case(0, starts=(512,))
    m = harness.load_model(case["dims"], case["layers"], case["head"], max_tokens=512, max_decodes=64)
    yield case, m
    m.close()


def test_graph_step_equals_kernel_by_kernel_and_oracle(mistral):
    case, m = mistral
    dims, lp, start = case["dims"], case["lp"], 512
    prompt = case["prompts"][start]
    outs = {}
    for mode in ("eager", "graph"):
        kv, dec_bt, bt = mistral_kv(case, m)
        m.step(kv, sar.Batch((0, 0, 512, bt), []), prompt[:512].cuda())
        decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])]
        b = sar.Batch((0, start, lp, bt), decs)
        x = torch.cat([prompt[start:start + lp], case["decode_inputs"]]).cuda().contiguous()
        hid = torch.empty(512, dims.hidden, dtype=torch.float32, device="cuda")
        logits = torch.empty(65, dims.vocab, dtype=torch.float32, device="cuda")
        if mode == "eager":
            m.step(kv, b, x, hidden_out=hid, logits_out=logits)
        else:
            g = sar.StepGraph(m, kv, b, x, hidden_out=hid, logits_out=logits)
            hid.fill_(float("nan"))
            g.launch()
            torch.cuda.synchronize()
            g.close()
        m.sync_status()
        torch.cuda.synchronize()
        outs[mode] = (hid.cpu(), logits.cpu())
        kv.close()
    assert rel(outs["graph"][0], outs["eager"][0]) <= RUN_TO_RUN
    assert rel(outs["graph"][1], outs["eager"][1]) <= RUN_TO_RUN
    w = om.layer_weights_np(case["layers"][0])
    head = om.layer_weights_np(case["head"])
    parts = [om.Part(x=om.to_np(prompt), lo=start, is_prefill=True)]
    for i, c in enumerate(case["ctxs"]):
        k, v = case["histories"][i]
        parts.append(om.Part(x=om.to_np(case["decode_inputs"][i:i + 1]), lo=c,
                             given=[om.LayerCache(om.to_np(k), om.to_np(v))]))
    ref_h, ref_l = om.hybrid_step([w], head, dims, parts)
    assert_close(outs["graph"][0].numpy(), ref_h[0], "graph hidden rows")
    assert_close(outs["graph"][1].numpy(), ref_l, "graph logits")


def test_graph_update_replays_the_next_decode_step(mistral):
    """A decode-only step captured once, then re-pointed at the decodes one token
    further (same page counts, so the same plan shape) and launched again."""
    case, m = mistral
    dims = case["dims"]
    ctxs = case["ctxs"]
    keep = [i for i, c in enumerate(ctxs) if (c + 1) % 16 != 0]  # ctx+1 stays in the same page count
    runs = {}
    for mode in ("eager", "graph"):
        kv, dec_bt, _ = mistral_kv(case, m)
        hid = torch.empty(len(keep), dims.hidden, dtype=torch.float32, device="cuda")
        logits = torch.empty(len(keep), dims.vocab, dtype=torch.float32, device="cuda")
        x = case["decode_inputs"][keep].cuda().contiguous()
        got = []
        g = None
        for t in range(2):
            b = sar.Batch(None, [(100 + i, ctxs[i] + t, dec_bt[i]) for i in keep])
            if mode == "eager":
                m.step(kv, b, x, hidden_out=hid, logits_out=logits)
            else:
                if g is None:
                    g = sar.StepGraph(m, kv, b, x, hidden_out=hid, logits_out=logits)
                else:
                    g.update(b)
                g.launch()
            torch.cuda.synchronize()
            got.append((hid.cpu().clone(), logits.cpu().clone()))
        if g is not None:
            g.close()
        m.sync_status()
        runs[mode] = got
        kv.close()
    for t in range(2):
        assert rel(runs["graph"][t][0], runs["eager"][t][0]) <= RUN_TO_RUN, t
        assert rel(runs["graph"][t][1], runs["eager"][t][1]) <= RUN_TO_RUN, t
    # the second step differs from the first (the keys written by the first are attended)
    assert rel(runs["graph"][1][0], runs["graph"][0][0]) > RUN_TO_RUN


def test_graph_update_refuses_another_shape(mistral):
    case, m = mistral
    dims = case["dims"]
    kv, dec_bt, bt = mistral_kv(case, m)
    x = case["decode_inputs"][:4].cuda().contiguous()
    hid = torch.empty(4, dims.hidden, dtype=torch.float32, device="cuda")
    g = sar.StepGraph(m, kv, sar.Batch(None, [(100 + i, case["ctxs"][i], dec_bt[i]) for i in range(4)]), x,
                      hidden_out=hid)
    with pytest.raises(sar.SarError):  # three decodes instead of four
        g.update(sar.Batch(None, [(100 + i, case["ctxs"][i], dec_bt[i]) for i in range(3)]))
    with pytest.raises(sar.SarError):  # a chunk added
        g.update(sar.Batch((0, 0, 16, bt), [(100 + i, case["ctxs"][i], dec_bt[i]) for i in range(4)]))
    g.launch()
    torch.cuda.synchronize()
    m.sync_status()
    g.close()
    kv.close()


def test_graph_launch_host_copies_in_and_out(mistral):
    """Host input rows in, the captured step, host logits and hidden rows out."""
    case, m = mistral
    dims, lp, start = case["dims"], case["lp"], 512
    prompt = case["prompts"][start]
    kv, dec_bt, bt = mistral_kv(case, m)
    m.step(kv, sar.Batch((0, 0, 512, bt), []), prompt[:512].cuda())
    decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])]
    b = sar.Batch((0, start, lp, bt), decs)
    x_host = torch.cat([prompt[start:start + lp], case["decode_inputs"]]).contiguous().pin_memory()
    x_dev = torch.zeros_like(x_host, device="cuda")
    hid = torch.empty(512, dims.hidden, dtype=torch.float32, device="cuda")
    logits = torch.empty(65, dims.vocab, dtype=torch.float32, device="cuda")
    g = sar.StepGraph(m, kv, b, x_dev, hidden_out=hid, logits_out=logits)
    h_log = torch.full((65, dims.vocab), float("nan")).pin_memory()
    h_hid = torch.full((512, dims.hidden), float("nan")).pin_memory()
    g.launch_host(x_host, logits_out=h_log, hidden_out=h_hid)
    assert torch.equal(x_dev.cpu(), x_host)
    ref_l, ref_h = logits.cpu(), hid.cpu()
    assert torch.equal(h_log, ref_l) and torch.equal(h_hid, ref_h)
    # greedy token ids instead of logits: each captured row's argmax, lowest index on ties
    toks = torch.full((65,), -1, dtype=torch.int32).pin_memory()
    g.launch_host_tokens(x_host, toks)
    assert torch.equal(toks, logits.cpu().argmax(dim=1).to(torch.int32))
    # enqueued steps (the input copied on the graph's own copy stream while
    # the previous step runs), two graphs of the batch alternating with
    # different input rows, each step waited for one step late: the same token
    # ids as the waited launches of the same inputs
    g.wait()  # nothing enqueued yet
    x_dev2 = torch.zeros_like(x_host, device="cuda")
    logits2 = torch.empty_like(logits)
    g2 = sar.StepGraph(m, kv, b, x_dev2, logits_out=logits2)
    x_host2 = torch.flip(x_host, dims=(1,)).contiguous().pin_memory()
    ref2 = torch.full((65,), -1, dtype=torch.int32).pin_memory()
    g2.launch_host_tokens(x_host2, ref2)
    assert torch.equal(ref2, logits2.cpu().argmax(dim=1).to(torch.int32))
    assert not torch.equal(ref2, toks)
    outs = [torch.full((65,), -1, dtype=torch.int32).pin_memory() for _ in range(6)]
    prev = None
    for i in range(6):
        gi, xi = (g, x_host) if i % 2 == 0 else (g2, x_host2)
        gi.enqueue_host_tokens(xi, outs[i])
        if prev is not None:
            prev.wait()
        prev = gi
    prev.wait()
    for i in range(6):
        assert torch.equal(outs[i], toks if i % 2 == 0 else ref2), i
    assert torch.equal(x_dev.cpu(), x_host) and torch.equal(x_dev2.cpu(), x_host2)
    with pytest.raises(sar.SarError):  # no logits captured: nothing to pick tokens from
        nolog2 = sar.StepGraph(m, kv, b, x_dev2, hidden_out=hid)
        try:
            nolog2.enqueue_host_tokens(x_host2, toks)
        finally:
            nolog2.close()
    g2.close()
    nolog = sar.StepGraph(m, kv, b, x_dev, hidden_out=hid)
    with pytest.raises(sar.SarError):  # no logits captured
        nolog.launch_host_tokens(x_host, toks)
    nolog.close()
    # pageable host buffers take the copy engine instead of the copy kernel
    p_log = torch.full((65, dims.vocab), float("nan"))
    g.launch_host(x_host.clone(), logits_out=p_log)
    assert rel(p_log, ref_l) <= RUN_TO_RUN
    # the same step launched on the device buffers agrees
    eh = torch.empty_like(hid)
    el = torch.empty_like(logits)
    m.step(kv, b, x_dev, hidden_out=eh, logits_out=el)
    torch.cuda.synchronize()
    assert rel(el.cpu(), ref_l) <= RUN_TO_RUN and rel(eh.cpu(), ref_h) <= RUN_TO_RUN
    m.sync_status()
    g.close()
    kv.close()
