"""Batches with several prefill chunks (Algorithm 3's admission loop) through
the C ABI against the oracle.

One batch holds the ongoing prompt's completing chunk, a new prompt whole and
the first chunk of another new prompt, then four decodes: the chunk rows are
stacked in that order, each chunk attends to its own prompt's earlier keys and
its own, and the logits rows are every chunk's last row then every decode
(Sarathi-Serve digest, section 3 flowchart of Algorithm 3).  Run on head_dim
128 (tcgen05 chunk kernel) and head_dim 64 (warp-MMA chunk kernel).  Bars:
per-layer hidden and logits max-abs <= 3e-2, relative L2 <= 1e-2; the
several-chunk batch against the same chunks in separate steps, relative L2
<= 1e-3.
"""

import dataclasses

import numpy as np
import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth
from chunked_prefill_hybrid_sar_gb300 import harness
from oracle import model as om

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 3e-2, 1e-2
PS = 16


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref).max()
    r = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS and r <= REL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {r:.3e}"


def np64(t):
    return om.to_np(t)


@pytest.fixture(scope="module", params=["head_dim128", "head_dim64"])
def mc(request):
    d = synth.SMALL_128_HEAD if request.param == "head_dim128" else dataclasses.replace(synth.TINY, vocab=512)
    case = synth.multi_chunk_case(0, d)
    m = harness.load_model(d, case["layers"], case["head"], max_tokens=512, max_decodes=8)
    yield case, m
    m.close()


def make_kv(case, m):
    dims = case["dims"]
    n_pages = sum(-(-(c + 1) // PS) for c in case["ctxs"]) + sum(-(-p.shape[0] // PS) for p in case["prompts"]) + 8
    kv = sar.KVCache(m, PS, n_pages)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(5), n_pages))
    dec_bt = []
    for i, c in enumerate(case["ctxs"]):
        bt = alloc.take(-(-(c + 1) // PS))
        k, v = case["histories"][i]
        harness.write_history(kv, dims, 0, k, v, bt)
        dec_bt.append(bt)
    pbt = [alloc.take(-(-p.shape[0] // PS)) for p in case["prompts"]]
    return kv, dec_bt, pbt


def run(m, kv, chunks, decs, x, n_logits):
    dims = m.dims
    hid = torch.empty(x.shape[0], dims.hidden, dtype=torch.float32, device="cuda")
    logits = torch.empty(n_logits, dims.vocab, dtype=torch.float32, device="cuda")
    b = sar.Batch(chunks, decs)
    assert b.logit_rows == n_logits
    m.step(kv, b, x.cuda().contiguous(), hidden_out=hid, logits_out=logits)
    m.sync_status()
    torch.cuda.synchronize()
    return hid.cpu().numpy(), logits.cpu().numpy()


def oracle(case, chunks, with_decodes):
    """chunks: (prompt index, start, len) in batch order."""
    w = om.layer_weights_np(case["layers"][0])
    head = om.layer_weights_np(case["head"])
    parts = [om.Part(x=np64(case["prompts"][i][:s + n]), lo=s, is_prefill=True) for i, s, n in chunks]
    if with_decodes:
        for i, c in enumerate(case["ctxs"]):
            k, v = case["histories"][i]
            parts.append(om.Part(x=np64(case["decode_inputs"][i:i + 1]), lo=c,
                                 given=[om.LayerCache(np64(k), np64(v))]))
    h, lg = om.hybrid_step([w], head, case["dims"], parts)
    return h[0], lg


def test_three_chunks_and_decodes(mc):
    case, m = mc
    P = case["prompts"]
    kv, dec_bt, pbt = make_kv(case, m)
    # step 1: the first 128 rows of prompt 0 alone
    run(m, kv, [(0, 0, 128, pbt[0])], [], P[0][:128], 1)
    # step 2: prompt 0 completes, prompt 1 whole, prompt 2's first 50 rows, four decodes
    plan = [(0, 128, 172), (1, 0, 180), (2, 0, 50)]
    chunks = [(i, s, n, pbt[i]) for i, s, n in plan]
    decs = [(10 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])]
    x = torch.cat([P[i][s:s + n] for i, s, n in plan] + [case["decode_inputs"]])
    hid, lg = run(m, kv, chunks, decs, x, 3 + 4)
    ref_h, ref_l = oracle(case, plan, True)
    lp = 172 + 180 + 50
    assert_close(hid[:172], ref_h[:172], "chunk 0 rows")
    assert_close(hid[172:352], ref_h[172:352], "chunk 1 rows")
    assert_close(hid[352:lp], ref_h[352:lp], "chunk 2 rows")
    assert_close(hid[lp:], ref_h[lp:], "decode rows")
    assert_close(lg, ref_l, "logits (each chunk's last row, then the decodes)")
    # step 3: prompt 2 continues from its first chunk's keys
    hid3, lg3 = run(m, kv, [(2, 50, 40, pbt[2])], [], P[2][50:90], 1)
    ref_h3, ref_l3 = oracle(case, [(2, 50, 40)], False)
    assert_close(hid3, ref_h3, "prompt 2 second chunk")
    assert_close(lg3, ref_l3, "prompt 2 second chunk logits")
    kv.close()


def test_several_chunks_equal_separate_steps(mc):
    case, m = mc
    P = case["prompts"]
    plan = [(0, 128, 172), (1, 0, 180), (2, 0, 50)]
    kv, _, pbt = make_kv(case, m)
    run(m, kv, [(0, 0, 128, pbt[0])], [], P[0][:128], 1)
    together, lg = run(m, kv, [(i, s, n, pbt[i]) for i, s, n in plan], [],
                       torch.cat([P[i][s:s + n] for i, s, n in plan]), 3)
    kv.close()
    kv, _, pbt = make_kv(case, m)
    run(m, kv, [(0, 0, 128, pbt[0])], [], P[0][:128], 1)
    alone, lgs = [], []
    for i, s, n in plan:
        h, l1 = run(m, kv, [(i, s, n, pbt[i])], [], P[i][s:s + n], 1)
        alone.append(h)
        lgs.append(l1)
    kv.close()
    alone = np.concatenate(alone)
    rel = np.linalg.norm(together - alone) / np.linalg.norm(alone)
    assert rel <= 1e-3, rel
    lgs = np.concatenate(lgs)
    assert np.linalg.norm(lg - lgs) / np.linalg.norm(lgs) <= 1e-3


def test_chunk_list_is_validated(mc):
    case, m = mc
    kv = sar.KVCache(m, PS, 16)
    x = torch.zeros(40, case["dims"].hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sar.SarError):  # the second chunk's block table is too short
        m.step(kv, sar.Batch([(0, 0, 8, [0]), (1, 0, 32, [1])], []), x)
    with pytest.raises(sar.SarError):  # an empty chunk
        m.step(kv, sar.Batch([(0, 0, 8, [0]), (1, 0, 0, [1])], []), x)
    with pytest.raises(sar.SarError):  # more rows than the workspace holds
        m.step(kv, sar.Batch([(0, 0, 300, list(range(16)) * 2), (1, 0, 300, list(range(16)) * 2)], []), x)
    kv.close()
