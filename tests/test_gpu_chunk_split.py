"""Chunk attention with key-range splits (sar_model_set_chunk_split) through
the C ABI against the oracle.

A short chunk deep into a long prompt has few 128-row query tiles; with the
option on, each tile's key blocks are shared out over up to four CTAs whose
unnormalised partial outputs and (running maximum, sum) pairs are merged
afterwards: the same identity the decode split uses, applied to the chunk
rows (Sarathi-Serve digest, section 3: a chunk attends to its prompt's earlier
keys and its own).  Bars: per-layer hidden max-abs <= 3e-2 and relative L2
<= 1e-2 against the oracle; split vs unsplit on the same step, relative L2
<= 1e-3 (one layer: only the summation order differs).
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
PROMPT = 2048


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref).max()
    r = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS and r <= REL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {r:.3e}"


def np64(t):
    return om.to_np(t)


@pytest.fixture(scope="module")
def case():
    return synth.window_case(0, prompt_len=PROMPT)


def scaled(case, f):
    c = dict(case)
    c["layers"] = [dict(w) for w in case["layers"]]
    for n in ("wq", "wk"):
        c["layers"][0][n] = (case["layers"][0][n].float() * f).to(torch.bfloat16)
    return c


def run(case, window, split, chunks, ps=16):
    """The prompt in ``chunks`` (boundaries), the decodes piggybacked on the
    last chunk; returns (last step's hidden rows, dims, that step's batch)."""
    dims = dataclasses.replace(case["dims"], sliding_window=window)
    m = harness.load_model(dims, case["layers"], None, max_tokens=512, max_decodes=8)
    m.set_chunk_split(split)
    n_pages = sum(-(-(c + 1) // ps) for c in case["ctxs"]) + PROMPT // ps + 4
    kv = sar.KVCache(m, ps, n_pages)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(3), n_pages))
    dec_bt = []
    for i, c in enumerate(case["ctxs"]):
        bt = alloc.take(-(-(c + 1) // ps))
        k, v = case["histories"][i]
        harness.write_history(kv, dims, 0, k, v, bt)
        dec_bt.append(bt)
    pbt = alloc.take(PROMPT // ps)
    prompt = case["prompt"]
    for a, b in zip(chunks[:-1], chunks[1:]):
        last = b == chunks[-1]
        decs = [(10 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])] if last else []
        x = prompt[a:b]
        if last:
            x = torch.cat([x, case["decode_inputs"]])
        hid = torch.empty(x.shape[0], dims.hidden, dtype=torch.float32, device="cuda")
        batch = sar.Batch((0, a, b - a, pbt), decs)
        m.step(kv, batch, x.cuda().contiguous(), hidden_out=hid)
        m.sync_status()
    torch.cuda.synchronize()
    out = hid.cpu()
    kv.close()
    m.close()
    return out, dims, batch


def oracle(case, dims, start, end):
    w = om.layer_weights_np(case["layers"][0])
    parts = [om.Part(x=np64(case["prompt"][:end]), lo=start, is_prefill=True)]
    for i, c in enumerate(case["ctxs"]):
        k, v = case["histories"][i]
        parts.append(om.Part(x=np64(case["decode_inputs"][i:i + 1]), lo=c,
                             given=[om.LayerCache(np64(k), np64(v))]))
    ref, _ = om.hybrid_step([w], None, dims, parts)
    return ref[0]


def n_merges(dims, batch):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return sar.plan_inspect(dims, batch, 16, 20000, sms, 512, 8, chunk_split=True)["n_comb"]


# (window, chunk boundaries of the prompt): the last chunk is the one checked
CASES = [
    (0, (0, 512, 1024, 1536, 1792, 2048)),   # two full tiles, 14 and 15 key blocks
    (0, (0, 512, 1024, 1536, 1800, 1990)),   # a ragged second tile, a ragged last key block
    (0, (0, 512, 1024, 1536, 1900, 1950)),   # one ragged tile
    (700, (0, 512, 1024, 1536, 1792, 2048)),  # a window: the shares start at the window's first block
]


@pytest.mark.parametrize("window,chunks", CASES, ids=["full", "ragged", "one_tile", "w700"])
def test_split_step_matches_oracle_and_unsplit(case, window, chunks):
    got, dims, batch = run(case, window, True, chunks)
    assert n_merges(dims, batch) > 0  # the step really is split
    plain, _, _ = run(case, window, False, chunks)
    start, end = chunks[-2], chunks[-1]
    ref = oracle(case, dims, start, end)
    lp = end - start
    assert_close(got[:lp].numpy(), ref[:lp], "split chunk rows")
    assert_close(got[lp:].numpy(), ref[lp:], "decode rows")
    rel = ((got.double() - plain.double()).norm() / plain.double().norm()).item()
    assert rel <= 1e-3, rel


def test_split_with_large_scores(case):
    # Wq and Wk scaled by 6: the shares' maxima differ widely, and a share whose
    # keys all sit far below another's maximum must merge with a vanishing weight
    c = scaled(case, 6)
    chunks = (0, 512, 1024, 1536, 1792, 2048)
    got, dims, batch = run(c, 0, True, chunks)
    assert n_merges(dims, batch) > 0
    ref = oracle(c, dims, 1792, 2048)
    assert_close(got[:256].numpy(), ref[:256], "split chunk rows, large scores")
