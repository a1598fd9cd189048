"""Sliding-window attention through the C ABI against the oracle.

Mistral-7B's attention is listed as GQA with a sliding window (Sarathi-Serve
digest, appendix table of evaluated models); a query at position p sees the
keys at positions (p - W, p].  The chunk rows run on the tcgen05 chunk kernel
(head_dim 128) or the warp-MMA one (head_dim 64), the decode rows on the paged
decode kernel; windows below, at and above the 128-key block and the 16-key
page exercise the block skip, whole blocks outside a row's window and the
per-key mask.  Bars as for the full-causal step: per-layer hidden max-abs
<= 3e-2 and relative L2 <= 1e-2; GPU chunked vs unchunked relative L2 <= 1e-3.
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


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref).max()
    r = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS and r <= REL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {r:.3e}"


def np64(t):
    return om.to_np(t)


# ---------------------------------------------------------------- head_dim 128 (tcgen05 chunk kernel)

@pytest.fixture(scope="module")
def small_case():
    return synth.window_case(0, prompt_len=600)


def _small_run(case, window, page_size, chunks, with_decodes=True):
    """Runs the prompt in ``chunks`` (boundaries), the last chunk with the
    decodes piggybacked unless ``with_decodes`` is false; returns (hidden rows
    of every step, model dims)."""
    dims = dataclasses.replace(case["dims"], sliding_window=window)
    m = harness.load_model(dims, case["layers"], None, max_tokens=512, max_decodes=8)
    ps = page_size
    n_pages = sum((c + 1 + ps - 1) // ps for c in case["ctxs"]) + 600 // ps + 4
    kv = sar.KVCache(m, ps, n_pages)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(3), n_pages))
    dec_bt = []
    for i, c in enumerate(case["ctxs"]):
        bt = alloc.take((c + 1 + ps - 1) // ps)
        k, v = case["histories"][i]
        harness.write_history(kv, dims, 0, k, v, bt)
        dec_bt.append(bt)
    pbt = alloc.take((600 + ps - 1) // ps)
    prompt = case["prompt"]
    outs = []
    for a, b in zip(chunks[:-1], chunks[1:]):
        last = b == chunks[-1] and with_decodes
        decs = [(10 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])] if last else []
        x = prompt[a:b]
        if last:
            x = torch.cat([x, case["decode_inputs"]])
        hid = torch.empty(x.shape[0], dims.hidden, dtype=torch.float32, device="cuda")
        m.step(kv, sar.Batch((0, a, b - a, pbt), decs), x.cuda().contiguous(), hidden_out=hid)
        m.sync_status()
        outs.append(hid)
    torch.cuda.synchronize()
    res = [o.cpu() for o in outs]
    kv.close()
    m.close()
    return res, dims


def _small_ref(case, dims, start):
    w = om.layer_weights_np(case["layers"][0])
    parts = [om.Part(x=np64(case["prompt"]), lo=start, is_prefill=True)]
    for i, c in enumerate(case["ctxs"]):
        k, v = case["histories"][i]
        parts.append(om.Part(x=np64(case["decode_inputs"][i:i + 1]), lo=c,
                             given=[om.LayerCache(np64(k), np64(v))]))
    ref, _ = om.hybrid_step([w], None, dims, parts)
    return ref[0]


@pytest.mark.parametrize("window,page_size", [(1, 16), (100, 16), (129, 16), (300, 32), (100, 64), (4096, 16)])
def test_windowed_step_head_dim_128(small_case, window, page_size):
    # second chunk [256, 600): three query tiles, the last one ragged (88 rows)
    outs, dims = _small_run(small_case, window, page_size, (0, 256, 600))
    ref = _small_ref(small_case, dims, 256)
    got = outs[-1].numpy()
    lp = 600 - 256
    assert_close(got[:lp], ref[:lp], what=f"W={window} chunk rows")
    assert_close(got[lp:], ref[lp:], what=f"W={window} decode rows")


@pytest.mark.parametrize("window", [100, 300])
def test_windowed_step_large_scores_head_dim_128(small_case, window):
    # Wq and Wk scaled by 6: scores large enough that a row's running maximum
    # grows past the rescale threshold after a block in which one key half was
    # still entirely outside the window (the other half already in O)
    case = dict(small_case)
    case["layers"] = [dict(w) for w in small_case["layers"]]
    for n in ("wq", "wk"):
        case["layers"][0][n] = (small_case["layers"][0][n].float() * 6).to(torch.bfloat16)
    outs, dims = _small_run(case, window, 16, (0, 256, 600))
    ref = _small_ref(case, dims, 256)
    got = outs[-1].numpy()
    lp = 600 - 256
    assert_close(got[:lp], ref[:lp], what=f"W={window} chunk rows")
    assert_close(got[lp:], ref[lp:], what=f"W={window} decode rows")


def test_window_changes_the_result_head_dim_128(small_case):
    # the windowed step differs from the full-causal oracle by several times the bar
    outs, dims = _small_run(small_case, 100, 16, (0, 256, 600))
    full = _small_ref(small_case, dataclasses.replace(dims, sliding_window=0), 256)
    assert np.abs(outs[-1].numpy() - full).max() > 3 * MAX_ABS


def test_windowed_chunked_equals_unchunked_head_dim_128(small_case):
    base, _ = _small_run(small_case, 129, 16, (0, 512), with_decodes=False)
    base = base[0].double()
    for chunks in ((0, 128, 512), (0, 200, 384, 512)):
        outs, _ = _small_run(small_case, 129, 16, chunks, with_decodes=False)
        rows = torch.cat([o[:b - a] for o, a, b in zip(outs, chunks[:-1], chunks[1:])]).double()
        rel = ((rows - base).norm() / base.norm()).item()
        assert rel <= 1e-3, (chunks, rel)


# ---------------------------------------------------------------- head_dim 64 (warp-MMA chunk kernel)

@pytest.fixture(scope="module", params=[sar.SAR_STORAGE_F16, sar.SAR_STORAGE_BF16], ids=["f16", "bf16"])
def tiny_w(request):
    case = synth.tiny_case(0, dtype=torch.bfloat16)
    dims = dataclasses.replace(case["dims"], sliding_window=100)
    m = harness.load_model(dims, case["layers"], None, max_tokens=512, max_decodes=8, storage=request.param)
    w = om.layer_weights_np(case["layers"][0])
    yield case, dims, m, w
    m.close()


def test_tiny_windowed_two_chunks_with_piggybacked_decodes(tiny_w):
    case, dims, m, w = tiny_w
    kv = sar.KVCache(m, 16, 256)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(1), 256))
    pbt = alloc.take(32)
    dbt = [alloc.take(20) for _ in case["ctxs"]]
    for i, c in enumerate(case["ctxs"]):  # decode histories from their own prompts, windowed too
        m.step(kv, sar.Batch((10 + i, 0, c, dbt[i]), []), case["decode_prompts"][i].cuda())
    for step in range(2):
        b = sar.Batch((0, step * 256, 256, pbt), [(10 + i, c + step, dbt[i]) for i, c in enumerate(case["ctxs"])])
        x = torch.cat([case["prompt"][step * 256:(step + 1) * 256]] +
                      [case["decode_inputs"][step][i] for i in range(4)]).cuda()
        hid = torch.empty(260, dims.hidden, dtype=torch.float32, device="cuda")
        m.step(kv, b, x, hidden_out=hid)
        m.sync_status()
        parts = [om.Part(x=np64(case["prompt"][: (step + 1) * 256]), lo=step * 256, is_prefill=True)]
        for i, c in enumerate(case["ctxs"]):
            xs = [case["decode_prompts"][i]] + [case["decode_inputs"][s][i] for s in range(step + 1)]
            parts.append(om.Part(x=np64(torch.cat(xs)), lo=c + step))
        ref, _ = om.hybrid_step([w], None, dims, parts)
        assert_close(hid.cpu(), ref[0], what=f"step {step}")
    kv.close()


def test_tiny_windowed_chunked_equals_unchunked(tiny_w):
    case, dims, m, w = tiny_w
    prompt = case["prompt"].cuda()
    outs = []
    for chunks in ((0, 512), (0, 256, 512), (0, 96, 160, 512)):
        kv = sar.KVCache(m, 16, 64)
        bt = list(range(32))
        rows = []
        for a, bnd in zip(chunks[:-1], chunks[1:]):
            hid = torch.empty(bnd - a, dims.hidden, dtype=torch.float32, device="cuda")
            m.step(kv, sar.Batch((0, a, bnd - a, bt), []), prompt[a:bnd].contiguous(), hidden_out=hid)
            rows.append(hid)
        outs.append(torch.cat(rows).double())
        kv.close()
    for o in outs[1:]:
        rel = ((o - outs[0]).norm() / outs[0].norm()).item()
        assert rel <= 1e-3, rel


# ---------------------------------------------------------------- Mistral-shaped layer

@pytest.fixture(scope="module")
def mistral_case():
    return synth.mistral_layer_case(0, starts=(1536,))


@pytest.mark.parametrize("window", [1000, 4096])
def test_mistral_layer_windowed_step(mistral_case, window):
    case = mistral_case
    dims = dataclasses.replace(case["dims"], sliding_window=window)
    m = harness.load_model(dims, case["layers"], case["head"], max_tokens=512, max_decodes=64)
    ps = 16
    need = sum((c + 1 + ps - 1) // ps for c in case["ctxs"]) + 2048 // ps
    kv = sar.KVCache(m, ps, need + 8)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(7), need + 8))
    dec_bt = []
    for i, c in enumerate(case["ctxs"]):
        bt = alloc.take((c + 1 + ps - 1) // ps)
        k, v = case["histories"][i]
        harness.write_history(kv, dims, 0, k, v, bt)
        dec_bt.append(bt)
    start, lp = 1536, case["lp"]
    bt = alloc.take(2048 // ps)
    prompt = case["prompts"][start]
    for s0 in range(0, start, 512):
        m.step(kv, sar.Batch((0, s0, 512, bt), []), prompt[s0:s0 + 512].cuda())
    decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])]
    x = torch.cat([prompt[start:start + lp], case["decode_inputs"]]).cuda()
    hid = torch.empty(512, dims.hidden, dtype=torch.float32, device="cuda")
    logits = torch.empty(65, dims.vocab, dtype=torch.float32, device="cuda")
    m.step(kv, sar.Batch((0, start, lp, bt), decs), x, hidden_out=hid, logits_out=logits)
    m.sync_status()
    torch.cuda.synchronize()
    w = om.layer_weights_np(case["layers"][0])
    head = om.layer_weights_np(case["head"])
    parts = [om.Part(x=np64(prompt), lo=start, is_prefill=True)]
    for i, c in enumerate(case["ctxs"]):
        k, v = case["histories"][i]
        parts.append(om.Part(x=np64(case["decode_inputs"][i:i + 1]), lo=c,
                             given=[om.LayerCache(np64(k), np64(v))]))
    ref_h, ref_l = om.hybrid_step([w], head, dims, parts)
    got = hid.cpu().numpy()
    assert_close(got[:lp], ref_h[0][:lp], what=f"W={window} chunk rows")
    assert_close(got[lp:], ref_h[0][lp:], what=f"W={window} decode rows")
    assert_close(logits.cpu().numpy(), ref_l, what=f"W={window} logits")
    kv.close()
    m.close()
