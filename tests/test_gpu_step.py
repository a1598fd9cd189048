"""Parity of the hybrid step (through the C ABI) with the oracle.

Bars: per-layer hidden states max-abs <= 3e-2 and relative L2 <= 1e-2 (16-bit
storage, fp32 accumulation and residual); GPU chunked vs GPU unchunked
relative L2 <= 1e-3.  The default storage is fp16; the tiny layer also runs
with bf16 storage.
"""

import numpy as np
import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth
from chunked_prefill_hybrid_sar_gb300 import harness
from oracle import model as om

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 3e-2, 1e-2


def assert_close(got, ref, max_abs=MAX_ABS, rel=REL_L2, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref).max()
    r = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= max_abs and r <= rel, f"{what}: max-abs {err:.3e}, rel-L2 {r:.3e}"


def np64(t):
    return om.to_np(t)


def oracle_intermediates(w, dims, parts):
    """Normed rows, rotated q|k|v rows and attention rows of a one-layer hybrid batch."""
    xs, poss, caches = [], [], []
    for p in parts:
        pre = p.lo - p.given_len
        if pre > 0:
            _, c = om.forward([w], dims, p.x[:pre], p.given)
            c = c[0]
        elif p.given is not None:
            c = p.given[0]
        else:
            c = om.empty_cache(dims)
        caches.append(c)
        xs.append(p.x[pre:])
        poss.append(np.arange(p.lo, p.end))
    x = np.concatenate(xs)
    pos = np.concatenate(poss)
    y = om.rms_norm(x, w["norm1"], dims.rms_eps)
    q, k, v = om.qkv_rope(x, pos, w, dims)
    a = np.empty_like(q)
    r0 = 0
    for p, c in zip(parts, caches):
        r1 = r0 + p.n_rows
        K = np.concatenate([c.k, k[r0:r1]])
        V = np.concatenate([c.v, v[r0:r1]])
        a[r0:r1] = om.attention(q[r0:r1], K, V, pos[r0:r1], np.arange(K.shape[0]))
        r0 = r1
    M = x.shape[0]
    h_mid = x + a.reshape(M, -1) @ w["wo"].T
    y2 = om.rms_norm(h_mid, w["norm2"], dims.rms_eps)
    return y2, np.concatenate([q.reshape(M, -1), k.reshape(M, -1), v.reshape(M, -1)], 1), a.reshape(M, -1)


def debug_tensor(model, which, rows, cols):
    ptr = model.debug_buffer(which)
    return harness.wrap(ptr, rows * cols, sar.storage_dtype(model.storage)).view(rows, cols)


# ---------------------------------------------------------------- tiny layer

@pytest.fixture(scope="module", params=[sar.SAR_STORAGE_F16, sar.SAR_STORAGE_BF16], ids=["f16", "bf16"])
def tiny(request):
    case = synth.tiny_case(0, dtype=torch.bfloat16)
    dims = case["dims"]
    m = harness.load_model(dims, case["layers"], None, max_tokens=512, max_decodes=8, storage=request.param)
    w = om.layer_weights_np(case["layers"][0])
    return case, m, w


def tiny_setup(case, m, n_pages=256, seed=1):
    dims = case["dims"]
    kv = sar.KVCache(m, 16, n_pages)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(seed), n_pages))
    prompt_bt = alloc.take(32)
    dec_bt = [alloc.take(20) for _ in case["ctxs"]]
    for i, c in enumerate(case["ctxs"]):  # decode histories from their own prompts
        m.step(kv, sar.Batch((10 + i, 0, c, dec_bt[i]), []), case["decode_prompts"][i].cuda())
    return kv, prompt_bt, dec_bt


def tiny_parts(case, step):
    parts = [om.Part(x=np64(case["prompt"][: (step + 1) * 256]), lo=step * 256, is_prefill=True)]
    for i, c in enumerate(case["ctxs"]):
        xs = [case["decode_prompts"][i]] + [case["decode_inputs"][s][i] for s in range(step + 1)]
        parts.append(om.Part(x=np64(torch.cat(xs)), lo=c + step))
    return parts


def test_tiny_intermediates_first_step(tiny):
    case, m, w = tiny
    dims = case["dims"]
    kv, pbt, dbt = tiny_setup(case, m)
    b = sar.Batch((0, 0, 256, pbt), [(10 + i, c, dbt[i]) for i, c in enumerate(case["ctxs"])])
    x = torch.cat([case["prompt"][:256]] + [case["decode_inputs"][0][i] for i in range(4)]).cuda()
    m.step(kv, b, x)
    m.sync_status()
    torch.cuda.synchronize()
    y2, qkv, attn = oracle_intermediates(w, dims, tiny_parts(case, 0))
    M = 260
    # the normed-rows buffer holds the second norm (ahead of the FFN) after the step
    assert_close(debug_tensor(m, 0, M, dims.hidden).float().cpu(), y2, what="rmsnorm before FFN")
    qkv32 = harness.wrap(m.debug_buffer(5), M * 3 * dims.hidden, torch.float32).view(M, 3 * dims.hidden)
    assert_close(qkv32.cpu(), qkv, what="qkv+rope")
    got_attn = debug_tensor(m, 2, M, dims.hidden).float().cpu().numpy()
    assert_close(got_attn[:256], attn[:256], what="chunk attention")
    assert_close(got_attn[256:], attn[256:], what="decode attention")
    # the new keys sit in the pages at their slots
    k_pages = harness.read_history(kv, dims, 0, 0, pbt, 256).float().cpu().numpy()
    assert_close(k_pages.reshape(256, -1), qkv[:256, dims.hidden:2 * dims.hidden], what="appended keys")


def test_tiny_two_chunks_with_piggybacked_decodes(tiny):
    case, m, w = tiny
    dims = case["dims"]
    kv, pbt, dbt = tiny_setup(case, m)
    for step in range(2):
        b = sar.Batch((0, step * 256, 256, pbt), [(10 + i, c + step, dbt[i]) for i, c in enumerate(case["ctxs"])])
        x = torch.cat([case["prompt"][step * 256:(step + 1) * 256]] +
                      [case["decode_inputs"][step][i] for i in range(4)]).cuda()
        lo = torch.empty(1, 260, dims.hidden, dtype=torch.float32, device="cuda")
        hid = torch.empty(260, dims.hidden, dtype=torch.float32, device="cuda")
        m.step(kv, b, x, hidden_out=hid, layer_out=lo)
        m.sync_status()
        ref, _ = om.hybrid_step([w], None, dims, tiny_parts(case, step))
        assert_close(lo[0].float().cpu(), ref[0], what=f"step {step} layer 0")
        assert_close(hid.float().cpu(), ref[0], what=f"step {step} hidden")


def test_tiny_chunked_equals_unchunked_on_gpu(tiny):
    case, m, w = tiny
    dims = case["dims"]
    prompt = case["prompt"].cuda()
    outs = []
    for chunks in ((0, 512), (0, 256, 512), (0, 128, 384, 512)):
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


def test_tiny_hybrid_rows_equal_rows_run_alone(tiny):
    """Hybrid batch == serial execution of its parts, on the GPU."""
    case, m, w = tiny
    dims = case["dims"]
    kv, pbt, dbt = tiny_setup(case, m)
    decs = [(10 + i, c, dbt[i]) for i, c in enumerate(case["ctxs"])]
    x = torch.cat([case["prompt"][:256]] + [case["decode_inputs"][0][i] for i in range(4)]).cuda()
    hyb = torch.empty(260, dims.hidden, dtype=torch.float32, device="cuda")
    m.step(kv, sar.Batch((0, 0, 256, pbt), decs), x, hidden_out=hyb)
    alone = []
    hid = torch.empty(256, dims.hidden, dtype=torch.float32, device="cuda")
    m.step(kv, sar.Batch((0, 0, 256, pbt), []), x[:256].contiguous(), hidden_out=hid)
    alone.append(hid)
    for i, d in enumerate(decs):
        h1 = torch.empty(1, dims.hidden, dtype=torch.float32, device="cuda")
        m.step(kv, sar.Batch(None, [d]), x[256 + i:257 + i].contiguous(), hidden_out=h1)
        alone.append(h1)
    alone = torch.cat(alone).double()
    rel = ((hyb.double() - alone).norm() / alone.norm()).item()
    assert rel <= 1e-3, rel


def test_invalid_batches_are_rejected_before_launch(tiny):
    case, m, w = tiny
    kv = sar.KVCache(m, 16, 8)
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sar.SarError):  # block table too short
        m.step(kv, sar.Batch((0, 0, 4, []), []), x)
    with pytest.raises(sar.SarError):  # page id out of range
        m.step(kv, sar.Batch(None, [(0, 3, [99])]), x[:1])
    with pytest.raises(sar.SarError):  # more rows than the workspace holds
        big = torch.zeros(600, 256, dtype=torch.bfloat16, device="cuda")
        m.step(kv, sar.Batch((0, 0, 600, list(range(8)) * 5), []), big)
    with pytest.raises(sar.SarError):  # empty batch
        m.step(kv, sar.Batch(None, []), x)


# ---------------------------------------------------------------- Mistral-shaped layer

@pytest.fixture(scope="module")
def mistral():
    case = synth.mistral_layer_case(0)
    dims = case["dims"]
    m = harness.load_model(dims, case["layers"], case["head"], max_tokens=512, max_decodes=64)
    ps = 16
    need = sum((c + 1 + ps - 1) // ps for c in case["ctxs"]) + 3 * (2048 // ps)
    kv = sar.KVCache(m, ps, need + 8)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(7), need + 8))
    dec_bt = []
    for i, c in enumerate(case["ctxs"]):
        bt = alloc.take((c + 1 + ps - 1) // ps)
        k, v = case["histories"][i]
        harness.write_history(kv, dims, 0, k, v, bt)
        dec_bt.append(bt)
    prompt_bt = {s: alloc.take(2048 // ps) for s in case["starts"]}
    torch.cuda.synchronize()
    w = om.layer_weights_np(case["layers"][0])
    head = om.layer_weights_np(case["head"])
    return case, m, kv, dec_bt, prompt_bt, w, head


@pytest.mark.parametrize("start", [0, 512, 1536])
def test_mistral_layer_hybrid_step(mistral, start):
    case, m, kv, dec_bt, prompt_bt, w, head = mistral
    dims, lp = case["dims"], case["lp"]
    prompt = case["prompts"][start]
    bt = prompt_bt[start]
    for s0 in range(0, start, 512):  # the prompt's earlier chunks
        m.step(kv, sar.Batch((start, s0, 512, bt), []), prompt[s0:s0 + 512].cuda())
    decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])]
    b = sar.Batch((start, start, lp, bt), decs)
    x = torch.cat([prompt[start:start + lp], case["decode_inputs"]]).cuda()
    hid = torch.empty(512, dims.hidden, dtype=torch.float32, device="cuda")
    logits = torch.empty(65, dims.vocab, dtype=torch.float32, device="cuda")
    m.step(kv, b, x, hidden_out=hid, logits_out=logits)
    m.sync_status()
    torch.cuda.synchronize()
    parts = [om.Part(x=np64(prompt), lo=start, is_prefill=True)]
    for i, c in enumerate(case["ctxs"]):
        k, v = case["histories"][i]
        parts.append(om.Part(x=np64(case["decode_inputs"][i:i + 1]), lo=c,
                             given=[om.LayerCache(np64(k), np64(v))]))
    ref_h, ref_l = om.hybrid_step([w], head, dims, parts)
    got = hid.float().cpu().numpy()
    assert_close(got[:lp], ref_h[0][:lp], what="chunk rows")
    assert_close(got[lp:], ref_h[0][lp:], what="decode rows")
    assert_close(logits.cpu().numpy(), ref_l, what="logits")


def test_mistral_layer_launch_orders_give_identical_attention(mistral):
    """The step launches decode attention first and the chunk kernel right
    behind it, without a start wait (it takes the SMs of the decode grid's
    draining tail); kernel-by-kernel profiling keeps the chunk-then-decode
    order.  The attention kernels and their inputs are the same, so the
    attention rows of both orders are bit-identical."""
    case, m, kv, dec_bt, prompt_bt, w, head = mistral
    dims, lp = case["dims"], case["lp"]
    start = 1536
    prompt = case["prompts"][start]
    bt = prompt_bt[start]
    for s0 in range(0, start, 512):
        m.step(kv, sar.Batch((start, s0, 512, bt), []), prompt[s0:s0 + 512].cuda())
    decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])]
    b = sar.Batch((start, start, lp, bt), decs)
    x = torch.cat([prompt[start:start + lp], case["decode_inputs"]]).cuda()
    rows = []
    for prof in (False, True, False):
        m.profile(prof)
        m.step(kv, b, x)
        m.sync_status()
        torch.cuda.synchronize()
        rows.append(debug_tensor(m, 2, lp + len(decs), dims.q_dim).clone())
    m.profile(False)
    m.profile_read()
    assert torch.isfinite(rows[0].float()).all()
    assert torch.equal(rows[0], rows[1]) and torch.equal(rows[0], rows[2])


def test_mistral_layer_attention_overlap_is_identical(mistral):
    """Chunk attention on a second stream, concurrent with decode attention:
    the same kernels write the same disjoint rows, so the step agrees with the
    one-stream step up to the order of the split-K atomic adds in the O and
    down projections (which differs from run to run on one stream too)."""
    case, m, kv, dec_bt, prompt_bt, w, head = mistral
    dims, lp = case["dims"], case["lp"]
    start = 1536
    prompt = case["prompts"][start]
    bt = prompt_bt[start]
    for s0 in range(0, start, 512):
        m.step(kv, sar.Batch((start, s0, 512, bt), []), prompt[s0:s0 + 512].cuda())
    decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(case["ctxs"])]
    b = sar.Batch((start, start, lp, bt), decs)
    x = torch.cat([prompt[start:start + lp], case["decode_inputs"]]).cuda()
    outs = []
    for on in (False, True, False):
        m.set_overlap(on)
        hid = torch.empty(512, dims.hidden, dtype=torch.float32, device="cuda")
        logits = torch.empty(65, dims.vocab, dtype=torch.float32, device="cuda")
        m.step(kv, b, x, hidden_out=hid, logits_out=logits)
        m.sync_status()
        outs.append((hid, logits))
    m.set_overlap(False)
    torch.cuda.synchronize()
    for hid, logits in outs[1:]:
        for got, ref in ((hid, outs[0][0]), (logits, outs[0][1])):
            rel = ((got.double() - ref.double()).norm() / ref.double().norm()).item()
            assert rel <= 1e-4, rel
