"""The Yi-34B shape (H = 7168, 56 query / 8 KV heads of 128, FFN 20480):
a long prompt prefilled in chunks with 128 piggybacked decodes.

* layers 0 and 1 against the oracle (max-abs 0.1, relative L2 1e-2; the
  absolute bound is wider than the Mistral-shaped layers' 3e-2 because fp16
  rounding of the stored activations alone exceeds 3e-2 at this width, as
  test_yi_tolerance.py shows) over the prompt's first two 512-token
  chunks, each step carrying all 128 decodes (contexts uniform in
  [512, 8192], random histories, the same context in both steps);
* the full 60-layer model: the prompt prefilled in 512-token chunks with
  piggybacked decodes equals the same prompt prefilled in one step (relative
  L2 <= 1e-3 over every row, and over the last row's logits).
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

# max-abs bound at this shape: rounding the stored activations to fp16 alone
# exceeds 3e-2 here (see test_yi_tolerance.py); relative L2 as stated
MAX_ABS, REL_L2 = 0.1, 1e-2
PS = 16
CHUNK = 512


def assert_close(got, ref, what, max_abs=MAX_ABS, rel_l2=REL_L2):
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= max_abs and rel <= rel_l2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"


def test_first_two_chunks_with_all_decodes_layers_0_1():
    dims = dataclasses.replace(synth.YI_34B, n_layers=2, vocab=0)
    m, kept = harness.load_synthetic_model(0, dims, max_tokens=CHUNK + 128, max_decodes=128,
                                           keep_layers=(0, 1))
    gen = synth.generator(1)
    ctxs = synth.uniform_int(gen, 128, 512, 8192)
    prompt = synth.normal(gen, (2 * CHUNK, dims.hidden), dtype=torch.bfloat16)
    dec_in = synth.normal(gen, (2, 128, dims.hidden), dtype=torch.bfloat16)
    n_pages = sum(c // PS + 1 for c in ctxs) + 2 * CHUNK // PS + 8
    kv = sar.KVCache(m, PS, n_pages)
    alloc = harness.PageAllocator(range(n_pages))
    dec_bt = []
    for i, c in enumerate(ctxs):
        bt = alloc.take(c // PS + 1)
        for l, (k, v) in enumerate(synth.decode_history(1000 + i, 2, c, dims)):
            harness.write_history(kv, dims, l, k, v, bt)
        dec_bt.append(bt)
    pbt = alloc.take(2 * CHUNK // PS)
    outs = []
    for s in range(2):
        # both steps carry the decodes at the same context (the slot is rewritten)
        decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(ctxs)]
        x = torch.cat([prompt[s * CHUNK:(s + 1) * CHUNK], dec_in[s]]).cuda()
        lo = torch.empty(2, CHUNK + 128, dims.hidden, dtype=torch.float32, device="cuda")
        m.step(kv, sar.Batch((0, s * CHUNK, CHUNK, pbt), decs), x, layer_out=lo)
        outs.append(lo.cpu().numpy().astype(np.float64))
    m.sync_status()
    layers = [om.layer_weights_np(kept[0]), om.layer_weights_np(kept[1])]
    ref, _ = om.forward(layers, dims, om.to_np(prompt))
    for s in range(2):
        for l in range(2):
            assert_close(outs[s][l, :CHUNK], ref[l][s * CHUNK:(s + 1) * CHUNK], f"chunk {s} layer {l}")
    # decode rows: independent of the chunk and of each other, so the oracle
    # takes them 32 decodes (both steps' rows) at a time
    got = np.stack([outs[s][:, CHUNK:] for s in range(2)])  # [step, layer, decode, H]
    want = np.empty_like(got)
    for g0 in range(0, 128, 32):
        parts = []
        for i in range(g0, g0 + 32):
            hist = [om.LayerCache(om.to_np(k), om.to_np(v))
                    for k, v in synth.decode_history(1000 + i, 2, ctxs[i], dims)]
            for s in range(2):
                parts.append(om.Part(x=om.to_np(dec_in[s, i:i + 1]), lo=ctxs[i], given=hist))
        r, _ = om.hybrid_step(layers, None, dims, parts)
        for l in range(2):
            want[:, l, g0:g0 + 32] = r[l].reshape(32, 2, dims.hidden).transpose(1, 0, 2)
    for s in range(2):
        for l in range(2):
            assert_close(got[s, l], want[s, l], f"decodes step {s} layer {l}")


def test_full_depth_chunked_prefill_equals_one_step():
    dims = synth.YI_34B
    n_dec = 8
    m, _ = harness.load_synthetic_model(0, dims, max_tokens=2048, max_decodes=n_dec)
    tokens, ctxs = synth.long_prompt_case(0, dims, prompt_len=2048, n_decode=n_dec, ctx_range=(512, 2048))
    n_pages = 2 * 2048 // PS + sum(c // PS + 1 for c in ctxs) + 8
    kv = sar.KVCache(m, PS, n_pages)
    gen = synth.generator(2, "cuda")
    for l in range(dims.n_layers):  # random histories everywhere; prompt pages are rewritten
        for kind in (0, 1):
            pv = harness.page_view(kv, l, kind, dims)
            pv.copy_(torch.randn(pv.shape, generator=gen, device="cuda").to(pv.dtype))
    alloc = harness.PageAllocator(range(n_pages))
    bt_one, bt_chunked = alloc.take(2048 // PS), alloc.take(2048 // PS)
    dec_bt = [alloc.take(c // PS + 1) for c in ctxs]
    tok = tokens.cuda()
    one = torch.empty(2048, dims.hidden, dtype=torch.float32, device="cuda")
    one_logits = torch.empty(1, dims.vocab, dtype=torch.float32, device="cuda")
    m.step(kv, sar.Batch((0, 0, 2048, bt_one), [], in_kind=sar.SAR_IN_TOKENS), tok, hidden_out=one,
           logits_out=one_logits)
    rows = []
    logits = torch.empty(1 + n_dec, dims.vocab, dtype=torch.float32, device="cuda")
    dec_tok = torch.arange(n_dec, dtype=torch.int32, device="cuda") * 7 + 3
    for s in range(0, 2048, CHUNK):
        decs = [(100 + i, c, dec_bt[i]) for i, c in enumerate(ctxs)]
        hid = torch.empty(CHUNK + n_dec, dims.hidden, dtype=torch.float32, device="cuda")
        m.step(kv, sar.Batch((1, s, CHUNK, bt_chunked), decs, in_kind=sar.SAR_IN_TOKENS),
               torch.cat([tok[s:s + CHUNK], dec_tok]), hidden_out=hid, logits_out=logits)
        rows.append(hid[:CHUNK].clone())
    m.sync_status()
    torch.cuda.synchronize()
    chunked = torch.cat(rows).double()
    ref = one.double()
    rel = ((chunked - ref).norm() / ref.norm()).item()
    lg, lr = logits[0].double(), one_logits[0].double()
    rel_logits = ((lg - lr).norm() / lr.norm()).item()
    print(f"chunked vs one step: hidden rel-L2 {rel:.3e}, logits rel-L2 {rel_logits:.3e}")
    assert rel <= 1e-3, rel
    assert rel_logits <= 1e-3, rel_logits
    assert torch.isfinite(logits).all()
