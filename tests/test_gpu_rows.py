"""The Mistral-shaped layer stepped at batch sizes on both sides of the GEMM
tile edges (M = Lp + 32 in {128, 255, 256, 257, 384, 511, 512, 1024, 2048}):
32 decodes at context 2048 with random histories plus one chunk at start 0.
Every row of every step is compared with the oracle (same bars as the step
tests).

The oracle runs once, over the longest chunk and the decodes: attention is
causal, so the first Lp rows of a one-shot forward over the longest prompt are
the rows a chunk of Lp rows at start 0 emits, and a decode row depends only on
its own history and input.
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
PS = 16


def assert_close(got, ref, what):
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"


@pytest.fixture(scope="module")
def sweep():
    case = synth.tile_sweep_case(0)
    dims, bd, ctx = case["dims"], len(case["histories"]), case["ctx"]
    m = harness.load_model(dims, case["layers"], None, max_tokens=max(case["rows"]), max_decodes=bd)
    n_pages = bd * (ctx // PS + 1) + max(case["rows"]) // PS + 8
    kv = sar.KVCache(m, PS, n_pages)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(5), n_pages))
    dec_bt = []
    for k, v in case["histories"]:
        bt = alloc.take(ctx // PS + 1)
        harness.write_history(kv, dims, 0, k, v, bt)
        dec_bt.append(bt)
    prompt_bt = alloc.take(max(case["rows"]) // PS)
    torch.cuda.synchronize()
    w = om.layer_weights_np(case["layers"][0])
    chunk_ref, _ = om.forward([w], dims, om.to_np(case["prompt"]))
    parts = [om.Part(x=om.to_np(case["decode_inputs"][i:i + 1]), lo=ctx,
                     given=[om.LayerCache(om.to_np(k), om.to_np(v))])
             for i, (k, v) in enumerate(case["histories"])]
    dec_ref, _ = om.hybrid_step([w], None, dims, parts)
    return case, m, kv, dec_bt, prompt_bt, chunk_ref[0], dec_ref[0]


@pytest.mark.parametrize("M", synth.SWEEP_ROWS)
def test_rows_at_tile_edges_match_oracle(sweep, M):
    case, m, kv, dec_bt, prompt_bt, chunk_ref, dec_ref = sweep
    dims, ctx = case["dims"], case["ctx"]
    bd = len(dec_bt)
    lp = M - bd
    decs = [(100 + i, ctx, dec_bt[i]) for i in range(bd)]
    x = torch.cat([case["prompt"][:lp], case["decode_inputs"]]).cuda()
    hid = torch.empty(M, dims.hidden, dtype=torch.float32, device="cuda")
    m.step(kv, sar.Batch((0, 0, lp, prompt_bt), decs), x, hidden_out=hid)
    m.sync_status()
    torch.cuda.synchronize()
    got = hid.cpu().numpy().astype(np.float64)
    assert_close(got[:lp], chunk_ref[:lp], f"M={M} chunk rows")
    assert_close(got[lp:], dec_ref, f"M={M} decode rows")


@pytest.mark.parametrize("bd", [1, 8, 32])
def test_decode_only_steps_match_oracle(sweep, bd):
    """Decode-only steps (the small-row regime: QKV and gate/up accumulate
    split-K in fp32, then the rotary/append and SwiGLU kernels)."""
    case, m, kv, dec_bt, prompt_bt, chunk_ref, dec_ref = sweep
    dims, ctx = case["dims"], case["ctx"]
    decs = [(100 + i, ctx, dec_bt[i]) for i in range(bd)]
    x = case["decode_inputs"][:bd].cuda().contiguous()
    hid = torch.empty(bd, dims.hidden, dtype=torch.float32, device="cuda")
    m.step(kv, sar.Batch(None, decs), x, hidden_out=hid)
    m.sync_status()
    torch.cuda.synchronize()
    assert_close(hid.cpu().numpy().astype(np.float64), dec_ref[:bd], f"Bd={bd} decode rows")


@pytest.mark.parametrize("storage", [sar.SAR_STORAGE_F16, sar.SAR_STORAGE_BF16], ids=["f16", "bf16"])
def test_small_step_split_path_both_storage_types(storage):
    """A decode-only step of a layer wide enough (H 1024, K = 16 slabs) that the
    small-step QKV and gate/up projections split K, in fp16 and in bf16
    storage (the rotary/append and SwiGLU finishing kernels of each type)."""
    import dataclasses
    dims = synth.Dims(n_layers=1, hidden=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=2048, vocab=0)
    case = synth.window_case(3, d=dims, prompt_len=16, ctxs=(40, 200, 333, 517, 700, 64, 129, 999))
    m = harness.load_model(dims, case["layers"], None, max_tokens=64, max_decodes=8, storage=storage)
    n_pages = sum(c // PS + 1 for c in case["ctxs"]) + 4
    kv = sar.KVCache(m, PS, n_pages)
    alloc = harness.PageAllocator(synth.page_permutation(synth.generator(9), n_pages))
    decs = []
    for i, c in enumerate(case["ctxs"]):
        bt = alloc.take(c // PS + 1)
        k, v = case["histories"][i]
        harness.write_history(kv, dims, 0, k, v, bt)
        decs.append((10 + i, c, bt))
    x = case["decode_inputs"].cuda().contiguous()
    hid = torch.empty(len(decs), dims.hidden, dtype=torch.float32, device="cuda")
    m.step(kv, sar.Batch(None, decs), x, hidden_out=hid)
    m.sync_status()
    torch.cuda.synchronize()
    w = om.layer_weights_np(case["layers"][0])
    parts = [om.Part(x=om.to_np(case["decode_inputs"][i:i + 1]), lo=c,
                     given=[om.LayerCache(om.to_np(k), om.to_np(v))])
             for i, (c, (k, v)) in enumerate(zip(case["ctxs"], case["histories"]))]
    ref, _ = om.hybrid_step([w], None, dims, parts)
    assert_close(hid.cpu().numpy().astype(np.float64), ref[0], f"storage {storage}")
    # the new keys were appended into the pages (rotary applied): read one back
    got_k = harness.read_history(kv, dims, 0, 0, decs[0][2], case["ctxs"][0] + 1)[-1].float().cpu().numpy()
    y = om.rms_norm(om.to_np(case["decode_inputs"][0:1]), w["norm1"], dims.rms_eps)
    k_ref = om.apply_rope((y @ w["wk"].T).reshape(1, dims.n_kv_heads, dims.head_dim), [case["ctxs"][0]],
                          dims.rope_base)[0]
    tol = 2e-2 if storage == sar.SAR_STORAGE_BF16 else 4e-3
    assert np.abs(got_k - k_ref).max() <= tol * max(1.0, np.abs(k_ref).max())
    kv.close()
    m.close()
