"""Chunk attention with two query tiles per CTA (the planner's tile pairs,
taken when one-tile CTAs would need more waves of the SMs than pairs do)
against the one-tile kernel and the oracle.

A pair's two tiles read the same key blocks; each tile does exactly the
one-tile kernel's arithmetic (the later tile's last block is fully masked for
the earlier one, where P is exactly 0), so the attention rows are
bit-identical to the same tiles run one per CTA (the chunk-attention step of
the hybrid batch, SARATHI technique write-up section 3.1; chunk k re-reads the
KV of the k earlier chunks, Sarathi-Serve digest section 4).  The rows are
also checked against the oracle's attention, in fp64 on the step's own fp32
queries and the keys and values read back from the pages: max-abs <= 3e-2,
relative L2 <= 1e-2 (the per-layer bars).
"""

import numpy as np
import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth
from chunked_prefill_hybrid_sar_gb300 import harness
from oracle import model as om

pytestmark = pytest.mark.gpu

PS = 16
PROMPT = 2048
MAX_ABS, REL_L2 = 3e-2, 1e-2


@pytest.fixture(scope="module", params=[sar.SAR_STORAGE_F16, sar.SAR_STORAGE_BF16], ids=["f16", "bf16"])
def layer(request):
    # one Mistral-shaped layer (32 query heads over 8 KV heads x 128), no head,
    # in either storage type (the kernels' two instantiations)
    case = synth.tile_sweep_case(0, rows=(PROMPT,), n_decode=0)
    dims = case["dims"]
    m = harness.load_model(dims, case["layers"], None, max_tokens=1024, max_decodes=8, storage=request.param)
    n_pages = PROMPT // PS + 8
    bt = list(synth.page_permutation(synth.generator(11), n_pages))[:PROMPT // PS]
    kv = sar.KVCache(m, PS, n_pages)
    yield case, m, kv, bt
    kv.close()
    m.close()


def chunk_rows(m, kv, bt, prompt, start, n):
    """The attention rows (storage type) of one chunk step."""
    dims = m.dims
    m.step(kv, sar.Batch((0, start, n, bt), []), prompt[start:start + n].cuda().contiguous())
    m.sync_status()
    torch.cuda.synchronize()
    ptr = m.debug_buffer(2)
    return harness.wrap(ptr, n * dims.q_dim, sar.storage_dtype(m.storage)).view(n, dims.q_dim).clone()


def pairs_planned(m, bt, start, n):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = sar.plan_inspect(m.dims, sar.Batch((0, start, n, bt), []), PS, PROMPT // PS + 8, sms, 1024, 8)
    return p["chunk_pairs"] == 1


def test_tile_pairs_match_one_tile_ctas_bit_for_bit(layer):
    case, m, kv, bt = layer
    prompt = case["prompt"]
    # 512-row chunks: 4 tiles x 32 heads = 128 CTAs, one per tile; 1024-row
    # chunks: 8 tiles x 32 heads, more than the SMs -> 4 pairs x 32 heads
    assert not pairs_planned(m, bt, 512, 512)
    assert pairs_planned(m, bt, 1024, 1024)
    single = torch.cat([chunk_rows(m, kv, bt, prompt, s, 512) for s in range(0, PROMPT, 512)])
    pairs = torch.cat([chunk_rows(m, kv, bt, prompt, s, 1024) for s in (0, 1024)])
    assert torch.isfinite(single.float()).all()
    assert torch.equal(pairs, single)
    # five tiles, the last one ragged (600 rows at position 1024: four pairs'
    # worth of CTAs would not fit one wave, three do): the fifth tile pairs
    # with an empty one; the same tiles one per CTA come from a 512-row and an
    # 88-row chunk
    assert pairs_planned(m, bt, 1024, 600)
    odd = chunk_rows(m, kv, bt, prompt, 1024, 600)
    one = torch.cat([chunk_rows(m, kv, bt, prompt, 1024, 512), chunk_rows(m, kv, bt, prompt, 1536, 88)])
    assert torch.equal(odd, one)


def test_tile_pairs_against_the_oracle(layer):
    case, m, kv, bt = layer
    if m.storage != sar.SAR_STORAGE_F16:
        # the kernel rounds the queries and probabilities to the storage type;
        # with bf16's 8-bit mantissa the scores of this layer's magnitudes are
        # off by up to ~2e-2 (log2 units), beyond the per-layer bars -- the
        # bf16 instantiation is held to the one-tile kernel bit for bit above
        pytest.skip("oracle comparison in f16 storage")
    dims = m.dims
    prompt = case["prompt"]
    chunk_rows(m, kv, bt, prompt, 0, 1024)
    start, n = 1024, 1000  # 8 tiles, the last of 104 rows
    assert pairs_planned(m, bt, start, n)
    got = chunk_rows(m, kv, bt, prompt, start, n).float().cpu().numpy()
    qkv_n = dims.q_dim + 2 * dims.kv_dim
    q32 = harness.wrap(m.debug_buffer(5), n * qkv_n, torch.float32).view(n, qkv_n)[:, :dims.q_dim]
    q = q32.cpu().double().numpy().reshape(n, dims.n_q_heads, dims.head_dim)
    keys = start + n
    k = harness.read_history(kv, dims, 0, 0, bt, keys).double().cpu().numpy()
    v = harness.read_history(kv, dims, 0, 1, bt, keys).double().cpu().numpy()
    # every tile's first and last rows, and a stride through the rest
    sel = sorted(set(list(range(0, n, 37)) + [t * 128 for t in range(8)] +
                     [min(n, t * 128 + 128) - 1 for t in range(8)]))
    ref = om.attention(q[sel], k, v, start + np.array(sel), np.arange(keys)).reshape(len(sel), -1)
    g = got[sel]
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert err <= MAX_ABS and rel <= REL_L2, f"max-abs {err:.3e}, rel-L2 {rel:.3e}"


def test_tile_pairs_of_two_prompts_in_one_batch(layer):
    """Two prompts' 512-row chunks in one batch (8 tiles x 32 heads: pairs,
    each within one prompt) against each chunk stepped alone (4 tiles x 32
    heads: one tile per CTA): bit-identical attention rows."""
    case, m, _, _ = layer
    dims = m.dims
    prompt = case["prompt"]
    n_pages = PROMPT // PS + 8
    perm = list(synth.page_permutation(synth.generator(12), n_pages))
    bts = [perm[:1024 // PS], perm[1024 // PS:2048 // PS]]
    xs = [prompt[:1024], prompt[1024:2048]]  # two different prompts of 1024 tokens
    kv = sar.KVCache(m, PS, n_pages)
    try:
        for i in range(2):  # their first chunks, one per step
            chunk_rows(m, kv, bts[i], xs[i], 0, 512)
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        both = sar.Batch([(0, 512, 512, bts[0]), (1, 512, 512, bts[1])], [])
        p = sar.plan_inspect(dims, both, PS, n_pages, sms, 1024, 8)
        assert p["chunk_pairs"] == 1 and p["n_tiles"] == 8
        x = torch.cat([xs[0][512:1024], xs[1][512:1024]]).cuda().contiguous()
        m.step(kv, both, x)
        m.sync_status()
        torch.cuda.synchronize()
        pairs = harness.wrap(m.debug_buffer(2), 1024 * dims.q_dim, sar.storage_dtype(m.storage)).view(
            1024, dims.q_dim).clone()
        alone = torch.cat([chunk_rows(m, kv, bts[i], xs[i], 512, 512) for i in range(2)])
        assert torch.isfinite(alone.float()).all()
        assert torch.equal(pairs, alone)
    finally:
        kv.close()
