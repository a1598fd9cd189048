"""Decode attention through the entry point that allocates nothing.

Callers that cannot call cudaMalloc -- code running while another component
captures a CUDA graph on the same stream, runtimes with a fixed memory budget
that own every allocation -- use ``sar_decode_attention_noalloc``; it keeps its
split partials in a fixed file-scope device array.  Its output must equal the
decode-attention rows that ``sar_step`` writes for the same queries and pages,
call after call.  Given the step's own fp32 queries the two differ only in
where the key ranges are cut: each range rounds its probabilities to 16 bits
relative to its own running maximum and the partial sums merge in another
order, which moves the output by about 2^-12 relative (the output is an
average of N(0,1) values that nearly cancel, so the relative error does not
shrink with the number of keys).  A dropped, doubled or misplaced range
would move it by whole percents.
"""

import ctypes

import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth
from chunked_prefill_hybrid_sar_gb300 import _lib, harness

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 2 << 20  # the entry point's 8 MiB of fp32 partials


def _split_for(n, qh, hd, max_ctx):
    """The split length the entry point documents: the smallest power of two
    in [256, 4096] whose partials fit its scratch (None: rejected)."""
    per = n * qh * (hd + 2)
    for sp in (256, 512, 1024, 2048, 4096):
        ns = (max_ctx + sp) // sp
        if ns <= 1 or ns * per <= SCRATCH_FLOATS:
            return sp
    return None


def _step_then_noalloc(dims, ctxs, seed, history):
    """Runs one decode-only step, then the allocation-free entry twice on the
    step's own queries and pages; returns the step's rows and both calls'."""
    layers, _, gen = synth.model_weights(seed, dims, torch.bfloat16)
    n = len(ctxs)
    m = harness.load_model(dims, layers, None, max_tokens=128, max_decodes=n)
    ps = 16
    stride = max(c // ps + 1 for c in ctxs)
    kv = sar.KVCache(m, ps, n * stride + 8)
    alloc = harness.PageAllocator(synth.page_permutation(gen, n * stride + 8))
    tables = [alloc.take(c // ps + 1) for c in ctxs]
    if history == "per-decode":
        for c, bt in zip(ctxs, tables):
            k, v = synth.kv_history(gen, 1, c, dims)[0]
            harness.write_history(kv, dims, 0, k, v, bt)
    else:  # every page random N(0,1), drawn on the device
        g = synth.generator(seed + 1, "cuda")
        for kind in (0, 1):
            pv = harness.page_view(kv, 0, kind, dims)
            pv.copy_(torch.randn(pv.shape, generator=g, device="cuda", dtype=torch.float32).to(pv.dtype))
    x = synth.normal(gen, (n, dims.hidden), dtype=torch.bfloat16).cuda()
    m.step(kv, sar.Batch(None, [(i, c, tables[i]) for i, c in enumerate(ctxs)]), x)
    m.sync_status()
    torch.cuda.synchronize()
    qkv_n = (dims.n_q_heads + 2 * dims.n_kv_heads) * dims.head_dim
    dt = sar.storage_dtype(m.storage)
    # the step's own decode-attention rows (it split and merged them through its workspace)
    ref = harness.wrap(m.debug_buffer(2), n * dims.q_dim, dt).view(n, dims.q_dim).clone()
    # rotated q|k|v rows of the same step, kept in fp32
    q32 = harness.wrap(m.debug_buffer(5), n * qkv_n, torch.float32).view(n, qkv_n).clone()
    ctx_dev = torch.tensor(ctxs, dtype=torch.int32, device="cuda")
    bt_dev = torch.zeros(n, stride, dtype=torch.int32, device="cuda")
    for i, bt in enumerate(tables):
        bt_dev[i, :len(bt)] = torch.tensor(bt, dtype=torch.int32)
    lib = sar.lib()
    outs = {}
    for qkind, q in (("f32", q32), ("16-bit", q32.to(dt).contiguous())):
        flag = _lib.SAR_Q_F32 if qkind == "f32" else 0
        for call in range(2):
            err = torch.zeros(4, dtype=torch.int32, device="cuda")
            out = torch.full((n, dims.q_dim), float("nan"), dtype=dt, device="cuda")
            rc = lib.sar_decode_attention_noalloc(
                q.data_ptr(), qkv_n, kv.layer_ptr(0, 0), kv.layer_ptr(0, 1), kv.num_pages, ps, dims.n_q_heads,
                dims.n_kv_heads, dims.head_dim, n, ctx_dev.data_ptr(), max(ctxs), bt_dev.data_ptr(),
                stride, out.data_ptr(), dims.q_dim, m.storage | flag, err.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
            sar.check(rc)
            torch.cuda.synchronize()
            assert err.tolist() == [0, 0, 0, 0], (qkind, call)
            outs[(qkind, call)] = out
    return ref, outs


def _assert_matches(ref, outs):
    ref = ref.double()
    for call in range(2):
        # fp32 queries, as the step: only the key-range cuts and the merge order differ
        d = outs[("f32", call)].double() - ref
        assert torch.isfinite(d).all(), call
        assert d.abs().max().item() <= 1e-3, (call, d.abs().max().item())
        assert (d.norm() / ref.norm()).item() <= 5e-4, (call, (d.norm() / ref.norm()).item())
        # queries rounded once to 16 bits: the scores move by about 2^-12 relative
        d = outs[("16-bit", call)].double() - ref
        assert d.abs().max().item() <= 3e-2 and (d.norm() / ref.norm()).item() <= 1e-2, call
    # the second call over the same shared scratch gives the first call's rows
    assert torch.equal(outs[("f32", 0)], outs[("f32", 1)])
    assert torch.equal(outs[("16-bit", 0)], outs[("16-bit", 1)])


def test_noalloc_decode_attention_matches_the_step_twice():
    dims = synth.Dims(n_layers=1, hidden=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=1024)
    gen = synth.generator(11)
    ctxs = synth.uniform_int(gen, 12, 1, 3000)
    assert _split_for(12, 8, 128, max(ctxs)) == 256
    ref, outs = _step_then_noalloc(dims, ctxs, 11, "per-decode")
    _assert_matches(ref, outs)


def test_noalloc_doubles_the_split_when_partials_would_not_fit():
    """64 decodes x 32 query heads near 4000 keys: at 256 or 512 keys per
    range the partials would exceed the 8 MiB scratch, so the entry point
    cuts 1024-key ranges."""
    dims = synth.Dims(n_layers=1, hidden=1024, n_q_heads=32, n_kv_heads=8, head_dim=128, ffn=1024)
    gen = synth.generator(12)
    ctxs = synth.uniform_int(gen, 64, 3900, 4000)
    assert _split_for(64, 32, 128, max(ctxs)) == 1024
    ref, outs = _step_then_noalloc(dims, ctxs, 12, "random-pages")
    _assert_matches(ref, outs)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = sar.lib()
    dummy = ctypes.c_void_p(16)
    # 4096 decodes x 64 heads over 2^20 keys: partials far beyond 8 MiB at any allowed split;
    # rejected before anything touches the device
    rc = lib.sar_decode_attention_noalloc(dummy, 8192, dummy, dummy, 1 << 20, 16, 64, 8, 128, 4096,
                                          dummy, 1 << 20, dummy, (1 << 16) + 1, dummy, 8192, 0, None, None)
    assert rc == _lib.SAR_ERR_INVALID_ARG
    assert b"8 MiB" in lib.sar_last_error()
