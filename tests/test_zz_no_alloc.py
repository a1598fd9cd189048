"""Decode attention through the entry point that allocates nothing.

Callers that cannot call cudaMalloc -- code running while another component
captures a CUDA graph on the same stream, runtimes with a fixed memory budget
that own every allocation -- use ``sar_decode_attention_noalloc``; it keeps its
split partials in a fixed file-scope device array.  Its output must equal the
decode-attention rows that ``sar_step`` writes for the same queries and pages,
call after call.
"""

import ctypes

import pytest
import torch

import chunked_prefill_hybrid_sar_gb300 as sar
import synth
from chunked_prefill_hybrid_sar_gb300 import _lib, harness

pytestmark = pytest.mark.gpu


def test_noalloc_decode_attention_matches_the_step_twice():
    dims = synth.Dims(n_layers=1, hidden=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=1024)
    layers, _, gen = synth.model_weights(11, dims, torch.bfloat16)
    m = harness.load_model(dims, layers, None, max_tokens=128, max_decodes=16)
    n = 12
    ctxs = synth.uniform_int(gen, n, 1, 3000)
    ps = 16
    stride = max(c // ps + 1 for c in ctxs)
    kv = sar.KVCache(m, ps, n * stride + 8)
    alloc = harness.PageAllocator(synth.page_permutation(gen, n * stride + 8))
    tables = []
    for c in ctxs:
        bt = alloc.take(c // ps + 1)
        k, v = synth.kv_history(gen, 1, c, dims)[0]
        harness.write_history(kv, dims, 0, k, v, bt)
        tables.append(bt)
    x = synth.normal(gen, (n, dims.hidden), dtype=torch.bfloat16).cuda()
    m.step(kv, sar.Batch(None, [(i, c, tables[i]) for i, c in enumerate(ctxs)]), x)
    m.sync_status()
    torch.cuda.synchronize()
    qkv_n = (dims.n_q_heads + 2 * dims.n_kv_heads) * dims.head_dim
    dt = sar.storage_dtype(m.storage)
    # the step's own decode-attention rows (it split and merged them through its workspace)
    ref = harness.wrap(m.debug_buffer(2), n * dims.q_dim, dt).view(n, dims.q_dim).clone()
    # rotated q|k|v rows of the same step (kept in fp32), in the storage type
    qkv_rows = harness.wrap(m.debug_buffer(5), n * qkv_n, torch.float32).view(n, qkv_n).to(dt).contiguous()
    q_ptr = qkv_rows.data_ptr()
    ctx_dev = torch.tensor(ctxs, dtype=torch.int32, device="cuda")
    bt_dev = torch.zeros(n, stride, dtype=torch.int32, device="cuda")
    for i, bt in enumerate(tables):
        bt_dev[i, :len(bt)] = torch.tensor(bt, dtype=torch.int32)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    lib = sar.lib()
    for call in range(2):
        out = torch.full((n, dims.q_dim), float("nan"), dtype=dt, device="cuda")
        rc = lib.sar_decode_attention_noalloc(
            q_ptr, qkv_n, kv.layer_ptr(0, 0), kv.layer_ptr(0, 1), kv.num_pages, ps, dims.n_q_heads,
            dims.n_kv_heads, dims.head_dim, n, ctx_dev.data_ptr(), max(ctxs), bt_dev.data_ptr(),
            stride, out.data_ptr(), dims.q_dim, m.storage, err.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        sar.check(rc)
        torch.cuda.synchronize()
        assert err.tolist() == [0, 0, 0, 0]
        diff = out.double() - ref.double()
        assert diff.abs().max().item() <= 3e-2, call
        assert (diff.norm() / ref.double().norm()).item() <= 1e-2, call


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = sar.lib()
    dummy = ctypes.c_void_p(16)
    # 4096 decodes x 64 heads over 2^20 keys: partials far beyond 8 MiB at any allowed split;
    # rejected before anything touches the device
    rc = lib.sar_decode_attention_noalloc(dummy, 8192, dummy, dummy, 1 << 20, 16, 64, 8, 128, 4096,
                                          dummy, 1 << 20, dummy, (1 << 16) + 1, dummy, 8192, 0, None, None)
    assert rc == _lib.SAR_ERR_INVALID_ARG
    assert b"8 MiB" in lib.sar_last_error()
