"""Hybrid-batch decoder step (chunked prefill + piggybacked decodes) on GB300.

Thin Python face of ``libsar.so``: the classes below only marshal torch
tensors (device memory and streams) and host lists into the C ABI of
``include/sar.h``; every step runs in the library's CUDA kernels.
"""

from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (SAR_EPI_F32, SAR_EPI_RESIDUAL, SAR_EPI_STORE, SAR_EPI_SWIGLU, SAR_GEMM_AUTO,
                   SAR_GEMM_PAIR_N128, SAR_GEMM_PAIR_N192,
                   SAR_GEMM_PAIR_N256, SAR_GEMM_STREAM_K, SAR_GEMM_TWO_CTAS,
                   SAR_GEMM_M128_N128, SAR_GEMM_M128_N256, SAR_GEMM_M256_N128, SAR_GEMM_SWAP,
                   SAR_IN_HIDDEN, SAR_IN_TOKENS, SAR_STORAGE_BF16, SAR_STORAGE_F16, KERNEL_KINDS,
                   SarError, check, lib)

__all__ = ["Model", "KVCache", "Scheduler", "Batch", "StepGraph", "SarError", "lib", "check", "gemm", "rmsnorm",
           "op_sync_status", "op_wait_check",
           "launch_count", "KERNEL_KINDS", "SAR_IN_HIDDEN", "SAR_IN_TOKENS", "SAR_STORAGE_F16",
           "SAR_STORAGE_BF16", "storage_dtype"]


def storage_dtype(storage: int):
    """torch dtype of a storage code."""
    import torch
    return torch.bfloat16 if storage == SAR_STORAGE_BF16 else torch.float16


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def launch_count() -> int:
    return int(lib().sar_launch_count())


class Batch:
    """Owns the ctypes descriptor of one hybrid batch (chunks first, then decodes).

    ``prefill``: ``(req, start_pos, len, block_table)``, a list of such chunks
    (each of a different request, rows stacked in list order) or ``None``;
    ``decodes``: iterable of ``(req, ctx_len, block_table)``.
    """

    def __init__(self, prefill, decodes, in_kind=SAR_IN_HIDDEN):
        self._keep = []
        b = _lib.sar_batch()
        b.in_kind = in_kind
        if prefill is None:
            chunks = []
        elif isinstance(prefill, tuple):
            chunks = [prefill]
        else:
            chunks = list(prefill)
        pre = []
        for req, start, n, bt in chunks:
            arr = _lib.i32_array(bt)
            self._keep.append(arr)
            pre.append(_lib.sar_prefill(req, start, n, arr, len(bt)))
        if pre:
            b.has_prefill = 1
            b.prefill = pre[0]
        if len(pre) > 1:
            more = (_lib.sar_prefill * (len(pre) - 1))(*pre[1:])
            self._keep.append(more)
            b.n_more_prefill = len(pre) - 1
            b.more_prefill = more
        decodes = list(decodes)
        dec = (_lib.sar_decode * max(1, len(decodes)))()
        for i, (req, ctx, bt) in enumerate(decodes):
            arr = _lib.i32_array(bt)
            self._keep.append(arr)
            dec[i] = _lib.sar_decode(req, ctx, arr, len(bt))
        self._keep.append(dec)
        b.n_decode = len(decodes)
        b.decode = dec
        self.c = b
        self.chunks = chunks
        self.lp = sum(c[2] for c in chunks)
        self.bd = len(decodes)

    @property
    def rows(self) -> int:
        return self.lp + self.bd

    @property
    def logit_rows(self) -> int:
        """The last row of every chunk, then every decode row."""
        return len(self.chunks) + self.bd


class Model:
    """Weights are given in bf16; ``storage`` picks the internal 16-bit type."""

    def __init__(self, dims, max_tokens: int, max_decodes: int, storage: int = SAR_STORAGE_F16):
        self.dims = dims
        self.storage = storage
        d = _lib.sar_dims(dims.n_layers, dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim,
                          dims.ffn, dims.vocab, dims.rms_eps, dims.rope_base, max_tokens, max_decodes,
                          storage, getattr(dims, "sliding_window", 0))
        h = ctypes.c_void_p()
        check(lib().sar_model_create(ctypes.byref(d), ctypes.byref(h)))
        self.h = h

    def set_layer(self, layer: int, w: dict, stream=None) -> None:
        lw = _lib.sar_layer_weights(*[_ptr(w[n]) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd",
                                                          "norm1", "norm2")])
        check(lib().sar_model_set_layer(self.h, layer, ctypes.byref(lw), _stream(stream)))

    def set_head(self, embed=None, final_norm=None, lm_head=None, stream=None) -> None:
        check(lib().sar_model_set_head(self.h, _ptr(embed), _ptr(final_norm), _ptr(lm_head),
                                       _stream(stream)))

    def step(self, kv: "KVCache", batch: Batch, inp, hidden_out=None, logits_out=None,
             layer_out=None, stream=None) -> None:
        check(lib().sar_step(self.h, kv.h, ctypes.byref(batch.c), _ptr(inp), _ptr(hidden_out),
                             _ptr(logits_out), _ptr(layer_out), _stream(stream)))

    def step_host(self, kv: "KVCache", batch: Batch, inp, hidden_out=None, logits_out=None,
                  stream=None) -> None:
        check(lib().sar_step_host(self.h, kv.h, ctypes.byref(batch.c), _ptr(inp), _ptr(hidden_out),
                                  _ptr(logits_out), None, _stream(stream)))

    def sample_greedy(self, logits, rows: int, out, stream=None) -> None:
        check(lib().sar_sample_greedy(self.h, _ptr(logits), rows, _ptr(out), _stream(stream)))

    def sync_status(self) -> None:
        check(lib().sar_sync_status(self.h))

    def profile(self, on: bool) -> None:
        check(lib().sar_profile_enable(self.h, 1 if on else 0))

    def set_chunk_split(self, on: bool) -> None:
        """Key-range splits of chunk-attention tiles when they leave SMs idle."""
        check(lib().sar_model_set_chunk_split(self.h, 1 if on else 0))

    def set_overlap(self, on: bool) -> None:
        """Chunk attention on a second stream, concurrent with decode attention."""
        check(lib().sar_model_set_overlap(self.h, 1 if on else 0))

    def profile_read(self) -> dict:
        n = len(KERNEL_KINDS)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        check(lib().sar_profile_read(self.h, ms, cnt, n))
        return {k: (ms[i], int(cnt[i])) for i, k in enumerate(KERNEL_KINDS)}

    def debug_buffer(self, which: int) -> int:
        p = ctypes.c_void_p()
        check(lib().sar_model_debug_buffer(self.h, which, ctypes.byref(p)))
        return p.value

    def close(self) -> None:
        if self.h:
            check(lib().sar_model_destroy(self.h))
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepGraph:
    """One step captured as a CUDA graph (``sar_graph_*``): fixed input and
    output buffers; ``update`` re-points it at a batch whose plan has the same
    shape, ``launch`` runs it."""

    def __init__(self, model: "Model", kv: "KVCache", batch: Batch, inp, hidden_out=None, logits_out=None,
                 layer_out=None, stream=None):
        self._keep = (batch, inp, hidden_out, logits_out, layer_out)
        h = ctypes.c_void_p()
        check(lib().sar_graph_create(model.h, kv.h, ctypes.byref(batch.c), _ptr(inp), _ptr(hidden_out),
                                     _ptr(logits_out), _ptr(layer_out), _stream(stream), ctypes.byref(h)))
        self.h = h

    def update(self, batch: Batch, stream=None) -> None:
        check(lib().sar_graph_update(self.h, ctypes.byref(batch.c), _stream(stream)))
        self._keep = (batch,) + self._keep[1:]

    def launch(self, stream=None) -> None:
        check(lib().sar_graph_launch(self.h, _stream(stream)))

    def launch_host(self, inp, logits_out=None, hidden_out=None, stream=None) -> None:
        """Host input in, the captured step, host logits / hidden rows out (synchronous)."""
        check(lib().sar_graph_launch_host(self.h, _ptr(inp), _ptr(logits_out), _ptr(hidden_out), _stream(stream)))

    def launch_host_tokens(self, inp, tokens_out, stream=None) -> None:
        """Host input in, the captured step, each logits row's greedy pick out
        (host int32 [R], synchronous)."""
        check(lib().sar_graph_launch_host_tokens(self.h, _ptr(inp), ctypes.cast(_ptr(tokens_out), _lib.P_i32),
                                                 _stream(stream)))

    def enqueue_host_tokens(self, inp, tokens_out, stream=None) -> None:
        """As launch_host_tokens, but returns once the step is enqueued (the
        input copy on the graph's own copy stream); ``wait`` then waits for
        it.  ``inp`` must stay unchanged and ``tokens_out`` unread until then."""
        check(lib().sar_graph_enqueue_host_tokens(self.h, _ptr(inp), ctypes.cast(_ptr(tokens_out), _lib.P_i32),
                                                  _stream(stream)))
        self._pending = (inp, tokens_out)

    def wait(self) -> None:
        """Waits for the last enqueue_host_tokens step of this graph."""
        check(lib().sar_graph_wait(self.h))
        self._pending = None

    def close(self) -> None:
        if self.h:
            check(lib().sar_graph_destroy(self.h))
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KVCache:
    def __init__(self, model: Model, page_size: int, num_pages: int):
        h = ctypes.c_void_p()
        check(lib().sar_kv_create(model.h, page_size, num_pages, ctypes.byref(h)))
        self.h = h
        self.model = model
        self.storage = model.storage
        self.page_size = page_size
        self.num_pages = num_pages

    def layer_ptr(self, layer: int, kind: int) -> int:
        p = ctypes.c_void_p()
        check(lib().sar_kv_layer_ptr(self.h, layer, kind, ctypes.byref(p)))
        return p.value

    def close(self) -> None:
        if self.h:
            check(lib().sar_kv_destroy(self.h))
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Scheduler:
    """Stall-free scheduler (host only)."""

    def __init__(self, tau: int, tile: int, page_size: int, num_pages: int, max_batch: int,
                 max_chunks: int = 0):
        cfg = _lib.sar_sched_cfg(tau, tile, page_size, num_pages, max_batch, max_chunks)
        h = ctypes.c_void_p()
        check(lib().sar_sched_create(ctypes.byref(cfg), ctypes.byref(h)))
        self.h = h

    def add(self, req: int, arrival: float, prompt_len: int, output_len: int, prompt_tokens=None):
        arr = _lib.i32_array(prompt_tokens) if prompt_tokens is not None else None
        check(lib().sar_sched_add(self.h, req, arrival, prompt_len, output_len, arr))

    def next(self, now: float):
        """Returns ``(chunks, decodes, tokens, c_batch)`` with Python lists copied
        out; ``chunks`` lists ``(req, start_pos, len, block_table)`` in row order."""
        b = _lib.sar_batch()
        tok = _lib.P_i32()
        check(lib().sar_sched_next(self.h, now, ctypes.byref(b), ctypes.byref(tok)))

        def chunk(p):
            return (p.req, p.start_pos, p.len, [p.block_table[i] for i in range(p.n_blocks)])

        chunks = []
        if b.has_prefill:
            chunks.append(chunk(b.prefill))
            chunks += [chunk(b.more_prefill[i]) for i in range(b.n_more_prefill)]
        decs = []
        for i in range(b.n_decode):
            dd = b.decode[i]
            decs.append((dd.req, dd.ctx_len, [dd.block_table[j] for j in range(dd.n_blocks)]))
        m = sum(c[2] for c in chunks) + len(decs)
        tokens = [tok[i] for i in range(m)] if bool(tok) else None
        return chunks, decs, tokens, b

    def commit(self, sampled) -> int:
        arr = _lib.i32_array(sampled)
        n = ctypes.c_int32()
        check(lib().sar_sched_commit(self.h, arr, len(list(sampled)), ctypes.byref(n)))
        return n.value

    def stats(self):
        v = [ctypes.c_int32() for _ in range(4)]
        check(lib().sar_sched_stats(self.h, *[ctypes.byref(x) for x in v]))
        return tuple(x.value for x in v)

    def close(self) -> None:
        if self.h:
            check(lib().sar_sched_destroy(self.h))
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_LAYOUT = ("M", "Lp", "Bd", "R", "n_items", "n_parts", "n_tiles", "tile_rows", "o_pos", "o_slot", "o_pbt",
           "o_nkeys", "o_btoff", "o_btlen", "o_pbeg", "o_pcnt", "o_items", "o_bt", "o_rows", "o_tiles", "total",
           "n_comb", "n_cparts", "o_comb", "chunk_pairs")


def plan_inspect(dims, batch: Batch, page_size: int, num_pages: int, sms: int, max_tokens: int,
                 max_decodes: int, storage: int = SAR_STORAGE_F16, chunk_split: bool = False) -> dict:
    """The step planner on the host alone (``sar_plan_inspect``): the plan's
    sizes and array offsets, and the metadata block as a list of int32."""
    d = _lib.sar_dims(dims.n_layers, dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim,
                      dims.ffn, dims.vocab, dims.rms_eps, dims.rope_base, max_tokens, max_decodes,
                      storage, getattr(dims, "sliding_window", 0))
    lay = (ctypes.c_int32 * len(_LAYOUT))()
    n = ctypes.c_int64()
    cs = 1 if chunk_split else 0
    check(lib().sar_plan_inspect(ctypes.byref(d), page_size, num_pages, sms, cs, ctypes.byref(batch.c), lay, None,
                                 0, ctypes.byref(n)))
    meta = (ctypes.c_int32 * max(1, n.value))()
    check(lib().sar_plan_inspect(ctypes.byref(d), page_size, num_pages, sms, cs, ctypes.byref(batch.c), lay, meta,
                                 n.value, ctypes.byref(n)))
    out = dict(zip(_LAYOUT, list(lay)))
    out["meta"] = list(meta)[:n.value]
    return out


def _storage_of(t) -> int:
    import torch
    return SAR_STORAGE_BF16 if t.dtype == torch.bfloat16 else SAR_STORAGE_F16


def gemm(a, w, c, residual=None, epilogue=SAR_EPI_STORE, variant=SAR_GEMM_AUTO, stream=None) -> None:
    """C = epilogue(a . w^T); the storage type is taken from ``a`` (fp16 or bf16)."""
    M, K = a.shape
    N = w.shape[0]
    check(lib().sar_op_gemm(_ptr(a), _ptr(w), _ptr(c), _ptr(residual), M, N, K, epilogue, variant,
                            _storage_of(a), _stream(stream)))


def op_sync_status() -> None:
    """Synchronise the device and raise if a single-kernel entry point's
    kernel recorded a failure (timeout or bounds) since the last call."""
    check(lib().sar_op_sync_status())


def op_wait_check(limit_ns: int, arrivals: int, stream=None) -> None:
    """Run the bounded-wait check kernel (see ``sar_op_wait_check``)."""
    check(lib().sar_op_wait_check(int(limit_ns), int(arrivals), _stream(stream)))


def rmsnorm(x, gain, y, eps: float, stream=None) -> None:
    """y (fp16/bf16) = rmsnorm of fp32 rows x with fp32 gain."""
    check(lib().sar_op_rmsnorm(_ptr(x), _ptr(gain), _ptr(y), x.shape[0], x.shape[1], eps,
                               _storage_of(y), _stream(stream)))
