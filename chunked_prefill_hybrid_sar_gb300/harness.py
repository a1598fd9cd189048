"""Convenience glue around the C ABI for callers that hold weights and cache
state as torch tensors: loading a model layer by layer, writing a recorded
K/V history into pages, handing out block tables.  Data movement only."""

from __future__ import annotations

import torch

from . import SAR_STORAGE_F16, KVCache, Model, storage_dtype


def load_model(dims, layers, head, max_tokens: int, max_decodes: int, device="cuda",
               storage: int = SAR_STORAGE_F16) -> Model:
    """Creates a model and copies each layer's bf16 tensors through the device
    one layer at a time (the library keeps its own packed copy)."""
    m = Model(dims, max_tokens=max_tokens, max_decodes=max_decodes, storage=storage)
    for l, w in enumerate(layers):
        wd = {k: v.to(device, torch.bfloat16).contiguous() for k, v in w.items()}
        m.set_layer(l, wd)
        torch.cuda.current_stream().synchronize()
        del wd
    if head:
        hd = {k: v.to(device, torch.bfloat16).contiguous() for k, v in head.items()}
        m.set_head(hd["embed"], hd["final_norm"], hd["lm_head"])
        torch.cuda.current_stream().synchronize()
    return m


def load_synthetic_model(seed: int, dims, max_tokens: int, max_decodes: int,
                         storage: int = SAR_STORAGE_F16, keep_layers=()) -> tuple:
    """Draws the seeded N(0, 0.02) weights of ``dims`` on the device layer by
    layer (the draw order of ``synth.model_weights``) and loads each into a
    new model as it is drawn, so a large model never exists twice in memory.
    Returns ``(model, kept)`` where ``kept`` maps the layer indices in
    ``keep_layers`` (and "head") to CPU copies of their bf16 tensors."""
    import synth

    m = Model(dims, max_tokens=max_tokens, max_decodes=max_decodes, storage=storage)
    gen = synth.generator(seed, "cuda")
    kept = {}
    for l in range(dims.n_layers):
        w = synth.layer_weights(gen, dims, torch.bfloat16, "cuda")
        m.set_layer(l, w)
        torch.cuda.current_stream().synchronize()
        if l in keep_layers:
            kept[l] = {k: v.cpu() for k, v in w.items()}
        del w
    head = synth.head_weights(gen, dims, torch.bfloat16, "cuda")
    if head:
        m.set_head(head["embed"], head["final_norm"], head["lm_head"])
        torch.cuda.current_stream().synchronize()
        if "head" in keep_layers:
            kept["head"] = {k: v.cpu() for k, v in head.items()}
    return m, kept


def page_view(kv: KVCache, layer: int, kind: int, dims) -> torch.Tensor:
    """The layer's K (0) or V (1) pages as a [pages, kvh, page, head_dim] tensor
    of the model's storage type."""
    ptr = kv.layer_ptr(layer, kind)
    n = kv.num_pages * dims.n_kv_heads * kv.page_size * dims.head_dim
    t = wrap(ptr, n, storage_dtype(kv.storage))
    return t.view(kv.num_pages, dims.n_kv_heads, kv.page_size, dims.head_dim)


def wrap(ptr: int, numel: int, dtype) -> torch.Tensor:
    """A tensor view of library-owned device memory (no copy, no ownership)."""
    typestr = {torch.float16: "<f2", torch.bfloat16: "<i2", torch.float32: "<f4", torch.int32: "<i4"}[dtype]

    class _Arr:
        __cuda_array_interface__ = {"shape": (numel,), "typestr": typestr, "data": (ptr, False),
                                    "version": 3, "strides": None}
    t = torch.as_tensor(_Arr(), device=f"cuda:{torch.cuda.current_device()}")
    return t.view(dtype) if dtype == torch.bfloat16 else t


def write_history(kv: KVCache, dims, layer: int, k, v, block_table) -> None:
    """Writes K/V of positions [0, ctx) (``[ctx, kvh, head_dim]``) into the
    request's pages in block-table order."""
    ctx = k.shape[0]
    if ctx == 0:
        return
    ps = kv.page_size
    nb = (ctx + ps - 1) // ps
    pages = torch.tensor(block_table[:nb], dtype=torch.long, device="cuda")
    for kind, src in ((0, k), (1, v)):
        dst = page_view(kv, layer, kind, dims)
        pad = torch.zeros(nb * ps, dims.n_kv_heads, dims.head_dim, dtype=dst.dtype, device="cuda")
        pad[:ctx] = src.to("cuda").to(dst.dtype)
        dst[pages] = pad.view(nb, ps, dims.n_kv_heads, dims.head_dim).permute(0, 2, 1, 3)


def read_history(kv: KVCache, dims, layer: int, kind: int, block_table, ctx: int) -> torch.Tensor:
    """Gathers positions [0, ctx) of a request back out of the pages: [ctx, kvh, head_dim]."""
    ps = kv.page_size
    nb = (ctx + ps - 1) // ps
    pages = torch.tensor(block_table[:nb], dtype=torch.long, device="cuda")
    src = page_view(kv, layer, kind, dims)[pages]  # [nb, kvh, ps, d]
    return src.permute(0, 2, 1, 3).reshape(nb * ps, dims.n_kv_heads, dims.head_dim)[:ctx]


class PageAllocator:
    """Hands out page ids from a seeded shuffle, so block tables are not contiguous."""

    def __init__(self, order):
        self.order = list(order)
        self.next = 0

    def take(self, n: int) -> list[int]:
        out = self.order[self.next:self.next + n]
        if len(out) < n:
            raise RuntimeError("out of pages")
        self.next += n
        return out
