"""Convenience glue around the C ABI for callers that hold weights and cache
state as torch tensors: loading a model layer by layer, writing a recorded
K/V history into pages, handing out block tables.  Data movement only."""

from __future__ import annotations

import torch

from . import KVCache, Model


def load_model(dims, layers, head, max_tokens: int, max_decodes: int, device="cuda") -> Model:
    """Creates a model and copies each layer's tensors through the device one
    layer at a time (the library keeps its own packed copy)."""
    m = Model(dims, max_tokens=max_tokens, max_decodes=max_decodes)
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


def page_view(kv: KVCache, layer: int, kind: int, dims) -> torch.Tensor:
    """The layer's K (0) or V (1) pages as a [pages, kvh, page, head_dim] bf16 tensor."""
    ptr = kv.layer_ptr(layer, kind)
    n = kv.num_pages * dims.n_kv_heads * kv.page_size * dims.head_dim
    storage = torch.cuda.current_device()
    t = _wrap(ptr, n, storage)
    return t.view(kv.num_pages, dims.n_kv_heads, kv.page_size, dims.head_dim)


def _wrap(ptr: int, numel: int, device: int) -> torch.Tensor:
    class _Arr:
        __cuda_array_interface__ = {"shape": (numel,), "typestr": "<i2", "data": (ptr, False),
                                    "version": 3, "strides": None}
    return torch.as_tensor(_Arr(), device=f"cuda:{device}").view(torch.bfloat16)


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
        pad = torch.zeros(nb * ps, dims.n_kv_heads, dims.head_dim, dtype=torch.bfloat16, device="cuda")
        pad[:ctx] = src.to("cuda", torch.bfloat16)
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
