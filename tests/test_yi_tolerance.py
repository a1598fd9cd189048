"""Where the absolute hidden-state bar comes from at the Yi-34B shape.

The hidden-state bar (max-abs 3e-2, relative L2 1e-2, 16-bit activation
storage with fp32 accumulation) holds as stated for the tiny and the
Mistral-shaped layers.  At the Yi-34B shape (H 7168, FFN 20480) the
random-init residual stream is larger (RMS about 5.6 after layer 0 and 7.8
after layer 1, peaks near 39), and rounding the stored activations to fp16
*alone* -- the normalised rows, K and V, the attention rows, the SwiGLU
product, each rounded once in an otherwise float64 computation -- already
moves layer 1 by more than 3e-2.  No 16-bit storage can meet the absolute bar
there (bf16 rounds 8x coarser than fp16), so the Yi tests bound max-abs by
YI_MAX_ABS, about twice what this rounding alone produces, and keep the
relative-L2 bar as stated.

This test recomputes that rounding-only error from the oracle's own steps.
"""

import dataclasses

import numpy as np
import torch

import synth
from oracle import model as om

YI_MAX_ABS = 0.1


def f16(a):
    return a.astype(np.float16).astype(np.float64)


def f32(a):
    return a.astype(np.float32).astype(np.float64)


def layer_with_fp16_storage(x, w, dims, pos):
    """One decoder layer in float64 with the activations that a 16-bit
    storage path keeps between kernels rounded to fp16 (queries kept in fp32,
    the residual stream in fp32 before rounding effects, which are far below
    fp16's)."""
    T = x.shape[0]
    y = f16(om.rms_norm(x, w["norm1"], dims.rms_eps))
    q = (y @ w["wq"].T).reshape(T, dims.n_q_heads, dims.head_dim)
    k = (y @ w["wk"].T).reshape(T, dims.n_kv_heads, dims.head_dim)
    v = (y @ w["wv"].T).reshape(T, dims.n_kv_heads, dims.head_dim)
    q = f32(om.apply_rope(q, pos, dims.rope_base))
    k = f16(om.apply_rope(k, pos, dims.rope_base))
    v = f16(v)
    a = f16(om.attention(q, k, v, pos, pos).reshape(T, -1))
    h = x + a @ w["wo"].T
    y2 = f16(om.rms_norm(h, w["norm2"], dims.rms_eps))
    act = f16(om.silu(y2 @ w["wg"].T) * (y2 @ w["wu"].T))
    return h + act @ w["wd"].T


def test_fp16_storage_alone_exceeds_the_absolute_bar_at_yi_shape():
    dims = dataclasses.replace(synth.YI_34B, n_layers=2, vocab=0)
    layers, _, gen = synth.model_weights(0, dims)
    w = [om.layer_weights_np(l) for l in layers]
    x = om.to_np(synth.normal(gen, (512, dims.hidden), dtype=torch.bfloat16))
    ref, _ = om.forward(w, dims, x)
    pos = np.arange(512)
    h = x
    errs = []
    for l in range(2):
        h = layer_with_fp16_storage(h, w[l], dims, pos)
        errs.append((np.abs(h - ref[l]).max(), np.linalg.norm(h - ref[l]) / np.linalg.norm(ref[l])))
    # rounding alone breaks the absolute bar at layer 1, not the relative one
    assert errs[1][0] > 3e-2
    assert all(r < 1e-2 for _, r in errs)
    # the bound used on the GPU leaves a margin of about 2 over it
    assert all(e < YI_MAX_ABS / 1.5 for e, _ in errs)
