"""Oracle decoder layer, chunked prefill and hybrid-batch step (test infrastructure only).

Plain NumPy, float64 by default.  Every function states the passage it
follows.  Where the pages leave a step open the plainest Llama/Mistral
reading is taken (the pages evaluate Mistral-7B, Yi-34B, LLaMA2-70B and
Falcon-180B decoder-only transformers with GQA: *Sarathi-Serve digest*,
Appendix table of evaluated models):

* RMSNorm ``x / sqrt(mean(x^2) + eps) * g`` before attention and before the FFN;
* rotary embedding, rotate-half pairing (dimension i with i + d/2),
  ``theta_i = base^(-2i/d)``, at absolute positions;
* causal grouped-query attention, query head h reads KV head ``h // (qh/kvh)``,
  scale ``1/sqrt(d)``;
* SwiGLU FFN ``(silu(y Wg^T) * (y Wu^T)) Wd^T``; residual adds after attention
  and after the FFN.

Parity status: rms_norm, apply_rope, silu, attention (full causal and
sliding-window), decoder_layer, final_logits (with the sampled-row choice)
and the hybrid step are pinned by ``tests/test_oracle_*.py`` (closed forms,
library special cases, brute force, chunked == one-shot, hybrid == serial).  The
absolute hidden values of a random-initialised model have no printed worked
example and are otherwise parity unpinned.
"""

from __future__ import annotations

import dataclasses

import numpy as np


def to_np(t, dtype=np.float64) -> np.ndarray:
    """Torch tensor (any dtype, incl. bf16) or array -> NumPy array of ``dtype``."""
    if hasattr(t, "detach"):
        t = t.detach().to("cpu")
        if str(t.dtype) in ("torch.bfloat16", "torch.float16"):
            t = t.float()
        t = t.numpy()
    return np.asarray(t, dtype=dtype)


def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """Root-mean-square normalisation over the last axis.

    The pages place a normalisation ahead of each sub-block ("insert an explicit
    sync before LayerNorm", *SARATHI technique write-up* §6.1); the evaluated
    models use RMSNorm, so ``x / sqrt(mean(x^2) + eps) * gain``.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gain


def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """Rotary frequencies ``base^(-2i/d)`` for ``i < d/2`` (float64)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return base ** (-2.0 * i / head_dim)


def apply_rope(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotate ``x[T, heads, d]`` at absolute positions ``pos[T]``.

    Each chunk keeps the absolute position ids of its tokens, so that a chunk
    starting at ``start_pos`` continues the prompt's numbering ("maintain an
    independent position_id for each chunk", *SARATHI technique write-up* §6.1).
    Pairing is rotate-half: dimension ``i`` with ``i + d/2``.
    """
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(d, base)[None, :]
    c = np.cos(ang).astype(x.dtype)[:, None, :]
    s = np.sin(ang).astype(x.dtype)[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    """``x * sigmoid(x)``."""
    return x / (1.0 + np.exp(-x))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos, k_pos, window: int = 0) -> np.ndarray:
    """Causal grouped-query attention, optionally over a sliding window.

    ``q[T, qh, d]``, ``k, v[S, kvh, d]``; query ``t`` attends to key ``s`` iff
    ``k_pos[s] <= q_pos[t]`` (the causal mask whose correctness across chunks
    the *SARATHI technique write-up* §6.1 asks to check) and, when
    ``window > 0``, also ``k_pos[s] > q_pos[t] - window``: the query sees the
    ``window`` most recent positions, itself included.  The pages list
    Mistral-7B's attention as GQA with a sliding window (*Sarathi-Serve
    digest*, Appendix table of evaluated models) without stating the window or
    its edge; this "W latest keys, self included" edge is the reading taken.
    Query head ``h`` reads KV head ``h // (qh // kvh)``.  Scale ``1/sqrt(d)``,
    softmax over the visible keys.
    """
    T, qh, d = q.shape
    S, kvh, _ = k.shape
    group = qh // kvh
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    visible = k_pos[None, :] <= q_pos[:, None]
    if window > 0:
        visible &= k_pos[None, :] > q_pos[:, None] - window
    out = np.empty_like(q)
    scale = 1.0 / np.sqrt(d)
    for h in range(qh):
        kh = h // group
        s = (q[:, h, :] @ k[:, kh, :].T) * scale
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, kh, :]
    return out


def window_of(dims) -> int:
    """The model's sliding window (0 = full causal attention)."""
    return int(getattr(dims, "sliding_window", 0) or 0)


@dataclasses.dataclass
class LayerCache:
    """Post-rotary K and V of positions ``[0, n)`` for one layer, contiguous."""

    k: np.ndarray  # [n, kvh, d]
    v: np.ndarray

    @property
    def n(self) -> int:
        return self.k.shape[0]


def empty_cache(dims, dtype=np.float64) -> LayerCache:
    z = np.zeros((0, dims.n_kv_heads, dims.head_dim), dtype=dtype)
    return LayerCache(z, z.copy())


def layer_weights_np(w: dict, dtype=np.float64) -> dict:
    return {name: to_np(t, dtype) for name, t in w.items()}


def qkv_rope(x: np.ndarray, pos, w: dict, dims) -> tuple:
    """Pre-attention part of a layer: norm, Q/K/V projections, rotary."""
    T = x.shape[0]
    y = rms_norm(x, w["norm1"], dims.rms_eps)
    q = (y @ w["wq"].T).reshape(T, dims.n_q_heads, dims.head_dim)
    k = (y @ w["wk"].T).reshape(T, dims.n_kv_heads, dims.head_dim)
    v = (y @ w["wv"].T).reshape(T, dims.n_kv_heads, dims.head_dim)
    q = apply_rope(q, pos, dims.rope_base)
    k = apply_rope(k, pos, dims.rope_base)
    return q, k, v


def post_attention(x: np.ndarray, a: np.ndarray, w: dict, dims) -> np.ndarray:
    """Output projection + residual, then norm, SwiGLU FFN + residual."""
    h = x + a @ w["wo"].T
    y = rms_norm(h, w["norm2"], dims.rms_eps)
    f = (silu(y @ w["wg"].T) * (y @ w["wu"].T)) @ w["wd"].T
    return h + f


def decoder_layer(x: np.ndarray, pos, w: dict, dims, cache: LayerCache) -> tuple:
    """One decoder layer over rows ``x[T, H]`` at absolute positions ``pos``
    that follow the ``cache.n`` positions already in ``cache``.

    Returns ``(h_out[T, H], LayerCache of positions [0, cache.n + T))``.
    """
    pos = np.asarray(pos)
    q, k, v = qkv_rope(x, pos, w, dims)
    K = np.concatenate([cache.k, k.astype(cache.k.dtype)], axis=0)
    V = np.concatenate([cache.v, v.astype(cache.v.dtype)], axis=0)
    k_pos = np.arange(K.shape[0])
    a = attention(q, K, V, pos, k_pos, window_of(dims)).reshape(x.shape[0], dims.q_dim)
    return post_attention(x, a, w, dims), LayerCache(K, V)


def forward(layers: list, dims, x: np.ndarray, caches: list | None = None) -> tuple:
    """All layers over one request's rows ``x`` (layer-0 inputs) that continue
    the positions held in ``caches`` (one ``LayerCache`` per layer; ``None`` =
    start of the prompt).  Returns ``(outputs per layer, caches after)``."""
    if caches is None:
        caches = [empty_cache(dims, x.dtype) for _ in layers]
    start = caches[0].n
    pos = np.arange(start, start + x.shape[0])
    outs, new = [], []
    h = x
    for w, c in zip(layers, caches):
        h, c2 = decoder_layer(h, pos, w, dims, c)
        outs.append(h)
        new.append(c2)
    return outs, new


def chunked_prefill(layers: list, dims, x: np.ndarray, chunk: int) -> tuple:
    """Prefill ``x`` chunk by chunk: each chunk attends to the KV of the earlier
    chunks held in the cache and to itself (*SARATHI reading notes*, part 2 §1;
    *Sarathi-Serve digest* §2 Q2 item 1).

    Returns ``(outputs per layer over all rows, prior_chunk_loads)`` where
    ``prior_chunk_loads`` counts, for layer 0, how many earlier chunks each
    chunk's attention read back from the cache (chunk k reads k of them).
    """
    caches = None
    outs = [[] for _ in layers]
    loads = 0
    for lo in range(0, x.shape[0], chunk):
        if caches is not None:
            loads += caches[0].n // chunk
        o, caches = forward(layers, dims, x[lo:lo + chunk], caches)
        for l, ol in enumerate(o):
            outs[l].append(ol)
    return [np.concatenate(o, axis=0) for o in outs], loads


def final_logits(h_rows: np.ndarray, head: dict, dims) -> np.ndarray:
    """Final RMSNorm and LM head on the rows whose next token is sampled
    (after the last layer, each sequence's last position feeds the sampler:
    *Sarathi-Serve overview* §3.2, logits then sampling)."""
    y = rms_norm(h_rows, head["final_norm"], dims.rms_eps)
    return y @ head["lm_head"].T


@dataclasses.dataclass
class Part:
    """One sequence's share of a hybrid batch.

    ``x``: layer-0 inputs of positions ``[given_len, end)``; ``given``: per
    layer ``LayerCache`` of positions ``[0, given_len)`` supplied as state
    (random histories), or ``None``; ``lo``: first position emitted as a
    batch row (a chunk emits ``[start_pos, end)``, a decode ``[ctx, ctx+1)``).
    """

    x: np.ndarray
    lo: int
    given: list | None = None
    is_prefill: bool = False

    @property
    def given_len(self) -> int:
        return 0 if self.given is None else self.given[0].n

    @property
    def end(self) -> int:
        return self.given_len + self.x.shape[0]

    @property
    def n_rows(self) -> int:
        return self.end - self.lo


def serial_step(layers, head, dims, parts: list) -> tuple:
    """Each part run by itself, one-shot over its whole un-cached span; the
    emitted rows are sliced out and stacked chunk-first.  This is what a hybrid
    batch must equal ("hybrid batch output differs from serial execution" is
    the failure the *SARATHI technique write-up* §6.1 debugs)."""
    per_layer = [[] for _ in layers]
    last_rows = []
    for p in parts:
        outs, _ = forward(layers, dims, p.x, p.given)
        off = p.lo - p.given_len
        for l, o in enumerate(outs):
            per_layer[l].append(o[off:])
        last_rows.append(outs[-1][-1])
    hidden = [np.concatenate(r, axis=0) for r in per_layer]
    logits = final_logits(np.stack(last_rows), head, dims) if head else None
    return hidden, logits


def hybrid_step(layers, head, dims, parts: list) -> tuple:
    """The hybrid batch computed the pages' way, "merge -> split -> merge"
    (*SARATHI reading notes* part 2 §3; *SARATHI technique write-up* §3.3):

    1. stack every part's batch rows into one ``[Lp+Bd, H]`` activation
       (chunk rows first, then decodes);
    2. per layer, one projection per weight over all stacked rows;
    3. split attention by row range, each range against its own KV (cache of
       earlier positions, then its own new keys);
    4. write the attention rows back into one contiguous buffer and continue
       with shared projections.

    The KV of positions before a part's first batch row (earlier chunks of a
    prompt, or a decode's own prompt) is built first by ``forward`` and serves
    as that part's cache.  Returns ``(hidden per layer [M, H], logits)`` where
    logits cover the last row of every part.
    """
    caches, xs, poss = [], [], []
    for p in parts:
        pre = p.lo - p.given_len
        if pre > 0:
            _, c = forward(layers, dims, p.x[:pre], p.given)
        elif p.given is not None:
            c = p.given
        else:
            c = [empty_cache(dims, p.x.dtype) for _ in layers]
        caches.append(c)
        xs.append(p.x[pre:])
        poss.append(np.arange(p.lo, p.end))
    h = np.concatenate(xs, axis=0)
    pos = np.concatenate(poss)
    bounds = np.cumsum([0] + [p.n_rows for p in parts])
    hidden = []
    for l, w in enumerate(layers):
        q, k, v = qkv_rope(h, pos, w, dims)
        a = np.empty((h.shape[0], dims.n_q_heads, dims.head_dim), dtype=h.dtype)
        for i, p in enumerate(parts):
            r0, r1 = bounds[i], bounds[i + 1]
            c = caches[i][l]
            K = np.concatenate([c.k, k[r0:r1].astype(c.k.dtype)], axis=0)
            V = np.concatenate([c.v, v[r0:r1].astype(c.v.dtype)], axis=0)
            a[r0:r1] = attention(q[r0:r1], K, V, pos[r0:r1], np.arange(K.shape[0]), window_of(dims))
        h = post_attention(h, a.reshape(h.shape[0], dims.q_dim), w, dims)
        hidden.append(h)
    logits = None
    if head:
        logits = final_logits(h[sampled_rows(parts)], head, dims)
    return hidden, logits


def sampled_rows(parts: list) -> np.ndarray:
    """Stacked-row index of each part's last position, the one whose next
    token is sampled: a chunk's last row (rows are chunk-first, then decodes
    in order: *SARATHI reading notes* part 2 §3), and each decode's only row."""
    return np.cumsum([p.n_rows for p in parts]) - 1
