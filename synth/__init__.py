"""Seeded synthetic inputs for the hybrid-batch step.

This module draws random numbers and arranges them into the shapes the
decoder-layer step consumes; it computes no part of the step itself (no
normalisation, projection, rotary embedding, attention or scheduling).  Both
the oracle checks and the CUDA path take their inputs from here, so that the
two sides see identical values and share nothing else.

Recipe (all draws from ``torch.Generator`` seeded explicitly, CPU unless a
device generator is asked for):

* weight matrices ``N(0, 0.02)``, drawn layer-major in the order
  Wq, Wk, Wv, Wo, Wg, Wu, Wd, then the embedding and the LM head;
  RMSNorm gains are ones (they are not random);
* layer-0 hidden inputs and random key/value histories ``N(0, 1)``;
* decode context lengths uniform integers in a closed range;
* request traces: Poisson arrivals (exponential gaps) and lognormal prompt /
  output lengths with ``mu = ln(median)``, clipped, from a NumPy PCG64
  generator.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Dims:
    """Decoder shape: Llama/Mistral-style layer with GQA and SwiGLU."""

    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int = 0
    rms_eps: float = 1e-5
    rope_base: float = 10000.0
    # keys a query may see, itself included (0 = the whole causal prefix)
    sliding_window: int = 0

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim


# Tiny single layer: H=256, 4 heads x 64 (MHA), FFN 1024, no vocabulary.
TINY = Dims(n_layers=1, hidden=256, n_q_heads=4, n_kv_heads=4, head_dim=64, ffn=1024, vocab=0)
# One Mistral-7B-shaped layer with its 32000-entry head.
MISTRAL_LAYER = Dims(n_layers=1, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                     ffn=14336, vocab=32000)
# The full 32-layer Mistral-7B shape.
MISTRAL_7B = dataclasses.replace(MISTRAL_LAYER, n_layers=32)
# Yi-34B shape, 60 layers; the vocabulary size is not given with the shape, 64000 is used.
YI_34B = Dims(n_layers=60, hidden=7168, n_q_heads=56, n_kv_heads=8, head_dim=128, ffn=20480,
              vocab=64000)

WEIGHT_STD = 0.02
LAYER_WEIGHT_NAMES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def generator(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(gen: torch.Generator, shape, std: float = 1.0, dtype=torch.float32,
           device: str = "cpu") -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def layer_shapes(d: Dims) -> dict:
    """Shapes of one layer's weights, ``[out, in]`` row-major like a linear layer."""
    return {
        "wq": (d.q_dim, d.hidden),
        "wk": (d.kv_dim, d.hidden),
        "wv": (d.kv_dim, d.hidden),
        "wo": (d.hidden, d.q_dim),
        "wg": (d.ffn, d.hidden),
        "wu": (d.ffn, d.hidden),
        "wd": (d.hidden, d.ffn),
    }


def layer_weights(gen: torch.Generator, d: Dims, dtype=torch.bfloat16, device: str = "cpu") -> dict:
    """One layer's weights in the documented draw order, plus unit norm gains."""
    out = {}
    for name, shape in layer_shapes(d).items():
        out[name] = normal(gen, shape, WEIGHT_STD, dtype, device)
    out["norm1"] = torch.ones(d.hidden, dtype=dtype, device=device)
    out["norm2"] = torch.ones(d.hidden, dtype=dtype, device=device)
    return out


def head_weights(gen: torch.Generator, d: Dims, dtype=torch.bfloat16, device: str = "cpu") -> dict:
    """Embedding ``[V, H]``, final norm gain (ones) and LM head ``[V, H]``."""
    if d.vocab == 0:
        return {}
    return {
        "embed": normal(gen, (d.vocab, d.hidden), WEIGHT_STD, dtype, device),
        "final_norm": torch.ones(d.hidden, dtype=dtype, device=device),
        "lm_head": normal(gen, (d.vocab, d.hidden), WEIGHT_STD, dtype, device),
    }


def model_weights(seed: int, d: Dims, dtype=torch.bfloat16, device: str = "cpu"):
    """All layers then the head, from one generator (layer-major draw order)."""
    gen = generator(seed, device)
    layers = [layer_weights(gen, d, dtype, device) for _ in range(d.n_layers)]
    head = head_weights(gen, d, dtype, device)
    return layers, head, gen


def uniform_int(gen: torch.Generator, n: int, lo: int, hi: int) -> list[int]:
    """``n`` integers uniform on the closed range ``[lo, hi]``."""
    return [int(v) for v in torch.randint(lo, hi + 1, (n,), generator=gen)]


def kv_history(gen: torch.Generator, n_layers: int, ctx: int, d: Dims, dtype=torch.bfloat16,
               device: str = "cpu"):
    """Random post-rotary key/value history ``[(K[ctx,kvh,dh], V[ctx,kvh,dh])] * n_layers``."""
    out = []
    for _ in range(n_layers):
        k = normal(gen, (ctx, d.n_kv_heads, d.head_dim), 1.0, dtype, device)
        v = normal(gen, (ctx, d.n_kv_heads, d.head_dim), 1.0, dtype, device)
        out.append((k, v))
    return out


def page_permutation(gen: torch.Generator, num_pages: int) -> list[int]:
    """A seeded shuffle of page ids, so that block tables are not contiguous."""
    return [int(v) for v in torch.randperm(num_pages, generator=gen)]


@dataclasses.dataclass(frozen=True)
class TraceRequest:
    req: int
    arrival: float
    prompt_len: int
    output_len: int


def request_trace(seed: int, n: int, rate: float, prompt_median: float, prompt_clip: tuple,
                  out_median: float, out_clip: tuple, sigma: float = 1.0) -> list[TraceRequest]:
    """Poisson arrivals at ``rate`` req/s and clipped lognormal lengths."""
    rng = np.random.Generator(np.random.PCG64(seed))
    gaps = rng.exponential(1.0 / rate, size=n)
    arrivals = np.cumsum(gaps) - gaps[0]
    p = rng.lognormal(math.log(prompt_median), sigma, size=n)
    o = rng.lognormal(math.log(out_median), sigma, size=n)
    p = np.clip(np.rint(p), prompt_clip[0], prompt_clip[1]).astype(np.int64)
    o = np.clip(np.rint(o), out_clip[0], out_clip[1]).astype(np.int64)
    return [TraceRequest(i, float(arrivals[i]), int(p[i]), int(o[i])) for i in range(n)]


def prompt_tokens(seed: int, trace: list[TraceRequest], vocab: int) -> dict[int, list[int]]:
    """Prompt token ids uniform in ``[0, vocab)`` for every request of a trace."""
    gen = generator(seed)
    return {r.req: [int(t) for t in torch.randint(0, vocab, (r.prompt_len,), generator=gen)]
            for r in trace}


# ---------------------------------------------------------------------------
# Workload cases.  Each returns plain tensors; what is computed from them is
# the business of the oracle on one side and the library on the other.
# ---------------------------------------------------------------------------

def tiny_case(seed: int = 0, dtype=torch.float32):
    """Tiny layer: one 512-token prompt in two 256-token chunks with four
    piggybacked decodes whose contexts 100/180/250/300 come from their own
    prompts.  Draw order after the weights: the long prompt, each decode
    prompt, then one decode input per decode per step (step-major)."""
    d = TINY
    layers, head, gen = model_weights(seed, d, dtype)
    prompt = normal(gen, (512, d.hidden), 1.0, dtype)
    ctxs = [100, 180, 250, 300]
    decode_prompts = [normal(gen, (c, d.hidden), 1.0, dtype) for c in ctxs]
    n_steps = 2
    decode_inputs = [[normal(gen, (1, d.hidden), 1.0, dtype) for _ in ctxs] for _ in range(n_steps)]
    return dict(dims=d, layers=layers, head=head, prompt=prompt, chunk=256, ctxs=ctxs,
                decode_prompts=decode_prompts, decode_inputs=decode_inputs)


SMALL_128 = Dims(n_layers=1, hidden=512, n_q_heads=4, n_kv_heads=2, head_dim=128, ffn=1024, vocab=0)


def window_case(seed: int = 0, d: Dims = SMALL_128, prompt_len: int = 640, ctxs=(90, 200, 333, 700)):
    """A one-layer case for sliding-window checks: a prompt of ``prompt_len``
    N(0,1) rows (chunked by the caller) and decodes at contexts ``ctxs`` with
    random N(0,1) K/V histories and one N(0,1) input row each.  Draw order
    after the weights: the prompt, the decode inputs, then the histories."""
    layers, _, gen = model_weights(seed, d, torch.bfloat16)
    prompt = normal(gen, (prompt_len, d.hidden), 1.0, torch.bfloat16)
    decode_inputs = normal(gen, (len(ctxs), d.hidden), 1.0, torch.bfloat16)
    hist = [kv_history(gen, 1, c, d, torch.bfloat16)[0] for c in ctxs]
    return dict(dims=d, layers=layers, prompt=prompt, ctxs=list(ctxs), decode_inputs=decode_inputs,
                histories=hist)


SMALL_128_HEAD = dataclasses.replace(SMALL_128, vocab=1024)


def multi_chunk_case(seed: int = 0, d: Dims = SMALL_128_HEAD, prompt_lens=(300, 180, 90),
                     ctxs=(70, 150, 260, 333)):
    """A one-layer case for batches of several prefill chunks: prompts of
    ``prompt_lens`` N(0,1) rows and decodes at contexts ``ctxs`` with random
    N(0,1) K/V histories and one N(0,1) input row each.  Draw order after the
    weights (and head): the prompts, the decode inputs, then the histories."""
    layers, head, gen = model_weights(seed, d, torch.bfloat16)
    prompts = [normal(gen, (n, d.hidden), 1.0, torch.bfloat16) for n in prompt_lens]
    decode_inputs = normal(gen, (len(ctxs), d.hidden), 1.0, torch.bfloat16)
    hist = [kv_history(gen, 1, c, d, torch.bfloat16)[0] for c in ctxs]
    return dict(dims=d, layers=layers, head=head, prompts=prompts, ctxs=list(ctxs),
                decode_inputs=decode_inputs, histories=hist)


MISTRAL_STARTS = (0, 512, 1536)


def mistral_layer_case(seed: int = 0, n_decode: int = 64, tau: int = 512, starts=MISTRAL_STARTS,
                       ctx_range=(128, 4096), with_history: bool = True, device: str = "cpu"):
    """One Mistral-shaped layer (+ head) at token budget ``tau``: for each start
    position a prompt of ``start + tau - n_decode`` N(0,1) rows, plus
    ``n_decode`` decodes with uniform contexts, random N(0,1) K/V histories
    and one N(0,1) input row each.  Draw order after the weights: decode
    contexts, prompts (by start), decode inputs, then histories."""
    d = MISTRAL_LAYER
    layers, head, gen = model_weights(seed, d, torch.bfloat16, device)
    lp = tau - n_decode
    ctxs = uniform_int(gen, n_decode, ctx_range[0], ctx_range[1]) if n_decode else []
    prompts = {s: normal(gen, (s + lp, d.hidden), 1.0, torch.bfloat16, device) for s in starts}
    decode_inputs = normal(gen, (n_decode, d.hidden), 1.0, torch.bfloat16, device)
    hist = [kv_history(gen, 1, c, d, torch.bfloat16, device)[0] for c in ctxs] if with_history else None
    return dict(dims=d, layers=layers, head=head, lp=lp, tau=tau, starts=tuple(starts),
                prompts=prompts, ctxs=ctxs, decode_inputs=decode_inputs, histories=hist)


SWEEP_ROWS = (128, 255, 256, 257, 384, 511, 512, 1024, 2048)


def tile_sweep_case(seed: int = 0, rows=SWEEP_ROWS, n_decode: int = 32, ctx: int = 2048,
                    device: str = "cpu"):
    """One Mistral-shaped layer (no head) stepped at several batch sizes
    ``M = Lp + n_decode``: a prompt of ``max(rows) - n_decode`` N(0,1) rows
    whose first ``Lp`` rows form the chunk (start 0) of each step, plus
    ``n_decode`` decodes at context ``ctx`` with random N(0,1) K/V histories
    and one N(0,1) input row each.  Draw order after the weights: the prompt,
    the decode inputs, then the histories."""
    d = dataclasses.replace(MISTRAL_LAYER, vocab=0)
    layers, _, gen = model_weights(seed, d, torch.bfloat16, device)
    prompt = normal(gen, (max(rows) - n_decode, d.hidden), 1.0, torch.bfloat16, device)
    decode_inputs = normal(gen, (n_decode, d.hidden), 1.0, torch.bfloat16, device)
    hist = [kv_history(gen, 1, ctx, d, torch.bfloat16, device)[0] for _ in range(n_decode)]
    return dict(dims=d, layers=layers, rows=tuple(rows), prompt=prompt, ctx=ctx,
                decode_inputs=decode_inputs, histories=hist)


def long_prompt_case(seed: int, d: Dims, prompt_len: int = 16384, n_decode: int = 128,
                     ctx_range=(512, 8192)):
    """Token ids of one long prompt (uniform in ``[0, vocab)``) and the context
    lengths of the decodes piggybacked on each of its chunks (uniform in
    ``ctx_range``), drawn in that order from a CPU generator seeded ``seed``."""
    gen = generator(seed)
    prompt = torch.randint(0, d.vocab, (prompt_len,), generator=gen, dtype=torch.int64).to(torch.int32)
    ctxs = uniform_int(gen, n_decode, ctx_range[0], ctx_range[1])
    return prompt, ctxs


def decode_history(seed: int, n_layers: int, ctx: int, d: Dims):
    """Random N(0,1) K/V history of one decode, from its own CPU generator
    seeded ``seed``, so that either side can draw it again when it needs it
    instead of holding every decode's history at once."""
    return kv_history(generator(seed), n_layers, ctx, d, torch.bfloat16)
