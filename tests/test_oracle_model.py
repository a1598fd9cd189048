"""Pins of the oracle's decoder-layer arithmetic against things other than itself:
library routines, closed forms, brute force and the method's invariants."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import model as om

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def small_dims(qh=4, kvh=2, d=16, h=64, f=96, layers=1):
    return synth.Dims(n_layers=layers, hidden=h, n_q_heads=qh, n_kv_heads=kvh, head_dim=d,
                      ffn=f, vocab=50)


def np_layers(seed, dims, dtype=np.float64, gain_noise=False):
    layers, head, gen = synth.model_weights(seed, dims, torch.float32)
    out = []
    for w in layers:
        w = om.layer_weights_np(w, dtype)
        if gain_noise:  # non-unit gains so that a dropped gain is caught
            rng = np.random.default_rng(seed)
            w["norm1"] = (1 + 0.3 * rng.standard_normal(dims.hidden)).astype(dtype)
            w["norm2"] = (1 + 0.3 * rng.standard_normal(dims.hidden)).astype(dtype)
        out.append(w)
    hd = om.layer_weights_np(head, dtype)
    return out, hd, gen


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_matches_torch_library():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 33))
    g = rng.standard_normal(33)
    ref = F.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), eps=1e-5).numpy()
    np.testing.assert_allclose(om.rms_norm(x, g, 1e-5), ref, rtol=1e-12, atol=1e-12)


def test_rms_norm_closed_form_constant_row():
    # a row of constant c normalises to sign(c) * c / sqrt(c^2 + eps)
    x = np.full((1, 8), 3.0)
    y = om.rms_norm(x, np.ones(8), 1e-5)
    np.testing.assert_allclose(y, 3.0 / math.sqrt(9.0 + 1e-5))


# ---------------------------------------------------------------- rotary

def test_rope_identity_at_position_zero():
    x = np.random.default_rng(2).standard_normal((1, 3, 16))
    np.testing.assert_allclose(om.apply_rope(x, [0], 1e4), x, atol=0)


def test_rope_is_complex_rotation_of_half_pairs():
    # closed form: (x_i + j x_{i+d/2}) * exp(j * p * base^(-2i/d))
    rng = np.random.default_rng(3)
    d, base = 32, 10000.0
    x = rng.standard_normal((5, 2, d))
    pos = np.array([0, 1, 7, 100, 4095])
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    theta = np.array([base ** (-2 * i / d) for i in range(d // 2)])
    zr = z * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    ref = np.concatenate([zr.real, zr.imag], axis=-1)
    np.testing.assert_allclose(om.apply_rope(x, pos, base), ref, rtol=1e-12, atol=1e-12)


def test_rope_preserves_pair_norms_and_is_relative():
    rng = np.random.default_rng(4)
    d = 64
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    qr = om.apply_rope(q, [37], 1e4)
    half = d // 2
    n0 = q[..., :half] ** 2 + q[..., half:] ** 2
    n1 = qr[..., :half] ** 2 + qr[..., half:] ** 2
    np.testing.assert_allclose(n0, n1, rtol=1e-12)
    # <R_m q, R_n k> depends on m - n only
    dots = []
    for m, n in [(10, 3), (107, 100), (2007, 2000)]:
        dots.append(float(np.sum(om.apply_rope(q, [m], 1e4) * om.apply_rope(k, [n], 1e4))))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# ---------------------------------------------------------------- SwiGLU pieces

def test_silu_matches_torch_library():
    x = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(om.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- attention

def brute_attention(q, k, v, q_pos, k_pos, window=0):
    """Triple loop in float64: softmax over visible keys, one query/head at a time.
    A key is visible when its distance back from the query, ``q_pos - k_pos``,
    is in ``[0, window)`` (any non-negative distance when ``window`` is 0)."""
    T, qh, d = q.shape
    S, kvh, _ = k.shape
    g = qh // kvh
    out = np.zeros_like(q)
    for t in range(T):
        for h in range(qh):
            kh = h // g
            sc = []
            for s in range(S):
                dist = q_pos[t] - k_pos[s]
                if dist >= 0 and (window == 0 or dist < window):
                    sc.append((s, sum(q[t, h, i] * k[s, kh, i] for i in range(d)) / math.sqrt(d)))
            m = max(v_ for _, v_ in sc)
            den = sum(math.exp(v_ - m) for _, v_ in sc)
            for s, v_ in sc:
                out[t, h] += math.exp(v_ - m) / den * v[s, kh]
    return out


@pytest.mark.parametrize("qh,kvh", [(4, 4), (4, 2), (6, 2), (7, 1)])
def test_attention_matches_brute_force(qh, kvh):
    rng = np.random.default_rng(5)
    d, S, T = 8, 11, 4
    q = rng.standard_normal((T, qh, d))
    k = rng.standard_normal((S, kvh, d))
    v = rng.standard_normal((S, kvh, d))
    q_pos = np.array([7, 8, 9, 10])  # a chunk starting at position 7 after 7 cached keys
    k_pos = np.arange(S)
    np.testing.assert_allclose(om.attention(q, k, v, q_pos, k_pos),
                               brute_attention(q, k, v, q_pos, k_pos), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("qh,kvh", [(4, 4), (8, 2)])
def test_attention_matches_torch_sdpa_causal(qh, kvh):
    # a prefill with no cache and no decodes reduces to library causal SDPA
    rng = np.random.default_rng(6)
    T, d = 33, 16
    q = rng.standard_normal((T, qh, d))
    k = rng.standard_normal((T, kvh, d))
    v = rng.standard_normal((T, kvh, d))
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(qh // kvh, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(qh // kvh, dim=0)
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True).permute(1, 0, 2).numpy()
    out = om.attention(q, k, v, np.arange(T), np.arange(T))
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_decode_row_equals_library_attention_over_full_history():
    # one decode query at position ctx sees all ctx+1 keys (no mask)
    rng = np.random.default_rng(7)
    ctx, qh, kvh, d = 40, 4, 1, 16
    q = rng.standard_normal((1, qh, d))
    k = rng.standard_normal((ctx + 1, kvh, d))
    v = rng.standard_normal((ctx + 1, kvh, d))
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).expand(qh, -1, -1)
    tv = torch.from_numpy(v).permute(1, 0, 2).expand(qh, -1, -1)
    ref = F.scaled_dot_product_attention(tq, tk, tv).permute(1, 0, 2).numpy()
    out = om.attention(q, k, v, [ctx], np.arange(ctx + 1))
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- sliding window


def test_window_one_sees_only_its_own_key():
    # closed form: with one visible key the softmax is 1 there, the output is that value
    rng = np.random.default_rng(21)
    T, S, qh, kvh, d = 5, 12, 4, 2, 8
    q = rng.standard_normal((T, qh, d))
    k = rng.standard_normal((S, kvh, d))
    v = rng.standard_normal((S, kvh, d))
    q_pos = np.arange(7, 12)
    out = om.attention(q, k, v, q_pos, np.arange(S), window=1)
    for t in range(T):
        for h in range(qh):
            np.testing.assert_allclose(out[t, h], v[q_pos[t], h // (qh // kvh)], rtol=0, atol=1e-15)


def test_window_two_is_a_two_key_softmax():
    # closed form: the query mixes its own value and the previous one by sigmoid weights
    rng = np.random.default_rng(22)
    d = 16
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((9, 1, d))
    v = rng.standard_normal((9, 1, d))
    out = om.attention(q, k, v, [8], np.arange(9), window=2)
    s7 = q[0, 0] @ k[7, 0] / math.sqrt(d)
    s8 = q[0, 0] @ k[8, 0] / math.sqrt(d)
    w8 = 1.0 / (1.0 + math.exp(s7 - s8))
    np.testing.assert_allclose(out[0, 0], w8 * v[8, 0] + (1 - w8) * v[7, 0], rtol=1e-13, atol=1e-14)


def test_window_covering_the_prefix_is_full_causal():
    rng = np.random.default_rng(23)
    T, S, qh, kvh, d = 6, 20, 4, 2, 8
    q = rng.standard_normal((T, qh, d))
    k = rng.standard_normal((S, kvh, d))
    v = rng.standard_normal((S, kvh, d))
    q_pos = np.arange(14, 20)
    full = om.attention(q, k, v, q_pos, np.arange(S))
    for w in (20, 21, 1000):
        np.testing.assert_array_equal(om.attention(q, k, v, q_pos, np.arange(S), window=w), full)
    assert np.abs(om.attention(q, k, v, q_pos, np.arange(S), window=19) - full).max() > 1e-6


@pytest.mark.parametrize("window", [1, 3, 5, 9])
def test_window_matches_brute_force(window):
    rng = np.random.default_rng(24)
    d, S, T, qh, kvh = 8, 13, 5, 6, 2
    q = rng.standard_normal((T, qh, d))
    k = rng.standard_normal((S, kvh, d))
    v = rng.standard_normal((S, kvh, d))
    q_pos = np.arange(8, 13)
    np.testing.assert_allclose(om.attention(q, k, v, q_pos, np.arange(S), window=window),
                               brute_attention(q, k, v, q_pos, np.arange(S), window), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("window", [4, 16, 31])
def test_window_matches_torch_sdpa_band_mask(window):
    # the library's attention with an explicit band mask (i - j in [0, window))
    rng = np.random.default_rng(25)
    T, d, qh, kvh = 40, 16, 8, 2
    q = rng.standard_normal((T, qh, d))
    k = rng.standard_normal((T, kvh, d))
    v = rng.standard_normal((T, kvh, d))
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    band = (i - j >= 0) & (i - j < window)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(qh // kvh, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(qh // kvh, dim=0)
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=band).permute(1, 0, 2).numpy()
    out = om.attention(q, k, v, np.arange(T), np.arange(T), window=window)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_window_off_by_one_is_caught():
    # a window that admits one key too many (>= instead of >) disagrees with the band reference
    rng = np.random.default_rng(26)
    T, d = 12, 8
    q = rng.standard_normal((T, 1, d))
    k = rng.standard_normal((T, 1, d))
    v = rng.standard_normal((T, 1, d))
    ref = brute_attention(q, k, v, np.arange(T), np.arange(T), 4)
    wide = brute_attention(q, k, v, np.arange(T), np.arange(T), 5)
    np.testing.assert_allclose(om.attention(q, k, v, np.arange(T), np.arange(T), window=4), ref,
                               rtol=1e-10, atol=1e-12)
    assert np.abs(wide - ref).max() > 1e-3


@pytest.mark.parametrize("window", [5, 16, 40])
def test_windowed_chunked_prefill_equals_one_shot(window):
    import dataclasses
    dims = dataclasses.replace(small_dims(layers=2), sliding_window=window)
    layers, _, gen = np_layers(27, dims)
    x = synth.normal(gen, (64, dims.hidden)).double().numpy()
    one, _ = om.forward(layers, dims, x)
    full, _ = om.forward(layers, small_dims(layers=2), x)
    assert np.abs(one[-1] - full[-1]).max() > 1e-6  # the window changes the result
    for chunk in (8, 24, 48):
        ch, _ = om.chunked_prefill(layers, dims, x, chunk)
        for a, b in zip(ch, one):
            np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("with_given", [False, True])
def test_windowed_hybrid_batch_equals_serial_execution(with_given):
    import dataclasses
    dims = dataclasses.replace(small_dims(layers=2), sliding_window=7)
    layers, head, gen = np_layers(28, dims)
    parts = _parts_for(dims, layers, gen, with_given)
    hyb, lh = om.hybrid_step(layers, head, dims, parts)
    ser, ls = om.serial_step(layers, head, dims, parts)
    for a, b in zip(hyb, ser):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(lh, ls, rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------- whole layer

def torch_layer(x, w, dims):
    """Llama-style layer composed from torch library routines only."""
    t = {k: torch.from_numpy(v) for k, v in w.items()}
    x = torch.from_numpy(x)
    T = x.shape[0]
    y = F.rms_norm(x, (dims.hidden,), t["norm1"], eps=dims.rms_eps)
    q = F.linear(y, t["wq"]).view(T, dims.n_q_heads, dims.head_dim)
    k = F.linear(y, t["wk"]).view(T, dims.n_kv_heads, dims.head_dim)
    v = F.linear(y, t["wv"]).view(T, dims.n_kv_heads, dims.head_dim)
    # rotary via complex multiplication of half pairs
    half = dims.head_dim // 2
    inv = dims.rope_base ** (-torch.arange(half, dtype=torch.float64) * 2 / dims.head_dim)
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64),
                      torch.arange(T, dtype=torch.float64)[:, None] * inv[None])

    def rope(z):
        c = torch.complex(z[..., :half], z[..., half:]) * rot[:, None, :]
        return torch.cat([c.real, c.imag], dim=-1)

    q, k = rope(q), rope(k)
    g = dims.n_q_heads // dims.n_kv_heads
    a = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1).repeat_interleave(g, 0),
                                       v.transpose(0, 1).repeat_interleave(g, 0), is_causal=True)
    h = x + F.linear(a.transpose(0, 1).reshape(T, -1), t["wo"])
    y = F.rms_norm(h, (dims.hidden,), t["norm2"], eps=dims.rms_eps)
    return (h + F.linear(F.silu(F.linear(y, t["wg"])) * F.linear(y, t["wu"]), t["wd"])).numpy()


@pytest.mark.parametrize("qh,kvh", [(4, 4), (4, 2), (7, 1)])
def test_decoder_layer_matches_torch_composition(qh, kvh):
    dims = small_dims(qh=qh, kvh=kvh)
    layers, _, gen = np_layers(11, dims, gain_noise=True)
    x = synth.normal(gen, (21, dims.hidden)).double().numpy()
    out, _ = om.decoder_layer(x, np.arange(21), layers[0], dims, om.empty_cache(dims))
    np.testing.assert_allclose(out, torch_layer(x, layers[0], dims), rtol=1e-9, atol=1e-10)


# ---------------------------------------------------------------- method invariants

@pytest.mark.parametrize("dtype,tol", [(np.float64, 1e-11), (np.float32, 1e-5)])
def test_chunked_prefill_equals_one_shot(dtype, tol):
    dims = small_dims(layers=2)
    layers, _, gen = np_layers(12, dims, dtype)
    x = synth.normal(gen, (64, dims.hidden)).numpy().astype(dtype)
    one, _ = om.forward(layers, dims, x)
    for chunk in (16, 32, 48):
        ch, _ = om.chunked_prefill(layers, dims, x, chunk)
        for a, b in zip(ch, one):
            rel = np.linalg.norm(a - b) / np.linalg.norm(b)
            assert rel <= tol, (chunk, rel)


def test_causality_future_rows_do_not_change_past_rows():
    dims = small_dims()
    layers, _, gen = np_layers(13, dims)
    x = synth.normal(gen, (20, dims.hidden)).double().numpy()
    a, _ = om.forward(layers, dims, x)
    x2 = x.copy()
    x2[12:] += 5.0
    b, _ = om.forward(layers, dims, x2)
    np.testing.assert_array_equal(a[0][:12], b[0][:12])
    assert np.abs(a[0][12:] - b[0][12:]).max() > 1e-3


def test_position_continuity_across_chunks():
    # a chunk processed at start_pos s with the cache equals rows s.. of one-shot,
    # and shifting its position ids breaks it
    dims = small_dims()
    layers, _, gen = np_layers(14, dims)
    x = synth.normal(gen, (24, dims.hidden)).double().numpy()
    one, _ = om.forward(layers, dims, x)
    _, cache = om.forward(layers, dims, x[:16])
    second, _ = om.forward(layers, dims, x[16:], cache)
    np.testing.assert_allclose(second[0], one[0][16:], rtol=1e-11, atol=1e-12)
    q, k, v = om.qkv_rope(x[16:], np.arange(0, 8), layers[0], dims)  # wrong ids: restart at 0
    K = np.concatenate([cache[0].k, k])
    V = np.concatenate([cache[0].v, v])
    a = om.attention(q, K, V, np.arange(16, 24), np.arange(24)).reshape(8, -1)
    wrong = om.post_attention(x[16:], a, layers[0], dims)
    assert np.abs(wrong - one[0][16:]).max() > 1e-6  # far above float64 rounding


def test_prior_chunk_loads_count_is_n_n_minus_1_over_2():
    dims = small_dims(h=32, f=32, qh=2, kvh=1, d=8)
    layers, _, gen = np_layers(15, dims)
    x = synth.normal(gen, (48, dims.hidden)).double().numpy()
    for chunk in (4, 6, 8, 12, 16, 24, 48):
        n = 48 // chunk
        _, loads = om.chunked_prefill(layers, dims, x, chunk)
        brute = sum(1 for k in range(n) for later in range(k + 1, n))
        assert loads == brute == n * (n - 1) // 2


def _parts_for(dims, layers, gen, with_given):
    """A chunk at start 24 (len 12) and three decodes."""
    prompt = synth.normal(gen, (36, dims.hidden)).double().numpy()
    parts = [om.Part(x=prompt, lo=24, is_prefill=True)]
    for ctx in (5, 17, 30):
        if with_given:
            given = []
            for _ in layers:
                k = synth.normal(gen, (ctx, dims.n_kv_heads, dims.head_dim)).double().numpy()
                v = synth.normal(gen, (ctx, dims.n_kv_heads, dims.head_dim)).double().numpy()
                given.append(om.LayerCache(k, v))
            x = synth.normal(gen, (1, dims.hidden)).double().numpy()
            parts.append(om.Part(x=x, lo=ctx, given=given))
        else:
            x = synth.normal(gen, (ctx + 1, dims.hidden)).double().numpy()
            parts.append(om.Part(x=x, lo=ctx))
    return parts


@pytest.mark.parametrize("with_given", [False, True])
def test_hybrid_batch_equals_serial_execution(with_given):
    dims = small_dims(layers=2)
    layers, head, gen = np_layers(16, dims)
    parts = _parts_for(dims, layers, gen, with_given)
    hyb, lh = om.hybrid_step(layers, head, dims, parts)
    ser, ls = om.serial_step(layers, head, dims, parts)
    assert hyb[0].shape == (12 + 3, dims.hidden)
    for a, b in zip(hyb, ser):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(lh, ls, rtol=1e-10, atol=1e-11)


def test_hybrid_rows_are_chunk_first_then_decodes_in_order():
    dims = small_dims()
    layers, head, gen = np_layers(17, dims)
    parts = _parts_for(dims, layers, gen, False)
    hyb, _ = om.hybrid_step(layers, head, dims, parts)
    alone, _ = om.forward(layers, dims, parts[2].x)  # the second decode by itself
    np.testing.assert_allclose(hyb[0][12 + 1], alone[0][-1], rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------- final norm + LM head

def torch_logits(h_rows, head, dims):
    """Final norm and LM head composed from library routines (float64)."""
    h = torch.from_numpy(np.asarray(h_rows, dtype=np.float64))
    g = torch.from_numpy(head["final_norm"])
    return F.linear(F.rms_norm(h, (dims.hidden,), g, eps=dims.rms_eps), torch.from_numpy(head["lm_head"])).numpy()


def _head_with_gain(head, dims, seed):
    rng = np.random.default_rng(seed)
    head = dict(head)
    head["final_norm"] = 1 + 0.3 * rng.standard_normal(dims.hidden)  # non-unit: a dropped norm shows
    return head


def test_final_logits_match_torch_composition():
    dims = small_dims()
    _, head, gen = np_layers(21, dims)
    head = _head_with_gain(head, dims, 21)
    h = 3.0 * synth.normal(gen, (6, dims.hidden)).double().numpy()
    np.testing.assert_allclose(om.final_logits(h, head, dims), torch_logits(h, head, dims), rtol=1e-11, atol=1e-12)


def test_final_logits_closed_form_constant_row():
    # a row of constant c normalises to c / sqrt(c^2 + eps) in every column,
    # so its logits are that factor times lm_head @ gain
    dims = small_dims()
    _, head, _ = np_layers(22, dims)
    head = _head_with_gain(head, dims, 22)
    for c in (-2.5, 0.01, 7.0):
        got = om.final_logits(np.full((1, dims.hidden), c), head, dims)[0]
        want = c / math.sqrt(c * c + dims.rms_eps) * (head["lm_head"] @ head["final_norm"])
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def _logits_pin_holds(parts, hidden, logits, head, dims):
    """The hybrid step's logits are the library composition on each part's
    last stacked row; the rows are counted here from the parts' own lengths."""
    rows, r = [], 0
    for p in parts:
        r += (p.end - p.lo)
        rows.append(r - 1)
    want = torch_logits(hidden[-1][rows], head, dims)
    return logits.shape == want.shape and np.allclose(logits, want, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("with_given", [False, True])
def test_hybrid_logits_are_last_row_of_each_part(with_given):
    dims = small_dims(layers=2)
    layers, head, gen = np_layers(23, dims)
    head = _head_with_gain(head, dims, 23)
    parts = _parts_for(dims, layers, gen, with_given)
    hyb, lg = om.hybrid_step(layers, head, dims, parts)
    assert lg.shape == (len(parts), dims.vocab)
    assert _logits_pin_holds(parts, hyb, lg, head, dims)


def test_planted_head_mistakes_are_caught(monkeypatch):
    """Each planted mistake in the oracle's head breaks one of the pins above."""
    dims = small_dims(layers=2)
    layers, head, gen = np_layers(24, dims)
    head = _head_with_gain(head, dims, 24)
    parts = _parts_for(dims, layers, gen, False)
    h = 3.0 * synth.normal(gen, (5, dims.hidden)).double().numpy()
    # the final norm dropped
    with monkeypatch.context() as m:
        m.setattr(om, "final_logits", lambda rows, hd, d: rows @ hd["lm_head"].T)
        assert not np.allclose(om.final_logits(h, head, dims), torch_logits(h, head, dims), rtol=1e-6)
        hyb, lg = om.hybrid_step(layers, head, dims, parts)
        assert not _logits_pin_holds(parts, hyb, lg, head, dims)
    # the gain dropped from the final norm
    with monkeypatch.context() as m:
        m.setattr(om, "final_logits",
                  lambda rows, hd, d: om.rms_norm(rows, np.ones(d.hidden), d.rms_eps) @ hd["lm_head"].T)
        assert not np.allclose(om.final_logits(h, head, dims), torch_logits(h, head, dims), rtol=1e-6)
    # the chunk's first row sampled instead of its last
    with monkeypatch.context() as m:
        m.setattr(om, "sampled_rows", lambda ps: np.cumsum([0] + [p.n_rows for p in ps])[:-1])
        hyb, lg = om.hybrid_step(layers, head, dims, parts)
        assert not _logits_pin_holds(parts, hyb, lg, head, dims)
    # unpatched, every pin holds
    hyb, lg = om.hybrid_step(layers, head, dims, parts)
    assert _logits_pin_holds(parts, hyb, lg, head, dims)


# ---------------------------------------------------------------- planted mistakes

def _mutant_cases():
    def drop_residual(x, a, w, dims):
        y = om.rms_norm(x + a @ w["wo"].T, w["norm2"], dims.rms_eps)
        return (om.silu(y @ w["wg"].T) * (y @ w["wu"].T)) @ w["wd"].T

    def transposed_pairing(x, pos, base):
        d = x.shape[-1]
        ang = np.asarray(pos, float)[:, None] * om.rope_inv_freq(d, base)[None]
        c, s = np.cos(ang)[:, None], np.sin(ang)[:, None]
        x1, x2 = x[..., 0::2], x[..., 1::2]  # interleaved pairing instead of rotate-half
        out = np.empty_like(x)
        out[..., 0::2] = x1 * c - x2 * s
        out[..., 1::2] = x2 * c + x1 * s
        return out

    def wrong_sign(x, pos, base):
        return _orig_rope(x, -np.asarray(pos), base)

    def no_eps_gain(x, g, eps):
        return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)

    return [("post_attention", drop_residual), ("apply_rope", transposed_pairing),
            ("apply_rope", wrong_sign), ("rms_norm", no_eps_gain)]


_orig_rope = om.apply_rope


@pytest.mark.parametrize("name,fn", _mutant_cases())
def test_planted_oracle_mistakes_are_caught(monkeypatch, name, fn):
    dims = small_dims(qh=4, kvh=2)
    layers, _, gen = np_layers(18, dims, gain_noise=True)
    x = synth.normal(gen, (9, dims.hidden)).double().numpy()
    ref = torch_layer(x, layers[0], dims)
    monkeypatch.setattr(om, name, fn)
    out, _ = om.decoder_layer(x, np.arange(9), layers[0], dims, om.empty_cache(dims))
    assert not np.allclose(out, ref, rtol=1e-6, atol=1e-6)
