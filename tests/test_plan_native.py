"""The library's step planner on the host (sar_plan_inspect), no GPU: every
batch row's position and page slot, the chunk-attention tiles, the decode
work split (key ranges, partials, sliding-window start), the logits rows, and
the plan shape a captured step graph relies on."""

import dataclasses

import numpy as np
import pytest

import chunked_prefill_hybrid_sar_gb300 as sar
import synth

PS = 16


def unpack(r):
    m = r["meta"]

    def arr(off, n):
        return m[off:off + n]

    out = dict(r)
    out["pos"] = arr(r["o_pos"], r["M"])
    out["slot"] = arr(r["o_slot"], r["M"])
    bd = r["Bd"]
    out["nkeys"] = arr(r["o_nkeys"], bd)
    out["btoff"] = arr(r["o_btoff"], bd)
    out["btlen"] = arr(r["o_btlen"], bd)
    out["pbeg"] = arr(r["o_pbeg"], bd)
    out["pcnt"] = arr(r["o_pcnt"], bd)
    out["items"] = [tuple(arr(r["o_items"] + 4 * i, 4)) for i in range(r["n_items"])]
    out["bt"] = arr(r["o_bt"], sum(out["btlen"]))
    out["rows"] = arr(r["o_rows"], r["R"])
    out["tiles"] = [tuple(arr(r["o_tiles"] + 8 * i, 8)) for i in range(r["n_tiles"])]
    out["comb"] = [tuple(arr(r["o_comb"] + 4 * i, 4)) for i in range(r["n_comb"])]
    out["pbt"] = m[r["o_pbt"]:r["o_nkeys"]]
    return out


def random_batch(rng, n_chunks, n_dec, max_ctx=3000, pages=20000):
    perm = rng.permutation(pages).tolist()
    nxt = 0

    def take(n):
        nonlocal nxt
        out = perm[nxt:nxt + n]
        nxt += n
        return out

    chunks, decs = [], []
    for i in range(n_chunks):
        start = int(rng.integers(0, 1500))
        ln = int(rng.integers(1, 200))
        chunks.append((i, start, ln, take((start + ln - 1) // PS + 1 + int(rng.integers(0, 3)))))
    for i in range(n_dec):
        ctx = int(rng.integers(0, max_ctx))
        decs.append((100 + i, ctx, take(ctx // PS + 1 + int(rng.integers(0, 2)))))
    return chunks, decs


def plan(dims, chunks, decs, sms=152, max_tokens=1024, max_decodes=128, pages=20000, chunk_split=True):
    b = sar.Batch(chunks if chunks else None, decs)
    return unpack(sar.plan_inspect(dims, b, PS, pages, sms, max_tokens, max_decodes, chunk_split=chunk_split))


DIMS = [synth.MISTRAL_LAYER, dataclasses.replace(synth.MISTRAL_LAYER, sliding_window=1000),
        dataclasses.replace(synth.MISTRAL_LAYER, sliding_window=100), synth.TINY]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("dims", DIMS, ids=["full", "w1000", "w100", "tiny"])
def test_plan_invariants_on_random_batches(seed, dims):
    rng = np.random.default_rng(seed)
    chunks, decs = random_batch(rng, int(rng.integers(0, 4)), int(rng.integers(0 if seed else 1, 70)))
    if not chunks and not decs:
        decs = [(1, 5, [0])]
    p = plan(dims, chunks, decs)
    W = dims.sliding_window
    # rows: chunks in order, then decodes; positions and page slots
    row = 0
    for req, start, ln, bt in chunks:
        for i in range(ln):
            pos = start + i
            assert p["pos"][row] == pos and p["slot"][row] == bt[pos // PS] * PS + pos % PS
            row += 1
    for req, ctx, bt in decs:
        assert p["pos"][row] == ctx and p["slot"][row] == bt[ctx // PS] * PS + ctx % PS
        row += 1
    assert row == p["M"] == p["Lp"] + p["Bd"]
    # logits rows: each chunk's last row, then every decode row
    ends = np.cumsum([c[2] for c in chunks]).tolist()
    assert p["rows"] == [e - 1 for e in ends] + [p["Lp"] + i for i in range(len(decs))]
    # chunk tiles: each chunk's rows exactly once, consecutive positions, its own block table
    covered = {}
    r0 = 0
    chunk_of_row = {}
    for ci, (req, start, ln, bt) in enumerate(chunks):
        for i in range(ln):
            chunk_of_row[r0 + i] = (ci, start + i)
        r0 += ln
    if p["chunk_pairs"]:  # no key-range splits planned, and enough tiles for pairs
        check_pair_table(p, chunks)
        return
    keys = []
    shares = {}
    for t in p["tiles"]:
        row0, pos0, rows, off, blen, kb0, kb1, part = t
        assert 0 < rows <= p["tile_rows"]
        ci, pfirst = chunk_of_row[row0]
        req, start, ln, bt = chunks[ci]
        assert pos0 == pfirst
        nb = (start + ln - 1) // PS + 1
        assert blen == nb and p["pbt"][off:off + nb] == bt[:nb]
        first = max(0, pos0 - W + 1) if W else 0
        assert kb0 < kb1
        if part < 0:  # the tile's whole key range, 128-key blocks
            assert (kb0, kb1) == (first // 128, -(-(pos0 + rows) // 128))
            for i in range(rows):
                assert chunk_of_row[row0 + i] == (ci, pos0 + i)
                assert row0 + i not in covered
                covered[row0 + i] = True
            keys.append(pos0 + rows - first)
        else:
            shares[part] = t
            keys.append((kb1 - kb0) * 128)
    assert keys == sorted(keys, reverse=True)  # the most keys first
    # split tiles: each merge's shares partition the tile's key blocks
    seen = set()
    for row0, rows, p0, cnt in p["comb"]:
        assert cnt >= 2
        grp = [shares[q] for q in range(p0, p0 + cnt)]
        seen |= set(range(p0, p0 + cnt))
        assert all(g[0] == row0 and g[2] == rows for g in grp)
        pos0 = grp[0][1]
        first = max(0, pos0 - W + 1) if W else 0
        lo, hi = first // 128, -(-(pos0 + rows) // 128)
        rng_ = sorted((g[5], g[6]) for g in grp)
        assert rng_[0][0] == lo and rng_[-1][1] == hi
        assert all(a[1] == b[0] for a, b in zip(rng_, rng_[1:])) and all(b - a >= 2 for a, b in rng_)
        ci, _ = chunk_of_row[row0]
        for i in range(rows):
            assert chunk_of_row[row0 + i] == (ci, pos0 + i)
            assert row0 + i not in covered
            covered[row0 + i] = True
    assert seen == set(shares) == set(range(p["n_cparts"]))
    assert sorted(covered) == list(range(p["Lp"]))
    # decode work: each decode's visible keys [first, nk) covered once by 16-aligned ranges
    by_dec = {}
    for d, k0, k1, part in p["items"]:
        by_dec.setdefault(d, []).append((k0, k1, part))
    lengths = [k1 - k0 for _, k0, k1, _ in p["items"]]
    assert lengths == sorted(lengths, reverse=True)  # longest first
    seen_parts = set()
    for i, (req, ctx, bt) in enumerate(decs):
        nk = ctx + 1
        assert p["nkeys"][i] == nk
        nb = ctx // PS + 1
        assert p["btlen"][i] == nb and p["bt"][p["btoff"][i]:p["btoff"][i] + nb] == bt[:nb]
        first = max(0, nk - W) // 16 * 16 if W else 0
        rs = sorted(by_dec[i])
        assert len(rs) == p["pcnt"][i]
        assert rs[0][0] == first and all(k0 % 16 == 0 for k0, _, _ in rs)
        at = first
        for k0, k1, part in rs:
            assert k1 >= k0
            if k1 > k0:
                assert k0 == at
                at = k1
        assert at == nk
        if len(rs) == 1:
            assert rs[0][2] == -1 and p["pbeg"][i] == -1
        else:
            parts = sorted(part for _, _, part in rs)
            assert parts == list(range(p["pbeg"][i], p["pbeg"][i] + len(rs)))
            seen_parts |= set(parts)
    assert seen_parts == set(range(p["n_parts"]))


def test_key_ranges_split_only_when_tiles_leave_sms_idle():
    # the tau = 512 step: 4 tiles x 32 heads = 128 CTAs -- splitting would not shorten it
    p = plan(synth.MISTRAL_LAYER, [(0, 1536, 448, list(range(125)))], [])
    assert p["n_comb"] == 0 and p["n_tiles"] == 4
    # a 256-row chunk deep into a long prompt: 2 tiles x 32 heads = 64 CTAs -> two shares each
    p = plan(synth.MISTRAL_LAYER, [(0, 8192, 256, list(range(528)))], [])
    assert p["n_comb"] == 2 and p["n_tiles"] == 4 and p["n_cparts"] == 4
    # a 128-row chunk: 1 tile x 32 heads = 32 CTAs -> four shares
    p = plan(synth.MISTRAL_LAYER, [(0, 8192, 128, list(range(520)))], [])
    assert p["n_comb"] == 1 and p["n_tiles"] == 4 and p["n_cparts"] == 4
    # the Yi-34B shape (56 heads): 2 tiles -> 112 CTAs, more than half the SMs: not split
    yi = dataclasses.replace(synth.YI_34B, n_layers=1)
    p = plan(yi, [(0, 8192, 256, list(range(528)))], [])
    assert p["n_comb"] == 0 and p["n_tiles"] == 2
    # a tile with fewer than four key blocks is not split
    p = plan(synth.MISTRAL_LAYER, [(0, 0, 200, list(range(13)))], [])
    assert p["n_comb"] == 0
    # and nothing is split unless the model asks for it
    p = plan(synth.MISTRAL_LAYER, [(0, 8192, 256, list(range(528)))], [], chunk_split=False)
    assert p["n_comb"] == 0 and p["n_tiles"] == 2


def test_tile_rows_follow_the_chunk_kernel():
    p = plan(synth.MISTRAL_LAYER, [(0, 0, 300, list(range(19)))], [])
    assert p["tile_rows"] == 128 and p["n_tiles"] == 3
    p = plan(synth.TINY, [(0, 0, 300, list(range(19)))], [])
    assert p["tile_rows"] == 64 and p["n_tiles"] == 5


def test_plan_shape_is_stable_while_contexts_grow_within_their_pages():
    """What sar_graph_update needs: the next decode step of the same requests,
    one token further within the same page counts, has the same plan shape."""
    rng = np.random.default_rng(3)
    ctxs = [int(c) for c in rng.integers(100, 4000, 64)]
    ctxs = [c - (c % 16) for c in ctxs]  # room for one more token in the last page
    bts = [list(range(1000 * i, 1000 * i + c // PS + 1)) for i, c in enumerate(ctxs)]
    a = plan(synth.MISTRAL_LAYER, [], [(i, c, bts[i]) for i, c in enumerate(ctxs)], pages=70000)
    b = plan(synth.MISTRAL_LAYER, [], [(i, c + 1, bts[i]) for i, c in enumerate(ctxs)], pages=70000)
    keys = [k for k in a if k.startswith("o_") or k in ("M", "Lp", "Bd", "R", "n_items", "n_parts", "n_tiles",
                                                         "total")]
    assert all(a[k] == b[k] for k in keys)
    assert a["items"] != b["items"]  # the ranges themselves follow the contexts


def test_plan_rejects_bad_batches():
    d = synth.MISTRAL_LAYER
    with pytest.raises(sar.SarError):  # block table too short for the chunk
        plan(d, [(0, 0, 40, [1, 2])], [])
    with pytest.raises(sar.SarError) as e:  # page id out of range
        plan(d, [], [(0, 20, [5, 99999])])
    assert e.value.code == 5
    with pytest.raises(sar.SarError):  # more rows than max_tokens
        plan(d, [(0, 0, 600, list(range(40))), (1, 0, 600, list(range(40, 80)))], [])
    with pytest.raises(sar.SarError):  # more decodes than max_decodes
        plan(d, [], [(i, 3, [i]) for i in range(200)], max_decodes=128)
    with pytest.raises(sar.SarError):  # an empty chunk
        plan(d, [(0, 0, 8, [0]), (1, 0, 0, [1])], [])


def test_decode_ranges_are_a_resident_slots_share():
    """The tau = 512 workload's 64 decodes (contexts uniform in [128, 4096]):
    ranges of at most 4096 keys, each about one resident slot's share of the
    launch (two CTAs resident per SM), so that with every decode's ranges
    rounded up the (range x KV head) CTAs come to two to four per SM."""
    rng = np.random.default_rng(0)
    ctxs = [int(c) for c in rng.integers(128, 4097, 64)]
    bts = [list(range(300 * i, 300 * i + c // PS + 1)) for i, c in enumerate(ctxs)]
    for sms in (152, 148, 132):
        p = plan(synth.MISTRAL_LAYER, [], [(i, c, bts[i]) for i, c in enumerate(ctxs)], sms=sms, pages=20000)
        lengths = [k1 - k0 for _, k0, k1, _ in p["items"]]
        assert max(lengths) <= 4096
        ctas = len(p["items"]) * synth.MISTRAL_LAYER.n_kv_heads
        assert 2 * sms <= ctas <= 4 * sms, (sms, ctas)


def check_pair_table(p, chunks):
    """A pair table: entries 2i, 2i + 1 are two consecutive query tiles of one
    chunk (or a chunk's odd last tile and an empty partner over the same key
    blocks); every chunk row once; pairs with the most keys first."""
    tiles = p["tiles"]
    assert len(tiles) % 2 == 0 and p["n_comb"] == 0
    chunk_of_row = {}
    r0 = 0
    for ci, (req, start, ln, bt) in enumerate(chunks):
        for i in range(ln):
            chunk_of_row[r0 + i] = (ci, start + i)
        r0 += ln
    covered = set()
    keys = []
    for i in range(0, len(tiles), 2):
        a, b = tiles[i], tiles[i + 1]
        ra0, pa0, rows_a, off_a, blen_a, kb0_a, kb1_a, part_a = a
        rb0, pb0, rows_b, off_b, blen_b, kb0_b, kb1_b, part_b = b
        assert part_a == part_b == -1 and kb0_a == kb0_b == 0
        ci, pfirst = chunk_of_row[ra0]
        req, start, ln, bt = chunks[ci]
        nb = (start + ln - 1) // PS + 1
        assert pa0 == pfirst and blen_a == nb and p["pbt"][off_a:off_a + nb] == bt[:nb]
        assert 0 < rows_a <= 128 and kb1_a == -(-(pa0 + rows_a) // 128)
        if rows_b == 0:  # an odd last tile's empty partner: the first tile's key blocks
            assert b == (ra0, pa0, 0, off_a, blen_a, kb0_a, kb1_a, -1)
            assert pa0 + rows_a == start + ln
        else:  # the chunk's next tile
            assert rows_a == 128 and (rb0, pb0) == (ra0 + 128, pa0 + 128)
            assert (off_b, blen_b) == (off_a, blen_a) and kb1_b == -(-(pb0 + rows_b) // 128)
        for t in (a, b):
            for r in range(t[0], t[0] + t[2]):
                assert r not in covered and chunk_of_row[r] == (ci, t[1] + r - t[0])
                covered.add(r)
        keys.append(max(pa0 + rows_a, pb0 + rows_b))
    assert covered == set(chunk_of_row)
    assert keys == sorted(keys, reverse=True)


def test_chunk_tiles_run_in_pairs_where_that_saves_a_wave():
    yi = dataclasses.replace(synth.YI_34B, n_layers=1)
    # a 512-row chunk of a long Yi-34B prompt: 4 tiles x 56 heads = 224 CTAs
    # (two waves on 152 SMs) -> 2 pairs x 56 = 112 CTAs (one)
    chunks = [(0, 8192, 512, list(range(544)))]
    p = plan(yi, chunks, [], chunk_split=False)
    assert p["chunk_pairs"] == 1 and p["n_tiles"] == 4
    check_pair_table(p, chunks)
    # three tiles: the last one pairs with an empty tile
    chunks = [(0, 4096, 384, list(range(280)))]
    p = plan(yi, chunks, [(9, 100, [600, 601, 602, 603, 604, 605, 606])], chunk_split=False)
    assert p["chunk_pairs"] == 1 and p["n_tiles"] == 4
    check_pair_table(p, chunks)
    # two chunks of two tiles each: pairs never mix prompts
    chunks = [(0, 2048, 256, list(range(144))), (1, 6000, 256, list(range(200, 592)))]
    p = plan(yi, chunks, [], chunk_split=False)
    assert p["chunk_pairs"] == 1 and p["n_tiles"] == 4
    check_pair_table(p, chunks)
    # one-tile CTAs that fit one wave stay one per CTA: the tau = 512 Mistral
    # step (4 x 32 = 128 CTAs), a 256-row Yi chunk (2 x 56 = 112)
    p = plan(synth.MISTRAL_LAYER, [(0, 1536, 448, list(range(125)))], [], chunk_split=False)
    assert p["chunk_pairs"] == 0
    p = plan(yi, [(0, 8192, 256, list(range(528)))], [], chunk_split=False)
    assert p["chunk_pairs"] == 0
    # three waves of one-tile CTAs against two of pairs: not worth the pairs'
    # longer blocks (8 tiles x 56 = 448 CTAs, 224 pairs)
    p = plan(yi, [(0, 8192, 1024, list(range(576)))], [], chunk_split=False, max_tokens=1024)
    assert p["chunk_pairs"] == 0
    # a whole 2048-token prompt at once (16 tiles x 56): pairs
    chunks = [(0, 0, 2048, list(range(128)))]
    p = plan(yi, chunks, [], chunk_split=False, max_tokens=2048)
    assert p["chunk_pairs"] == 1 and p["n_tiles"] == 16
    check_pair_table(p, chunks)
    # no pairs with a sliding window or with key-range splits planned
    w = dataclasses.replace(yi, sliding_window=4096)
    assert plan(w, [(0, 8192, 512, list(range(544)))], [], chunk_split=False)["chunk_pairs"] == 0
    p = plan(synth.MISTRAL_LAYER, [(0, 8192, 256, list(range(528)))], [], chunk_split=True)
    assert p["chunk_pairs"] == 0 and p["n_comb"] == 2


@pytest.mark.parametrize("seed", range(8))
def test_pair_tables_on_random_batches(seed):
    rng = np.random.default_rng(100 + seed)
    yi = dataclasses.replace(synth.YI_34B, n_layers=1)
    # few SMs, so that small random batches take pairs too
    chunks, decs = random_batch(rng, int(rng.integers(1, 4)), int(rng.integers(0, 20)))
    for sms in (8, 40, 152):
        p = plan(yi, chunks, decs, chunk_split=False, sms=sms)
        if p["chunk_pairs"]:
            check_pair_table(p, chunks)
        else:
            assert all(t[2] > 0 for t in p["tiles"])


@pytest.mark.parametrize("ps", [16, 48, 64])
def test_row_slots_for_other_page_sizes(ps):
    """Positions map to (page, offset) slots for any page size the kernels
    take (multiples of 16; powers of two take the shift-and-mask path, others
    the division), for chunk rows that cross pages and for decode rows."""
    rng = np.random.default_rng(ps)
    pages = 4000
    perm = rng.permutation(pages).tolist()
    start, ln = 3 * ps - 5, 2 * ps + 9  # starts inside a page, ends inside another
    cbt = perm[:(start + ln - 1) // ps + 1]
    decs = []
    o = len(cbt)
    for i, ctx in enumerate([0, ps - 1, ps, 5 * ps + 3]):
        n = ctx // ps + 1
        decs.append((10 + i, ctx, perm[o:o + n]))
        o += n
    b = sar.Batch((0, start, ln, cbt), decs)
    r = unpack(sar.plan_inspect(synth.MISTRAL_LAYER, b, ps, pages, 152, 512, 8))
    for i in range(ln):
        pos = start + i
        assert r["pos"][i] == pos and r["slot"][i] == cbt[pos // ps] * ps + pos % ps
    for k, (req, ctx, bt) in enumerate(decs):
        assert r["pos"][ln + k] == ctx and r["slot"][ln + k] == bt[ctx // ps] * ps + ctx % ps
