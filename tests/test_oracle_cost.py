"""Pins of the oracle's cost helpers against the pages' printed numbers and brute force."""

import json
import os

import pytest

import synth
from oracle import cost

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_toy_batches_roofline_totals_match_printed_values():
    g = load("toy_batches.json")
    for scheme in ("scheme_a", "scheme_b"):
        ops = []
        for b in g[scheme]["batches"]:
            ops += [(b["t_math"], b["t_mem"])] * b["count"]
        assert cost.roofline_time(ops) == g[scheme]["total"]


def test_toy_batches_carry_every_prefill_and_decode():
    g = load("toy_batches.json")
    # scheme B: six 256-token chunks with 15 decodes each cover 1536 prefill and 90 decodes
    assert 6 * 256 == g["prefill_tokens"]
    assert 6 * g["decodes_per_batch"] == g["decodes"]


def test_tile_count_matches_printed_example():
    g = load("tile_quantisation.json")
    for c in g["cases"]:
        n = cost.n_row_tiles(c["rows"], g["tile"])
        assert n == c["tiles"]
        assert c["rows"] - (n - 1) * g["tile"] == c["valid_rows_in_last_tile"]


@pytest.mark.parametrize("mg,ms,L,mkv,res", [(80e9, 14.5e9, 4096, 131072, 0.0),
                                              (80e9, 14.5e9, 4096, 131072, 0.2),
                                              (288e9, 69e9, 16384, 60 * 4096, 0.2),
                                              (1000, 100, 7, 3, 0.0)])
def test_max_batch_is_the_largest_fitting_batch(mg, ms, L, mkv, res):
    b = cost.max_batch(mg, ms, L, mkv, res)
    budget = mg * (1 - res) - ms
    assert b * L * mkv <= budget < (b + 1) * L * mkv


def test_prior_chunk_loads_closed_form_matches_enumeration():
    for n in range(1, 70):
        brute = sum(n - k for k in range(1, n + 1))  # chunk k re-read by N-k later chunks
        assert cost.prior_chunk_loads(n) == brute


def test_mistral_layer_parameter_count():
    # 4096*(4096+2*1024) + 4096*4096 + 3*4096*14336 = 218.1 M parameters per layer
    d = synth.MISTRAL_LAYER
    params = cost.layer_weight_bytes(d) / 2
    assert params == 4096 * 6144 + 4096 * 4096 + 3 * 4096 * 14336
    assert cost.layer_flops(d, 1) == 2 * params
    assert cost.kv_bytes_per_token(d) == 4096
