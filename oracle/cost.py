"""Oracle cost model helpers (test infrastructure only).

* ``roofline_time`` -- ``T = max(T_math, T_mem)`` per operator (*Sarathi-Serve
  digest* §4, roofline equation), summed over a sequence of operators.
* ``n_row_tiles`` -- thread blocks a GEMM needs along its row dimension
  (*SARATHI reading notes* part 3 §3: 257 rows need 3 blocks of 128).
* ``max_batch`` -- ``B = floor((MG - MS) / (L * mkv))`` (*SARATHI technique
  write-up* §4.1), optionally after holding back a reserve fraction of MG.
* ``prior_chunk_loads`` -- chunk k of N is re-read by the N-k later chunks, in
  total ``N(N-1)/2`` chunk loads (*Sarathi-Serve digest* §4, check 4).
* ``layer_flops`` / ``layer_weight_bytes`` -- algorithmic work of the linear
  layers of one decoder layer (2 flops per multiply-add).

Parity pins: the printed toy batches (123 ms vs 96 ms), 257 -> 3 tiles, the
closed-form sum, and brute-force enumeration (``tests/test_oracle_cost.py``).
"""

from __future__ import annotations

import math


def roofline_time(ops) -> float:
    """Sum over ``ops`` of ``max(t_math, t_mem)``; ``ops`` yields pairs."""
    return sum(max(tm, tb) for tm, tb in ops)


def op_time(flops: float, bytes_: float, peak_flops: float, peak_bw: float) -> float:
    return max(flops / peak_flops, bytes_ / peak_bw)


def n_row_tiles(rows: int, tile: int) -> int:
    return -(-rows // tile)


def max_batch(mg: float, ms: float, max_len: int, mkv: float, reserve: float = 0.0) -> int:
    """Largest batch whose worst-case KV fits in ``mg*(1-reserve) - ms``."""
    return int(math.floor((mg * (1.0 - reserve) - ms) / (max_len * mkv)))


def prior_chunk_loads(n_chunks: int) -> int:
    """Closed form of the extra KV loads when a prompt is cut into N chunks."""
    return n_chunks * (n_chunks - 1) // 2


def layer_flops(dims, rows: int) -> float:
    """Linear-layer flops of one decoder layer over ``rows`` tokens."""
    h, qd, kvd, f = dims.hidden, dims.q_dim, dims.kv_dim, dims.ffn
    macs = h * (qd + 2 * kvd) + qd * h + 2 * h * f + f * h
    return 2.0 * rows * macs


def layer_weight_bytes(dims, elem_bytes: int = 2) -> float:
    h, qd, kvd, f = dims.hidden, dims.q_dim, dims.kv_dim, dims.ffn
    return float(elem_bytes * (h * (qd + 2 * kvd) + qd * h + 3 * h * f))


def kv_bytes_per_token(dims, elem_bytes: int = 2) -> int:
    """K and V of one token for one layer."""
    return 2 * dims.kv_dim * elem_bytes
