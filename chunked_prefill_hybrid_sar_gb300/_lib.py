"""ctypes binding of ``libsar.so`` (include/sar.h, include/sar_ops.h).

Argument marshalling only: every step of the hybrid batch runs in the
library's CUDA kernels.  Loading fails loudly when the library has not been
built -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsar.so")

# status codes
SAR_OK = 0
SAR_ERR_INVALID_ARG = 1
SAR_ERR_NO_PAGES = 2
SAR_ERR_OOM = 3
SAR_ERR_CUDA = 4
SAR_ERR_BOUNDS = 5
SAR_ERR_TIMEOUT = 6
SAR_ERR_UNSUPPORTED = 7

SAR_IN_HIDDEN = 0
SAR_IN_TOKENS = 1

SAR_STORAGE_F16, SAR_STORAGE_BF16 = 0, 1
SAR_EPI_STORE, SAR_EPI_RESIDUAL, SAR_EPI_SWIGLU, SAR_EPI_F32 = 0, 1, 2, 3
SAR_GEMM_AUTO, SAR_GEMM_M128_N128, SAR_GEMM_M128_N256, SAR_GEMM_SWAP, SAR_GEMM_M256_N128 = 0, 1, 2, 3, 4
SAR_GEMM_PAIR_N256, SAR_GEMM_PAIR_N128, SAR_GEMM_PAIR_N192 = 5, 6, 7
SAR_GEMM_TWO_CTAS = 0x1000
SAR_Q_F32 = 0x100
SAR_GEMM_STREAM_K = 0x2000

KERNEL_KINDS = ("embed", "rmsnorm", "gemm_qkv", "rope_append", "chunk_attn", "decode_attn", "gemm_o",
                "gemm_gateup", "gemm_down", "head_norm", "gemm_head", "decode_combine")

i32 = ctypes.c_int32
i64 = ctypes.c_int64
vp = ctypes.c_void_p
P_i32 = ctypes.POINTER(ctypes.c_int32)


class sar_dims(ctypes.Structure):
    _fields_ = [("n_layers", i32), ("hidden", i32), ("n_q_heads", i32), ("n_kv_heads", i32),
                ("head_dim", i32), ("ffn", i32), ("vocab", i32), ("rms_eps", ctypes.c_float),
                ("rope_base", ctypes.c_float), ("max_tokens", i32), ("max_decodes", i32),
                ("storage", i32), ("sliding_window", i32)]


class sar_layer_weights(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "norm1", "norm2")]


class sar_prefill(ctypes.Structure):
    _fields_ = [("req", i32), ("start_pos", i32), ("len", i32), ("block_table", P_i32),
                ("n_blocks", i32)]


class sar_decode(ctypes.Structure):
    _fields_ = [("req", i32), ("ctx_len", i32), ("block_table", P_i32), ("n_blocks", i32)]


class sar_batch(ctypes.Structure):
    _fields_ = [("has_prefill", i32), ("prefill", sar_prefill), ("n_decode", i32),
                ("decode", ctypes.POINTER(sar_decode)), ("in_kind", i32), ("n_more_prefill", i32),
                ("more_prefill", ctypes.POINTER(sar_prefill))]


class sar_sched_cfg(ctypes.Structure):
    _fields_ = [("tau", i32), ("tile", i32), ("page_size", i32), ("num_pages", i32),
                ("max_batch", i32), ("max_chunks", i32)]


# name -> (restype, argtypes)
SIGNATURES = {
    "sar_last_error": (ctypes.c_char_p, []),
    "sar_launch_count": (i64, []),
    "sar_model_create": (i32, [ctypes.POINTER(sar_dims), ctypes.POINTER(vp)]),
    "sar_model_set_layer": (i32, [vp, i32, ctypes.POINTER(sar_layer_weights), vp]),
    "sar_model_set_head": (i32, [vp, vp, vp, vp, vp]),
    "sar_model_destroy": (i32, [vp]),
    "sar_sync_status": (i32, [vp]),
    "sar_kv_create": (i32, [vp, i32, i32, ctypes.POINTER(vp)]),
    "sar_kv_layer_ptr": (i32, [vp, i32, i32, ctypes.POINTER(vp)]),
    "sar_kv_destroy": (i32, [vp]),
    "sar_step": (i32, [vp, vp, ctypes.POINTER(sar_batch), vp, vp, vp, vp, vp]),
    "sar_step_host": (i32, [vp, vp, ctypes.POINTER(sar_batch), vp, vp, vp, vp, vp]),
    "sar_sample_greedy": (i32, [vp, vp, i32, vp, vp]),
    "sar_profile_enable": (i32, [vp, i32]),
    "sar_model_set_overlap": (i32, [vp, i32]),
    "sar_model_set_chunk_split": (i32, [vp, i32]),
    "sar_graph_launch_host_tokens": (i32, [vp, vp, P_i32, vp]),
    "sar_graph_enqueue_host_tokens": (i32, [vp, vp, P_i32, vp]),
    "sar_graph_wait": (i32, [vp]),
    "sar_graph_create": (i32, [vp, vp, ctypes.POINTER(sar_batch), vp, vp, vp, vp, vp, ctypes.POINTER(vp)]),
    "sar_graph_update": (i32, [vp, ctypes.POINTER(sar_batch), vp]),
    "sar_graph_launch": (i32, [vp, vp]),
    "sar_graph_launch_host": (i32, [vp, vp, vp, vp, vp]),
    "sar_graph_destroy": (i32, [vp]),
    "sar_profile_read": (i32, [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64), i32]),
    "sar_sched_create": (i32, [ctypes.POINTER(sar_sched_cfg), ctypes.POINTER(vp)]),
    "sar_sched_add": (i32, [vp, i32, ctypes.c_double, i32, i32, P_i32]),
    "sar_sched_next": (i32, [vp, ctypes.c_double, ctypes.POINTER(sar_batch), ctypes.POINTER(P_i32)]),
    "sar_sched_commit": (i32, [vp, P_i32, i32, P_i32]),
    "sar_sched_stats": (i32, [vp, P_i32, P_i32, P_i32, P_i32]),
    "sar_sched_destroy": (i32, [vp]),
    "sar_op_gemm": (i32, [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]),
    "sar_op_rmsnorm": (i32, [vp, vp, vp, i32, i32, ctypes.c_float, i32, vp]),
    "sar_op_sync_status": (i32, []),
    "sar_op_wait_check": (i32, [i64, i32, vp]),
    "sar_plan_inspect": (i32, [ctypes.POINTER(sar_dims), i32, i32, i32, i32, ctypes.POINTER(sar_batch), P_i32,
                               P_i32, i64, ctypes.POINTER(i64)]),
    "sar_model_debug_buffer": (i32, [vp, i32, ctypes.POINTER(vp)]),
    "sar_decode_attention_noalloc": (i32, [vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, vp, i32,
                                           vp, i32, vp, i32, i32, vp, vp]),
}

_lib = None


class SarError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"sar error {code}: {msg}")
        self.code = code


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def check(rc: int) -> None:
    if rc != SAR_OK:
        raise SarError(rc, lib().sar_last_error().decode())


def i32_array(values):
    vals = list(values)
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)
