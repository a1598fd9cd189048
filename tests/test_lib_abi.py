"""The C-ABI library loads without a GPU and exports every entry point its headers declare."""

import ctypes
import os
import re

import pytest

import chunked_prefill_hybrid_sar_gb300 as sar
from chunked_prefill_hybrid_sar_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(sar_\w+)\s*\(", text, flags=re.M))
    return names


def test_headers_declare_the_boundary():
    names = declared_functions()
    for n in ("sar_model_create", "sar_kv_create", "sar_step", "sar_sched_next", "sar_sched_commit"):
        assert n in names


def test_library_exports_every_declared_function():
    lib = sar.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_function():
    assert declared_functions() == set(_lib.SIGNATURES)


def test_invalid_arguments_are_rejected_with_a_message():
    lib = sar.lib()
    h = ctypes.c_void_p()
    cfg = _lib.sar_sched_cfg(100, 128, 16, 10, 4)  # budget below one tile
    rc = lib.sar_sched_create(ctypes.byref(cfg), ctypes.byref(h))
    assert rc == _lib.SAR_ERR_INVALID_ARG
    assert b"tile" in lib.sar_last_error()
    assert lib.sar_model_create(None, ctypes.byref(h)) == _lib.SAR_ERR_INVALID_ARG
    assert lib.sar_step(None, None, None, None, None, None, None, None) == _lib.SAR_ERR_INVALID_ARG
    # argument checks come before any device work
    assert lib.sar_op_wait_check(0, 1, None) == _lib.SAR_ERR_INVALID_ARG
    assert lib.sar_op_wait_check(1000, 3, None) == _lib.SAR_ERR_INVALID_ARG


def test_launch_counter_starts_without_gpu_work():
    assert sar.launch_count() >= 0
