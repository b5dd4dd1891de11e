"""C ABI checks that need no GPU: the library loads, exports every entry point
include/kda.h declares, and rejects bad arguments on the host before any CUDA
call."""
import ctypes
import os
import re

import pytest

import kda_delta_rule_token_gb300 as kda
from kda_delta_rule_token_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(kda_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kda.load()


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("kda_create", "kda_decode_step", "kda_prefill", "kda_prefill_varlen", "kda_destroy",
              "kda_strerror", "kda_prefill_workspace_bytes", "kda_sync_status", "kda_bind_lowrank",
              "kda_lowrank", "kda_decode_step_lowrank", "kda_decode_step_bf16state"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(build.LIB)
    for n in declared_functions():
        assert hasattr(raw, n), f"{n} declared in include/ but not exported"


def test_strerror_names_every_status(lib):
    for s in range(6):
        assert kda.kda_strerror(s).startswith("KDA_")
    assert "unknown" in kda.kda_strerror(99)


def test_host_side_rejections(lib):
    null = None
    # kda_create: NULL out / config / params
    assert lib.kda_create(null, null, null, null, null, null) == kda.KDA_ERR_INVALID_ARG
    out = ctypes.c_void_p()
    assert lib.kda_create(null, 16, 16, 16, 16, ctypes.byref(out)) == kda.KDA_ERR_INVALID_ARG
    cfg = kda._Config(0, 128, 64, 1e-6, 1e-6)
    assert lib.kda_create(ctypes.byref(cfg), 16, 16, 16, 16, ctypes.byref(out)) == \
        kda.KDA_ERR_INVALID_ARG
    cfg = kda._Config(4, 64, 64, 1e-6, 1e-6)
    assert lib.kda_create(ctypes.byref(cfg), 16, 16, 16, 16, ctypes.byref(out)) == \
        kda.KDA_ERR_UNSUPPORTED
    cfg = kda._Config(4, 128, 32, 1e-6, 1e-6)
    assert lib.kda_create(ctypes.byref(cfg), 16, 16, 16, 16, ctypes.byref(out)) == \
        kda.KDA_ERR_UNSUPPORTED
    cfg = kda._Config(4, 128, 64, -1.0, 1e-6)
    assert lib.kda_create(ctypes.byref(cfg), 16, 16, 16, 16, ctypes.byref(out)) == \
        kda.KDA_ERR_INVALID_ARG
    cfg = kda._Config(4, 128, 64, 1e-6, 1e-6)
    assert lib.kda_create(ctypes.byref(cfg), 18, 16, 16, 16, ctypes.byref(out)) == \
        kda.KDA_ERR_ALIGNMENT
    assert out.value is None
    # calls without a context
    assert lib.kda_decode_step(null, 1, *([16] * 10), null) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_step_bf16state(null, 1, *([16] * 10), null) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill(null, 1, 1, *([16] * 10), 0, null) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_varlen(null, 1, 16, 1, *([16] * 9), null) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_sync_status(null, null) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_workspace_bytes(null, 1, 1) == 0
    assert lib.kda_bind_lowrank(null, 64, 32, 16, 16, 16) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_lowrank(null, 1, 16, 16, 16, 16, 1 << 20, null) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_step_lowrank(null, 1, *([16] * 10), 1 << 20, null) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_lowrank_workspace_bytes(null, 8) == 0
    assert lib.kda_decode_lowrank_workspace_bytes(null, 8) == 0
    lib.kda_destroy(null)  # ignored

