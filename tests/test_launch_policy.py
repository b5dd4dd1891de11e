"""Launch policies of the library, on the host (no GPU): which prefill heads
run as relay pairs, and when the output projection splits K.  Both are
computed by the library itself (test hooks of csrc/kda_testing.h)."""
import ctypes

import pytest

from kda_delta_rule_token_gb300 import build


@pytest.fixture(scope="module")
def lib():
    build.build()
    raw = ctypes.CDLL(build.LIB)
    raw.kda_testing_prefill_relay_heads.argtypes = [ctypes.c_longlong, ctypes.c_int, ctypes.c_int]
    raw.kda_testing_prefill_relay_heads.restype = ctypes.c_longlong
    raw.kda_testing_project_o_ksplit.argtypes = [ctypes.c_int] * 4
    raw.kda_testing_project_o_ksplit.restype = ctypes.c_int
    return raw


@pytest.mark.parametrize("heads,T,sms,want", [
    (32, 4096, 152, 32),      # single sequence, 32 heads: every head as a pair (64 CTAs)
    (76, 128, 152, 76),       # two CTAs per head still fit on the SMs
    (77, 128, 152, 0),        # they do not; one partial wave of 77 > 76: no pairs
    (512, 8192, 152, 56),     # 3 full waves + 56: the tail as pairs
    (456, 8192, 152, 0),      # exactly 3 waves: no tail
    (200, 200, 152, 48),      # 1 wave + 48
    (229, 4096, 152, 0),      # 1 wave + 77: the tail would not fit twice
    (32, 64, 152, 0),         # one chunk: nothing to relay
    (32, 1, 152, 0),
    (32, 65, 152, 32),        # two chunks (the second of one token)
    (4, 4096, 1, 0),          # one SM
    (0, 4096, 152, 0),
])
def test_prefill_relay_heads(lib, heads, T, sms, want):
    assert lib.kda_testing_prefill_relay_heads(heads, T, sms) == want


@pytest.mark.parametrize("hidden,N,HD,sms,want", [
    (7168, 64, 4096, 152, 2),     # decode batch: 56 tiles on 152 SMs
    (7168, 1, 4096, 152, 2),      # one token
    (7168, 64, 8192, 152, 2),
    (1024, 64, 8192, 152, 2),     # 8 tiles
    (7168, 65536, 8192, 152, 1),  # prefill batch: thousands of tiles
    (7168, 300, 4096, 152, 1),    # 2 token tiles x 56 = 112 tiles > 76
    (16384, 64, 4096, 152, 1),    # 128 tiles
    (128, 5, 256, 152, 1),        # K of 4 slices: too short to split
    (128, 5, 1024, 152, 2),       # K of 16 slices
])
def test_project_o_ksplit(lib, hidden, N, HD, sms, want):
    assert lib.kda_testing_project_o_ksplit(hidden, N, HD, sms) == want


def test_policies_reject_negative_arguments(lib):
    assert lib.kda_testing_prefill_relay_heads(-1, 64, 152) == -1
    assert lib.kda_testing_project_o_ksplit(128, 0, 256, 152) == -1
