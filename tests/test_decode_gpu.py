"""Decode kernel vs the fp64 oracle (GPU).

Tolerance: max relative error 1e-4, measured per (sequence, head) and
tensor as max|x - r| / max|r|, on o at every call and on S and the conv
window after the last call.
"""
import numpy as np
import pytest
import torch

import kda_delta_rule_token_gb300 as kda
from kda_delta_rule_token_gb300 import synth
from harness import (Guarded, max_rel_err, np64, oracle_pairs, pair_window, set_pair_window)

pytestmark = pytest.mark.gpu
TOL = 1e-4
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_delta_rule_token_gb300 import build
    build.build()
    kda.load()


def gpu_decode(wl, params, tokens, S, conv, *, o_pre=True, stream=None):
    """Run the calls of ``tokens`` (call-major) in place on S / conv.

    o, o_pre, S and the window live inside poisoned guard regions during the
    calls; the guards are checked bit for bit after every call.
    """
    T, B, H, d = tokens["q"].shape
    go = Guarded(torch.zeros((B, H, d), device=DEV))
    gp = Guarded(torch.zeros((B, H, d), device=DEV)) if o_pre else None
    gS, gc = Guarded(S), Guarded(conv)
    o = torch.empty((T, B, H, d), device=DEV)
    op = torch.empty((T, B, H, d), device=DEV) if o_pre else None
    ctx = kda.kda_create(H, params["conv_w"], params["dt_bias"], params["A_log"],
                         params["gamma"])
    try:
        for t in range(T):
            kda.kda_decode_step(ctx, B, tokens["q"][t], tokens["k"][t], tokens["v"][t],
                                tokens["z"][t], tokens["beta_logit"][t],
                                tokens["gate_logit"][t], gc.t, gS.t, go.t,
                                gp.t if o_pre else None, stream=stream)
            o[t].copy_(go.t)
            if o_pre:
                op[t].copy_(gp.t)
            if t == 0 or t == T - 1 or T <= 32:
                torch.cuda.synchronize()
                for g in (go, gp, gS, gc):
                    assert g is None or g.intact(), f"a guard region was written at call {t}"
        assert kda.kda_sync_status(ctx, stream) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    S.copy_(gS.t)
    conv.copy_(gc.t)
    for g in (go, gp, gS, gc):
        assert g is None or g.intact()
    return o, op


def check_pairs(ref, o, op, S, conv, pairs, tol=TOL):
    worst = 0.0
    for (b, h) in pairs:
        r = ref[(b, h)]
        o_g = np64(o[:, b, h])
        for t in range(o_g.shape[0]):
            e = max_rel_err(o_g[t], r.o[0, t, 0])
            worst = max(worst, e)
            assert e <= tol, f"o at call {t}, pair {(b, h)}: {e:.3e}"
            if op is not None:
                e = max_rel_err(np64(op[t, b, h]), r.o_pre[0, t, 0])
                assert e <= tol, f"o_pre at call {t}, pair {(b, h)}: {e:.3e}"
        e = max_rel_err(np64(S[b, h]), r.S[0, 0])
        worst = max(worst, e)
        assert e <= tol, f"S of pair {(b, h)}: {e:.3e}"
        e = max_rel_err(pair_window(conv, b, h), r.conv_state)
        assert e == 0.0, f"conv window of pair {(b, h)} differs: {e:.3e}"
    return worst


def _all_pairs(wl):
    return [(b, h) for b in range(wl.B) for h in range(wl.H)]


def _setup(wl, T=None):
    params = synth.make_params(wl, DEV)
    tokens = synth.make_tokens(wl, DEV, T=T)
    st = synth.make_state(wl, DEV)
    return params, tokens, st["S"], st["conv_state"]


def test_tiny_decode_every_output():
    wl = synth.TINY
    params, tokens, S, conv = _setup(wl)
    S0, c0 = S.clone(), conv.clone()
    o, op = gpu_decode(wl, params, tokens, S, conv)
    ref = oracle_pairs(params, tokens, S0, c0, _all_pairs(wl), call_major=True)
    check_pairs(ref, o, op, S, conv, _all_pairs(wl))


def test_ragged_batch_and_heads():
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=3, H=5, T=9)
    params, tokens, S, conv = _setup(wl)
    S0, c0 = S.clone(), conv.clone()
    o, op = gpu_decode(wl, params, tokens, S, conv)
    ref = oracle_pairs(params, tokens, S0, c0, _all_pairs(wl), call_major=True)
    check_pairs(ref, o, op, S, conv, _all_pairs(wl))


def test_decode_b64_h32_256_calls_sampled():
    """Full batched-decode workload: 64 x 32 heads, 256 calls, fp32 state."""
    wl = synth.WORKLOADS["decode_b64_h32_x256"]
    params, tokens, S, conv = _setup(wl)
    S0, c0 = S.clone(), conv.clone()
    pairs = synth.sample_heads(wl, 12)
    o, _ = gpu_decode(wl, params, tokens, S, conv, o_pre=False)
    ref = oracle_pairs(params, tokens, S0, c0, pairs, call_major=True)
    check_pairs(ref, o, None, S, conv, pairs)


def test_decode_b256_h64_128_calls_sampled():
    """Serving-scale decode (1 GiB state): initial state from 32 warm-up tokens.

    The warm-up of the sampled pairs is the oracle's (rounded to fp32) and is
    written into the device state before the timed-shape run; the other pairs
    keep the GPU's own warm-up (they do not interact with the sampled ones).
    """
    wl = synth.WORKLOADS["decode_b256_h64_x128"]
    params = synth.make_params(wl, DEV)
    st = synth.make_state(wl, DEV)
    S, conv = st["S"], st["conv_state"]
    warm = synth.make_tokens(wl, DEV, T=wl.warmup_tokens, warm=True)
    pairs = synth.sample_heads(wl, 8)
    S_zero, c_zero = S.clone(), conv.clone()
    gpu_decode(wl, params, warm, S, conv, o_pre=False)
    wref = oracle_pairs(params, warm, S_zero, c_zero, pairs, call_major=True)
    del S_zero, c_zero
    for (b, h) in pairs:   # GPU warm-up agrees with the oracle's...
        assert max_rel_err(np64(S[b, h]), wref[(b, h)].S[0, 0]) <= TOL
        # ...and the oracle's own warm-up state is what both sides start from.
        S[b, h] = torch.as_tensor(wref[(b, h)].S[0, 0], dtype=torch.float32, device=DEV)
        set_pair_window(conv, b, h, wref[(b, h)].conv_state)
    tokens = synth.make_tokens(wl, DEV)
    S0, c0 = S.clone(), conv.clone()
    o, _ = gpu_decode(wl, params, tokens, S, conv, o_pre=False)
    ref = oracle_pairs(params, tokens, S0, c0, pairs, call_major=True)
    check_pairs(ref, o, None, S, conv, pairs)


def test_zero_batch_is_noop():
    wl = synth.TINY
    params, tokens, S, conv = _setup(wl, T=1)
    S1, c1 = S.clone(), conv.clone()
    ctx = kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"],
                         params["gamma"])
    try:
        o = torch.full((1, wl.H, 128), 7.0, device=DEV)
        kda.kda_decode_step(ctx, 0, tokens["q"][0], tokens["k"][0], tokens["v"][0],
                            tokens["z"][0], tokens["beta_logit"][0], tokens["gate_logit"][0],
                            conv, S, o)
        torch.cuda.synchronize()
        assert torch.equal(S, S1) and torch.equal(conv, c1) and bool((o == 7.0).all())
    finally:
        kda.kda_destroy(ctx)


def test_no_write_no_decay_keeps_state_exactly():
    """beta = 0 and gk = 0 leave S bit-for-bit unchanged on the GPU too."""
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=2, H=3, T=4)
    params, tokens, S, conv = _setup(wl)
    params["A_log"].fill_(-float("inf"))
    tokens["beta_logit"].fill_(-float("inf"))
    S0 = S.clone()
    gpu_decode(wl, params, tokens, S, conv)
    assert torch.equal(S, S0)


def test_extreme_inputs():
    """Saturated gates, strong decay, a zero input, large values."""
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=2, H=2, T=6)
    params, tokens, S, conv = _setup(wl)
    params["A_log"][0].fill_(0.0)
    tokens["z"][:, 0].fill_(30.0)          # gk = -30: state wiped
    tokens["beta_logit"][:, 1, 0] = 40.0    # beta -> 1
    tokens["beta_logit"][:, 1, 1] = -40.0   # beta -> 0
    tokens["gate_logit"][2] = 60.0
    tokens["gate_logit"][3] = -60.0
    tokens["q"][4, 0].zero_()               # zero q input at one call
    tokens["v"][5].mul_(1e3)
    S0, c0 = S.clone(), conv.clone()
    o, op = gpu_decode(wl, params, tokens, S, conv)
    ref = oracle_pairs(params, tokens, S0, c0, _all_pairs(wl), call_major=True)
    for (b, h) in _all_pairs(wl):
        r = ref[(b, h)]
        np.testing.assert_allclose(np64(o[:, b, h]), r.o[0, :, 0], rtol=0, atol=1e-4 * max(
            1.0, float(np.abs(r.o).max())))
        assert max_rel_err(np64(S[b, h]), r.S[0, 0]) <= TOL


def test_side_stream_matches_default_stream():
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=4, H=4, T=5)
    params, tokens, S, conv = _setup(wl)
    S2, c2 = S.clone(), conv.clone()
    o1, _ = gpu_decode(wl, params, tokens, S, conv)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, _ = gpu_decode(wl, params, tokens, S2, c2, stream=s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S, S2) and torch.equal(conv, c2)


def test_misaligned_pointer_is_rejected_before_launch():
    wl = synth.TINY
    params, tokens, S, conv = _setup(wl, T=1)
    ctx = kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"],
                         params["gamma"])
    try:
        buf = torch.zeros(wl.H * 128 + 1, device=DEV)
        q_bad = buf[1:]                     # 4-byte offset
        o = torch.empty((1, wl.H, 128), device=DEV)
        with pytest.raises(kda.KDAError) as ei:
            kda.kda_decode_step(ctx, 1, q_bad, tokens["k"][0], tokens["v"][0], tokens["z"][0],
                                tokens["beta_logit"][0], tokens["gate_logit"][0], conv, S, o)
        assert ei.value.status == kda.KDA_ERR_ALIGNMENT
    finally:
        kda.kda_destroy(ctx)


def test_graph_replay_equals_launches():
    """Calls captured in a CUDA graph and replayed give exactly what launching them does.

    The entry point does no host synchronisation and no allocation, so a
    sequence of decode calls can be captured once and replayed; the replay
    must run the same kernels on the same buffers (bit-for-bit o, S, window).
    """
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=4, H=3, T=8)
    params, tokens, S, conv = _setup(wl)
    S2, c2 = S.clone(), conv.clone()
    o_l, _ = gpu_decode(wl, params, tokens, S, conv, o_pre=False)

    T, B, H, d = tokens["q"].shape
    o_g = torch.full((T, B, H, d), float("nan"), device=DEV)
    ctx = kda.kda_create(H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=side):
            for t in range(T):
                kda.kda_decode_step(ctx, B, tokens["q"][t], tokens["k"][t], tokens["v"][t],
                                    tokens["z"][t], tokens["beta_logit"][t],
                                    tokens["gate_logit"][t], c2, S2, o_g[t], None,
                                    stream=torch.cuda.current_stream())
        torch.cuda.current_stream().wait_stream(side)
        assert bool(torch.isnan(o_g).all())   # the capture itself ran nothing
        g.replay()
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    assert torch.equal(o_g, o_l)
    assert torch.equal(S2, S)
    assert torch.equal(c2, conv)
