"""Prefill vs the fp64 oracle (GPU).

Tolerance: relative L2 error 2e-3 over all of o and, separately, over the
final state S (bf16 q/k/v inputs, fp32 everything else), for every
(sequence, head) pair on its own as well as pooled over the checked pairs.
The conv window after the prefill holds raw inputs and must match exactly.
o, S and the window sit inside poisoned guard regions during each call; the
guards are checked bit for bit afterwards.
"""
import numpy as np
import pytest
import torch

import kda_delta_rule_token_gb300 as kda
from kda_delta_rule_token_gb300 import synth
from harness import Guarded, max_rel_err, np64, oracle_pairs, pair_window, rel_l2

pytestmark = pytest.mark.gpu
TOL = 2e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_delta_rule_token_gb300 import build
    build.build()
    kda.load()


def bits(x: torch.Tensor) -> torch.Tensor:
    assert x.dtype == torch.bfloat16
    return x.view(torch.int16)


def gpu_prefill(wl, params, tokens, S, conv, T=None, t0=0, stream=None, schedule="split"):
    """Prefill tokens [t0, t0+T) of ``tokens`` ([B, T, H, d]) in place on S / conv.
    schedule "split": with the workspace kda_prefill_workspace_bytes asks for
    (few-head calls split producers from consumers); "relay": without one
    (those heads run as relay pairs)."""
    B, Tall, H, d = tokens["q"].shape
    T = Tall - t0 if T is None else T
    sl = lambda x: x[:, t0:t0 + T].contiguous()
    q, k, v = (bits(sl(tokens[n])) for n in ("q", "k", "v"))
    z, g = sl(tokens["z"]), sl(tokens["gate_logit"])
    bl = tokens["beta_logit"][:, t0:t0 + T].contiguous()
    go = Guarded(torch.zeros((B, T, H, d), device=DEV))
    gS, gc = Guarded(S), Guarded(conv)
    ctx = kda.kda_create(H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        nws = kda.kda_prefill_workspace_bytes(ctx, B, T)
        if schedule == "relay":
            nws = 0
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=DEV) if nws else None
        kda.kda_prefill(ctx, B, T, q, k, v, z, bl, g, gc.t, gS.t, go.t, ws, nws, stream=stream)
        assert kda.kda_sync_status(ctx, stream) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    assert go.intact() and gS.intact() and gc.intact(), "a guard region was written"
    S.copy_(gS.t)
    conv.copy_(gc.t)
    return go.t.clone()


def check(ref, o, S, conv, pairs, tol=TOL):
    """rel-L2 of o and of S per (sequence, head) pair and pooled; the worst
    pair and the worst element-wise |x - r| / max|r| are printed."""
    per = {}
    for b, h in pairs:
        og, orf = np64(o[b, :, h]), ref[(b, h)].o[0, :, 0]
        sg, srf = np64(S[b, h]), ref[(b, h)].S[0, 0]
        per[(b, h)] = (rel_l2(og, orf), rel_l2(sg, srf), max_rel_err(og, orf), max_rel_err(sg, srf))
        assert max_rel_err(pair_window(conv, b, h), ref[(b, h)].conv_state) == 0.0
    wo = max(per, key=lambda p: per[p][0])
    ws = max(per, key=lambda p: per[p][1])
    print(f"\n  worst pair o {wo}: rel-L2 {per[wo][0]:.3e}, element-wise {max(v[2] for v in per.values()):.3e}; "
          f"worst pair S {ws}: rel-L2 {per[ws][1]:.3e}, element-wise {max(v[3] for v in per.values()):.3e}")
    for p, (eo, es, _, _) in per.items():
        assert eo <= tol, f"o rel-L2 of pair {p}: {eo:.3e}"
        assert es <= tol, f"S rel-L2 of pair {p}: {es:.3e}"
    o_g = np.stack([np64(o[b, :, h]) for b, h in pairs])
    o_r = np.stack([ref[p].o[0, :, 0] for p in pairs])
    S_g = np.stack([np64(S[b, h]) for b, h in pairs])
    S_r = np.stack([ref[p].S[0, 0] for p in pairs])
    eo, es = rel_l2(o_g, o_r), rel_l2(S_g, S_r)
    assert eo <= tol, f"pooled o rel-L2 {eo:.3e}"
    assert es <= tol, f"pooled S rel-L2 {es:.3e}"
    return eo, es


def _setup(wl, T=None):
    return (synth.make_params(wl, DEV), synth.make_tokens(wl, DEV, T=T),
            *synth.make_state(wl, DEV).values())


SMALL = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], B=2, H=3, T=130,
                     s0_std=0.05, win_std=1.0)


@pytest.mark.parametrize("schedule", ["split", "relay"])
@pytest.mark.parametrize("T", [1, 2, 16, 63, 64, 65, 100, 128, 130, 192, 320])
def test_small_prefill_every_output(T, schedule):
    """6 heads: one CTA per head for T <= 64; from two chunks on, producers
    and one consumer per head (split) or two CTAs per head taking alternate
    chunks (relay); nonzero initial state and window.  T = 320 (five chunks)
    wraps the split schedule's ring of four slots per head."""
    wl = synth.shrink(SMALL, T=T)
    params, tokens, S, conv = _setup(wl)
    S0, c0 = S.clone(), conv.clone()
    o = gpu_prefill(wl, params, tokens, S, conv, schedule=schedule)
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    ref = oracle_pairs(params, tokens, S0, c0, pairs, call_major=False)
    check(ref, o, S, conv, pairs)


def test_prefill_equals_decode_calls():
    """Prefill of T tokens = T decode calls on the same (bf16-valued) inputs."""
    wl = synth.shrink(SMALL, T=70)
    params, tokens, S, conv = _setup(wl)
    Sd, cd = S.clone(), conv.clone()
    o_p = gpu_prefill(wl, params, tokens, S, conv)
    ctx = kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"],
                         params["gamma"])
    try:
        od = torch.empty_like(o_p)
        f32 = {n: tokens[n].float().transpose(0, 1).contiguous()
               for n in ("q", "k", "v", "z", "gate_logit")}
        bl = tokens["beta_logit"].transpose(0, 1).contiguous()
        ot = torch.empty((wl.T, wl.B, wl.H, 128), device=DEV)
        for t in range(wl.T):
            kda.kda_decode_step(ctx, wl.B, f32["q"][t], f32["k"][t], f32["v"][t], f32["z"][t],
                                bl[t], f32["gate_logit"][t], cd, Sd, ot[t])
        od.copy_(ot.transpose(0, 1))
        torch.cuda.synchronize()
    finally:
        kda.kda_destroy(ctx)
    assert rel_l2(np64(o_p), np64(od)) <= TOL
    assert rel_l2(np64(S), np64(Sd)) <= TOL
    assert torch.equal(conv, cd)


def test_resume_split_equals_whole():
    """prefill(T1) then prefill(T2) continues exactly like prefill(T1 + T2)."""
    wl = synth.shrink(SMALL, T=150)
    params, tokens, S, conv = _setup(wl)
    S2, c2 = S.clone(), conv.clone()
    o_all = gpu_prefill(wl, params, tokens, S, conv)
    o_a = gpu_prefill(wl, params, tokens, S2, c2, T=77, t0=0)
    o_b = gpu_prefill(wl, params, tokens, S2, c2, T=73, t0=77)
    assert rel_l2(np64(torch.cat([o_a, o_b], 1)), np64(o_all)) <= TOL
    assert rel_l2(np64(S2), np64(S)) <= TOL
    assert torch.equal(c2, conv)


def test_strong_and_extreme_decay():
    """Channels with gk near -30 per token, beta saturated, huge values."""
    wl = synth.shrink(SMALL, T=100)
    params, tokens, S, conv = _setup(wl)
    params["A_log"][0, :32].fill_(0.0)
    tokens["z"][:, :, 0, :32] = 30.0
    tokens["z"][:, 40:60, 1] = 80.0
    tokens["beta_logit"][:, 10:20] = 50.0
    tokens["beta_logit"][:, 20:30] = -50.0
    S0, c0 = S.clone(), conv.clone()
    o = gpu_prefill(wl, params, tokens, S, conv)
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    ref = oracle_pairs(params, tokens, S0, c0, pairs, call_major=False)
    check(ref, o, S, conv, pairs)


def test_zero_sizes_are_noops():
    wl = synth.shrink(SMALL, T=4)
    params, tokens, S, conv = _setup(wl)
    S1, c1 = S.clone(), conv.clone()
    ctx = kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"],
                         params["gamma"])
    try:
        o = torch.empty((wl.B, 4, wl.H, 128), device=DEV)
        for B, T in ((0, 4), (wl.B, 0)):
            kda.kda_prefill(ctx, B, T, bits(tokens["q"]), bits(tokens["k"]), bits(tokens["v"]),
                            tokens["z"], tokens["beta_logit"], tokens["gate_logit"], conv, S, o)
        torch.cuda.synchronize()
        assert torch.equal(S, S1) and torch.equal(conv, c1)
    finally:
        kda.kda_destroy(ctx)


def test_prefill_b1_h32_t4096_sampled():
    """Single-sequence prefill workload at full size."""
    wl = synth.WORKLOADS["prefill_b1_h32_t4096"]
    params, tokens, S, conv = _setup(wl)
    S0, c0 = S.clone(), conv.clone()
    o = gpu_prefill(wl, params, tokens, S, conv)
    pairs = synth.sample_heads(wl, 6)
    ref = oracle_pairs(params, tokens, S0, c0, pairs, call_major=False)
    check(ref, o, S, conv, pairs)


def test_prefill_b8_h64_t8192_sampled():
    """Batched prefill workload at full size (long-memory channels)."""
    wl = synth.WORKLOADS["prefill_b8_h64_t8192"]
    params, tokens, S, conv = _setup(wl)
    S0, c0 = S.clone(), conv.clone()
    o = gpu_prefill(wl, params, tokens, S, conv)
    pairs = synth.sample_heads(wl, 6)
    ref = oracle_pairs(params, tokens, S0, c0, pairs, call_major=False)
    check(ref, o, S, conv, pairs)


def test_graph_replay_equals_launch():
    """A prefill call captured in a CUDA graph and replayed gives bit for bit
    what launching it gives (the entry point neither synchronises nor
    allocates, so it can be captured)."""
    params, tokens, S, conv = _setup(SMALL)
    S2, c2 = S.clone(), conv.clone()
    o_l = gpu_prefill(SMALL, params, tokens, S, conv)

    B, T, H, d = tokens["q"].shape
    q, k, v = (bits(tokens[n]) for n in ("q", "k", "v"))
    o_g = torch.full((B, T, H, d), float("nan"), device=DEV)
    ctx = kda.kda_create(H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        nws = kda.kda_prefill_workspace_bytes(ctx, B, T)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=DEV) if nws else None
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=side):
            kda.kda_prefill(ctx, B, T, q, k, v, tokens["z"], tokens["beta_logit"],
                            tokens["gate_logit"], c2, S2, o_g, ws, nws,
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


@pytest.mark.parametrize("schedule", ["split", "relay"])
def test_tail_wave_matches_oracle(schedule):
    """More heads than SMs: the last partial wave runs on the few-head
    schedule (split, or relay pairs without a workspace).  200 heads = one
    full wave of single CTAs plus a 48-head tail on 152 SMs; sampled heads
    from both parts against the oracle."""
    wl = synth.shrink(synth.WORKLOADS["prefill_b8_h64_t8192"], B=2, H=100, T=200)
    params, tokens, S, conv = _setup(wl)
    S0, c0 = S.clone(), conv.clone()
    o = gpu_prefill(wl, params, tokens, S, conv, schedule=schedule)
    pairs = [(0, 0), (0, 57), (1, 51), (1, 52), (1, 99)]
    ref = oracle_pairs(params, tokens, S0, c0, pairs, call_major=False)
    check(ref, o, S, conv, pairs)


@pytest.mark.parametrize("shape", [dict(B=1, H=32, T=4096), dict(B=2, H=100, T=333), dict(B=1, H=1, T=333),
                                   dict(B=1, H=76, T=1000), dict(B=4, H=16, T=700), dict(B=1, H=2, T=8192)],
                         ids=["single_seq", "tail", "one_head", "h76", "b4_h16", "long_ring"])
def test_schedules_agree_bit_for_bit(shape):
    """The split schedule, the relay pairs and single CTAs (the packed entry
    point runs one CTA per sequence-head) compute the same arithmetic in the
    same order: o, S and the window agree bit for bit.  Shapes: the
    single-sequence workload's full size; a tail wave with a ragged last
    chunk; one head (one consumer, as many producers as it has chunks); 76
    heads (as many producers as consumers: the producers set the pace); four
    sequences of 16 heads; two heads of 128 chunks each (every head's ring of
    four slots is refilled 32 times)."""
    wl = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], **shape)
    params, tokens, S, conv = _setup(wl)
    S0, c0 = S.clone(), conv.clone()
    res = {}
    for schedule in ("split", "relay"):
        S1, c1 = S0.clone(), c0.clone()
        res[schedule] = (gpu_prefill(wl, params, tokens, S1, c1, schedule=schedule), S1, c1)
    B, T, H, d = tokens["q"].shape
    cu = torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device=DEV)
    flat = {n: tokens[n].reshape((B * T,) + tuple(tokens[n].shape[2:])).contiguous() for n in tokens}
    o_v = torch.zeros((B * T, H, d), device=DEV)
    S_v, c_v = S0.clone(), c0.clone()
    ctx = kda.kda_create(H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        kda.kda_prefill_varlen(ctx, B, cu, B * T, bits(flat["q"]), bits(flat["k"]), bits(flat["v"]), flat["z"],
                               flat["beta_logit"], flat["gate_logit"], c_v, S_v, o_v)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    for schedule, (o, S1, c1) in res.items():
        assert torch.equal(o.reshape(B * T, H, d), o_v), schedule
        assert torch.equal(S1, S_v), schedule
        assert torch.equal(c1, c_v), schedule
