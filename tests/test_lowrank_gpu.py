"""Low-rank front-end (kda_lowrank, kda_decode_step_lowrank) vs the fp64 oracle (GPU).

Tolerances.  kda_lowrank: max|x - r| / max|r| <= 2e-5 on z and on beta_logit,
per output tensor.  Each product runs as three tf32 products (hi*hi + hi*lo
+ lo*hi of the split a = hi + lo), whose error is below 2^-19 of |a b|, and
the fp32 accumulation adds about K * 2^-24 of the sum of |a b| at worst; for
N(0, 1) inputs with the 1/sqrt(K) weight scale that is a few 1e-6 of
max|z| at K = 7168, so 2e-5 leaves a margin of several times.  The cases
span one to 1,000 tokens (token tiles of 32 to 256), ragged hidden, rank and
H, and the largest rank (512).
kda_decode_step_lowrank: the decode tolerance, max relative error 1e-4 on o
at every call and on S after the last call, per (sequence, head), against
the oracle's front-end followed by the oracle's token step.
"""
import numpy as np
import pytest
import torch

import kda_delta_rule_token_gb300 as kda
from kda_delta_rule_token_gb300 import synth
import oracle
from harness import Guarded, max_rel_err, np64, pair_params, pair_window

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_FE = 2e-5
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_delta_rule_token_gb300 import build
    build.build()
    kda.load()


def _ctx(wl, params, lr):
    ctx = kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    kda.kda_bind_lowrank(ctx, lr["hidden"], lr["rank"], lr["W_fa"], lr["W_fb"], lr["W_bp"])
    return ctx


def run_lowrank(ctx, H, x2d):
    N = x2d.shape[0]
    gz = Guarded(torch.zeros((N, H, 128), device=DEV))
    gb = Guarded(torch.zeros((N, H), device=DEV))
    nws = kda.kda_lowrank_workspace_bytes(ctx, N)
    ws = torch.empty(nws, dtype=torch.uint8, device=DEV)
    kda.kda_lowrank(ctx, N, x2d, gz.t, gb.t, ws)
    assert kda.kda_sync_status(ctx) == kda.KDA_OK
    assert gz.intact() and gb.intact(), "a guard region was written"
    return gz.t.clone(), gb.t.clone()


@pytest.mark.parametrize("N,hidden,rank,H", [(5, 96, 32, 3), (64, 7168, 128, 32), (256, 7168, 128, 64),
                                             (1000, 512, 64, 4), (300, 100, 36, 2), (64, 100, 36, 3),
                                             (65, 7168, 128, 32), (1, 7168, 512, 5), (33, 2052, 508, 7)])
def test_lowrank_matches_oracle(N, hidden, rank, H):
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=N, H=H, T=1)
    params = synth.make_params(wl, DEV)
    lr = synth.make_lowrank(wl, DEV, hidden=hidden, rank=rank)
    ctx = _ctx(wl, params, lr)
    try:
        x = lr["x"][0]
        z, bl = run_lowrank(ctx, H, x)
    finally:
        kda.kda_destroy(ctx)
    zr, br = oracle.lowrank(np64(x), np64(lr["W_fa"]), np64(lr["W_fb"]), np64(lr["W_bp"]), H)
    ez, eb = max_rel_err(np64(z), zr), max_rel_err(np64(bl), br)
    print(f"\n  N={N} hidden={hidden} rank={rank} H={H}: z {ez:.2e}, beta_logit {eb:.2e}")
    assert ez <= TOL_FE and eb <= TOL_FE


def _decode_lowrank(wl, params, lr, tokens, S, conv, o_pre=False):
    T, B, H, d = tokens["q"].shape
    gS, gc = Guarded(S), Guarded(conv)
    go = Guarded(torch.zeros((B, H, d), device=DEV))
    o = torch.empty((T, B, H, d), device=DEV)
    ctx = _ctx(wl, params, lr)
    try:
        nws = kda.kda_decode_lowrank_workspace_bytes(ctx, B)
        ws = torch.empty(nws, dtype=torch.uint8, device=DEV)
        for t in range(T):
            kda.kda_decode_step_lowrank(ctx, B, lr["x"][t], tokens["q"][t], tokens["k"][t], tokens["v"][t],
                                        tokens["gate_logit"][t], gc.t, gS.t, go.t, None, ws)
            o[t].copy_(go.t)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    assert gS.intact() and gc.intact() and go.intact(), "a guard region was written"
    S.copy_(gS.t)
    conv.copy_(gc.t)
    return o


def _check(wl, params, lr, tokens, S0, c0, S, conv, o, pairs):
    """Oracle: front-end in fp64, then the token step in fp64 on exactly those
    (unrounded) z / beta_logit values."""
    seqs = sorted({b for b, _ in pairs})
    for b in seqs:
        x = np64(lr["x"][:, b])
        z, bl = oracle.lowrank(x, np64(lr["W_fa"]), np64(lr["W_fb"]), np64(lr["W_bp"]), wl.H)
        for h in [hh for bb, hh in pairs if bb == b]:
            tk = {n: np64(tokens[n][:, b, h])[None, :, None, :] for n in ("q", "k", "v", "gate_logit")}
            tk["z"] = z[:, h][None, :, None, :]
            tk["beta_logit"] = bl[:, h][None, :, None]
            ref = oracle.run(**tk, **pair_params(params, h), conv_state=pair_window(c0, b, h),
                             S=np64(S0[b, h])[None, None])
            og = np64(o[:, b, h])
            for t in range(og.shape[0]):
                e = max_rel_err(og[t], ref.o[0, t, 0])
                assert e <= TOL, f"o at call {t}, pair {(b, h)}: {e:.3e}"
            e = max_rel_err(np64(S[b, h]), ref.S[0, 0])
            assert e <= TOL, f"S of pair {(b, h)}: {e:.3e}"
            assert max_rel_err(pair_window(conv, b, h), ref.conv_state) == 0.0


def test_decode_lowrank_small_every_output():
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=3, H=5, T=9)
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    lr = synth.make_lowrank(wl, DEV, hidden=256, rank=32)
    S, conv = st["S"], st["conv_state"]
    S0, c0 = S.clone(), conv.clone()
    o = _decode_lowrank(wl, params, lr, tokens, S, conv)
    _check(wl, params, lr, tokens, S0, c0, S, conv, o, [(b, h) for b in range(wl.B) for h in range(wl.H)])


def test_decode_lowrank_b64_h32_256_calls_sampled():
    """Batched-decode workload through the front-end (hidden 7168, rank 128):
    256 calls, sampled pairs vs the oracle."""
    wl = synth.WORKLOADS["decode_b64_h32_x256"]
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    lr = synth.make_lowrank(wl, DEV)
    S, conv = st["S"], st["conv_state"]
    S0, c0 = S.clone(), conv.clone()
    o = _decode_lowrank(wl, params, lr, tokens, S, conv)
    _check(wl, params, lr, tokens, S0, c0, S, conv, o, synth.sample_heads(wl, 6))


def test_decode_lowrank_equals_frontend_then_decode():
    """The fused entry point gives bit for bit what kda_lowrank followed by
    kda_decode_step gives."""
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=8, H=4, T=3)
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    lr = synth.make_lowrank(wl, DEV, hidden=512, rank=64)
    S, conv = st["S"], st["conv_state"]
    S2, c2 = S.clone(), conv.clone()
    o = _decode_lowrank(wl, params, lr, tokens, S, conv)
    ctx = _ctx(wl, params, lr)
    try:
        B, H = wl.B, wl.H
        ws = torch.empty(kda.kda_lowrank_workspace_bytes(ctx, B), dtype=torch.uint8, device=DEV)
        z = torch.empty((B, H, 128), device=DEV)
        bl = torch.empty((B, H), device=DEV)
        o2 = torch.empty_like(o)
        for t in range(wl.T):
            kda.kda_lowrank(ctx, B, lr["x"][t], z, bl, ws)
            kda.kda_decode_step(ctx, B, tokens["q"][t], tokens["k"][t], tokens["v"][t], z, bl,
                                tokens["gate_logit"][t], c2, S2, o2[t])
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    assert torch.equal(o, o2) and torch.equal(S, S2) and torch.equal(conv, c2)


def test_decode_lowrank_graph_replay_equals_launches():
    """kda_decode_step_lowrank launches its later kernels as programmatic
    dependents (they start early and wait for their inputs); captured in a
    CUDA graph and replayed, the calls give bit for bit what launching them
    gives."""
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=16, H=4, T=4)
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    lr = synth.make_lowrank(wl, DEV, hidden=512, rank=64)
    S, conv = st["S"], st["conv_state"]
    S2, c2 = S.clone(), conv.clone()
    o = _decode_lowrank(wl, params, lr, tokens, S, conv)
    B, H = wl.B, wl.H
    og = torch.full((wl.T, B, H, 128), float("nan"), device=DEV)
    ctx = _ctx(wl, params, lr)
    try:
        ws = torch.empty(kda.kda_decode_lowrank_workspace_bytes(ctx, B), dtype=torch.uint8, device=DEV)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=side):
            for t in range(wl.T):
                kda.kda_decode_step_lowrank(ctx, B, lr["x"][t], tokens["q"][t], tokens["k"][t], tokens["v"][t],
                                            tokens["gate_logit"][t], c2, S2, og[t], None, ws,
                                            stream=torch.cuda.current_stream())
        torch.cuda.current_stream().wait_stream(side)
        assert bool(torch.isnan(og).all())   # the capture itself ran nothing
        g.replay()
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
        del g
    finally:
        kda.kda_destroy(ctx)
    assert torch.equal(o, og) and torch.equal(S, S2) and torch.equal(conv, c2)


def test_lowrank_argument_errors():
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=4, H=2, T=1)
    params = synth.make_params(wl, DEV)
    lr = synth.make_lowrank(wl, DEV, hidden=64, rank=32)
    ctx = kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        z = torch.empty((4, 2, 128), device=DEV)
        bl = torch.empty((4, 2), device=DEV)
        ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
        with pytest.raises(kda.KDAError) as ei:                      # nothing bound yet
            kda.kda_lowrank(ctx, 4, lr["x"][0], z, bl, ws)
        assert ei.value.status == kda.KDA_ERR_INVALID_ARG
        for hidden, rank in ((66, 32), (64, 30), (64, 516)):
            with pytest.raises(kda.KDAError) as ei:
                kda.kda_bind_lowrank(ctx, hidden, rank, lr["W_fa"], lr["W_fb"], lr["W_bp"])
            assert ei.value.status == kda.KDA_ERR_INVALID_ARG
        kda.kda_bind_lowrank(ctx, 64, 32, lr["W_fa"], lr["W_fb"], lr["W_bp"])
        need = kda.kda_lowrank_workspace_bytes(ctx, 4)
        with pytest.raises(kda.KDAError) as ei:                      # workspace too small
            kda.kda_lowrank(ctx, 4, lr["x"][0], z, bl, ws, need - 16)
        assert ei.value.status == kda.KDA_ERR_INVALID_ARG
        kda.kda_lowrank(ctx, 0, lr["x"][0], z, bl, ws)               # N = 0: no-op
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
