"""Failure paths on the GPU, made to happen without faulting anything.

* A bounded wait that runs out: a test-only kernel waits on an mbarrier that
  nothing arrives on (no copy or MMA pending) for one millisecond and gives
  up; kda_sync_status must report KDA_ERR_TIMEOUT once, then KDA_OK, and the
  context must keep working.
* An injected launch failure: with KDA_FAULT_INJECT naming an entry point,
  the context's launches of it are replaced on the host by
  cudaErrorLaunchFailure; the call must return KDA_ERR_CUDA, launch nothing
  and leave every buffer as it was.
* A relay hand-over that never comes: with KDA_FAULT_INJECT=relay_drop the
  first CTA of each prefill relay pair skips its first state hand-over, so
  the second CTA's bounded wait (1 s) runs out, then the first one's wait for
  a state the second never sends; both give up, drain what they issued and
  leave; kda_sync_status reports KDA_ERR_TIMEOUT, S and the window keep their
  old contents, and the device keeps working.
* A split launch that does not fit: with KDA_FAULT_INJECT=split_nofit the
  split schedule's cooperative launch is treated as not fitting on the
  device; the call runs the relay pairs instead, one launch, and gives the
  same results bit for bit.
* A chunk that is never published: with KDA_FAULT_INJECT=split_drop the
  producers of the split schedule skip publishing their first chunk, so each
  consumer's bounded wait for its head's first chunk runs out; the same
  report, S and the window unchanged, the device still working.
"""
import os

import pytest
import torch

from harness import Guarded

import kda_delta_rule_token_gb300 as kda
from kda_delta_rule_token_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_delta_rule_token_gb300 import build
    build.build()
    kda.load()


def _create(wl, params):
    return kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])


def _decode_once(ctx, wl, tokens, S, conv, o):
    kda.kda_decode_step(ctx, wl.B, tokens["q"][0], tokens["k"][0], tokens["v"][0], tokens["z"][0],
                        tokens["beta_logit"][0], tokens["gate_logit"][0], conv, S, o)


def test_bounded_wait_gives_up_and_is_reported_once():
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=2, H=2, T=1)
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    S, conv = st["S"], st["conv_state"]
    ctx = _create(wl, params)
    try:
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
        kda.kda_testing_bounded_wait(ctx, 1000)          # gives up after 1 ms
        assert kda.kda_sync_status(ctx) == kda.KDA_ERR_TIMEOUT
        assert "error word" in kda.kda_last_error_detail()
        assert kda.kda_sync_status(ctx) == kda.KDA_OK    # the word was cleared
        # the context and the device keep working
        o = torch.empty((wl.B, wl.H, 128), device=DEV)
        _decode_once(ctx, wl, tokens, S, conv, o)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
        assert bool(torch.isfinite(o).all())
    finally:
        kda.kda_destroy(ctx)


def test_bounded_wait_limit_is_validated():
    wl = synth.TINY
    params = synth.make_params(wl, DEV)
    ctx = _create(wl, params)
    try:
        for bad in (0, 1000001):
            with pytest.raises(kda.KDAError) as ei:
                kda.kda_testing_bounded_wait(ctx, bad)
            assert ei.value.status == kda.KDA_ERR_INVALID_ARG
    finally:
        kda.kda_destroy(ctx)


@pytest.fixture
def inject(monkeypatch):
    def set_(what):
        monkeypatch.setenv("KDA_FAULT_INJECT", what)
    return set_


@pytest.mark.parametrize("what", ["decode", "all", "prefill,decode"])
def test_injected_decode_launch_failure(inject, what):
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=2, H=3, T=1)
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    S, conv = st["S"], st["conv_state"]
    S0, c0 = S.clone(), conv.clone()
    o = torch.full((wl.B, wl.H, 128), 3.0, device=DEV)
    inject(what)
    ctx = _create(wl, params)
    try:
        n0 = kda.kda_launch_count()
        with pytest.raises(kda.KDAError) as ei:
            _decode_once(ctx, wl, tokens, S, conv, o)
        assert ei.value.status == kda.KDA_ERR_CUDA
        detail = kda.kda_last_error_detail()
        assert "cudaErrorLaunchFailure" in detail and "KDA_FAULT_INJECT" in detail
        assert kda.kda_launch_count() == n0                 # nothing was launched
        torch.cuda.synchronize()
        assert torch.equal(S, S0) and torch.equal(conv, c0) and bool((o == 3.0).all())
        assert kda.kda_sync_status(ctx) == kda.KDA_OK       # no kernel reported anything
    finally:
        kda.kda_destroy(ctx)


def test_injected_prefill_launch_failures(inject):
    wl = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], B=2, H=2, T=70)
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    S, conv = st["S"], st["conv_state"]
    S0, c0 = S.clone(), conv.clone()
    q, k, v = (tokens[n].view(torch.int16) for n in ("q", "k", "v"))
    o = torch.full((wl.B, wl.T, wl.H, 128), 3.0, device=DEV)
    cu = torch.tensor([0, wl.T], dtype=torch.int32, device=DEV)
    inject("prefill,prefill_varlen")
    ctx = _create(wl, params)
    try:
        nws = kda.kda_prefill_workspace_bytes(ctx, wl.B, wl.T)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=DEV)
        n0 = kda.kda_launch_count()
        with pytest.raises(kda.KDAError) as ei:
            kda.kda_prefill(ctx, wl.B, wl.T, q, k, v, tokens["z"], tokens["beta_logit"],
                            tokens["gate_logit"], conv, S, o, ws, nws)
        assert ei.value.status == kda.KDA_ERR_CUDA
        with pytest.raises(kda.KDAError) as ei:
            kda.kda_prefill_varlen(ctx, 1, cu, wl.T, q[0], k[0], v[0], tokens["z"][0],
                                   tokens["beta_logit"][0], tokens["gate_logit"][0], conv[:1], S[:1], o[0])
        assert ei.value.status == kda.KDA_ERR_CUDA
        assert "KDA_FAULT_INJECT" in kda.kda_last_error_detail()
        assert kda.kda_launch_count() == n0
        torch.cuda.synchronize()
        assert torch.equal(S, S0) and torch.equal(conv, c0) and bool((o == 3.0).all())
        # decode is not named: it still runs
        od = torch.empty((wl.B, wl.H, 128), device=DEV)
        f32 = {n: tokens[n][:, 0].float().contiguous() for n in ("q", "k", "v", "z", "gate_logit")}
        kda.kda_decode_step(ctx, wl.B, f32["q"], f32["k"], f32["v"], f32["z"],
                            tokens["beta_logit"][:, 0].contiguous(), f32["gate_logit"], conv, S, od)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
        assert kda.kda_launch_count() == n0 + 1
    finally:
        kda.kda_destroy(ctx)


def test_injection_is_off_when_unset(monkeypatch):
    monkeypatch.delenv("KDA_FAULT_INJECT", raising=False)
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=1, H=1, T=1)
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    ctx = _create(wl, params)
    try:
        o = torch.empty((1, 1, 128), device=DEV)
        _decode_once(ctx, wl, tokens, st["S"], st["conv_state"], o)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)


def test_injected_lowrank_launch_failure(inject):
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=4, H=2, T=1)
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    lr = synth.make_lowrank(wl, DEV, hidden=64, rank=32)
    S, conv = st["S"], st["conv_state"]
    S0, c0 = S.clone(), conv.clone()
    inject("lowrank")
    ctx = _create(wl, params)
    try:
        kda.kda_bind_lowrank(ctx, 64, 32, lr["W_fa"], lr["W_fb"], lr["W_bp"])
        z = torch.full((4, 2, 128), 3.0, device=DEV)
        bl = torch.full((4, 2), 3.0, device=DEV)
        ws = torch.empty(kda.kda_decode_lowrank_workspace_bytes(ctx, 4), dtype=torch.uint8, device=DEV)
        o = torch.full((4, 2, 128), 3.0, device=DEV)
        n0 = kda.kda_launch_count()
        with pytest.raises(kda.KDAError) as ei:
            kda.kda_lowrank(ctx, 4, lr["x"][0], z, bl, ws)
        assert ei.value.status == kda.KDA_ERR_CUDA
        with pytest.raises(kda.KDAError) as ei:
            kda.kda_decode_step_lowrank(ctx, 4, lr["x"][0], tokens["q"][0], tokens["k"][0], tokens["v"][0],
                                        tokens["gate_logit"][0], conv, S, o, None, ws)
        assert ei.value.status == kda.KDA_ERR_CUDA
        assert kda.kda_launch_count() == n0
        torch.cuda.synchronize()
        assert bool((z == 3.0).all()) and bool((bl == 3.0).all()) and bool((o == 3.0).all())
        assert torch.equal(S, S0) and torch.equal(conv, c0)
    finally:
        kda.kda_destroy(ctx)


def test_relay_hand_over_that_never_comes_times_out(inject, monkeypatch):
    wl = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], B=1, H=2, T=192)   # relay pairs, 3 chunks
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    S, conv = st["S"], st["conv_state"]
    S.normal_(0.0, 0.01)
    q, k, v = (tokens[n].view(torch.int16) for n in ("q", "k", "v"))
    gS, gc = Guarded(S), Guarded(conv)
    S0, c0 = S.clone(), conv.clone()
    o = torch.zeros((wl.B, wl.T, wl.H, 128), device=DEV)
    inject("relay_drop")
    ctx = _create(wl, params)
    try:
        kda.kda_prefill(ctx, wl.B, wl.T, q, k, v, tokens["z"], tokens["beta_logit"], tokens["gate_logit"],
                        gc.t, gS.t, o)
        assert kda.kda_sync_status(ctx) == kda.KDA_ERR_TIMEOUT
        assert kda.kda_sync_status(ctx) == kda.KDA_OK          # reported once
        assert torch.equal(gS.t, S0) and torch.equal(gc.t, c0)
        assert gS.intact() and gc.intact()
    finally:
        kda.kda_destroy(ctx)
    # a context without the injection computes the same call normally
    monkeypatch.delenv("KDA_FAULT_INJECT", raising=False)
    ctx = _create(wl, params)
    try:
        kda.kda_prefill(ctx, wl.B, wl.T, q, k, v, tokens["z"], tokens["beta_logit"], tokens["gate_logit"],
                        conv, S, o)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
        assert not torch.equal(S, S0)
    finally:
        kda.kda_destroy(ctx)


def test_split_chunk_that_is_never_published_times_out(inject, monkeypatch):
    wl = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], B=1, H=2, T=192)   # split schedule, 3 chunks
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    S, conv = st["S"], st["conv_state"]
    S.normal_(0.0, 0.01)
    q, k, v = (tokens[n].view(torch.int16) for n in ("q", "k", "v"))
    gS, gc = Guarded(S), Guarded(conv)
    S0, c0 = S.clone(), conv.clone()
    o = torch.zeros((wl.B, wl.T, wl.H, 128), device=DEV)
    inject("split_drop")
    ctx = _create(wl, params)
    try:
        nws = kda.kda_prefill_workspace_bytes(ctx, wl.B, wl.T)
        assert nws > 0
        ws = torch.empty(nws, dtype=torch.uint8, device=DEV)
        kda.kda_prefill(ctx, wl.B, wl.T, q, k, v, tokens["z"], tokens["beta_logit"], tokens["gate_logit"],
                        gc.t, gS.t, o, ws, nws)
        assert kda.kda_sync_status(ctx) == kda.KDA_ERR_TIMEOUT
        assert kda.kda_sync_status(ctx) == kda.KDA_OK          # reported once
        assert torch.equal(gS.t, S0) and torch.equal(gc.t, c0)
        assert gS.intact() and gc.intact()
    finally:
        kda.kda_destroy(ctx)
    # a context without the injection computes the same call normally
    monkeypatch.delenv("KDA_FAULT_INJECT", raising=False)
    ctx = _create(wl, params)
    try:
        kda.kda_prefill(ctx, wl.B, wl.T, q, k, v, tokens["z"], tokens["beta_logit"], tokens["gate_logit"],
                        conv, S, o, ws, nws)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
        assert not torch.equal(S, S0)
    finally:
        kda.kda_destroy(ctx)


def test_split_launch_that_does_not_fit_falls_back_to_relay_pairs(inject, monkeypatch):
    wl = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], B=2, H=8, T=300)   # 16 heads, split schedule
    params, tokens = synth.make_params(wl, DEV), synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    S0, c0 = st["S"].normal_(0.0, 0.01).clone(), st["conv_state"].clone()
    q, k, v = (tokens[n].view(torch.int16) for n in ("q", "k", "v"))
    res = {}
    for what in ("", "split_nofit"):
        if what:
            inject(what)
        else:
            monkeypatch.delenv("KDA_FAULT_INJECT", raising=False)
        S, conv = S0.clone(), c0.clone()
        o = torch.zeros((wl.B, wl.T, wl.H, 128), device=DEV)
        ctx = _create(wl, params)
        try:
            nws = kda.kda_prefill_workspace_bytes(ctx, wl.B, wl.T)
            assert nws > 0
            ws = torch.empty(nws, dtype=torch.uint8, device=DEV)
            n0 = kda.kda_launch_count()
            kda.kda_prefill(ctx, wl.B, wl.T, q, k, v, tokens["z"], tokens["beta_logit"], tokens["gate_logit"],
                            conv, S, o, ws, nws)
            assert kda.kda_sync_status(ctx) == kda.KDA_OK
            assert kda.kda_launch_count() == n0 + 1
        finally:
            kda.kda_destroy(ctx)
        res[what] = (o, S, conv)
    for a, b in zip(res[""], res["split_nofit"]):
        assert torch.equal(a, b)
