"""Packed sequences of different lengths (kda_prefill_varlen) on the GPU.

Each sequence is checked against the fp64 oracle run on that sequence alone
(rel-L2 2e-3 over o and the final S; the conv window exactly), and the packed
call must give exactly what one kda_prefill call per sequence gives: the
same arithmetic, only the addressing differs (a few-head kda_prefill call
runs its heads as CTA pairs that relay the state; the relay carries the
state in the form a single CTA keeps it, so the results stay bit for bit
equal).  o, S and
the windows sit inside poisoned guard regions during each packed call.
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


def bits(x):
    return x.view(torch.int16)


def packed(tokens, lengths):
    """[B, Tmax, ...] per-sequence tokens -> packed [total, ...] (first L_b of each)."""
    out = {n: torch.cat([tokens[n][b, :L] for b, L in enumerate(lengths)], 0).contiguous()
           for n in ("q", "k", "v", "z", "gate_logit", "beta_logit")}
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=DEV)
    return out, cu


def run_varlen(H, params, pk, cu, S, conv):
    total = int(cu[-1].item())
    go = Guarded(torch.full((total, H, 128), float("nan"), device=DEV))
    gS, gc = Guarded(S), Guarded(conv)
    ctx = kda.kda_create(H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        kda.kda_prefill_varlen(ctx, len(cu) - 1, cu, total, bits(pk["q"]), bits(pk["k"]), bits(pk["v"]),
                               pk["z"], pk["beta_logit"], pk["gate_logit"], gc.t, gS.t, go.t)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    assert go.intact() and gS.intact() and gc.intact(), "a guard region was written"
    S.copy_(gS.t)
    conv.copy_(gc.t)
    return go.t.clone()


def run_separate(H, params, tokens, lengths, S, conv):
    """One kda_prefill call per (non-empty) sequence, B = 1 each."""
    outs = []
    ctx = kda.kda_create(H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        for b, L in enumerate(lengths):
            if L == 0:
                continue
            sl = {n: tokens[n][b:b + 1, :L].contiguous() for n in tokens}
            o = torch.empty((1, L, H, 128), device=DEV)
            Sb, cb = S[b:b + 1].clone(), conv[b:b + 1].clone()
            nws = kda.kda_prefill_workspace_bytes(ctx, 1, L)
            ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=DEV)
            kda.kda_prefill(ctx, 1, L, bits(sl["q"]), bits(sl["k"]), bits(sl["v"]), sl["z"],
                            sl["beta_logit"], sl["gate_logit"], cb, Sb, o, ws, nws)
            S[b:b + 1].copy_(Sb)
            conv[b:b + 1].copy_(cb)
            outs.append(o[0])
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    return torch.cat(outs, 0) if outs else torch.empty((0, H, 128), device=DEV)


LENGTHS = [0, 1, 2, 63, 64, 65, 130, 5]


def _setup(lengths, H=2):
    wl = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], B=len(lengths), H=H, T=max(lengths),
                      s0_std=0.05, win_std=1.0)
    params = synth.make_params(wl, DEV)
    tokens = synth.make_tokens(wl, DEV)
    st = synth.make_state(wl, DEV)
    return wl, params, tokens, st["S"], st["conv_state"]


def test_varlen_matches_oracle_per_sequence():
    wl, params, tokens, S, conv = _setup(LENGTHS)
    S0, c0 = S.clone(), conv.clone()
    pk, cu = packed(tokens, LENGTHS)
    o = run_varlen(wl.H, params, pk, cu, S, conv)
    start = 0
    for b, L in enumerate(LENGTHS):
        if L == 0:
            assert torch.equal(S[b], S0[b]) and torch.equal(conv[b], c0[b])
            continue
        tk = {n: tokens[n][b:b + 1, :L] for n in tokens}
        ref = oracle_pairs(params, tk, S0[b:b + 1], c0[b:b + 1], [(0, h) for h in range(wl.H)],
                           call_major=False)
        for h in range(wl.H):
            eo = rel_l2(np64(o[start:start + L, h]), ref[(0, h)].o[0, :, 0])
            es = rel_l2(np64(S[b, h]), ref[(0, h)].S[0, 0])
            assert eo <= TOL, f"seq {b} head {h}: o rel-L2 {eo:.3e}"
            assert es <= TOL, f"seq {b} head {h}: S rel-L2 {es:.3e}"
            assert max_rel_err(pair_window(conv, b, h), ref[(0, h)].conv_state) == 0.0
        start += L


def test_varlen_equals_separate_calls():
    wl, params, tokens, S, conv = _setup(LENGTHS)
    S2, c2 = S.clone(), conv.clone()
    pk, cu = packed(tokens, LENGTHS)
    o_v = run_varlen(wl.H, params, pk, cu, S, conv)
    o_s = run_separate(wl.H, params, tokens, LENGTHS, S2, c2)
    assert torch.equal(o_v, o_s)
    assert torch.equal(S, S2)
    assert torch.equal(conv, c2)


def test_varlen_all_empty_or_zero_total_is_noop():
    wl, params, tokens, S, conv = _setup([0, 0, 3])
    S0, c0 = S.clone(), conv.clone()
    cu = torch.zeros(4, dtype=torch.int32, device=DEV)
    o = torch.empty((1, wl.H, 128), device=DEV)
    ctx = kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        t = tokens
        kda.kda_prefill_varlen(ctx, 3, cu, 0, bits(t["q"]), bits(t["k"]), bits(t["v"]), t["z"],
                               t["beta_logit"], t["gate_logit"], conv, S, o)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    assert torch.equal(S, S0) and torch.equal(conv, c0)


def test_varlen_long_sequences_sampled():
    """Mixed long lengths (several chunks, ragged tails), sampled heads vs the oracle."""
    lengths = [1000, 333, 0, 2049]
    wl, params, tokens, S, conv = _setup(lengths, H=4)
    S0, c0 = S.clone(), conv.clone()
    pk, cu = packed(tokens, lengths)
    o = run_varlen(wl.H, params, pk, cu, S, conv)
    starts = np.concatenate([[0], np.cumsum(lengths)])
    for b, h in [(0, 1), (1, 3), (3, 0)]:
        L = lengths[b]
        tk = {n: tokens[n][b:b + 1, :L] for n in tokens}
        ref = oracle_pairs(params, tk, S0[b:b + 1], c0[b:b + 1], [(0, h)], call_major=False)[(0, h)]
        s = starts[b]
        assert rel_l2(np64(o[s:s + L, h]), ref.o[0, :, 0]) <= TOL
        assert rel_l2(np64(S[b, h]), ref.S[0, 0]) <= TOL
        assert max_rel_err(pair_window(conv, b, h), ref.conv_state) == 0.0
    assert torch.equal(S[2], S0[2]) and torch.equal(conv[2], c0[2])


def test_varlen_bench_workload_sampled():
    """The packed workload the benchmark times (32 sequences, 80,371 tokens,
    64 heads, one launch), sampled (sequence, head) pairs vs the oracle: the
    shortest and the longest sequence, the first and the last."""
    lengths = synth.packed_lengths()
    wl = synth.packed_workload(lengths)
    params = synth.make_params(wl, DEV)
    tk = synth.make_tokens(wl, DEV)
    Bs, H, total = len(lengths), wl.H, wl.T
    S = torch.zeros((Bs, H, 128, 128), device=DEV)
    conv = torch.zeros((Bs, 3, 3 * H * 128), device=DEV)
    pk = {n: tk[n][0] for n in tk}
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=DEV)
    o = run_varlen(H, params, pk, cu, S, conv)
    starts = np.concatenate([[0], np.cumsum(lengths)])
    picks = [(int(np.argmin(lengths)), 5), (int(np.argmax(lengths)), 63), (0, 0), (Bs - 1, 31)]
    zS = torch.zeros((1, H, 128, 128))
    zc = torch.zeros((1, 3, 3 * H * 128))
    for b, h in picks:
        s, L = int(starts[b]), int(lengths[b])
        seq = {n: tk[n][:, s:s + L] for n in tk}
        ref = oracle_pairs(params, seq, zS, zc, [(0, h)], call_major=False)[(0, h)]
        assert rel_l2(np64(o[s:s + L, h]), ref.o[0, :, 0]) <= TOL, f"seq {b} head {h}"
        assert rel_l2(np64(S[b, h]), ref.S[0, 0]) <= TOL, f"seq {b} head {h}"
        assert max_rel_err(pair_window(conv, b, h), ref.conv_state) == 0.0


def test_varlen_nonfinite_next_sequence_does_not_leak():
    """The last chunk of a packed sequence is partial and its tile rows past
    the end hold the next sequence's tokens; NaN / Inf there must change
    nothing of the earlier sequence (o, S and window bit for bit)."""
    lengths = [70, 50]
    wl, params, tokens, S, conv = _setup(lengths)
    S2, c2 = S.clone(), conv.clone()
    pk, cu = packed(tokens, lengths)
    o_ref = run_varlen(wl.H, params, pk, cu, S, conv)
    bad = {n: t.clone() for n, t in pk.items()}
    for n in ("q", "k", "v", "gate_logit", "beta_logit"):
        bad[n][lengths[0]:] = float("nan")
    bad["z"][lengths[0]:] = float("inf")
    o_bad = run_varlen(wl.H, params, bad, cu, S2, c2)
    L = lengths[0]
    assert torch.equal(o_bad[:L], o_ref[:L])
    assert torch.equal(S2[0], S[0])
    assert torch.equal(c2[0], conv[0])
