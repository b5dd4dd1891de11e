"""Decode with the state stored as bfloat16 vs the fp64 oracle (GPU).

The variant runs each token in fp32 from the stored bf16 state and rounds the
new state to nearest-even bf16 as it stores it; the read-out uses the new
state as computed.  Rounding decides an integer (the bf16 pattern) from a
floating-point value, and the kernel's fp32 value differs from the oracle's
fp64 one by a few fp32 units, so the checks are:

* one call from the same stored state on both sides: o and o_pre within the
  fp32 decode's 1e-4 (max |x - r| / max |r|, per sequence and head); every
  stored element is the bf16 rounding of a value within EPS_REL * max|S_new|
  of the oracle's exact new state (EPS_REL = 2^-18, about 40 fp32 units of
  the head's largest element: the kernel's fp32 state error is a few units),
  and it equals the round-to-nearest-even pattern of the exact value except
  at a few near-ties (at most TIE_FRAC of the elements);
* many calls, each side keeping its own bf16 state: a near-tie that went the
  other way leaves the two states one bf16 unit apart in one element, and
  later tokens carry such differences on, so the states drift apart by up to
  the size of the variant's own rounding error.  That error is measured on
  the oracle itself: E = the distance of the oracle's bf16-state run from
  its exact (no rounding) run, per pair, max over the calls.  The GPU must
  be no farther from the exact run than 1.25 E (+ the fp32 decode's 1e-4),
  i.e. as accurate as the variant's definition, and within 2 E (+ 1e-4) of
  the oracle's bf16-state run at every call.
"""
import numpy as np
import pytest
import torch

import oracle
import kda_delta_rule_token_gb300 as kda
from kda_delta_rule_token_gb300 import synth
from harness import Guarded, max_rel_err, np64, pair_params, pair_tokens, pair_window, set_pair_window

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_O = 1e-4
EPS_REL = 2.0 ** -18
TIE_FRAC = 1e-3
ACC_FACTOR = 1.25   # GPU error vs exact <= ACC_FACTOR * E + TOL_O
GAP_FACTOR = 2.0    # GPU vs the oracle's bf16-state run <= GAP_FACTOR * E + TOL_O


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_delta_rule_token_gb300 import build
    build.build()
    kda.load()


def bf16_of(S32: torch.Tensor) -> torch.Tensor:
    """fp32 state -> bf16 patterns (int16) rounded to nearest even, by the oracle's rounding."""
    if not bool(S32.any()):
        return torch.zeros(S32.shape, dtype=torch.int16, device=DEV)
    pat = oracle.bf16_round(np64(S32))
    return torch.from_numpy(pat.view(np.int16)).to(DEV)


def values(S16: torch.Tensor) -> np.ndarray:
    return oracle.bf16_value(S16.detach().cpu().numpy().view(np.uint16))


class GuardedBF16:
    """A bf16 tensor inside poisoned guard margins (a float32 Guarded of the same bytes)."""

    def __init__(self, S16: torch.Tensor):
        assert S16.dtype == torch.int16 and S16.numel() % 2 == 0
        self.g = Guarded(torch.zeros(S16.numel() // 2, device=DEV))
        self.t = self.g.t.view(torch.int16).view(S16.shape)
        self.t.copy_(S16)

    def intact(self):
        return self.g.intact()


def run_calls(wl, params, tokens, S16, conv, *, every=None):
    """Run the calls of ``tokens`` (call-major) on the bf16 state in place.

    every(t, S16_before, conv_before, o, o_pre, S16_after) is called after each
    call when given (the tensors are copies).  Returns o [T, B, H, d].
    """
    T, B, H, d = tokens["q"].shape
    go, gp = Guarded(torch.zeros((B, H, d), device=DEV)), Guarded(torch.zeros((B, H, d), device=DEV))
    gS, gc = GuardedBF16(S16), Guarded(conv)
    o = torch.empty((T, B, H, d), device=DEV)
    ctx = kda.kda_create(H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        for t in range(T):
            before = (gS.t.clone(), gc.t.clone()) if every else None
            kda.kda_decode_step_bf16state(ctx, B, tokens["q"][t], tokens["k"][t], tokens["v"][t],
                                          tokens["z"][t], tokens["beta_logit"][t],
                                          tokens["gate_logit"][t], gc.t, gS.t, go.t, gp.t)
            o[t].copy_(go.t)
            if every:
                torch.cuda.synchronize()
                every(t, *before, go.t.clone(), gp.t.clone(), gS.t.clone())
            if t == 0 or t == T - 1 or every:
                torch.cuda.synchronize()
                for g in (go, gp, gS, gc):
                    assert g.intact(), f"a guard region was written at call {t}"
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    S16.copy_(gS.t)
    conv.copy_(gc.t)
    return o


def _one_call_ref(params, tokens, t, S_vals, conv_before, b, h):
    """The oracle's exact (unrounded) call t of pair (b, h) from the given stored state."""
    tk = pair_tokens({k: v[t:t + 1] for k, v in tokens.items()}, b, h, call_major=True)
    return oracle.run(**tk, **pair_params(params, h), conv_state=pair_window(conv_before, b, h),
                      S=S_vals[b, h][None, None])


def _setup(wl, T=None):
    params = synth.make_params(wl, DEV)
    tokens = synth.make_tokens(wl, DEV, T=T)
    st = synth.make_state(wl, DEV)
    return params, tokens, bf16_of(st["S"]), st["conv_state"]


def _extreme(params, tokens):
    """Strong decay (gk about -30 per token: the state walks down into the
    subnormal range), saturated beta, a zero q, large v."""
    params["A_log"][0].fill_(0.0)
    tokens["z"][:, 0, 0].fill_(30.0)
    tokens["beta_logit"][:, 1, 0] = 40.0
    tokens["beta_logit"][:, 1, 1] = -40.0
    tokens["q"][2, 0].zero_()
    tokens["v"][3].mul_(1e3)


@pytest.mark.parametrize("shape", [dict(B=1, H=2, T=16), dict(B=3, H=5, T=9), dict(B=2, H=2, T=8)],
                         ids=["tiny", "ragged", "extreme"])
def test_each_call_is_a_valid_rounding(shape):
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], **shape)
    params, tokens, S16, conv = _setup(wl)
    if shape["T"] == 8:
        _extreme(params, tokens)
    # a nonzero starting state (from fp32 warm tokens) so that decay, erase and write all matter
    warm = synth.make_tokens(wl, DEV, T=6, warm=True)
    run_calls(wl, params, warm, S16, conv)
    stats = {"elems": 0, "off_rne": 0, "worst_o": 0.0}

    def every(t, S_before, conv_before, o, o_pre, S_after):
        S_vals = values(S_before)
        S_new = values(S_after)
        pat_new = S_after.cpu().numpy().view(np.uint16)
        for b in range(wl.B):
            for h in range(wl.H):
                r = _one_call_ref(params, tokens, t, S_vals, conv_before, b, h)
                e = max_rel_err(np64(o[b, h]), r.o[0, 0, 0])
                stats["worst_o"] = max(stats["worst_o"], e)
                assert e <= TOL_O, f"o at call {t}, pair {(b, h)}: {e:.3e}"
                assert max_rel_err(np64(o_pre[b, h]), r.o_pre[0, 0, 0]) <= TOL_O
                ex = r.S[0, 0]
                eps = EPS_REL * np.abs(ex).max()
                lo, hi = oracle.bf16_round(ex - eps), oracle.bf16_round(ex + eps)
                got = S_new[b, h]
                ok = (got >= oracle.bf16_value(lo)) & (got <= oracle.bf16_value(hi))
                assert ok.all(), f"call {t}, pair {(b, h)}: {int((~ok).sum())} elements are no rounding of the exact state"
                stats["off_rne"] += int((pat_new[b, h] != oracle.bf16_round(ex)).sum())
                stats["elems"] += ex.size

    run_calls(wl, params, tokens, S16, conv, every=every)
    frac = stats["off_rne"] / stats["elems"]
    print(f"\n  worst o {stats['worst_o']:.3e}; {stats['off_rne']} of {stats['elems']} elements "
          f"off the nearest-even pattern of the exact state ({frac:.2e})")
    assert frac <= TIE_FRAC


def test_no_write_no_decay_keeps_state_exactly():
    """beta = 0 and gk = 0: the stored bf16 state comes back bit for bit."""
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=2, H=3, T=4)
    params, tokens, S16, conv = _setup(wl)
    S16.copy_(bf16_of(torch.randn(S16.shape, device=DEV)))
    params["A_log"].fill_(-float("inf"))
    tokens["beta_logit"].fill_(-float("inf"))
    S0 = S16.clone()
    run_calls(wl, params, tokens, S16, conv)
    assert torch.equal(S16, S0)


def test_zero_batch_is_noop_and_misaligned_is_rejected():
    wl = synth.TINY
    params, tokens, S16, conv = _setup(wl, T=1)
    S1 = S16.clone()
    ctx = kda.kda_create(wl.H, params["conv_w"], params["dt_bias"], params["A_log"], params["gamma"])
    try:
        o = torch.full((1, wl.H, 128), 7.0, device=DEV)
        kda.kda_decode_step_bf16state(ctx, 0, tokens["q"][0], tokens["k"][0], tokens["v"][0],
                                      tokens["z"][0], tokens["beta_logit"][0], tokens["gate_logit"][0],
                                      conv, S16, o)
        torch.cuda.synchronize()
        assert torch.equal(S16, S1) and bool((o == 7.0).all())
        buf = torch.zeros(S16.numel() + 4, dtype=torch.int16, device=DEV)
        with pytest.raises(kda.KDAError) as ei:
            kda.kda_decode_step_bf16state(ctx, 1, tokens["q"][0], tokens["k"][0], tokens["v"][0],
                                          tokens["z"][0], tokens["beta_logit"][0], tokens["gate_logit"][0],
                                          conv, buf[2:], o)   # 4-byte offset
        assert ei.value.status == kda.KDA_ERR_ALIGNMENT
    finally:
        kda.kda_destroy(ctx)


def _oracle_bf16_pairs(params, tokens, S16_0, conv0, pairs):
    """{pair: (bf16-state run, exact run)} of the oracle from the same stored state."""
    ref = {}
    vals = values(S16_0)
    for (b, h) in pairs:
        tk = pair_tokens(tokens, b, h, call_major=True)
        kw = dict(**tk, **pair_params(params, h), conv_state=pair_window(conv0, b, h),
                  S=vals[b, h][None, None], nthreads=1)
        ref[(b, h)] = (oracle.run(**kw, state_bf16=True), oracle.run(**kw))
    return ref


def _check_multi(ref, o, S16, conv, pairs):
    S_vals = values(S16)
    report = []
    for (b, h) in pairs:
        rb, rx = ref[(b, h)]
        o_g = np64(o[:, b, h])
        T = o_g.shape[0]
        E = max(max_rel_err(rb.o[0, t, 0], rx.o[0, t, 0]) for t in range(T))
        E_S = max_rel_err(rb.S[0, 0], rx.S[0, 0])
        acc = max(max_rel_err(o_g[t], rx.o[0, t, 0]) for t in range(T))
        gap = max(max_rel_err(o_g[t], rb.o[0, t, 0]) for t in range(T))
        report.append((b, h, E, acc, gap))
        assert acc <= ACC_FACTOR * E + TOL_O, f"pair {(b, h)}: o vs exact {acc:.3e}, variant's own error {E:.3e}"
        assert gap <= GAP_FACTOR * E + TOL_O, f"pair {(b, h)}: o vs the bf16-state oracle {gap:.3e} (E {E:.3e})"
        acc_S = max_rel_err(S_vals[b, h], rx.S[0, 0])
        assert acc_S <= ACC_FACTOR * E_S + TOL_O, f"pair {(b, h)}: S vs exact {acc_S:.3e} (E_S {E_S:.3e})"
        assert max_rel_err(S_vals[b, h], rb.S[0, 0]) <= GAP_FACTOR * E_S + TOL_O
        assert max_rel_err(pair_window(conv, b, h), rb.conv_state) == 0.0
    return report


def test_b64_h32_256_calls_sampled():
    """Batched decode, 64 x 32 heads, 256 calls, each side keeping its bf16 state."""
    wl = synth.WORKLOADS["decode_b64_h32_x256"]
    params, tokens, S16, conv = _setup(wl)
    S0, c0 = S16.clone(), conv.clone()
    pairs = synth.sample_heads(wl, 12)
    o = run_calls(wl, params, tokens, S16, conv)
    ref = _oracle_bf16_pairs(params, tokens, S0, c0, pairs)
    for b, h, E, acc, gap in _check_multi(ref, o, S16, conv, pairs):
        print(f"\n  pair {(b, h)}: variant error E {E:.3e}, GPU vs exact {acc:.3e}, vs bf16 oracle {gap:.3e}", end="")


def test_b256_h64_128_calls_sampled():
    """Serving-scale decode (256 x 64 heads, 512 MiB of bf16 state) after 32 warm-up tokens;
    the sampled pairs start from the oracle's own warm-up state on both sides."""
    wl = synth.WORKLOADS["decode_b256_h64_x128"]
    params = synth.make_params(wl, DEV)
    st = synth.make_state(wl, DEV)
    S16, conv = bf16_of(st["S"]), st["conv_state"]
    del st
    warm = synth.make_tokens(wl, DEV, T=wl.warmup_tokens, warm=True)
    pairs = synth.sample_heads(wl, 8)
    S_zero, c_zero = S16.clone(), conv.clone()
    ow = run_calls(wl, params, warm, S16, conv)
    wref = _oracle_bf16_pairs(params, warm, S_zero, c_zero, pairs)
    del S_zero, c_zero
    _check_multi(wref, ow, S16, conv, pairs)   # the warm-up itself
    del ow
    for (b, h) in pairs:
        S16[b, h] = torch.from_numpy(oracle.bf16_round(wref[(b, h)][0].S[0, 0]).view(np.int16)).to(DEV)
        set_pair_window(conv, b, h, wref[(b, h)][0].conv_state)
    tokens = synth.make_tokens(wl, DEV)
    S0, c0 = S16.clone(), conv.clone()
    o = run_calls(wl, params, tokens, S16, conv)
    ref = _oracle_bf16_pairs(params, tokens, S0, c0, pairs)
    for b, h, E, acc, gap in _check_multi(ref, o, S16, conv, pairs):
        print(f"\n  pair {(b, h)}: variant error E {E:.3e}, GPU vs exact {acc:.3e}, vs bf16 oracle {gap:.3e}", end="")
