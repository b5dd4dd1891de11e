"""The chunked (WY/UT) form of the gated delta rule, in plain fp64 numpy, equals
the sequential recurrence of the oracle up to rounding.

This pins the algebra the prefill kernel computes with its tensor-core MMAs,
separately from its tf32 precision (the pages give no chunked algorithm; it is
derived from the recurrence row of "Kimi K3 Metal Gap Analysis", section 2).
Per chunk of C tokens with state S0 and per-channel cumulative decay G_t:

    K_g = k^ e^{G - rho},  Q_g = q^ e^{G - rho},  R = k^ e^{rho - G}
    A'  = strictly_lower(K_g R^T),  P = lower(Q_g R^T)
    U   = (I + Diag(beta) A')^{-1} Diag(beta) (V - K_g e^{rho} S0)
    O   = Q_g e^{rho} S0 + P U
    S   = e^{G_last} S0 + (k^ e^{G_last - G})^T U

for any per-channel rho (the kernel takes G_last / 2, or 0 and G_last on its
exact fallback).  The same form split into a state-independent part for all
chunks (W = Minv Diag(beta) K_g, U' = Minv Diag(beta) V) and a sequential
state pass (U = U' - W e^{rho} S0) is checked too.  Inputs are the oracle's
own conv / norm / decay intermediates, so only the recurrence is restated.
"""
import numpy as np
import pytest

import oracle
from kda_delta_rule_token_gb300 import synth
from harness import np64, pair_params, pair_tokens, pair_window

D = 128


def chunk_recurrence(qh, kh, v, gk, beta, S0, C, rho="half"):
    """o_pre [T, d] and the final S [d, d] by chunks of C tokens."""
    T = qh.shape[0]
    S = S0.copy()
    o = np.zeros((T, D))
    for t0 in range(0, T, C):
        n = min(C, T - t0)
        k, q, vv = kh[t0:t0 + n], qh[t0:t0 + n], v[t0:t0 + n]
        b = beta[t0:t0 + n]
        G = np.cumsum(gk[t0:t0 + n], axis=0)           # [n, d], G_t = sum_{i <= t} gk_i
        Gl = G[-1]
        if rho == "half":
            rl = rr = 0.5 * Gl
        elif rho == "zero":
            rl = rr = np.zeros(D)
        else:                                          # the kernel's exact-fallback split
            rl, rr = np.zeros(D), Gl
        Kg = k * np.exp(G - rl)
        Qg = q * np.exp(G - rl)
        R = k * np.exp(rr - G)
        S0s = np.exp(rl)[:, None] * S                  # Diag(e^rho_L) S0
        A = np.tril(Kg @ (k * np.exp(rl - G)).T, -1)   # A'_{ti} = sum_c k_t k_i e^{G_t - G_i}, i < t
        P = np.tril(Qg @ (k * np.exp(rl - G)).T)       # P_{ti}, i <= t
        M = np.eye(n) + b[:, None] * A
        U = np.linalg.solve(M, b[:, None] * (vv - Kg @ S0s))
        o[t0:t0 + n] = Qg @ S0s + P @ U
        # S_end = e^{G_last - rho_R} (e^{rho_R} S0 + R^T U)
        S = np.exp(Gl - rr)[:, None] * (np.exp(rr)[:, None] * S + R.T @ U)
    return o, S


def chunk_recurrence_wu(qh, kh, v, gk, beta, S0, C):
    """The same chunk form split into a state-independent part, computable for
    every chunk at once (W = Minv Diag(beta) K_g, U' = Minv Diag(beta) V, P),
    and the sequential state pass U = U' - W e^{rho} S0."""
    T = qh.shape[0]
    parts = []
    for t0 in range(0, T, C):                          # independent of the state
        n = min(C, T - t0)
        k, q, vv, b = kh[t0:t0 + n], qh[t0:t0 + n], v[t0:t0 + n], beta[t0:t0 + n]
        G = np.cumsum(gk[t0:t0 + n], axis=0)
        rho = 0.5 * G[-1]
        Kg, Qg, Rm = k * np.exp(G - rho), q * np.exp(G - rho), k * np.exp(rho - G)
        Minv = np.linalg.inv(np.eye(n) + b[:, None] * np.tril(Kg @ Rm.T, -1))
        parts.append((Minv @ (b[:, None] * Kg), Minv @ (b[:, None] * vv), Qg, np.tril(Qg @ Rm.T),
                      Rm, G[-1], rho))
    S = S0.copy()
    o = np.zeros((T, D))
    for c, (W, Up, Qg, P, Rm, Gl, rho) in enumerate(parts):   # sequential over chunks
        S0s = np.exp(rho)[:, None] * S
        U = Up - W @ S0s
        o[c * C:c * C + Qg.shape[0]] = Qg @ S0s + P @ U
        S = np.exp(Gl - rho)[:, None] * (S0s + Rm.T @ U)
    return o, S


def _oracle_case(T, s0_std=0.05, a_log_low=-4.0, seed=2):
    wl = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], B=1, H=2, T=T,
                      s0_std=s0_std, win_std=1.0, seed=seed, a_log_low=a_log_low)
    params = synth.make_params(wl, "cpu")
    tokens = synth.make_tokens(wl, "cpu")
    st = synth.make_state(wl, "cpu")
    out = {}
    for h in range(wl.H):
        tk = pair_tokens(tokens, 0, h, call_major=False)
        S0 = np64(st["S"][0, h])
        r = oracle.run(**tk, **pair_params(params, h), conv_state=pair_window(st["conv_state"], 0, h),
                       S=S0[None, None], intermediates=True)
        out[h] = (r, S0)
    return out


@pytest.mark.parametrize("C", [1, 16, 64])
@pytest.mark.parametrize("rho", ["half", "zero", "fallback"])
def test_chunk_form_equals_sequential(C, rho):
    for h, (r, S0) in _oracle_case(T=150).items():      # two full chunks and a ragged tail at C = 64
        qh, kh, vc = r.qhat[0, :, 0], r.khat[0, :, 0], r.vconv[0, :, 0]
        gk, beta = r.gk[0, :, 0], r.beta[0, :, 0]
        o, S = chunk_recurrence(qh, kh, vc, gk, beta, S0, C, rho)
        ref_o, ref_S = r.o_pre[0, :, 0], r.S[0, 0]
        assert np.max(np.abs(o - ref_o)) <= 1e-11 * np.max(np.abs(ref_o)), (h, C, rho)
        assert np.max(np.abs(S - ref_S)) <= 1e-11 * np.max(np.abs(ref_S)), (h, C, rho)


def test_chunk_form_strong_decay():
    """Long-memory and fast-forgetting channels together (A_log up to 0 on
    z ~ N(0, 1)): the chunk's decay spans tens of nats, as in the batched
    prefill; the fallback split keeps every factor <= 1."""
    for h, (r, S0) in _oracle_case(T=130, a_log_low=-6.0, seed=3).items():
        qh, kh, vc = r.qhat[0, :, 0], r.khat[0, :, 0], r.vconv[0, :, 0]
        gk, beta = r.gk[0, :, 0], r.beta[0, :, 0]
        for rho in ("half", "fallback"):
            o, S = chunk_recurrence(qh, kh, vc, gk, beta, S0, 64, rho)
            assert np.max(np.abs(o - r.o_pre[0, :, 0])) <= 1e-10 * np.max(np.abs(r.o_pre[0, :, 0]))
            assert np.max(np.abs(S - r.S[0, 0])) <= 1e-10 * np.max(np.abs(r.S[0, 0]))


def test_state_independent_split_equals_sequential():
    """W and U' of every chunk first, the state pass after: same result."""
    for h, (r, S0) in _oracle_case(T=150).items():
        o, S = chunk_recurrence_wu(r.qhat[0, :, 0], r.khat[0, :, 0], r.vconv[0, :, 0],
                                   r.gk[0, :, 0], r.beta[0, :, 0], S0, 64)
        assert np.max(np.abs(o - r.o_pre[0, :, 0])) <= 1e-11 * np.max(np.abs(r.o_pre[0, :, 0]))
        assert np.max(np.abs(S - r.S[0, 0])) <= 1e-11 * np.max(np.abs(r.S[0, 0]))
