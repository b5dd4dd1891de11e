"""Pins for the fp64 oracle: facts fixed by the sources and by mathematics.

Each ``pin_*`` takes the path of an oracle build (None = the real one) and
raises AssertionError when the oracle breaks the fact.  The same functions
run against mutated builds of the oracle in ``test_oracle_mutants.py`` to show
that a plausible slip (dropped term, wrong sign, wrong index, transposed
operand) is caught by at least one of them.

Sources: "Kimi K3 Metal Gap Analysis" section 2 "KDA Attention" (rows Conv4 +
SiLU, L2 normalize q/k, Decay compute, Recurrence, O projection) and "Metal
(Apple GPU) backend for Kimi K3" section "Correctness" (token-0 zero-state
identity o / (v * beta) = q_hat . k_hat) and table "What runs where (per
layer)" (the low-rank fa, fb, bp matmuls feeding the decay and beta, and
the q, k, v, g, o projections).
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import expit

import oracle

D = 128


def _inputs(seed, B=1, T=4, H=2, d=D, s0=0.0, win=0.0):
    rng = np.random.default_rng(seed)
    n = rng.standard_normal
    return dict(
        q=n((B, T, H, d)), k=n((B, T, H, d)), v=n((B, T, H, d)), z=n((B, T, H, d)),
        beta_logit=n((B, T, H)), gate_logit=n((B, T, H, d)),
        conv_w=0.25 * n((3, H * d, 4)), dt_bias=0.1 * n((H, d)),
        A_log=rng.uniform(-4.0, 0.0, (H, d)), gamma=1.0 + 0.1 * n((H, d)),
        conv_state=win * n((B, 3, 3 * H * d)), S=s0 * n((B, H, d, d)))


def _run(inp, lib_path, **kw):
    return oracle.run(**inp, lib_path=lib_path, **kw)


def _silu(x):
    return x * expit(x)


def pin_token0_identity(lib_path=None):
    """Zero state and window: o_pre = beta * v_conv * (q_hat . k_hat) and
    S_1 = beta k_hat v_conv^T ("Correctness", token-0 zero-state check)."""
    inp = _inputs(101, T=1, H=3)
    out = _run(inp, lib_path, intermediates=True)
    H = 3
    for h in range(H):
        qh, kh, vc = out.qhat[0, 0, h], out.khat[0, 0, h], out.vconv[0, 0, h]
        beta = out.beta[0, 0, h]
        qk = float(qh @ kh)
        np.testing.assert_allclose(out.o_pre[0, 0, h], beta * vc * qk, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(out.S[0, h], beta * np.outer(kh, vc), rtol=1e-12, atol=1e-16)
    # With a zero window the conv keeps only the current-token tap.
    w3 = inp["conv_w"][..., 3]                       # [3, H*d]
    x = np.stack([inp["q"][0, 0], inp["k"][0, 0], inp["v"][0, 0]]).reshape(3, -1)
    y = _silu(w3 * x).reshape(3, H, D)
    np.testing.assert_allclose(out.vconv[0, 0], y[2], rtol=1e-13, atol=1e-15)
    for i, got in ((0, out.qhat), (1, out.khat)):
        ref = y[i] / np.sqrt((y[i] ** 2).sum(-1, keepdims=True) + 1e-6)
        np.testing.assert_allclose(got[0, 0], ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(out.beta[0, 0], expit(inp["beta_logit"][0, 0]), rtol=1e-14)


def pin_identity_when_no_write_no_decay(lib_path=None):
    """beta = 0 (logit -inf) and gk = 0 (A_log = -inf) leave S exactly unchanged."""
    inp = _inputs(102, T=5, s0=0.3, win=1.0)
    inp["beta_logit"][:] = -np.inf
    inp["A_log"][:] = -np.inf
    out = _run(inp, lib_path, intermediates=True)
    assert np.array_equal(out.S, inp["S"]), "state moved with beta = 0 and gk = 0"
    assert np.all(out.gk == 0.0) and np.all(out.beta == 0.0)


def pin_decay_only_closed_form(lib_path=None):
    """beta = 0 and softplus(z + dt_bias) = 1 (z + dt_bias = ln(e - 1)) with
    A_log = ln c per channel: gk = -c, and S_T = Diag(exp(-T c)) S_0."""
    T = 7
    inp = _inputs(103, T=T, s0=1.0, win=1.0)
    rng = np.random.default_rng(7)
    c = rng.uniform(0.01, 1.0, inp["A_log"].shape)
    inp["A_log"] = np.log(c)
    inp["beta_logit"][:] = -np.inf
    inp["z"] = np.broadcast_to(math.log(math.e - 1.0) - inp["dt_bias"], inp["z"].shape).copy()
    out = _run(inp, lib_path, intermediates=True)
    np.testing.assert_allclose(out.gk, np.broadcast_to(-c, out.gk.shape), rtol=1e-12)
    ref = inp["S"] * np.exp(-T * c)[None, :, :, None]
    np.testing.assert_allclose(out.S, ref, rtol=1e-11, atol=0)


def pin_delta_rule_write(lib_path=None):
    """With ||k_hat|| = 1 (l2_eps = 0): S_new^T k_hat = (1 - beta) S'^T k_hat
    + beta v_conv, S' = Diag(e^gk) S; beta = 1 and gk = 0 give exactly v_conv."""
    inp = _inputs(104, T=1, s0=0.5, win=1.0)
    inp["A_log"][:] = -np.inf
    inp["beta_logit"][:] = np.inf
    out = _run(inp, lib_path, intermediates=True, l2_eps=0.0)
    for h in range(2):
        kh, vc = out.khat[0, 0, h], out.vconv[0, 0, h]
        np.testing.assert_allclose(out.S[0, h].T @ kh, vc, rtol=1e-11, atol=1e-12)
    inp = _inputs(105, T=1, s0=0.5, win=1.0)
    out = _run(inp, lib_path, intermediates=True, l2_eps=0.0)
    for h in range(2):
        kh, vc, b = out.khat[0, 0, h], out.vconv[0, 0, h], out.beta[0, 0, h]
        a = np.exp(out.gk[0, 0, h])
        Sp = a[:, None] * inp["S"][0, h]
        np.testing.assert_allclose(out.S[0, h].T @ kh, (1 - b) * (Sp.T @ kh) + b * vc,
                                   rtol=1e-11, atol=1e-12)


def pin_bruteforce_products(lib_path=None):
    """T <= 4: S_T = M_T...M_1 S_0 + sum_t M_T...M_{t+1} beta_t k_t v_t^T with
    dense M_t = (I - beta_t k_t k_t^T) Diag(e^{gk_t}); o_pre_t = S_t^T q_t."""
    T, H = 4, 2
    inp = _inputs(106, T=T, H=H, s0=0.2, win=1.0)
    out = _run(inp, lib_path, intermediates=True)
    I = np.eye(D)
    for h in range(H):
        k = out.khat[0, :, h]
        q = out.qhat[0, :, h]
        v = out.vconv[0, :, h]
        a = np.exp(out.gk[0, :, h])
        b = out.beta[0, :, h]
        M = [(I - b[t] * np.outer(k[t], k[t])) @ np.diag(a[t]) for t in range(T)]
        for tt in range(1, T + 1):
            P = I.copy()
            for t in range(tt):
                P = M[t] @ P
            St = P @ inp["S"][0, h]
            for t in range(tt):
                Pt = I.copy()
                for s in range(t + 1, tt):
                    Pt = M[s] @ Pt
                St = St + Pt @ (b[t] * np.outer(k[t], v[t]))
            np.testing.assert_allclose(out.o_pre[0, tt - 1, h], St.T @ q[tt - 1],
                                       rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(out.S[0, h], St, rtol=1e-9, atol=1e-12)


def pin_conv_one_hot_tap(lib_path=None):
    """Tap weights e_3 (current token only): v_conv_t = SiLU(v_t) whatever the
    window holds; q_hat_t = SiLU(q_t) / ||SiLU(q_t)|| (l2_eps = 0)."""
    inp = _inputs(107, T=5, win=3.0)
    inp["conv_w"][:] = 0.0
    inp["conv_w"][..., 3] = 1.0
    out = _run(inp, lib_path, intermediates=True, l2_eps=0.0)
    np.testing.assert_allclose(out.vconv, _silu(inp["v"]), rtol=1e-13, atol=1e-15)
    y = _silu(inp["q"])
    np.testing.assert_allclose(out.qhat, y / np.linalg.norm(y, axis=-1, keepdims=True),
                               rtol=1e-12, atol=1e-15)


def pin_conv_impulse(lib_path=None):
    """Unit impulse at t = 0 on v through a zero window: v_conv_t = SiLU(w[3 - t])
    for t <= 3 and 0 afterwards (causal, width 4, newest tap last)."""
    T, H = 6, 2
    inp = _inputs(108, T=T, H=H)
    inp["v"][:] = 0.0
    inp["v"][:, 0] = 1.0
    out = _run(inp, lib_path, intermediates=True)
    w = inp["conv_w"][2].reshape(H, D, 4)
    for t in range(T):
        ref = _silu(w[..., 3 - t]) if t <= 3 else np.zeros((H, D))
        np.testing.assert_allclose(out.vconv[0, t], ref, rtol=1e-13, atol=1e-300)


def pin_window_continuity(lib_path=None):
    """Running 8 tokens in one call equals 3 then 5 tokens with the state and
    window carried over; the window ends as the last 3 raw inputs."""
    inp = _inputs(109, T=8, s0=0.1, win=1.0)
    full = _run(inp, lib_path)
    a = {k: (v[:, :3] if v.ndim >= 2 and v.shape[:2] == (1, 8) else v) for k, v in inp.items()}
    first = _run(a, lib_path)
    b = {k: (v[:, 3:] if v.ndim >= 2 and v.shape[:2] == (1, 8) else v) for k, v in inp.items()}
    b["S"], b["conv_state"] = first.S, first.conv_state
    second = _run(b, lib_path)
    assert np.array_equal(second.S, full.S)
    assert np.array_equal(second.conv_state, full.conv_state)
    assert np.array_equal(np.concatenate([first.o, second.o], axis=1), full.o)
    raw = np.stack([inp["q"], inp["k"], inp["v"]], axis=2)   # [B, T, 3, H, d]
    last3 = raw[0, -3:].reshape(3, -1)                          # oldest first
    assert np.array_equal(full.conv_state[0], last3)
    # Two tokens: the oldest saved input moves to the front.
    two = {k: (v[:, :2] if v.ndim >= 2 and v.shape[:2] == (1, 8) else v) for k, v in inp.items()}
    o2 = _run(two, lib_path)
    assert np.array_equal(o2.conv_state[0, 0], inp["conv_state"][0, 2])
    assert np.array_equal(o2.conv_state[0, 1:], raw[0, :2].reshape(2, -1))


def pin_l2_norm(lib_path=None):
    """||q_hat||^2 = s / (s + eps) with s = ||conv output||^2 (one-hot taps)."""
    eps = 10.0
    inp = _inputs(110, T=3)
    inp["conv_w"][:] = 0.0
    inp["conv_w"][..., 3] = 1.0
    out = _run(inp, lib_path, intermediates=True, l2_eps=eps)
    for name, x in (("qhat", inp["q"]), ("khat", inp["k"])):
        s = (_silu(x) ** 2).sum(-1)
        n2 = (getattr(out, name) ** 2).sum(-1)
        np.testing.assert_allclose(n2, s / (s + eps), rtol=1e-12)


def pin_rmsnorm_gate_gamma(lib_path=None):
    """Head RMSNorm: with gate -> 1, o_j / (gamma_j o_pre_j) is one constant per
    head equal to 1/sqrt(mean(o_pre^2) + eps); o is linear in gamma and a zero
    gate logit halves it."""
    eps = 0.05
    inp = _inputs(111, T=3, s0=0.2, win=1.0)
    inp["gate_logit"][:] = np.inf
    out = _run(inp, lib_path, rms_eps=eps)
    ms = (out.o_pre ** 2).mean(-1, keepdims=True)
    np.testing.assert_allclose(out.o, inp["gamma"] * out.o_pre / np.sqrt(ms + eps), rtol=1e-12)
    inp2 = dict(inp, gamma=2.0 * inp["gamma"])
    np.testing.assert_allclose(_run(inp2, lib_path, rms_eps=eps).o, 2.0 * out.o, rtol=1e-14)
    inp3 = dict(inp, gate_logit=np.zeros_like(inp["gate_logit"]))
    np.testing.assert_allclose(_run(inp3, lib_path, rms_eps=eps).o, 0.5 * out.o, rtol=1e-14)


def pin_contraction_bound(lib_path=None):
    """(I - beta k k^T) has eigenvalues {1 - beta, 1}, e^gk <= 1: ||S_t||_F <=
    ||S_0||_F + sum_t beta_t ||v_conv_t||."""
    inp = _inputs(112, T=16, s0=0.3, win=1.0)
    out = _run(inp, lib_path, intermediates=True)
    for h in range(2):
        bound = np.linalg.norm(inp["S"][0, h]) + np.sum(
            out.beta[0, :, h] * np.linalg.norm(out.vconv[0, :, h], axis=-1))
        assert np.linalg.norm(out.S[0, h]) <= bound * (1 + 1e-12)


def pin_decay_values(lib_path=None):
    """Closed-form decay values: gk = -exp(A_log) * ln(1 + e^(z + dt_bias))."""
    inp = _inputs(113, T=3, H=1)
    inp["dt_bias"][:] = 0.0
    inp["A_log"][0, :64] = 0.0
    inp["A_log"][0, 64:] = math.log(0.5)
    zs = [0.0, 40.0, -40.0]
    for t, zv in enumerate(zs):
        inp["z"][0, t] = zv
    out = _run(inp, lib_path, intermediates=True)
    for t, zv in enumerate(zs):
        sp = zv + math.log1p(math.exp(-zv)) if zv > 0 else math.log1p(math.exp(zv))
        np.testing.assert_allclose(out.gk[0, t, 0, :64], -sp, rtol=1e-13)
        np.testing.assert_allclose(out.gk[0, t, 0, 64:], -0.5 * sp, rtol=1e-13)
    inp["beta_logit"][0, :, 0] = [0.0, math.log(3.0), -math.log(3.0)]
    out = _run(inp, lib_path, intermediates=True)
    np.testing.assert_allclose(out.beta[0, :, 0], [0.5, 0.75, 0.25], rtol=1e-14)


def _lowrank_inputs(seed, N=5, hidden=40, rank=6, H=3):
    rng = np.random.default_rng(seed)
    n = rng.standard_normal
    return dict(x=n((N, hidden)), W_fa=n((rank, hidden)) / math.sqrt(hidden),
                W_fb=n((H * D, rank)) / math.sqrt(rank), W_bp=n((H, hidden)) / math.sqrt(hidden))


def pin_lowrank_one_hot(lib_path=None):
    """Low-rank front-end ("What runs where (per layer)", row "KDA low-rank
    (fa,fb,bp)"; "Decay compute" row, z = W_fb W_fa x): a single nonzero
    weight in each matrix routes one input value to one output.  With
    W_fa = e_2 e_17^T, W_fb = 3 e_(1*d+5) e_2^T and W_bp = -2 e_2 e_9^T, the
    only nonzero outputs are z[head 1, channel 5] = 3 x_17 and
    beta_logit[head 2] = -2 x_9, exactly."""
    inp = _lowrank_inputs(301)
    N, hidden = inp["x"].shape
    W_fa = np.zeros_like(inp["W_fa"]); W_fa[2, 17] = 1.0
    W_fb = np.zeros_like(inp["W_fb"]); W_fb[1 * D + 5, 2] = 3.0
    W_bp = np.zeros_like(inp["W_bp"]); W_bp[2, 9] = -2.0
    z, bl = oracle.lowrank(inp["x"], W_fa, W_fb, W_bp, H=3, lib_path=lib_path)
    ez = np.zeros((N, 3, D)); ez[:, 1, 5] = 3.0 * inp["x"][:, 17]
    eb = np.zeros((N, 3)); eb[:, 2] = -2.0 * inp["x"][:, 9]
    assert np.array_equal(z, ez) and np.array_equal(bl, eb)


def pin_lowrank_zero_fa(lib_path=None):
    """W_fa = 0 makes z = 0 whatever W_fb and x are; beta_logit does not
    depend on W_fa (the same with W_fa random)."""
    inp = _lowrank_inputs(302)
    z0, b0 = oracle.lowrank(inp["x"], np.zeros_like(inp["W_fa"]), inp["W_fb"], inp["W_bp"], H=3,
                            lib_path=lib_path)
    z1, b1 = oracle.lowrank(inp["x"], inp["W_fa"], inp["W_fb"], inp["W_bp"], H=3, lib_path=lib_path)
    assert np.array_equal(z0, np.zeros_like(z0))
    assert np.array_equal(b0, b1) and np.abs(z1).max() > 0


def pin_lowrank_rank_and_linearity(lib_path=None):
    """z is a linear map of x of rank at most `rank`: z(a x1 + b x2) =
    a z(x1) + b z(x2) to rounding, and the z of 40 tokens span exactly `rank`
    dimensions (W_fb W_fa has rank `rank` for generic weights); beta_logit is
    linear in x too."""
    inp = _lowrank_inputs(303, N=40)
    rank = inp["W_fa"].shape[0]
    x1, x2 = inp["x"][:20], inp["x"][20:]
    f = lambda x: oracle.lowrank(x, inp["W_fa"], inp["W_fb"], inp["W_bp"], H=3, lib_path=lib_path)
    (z1, b1), (z2, b2), (z3, b3) = f(x1), f(x2), f(0.5 * x1 - 2.0 * x2)
    np.testing.assert_allclose(z3, 0.5 * z1 - 2.0 * z2, rtol=0, atol=1e-12 * np.abs(z1).max())
    np.testing.assert_allclose(b3, 0.5 * b1 - 2.0 * b2, rtol=0, atol=1e-12 * np.abs(b1).max())
    zs, _ = f(inp["x"])
    sv = np.linalg.svd(zs.reshape(40, -1), compute_uv=False)
    assert sv[rank - 1] > 1e-6 * sv[0] and sv[rank] < 1e-10 * sv[0]


def pin_project_one_hot_and_linearity(lib_path=None):
    """Projections ("What runs where (per layer)", row "KDA projections
    (q,k,v,g,o)"; "O projection" row): y = W x.  A single nonzero weight
    W[i][j] = c routes c x_j to output i alone (exactly), and y is linear in
    x and in W (to rounding)."""
    rng = np.random.default_rng(401)
    N, n_in, n_out = 6, 24, 10
    x = rng.standard_normal((N, n_in))
    W = np.zeros((n_out, n_in)); W[7, 3] = -1.5
    y = oracle.project(x, W, lib_path=lib_path)
    e = np.zeros((N, n_out)); e[:, 7] = -1.5 * x[:, 3]
    assert np.array_equal(y, e)
    W1, W2 = rng.standard_normal((n_out, n_in)), rng.standard_normal((n_out, n_in))
    x2 = rng.standard_normal((N, n_in))
    f = lambda xx, ww: oracle.project(xx, ww, lib_path=lib_path)
    y1 = f(x, W1)
    tol = 1e-12 * np.abs(y1).max()
    np.testing.assert_allclose(f(2.0 * x - x2, W1), 2.0 * y1 - f(x2, W1), rtol=0, atol=tol)
    np.testing.assert_allclose(f(x, W1 + 3.0 * W2), y1 + 3.0 * f(x, W2), rtol=0, atol=10 * tol)


def pin_project_orthogonal(lib_path=None):
    """With W orthogonal (from a QR factorisation) the projection keeps
    every token's norm, and W^T applied to y gives x back."""
    rng = np.random.default_rng(402)
    Q, _ = np.linalg.qr(rng.standard_normal((16, 16)))
    x = rng.standard_normal((5, 16))
    y = oracle.project(x, Q, lib_path=lib_path)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    np.testing.assert_allclose(oracle.project(y, Q.T.copy(), lib_path=lib_path), x, rtol=0, atol=1e-12)


# ---- bfloat16 state storage -------------------------------------------------
# bfloat16 = IEEE binary32's sign and 8 exponent bits with 7 stored fraction
# bits: normal values m * 2^(E-7), m in [128, 255], E in [-126, 127];
# subnormals m * 2^-133, m in [0, 127]; pattern = upper half of the binary32
# pattern.  Rounding to nearest, ties to the even m, overflow to infinity.

_BF16_TABLE = [   # (value, pattern), each worked out from the format by hand
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -7, 0x3F81),                  # next value above 1
    (1.0 + 2.0 ** -8, 0x3F80),                  # tie between m = 128 and 129: even 128
    (1.0 + 3 * 2.0 ** -8, 0x3F82),              # tie between m = 129 and 130: even 130
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),     # just above the tie
    (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
    (2.0 - 2.0 ** -9, 0x4000),                  # rounds up across the exponent: 2.0
    (-2.5, 0xC020),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (2.0 ** -126, 0x0080),                      # smallest normal
    (2.0 ** -133, 0x0001),                      # smallest subnormal
    (2.0 ** -134, 0x0000),                      # tie between 0 and 2^-133: even 0
    (3 * 2.0 ** -134, 0x0002),                  # tie between m = 1 and 2: even 2
    (127 * 2.0 ** -133 + 2.0 ** -134, 0x0080),  # tie between m = 127 and 128: even 128
    ((2.0 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),   # largest finite
    ((2.0 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),   # tie between largest (m odd) and 2^128: infinity
    (-1e39, 0xFF80),
]


def pin_bf16_round_table(lib_path=None):
    """Rounding to bfloat16 at ties, carries, subnormals and overflow,
    against values worked out from the format's definition."""
    vals = np.array([v for v, _ in _BF16_TABLE])
    want = np.array([b for _, b in _BF16_TABLE], dtype=np.uint16)
    got = oracle.bf16_round(vals, lib_path=lib_path)
    assert np.array_equal(got, want), [(v, hex(g), hex(w)) for v, g, w in zip(vals, got, want) if g != w]
    finite = want[(want & 0x7F80) != 0x7F80]
    back = oracle.bf16_value(finite, lib_path=lib_path)
    assert np.array_equal(oracle.bf16_round(back, lib_path=lib_path), finite)   # values round to themselves


def pin_bf16_round_matches_library(lib_path=None):
    """On binary32 inputs (exact in double) the rounding equals the
    library's float32 -> bfloat16 conversion (round to nearest even), across
    normal, subnormal and near-overflow magnitudes."""
    import torch
    rng = np.random.default_rng(501)
    bits = rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    got = oracle.bf16_round(f.astype(np.float64), lib_path=lib_path)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref), int((got != ref).sum())
    assert np.array_equal(oracle.bf16_value(got, lib_path=lib_path),
                          torch.from_numpy(ref.view(np.int16).copy()).view(torch.bfloat16).double().numpy())


def pin_bf16_state_halving(lib_path=None):
    """bfloat16 state storage, beta = 0 and a = e^gk = 1/2 exactly (A_log =
    z = dt_bias = 0: gk = -softplus(0) = -ln 2): every token halves the
    state and stores the rounding, so subnormal states walk down their own
    sequences with ties to even (3 -> 2 -> 1 -> 0, 7 -> 4 -> 2 -> 1 units of
    2^-133), while normal values halve exactly.  Without bfloat16 storage
    the same run gives S0 * 2^-T exactly."""
    T, H = 4, 1
    inp = _inputs(503, T=T, H=H)
    inp["beta_logit"] = np.full((1, T, H), -np.inf)
    inp["A_log"] = np.zeros((H, D))
    inp["dt_bias"] = np.zeros((H, D))
    inp["z"] = np.zeros((1, T, H, D))
    S0 = np.zeros((1, H, D, D))
    unit = 2.0 ** -133
    S0[0, 0, 0, :4] = np.array([3, 5, 6, 7]) * unit
    S0[0, 0, 1, :3] = [1.0, -0.75, 2.0 ** -120]
    inp["S"] = S0
    walk = {3: [2, 1, 0, 0], 5: [2, 1, 0, 0], 6: [3, 2, 1, 0], 7: [4, 2, 1, 0]}
    for t in range(1, T + 1):
        step = dict(inp, q=inp["q"][:, :t], k=inp["k"][:, :t], v=inp["v"][:, :t], z=inp["z"][:, :t],
                    beta_logit=inp["beta_logit"][:, :t], gate_logit=inp["gate_logit"][:, :t])
        Sb = _run(step, lib_path, state_bf16=True).S[0, 0]
        np.testing.assert_array_equal(Sb[0, :4], [walk[m][t - 1] * unit for m in (3, 5, 6, 7)])
        np.testing.assert_array_equal(Sb[1, :3], np.array([1.0, -0.75, 2.0 ** -120]) * 2.0 ** -t)
        assert not Sb[2:].any() and not Sb[:2, 4:].any()
        Sf = _run(step, lib_path).S[0, 0]
        np.testing.assert_array_equal(Sf, S0[0, 0] * 2.0 ** -t)


def pin_bf16_state_readout_unrounded(lib_path=None):
    """bfloat16 state storage keeps the read-out of the token on the new
    state as computed: from a zero state and window, o_pre = beta v_conv
    (q_hat . k_hat) to double rounding, while the stored S_1 is the
    bfloat16 rounding of beta k_hat v_conv^T."""
    inp = _inputs(505, T=1, H=2)
    full = _run(inp, lib_path, intermediates=True)
    out = _run(inp, lib_path, intermediates=True, state_bf16=True)
    for h in range(2):
        qh, kh, vc = out.qhat[0, 0, h], out.khat[0, 0, h], out.vconv[0, 0, h]
        beta = out.beta[0, 0, h]
        np.testing.assert_allclose(out.o_pre[0, 0, h], beta * vc * float(qh @ kh), rtol=1e-12, atol=1e-15)
        want = oracle.bf16_value(oracle.bf16_round(full.S[0, h], lib_path=lib_path), lib_path=lib_path)
        np.testing.assert_array_equal(out.S[0, h], want)
        assert not np.array_equal(out.S[0, h], full.S[0, h])   # the rounding did happen


PINS = [pin_token0_identity, pin_identity_when_no_write_no_decay, pin_decay_only_closed_form,
        pin_delta_rule_write, pin_bruteforce_products, pin_conv_one_hot_tap, pin_conv_impulse,
        pin_window_continuity, pin_l2_norm, pin_rmsnorm_gate_gamma, pin_contraction_bound,
        pin_decay_values, pin_lowrank_one_hot, pin_lowrank_zero_fa, pin_lowrank_rank_and_linearity,
        pin_project_one_hot_and_linearity, pin_project_orthogonal, pin_bf16_round_table,
        pin_bf16_round_matches_library, pin_bf16_state_halving, pin_bf16_state_readout_unrounded]
