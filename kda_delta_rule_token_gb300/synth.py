"""Seeded synthetic inputs for the KDA token step (no KDA arithmetic here).

Every tensor is drawn from its own ``torch.Generator`` seeded from the
workload seed and a fixed per-tensor id, on the device the caller names, so
one process can hand bit-identical inputs to both the CUDA library and the
fp64 oracle (copying device tensors to the host for the latter).  ``N(mu, s)``
in the workload descriptions is read with ``s`` the standard deviation.

Workloads are shaped like Kimi K3's KDA layers: d_k = d_v = 128 per head.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

import torch

D = 128

# Fixed per-tensor stream ids: a tensor's values never depend on which other
# tensors were drawn before it.
_IDS = {
    "conv_w": 1, "dt_bias": 2, "A_log": 3, "gamma": 4,
    "q": 10, "k": 11, "v": 12, "z": 13, "beta_logit": 14, "gate_logit": 15,
    "S0": 20, "conv0": 21,
    "x": 30, "W_fa": 31, "W_fb": 32, "W_bp": 33,
    "xh": 40, "W_qkvg": 41, "W_o": 42, "o_in": 43,
}

# Low-rank front-end widths: the pages give none; the hidden width of the
# Kimi K2 / K3 family (7168) and a rank of one head width (128).
LOWRANK_HIDDEN = 7168
LOWRANK_RANK = 128
_WARM_OFFSET = 100


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "decode" (one token per call) or "prefill"
    B: int
    H: int
    T: int               # decode: number of calls; prefill: tokens per sequence
    seed: int
    qkv_bf16: bool = False
    a_log_low: float = -4.0
    s0_std: float = 0.0  # 0 => zero initial state
    win_std: float = 0.0  # 0 => zero initial conv window
    warmup_tokens: int = 0
    chunk: int = 64
    d: int = D

    @property
    def heads(self) -> int:
        return self.B * self.H


WORKLOADS = {
    # Tiny oracle check: 1 sequence, 2 heads, 16 sequential decode steps, fp32.
    "tiny_decode_b1_h2_t16": Workload("tiny_decode_b1_h2_t16", "decode", 1, 2, 16, 0),
    # Batched decode: 64 sequences x 32 heads, 256 calls; fp32 state (128 MiB).
    "decode_b64_h32_x256": Workload("decode_b64_h32_x256", "decode", 64, 32, 256, 1,
                                    s0_std=0.01, win_std=1.0),
    # Single-sequence prefill: 32 heads, 4096 tokens, bf16 q/k/v.
    "prefill_b1_h32_t4096": Workload("prefill_b1_h32_t4096", "prefill", 1, 32, 4096, 2,
                                     qkv_bf16=True),
    # Batched prefill: 8 x 64 heads, 8192 tokens, long-memory channels.
    "prefill_b8_h64_t8192": Workload("prefill_b8_h64_t8192", "prefill", 8, 64, 8192, 3,
                                     qkv_bf16=True, a_log_low=-6.0),
    # Serving-scale decode: 256 x 64 heads (1 GiB state), 128 calls, state from
    # 32 warm-up tokens.
    "decode_b256_h64_x128": Workload("decode_b256_h64_x128", "decode", 256, 64, 128, 4,
                                     warmup_tokens=32),
}
TINY = WORKLOADS["tiny_decode_b1_h2_t16"]


def packed_lengths(n: int = 32, seed: int = 5, lo: float = 8.0, hi: float = 13.0) -> np.ndarray:
    """Sequence lengths of the packed-sequence prefill workload: round(2^U(lo, hi))."""
    rng = np.random.default_rng(seed)
    return np.round(2.0 ** rng.uniform(lo, hi, n)).astype(np.int64)


def packed_workload(lengths) -> "Workload":
    """One token axis of sum(lengths) tokens with the 8 x 64-head prefill recipe
    (bf16 q/k/v, A_log U(-6, 0)); the caller packs sequences along it."""
    return replace(WORKLOADS["prefill_b8_h64_t8192"], B=1, T=int(np.sum(lengths)))


def shrink(wl: Workload, **kw) -> Workload:
    """Same distributions, other sizes (used for small parity cases)."""
    return replace(wl, **kw)


def _gen(wl: Workload, key: str, device, warm: bool = False) -> torch.Generator:
    g = torch.Generator(device=device)
    sid = _IDS[key] + (_WARM_OFFSET if warm else 0)
    g.manual_seed(wl.seed * 1_000_003 + sid)
    return g


def _normal(shape, std, mean, g, device):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def make_params(wl: Workload, device="cpu") -> dict:
    """conv_w [3, H*d, 4] (q, k, v), dt_bias / A_log / gamma [H, d], fp32."""
    H, d = wl.H, wl.d
    conv_w = _normal((3, H * d, 4), 0.25, 0.0, _gen(wl, "conv_w", device), device)
    dt_bias = _normal((H, d), 0.1, 0.0, _gen(wl, "dt_bias", device), device)
    u = torch.rand((H, d), generator=_gen(wl, "A_log", device), device=device,
                   dtype=torch.float32)
    A_log = u * (0.0 - wl.a_log_low) + wl.a_log_low
    gamma = _normal((H, d), 0.1, 1.0, _gen(wl, "gamma", device), device)
    return {"conv_w": conv_w, "dt_bias": dt_bias, "A_log": A_log, "gamma": gamma}


def make_tokens(wl: Workload, device="cpu", T: int | None = None,
                warm: bool = False) -> dict:
    """Per-token inputs.

    decode:  q, k, v, z, gate_logit [T, B, H, d]; beta_logit [T, B, H]  (call-major)
    prefill: q, k, v, z, gate_logit [B, T, H, d]; beta_logit [B, T, H]
    q/k/v are bf16 when the workload says so (round-to-nearest-even from fp32
    normals), everything else fp32.
    """
    T = wl.T if T is None else T
    B, H, d = wl.B, wl.H, wl.d
    if wl.mode == "decode" or warm:
        shp, shb = (T, B, H, d), (T, B, H)
    else:
        shp, shb = (B, T, H, d), (B, T, H)
    out = {}
    for key in ("q", "k", "v"):
        x = _normal(shp, 1.0, 0.0, _gen(wl, key, device, warm), device)
        out[key] = x.to(torch.bfloat16) if (wl.qkv_bf16 and not warm) else x
    out["z"] = _normal(shp, 1.0, 0.0, _gen(wl, "z", device, warm), device)
    out["beta_logit"] = _normal(shb, 1.0, 0.0, _gen(wl, "beta_logit", device, warm), device)
    out["gate_logit"] = _normal(shp, 1.0, 0.0, _gen(wl, "gate_logit", device, warm), device)
    return out


def make_state(wl: Workload, device="cpu") -> dict:
    """Initial S [B, H, d, d] and conv window [B, 3, 3*H*d], fp32."""
    B, H, d = wl.B, wl.H, wl.d
    if wl.s0_std > 0:
        S0 = _normal((B, H, d, d), wl.s0_std, 0.0, _gen(wl, "S0", device), device)
    else:
        S0 = torch.zeros((B, H, d, d), device=device, dtype=torch.float32)
    if wl.win_std > 0:
        c0 = _normal((B, 3, 3 * H * d), wl.win_std, 0.0, _gen(wl, "conv0", device), device)
    else:
        c0 = torch.zeros((B, 3, 3 * H * d), device=device, dtype=torch.float32)
    return {"S": S0, "conv_state": c0}


def sample_heads(wl: Workload, n: int) -> list[tuple[int, int]]:
    """n (sequence, head) pairs spread over the batch, first and last included."""
    total = wl.B * wl.H
    n = min(n, total)
    if n <= 1:
        return [(0, 0)]
    idx = sorted({round(i * (total - 1) / (n - 1)) for i in range(n)})
    return [(p // wl.H, p % wl.H) for p in idx]


def make_lowrank(wl: Workload, device="cpu", hidden: int = LOWRANK_HIDDEN, rank: int = LOWRANK_RANK,
                 T: int | None = None) -> dict:
    """Low-rank front-end weights and hidden inputs, fp32.

    W_fa [rank, hidden] ~ N(0, 1/hidden), W_fb [H*d, rank] ~ N(0, 1/rank),
    W_bp [H, hidden] ~ N(0, 1/hidden) and x ~ N(0, 1), so that z = W_fb W_fa x
    and beta_logit = W_bp x come out about N(0, 1), the distribution the
    workloads give those inputs directly.  x is [T, B, hidden] (call-major)
    for decode workloads and [B, T, hidden] for prefill ones.
    """
    T = wl.T if T is None else T
    H, d = wl.H, wl.d
    W_fa = _normal((rank, hidden), hidden ** -0.5, 0.0, _gen(wl, "W_fa", device), device)
    W_fb = _normal((H * d, rank), rank ** -0.5, 0.0, _gen(wl, "W_fb", device), device)
    W_bp = _normal((H, hidden), hidden ** -0.5, 0.0, _gen(wl, "W_bp", device), device)
    shp = (T, wl.B, hidden) if wl.mode == "decode" else (wl.B, T, hidden)
    x = _normal(shp, 1.0, 0.0, _gen(wl, "x", device), device)
    return {"W_fa": W_fa, "W_fb": W_fb, "W_bp": W_bp, "x": x, "hidden": hidden, "rank": rank}


def make_projections(wl: Workload, device="cpu", hidden: int = LOWRANK_HIDDEN, N: int | None = None) -> dict:
    """Projection weights and inputs, bf16 (round to nearest even).

    W_qkvg [4*H*d, hidden] ~ N(0, 1/hidden) (W_q, W_k, W_v, W_g stacked by
    rows), W_o [hidden, H*d] ~ N(0, 1/(H*d)), x [N, hidden] ~ N(0, 1), so that
    q, k, v and the gate logits come out about N(0, 1) like the workloads'
    direct draws; o_in [N, H, d] ~ N(0, 1) fp32 stands in for the token
    step's output when the output projection is checked alone.  N defaults to
    the workload's tokens per call (B for decode, B*T for prefill).
    """
    H, d = wl.H, wl.d
    HD = H * d
    N = (wl.B if wl.mode == "decode" else wl.B * wl.T) if N is None else N
    W_qkvg = _normal((4 * HD, hidden), hidden ** -0.5, 0.0, _gen(wl, "W_qkvg", device), device).to(torch.bfloat16)
    W_o = _normal((hidden, HD), HD ** -0.5, 0.0, _gen(wl, "W_o", device), device).to(torch.bfloat16)
    x = _normal((N, hidden), 1.0, 0.0, _gen(wl, "xh", device), device).to(torch.bfloat16)
    o_in = _normal((N, H, d), 1.0, 0.0, _gen(wl, "o_in", device), device)
    return {"W_qkvg": W_qkvg, "W_o": W_o, "x": x, "o_in": o_in, "hidden": hidden}
