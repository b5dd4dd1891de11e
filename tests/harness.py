"""Test helpers: run the fp64 oracle on chosen (sequence, head) pairs of a
workload and compare against the CUDA library's outputs.

Inputs always come from ``kda_delta_rule_token_gb300.synth`` (one process,
one device), so both sides see the same bytes; outputs of the CUDA library
are only ever compared, never fed to the oracle.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle

D = 128


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def max_rel_err(x, r) -> float:
    """max |x - r| / max |r| (the decode tolerance measure)."""
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    den = np.max(np.abs(r))
    return float(np.max(np.abs(x - r)) / den) if den > 0 else float(np.max(np.abs(x)))


def rel_l2(x, r) -> float:
    """||x - r||_2 / ||r||_2 (the prefill tolerance measure)."""
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    den = np.linalg.norm(r)
    return float(np.linalg.norm(x - r) / den) if den > 0 else float(np.linalg.norm(x))


def pair_params(params: dict, h: int) -> dict:
    """Parameters of one head as an H = 1 layer (float64 numpy)."""
    H = params["dt_bias"].shape[0]
    cw = params["conv_w"].reshape(3, H, D, 4)[:, h]
    return {"conv_w": np64(cw.reshape(3, D, 4)), "dt_bias": np64(params["dt_bias"][h:h + 1]),
            "A_log": np64(params["A_log"][h:h + 1]), "gamma": np64(params["gamma"][h:h + 1])}


def pair_window(conv_state: torch.Tensor, b: int, h: int) -> np.ndarray:
    """[1, 3, 3*d] window of (b, h) out of a [B, 3, 3*H*d] tensor."""
    B, _, C = conv_state.shape
    H = C // (3 * D)
    w = conv_state[b].reshape(3, 3, H, D)[:, :, h]       # [tap, tensor, d]
    return np64(w.reshape(1, 3, 3 * D))


def set_pair_window(conv_state: torch.Tensor, b: int, h: int, w: np.ndarray):
    B, _, C = conv_state.shape
    H = C // (3 * D)
    view = conv_state[b].view(3, 3, H, D)
    view[:, :, h] = torch.as_tensor(w.reshape(3, 3, D), dtype=conv_state.dtype,
                                    device=conv_state.device)


def pair_tokens(tokens: dict, b: int, h: int, call_major: bool) -> dict:
    """Per-token inputs of (b, h) as [1, T, 1, d] / [1, T, 1] float64."""
    out = {}
    for key in ("q", "k", "v", "z", "gate_logit"):
        x = tokens[key][:, b, h] if call_major else tokens[key][b, :, h]
        out[key] = np64(x)[None, :, None, :]
    x = tokens["beta_logit"][:, b, h] if call_major else tokens["beta_logit"][b, :, h]
    out["beta_logit"] = np64(x)[None, :, None]
    return out


def oracle_pairs(params, tokens, S0, conv0, pairs, *, call_major, l2_eps=1e-6, rms_eps=1e-6,
                 workers=None):
    """Run the oracle for each (b, h) in ``pairs`` (threads across pairs).

    Returns {pair: OracleOut} with o/o_pre of shape [1, T, 1, d] and S [1, 1, d, d].
    S0 / conv0 are the initial device or host tensors of the whole batch.
    """
    workers = workers or max(1, min(len(pairs), os.cpu_count() or 1))

    def one(pair):
        b, h = pair
        tk = pair_tokens(tokens, b, h, call_major)
        return pair, oracle.run(**tk, **pair_params(params, h),
                                conv_state=pair_window(conv0, b, h),
                                S=np64(S0[b, h])[None, None], l2_eps=l2_eps, rms_eps=rms_eps)

    with cf.ThreadPoolExecutor(workers) as ex:
        return dict(ex.map(one, pairs))


POISON = 0x7FADBEEF          # a quiet NaN with a payload no computation produces
GUARD_BYTES = 4096


class Guarded:
    """A float32 tensor placed inside a larger device buffer whose margins
    (GUARD_BYTES before and after) hold the NaN pattern POISON.

    ``t`` is the interior view (contiguous, 16-byte aligned: torch buffers
    are 256-byte aligned and the margin is a multiple of 16 bytes);
    ``intact()`` says whether every margin word still holds the pattern bit
    for bit, i.e. no kernel wrote outside the tensor it was given.
    """

    def __init__(self, like: torch.Tensor):
        assert like.dtype == torch.float32 and like.is_contiguous()
        n, m = like.numel(), GUARD_BYTES // 4
        self.m = m
        self.buf = torch.empty(n + 2 * m, dtype=torch.float32, device=like.device)
        self.buf.view(torch.int32).fill_(POISON)
        self.t = self.buf[m:m + n].view(like.shape)
        self.t.copy_(like)

    def intact(self) -> bool:
        w = self.buf.view(torch.int32)
        return bool((w[:self.m] == POISON).all()) and bool((w[-self.m:] == POISON).all())
