"""Projections (kda_project_qkvg, kda_project_o) vs the fp64 oracle (GPU).

The products run on tensor cores with bf16 operands and fp32 accumulation.
Tolerances, from that arithmetic:
* fp32 outputs of bf16-exact inputs (gate logits; q, k, v in the decode
  format): max|x - r| / max|r| <= 5e-5 per output tensor.  The products are
  exact; the tensor core adds each group of 16 of them and the group sums
  into the fp32 accumulator, each addition truncating to fp32 (relative
  error up to 2^-23, always towards zero, so the errors add up): at
  K = 7168 that is 448 additions, at most about 448 * 2^-23 = 5.3e-5 of the
  accumulator's scale (measured 8e-6);
* bf16 outputs (q, k, v in the prefill format) are that result rounded to
  nearest even: each element within one bf16 step of the exact value,
  |x - r| <= 2^-8 |r| + 5e-5 max|r|;
* the output projection rounds o to bf16 first: against the oracle's product
  of that rounded o, max-rel <= 5e-5 (the same accumulation bound); against
  the unrounded o, the bf16 rounding itself, RMS relative error 2^-8 /
  sqrt(12) times the mean of 1/mantissa (about 1.6e-3 for normal inputs),
  must stay within rel-L2 2.5e-3.
The cases span the token tiles 32, 64, 128 and 256 (rings of 8, 8, 6 and 4
stages) and K ranges shorter than the ring.
"""
import numpy as np
import pytest
import torch

import kda_delta_rule_token_gb300 as kda
from kda_delta_rule_token_gb300 import synth
import oracle
from harness import Guarded, max_rel_err, np64, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_delta_rule_token_gb300 import build
    build.build()
    kda.load()


def _ctx(wl, pr):
    p = synth.make_params(wl, DEV)
    ctx = kda.kda_create(wl.H, p["conv_w"], p["dt_bias"], p["A_log"], p["gamma"])
    kda.kda_bind_projections(ctx, pr["hidden"], pr["W_qkvg"].view(torch.int16), pr["W_o"].view(torch.int16))
    return ctx


def _wl(N, H):
    return synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=N, H=H, T=1)


@pytest.mark.parametrize("N,hidden,H", [(5, 128, 2), (300, 256, 3), (64, 7168, 32), (1000, 384, 1), (100, 512, 2)])
@pytest.mark.parametrize("qkv_f32", [False, True])
def test_project_qkvg_matches_oracle(N, hidden, H, qkv_f32):
    wl = _wl(N, H)
    pr = synth.make_projections(wl, DEV, hidden=hidden)
    HD = H * 128
    ctx = _ctx(wl, pr)
    dt = torch.float32 if qkv_f32 else torch.bfloat16
    try:
        gq, gk, gv = (Guarded(torch.zeros((N, HD), device=DEV)) for _ in range(3)) if qkv_f32 else (None,) * 3
        if qkv_f32:
            q, k, v = gq.t, gk.t, gv.t
        else:
            q, k, v = (torch.zeros((N, HD), device=DEV, dtype=dt) for _ in range(3))
        gg = Guarded(torch.zeros((N, HD), device=DEV))
        kda.kda_project_qkvg(ctx, N, pr["x"].view(torch.int16), q, k, v, gg.t, qkv_f32=qkv_f32)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
        assert gg.intact() and all(g is None or g.intact() for g in (gq, gk, gv)), "a guard region was written"
    finally:
        kda.kda_destroy(ctx)
    ref = oracle.project(np64(pr["x"]), np64(pr["W_qkvg"]))          # [N, 4 HD]
    eg = max_rel_err(np64(gg.t), ref[:, 3 * HD:])
    assert eg <= 5e-5, f"gate logits {eg:.2e}"
    for j, t in enumerate((q, k, v)):
        r = ref[:, j * HD:(j + 1) * HD]
        x = np64(t)
        if qkv_f32:
            e = max_rel_err(x, r)
            assert e <= 5e-5, f"output {j}: {e:.2e}"
        else:
            bound = 2.0 ** -8 * np.abs(r) + 5e-5 * np.abs(r).max()
            assert np.all(np.abs(x - r) <= bound), f"output {j}: beyond one bf16 step"
    print(f"\n  N={N} hidden={hidden} H={H} qkv_f32={qkv_f32}: gate {eg:.2e}")


@pytest.mark.parametrize("N,hidden,H", [(5, 128, 2), (64, 7168, 32), (700, 256, 4), (1, 7168, 32), (64, 1024, 64),
                                        (120, 768, 3)])
def test_project_o_matches_oracle(N, hidden, H):
    """Includes calls that split K in two halves across CTAs (64 and 1 tokens
    at hidden 7168: 56 output tiles; hidden 1024 at H = 64: 8 tiles)."""
    wl = _wl(N, H)
    pr = synth.make_projections(wl, DEV, hidden=hidden)
    HD = H * 128
    ctx = _ctx(wl, pr)
    try:
        gy = Guarded(torch.zeros((N, hidden), device=DEV))
        ws = torch.empty(kda.kda_project_o_workspace_bytes(ctx, N), dtype=torch.uint8, device=DEV)
        kda.kda_project_o(ctx, N, pr["o_in"], gy.t, ws)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
        assert gy.intact(), "a guard region was written"
    finally:
        kda.kda_destroy(ctx)
    o = np64(pr["o_in"]).reshape(N, HD)
    o_b = np64(pr["o_in"].to(torch.bfloat16)).reshape(N, HD)    # the kernel's rounding of o
    W = np64(pr["W_o"])
    e_b = max_rel_err(np64(gy.t), oracle.project(o_b, W))
    e_u = rel_l2(np64(gy.t), oracle.project(o, W))
    print(f"\n  N={N} hidden={hidden} H={H}: vs rounded o {e_b:.2e} (max-rel), vs o {e_u:.2e} (rel-L2)")
    assert e_b <= 5e-5 and e_u <= 2.5e-3


def test_project_argument_errors():
    wl = _wl(4, 2)
    pr = synth.make_projections(wl, DEV, hidden=128)
    p = synth.make_params(wl, DEV)
    ctx = kda.kda_create(wl.H, p["conv_w"], p["dt_bias"], p["A_log"], p["gamma"])
    try:
        buf = torch.empty((4, 256), device=DEV)
        with pytest.raises(kda.KDAError) as ei:                      # nothing bound yet
            kda.kda_project_qkvg(ctx, 4, pr["x"].view(torch.int16), buf, buf, buf, buf)
        assert ei.value.status == kda.KDA_ERR_INVALID_ARG
        with pytest.raises(kda.KDAError) as ei:                      # hidden not a multiple of 128
            kda.kda_bind_projections(ctx, 96, pr["W_qkvg"].view(torch.int16), pr["W_o"].view(torch.int16))
        assert ei.value.status == kda.KDA_ERR_INVALID_ARG
        kda.kda_bind_projections(ctx, 128, pr["W_qkvg"].view(torch.int16), pr["W_o"].view(torch.int16))
        ws = torch.empty(16, dtype=torch.uint8, device=DEV)
        with pytest.raises(kda.KDAError) as ei:                      # workspace too small
            kda.kda_project_o(ctx, 4, pr["o_in"], torch.empty((4, 128), device=DEV), ws)
        assert ei.value.status == kda.KDA_ERR_INVALID_ARG
    finally:
        kda.kda_destroy(ctx)


def test_project_o_split_is_deterministic_and_overwrites_y():
    """Split K (64 tokens, hidden 7168, H = 32: 56 output tiles, two K halves
    added into y): y starts as NaN and is fully overwritten; two calls give
    the same y bit for bit (two addends onto zero commute exactly)."""
    N, hidden, H = 64, 7168, 32
    wl = _wl(N, H)
    pr = synth.make_projections(wl, DEV, hidden=hidden)
    ctx = _ctx(wl, pr)
    try:
        ws = torch.full((kda.kda_project_o_workspace_bytes(ctx, N),), 0x7F, dtype=torch.uint8, device=DEV)
        y1 = torch.full((N, hidden), float("nan"), device=DEV)
        y2 = torch.full((N, hidden), float("nan"), device=DEV)
        kda.kda_project_o(ctx, N, pr["o_in"], y1, ws)
        kda.kda_project_o(ctx, N, pr["o_in"], y2, ws)
        assert kda.kda_sync_status(ctx) == kda.KDA_OK
    finally:
        kda.kda_destroy(ctx)
    assert bool(torch.isfinite(y1).all())
    assert torch.equal(y1, y2)
