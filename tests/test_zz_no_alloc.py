"""kda_lowrank_noalloc: the low-rank front-end for callers that cannot give
the library device memory for a call.

Such a caller (a host runtime that hands a plugin only the layer's tensors,
or a serving loop that must not allocate once it runs) gets the same z and
beta_logit as kda_lowrank, with the scratch kept in the library's own static
device array instead of a workspace argument.  Checked here through the C
ABI against kda_lowrank on two calls in a row (different inputs, and the
second at another batch size, so the array holds the first call's contents
when the second starts), within the front-end tolerance of the other GPU
tests (max|x - r| / max|r| <= 2e-5), with guard regions around the outputs;
and a batch whose scratch would not fit the array is refused on the host.

This file is collected last on purpose: when it fails, a run that stops at
the first failure has already run every other test.
"""
import pytest
import torch

import kda_delta_rule_token_gb300 as kda
from kda_delta_rule_token_gb300 import synth
from harness import Guarded, max_rel_err, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_FE = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_delta_rule_token_gb300 import build
    build.build()
    kda.load()


def _ctx(wl, lr):
    p = synth.make_params(wl, DEV)
    ctx = kda.kda_create(wl.H, p["conv_w"], p["dt_bias"], p["A_log"], p["gamma"])
    kda.kda_bind_lowrank(ctx, lr["hidden"], lr["rank"], lr["W_fa"], lr["W_fb"], lr["W_bp"])
    return ctx


def _with_workspace(ctx, H, x):
    N = x.shape[0]
    z = torch.empty((N, H, 128), device=DEV)
    bl = torch.empty((N, H), device=DEV)
    ws = torch.empty(kda.kda_lowrank_workspace_bytes(ctx, N), dtype=torch.uint8, device=DEV)
    kda.kda_lowrank(ctx, N, x, z, bl, ws)
    return z, bl


def _no_alloc(ctx, H, x):
    N = x.shape[0]
    gz = Guarded(torch.zeros((N, H, 128), device=DEV))
    gb = Guarded(torch.zeros((N, H), device=DEV))
    kda.kda_lowrank_noalloc(ctx, N, x, gz.t, gb.t)
    return gz, gb


@pytest.mark.parametrize("B,H", [(64, 32), (256, 64)])
def test_no_alloc_matches_workspace_entry_point_on_two_calls(B, H):
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=B, H=H, T=2)
    lr = synth.make_lowrank(wl, DEV)
    ctx = _ctx(wl, lr)
    try:
        for x in (lr["x"][0], lr["x"][1][: B // 2 + 3]):     # second call: other inputs, another size
            z_ref, b_ref = _with_workspace(ctx, H, x)
            gz, gb = _no_alloc(ctx, H, x)
            assert kda.kda_sync_status(ctx) == kda.KDA_OK
            assert gz.intact() and gb.intact(), "a guard region was written"
            ez, eb = max_rel_err(np64(gz.t), np64(z_ref)), max_rel_err(np64(gb.t), np64(b_ref))
            print(f"\n  B={B} H={H} N={x.shape[0]}: z {ez:.2e}, beta_logit {eb:.2e}")
            assert ez <= TOL_FE and eb <= TOL_FE
    finally:
        kda.kda_destroy(ctx)


def test_no_alloc_refuses_a_batch_beyond_its_array():
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=8192, H=4, T=1)
    lr = synth.make_lowrank(wl, DEV, hidden=64, rank=128)       # u alone is 4 MiB at 8192 tokens
    ctx = _ctx(wl, lr)
    try:
        z = torch.full((8192, 4, 128), 3.0, device=DEV)
        bl = torch.full((8192, 4), 3.0, device=DEV)
        n0 = kda.kda_launch_count()
        with pytest.raises(kda.KDAError) as ei:
            kda.kda_lowrank_noalloc(ctx, 8192, lr["x"][0], z, bl)
        assert ei.value.status == kda.KDA_ERR_INVALID_ARG
        assert str(kda.LOWRANK_NOALLOC_SCRATCH_BYTES) in kda.kda_last_error_detail()
        assert kda.kda_launch_count() == n0
        torch.cuda.synchronize()
        assert bool((z == 3.0).all()) and bool((bl == 3.0).all())
    finally:
        kda.kda_destroy(ctx)
