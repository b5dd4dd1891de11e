"""The seeded input generators (no KDA arithmetic in them): the same workload
gives the same bytes on every call, each tensor has a stream of its own, and
shapes, dtypes and distributions follow the stated recipe."""
import numpy as np
import torch

from kda_delta_rule_token_gb300 import synth


def test_same_workload_same_bytes():
    wl = synth.shrink(synth.WORKLOADS["prefill_b1_h32_t4096"], H=2, T=70)
    a, b = synth.make_tokens(wl), synth.make_tokens(wl)
    for n in a:
        assert torch.equal(a[n].view(torch.int16) if a[n].dtype == torch.bfloat16 else a[n],
                           b[n].view(torch.int16) if b[n].dtype == torch.bfloat16 else b[n])
    pa, pb = synth.make_params(wl), synth.make_params(wl)
    for n in pa:
        assert torch.equal(pa[n], pb[n])


def test_tensors_and_seeds_have_their_own_streams():
    wl = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=2, H=2, T=3)
    t = synth.make_tokens(wl)
    assert not torch.equal(t["q"], t["k"]) and not torch.equal(t["z"], t["gate_logit"])
    w2 = synth.shrink(wl, seed=wl.seed + 1)
    assert not torch.equal(t["q"], synth.make_tokens(w2)["q"])
    warm = synth.make_tokens(wl, warm=True)
    assert not torch.equal(t["q"], warm["q"])


def test_layouts_and_dtypes():
    dec = synth.shrink(synth.WORKLOADS["decode_b64_h32_x256"], B=3, H=2, T=5)
    t = synth.make_tokens(dec)
    assert t["q"].shape == (5, 3, 2, 128) and t["q"].dtype == torch.float32   # call-major
    assert t["beta_logit"].shape == (5, 3, 2)
    pre = synth.shrink(synth.WORKLOADS["prefill_b8_h64_t8192"], B=2, H=2, T=7)
    t = synth.make_tokens(pre)
    assert t["q"].shape == (2, 7, 2, 128) and t["q"].dtype == torch.bfloat16
    assert t["z"].dtype == torch.float32 and t["beta_logit"].shape == (2, 7, 2)
    st = synth.make_state(synth.WORKLOADS["decode_b64_h32_x256"])
    assert st["S"].shape == (64, 32, 128, 128) and st["conv_state"].shape == (64, 3, 3 * 32 * 128)


def test_distributions():
    wl = synth.WORKLOADS["prefill_b8_h64_t8192"]
    p = synth.make_params(wl)
    assert abs(p["conv_w"].std().item() - 0.25) < 0.01
    assert abs(p["dt_bias"].std().item() - 0.1) < 0.005
    assert -6.0 <= p["A_log"].min().item() and p["A_log"].max().item() < 0.0
    assert p["A_log"].min().item() < -5.9                      # U(-6, 0) for this workload
    assert abs(p["gamma"].mean().item() - 1.0) < 0.01
    d = synth.make_params(synth.WORKLOADS["decode_b64_h32_x256"])["A_log"]
    assert -4.0 <= d.min().item() < -3.9                       # U(-4, 0) otherwise
    st = synth.make_state(synth.WORKLOADS["decode_b64_h32_x256"])
    assert abs(st["S"].std().item() - 0.01) < 0.001 and abs(st["conv_state"].std().item() - 1.0) < 0.01
    z = synth.make_state(synth.shrink(wl, B=1, H=1))
    assert not bool(z["S"].any()) and not bool(z["conv_state"].any())   # zero initial state


def test_packed_lengths_recipe():
    L = synth.packed_lengths()
    assert len(L) == 32 and int(L.sum()) == 80371 and int(L.min()) == 257 and int(L.max()) == 8169
    assert np.array_equal(L, synth.packed_lengths())
    wl = synth.packed_workload(L)
    assert (wl.B, wl.H, wl.T, wl.a_log_low, wl.qkv_bf16) == (1, 64, 80371, -6.0, True)
