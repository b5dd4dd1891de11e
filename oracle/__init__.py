"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle of the KDA token step.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The CUDA library never calls it
and shares no code with it.

``build()`` compiles ``kda_oracle.c`` with gcc into ``oracle/_build``;
``run()`` wraps the C entry point for numpy float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")
_libs: dict = {}


def build(force: bool = False) -> str:
    """Compile the oracle (plain C, IEEE double, no fast-math) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    hdr = os.path.join(_HERE, "kda_oracle.h")
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(hdr))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
             "-fno-fast-math", "-ffp-contract=off",
             "-o", tmp, _SRC, "-lm", "-lpthread"],
            check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_variant(src_text: str, tag: str) -> str:
    """Compile another version of the oracle source (used by the mutation tests
    that check the pins catch planted mistakes).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_BUILD, f"variant_{tag}.c")
    with open(src, "w") as f:
        f.write(src_text)
    out = os.path.join(_BUILD, f"libkda_oracle_{tag}.so")
    subprocess.run(
        ["gcc", "-O1", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
         "-fno-fast-math", "-ffp-contract=off", f"-I{_HERE}",
         "-o", out, src, "-lm", "-lpthread"], check=True)
    return out


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _load(lib_path: str | None = None):
    path = lib_path or build()
    if path not in _libs:
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.kda_oracle_run.restype = ctypes.c_int
        lib.kda_oracle_run.argtypes = (
            [ctypes.c_int] * 4 + [dp] * 10 + [ctypes.c_double] * 2 + [dp] * 9 + [ctypes.c_int])
        lib.kda_oracle_run_bf16_state.restype = ctypes.c_int
        lib.kda_oracle_run_bf16_state.argtypes = lib.kda_oracle_run.argtypes
        u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.kda_oracle_bf16_round_n.restype = None
        lib.kda_oracle_bf16_round_n.argtypes = [ctypes.c_size_t, dp, u16p]
        lib.kda_oracle_bf16_value_n.restype = None
        lib.kda_oracle_bf16_value_n.argtypes = [ctypes.c_size_t, u16p, dp]
        lib.kda_oracle_cpu_count.restype = ctypes.c_int
        lib.kda_oracle_cpu_count.argtypes = []
        lib.kda_oracle_lowrank.restype = ctypes.c_int
        lib.kda_oracle_lowrank.argtypes = [ctypes.c_int] * 5 + [dp] * 6
        lib.kda_oracle_project.restype = ctypes.c_int
        lib.kda_oracle_project.argtypes = [ctypes.c_int] * 3 + [dp] * 3
        _libs[path] = lib
    return _libs[path]


def cpu_count() -> int:
    return int(_load().kda_oracle_cpu_count())


def _ptr(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous float64"
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


@dataclass
class OracleOut:
    o: np.ndarray
    o_pre: np.ndarray
    S: np.ndarray
    conv_state: np.ndarray
    qhat: np.ndarray | None = None
    khat: np.ndarray | None = None
    vconv: np.ndarray | None = None
    gk: np.ndarray | None = None
    beta: np.ndarray | None = None


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def run(q, k, v, z, beta_logit, gate_logit, conv_w, dt_bias, A_log, gamma,
        conv_state, S, *, l2_eps=1e-6, rms_eps=1e-6, intermediates=False,
        nthreads=1, state_bf16=False, lib_path: str | None = None) -> OracleOut:
    """Run T tokens of the KDA step for every (sequence, head).

    q, k, v, z, gate_logit: [B, T, H, d]; beta_logit: [B, T, H];
    conv_w: [3, H*d, 4]; dt_bias, A_log, gamma: [H, d];
    conv_state: [B, 3, 3*H*d]; S: [B, H, d, d].  Inputs are copied to
    float64 (exact for fp32 and bf16 values); S and conv_state are returned
    updated, the caller's arrays are left untouched.  With state_bf16 the
    state is stored as bfloat16 between tokens (S must hold bfloat16 values
    on entry and is returned rounded); the read-outs are unchanged in form.
    """
    q, k, v, z, gate_logit = (_f64(a) for a in (q, k, v, z, gate_logit))
    beta_logit, conv_w, dt_bias, A_log, gamma = (
        _f64(a) for a in (beta_logit, conv_w, dt_bias, A_log, gamma))
    B, T, H, d = q.shape
    for a in (k, v, z, gate_logit):
        assert a.shape == (B, T, H, d)
    assert beta_logit.shape == (B, T, H)
    assert conv_w.shape == (3, H * d, 4)
    for a in (dt_bias, A_log, gamma):
        assert a.shape == (H, d)
    cs = _f64(conv_state).copy()
    St = _f64(S).copy()
    assert cs.shape == (B, 3, 3 * H * d) and St.shape == (B, H, d, d)
    o = np.zeros((B, T, H, d))
    o_pre = np.zeros((B, T, H, d))
    extra = [np.zeros((B, T, H, d)) for _ in range(4)] + [np.zeros((B, T, H))] \
        if intermediates else [None] * 5
    lib = _load(lib_path)
    if state_bf16:
        assert np.array_equal(bf16_value(bf16_round(St, lib_path=lib_path), lib_path=lib_path), St), \
            "state_bf16 wants S made of bfloat16 values"
    rc = (lib.kda_oracle_run_bf16_state if state_bf16 else lib.kda_oracle_run)(
        B, T, H, d, _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta_logit),
        _ptr(gate_logit), _ptr(conv_w), _ptr(dt_bias), _ptr(A_log), _ptr(gamma),
        float(l2_eps), float(rms_eps), _ptr(cs), _ptr(St), _ptr(o), _ptr(o_pre),
        *[_ptr(e) for e in extra], int(nthreads))
    if rc != 0:
        raise ValueError(f"kda_oracle_run rejected its arguments (rc={rc})")
    return OracleOut(o, o_pre, St, cs, *extra)


def bf16_round(x, *, lib_path: str | None = None) -> np.ndarray:
    """bfloat16 patterns (uint16) of x rounded to nearest, ties to even."""
    x = _f64(x)
    out = np.empty(x.shape, dtype=np.uint16)
    _load(lib_path).kda_oracle_bf16_round_n(
        x.size, _ptr(x), out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)))
    return out


def bf16_value(b, *, lib_path: str | None = None) -> np.ndarray:
    """Exact float64 values of bfloat16 patterns."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    out = np.empty(b.shape, dtype=np.float64)
    _load(lib_path).kda_oracle_bf16_value_n(
        b.size, b.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), _ptr(out))
    return out


def lowrank(x, W_fa, W_fb, W_bp, H, d=128, *, lib_path: str | None = None):
    """Low-rank front-end: z = W_fb (W_fa x), beta_logit = W_bp x per token.

    x: [..., hidden]; W_fa: [rank, hidden]; W_fb: [H*d, rank]; W_bp: [H, hidden].
    Returns (z [..., H, d], beta_logit [..., H]) as float64.
    """
    x = _f64(x)
    lead = x.shape[:-1]
    hidden = x.shape[-1]
    W_fa, W_fb, W_bp = _f64(W_fa), _f64(W_fb), _f64(W_bp)
    rank = W_fa.shape[0]
    assert W_fa.shape == (rank, hidden) and W_fb.shape == (H * d, rank) and W_bp.shape == (H, hidden)
    N = int(np.prod(lead)) if lead else 1
    xf = np.ascontiguousarray(x.reshape(N, hidden))
    z = np.zeros((N, H * d))
    bl = np.zeros((N, H))
    rc = _load(lib_path).kda_oracle_lowrank(N, hidden, rank, H, d, _ptr(xf), _ptr(W_fa), _ptr(W_fb),
                                            _ptr(W_bp), _ptr(z), _ptr(bl))
    if rc != 0:
        raise ValueError(f"kda_oracle_lowrank rejected its arguments (rc={rc})")
    return z.reshape(*lead, H, d), bl.reshape(*lead, H)


def project(x, W, *, lib_path: str | None = None):
    """Projection y = W x per token: x [..., in], W [out, in] -> y [..., out], float64."""
    x = _f64(x)
    W = _f64(W)
    lead = x.shape[:-1]
    n_in = x.shape[-1]
    n_out = W.shape[0]
    assert W.shape == (n_out, n_in)
    N = int(np.prod(lead)) if lead else 1
    xf = np.ascontiguousarray(x.reshape(N, n_in))
    y = np.zeros((N, n_out))
    rc = _load(lib_path).kda_oracle_project(N, n_in, n_out, _ptr(xf), _ptr(W), _ptr(y))
    if rc != 0:
        raise ValueError(f"kda_oracle_project rejected its arguments (rc={rc})")
    return y.reshape(*lead, n_out)
