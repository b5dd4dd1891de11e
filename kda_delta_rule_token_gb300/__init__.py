"""Python binding of the GB300 KDA token-step library (libkda.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI of ``include/kda.h``.  The functions carry the C
names; tensors are PyTorch CUDA tensors (PyTorch supplies device memory and
streams).  There is no fallback: if libkda.so is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build_mod

__all__ = [
    "KDAError", "load", "kda_create", "kda_destroy", "kda_strerror", "kda_last_error_detail",
    "kda_decode_step", "kda_decode_step_bf16state", "kda_prefill", "kda_prefill_varlen", "kda_prefill_workspace_bytes", "kda_sync_status",
    "kda_launch_count", "kda_bind_lowrank", "kda_lowrank", "kda_lowrank_workspace_bytes",
    "kda_decode_step_lowrank", "kda_decode_lowrank_workspace_bytes", "kda_lowrank_noalloc",
    "LOWRANK_NOALLOC_SCRATCH_BYTES", "kda_bind_projections", "kda_project_qkvg", "kda_project_o",
    "kda_project_o_workspace_bytes", "KDA_OK", "KDA_ERR_INVALID_ARG", "KDA_ERR_ALIGNMENT",
    "KDA_ERR_UNSUPPORTED", "KDA_ERR_CUDA", "KDA_ERR_TIMEOUT", "HEAD_DIM", "CHUNK",
]

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_ALIGNMENT, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, \
    KDA_ERR_TIMEOUT = range(6)
HEAD_DIM = 128
CHUNK = 64
LOWRANK_NOALLOC_SCRATCH_BYTES = 4 << 20   # KDA_LOWRANK_NOALLOC_SCRATCH_BYTES of include/kda.h

_lib = None


class KDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if _lib is not None:
            d = _lib.kda_last_error_detail()
            detail = d.decode() if d else ""
        msg = f"{where}: {kda_strerror(status)}" + (f" [{detail}]" if detail else "")
        super().__init__(msg)


class _Config(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("chunk_size", ctypes.c_int), ("l2_eps", ctypes.c_float),
                ("rms_eps", ctypes.c_float)]


def library_path() -> str:
    return _build_mod.LIB


def load(path: str | None = None):
    """Load libkda.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -m kda_delta_rule_token_gb300.build)")
    lib = ctypes.CDLL(path)
    vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
    lib.kda_create.argtypes = [ctypes.POINTER(_Config), vp, vp, vp, vp, ctypes.POINTER(vp)]
    lib.kda_create.restype = i32
    lib.kda_destroy.argtypes = [vp]
    lib.kda_destroy.restype = None
    lib.kda_strerror.argtypes = [i32]
    lib.kda_strerror.restype = ctypes.c_char_p
    lib.kda_last_error_detail.argtypes = []
    lib.kda_last_error_detail.restype = ctypes.c_char_p
    lib.kda_decode_step.argtypes = [vp, i32] + [vp] * 11
    lib.kda_decode_step.restype = i32
    lib.kda_decode_step_bf16state.argtypes = [vp, i32] + [vp] * 11
    lib.kda_decode_step_bf16state.restype = i32
    lib.kda_prefill_workspace_bytes.argtypes = [vp, i32, i32]
    lib.kda_prefill_workspace_bytes.restype = sz
    lib.kda_prefill.argtypes = [vp, i32, i32] + [vp] * 10 + [sz, vp]
    lib.kda_prefill.restype = i32
    lib.kda_prefill_varlen.argtypes = [vp, i32, vp, i32] + [vp] * 10
    lib.kda_prefill_varlen.restype = i32
    lib.kda_sync_status.argtypes = [vp, vp]
    lib.kda_sync_status.restype = i32
    lib.kda_launch_count.argtypes = []
    lib.kda_launch_count.restype = u64
    lib.kda_bind_lowrank.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.kda_bind_lowrank.restype = i32
    lib.kda_lowrank_workspace_bytes.argtypes = [vp, i32]
    lib.kda_lowrank_workspace_bytes.restype = sz
    lib.kda_lowrank.argtypes = [vp, i32, vp, vp, vp, vp, sz, vp]
    lib.kda_lowrank.restype = i32
    lib.kda_decode_lowrank_workspace_bytes.argtypes = [vp, i32]
    lib.kda_decode_lowrank_workspace_bytes.restype = sz
    lib.kda_decode_step_lowrank.argtypes = [vp, i32] + [vp] * 10 + [sz, vp]
    lib.kda_decode_step_lowrank.restype = i32
    lib.kda_lowrank_noalloc.argtypes = [vp, i32, vp, vp, vp, vp]
    lib.kda_lowrank_noalloc.restype = i32
    lib.kda_bind_projections.argtypes = [vp, i32, vp, vp]
    lib.kda_bind_projections.restype = i32
    lib.kda_project_qkvg.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, vp]
    lib.kda_project_qkvg.restype = i32
    lib.kda_project_o_workspace_bytes.argtypes = [vp, i32]
    lib.kda_project_o_workspace_bytes.restype = sz
    lib.kda_project_o.argtypes = [vp, i32, vp, vp, vp, sz, vp]
    lib.kda_project_o.restype = i32
    lib.kda_testing_bounded_wait.argtypes = [vp, ctypes.c_uint, vp]
    lib.kda_testing_bounded_wait.restype = i32
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != KDA_OK:
        raise KDAError(status, where)


def _p(t):
    """Device address of a tensor (None -> NULL); ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kda_strerror(status: int) -> str:
    return load().kda_strerror(int(status)).decode()


def kda_last_error_detail() -> str:
    d = load().kda_last_error_detail()
    return d.decode() if d else ""


def kda_launch_count() -> int:
    return int(load().kda_launch_count())


def kda_create(num_heads, conv_w, dt_bias, A_log, rms_gamma, *, head_dim=HEAD_DIM,
               chunk_size=CHUNK, l2_eps=1e-6, rms_eps=1e-6) -> int:
    """Returns an opaque context handle (int).  Parameters are borrowed."""
    cfg = _Config(int(num_heads), int(head_dim), int(chunk_size), float(l2_eps), float(rms_eps))
    out = ctypes.c_void_p()
    _check(load().kda_create(ctypes.byref(cfg), _p(conv_w), _p(dt_bias), _p(A_log),
                             _p(rms_gamma), ctypes.byref(out)), "kda_create")
    return out.value


def kda_destroy(ctx: int) -> None:
    load().kda_destroy(ctx)


def kda_decode_step(ctx, B, q, k, v, z, beta_logit, gate_logit, conv_state, S, o,
                    o_pre=None, stream=None) -> None:
    _check(load().kda_decode_step(ctx, int(B), _p(q), _p(k), _p(v), _p(z), _p(beta_logit),
                                  _p(gate_logit), _p(conv_state), _p(S), _p(o), _p(o_pre),
                                  _stream(stream)), "kda_decode_step")


def kda_decode_step_bf16state(ctx, B, q, k, v, z, beta_logit, gate_logit, conv_state, S, o,
                              o_pre=None, stream=None) -> None:
    """kda_decode_step with S held as bf16 (a 16-bit tensor of raw patterns)."""
    _check(load().kda_decode_step_bf16state(ctx, int(B), _p(q), _p(k), _p(v), _p(z), _p(beta_logit),
                                            _p(gate_logit), _p(conv_state), _p(S), _p(o), _p(o_pre),
                                            _stream(stream)), "kda_decode_step_bf16state")


def kda_prefill_workspace_bytes(ctx, B, T) -> int:
    return int(load().kda_prefill_workspace_bytes(ctx, int(B), int(T)))


def kda_prefill(ctx, B, T, q, k, v, z, beta_logit, gate_logit, conv_state, S, o,
                workspace=None, workspace_bytes=0, stream=None) -> None:
    if workspace is not None and not isinstance(workspace, int) and workspace_bytes == 0:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load().kda_prefill(ctx, int(B), int(T), _p(q), _p(k), _p(v), _p(z), _p(beta_logit),
                              _p(gate_logit), _p(conv_state), _p(S), _p(o), _p(workspace),
                              int(workspace_bytes), _stream(stream)), "kda_prefill")


def kda_prefill_varlen(ctx, B, cu_seqlens, total_T, q, k, v, z, beta_logit, gate_logit, conv_state,
                       S, o, stream=None) -> None:
    """Packed sequences: cu_seqlens is a device int32 tensor of B + 1 offsets."""
    _check(load().kda_prefill_varlen(ctx, int(B), _p(cu_seqlens), int(total_T), _p(q), _p(k), _p(v),
                                     _p(z), _p(beta_logit), _p(gate_logit), _p(conv_state), _p(S),
                                     _p(o), _stream(stream)), "kda_prefill_varlen")


def _nbytes(buf, given):
    if buf is None or isinstance(buf, int) or given:
        return int(given)
    return buf.numel() * buf.element_size()


def kda_bind_lowrank(ctx, hidden, rank, W_fa, W_fb, W_bp) -> None:
    _check(load().kda_bind_lowrank(ctx, int(hidden), int(rank), _p(W_fa), _p(W_fb), _p(W_bp)),
           "kda_bind_lowrank")


def kda_lowrank_workspace_bytes(ctx, N) -> int:
    return int(load().kda_lowrank_workspace_bytes(ctx, int(N)))


def kda_lowrank(ctx, N, x, z, beta_logit, workspace, workspace_bytes=0, stream=None) -> None:
    _check(load().kda_lowrank(ctx, int(N), _p(x), _p(z), _p(beta_logit), _p(workspace),
                              _nbytes(workspace, workspace_bytes), _stream(stream)), "kda_lowrank")


def kda_lowrank_noalloc(ctx, N, x, z, beta_logit, stream=None) -> None:
    """The front-end with its scratch in the library's static device array
    (no workspace argument; see kda.h)."""
    _check(load().kda_lowrank_noalloc(ctx, int(N), _p(x), _p(z), _p(beta_logit), _stream(stream)),
           "kda_lowrank_noalloc")


def kda_decode_lowrank_workspace_bytes(ctx, B) -> int:
    return int(load().kda_decode_lowrank_workspace_bytes(ctx, int(B)))


def kda_decode_step_lowrank(ctx, B, x, q, k, v, gate_logit, conv_state, S, o, o_pre, workspace,
                            workspace_bytes=0, stream=None) -> None:
    _check(load().kda_decode_step_lowrank(ctx, int(B), _p(x), _p(q), _p(k), _p(v), _p(gate_logit),
                                          _p(conv_state), _p(S), _p(o), _p(o_pre), _p(workspace),
                                          _nbytes(workspace, workspace_bytes), _stream(stream)),
           "kda_decode_step_lowrank")


def kda_bind_projections(ctx, hidden, W_qkvg, W_o) -> None:
    """W_qkvg [4*H*d, hidden] and W_o [hidden, H*d]: bf16 tensors (or their int16 views)."""
    _check(load().kda_bind_projections(ctx, int(hidden), _p(W_qkvg), _p(W_o)), "kda_bind_projections")


def kda_project_qkvg(ctx, N, x, q, k, v, gate_logit, qkv_f32=False, stream=None) -> None:
    _check(load().kda_project_qkvg(ctx, int(N), _p(x), _p(q), _p(k), _p(v), _p(gate_logit),
                                   1 if qkv_f32 else 0, _stream(stream)), "kda_project_qkvg")


def kda_project_o_workspace_bytes(ctx, N) -> int:
    return int(load().kda_project_o_workspace_bytes(ctx, int(N)))


def kda_project_o(ctx, N, o, y, workspace, workspace_bytes=0, stream=None) -> None:
    _check(load().kda_project_o(ctx, int(N), _p(o), _p(y), _p(workspace),
                                _nbytes(workspace, workspace_bytes), _stream(stream)), "kda_project_o")


def kda_sync_status(ctx, stream=None) -> int:
    """Synchronise and return the status code (does not raise)."""
    return int(load().kda_sync_status(ctx, _stream(stream)))


def kda_testing_bounded_wait(ctx, limit_us, stream=None) -> None:
    """Test hook (not part of the public API): launch a kernel whose bounded
    wait runs out after ``limit_us`` microseconds; the next kda_sync_status
    reports KDA_ERR_TIMEOUT."""
    _check(load().kda_testing_bounded_wait(ctx, int(limit_us), _stream(stream)),
           "kda_testing_bounded_wait")
