"""Thin ctypes binding of ``libkda.so`` (the C ABI in ``include/kda.h``).

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream, and every step of the computation runs in the library's
kernels.  Importing this module loads the library and raises ``ImportError``
when it has not been built (``python -m gated_delta_rule_kda_gb300.build``):
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from .build import LIB as _LIB_PATH

KDA_OK = 0
KDA_BF16 = 0
KDA_FP32 = 1
HEAD_DIM = 128
DEFAULT_SCALE = 1.0 / math.sqrt(128.0)

STATUS_NAMES = {
    0: "KDA_OK",
    1: "KDA_ERR_INVALID_ARGUMENT",
    2: "KDA_ERR_UNSUPPORTED",
    3: "KDA_ERR_WORKSPACE",
    4: "KDA_ERR_CUDA",
    5: "KDA_ERR_DEVICE_TIMEOUT",
    6: "KDA_ERR_DEVICE_CHECK",
}

# Every entry point include/kda.h declares (checked by tests on CPU).
EXPORTED = (
    "kda_status_string",
    "kda_version",
    "kda_prefill_workspace_size",
    "kda_prefill",
    "kda_prefill_with_checkpoints",
    "kda_prefill_head_decay",
    "kda_prefill_unbounded_decay",
    "kda_decode_step",
    "kda_decode_step_head_decay",
    "kda_frontend",
    "kda_frontend_unbounded_decay",
    "kda_output_gate",
    "kda_layer_core_workspace_size",
    "kda_layer_core",
    "kda_layer_core_unbounded_decay",
    "kda_layer_core_noalloc",
    "kda_layer_core_fused",
    "kda_layer_core_fused_unbounded_decay",
    "kda_layer_core_fused_with_checkpoints",
    "kda_decode_layer",
    "kda_decode_tokens",
    "kda_decode_layer_tokens",
    "kda_check_prefill_inputs",
    "kda_get_device_status",
    "kda_debug_inject_handoff_timeout",
)

# Capacity of the fixed scratch array behind kda_layer_core_noalloc (include/kda.h).
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class KdaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libkda.so is not built ({_LIB_PATH}); run "
                          "`python -m gated_delta_rule_kda_gb300.build` first")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I32, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                          ctypes.c_size_t)
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_version.argtypes = []
    lib.kda_version.restype = I32
    lib.kda_prefill_workspace_size.argtypes = [I32, I32, I32, ctypes.c_int]
    lib.kda_prefill_workspace_size.restype = SZ
    lib.kda_prefill.argtypes = [ctypes.c_int, ctypes.c_int, I32, I32, I32, P, P, P, P, P, P, P,
                                F, P, P, P, SZ, P]
    lib.kda_prefill.restype = ctypes.c_int
    lib.kda_prefill_with_checkpoints.argtypes = [ctypes.c_int, ctypes.c_int, I32, I32, I32, P, P,
                                                 P, P, P, P, P, F, P, P, P, SZ, I32, P, P, P]
    lib.kda_prefill_with_checkpoints.restype = ctypes.c_int
    lib.kda_prefill_head_decay.argtypes = lib.kda_prefill_with_checkpoints.argtypes
    lib.kda_prefill_head_decay.restype = ctypes.c_int
    lib.kda_prefill_unbounded_decay.argtypes = lib.kda_prefill.argtypes
    lib.kda_prefill_unbounded_decay.restype = ctypes.c_int
    lib.kda_decode_step.argtypes = [ctypes.c_int, ctypes.c_int, I32, I32, P, P, P, P, P, P, F,
                                    P, P]
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_decode_step_head_decay.argtypes = lib.kda_decode_step.argtypes
    lib.kda_decode_step_head_decay.restype = ctypes.c_int
    lib.kda_frontend.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, P, P, F, ctypes.c_int,
                                 P, P, P, P, P, P]
    lib.kda_frontend.restype = ctypes.c_int
    lib.kda_frontend_unbounded_decay.argtypes = lib.kda_frontend.argtypes
    lib.kda_frontend_unbounded_decay.restype = ctypes.c_int
    lib.kda_output_gate.argtypes = [I64, ctypes.c_int, P, P, F, ctypes.c_int, P, P]
    lib.kda_output_gate.restype = ctypes.c_int
    lib.kda_layer_core_workspace_size.argtypes = [I32, I32, I32]
    lib.kda_layer_core_workspace_size.restype = SZ
    lib.kda_layer_core.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, F, F, F,
                                   ctypes.c_int, P, P, P, SZ, P]
    lib.kda_layer_core.restype = ctypes.c_int
    lib.kda_layer_core_unbounded_decay.argtypes = lib.kda_layer_core.argtypes
    lib.kda_layer_core_unbounded_decay.restype = ctypes.c_int
    lib.kda_layer_core_noalloc.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, F, F,
                                           F, ctypes.c_int, P, P, P]
    lib.kda_layer_core_noalloc.restype = ctypes.c_int
    lib.kda_layer_core_fused.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, F, F,
                                         F, ctypes.c_int, P, P, P]
    lib.kda_layer_core_fused.restype = ctypes.c_int
    lib.kda_layer_core_fused_unbounded_decay.argtypes = lib.kda_layer_core_fused.argtypes
    lib.kda_layer_core_fused_unbounded_decay.restype = ctypes.c_int
    lib.kda_layer_core_fused_with_checkpoints.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, P,
                                                          P, P, P, F, F, F, ctypes.c_int, P, P,
                                                          I32, P, P, P]
    lib.kda_layer_core_fused_with_checkpoints.restype = ctypes.c_int
    lib.kda_decode_layer.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P, F, F, F,
                                     ctypes.c_int, P, P]
    lib.kda_decode_layer.restype = ctypes.c_int
    lib.kda_decode_tokens.argtypes = [ctypes.c_int, ctypes.c_int, I32, I32, I32, I32, P, P, P, P,
                                      P, P, P, P, I32, P, F, P, P]
    lib.kda_decode_tokens.restype = ctypes.c_int
    lib.kda_decode_layer_tokens.argtypes = [I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P,
                                            P, P, I32, F, F, F, ctypes.c_int, P, P]
    lib.kda_decode_layer_tokens.restype = ctypes.c_int
    lib.kda_check_prefill_inputs.argtypes = [I32, I32, I32, P, I32, P, P]
    lib.kda_check_prefill_inputs.restype = ctypes.c_int
    lib.kda_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.kda_get_device_status.restype = ctypes.c_int
    lib.kda_debug_inject_handoff_timeout.argtypes = []
    lib.kda_debug_inject_handoff_timeout.restype = ctypes.c_int
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def library_path() -> str:
    return _LIB_PATH


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dtype_code(d: torch.dtype) -> int:
    return KDA_BF16 if d == torch.bfloat16 else KDA_FP32


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, rc: int):
    if rc != KDA_OK:
        raise KdaError(fn, rc)


def kda_prefill_workspace_size(num_seqs: int, total_tokens: int, num_heads: int,
                               in_dtype: torch.dtype = torch.bfloat16) -> int:
    return int(_lib.kda_prefill_workspace_size(num_seqs, total_tokens, num_heads,
                                               _dtype_code(in_dtype)))


def kda_prefill(q, k, v, log_alpha, beta, cu_seqlens, S0=None, scale=DEFAULT_SCALE, *,
                out_dtype=None, o=None, S_final=None, want_state=True, workspace=None,
                stream=None, _entry="kda_prefill"):
    """Packed-varlen prefill.  Returns (o, S_final or None).

    q, k, v [T, H, 128] (bf16 or fp32); log_alpha [T, H, 128] fp32; beta [T, H] fp32;
    cu_seqlens [N+1] int32 (device); S0 [N, H, 128, 128] fp32 or None.
    S_final may be S0 itself (in-place resume)."""
    T, H, _ = q.shape
    N = cu_seqlens.shape[0] - 1
    out_dtype = out_dtype or q.dtype
    if o is None:
        o = torch.empty((T, H, HEAD_DIM), dtype=out_dtype, device=q.device)
    if S_final is None and want_state:
        S_final = torch.empty((N, H, HEAD_DIM, HEAD_DIM), dtype=torch.float32, device=q.device)
    need = kda_prefill_workspace_size(N, T, H, q.dtype)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = getattr(_lib, _entry)(_dt(q), _dtype_code(o.dtype), N, T, H, _p(q), _p(k), _p(v),
                          _p(log_alpha), _p(beta), _p(S0), _p(cu_seqlens), float(scale), _p(o),
                          _p(S_final), _p(workspace), wbytes, _stream(stream))
    _check(_entry, rc)
    return o, S_final


def kda_prefill_unbounded_decay(q, k, v, log_alpha, beta, cu_seqlens, S0=None,
                                scale=DEFAULT_SCALE, **kw):
    """kda_prefill for any log_alpha <= 0 (-inf included) on the token-by-token kernel."""
    return kda_prefill(q, k, v, log_alpha, beta, cu_seqlens, S0, scale,
                       _entry="kda_prefill_unbounded_decay", **kw)


def checkpoint_offsets(cu_seqlens, every: int) -> torch.Tensor:
    """Snapshot offsets [N+1] int32 (host) for one snapshot per `every` tokens of each
    sequence: base[n+1] - base[n] = len_n // every."""
    cu = torch.as_tensor(cu_seqlens).to("cpu", torch.int64)
    counts = torch.div(cu[1:] - cu[:-1], every, rounding_mode="floor")
    return torch.cat([torch.zeros(1, dtype=torch.int64), counts.cumsum(0)]).to(torch.int32)


def _checkpoint_args(cu_seqlens, H, every, ckpt_base, ckpt_states, device):
    if ckpt_base is None:
        ckpt_base = checkpoint_offsets(cu_seqlens, every).to(device)
    if ckpt_states is None:
        total = int(ckpt_base[-1])
        ckpt_states = torch.empty((total, H, HEAD_DIM, HEAD_DIM), dtype=torch.float32,
                                  device=device)
    return ckpt_base, ckpt_states


def kda_prefill_with_checkpoints(q, k, v, log_alpha, beta, cu_seqlens, every, S0=None,
                                 scale=DEFAULT_SCALE, *, ckpt_base=None, ckpt_states=None,
                                 out_dtype=None, o=None, S_final=None, want_state=True,
                                 workspace=None, stream=None, _entry="kda_prefill_with_checkpoints"):
    """kda_prefill that also writes the state after every `every` tokens of each sequence
    (every: a positive multiple of 32).  ckpt_base [N+1] int32 (device) defaults to
    checkpoint_offsets(cu_seqlens, every).  Returns (o, S_final, ckpt_base, ckpt_states)."""
    T, H, _ = q.shape
    N = cu_seqlens.shape[0] - 1
    out_dtype = out_dtype or q.dtype
    if o is None:
        o = torch.empty((T, H, HEAD_DIM), dtype=out_dtype, device=q.device)
    if S_final is None and want_state:
        S_final = torch.empty((N, H, HEAD_DIM, HEAD_DIM), dtype=torch.float32, device=q.device)
    if every:
        ckpt_base, ckpt_states = _checkpoint_args(cu_seqlens, H, every, ckpt_base, ckpt_states,
                                                  q.device)
    need = kda_prefill_workspace_size(N, T, H, q.dtype)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = getattr(_lib, _entry)(
        _dt(q), _dtype_code(o.dtype), N, T, H, _p(q), _p(k), _p(v), _p(log_alpha), _p(beta),
        _p(S0), _p(cu_seqlens), float(scale), _p(o), _p(S_final), _p(workspace), wbytes,
        int(every), _p(ckpt_base), _p(ckpt_states), _stream(stream))
    _check(_entry, rc)
    return o, S_final, ckpt_base, ckpt_states


def kda_prefill_head_decay(q, k, v, log_alpha, beta, cu_seqlens, S0=None, scale=DEFAULT_SCALE, *,
                           every=0, ckpt_base=None, ckpt_states=None, out_dtype=None, o=None,
                           S_final=None, want_state=True, workspace=None, stream=None):
    """The Gated DeltaNet case: log_alpha [T, H] fp32, one decay per (token, head).
    Returns (o, S_final, ckpt_base, ckpt_states) (the last two None without snapshots)."""
    return kda_prefill_with_checkpoints(q, k, v, log_alpha, beta, cu_seqlens, every, S0, scale,
                                        ckpt_base=ckpt_base, ckpt_states=ckpt_states,
                                        out_dtype=out_dtype, o=o, S_final=S_final,
                                        want_state=want_state, workspace=workspace, stream=stream,
                                        _entry="kda_prefill_head_decay")


def kda_decode_step(q, k, v, log_alpha, beta, S_inout, scale=DEFAULT_SCALE, *, out_dtype=None,
                    o=None, stream=None, _entry="kda_decode_step"):
    """One decode step; S_inout [B, H, 128, 128] fp32 is updated in place.  Returns o."""
    B, H, _ = q.shape
    out_dtype = out_dtype or q.dtype
    if o is None:
        o = torch.empty((B, H, HEAD_DIM), dtype=out_dtype, device=q.device)
    rc = getattr(_lib, _entry)(_dt(q), _dtype_code(o.dtype), B, H, _p(q), _p(k), _p(v),
                               _p(log_alpha), _p(beta), _p(S_inout), float(scale), _p(o),
                               _stream(stream))
    _check(_entry, rc)
    return o


def kda_decode_step_head_decay(q, k, v, log_alpha, beta, S_inout, scale=DEFAULT_SCALE, *,
                               out_dtype=None, o=None, stream=None):
    """kda_decode_step with log_alpha [B, H] fp32 (one decay per request and head)."""
    return kda_decode_step(q, k, v, log_alpha, beta, S_inout, scale, out_dtype=out_dtype, o=o,
                           stream=stream, _entry="kda_decode_step_head_decay")


def kda_frontend(qp, kp, vp, conv_w, z, A, b, beta_logit, cu_seqlens, l2_eps=1e-6, *,
                 out_dtype=torch.bfloat16, stream=None, _entry="kda_frontend"):
    """Returns (q_hat, k_hat, v, log_alpha, beta)."""
    T, H, _ = qp.shape
    N = cu_seqlens.shape[0] - 1
    dev = qp.device
    q_hat = torch.empty((T, H, HEAD_DIM), dtype=out_dtype, device=dev)
    k_hat = torch.empty_like(q_hat)
    v_out = torch.empty_like(q_hat)
    log_alpha = torch.empty((T, H, HEAD_DIM), dtype=torch.float32, device=dev)
    beta = torch.empty((T, H), dtype=torch.float32, device=dev)
    rc = getattr(_lib, _entry)(N, T, H, _p(qp), _p(kp), _p(vp), _p(conv_w), _p(z), _p(A), _p(b),
                           _p(beta_logit), _p(cu_seqlens), float(l2_eps),
                           _dtype_code(out_dtype), _p(q_hat), _p(k_hat), _p(v_out),
                           _p(log_alpha), _p(beta), _stream(stream))
    _check(_entry, rc)
    return q_hat, k_hat, v_out, log_alpha, beta


def kda_frontend_unbounded_decay(qp, kp, vp, conv_w, z, A, b, beta_logit, cu_seqlens, l2_eps=1e-6,
                                 **kw):
    """kda_frontend with Kimi Linear's gate log_alpha = -e^A softplus(z + b)."""
    return kda_frontend(qp, kp, vp, conv_w, z, A, b, beta_logit, cu_seqlens, l2_eps,
                        _entry="kda_frontend_unbounded_decay", **kw)


def kda_output_gate(o_tilde, g, eps=1e-6, *, out_dtype=torch.bfloat16, out=None, stream=None):
    rows = o_tilde.numel() // HEAD_DIM
    if out is None:
        out = torch.empty(o_tilde.shape, dtype=out_dtype, device=o_tilde.device)
    rc = _lib.kda_output_gate(rows, _dt(o_tilde), _p(o_tilde), _p(g), float(eps),
                              _dtype_code(out.dtype), _p(out), _stream(stream))
    _check("kda_output_gate", rc)
    return out


def kda_layer_core_workspace_size(num_seqs: int, total_tokens: int, num_heads: int) -> int:
    return int(_lib.kda_layer_core_workspace_size(num_seqs, total_tokens, num_heads))


def kda_layer_core(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens, S0=None,
                   scale=DEFAULT_SCALE, l2_eps=1e-6, rms_eps=1e-6, *, out_dtype=torch.bfloat16,
                   o=None, S_final=None, want_state=True, workspace=None, stream=None,
                   _entry="kda_layer_core"):
    """Front end -> recurrence -> output gate.  Returns (o_gated, S_final or None)."""
    T, H, _ = qp.shape
    N = cu_seqlens.shape[0] - 1
    if o is None:
        o = torch.empty((T, H, HEAD_DIM), dtype=out_dtype, device=qp.device)
    if S_final is None and want_state:
        S_final = torch.empty((N, H, HEAD_DIM, HEAD_DIM), dtype=torch.float32, device=qp.device)
    need = kda_layer_core_workspace_size(N, T, H)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=qp.device)
    wbytes = workspace.numel() * workspace.element_size()
    rc = getattr(_lib, _entry)(N, T, H, _p(qp), _p(kp), _p(vp), _p(conv_w), _p(z), _p(A), _p(b),
                             _p(beta_logit), _p(g), _p(cu_seqlens), _p(S0), float(scale),
                             float(l2_eps), float(rms_eps), _dtype_code(o.dtype), _p(o),
                             _p(S_final), _p(workspace), wbytes, _stream(stream))
    _check(_entry, rc)
    return o, S_final


def kda_layer_core_unbounded_decay(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens, S0=None,
                                   **kw):
    """kda_layer_core with Kimi Linear's unbounded decay gate (staged, fp32 intermediates)."""
    return kda_layer_core(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens, S0,
                          _entry="kda_layer_core_unbounded_decay", **kw)


def kda_layer_core_noalloc(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens, S0=None,
                           scale=DEFAULT_SCALE, l2_eps=1e-6, rms_eps=1e-6, *, o, S_final=None,
                           stream=None):
    """kda_layer_core for callers that cannot allocate device memory: the library
    supplies the scratch from a fixed array of NOALLOC_SCRATCH_BYTES bytes.
    `o` (and `S_final` if wanted) must be provided by the caller; nothing is
    allocated here.  Calls that overlap on the GPU race on the shared scratch."""
    T, H, _ = qp.shape
    N = cu_seqlens.shape[0] - 1
    rc = _lib.kda_layer_core_noalloc(N, T, H, _p(qp), _p(kp), _p(vp), _p(conv_w), _p(z), _p(A),
                                     _p(b), _p(beta_logit), _p(g), _p(cu_seqlens), _p(S0),
                                     float(scale), float(l2_eps), float(rms_eps),
                                     _dtype_code(o.dtype), _p(o), _p(S_final), _stream(stream))
    _check("kda_layer_core_noalloc", rc)
    return o, S_final


def kda_layer_core_fused(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens, S0=None,
                         scale=DEFAULT_SCALE, l2_eps=1e-6, rms_eps=1e-6, *,
                         out_dtype=torch.bfloat16, o=None, S_final=None, want_state=True,
                         stream=None, _entry="kda_layer_core_fused"):
    """The layer core in one tensor-core kernel.  Returns (o_gated, S_final or None)."""
    T, H, _ = qp.shape
    N = cu_seqlens.shape[0] - 1
    if o is None:
        o = torch.empty((T, H, HEAD_DIM), dtype=out_dtype, device=qp.device)
    if S_final is None and want_state:
        S_final = torch.empty((N, H, HEAD_DIM, HEAD_DIM), dtype=torch.float32, device=qp.device)
    rc = getattr(_lib, _entry)(N, T, H, _p(qp), _p(kp), _p(vp), _p(conv_w), _p(z), _p(A),
                               _p(b), _p(beta_logit), _p(g), _p(cu_seqlens), _p(S0),
                               float(scale), float(l2_eps), float(rms_eps),
                               _dtype_code(o.dtype), _p(o), _p(S_final), _stream(stream))
    _check(_entry, rc)
    return o, S_final


def kda_layer_core_fused_unbounded_decay(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens,
                                         S0=None, scale=DEFAULT_SCALE, l2_eps=1e-6, rms_eps=1e-6,
                                         *, out_dtype=torch.bfloat16, o=None, S_final=None,
                                         want_state=True, stream=None):
    """kda_layer_core_fused with Kimi Linear's decay gate -e^A softplus(z + b) (no floor)."""
    return kda_layer_core_fused(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens, S0,
                                scale, l2_eps, rms_eps, out_dtype=out_dtype, o=o,
                                S_final=S_final, want_state=want_state, stream=stream,
                                _entry="kda_layer_core_fused_unbounded_decay")


def kda_layer_core_fused_with_checkpoints(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens,
                                          every, S0=None, scale=DEFAULT_SCALE, l2_eps=1e-6,
                                          rms_eps=1e-6, *, ckpt_base=None, ckpt_states=None,
                                          out_dtype=torch.bfloat16, o=None, S_final=None,
                                          want_state=True, stream=None):
    """kda_layer_core_fused that also writes the recurrent state after every `every` tokens
    of each sequence.  Returns (o_gated, S_final, ckpt_base, ckpt_states)."""
    T, H, _ = qp.shape
    N = cu_seqlens.shape[0] - 1
    if o is None:
        o = torch.empty((T, H, HEAD_DIM), dtype=out_dtype, device=qp.device)
    if S_final is None and want_state:
        S_final = torch.empty((N, H, HEAD_DIM, HEAD_DIM), dtype=torch.float32, device=qp.device)
    ckpt_base, ckpt_states = _checkpoint_args(cu_seqlens, H, every, ckpt_base, ckpt_states,
                                              qp.device)
    rc = _lib.kda_layer_core_fused_with_checkpoints(
        N, T, H, _p(qp), _p(kp), _p(vp), _p(conv_w), _p(z), _p(A), _p(b), _p(beta_logit), _p(g),
        _p(cu_seqlens), _p(S0), float(scale), float(l2_eps), float(rms_eps),
        _dtype_code(o.dtype), _p(o), _p(S_final), int(every), _p(ckpt_base), _p(ckpt_states),
        _stream(stream))
    _check("kda_layer_core_fused_with_checkpoints", rc)
    return o, S_final, ckpt_base, ckpt_states


def kda_decode_layer(qp, kp, vp, conv_w, z, A, b, beta_logit, g, slot, S_pool, conv_pool,
                     scale=DEFAULT_SCALE, l2_eps=1e-6, rms_eps=1e-6, *, out_dtype=torch.bfloat16,
                     o=None, stream=None):
    """One decode step of the layer core for requests whose states sit in pools.

    qp, kp, vp, z, g: [B, H, 128] bf16; beta_logit: [B, H] bf16; slot: [B] int32 (distinct
    pool rows); S_pool: [P, H, 128, 128] fp32 and conv_pool: [P, 3, 3, H, 128] bf16, both
    updated in place.  Returns o [B, H, 128].
    """
    B, H, _ = qp.shape
    P = S_pool.shape[0]
    if o is None:
        o = torch.empty((B, H, HEAD_DIM), dtype=out_dtype, device=qp.device)
    rc = _lib.kda_decode_layer(B, H, P, _p(qp), _p(kp), _p(vp), _p(conv_w), _p(z), _p(A), _p(b),
                               _p(beta_logit), _p(g), _p(slot), _p(S_pool), _p(conv_pool),
                               float(scale), float(l2_eps), float(rms_eps), _dtype_code(o.dtype),
                               _p(o), _stream(stream))
    _check("kda_decode_layer", rc)
    return o


def kda_decode_tokens(q, k, v, log_alpha, beta, cu_tokens, slot, S_pool, write_back,
                      scale=DEFAULT_SCALE, *, S_final=None, out_dtype=None, o=None, stream=None):
    """A few tokens per request from pool rows (speculative verify: write_back=False;
    replay of accepted tokens: write_back=True).  q, k, v [T, H, 128]; log_alpha
    [T, H, 128] fp32; beta [T, H] fp32; cu_tokens [B+1] int32 and slot [B] int32 (device);
    S_pool [P, H, 128, 128] fp32.  Returns o [T, H, 128]."""
    T, H, _ = q.shape
    B = slot.shape[0]
    P = S_pool.shape[0]
    out_dtype = out_dtype or q.dtype
    if o is None:
        o = torch.empty((T, H, HEAD_DIM), dtype=out_dtype, device=q.device)
    rc = _lib.kda_decode_tokens(_dt(q), _dtype_code(o.dtype), B, H, P, T, _p(cu_tokens),
                                _p(slot), _p(q), _p(k), _p(v), _p(log_alpha), _p(beta),
                                _p(S_pool), int(bool(write_back)), _p(S_final), float(scale),
                                _p(o), _stream(stream))
    _check("kda_decode_tokens", rc)
    return o


DECODE_LAYER_MAX_TOKENS = 16  # KDA_DECODE_LAYER_MAX_TOKENS in include/kda.h


def kda_decode_layer_tokens(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_tokens, slot, S_pool,
                            conv_pool, write_back, scale=DEFAULT_SCALE, l2_eps=1e-6, rms_eps=1e-6,
                            *, out_dtype=torch.bfloat16, o=None, stream=None):
    """The layer core for a few tokens per request from pooled states (verify:
    write_back=False; replay: write_back=True).  Returns o_gated [T, H, 128]."""
    T, H, _ = qp.shape
    B = slot.shape[0]
    P = S_pool.shape[0]
    if o is None:
        o = torch.empty((T, H, HEAD_DIM), dtype=out_dtype, device=qp.device)
    rc = _lib.kda_decode_layer_tokens(B, H, P, T, _p(cu_tokens), _p(slot), _p(qp), _p(kp), _p(vp),
                                      _p(conv_w), _p(z), _p(A), _p(b), _p(beta_logit), _p(g),
                                      _p(S_pool), _p(conv_pool), int(bool(write_back)),
                                      float(scale), float(l2_eps), float(rms_eps),
                                      _dtype_code(o.dtype), _p(o), _stream(stream))
    _check("kda_decode_layer_tokens", rc)
    return o


def kda_check_prefill_inputs(cu_seqlens, log_alpha=None, total_tokens=None, num_heads=1,
                             stream=None):
    """Queue the contents checks of prefill inputs (offsets, decay range); read the result
    with kda_get_device_status.  log_alpha [T, H, 128] or [T, H] (per-head decay), or None
    to check the offsets alone against total_tokens."""
    N = cu_seqlens.shape[0] - 1
    if log_alpha is None:
        T, H, head = int(total_tokens), int(num_heads), 0
    else:
        T, H = log_alpha.shape[:2]
        head = 1 if log_alpha.dim() == 2 else 0
    rc = _lib.kda_check_prefill_inputs(N, T, H, _p(log_alpha), head, _p(cu_seqlens),
                                       _stream(stream))
    _check("kda_check_prefill_inputs", rc)


def kda_get_device_status(stream=None):
    """Synchronises the stream; returns (status_code, detail) and clears the word."""
    detail = ctypes.c_uint32(0)
    rc = _lib.kda_get_device_status(_stream(stream), ctypes.byref(detail))
    return int(rc), int(detail.value)
