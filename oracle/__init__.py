"""Plain fp64 CPU oracle for the KDA layer core.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
calls it, shares no code with it, and has no CPU fallback.

The arithmetic lives in ``kda_oracle.c`` (sequential double-precision loops,
one routine per step of the method, each citing the page it follows).  This
module only compiles that file with the host C compiler (``gcc -O2``, no
fast-math), and marshals numpy arrays into it.  ``chunked.py`` holds a second,
chunk-wise fp64 form of the recurrence that exists only to pin the chunk
algebra (it is compared against the recurrence for every chunk size).

Parity status: every routine here is pinned by ``tests/test_oracle_pins.py``
(invariants, closed forms, library special cases and brute force on tiny
inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (if stale)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_kda_prefill.argtypes = [I, I, I, I, P, P, P, P, P, P, P, D, P, P, I]
        lib.oracle_kda_decode_step.argtypes = [I, I, I, I, P, P, P, P, P, P, D, P, I]
        lib.oracle_kda_frontend.argtypes = [I, I, I, P, P, P, P, P, P, P, P, P, D,
                                            P, P, P, P, P, I]
        lib.oracle_kda_output_gate.argtypes = [ctypes.c_long, I, P, P, D, P, I]
        for f in (lib.oracle_kda_prefill, lib.oracle_kda_decode_step,
                  lib.oracle_kda_frontend, lib.oracle_kda_output_gate):
            f.restype = I
        _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def kda_prefill(q, k, v, log_alpha, beta, cu_seqlens, S0=None, scale=None,
                n_threads=None):
    """Token-by-token KDA recurrence over packed sequences (fp64).

    q, k: [T, H, dk]; v: [T, H, dv]; log_alpha: [T, H, dk]; beta: [T, H];
    cu_seqlens: [N+1] int; S0: [N, H, dk, dv] or None (zeros).
    Returns (o [T, H, dv], S_final [N, H, dk, dv]) as float64.
    """
    q, k, v, la, beta = map(_f64, (q, k, v, log_alpha, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    if scale is None:
        scale = 1.0 / np.sqrt(128.0)
    S0a = None if S0 is None else _f64(S0)
    o = np.zeros((T, H, dv), np.float64)
    Sf = np.zeros((N, H, dk, dv), np.float64)
    rc = _load().oracle_kda_prefill(N, H, dk, dv, _ptr(cu), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(la), _ptr(beta), _ptr(S0a), float(scale),
                                    _ptr(o), _ptr(Sf), n_threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_kda_prefill: invalid arguments")
    return o, Sf


def kda_decode_step(q, k, v, log_alpha, beta, S, scale=None, n_threads=None):
    """One recurrence step per (request, head).  Returns (o, S_new); S is not modified.

    q, k: [B, H, dk]; v: [B, H, dv]; log_alpha: [B, H, dk]; beta: [B, H];
    S: [B, H, dk, dv].
    """
    q, k, v, la, beta = map(_f64, (q, k, v, log_alpha, beta))
    S_new = _f64(S).copy()
    B, H, dk = q.shape
    dv = v.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(128.0)
    o = np.zeros((B, H, dv), np.float64)
    rc = _load().oracle_kda_decode_step(B, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(la),
                                        _ptr(beta), _ptr(S_new), float(scale), _ptr(o),
                                        n_threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_kda_decode_step: invalid arguments")
    return o, S_new


def kda_frontend(qp, kp, vp, conv_w, z, A, b, beta_logit, cu_seqlens, l2_eps=1e-6,
                 n_threads=None):
    """ShortConv + SiLU + L2 (q, k), ShortConv + SiLU (v), decay and write strength.

    qp, kp, vp, z: [T, H, d]; conv_w: [3, H*d, 4]; A: [H]; b: [H, d];
    beta_logit: [T, H].  Returns (q_hat, k_hat, v, log_alpha, beta) as float64.
    """
    qp, kp, vp, conv_w, z, A, b, bl = map(_f64, (qp, kp, vp, conv_w, z, A, b, beta_logit))
    T, H, d = qp.shape
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    outs = [np.zeros((T, H, d)) for _ in range(4)]
    beta = np.zeros((T, H))
    rc = _load().oracle_kda_frontend(N, H, d, _ptr(cu), _ptr(qp), _ptr(kp), _ptr(vp),
                                     _ptr(conv_w), _ptr(z), _ptr(A), _ptr(b), _ptr(bl),
                                     float(l2_eps), _ptr(outs[0]), _ptr(outs[1]),
                                     _ptr(outs[2]), _ptr(outs[3]), _ptr(beta),
                                     n_threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_kda_frontend: invalid arguments")
    return outs[0], outs[1], outs[2], outs[3], beta


def kda_output_gate(o_tilde, g, eps=1e-6, n_threads=None):
    """sigma(g) * RMSNorm(o~) per head over the last axis (unit weight)."""
    ot, g = _f64(o_tilde), _f64(g)
    d = ot.shape[-1]
    rows = ot.size // d
    out = np.zeros_like(ot)
    rc = _load().oracle_kda_output_gate(rows, d, _ptr(ot), _ptr(g), float(eps), _ptr(out),
                                        n_threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_kda_output_gate: invalid arguments")
    return out


def kda_layer_core(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens, S0=None,
                   scale=None, l2_eps=1e-6, rms_eps=1e-6, n_threads=None):
    """Front end, then the recurrence, then the output gate (all fp64).

    Returns (o_gated [T, H, d], S_final [N, H, d, d]).
    """
    qh, kh, vv, la, beta = kda_frontend(qp, kp, vp, conv_w, z, A, b, beta_logit,
                                        cu_seqlens, l2_eps, n_threads)
    ot, Sf = kda_prefill(qh, kh, vv, la, beta, cu_seqlens, S0, scale, n_threads)
    return kda_output_gate(ot, g, rms_eps, n_threads), Sf


def kda_decode_layer(qp, kp, vp, conv_w, z, A, b, beta_logit, g, slot, S_pool, conv_pool,
                     scale=None, l2_eps=1e-6, rms_eps=1e-6, n_threads=None):
    """One decode step of the layer core over pooled states (fp64); inputs are not modified.

    Follows the KDA equation list ("Kimi K3 · KDA layer") for one new token per request,
    with the request's short-convolution state (its last three pre-convolution inputs per
    channel; "Inside Kimi K3: How KDA, AttnRes, and 896 Experts Work", section "KDA writes
    corrections into a recurrent matrix") and recurrent state taken from pool row slot[b].

    qp, kp, vp, z, g: [B, H, d]; beta_logit: [B, H]; slot: [B] distinct rows of the pools;
    S_pool: [P, H, d, d]; conv_pool: [P, 3 (q, k, v), 3 (taps t-1, t-2, t-3), H, d].
    Returns (o_gated [B, H, d], S_pool_new, conv_pool_new).

    The front end of request b is the pinned sequence front end run on the 4-token
    window (x_{t-3}, x_{t-2}, x_{t-1}, x_t) as one sequence: the convolution of its last
    token is the decode convolution.  Then one recurrence step on row slot[b] of S_pool,
    then the output gate; row slot[b] of conv_pool shifts by one token.
    """
    qp, kp, vp, conv_w, z, A, b, bl, g = map(_f64, (qp, kp, vp, conv_w, z, A, b, beta_logit, g))
    S_pool, conv_pool = _f64(S_pool), _f64(conv_pool)
    slot = np.asarray(slot, dtype=np.int64)
    B, H, d = qp.shape
    P = S_pool.shape[0]
    if slot.shape != (B,) or len(set(slot.tolist())) != B or slot.min() < 0 or slot.max() >= P:
        raise ValueError("kda_decode_layer: slots must be B distinct rows in [0, P)")
    windows = []
    for s, xp in enumerate((qp, kp, vp)):
        w = np.zeros((B, 4, H, d))
        w[:, 0] = conv_pool[slot, s, 2]  # t-3
        w[:, 1] = conv_pool[slot, s, 1]  # t-2
        w[:, 2] = conv_pool[slot, s, 0]  # t-1
        w[:, 3] = xp
        windows.append(w.reshape(4 * B, H, d))
    zw = np.zeros((B, 4, H, d)); zw[:, 3] = z
    blw = np.zeros((B, 4, H)); blw[:, 3] = bl
    cu = np.arange(0, 4 * B + 1, 4, dtype=np.int32)
    qh, kh, vv, la, beta = kda_frontend(windows[0], windows[1], windows[2], conv_w,
                                        zw.reshape(4 * B, H, d), A, b, blw.reshape(4 * B, H),
                                        cu, l2_eps, n_threads)
    last = np.arange(3, 4 * B, 4)
    o_t, S_rows = kda_decode_step(qh[last], kh[last], vv[last], la[last], beta[last], S_pool[slot],
                                  scale, n_threads)
    o = kda_output_gate(o_t, g, rms_eps, n_threads)
    S_new = S_pool.copy()
    S_new[slot] = S_rows
    conv_new = conv_pool.copy()
    for s, xp in enumerate((qp, kp, vp)):
        conv_new[slot, s, 2] = conv_pool[slot, s, 1]
        conv_new[slot, s, 1] = conv_pool[slot, s, 0]
        conv_new[slot, s, 0] = xp
    return o, S_new, conv_new


def kda_decode_tokens(q, k, v, log_alpha, beta, cu_tokens, slot, S_pool, write_back, scale=None,
                      n_threads=None):
    """A few tokens per request from pooled states (fp64); inputs are not modified.

    Request b runs the recurrence over its tokens [cu_tokens[b], cu_tokens[b+1]) from
    S_pool[slot[b]]: the prefill recurrence with S0 = that row.  Speculative verify leaves
    the pool as it is (write_back false); replay of the accepted tokens writes the state
    after each request's last token back to its row (write_back true; "Inside Kimi K3: How
    KDA, AttnRes, and 896 Experts Work", section "What could go wrong").

    q, k: [T, H, dk]; v: [T, H, dv]; log_alpha: [T, H, dk]; beta: [T, H];
    cu_tokens: [B+1]; slot: [B] rows in [0, P) (distinct when write_back);
    S_pool: [P, H, dk, dv].  Returns (o [T, H, dv], S_pool_new, S_final [B, H, dk, dv]).
    """
    S_pool = _f64(S_pool)
    slot = np.asarray(slot, dtype=np.int64)
    P = S_pool.shape[0]
    B = slot.shape[0]
    cu = np.asarray(cu_tokens, dtype=np.int64)
    if cu.shape != (B + 1,) or slot.size == 0 or slot.min() < 0 or slot.max() >= P:
        raise ValueError("kda_decode_tokens: slots must lie in [0, P), one per request")
    if write_back and len(set(slot.tolist())) != B:
        raise ValueError("kda_decode_tokens: write-back needs distinct slots")
    o, S_final = kda_prefill(q, k, v, log_alpha, beta, cu.astype(np.int32), S0=S_pool[slot],
                             scale=scale, n_threads=n_threads)
    S_new = S_pool.copy()
    if write_back:
        S_new[slot] = S_final
    return o, S_new, S_final


def kda_prefill_head_decay(q, k, v, log_alpha, beta, cu_seqlens, S0=None, scale=None,
                           n_threads=None):
    """The Gated DeltaNet case (fp64): one log-decay per (token, head), log_alpha [T, H],
    shared by every key channel ("Kimi K3's Architecture: Kimi Delta Attention, Attention
    Residuals, and 896 Experts", section "Channel-wise decay, and the floor K3 puts under
    it").  The per-channel recurrence with the decay repeated over the channels."""
    la = _f64(log_alpha)
    dk = _f64(q).shape[2]
    return kda_prefill(q, k, v, np.repeat(la[:, :, None], dk, axis=2), beta, cu_seqlens, S0,
                       scale, n_threads)


def kda_decode_layer_tokens(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_tokens, slot, S_pool,
                            conv_pool, write_back, scale=None, l2_eps=1e-6, rms_eps=1e-6,
                            n_threads=None, return_o_tilde=False):
    """A few tokens per request through the whole layer core from pooled states (fp64):
    the layer-level speculative verify (write_back false: both pools unchanged) and replay
    (write_back true: each request's rows advance past its tokens).  Inputs not modified.

    Request b's tokens are rows [cu_tokens[b], cu_tokens[b+1]) of qp, kp, vp, z, g
    [T, H, d] and beta_logit [T, H]; its recurrent state is S_pool[slot[b]] and its
    short-convolution state conv_pool[slot[b]] ([3 streams][3 taps (t-1, t-2, t-3)][H][d]).
    The pinned sequence front end runs on the window (the three earlier inputs, then the
    request's tokens) as one sequence, the recurrence from the row's state over the tokens,
    then the output gate ("Kimi K3 · KDA layer", KDA equation list; "Inside Kimi K3: How
    KDA, AttnRes, and 896 Experts Work", sections "KDA writes corrections into a recurrent
    matrix" and "What could go wrong").
    Returns (o_gated [T, H, d], S_pool_new, conv_pool_new), and o~ [T, H, d] (the
    readout before the gate) as a fourth value with return_o_tilde.
    """
    qp, kp, vp, conv_w, z, A, b, bl, g = map(_f64, (qp, kp, vp, conv_w, z, A, b, beta_logit, g))
    S_pool, conv_pool = _f64(S_pool), _f64(conv_pool)
    slot = np.asarray(slot, dtype=np.int64)
    cu = np.asarray(cu_tokens, dtype=np.int64)
    B = slot.shape[0]
    T, H, d = qp.shape
    P = S_pool.shape[0]
    if cu.shape != (B + 1,) or B == 0 or slot.min() < 0 or slot.max() >= P:
        raise ValueError("kda_decode_layer_tokens: slots must lie in [0, P), one per request")
    if write_back and len(set(slot.tolist())) != B:
        raise ValueError("kda_decode_layer_tokens: write-back needs distinct slots")
    o = np.zeros((T, H, d))
    o_tilde = np.zeros((T, H, d))
    S_new, conv_new = S_pool.copy(), conv_pool.copy()
    for r in range(B):
        n, t0, t1 = slot[r], cu[r], cu[r + 1]
        m = t1 - t0
        if m == 0:
            continue
        win = []
        for s, xp in enumerate((qp, kp, vp)):
            w = np.zeros((m + 3, H, d))
            w[0], w[1], w[2] = conv_pool[n, s, 2], conv_pool[n, s, 1], conv_pool[n, s, 0]
            w[3:] = xp[t0:t1]
            win.append(w)
        zw = np.zeros((m + 3, H, d)); zw[3:] = z[t0:t1]
        blw = np.zeros((m + 3, H)); blw[3:] = bl[t0:t1]
        qh, kh, vv, la, beta = kda_frontend(win[0], win[1], win[2], conv_w, zw, A, b, blw,
                                            np.array([0, m + 3], np.int32), l2_eps, n_threads)
        ot, Sf = kda_prefill(qh[3:], kh[3:], vv[3:], la[3:], beta[3:], np.array([0, m], np.int32),
                             S0=S_pool[n:n + 1], scale=scale, n_threads=n_threads)
        o[t0:t1] = kda_output_gate(ot, g[t0:t1], rms_eps, n_threads)
        o_tilde[t0:t1] = ot
        if write_back:
            S_new[n] = Sf[0]
            for s in range(3):
                for tap in range(3):
                    conv_new[n, s, tap] = win[s][m + 2 - tap]
    if return_o_tilde:
        return o, S_new, conv_new, o_tilde
    return o, S_new, conv_new


def kimi_linear_log_decay(z, A, b):
    """Kimi Linear's unbounded decay gate (fp64): log alpha = -e^{A_h} softplus(z + b),
    in (-inf, 0) ("Kimi K3's Architecture: Kimi Delta Attention, Attention Residuals, and
    896 Experts", section "Channel-wise decay, and the floor K3 puts under it").
    z: [T, H, d]; A: [H]; b: [H, d] or None.  softplus(x) = log(1 + e^x) = logaddexp(0, x)."""
    z = _f64(z)
    x = z + (0.0 if b is None else _f64(b)[None])
    return -np.exp(_f64(A))[None, :, None] * np.logaddexp(0.0, x)


def kda_frontend_unbounded_decay(qp, kp, vp, conv_w, z, A, b, beta_logit, cu_seqlens,
                                 l2_eps=1e-6, n_threads=None):
    """The front end with Kimi Linear's decay gate: q^, k^, v and beta as kda_frontend,
    log alpha from kimi_linear_log_decay."""
    qh, kh, vv, _, beta = kda_frontend(qp, kp, vp, conv_w, z, A, b, beta_logit, cu_seqlens,
                                       l2_eps, n_threads)
    return qh, kh, vv, kimi_linear_log_decay(z, A, b), beta


def kda_layer_core_unbounded_decay(qp, kp, vp, conv_w, z, A, b, beta_logit, g, cu_seqlens,
                                   S0=None, scale=None, l2_eps=1e-6, rms_eps=1e-6,
                                   n_threads=None):
    """The layer core with Kimi Linear's decay gate (fp64): front end, the recurrence
    (which takes any log alpha <= 0), the output gate.  Returns (o_gated, S_final)."""
    qh, kh, vv, la, beta = kda_frontend_unbounded_decay(qp, kp, vp, conv_w, z, A, b, beta_logit,
                                                        cu_seqlens, l2_eps, n_threads)
    ot, Sf = kda_prefill(qh, kh, vv, la, beta, cu_seqlens, S0, scale, n_threads)
    return kda_output_gate(ot, g, rms_eps, n_threads), Sf
