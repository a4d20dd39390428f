"""Pins for the fp64 oracle: each check ties it to something other than itself.

A plausible slip in the oracle (readout before the write, decay of columns
instead of rows, a transposed state, a dropped beta, conv taps reversed, no
zero history at a sequence start, RMS over the wrong axis) fails at least one
of these.  Sources, by page:
  [SGLang]     "Kimi K3: Architecture and SGLang Day-0 Support"
  [Arch-K3]    "Kimi K3's Architecture: Kimi Delta Attention, Attention Residuals,
               and 896 Experts"
  [KDA-layer]  "Kimi K3 · KDA layer" (OpenModelAtlas), the KDA equation list
  [Inside-K3]  "Inside Kimi K3: How KDA, AttnRes, and 896 Experts Work"
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.chunked import kda_chunked_single

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(20261202)


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_problem(T, H, dk, dv, la_lo=-5.0, s0=True, rng=RNG):
    q = unit(rng.standard_normal((T, H, dk)))
    k = unit(rng.standard_normal((T, H, dk)))
    v = rng.standard_normal((T, H, dv))
    la = rng.uniform(la_lo, 0.0, (T, H, dk))
    beta = rng.uniform(0.0, 1.0, (T, H))
    S0 = rng.standard_normal((1, H, dk, dv)) * 0.3 if s0 else None
    return q, k, v, la, beta, S0


# --------------------------------------------------------------------------
# P1  read-after-write [SGLang, "Math details: how KDA gates ..."], [Arch-K3,
#     "Deriving the delta rule"]: for unit k, S_t^T k_t = (1-b) r_old + b v_t,
#     r_old = (Diag(alpha_t) S_{t-1})^T k_t.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dk,dv", [(128, 128), (4, 3), (2, 1)])
def test_read_after_write(dk, dv):
    B, H = 3, 2
    q = unit(RNG.standard_normal((B, H, dk)))
    k = unit(RNG.standard_normal((B, H, dk)))
    v = RNG.standard_normal((B, H, dv))
    la = RNG.uniform(-5, 0, (B, H, dk))
    beta = RNG.uniform(0, 1, (B, H))
    S = RNG.standard_normal((B, H, dk, dv))
    _, S_new = oracle.kda_decode_step(q, k, v, la, beta, S, scale=1.0)
    for b in range(B):
        for h in range(H):
            r_old = (np.exp(la[b, h])[:, None] * S[b, h]).T @ k[b, h]
            want = (1 - beta[b, h]) * r_old + beta[b, h] * v[b, h]
            got = S_new[b, h].T @ k[b, h]
            np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * (1 + np.abs(want).max()))


# --------------------------------------------------------------------------
# P2  alpha = 1, beta = 1, orthonormal keys: every key reads back the value it
#     was last written with, in any write order [SGLang crosstalk term: the
#     readout is crosstalk-free iff keys are pairwise orthogonal, at most d_k
#     of them], [Arch-K3]: at beta = 1 the read returns v_t exactly.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("d", [8, 128])
def test_orthonormal_keys_exact_recall(d):
    Qm, _ = np.linalg.qr(RNG.standard_normal((d, d)))
    keys = Qm.T                                  # rows are orthonormal
    order = list(RNG.permutation(d)) + list(RNG.permutation(d)[: d // 2])
    T = len(order)
    k = keys[order][:, None, :]
    v = RNG.standard_normal((T, 1, d))
    last = {}
    for t, i in enumerate(order):
        last[i] = v[t, 0]
    q = k.copy()
    la = np.zeros((T, 1, d))
    beta = np.ones((T, 1))
    o, Sf = oracle.kda_prefill(q, k, v, la, beta, [0, T], S0=None, scale=1.0)
    for i, val in last.items():
        np.testing.assert_allclose(Sf[0, 0].T @ keys[i], val, atol=1e-10)
    # the readout of the token just written is its own value (newest write is exact)
    np.testing.assert_allclose(o[:, 0, :], v[:, 0, :], atol=1e-10)


# --------------------------------------------------------------------------
# P3  beta = 0: no rewrite, the state only decays [SGLang: "beta_t = 0 keeps
#     everything"].  S_T = Diag(prod alpha) S0 and o_t = scale (Diag(prod_{u<=t}
#     alpha_u) S0)^T q_t.
# --------------------------------------------------------------------------
def test_beta_zero_pure_decay():
    T, H, dk, dv = 9, 2, 6, 5
    q, k, v, la, _, S0 = rand_problem(T, H, dk, dv)
    beta = np.zeros((T, H))
    o, Sf = oracle.kda_prefill(q, k, v, la, beta, [0, T], S0=S0, scale=0.5)
    for h in range(H):
        cum = np.cumsum(la[:, h, :], axis=0)
        for t in range(T):
            St = np.exp(cum[t])[:, None] * S0[0, h]
            np.testing.assert_allclose(o[t, h], 0.5 * St.T @ q[t, h], atol=1e-13)
        np.testing.assert_allclose(Sf[0, h], np.exp(cum[-1])[:, None] * S0[0, h], atol=1e-13)


# --------------------------------------------------------------------------
# P4  alpha = 0 (log alpha = -inf): the old state is wiped, S_t = beta k v^T.
# --------------------------------------------------------------------------
def test_alpha_zero_resets_state():
    B, H, dk, dv = 2, 3, 5, 4
    q = unit(RNG.standard_normal((B, H, dk)))
    k = unit(RNG.standard_normal((B, H, dk)))
    v = RNG.standard_normal((B, H, dv))
    la = np.full((B, H, dk), -np.inf)
    beta = RNG.uniform(0, 1, (B, H))
    S = RNG.standard_normal((B, H, dk, dv)) * 10
    o, S_new = oracle.kda_decode_step(q, k, v, la, beta, S, scale=0.25)
    for b in range(B):
        for h in range(H):
            want = beta[b, h] * np.outer(k[b, h], v[b, h])
            np.testing.assert_allclose(S_new[b, h], want, atol=1e-14)
            np.testing.assert_allclose(o[b, h], 0.25 * beta[b, h] * (k[b, h] @ q[b, h]) * v[b, h],
                                       atol=1e-14)


# --------------------------------------------------------------------------
# P5  the 2-D worked example [SGLang, DeltaNet / KDA diagrams and the crosstalk
#     term], values stored under tests/golden with their citation.
# --------------------------------------------------------------------------
def test_worked_example_2d():
    with open(os.path.join(GOLDEN, "worked_example_2d.json")) as f:
        ex = json.load(f)
    keys = {n: np.array(x) for n, x in ex["keys"].items()}
    for case in ex["cases"]:
        T = len(case["writes"])
        k = np.array([keys[n] for n, _ in case["writes"]])[:, None, :]
        v = np.array([[val] for _, val in case["writes"]])[:, None, :]
        la = np.array(case["log_alpha"], dtype=np.float64)[:, None, :]
        beta = np.array(case["beta"])[:, None]
        _, Sf = oracle.kda_prefill(k, k, v, la, beta, [0, T], S0=None, scale=1.0)
        got = float((Sf[0, 0].T @ keys[case["query"]])[0])
        assert got == pytest.approx(case["kda_expected"], abs=1e-12), case["name"]
        if "naive_expected" in case:   # contrast: plain accumulation S = sum k v^T
            S_naive = sum(np.outer(k[t, 0], v[t, 0]) for t in range(T))
            assert float((S_naive.T @ keys[case["query"]])[0]) == pytest.approx(
                case["naive_expected"], abs=1e-12)


def test_crosstalk_non_orthogonal():
    """Write (k_a, v_a) then (k_b, v_b), beta = alpha = 1, cos(theta) = c.
    The delta write along k_b first removes its prediction c v_a, so reading k_a
    gives v_a + c (v_b - c v_a) = (1 - c^2) v_a + c v_b (from the crosstalk term
    o_a = v_a + cos(theta) v_b of [SGLang] applied to the corrected write)."""
    for theta in (0.3, 1.0, math.pi / 2):
        c = math.cos(theta)
        ka = np.array([1.0, 0.0])
        kb = np.array([c, math.sin(theta)])
        va, vb = 1.5, -0.7
        k = np.stack([ka, kb])[:, None, :]
        v = np.array([[va], [vb]])[:, None, :]
        _, Sf = oracle.kda_prefill(k, k, v, np.zeros((2, 1, 2)), np.ones((2, 1)), [0, 2],
                                   scale=1.0)
        assert float((Sf[0, 0].T @ ka)[0]) == pytest.approx((1 - c * c) * va + c * vb, abs=1e-12)


# --------------------------------------------------------------------------
# P6  unrolled product form [SGLang]: S_t = sum_{s<=t} [prod_{u=s+1..t}
#     (I - b_u k_u k_u^T) Diag(alpha_u)] b_s k_s v_s^T  (S0 = 0), by explicit
#     d x d matrix products; single-form update (I - b k k^T) Diag(alpha) S + b k v^T
#     [Inside-K3] also checked step by step.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dk,dv,T", [(2, 1, 5), (3, 2, 8), (4, 4, 8)])
def test_unrolled_product_form(dk, dv, T):
    q, k, v, la, beta, _ = rand_problem(T, 1, dk, dv, s0=False)
    o, Sf = oracle.kda_prefill(q, k, v, la, beta, [0, T], S0=None, scale=1.0)
    I = np.eye(dk)
    for t in range(T):
        St = np.zeros((dk, dv))
        for s in range(t + 1):
            M = I.copy()
            for u in range(s + 1, t + 1):
                M = (I - beta[u, 0] * np.outer(k[u, 0], k[u, 0])) @ np.diag(np.exp(la[u, 0])) @ M
            St += M @ (beta[s, 0] * np.outer(k[s, 0], v[s, 0]))
        np.testing.assert_allclose(o[t, 0], St.T @ q[t, 0], atol=1e-12)
    # single-form step
    S = np.zeros((dk, dv))
    for t in range(T):
        S = (I - beta[t, 0] * np.outer(k[t, 0], k[t, 0])) @ np.diag(np.exp(la[t, 0])) @ S \
            + beta[t, 0] * np.outer(k[t, 0], v[t, 0])
    np.testing.assert_allclose(Sf[0, 0], S, atol=1e-12)


# --------------------------------------------------------------------------
# P7  the delta write is one gradient step [Arch-K3, "Deriving the delta rule"]:
#     S_t = S' - beta grad_S 1/2 ||S^T k - v||^2 at S' = Diag(alpha) S_{t-1}.
#     The gradient comes from autograd, not from the formula.
# --------------------------------------------------------------------------
def test_gradient_step_form():
    dk, dv = 6, 5
    S = RNG.standard_normal((1, 1, dk, dv))
    k = RNG.standard_normal((1, 1, dk))        # no unit norm needed for this identity
    v = RNG.standard_normal((1, 1, dv))
    q = RNG.standard_normal((1, 1, dk))
    la = RNG.uniform(-2, 0, (1, 1, dk))
    beta = np.array([[0.37]])
    _, S_new = oracle.kda_decode_step(q, k, v, la, beta, S, scale=1.0)
    Sd = torch.tensor(np.exp(la[0, 0])[:, None] * S[0, 0], requires_grad=True)
    loss = 0.5 * ((Sd.T @ torch.tensor(k[0, 0]) - torch.tensor(v[0, 0])) ** 2).sum()
    loss.backward()
    want = (Sd - 0.37 * Sd.grad).detach().numpy()
    np.testing.assert_allclose(S_new[0, 0], want, atol=1e-13)


# --------------------------------------------------------------------------
# P8  chunk-wise fp64 form == token-by-token recurrence for EVERY chunk size,
#     with S0 != 0 and partial last chunks.  Pins the chunk algebra the GPU uses.
# --------------------------------------------------------------------------
def test_chunked_equals_recurrent_every_chunk_size():
    T, dk, dv = 37, 8, 8
    q, k, v, la, beta, S0 = rand_problem(T, 1, dk, dv)
    o_ref, S_ref = oracle.kda_prefill(q, k, v, la, beta, [0, T], S0=S0, scale=0.3)
    for C in range(1, T + 1):
        o, S = kda_chunked_single(q[:, 0], k[:, 0], v[:, 0], la[:, 0], beta[:, 0], S0[0, 0],
                                  C, 0.3)
        np.testing.assert_allclose(o, o_ref[:, 0], atol=1e-11, err_msg=f"C={C}")
        np.testing.assert_allclose(S, S_ref[0, 0], atol=1e-11, err_msg=f"C={C}")


@pytest.mark.parametrize("C", [16, 64])
def test_chunked_equals_recurrent_d128(C):
    T, d = 200, 128
    q, k, v, la, beta, S0 = rand_problem(T, 1, d, d)
    o_ref, S_ref = oracle.kda_prefill(q, k, v, la, beta, [0, T], S0=S0)
    o, S = kda_chunked_single(q[:, 0], k[:, 0], v[:, 0], la[:, 0], beta[:, 0], S0[0, 0], C,
                              1 / math.sqrt(128))
    np.testing.assert_allclose(o, o_ref[:, 0], atol=1e-11)
    np.testing.assert_allclose(S, S_ref[0, 0], atol=1e-11)


# --------------------------------------------------------------------------
# P11 the decay floor [Arch-K3, "Channel-wise decay ..."]: log alpha = -5
#     everywhere keeps every quantity finite; a 16-token tile sums to -80 at
#     most and e^80 < bf16/fp32 max.
# --------------------------------------------------------------------------
def test_decay_floor_finite():
    assert 16 * -5.0 == -80.0
    assert math.exp(80.0) < float(torch.finfo(torch.bfloat16).max)
    assert math.exp(80.0) < float(torch.finfo(torch.float32).max)
    T, H, d = 70, 1, 16
    q, k, v, _, beta, S0 = rand_problem(T, H, d, d)
    la = np.full((T, H, d), -5.0)
    o, Sf = oracle.kda_prefill(q, k, v, la, beta, [0, T], S0=S0)
    assert np.isfinite(o).all() and np.isfinite(Sf).all()
    o2, S2 = kda_chunked_single(q[:, 0], k[:, 0], v[:, 0], la[:, 0], beta[:, 0], S0[0, 0], 64,
                                1 / math.sqrt(128))
    np.testing.assert_allclose(o2, o[:, 0], atol=1e-11)


# --------------------------------------------------------------------------
# P12 splitting a sequence: prefill(T1) then prefill(T2) from its final state
#     == prefill(T1 + T2); decode applied T times == prefill(T).
# --------------------------------------------------------------------------
def test_resume_and_decode_equal_prefill():
    T, H, d = 12, 2, 8
    q, k, v, la, beta, S0 = rand_problem(T, H, d, d)
    o_ref, S_ref = oracle.kda_prefill(q, k, v, la, beta, [0, T], S0=S0)
    o1, S1 = oracle.kda_prefill(q[:5], k[:5], v[:5], la[:5], beta[:5], [0, 5], S0=S0)
    o2, S2 = oracle.kda_prefill(q[5:], k[5:], v[5:], la[5:], beta[5:], [0, T - 5], S0=S1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o_ref, atol=1e-13)
    np.testing.assert_allclose(S2, S_ref, atol=1e-13)
    S = S0.copy()
    for t in range(T):
        o_t, S = oracle.kda_decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1],
                                        beta[t:t + 1], S)
        np.testing.assert_allclose(o_t[0], o_ref[t], atol=1e-13)
    np.testing.assert_allclose(S, S_ref, atol=1e-13)


# --------------------------------------------------------------------------
# P13 varlen packing: sequences are independent; a zero-length sequence keeps
#     its S0 and writes nothing.
# --------------------------------------------------------------------------
def test_varlen_independence_and_empty():
    lens = [5, 0, 9, 1]
    T, H, d = sum(lens), 2, 4
    q, k, v, la, beta, _ = rand_problem(T, H, d, d)
    S0 = RNG.standard_normal((len(lens), H, d, d))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, Sf = oracle.kda_prefill(q, k, v, la, beta, cu, S0=S0)
    for n, L in enumerate(lens):
        a, b = cu[n], cu[n + 1]
        o_n, S_n = oracle.kda_prefill(q[a:b], k[a:b], v[a:b], la[a:b], beta[a:b], [0, L],
                                      S0=S0[n:n + 1])
        np.testing.assert_array_equal(o[a:b], o_n)
        np.testing.assert_array_equal(Sf[n], S_n[0])
    np.testing.assert_array_equal(Sf[1], S0[1])


# --------------------------------------------------------------------------
# Front end [KDA-layer]; [Inside-K3, "Short convolutions ..."].
# --------------------------------------------------------------------------
def _frontend_inputs(lens, H, d, rng=RNG):
    T = sum(lens)
    qp, kp, vp, z = (rng.standard_normal((T, H, d)) for _ in range(4))
    conv_w = rng.standard_normal((3, H * d, 4)) * 0.5
    A = rng.standard_normal(H) * 0.5
    b = rng.standard_normal((H, d)) * 0.1
    bl = rng.standard_normal((T, H))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return qp, kp, vp, conv_w, z, A, b, bl, cu


def test_frontend_conv_matches_library_filter():
    """Depthwise causal conv == scipy.signal.lfilter per channel and sequence
    (zero initial conditions at each sequence start), SiLU == torch silu,
    L2 == division by numpy's norm."""
    from scipy.signal import lfilter
    lens = [7, 1, 12]
    H, d = 2, 8
    qp, kp, vp, conv_w, z, A, b, bl, cu = _frontend_inputs(lens, H, d)
    qh, kh, vv, la, beta = oracle.kda_frontend(qp, kp, vp, conv_w, z, A, b, bl, cu, l2_eps=0.0)
    for s, (xp, out) in enumerate(((qp, qh), (kp, kh), (vp, vv))):
        pre = np.zeros_like(xp)
        for n in range(len(lens)):
            a_, b_ = cu[n], cu[n + 1]
            for h in range(H):
                for i in range(d):
                    pre[a_:b_, h, i] = lfilter(conv_w[s, h * d + i], [1.0], xp[a_:b_, h, i])
        act = torch.nn.functional.silu(torch.tensor(pre)).numpy()
        if s < 2:
            act = act / np.linalg.norm(act, axis=-1, keepdims=True)
        np.testing.assert_allclose(out, act, atol=1e-12)


def test_frontend_one_hot_taps_shift():
    """Tap j alone reproduces SiLU(x_{t-j}), zero before each sequence start
    (catches reversed taps and history leaking across sequences)."""
    lens = [6, 5]
    H, d = 1, 4
    qp, kp, vp, conv_w, z, A, b, bl, cu = _frontend_inputs(lens, H, d)
    for j in range(4):
        w = np.zeros((3, H * d, 4))
        w[:, :, j] = 1.0
        _, _, vv, _, _ = oracle.kda_frontend(qp, kp, vp, w, z, A, b, bl, cu)
        for n in range(2):
            for t in range(cu[n], cu[n + 1]):
                src = vp[t - j] if t - j >= cu[n] else np.zeros((H, d))
                want = torch.nn.functional.silu(torch.tensor(src)).numpy()
                np.testing.assert_allclose(vv[t], want, atol=1e-14)


def test_frontend_gate_parameters():
    """log alpha in (-5, 0) with the special values -5 sigma(0) = -2.5 at
    z + b = 0 and the limits -5 / 0; beta = sigma(w) == scipy expit."""
    from scipy.special import expit
    lens = [10]
    H, d = 3, 8
    qp, kp, vp, conv_w, z, A, b, bl, cu = _frontend_inputs(lens, H, d)
    _, _, _, la, beta = oracle.kda_frontend(qp, kp, vp, conv_w, z, A, b, bl, cu)
    np.testing.assert_allclose(beta, expit(bl), atol=1e-15)
    assert (la < 0).all() and (la > -5).all()
    z0 = -np.broadcast_to(b, z.shape).copy()
    _, _, _, la0, _ = oracle.kda_frontend(qp, kp, vp, conv_w, z0, A, b, bl, cu)
    np.testing.assert_allclose(la0, -2.5, atol=1e-15)
    big = np.full_like(z, 50.0)
    _, _, _, la_hi, _ = oracle.kda_frontend(qp, kp, vp, conv_w, big, np.full(H, 2.0), b, bl, cu)
    np.testing.assert_allclose(la_hi, -5.0, atol=1e-12)
    _, _, _, la_lo, _ = oracle.kda_frontend(qp, kp, vp, conv_w, -big, np.full(H, 2.0), b, bl, cu)
    np.testing.assert_allclose(la_lo, 0.0, atol=1e-12)
    # the scale e^{A_h} is per head: compare sigma through scipy for each head
    for h in range(H):
        want = -5.0 * expit(np.exp(A[h]) * (z[:, h, :] + b[h]))
        np.testing.assert_allclose(la[:, h, :], want, atol=1e-14)


# --------------------------------------------------------------------------
# Output gate [KDA-layer]: o^g = sigma(g) RMSNorm(o~) per head.
# --------------------------------------------------------------------------
def test_output_gate_matches_torch_rms_norm():
    from scipy.special import expit
    ot = RNG.standard_normal((5, 3, 128)) * 0.01
    g = RNG.standard_normal((5, 3, 128))
    out = oracle.kda_output_gate(ot, g, eps=1e-6)
    rms = torch.nn.functional.rms_norm(torch.tensor(ot), (128,), eps=1e-6).numpy()
    np.testing.assert_allclose(out, expit(g) * rms, atol=1e-13)


def test_output_gate_scale_invariance_and_constant():
    ot = RNG.standard_normal((4, 2, 128))
    g = RNG.standard_normal((4, 2, 128))
    a = oracle.kda_output_gate(ot, g, eps=0.0)
    b = oracle.kda_output_gate(ot * 37.0, g, eps=0.0)
    np.testing.assert_allclose(a, b, atol=1e-13)
    c = oracle.kda_output_gate(np.full((1, 1, 128), -3.0), np.zeros((1, 1, 128)), eps=0.0)
    np.testing.assert_allclose(c, -0.5, atol=1e-15)


def test_state_size_figures():
    """Per layer 96 heads x 128 x 128 = 1,572,864 state elements [Inside-K3];
    69 KDA layers x 12 heads per GPU (TP 8) x 128^2 x 4 bytes = 54.3 MB, which
    matches the quoted ~54 MB per request per GPU [SGLang] only for fp32 state."""
    assert 96 * 128 * 128 == 1_572_864
    mb = 69 * (96 // 8) * 128 * 128 * 4 / 1e6
    assert 53.5 < mb < 55.0
    assert not (53.5 < mb / 2 < 55.0)


# --------------------------------------------------------------------------
# P15 decode step of the layer core over pooled states: the layer core over
#     T0 tokens, then one decode_layer step per further token (convolution
#     state = the last three pre-convolution inputs, zero before the sequence
#     start; recurrent state = the layer core's S_final, placed in an arbitrary
#     pool row) reproduces the layer core over all T tokens, output by output;
#     pool rows of other requests are untouched; the convolution state shifts.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T0", [0, 1, 2, 5])
def test_decode_layer_continues_the_layer_core(T0):
    T, H, d, P = T0 + 4, 2, 8, 3
    rng = np.random.default_rng(700 + T0)
    qp, kp, vp, z, g = (rng.standard_normal((T, H, d)) for _ in range(5))
    conv_w = rng.standard_normal((3, H * d, 4)) * 0.5
    A = rng.standard_normal(H) * 0.5
    b = rng.standard_normal((H, d)) * 0.3
    bl = rng.standard_normal((T, H))
    S0 = rng.standard_normal((1, H, d, d)) * 0.3
    ref_o, ref_S = oracle.kda_layer_core(qp, kp, vp, conv_w, z, A, b, bl, g, [0, T], S0=S0)
    row = 1  # this request's pool row; rows 0 and 2 belong to other requests
    S_pool = rng.standard_normal((P, H, d, d))
    conv_pool = rng.standard_normal((P, 3, 3, H, d))
    if T0 > 0:
        o0, S_T0 = oracle.kda_layer_core(qp[:T0], kp[:T0], vp[:T0], conv_w, z[:T0], A, b, bl[:T0],
                                         g[:T0], [0, T0], S0=S0)
        np.testing.assert_allclose(o0, ref_o[:T0], atol=1e-12)
        S_pool[row] = S_T0[0]
    else:
        S_pool[row] = S0[0]
    for s, xp in enumerate((qp, kp, vp)):  # the last three inputs before token T0
        for tap in range(3):
            t = T0 - 1 - tap
            conv_pool[row, s, tap] = xp[t] if t >= 0 else 0.0
    others = [r for r in range(P) if r != row]
    S_others, conv_others = S_pool[others].copy(), conv_pool[others].copy()
    for t in range(T0, T):
        sl = slice(t, t + 1)
        o, S_pool_new, conv_new = oracle.kda_decode_layer(qp[sl], kp[sl], vp[sl], conv_w, z[sl], A, b,
                                                          bl[sl], g[sl], [row], S_pool, conv_pool)
        np.testing.assert_allclose(o[0], ref_o[t], atol=1e-12)
        for s, xp in enumerate((qp, kp, vp)):
            np.testing.assert_array_equal(conv_new[row, s, 0], xp[t])
            np.testing.assert_array_equal(conv_new[row, s, 1], conv_pool[row, s, 0])
            np.testing.assert_array_equal(conv_new[row, s, 2], conv_pool[row, s, 1])
        S_pool, conv_pool = S_pool_new, conv_new
    np.testing.assert_allclose(S_pool[row], ref_S[0], atol=1e-12)
    np.testing.assert_array_equal(S_pool[others], S_others)
    np.testing.assert_array_equal(conv_pool[others], conv_others)


def test_decode_layer_rejects_repeated_or_out_of_range_slots():
    H, d, P = 1, 4, 2
    x = np.zeros((2, H, d))
    args = (x, x, x, np.zeros((3, H * d, 4)), x, np.zeros(H), np.zeros((H, d)), np.zeros((2, H)), x)
    S_pool, conv_pool = np.zeros((P, H, d, d)), np.zeros((P, 3, 3, H, d))
    for slots in ([0, 0], [0, 2], [-1, 1]):
        with pytest.raises(ValueError):
            oracle.kda_decode_layer(*args, slots, S_pool, conv_pool)


# P16 several tokens per request from pooled states (speculative verify and replay):
#     the same as one decode step per token on the request's row, taken in order;
#     verify leaves the pool untouched (and may share a row), replay advances only the
#     rows it names ("Inside Kimi K3: How KDA, AttnRes, and 896 Experts Work", section
#     "What could go wrong": accepted inputs are replayed).
def test_decode_tokens_equals_decode_steps():
    H, d, P = 2, 8, 5
    lens, slot = [3, 0, 1, 4], [4, 0, 2, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    rng = np.random.default_rng(800)
    q, k = (unit(rng.standard_normal((T, H, d))) for _ in range(2))
    v = rng.standard_normal((T, H, d))
    la = -5.0 / (1.0 + np.exp(-rng.standard_normal((T, H, d)) * 2))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S_pool = rng.standard_normal((P, H, d, d)) * 0.3
    for wb in (False, True):
        o, S_new, S_fin = oracle.kda_decode_tokens(q, k, v, la, beta, cu, slot, S_pool, wb)
        for b, n in enumerate(slot):
            S = S_pool[n:n + 1]
            for t in range(cu[b], cu[b + 1]):
                sl = slice(t, t + 1)
                ot, S = oracle.kda_decode_step(q[sl], k[sl], v[sl], la[sl], beta[sl], S)
                np.testing.assert_allclose(o[t], ot[0], atol=1e-12)
            np.testing.assert_allclose(S_fin[b], S[0], atol=1e-12)
            np.testing.assert_array_equal(S_new[n], S[0] if wb else S_pool[n])
        untouched = sorted(set(range(P)) - set(slot))
        np.testing.assert_array_equal(S_new[untouched], S_pool[untouched])


def test_decode_tokens_verify_then_replay():
    """Verify a 4-token draft from a row, accept the first 2 (the draft's outputs for them
    are the accepted outputs), replay them: the row equals the prefill over the accepted
    prefix, and verifying the rest of the draft from it reproduces the draft's outputs."""
    H, d = 2, 8
    rng = np.random.default_rng(801)
    q, k = (unit(rng.standard_normal((4, H, d))) for _ in range(2))
    v = rng.standard_normal((4, H, d))
    la = -5.0 / (1.0 + np.exp(-rng.standard_normal((4, H, d)) * 2))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((4, H))))
    S_pool = rng.standard_normal((2, H, d, d)) * 0.3
    o_draft, S_v, _ = oracle.kda_decode_tokens(q, k, v, la, beta, [0, 4], [1], S_pool, False)
    np.testing.assert_array_equal(S_v, S_pool)
    a = slice(0, 2)
    _, S_r, _ = oracle.kda_decode_tokens(q[a], k[a], v[a], la[a], beta[a], [0, 2], [1], S_pool, True)
    _, S_pre = oracle.kda_prefill(q[a], k[a], v[a], la[a], beta[a], [0, 2], S0=S_pool[1:2])
    np.testing.assert_allclose(S_r[1], S_pre[0], atol=1e-12)
    np.testing.assert_array_equal(S_r[0], S_pool[0])
    r = slice(2, 4)
    o_rest, _, _ = oracle.kda_decode_tokens(q[r], k[r], v[r], la[r], beta[r], [0, 2], [1], S_r, False)
    np.testing.assert_allclose(o_rest, o_draft[2:], atol=1e-12)


def test_decode_tokens_rejects_bad_slots():
    z = np.zeros((2, 1, 4))
    S = np.zeros((3, 1, 4, 4))
    zb = np.zeros((2, 1))
    with pytest.raises(ValueError):
        oracle.kda_decode_tokens(z, z, z, z, zb, [0, 1, 2], [0, 3], S, False)
    with pytest.raises(ValueError):
        oracle.kda_decode_tokens(z, z, z, z, zb, [0, 1, 2], [1, 1], S, True)
    oracle.kda_decode_tokens(z, z, z, z, zb, [0, 1, 2], [1, 1], S, False)  # shared row: verify only


# P17 the Gated DeltaNet case [Arch-K3, "Channel-wise decay, and the floor K3 puts under
#     it": one decay per head]: with Diag(alpha) = alpha I the recurrence is the scalar-gated
#     delta rule S_t = alpha_t (I - beta_t k k^T) S_{t-1} + beta_t k v^T, written here with
#     plain matrix products, and o_t = scale S_t^T q_t.
def test_head_decay_is_the_scalar_gated_delta_rule():
    T, H, d = 9, 2, 6
    rng = np.random.default_rng(900)
    q = unit(rng.standard_normal((T, H, d)))
    k = unit(rng.standard_normal((T, H, d)))
    v = rng.standard_normal((T, H, d))
    la = -5.0 / (1.0 + np.exp(-rng.standard_normal((T, H)) * 2))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    S0 = rng.standard_normal((1, H, d, d)) * 0.3
    o, Sf = oracle.kda_prefill_head_decay(q, k, v, la, beta, [0, T], S0=S0, scale=0.5)
    for h in range(H):
        S = S0[0, h].copy()
        for t in range(T):
            kk = k[t, h][:, None]
            S = np.exp(la[t, h]) * (np.eye(d) - beta[t, h] * kk @ kk.T) @ S + beta[t, h] * kk @ v[t, h][None, :]
            np.testing.assert_allclose(o[t, h], 0.5 * S.T @ q[t, h], atol=1e-12)
        np.testing.assert_allclose(Sf[0, h], S, atol=1e-12)


# P18 a few tokens per request through the layer core from pooled states == one
#     decode-layer step (P15) per token, in order; verify leaves both pools as they are.
def test_decode_layer_tokens_equals_decode_layer_steps():
    H, d, P = 2, 8, 5
    lens, slot = [3, 0, 1, 5], [4, 0, 2, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    rng = np.random.default_rng(1000)
    qp, kp, vp, z, g = (rng.standard_normal((T, H, d)) for _ in range(5))
    conv_w = rng.standard_normal((3, H * d, 4)) * 0.5
    A = rng.standard_normal(H) * 0.5
    b = rng.standard_normal((H, d)) * 0.3
    bl = rng.standard_normal((T, H))
    S_pool = rng.standard_normal((P, H, d, d)) * 0.3
    conv_pool = rng.standard_normal((P, 3, 3, H, d))
    for wb in (False, True):
        o, S_new, conv_new = oracle.kda_decode_layer_tokens(qp, kp, vp, conv_w, z, A, b, bl, g, cu,
                                                            slot, S_pool, conv_pool, wb)
        if not wb:
            np.testing.assert_array_equal(S_new, S_pool)
            np.testing.assert_array_equal(conv_new, conv_pool)
        for r, n in enumerate(slot):
            S_row, c_row = S_pool.copy(), conv_pool.copy()
            for t in range(cu[r], cu[r + 1]):
                sl = slice(t, t + 1)
                ot, S_row, c_row = oracle.kda_decode_layer(qp[sl], kp[sl], vp[sl], conv_w, z[sl], A, b,
                                                           bl[sl], g[sl], [n], S_row, c_row)
                np.testing.assert_allclose(o[t], ot[0], atol=1e-12)
            if wb:
                np.testing.assert_allclose(S_new[n], S_row[n], atol=1e-12)
                np.testing.assert_array_equal(conv_new[n], c_row[n])
        untouched = sorted(set(range(P)) - set(slot))
        np.testing.assert_array_equal(S_new[untouched], S_pool[untouched])
        np.testing.assert_array_equal(conv_new[untouched], conv_pool[untouched])


# P19 Kimi Linear's unbounded decay gate [Arch-K3, "Channel-wise decay, and the floor K3
#     puts under it": g = -e^A softplus(z)]: closed forms of softplus (ln 2 at 0; x + e^-x
#     to first order for large x; e^x for very negative x), the range (-inf, 0), per-head
#     scaling by e^A, b added before the softplus; and decays far below K3's floor of -5
#     (and -inf) go through the recurrence exactly as P3/P4 say.
def test_kimi_linear_gate_closed_forms():
    A = np.array([0.0, np.log(3.0)])
    z = np.zeros((1, 2, 4))
    z[0, :, 1] = 30.0
    z[0, :, 2] = -30.0
    z[0, :, 3] = 1.0
    la = oracle.kimi_linear_log_decay(z, A, None)
    for h, eA in enumerate([1.0, 3.0]):
        np.testing.assert_allclose(la[0, h, 0], -eA * np.log(2.0), rtol=1e-15)
        np.testing.assert_allclose(la[0, h, 1], -eA * (30.0 + np.exp(-30.0)), rtol=1e-15)
        np.testing.assert_allclose(la[0, h, 2], -eA * np.exp(-30.0), rtol=1e-12)
        np.testing.assert_allclose(la[0, h, 3], -eA * np.log(1.0 + np.e), rtol=1e-15)
    b = np.full((2, 4), 0.5)
    np.testing.assert_allclose(oracle.kimi_linear_log_decay(z - 0.5, A, b), la, rtol=1e-15)
    zz = np.random.default_rng(1100).standard_normal((50, 2, 4)) * 10
    assert (oracle.kimi_linear_log_decay(zz, A, None) < 0).all()


def test_unbounded_decays_in_the_recurrence():
    T, H, d = 6, 1, 4
    rng = np.random.default_rng(1101)
    q = unit(rng.standard_normal((T, H, d)))
    k = unit(rng.standard_normal((T, H, d)))
    v = rng.standard_normal((T, H, d))
    beta = np.full((T, H), 0.5)
    S0 = rng.standard_normal((1, H, d, d))
    la = np.full((T, H, d), -40.0)   # far below the floor: e^-40 ~ 4e-18 per step
    la[3] = -np.inf                  # a full reset at token 3
    o, Sf = oracle.kda_prefill(q, k, v, la, beta, [0, T], S0=S0)
    assert np.isfinite(o).all() and np.isfinite(Sf).all()
    # after the reset only tokens 3..5 write; each earlier state is scaled by e^-40 per step
    S = np.zeros((d, d))
    for t in range(3, T):
        a = 0.0 if t == 3 else np.exp(-40.0)
        S = a * S
        S = S + beta[t, 0] * np.outer(k[t, 0], v[t, 0] - S.T @ k[t, 0])
    np.testing.assert_allclose(Sf[0, 0], S, atol=1e-12)
