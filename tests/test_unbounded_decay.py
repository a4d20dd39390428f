"""GPU Kimi Linear case (decays without the -5 floor) vs the fp64 oracle: the front end with
the unbounded gate -e^A softplus(z + b); the prefill for any log alpha <= 0 (-inf included),
bf16 inputs on the tensor-core kernel (chunks out of its range run token by token inside it)
and fp32 inputs on the token-by-token kernel; the staged layer core; and the fused layer core
with the unbounded gate."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_kda_gb300 import synthetic
from tests._parity import TOL_BF16, TOL_FP32, assert_close, assert_gated_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import build
    build.build()
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


def strong_decay_layer(lens, H, seed):
    """Layer inputs with A ~ N(1.5, 0.5) and a nonzero b: e^A softplus(z + b) reaches far
    below K3's floor of -5."""
    inp = synthetic.layer_inputs(lens, H, seed=seed, s0_std=0.1, device="cuda")
    gen = torch.Generator("cuda").manual_seed(seed)
    inp.A.copy_(torch.randn(inp.A.shape, generator=gen, device="cuda") * 0.5 + 1.5)
    inp.b.copy_(torch.randn(inp.b.shape, generator=gen, device="cuda") * 0.3)
    return inp


def test_frontend_gate(kda):
    inp = strong_decay_layer([37, 1, 0, 90], 3, seed=101)
    outs = kda.kda_frontend_unbounded_decay(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A,
                                            inp.b, inp.beta_logit, inp.cu_seqlens,
                                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    refs = oracle.kda_frontend_unbounded_decay(to64(inp.qp), to64(inp.kp), to64(inp.vp),
                                               to64(inp.conv_w), to64(inp.z), to64(inp.A),
                                               to64(inp.b), to64(inp.beta_logit),
                                               inp.cu_seqlens.cpu().numpy())
    for name, g, r in zip(["q_hat", "k_hat", "v", "log_alpha", "beta"], outs, refs):
        assert_close(to64(g), r, TOL_FP32, name)
    la = to64(outs[3])
    assert (la < 0).all() and la.min() < -10.0, "the test should reach well below the floor"
    # the other outputs are the bounded front end's
    bounded = kda.kda_frontend(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                               inp.beta_logit, inp.cu_seqlens, out_dtype=torch.float32)
    for i in (0, 1, 2, 4):
        assert torch.equal(outs[i], bounded[i])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_prefill_any_decay(kda, dtype):
    """log alpha uniform in [-40, 0] with every 7th token -inf (a reset), ragged sequences."""
    inp = synthetic.prefill_inputs([150, 0, 33, 64], 2, dtype, seed=102, s0_std=0.1, device="cuda")
    gen = torch.Generator("cuda").manual_seed(102)
    la = -40.0 * torch.rand(inp.log_alpha.shape, generator=gen, device="cuda")
    la[::7] = -float("inf")
    o, Sf = kda.kda_prefill_unbounded_decay(inp.q, inp.k, inp.v, la.contiguous(), inp.beta,
                                            inp.cu_seqlens, inp.S0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S = oracle.kda_prefill(to64(inp.q), to64(inp.k), to64(inp.v), to64(la),
                                      to64(inp.beta), inp.cu_seqlens.cpu().numpy(), S0=to64(inp.S0))
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
    assert_close(to64(o), ref_o, tol, "o")
    assert_close(to64(Sf), ref_S, tol, "S_final")


def test_layer_core(kda):
    inp = strong_decay_layer([70, 1, 0, 129], 3, seed=103)
    og, Sf = kda.kda_layer_core_unbounded_decay(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A,
                                                inp.b, inp.beta_logit, inp.g, inp.cu_seqlens,
                                                inp.S0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    x = [to64(t) for t in (inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                           inp.beta_logit)]
    cu = inp.cu_seqlens.cpu().numpy()
    ref_o, ref_S = oracle.kda_layer_core_unbounded_decay(*x, to64(inp.g), cu, S0=to64(inp.S0))
    assert_gated_close(to64(og), ref_o, False)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")


def test_prefill_mixed_chunks(kda):
    """bf16 prefill where most 32-token chunks stay in the tensor-core range and some do not
    (a token of -40 or -inf inside them): both forms, and the hand-over of the state between
    them, against the oracle."""
    inp = synthetic.prefill_inputs([300, 77, 1, 0, 129], 3, torch.bfloat16, seed=104,
                                   s0_std=0.1, device="cuda")
    la = inp.log_alpha.clone()
    la[40, 0, 5] = -40.0          # sequence 0, chunk 1, one channel of head 0
    la[100, :, :] = -float("inf")  # sequence 0, chunk 3: a reset of every channel and head
    la[200, 2, 7] = -25.0         # sequence 0, chunk 6, head 2
    la[310, 1, 100] = -60.0       # sequence 1, chunk 0
    la[400, 0, 3] = -float("inf")  # sequence 4, chunk 0, one channel
    o, Sf = kda.kda_prefill_unbounded_decay(inp.q, inp.k, inp.v, la, inp.beta, inp.cu_seqlens,
                                            inp.S0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S = oracle.kda_prefill(to64(inp.q), to64(inp.k), to64(inp.v), to64(la),
                                      to64(inp.beta), inp.cu_seqlens.cpu().numpy(), S0=to64(inp.S0))
    assert_close(to64(o), ref_o, TOL_BF16, "o")
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")
    # in-range chunks take the tensor-core form: same output as kda_prefill where no chunk of
    # the sequence leaves the range (sequence 2 and 3 are one token or empty; check sequence 4's
    # heads 1 and 2, whose decays stay above the floor)
    o_b, _ = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens,
                             inp.S0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o[377:, 1:], o_b[377:, 1:])


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fused_layer_core(kda, out_dtype):
    """The whole layer core in the tensor-core kernel with the unbounded gate (chunks both in
    and out of range), ragged sequences, a carried state."""
    inp = strong_decay_layer([300, 70, 1, 0, 129], 3, seed=105)
    og, Sf = kda.kda_layer_core_fused_unbounded_decay(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z,
                                                      inp.A, inp.b, inp.beta_logit, inp.g,
                                                      inp.cu_seqlens, inp.S0, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    x = [to64(t) for t in (inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                           inp.beta_logit)]
    cu = inp.cu_seqlens.cpu().numpy()
    ref_o, ref_S = oracle.kda_layer_core_unbounded_decay(*x, to64(inp.g), cu, S0=to64(inp.S0))
    assert_gated_close(to64(og), ref_o, out_dtype == torch.bfloat16)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")


def test_fused_layer_core_in_range(kda):
    """The unbounded gate on inputs whose decays keep every chunk in range (A ~ N(0, 0.5)):
    every chunk takes the tensor-core form, against the unbounded oracle."""
    inp = synthetic.layer_inputs([150, 33], 2, seed=106, s0_std=0.1, device="cuda")
    og, Sf = kda.kda_layer_core_fused_unbounded_decay(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z,
                                                      inp.A, inp.b, inp.beta_logit, inp.g,
                                                      inp.cu_seqlens, inp.S0,
                                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    x = [to64(t) for t in (inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                           inp.beta_logit)]
    ref_o, ref_S = oracle.kda_layer_core_unbounded_decay(*x, to64(inp.g),
                                                         inp.cu_seqlens.cpu().numpy(),
                                                         S0=to64(inp.S0))
    assert_gated_close(to64(og), ref_o, False)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")


def test_fused_layer_core_full_varlen_sampled_heads(kda):
    """Workload 5's layer inputs with Kimi Linear's gate (16 sequences, ~317K tokens, 96
    heads); oracle on heads 0, 47, 95 over every sequence."""
    inp = synthetic.workload(5, device="cuda")
    og, Sf = kda.kda_layer_core_fused_unbounded_decay(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z,
                                                      inp.A, inp.b, inp.beta_logit, inp.g,
                                                      inp.cu_seqlens, None,
                                                      out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    heads = [0, 47, 95]
    H_all = inp.qp.shape[1]
    sel = lambda t: to64(t[:, heads])
    conv_w = to64(inp.conv_w).reshape(3, H_all, 128, 4)[:, heads].reshape(3, len(heads) * 128, 4)
    ref_o, ref_S = oracle.kda_layer_core_unbounded_decay(
        sel(inp.qp), sel(inp.kp), sel(inp.vp), conv_w, sel(inp.z), to64(inp.A)[heads],
        to64(inp.b)[heads], sel(inp.beta_logit), sel(inp.g), inp.cu_seqlens.cpu().numpy())
    assert_gated_close(to64(og[:, heads]), ref_o, True)
    assert_close(to64(Sf[:, heads]), ref_S, TOL_BF16, "S_final")
