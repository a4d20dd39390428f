"""GPU Kimi Linear case (decays without the -5 floor) vs the fp64 oracle: the front end with
the unbounded gate -e^A softplus(z + b), the token-by-token prefill for any log alpha <= 0
(-inf included), and the staged layer core that composes them."""
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
