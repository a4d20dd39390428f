"""GPU front end and output gate vs the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_kda_gb300 import synthetic
from tests._parity import TOL_BF16, TOL_FP32, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import build
    build.build()
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


def small_layer(lens, H=4, seed=31):
    inp = synthetic.layer_inputs(lens, H, seed=seed, device="cuda")
    # give b a nonzero value so the bias path is exercised
    inp.b.copy_(torch.randn(inp.b.shape, generator=torch.Generator("cuda").manual_seed(5),
                            device="cuda") * 0.3)
    return inp


# the second list puts several sequence starts (and an empty sequence) inside one warp's
# group of consecutive tokens
@pytest.mark.parametrize("lens", [[37, 1, 0, 90, 3], [1, 2, 1, 1, 0, 3, 1, 7, 1, 2, 5, 1]])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_frontend_matches_oracle(kda, out_dtype, lens):
    inp = small_layer(lens)
    outs = kda.kda_frontend(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                            inp.beta_logit, inp.cu_seqlens, 1e-6, out_dtype=out_dtype)
    torch.cuda.synchronize()
    refs = oracle.kda_frontend(to64(inp.qp), to64(inp.kp), to64(inp.vp), to64(inp.conv_w),
                               to64(inp.z), to64(inp.A), to64(inp.b), to64(inp.beta_logit),
                               inp.cu_seqlens.cpu().numpy(), 1e-6)
    bf = out_dtype == torch.bfloat16
    for name, g, r in zip(["q_hat", "k_hat", "v"], outs[:3], refs[:3]):
        assert_close(to64(g), r, TOL_FP32, name, out_is_bf16=bf)
    assert_close(to64(outs[3]), refs[3], TOL_FP32, "log_alpha")
    assert_close(to64(outs[4]), refs[4], TOL_FP32, "beta")
    # unit norm per head for q^, k^ (fp32 output)
    if not bf:
        n = outs[0].norm(dim=-1)
        assert torch.allclose(n, torch.ones_like(n), atol=1e-5)


def test_frontend_without_bias(kda):
    inp = small_layer([20, 11], H=2, seed=32)
    a = kda.kda_frontend(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, None,
                         inp.beta_logit, inp.cu_seqlens, out_dtype=torch.float32)
    zeros = torch.zeros_like(inp.b)
    b = kda.kda_frontend(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, zeros,
                         inp.beta_logit, inp.cu_seqlens, out_dtype=torch.float32)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("in_dtype,out_dtype", [(torch.float32, torch.float32),
                                                (torch.float32, torch.bfloat16),
                                                (torch.bfloat16, torch.bfloat16)])
def test_output_gate_matches_oracle(kda, in_dtype, out_dtype):
    g_ = torch.Generator("cuda").manual_seed(33)
    ot = (torch.randn((300, 5, 128), generator=g_, device="cuda") * 0.02).to(in_dtype)
    g = torch.randn((300, 5, 128), generator=g_, device="cuda").to(torch.bfloat16)
    out = kda.kda_output_gate(ot, g, 1e-6, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = oracle.kda_output_gate(to64(ot), to64(g), 1e-6)
    assert_close(to64(out), ref, TOL_FP32, "o_gated", out_is_bf16=out_dtype == torch.bfloat16)


def test_layer_core_unfused_small(kda):
    """Front end -> prefill -> gate through the library, against the oracle's
    composition.  The intermediate q^, k^, v are kept in fp32 here so that the
    only rounding is the kernels' own."""
    inp = small_layer([130, 64, 7], H=3, seed=34)
    qh, kh, vv, la, beta = kda.kda_frontend(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A,
                                            inp.b, inp.beta_logit, inp.cu_seqlens,
                                            out_dtype=torch.float32)
    ot, Sf = kda.kda_prefill(qh, kh, vv, la, beta, inp.cu_seqlens, None,
                             out_dtype=torch.float32)
    og = kda.kda_output_gate(ot, inp.g, 1e-6, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref_o, ref_S = oracle.kda_layer_core(to64(inp.qp), to64(inp.kp), to64(inp.vp),
                                         to64(inp.conv_w), to64(inp.z), to64(inp.A),
                                         to64(inp.b), to64(inp.beta_logit), to64(inp.g),
                                         inp.cu_seqlens.cpu().numpy())
    assert_close(to64(og), ref_o, TOL_BF16, "o_gated")
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")
