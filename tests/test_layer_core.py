"""GPU layer core (front end -> recurrence -> output gate) vs the fp64 oracle.

The library hands q^, k^, v from the front end to the recurrence in bf16 (the
kernel interface the pages describe takes bf16 q/k/v).  The oracle composition
below rounds at the same point (torch's bf16 rounding of the oracle's own fp64
front-end outputs); every other step is fp64.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_kda_gb300 import synthetic
from tests._parity import TOL_BF16, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


def bf16_round(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def oracle_layer_core(inp, heads=None):
    sel = (lambda t: t) if heads is None else (lambda t: t[:, heads])
    H_all = inp.qp.shape[1]
    hs = list(range(H_all)) if heads is None else heads
    conv_w = to64(inp.conv_w).reshape(3, H_all, 128, 4)[:, hs].reshape(3, len(hs) * 128, 4)
    cu = inp.cu_seqlens.cpu().numpy()
    qh, kh, vv, la, beta = oracle.kda_frontend(to64(sel(inp.qp)), to64(sel(inp.kp)),
                                               to64(sel(inp.vp)), conv_w, to64(sel(inp.z)),
                                               to64(inp.A)[hs], to64(inp.b)[hs],
                                               to64(sel(inp.beta_logit)), cu)
    S0 = None if inp.S0 is None else to64(inp.S0)[:, hs]
    ot, Sf = oracle.kda_prefill(bf16_round(qh), bf16_round(kh), bf16_round(vv), la, beta, cu,
                                S0=S0)
    return oracle.kda_output_gate(ot, to64(sel(inp.g))), Sf


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_layer_core_small_varlen(kda, out_dtype):
    inp = synthetic.layer_inputs([70, 1, 0, 33, 129], 4, seed=41, s0_std=0.1, device="cuda")
    og, Sf = kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0,
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref_o, ref_S = oracle_layer_core(inp)
    assert_close(to64(og), ref_o, TOL_BF16, "o_gated", out_is_bf16=out_dtype == torch.bfloat16)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")


def test_layer_core_matches_its_three_calls(kda):
    """The composed entry point equals kda_frontend -> kda_prefill -> kda_output_gate, bit for bit."""
    inp = synthetic.layer_inputs([90, 41], 3, seed=42, device="cuda")
    og, Sf = kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                inp.beta_logit, inp.g, inp.cu_seqlens, None,
                                out_dtype=torch.float32)
    qh, kh, vv, la, beta = kda.kda_frontend(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A,
                                            inp.b, inp.beta_logit, inp.cu_seqlens)
    ot, Sf2 = kda.kda_prefill(qh, kh, vv, la, beta, inp.cu_seqlens, None,
                              out_dtype=torch.float32)
    og2 = kda.kda_output_gate(ot, inp.g, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(og, og2) and torch.equal(Sf, Sf2)


def test_layer_core_full_varlen_sampled_heads(kda):
    """16 sequences, log-uniform lengths in [1K, 64K] (~248K tokens), 96 heads;
    oracle on heads 0, 47, 95 over every sequence."""
    inp = synthetic.workload(5, device="cuda")
    og, Sf = kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                inp.beta_logit, inp.g, inp.cu_seqlens, None,
                                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    heads = [0, 47, 95]
    ref_o, ref_S = oracle_layer_core(inp, heads)
    assert_close(to64(og[:, heads]), ref_o, TOL_BF16, "o_gated", out_is_bf16=True)
    assert_close(to64(Sf[:, heads]), ref_S, TOL_BF16, "S_final")


def test_layer_core_rejects_small_workspace(kda):
    inp = synthetic.layer_inputs([20], 2, seed=43, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError):
        kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                           inp.beta_logit, inp.g, inp.cu_seqlens, None, workspace=ws)
