"""GPU prefill and decode with one decay per (token, head) (the Gated DeltaNet case) vs the
fp64 oracle, through the C ABI: the tensor-core kernel (bf16 inputs), the recurrent kernel
(fp32 inputs), snapshots, and the decode step."""
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


@pytest.mark.parametrize("dtype,out_dtype", [(torch.bfloat16, torch.float32),
                                             (torch.bfloat16, torch.bfloat16),
                                             (torch.float32, torch.float32)])
def test_prefill_varlen(kda, dtype, out_dtype):
    inp = synthetic.prefill_inputs([229, 64, 1, 0, 130], 3, dtype, seed=81, s0_std=0.1,
                                   device="cuda", head_decay=True)
    assert inp.log_alpha.shape == (424, 3)
    o, Sf, _, _ = kda.kda_prefill_head_decay(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                             inp.cu_seqlens, inp.S0, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S = oracle.kda_prefill_head_decay(to64(inp.q), to64(inp.k), to64(inp.v),
                                                 to64(inp.log_alpha), to64(inp.beta),
                                                 inp.cu_seqlens.cpu().numpy(), S0=to64(inp.S0))
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
    assert_close(to64(o), ref_o, tol, "o", out_is_bf16=out_dtype == torch.bfloat16)
    assert_close(to64(Sf), ref_S, tol, "S_final")


def test_prefill_equals_per_channel_call_with_repeated_decay(kda):
    """The per-head path and the per-channel path fed the same decay repeated over the
    channels compute the same products: outputs agree to rounding."""
    inp = synthetic.prefill_inputs([300, 77], 2, torch.bfloat16, seed=82, s0_std=0.1,
                                   device="cuda", head_decay=True)
    o1, S1, _, _ = kda.kda_prefill_head_decay(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                              inp.cu_seqlens, inp.S0, out_dtype=torch.float32)
    la_full = inp.log_alpha[:, :, None].expand(-1, -1, 128).contiguous()
    o2, S2 = kda.kda_prefill(inp.q, inp.k, inp.v, la_full, inp.beta, inp.cu_seqlens, inp.S0,
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


def test_prefill_snapshots(kda):
    inp = synthetic.prefill_inputs([160, 96], 2, torch.bfloat16, seed=83, device="cuda",
                                   head_decay=True)
    _, Sf, base, ck = kda.kda_prefill_head_decay(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                                 inp.cu_seqlens, every=64)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    assert base.tolist() == [0, 2, 3]
    x = [to64(t) for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    for slot, (t0, m) in enumerate([(0, 64), (0, 128), (160, 64)]):
        sub = [t[t0:t0 + m] for t in x]
        _, S = oracle.kda_prefill_head_decay(*sub, [0, m])
        assert_close(to64(ck[slot]), S[0], TOL_BF16, f"snapshot {slot}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_step(kda, dtype):
    inp = synthetic.decode_inputs(24, 3, dtype, seed=84, device="cuda", head_decay=True)
    S = inp.S.clone()
    o = kda.kda_decode_step_head_decay(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, S,
                                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    la = to64(inp.log_alpha)[:, :, None].repeat(128, axis=2)
    ref_o, ref_S = oracle.kda_decode_step(to64(inp.q), to64(inp.k), to64(inp.v), la,
                                          to64(inp.beta), to64(inp.S))
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
    assert_close(to64(o), ref_o, tol, "o")
    assert_close(to64(S), ref_S, tol, "S")
