"""GPU decode step vs the fp64 oracle (through the C ABI)."""
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


@pytest.mark.parametrize("dtype,out_dtype,tol", [
    (torch.float32, torch.float32, TOL_FP32),
    (torch.bfloat16, torch.float32, TOL_BF16),
    (torch.bfloat16, torch.bfloat16, TOL_BF16),
])
def test_decode_small(kda, dtype, out_dtype, tol):
    inp = synthetic.decode_inputs(5, 3, dtype, seed=11, device="cuda")
    S_ref_in = to64(inp.S)
    S = inp.S.clone()
    o = kda.kda_decode_step(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, S,
                            out_dtype=out_dtype)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.kda_decode_step(to64(inp.q), to64(inp.k), to64(inp.v),
                                          to64(inp.log_alpha), to64(inp.beta), S_ref_in)
    assert_close(to64(o), o_ref, tol, "o", out_is_bf16=out_dtype == torch.bfloat16)
    assert_close(to64(S), S_ref, TOL_FP32, "S")


def test_decode_alpha_zero_resets(kda):
    inp = synthetic.decode_inputs(2, 2, torch.float32, seed=12, device="cuda")
    la = torch.full_like(inp.log_alpha, float("-inf"))
    S = inp.S.clone()
    o = kda.kda_decode_step(inp.q, inp.k, inp.v, la, inp.beta, S, out_dtype=torch.float32)
    want = inp.beta[..., None, None] * inp.k[..., :, None] * inp.v[..., None, :]
    torch.testing.assert_close(S, want, rtol=0, atol=1e-6)
    assert torch.isfinite(o).all()


def test_decode_repeated_equals_prefill(kda):
    """T decode steps == one prefill over the same T tokens (P12)."""
    T, H = 9, 2
    p = synthetic.prefill_inputs([T], H, torch.float32, seed=13, s0_std=0.1, device="cuda")
    o_pre, S_pre = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0,
                                   out_dtype=torch.float32)
    S = p.S0[0:1].clone()
    outs = []
    for t in range(T):
        outs.append(kda.kda_decode_step(p.q[t:t + 1], p.k[t:t + 1], p.v[t:t + 1],
                                        p.log_alpha[t:t + 1].contiguous(),
                                        p.beta[t:t + 1].contiguous(), S,
                                        out_dtype=torch.float32))
    torch.testing.assert_close(torch.cat(outs), o_pre, rtol=0, atol=2e-6)
    torch.testing.assert_close(S, S_pre, rtol=0, atol=2e-6)


def test_decode_full_size_sampled(kda):
    """256 requests x 96 heads (1.6 GB of state), the benchmark's launch;
    oracle on a sample of (request, head) units."""
    inp = synthetic.workload(3, device="cuda")
    B, H = inp.q.shape[:2]
    rng = np.random.default_rng(3)
    units = [(int(b), int(h)) for b, h in zip(rng.integers(0, B, 48), rng.integers(0, H, 48))]
    units += [(0, 0), (B - 1, H - 1)]
    before = {u: to64(inp.S[u[0], u[1]]) for u in units}
    o = kda.kda_decode_step(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S,
                            out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    bi = [u[0] for u in units]
    hi = [u[1] for u in units]
    sel = lambda t: to64(t[bi, hi])[:, None]
    o_ref, S_ref = oracle.kda_decode_step(sel(inp.q), sel(inp.k), sel(inp.v),
                                          sel(inp.log_alpha), to64(inp.beta[bi, hi])[:, None],
                                          np.stack([before[u] for u in units])[:, None])
    assert_close(to64(o[bi, hi]), o_ref[:, 0], TOL_BF16, "o", out_is_bf16=True)
    assert_close(to64(inp.S[bi, hi]), S_ref[:, 0], TOL_BF16, "S")
