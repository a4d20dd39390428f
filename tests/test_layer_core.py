"""GPU layer core (front end -> recurrence -> output gate) vs the fp64 oracle.

The library keeps every intermediate of the layer in fp32, and the oracle is
the plain fp64 composition.  (Rounding q^, k^, v to bf16 between the stages
moves the output of these inputs by ~10%: the conv-smoothed keys are close to
parallel and the recurrence is ill-conditioned.)

Tolerance: the plain contract bound, max-abs over rms <= 2e-3, on the gated
output o^g and on S_final (plus the bf16 half-ulp per element for a bf16
output).  The pre-gate o~ of the fused kernel is checked on its own through
the same entry point: with g = 0 and rms_eps = 1e6 the gate is
0.5 o~ / sqrt(mean(o~^2) + 1e6), linear in o~ to about 1e-6 for |o~| of order
one, so the plain error of that output is the plain error of o~.
"""
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
    ot, Sf = oracle.kda_prefill(qh, kh, vv, la, beta, cu, S0=S0)
    return oracle.kda_output_gate(ot, to64(sel(inp.g))), Sf, ot


def assert_fused_o_tilde_close(kda, inp, ref_ot, heads=None):
    """The fused kernel's pre-gate o~ against the oracle's, through the same entry point:
    g = 0 and rms_eps = 1e6 make the gate 0.5 o~ / sqrt(mean(o~^2) + 1e6), linear in o~ to
    about 1e-6, and the oracle applies the same gate to its own o~."""
    og0, _ = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                      inp.beta_logit, torch.zeros_like(inp.g), inp.cu_seqlens,
                                      inp.S0, rms_eps=1e6, out_dtype=torch.float32)
    torch.cuda.synchronize()
    gpu = to64(og0 if heads is None else og0[:, heads])
    ref = oracle.kda_output_gate(ref_ot, np.zeros_like(ref_ot), eps=1e6)
    return assert_close(gpu, ref, TOL_BF16, "o~ (fused, before the gate)")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_layer_core_small_varlen(kda, out_dtype):
    inp = synthetic.layer_inputs([70, 1, 0, 33, 129], 4, seed=41, s0_std=0.1, device="cuda")
    og, Sf = kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0,
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref_o, ref_S, _ = oracle_layer_core(inp)
    assert_gated_close(to64(og), ref_o, out_dtype == torch.bfloat16)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")


def test_layer_core_matches_its_three_calls(kda):
    """The composed entry point equals kda_frontend -> kda_prefill -> kda_output_gate, bit for bit."""
    inp = synthetic.layer_inputs([90, 41], 3, seed=42, device="cuda")
    og, Sf = kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                inp.beta_logit, inp.g, inp.cu_seqlens, None,
                                out_dtype=torch.float32)
    qh, kh, vv, la, beta = kda.kda_frontend(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A,
                                            inp.b, inp.beta_logit, inp.cu_seqlens,
                                            out_dtype=torch.float32)
    ot, Sf2 = kda.kda_prefill(qh, kh, vv, la, beta, inp.cu_seqlens, None,
                              out_dtype=torch.float32)
    og2 = kda.kda_output_gate(ot, inp.g, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(og, og2) and torch.equal(Sf, Sf2)
    _, _, ref_ot = oracle_layer_core(inp)
    assert_close(to64(ot), ref_ot, TOL_FP32 * 10, "o~ (before the gate)")


def test_layer_core_full_varlen_sampled_heads(kda):
    """16 sequences, log-uniform lengths in [1K, 64K] (~248K tokens), 96 heads;
    oracle on heads 0, 47, 95 over every sequence."""
    inp = synthetic.workload(5, device="cuda")
    og, Sf = kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                inp.beta_logit, inp.g, inp.cu_seqlens, None,
                                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    heads = [0, 47, 95]
    ref_o, ref_S, _ = oracle_layer_core(inp, heads)
    assert_gated_close(to64(og[:, heads]), ref_o, True)
    assert_close(to64(Sf[:, heads]), ref_S, TOL_BF16, "S_final")


def test_layer_core_rejects_small_workspace(kda):
    inp = synthetic.layer_inputs([20], 2, seed=43, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError):
        kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                           inp.beta_logit, inp.g, inp.cu_seqlens, None, workspace=ws)


# ---------------------------------------------------------------------------
# kda_layer_core_fused: the same layer core in one tensor-core kernel.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fused_small_varlen(kda, out_dtype):
    """Ragged lengths (1, 0, 33, 70, 129 tokens: partial chunks, an empty sequence,
    conv history across chunk boundaries) with a carried state."""
    inp = synthetic.layer_inputs([70, 1, 0, 33, 129], 4, seed=41, s0_std=0.1, device="cuda")
    og, Sf = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                      inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0,
                                      out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S, ref_ot = oracle_layer_core(inp)
    assert_gated_close(to64(og), ref_o, out_dtype == torch.bfloat16)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")
    assert_fused_o_tilde_close(kda, inp, ref_ot)


def test_fused_long_sequence_nonzero_bias(kda):
    """One 3000-token sequence (94 chunks) plus a short one, with a nonzero decay bias b."""
    inp = synthetic.layer_inputs([3000, 45], 2, seed=44, s0_std=0.1, device="cuda")
    b = torch.randn(inp.b.shape, generator=torch.Generator().manual_seed(7)).to(inp.b.device) * 0.5
    og, Sf = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, b,
                                      inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0,
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    inp.b = b
    ref_o, ref_S, _ = oracle_layer_core(inp)
    assert_gated_close(to64(og), ref_o, False)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")


def test_fused_full_varlen_sampled_heads(kda):
    """Workload 5 (16 sequences, lengths log-uniform in [1K, 64K], 96 heads); oracle on
    heads 0, 47, 95 over every sequence."""
    inp = synthetic.workload(5, device="cuda")
    og, Sf = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                      inp.beta_logit, inp.g, inp.cu_seqlens, None,
                                      out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    heads = [0, 47, 95]
    ref_o, ref_S, ref_ot = oracle_layer_core(inp, heads)
    assert_gated_close(to64(og[:, heads]), ref_o, True)
    assert_close(to64(Sf[:, heads]), ref_S, TOL_BF16, "S_final")
    del og, Sf
    assert_fused_o_tilde_close(kda, inp, ref_ot, heads)


@pytest.mark.parametrize("entry", ["kda_layer_core_fused", "kda_layer_core_fused_unbounded_decay"])
def test_fused_varlen_bit_exact_packing(kda, entry):
    """The fused layer core gives a sequence the same bits alone, packed, or packed in another
    order (so its convolution never reads across a sequence boundary of the packed layout), and
    leaves the output rows around the batch untouched; for both gates."""
    fn = getattr(kda, entry)
    lens = [77, 200, 3, 64, 0, 129, 33]
    H = 3
    inp = synthetic.layer_inputs(lens, H, seed=46, s0_std=0.1, device="cuda")
    T = int(inp.cu_seqlens[-1])
    canary = 8
    o_buf = torch.full((T + 2 * canary, H, 128), 1234.5, dtype=torch.bfloat16, device="cuda")
    o = o_buf[canary:canary + T]
    _, Sf = fn(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b, inp.beta_logit, inp.g,
               inp.cu_seqlens, inp.S0, o=o)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    assert (o_buf[:canary] == 1234.5).all() and (o_buf[canary + T:] == 1234.5).all()
    cu = inp.cu_seqlens.tolist()
    for n, L in enumerate(lens):  # each sequence alone
        a, b = cu[n], cu[n + 1]
        solo_cu = torch.tensor([0, L], dtype=torch.int32, device="cuda")
        o_n, S_n = fn(inp.qp[a:b], inp.kp[a:b], inp.vp[a:b], inp.conv_w, inp.z[a:b], inp.A, inp.b,
                      inp.beta_logit[a:b], inp.g[a:b], solo_cu, inp.S0[n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(o_n, o[a:b]), f"sequence {n} output differs when run alone"
        assert torch.equal(S_n[0], Sf[n]), f"sequence {n} state differs when run alone"
    perm = [5, 2, 0, 6, 4, 3, 1]  # the same sequences packed in another order
    idx = torch.cat([torch.arange(cu[n], cu[n + 1]) for n in perm]).cuda()
    cu_p = synthetic.cu_from_lengths([lens[n] for n in perm], "cuda")
    pick = lambda t: t[idx].contiguous()
    o_p, S_p = fn(pick(inp.qp), pick(inp.kp), pick(inp.vp), inp.conv_w, pick(inp.z), inp.A, inp.b,
                  pick(inp.beta_logit), pick(inp.g), cu_p, inp.S0[perm].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(o_p, o[idx]) and torch.equal(S_p, Sf[perm])


def test_fused_deterministic(kda):
    inp = synthetic.layer_inputs([300, 77], 3, seed=45, device="cuda")
    a, Sa = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                     inp.beta_logit, inp.g, inp.cu_seqlens, None)
    b, Sb = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                     inp.beta_logit, inp.g, inp.cu_seqlens, None)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(Sa, Sb)


def test_fused_sequences_shorter_than_the_convolution(kda):
    """Sequences of 1 to 5 tokens (shorter than or equal to the width-4 convolution, so
    the zero history before each start matters on every row) beside 8, 9 and 40, with a
    carried state."""
    inp = synthetic.layer_inputs([2, 3, 1, 4, 5, 8, 9, 40], 3, seed=46, s0_std=0.1, device="cuda")
    og, Sf = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                      inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0,
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S, _ = oracle_layer_core(inp)
    assert_gated_close(to64(og), ref_o, False)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")


def test_fused_many_heads_several_waves(kda):
    """H=160 heads x 2 sequences = 320 CTAs (several waves of the grid), lengths 70 and 41
    (history boxes across chunk boundaries); oracle on four heads, the last included."""
    inp = synthetic.layer_inputs([70, 41], 160, seed=47, s0_std=0.1, device="cuda")
    og, Sf = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                      inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0,
                                      out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    heads = [0, 63, 152, 159]
    ref_o, ref_S, _ = oracle_layer_core(inp, heads)
    assert_gated_close(to64(og[:, heads]), ref_o, True)
    assert_close(to64(Sf[:, heads]), ref_S, TOL_BF16, "S_final")


def test_fused_many_short_sequences(kda):
    """200 sequences of 0 to 50 tokens through the fused layer core (index-order CTAs, many
    sequences shorter than the convolution or a chunk)."""
    lens = np.random.default_rng(44).integers(0, 51, size=200).tolist()
    inp = synthetic.layer_inputs(lens, 2, seed=45, s0_std=0.1, device="cuda")
    og, Sf = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                      inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0,
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S, _ = oracle_layer_core(inp)
    assert_gated_close(to64(og), ref_o, False)
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final")
