"""GPU decode step of the layer core over pooled states vs the fp64 oracle.

The gated output and the state rows are checked with the plain 2e-3 max-abs/rms bound;
the convolution state is bit-exact (it only moves bf16 inputs); rows of the pools
that no request names are untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_kda_gb300 import synthetic
from tests._parity import TOL_BF16, assert_close, assert_gated_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import build
    build.build()
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


def oracle_step(inp, heads=None):
    sel = (lambda t: t) if heads is None else (lambda t: t[:, heads])
    H_all = inp.qp.shape[1]
    hs = list(range(H_all)) if heads is None else heads
    conv_w = to64(inp.conv_w).reshape(3, H_all, 128, 4)[:, hs].reshape(3, len(hs) * 128, 4)
    S_pool = to64(inp.S_pool)[:, hs]
    conv_pool = to64(inp.conv_pool)[:, :, :, hs]
    slot = inp.slot.cpu().numpy()
    o, S_new, conv_new = oracle.kda_decode_layer(
        to64(sel(inp.qp)), to64(sel(inp.kp)), to64(sel(inp.vp)), conv_w, to64(sel(inp.z)),
        to64(inp.A)[hs], to64(inp.b)[hs], to64(sel(inp.beta_logit)), to64(sel(inp.g)), slot,
        S_pool, conv_pool)
    return o, S_new, conv_new



def run(kda, inp, out_dtype=torch.float32):
    S_pool, conv_pool = inp.S_pool.clone(), inp.conv_pool.clone()
    o = kda.kda_decode_layer(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                             inp.beta_logit, inp.g, inp.slot, S_pool, conv_pool,
                             out_dtype=out_dtype)
    torch.cuda.synchronize()
    return o, S_pool, conv_pool


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_layer_small_pool(kda, out_dtype):
    """B=12 requests in shuffled rows of a 20-row pool, H=3."""
    inp = synthetic.decode_layer_inputs(12, 3, 20, seed=51, device="cuda")
    o, S_pool, conv_pool = run(kda, inp, out_dtype)
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S, ref_conv = oracle_step(inp)
    assert_gated_close(to64(o), ref_o, out_dtype == torch.bfloat16)
    slot = inp.slot.cpu().numpy()
    assert_close(to64(S_pool)[slot], ref_S[slot], TOL_BF16, "S_pool rows")
    assert torch.equal(conv_pool.float().cpu(), torch.from_numpy(ref_conv).float()), "conv_pool"
    free = sorted(set(range(20)) - set(slot.tolist()))
    assert torch.equal(S_pool[free], inp.S_pool[free]), "rows no request names changed"


def test_decode_layer_full_batch_sampled_heads(kda):
    """B=256 requests, H=96, a 320-row pool (the decode workload's size with the layer's
    front end and gate); oracle on heads 0, 47, 95 for every request."""
    inp = synthetic.decode_layer_inputs(256, 96, 320, device="cuda")
    o, S_pool, conv_pool = run(kda, inp, torch.bfloat16)
    assert kda.kda_get_device_status()[0] == 0
    heads = [0, 47, 95]
    ref_o, ref_S, ref_conv = oracle_step(inp, heads)
    assert_gated_close(to64(o[:, heads]), ref_o, True)
    slot = inp.slot.cpu().numpy()
    assert_close(to64(S_pool[:, heads])[slot], ref_S[slot], TOL_BF16, "S_pool rows")
    assert torch.equal(conv_pool[:, :, :, heads].float().cpu(), torch.from_numpy(ref_conv).float())


def test_decode_layer_continues_the_fused_prefill(kda):
    """The fused layer core over the first T0 tokens of two sequences, then T - T0
    decode-layer steps on pool rows 3 and 0 (state = S_final, convolution state = the
    last three pre-convolution inputs), against the oracle layer core over all T
    tokens of each sequence."""
    lens, T0, steps, H = [37, 70], [33, 64], 4, 2
    inp = synthetic.layer_inputs(lens, H, seed=52, s0_std=0.1, device="cuda")
    cu = inp.cu_seqlens.tolist()
    # prefill of the first T0 tokens of each sequence
    idx = torch.cat([torch.arange(cu[n], cu[n] + T0[n]) for n in range(2)]).cuda()
    cu0 = synthetic.cu_from_lengths(T0, "cuda")
    sub = lambda t: t[idx].contiguous()
    _, Sf = kda.kda_layer_core_fused(sub(inp.qp), sub(inp.kp), sub(inp.vp), inp.conv_w, sub(inp.z),
                                     inp.A, inp.b, sub(inp.beta_logit), sub(inp.g), cu0, inp.S0,
                                     out_dtype=torch.float32)
    rows = [3, 0]
    S_pool = torch.zeros((5, H, 128, 128), device="cuda")
    conv_pool = torch.zeros((5, 3, 3, H, 128), dtype=torch.bfloat16, device="cuda")
    for n in range(2):
        S_pool[rows[n]] = Sf[n]
        for s, xp in enumerate((inp.qp, inp.kp, inp.vp)):
            for tap in range(3):
                conv_pool[rows[n], s, tap] = xp[cu[n] + T0[n] - 1 - tap]
    slot = torch.tensor(rows, dtype=torch.int32, device="cuda")
    outs = []
    for i in range(steps):
        t = [cu[n] + T0[n] + i for n in range(2)]
        pick = lambda x: x[t].contiguous()
        outs.append(kda.kda_decode_layer(pick(inp.qp), pick(inp.kp), pick(inp.vp), inp.conv_w,
                                         pick(inp.z), inp.A, inp.b, pick(inp.beta_logit),
                                         pick(inp.g), slot, S_pool, conv_pool,
                                         out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S = oracle.kda_layer_core(to64(inp.qp), to64(inp.kp), to64(inp.vp), to64(inp.conv_w),
                                         to64(inp.z), to64(inp.A), to64(inp.b), to64(inp.beta_logit),
                                         to64(inp.g), inp.cu_seqlens.cpu().numpy(), S0=to64(inp.S0))
    gpu = np.stack([to64(x) for x in outs], 1)          # [2, steps, H, 128]
    want = np.stack([ref_o[cu[n] + T0[n]:cu[n] + T0[n] + steps] for n in range(2)])
    assert_gated_close(gpu, want, False)
    for n in range(2):
        if T0[n] + steps == lens[n]:
            assert_close(to64(S_pool[rows[n]]), ref_S[n], TOL_BF16, "S after the last token")


def test_decode_layer_slot_out_of_range_is_reported(kda):
    """A pool row outside [0, P) is refused by the kernel's bounds check: that request's
    output and every pool row stay untouched, KDA_ERR_DEVICE_CHECK names the request."""
    inp = synthetic.decode_layer_inputs(3, 2, 4, seed=53, device="cuda")
    inp.slot[1] = 7
    o = torch.full((3, 2, 128), -7.0, device="cuda")
    S_pool, conv_pool = inp.S_pool.clone(), inp.conv_pool.clone()
    kda.kda_decode_layer(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b, inp.beta_logit,
                         inp.g, inp.slot, S_pool, conv_pool, o=o)
    code, detail = kda.kda_get_device_status()
    assert code == 6 and detail == 1
    assert bool((o[1] == -7.0).all())
    assert bool((o[0] != -7.0).any()) and bool((o[2] != -7.0).any())
    untouched = sorted(set(range(4)) - {int(inp.slot[0]), int(inp.slot[2])})
    assert torch.equal(S_pool[untouched], inp.S_pool[untouched])
    assert torch.equal(conv_pool[untouched], inp.conv_pool[untouched])
