"""GPU layer core for a few tokens per request from pooled states (layer-level speculative
verify and replay) vs the fp64 oracle, through the C ABI.

Gated outputs and state rows are checked with the plain 2e-3 max-abs/rms bound; convolution-state rows are bit-exact (they only move bf16 inputs); rows that no
request advances stay bit-identical.
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


def reference(inp, write_back, heads=None):
    H_all = inp.qp.shape[1]
    hs = list(range(H_all)) if heads is None else heads
    sel = lambda t: to64(t)[:, hs]
    conv_w = to64(inp.conv_w).reshape(3, H_all, 128, 4)[:, hs].reshape(3, len(hs) * 128, 4)
    return oracle.kda_decode_layer_tokens(
        sel(inp.qp), sel(inp.kp), sel(inp.vp), conv_w, sel(inp.z), to64(inp.A)[hs],
        to64(inp.b)[hs], sel(inp.beta_logit), sel(inp.g), inp.cu_tokens.cpu().numpy(),
        inp.slot.cpu().numpy(), to64(inp.S_pool)[:, hs], to64(inp.conv_pool)[:, :, :, hs],
        write_back)


def run(kda, inp, write_back, out_dtype=torch.float32):
    S_pool, conv_pool = inp.S_pool.clone(), inp.conv_pool.clone()
    o = kda.kda_decode_layer_tokens(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                    inp.beta_logit, inp.g, inp.cu_tokens, inp.slot, S_pool,
                                    conv_pool, write_back, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return o, S_pool, conv_pool


@pytest.mark.parametrize("out_dtype,write_back", [(torch.float32, False), (torch.float32, True),
                                                  (torch.bfloat16, True)])
def test_ragged_requests_shuffled_pools(kda, out_dtype, write_back):
    """Requests of 3, 0, 1, 16, 5 and 2 tokens in shuffled rows of 9-row pools, H=3."""
    inp = synthetic.decode_layer_tokens_inputs([3, 0, 1, 16, 5, 2], 3, 9, seed=91, device="cuda")
    o, S_pool, conv_pool = run(kda, inp, write_back, out_dtype)
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S, ref_conv = reference(inp, write_back)
    assert_gated_close(to64(o), ref_o, out_dtype == torch.bfloat16)
    slot = inp.slot.cpu().numpy()
    if write_back:
        assert_close(to64(S_pool)[slot], ref_S[slot], TOL_BF16, "S_pool rows")
        assert torch.equal(conv_pool.float().cpu(), torch.from_numpy(ref_conv).float())
    else:
        assert torch.equal(S_pool, inp.S_pool) and torch.equal(conv_pool, inp.conv_pool)
    free = sorted(set(range(9)) - set(slot.tolist()))
    assert torch.equal(S_pool[free], inp.S_pool[free])
    assert torch.equal(conv_pool[free], inp.conv_pool[free])


def test_verify_may_share_rows(kda):
    inp = synthetic.decode_layer_tokens_inputs([4, 2, 7], 2, 4, seed=92, device="cuda")
    inp.slot[:] = 1
    o, S_pool, conv_pool = run(kda, inp, False)
    assert kda.kda_get_device_status()[0] == 0
    ref_o, _, _ = reference(inp, False)
    assert_gated_close(to64(o), ref_o, False)
    assert torch.equal(S_pool, inp.S_pool) and torch.equal(conv_pool, inp.conv_pool)


def test_continues_the_fused_prefill_in_drafts(kda):
    """The fused layer core over the first T0 tokens of two sequences, their states moved
    into pool rows 3 and 0, then the remaining tokens as verify-then-replay rounds of up to
    5 tokens (4 accepted, or all of the last ones): the outputs of the accepted tokens and
    the final rows against the oracle layer core over whole sequences."""
    lens, T0, H = [41, 60], [9, 30], 2
    inp = synthetic.layer_inputs(lens, H, seed=93, s0_std=0.1, device="cuda")
    cu = inp.cu_seqlens.tolist()
    idx = torch.cat([torch.arange(cu[n], cu[n] + T0[n]) for n in range(2)]).cuda()
    sub = lambda t: t[idx].contiguous()
    _, Sf = kda.kda_layer_core_fused(sub(inp.qp), sub(inp.kp), sub(inp.vp), inp.conv_w, sub(inp.z),
                                     inp.A, inp.b, sub(inp.beta_logit), sub(inp.g),
                                     synthetic.cu_from_lengths(T0, "cuda"), inp.S0,
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
    pos = [cu[n] + T0[n] for n in range(2)]
    got = {}
    while any(pos[n] < cu[n + 1] for n in range(2)):
        draft = [list(range(pos[n], min(pos[n] + 5, cu[n + 1]))) for n in range(2)]
        ids = torch.tensor(draft[0] + draft[1], dtype=torch.long, device="cuda")
        cu_d = synthetic.cu_from_lengths([len(d) for d in draft], "cuda")
        pick = lambda x: x[ids].contiguous()
        args = (pick(inp.qp), pick(inp.kp), pick(inp.vp), inp.conv_w, pick(inp.z), inp.A, inp.b,
                pick(inp.beta_logit), pick(inp.g), cu_d, slot, S_pool, conv_pool)
        o_draft = kda.kda_decode_layer_tokens(*args, False, out_dtype=torch.float32)
        acc = [min(4, len(d)) if pos[n] + len(d) < cu[n + 1] else len(d) for n, d in enumerate(draft)]
        ids_a = torch.tensor(draft[0][:acc[0]] + draft[1][:acc[1]], dtype=torch.long, device="cuda")
        pick_a = lambda x: x[ids_a].contiguous()
        kda.kda_decode_layer_tokens(pick_a(inp.qp), pick_a(inp.kp), pick_a(inp.vp), inp.conv_w,
                                    pick_a(inp.z), inp.A, inp.b, pick_a(inp.beta_logit),
                                    pick_a(inp.g), synthetic.cu_from_lengths(acc, "cuda"), slot,
                                    S_pool, conv_pool, True, out_dtype=torch.float32)
        off = 0
        for n in range(2):
            for j in range(acc[n]):
                got[draft[n][j]] = o_draft[off + j]
            off += len(draft[n])
            pos[n] += acc[n]
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    ref_o, ref_S = oracle.kda_layer_core(to64(inp.qp), to64(inp.kp), to64(inp.vp), to64(inp.conv_w),
                                         to64(inp.z), to64(inp.A), to64(inp.b), to64(inp.beta_logit),
                                         to64(inp.g), inp.cu_seqlens.cpu().numpy(), S0=to64(inp.S0))
    ts = sorted(got)
    gpu = np.stack([to64(got[t]) for t in ts])
    assert_gated_close(gpu, ref_o[ts], False)
    for n in range(2):
        assert_close(to64(S_pool[rows[n]]), ref_S[n], TOL_BF16, "row after the last token")


def test_full_batch_sampled_heads(kda):
    """256 requests x 4 tokens x 96 heads in 320-row pools; the oracle on heads 0, 47, 95."""
    inp = synthetic.decode_layer_tokens_inputs([4] * 256, 96, 320, device="cuda")
    o, S_pool, conv_pool = run(kda, inp, True, torch.bfloat16)
    assert kda.kda_get_device_status()[0] == 0
    heads = [0, 47, 95]
    ref_o, ref_S, ref_conv = reference(inp, True, heads)
    assert_gated_close(to64(o[:, heads]), ref_o, True)
    slot = inp.slot.cpu().numpy()
    assert_close(to64(S_pool[:, heads])[slot], ref_S[slot], TOL_BF16, "S_pool rows")
    assert torch.equal(conv_pool[:, :, :, heads].float().cpu(), torch.from_numpy(ref_conv).float())


@pytest.mark.parametrize("bad", ["slot", "range", "too_many"])
def test_refused_requests_are_reported(kda, bad):
    lens = [2, 17, 3] if bad == "too_many" else [2, 3, 3]
    inp = synthetic.decode_layer_tokens_inputs(lens, 2, 4, seed=94, device="cuda")
    if bad == "slot":
        inp.slot[1] = -1
    elif bad == "range":
        inp.cu_tokens[2] = int(inp.cu_tokens[3]) + 4
        inp.cu_tokens[3] = int(inp.cu_tokens[3]) + 4
    T = inp.qp.shape[0]
    S_pool, conv_pool = inp.S_pool.clone(), inp.conv_pool.clone()
    o = torch.full((T, 2, 128), -7.0, device="cuda")
    kda.kda_decode_layer_tokens(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                inp.beta_logit, inp.g, inp.cu_tokens, inp.slot, S_pool, conv_pool,
                                True, o=o)
    code, detail = kda.kda_get_device_status()
    assert code == 6
    assert detail in ((1,) if bad != "range" else (1, 2))
    t0 = int(inp.cu_tokens[0]), int(inp.cu_tokens[1])
    assert bool((o[t0[0]:t0[1]] != -7.0).all())  # request 0 ran
    if bad != "range":
        t1 = int(inp.cu_tokens[1]), int(inp.cu_tokens[2])
        assert bool((o[t1[0]:t1[1]] == -7.0).all())  # request 1 refused
        n1 = int(inp.slot[1])
        if 0 <= n1 < 4:
            assert torch.equal(S_pool[n1], inp.S_pool[n1]) and torch.equal(conv_pool[n1], inp.conv_pool[n1])
