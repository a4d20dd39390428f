"""GPU decode of a few tokens per request from pooled states (speculative verify and
replay) vs the fp64 oracle, through the C ABI.

Outputs and states use the contract's bounds (2e-3 max-abs/rms for bf16 inputs, 1e-5 for
fp32); pool rows that no request advances stay bit-identical.
"""
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


def reference(inp, write_back, heads=None):
    sl = (lambda t: t) if heads is None else (lambda t: t[:, heads])
    return oracle.kda_decode_tokens(to64(sl(inp.q)), to64(sl(inp.k)), to64(sl(inp.v)),
                                    to64(sl(inp.log_alpha)), to64(sl(inp.beta)),
                                    inp.cu_tokens.cpu().numpy(), inp.slot.cpu().numpy(),
                                    to64(sl(inp.S_pool)), write_back)


def run(kda, inp, write_back, out_dtype=torch.float32, with_final=True):
    S_pool = inp.S_pool.clone()
    B, H = inp.slot.shape[0], inp.q.shape[1]
    Sf = torch.full((B, H, 128, 128), -7.0, device="cuda") if with_final else None
    o = kda.kda_decode_tokens(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_tokens,
                              inp.slot, S_pool, write_back, S_final=Sf, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    return o, S_pool, Sf


@pytest.mark.parametrize("dtype,out_dtype,write_back", [
    (torch.bfloat16, torch.float32, False), (torch.bfloat16, torch.float32, True),
    (torch.bfloat16, torch.bfloat16, True), (torch.float32, torch.float32, True)])
def test_ragged_requests_shuffled_pool(kda, dtype, out_dtype, write_back):
    """Requests of 3, 0, 1, 8, 13 and 4 tokens (13 spans two staged batches) in shuffled
    rows of a 9-row pool, H=3."""
    inp = synthetic.decode_tokens_inputs([3, 0, 1, 8, 13, 4], 3, 9, dtype, seed=71, device="cuda")
    o, S_pool, Sf = run(kda, inp, write_back, out_dtype)
    ref_o, ref_pool, ref_f = reference(inp, write_back)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
    assert_close(to64(o), ref_o, tol, "o", out_is_bf16=out_dtype == torch.bfloat16)
    assert_close(to64(Sf), ref_f, tol, "S_final")
    slot = inp.slot.cpu().numpy()
    if write_back:
        assert_close(to64(S_pool)[slot], ref_pool[slot], tol, "advanced pool rows")
        assert torch.equal(S_pool[slot], Sf), "pool rows and S_final differ"
    else:
        assert torch.equal(S_pool, inp.S_pool), "verify changed the pool"
    free = sorted(set(range(9)) - set(slot.tolist()))
    assert torch.equal(S_pool[free], inp.S_pool[free])


def test_verify_may_share_a_row(kda):
    """Three draft branches verified from the same cached row (no write-back)."""
    inp = synthetic.decode_tokens_inputs([4, 2, 5], 2, 4, seed=72, device="cuda")
    inp.slot[:] = 2
    o, S_pool, Sf = run(kda, inp, False)
    ref_o, _, ref_f = reference(inp, False)
    assert_close(to64(o), ref_o, TOL_BF16, "o")
    assert_close(to64(Sf), ref_f, TOL_BF16, "S_final")
    assert torch.equal(S_pool, inp.S_pool)


def test_verify_accept_replay_cycle(kda):
    """Verify a 5-token draft per request, accept 0, 2, 5 and 3 tokens, replay the accepted
    ones into the rows, then verify the next draft: everything against the oracle prefill of
    the accepted stream."""
    lens, acc = [5, 5, 5, 5], [0, 2, 5, 3]
    inp = synthetic.decode_tokens_inputs(lens, 2, 6, seed=73, device="cuda")
    S_pool = inp.S_pool.clone()
    o_draft = kda.kda_decode_tokens(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_tokens,
                                    inp.slot, S_pool, False, out_dtype=torch.float32)
    idx = torch.cat([torch.arange(5 * b, 5 * b + acc[b]) for b in range(4)]).cuda()
    cu_acc = synthetic.cu_from_lengths(acc, "cuda")
    pick = lambda t: t[idx].contiguous()
    kda.kda_decode_tokens(pick(inp.q), pick(inp.k), pick(inp.v), pick(inp.log_alpha),
                          pick(inp.beta), cu_acc, inp.slot, S_pool, True)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    x = [to64(t) for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    slot = inp.slot.cpu().numpy()
    S0 = to64(inp.S_pool)[slot]
    ref_o, ref_S = oracle.kda_prefill(*x, inp.cu_tokens.cpu().numpy(), S0=S0)
    assert_close(to64(o_draft), ref_o, TOL_BF16, "draft outputs")
    idx_np = idx.cpu().numpy()
    _, ref_acc = oracle.kda_prefill(*[t[idx_np] for t in x], cu_acc.cpu().numpy(), S0=S0)
    assert_close(to64(S_pool)[slot], ref_acc, TOL_BF16, "rows after the replay")
    assert torch.equal(S_pool[slot[0]], inp.S_pool[slot[0]])  # nothing accepted: row unchanged


def test_full_batch_sampled_heads(kda):
    """256 requests x 4 tokens x 96 heads in a 320-row pool (the decode workload with a
    3-token draft); the oracle on heads 0, 47 and 95."""
    inp = synthetic.decode_tokens_inputs([4] * 256, 96, 320, device="cuda")
    o, S_pool, _ = run(kda, inp, True, torch.bfloat16, with_final=False)
    heads = [0, 47, 95]
    ref_o, ref_pool, _ = reference(inp, True, heads)
    assert_close(to64(o[:, heads]), ref_o, TOL_BF16, "o", out_is_bf16=True)
    slot = inp.slot.cpu().numpy()
    assert_close(to64(S_pool[:, heads])[slot], ref_pool[slot], TOL_BF16, "pool rows")


@pytest.mark.parametrize("bad", ["slot", "range"])
def test_refused_requests_are_reported(kda, bad):
    """A pool row outside [0, P) (request 1), or a token range past T (request 2), is
    refused by the kernel: that request's outputs and row stay untouched, the others run,
    KDA_ERR_DEVICE_CHECK names it."""
    inp = synthetic.decode_tokens_inputs([2, 3, 2], 2, 4, seed=74, device="cuda")
    if bad == "slot":
        b_bad, rows = 1, slice(2, 5)
        inp.slot[1] = 4
    else:
        b_bad, rows = 2, slice(5, 7)
        inp.cu_tokens[3] = 9  # request 2 claims tokens 5..8 of 7
    S_pool = inp.S_pool.clone()
    o = torch.full((7, 2, 128), -7.0, device="cuda")
    kda.kda_decode_tokens(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_tokens, inp.slot,
                          S_pool, True, o=o)
    code, detail = kda.kda_get_device_status()
    assert code == 6 and detail == b_bad
    assert bool((o[rows] == -7.0).all())
    ok = [b for b in range(3) if b != b_bad]
    for b in ok:
        t0, t1 = int(inp.cu_tokens[b]), int(inp.cu_tokens[b + 1])
        assert bool((o[t0:t1] != -7.0).all())
    advanced = {int(inp.slot[b]) for b in ok}
    untouched = sorted(set(range(4)) - advanced)
    assert torch.equal(S_pool[untouched], inp.S_pool[untouched])


def test_many_units_with_refused_and_empty_requests(kda):
    """More units than resident CTAs (each CTA walks several, prefetching the next one's
    state), with empty requests and one refused request among them."""
    rng = np.random.default_rng(75)
    lens = rng.integers(0, 7, size=700).tolist()
    inp = synthetic.decode_tokens_inputs(lens, 1, 800, seed=75, device="cuda")
    inp.slot[333] = 800
    S_pool = inp.S_pool.clone()
    T = int(inp.cu_tokens[-1])
    o = torch.full((T, 1, 128), -7.0, device="cuda")
    kda.kda_decode_tokens(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_tokens, inp.slot,
                          S_pool, True, o=o, out_dtype=torch.float32)
    code, detail = kda.kda_get_device_status()
    assert code == 6 and detail == 333
    cu = inp.cu_tokens.cpu().numpy()
    keep = [b for b in range(700) if b != 333]
    slot = inp.slot.cpu().numpy()
    ref_o, _, _ = oracle.kda_decode_tokens(
        to64(inp.q), to64(inp.k), to64(inp.v), to64(inp.log_alpha), to64(inp.beta), cu,
        np.where(np.arange(700) == 333, 0, slot), to64(inp.S_pool), False)  # outputs only
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in keep])
    assert_close(to64(o)[rows], ref_o[rows], TOL_BF16, "o")
    assert bool((o[cu[333]:cu[334]] == -7.0).all())
    # advanced rows (a sample) against the oracle prefill of each request's tokens
    for b in keep[::37]:
        n = slot[b]
        t0, t1 = cu[b], cu[b + 1]
        _, S_ref = oracle.kda_prefill(to64(inp.q)[t0:t1], to64(inp.k)[t0:t1], to64(inp.v)[t0:t1],
                                      to64(inp.log_alpha)[t0:t1], to64(inp.beta)[t0:t1],
                                      [0, t1 - t0], S0=to64(inp.S_pool)[n:n + 1])
        assert_close(to64(S_pool[n]), S_ref[0], TOL_BF16, f"row of request {b}")
    untouched = sorted(set(range(800)) - {int(slot[b]) for b in keep})
    assert torch.equal(S_pool[untouched], inp.S_pool[untouched])


def test_decay_reset_minus_infinity(kda):
    """log alpha = -inf (alpha = 0) clears the row's state at that token; decode accepts it."""
    inp = synthetic.decode_tokens_inputs([3, 5, 2], 2, 4, torch.float32, seed=76, device="cuda")
    inp.log_alpha[1] = -float("inf")   # request 0, token 1
    inp.log_alpha[6, 1] = -float("inf")  # request 1, token 3, head 1
    o, S_pool, Sf = run(kda, inp, True)
    ref_o, ref_pool, ref_f = reference(inp, True)
    assert_close(to64(o), ref_o, TOL_FP32, "o")
    assert_close(to64(Sf), ref_f, TOL_FP32, "S_final")
