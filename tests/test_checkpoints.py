"""GPU state snapshots during a prefill (prefix-cache checkpoints) vs the fp64 oracle.

A snapshot of sequence n taken after its first m tokens must equal the final state of
the oracle's prefill over that m-token prefix alone (same S0).  Taking snapshots must
not change the prefill's own outputs, a snapshot at a sequence's last token is the
S_final of the same run bit for bit, snapshot slots that the offsets leave out (or that
lie past the sequence's end) stay untouched, and a prefill restarted from a snapshot
continues the sequence (the copy-on-write restore of a prefix-cache hit).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_kda_gb300 import synthetic
from tests._parity import TOL_BF16, TOL_FP32, assert_close, to64

pytestmark = pytest.mark.gpu

SENTINEL = -1234.5


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import build
    build.build()
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


def prefixes(cu, base, every):
    """(n, i, m): snapshot slot base[n] + i holds sequence n after m = (i + 1) every tokens,
    for every slot the offsets give whose token count lies inside the sequence."""
    out = []
    for n in range(len(cu) - 1):
        for i in range(base[n + 1] - base[n]):
            m = (i + 1) * every
            if m <= cu[n + 1] - cu[n]:
                out.append((n, i, m))
    return out


def gather_prefixes(cu, pre):
    """Token indices and cu_seqlens of the packed prefixes."""
    idx = np.concatenate([np.arange(cu[n], cu[n] + m) for n, _, m in pre]) if pre else \
        np.zeros(0, np.int64)
    cu_p = np.concatenate([[0], np.cumsum([m for _, _, m in pre])]).astype(np.int32)
    return idx, cu_p


def oracle_prefix_states(x, cu, S0, pre, heads):
    """Final states of the oracle prefill over each prefix.  x = (q, k, v, la, beta) fp64."""
    idx, cu_p = gather_prefixes(cu, pre)
    sub = [t[idx][:, heads] for t in x]
    S0p = None if S0 is None else S0[[n for n, _, _ in pre]][:, heads]
    return oracle.kda_prefill(*sub, cu_p, S0=S0p)[1]


def check_snapshots(ckpt, base, pre, ref, tol, heads):
    for j, (n, i, _) in enumerate(pre):
        assert_close(to64(ckpt[base[n] + i][heads]), ref[j], tol, f"snapshot seq {n} #{i}")


@pytest.mark.parametrize("dtype,every", [(torch.bfloat16, 32), (torch.bfloat16, 96),
                                         (torch.float32, 32), (torch.float32, 64)])
def test_prefill_snapshots_match_prefix_prefills(kda, dtype, every):
    lens = [229, 64, 31, 0, 130, 96, 1]
    inp = synthetic.prefill_inputs(lens, 3, dtype, seed=61, s0_std=0.1, device="cuda")
    o0, S0f = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens,
                              inp.S0, out_dtype=torch.float32)
    base = kda.checkpoint_offsets(inp.cu_seqlens, every)
    ckpt = torch.full((int(base[-1]), 3, 128, 128), SENTINEL, device="cuda")
    o, Sf, _, _ = kda.kda_prefill_with_checkpoints(
        inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens, every, inp.S0,
        ckpt_base=base.cuda(), ckpt_states=ckpt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    assert torch.equal(o, o0) and torch.equal(Sf, S0f), "snapshots changed the prefill's results"
    cu, b = inp.cu_seqlens.tolist(), base.tolist()
    pre = prefixes(cu, b, every)
    assert len(pre) == b[-1] == sum(l // every for l in lens)
    x = [to64(t) for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    ref = oracle_prefix_states(x, cu, to64(inp.S0), pre, [0, 1, 2])
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
    check_snapshots(ckpt, b, pre, ref, tol, [0, 1, 2])
    for n, i, m in pre:  # a snapshot at the last token is that run's S_final, bit for bit
        if m == lens[n]:
            assert torch.equal(ckpt[b[n] + i], Sf[n])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_slots_the_offsets_leave_out_stay_untouched(kda, dtype):
    """Sequence 0 gets one slot of three possible, sequence 1 four slots for two possible
    snapshots, sequence 2 (shorter than the interval) two slots: only the slots inside
    the sequences are written."""
    lens, every = [100, 70, 20], 32
    inp = synthetic.prefill_inputs(lens, 2, dtype, seed=62, s0_std=0.1, device="cuda")
    base = torch.tensor([0, 1, 5, 7], dtype=torch.int32)
    ckpt = torch.full((7, 2, 128, 128), SENTINEL, device="cuda")
    kda.kda_prefill_with_checkpoints(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta,
                                     inp.cu_seqlens, every, inp.S0, ckpt_base=base.cuda(),
                                     ckpt_states=ckpt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    written = [0, 1, 2]
    for slot in range(7):
        untouched = bool((ckpt[slot] == SENTINEL).all())
        assert untouched == (slot not in written), f"slot {slot}"
    cu = inp.cu_seqlens.tolist()
    pre = prefixes(cu, base.tolist(), every)
    assert [(n, i) for n, i, _ in pre] == [(0, 0), (1, 0), (1, 1)]
    x = [to64(t) for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    ref = oracle_prefix_states(x, cu, to64(inp.S0), pre, [0, 1])
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_FP32
    check_snapshots(ckpt, base.tolist(), pre, ref, tol, [0, 1])


def test_restart_from_a_snapshot_continues_the_sequence(kda):
    """Copy-on-write restore: a prefill of the last 77 tokens of a 237-token sequence from
    its snapshot after 160 tokens gives the full prefill's outputs and final state."""
    L, every, m = 237, 32, 160
    inp = synthetic.prefill_inputs([L], 4, torch.bfloat16, seed=63, s0_std=0.1, device="cuda")
    _, _, base, ckpt = kda.kda_prefill_with_checkpoints(
        inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens, every, inp.S0,
        out_dtype=torch.float32)
    slot = m // every - 1
    restored = ckpt[slot:slot + 1].clone()  # the request's private copy
    tail = lambda t: t[m:].contiguous()
    o_t, S_t = kda.kda_prefill(tail(inp.q), tail(inp.k), tail(inp.v), tail(inp.log_alpha),
                               tail(inp.beta), synthetic.cu_from_lengths([L - m], "cuda"),
                               restored, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    o_ref, S_ref = oracle.kda_prefill(*[to64(t) for t in (inp.q, inp.k, inp.v, inp.log_alpha,
                                                          inp.beta)],
                                      inp.cu_seqlens.cpu().numpy(), S0=to64(inp.S0))
    assert_close(to64(o_t), o_ref[m:], TOL_BF16, "o after the restore")
    assert_close(to64(S_t), S_ref, TOL_BF16, "S_final after the restore")
    assert bool((ckpt[slot] == restored[0]).all()), "the shared snapshot was modified"


@pytest.mark.parametrize("every", [32, 64])
def test_fused_layer_core_snapshots(kda, every):
    """The fused layer core's snapshots against the oracle layer core over each prefix (the
    short convolution is causal inside a sequence, so a prefix's final state is the state
    after that many tokens)."""
    lens = [150, 33, 0, 96, 5]
    inp = synthetic.layer_inputs(lens, 2, seed=64, s0_std=0.1, device="cuda")
    o0, Sf0 = kda.kda_layer_core_fused(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                       inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0)
    base = kda.checkpoint_offsets(inp.cu_seqlens, every)
    ckpt = torch.full((int(base[-1]), 2, 128, 128), SENTINEL, device="cuda")
    o, Sf, _, _ = kda.kda_layer_core_fused_with_checkpoints(
        inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b, inp.beta_logit, inp.g,
        inp.cu_seqlens, every, inp.S0, ckpt_base=base.cuda(), ckpt_states=ckpt)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    assert torch.equal(o, o0) and torch.equal(Sf, Sf0)
    cu, b = inp.cu_seqlens.tolist(), base.tolist()
    pre = prefixes(cu, b, every)
    assert len(pre) == b[-1]
    idx, cu_p = gather_prefixes(cu, pre)
    sub = lambda t: to64(t)[idx]
    S0p = to64(inp.S0)[[n for n, _, _ in pre]]
    _, ref = oracle.kda_layer_core(sub(inp.qp), sub(inp.kp), sub(inp.vp), to64(inp.conv_w),
                                   sub(inp.z), to64(inp.A), to64(inp.b), sub(inp.beta_logit),
                                   sub(inp.g), cu_p, S0=S0p)
    check_snapshots(ckpt, b, pre, ref, TOL_BF16, [0, 1])
    for n, i, m in pre:
        if m == lens[n]:
            assert torch.equal(ckpt[b[n] + i], Sf[n])


def test_full_size_snapshots_sampled_heads(kda):
    """1 x 8192 tokens x 96 heads (the prefill workload) with a snapshot every 1024 tokens:
    snapshots 0, 3 and 7 of heads 0, 50 and 95 against the oracle."""
    every, heads = 1024, [0, 50, 95]
    inp = synthetic.prefill_inputs([8192], 96, torch.bfloat16, device="cuda")
    _, Sf, base, ckpt = kda.kda_prefill_with_checkpoints(
        inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens, every, inp.S0)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status()[0] == 0
    assert base.tolist() == [0, 8]
    x = [to64(t[:, heads]) for t in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta)]
    S = None
    for i in range(8):  # the oracle segment by segment: each segment resumes from the last
        seg = [t[i * every:(i + 1) * every] for t in x]
        S = oracle.kda_prefill(*seg, np.array([0, every], np.int32), S0=S)[1]
        if i in (0, 3, 7):
            assert_close(to64(ckpt[i][heads]), S[0], TOL_BF16, f"snapshot {i}")
    assert torch.equal(ckpt[7], Sf[0])
