"""kda_layer_core_noalloc: the layer core for callers that cannot allocate device memory.

Such callers (a plugin that may not allocate outside its host's memory pool, a
latency-critical path that cannot afford an allocation) cannot hand
kda_layer_core a workspace; kda_layer_core_noalloc takes its scratch from a
fixed array inside the library instead.  These tests call it through the C ABI
and compare it with kda_layer_core, twice in a row with different inputs so
that whatever the first call left in the shared scratch cannot leak into the
second.  Both run the same kernels in the same order on the same inputs, only
with the scratch at another address, so the results must be identical bit for
bit.  The file is named to be collected last.
"""
import pytest
import torch

from gated_delta_rule_kda_gb300 import synthetic


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import build
    build.build()
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


@pytest.mark.gpu
def test_noalloc_matches_layer_core_twice(kda):
    cases = [([70, 1, 0, 33, 129], 4, 51, 0.1), ([200, 17], 3, 52, None)]
    for lens, H, seed, s0 in cases:
        inp = synthetic.layer_inputs(lens, H, seed=seed, s0_std=s0, device="cuda")
        T = inp.qp.shape[0]
        N = len(lens)
        assert kda.kda_layer_core_workspace_size(N, T, H) <= kda.NOALLOC_SCRATCH_BYTES
        ref_o, ref_S = kda.kda_layer_core(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A,
                                          inp.b, inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0,
                                          out_dtype=torch.float32)
        o = torch.full((T, H, 128), float("nan"), dtype=torch.float32, device="cuda")
        S = torch.full((N, H, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
        kda.kda_layer_core_noalloc(inp.qp, inp.kp, inp.vp, inp.conv_w, inp.z, inp.A, inp.b,
                                   inp.beta_logit, inp.g, inp.cu_seqlens, inp.S0, o=o,
                                   S_final=S)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o), "o_gated differs from kda_layer_core's"
        assert torch.equal(S, ref_S), "S_final differs from kda_layer_core's"
    status, _ = kda.kda_get_device_status()
    assert status == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(kda):
    """Too large for the fixed scratch: rejected on the host before any launch."""
    lib = kda.library()
    fake = 0x10000  # never dereferenced: the size check comes first
    rc = lib.kda_layer_core_noalloc(1, 1 << 20, 96, fake, fake, fake, fake, fake, fake, None,
                                    fake, fake, fake, None, 0.1, 1e-6, 1e-6, 0, fake, None, None)
    assert rc == 2  # KDA_ERR_UNSUPPORTED
