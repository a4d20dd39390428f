"""A device-side wait that runs out, on purpose, in the one safe form.

Every wait inside the tensor-core prefill is bounded; when one gives up, the kernel records
KDA_ERR_DEVICE_TIMEOUT with the place it waited, leaves through its normal exit (the final
barrier and the release of its tensor memory), and the context stays usable.  The debug
library (KDA_DEBUG) can arm one launch in which the warps that build a chunk's operands skip
their first "chunk ready" hand-off before anything is issued into that chunk's slot, with
every wait limited to 1 ms, so that the consuming warps' wait for the chunk runs out with no
copy or tensor-core product in flight.  Nothing faults, traps or hangs: the test checks the
reported status, then that the next prefill through the same library is correct.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_kda_gb300 import synthetic
from tests._parity import TOL_BF16, assert_close, to64

TIMEOUT = 5
UNSUPPORTED = 2
WAIT_FOR_READY_CHUNK = 20


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import build
    build.build()
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


def test_normal_library_refuses_the_injection(kda):
    """Only the debug library arms anything; the normal one says so and changes nothing."""
    assert kda.library().kda_debug_inject_handoff_timeout() == UNSUPPORTED


def _prefill(lib, inp, o, S_final, stream):
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    T, H = inp.q.shape[:2]
    N = inp.cu_seqlens.numel() - 1
    return lib.kda_prefill(0, 1, N, T, H, P(inp.q), P(inp.k), P(inp.v), P(inp.log_alpha),
                           P(inp.beta), None, P(inp.cu_seqlens), 1.0 / np.sqrt(128.0), P(o),
                           P(S_final), None, 0, stream)


@pytest.mark.gpu
def test_debug_library_reports_a_wait_that_runs_out(kda):
    from gated_delta_rule_kda_gb300 import build
    lib = ctypes.CDLL(build.build(debug=True))
    lib.kda_prefill.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32] + [ctypes.c_void_p] * 7 + [
                                ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.kda_get_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    lib.kda_debug_inject_handoff_timeout.argtypes = []
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    detail = ctypes.c_uint32(0)
    assert lib.kda_get_device_status(stream, ctypes.byref(detail)) == 0

    # two chunks (50 tokens) per (sequence, head): the skipped hand-off is the only one the
    # consuming warps wait for, and the building warps finish on their own
    inp = synthetic.prefill_inputs([50], 2, torch.bfloat16, seed=61, device="cuda")
    o = torch.zeros((50, 2, 128), dtype=torch.float32, device="cuda")
    Sf = torch.zeros((1, 2, 128, 128), dtype=torch.float32, device="cuda")
    assert lib.kda_debug_inject_handoff_timeout() == 0
    assert _prefill(lib, inp, o, Sf, stream) == 0
    assert lib.kda_get_device_status(stream, ctypes.byref(detail)) == TIMEOUT
    assert detail.value == WAIT_FOR_READY_CHUNK

    # the injection was for that launch only: the next prefill is whole and correct
    assert _prefill(lib, inp, o, Sf, stream) == 0
    assert lib.kda_get_device_status(stream, ctypes.byref(detail)) == 0
    f = to64
    ref_o, ref_S = oracle.kda_prefill(f(inp.q), f(inp.k), f(inp.v), f(inp.log_alpha),
                                      f(inp.beta), inp.cu_seqlens.cpu().numpy())
    assert_close(to64(o), ref_o, TOL_BF16, "o after the timed-out launch")
    assert_close(to64(Sf), ref_S, TOL_BF16, "S_final after the timed-out launch")
