"""GPU contents checks of prefill inputs (kda_check_prefill_inputs): offsets that do not
start at 0, decrease or miss T, and log alpha outside [-5, 0] (or NaN), reported through the
device status word as KDA_ERR_DEVICE_CHECK with (kind << 28) | index."""
import pytest
import torch

from gated_delta_rule_kda_gb300 import synthetic

pytestmark = pytest.mark.gpu
CHECK = 6


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import build
    build.build()
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


def status(kda):
    return kda.kda_get_device_status()


@pytest.mark.parametrize("head_decay", [False, True])
def test_valid_inputs_pass(kda, head_decay):
    inp = synthetic.prefill_inputs([100, 0, 37], 3, device="cuda", head_decay=head_decay)
    inp.log_alpha[0].fill_(-5.0)
    inp.log_alpha[1].fill_(0.0)
    kda.kda_check_prefill_inputs(inp.cu_seqlens, inp.log_alpha)
    assert status(kda) == (0, 0)


@pytest.mark.parametrize("cu,n", [([1, 5, 9], 0), ([0, 6, 5, 9], 2), ([0, 4, 8], 2)])
def test_bad_offsets(kda, cu, n):
    c = torch.tensor(cu, dtype=torch.int32, device="cuda")
    kda.kda_check_prefill_inputs(c, total_tokens=9, num_heads=2)
    assert status(kda) == (CHECK, (1 << 28) | n)


@pytest.mark.parametrize("head_decay", [False, True])
@pytest.mark.parametrize("value", [-6.0, 0.5, float("nan")])
def test_decay_out_of_range(kda, head_decay, value):
    inp = synthetic.prefill_inputs([64, 50], 2, device="cuda", head_decay=head_decay)
    inp.log_alpha[77, 1] = value  # token 77, head 1 (all channels when per-channel)
    kda.kda_check_prefill_inputs(inp.cu_seqlens, inp.log_alpha)
    assert status(kda) == (CHECK, (2 << 28) | 77)
    # cleared by the read: a second valid check passes
    inp.log_alpha[77, 1] = -1.0
    kda.kda_check_prefill_inputs(inp.cu_seqlens, inp.log_alpha)
    assert status(kda) == (0, 0)


def test_debug_library_checks_inside_prefill(kda):
    """The debug build (KDA_DEBUG defined) runs the checks inside kda_prefill: a decay below
    the floor is reported although the caller made no check call."""
    import ctypes
    from gated_delta_rule_kda_gb300 import build
    lib = ctypes.CDLL(build.build(debug=True))
    inp = synthetic.prefill_inputs([40], 2, device="cuda")
    inp.log_alpha[13, 0, 5] = -7.0
    o = torch.empty((40, 2, 128), dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    lib.kda_prefill.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32] + [ctypes.c_void_p] * 7 + [
                                ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.kda_prefill(0, 0, 1, 40, 2, P(inp.q), P(inp.k), P(inp.v), P(inp.log_alpha),
                         P(inp.beta), None, P(inp.cu_seqlens), 0.0883883, P(o), None, None, 0,
                         stream)
    assert rc == 0
    detail = ctypes.c_uint32(0)
    lib.kda_get_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    assert lib.kda_get_device_status(stream, ctypes.byref(detail)) == CHECK
    assert detail.value == (2 << 28) | 13
