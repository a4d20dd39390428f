"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every entry point include/kda.h declares, and rejects bad arguments
on the host before any launch (nothing is dereferenced in these calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_kda_gb300 import build
    build.build()
    from gated_delta_rule_kda_gb300 import kda as mod
    return mod


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(kda_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(kda):
    declared = declared_symbols()
    assert declared, "no declarations parsed"
    assert declared == set(kda.EXPORTED)
    lib = kda.library()
    for name in declared:
        assert hasattr(lib, name), name
    # and the shared object's dynamic symbol table really has them
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", kda.library_path()], capture_output=True,
                         text=True).stdout
    for name in declared:
        assert re.search(rf"\bT {name}$", out, re.M), f"{name} not exported"


def test_status_strings(kda):
    lib = kda.library()
    for code, name in kda.STATUS_NAMES.items():
        assert lib.kda_status_string(code).decode() == name
    assert lib.kda_version() >= 100


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first
MIS = 0x10008   # misaligned


def _prefill(lib, **kw):
    a = dict(in_dt=0, out_dt=0, N=1, T=4, H=2, q=FAKE, k=FAKE, v=FAKE, la=FAKE, beta=FAKE,
             S0=None, cu=FAKE, scale=0.1, o=FAKE, Sf=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.kda_prefill(a["in_dt"], a["out_dt"], a["N"], a["T"], a["H"], a["q"], a["k"],
                           a["v"], a["la"], a["beta"], a["S0"], a["cu"], a["scale"], a["o"],
                           a["Sf"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("bad", [
    dict(in_dt=7), dict(out_dt=-1), dict(N=0), dict(H=0), dict(T=-1),
    dict(q=None), dict(k=MIS), dict(v=None), dict(la=MIS), dict(beta=None), dict(o=None),
    dict(cu=None), dict(S0=MIS), dict(Sf=MIS),
    dict(S0=FAKE, Sf=FAKE + 64),   # partial overlap of S0 and S_final
])
def test_prefill_rejects_bad_arguments(kda, bad):
    assert _prefill(kda.library(), **bad) == 1  # KDA_ERR_INVALID_ARGUMENT


def test_prefill_too_many_heads_unsupported(kda):
    assert _prefill(kda.library(), H=70000) == 2


@pytest.mark.parametrize("bad", [dict(B=0), dict(H=0), dict(q=None), dict(S=MIS), dict(o=None),
                                 dict(in_dt=3)])
def test_decode_rejects_bad_arguments(kda, bad):
    a = dict(in_dt=0, out_dt=0, B=2, H=2, q=FAKE, k=FAKE, v=FAKE, la=FAKE, beta=FAKE, S=FAKE,
             o=FAKE)
    a.update(bad)
    rc = kda.library().kda_decode_step(a["in_dt"], a["out_dt"], a["B"], a["H"], a["q"], a["k"],
                                       a["v"], a["la"], a["beta"], a["S"], 0.1, a["o"], None)
    assert rc == 1


def test_frontend_and_gate_reject_bad_arguments(kda):
    lib = kda.library()
    rc = lib.kda_frontend(1, 4, 2, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, FAKE, 1e-6, 0,
                          FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert rc == 1
    rc = lib.kda_frontend(1, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, MIS, FAKE, FAKE, 1e-6, 0,
                          FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert rc == 1
    assert lib.kda_output_gate(8, 0, None, FAKE, 1e-6, 0, FAKE, None) == 1
    assert lib.kda_output_gate(8, 0, FAKE, FAKE, 1e-6, 9, FAKE, None) == 1
    assert lib.kda_output_gate(-1, 0, FAKE, FAKE, 1e-6, 0, FAKE, None) == 1


def test_workspace_size_is_callable(kda):
    assert kda.kda_prefill_workspace_size(1, 8192, 96) >= 0


def test_layer_core_rejects_missing_workspace(kda):
    lib = kda.library()
    rc = lib.kda_layer_core(1, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE,
                            None, 0.1, 1e-6, 1e-6, 0, FAKE, None, None, 0, None)
    assert rc == 3  # KDA_ERR_WORKSPACE
    rc = lib.kda_layer_core(1, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE,
                            None, 0.1, 1e-6, 1e-6, 0, FAKE, None, FAKE, 1 << 20, None)
    assert rc == 1  # g missing
    assert kda.kda_layer_core_workspace_size(16, 1000, 96) > 1000 * 96 * 128 * 2 * 3


def _fused(lib, **kw):
    a = dict(N=1, T=4, H=2, qp=FAKE, kp=FAKE, vp=FAKE, w=FAKE, z=FAKE, A=FAKE, b=None, bl=FAKE,
             g=FAKE, cu=FAKE, S0=None, out_dt=0, o=FAKE, Sf=None)
    a.update(kw)
    return lib.kda_layer_core_fused(a["N"], a["T"], a["H"], a["qp"], a["kp"], a["vp"], a["w"],
                                    a["z"], a["A"], a["b"], a["bl"], a["g"], a["cu"], a["S0"], 0.1,
                                    1e-6, 1e-6, a["out_dt"], a["o"], a["Sf"], None)


@pytest.mark.parametrize("bad", [
    dict(out_dt=5), dict(N=0), dict(H=0), dict(T=-1), dict(qp=None), dict(kp=MIS), dict(vp=None),
    dict(w=MIS), dict(z=None), dict(A=None), dict(b=MIS), dict(bl=None), dict(g=None),
    dict(o=MIS), dict(cu=None), dict(S0=MIS), dict(S0=FAKE, Sf=FAKE + 64),
])
def test_layer_core_fused_rejects_bad_arguments(kda, bad):
    assert _fused(kda.library(), **bad) == 1  # KDA_ERR_INVALID_ARGUMENT, before any launch


def test_layer_core_fused_too_many_heads_unsupported(kda):
    assert _fused(kda.library(), H=70000) == 2


# Checkpoint arguments: every must be 0 or a positive multiple of 32; with every > 0 the
# offsets need 4-byte and the snapshot states 16-byte alignment.
BAD_CKPT = [dict(every=-32), dict(every=16), dict(every=48), dict(every=1),
            dict(every=32, base=None), dict(every=32, base=FAKE + 2),
            dict(every=32, states=None), dict(every=64, states=MIS)]


def _ckpt(kw):
    c = dict(every=32, base=FAKE, states=FAKE + (1 << 30))
    c.update(kw)
    return c


@pytest.mark.parametrize("bad", BAD_CKPT)
def test_prefill_with_checkpoints_rejects_bad_checkpoint_arguments(kda, bad):
    c = _ckpt(bad)
    rc = kda.library().kda_prefill_with_checkpoints(
        0, 0, 1, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 0.1, FAKE, None, None, 0,
        c["every"], c["base"], c["states"], None)
    assert rc == 1


@pytest.mark.parametrize("bad", BAD_CKPT)
def test_layer_core_fused_with_checkpoints_rejects_bad_checkpoint_arguments(kda, bad):
    c = _ckpt(bad)
    rc = kda.library().kda_layer_core_fused_with_checkpoints(
        1, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, 0.1, 1e-6,
        1e-6, 0, FAKE, None, c["every"], c["base"], c["states"], None)
    assert rc == 1


def test_with_checkpoints_still_validates_the_prefill_arguments(kda):
    lib = kda.library()
    rc = lib.kda_prefill_with_checkpoints(0, 0, 1, 4, 2, None, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                          0.1, FAKE, None, None, 0, 32, FAKE, FAKE + (1 << 30),
                                          None)
    assert rc == 1  # q missing
    rc = lib.kda_layer_core_fused_with_checkpoints(1, 4, 70000, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                                   None, FAKE, FAKE, FAKE, None, 0.1, 1e-6, 1e-6,
                                                   0, FAKE, None, 32, FAKE, FAKE + (1 << 30), None)
    assert rc == 2  # too many heads


def test_checkpoint_offsets(kda):
    base = kda.checkpoint_offsets([0, 100, 100, 164, 500], 32)
    assert base.tolist() == [0, 3, 3, 5, 15]
    assert kda.checkpoint_offsets([0, 31], 32).tolist() == [0, 0]


def _decode_layer(lib, **kw):
    a = dict(B=2, H=2, P=4, qp=FAKE, kp=FAKE, vp=FAKE, w=FAKE, z=FAKE, A=FAKE, b=None, bl=FAKE,
             g=FAKE, slot=FAKE, S=FAKE, conv=FAKE + (1 << 24), out_dt=0, o=FAKE)
    a.update(kw)
    return lib.kda_decode_layer(a["B"], a["H"], a["P"], a["qp"], a["kp"], a["vp"], a["w"], a["z"],
                                a["A"], a["b"], a["bl"], a["g"], a["slot"], a["S"], a["conv"],
                                0.1, 1e-6, 1e-6, a["out_dt"], a["o"], None)


@pytest.mark.parametrize("bad", [
    dict(out_dt=5), dict(B=0), dict(H=0), dict(P=0), dict(qp=None), dict(kp=MIS), dict(vp=None),
    dict(w=MIS), dict(z=None), dict(A=None), dict(b=MIS), dict(bl=None), dict(g=MIS),
    dict(slot=None), dict(S=None), dict(conv=MIS), dict(o=None),
    dict(conv=FAKE + 1024),  # the convolution pool inside the state pool
])
def test_decode_layer_rejects_bad_arguments(kda, bad):
    assert _decode_layer(kda.library(), **bad) == 1  # KDA_ERR_INVALID_ARGUMENT, before any launch


def test_decode_layer_grid_too_large_unsupported(kda):
    assert _decode_layer(kda.library(), B=1 << 20, H=1 << 12, conv=FAKE + (1 << 40)) == 2


def _decode_tokens(lib, **kw):
    a = dict(in_dt=0, out_dt=0, B=2, H=2, P=4, T=6, cu=FAKE, slot=FAKE, q=FAKE, k=FAKE, v=FAKE,
             la=FAKE, beta=FAKE, S=FAKE, wb=1, Sf=None, o=FAKE)
    a.update(kw)
    return lib.kda_decode_tokens(a["in_dt"], a["out_dt"], a["B"], a["H"], a["P"], a["T"], a["cu"],
                                 a["slot"], a["q"], a["k"], a["v"], a["la"], a["beta"], a["S"],
                                 a["wb"], a["Sf"], 0.1, a["o"], None)


@pytest.mark.parametrize("bad", [
    dict(in_dt=4), dict(out_dt=2), dict(B=0), dict(H=0), dict(P=0), dict(T=-1), dict(wb=2),
    dict(cu=None), dict(cu=FAKE + 2), dict(slot=None), dict(q=None), dict(k=MIS), dict(v=None),
    dict(la=MIS), dict(beta=None), dict(S=None), dict(S=MIS), dict(Sf=MIS), dict(o=None),
    dict(Sf=FAKE + 4 * 2 * 128 * 128 * 4 - 16),  # S_final starts inside the pool's last row
    dict(S=FAKE + (1 << 30), Sf=FAKE + (1 << 30) - 16),  # S_final ends inside the pool
])
def test_decode_tokens_rejects_bad_arguments(kda, bad):
    assert _decode_tokens(kda.library(), **bad) == 1


def test_decode_tokens_too_large_unsupported(kda):
    assert _decode_tokens(kda.library(), B=1 << 20, H=1 << 12, Sf=None) == 2
    assert _decode_tokens(kda.library(), T=1 << 30, H=4) == 2


def test_head_decay_entries_validate(kda):
    lib = kda.library()
    # log_alpha needs only 4-byte alignment here: a 4-byte-aligned pointer passes that check
    # and the call fails on the next one (o missing), never reaching a launch
    rc = lib.kda_prefill_head_decay(0, 0, 1, 4, 2, FAKE, FAKE, FAKE, FAKE + 4, FAKE, None, FAKE,
                                    0.1, None, None, None, 0, 0, None, None, None)
    assert rc == 1
    rc = lib.kda_prefill_head_decay(0, 0, 1, 4, 2, FAKE, FAKE, FAKE, FAKE + 2, FAKE, None, FAKE,
                                    0.1, FAKE, None, None, 0, 0, None, None, None)
    assert rc == 1  # log_alpha misaligned
    rc = lib.kda_prefill_head_decay(0, 0, 1, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                    0.1, FAKE, None, None, 0, 16, FAKE, FAKE, None)
    assert rc == 1  # checkpoint interval not a multiple of 32
    rc = lib.kda_decode_step_head_decay(0, 0, 2, 2, FAKE, FAKE, FAKE, FAKE + 2, FAKE, FAKE, 0.1,
                                        FAKE, None)
    assert rc == 1
    rc = lib.kda_decode_step_head_decay(0, 0, 0, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1,
                                        FAKE, None)
    assert rc == 1


def test_check_prefill_inputs_validates(kda):
    lib = kda.library()
    assert lib.kda_check_prefill_inputs(0, 4, 2, FAKE, 0, FAKE, None) == 1      # no sequences
    assert lib.kda_check_prefill_inputs(1, -1, 2, FAKE, 0, FAKE, None) == 1     # negative T
    assert lib.kda_check_prefill_inputs(1, 4, 2, FAKE, 2, FAKE, None) == 1      # bad flag
    assert lib.kda_check_prefill_inputs(1, 4, 2, FAKE, 0, None, None) == 1      # no offsets
    assert lib.kda_check_prefill_inputs(1, 4, 2, FAKE + 4, 0, FAKE, None) == 1  # misaligned
    assert lib.kda_check_prefill_inputs(1, 4, 2, FAKE + 2, 1, FAKE, None) == 1  # misaligned


def _decode_layer_tokens(lib, **kw):
    a = dict(B=2, H=2, P=4, T=6, cu=FAKE, slot=FAKE, qp=FAKE, kp=FAKE, vp=FAKE, w=FAKE, z=FAKE,
             A=FAKE, b=None, bl=FAKE, g=FAKE, S=FAKE, conv=FAKE + (1 << 24), wb=1, out_dt=0, o=FAKE)
    a.update(kw)
    return lib.kda_decode_layer_tokens(a["B"], a["H"], a["P"], a["T"], a["cu"], a["slot"], a["qp"],
                                       a["kp"], a["vp"], a["w"], a["z"], a["A"], a["b"], a["bl"],
                                       a["g"], a["S"], a["conv"], a["wb"], 0.1, 1e-6, 1e-6,
                                       a["out_dt"], a["o"], None)


@pytest.mark.parametrize("bad", [
    dict(B=0), dict(H=0), dict(P=0), dict(T=-1), dict(wb=3), dict(out_dt=4), dict(cu=None),
    dict(slot=FAKE + 1), dict(qp=None), dict(kp=MIS), dict(vp=None), dict(w=MIS), dict(z=None),
    dict(A=None), dict(b=MIS), dict(bl=FAKE + 1), dict(g=None), dict(S=None), dict(conv=MIS),
    dict(o=None), dict(conv=FAKE + 1024),  # the convolution pool inside the state pool
])
def test_decode_layer_tokens_rejects_bad_arguments(kda, bad):
    assert _decode_layer_tokens(kda.library(), **bad) == 1


def test_decode_layer_tokens_too_large_unsupported(kda):
    assert _decode_layer_tokens(kda.library(), B=1 << 20, H=1 << 12, conv=FAKE + (1 << 40)) == 2


def test_unbounded_decay_entries_validate(kda):
    lib = kda.library()
    a = dict(in_dt=0, out_dt=0, N=1, T=4, H=2, q=FAKE, k=FAKE, v=FAKE, la=FAKE, beta=FAKE,
             S0=None, cu=FAKE, scale=0.1, o=FAKE, Sf=None, ws=None, wsb=0, stream=None)
    for bad in (dict(q=None), dict(la=MIS), dict(H=0), dict(S0=FAKE, Sf=FAKE + 64)):
        c = dict(a, **bad)
        assert lib.kda_prefill_unbounded_decay(c["in_dt"], c["out_dt"], c["N"], c["T"], c["H"],
                                               c["q"], c["k"], c["v"], c["la"], c["beta"], c["S0"],
                                               c["cu"], c["scale"], c["o"], c["Sf"], c["ws"],
                                               c["wsb"], c["stream"]) == 1
    assert lib.kda_frontend_unbounded_decay(1, 4, 2, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE,
                                            FAKE, 1e-6, 0, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert lib.kda_layer_core_unbounded_decay(1, 4, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                              FAKE, FAKE, FAKE, None, 0.1, 1e-6, 1e-6, 0, FAKE,
                                              None, None, 0, None) == 3  # no workspace
