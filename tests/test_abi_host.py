"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point include/gdn.h declares, and rejects bad arguments with a typed
status BEFORE touching CUDA (fake, never-dereferenced pointers are enough to
reach each check)."""
import ctypes

import pytest

from gateddeltanet_linear_attention_gb300 import gdn

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
P = ctypes.c_void_p
A16 = P(0x100000)          # 16-byte aligned fake device address
A16b = P(0x200000)
MIS = P(0x100004)          # misaligned


@pytest.fixture(scope="module")
def lib():
    return gdn.load()


def cfg(**kw):
    base = dict(HK=16, HV=32, dk=128, dv=128, chunk=64, act="bf16", n_slots=4)
    base.update(kw)
    return gdn.make_config(**base)


def test_exports_every_declared_entry_point(lib):
    names = gdn.header_entry_points()
    assert {"gdn_conv1d_prefill", "gdn_conv1d_step", "gdn_chunk_prefill", "gdn_recurrent_decode",
            "gdn_gated_rmsnorm", "gdn_mixer_prefill", "gdn_mixer_decode", "gdn_gate_prep",
            "gdn_workspace_size", "gdn_device_error", "gdn_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(6):
        assert gdn.gdn_status_string(s) != "unknown status"
    assert gdn.gdn_status_string(99) == "unknown status"


@pytest.mark.parametrize("kw,expect", [
    (dict(chunk=32), UNSUPPORTED), (dict(dk=128, dv=64), UNSUPPORTED), (dict(dk=96, dv=96), UNSUPPORTED),
    (dict(HK=16, HV=24), INVALID), (dict(HK=4, HV=32), UNSUPPORTED), (dict(HK=0), INVALID),
    (dict(n_slots=-1), INVALID), (dict(chunk=0), INVALID),
])
def test_config_validation(lib, kw, expect):
    c = cfg(**kw)
    st = lib.gdn_gate_prep(ctypes.byref(c), A16, A16b, 32, 10, A16, A16, A16, A16, None)
    assert st == expect
    assert lib.gdn_workspace_size(ctypes.byref(c), 100, 1) == 0


def test_null_config(lib):
    assert lib.gdn_gate_prep(None, A16, A16, 32, 1, A16, A16, A16, A16, None) == INVALID
    assert lib.gdn_workspace_size(None, 1, 1) == 0


def test_view_checks(lib):
    c = cfg()
    # u / b_logit: ld smaller than HV, misaligned, null
    assert lib.gdn_gate_prep(ctypes.byref(c), A16, A16, 16, 1, A16, A16, A16, A16, None) == INVALID
    odd = P(0x100002)      # not even element-aligned for fp32 / 4-byte loads
    assert lib.gdn_gate_prep(ctypes.byref(c), odd, A16, 32, 1, A16, A16, A16, A16, None) == INVALID
    assert lib.gdn_gate_prep(ctypes.byref(c), None, A16, 32, 1, A16, A16, A16, A16, None) == INVALID
    # T = 0 is a no-op that never touches the GPU
    assert lib.gdn_gate_prep(ctypes.byref(c), None, None, 0, 0, None, None, None, None, None) == OK
    assert lib.gdn_gate_prep(ctypes.byref(c), A16, A16, 32, -1, A16, A16, A16, A16, None) == INVALID


def test_chunk_prefill_validation(lib):
    c = cfg()
    ch = ctypes.byref(c)
    # bad flag bit
    assert lib.gdn_chunk_prefill(ch, A16, A16, 2048, A16, 4096, 0, A16, A16, A16, 1, 64, None, None,
                                 None, A16, 1, 0x10, None, 0, None) == INVALID
    # q/k row stride narrower than HK*dk
    assert lib.gdn_chunk_prefill(ch, A16, A16, 1024, A16, 4096, 0, A16, A16, A16, 1, 64, None, None,
                                 None, A16, 1, 1, None, 0, None) == INVALID
    # misaligned state
    assert lib.gdn_chunk_prefill(ch, A16, A16, 2048, A16, 4096, 0, A16, A16, A16, 1, 64, MIS, None,
                                 None, A16, 1, 1, None, 0, None) == INVALID
    # state without slots
    c0 = cfg(n_slots=0)
    assert lib.gdn_chunk_prefill(ctypes.byref(c0), A16, A16, 2048, A16, 4096, 0, A16, A16, A16, 1, 64,
                                 A16, A16, None, A16, 1, 1, None, 0, None) == INVALID
    # zero sequences with tokens is inconsistent; zero of both is a no-op
    assert lib.gdn_chunk_prefill(ch, A16, A16, 2048, A16, 4096, 0, A16, A16, A16, 0, 5, None, None,
                                 None, A16, 1, 1, None, 0, None) == INVALID
    assert lib.gdn_chunk_prefill(ch, None, None, 0, None, 0, 0, None, None, None, 0, 0, None, None,
                                 None, None, 1, 1, None, 0, None) == OK
    # the tensor-core path (bf16, d = 128, chunk 64) needs its [T ; PT] workspace
    need = lib.gdn_workspace_size(ch, 64, 1)
    assert lib.gdn_chunk_prefill(ch, A16, A16, 2048, A16, 4096, 0, A16, A16, A16, 1, 64, None, None,
                                 None, A16, 1, 1, None, 0, None) == WORKSPACE
    assert lib.gdn_chunk_prefill(ch, A16, A16, 2048, A16, 4096, 0, A16, A16, A16, 1, 64, None, None,
                                 None, A16, 1, 1, MIS, need, None) == WORKSPACE
    # one (chunk, v-head) operand of 32 KB each, plus the chunk map
    assert need >= 32 * 32768
    # the fp32 mode runs the SIMT kernel and needs none
    c32 = cfg(act="fp32")
    assert lib.gdn_chunk_prefill(ctypes.byref(c32), A16, A16, 2048, A16, 4096, 1, A16, A16, A16, 0, 5,
                                 None, None, None, A16, 1, 1, None, 0, None) == INVALID


def _io(T=64, n=1, **kw):
    io = gdn.MixerIO(A16, 8192, A16, 4096, A16, A16, 32, A16, A16, A16, A16, A16, n, T, None, None,
                     None, None, A16, 1)
    for k, v in kw.items():
        setattr(io, k, v)
    return io


def test_mixer_validation_and_workspace(lib):
    c = cfg()
    ch = ctypes.byref(c)
    need = lib.gdn_workspace_size(ch, 64, 1)
    assert need >= 64 * (8192 + 4096 + 64) * 4
    io = _io()
    assert lib.gdn_mixer_prefill(ch, ctypes.byref(io), None, 0, None) == WORKSPACE
    assert lib.gdn_mixer_prefill(ch, ctypes.byref(io), A16, 1024, None) == WORKSPACE
    assert lib.gdn_mixer_prefill(ch, ctypes.byref(io), MIS, need, None) == WORKSPACE
    bad = _io(ld_x=8000)                       # narrower than CH
    assert lib.gdn_mixer_prefill(ch, ctypes.byref(bad), A16, need, None) == INVALID
    bad = _io(ld_z=4100)                       # wide view stride not a multiple of 8
    assert lib.gdn_mixer_prefill(ch, ctypes.byref(bad), A16, need, None) == INVALID
    bad = _io(x=MIS)                           # wide view base not 16-byte aligned
    assert lib.gdn_mixer_prefill(ch, ctypes.byref(bad), A16, need, None) == INVALID
    bad = _io(cu_seqlens=None)
    assert lib.gdn_mixer_prefill(ch, ctypes.byref(bad), A16, need, None) == INVALID
    bad = _io(y_dtype=7)
    assert lib.gdn_mixer_prefill(ch, ctypes.byref(bad), A16, need, None) == INVALID
    assert lib.gdn_mixer_prefill(ch, None, A16, need, None) == INVALID
    # decode: T must equal n_seqs, state in place and required, conv history required
    d = _io(T=4, n=4, state_in=A16, state_out=A16, conv_state=A16b)
    dneed = lib.gdn_workspace_size(ch, 4, 4)
    bad = _io(T=5, n=4, state_in=A16, state_out=A16, conv_state=A16b)
    assert lib.gdn_mixer_decode(ch, ctypes.byref(bad), A16, dneed, None) == INVALID
    bad = _io(T=4, n=4, state_in=A16, state_out=A16b, conv_state=A16b)
    assert lib.gdn_mixer_decode(ch, ctypes.byref(bad), A16, dneed, None) == INVALID
    bad = _io(T=4, n=4, state_in=A16, state_out=A16, conv_state=None)
    assert lib.gdn_mixer_decode(ch, ctypes.byref(bad), A16, dneed, None) == INVALID
    c0 = cfg(n_slots=0)
    assert lib.gdn_mixer_decode(ctypes.byref(c0), ctypes.byref(d), A16, dneed, None) == INVALID
    # decode workspace: one record per (sequence, q/k head), missing / short / misaligned rejected
    assert dneed >= 4 * 16 * (2 * 128 + 2 * 2 * 128) * 4
    assert lib.gdn_mixer_decode(ch, ctypes.byref(d), None, 0, None) == WORKSPACE
    assert lib.gdn_mixer_decode(ch, ctypes.byref(d), A16, 1024, None) == WORKSPACE
    assert lib.gdn_mixer_decode(ch, ctypes.byref(d), MIS, dneed, None) == WORKSPACE


def test_decode_and_norm_validation(lib):
    c = cfg()
    ch = ctypes.byref(c)
    assert lib.gdn_recurrent_decode(ch, A16, A16, 2048, A16, 4096, 0, A16, A16, 4, None, None, A16, 1,
                                    1, None) == INVALID          # no state
    assert lib.gdn_recurrent_decode(ch, A16, A16, 2048, A16, 4096, 0, A16, A16, 4, MIS, None, A16, 1,
                                    1, None) == INVALID          # misaligned state
    assert lib.gdn_gated_rmsnorm(ch, A16, 1, A16, 100, A16, 4, A16, 1, None) == INVALID
    assert lib.gdn_gated_rmsnorm(ch, A16, 3, A16, 4096, A16, 4, A16, 1, None) == INVALID
    assert lib.gdn_conv1d_step(ch, A16, 8192, 2, A16, None, None, A16, 1, None) == INVALID
    assert lib.gdn_conv1d_prefill(ch, A16, 8192, None, 1, 10, A16, None, None, A16, 1, None) == INVALID


def test_state_copy_validation(lib):
    c = cfg()
    ch = ctypes.byref(c)
    # n < 0, negative pool sizes, missing index buffers, misaligned pools
    assert lib.gdn_state_copy(ch, A16, A16, 4, A16b, A16b, 4, A16, A16, -1, None) == INVALID
    assert lib.gdn_state_copy(ch, A16, A16, -1, A16b, A16b, 4, A16, A16, 1, None) == INVALID
    assert lib.gdn_state_copy(ch, A16, A16, 4, A16b, A16b, -2, A16, A16, 1, None) == INVALID
    assert lib.gdn_state_copy(ch, A16, A16, 4, A16b, A16b, 4, None, A16, 1, None) == INVALID
    assert lib.gdn_state_copy(ch, A16, A16, 4, A16b, A16b, 4, A16, None, 1, None) == INVALID
    assert lib.gdn_state_copy(ch, MIS, None, 4, A16b, None, 4, A16, A16, 1, None) == INVALID
    assert lib.gdn_state_copy(ch, A16, None, 4, P(0x200008), None, 4, A16, A16, 1, None) == INVALID
    assert lib.gdn_state_copy(ch, None, MIS, 4, None, A16b, 4, A16, A16, 1, None) == INVALID
    # nothing to do: no pairs, or no destination pool -- never touches the GPU
    assert lib.gdn_state_copy(ch, A16, A16, 4, A16b, A16b, 4, A16, A16, 0, None) == OK
    assert lib.gdn_state_copy(ch, A16, A16, 4, None, None, 4, A16, A16, 3, None) == OK
    # an invalid configuration is refused first
    bad = cfg(dk=96, dv=96)
    assert lib.gdn_state_copy(ctypes.byref(bad), A16, A16, 4, A16b, A16b, 4, A16, A16, 1, None) == UNSUPPORTED


def test_mixer_verify_validation(lib):
    c = cfg()
    ch = ctypes.byref(c)
    k, n = 4, 3
    good = dict(state_in=A16b, state_out=A16b, conv_state=A16)
    need = lib.gdn_workspace_size(ch, n * k, n)
    io = _io(T=n * k, n=n, **good)
    for kk in (0, 9, -1):                                               # 1 <= k <= 8
        assert lib.gdn_mixer_verify(ch, ctypes.byref(io), kk, A16, A16, need, None) == INVALID
    bad = _io(T=n * k + 1, n=n, **good)                                 # T != n * k
    assert lib.gdn_mixer_verify(ch, ctypes.byref(bad), k, A16, A16, need, None) == INVALID
    assert lib.gdn_mixer_verify(ch, ctypes.byref(io), k, None, A16, need, None) == INVALID
    bad = _io(T=n * k, n=n, state_in=A16b, state_out=A16, conv_state=A16)   # two pools
    assert lib.gdn_mixer_verify(ch, ctypes.byref(bad), k, A16, A16, need, None) == INVALID
    bad = _io(T=n * k, n=n, state_in=A16b, state_out=A16b, conv_state=None)  # no histories
    assert lib.gdn_mixer_verify(ch, ctypes.byref(bad), k, A16, A16, need, None) == INVALID
    bad = _io(T=n * k, n=n, ld_x=8000, **good)                          # narrower than CH
    assert lib.gdn_mixer_verify(ch, ctypes.byref(bad), k, A16, A16, need, None) == INVALID
    # the workspace is not used: none, a small one or a misaligned one is no workspace error
    # (without a GPU the call then stops at the CUDA runtime)
    for ws, nb in ((None, 0), (A16, 16), (MIS, need)):
        assert lib.gdn_mixer_verify(ch, ctypes.byref(io), k, A16, ws, nb, None) not in (OK, WORKSPACE,
                                                                                      INVALID)
    empty = _io(T=0, n=0, **good)
    assert lib.gdn_mixer_verify(ch, ctypes.byref(empty), k, None, None, 0, None) == OK


def test_q8_validation(lib):
    c = cfg()
    ch = ctypes.byref(c)
    assert lib.gdn_state_to_q8(ch, None, A16, A16b, None, 0, None) == INVALID
    assert lib.gdn_state_to_q8(ch, A16, MIS, A16b, None, 0, None) == INVALID
    assert lib.gdn_state_from_q8(ch, A16, None, A16b, None) == INVALID
    assert lib.gdn_state_from_q8(ch, A16, A16b, MIS, None) == INVALID
    c0 = cfg(n_slots=0)                                                 # an empty pool: nothing to do
    assert lib.gdn_state_to_q8(ctypes.byref(c0), A16, A16, A16b, None, 0, None) == OK
    need = lib.gdn_workspace_size(ch, 4, 4)
    q8io = _io(T=4, n=4, conv_state=A16b)                               # no fp32 state pointers
    bad = _io(T=4, n=4, state_in=A16, state_out=A16, conv_state=A16b)   # fp32 state given
    assert lib.gdn_mixer_decode_q8(ch, ctypes.byref(bad), A16, A16b, None, 0, A16, need, None) == INVALID
    bad = _io(T=4, n=4)                                                 # no conv history
    assert lib.gdn_mixer_decode_q8(ch, ctypes.byref(bad), A16, A16b, None, 0, A16, need, None) == INVALID
    bad = _io(T=5, n=4, conv_state=A16b)                                # T != n_seqs
    assert lib.gdn_mixer_decode_q8(ch, ctypes.byref(bad), A16, A16b, None, 0, A16, need, None) == INVALID
    assert lib.gdn_mixer_decode_q8(ch, ctypes.byref(q8io), None, A16b, None, 0, A16, need, None) == INVALID
    assert lib.gdn_mixer_decode_q8(ch, ctypes.byref(q8io), A16, MIS, None, 0, A16, need, None) == INVALID
    assert lib.gdn_mixer_decode_q8(ch, ctypes.byref(q8io), A16, A16b, MIS, 0, A16, need, None) == INVALID
    assert lib.gdn_state_to_q8(ch, A16, A16, A16b, MIS, 0, None) == INVALID   # misaligned residual
    assert lib.gdn_mixer_decode_q8(ch, ctypes.byref(q8io), A16, A16b, None, 0, A16, 64, None) == WORKSPACE
    assert lib.gdn_mixer_decode_q8(ctypes.byref(c0), ctypes.byref(q8io), A16, A16b, None, 0, A16, need, None) == INVALID


def test_backward_validation(lib):
    """gdn_chunk_states / gdn_chunk_backward: every pointer check, the retained p and w
    (token_pw) included, and the workspace size, before any CUDA call."""
    c = cfg()
    ch = ctypes.byref(c)
    T, n = 64, 1
    need = lib.gdn_backward_workspace_size(ch, T, n)
    assert need > 0
    assert lib.gdn_backward_workspace_size(ch, -1, n) == 0

    def states(bnd=A16, pw=None, ws_bytes=need, T=T, k=A16, state_in=None):
        return lib.gdn_chunk_states(ch, k, 2048, A16b, 4096, 0, A16, A16b, A16, n, T, state_in, None,
                                    bnd, pw, A16, ws_bytes, None)

    assert states(pw=MIS) == INVALID                   # misaligned p/w rows
    assert states(bnd=None) == INVALID
    assert states(bnd=MIS) == INVALID
    assert states(k=MIS) == INVALID
    assert states(state_in=MIS) == INVALID
    assert states(ws_bytes=64) == WORKSPACE
    assert states(pw=A16b, ws_bytes=64) == WORKSPACE   # an aligned buffer passes to the next check
    assert states(T=0, bnd=None) == OK                 # nothing to do

    def backward(pw=None, d_o=A16, dq=A16, ld_dqk=2048, ws_bytes=need, T=T, d_state_in=None):
        return lib.gdn_chunk_backward(ch, A16, A16, 2048, A16b, 4096, 0, A16, A16b, A16, n, T, None,
                                      A16b, pw, d_o, None, dq, A16, ld_dqk, A16b, A16, A16b, d_state_in,
                                      A16, ws_bytes, None)

    assert backward(pw=MIS) == INVALID
    assert backward(d_o=MIS) == INVALID
    assert backward(dq=None) == INVALID
    assert backward(ld_dqk=1024) == INVALID            # narrower than HK * dk
    assert backward(d_state_in=MIS) == INVALID
    assert backward(ws_bytes=need - 257) == WORKSPACE   # (the size includes 256 bytes of slack)
    assert backward(pw=A16b, ws_bytes=64) == WORKSPACE
    assert backward(T=0) == OK
