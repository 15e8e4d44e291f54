"""ctypes binding of the C ABI in include/gdn.h.

Argument marshalling only: each function takes torch tensors that already
live on the GPU (or None), passes their device pointers, row strides and the
current stream to the entry point of the same name, and raises GDNError on a
non-OK status.  Every step of the mixer runs in the library's CUDA kernels;
if the compiled library is missing, loading it raises -- there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build_lib

GDN_BF16, GDN_FP32 = 0, 1
GDN_FLAG_L2NORM_QK = 1
DEVERR_CU_SEQLENS, DEVERR_SLOT, DEVERR_TIMEOUT = 1, 2, 4
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED",
          3: "GDN_ERR_WORKSPACE", 4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE"}


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, STATUS.get(status, str(status))))


class Config(ctypes.Structure):
    _fields_ = [("hk", ctypes.c_int32), ("hv", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("chunk", ctypes.c_int32), ("act", ctypes.c_int32),
                ("n_slots", ctypes.c_int32), ("q_scale", ctypes.c_float),
                ("l2_eps", ctypes.c_float), ("norm_eps", ctypes.c_float)]


class MixerIO(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("ld_x", ctypes.c_int64),
                ("z", ctypes.c_void_p), ("ld_z", ctypes.c_int64),
                ("u", ctypes.c_void_p), ("b_logit", ctypes.c_void_p), ("ld_ub", ctypes.c_int64),
                ("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("norm_w", ctypes.c_void_p),
                ("cu_seqlens", ctypes.c_void_p), ("n_seqs", ctypes.c_int32), ("T", ctypes.c_int64),
                ("state_idx", ctypes.c_void_p), ("state_in", ctypes.c_void_p),
                ("state_out", ctypes.c_void_p), ("conv_state", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("y_dtype", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()
LIB_PATH = build_lib.LIB


def header_entry_points():
    """Names of the functions declared in include/gdn.h."""
    txt = open(os.path.join(build_lib.INCLUDE, "gdn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", txt)))


def load(path: str | None = None):
    """Load the compiled library (building it first if sources are newer)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if path is None and build_lib.needs_build():
            build_lib.build()
        if not os.path.exists(p):
            raise RuntimeError("GDN CUDA library not found at %s; run build()" % p)
        lib = ctypes.CDLL(p)
        V, P, I32, I64, U32, SZ = (ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                   ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t)
        CP = ctypes.POINTER(Config)
        sig = {
            "gdn_workspace_size": ([CP, I64, I32], SZ),
            "gdn_gate_prep": ([CP, P, P, I64, I64, P, P, P, P, V], I32),
            "gdn_conv1d_prefill": ([CP, P, I64, P, I32, I64, P, P, P, P, I32, V], I32),
            "gdn_conv1d_step": ([CP, P, I64, I32, P, P, P, P, I32, V], I32),
            "gdn_chunk_prefill": ([CP, P, P, I64, P, I64, I32, P, P, P, I32, I64, P, P, P, P, I32,
                                   U32, P, SZ, V], I32),
            "gdn_recurrent_decode": ([CP, P, P, I64, P, I64, I32, P, P, I32, P, P, P, I32, U32, V],
                                     I32),
            "gdn_gated_rmsnorm": ([CP, P, I32, P, I64, P, I64, P, I32, V], I32),
            "gdn_mixer_prefill": ([CP, ctypes.POINTER(MixerIO), P, SZ, V], I32),
            "gdn_mixer_decode": ([CP, ctypes.POINTER(MixerIO), P, SZ, V], I32),
            "gdn_mixer_prefill_static": ([CP, ctypes.POINTER(MixerIO), V], I32),
            "gdn_state_copy": ([CP, P, P, I32, P, P, I32, P, P, I32, V], I32),
            "gdn_mixer_verify": ([CP, ctypes.POINTER(MixerIO), I32, P, P, SZ, V], I32),
            "gdn_backward_workspace_size": ([CP, I64, I32], SZ),
            "gdn_state_to_q8": ([CP, P, P, P, P, U32, V], I32),
            "gdn_state_from_q8": ([CP, P, P, P, V], I32),
            "gdn_mixer_decode_q8": ([CP, ctypes.POINTER(MixerIO), P, P, P, U32, P, SZ, V], I32),
            "gdn_chunk_states": ([CP, P, I64, P, I64, I32, P, P, P, I32, I64, P, P, P, P, P, SZ, V], I32),
            "gdn_chunk_backward": ([CP, P, P, I64, P, I64, I32, P, P, P, I32, I64, P, P, P, P, P, P, P,
                                    I64, P, P, P, P, P, SZ, V], I32),
            "gdn_device_error": ([V, ctypes.POINTER(U32)], I32),
            "gdn_debug_set_wait": ([ctypes.c_uint64, U32], I32),
            "gdn_status_string": ([I32], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


# ---------------------------------------------------------------- helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _ld(t):
    if t is None:
        return 0
    return t.stride(0) if t.dim() > 1 else t.shape[0]


def _dt(t):
    import torch
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_FP32
    raise TypeError("unsupported dtype %s" % t.dtype)


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


def _check(st, where):
    if st != 0:
        raise GDNError(st, where)


def make_config(HK, HV, dk, dv, chunk=64, act="bf16", n_slots=0, q_scale=1.0, l2_eps=1e-6,
                norm_eps=1e-6) -> Config:
    return Config(HK, HV, dk, dv, chunk, GDN_BF16 if act == "bf16" else GDN_FP32, n_slots,
                  q_scale, l2_eps, norm_eps)


# ------------------------------------------------------------ entry points

def gdn_workspace_size(cfg, max_tokens, max_seqs):
    return load().gdn_workspace_size(ctypes.byref(cfg), max_tokens, max_seqs)


def gdn_gate_prep(cfg, u, b_logit, A_log, dt_bias, g, beta, stream=None):
    T = u.shape[0]
    _check(load().gdn_gate_prep(ctypes.byref(cfg), _ptr(u), _ptr(b_logit), _ld(u), T,
                                _ptr(A_log), _ptr(dt_bias), _ptr(g), _ptr(beta),
                                _stream(stream)), "gdn_gate_prep")


def gdn_conv1d_prefill(cfg, x, cu_seqlens, w, conv_state, state_idx, out, stream=None):
    _check(load().gdn_conv1d_prefill(ctypes.byref(cfg), _ptr(x), _ld(x), _ptr(cu_seqlens),
                                     cu_seqlens.shape[0] - 1, x.shape[0], _ptr(w),
                                     _ptr(conv_state), _ptr(state_idx), _ptr(out), _dt(out),
                                     _stream(stream)), "gdn_conv1d_prefill")


def gdn_conv1d_step(cfg, x, w, conv_state, state_idx, out, stream=None):
    _check(load().gdn_conv1d_step(ctypes.byref(cfg), _ptr(x), _ld(x), x.shape[0], _ptr(w),
                                  _ptr(conv_state), _ptr(state_idx), _ptr(out), _dt(out),
                                  _stream(stream)), "gdn_conv1d_step")


def gdn_chunk_prefill(cfg, q, k, v, g, beta, cu_seqlens, state_in, state_out, state_idx, o,
                      flags=GDN_FLAG_L2NORM_QK, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_chunk_prefill(ctypes.byref(cfg), _ptr(q), _ptr(k), _ld(q), _ptr(v), _ld(v),
                                    _dt(q), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                    cu_seqlens.shape[0] - 1, q.shape[0], _ptr(state_in),
                                    _ptr(state_out), _ptr(state_idx), _ptr(o), _dt(o), flags,
                                    _ptr(workspace), ws_bytes, _stream(stream)),
           "gdn_chunk_prefill")


def gdn_recurrent_decode(cfg, q, k, v, g, beta, state, state_idx, o, flags=GDN_FLAG_L2NORM_QK,
                         stream=None):
    _check(load().gdn_recurrent_decode(ctypes.byref(cfg), _ptr(q), _ptr(k), _ld(q), _ptr(v),
                                       _ld(v), _dt(q), _ptr(g), _ptr(beta), q.shape[0],
                                       _ptr(state), _ptr(state_idx), _ptr(o), _dt(o), flags,
                                       _stream(stream)), "gdn_recurrent_decode")


def gdn_gated_rmsnorm(cfg, o, z, w, y, stream=None):
    _check(load().gdn_gated_rmsnorm(ctypes.byref(cfg), _ptr(o), _dt(o), _ptr(z), _ld(z), _ptr(w),
                                    o.shape[0], _ptr(y), _dt(y), _stream(stream)),
           "gdn_gated_rmsnorm")


def _mixer_io(x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, cu_seqlens, state_in, state_out,
              conv_state, state_idx, y, n_seqs):
    return MixerIO(_ptr(x), _ld(x), _ptr(z), _ld(z), _ptr(u), _ptr(b_logit), _ld(u),
                   _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w), _ptr(cu_seqlens),
                   n_seqs, x.shape[0], _ptr(state_idx), _ptr(state_in), _ptr(state_out),
                   _ptr(conv_state), _ptr(y), _dt(y))


def gdn_mixer_prefill(cfg, x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, cu_seqlens, y,
                      state_in=None, state_out=None, conv_state=None, state_idx=None,
                      workspace=None, stream=None):
    io = _mixer_io(x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, cu_seqlens, state_in,
                   state_out, conv_state, state_idx, y, cu_seqlens.shape[0] - 1)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_mixer_prefill(ctypes.byref(cfg), ctypes.byref(io), _ptr(workspace),
                                    ws_bytes, _stream(stream)), "gdn_mixer_prefill")


def gdn_mixer_prefill_static(cfg, x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, cu_seqlens, y,
                             state_in=None, state_out=None, conv_state=None, state_idx=None,
                             stream=None):
    """gdn_mixer_prefill without a workspace: the library's fixed scratch is used."""
    io = _mixer_io(x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, cu_seqlens, state_in,
                   state_out, conv_state, state_idx, y, cu_seqlens.shape[0] - 1)
    _check(load().gdn_mixer_prefill_static(ctypes.byref(cfg), ctypes.byref(io), _stream(stream)),
           "gdn_mixer_prefill_static")


def gdn_mixer_decode(cfg, x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, y, state,
                     conv_state, workspace, state_idx=None, stream=None):
    """workspace: a device byte tensor of gdn_workspace_size(cfg, n, n) bytes or more."""
    io = _mixer_io(x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, None, state, state,
                   conv_state, state_idx, y, x.shape[0])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_mixer_decode(ctypes.byref(cfg), ctypes.byref(io), _ptr(workspace), ws_bytes,
                                   _stream(stream)), "gdn_mixer_decode")


def gdn_state_to_q8(cfg, state, codes, scales, frame, stream=None, residual=None):
    """residual (bf16 [slots][HV][dk][dv], optional): written for an error-feedback pool."""
    _check(load().gdn_state_to_q8(ctypes.byref(cfg), _ptr(state), _ptr(codes), _ptr(scales),
                                  _ptr(residual), frame, _stream(stream)), "gdn_state_to_q8")


def gdn_state_from_q8(cfg, codes, scales, state, stream=None):
    _check(load().gdn_state_from_q8(ctypes.byref(cfg), _ptr(codes), _ptr(scales), _ptr(state),
                                    _stream(stream)), "gdn_state_from_q8")


def gdn_mixer_decode_q8(cfg, x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, y, codes, scales,
                        conv_state, frame, workspace, state_idx=None, stream=None, residual=None):
    """gdn_mixer_decode on a Q8 state pool (codes int8 [slots][HV][dk][dv], scales fp32
    [slots][HV][dk]); `frame` keys the rounding dither and should change every step.  A bf16
    `residual` pool of the codes' shape turns error feedback on."""
    io = _mixer_io(x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, None, None, None,
                   conv_state, state_idx, y, x.shape[0])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_mixer_decode_q8(ctypes.byref(cfg), ctypes.byref(io), _ptr(codes), _ptr(scales),
                                      _ptr(residual), frame, _ptr(workspace), ws_bytes, _stream(stream)),
           "gdn_mixer_decode_q8")


def gdn_backward_workspace_size(cfg, max_tokens, max_seqs) -> int:
    return load().gdn_backward_workspace_size(ctypes.byref(cfg), max_tokens, max_seqs)


def chunk_count(seqlens, chunk):
    """Boundary states of a batch: sum over sequences of ceil(len / chunk)."""
    return sum((int(L) + chunk - 1) // chunk for L in seqlens)


def gdn_chunk_states(cfg, k, v, g, beta, cu_seqlens, boundary_states, workspace, state_in=None,
                     state_idx=None, token_pw=None, stream=None):
    """token_pw: optional fp32 [T, HV, 2, dv] that receives every token's p and w, for
    gdn_chunk_backward's token_pw."""
    T = k.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_chunk_states(ctypes.byref(cfg), _ptr(k), _ld(k), _ptr(v), _ld(v), _dt(k),
                                   _ptr(g), _ptr(beta), _ptr(cu_seqlens), cu_seqlens.shape[0] - 1, T,
                                   _ptr(state_in), _ptr(state_idx), _ptr(boundary_states),
                                   _ptr(token_pw), _ptr(workspace), ws_bytes, _stream(stream)),
           "gdn_chunk_states")


def gdn_chunk_backward(cfg, q, k, v, g, beta, cu_seqlens, boundary_states, d_o, dq, dk, dv, dg,
                       dbeta, workspace, d_state_out=None, d_state_in=None, state_idx=None,
                       token_pw=None, stream=None):
    """token_pw: None, or the buffer gdn_chunk_states filled for the same batch."""
    T = q.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_chunk_backward(ctypes.byref(cfg), _ptr(q), _ptr(k), _ld(q), _ptr(v), _ld(v),
                                     _dt(q), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                     cu_seqlens.shape[0] - 1, T, _ptr(state_idx),
                                     _ptr(boundary_states), _ptr(token_pw), _ptr(d_o),
                                     _ptr(d_state_out), _ptr(dq),
                                     _ptr(dk), _ld(dq), _ptr(dv), _ptr(dg), _ptr(dbeta),
                                     _ptr(d_state_in), _ptr(workspace), ws_bytes, _stream(stream)),
           "gdn_chunk_backward")


def gdn_mixer_verify(cfg, x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, y, state,
                     conv_state, ckpt_idx, k, workspace, state_idx=None, stream=None):
    """k tokens per sequence (rows n*k .. n*k+k-1 of x, z, u, b_logit, y); the state and conv
    history after token j go to slot ckpt_idx[n] + j of the same pools."""
    n = x.shape[0] // k
    if n * k != x.shape[0]:
        raise ValueError("x holds %d rows, not a multiple of k=%d" % (x.shape[0], k))
    io = _mixer_io(x, z, u, b_logit, conv_w, A_log, dt_bias, norm_w, None, state, state,
                   conv_state, state_idx, y, x.shape[0])
    io.n_seqs = n
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().gdn_mixer_verify(ctypes.byref(cfg), ctypes.byref(io), k, _ptr(ckpt_idx),
                                   _ptr(workspace), ws_bytes, _stream(stream)), "gdn_mixer_verify")


def gdn_state_copy(cfg, src_state, src_conv, dst_state, dst_conv, src_idx, dst_idx, stream=None):
    """Snapshot / restore / reset: slot src_idx[i] -> slot dst_idx[i] (src < 0: reset to zeros,
    dst < 0: nothing).  The slot counts come from the pools' first dimension; src and dst may be
    the same tensors."""
    import torch
    CH = 2 * cfg.hk * cfg.dk + cfg.hv * cfg.dv
    act = torch.bfloat16 if cfg.act == GDN_BF16 else torch.float32
    for t in (src_state, dst_state):
        if t is not None and (tuple(t.shape[1:]) != (cfg.hv, cfg.dk, cfg.dv) or t.dtype != torch.float32
                              or not t.is_contiguous()):
            raise ValueError("state pools are contiguous fp32 [slots][HV][dk][dv]")
    for t in (src_conv, dst_conv):
        if t is not None and (tuple(t.shape[1:]) != (CH, 3) or t.dtype != act or not t.is_contiguous()):
            raise ValueError("history pools are contiguous [slots][CH][3] in the activation dtype")
    for t in (src_idx, dst_idx):
        if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
            raise ValueError("slot indices are contiguous int32")
    if src_idx is not None and dst_idx is not None and src_idx.numel() != dst_idx.numel():
        raise ValueError("src_idx and dst_idx differ in length")

    def slots(*ts):
        return min([t.shape[0] for t in ts if t is not None] or [0])
    n = 0 if dst_idx is None else dst_idx.numel()
    _check(load().gdn_state_copy(ctypes.byref(cfg), _ptr(src_state), _ptr(src_conv),
                                 slots(src_state, src_conv), _ptr(dst_state), _ptr(dst_conv),
                                 slots(dst_state, dst_conv), _ptr(src_idx), _ptr(dst_idx), n,
                                 _stream(stream)), "gdn_state_copy")


def gdn_device_error(stream=None) -> int:
    code = ctypes.c_uint32(0)
    st = load().gdn_device_error(_stream(stream), ctypes.byref(code))
    if st not in (0, 5):
        raise GDNError(st, "gdn_device_error")
    return code.value


def gdn_debug_set_wait(wait_ns=2_000_000_000, lose=0):
    """Limit of every bounded device wait (ns) and the test hook that drops one operand copy
    (bit 0: decode, bit 1: state chain); gdn_debug_set_wait() restores the defaults."""
    _check(load().gdn_debug_set_wait(wait_ns, lose), "gdn_debug_set_wait")


def gdn_status_string(status: int) -> str:
    return load().gdn_status_string(status).decode()
