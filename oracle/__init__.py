"""fp64 CPU oracle for the GatedDeltaNet mixer (ctypes binding of gdn_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library; the only thing both sides share is the seeded
input generator, which holds none of the method's arithmetic.

The C file computes, in double precision and in the order the definition
states: the width-4 causal conv1d with history and SiLU, the per-head L2 norm
of q and k, the gates, the gated delta rule token by token (plus a separate
chunked restatement used only to check chunk algebra), and the gated RMSNorm.
Citations to the pages are in the C file's header.

Arrays are numpy float64 (bf16 or fp32 inputs are widened exactly).  Layouts
are the library's: state ``[slots, HV, dk, dv]`` holding S transposed, conv
history ``[slots, CH, 3]`` oldest first, activations ``[T, ...]`` packed.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c with gcc into oracle/_build/libgdn_oracle.so."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_conv1d_silu.argtypes = [I, P, P, I, P, P, P, P]
            lib.oracle_gates.argtypes = [I, I, P, P, P, P, P, P]
            lib.oracle_l2norm_qk.argtypes = [I, I, I, I, D, D, P]
            lib.oracle_delta_rule.argtypes = [I, P, P, I, I, I, I, P, P, P, P, P, I, I]
            lib.oracle_gated_rmsnorm.argtypes = [I, I, I, P, P, P, D, P]
            lib.oracle_mixer.argtypes = [I, P, P, I, I, I, I, P, P, P, P, P, P, P, P, P, D, D, D,
                                         P, P, P, P, I, I]
            lib.oracle_mixer.restype = I
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor (CPU): widen exactly
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def conv1d_silu(x, cu_seqlens, w, conv_state=None, slot_idx=None):
    """Causal conv1d (width 4) + SiLU.  Returns (out [T, CH], new conv_state or None)."""
    lib = _load()
    x = _f64(x); w = _f64(w); cu = _i32(cu_seqlens); si = _i32(slot_idx)
    cs = None if conv_state is None else _f64(conv_state).copy()
    T, CH = x.shape
    out = np.zeros((T, CH))
    lib.oracle_conv1d_silu(CH, _p(x), _p(cu), len(cu) - 1, _p(w), _p(cs), _p(si), _p(out))
    return out, cs


def gates(u, b_logit, A_log, dt_bias):
    """Returns (g, beta), both [T, HV]."""
    lib = _load()
    u = _f64(u); b = _f64(b_logit); A = _f64(A_log); dt = _f64(dt_bias)
    T, HV = u.shape
    g = np.zeros((T, HV)); beta = np.zeros((T, HV))
    lib.oracle_gates(T, HV, _p(u), _p(b), _p(A), _p(dt), _p(g), _p(beta))
    return g, beta


def l2norm_qk(xa, HK, dk, eps=1e-6, q_scale=1.0):
    """L2-normalise the q and k heads of [T, CH] activations (returns a copy)."""
    lib = _load()
    xa = _f64(xa).copy()
    T, CH = xa.shape
    lib.oracle_l2norm_qk(T, CH, HK, dk, eps, q_scale, _p(xa))
    return xa


def delta_rule(xa, g, beta, cu_seqlens, HK, HV, dk, dv, state=None, slot_idx=None, chunk=0,
               n_threads=None):
    """Gated delta rule over packed, already normalised activations.

    Returns (o [T, HV*dv], final state or None).  chunk=0 is the token-by-token
    definition; chunk>0 the chunked restatement (for checking chunk algebra)."""
    lib = _load()
    xa = _f64(xa); g = _f64(g); beta = _f64(beta); cu = _i32(cu_seqlens); si = _i32(slot_idx)
    st = None if state is None else _f64(state).copy()
    T = xa.shape[0]
    o = np.zeros((T, HV * dv))
    lib.oracle_delta_rule(len(cu) - 1, _p(cu), _p(si), HK, HV, dk, dv, _p(xa), _p(g), _p(beta),
                          _p(st), _p(o), int(chunk), int(n_threads or default_threads()))
    return o, st


def gated_rmsnorm(o, z, w, HV, dv, eps=1e-6):
    lib = _load()
    o = _f64(o); z = _f64(z); w = _f64(w)
    T = o.shape[0]
    y = np.zeros((T, HV * dv))
    lib.oracle_gated_rmsnorm(T, HV, dv, _p(o), _p(z), _p(w), eps, _p(y))
    return y


def mixer(x, conv_w, u, b_logit, A_log, dt_bias, z, norm_w, cu_seqlens, HK, HV, dk, dv,
          state=None, conv_state=None, slot_idx=None, q_scale=1.0, l2_eps=1e-6, norm_eps=1e-6,
          dumps=False, chunk=0, n_threads=None):
    """The whole mixer over a packed batch.

    Returns a dict with y [T, HV*dv], state (final, or None), conv_state (new,
    or None) and, with dumps=True, xa (post-SiLU, q/k normalised) and o."""
    lib = _load()
    x = _f64(x); T, CH = x.shape
    assert CH == 2 * HK * dk + HV * dv
    cw = _f64(conv_w); u = _f64(u); b = _f64(b_logit); A = _f64(A_log); dt = _f64(dt_bias)
    z = _f64(z); nw = _f64(norm_w); cu = _i32(cu_seqlens); si = _i32(slot_idx)
    st = None if state is None else _f64(state).copy()
    cs = None if conv_state is None else _f64(conv_state).copy()
    y = np.zeros((T, HV * dv))
    xa = np.zeros((T, CH)) if dumps else None
    o = np.zeros((T, HV * dv)) if dumps else None
    rc = lib.oracle_mixer(len(cu) - 1, _p(cu), _p(si), HK, HV, dk, dv, _p(x), _p(cw), _p(cs),
                          _p(u), _p(b), _p(A), _p(dt), _p(z), _p(nw), q_scale, l2_eps, norm_eps,
                          _p(st), _p(y), _p(xa), _p(o), int(chunk),
                          int(n_threads or default_threads()))
    if rc != 0:
        raise MemoryError("oracle_mixer: allocation failed")
    out = {"y": y, "state": st, "conv_state": cs}
    if dumps:
        out["xa"] = xa
        out["o"] = o
    return out


def head_channels(HK, HV, dk, dv, kheads):
    """For a subset of q/k heads (with their HV/HK v-heads each): the channel indices into the raw
    projection [q (HK*dk) | k (HK*dk) | v (HV*dv)], the v-head indices, and the columns of
    [T, HV*dv] outputs they own.  Heads never interact, so running the mixer on such a subset
    gives exactly the subset's share of the full result."""
    G = HV // HK
    vheads = [kh * G + j for kh in kheads for j in range(G)]
    q = [kh * dk + i for kh in kheads for i in range(dk)]
    k = [HK * dk + kh * dk + i for kh in kheads for i in range(dk)]
    v = [2 * HK * dk + h * dv + j for h in vheads for j in range(dv)]
    cols = [h * dv + j for h in vheads for j in range(dv)]
    return np.array(q + k + v), np.array(vheads), np.array(cols)


def mixer_heads(x, conv_w, u, b_logit, A_log, dt_bias, z, norm_w, cu_seqlens, HK, HV, dk, dv,
                kheads, state=None, conv_state=None, **kw):
    """mixer() on the q/k heads `kheads` only: the inputs are the full-width tensors, sliced
    here; state [slots, HV, dk, dv] and conv_state [slots, CH, 3] likewise (absent: zeros)."""
    chs, vh, cols = head_channels(HK, HV, dk, dv, list(kheads))
    n_seqs = len(np.asarray(cu_seqlens)) - 1
    st = np.zeros((n_seqs, len(vh), dk, dv)) if state is None else _f64(state)[:, vh]
    cs = np.zeros((n_seqs, len(chs), 3)) if conv_state is None else _f64(conv_state)[:, chs]
    return mixer(_f64(x)[:, chs], _f64(conv_w)[chs], _f64(u)[:, vh], _f64(b_logit)[:, vh],
                 _f64(A_log)[vh], _f64(dt_bias)[vh], _f64(z)[:, cols], norm_w, cu_seqlens,
                 len(list(kheads)), len(vh), dk, dv, state=st, conv_state=cs, **kw)


def state_copy(src_state, src_conv, dst_state, dst_conv, src_idx, dst_idx):
    """Slot maintenance (hyperflare core-design, "State operations": snapshot, restore and
    reset as indirect copies over slot indices).  For each pair (s, t): t < 0 does nothing;
    s >= 0 copies source slot s to destination slot t exactly; s < 0 resets slot t to zeros.
    A pair whose t is past the destination pool, or whose s is past a given source pool, is
    skipped and flagged.  The pairs are applied in order, each reading the sources as they were
    before the call (the library's contract keeps sources and destinations apart, where order
    cannot matter).  Works on any array dtype (bit-exact: plain element copies).

    Returns (new dst_state or None, new dst_conv or None, slot_error)."""
    out_s = None if dst_state is None else np.array(dst_state, copy=True)
    out_c = None if dst_conv is None else np.array(dst_conv, copy=True)
    srcs = [a for a in (src_state, src_conv) if a is not None]
    dsts = [a for a in (out_s, out_c) if a is not None]
    n_src = min((a.shape[0] for a in srcs), default=0)
    n_dst = min((a.shape[0] for a in dsts), default=0)
    src_s0 = None if src_state is None else np.array(src_state, copy=True)
    src_c0 = None if src_conv is None else np.array(src_conv, copy=True)
    err = False
    for s, t in zip(np.asarray(src_idx).tolist(), np.asarray(dst_idx).tolist()):
        if t < 0:
            continue
        if t >= n_dst or (s >= n_src and srcs):
            err = True
            continue
        for src, dst in ((src_s0, out_s), (src_c0, out_c)):
            if dst is None:
                continue
            if s >= 0 and src is not None:
                dst[t] = src[s]
            else:
                dst[t] = 0
    return out_s, out_c, err


def mixer_verify(x, conv_w, u, b_logit, A_log, dt_bias, z, norm_w, k, HK, HV, dk, dv, state,
                 conv_state, src_idx=None, q_scale=1.0, l2_eps=1e-6, norm_eps=1e-6, n_threads=None):
    """Multi-token verification (hyperflare core-design, speculative target state: a round
    writes one recurrent checkpoint column per verification input).  Sequence n holds rows
    n*k .. n*k+k-1; it starts from slot src_idx[n] (default n) of state / conv_state, and the
    checkpoint column j is the state and conv history after its first j+1 tokens.

    Computed as the plain mixer over the k prefixes of each sequence (lengths 1..k, each from
    its own copy of the source slot).  Returns y [n*k, HV*dv], states [n, k, HV, dk, dv] and
    convs [n, k, CH, 3]."""
    x = _f64(x); T, CH = x.shape
    n = T // k
    assert n * k == T
    st0 = _f64(state); cs0 = _f64(conv_state)
    src = list(range(n)) if src_idx is None else [int(s) for s in np.asarray(src_idx)]
    y = np.zeros((T, HV * dv))
    states = np.zeros((n, k, HV, dk, dv))
    convs = np.zeros((n, k, CH, 3))
    for i in range(n):
        rows = np.concatenate([np.arange(i * k, i * k + j + 1) for j in range(k)])
        cu = np.concatenate([[0], np.cumsum(np.arange(1, k + 1))]).astype(np.int32)
        out = mixer(x[rows], conv_w, _f64(u)[rows], _f64(b_logit)[rows], A_log, dt_bias,
                    _f64(z)[rows], norm_w, cu, HK, HV, dk, dv,
                    state=np.repeat(st0[src[i]][None], k, axis=0),
                    conv_state=np.repeat(cs0[src[i]][None], k, axis=0),
                    q_scale=q_scale, l2_eps=l2_eps, norm_eps=norm_eps, n_threads=n_threads)
        for j in range(k):
            y[i * k + j] = out["y"][cu[j + 1] - 1]
        states[i] = out["state"]
        convs[i] = out["conv_state"]
    return y, states, convs


def delta_rule_backward(xa, g, beta, cu_seqlens, HK, HV, dk, dv, d_o, state=None, slot_idx=None,
                        d_state=None):
    """Reverse-mode gradient of the gated delta rule (the token-by-token definition of
    `delta_rule`), per sequence and v-head, in numpy fp64 (hyperflare core-design, training
    plan: a backward per region, the GDN core one among them, from retained chunk-boundary
    states).  With S the dv x dk state (the buffers hold M = S^T) and per token
    p = S k, S' = a S + beta (v - a p) k^T, o = S' q, a = exp(g), the loss is
    sum(d_o * o) + sum(d_state * M_final).

    Returns (dxa [T, CH] = (dq | dk | dv) in the layout of xa, with dq and dk summed over the
    v-heads of each q/k head; dg [T, HV]; dbeta [T, HV]; d_state_in [slots, HV, dk, dv] or None).
    The state before every token is kept, so this is for small cases only."""
    xa = _f64(xa); g = _f64(g); beta = _f64(beta); d_o = _f64(d_o)
    cu = [int(c) for c in np.asarray(cu_seqlens)]
    T = xa.shape[0]
    G = HV // HK
    n_seqs = len(cu) - 1
    dxa = np.zeros_like(xa)
    dg = np.zeros((T, HV)); db = np.zeros((T, HV))
    d_state_in = None if state is None else np.zeros_like(_f64(state))
    for n in range(n_seqs):
        slot = n if slot_idx is None else int(np.asarray(slot_idx)[n])
        if slot < 0:          # a padding lane: its outputs are zero, so are its gradients
            continue
        for h in range(HV):
            kh = h // G
            qc = slice(kh * dk, (kh + 1) * dk)
            kc = slice(HK * dk + kh * dk, HK * dk + (kh + 1) * dk)
            vc = slice(2 * HK * dk + h * dv, 2 * HK * dk + (h + 1) * dv)
            S = np.zeros((dv, dk)) if state is None else _f64(state)[slot, h].T.copy()
            prev = []
            for t in range(cu[n], cu[n + 1]):                       # forward, keeping S_{t-1}
                a = np.exp(g[t, h]); b = beta[t, h]; k = xa[t, kc]; v = xa[t, vc]
                prev.append(S.copy())
                p = S @ k
                S = a * S + b * np.outer(v - a * p, k)
            GS = np.zeros((dv, dk))
            if d_state is not None:
                GS = _f64(d_state)[slot, h].T.copy()
            for i, t in reversed(list(enumerate(range(cu[n], cu[n + 1])))):
                a = np.exp(g[t, h]); b = beta[t, h]
                q = xa[t, qc]; k = xa[t, kc]; v = xa[t, vc]; do = d_o[t, h * dv:(h + 1) * dv]
                Sp = prev[i]
                p = Sp @ k
                r = v - a * p
                St = a * Sp + b * np.outer(r, k)
                GS = GS + np.outer(do, q)                           # o = S_t q
                dxa[t, qc] += St.T @ do
                dw = GS @ k                                         # w = b r, S_t = a Sp + w k^T
                dxa[t, kc] += GS.T @ (b * r)
                da = np.sum(GS * Sp)
                dxa[t, vc] += b * dw
                db[t, h] = dw @ r
                dp = -a * b * dw                                    # r = v - a p
                da += -b * (dw @ p)
                dxa[t, kc] += Sp.T @ dp                             # p = Sp k
                GS = a * GS + np.outer(dp, k)
                dg[t, h] = da * a
            if d_state_in is not None:
                d_state_in[slot, h] = GS.T
    return dxa, dg, db, d_state_in


# ------------------------------------------------------------------ Q8 state

def pcg_hash(v):
    """The PCG hash of Jarzynski and Olano ("Hash Functions for GPU Rendering", JCGT 2020): one
    step of the PCG32 LCG followed by its RXS-M-XS output permutation, on uint32 (wrapping)."""
    v = np.asarray(v, dtype=np.uint32)
    with np.errstate(over="ignore"):
        state = v * np.uint32(747796405) + np.uint32(2891336453)
        word = ((state >> ((state >> np.uint32(28)) + np.uint32(4))) ^ state) * np.uint32(277803737)
    return (word >> np.uint32(22)) ^ word


def q8_dither(frame, slot, HV, h, dk, dv):
    """The rounding offsets u in [0, 1) of one head's [dk, dv] codes at a given frame.  Every code
    draws its own: with index = ((slot*HV + h)*dk + i)*dv + j (uint32) and
    r = pcg_hash(index ^ pcg_hash(frame)), u = (r >> 8) * 2^-24 (24 bits, exact in fp32)."""
    i = np.arange(dk, dtype=np.uint64)[:, None]
    j = np.arange(dv, dtype=np.uint64)[None, :]
    idx = ((((np.uint64(slot) * np.uint64(HV) + np.uint64(h)) * np.uint64(dk) + i) * np.uint64(dv) + j)
           & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    r = pcg_hash(idx ^ pcg_hash(np.uint32(frame)))
    return (r >> np.uint32(8)).astype(np.float32) * np.float32(1.0 / 16777216.0)


def bf16_round(x):
    """fp32 -> the nearest bf16 value (ties to even), returned as fp32: the top 16 bits of the
    fp32 pattern after adding 0x7FFF plus the lowest kept bit (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
    return (r & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)


def q8_encode_head(M, frame, slot, HV, h, residual=None):
    """One head's fp32 [dk, dv] state (M = S^T) to int8 codes and per-row scales, every step in
    fp32 with round-to-nearest.  The value encoded is x = M, or x = M + residual with error
    feedback (residual: the bf16 [dk, dv] left by the previous encode).  Absmax a_i of row i of
    x, scale s_i = a_i / 127, code = clamp(floor(x * (127 / a_i) + u), -127, 127) with the dither
    u of q8_dither (stochastic rounding: the expected code is x * 127 / a_i).  A zero row gets
    scale 0 and codes 0.  Returns (codes int8 [dk, dv], scales fp32 [dk]); with a residual also
    the new residual bf16(x - code * s_i) (as fp32 values), the rounding error this encode
    leaves for the next one."""
    M = np.asarray(M, dtype=np.float32)
    if residual is not None:
        M = (M + np.asarray(residual, dtype=np.float32)).astype(np.float32)
    dk, dv = M.shape
    amax = np.max(np.abs(M), axis=1).astype(np.float32)
    nz = amax > 0
    scale = np.zeros(dk, np.float32)
    scale[nz] = amax[nz] / np.float32(127)
    inv = np.zeros(dk, np.float32)
    inv[nz] = np.float32(127) / amax[nz]
    x = (M * inv[:, None]).astype(np.float32)
    u = q8_dither(frame, slot, HV, h, dk, dv)
    c = np.floor((x + u).astype(np.float32))
    c = np.clip(c, -127, 127)
    c[~nz] = 0
    codes = c.astype(np.int8)
    if residual is None:
        return codes, scale
    back = (codes.astype(np.float32) * scale[:, None]).astype(np.float32)
    return codes, scale, bf16_round((M - back).astype(np.float32))


def q8_encode(state, frame, residual=None):
    """A whole fp32 pool [slots, HV, dk, dv] -> (codes int8, scales [slots, HV, dk]), plus the
    new residual pool when a residual pool (error feedback) is given."""
    state = np.asarray(state, dtype=np.float32)
    S, HV, dk, dv = state.shape
    codes = np.zeros(state.shape, np.int8)
    scales = np.zeros((S, HV, dk), np.float32)
    res = None if residual is None else np.zeros(state.shape, np.float32)
    for s in range(S):
        for h in range(HV):
            if residual is None:
                codes[s, h], scales[s, h] = q8_encode_head(state[s, h], frame, s, HV, h)
            else:
                codes[s, h], scales[s, h], res[s, h] = q8_encode_head(state[s, h], frame, s, HV, h,
                                                                      residual[s, h])
    return (codes, scales) if residual is None else (codes, scales, res)


def q8_decode(codes, scales):
    """Dequantise: M = code * scale (fp32)."""
    return (np.asarray(codes, np.float32) * np.asarray(scales, np.float32)[..., None]).astype(np.float32)


def mixer_decode_q8(x, conv_w, u, b_logit, A_log, dt_bias, z, norm_w, HK, HV, dk, dv, codes, scales,
                    conv_state, frame, slot_idx=None, q_scale=1.0, l2_eps=1e-6, norm_eps=1e-6,
                    residual=None):
    """One decode step (one token for each of n sequences) on a Q8 state pool: the state of
    each sequence's slot is dequantised, the plain mixer (fp64) runs one token, and the new
    state is cast to fp32 and quantised again at `frame`.  With a residual pool (error
    feedback), the slot's residual is added to the new state before it is quantised and is
    replaced by the rounding error of that encode; the recurrence itself reads only the
    dequantised codes.  Returns (y, codes, scales, conv), plus the residual pool when given."""
    n = _f64(x).shape[0]
    slots = list(range(n)) if slot_idx is None else [int(s) for s in np.asarray(slot_idx)]
    codes = np.array(codes, copy=True); scales = np.array(scales, copy=True)
    res = None if residual is None else np.array(residual, dtype=np.float32, copy=True)
    conv = _f64(conv_state).copy()
    y = np.zeros((n, HV * dv))
    for i, s in enumerate(slots):
        if s < 0:
            continue
        st = q8_decode(codes[s:s + 1], scales[s:s + 1]).astype(np.float64)
        out = mixer(_f64(x)[i:i + 1], conv_w, _f64(u)[i:i + 1], _f64(b_logit)[i:i + 1], A_log, dt_bias,
                    _f64(z)[i:i + 1], norm_w, np.array([0, 1], np.int32), HK, HV, dk, dv,
                    state=st, conv_state=conv[s:s + 1], q_scale=q_scale, l2_eps=l2_eps,
                    norm_eps=norm_eps, n_threads=1)
        y[i] = out["y"][0]
        conv[s] = out["conv_state"][0]
        for h in range(HV):
            Mh = out["state"][0, h].astype(np.float32)
            if res is None:
                codes[s, h], scales[s, h] = q8_encode_head(Mh, frame, s, HV, h)
            else:
                codes[s, h], scales[s, h], res[s, h] = q8_encode_head(Mh, frame, s, HV, h, res[s, h])
    return (y, codes, scales, conv) if res is None else (y, codes, scales, conv, res)
