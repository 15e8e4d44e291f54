"""Pins of the fp64 oracle to facts the mathematics fixes (CPU only).

Each test checks the oracle against something other than itself: a closed
form, a hand-worked example, brute force with dense matrices, a library
routine that computes a special case, or an invariant (linearity, chunked ==
sequential, split invariance).  Together they are chosen so that a dropped
term, a wrong sign, a wrong index or a transposed operand in the oracle fails
at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pack(q, k, v):
    """[T, HK*dk], [T, HK*dk], [T, HV*dv] -> xa [T, CH]."""
    return np.concatenate([q, k, v], axis=1)


def _run(q, k, v, g, beta, S0T=None, HK=1, HV=1, cu=None, chunk=0, slot_idx=None):
    T = q.shape[0]
    dk = q.shape[1] // HK
    dv = v.shape[1] // HV
    cu = np.array([0, T] if cu is None else cu, np.int32)
    return oracle.delta_rule(_pack(q, k, v), g, beta, cu, HK, HV, dk, dv, state=S0T,
                             slot_idx=slot_idx, chunk=chunk, n_threads=2)


def _rand_unit(rng, T, d):
    x = rng.standard_normal((T, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


# ----------------------------------------------------------- hand example

def test_hand_worked_example_d2():
    G = json.load(open(os.path.join(GOLDEN, "hand_rule_d2.json")))
    q = np.array(G["q"]); k = np.array(G["k"]); v = np.array(G["v"])
    g = np.log(np.array(G["a"]))[:, None]
    b = np.array(G["b"])[:, None]
    S0 = np.array(G["S0"])
    o, st = _run(q, k, v, g, b, S0T=S0.T[None, None].copy())
    np.testing.assert_allclose(o, np.array(G["o"]), atol=1e-14)
    np.testing.assert_allclose(st[0, 0].T, np.array(G["S_final"]), atol=1e-14)


# ------------------------------------------------------------ special cases

def test_beta0_a1_leaves_state_unchanged():
    rng = np.random.default_rng(1)
    T, d = 7, 8
    q, k, v = rng.standard_normal((T, d)), _rand_unit(rng, T, d), rng.standard_normal((T, d))
    S0T = rng.standard_normal((1, 1, d, d))
    o, st = _run(q, k, v, np.zeros((T, 1)), np.zeros((T, 1)), S0T=S0T)
    np.testing.assert_array_equal(st, S0T)
    np.testing.assert_allclose(o, q @ S0T[0, 0], rtol=1e-13, atol=1e-13)  # o = S0 q


def test_a0_resets_state():
    rng = np.random.default_rng(2)
    T, d = 5, 6
    q, k, v = rng.standard_normal((T, d)), _rand_unit(rng, T, d), rng.standard_normal((T, d))
    b = rng.uniform(0.1, 0.9, (T, 1))
    S0T = rng.standard_normal((1, 1, d, d))
    o, st = _run(q, k, v, np.full((T, 1), -np.inf), b, S0T=S0T)
    S_last = b[-1, 0] * np.outer(v[-1], k[-1])          # S = b v k^T
    np.testing.assert_allclose(st[0, 0].T, S_last, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(o[-1], S_last @ q[-1], rtol=1e-13, atol=1e-14)


def test_beta1_unit_key_maps_key_to_value():
    rng = np.random.default_rng(3)
    T, d = 6, 16
    q, k, v = rng.standard_normal((T, d)), _rand_unit(rng, T, d), rng.standard_normal((T, d))
    g = -rng.uniform(0, 2, (T, 1))
    for t in range(1, T + 1):
        S0T = rng.standard_normal((1, 1, d, d))
        _, st = _run(q[:t], k[:t], v[:t], g[:t], np.ones((t, 1)), S0T=S0T)
        np.testing.assert_allclose(st[0, 0].T @ k[t - 1], v[t - 1], rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_build_associative_memory():
    rng = np.random.default_rng(4)
    d = 8
    K = np.eye(d)
    V = rng.standard_normal((d, d))
    Q = np.eye(d)[::-1].copy()
    _, st = _run(Q, K, V, np.zeros((d, 1)), np.ones((d, 1)), S0T=np.zeros((1, 1, d, d)))
    S = st[0, 0].T
    np.testing.assert_allclose(S, V.T @ K, atol=1e-14)          # S = sum_i v_i k_i^T
    for i in range(d):
        np.testing.assert_allclose(S @ np.eye(d)[i], V[i], atol=1e-14)


def test_linear_in_values_and_initial_state():
    rng = np.random.default_rng(5)
    T, d = 9, 8
    q, k = rng.standard_normal((T, d)), _rand_unit(rng, T, d)
    g, b = -rng.uniform(0, 1, (T, 1)), rng.uniform(0, 1, (T, 1))
    V1, V2 = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    S1, S2 = rng.standard_normal((1, 1, d, d)), rng.standard_normal((1, 1, d, d))
    o1, s1 = _run(q, k, V1, g, b, S0T=S1)
    o2, s2 = _run(q, k, V2, g, b, S0T=S2)
    o3, s3 = _run(q, k, 2.0 * V1 - 3.0 * V2, g, b, S0T=2.0 * S1 - 3.0 * S2)
    np.testing.assert_allclose(o3, 2 * o1 - 3 * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(s3, 2 * s1 - 3 * s2, rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------- brute force

@pytest.mark.parametrize("T,d", [(1, 1), (2, 3), (3, 4), (4, 4), (4, 2)])
def test_brute_force_product_form(T, d):
    """S_T = S0 prod_i a_i (I - b_i k_i k_i^T) + sum_i b_i v_i k_i^T prod_{j>i} a_j (I - b_j k_j k_j^T)."""
    rng = np.random.default_rng(10 + T * 7 + d)
    q, k, v = rng.standard_normal((T, d)), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    g, b = -rng.uniform(0, 2, (T, 1)), rng.uniform(0, 1, (T, 1))
    S0 = rng.standard_normal((d, d))
    o, st = _run(q, k, v, g, b, S0T=S0.T[None, None].copy())
    F = [np.exp(g[i, 0]) * (np.eye(d) - b[i, 0] * np.outer(k[i], k[i])) for i in range(T)]
    for t in range(1, T + 1):
        S = S0.copy()
        for i in range(t):
            S = S @ F[i]
        for i in range(t):
            term = b[i, 0] * np.outer(v[i], k[i])
            for j in range(i + 1, t):
                term = term @ F[j]
            S = S + term
        np.testing.assert_allclose(o[t - 1], S @ q[t - 1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(st[0, 0].T, S, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ chunked == sequential

@pytest.mark.parametrize("chunk", [1, 2, 16, 64])
def test_chunked_equals_sequential(chunk):
    rng = np.random.default_rng(20 + chunk)
    HK, HV, d = 2, 4, 16
    lens = [0, 1, 37, 130, 64]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = rng.standard_normal((T, HK * d))
    k = np.concatenate([_rand_unit(rng, T, d) for _ in range(HK)], 1)
    v = rng.standard_normal((T, HV * d))
    g, b = -rng.uniform(0, 1.5, (T, HV)), rng.uniform(0, 1, (T, HV))
    S0 = rng.standard_normal((len(lens), HV, d, d)) * 0.1
    o_s, s_s = _run(q, k, v, g, b, S0T=S0, HK=HK, HV=HV, cu=cu, chunk=0)
    o_c, s_c = _run(q, k, v, g, b, S0T=S0, HK=HK, HV=HV, cu=cu, chunk=chunk)
    scale = np.abs(o_s).max()
    assert np.abs(o_c - o_s).max() <= 1e-12 * scale
    assert np.abs(s_c - s_s).max() <= 1e-12 * np.abs(s_s).max()


def test_gqa_head_grouping_consecutive():
    """v-head h reads q/k head h // (HV/HK)."""
    rng = np.random.default_rng(30)
    HK, HV, d, T = 2, 4, 4, 5
    q = rng.standard_normal((T, HK * d)); k = rng.standard_normal((T, HK * d))
    v = rng.standard_normal((T, HV * d))
    g, b = -rng.uniform(0, 1, (T, HV)), rng.uniform(0, 1, (T, HV))
    o, _ = _run(q, k, v, g, b, HK=HK, HV=HV)
    for h in range(HV):
        kh = h // (HV // HK)
        oh, _ = _run(q[:, kh * d:(kh + 1) * d], k[:, kh * d:(kh + 1) * d], v[:, h * d:(h + 1) * d],
                     g[:, h:h + 1], b[:, h:h + 1])
        np.testing.assert_array_equal(o[:, h * d:(h + 1) * d], oh)


# ------------------------------------------------------------------- conv

def test_conv_impulse_response_and_library():
    rng = np.random.default_rng(40)
    CH, T = 5, 9
    w = rng.standard_normal((CH, 4))
    x = np.zeros((T, CH)); x[0] = 1.0
    out, _ = oracle.conv1d_silu(x, [0, T], w)
    silu = lambda t: t / (1 + np.exp(-t))
    for t in range(4):
        np.testing.assert_allclose(out[t], silu(w[:, 3 - t]), rtol=1e-15)
    np.testing.assert_allclose(out[4:], silu(np.zeros((T - 4, CH))))
    # random input, zero history == torch conv1d (cross-correlation) with left padding 3
    x = rng.standard_normal((T, CH))
    out, _ = oracle.conv1d_silu(x, [0, T], w)
    ref = torch.nn.functional.conv1d(torch.tensor(x.T[None]), torch.tensor(w[:, None, :]),
                                     padding=3, groups=CH)[0, :, :T].T
    np.testing.assert_allclose(out, torch.nn.functional.silu(ref).numpy(), rtol=1e-13, atol=1e-15)


def test_conv_history_and_split_invariance():
    rng = np.random.default_rng(41)
    CH = 6
    w = rng.standard_normal((CH, 4))
    hist = rng.standard_normal((1, CH, 3))
    x = rng.standard_normal((11, CH))
    full, h_full = oracle.conv1d_silu(x, [0, 11], w, conv_state=hist)
    # history behaves as the three tokens before the sequence
    ext = np.concatenate([hist[0].T, x])
    ref, _ = oracle.conv1d_silu(ext, [0, 14], w)
    np.testing.assert_allclose(full, ref[3:], rtol=1e-14)
    np.testing.assert_array_equal(h_full[0], x[-3:].T)       # new history = last 3 raw inputs
    # one call over 11 tokens == 11 one-token calls == calls of 1, 2 and 8 tokens
    h = hist.copy(); outs = []
    for t in range(11):
        o1, h = oracle.conv1d_silu(x[t:t + 1], [0, 1], w, conv_state=h)
        outs.append(o1)
    np.testing.assert_array_equal(np.concatenate(outs), full)
    np.testing.assert_array_equal(h, h_full)
    h = hist.copy(); outs = []
    for a, b in [(0, 1), (1, 3), (3, 11)]:
        o1, h = oracle.conv1d_silu(x[a:b], [0, b - a], w, conv_state=h)
        outs.append(o1)
    np.testing.assert_array_equal(np.concatenate(outs), full)
    np.testing.assert_array_equal(h, h_full)
    # a 2-token sequence keeps the newest old-history tap
    _, h2 = oracle.conv1d_silu(x[:2], [0, 2], w, conv_state=hist)
    np.testing.assert_array_equal(h2[0], np.stack([hist[0, :, 2], x[0], x[1]], 1))
    # empty sequence leaves the history unchanged
    _, h0 = oracle.conv1d_silu(np.zeros((0, CH)), [0, 0], w, conv_state=hist)
    np.testing.assert_array_equal(h0, hist)


def test_conv_varlen_no_leakage_and_padding_slot():
    rng = np.random.default_rng(42)
    CH = 4
    w = rng.standard_normal((CH, 4))
    hist = rng.standard_normal((3, CH, 3))
    x = rng.standard_normal((10, CH))
    cu = [0, 4, 4, 10]
    out, h = oracle.conv1d_silu(x, cu, w, conv_state=hist, slot_idx=[2, 0, -1])
    o0, h0 = oracle.conv1d_silu(x[:4], [0, 4], w, conv_state=hist[2:3])
    o2, _ = oracle.conv1d_silu(x[4:], [0, 6], w)                  # padding lane: zero history
    np.testing.assert_array_equal(out[:4], o0)
    np.testing.assert_array_equal(out[4:], o2)
    np.testing.assert_array_equal(h[2], h0[0])
    np.testing.assert_array_equal(h[0], hist[0])                  # empty sequence
    np.testing.assert_array_equal(h[1], hist[1])                  # untouched slot


# ----------------------------------------------------- gates, L2, gated norm

def test_gates_match_library_routines():
    rng = np.random.default_rng(50)
    T, HV = 33, 3
    u = rng.standard_normal((T, HV)) * 4; b = rng.standard_normal((T, HV)) * 4
    A = rng.uniform(-1, 1, HV); dt = rng.standard_normal(HV)
    g, beta = oracle.gates(u, b, A, dt)
    sp = torch.nn.functional.softplus(torch.tensor(u + dt)).numpy()
    np.testing.assert_allclose(g, -np.exp(A) * sp, rtol=1e-14)
    np.testing.assert_allclose(beta, torch.sigmoid(torch.tensor(b)).numpy(), rtol=1e-14)
    assert (g < 0).all() and (beta > 0).all() and (beta < 1).all()


def test_l2norm_closed_form():
    xa = np.zeros((1, 2 * 2 + 2))
    xa[0, :2] = [3.0, 4.0]            # q head (HK=1, dk=2)
    xa[0, 2:4] = [0.0, 2.0]           # k head
    xa[0, 4:] = [7.0, 8.0]            # v untouched
    eps, qs = 1e-6, 0.5
    out = oracle.l2norm_qk(xa, 1, 2, eps=eps, q_scale=qs)
    np.testing.assert_allclose(out[0, :2], qs * np.array([3, 4]) / np.sqrt(25 + eps), rtol=1e-15)
    np.testing.assert_allclose(out[0, 2:4], np.array([0, 2]) / np.sqrt(4 + eps), rtol=1e-15)
    np.testing.assert_array_equal(out[0, 4:], [7, 8])


def test_gated_rmsnorm_cases():
    rng = np.random.default_rng(60)
    T, HV, dv, eps = 4, 2, 8, 1e-6
    o = rng.standard_normal((T, HV * dv)); w = rng.standard_normal(dv)
    y = oracle.gated_rmsnorm(o, np.zeros_like(o), w, HV, dv, eps)
    np.testing.assert_array_equal(y, 0.0)                          # z = 0 => y = 0
    c = 0.37
    z = rng.standard_normal((T, HV * dv))
    y = oracle.gated_rmsnorm(np.full_like(o, c), z, np.ones(dv), HV, dv, eps)
    silu = z / (1 + np.exp(-z))
    np.testing.assert_allclose(y, c / np.sqrt(c * c + eps) * silu, rtol=1e-14)
    # library routine: torch rms_norm over each head, then the gate
    y = oracle.gated_rmsnorm(o, z, w, HV, dv, eps)
    ref = torch.nn.functional.rms_norm(torch.tensor(o).view(T, HV, dv), (dv,),
                                       weight=torch.tensor(w), eps=eps).view(T, -1).numpy() * silu
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------- whole mixer

def _mixer_inputs(rng, lens, HK=2, HV=4, d=8, with_state=True):
    CH = 2 * HK * d + HV * d
    T = sum(lens); N = len(lens)
    return dict(
        x=rng.standard_normal((T, CH)), conv_w=rng.standard_normal((CH, 4)) * 0.25,
        u=rng.standard_normal((T, HV)), b_logit=rng.standard_normal((T, HV)),
        A_log=rng.uniform(-1, 1, HV), dt_bias=np.zeros(HV), z=rng.standard_normal((T, HV * d)),
        norm_w=np.ones(d), cu_seqlens=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
        HK=HK, HV=HV, dk=d, dv=d,
        state=rng.standard_normal((N, HV, d, d)) * 0.02 if with_state else None,
        conv_state=rng.standard_normal((N, CH, 3)) if with_state else None)


def test_mixer_split_invariance():
    """prefill(T) == prefill(T1) then prefill(T2) == prefill(T1) then one-token steps."""
    rng = np.random.default_rng(70)
    I = _mixer_inputs(rng, [23])
    full = oracle.mixer(**I, n_threads=2)
    T1 = 9

    def sub(a, b, state, conv):
        J = dict(I)
        for key in ("x", "u", "b_logit", "z"):
            J[key] = I[key][a:b]
        J["cu_seqlens"] = np.array([0, b - a], np.int32)
        J["state"], J["conv_state"] = state, conv
        return oracle.mixer(**J, n_threads=2)

    p1 = sub(0, T1, I["state"], I["conv_state"])
    p2 = sub(T1, 23, p1["state"], p1["conv_state"])
    np.testing.assert_allclose(np.concatenate([p1["y"], p2["y"]]), full["y"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(p2["state"], full["state"], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(p2["conv_state"], full["conv_state"])
    st, cs, ys = p1["state"], p1["conv_state"], [p1["y"]]
    for t in range(T1, 23):
        r = sub(t, t + 1, st, cs)
        st, cs = r["state"], r["conv_state"]
        ys.append(r["y"])
    np.testing.assert_allclose(np.concatenate(ys), full["y"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(st, full["state"], rtol=1e-12, atol=1e-14)


def test_mixer_varlen_equals_separate_and_padding_lane():
    rng = np.random.default_rng(71)
    lens = [5, 0, 12, 3]
    I = _mixer_inputs(rng, lens)
    packed = oracle.mixer(**I, n_threads=2)
    cu = I["cu_seqlens"]
    for n, L in enumerate(lens):
        J = dict(I)
        for key in ("x", "u", "b_logit", "z"):
            J[key] = I[key][cu[n]:cu[n + 1]]
        J["cu_seqlens"] = np.array([0, L], np.int32)
        J["state"], J["conv_state"] = I["state"][n:n + 1], I["conv_state"][n:n + 1]
        r = oracle.mixer(**J, n_threads=1)
        np.testing.assert_array_equal(r["y"], packed["y"][cu[n]:cu[n + 1]])
        np.testing.assert_array_equal(r["state"][0], packed["state"][n])
        np.testing.assert_array_equal(r["conv_state"][0], packed["conv_state"][n])
    # slot mapping with a padding lane: zero output, its slot untouched
    pad = oracle.mixer(**I, slot_idx=np.array([3, 1, -1, 0], np.int32), n_threads=2)
    np.testing.assert_array_equal(pad["y"][cu[2]:cu[3]], 0.0)
    np.testing.assert_array_equal(pad["state"][2], I["state"][2])
    np.testing.assert_array_equal(pad["conv_state"][2], I["conv_state"][2])


def test_head_subset_channels_and_outputs():
    """The head map the full-size GPU checks sample with: HK=2, HV=4, d=2, q/k head 1 owns q
    channels 2-3, k channels 6-7, v-heads 2 and 3 (v channels 12-15, output columns 4-7); and the
    mixer over heads {1} or {0, 1} equals the full mixer's share exactly (heads never interact)."""
    chs, vh, cols = oracle.head_channels(2, 4, 2, 2, [1])
    assert chs.tolist() == [2, 3, 6, 7, 12, 13, 14, 15]
    assert vh.tolist() == [2, 3] and cols.tolist() == [4, 5, 6, 7]
    rng = np.random.default_rng(72)
    I = _mixer_inputs(rng, [7, 0, 19], HK=4, HV=8, d=4)
    full = oracle.mixer(**I, n_threads=2)
    J = {k: v for k, v in I.items() if k not in ("HK", "HV", "dk", "dv")}
    for heads in ([1], [0, 3], [2, 1]):
        r = oracle.mixer_heads(**J, HK=4, HV=8, dk=4, dv=4, kheads=heads, n_threads=1)
        chs, vh, cols = oracle.head_channels(4, 8, 4, 4, heads)
        np.testing.assert_array_equal(r["y"], full["y"][:, cols])
        np.testing.assert_array_equal(r["state"], full["state"][:, vh])
        np.testing.assert_array_equal(r["conv_state"], full["conv_state"][:, chs])


# ----------------------------------------------------------- slot maintenance

def test_state_copy_hand_example():
    """Snapshot / restore / reset on a hand-written pool: the expected pools are spelled out
    element by element (hyperflare core-design, "State operations")."""
    src = np.array([[[10., 11.]], [[20., 21.]], [[30., 31.]]])          # 3 slots of [1, 2]
    srcc = np.array([[[1, 2, 3]], [[4, 5, 6]], [[7, 8, 9]]], np.int16)  # 3 histories of [1, 3]
    dst = np.full((3, 1, 2), -1.0)
    dstc = np.full((3, 1, 3), -1, np.int16)
    # slot 2 -> 0 (copy), reset 1, inactive lane, out-of-range source (flagged, skipped)
    s, c, err = oracle.state_copy(src, srcc, dst, dstc, [2, -1, 0, 7], [0, 1, -1, 2])
    assert s.tolist() == [[[30., 31.]], [[0., 0.]], [[-1., -1.]]]
    assert c.tolist() == [[[7, 8, 9]], [[0, 0, 0]], [[-1, -1, -1]]]
    assert err
    assert dst.tolist() == [[[-1., -1.]]] * 3                         # inputs untouched
    # in one pool: snapshot then restore gives back the original slot bit for bit
    pool = np.array([[[1.5, -2.25]], [[0., 0.]]])
    snap, _, e1 = oracle.state_copy(pool, None, pool, None, [0], [1])
    assert snap.tolist() == [[[1.5, -2.25]], [[1.5, -2.25]]] and not e1
    live = snap.copy(); live[0] = 99.0
    back, _, e2 = oracle.state_copy(live, None, live, None, [1], [0])
    assert back[0].tolist() == [[1.5, -2.25]] and not e2
    # without a source pool every active pair resets; a destination index past the pool is flagged
    z, _, e3 = oracle.state_copy(None, None, pool, None, [5, -3], [0, 4])
    assert z.tolist() == [[[0., 0.]], [[0., 0.]]] and e3


def test_mixer_verify_columns_are_prefix_states():
    """Verification columns (hyperflare core-design, speculative target state): column j is the
    state after j+1 tokens, so the last column and every y row equal one plain pass over the k
    tokens, and column j of a k-token round equals the last column of a (j+1)-token round."""
    HK, HV, d, k = 1, 2, 4, 4
    CH = 2 * HK * d + HV * d
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2 * k, CH)); z = rng.standard_normal((2 * k, HV * d))
    u = rng.standard_normal((2 * k, HV)); b = rng.standard_normal((2 * k, HV))
    cw = rng.normal(0, 0.25, (CH, 4)); A = rng.uniform(-1, 1, HV); dt = np.zeros(HV); nw = np.ones(d)
    st = rng.normal(0, 0.02, (3, HV, d, d)); cs = rng.standard_normal((3, CH, 3))
    y, S, C = oracle.mixer_verify(x, cw, u, b, A, dt, z, nw, k, HK, HV, d, d, st, cs, src_idx=[2, 0],
                                  n_threads=1)
    for i, s in enumerate([2, 0]):
        one = oracle.mixer(x[i * k:(i + 1) * k], cw, u[i * k:(i + 1) * k], b[i * k:(i + 1) * k], A, dt,
                           z[i * k:(i + 1) * k], nw, np.array([0, k], np.int32), HK, HV, d, d,
                           state=st[s:s + 1].copy(), conv_state=cs[s:s + 1].copy(), n_threads=1)
        assert np.allclose(y[i * k:(i + 1) * k], one["y"], rtol=0, atol=1e-12)
        assert np.allclose(S[i, -1], one["state"][0], rtol=0, atol=1e-12)
        assert np.array_equal(C[i, -1], one["conv_state"][0])
        # the conv window after token j holds raw inputs j-2 .. j (history taps before token 0)
        X = np.concatenate([cs[s].T, x[i * k:(i + 1) * k]])          # [3 + k, CH]
        for j in range(k):
            assert np.array_equal(C[i, j], X[j + 1:j + 4].T)
    y2, S2, _ = oracle.mixer_verify(x[:2], cw, u[:2], b[:2], A, dt, z[:2], nw, 2, HK, HV, d, d, st, cs,
                                    src_idx=[2], n_threads=1)
    assert np.allclose(S2[0, 1], S[0, 1], rtol=0, atol=1e-12) and np.allclose(y2, y[:2], rtol=0, atol=1e-12)


def test_delta_rule_backward_matches_central_differences():
    """The oracle's reverse-mode gradient against central differences of the (pinned) forward:
    L = sum(d_o * o) + sum(d_state * M_final), over q, k, v, g, beta and the initial state, with
    GQA (two v-heads per q/k head), two sequences (one empty-ended, one of several tokens) and a
    padding-free slot map."""
    rng = np.random.default_rng(21)
    HK, HV, d = 1, 2, 3
    CH = 2 * HK * d + HV * d
    T, cu, slots = 7, np.array([0, 3, 7], np.int32), [1, 0]
    xa = rng.standard_normal((T, CH)) * 0.7
    g = -rng.uniform(0.05, 0.6, (T, HV)); beta = rng.uniform(0.2, 0.9, (T, HV))
    S0 = rng.standard_normal((2, HV, d, d)) * 0.3
    d_o = rng.standard_normal((T, HV * d)); d_S = rng.standard_normal((2, HV, d, d))

    def loss(xa_, g_, b_, S0_):
        o, st = oracle.delta_rule(xa_, g_, b_, cu, HK, HV, d, d, state=S0_.copy(), slot_idx=slots,
                                  n_threads=1)
        return float(np.sum(d_o * o) + np.sum(d_S * st))

    dxa, dg, db, dS0 = oracle.delta_rule_backward(xa, g, beta, cu, HK, HV, d, d, d_o, state=S0,
                                                  slot_idx=slots, d_state=d_S)
    eps = 1e-6
    for arr, grad in ((xa, dxa), (g, dg), (beta, db), (S0, dS0)):
        for idx in [tuple(rng.integers(0, s) for s in arr.shape) for _ in range(12)]:
            args_p = [a.copy() for a in (xa, g, beta, S0)]
            args_m = [a.copy() for a in (xa, g, beta, S0)]
            pos = [a is arr for a in (xa, g, beta, S0)].index(True)
            args_p[pos][idx] += eps
            args_m[pos][idx] -= eps
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (pos, idx, fd, grad[idx])


def test_delta_rule_backward_padding_lane_has_no_gradient():
    """A padding lane (negative slot) produces zero outputs and touches no state, so every
    gradient of its tokens is zero and the other lanes' gradients are those of the batch
    without it."""
    rng = np.random.default_rng(8)
    HK, HV, d = 1, 1, 2
    xa = rng.standard_normal((5, 2 * HK * d + HV * d))
    g = -rng.uniform(0.1, 0.5, (5, HV)); beta = rng.uniform(0.2, 0.8, (5, HV))
    d_o = rng.standard_normal((5, HV * d)); S0 = rng.standard_normal((1, HV, d, d))
    o, _ = oracle.delta_rule(xa, g, beta, np.array([0, 2, 5], np.int32), HK, HV, d, d, state=S0.copy(),
                             slot_idx=[-1, 0], n_threads=1)
    assert np.all(o[:2] == 0)                                    # the forward's padding rule
    full = oracle.delta_rule_backward(xa, g, beta, [0, 2, 5], HK, HV, d, d, d_o, state=S0, slot_idx=[-1, 0])
    alone = oracle.delta_rule_backward(xa[2:], g[2:], beta[2:], [0, 3], HK, HV, d, d, d_o[2:], state=S0,
                                       slot_idx=[0])
    assert np.all(full[0][:2] == 0) and np.all(full[1][:2] == 0) and np.all(full[2][:2] == 0)
    for a, b in zip(full[:3], alone[:3]):
        assert np.array_equal(a[2:], b)
    assert np.array_equal(full[3], alone[3])


# ----------------------------------------------------------- Q8 state

def test_q8_encoding_rules():
    """Every code lies in [-127, 127], the row's largest magnitude maps to +-127, the decoded
    value is within one step (the row scale max/127) of the original, and a zero row stays zero."""
    rng = np.random.default_rng(31)
    M = (rng.standard_normal((6, 16)) * rng.uniform(0.01, 3, (6, 1))).astype(np.float32)
    M[4] = 0
    c, s = oracle.q8_encode_head(M, frame=5, slot=2, HV=3, h=1)
    assert c.dtype == np.int8 and np.all(np.abs(c.astype(int)) <= 127)
    for i in range(6):
        if i == 4:
            assert s[i] == 0 and np.all(c[i] == 0)
            continue
        j = int(np.argmax(np.abs(M[i])))
        assert abs(int(c[i, j])) == 127 and np.sign(c[i, j]) == np.sign(M[i, j])
        assert s[i] == np.float32(np.abs(M[i]).max()) / np.float32(127)
    err = np.abs(oracle.q8_decode(c, s) - M)
    assert np.all(err < s[:, None] * 1.0001 + 1e-30)


def _golden(name):
    import json
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


def test_pcg_hash_matches_the_hand_evaluated_definition():
    """pcg_hash against values worked by hand from the published PCG hash (Jarzynski and Olano,
    JCGT 2020; intermediates in tests/golden/pcg_hash.json)."""
    cases = _golden("pcg_hash.json")["cases"]
    v = np.array([c["v"] for c in cases], dtype=np.uint32)
    want = np.array([int(c["hash"], 16) for c in cases], dtype=np.uint32)
    assert np.array_equal(oracle.pcg_hash(v), want)
    for c in cases:   # scalar calls too
        assert int(oracle.pcg_hash(np.uint32(c["v"]))) == int(c["hash"], 16)


def test_bf16_round_matches_torch_conversion():
    """The oracle's fp32 -> bf16 rounding against torch's CPU conversion (round to nearest even),
    on random values, exact ties and values next to ties."""
    rng = np.random.default_rng(34)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 5, 20000))).astype(np.float32)
    ties = (np.arange(1, 4000, dtype=np.uint32) << np.uint32(15)).view(np.float32)   # low half 0x8000
    x = np.concatenate([x, ties, -ties, np.nextafter(ties, np.float32(0)), np.float32([0.0, -0.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(oracle.bf16_round(x).view(np.uint32), want.view(np.uint32))


def test_q8_dither_per_code_24_bits():
    """Each code's dither is (pcg_hash(index ^ pcg_hash(frame)) >> 8) / 2^24: the hand-worked
    values of tests/golden/q8_encode_d2.json (slot 1, HV 2, head 1, frame 3: indices 12..15)."""
    u = oracle.q8_dither(3, 1, 2, 1, 2, 2)
    want = np.array([[2758547, 10522013], [9246080, 9519212]], np.float64) / 2.0 ** 24
    assert u.dtype == np.float32 and np.array_equal(u.astype(np.float64), want)


def test_q8_dither_uniform_and_rounding_unbiased():
    """The dither is uniform on [0, 1) (16-bin counts within 5 sigma over 65,536 draws, nearly all
    values distinct); the stochastic rounding is unbiased: the decoded value averaged over 400
    frames sits within a few standard errors of the input."""
    u = np.concatenate([oracle.q8_dither(f, 0, 4, 1, 64, 64).ravel() for f in range(16)])
    assert u.min() >= 0 and u.max() < 1 and len(np.unique(u)) > 0.99 * u.size
    counts = np.histogram(u, bins=16, range=(0, 1))[0]
    expect = u.size / 16
    assert np.all(np.abs(counts - expect) <= 5 * np.sqrt(expect))
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / u.size)
    rng = np.random.default_rng(32)
    M = rng.standard_normal((4, 32)).astype(np.float32)
    acc = np.zeros_like(M, dtype=np.float64)
    F = 400
    for f in range(F):
        c, s = oracle.q8_encode_head(M, frame=f, slot=0, HV=1, h=0)
        acc += oracle.q8_decode(c, s)
    step = (np.abs(M).max(axis=1) / 127)[:, None]
    assert np.all(np.abs(acc / F - M) <= 5 * step / (2 * np.sqrt(F)) + 1e-7)
    # round-to-nearest (no dither) would be biased for values between codes
    biased = np.round(M / step) * step
    assert np.abs(biased - M).max() > 10 * np.abs(acc / F - M).max() / 5


def test_q8_encode_hand_example_plain_and_error_feedback():
    g = _golden("q8_encode_d2.json")
    M = np.array(g["M"], np.float32)
    c, s = oracle.q8_encode_head(M, g["frame"], g["slot"], g["HV"], g["head"])
    assert np.array_equal(c, np.array(g["codes_plain"], np.int8))
    assert np.array_equal(s, np.array(g["scales_plain"], np.float32))
    c, s, r = oracle.q8_encode_head(M, g["frame"], g["slot"], g["HV"], g["head"],
                                    np.array(g["residual_in"], np.float32))
    assert np.array_equal(c, np.array(g["codes_ef"], np.int8))
    assert np.array_equal(s, np.array(g["scales_ef"], np.float32))
    assert np.array_equal(r, np.array(g["residual_out"], np.float32))


def test_q8_error_feedback_keeps_the_running_sum():
    """Error feedback (x_t = y_t + e_{t-1}, e_t = x_t - decode(code_t)) telescopes: the running
    sum of the decoded values equals the running sum of the inputs minus the last residual, up
    to the bf16 rounding of each stored residual (|rounding| <= 2^-9 |e|, |e| < one step).  Without
    it the running-sum error is a random walk that grows like sqrt(t) steps."""
    rng = np.random.default_rng(35)
    T = 300
    ys = [(rng.standard_normal((3, 16)) * [[1.0], [0.1], [3.0]]).astype(np.float32) for _ in range(T)]
    e = np.zeros((3, 16), np.float32)
    dec_sum = np.zeros((3, 16)); in_sum = np.zeros((3, 16)); plain_sum = np.zeros((3, 16))
    bound = np.zeros((3, 16))
    for t, y in enumerate(ys):
        c, s, e_new = oracle.q8_encode_head(y, frame=t, slot=0, HV=1, h=0, residual=e)
        x = (y + e).astype(np.float32)
        exact = x.astype(np.float64) - oracle.q8_decode(c, s).astype(np.float64)
        assert np.all(np.abs(exact) < s[:, None] * 1.0001)                  # within one step
        assert np.all(np.abs(e_new - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-12)   # bf16 of it
        bound += np.abs(e_new - exact) + np.abs(x.astype(np.float64) - (y.astype(np.float64) + e))
        dec_sum += oracle.q8_decode(c, s); in_sum += y
        c0, s0 = oracle.q8_encode_head(y, frame=t, slot=0, HV=1, h=0)
        plain_sum += oracle.q8_decode(c0, s0)
        e = e_new
    assert np.all(np.abs(dec_sum - (in_sum - e)) <= bound + 1e-9)
    step = np.mean([np.abs(y).max(axis=1) for y in ys], axis=0)[:, None] / 127
    assert np.abs(dec_sum - in_sum).max(axis=1).max() < 2 * step.max()
    assert np.mean(np.abs(plain_sum - in_sum) / step) > 3 * np.mean(np.abs(dec_sum - in_sum) / step)


def _q8_step_inputs(g):
    x = np.array([g["x"]]); z = np.array([g["z"]])
    cw = np.tile(np.array(g["conv_w"], np.float64), (6, 1))
    conv = np.zeros((2, 6, 3)); conv[1] = np.array(g["conv_state_slot1"])
    codes = np.zeros((2, 1, 2, 2), np.int8); codes[1, 0] = np.array(g["codes_in"], np.int8)
    scales = np.zeros((2, 1, 2), np.float32)
    scales[1, 0] = [np.float32(1) / np.float32(127), np.float32(0.5) / np.float32(127)]
    zeros = np.zeros((1, 1))
    return x, z, cw, conv, codes, scales, zeros


def test_mixer_decode_q8_hand_worked_step():
    """One decode step on a Q8 slot against tests/golden/q8_decode_step_d2.json (worked by hand):
    y, the new codes and scales of slot 1, slot 0 untouched, the history shifted; then the same
    step with an error-feedback residual."""
    g = _golden("q8_decode_step_d2.json")
    x, z, cw, conv, codes, scales, zeros = _q8_step_inputs(g)
    args = (x, cw, zeros, zeros, np.zeros(1), np.zeros(1), z, np.ones(2), 1, 1, 2, 2)
    y, c2, s2, conv2 = oracle.mixer_decode_q8(*args, codes, scales, conv, frame=g["frame"], slot_idx=[1])
    assert np.allclose(y[0], g["y"], rtol=1e-12, atol=0)
    assert np.array_equal(c2[1, 0], np.array(g["codes_plain"], np.int8))
    assert np.array_equal(s2[1, 0], np.array(g["scales_plain"], np.float32))
    assert np.array_equal(c2[0], codes[0]) and np.array_equal(s2[0], scales[0])
    hist = np.array(g["conv_state_slot1"])
    assert np.array_equal(conv2[1], np.concatenate([hist[:, 1:], x[0][:, None]], axis=1))
    res = np.zeros((2, 1, 2, 2), np.float32); res[1, 0] = g["residual_in"]
    y, c3, s3, conv3, r3 = oracle.mixer_decode_q8(*args, codes, scales, conv, frame=g["frame"], slot_idx=[1],
                                                   residual=res)
    assert np.allclose(y[0], g["y"], rtol=1e-12, atol=0)            # the rule reads the codes only
    assert np.array_equal(c3[1, 0], np.array(g["codes_ef"], np.int8))
    assert np.array_equal(s3[1, 0], np.array(g["scales_ef"], np.float32))
    assert np.array_equal(r3[1, 0], np.array(g["residual_out"], np.float32))
    assert np.array_equal(r3[0], res[0])
