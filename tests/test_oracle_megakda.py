"""Pins of the MegaKDA-style oracle (oracle/megakda.py) against closed forms
and a brute-force scalar loop, independent of the oracle's own code."""
import math

import numpy as np
import pytest

import oracle
from oracle import megakda


def test_silu_closed_forms():
    # sigmoid(log 3) = 3/4, so silu(log 3) = (3/4) log 3; silu(0) = 0
    assert megakda.silu(0.0) == 0.0
    assert abs(megakda.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert abs(megakda.silu(-math.log(3.0)) + 0.25 * math.log(3.0)) < 1e-15


def test_silu_odd_part_and_far_arguments():
    # sigmoid(x) + sigmoid(-x) = 1, so silu(x) - silu(-x) = x at any scale,
    # including the saturated arguments the fused kernels' tests reach
    x = np.array([0.5, 3.0, 40.0, 88.5, 300.0])
    np.testing.assert_allclose(megakda.silu(x) - megakda.silu(-x), x, rtol=1e-15)
    # far arguments: silu(x) = x for x >> 0 and -|x| e^{-|x|} for x << 0, to
    # fp64 precision (the corrections are of order e^{-|x|})
    assert megakda.silu(300.0) == 300.0
    np.testing.assert_allclose(megakda.silu(-300.0), -300.0 * math.exp(-300.0), rtol=1e-14)


def test_short_conv_taps_pick_the_right_inputs():
    rng = np.random.default_rng(0)
    d = 5
    hist = rng.standard_normal((3, d))
    x = rng.standard_normal(d)
    for tap, want in ((3, x), (2, hist[2]), (1, hist[1]), (0, hist[0])):
        w = np.zeros((d, 4))
        w[:, tap] = 1.0
        y, new = megakda.short_conv_step(hist, x, w)
        np.testing.assert_allclose(y, want / (1 + np.exp(-want)), rtol=0, atol=1e-15)
        np.testing.assert_array_equal(new, np.stack([hist[1], hist[2], x]))
    # a causal moving sum: w = 1 on every tap
    y, _ = megakda.short_conv_step(hist, x, np.ones((d, 4)))
    s = hist.sum(0) + x
    np.testing.assert_allclose(y, s / (1 + np.exp(-s)), rtol=1e-15)


def test_rms_norm_gate_closed_forms():
    w = np.array([1.0, 2.0, -0.5, 4.0])
    # a constant vector c 1 with eps = 0 normalises to 1 (c > 0)
    for c in (0.3, 7.0):
        o = np.full(4, c)
        np.testing.assert_allclose(megakda.rms_norm_gate(o, np.zeros(4), w, 0.0), 0.5 * w, rtol=1e-15)
    # the rms of (3, 4, 0, 0) is 5 / 2; sigmoid(log 3) = 3/4
    o = np.array([3.0, 4.0, 0.0, 0.0])
    z = np.full(4, math.log(3.0))
    np.testing.assert_allclose(megakda.rms_norm_gate(o, z, np.ones(4), 0.0),
                               o / 2.5 * 0.75, rtol=1e-15)
    # scale invariance up to eps
    o = np.random.default_rng(1).standard_normal(6)
    a = megakda.rms_norm_gate(o, np.zeros(6), np.ones(6), 0.0)
    b = megakda.rms_norm_gate(17.0 * o, np.zeros(6), np.ones(6), 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-14)


def _brute_decode_fused(q, k, v, g, b, z, wq, wk, wv, wo, slots, pool, cpool, eps, eps_o, scale):
    """Scalar loops over every element, written separately from the oracle."""
    B, H, dk = len(q), len(q[0]), len(q[0][0])
    dv = len(v[0][0])
    pool = [[[list(r) for r in pool[s][h]] for h in range(H)] for s in range(len(pool))]
    cpool = [[[list(r) for r in cpool[s][h]] for h in range(H)] for s in range(len(cpool))]
    out = [[[0.0] * dv for _ in range(H)] for _ in range(B)]
    for n in range(B):
        s = slots[n]
        for h in range(H):
            hist = cpool[s][h]

            def conv(col, x, w):
                acc = w[3] * x
                for t in range(3):
                    acc += w[t] * hist[t][col]
                return acc / (1.0 + math.exp(-acc))
            qc = [conv(c, q[n][h][c], wq[h][c]) for c in range(dk)]
            kc = [conv(dk + c, k[n][h][c], wk[h][c]) for c in range(dk)]
            vc = [conv(2 * dk + i, v[n][h][i], wv[h][i]) for i in range(dv)]
            raw = list(q[n][h]) + list(k[n][h]) + list(v[n][h])
            cpool[s][h] = [hist[1], hist[2], raw]
            nq = math.sqrt(sum(x * x for x in qc) + eps)
            nk = math.sqrt(sum(x * x for x in kc) + eps)
            qh = [x / nq for x in qc]
            kh = [x / nk for x in kc]
            beta = 1.0 / (1.0 + math.exp(-b[n][h]))
            S = pool[s][h]
            o = []
            for i in range(dv):
                row = [S[i][c] * math.exp(g[n][h][c]) for c in range(dk)]
                r = sum(row[c] * kh[c] for c in range(dk))
                u = beta * (vc[i] - r)
                row = [row[c] + u * kh[c] for c in range(dk)]
                S[i] = row
                o.append(scale * sum(row[c] * qh[c] for c in range(dk)))
            rms = math.sqrt(sum(x * x for x in o) / dv + eps_o)
            out[n][h] = [o[i] / rms * wo[i] / (1.0 + math.exp(-z[n][h][i])) for i in range(dv)]
    return out, pool, cpool


def test_decode_fused_matches_brute_force():
    rng = np.random.default_rng(2)
    B, H, dk, dv, S = 2, 2, 4, 3, 3
    q, k = rng.standard_normal((B, H, dk)), rng.standard_normal((B, H, dk))
    v, z = rng.standard_normal((B, H, dv)), rng.standard_normal((B, H, dv))
    g = -np.abs(rng.standard_normal((B, H, dk))) * 0.3
    b = rng.standard_normal((B, H))
    wq, wk = rng.standard_normal((H, dk, 4)), rng.standard_normal((H, dk, 4))
    wv, wo = rng.standard_normal((H, dv, 4)), rng.standard_normal(dv)
    pool = rng.standard_normal((S, H, dv, dk)) * 0.3
    cpool = rng.standard_normal((S, H, 3, 2 * dk + dv))
    slots = np.array([2, 0], dtype=np.int32)
    scale = dk ** -0.5
    out, P, C, err = megakda.decode_fused(q, k, v, g, b, z, wq, wk, wv, wo, slots, pool, cpool,
                                          eps=1e-6, eps_o=1e-5, scale=scale)
    assert err == 0
    bo, bp, bc = _brute_decode_fused(q.tolist(), k.tolist(), v.tolist(), g.tolist(), b.tolist(),
                                     z.tolist(), wq.tolist(), wk.tolist(), wv.tolist(), wo.tolist(),
                                     slots.tolist(), pool.tolist(), cpool.tolist(), 1e-6, 1e-5, scale)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(P, np.array(bp), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(C, np.array(bc), rtol=0, atol=0)
    # slot 1 is named by nobody: both pools keep it
    np.testing.assert_array_equal(P[1], pool[1])
    np.testing.assert_array_equal(C[1], cpool[1])


def test_prefill_fused_equals_sequential_fused_decodes():
    """A fused prefill of a sequence equals its tokens fed one by one to the
    fused decode (the conv history carried through the conv state, the KDA
    state through the pool): outputs, final state and final conv state.
    Sequences of 5, 2 (shorter than the conv history), 0 and 4 tokens, one
    of them padding; the prefill starts from the pools."""
    rng = np.random.default_rng(7)
    H, dk, dv, S = 2, 4, 3, 5
    lens = [5, 2, 0, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    q, k = rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dk))
    v, z = rng.standard_normal((T, H, dv)), rng.standard_normal((T, H, dv))
    g = -np.abs(rng.standard_normal((T, H, dk))) * 0.3
    b = rng.standard_normal((T, H))
    wq, wk = rng.standard_normal((H, dk, 4)), rng.standard_normal((H, dk, 4))
    wv, wo = rng.standard_normal((H, dv, 4)), rng.standard_normal(dv)
    pool = rng.standard_normal((S, H, dv, dk)) * 0.3
    cpool = rng.standard_normal((S, H, 3, 2 * dk + dv))
    slots = np.array([3, 0, 4, -1], dtype=np.int32)
    out, P, C, err = megakda.prefill_fused(q, k, v, g, b, z, wq, wk, wv, wo, cu, slots, pool, cpool,
                                           init_from_pool=True, eps_o=1e-5)
    assert err == 0
    P2, C2 = pool.copy(), cpool.copy()
    for s, L in enumerate(lens):
        for t in range(cu[s], cu[s] + L):
            sel = lambda a: a[t:t + 1]  # noqa: E731
            o1, P2, C2, e = megakda.decode_fused(sel(q), sel(k), sel(v), sel(g), sel(b), sel(z),
                                                 wq, wk, wv, wo, slots[s:s + 1], P2, C2, eps_o=1e-5)
            np.testing.assert_allclose(out[t], o1[0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(P, P2, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(C, C2)
    assert np.all(out[cu[3]:cu[4]] == 0)


def test_prefill_fused_from_zero_history():
    """Without init_from_pool the conv history and the state start at zero:
    the first token's conv output is silu(w3 x) and the new conv state of a
    two-token sequence is [0, x0, x1]."""
    rng = np.random.default_rng(8)
    H, dk, dv = 1, 4, 3
    q, k = rng.standard_normal((2, H, dk)), rng.standard_normal((2, H, dk))
    v, z = rng.standard_normal((2, H, dv)), rng.standard_normal((2, H, dv))
    g = -np.abs(rng.standard_normal((2, H, dk)))
    b = rng.standard_normal((2, H))
    wq, wk = rng.standard_normal((H, dk, 4)), rng.standard_normal((H, dk, 4))
    wv, wo = rng.standard_normal((H, dv, 4)), np.ones(dv)
    cpool = rng.standard_normal((1, H, 3, 2 * dk + dv))
    out, P, C, err = megakda.prefill_fused(q, k, v, g, b, z, wq, wk, wv, wo, [0, 2],
                                           np.array([0], np.int32), np.zeros((1, H, dv, dk)), cpool)
    raw = np.concatenate([q[:, 0], k[:, 0], v[:, 0]], axis=1)
    np.testing.assert_array_equal(C[0, 0], np.stack([np.zeros(2 * dk + dv), raw[0], raw[1]]))
    # token 0 alone: the zero state makes o = scale beta (k^.q^) v~ with the
    # convolved inputs silu(w3 x)
    qc = megakda.silu(wq[0, :, 3] * q[0, 0])
    kc = megakda.silu(wk[0, :, 3] * k[0, 0])
    vc = megakda.silu(wv[0, :, 3] * v[0, 0])
    qh = qc / np.sqrt(qc @ qc + 1e-6)
    kh = kc / np.sqrt(kc @ kc + 1e-6)
    o = dk ** -0.5 * (1 / (1 + np.exp(-b[0, 0]))) * (kh @ qh) * vc
    np.testing.assert_allclose(out[0, 0], megakda.rms_norm_gate(o, z[0, 0], wo, 1e-6), rtol=1e-12)
