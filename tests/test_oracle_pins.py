"""Pins for the fp64 oracle: checks against things other than the oracle itself.

The pages print no numeric KDA example, so the oracle is pinned by
  * hand-derived worked examples (tests/golden/kda_worked_examples_2x2.json),
  * closed forms (first token from a zero state),
  * exact rational brute force on tiny inputs (fractions.Fraction),
  * an independent matrix form of the transition,
    S_t = S_{t-1} diag(alpha) (I - beta k^ k^T) + beta v k^T,
  * invariants of the method (beta = 0, beta = 1, contraction, symmetry),
  * agreement of the record/replay and chunked re-associations with the
    token loop.
A mutation test (test_oracle_mutants.py) shows that plausible mistakes in
the oracle fail these pins.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import chunk_form

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "kda_worked_examples_2x2.json")


def _unit_rows(rng, n, d):
    x = rng.standard_normal((n, d))
    return x


# --------------------------------------------------------------- worked examples

def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c["name"])
def test_golden_worked_examples(case):
    toks = case["tokens"]
    q = np.array([t["q"] for t in toks], float)
    k = np.array([t["k"] for t in toks], float)
    v = np.array([t["v"] for t in toks], float)
    g = np.array([t["g"] for t in toks], float)
    b = np.array([t["b"] for t in toks], float)
    o, S = oracle.recurrence(q, k, v, g, b, S0=np.array(case["S0"], float),
                             eps=case["eps"], scale=1 / math.sqrt(2))
    np.testing.assert_allclose(o * math.sqrt(2), case["expected_o_times_sqrt2"],
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, case["expected_S"], rtol=0, atol=1e-12)


def test_golden_through_pool_decode():
    """The second worked example through the slot-addressed pool entry."""
    case = load_golden()[1]
    t = case["tokens"][0]
    rng = np.random.default_rng(7)
    pool = rng.standard_normal((3, 1, 2, 2))
    pool[1, 0] = np.array(case["S0"], float)
    before = pool.copy()
    out, new_pool, err = oracle.decode(
        np.array(t["q"], float).reshape(1, 1, 2),
        np.array(t["k"], float).reshape(1, 1, 2),
        np.array(t["v"], float).reshape(1, 1, 2),
        np.array(t["g"], float).reshape(1, 1, 2),
        np.array([[t["b"]]], float), np.array([1], np.int32), pool,
        eps=0.0, scale=1 / math.sqrt(2))
    assert err == 0
    np.testing.assert_allclose(out[0, 0] * math.sqrt(2),
                               case["expected_o_times_sqrt2"][0], atol=1e-12)
    np.testing.assert_allclose(new_pool[1, 0], case["expected_S"], atol=1e-12)
    # untouched slots are bit-identical
    assert np.array_equal(new_pool[0], before[0])
    assert np.array_equal(new_pool[2], before[2])
    assert np.array_equal(pool, before)  # the input pool is not modified


# --------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dk,dv", [(16, 16), (8, 24), (32, 8)])
def test_first_token_closed_form(dk, dv):
    """From S0 = 0: S1 = beta v k^T and o1 = dk^-1/2 beta (k^.q^) v."""
    rng = np.random.default_rng(dk * 100 + dv)
    q, k = rng.standard_normal((1, dk)), rng.standard_normal((1, dk))
    v = rng.standard_normal((1, dv))
    g = np.log(1 / (1 + np.exp(-rng.standard_normal((1, dk)) - 2)))
    b = rng.standard_normal(1)
    eps = 1e-6
    o, S = oracle.recurrence(q, k, v, g, b, eps=eps)
    kh = k[0] / math.sqrt((k[0] ** 2).sum() + eps)
    qh = q[0] / math.sqrt((q[0] ** 2).sum() + eps)
    beta = 1 / (1 + math.exp(-b[0]))
    np.testing.assert_allclose(S, beta * np.outer(v[0], kh), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o[0], dk ** -0.5 * beta * kh.dot(qh) * v[0],
                               rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------- exact brute force

# rational unit vectors (Pythagorean tuples): normalisation with eps = 0 is exact
_UNIT = {
    2: [(3, 4, 5), (5, 12, 13), (8, 15, 17), (1, 0, 1)],
    3: [(1, 2, 2, 3), (2, 3, 6, 7), (2, 6, 9, 11), (0, 0, 1, 1)],
    4: [(1, 1, 1, 1, 2), (1, 2, 2, 4, 5), (2, 4, 5, 6, 9), (1, 0, 0, 0, 1)],
}


def _rational_unit(rng, d):
    tup = _UNIT[d][rng.integers(len(_UNIT[d]))]
    comps, n = list(tup[:-1]), tup[-1]
    rng.shuffle(comps)
    signs = rng.choice([-1, 1], size=d)
    return [Fraction(int(s) * c, n) for s, c in zip(signs, comps)]


def _fraction_recurrence(S, toks, scale):
    """Exact rational token loop (independent of the oracle's C code)."""
    dv, dk = len(S), len(S[0])
    outs = []
    for q, k, v, alpha, beta in toks:
        S = [[S[i][c] * alpha[c] for c in range(dk)] for i in range(dv)]
        r = [sum(S[i][c] * k[c] for c in range(dk)) for i in range(dv)]
        u = [beta * (v[i] - r[i]) for i in range(dv)]
        S = [[S[i][c] + u[i] * k[c] for c in range(dk)] for i in range(dv)]
        outs.append([sum(S[i][c] * q[c] for c in range(dk)) for i in range(dv)])
    return outs, S


@pytest.mark.parametrize("d", [2, 3, 4])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fraction_bruteforce(d, seed):
    rng = np.random.default_rng(seed * 10 + d)
    dk = dv = d
    n = 6
    alphas = [Fraction(1), Fraction(1, 2), Fraction(3, 4), Fraction(7, 8)]
    betas = [Fraction(1, 2), Fraction(3, 4), Fraction(1, 4), Fraction(9, 10)]
    toks = []
    for _ in range(n):
        q = _rational_unit(rng, dk)
        k = _rational_unit(rng, dk)
        v = [Fraction(int(x), 4) for x in rng.integers(-8, 9, size=dv)]
        alpha = [alphas[i] for i in rng.integers(len(alphas), size=dk)]
        beta = betas[rng.integers(len(betas))]
        toks.append((q, k, v, alpha, beta))
    S0 = [[Fraction(int(x), 8) for x in rng.integers(-8, 9, size=dk)] for _ in range(dv)]
    outs, S = _fraction_recurrence(S0, toks, None)
    scale = 0.5  # passed explicitly; the exact outputs are multiplied by it
    q = np.array([[float(x) for x in t[0]] for t in toks])
    k = np.array([[float(x) for x in t[1]] for t in toks])
    v = np.array([[float(x) for x in t[2]] for t in toks])
    g = np.array([[math.log(float(a)) for a in t[3]] for t in toks])
    b = np.array([math.log(float(t[4]) / (1 - float(t[4]))) for t in toks])
    o, Sf = oracle.recurrence(q, k, v, g, b, S0=np.array(S0, float), eps=0.0,
                              scale=scale)
    np.testing.assert_allclose(o, scale * np.array(outs, float), rtol=0, atol=1e-13)
    np.testing.assert_allclose(Sf, np.array(S, float), rtol=0, atol=1e-13)


# --------------------------------------------------------------- matrix form

def _random_tokens(rng, n, dk, dv, g_mean=2.0):
    q = rng.standard_normal((n, dk))
    k = rng.standard_normal((n, dk))
    v = rng.standard_normal((n, dv))
    g = -np.log1p(np.exp(-(rng.standard_normal((n, dk)) + g_mean)))
    b = rng.standard_normal(n)
    return q, k, v, g, b


@pytest.mark.parametrize("dk,dv", [(24, 16), (16, 24), (32, 32)])
def test_matrix_form(dk, dv):
    """S_t = S_{t-1} diag(alpha_t) (I - beta_t k^ k^T) + beta_t v_t k^_t^T."""
    rng = np.random.default_rng(dk + 7 * dv)
    n, eps = 50, 1e-6
    q, k, v, g, b = _random_tokens(rng, n, dk, dv)
    S0 = 0.1 * rng.standard_normal((dv, dk))
    o, Sf = oracle.recurrence(q, k, v, g, b, S0=S0, eps=eps)
    S = S0.copy()
    for t in range(n):
        kh = k[t] / np.sqrt(k[t] @ k[t] + eps)
        qh = q[t] / np.sqrt(q[t] @ q[t] + eps)
        beta = 1 / (1 + np.exp(-b[t]))
        S = S @ np.diag(np.exp(g[t])) @ (np.eye(dk) - beta * np.outer(kh, kh)) \
            + beta * np.outer(v[t], kh)
        np.testing.assert_allclose(o[t], dk ** -0.5 * S @ qh, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(Sf, S, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------- invariants

def test_beta_zero_no_decay_leaves_state_bitwise():
    rng = np.random.default_rng(3)
    dk, dv, n = 16, 8, 5
    q, k, v, _, _ = _random_tokens(rng, n, dk, dv)
    g = np.zeros((n, dk))
    b = np.full(n, -np.inf)
    S0 = rng.standard_normal((dv, dk))
    _, S = oracle.recurrence(q, k, v, g, b, S0=S0)
    assert np.array_equal(S, S0)


def test_beta_one_writes_value_at_key():
    """With beta = 1 the updated state maps k^_t exactly to v_t."""
    rng = np.random.default_rng(4)
    dk, dv = 32, 16
    S = rng.standard_normal((dv, dk))
    for t in range(6):
        q, k, v, g, _ = _random_tokens(rng, 1, dk, dv)
        _, S = oracle.recurrence(q, k, v, g, np.array([np.inf]), S0=S, eps=0.0)
        kh = k[0] / np.linalg.norm(k[0])
        np.testing.assert_allclose(S @ kh, v[0], rtol=1e-12, atol=1e-12)


def test_transition_is_contractive():
    """With v = 0, alpha <= 1, 0 <= beta <= 1 the spectral norm never grows."""
    rng = np.random.default_rng(5)
    dk, dv = 16, 16
    S = rng.standard_normal((dv, dk))
    for t in range(20):
        q, k, _, g, b = _random_tokens(rng, 1, dk, dv)
        before = np.linalg.norm(S, 2)
        _, S = oracle.recurrence(q, k, np.zeros((1, dv)), g, b, S0=S)
        assert np.linalg.norm(S, 2) <= before * (1 + 1e-12)


def test_scale_invariance_of_q_and_k():
    rng = np.random.default_rng(6)
    dk, dv, n = 16, 8, 12
    q, k, v, g, b = _random_tokens(rng, n, dk, dv)
    o1, S1 = oracle.recurrence(q, k, v, g, b, eps=0.0)
    o2, S2 = oracle.recurrence(3.5 * q, 0.25 * k, v, g, b, eps=0.0)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S1, S2, rtol=1e-12, atol=1e-13)


def test_channel_permutation_equivariance():
    """Permuting value channels permutes outputs and state rows; permuting key
    channels (q, k, g and state columns together) changes nothing else."""
    rng = np.random.default_rng(8)
    dk, dv, n = 12, 10, 9
    q, k, v, g, b = _random_tokens(rng, n, dk, dv)
    S0 = rng.standard_normal((dv, dk))
    o, S = oracle.recurrence(q, k, v, g, b, S0=S0)
    pv, pk = rng.permutation(dv), rng.permutation(dk)
    o2, S2 = oracle.recurrence(q[:, pk], k[:, pk], v[:, pv], g[:, pk], b,
                               S0=S0[pv][:, pk])
    np.testing.assert_allclose(o2, o[:, pv], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S2, S[pv][:, pk], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------- decode / verify / replay

def _pool_case(rng, B, H, dk, dv, num_slots):
    pool = 0.3 * rng.standard_normal((num_slots, H, dv, dk))
    slots = rng.permutation(num_slots)[:B].astype(np.int32)
    return pool, slots


def test_decode_matches_recurrence_and_padding_rules():
    rng = np.random.default_rng(11)
    B, H, dk, dv, NS = 5, 3, 16, 8, 9
    pool, slots = _pool_case(rng, B, H, dk, dv, NS)
    slots[1] = -1          # padding
    slots[3] = NS + 2      # out of range
    q = rng.standard_normal((B, H, dk))
    k = rng.standard_normal((B, H, dk))
    v = rng.standard_normal((B, H, dv))
    g = -np.log1p(np.exp(-(rng.standard_normal((B, H, dk)) + 3)))
    b = rng.standard_normal((B, H))
    out, P, err = oracle.decode(q, k, v, g, b, slots, pool)
    assert err == H  # one error per head of the out-of-range sequence
    touched = set()
    for n in range(B):
        for h in range(H):
            if slots[n] < 0 or slots[n] >= NS:
                assert np.all(out[n, h] == 0)
                continue
            touched.add(int(slots[n]))
            o, S = oracle.recurrence(q[n, h][None], k[n, h][None], v[n, h][None],
                                     g[n, h][None], b[n, h][None], S0=pool[slots[n], h])
            np.testing.assert_array_equal(out[n, h], o[0])
            np.testing.assert_array_equal(P[slots[n], h], S)
    for s in range(NS):
        if s not in touched:
            assert np.array_equal(P[s], pool[s])


def _draft(rng, B, D, H, dk, dv, g_mean=3.0):
    q = rng.standard_normal((B, D, H, dk))
    k = rng.standard_normal((B, D, H, dk))
    v = rng.standard_normal((B, D, H, dv))
    g = -np.log1p(np.exp(-(rng.standard_normal((B, D, H, dk)) + g_mean)))
    b = rng.standard_normal((B, D, H))
    return q, k, v, g, b


def test_verify_equals_sequential_decode_and_keeps_pool():
    rng = np.random.default_rng(12)
    B, D, H, dk, dv, NS = 3, 7, 2, 16, 16, 6
    pool, slots = _pool_case(rng, B, H, dk, dv, NS)
    q, k, v, g, b = _draft(rng, B, D, H, dk, dv)
    out, rec, err = oracle.verify(q, k, v, g, b, slots, pool)
    assert err == 0
    P = pool.copy()
    for j in range(D):
        oj, P, _ = oracle.decode(q[:, j], k[:, j], v[:, j], g[:, j], b[:, j], slots, P)
        np.testing.assert_array_equal(out[:, j], oj)
    # the records are the token's normalised key, value, gate and beta
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(rec["k_hat"], kn, rtol=1e-15, atol=1e-16)
    np.testing.assert_array_equal(rec["v"], v)
    np.testing.assert_array_equal(rec["g"], g)
    np.testing.assert_allclose(rec["beta"], 1 / (1 + np.exp(-b)), rtol=1e-15)


@pytest.mark.parametrize("seed", [0, 1])
def test_replay_equals_recurrence_on_accepted_prefix(seed):
    rng = np.random.default_rng(20 + seed)
    B, D, H, dk, dv, NS = 6, 7, 2, 16, 8, 10
    pool, slots = _pool_case(rng, B, H, dk, dv, NS)
    q, k, v, g, b = _draft(rng, B, D, H, dk, dv)
    acc = np.array([0, 1, 3, 7, 5, 2], np.int32)
    _, rec, _ = oracle.verify(q, k, v, g, b, slots, pool)
    P, err = oracle.replay(rec, acc, slots, pool)
    assert err == 0
    for n in range(B):
        for h in range(H):
            a = acc[n]
            if a == 0:
                assert np.array_equal(P[slots[n], h], pool[slots[n], h])
                continue
            _, S = oracle.recurrence(q[n, :a, h], k[n, :a, h], v[n, :a, h],
                                     g[n, :a, h], b[n, :a, h], S0=pool[slots[n], h])
            np.testing.assert_allclose(P[slots[n], h], S, rtol=1e-13, atol=1e-15)


def test_replay_rejects_bad_lengths_and_slots():
    rng = np.random.default_rng(30)
    B, D, H, dk, dv, NS = 3, 4, 1, 8, 8, 4
    pool, slots = _pool_case(rng, B, H, dk, dv, NS)
    q, k, v, g, b = _draft(rng, B, D, H, dk, dv)
    _, rec, _ = oracle.verify(q, k, v, g, b, slots, pool)
    acc = np.array([D + 1, 2, 1], np.int32)
    slots2 = slots.copy()
    slots2[2] = NS
    P, err = oracle.replay(rec, acc, slots2, pool)
    assert err == 2
    assert np.array_equal(P[slots[0]], pool[slots[0]])
    assert not np.array_equal(P[slots[1]], pool[slots[1]])


# --------------------------------------------------------------- chunked form

@pytest.mark.parametrize("T", [1, 63, 64, 65, 150])
def test_chunk_form_equals_recurrence(T):
    rng = np.random.default_rng(T)
    dk, dv = 32, 24
    q, k, v, g, b = _random_tokens(rng, T, dk, dv, g_mean=3.0)
    S0 = 0.2 * rng.standard_normal((dv, dk))
    o_ref, S_ref = oracle.recurrence(q, k, v, g, b, S0=S0)
    o_c, S_c = chunk_form.prefill(q, k, v, g, b, S0=S0, chunk=64)
    np.testing.assert_allclose(o_c, o_ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S_c, S_ref, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("L", [64, 37])
def test_chunk_step_split_equals_chunk_step(L):
    """The state-independent split of the chunk step (G = W^T K^, Q' = Q~ - P W)
    is the same map as the U form, on a full and a partial chunk."""
    rng = np.random.default_rng(100 + L)
    dk, dv = 32, 24
    q, k, v, g, b = _random_tokens(rng, L, dk, dv, g_mean=3.0)
    S0 = 0.3 * rng.standard_normal((dv, dk))
    inter = chunk_form.chunk_intermediates(q, k, v, g, b)
    o1, s1 = chunk_form.chunk_step(S0, inter, dk ** -0.5)
    o2, s2 = chunk_form.chunk_step_split(S0, inter, dk ** -0.5)
    np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s2, s1, rtol=1e-11, atol=1e-13)
    # and both are the token loop
    o_ref, s_ref = oracle.recurrence(q, k, v, g, b, S0=S0)
    np.testing.assert_allclose(o2, o_ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(s2, s_ref, rtol=1e-9, atol=1e-11)


def test_chunk_form_strong_decay():
    """Large per-token decay (alpha ~ e^-3) stays finite and equal to the loop."""
    rng = np.random.default_rng(99)
    T, dk, dv = 130, 16, 16
    q, k, v, g, b = _random_tokens(rng, T, dk, dv, g_mean=-3.0)
    o_ref, S_ref = oracle.recurrence(q, k, v, g, b)
    o_c, S_c = chunk_form.prefill(q, k, v, g, b, chunk=64)
    np.testing.assert_allclose(o_c, o_ref, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(S_c, S_ref, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("D,g_mean", [(1, 3.0), (7, 3.0), (8, 3.0), (8, -6.0), (16, 0.0)])
@pytest.mark.parametrize("factored", [False, True])
def test_verify_window_form_equals_token_loop(D, g_mean, factored):
    """The draft-window chunk form (running or factored window products)
    equals the oracle's token-by-token verify on one (sequence, head)."""
    rng = np.random.default_rng(200 + D)
    dk, dv, NS = 16, 12, 3
    pool = 0.3 * rng.standard_normal((NS, 1, dv, dk))
    slots = np.array([2], np.int32)
    q, k, v, g, b = _draft(rng, 1, D, 1, dk, dv, g_mean=g_mean)
    o_ref, _, err = oracle.verify(q, k, v, g, b, slots, pool)
    assert err == 0
    o_w = chunk_form.verify_window(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], b[0, :, 0],
                                   pool[2, 0], factored=factored)
    np.testing.assert_allclose(o_w, o_ref[0, :, 0], rtol=1e-9, atol=1e-11)


def test_prefill_varlen_matches_recurrence():
    rng = np.random.default_rng(41)
    lens = [5, 0, 70, 64]
    H, dk, dv, NS = 2, 16, 8, 7
    T = sum(lens)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -np.log1p(np.exp(-(rng.standard_normal((T, H, dk)) + 3)))
    b = rng.standard_normal((T, H))
    cu = np.cumsum([0] + lens)
    slots = np.array([4, 1, -1, 2], np.int32)
    pool = rng.standard_normal((NS, H, dv, dk))
    for init in (False, True):
        out, P, err = oracle.prefill(q, k, v, g, b, cu, slots, pool,
                                     init_from_pool=init)
        assert err == 0
        for s, L in enumerate(lens):
            t0, t1 = cu[s], cu[s + 1]
            if slots[s] < 0:
                assert np.all(out[t0:t1] == 0)
                continue
            for h in range(H):
                S0 = pool[slots[s], h] if init else None
                o, S = oracle.recurrence(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h],
                                         g[t0:t1, h], b[t0:t1, h], S0=S0)
                np.testing.assert_array_equal(out[t0:t1, h], o)
                np.testing.assert_array_equal(P[slots[s], h], S)
        for s in (0, 3, 5, 6):
            assert np.array_equal(P[s], pool[s])
