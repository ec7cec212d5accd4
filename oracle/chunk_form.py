"""fp64 chunk-form (WY/UT) restatement of the KDA recurrence, one (sequence, head).

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Ascend day-0 support for Kimi K3" (hwcomputing.csdn.net/6a695b59...),
section "Fused-operator acceleration: KDA Prefill and Decode dual path",
describes the prefill as 64-token chunks in which Q/K normalisation, gate
accumulation and the chunk KDA are organised as batched computation.  The
page gives no formulas; this module writes out the chunk form that follows
from unrolling the token recurrence inside one chunk, step by step, with no
blocking or fusion beyond that:

  gamma_r  = sum_{j<=r} g_j                         (in-chunk cumulative gate)
  A[r,j]   = beta_r sum_c k^_r[c] k^_j[c] e^{gamma_r[c]-gamma_j[c]},  j < r
  P[r,j]   =        sum_c q^_r[c] k^_j[c] e^{gamma_r[c]-gamma_j[c]},  j <= r
  T        = (I + A)^-1                             (UT transform)
  K~_r     = k^_r (.) e^{gamma_r},  Q~_r = q^_r (.) e^{gamma_r}
  W        = T diag(beta) K~,       U' = T diag(beta) V   (WY factors)
  U        = U' - W S0^T
  O        = scale (Q~ S0^T + P U)
  K^_j     = k^_j (.) e^{gamma_C - gamma_j}
  S_C      = S0 diag(e^{gamma_C}) + U^T K^

Derivation: inside a chunk S_r = S0 diag(e^{gamma_r}) + sum_{j<=r} u_j
(k^_j (.) e^{gamma_r - gamma_j})^T with u_r = beta_r (v_r - S'_r k^_r);
substituting S'_r gives (I + A) U = diag(beta) (V - K~ S0^T).

It exists to show that the chunked re-association equals the token loop in
exact arithmetic (to fp64 rounding), and to expose per-chunk intermediates.

The same unrolling over a ReplaySSM draft window ("2.8x faster Kimi K3
inference on CANN", section 04 "ReplaySSM": verify emits an output for every
draft token and never writes the state; the page does not say how the
outputs are formed) gives `verify_window`, starting from the committed state
S0 with E_j = prod_{l<=j} alpha_l:

  K~_j = k^_j (.) E_j,   Q~_j = q^_j (.) E_j
  a_jm = sum_c k^_m[c] k^_j[c] prod_{l=m+1..j} alpha_l[c]       (m < j)
  p_jm = sum_c k^_m[c] q^_j[c] prod_{l=m+1..j} alpha_l[c]       (m <= j)
  u_j  = beta_j (v_j - S0 K~_j - sum_{m<j} a_jm u_m)
  o_j  = scale (S0 Q~_j + sum_{m<=j} p_jm u_m)

and, since prod_{l=m+1..j} alpha_l = E_j / E_m, the factored products
a_jm = K~_j . (k^_m / E_m) and p_jm = Q~_j . (k^_m / E_m).
"""
from __future__ import annotations

import numpy as np


def _l2norm(x: np.ndarray, eps: float) -> np.ndarray:
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + eps)


def chunk_intermediates(q, k, v, g, b, eps: float = 1e-6):
    """State-independent quantities of one chunk (all fp64).

    q, k, g: [C, dk]; v: [C, dv]; b: [C].  Returns a dict with gamma, A, P,
    T, W, U_prime, Q_tilde, K_hat_end (the K^ above), and beta.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    b = np.asarray(b, np.float64)
    C = k.shape[0]
    qh = _l2norm(q, eps)
    kh = _l2norm(k, eps)
    beta = 1.0 / (1.0 + np.exp(-b))
    gamma = np.cumsum(g, axis=0)                       # [C, dk]
    diff = gamma[:, None, :] - gamma[None, :, :]       # [r, j, c]
    strict = np.tril(np.ones((C, C), bool), k=-1)
    lower = np.tril(np.ones((C, C), bool), k=0)
    # exp only where j <= r; elsewhere the entry is masked out anyway
    decay = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], diff, 0.0)), 0.0)
    A = beta[:, None] * np.einsum("rc,jc,rjc->rj", kh, kh, decay) * strict
    P = np.einsum("rc,jc,rjc->rj", qh, kh, decay) * lower
    T = np.linalg.inv(np.eye(C) + A)
    K_tilde = kh * np.exp(gamma)
    Q_tilde = qh * np.exp(gamma)
    W = T @ (beta[:, None] * K_tilde)
    U_prime = T @ (beta[:, None] * v)
    K_hat_end = kh * np.exp(gamma[-1][None, :] - gamma)
    return dict(gamma=gamma, A=A, P=P, T=T, W=W, U_prime=U_prime,
                Q_tilde=Q_tilde, K_hat_end=K_hat_end, beta=beta)


def chunk_step(S0, inter, scale: float):
    """Apply one chunk to state S0 [dv, dk]; returns (O [C, dv], S_C)."""
    U = inter["U_prime"] - inter["W"] @ S0.T
    O = scale * (inter["Q_tilde"] @ S0.T + inter["P"] @ U)
    S_C = S0 * np.exp(inter["gamma"][-1])[None, :] + U.T @ inter["K_hat_end"]
    return O, S_C


def chunk_step_split(S0, inter, scale: float):
    """The same chunk step with every state-independent product formed first.

    Substituting U = U' - W S0^T into the two uses of U gives
      S_C = S0 diag(e^{gamma_C}) + U'^T K^ - S0 G,   G = W^T K^  (dk x dk)
      O   = scale (Q' S0^T + P U'),                   Q' = Q~ - P W
    so that the only product that needs the incoming state is S0 [G; Q']
    (exact algebra: the result differs from chunk_step by rounding only).
    """
    G = inter["W"].T @ inter["K_hat_end"]
    Qp = inter["Q_tilde"] - inter["P"] @ inter["W"]
    O = scale * (Qp @ S0.T + inter["P"] @ inter["U_prime"])
    S_C = S0 * np.exp(inter["gamma"][-1])[None, :] + inter["U_prime"].T @ inter["K_hat_end"] - S0 @ G
    return O, S_C


def prefill(q, k, v, g, b, S0=None, chunk: int = 64, eps: float = 1e-6,
            scale=None):
    """Chunked prefill of one (sequence, head); the last chunk may be partial.

    q, k, g: [T, dk]; v: [T, dv]; b: [T].  Returns (O [T, dv], S_final).
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    scale = dk ** -0.5 if scale is None else scale
    S = np.zeros((dv, dk)) if S0 is None else np.array(S0, np.float64)
    O = np.zeros((T, dv))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        inter = chunk_intermediates(q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1],
                                    np.asarray(b)[c0:c1], eps)
        O[c0:c1], S = chunk_step(S, inter, scale)
    return O, S


def verify_window(q, k, v, g, b, S0, eps: float = 1e-6, scale=None,
                  factored: bool = False):
    """Draft-window outputs of one (sequence, head) from the committed state.

    q, k, g: [D, dk]; v: [D, dv]; b: [D]; S0: [dv, dk].  The window products
    are running products of alpha, or with ``factored`` the dot products
    K~_j . (k^_m / E_m).  Returns O [D, dv]; S0 is not changed.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    b = np.asarray(b, np.float64)
    S0 = np.asarray(S0, np.float64)
    D, dk = k.shape
    scale = dk ** -0.5 if scale is None else scale
    qh = _l2norm(q, eps)
    kh = _l2norm(k, eps)
    beta = 1.0 / (1.0 + np.exp(-b))
    alpha = np.exp(g)
    E = np.cumprod(alpha, axis=0)                      # [D, dk]
    K_tilde = kh * E
    Q_tilde = qh * E
    A = np.zeros((D, D))
    P = np.zeros((D, D))
    for j in range(D):
        for m in range(j + 1):
            if factored:
                w_k = kh[m] / E[m]
                a, pp = K_tilde[j] @ w_k, Q_tilde[j] @ w_k
            else:
                w = np.prod(alpha[m + 1:j + 1], axis=0)   # empty product = 1
                a, pp = (kh[m] * w) @ kh[j], (kh[m] * w) @ qh[j]
            if m < j:
                A[j, m] = a
            P[j, m] = pp
    U = np.zeros((D, S0.shape[0]))
    O = np.zeros((D, S0.shape[0]))
    for j in range(D):
        U[j] = beta[j] * (v[j] - S0 @ K_tilde[j] - A[j, :j] @ U[:j])
        O[j] = scale * (S0 @ Q_tilde[j] + P[j, :j + 1] @ U[:j + 1])
    return O
