"""fp64 oracle of the MegaKDA-style fusion around the decode recurrence.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the test
suite, the smoke check and the benchmark's CPU-baseline leg use it, and it
shares nothing with the CUDA path.

"2.8x faster Kimi K3 inference on CANN", section 03 "MegaKDA": one operator
fuses the input side (projection and ShortConv) and the output-side compute
with the KDA recurrence.  The page gives no formulas; the readings taken:

  ShortConv  a causal depthwise convolution along the token axis, width 4,
             one weight vector per channel, followed by SiLU:
               y_t[c] = silu( sum_{i=0..3} w[c][i] x_{t-3+i}[c] )
             applied to q, k and v separately.  The three inputs before the
             current token come from the sequence's conv state (its last
             three raw inputs, oldest first), which the step then shifts.
  output     o' = o / sqrt(mean_i o_i^2 + eps_o) * w_o * sigmoid(z): an RMS
             norm over the head's dv outputs, a per-channel weight, and a
             sigmoid gate whose pre-activation z the caller supplies.

The projections are not part of it (they need trained weights): the conv
weights, w_o and z are inputs.  The recurrence itself is the C oracle's.

For a prefill the same ShortConv runs along each sequence: the history of
its first token is the slot's conv state when the prefill starts from the
pool, else zero, and the slot's conv state afterwards holds the last three
raw inputs of that history followed by the sequence.
"""
from __future__ import annotations

import numpy as np

from . import _f64, _i32, decode as _decode, prefill as _prefill

CONV_WIDTH = 4


def silu(x):
    x = np.asarray(x, np.float64)
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, np.float64)))


def short_conv_step(hist, x, w):
    """One token of the causal depthwise conv.

    hist: [3, d] the previous three raw inputs, oldest first; x: [d];
    w: [d, 4] (tap 0 multiplies the oldest input, tap 3 the current one).
    Returns (silu(conv) [d], the shifted history [3, d]).
    """
    hist = np.asarray(hist, np.float64)
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    win = np.concatenate([hist, x[None, :]], axis=0)  # [4, d], oldest first
    y = silu(np.einsum("td,dt->d", win, w))
    return y, win[1:]


def rms_norm_gate(o, z, w_o, eps_o):
    """o [.., dv] -> o / sqrt(mean(o^2) + eps_o) * w_o * sigmoid(z)."""
    o = np.asarray(o, np.float64)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return o / np.sqrt(ms + eps_o) * np.asarray(w_o, np.float64) * sigmoid(z)


def decode_fused(q, k, v, g, b, z, wq, wk, wv, w_o, slot_ids, pool, conv_pool,
                 eps: float = 1e-6, eps_o: float = 1e-6, scale=None):
    """One fused decode token per sequence.

    q, k: [B, H, dk]; v, z: [B, H, dv]; g: [B, H, dk]; b: [B, H];
    wq, wk: [H, dk, 4]; wv: [H, dv, 4]; w_o: [dv];
    pool: [S, H, dv, dk]; conv_pool: [S, H, 3, 2 dk + dv] (q, k, v channels).
    Returns (out [B, H, dv], new pool, new conv_pool, errors).  Padding
    entries (slot < 0) and errors (slot >= S) leave both pools alone and
    output zero.
    """
    q, k, v, g, b, z = (_f64(t) for t in (q, k, v, g, b, z))
    wq, wk, wv, w_o = (_f64(t) for t in (wq, wk, wv, w_o))
    slots = _i32(slot_ids)
    cpool = _f64(conv_pool).copy()
    B, H, dk = k.shape
    dv = v.shape[2]
    qc, kc, vc = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for n in range(B):
        sl = int(slots[n])
        if sl < 0 or sl >= cpool.shape[0]:
            continue
        for h in range(H):
            hist = cpool[sl, h]
            qc[n, h], hq = short_conv_step(hist[:, :dk], q[n, h], wq[h])
            kc[n, h], hk = short_conv_step(hist[:, dk:2 * dk], k[n, h], wk[h])
            vc[n, h], hv = short_conv_step(hist[:, 2 * dk:], v[n, h], wv[h])
            cpool[sl, h] = np.concatenate([hq, hk, hv], axis=1)
    o, P, err = _decode(qc, kc, vc, g, b, slots, pool, eps=eps, scale=scale)
    out = rms_norm_gate(o, z, w_o, eps_o)
    for n in range(B):
        sl = int(slots[n])
        if sl < 0 or sl >= cpool.shape[0]:
            out[n] = 0.0
    return out, P, cpool, err


def prefill_fused(q, k, v, g, b, z, wq, wk, wv, w_o, cu_seqlens, slot_ids, pool, conv_pool,
                  init_from_pool=False, eps: float = 1e-6, eps_o: float = 1e-6, scale=None):
    """Fused prefill of a variable-length batch.

    q, k, g: [T, H, dk]; v, z: [T, H, dv]; b: [T, H]; cu_seqlens: [n+1];
    conv_pool: [S, H, 3, 2 dk + dv].  Returns (out [T, H, dv], new pool,
    new conv_pool, errors).  Padding and out-of-range sequences output zero
    and leave both pools alone.
    """
    q, k, v, g, b, z = (_f64(t) for t in (q, k, v, g, b, z))
    wq, wk, wv, w_o = (_f64(t) for t in (wq, wk, wv, w_o))
    cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    slots = _i32(slot_ids)
    cpool = _f64(conv_pool).copy()
    T, H, dk = k.shape
    dv = v.shape[2]
    qc, kc, vc = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s in range(len(cu) - 1):
        sl = int(slots[s])
        if sl < 0 or sl >= cpool.shape[0]:
            continue
        a, e = cu[s], cu[s + 1]
        for h in range(H):
            hist = cpool[sl, h].copy() if init_from_pool else np.zeros((3, 2 * dk + dv))
            # the raw inputs of the sequence after its three-token history
            x = np.concatenate([hist, np.concatenate([q[a:e, h], k[a:e, h], v[a:e, h]], axis=1)])
            w = np.concatenate([wq[h], wk[h], wv[h]])          # [2 dk + dv, 4]
            L = e - a
            # y_t = silu(sum_i w[:, i] x_{t-3+i}): window i of x starts at row i
            y = silu(sum(w[:, i] * x[i:i + L] for i in range(4)))
            qc[a:e, h], kc[a:e, h], vc[a:e, h] = y[:, :dk], y[:, dk:2 * dk], y[:, 2 * dk:]
            cpool[sl, h] = x[-3:]
    o, P, err = _prefill(qc, kc, vc, g, b, cu, slots, pool, init_from_pool=init_from_pool,
                         eps=eps, scale=scale)
    out = rms_norm_gate(o, z, w_o, eps_o)
    for s in range(len(cu) - 1):
        sl = int(slots[s])
        if sl < 0 or sl >= cpool.shape[0]:
            out[cu[s]:cu[s + 1]] = 0.0
    return out, P, cpool, err
