"""Seeded synthetic inputs shaped like the KDA workloads.

This module draws random numbers and nothing else: it holds none of the
recurrence's arithmetic, so both the CUDA path and the fp64 oracle can be
fed from it.  Every draw goes through one ``torch.Generator`` per call, in a
fixed order (q, k, v, g, b, state pool, slot permutation, accepted lengths),
in fp32, then is rounded to the input dtype (round-to-nearest-even for bf16).

Distributions (the workloads of the decode, speculative-verify and prefill
paths): q, k, v ~ N(0, 1); g = log(sigmoid(x)) with x ~ N(g_mean, 1), drawn
per key channel and computed as -softplus(-x) in fp32; b ~ N(0, 1); state
pool ~ N(0, pool_std) with pool_std a standard deviation; slot ids are the
first B entries of a random permutation of the pool; accepted lengths are
uniform on 0..D.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


def _gen(seed: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return gen


def _normal(shape, gen, device, std=1.0, mean=0.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def log_sigmoid_gate(x: torch.Tensor) -> torch.Tensor:
    """g = log(sigmoid(x)) evaluated as -softplus(-x) in fp32."""
    return -torch.nn.functional.softplus(-x)


@dataclass
class DecodeInputs:
    q: torch.Tensor          # [B, H, dk] (input dtype)
    k: torch.Tensor          # [B, H, dk]
    v: torch.Tensor          # [B, H, dv]
    g: torch.Tensor          # [B, H, dk] fp32
    b: torch.Tensor          # [B, H] (input dtype)
    pool: torch.Tensor       # [num_slots, H, dv, dk] fp32
    slot_ids: torch.Tensor   # [B] int32


def decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=None, seed=0,
                  g_mean=3.0, pool_std=0.02, zero_state=False, device="cpu",
                  tokens=None):
    """Inputs for ``tokens`` decode steps (None: one step, no token axis).

    With ``tokens`` = n the per-token tensors gain a leading [n] axis.  When
    ``zero_state`` is set the slots named by slot_ids start at zero and every
    other slot holds N(0, 1) canary values.
    """
    num_slots = B if num_slots is None else num_slots
    gen = _gen(seed, device)
    dt = torch_dtype(dtype)
    lead = () if tokens is None else (tokens,)
    q = _normal(lead + (B, H, dk), gen, device).to(dt)
    k = _normal(lead + (B, H, dk), gen, device).to(dt)
    v = _normal(lead + (B, H, dv), gen, device).to(dt)
    g = log_sigmoid_gate(_normal(lead + (B, H, dk), gen, device, mean=g_mean))
    b = _normal(lead + (B, H), gen, device).to(dt)
    pool = _normal((num_slots, H, dv, dk), gen, device,
                   std=1.0 if zero_state else pool_std)
    perm = torch.randperm(num_slots, generator=gen, device=device)
    slot_ids = perm[:B].to(torch.int32)
    if zero_state:
        pool[slot_ids.long()] = 0.0
    return DecodeInputs(q, k, v, g, b, pool, slot_ids)


@dataclass
class FusedExtras:
    conv_state: torch.Tensor  # [num_slots, H, 3, 2 dk + dv] (input dtype)
    conv_w: torch.Tensor      # [H, 2 dk + dv, 4] fp32
    z: torch.Tensor           # [B, H, dv] (input dtype)
    norm_w: torch.Tensor      # [dv] fp32


def fused_extras(B, H, dk, dv, dtype="bf16", num_slots=None, seed=0, device="cpu"):
    """The fused decode's extra inputs, drawn after (and independently of)
    ``decode_inputs`` from their own generator: conv state ~ N(0, 1) (raw
    q/k/v-like inputs), conv taps ~ N(0, 0.5^2) (so that a width-4 conv of
    N(0, 1) inputs stays near unit variance), gate pre-activations
    z ~ N(0, 1), norm weight ~ N(1, 0.1^2)."""
    num_slots = B if num_slots is None else num_slots
    gen = _gen(seed + 7919, device)
    dt = torch_dtype(dtype)
    nc = 2 * dk + dv
    conv_state = _normal((num_slots, H, 3, nc), gen, device).to(dt)
    conv_w = _normal((H, nc, 4), gen, device, std=0.5)
    z = _normal((B, H, dv), gen, device).to(dt)
    norm_w = _normal((dv,), gen, device, std=0.1, mean=1.0)
    return FusedExtras(conv_state, conv_w, z, norm_w)


def fused_prefill_extras(T, n_seqs, H, dk, dv, dtype="bf16", num_slots=None, seed=0, device="cpu"):
    """The fused prefill's extra inputs: as ``fused_extras``, with z drawn per
    token ([T, H, dv])."""
    num_slots = n_seqs if num_slots is None else num_slots
    gen = _gen(seed + 7919, device)
    dt = torch_dtype(dtype)
    nc = 2 * dk + dv
    conv_state = _normal((num_slots, H, 3, nc), gen, device).to(dt)
    conv_w = _normal((H, nc, 4), gen, device, std=0.5)
    z = _normal((T, H, dv), gen, device).to(dt)
    norm_w = _normal((dv,), gen, device, std=0.1, mean=1.0)
    return FusedExtras(conv_state, conv_w, z, norm_w)


@dataclass
class VerifyInputs:
    q: torch.Tensor             # [B, D, H, dk]
    k: torch.Tensor             # [B, D, H, dk]
    v: torch.Tensor             # [B, D, H, dv]
    g: torch.Tensor             # [B, D, H, dk] fp32
    b: torch.Tensor             # [B, D, H]
    pool: torch.Tensor          # [num_slots, H, dv, dk] fp32
    slot_ids: torch.Tensor      # [B] int32
    num_accepted: torch.Tensor  # [B] int32, uniform on 0..D


def verify_inputs(B, D, H, dk, dv, dtype="bf16", num_slots=None, seed=0,
                  g_mean=3.0, pool_std=0.02, device="cpu"):
    num_slots = B if num_slots is None else num_slots
    gen = _gen(seed, device)
    dt = torch_dtype(dtype)
    q = _normal((B, D, H, dk), gen, device).to(dt)
    k = _normal((B, D, H, dk), gen, device).to(dt)
    v = _normal((B, D, H, dv), gen, device).to(dt)
    g = log_sigmoid_gate(_normal((B, D, H, dk), gen, device, mean=g_mean))
    b = _normal((B, D, H), gen, device).to(dt)
    pool = _normal((num_slots, H, dv, dk), gen, device, std=pool_std)
    perm = torch.randperm(num_slots, generator=gen, device=device)
    slot_ids = perm[:B].to(torch.int32)
    num_accepted = torch.randint(0, D + 1, (B,), generator=gen,
                                 device=device).to(torch.int32)
    return VerifyInputs(q, k, v, g, b, pool, slot_ids, num_accepted)


@dataclass
class PrefillInputs:
    q: torch.Tensor           # [T, H, dk]
    k: torch.Tensor           # [T, H, dk]
    v: torch.Tensor           # [T, H, dv]
    g: torch.Tensor           # [T, H, dk] fp32
    b: torch.Tensor           # [T, H]
    cu_seqlens: torch.Tensor  # [n+1] int32
    pool: torch.Tensor        # [num_slots, H, dv, dk] fp32
    slot_ids: torch.Tensor    # [n] int32


def prefill_inputs(seqlens, H, dk, dv, dtype="bf16", num_slots=None, seed=0,
                   g_mean=3.0, pool_std=0.02, zero_state=True, device="cpu"):
    """Variable-length prefill batch; ``seqlens`` is a list of token counts."""
    seqlens = [int(x) for x in seqlens]
    n = len(seqlens)
    T = sum(seqlens)
    num_slots = n if num_slots is None else num_slots
    gen = _gen(seed, device)
    dt = torch_dtype(dtype)
    q = _normal((T, H, dk), gen, device).to(dt)
    k = _normal((T, H, dk), gen, device).to(dt)
    v = _normal((T, H, dv), gen, device).to(dt)
    g = log_sigmoid_gate(_normal((T, H, dk), gen, device, mean=g_mean))
    b = _normal((T, H), gen, device).to(dt)
    pool = _normal((num_slots, H, dv, dk), gen, device,
                   std=1.0 if zero_state else pool_std)
    perm = torch.randperm(num_slots, generator=gen, device=device)
    slot_ids = perm[:n].to(torch.int32)
    cu = [0]
    for L in seqlens:
        cu.append(cu[-1] + L)
    cu_seqlens = torch.tensor(cu, dtype=torch.int32, device=device)
    return PrefillInputs(q, k, v, g, b, cu_seqlens, pool, slot_ids)


# The five workloads, by what they are.  Sizes are those of the decode,
# speculative-verify, prefill and long-context-mix measurements.
WORKLOADS = {
    "tiny_decode_2x2_d32_8tok_f32": dict(
        kind="decode_seq", B=2, H=2, dk=32, dv=32, tokens=8, dtype="f32",
        g_mean=2.0, num_slots=4, zero_state=True, seed=0),
    "decode_b256_h32_d128_pool4096_bf16": dict(
        kind="decode", B=256, H=32, dk=128, dv=128, dtype="bf16", g_mean=3.0,
        num_slots=4096, pool_std=0.02, seed=0),
    "verify_commit_b128_d7_h32_d128_bf16": dict(
        kind="verify", B=128, D=7, H=32, dk=128, dv=128, dtype="bf16",
        g_mean=3.0, num_slots=4096, pool_std=0.02, seed=0),
    "prefill_t8192_h32_d128_bf16": dict(
        kind="prefill", seqlens=[8192], H=32, dk=128, dv=128, dtype="bf16",
        g_mean=3.0, seed=0),
    "longmix_prefill_t102400_h32_decode256_b1024_h64_pool16384": dict(
        kind="longmix", T=102400, H=32, dk=128, dv=128, dtype="bf16",
        g_mean=3.0, decode_steps=256, B2=1024, H2=64, num_slots2=16384,
        seed=0),
}
