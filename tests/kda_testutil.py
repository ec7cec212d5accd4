"""Shared helpers for the parity tests (tolerances, conversions, sampling)."""
from __future__ import annotations

import numpy as np
import torch

# Element-wise |x - ref| <= atol + rtol * |ref|, against fp64 oracle values
# (outputs first rounded to the output dtype).  bf16 inputs: max-abs 2e-3 /
# rel 1e-2; fp32 inputs: 1e-4 / 1e-4.
TOL = {torch.bfloat16: (2e-3, 1e-2), torch.float32: (1e-4, 1e-4)}


def tol_for(dtype):
    return TOL[dtype]


def to_np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """Round fp64 oracle values to the output dtype (RNE), back to fp64."""
    return torch.from_numpy(np.asarray(x, np.float64)).to(dtype).to(torch.float64).numpy()


def assert_close(got, ref, atol, rtol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance "
            f"(atol {atol}, rtol {rtol}); first at {tuple(idx)}: got {got[tuple(idx)]}, "
            f"ref {ref[tuple(idx)]}; max abs err {err.max():.3e}")


def err_flag(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)


def segment_starts(chains: int, sms: int, per_seq: int) -> list[int]:
    """Local chunk indices where the pipelined tensor-core prefill starts its
    segments, by the library's rule (restated here so that tests can put
    snapshot requests on segment boundaries): a geometric series of ratio
    rho = 0.16 x (sms - chains) / chains summing to the mean chunks per
    sequence, each segment at least max(16, per_seq // 50) chunks and 256
    prep CTAs, as many segments as that allows (at most 64)."""
    lo = [0]
    if chains <= 0 or chains >= sms or per_seq < 2:
        return lo
    rho = 0.16 * (sms - chains) / chains
    m = max(16.0, float(per_seq // 50), float((256 + chains - 1) // chains))

    def first(k):
        return per_seq / k if abs(rho - 1.0) < 1e-9 else per_seq * (1.0 - rho) / (1.0 - rho ** k)

    K = 1
    for k in range(2, 65):
        n0 = first(k)
        if min(n0, n0 * rho ** (k - 1)) >= m:
            K = k
        else:
            break
    acc = 0.0
    for k in range(1, K):
        acc += first(K) * rho ** (k - 1)
        lo.append(int(acc + 0.5))
    return lo
