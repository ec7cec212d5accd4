"""fp64 CPU oracle for the KDA recurrence.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg import this package.  The product library
never imports, links or calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``kda_oracle.c`` (plain sequential fp64 C, one loop
per (sequence, head), optionally spread over host cores with OpenMP).  This
module compiles it with gcc on first use and exposes array-level wrappers.
Every wrapper takes arrays holding the exact values the GPU path receives
(bf16 or fp32 inputs upcast to float64) and returns float64 results.

``chunk_form`` holds the separate fp64 chunk-form (WY/UT) restatement used to
check that the chunked prefill is a re-association of this recurrence.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libkda_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.kda_oracle_set_threads.argtypes = [ctypes.c_int]
        lib.kda_oracle_set_threads.restype = ctypes.c_int
        lib.kda_oracle_recurrence.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int64, _D, _D, _D, _D, _D,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
            ctypes.c_double, _D, _D]
        lib.kda_oracle_recurrence.restype = None
        lib.kda_oracle_decode.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D, _D, _D,
            _D, _D, _I32, _D, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
            _D]
        lib.kda_oracle_decode.restype = ctypes.c_int64
        lib.kda_oracle_verify.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, _D, _D, _D, _D, _D, _I32, _D, ctypes.c_int64,
            ctypes.c_double, ctypes.c_double, _D, _D, _D, _D, _D]
        lib.kda_oracle_verify.restype = ctypes.c_int64
        lib.kda_oracle_replay.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, _D, _D, _D, _D, _I32, _I32, _D, ctypes.c_int64]
        lib.kda_oracle_replay.restype = ctypes.c_int64
        lib.kda_oracle_prefill.argtypes = [
            ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D,
            _D, _D, _D, _D, _I32, _D, ctypes.c_int64, ctypes.c_int,
            ctypes.c_double, ctypes.c_double, _D]
        lib.kda_oracle_prefill.restype = ctypes.c_int64
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    """Upcast to a C-contiguous float64 numpy array (torch tensors accepted)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: only for the dtype upcast of torch inputs
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _p(a: np.ndarray, ty=_D):
    return a.ctypes.data_as(ty)


def default_scale(dk: int) -> float:
    """The output scale dk^-1/2."""
    return float(dk) ** -0.5


def set_threads(n: int) -> int:
    """Set the OpenMP thread count of the oracle; returns the count in effect."""
    return _load().kda_oracle_set_threads(int(n))


def recurrence(q, k, v, g, b, S0=None, eps: float = 1e-6, scale=None):
    """Token-by-token recurrence for ONE (sequence, head).

    q, k, g: [n, dk]; v: [n, dv]; b: [n]; S0: [dv, dk] (zero if None).
    Returns (o [n, dv], S_final [dv, dk]).
    """
    lib = _load()
    k = _f64(k)
    n, dk = k.shape
    v = _f64(v)
    dv = v.shape[1]
    q = _f64(q)
    g = _f64(g)
    b = _f64(b).reshape(n)
    S = np.zeros((dv, dk)) if S0 is None else _f64(S0).copy()
    o = np.zeros((n, dv))
    scale = default_scale(dk) if scale is None else float(scale)
    lib.kda_oracle_recurrence(dk, dv, n, _p(q), _p(k), _p(v), _p(g), _p(b),
                              dk, dv, 1, eps, scale, _p(S), _p(o))
    return o, S


def decode(q, k, v, g, b, slot_ids, pool, eps: float = 1e-6, scale=None):
    """One decode token per sequence over the state pool (fp64).

    q, k, g: [B, H, dk]; v: [B, H, dv]; b: [B, H]; slot_ids: [B];
    pool: [num_slots, H, dv, dk].  Returns (out [B, H, dv], new_pool, errors).
    The input pool is not modified; a float64 copy is updated and returned.
    """
    lib = _load()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    B, H, dk = k.shape
    dv = v.shape[2]
    b = _f64(b).reshape(B, H)
    slots = _i32(slot_ids).reshape(B)
    P = _f64(pool).copy()
    out = np.zeros((B, H, dv))
    scale = default_scale(dk) if scale is None else float(scale)
    err = lib.kda_oracle_decode(B, H, dk, dv, _p(q), _p(k), _p(v), _p(g),
                                _p(b), _p(slots, _I32), _p(P), P.shape[0],
                                eps, scale, _p(out))
    return out, P, int(err)


def verify(q, k, v, g, b, slot_ids, pool, eps: float = 1e-6, scale=None):
    """Speculative verify over D draft tokens per sequence; pool is read only.

    q, k, g: [B, D, H, dk]; v: [B, D, H, dv]; b: [B, D, H].
    Returns (out [B, D, H, dv], records dict(k_hat, v, g, beta), errors).
    """
    lib = _load()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    B, D, H, dk = k.shape
    dv = v.shape[3]
    b = _f64(b).reshape(B, D, H)
    slots = _i32(slot_ids).reshape(B)
    P = _f64(pool)
    out = np.zeros((B, D, H, dv))
    khat = np.zeros((B, D, H, dk))
    vrec = np.zeros((B, D, H, dv))
    grec = np.zeros((B, D, H, dk))
    beta = np.zeros((B, D, H))
    scale = default_scale(dk) if scale is None else float(scale)
    err = lib.kda_oracle_verify(B, D, H, dk, dv, _p(q), _p(k), _p(v), _p(g),
                                _p(b), _p(slots, _I32), _p(P), P.shape[0],
                                eps, scale, _p(out), _p(khat), _p(vrec),
                                _p(grec), _p(beta))
    return out, dict(k_hat=khat, v=vrec, g=grec, beta=beta), int(err)


def replay(records, num_accepted, slot_ids, pool):
    """Commit: replay the first num_accepted[n] records onto the pool (fp64).

    records: dict(k_hat [B,D,H,dk], v [B,D,H,dv], g [B,D,H,dk], beta [B,D,H]).
    Returns (new_pool, errors); the input pool is not modified.
    """
    lib = _load()
    khat = _f64(records["k_hat"])
    B, D, H, dk = khat.shape
    vrec = _f64(records["v"])
    dv = vrec.shape[3]
    grec = _f64(records["g"])
    beta = _f64(records["beta"]).reshape(B, D, H)
    acc = _i32(num_accepted).reshape(B)
    slots = _i32(slot_ids).reshape(B)
    P = _f64(pool).copy()
    err = lib.kda_oracle_replay(B, D, H, dk, dv, _p(khat), _p(vrec), _p(grec),
                                _p(beta), _p(acc, _I32), _p(slots, _I32),
                                _p(P), P.shape[0])
    return P, int(err)


def prefill(q, k, v, g, b, cu_seqlens, slot_ids, pool, init_from_pool=False,
            eps: float = 1e-6, scale=None):
    """Token-by-token prefill of a variable-length batch (fp64).

    q, k, g: [T, H, dk]; v: [T, H, dv]; b: [T, H]; cu_seqlens: [n+1].
    Returns (out [T, H, dv], new_pool, errors); the input pool is not modified.
    """
    lib = _load()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(g)
    T, H, dk = k.shape
    dv = v.shape[2]
    b = _f64(b).reshape(T, H)
    cu = np.ascontiguousarray(
        cu_seqlens.detach().cpu().numpy() if hasattr(cu_seqlens, "detach")
        else cu_seqlens, dtype=np.int64)
    n = cu.shape[0] - 1
    slots = _i32(slot_ids).reshape(n)
    P = _f64(pool).copy()
    out = np.zeros((T, H, dv))
    scale = default_scale(dk) if scale is None else float(scale)
    err = lib.kda_oracle_prefill(n, _p(cu, _I64), H, dk, dv, _p(q), _p(k),
                                 _p(v), _p(g), _p(b), _p(slots, _I32), _p(P),
                                 P.shape[0], 1 if init_from_pool else 0, eps,
                                 scale, _p(out))
    return out, P, int(err)
