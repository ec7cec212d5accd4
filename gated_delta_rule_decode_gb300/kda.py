"""Thin Python binding of libkda.so (argument marshalling only).

Every function here checks tensor shapes, dtypes and devices, passes raw
device pointers and the current CUDA stream to the C ABI declared in
``include/kda.h``, and raises ``KdaError`` on a negative status.  All
arithmetic runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback, and importing this module fails loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_CUDA = -3
KDA_ERR_WORKSPACE = -4
KDA_DT_F32 = 0
KDA_DT_BF16 = 1
KDA_DEVERR_SLOT = 1
KDA_DEVERR_ACCEPTED = 2
KDA_DEVERR_SEQLENS = 4
KDA_DEVERR_TIMEOUT = 8
KDA_DEVERR_RANGE = 16
KDA_DEVERR_SNAPSHOT = 32
KDA_DEVERR_BOUNDS = 64  # checked builds (-DKDA_CHECKED) only
KDA_DEVERR_DUPLICATE = 128  # checked builds only

EXPORTED = ("kda_decode", "kda_verify_record", "kda_replay_commit",
            "kda_prefill_chunked", "kda_prefill_workspace_bytes",
            "kda_records_bytes", "kda_status_string", "kda_abi_version",
            "kda_prefill_chunked_static", "kda_static_scratch_bytes",
            "kda_verify_workspace_bytes", "kda_prefill_chunked_snapshots",
            "kda_records_u_bytes", "kda_verify_record_u", "kda_replay_commit_u",
            "kda_commit_verify_u", "kda_decode_fused", "kda_prefill_fused", "kda_checked_build")


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status}")


class KdaDims(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("eps", ctypes.c_float), ("scale", ctypes.c_float)]


class KdaRecords(ctypes.Structure):
    _fields_ = [("k_hat", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p)]


class KdaFusedIo(ctypes.Structure):
    _fields_ = [("conv_state", ctypes.c_void_p), ("conv_w", ctypes.c_void_p),
                ("z", ctypes.c_void_p), ("norm_w", ctypes.c_void_p), ("eps_o", ctypes.c_float)]


class KdaRecordsU(ctypes.Structure):
    _fields_ = [("k_hat", ctypes.c_void_p), ("g", ctypes.c_void_p), ("u", ctypes.c_void_p)]


_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_PD = ctypes.POINTER(KdaDims)
_PR = ctypes.POINTER(KdaRecords)
_PRU = ctypes.POINTER(KdaRecordsU)
_PF = ctypes.POINTER(KdaFusedIo)


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkda.so and declare the C signatures.  Raises if it is missing."""
    if not os.path.exists(path):
        raise ImportError(
            f"libkda.so not found at {path}; build it with "
            "`python -m gated_delta_rule_decode_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    lib.kda_decode.argtypes = [_PD, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                               _I64, _VP, _VP, _VP]
    lib.kda_decode_fused.argtypes = [_PD, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                     _I64, _PF, _VP, _VP, _VP]
    lib.kda_decode_fused.restype = ctypes.c_int
    lib.kda_prefill_fused.argtypes = [_PD, _I32, _VP, _I64, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64,
                                      _I32, _PF, _VP, _VP, _SZ, _VP, _VP]
    lib.kda_prefill_fused.restype = ctypes.c_int
    lib.kda_verify_record.argtypes = [_PD, _I32, _I32, _VP, _VP, _VP, _VP, _VP,
                                      _VP, _VP, _I64, _VP, _PR, _VP, _SZ, _VP, _VP]
    lib.kda_verify_workspace_bytes.argtypes = [_PD, _I32, _I32]
    lib.kda_verify_workspace_bytes.restype = _SZ
    lib.kda_replay_commit.argtypes = [_PD, _I32, _I32, _PR, _VP, _VP, _VP, _I64,
                                      _VP, _VP]
    lib.kda_prefill_chunked.argtypes = [_PD, _I32, _VP, _I64, _VP, _VP, _VP,
                                        _VP, _VP, _VP, _VP, _I64, _I32, _VP,
                                        _VP, _SZ, _VP, _VP]
    lib.kda_records_u_bytes.argtypes = [_PD, _I32, _I32]
    lib.kda_records_u_bytes.restype = _SZ
    lib.kda_verify_record_u.argtypes = [_PD, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64,
                                        _VP, _PRU, _VP, _SZ, _VP, _VP]
    lib.kda_verify_record_u.restype = ctypes.c_int
    lib.kda_replay_commit_u.argtypes = [_PD, _I32, _I32, _PRU, _VP, _VP, _VP, _I64, _VP, _VP]
    lib.kda_replay_commit_u.restype = ctypes.c_int
    lib.kda_commit_verify_u.argtypes = [_PD, _I32, _I32, _PRU, _VP, _I32, _VP, _VP, _VP, _VP, _VP,
                                        _VP, _VP, _I64, _VP, _PRU, _VP, _SZ, _VP, _VP]
    lib.kda_commit_verify_u.restype = ctypes.c_int
    lib.kda_prefill_chunked_snapshots.argtypes = [_PD, _I32, _VP, _I64, _VP, _VP, _VP, _VP, _VP, _VP,
                                                  _VP, _I64, _I32, _VP, _I32, _VP, _VP, _VP, _VP, _SZ,
                                                  _VP, _VP]
    lib.kda_prefill_chunked_snapshots.restype = ctypes.c_int
    lib.kda_prefill_chunked_static.argtypes = [_PD, _I32, _VP, _I64, _VP, _VP, _VP, _VP,
                                               _VP, _VP, _VP, _I64, _I32, _VP, _VP, _VP]
    lib.kda_prefill_chunked_static.restype = ctypes.c_int
    lib.kda_static_scratch_bytes.argtypes = []
    lib.kda_static_scratch_bytes.restype = _SZ
    lib.kda_prefill_workspace_bytes.argtypes = [_PD, _I32, _I64]
    lib.kda_prefill_workspace_bytes.restype = _SZ
    lib.kda_records_bytes.argtypes = [_PD, _I32, _I32]
    lib.kda_records_bytes.restype = _SZ
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_abi_version.argtypes = []
    lib.kda_checked_build.argtypes = []
    for name in ("kda_decode", "kda_verify_record", "kda_replay_commit",
                 "kda_prefill_chunked", "kda_abi_version", "kda_checked_build"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


_lib = load_library()


def lib() -> ctypes.CDLL:
    return _lib


def _check(status: int, what: str):
    if status != KDA_OK:
        msg = _lib.kda_status_string(status).decode()
        raise KdaError(status, f"{what} failed ({msg})")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_DT_BF16
    if t.dtype == torch.float32:
        return KDA_DT_F32
    raise TypeError(f"unsupported input dtype {t.dtype} (bf16 or fp32)")


def make_dims(num_heads: int, dk: int, dv: int, dtype_code: int,
              eps: float = 1e-6, scale: float | None = None) -> KdaDims:
    return KdaDims(int(num_heads), int(dk), int(dv), int(dtype_code), float(eps),
                   float(scale) if scale is not None else 0.0)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _scratch(nbytes: int, device, stream) -> torch.Tensor:
    """Device scratch for one call; when the call runs on a stream other than
    the current one, the allocator is told so it is not reused too early."""
    t = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if stream is not None:
        t.record_stream(stream)
    return t


def _need(t: torch.Tensor, name: str, shape, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


class _Prepared:
    """A C-ABI call with its arguments already marshalled; calling it launches
    again on the same buffers (used to time launches without Python overhead)."""

    def __init__(self, fn, args, name, keep, result):
        self._fn, self._args, self._name = fn, args, name
        self._keep = keep          # ctypes structs the arguments point to
        self.result = result

    def __call__(self):
        _check(self._fn(*self._args), self._name)
        return self.result


def decode(q, k, v, g, b, slot_ids, pool, out=None, *, eps=1e-6, scale=None,
           err_flag=None, stream=None, _prepare=False):
    """One fused decode token per sequence, in place on ``pool``.

    q, k: [B, H, dk]; v: [B, H, dv]; g: [B, H, dk] fp32; b: [B, H];
    slot_ids: [B] int32; pool: [num_slots, H, dv, dk] fp32.  Returns out.
    """
    B, H, dk = k.shape
    dv = v.shape[2]
    dt = q.dtype
    for name, t, shp, d in (("q", q, (B, H, dk), dt), ("k", k, (B, H, dk), dt),
                            ("v", v, (B, H, dv), dt), ("g", g, (B, H, dk), torch.float32),
                            ("b", b, (B, H), dt), ("slot_ids", slot_ids, (B,), torch.int32)):
        _need(t, name, shp, d)
    _need(pool, "pool", (pool.shape[0], H, dv, dk), torch.float32)
    if out is None:
        out = torch.empty((B, H, dv), dtype=dt, device=q.device)
    _need(out, "out", (B, H, dv), dt)
    dims = make_dims(H, dk, dv, _dtype_code(q), eps, scale)
    args = (ctypes.byref(dims), B, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(slot_ids),
            _ptr(pool), pool.shape[0], _ptr(out), _ptr(err_flag), _stream_handle(stream))
    if _prepare:
        return _Prepared(_lib.kda_decode, args, "kda_decode", (dims,), out)
    _check(_lib.kda_decode(*args), "kda_decode")
    return out


def decode_fused(q, k, v, g, b, z, slot_ids, pool, conv_state, conv_w, norm_w, out=None, *,
                 eps=1e-6, eps_o=1e-6, scale=None, err_flag=None, stream=None, _prepare=False):
    """MegaKDA-style fused decode: ShortConv of q, k, v (conv_state shifted in
    place), the decode step on ``pool``, then RMS norm x norm_w x sigmoid(z).

    q, k: [B, H, dk]; v, z: [B, H, dv]; g: [B, H, dk] fp32; b: [B, H];
    conv_state: [num_slots, H, 3, 2 dk + dv] (input dtype);
    conv_w: [H, 2 dk + dv, 4] fp32; norm_w: [dv] fp32.  Returns out.
    """
    B, H, dk = k.shape
    dv = v.shape[2]
    dt = q.dtype
    S = pool.shape[0]
    for name, t, shp, d in (("q", q, (B, H, dk), dt), ("k", k, (B, H, dk), dt),
                            ("v", v, (B, H, dv), dt), ("g", g, (B, H, dk), torch.float32),
                            ("b", b, (B, H), dt), ("z", z, (B, H, dv), dt),
                            ("slot_ids", slot_ids, (B,), torch.int32),
                            ("pool", pool, (S, H, dv, dk), torch.float32),
                            ("conv_state", conv_state, (S, H, 3, 2 * dk + dv), dt),
                            ("conv_w", conv_w, (H, 2 * dk + dv, 4), torch.float32),
                            ("norm_w", norm_w, (dv,), torch.float32)):
        _need(t, name, shp, d)
    if out is None:
        out = torch.empty((B, H, dv), dtype=dt, device=q.device)
    _need(out, "out", (B, H, dv), dt)
    dims = make_dims(H, dk, dv, _dtype_code(q), eps, scale)
    io = KdaFusedIo(conv_state.data_ptr(), conv_w.data_ptr(), z.data_ptr(), norm_w.data_ptr(),
                    float(eps_o))
    args = (ctypes.byref(dims), B, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(slot_ids),
            _ptr(pool), S, ctypes.byref(io), _ptr(out), _ptr(err_flag), _stream_handle(stream))
    if _prepare:
        return _Prepared(_lib.kda_decode_fused, args, "kda_decode_fused", (dims, io), out)
    _check(_lib.kda_decode_fused(*args), "kda_decode_fused")
    return out


def prefill_fused(q, k, v, g, b, z, cu_seqlens, slot_ids, pool, conv_state, conv_w, norm_w, out=None, *,
                  init_from_pool=False, workspace=None, eps=1e-6, eps_o=1e-6, scale=None, err_flag=None,
                  stream=None, _prepare=False):
    """MegaKDA-style fused prefill: ShortConv of q, k, v along each sequence
    (history from ``conv_state`` when ``init_from_pool``, else zero; the conv
    state is updated), the chunked prefill on ``pool``, then RMS norm x
    norm_w x sigmoid(z) per token.  bf16 with dk = dv = 128 only.

    q, k: [T, H, dk]; v, z: [T, H, dv]; g: [T, H, dk] fp32; b: [T, H];
    cu_seqlens: [n+1] int32; slot_ids: [n] int32; conv_state:
    [num_slots, H, 3, 2 dk + dv]; conv_w: [H, 2 dk + dv, 4] fp32;
    norm_w: [dv] fp32.  Returns out [T, H, dv].
    """
    T, H, dk = k.shape
    dv = v.shape[2]
    n = slot_ids.shape[0]
    dt = q.dtype
    S = pool.shape[0]
    for name, t, shp, d in (("q", q, (T, H, dk), dt), ("k", k, (T, H, dk), dt),
                            ("v", v, (T, H, dv), dt), ("g", g, (T, H, dk), torch.float32),
                            ("b", b, (T, H), dt), ("z", z, (T, H, dv), dt),
                            ("cu_seqlens", cu_seqlens, (n + 1,), torch.int32),
                            ("slot_ids", slot_ids, (n,), torch.int32),
                            ("pool", pool, (S, H, dv, dk), torch.float32),
                            ("conv_state", conv_state, (S, H, 3, 2 * dk + dv), dt),
                            ("conv_w", conv_w, (H, 2 * dk + dv, 4), torch.float32),
                            ("norm_w", norm_w, (dv,), torch.float32)):
        _need(t, name, shp, d)
    if out is None:
        out = torch.empty((T, H, dv), dtype=dt, device=q.device)
    _need(out, "out", (T, H, dv), dt)
    code = _dtype_code(q)
    need = prefill_workspace_bytes(H, dk, dv, code, n, T)
    if workspace is None and need > 0:
        workspace = _scratch(need, q.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dims = make_dims(H, dk, dv, code, eps, scale)
    io = KdaFusedIo(conv_state.data_ptr(), conv_w.data_ptr(), z.data_ptr(), norm_w.data_ptr(), float(eps_o))
    args = (ctypes.byref(dims), n, _ptr(cu_seqlens), T, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b),
            _ptr(slot_ids), _ptr(pool), S, 1 if init_from_pool else 0, ctypes.byref(io), _ptr(out),
            _ptr(workspace), ws_bytes, _ptr(err_flag), _stream_handle(stream))
    if _prepare:
        return _Prepared(_lib.kda_prefill_fused, args, "kda_prefill_fused", (dims, io, workspace), out)
    _check(_lib.kda_prefill_fused(*args), "kda_prefill_fused")
    return out


def alloc_records(B, D, H, dk, dv, dtype, device):
    """Allocate a ReplaySSM record set (dict of tensors) for (B, D)."""
    return dict(
        k_hat=torch.empty((B, D, H, dk), dtype=torch.float32, device=device),
        v=torch.empty((B, D, H, dv), dtype=dtype, device=device),
        g=torch.empty((B, D, H, dk), dtype=torch.float32, device=device),
        beta=torch.empty((B, D, H), dtype=torch.float32, device=device))


def _records_struct(rec) -> KdaRecords:
    return KdaRecords(rec["k_hat"].data_ptr(), rec["v"].data_ptr(),
                      rec["g"].data_ptr(), rec["beta"].data_ptr())


def verify_workspace_bytes(H, dk, dv, dtype_code, batch, draft_len) -> int:
    dims = make_dims(H, dk, dv, dtype_code)
    return int(_lib.kda_verify_workspace_bytes(ctypes.byref(dims), int(batch), int(draft_len)))


def verify_record(q, k, v, g, b, slot_ids, pool, out=None, records=None, *,
                  workspace=None, eps=1e-6, scale=None, err_flag=None, stream=None,
                  _prepare=False):
    """ReplaySSM verify of D draft tokens; pool is read only.

    q, k: [B, D, H, dk]; v: [B, D, H, dv]; g fp32; b: [B, D, H].
    ``workspace``: device uint8 scratch of verify_workspace_bytes(...) bytes,
    allocated here when omitted.  Returns (out [B, D, H, dv], records dict).
    """
    B, D, H, dk = k.shape
    dv = v.shape[3]
    dt = q.dtype
    for name, t, shp, d in (("q", q, (B, D, H, dk), dt), ("k", k, (B, D, H, dk), dt),
                            ("v", v, (B, D, H, dv), dt),
                            ("g", g, (B, D, H, dk), torch.float32),
                            ("b", b, (B, D, H), dt), ("slot_ids", slot_ids, (B,), torch.int32)):
        _need(t, name, shp, d)
    _need(pool, "pool", (pool.shape[0], H, dv, dk), torch.float32)
    if out is None:
        out = torch.empty((B, D, H, dv), dtype=dt, device=q.device)
    _need(out, "out", (B, D, H, dv), dt)
    if records is None:
        records = alloc_records(B, D, H, dk, dv, dt, q.device)
    rs = _records_struct(records)
    dims = make_dims(H, dk, dv, _dtype_code(q), eps, scale)
    need = int(_lib.kda_verify_workspace_bytes(ctypes.byref(dims), B, D))
    if workspace is None and need > 0:
        workspace = _scratch(need, q.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (ctypes.byref(dims), B, D, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b),
            _ptr(slot_ids), _ptr(pool), pool.shape[0], _ptr(out), ctypes.byref(rs),
            _ptr(workspace), ws_bytes, _ptr(err_flag), _stream_handle(stream))
    if _prepare:
        return _Prepared(_lib.kda_verify_record, args, "kda_verify_record", (dims, rs, workspace),
                         (out, records))
    _check(_lib.kda_verify_record(*args), "kda_verify_record")
    return out, records


def replay_commit(records, num_accepted, slot_ids, pool, *, err_flag=None,
                  stream=None, _prepare=False):
    """Replay the accepted prefix of each sequence's records onto ``pool``."""
    B, D, H, dk = records["k_hat"].shape
    dv = records["v"].shape[3]
    dt = records["v"].dtype
    _need(num_accepted, "num_accepted", (B,), torch.int32)
    _need(slot_ids, "slot_ids", (B,), torch.int32)
    _need(pool, "pool", (pool.shape[0], H, dv, dk), torch.float32)
    rs = _records_struct(records)
    dims = make_dims(H, dk, dv, _dtype_code(records["v"]))
    args = (ctypes.byref(dims), B, D, ctypes.byref(rs), _ptr(num_accepted), _ptr(slot_ids),
            _ptr(pool), pool.shape[0], _ptr(err_flag), _stream_handle(stream))
    del dt
    if _prepare:
        return _Prepared(_lib.kda_replay_commit, args, "kda_replay_commit", (dims, rs), None)
    _check(_lib.kda_replay_commit(*args), "kda_replay_commit")


def alloc_records_u(B, D, H, dk, dv, device):
    """Allocate a u-record set (dict of fp32 tensors) for (B, D)."""
    return dict(k_hat=torch.empty((B, D, H, dk), dtype=torch.float32, device=device),
                g=torch.empty((B, D, H, dk), dtype=torch.float32, device=device),
                u=torch.empty((B, D, H, dv), dtype=torch.float32, device=device))


def _records_u_struct(rec) -> KdaRecordsU:
    return KdaRecordsU(rec["k_hat"].data_ptr(), rec["g"].data_ptr(), rec["u"].data_ptr())


def _verify_u_args(q, k, v, g, b, slot_ids, pool, out, records, workspace, eps, scale, stream):
    B, D, H, dk = k.shape
    dv = v.shape[3]
    dt = q.dtype
    for name, t, shp, d in (("q", q, (B, D, H, dk), dt), ("k", k, (B, D, H, dk), dt),
                            ("v", v, (B, D, H, dv), dt),
                            ("g", g, (B, D, H, dk), torch.float32),
                            ("b", b, (B, D, H), dt), ("slot_ids", slot_ids, (B,), torch.int32)):
        _need(t, name, shp, d)
    _need(pool, "pool", (pool.shape[0], H, dv, dk), torch.float32)
    if out is None:
        out = torch.empty((B, D, H, dv), dtype=dt, device=q.device)
    _need(out, "out", (B, D, H, dv), dt)
    if records is None:
        records = alloc_records_u(B, D, H, dk, dv, q.device)
    dims = make_dims(H, dk, dv, _dtype_code(q), eps, scale)
    need = int(_lib.kda_verify_workspace_bytes(ctypes.byref(dims), B, D))
    if workspace is None and need > 0:
        workspace = _scratch(need, q.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return B, D, dims, out, records, workspace, ws_bytes


def verify_record_u(q, k, v, g, b, slot_ids, pool, out=None, records=None, *, workspace=None,
                    eps=1e-6, scale=None, err_flag=None, stream=None, _prepare=False):
    """ReplaySSM verify writing u records; pool is read only.  Returns (out, records)."""
    B, D, dims, out, records, workspace, ws_bytes = _verify_u_args(
        q, k, v, g, b, slot_ids, pool, out, records, workspace, eps, scale, stream)
    rs = _records_u_struct(records)
    args = (ctypes.byref(dims), B, D, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(slot_ids),
            _ptr(pool), pool.shape[0], _ptr(out), ctypes.byref(rs), _ptr(workspace), ws_bytes,
            _ptr(err_flag), _stream_handle(stream))
    if _prepare:
        return _Prepared(_lib.kda_verify_record_u, args, "kda_verify_record_u", (dims, rs, workspace),
                         (out, records))
    _check(_lib.kda_verify_record_u(*args), "kda_verify_record_u")
    return out, records


def replay_commit_u(records, num_accepted, slot_ids, pool, *, err_flag=None, stream=None,
                    _prepare=False):
    """Commit the accepted prefix of each sequence's u records onto ``pool``."""
    B, D, H, dk = records["k_hat"].shape
    dv = records["u"].shape[3]
    _need(num_accepted, "num_accepted", (B,), torch.int32)
    _need(slot_ids, "slot_ids", (B,), torch.int32)
    _need(pool, "pool", (pool.shape[0], H, dv, dk), torch.float32)
    rs = _records_u_struct(records)
    dims = make_dims(H, dk, dv, KDA_DT_F32)
    args = (ctypes.byref(dims), B, D, ctypes.byref(rs), _ptr(num_accepted), _ptr(slot_ids),
            _ptr(pool), pool.shape[0], _ptr(err_flag), _stream_handle(stream))
    if _prepare:
        return _Prepared(_lib.kda_replay_commit_u, args, "kda_replay_commit_u", (dims, rs), None)
    _check(_lib.kda_replay_commit_u(*args), "kda_replay_commit_u")


def commit_verify_u(prev_records, prev_accepted, q, k, v, g, b, slot_ids, pool, out=None,
                    records=None, *, workspace=None, eps=1e-6, scale=None, err_flag=None,
                    stream=None, _prepare=False):
    """Commit the previous window's accepted u records, then verify this
    window, in one call (the pool receives the committed state).
    Returns (out, records)."""
    B, D, dims, out, records, workspace, ws_bytes = _verify_u_args(
        q, k, v, g, b, slot_ids, pool, out, records, workspace, eps, scale, stream)
    Dp = prev_records["k_hat"].shape[1]
    _need(prev_accepted, "prev_accepted", (B,), torch.int32)
    prs = _records_u_struct(prev_records)
    rs = _records_u_struct(records)
    args = (ctypes.byref(dims), B, Dp, ctypes.byref(prs), _ptr(prev_accepted), D, _ptr(q), _ptr(k),
            _ptr(v), _ptr(g), _ptr(b), _ptr(slot_ids), _ptr(pool), pool.shape[0], _ptr(out),
            ctypes.byref(rs), _ptr(workspace), ws_bytes, _ptr(err_flag), _stream_handle(stream))
    if _prepare:
        return _Prepared(_lib.kda_commit_verify_u, args, "kda_commit_verify_u",
                         (dims, prs, rs, workspace), (out, records))
    _check(_lib.kda_commit_verify_u(*args), "kda_commit_verify_u")
    return out, records


def prefill_workspace_bytes(H, dk, dv, dtype_code, num_seqs, total_tokens) -> int:
    dims = make_dims(H, dk, dv, dtype_code)
    return int(_lib.kda_prefill_workspace_bytes(ctypes.byref(dims), int(num_seqs),
                                                int(total_tokens)))


def prefill_chunked(q, k, v, g, b, cu_seqlens, slot_ids, pool, out=None, *,
                    init_from_pool=False, workspace=None, snapshots=None, eps=1e-6,
                    scale=None, err_flag=None, stream=None, _prepare=False):
    """Chunked prefill of a packed variable-length batch.

    q, k: [T, H, dk]; v: [T, H, dv]; g: [T, H, dk] fp32; b: [T, H];
    cu_seqlens: [n+1] int32 (device); slot_ids: [n] int32.  The final state of
    each sequence goes to its slot.  ``snapshots``: optional (seq, tokens,
    slot) int32 device tensors of equal length, sorted by sequence then token
    count: the state after that many tokens of that sequence also goes to
    that slot (kda_prefill_chunked_snapshots).  Returns out [T, H, dv].
    """
    T, H, dk = k.shape
    dv = v.shape[2]
    n = slot_ids.shape[0]
    dt = q.dtype
    for name, t, shp, d in (("q", q, (T, H, dk), dt), ("k", k, (T, H, dk), dt),
                            ("v", v, (T, H, dv), dt), ("g", g, (T, H, dk), torch.float32),
                            ("b", b, (T, H), dt), ("cu_seqlens", cu_seqlens, (n + 1,), torch.int32),
                            ("slot_ids", slot_ids, (n,), torch.int32)):
        _need(t, name, shp, d)
    _need(pool, "pool", (pool.shape[0], H, dv, dk), torch.float32)
    if out is None:
        out = torch.empty((T, H, dv), dtype=dt, device=q.device)
    _need(out, "out", (T, H, dv), dt)
    code = _dtype_code(q)
    need = prefill_workspace_bytes(H, dk, dv, code, n, T)
    if workspace is None and need > 0:
        workspace = _scratch(need, q.device, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dims = make_dims(H, dk, dv, code, eps, scale)
    if snapshots is not None:
        sseq, stok, sslot = snapshots
        m = sseq.shape[0]
        for name, t in (("snapshot seq", sseq), ("snapshot tokens", stok), ("snapshot slot", sslot)):
            _need(t, name, (m,), torch.int32)
        args = (ctypes.byref(dims), n, _ptr(cu_seqlens), T, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                _ptr(b), _ptr(slot_ids), _ptr(pool), pool.shape[0], 1 if init_from_pool else 0,
                _ptr(out), m, _ptr(sseq), _ptr(stok), _ptr(sslot), _ptr(workspace), ws_bytes,
                _ptr(err_flag), _stream_handle(stream))
        fn, name = _lib.kda_prefill_chunked_snapshots, "kda_prefill_chunked_snapshots"
    else:
        args = (ctypes.byref(dims), n, _ptr(cu_seqlens), T, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                _ptr(b), _ptr(slot_ids), _ptr(pool), pool.shape[0], 1 if init_from_pool else 0,
                _ptr(out), _ptr(workspace), ws_bytes, _ptr(err_flag), _stream_handle(stream))
        fn, name = _lib.kda_prefill_chunked, "kda_prefill_chunked"
    if _prepare:
        return _Prepared(fn, args, name, (dims, workspace), out)
    _check(fn(*args), name)
    return out
