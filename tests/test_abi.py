"""CPU checks of the C ABI: the library loads, exports every entry point that
include/*.h declares, and rejects bad host-side arguments before any launch
(none of these calls reaches a kernel, so no GPU is needed)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    from gated_delta_rule_decode_gb300 import build
    build.build()
    from gated_delta_rule_decode_gb300 import kda as mod
    return mod


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kda_decode", "kda_verify_record", "kda_replay_commit", "kda_prefill_chunked"):
        assert n in names


def test_library_exports_every_declared_symbol(kda):
    lib = kda.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(kda.EXPORTED) <= set(declared_functions())
    assert lib.kda_abi_version() == 6


def test_status_strings(kda):
    lib = kda.lib()
    assert lib.kda_status_string(0) == b"ok"
    for s in (-1, -2, -3, -4):
        assert lib.kda_status_string(s) != b"unknown status"
    assert lib.kda_status_string(12345) == b"unknown status"


def test_sizing_helpers(kda):
    lib = kda.lib()
    d = kda.make_dims(32, 128, 128, kda.KDA_DT_BF16)
    # per (sequence, draft token, head): k_hat 512 + g 512 + v 256 + beta 4 bytes
    assert lib.kda_records_bytes(ctypes.byref(d), 128, 7) == 128 * 7 * 32 * 1284
    d32 = kda.make_dims(2, 32, 64, kda.KDA_DT_F32)
    assert lib.kda_records_bytes(ctypes.byref(d32), 3, 2) == 3 * 2 * 2 * (32 * 8 + 64 * 4 + 4)
    bad = kda.make_dims(2, 48, 64, kda.KDA_DT_F32)
    assert lib.kda_records_bytes(ctypes.byref(bad), 3, 2) == 0
    # verify scratch: one 12928-byte record per (sequence, head) for bf16
    # windows of 1..8 tokens at dk = dv = 128, none for any other shape
    for D in (1, 7, 8):
        assert lib.kda_verify_workspace_bytes(ctypes.byref(d), 128, D) == 128 * 32 * 12928
    assert lib.kda_verify_workspace_bytes(ctypes.byref(d), 128, 9) == 0
    assert lib.kda_verify_workspace_bytes(ctypes.byref(d), 0, 7) == 0
    assert lib.kda_verify_workspace_bytes(ctypes.byref(d32), 3, 2) == 0
    df = kda.make_dims(32, 128, 128, kda.KDA_DT_F32)
    assert lib.kda_verify_workspace_bytes(ctypes.byref(df), 128, 7) == 0
    d64 = kda.make_dims(32, 128, 64, kda.KDA_DT_BF16)
    assert lib.kda_verify_workspace_bytes(ctypes.byref(d64), 128, 7) == 0
    for D in (0, 17):
        assert lib.kda_verify_workspace_bytes(ctypes.byref(d), 128, D) == 0
    assert lib.kda_verify_workspace_bytes(ctypes.byref(bad), 128, 7) == 0
    assert lib.kda_prefill_workspace_bytes(ctypes.byref(bad), 1, 64) == 0


def test_host_side_argument_errors_launch_nothing(kda):
    lib = kda.lib()
    P = ctypes.c_void_p(256)  # never dereferenced: every call below fails validation
    good = kda.make_dims(4, 64, 64, kda.KDA_DT_BF16)
    call = lambda dims, batch, *ptrs: lib.kda_decode(  # noqa: E731
        dims, batch, *ptrs, 8, P, None, None)
    ptrs = (P, P, P, P, P, P, P)
    assert call(None, 1, *ptrs) == kda.KDA_ERR_INVALID_ARG
    assert call(ctypes.byref(kda.make_dims(0, 64, 64, 1)), 1, *ptrs) == kda.KDA_ERR_INVALID_ARG
    assert call(ctypes.byref(kda.make_dims(4, 96, 64, 1)), 1, *ptrs) == kda.KDA_ERR_UNSUPPORTED
    assert call(ctypes.byref(kda.make_dims(4, 64, 64, 7)), 1, *ptrs) == kda.KDA_ERR_UNSUPPORTED
    assert call(ctypes.byref(good), -1, *ptrs) == kda.KDA_ERR_INVALID_ARG
    assert call(ctypes.byref(good), 0, *ptrs) == kda.KDA_OK          # empty batch: no-op
    assert call(ctypes.byref(good), 1, None, P, P, P, P, P, P) == kda.KDA_ERR_INVALID_ARG
    mis = ctypes.c_void_p(258)                                          # not 16-byte aligned
    assert call(ctypes.byref(good), 1, mis, P, P, P, P, P, P) == kda.KDA_ERR_INVALID_ARG
    rec = kda.KdaRecords(256, 256, 256, 256)
    for D in (0, 17):
        assert lib.kda_verify_record(ctypes.byref(good), 1, D, P, P, P, P, P, P, P, 8, P,
                                     ctypes.byref(rec), None, 0, None, None) == kda.KDA_ERR_INVALID_ARG
        assert lib.kda_replay_commit(ctypes.byref(good), 1, D, ctypes.byref(rec), P, P, P, 8,
                                     None, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_verify_record(ctypes.byref(good), 1, 7, P, P, P, P, P, P, P, 8, P,
                                 None, None, 0, None, None) == kda.KDA_ERR_INVALID_ARG
    # the bf16 dk = dv = 128 window of <= 8 tokens needs its scratch: missing,
    # too small or unaligned is rejected before any launch
    big = kda.make_dims(2, 128, 128, kda.KDA_DT_BF16)
    need = lib.kda_verify_workspace_bytes(ctypes.byref(big), 1, 7)
    assert need > 0
    for ws, nbytes in ((None, 0), (P, need - 1), (ctypes.c_void_p(256 + 16), need)):
        assert lib.kda_verify_record(ctypes.byref(big), 1, 7, P, P, P, P, P, P, P, 8, P,
                                     ctypes.byref(rec), ws, nbytes, None,
                                     None) == kda.KDA_ERR_WORKSPACE
    assert lib.kda_replay_commit(ctypes.byref(good), 0, 7, ctypes.byref(rec), P, P, P, 8,
                                 None, None) == kda.KDA_OK
    assert lib.kda_prefill_chunked(ctypes.byref(good), 0, P, 0, P, P, P, P, P, P, P, 8, 0,
                                   P, None, 0, None, None) == kda.KDA_OK
    assert lib.kda_prefill_chunked(ctypes.byref(good), 1, None, 64, P, P, P, P, P, P, P, 8,
                                   0, P, None, 0, None, None) == kda.KDA_ERR_INVALID_ARG
