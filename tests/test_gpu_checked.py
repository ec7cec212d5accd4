"""The checked build (-DKDA_CHECKED), the stand-in for a memory checker.

A variant of the library is built with the kernels' bounds checks compiled
in: every kernel checks the ranges its CTA reads and writes (token vectors,
state rows, records, scratch records, operand images, conv states) against
the sizes its arguments give, and an access outside them would set
KDA_DEVERR_BOUNDS and be skipped.  Each entry point runs on the same inputs
through the normal and the checked library: the checked one must find
nothing (the error flag stays 0) and produce the same bits.  The checked
build also checks a precondition the normal one leaves undefined: a slot
id named twice in one call sets KDA_DEVERR_DUPLICATE."""
import pytest
import torch

from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import err_flag

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked(tmp_path_factory):
    from gated_delta_rule_decode_gb300 import build, kda
    path = build.build(force=True, extra_flags=["-DKDA_CHECKED"],
                       out_path=str(tmp_path_factory.mktemp("checked") / "libkda_checked.so"))
    lib = kda.load_library(path)
    assert lib.kda_checked_build() == 1 and kda.lib().kda_checked_build() == 0
    return lib


def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


def _both(checked, run):
    """run(flag) on fresh copies of its buffers with the normal library and
    with the checked one; returns the two results and the two flags."""
    kda = _kda()
    saved = kda._lib
    outs = []
    for lib in (saved, checked):
        kda._lib = lib
        try:
            flag = err_flag()
            res = run(flag)
            torch.cuda.synchronize()
            outs.append((res, flag.item()))
        finally:
            kda._lib = saved
    return outs


def _assert_same(a, b):
    if isinstance(a, (tuple, list)):
        for x, y in zip(a, b):
            _assert_same(x, y)
    elif isinstance(a, dict):
        for key in a:
            _assert_same(a[key], b[key])
    else:
        assert torch.equal(a, b)


def _check(outs):
    (r0, f0), (r1, f1) = outs
    assert f0 == 0 and f1 == 0, (f0, f1)
    _assert_same(r0, r1)


@pytest.mark.parametrize("dtype,dk,dv,B", [("bf16", 128, 128, 256), ("f32", 64, 32, 5), ("bf16", 32, 64, 9)])
def test_decode_checked(checked, dtype, dk, dv, B):
    kda = _kda()
    x = inputs.decode_inputs(B, 4, dk, dv, dtype=dtype, num_slots=2 * B, seed=11, device="cuda")

    def run(flag):
        pool = x.pool.clone()
        out = kda.decode(x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool, err_flag=flag)
        return out, pool
    _check(_both(checked, run))


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("bf16", 32)])
def test_fused_decode_checked(checked, dtype, d):
    kda = _kda()
    x = inputs.decode_inputs(7, 3, d, d, dtype=dtype, num_slots=9, seed=12, device="cuda")
    ex = inputs.fused_extras(7, 3, d, d, dtype=dtype, num_slots=9, seed=12, device="cuda")

    def run(flag):
        pool, cst = x.pool.clone(), ex.conv_state.clone()
        out = kda.decode_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.slot_ids, pool, cst, ex.conv_w, ex.norm_w,
                               err_flag=flag)
        return out, pool, cst
    _check(_both(checked, run))


@pytest.mark.parametrize("dtype,dk,dv,D", [("bf16", 128, 128, 7), ("bf16", 128, 128, 3), ("f32", 64, 64, 5),
                                           ("bf16", 128, 128, 12)])
def test_verify_commit_checked(checked, dtype, dk, dv, D):
    kda = _kda()
    B, H = 6, 3
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype=dtype, num_slots=8, seed=13, device="cuda")

    def run(flag):
        pool = x.pool.clone()
        out, rec = kda.verify_record(x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool, err_flag=flag)
        kda.replay_commit(rec, x.num_accepted, x.slot_ids, pool, err_flag=flag)
        out_u, rec_u = kda.verify_record_u(x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool, err_flag=flag)
        kda.replay_commit_u(rec_u, x.num_accepted, x.slot_ids, pool, err_flag=flag)
        out2, rec2 = kda.commit_verify_u(rec_u, x.num_accepted, x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool,
                                         err_flag=flag)
        return out, rec, out_u, rec_u, out2, rec2, pool
    _check(_both(checked, run))


@pytest.mark.parametrize("lens,H,dtype,dk,dv", [
    ([70, 0, 130, 64, 1], 2, "bf16", 128, 128),
    ([8192], 32, "bf16", 128, 128),           # pipelined segments
    ([3 * 8192 + 337], 16, "bf16", 128, 128),  # growing segments
    ([70, 0, 130, 64, 1], 2, "f32", 64, 64),
    ([200, 5], 3, "bf16", 32, 128),
])
def test_prefill_checked(checked, lens, H, dtype, dk, dv):
    kda = _kda()
    x = inputs.prefill_inputs(lens, H, dk, dv, dtype=dtype, num_slots=len(lens) + 2, seed=14, device="cuda",
                              zero_state=False)
    x.slot_ids = torch.arange(len(lens), dtype=torch.int32, device="cuda")  # the snapshot's slot is free
    first = next(i for i, L in enumerate(lens) if L >= 128)
    snaps = (torch.tensor([first], dtype=torch.int32, device="cuda"),
             torch.tensor([64], dtype=torch.int32, device="cuda"),
             torch.tensor([len(lens)], dtype=torch.int32, device="cuda"))

    def run(flag):
        pool = x.pool.clone()
        out = kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, pool, init_from_pool=True,
                                  snapshots=snaps, err_flag=flag)
        return out, pool
    _check(_both(checked, run))


@pytest.mark.parametrize("lens,H", [([100, 3, 200], 2), ([8192], 32)])
def test_prefill_fused_checked(checked, lens, H):
    kda = _kda()
    d = 128
    x = inputs.prefill_inputs(lens, H, d, d, dtype="bf16", num_slots=len(lens) + 1, seed=15, device="cuda",
                              zero_state=False)
    ex = inputs.fused_prefill_extras(sum(lens), len(lens), H, d, d, dtype="bf16", num_slots=len(lens) + 1,
                                     seed=15, device="cuda")

    def run(flag):
        pool, cst = x.pool.clone(), ex.conv_state.clone()
        out = kda.prefill_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.cu_seqlens, x.slot_ids, pool, cst, ex.conv_w,
                                ex.norm_w, init_from_pool=True, err_flag=flag)
        return out, pool, cst
    _check(_both(checked, run))


def test_duplicate_slots_flagged(checked):
    """Two sequences naming the same slot (a precondition violation: both
    would update that state) are flagged by the checked build, in every
    entry point that takes slot ids; the normal build does not look."""
    kda = _kda()
    x = inputs.decode_inputs(4, 2, 64, 64, dtype="f32", num_slots=6, seed=16, device="cuda")
    x.slot_ids = torch.tensor([3, 1, 3, 0], dtype=torch.int32, device="cuda")
    y = inputs.verify_inputs(4, 3, 2, 64, 64, dtype="f32", num_slots=6, seed=16, device="cuda")
    y.slot_ids = torch.tensor([2, 2, -1, 5], dtype=torch.int32, device="cuda")
    z = inputs.prefill_inputs([40, 70], 2, 64, 64, dtype="f32", num_slots=3, seed=16, device="cuda")
    z.slot_ids = torch.tensor([1, 1], dtype=torch.int32, device="cuda")
    calls = [
        lambda f: kda.decode(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool.clone(), err_flag=f),
        lambda f: kda.verify_record(y.q, y.k, y.v, y.g, y.b, y.slot_ids, y.pool, err_flag=f),
        lambda f: kda.prefill_chunked(z.q, z.k, z.v, z.g, z.b, z.cu_seqlens, z.slot_ids, z.pool.clone(),
                                      err_flag=f),
    ]
    for call in calls:
        (_, f0), (_, f1) = _both(checked, call)
        assert f0 == 0
        assert f1 == kda.KDA_DEVERR_DUPLICATE
