"""The bounded-wait timeout path, on the GPU, without a stuck copy.

A variant of the library is built with KDA_WAIT_LIMIT=1 and
KDA_WAIT_NONBLOCKING: every main-path mbarrier wait of the prefill and verify
kernels gives up after one non-suspending poll,
while the drain waits that follow keep their full limit (every copy and
product still in flight completes before a CTA releases its shared and
tensor memory).  The calls must return, report KDA_DEVERR_TIMEOUT, and leave
the context usable: the normal library, in the same process, still matches
the oracle afterwards."""
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def variant(tmp_path_factory):
    from gated_delta_rule_decode_gb300 import build, kda
    path = build.build(force=True, extra_flags=["-DKDA_WAIT_LIMIT=1", "-DKDA_WAIT_NONBLOCKING"],
                       out_path=str(tmp_path_factory.mktemp("waitlimit") / "libkda_wait1.so"))
    return kda.load_library(path)


def _with_lib(kda, lib, fn):
    saved = kda._lib
    kda._lib = lib
    try:
        return fn()
    finally:
        kda._lib = saved


def test_prefill_and_verify_time_out_and_return(variant):
    from gated_delta_rule_decode_gb300 import kda
    # tensor-core prefill (prep + chain)
    x = inputs.prefill_inputs([8192], 32, 128, 128, dtype="bf16", seed=0, device="cuda")
    flag = err_flag()
    _with_lib(kda, variant, lambda: kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens,
                                                        x.slot_ids, x.pool, err_flag=flag))
    torch.cuda.synchronize()
    assert flag.item() & kda.KDA_DEVERR_TIMEOUT
    # tensor-core verify (window + state kernels): its waits give up
    y = inputs.verify_inputs(64, 7, 16, 128, 128, dtype="bf16", num_slots=128, seed=1, device="cuda")
    flag = err_flag()
    _with_lib(kda, variant, lambda: kda.verify_record(y.q, y.k, y.v, y.g, y.b, y.slot_ids, y.pool,
                                                      err_flag=flag))
    torch.cuda.synchronize()
    assert flag.item() & kda.KDA_DEVERR_TIMEOUT
    # CUDA-core verify: its one wait is on the state copy it issued before
    # the coefficient work, which has usually landed by then; the call
    # returns either way, with no other error
    y = inputs.verify_inputs(64, 5, 16, 64, 64, dtype="bf16", num_slots=128, seed=1, device="cuda")
    flag = err_flag()
    _with_lib(kda, variant, lambda: kda.verify_record(y.q, y.k, y.v, y.g, y.b, y.slot_ids, y.pool,
                                                      err_flag=flag))
    torch.cuda.synchronize()
    assert flag.item() in (0, kda.KDA_DEVERR_TIMEOUT)


def test_context_still_usable_after_timeouts(variant):
    """Run after the timeouts: the normal library, same process, against the oracle."""
    from gated_delta_rule_decode_gb300 import kda
    x = inputs.prefill_inputs([130, 64], 2, 128, 128, dtype="bf16", num_slots=3, seed=2,
                              zero_state=False)
    pool = x.pool.cuda()
    flag = err_flag()
    out = kda.prefill_chunked(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(),
                              x.cu_seqlens.cuda(), x.slot_ids.cuda(), pool, init_from_pool=True,
                              err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    o_ref, p_ref, _ = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                                     init_from_pool=True)
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), atol, rtol, "outputs")
    assert_close(to_np64(pool), p_ref, atol, rtol, "states")
