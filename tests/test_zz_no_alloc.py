"""GPU check of kda_prefill_chunked_static, the prefill entry point that
allocates nothing.

Some callers cannot allocate device memory at the moment they call the
library: code running while a CUDA graph is being captured, an engine whose
memory is entirely pre-planned and owned by another allocator, or a plug-in
host that hands the library only its inputs and outputs.  For them the
library keeps its prefill scratch in a fixed-size device array of its own.
This test calls that entry point through the C ABI and checks it against
the ordinary, caller-provided-workspace entry point, twice in a row (the
scratch array is shared by every call and keeps the previous call's bytes).
Before the compared calls, a larger, different batch with NaN inputs runs
through the same array, so that nothing in it starts out clean.  It lives in
a file of its own so that it runs after every other test.
"""
import ctypes

import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, round_to, to_np64, tol_for

pytestmark = pytest.mark.gpu


def _call_static(kda, x, out, pool, init_from_pool):
    lib = kda.lib()
    T, H, dk = x.k.shape
    dv = x.v.shape[2]
    n = x.slot_ids.shape[0]
    code = kda.KDA_DT_BF16 if x.q.dtype == torch.bfloat16 else kda.KDA_DT_F32
    dims = kda.make_dims(H, dk, dv, code)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.kda_prefill_chunked_static(
        ctypes.byref(dims), n, P(x.cu_seqlens), T, P(x.q), P(x.k), P(x.v), P(x.g), P(x.b),
        P(x.slot_ids), P(pool), pool.shape[0], 1 if init_from_pool else 0, P(out), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _poison_scratch(kda, dtype, d):
    """Fill the shared scratch with another call's bytes: a bigger batch with
    other lengths and NaN inputs, on a pool of its own."""
    y = inputs.prefill_inputs([300, 7, 200], 3, d, d, dtype=dtype, num_slots=3, seed=77,
                              device="cuda")
    for t in (y.q, y.k, y.v, y.g):
        t.fill_(float("nan"))
    out = torch.empty_like(y.v)
    assert _call_static(kda, y, out, y.pool, False) == kda.KDA_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_static_scratch_prefill_matches_workspace_prefill(dtype, d):
    from gated_delta_rule_decode_gb300 import kda
    x = inputs.prefill_inputs([100, 64, 30], 2, d, d, dtype=dtype, num_slots=4, seed=3,
                              zero_state=False, device="cuda")
    ref_pool = x.pool.clone()
    ref_out = kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, ref_pool,
                                  init_from_pool=True)
    torch.cuda.synchronize()
    # the workspace entry point against the oracle, so that bit equality
    # below is equality with a checked result
    xc = inputs.PrefillInputs(x.q.cpu(), x.k.cpu(), x.v.cpu(), x.g.cpu(), x.b.cpu(),
                              x.cu_seqlens.cpu(), x.pool.cpu(), x.slot_ids.cpu())
    o_ref, p_ref, e = oracle.prefill(xc.q, xc.k, xc.v, xc.g, xc.b, xc.cu_seqlens, xc.slot_ids,
                                     xc.pool, init_from_pool=True)
    assert e == 0
    atol, rtol = tol_for(x.q.dtype)
    assert_close(to_np64(ref_out), round_to(o_ref, x.q.dtype), atol, rtol, "outputs vs oracle")
    assert_close(to_np64(ref_pool), p_ref, atol, rtol, "states vs oracle")

    _poison_scratch(kda, dtype, d)
    for _ in range(2):  # the second call finds the first call's bytes in the scratch
        pool = x.pool.clone()
        out = torch.full_like(ref_out, float("nan"))
        assert _call_static(kda, x, out, pool, True) == kda.KDA_OK
        torch.cuda.synchronize()
        # the same kernels as the workspace entry point: the same bits
        assert torch.equal(out, ref_out)
        assert torch.equal(pool, ref_pool)


def test_static_scratch_rejects_oversized_batches():
    from gated_delta_rule_decode_gb300 import kda
    T, H = 1 << 20, 64  # far beyond the fixed scratch
    dims = kda.make_dims(H, 128, 128, kda.KDA_DT_BF16)
    need = kda.lib().kda_prefill_workspace_bytes(ctypes.byref(dims), 1, T)
    assert need > kda.lib().kda_static_scratch_bytes()
    dummy = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    st = kda.lib().kda_prefill_chunked_static(ctypes.byref(dims), 1, dummy, T, dummy, dummy, dummy,
                                             dummy, dummy, dummy, dummy, 1, 0, dummy, None, None)
    assert st == kda.KDA_ERR_WORKSPACE
