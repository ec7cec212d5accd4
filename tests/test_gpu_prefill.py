"""GPU parity of kda_prefill_chunked against the fp64 token-by-token oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for

pytestmark = pytest.mark.gpu


def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


def _run(kda, x, init=False, flag=None, workspace=None):
    pool = x.pool.cuda()
    out = kda.prefill_chunked(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(),
                              x.cu_seqlens.cuda(), x.slot_ids.cuda(), pool,
                              init_from_pool=init, err_flag=flag, workspace=workspace)
    torch.cuda.synchronize()
    return out, pool


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 128), (64, 128), (128, 32)])
def test_prefill_varlen_parity(dtype, dk, dv):
    """Ragged batch: a partial chunk, exact chunks, a one-token and an empty
    sequence; states from zero and from the pool."""
    kda = _kda()
    lens = [100, 64, 1, 0, 130]
    x = inputs.prefill_inputs(lens, 2, dk, dv, dtype=dtype, num_slots=7, seed=dk + dv,
                              zero_state=False, pool_std=0.05)
    dt = inputs.torch_dtype(dtype)
    atol, rtol = tol_for(dt)
    for init in (False, True):
        flag = err_flag()
        out, pool = _run(kda, x, init=init, flag=flag)
        assert flag.item() == 0
        o_ref, p_ref, e = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids,
                                         x.pool, init_from_pool=init)
        assert e == 0
        assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, f"outputs (init={init})")
        assert_close(to_np64(pool), p_ref, atol, rtol, f"states (init={init})")
        touched = set(x.slot_ids.tolist())
        for sl in range(7):
            if sl not in touched:
                assert torch.equal(pool[sl].cpu(), x.pool[sl])


def test_prefill_padding_and_bad_slot():
    kda = _kda()
    x = inputs.prefill_inputs([70, 20, 33], 2, 64, 64, dtype="bf16", num_slots=4, seed=4,
                              zero_state=False)
    x.slot_ids = torch.tensor([-1, 2, 9], dtype=torch.int32)   # padding, ok, out of range
    flag = err_flag()
    out, pool = _run(kda, x, flag=flag)
    assert flag.item() == kda.KDA_DEVERR_SLOT
    o_ref, p_ref, e = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool)
    assert e == 2  # one per head of the out-of-range sequence
    atol, rtol = tol_for(torch.bfloat16)
    assert torch.all(out[:70] == 0) and torch.all(out[90:] == 0)
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), atol, rtol, "outputs")
    assert_close(to_np64(pool), p_ref, atol, rtol, "states")


def test_prefill_tensor_core_path_padding_and_bad_slot():
    """The same slot rules on the tensor-core path (bf16, dk = dv = 128):
    padding and out-of-range sequences get zero outputs and leave the pool
    alone; the others match the oracle."""
    kda = _kda()
    x = inputs.prefill_inputs([130, 64, 70, 1], 2, 128, 128, dtype="bf16", num_slots=5, seed=12,
                              zero_state=False)
    x.slot_ids = torch.tensor([3, -1, 7, 0], dtype=torch.int32)   # ok, padding, out of range, ok
    flag = err_flag()
    pool_before = x.pool.clone()
    out, pool = _run(kda, x, init=True, flag=flag)
    assert flag.item() == kda.KDA_DEVERR_SLOT
    o_ref, p_ref, e = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                                     init_from_pool=True)
    assert e == 2  # one per head of the out-of-range sequence
    atol, rtol = tol_for(torch.bfloat16)
    assert torch.all(out[130:194] == 0) and torch.all(out[194:264] == 0)
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), atol, rtol, "outputs")
    assert_close(to_np64(pool), p_ref, atol, rtol, "states")
    for sl in (1, 2, 4):
        assert torch.equal(pool[sl].cpu(), pool_before[sl])


def test_prefill_bad_seqlens_and_workspace():
    kda = _kda()
    x = inputs.prefill_inputs([40, 40], 1, 32, 32, dtype="bf16", num_slots=2, seed=5)
    bad = x.cu_seqlens.clone()
    bad[1] = 50
    bad[2] = 45  # decreasing
    x2 = inputs.PrefillInputs(x.q, x.k, x.v, x.g, x.b, bad, x.pool, x.slot_ids)
    flag = err_flag()
    _run(kda, x2, flag=flag)
    assert flag.item() == kda.KDA_DEVERR_SEQLENS
    need = kda.prefill_workspace_bytes(1, 32, 32, kda.KDA_DT_BF16, 2, 80)
    small = torch.empty(max(need - 256, 1), dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError) as ei:
        _run(kda, x, workspace=small)
    assert ei.value.status == kda.KDA_ERR_WORKSPACE


def test_prefill_deterministic():
    kda = _kda()
    x = inputs.prefill_inputs([300, 77], 4, 128, 128, dtype="bf16", num_slots=3, seed=6)
    o1, p1 = _run(kda, x)
    o2, p2 = _run(kda, x)
    assert torch.equal(o1, o2) and torch.equal(p1, p2)


def test_prefill_strong_decay():
    """g = log sigmoid(N(-3, 1)) (alpha ~ 0.05 per token) stays finite."""
    kda = _kda()
    x = inputs.prefill_inputs([150], 2, 64, 64, dtype="f32", num_slots=1, seed=8, g_mean=-3.0)
    out, pool = _run(kda, x)
    o_ref, p_ref, _ = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool)
    atol, rtol = tol_for(torch.float32)
    assert torch.isfinite(out).all()
    assert_close(to_np64(out), o_ref, atol, rtol, "outputs")
    assert_close(to_np64(pool), p_ref, atol, rtol, "states")


@pytest.mark.parametrize("g_mean", [-3.0, 0.0, 6.0])
def test_prefill_decay_range_bf16_d128(g_mean):
    """Strong decay (alpha ~ 0.05 per token: some chunks take the exact
    per-element decay path), moderate decay, and almost no decay, on the
    dk = dv = 128 bf16 shape."""
    kda = _kda()
    x = inputs.prefill_inputs([150, 64], 2, 128, 128, dtype="bf16", num_slots=2, seed=9,
                              g_mean=g_mean, zero_state=False)
    out, pool = _run(kda, x, init=True)
    o_ref, p_ref, _ = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                                     init_from_pool=True)
    atol, rtol = tol_for(torch.bfloat16)
    assert torch.isfinite(out.float()).all()
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), atol, rtol, "outputs")
    assert_close(to_np64(pool), p_ref, atol, rtol, "states")


def _full_size_sampled(T, heads_checked, seed=0):
    kda = _kda()
    H, dk, dv = 32, 128, 128
    x = inputs.prefill_inputs([T], H, dk, dv, dtype="bf16", seed=seed, device="cuda")
    flag = err_flag()
    out = kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                              err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    atol, rtol = tol_for(torch.bfloat16)
    for h in heads_checked:
        sel = lambda t: t[:, h].cpu()  # noqa: E731
        o_ref, S_ref = oracle.recurrence(sel(x.q), sel(x.k), sel(x.v), sel(x.g), sel(x.b))
        assert_close(to_np64(out[:, h].cpu()), round_to(o_ref, torch.bfloat16), atol, rtol,
                     f"T={T} head {h} outputs")
        assert_close(to_np64(x.pool[int(x.slot_ids[0]), h].cpu()), S_ref, atol, rtol,
                     f"T={T} head {h} final state")


def test_prefill_full_size_t8192_sampled_heads():
    """1 sequence x 8192 tokens x 32 heads (the benchmark's prefill shape);
    every output and the final state of two heads against the oracle."""
    _full_size_sampled(8192, [0, 19])


def test_prefill_full_size_t102400_sampled_head():
    """The long-context prefill (102400 tokens x 32 heads); one head checked
    over all 1600 chunks."""
    _full_size_sampled(102400, [7], seed=1)
