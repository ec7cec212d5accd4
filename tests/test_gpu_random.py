"""Seeded randomized parity sweeps over shapes, dtypes, lengths and slot
patterns (prefill, verify + commit) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for

pytestmark = pytest.mark.gpu

SHAPES = [(128, 128, "bf16"), (64, 64, "f32"), (128, 64, "bf16"), (32, 32, "f32")]


def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


@pytest.mark.parametrize("seed", [101, 202, 303])
def test_prefill_random_ragged_batches(seed):
    kda = _kda()
    rng = np.random.default_rng(seed)
    for dk, dv, dtype in SHAPES:
        n = int(rng.integers(1, 7))
        lens = [int(x) for x in rng.integers(0, 300, size=n)]
        H = int(rng.integers(1, 4))
        ns = n + 2
        x = inputs.prefill_inputs(lens, H, dk, dv, dtype=dtype, num_slots=ns, seed=seed + dk,
                                  zero_state=False, pool_std=0.05,
                                  g_mean=float(rng.choice([-2.0, 3.0, 6.0])))
        init = bool(rng.integers(0, 2))
        pool = x.pool.cuda()
        flag = err_flag()
        out = kda.prefill_chunked(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(),
                                  x.cu_seqlens.cuda(), x.slot_ids.cuda(), pool,
                                  init_from_pool=init, err_flag=flag)
        torch.cuda.synchronize()
        assert flag.item() == 0
        o_ref, p_ref, e = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                                         init_from_pool=init)
        assert e == 0
        dt = inputs.torch_dtype(dtype)
        atol, rtol = tol_for(dt)
        tag = f"{dk}x{dv} {dtype} lens {lens} H {H} init {init}"
        assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, f"outputs, {tag}")
        assert_close(to_np64(pool), p_ref, atol, rtol, f"states, {tag}")


@pytest.mark.parametrize("seed", [11, 22, 33])
def test_verify_commit_random(seed):
    kda = _kda()
    rng = np.random.default_rng(seed)
    for dk, dv, dtype in SHAPES:
        B = int(rng.integers(1, 24))
        D = int(rng.integers(1, 17))
        H = int(rng.integers(1, 4))
        NS = B + 4
        x = inputs.verify_inputs(B, D, H, dk, dv, dtype=dtype, num_slots=NS, seed=seed + D,
                                 g_mean=float(rng.choice([-2.0, 3.0])))
        slots = x.slot_ids.clone()
        if B > 2:
            slots[int(rng.integers(0, B))] = -1
        pool = x.pool.cuda()
        pool_before = pool.clone()
        out, rec = kda.verify_record(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(),
                                     slots.cuda(), pool)
        torch.cuda.synchronize()
        assert torch.equal(pool, pool_before)
        o_ref, _, e = oracle.verify(x.q, x.k, x.v, x.g, x.b, slots, x.pool)
        assert e == 0
        dt = inputs.torch_dtype(dtype)
        atol, rtol = tol_for(dt)
        tag = f"{dk}x{dv} {dtype} B {B} D {D} H {H}"
        assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, f"verify outputs, {tag}")
        acc = torch.as_tensor(rng.integers(0, D + 1, size=B), dtype=torch.int32)
        flag = err_flag()
        kda.replay_commit(rec, acc.cuda(), slots.cuda(), pool, err_flag=flag)
        torch.cuda.synchronize()
        assert flag.item() == 0
        p_ref = to_np64(x.pool)
        for nn in range(B):
            a, s = int(acc[nn]), int(slots[nn])
            if a == 0 or s < 0:
                continue
            for hh in range(H):
                _, S = oracle.recurrence(x.q[nn, :a, hh], x.k[nn, :a, hh], x.v[nn, :a, hh],
                                         x.g[nn, :a, hh], x.b[nn, :a, hh], S0=p_ref[s, hh])
                p_ref[s, hh] = S
        assert_close(to_np64(pool), p_ref, atol, rtol, f"committed states, {tag}")
