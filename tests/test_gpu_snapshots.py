"""GPU parity of kda_prefill_chunked_snapshots: the state at chosen chunk
boundaries written into pool slots (the KDA Prefix-Cache of "Ascend day-0
support for Kimi K3", Kimi K3 overview).  Each snapshot is compared with the
fp64 oracle's token recurrence over its prefix, and a prefill resumed from a
snapshot with init_from_pool is compared with the one-shot prefill."""
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for

pytestmark = pytest.mark.gpu

LENS = [300, 130, 64, 0]
# (sequence, tokens, destination slot), sorted by sequence then tokens
REQS = [(0, 64, 5), (0, 192, 6), (0, 256, 7), (1, 128, 8), (2, 64, 9)]


def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


def _snap_tensors(reqs):
    cols = list(zip(*reqs))
    return tuple(torch.tensor(c, dtype=torch.int32, device="cuda") for c in cols)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_snapshots_match_oracle_prefixes(dtype, d):
    kda = _kda()
    H = 3
    x = inputs.prefill_inputs(LENS, H, d, d, dtype=dtype, num_slots=11, seed=21, zero_state=False,
                              pool_std=0.05)
    x.slot_ids = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    pool = x.pool.cuda()
    flag = err_flag()
    out = kda.prefill_chunked(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(),
                              x.cu_seqlens.cuda(), x.slot_ids.cuda(), pool, init_from_pool=True,
                              snapshots=_snap_tensors(REQS), err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    dt = inputs.torch_dtype(dtype)
    atol, rtol = tol_for(dt)
    o_ref, p_ref, e = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                                     init_from_pool=True)
    assert e == 0
    assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, "outputs")
    assert_close(to_np64(pool[:4]), p_ref[:4], atol, rtol, "final states")
    cu = x.cu_seqlens.tolist()
    for s, t, sl in REQS:
        t0 = cu[s]
        for h in range(H):
            sel = lambda a: a[t0:t0 + t, h]  # noqa: E731
            _, S_ref = oracle.recurrence(sel(x.q), sel(x.k), sel(x.v), sel(x.g), sel(x.b),
                                         S0=x.pool[int(x.slot_ids[s]), h])
            assert_close(to_np64(pool[sl, h]), S_ref, atol, rtol, f"snapshot seq {s} at {t} head {h}")
    # untouched slots keep their bits
    assert torch.equal(pool[10].cpu(), x.pool[10])


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_resume_from_snapshot_matches_one_shot(dtype, d):
    """Prefill 300 tokens with a snapshot at 256, then prefill tokens 256..299
    from that snapshot: outputs and final state match the one-shot run."""
    kda = _kda()
    H = 2
    x = inputs.prefill_inputs([300], H, d, d, dtype=dtype, num_slots=3, seed=22, zero_state=False,
                              pool_std=0.05)
    x.slot_ids = torch.tensor([0], dtype=torch.int32)
    dev = lambda t: t.cuda()  # noqa: E731
    pool = dev(x.pool)
    out = kda.prefill_chunked(dev(x.q), dev(x.k), dev(x.v), dev(x.g), dev(x.b), dev(x.cu_seqlens),
                              dev(x.slot_ids), pool, init_from_pool=True,
                              snapshots=_snap_tensors([(0, 256, 1)]))
    tail = slice(256, 300)
    cu2 = torch.tensor([0, 44], dtype=torch.int32, device="cuda")
    out2 = kda.prefill_chunked(dev(x.q[tail]).contiguous(), dev(x.k[tail]).contiguous(),
                               dev(x.v[tail]).contiguous(), dev(x.g[tail]).contiguous(),
                               dev(x.b[tail]).contiguous(), cu2,
                               torch.tensor([1], dtype=torch.int32, device="cuda"), pool,
                               init_from_pool=True)
    torch.cuda.synchronize()
    atol, rtol = tol_for(inputs.torch_dtype(dtype))
    assert_close(to_np64(out2), to_np64(out[tail]), atol, rtol, "resumed outputs")
    assert_close(to_np64(pool[1]), to_np64(pool[0]), atol, rtol, "resumed final state")


@pytest.mark.parametrize("d", [128, 64])
def test_bad_snapshot_requests_are_skipped_and_flagged(d):
    kda = _kda()
    H = 2
    x = inputs.prefill_inputs([200, 64], H, d, d, dtype="bf16", num_slots=8, seed=23,
                              zero_state=False)
    x.slot_ids = torch.tensor([0, 1], dtype=torch.int32)
    reqs = [(0, 64, 2),    # valid
            (0, 100, 3),   # not a multiple of 64
            (0, 256, 4),   # beyond the sequence
            (1, 64, 9),    # slot out of range
            (1, 64, -1)]   # padding: skipped silently
    pool = x.pool.cuda()
    flag = err_flag()
    kda.prefill_chunked(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(),
                        x.cu_seqlens.cuda(), x.slot_ids.cuda(), pool, init_from_pool=True,
                        snapshots=_snap_tensors(reqs), err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == kda.KDA_DEVERR_SNAPSHOT
    atol, rtol = tol_for(torch.bfloat16)
    for h in range(H):
        _, S_ref = oracle.recurrence(x.q[:64, h], x.k[:64, h], x.v[:64, h], x.g[:64, h], x.b[:64, h],
                                     S0=x.pool[0, h])
        assert_close(to_np64(pool[2, h]), S_ref, atol, rtol, f"valid snapshot head {h}")
    for sl in (3, 4, 5, 6, 7):
        assert torch.equal(pool[sl].cpu(), x.pool[sl])


def test_snapshots_full_size_t8192():
    """The benchmark's 8192-token, 32-head prefill with a snapshot every 1024
    tokens; two snapshots of two heads against the oracle."""
    kda = _kda()
    T, H = 8192, 32
    x = inputs.prefill_inputs([T], H, 128, 128, dtype="bf16", num_slots=9, seed=24, device="cuda")
    x.slot_ids = torch.tensor([0], dtype=torch.int32, device="cuda")
    reqs = [(0, 1024 * (i + 1), 1 + i) for i in range(8)]
    flag = err_flag()
    kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                        snapshots=_snap_tensors(reqs), err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    atol, rtol = tol_for(torch.bfloat16)
    for t, sl in ((1024, 1), (5120, 5)):
        for h in (3, 30):
            sel = lambda a: a[:t, h].cpu()  # noqa: E731
            _, S_ref = oracle.recurrence(sel(x.q), sel(x.k), sel(x.v), sel(x.g), sel(x.b))
            assert_close(to_np64(x.pool[sl, h]), S_ref, atol, rtol, f"snapshot at {t} head {h}")
    # the last snapshot (8192 tokens) is the final state itself
    assert torch.equal(x.pool[8], x.pool[0])
