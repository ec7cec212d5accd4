"""GPU parity of the ReplaySSM verify/commit pair against the fp64 oracle."""
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


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv,D", [(32, 32, 1), (64, 64, 7), (128, 128, 7), (128, 64, 16)])
def test_verify_parity_records_and_pool_untouched(dtype, dk, dv, D):
    kda = _kda()
    B, H, NS = 5, 3, 9
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype=dtype, num_slots=NS, seed=dk + D)
    slots = x.slot_ids.clone()
    slots[1] = -1
    pool = x.pool.cuda()
    pool_before = pool.clone()
    flag = err_flag()
    out, rec = kda.verify_record(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(),
                                 x.b.cuda(), slots.cuda(), pool, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    assert torch.equal(pool, pool_before)
    o_ref, r_ref, e = oracle.verify(x.q, x.k, x.v, x.g, x.b, slots, x.pool)
    dt = inputs.torch_dtype(dtype)
    atol, rtol = tol_for(dt)
    assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, "verify outputs")
    assert torch.all(out[1] == 0)
    # records: normalised key (fp32 rounding of the fp64 value), bit copies of
    # v and g, and beta = sigmoid(b)
    assert_close(to_np64(rec["k_hat"]), r_ref["k_hat"], 1e-6, 1e-5, "k_hat records")
    assert torch.equal(rec["v"].cpu(), x.v)
    assert torch.equal(rec["g"].cpu(), x.g)
    assert_close(to_np64(rec["beta"]), r_ref["beta"], 1e-7, 1e-6, "beta records")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(32, 64), (128, 128)])
def test_replay_equals_decode_bitwise_and_oracle(dtype, dk, dv):
    kda = _kda()
    B, D, H, NS = 8, 7, 2, 12
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype=dtype, num_slots=NS, seed=3 + dk)
    acc = torch.tensor([0, 1, 2, 3, 4, 5, 6, 7], dtype=torch.int32)
    pool_v = x.pool.cuda()
    slots = x.slot_ids.cuda()
    _, rec = kda.verify_record(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(),
                               x.b.cuda(), slots, pool_v)
    pool_r = x.pool.cuda()
    flag = err_flag()
    kda.replay_commit(rec, acc.cuda(), slots, pool_r, err_flag=flag)
    # reference 1: the decode kernel applied a_n times (bit-exact expected)
    pool_d = x.pool.cuda()
    for j in range(D):
        live = (acc > j)
        if not live.any():
            break
        idx = torch.nonzero(live).flatten()
        kda.decode(*[t[idx, j].contiguous().cuda() for t in (x.q, x.k, x.v, x.g, x.b)],
                   slots[idx.cuda()].contiguous(), pool_d)
    torch.cuda.synchronize()
    assert flag.item() == 0
    assert torch.equal(pool_r, pool_d), "replay differs from repeated decode"
    # reference 2: fp64 recurrence over the accepted prefix of the ORIGINAL inputs
    p_ref = to_np64(x.pool)
    for n in range(B):
        a = int(acc[n])
        s = int(x.slot_ids[n])
        for h in range(H):
            if a == 0:
                continue
            _, S = oracle.recurrence(x.q[n, :a, h], x.k[n, :a, h], x.v[n, :a, h],
                                     x.g[n, :a, h], x.b[n, :a, h], S0=p_ref[s, h])
            p_ref[s, h] = S
    atol, rtol = tol_for(inputs.torch_dtype(dtype))
    assert_close(to_np64(pool_r), p_ref, atol, rtol, "committed states")
    # a = 0 leaves the slot's bytes untouched
    s0 = int(x.slot_ids[0])
    assert torch.equal(pool_r[s0].cpu(), x.pool[s0])


def test_verify_outputs_match_sequential_decode():
    """Verify evaluates the draft window in chunk form; its outputs agree with
    D sequential decode calls within the output tolerance (the committed
    state is what must match decode bit for bit, and does: see the replay
    test above)."""
    kda = _kda()
    B, D, H, dk, dv, NS = 6, 7, 4, 128, 128, 16
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype="bf16", num_slots=NS, seed=17)
    slots = x.slot_ids.cuda()
    out, _ = kda.verify_record(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(),
                               x.b.cuda(), slots, x.pool.cuda())
    pool_d = x.pool.cuda()
    atol, rtol = tol_for(torch.bfloat16)
    for j in range(D):
        oj = kda.decode(*[t[:, j].contiguous().cuda() for t in (x.q, x.k, x.v, x.g, x.b)],
                        slots, pool_d)
        assert_close(to_np64(out[:, j]), to_np64(oj), atol, rtol, f"draft token {j}")


@pytest.mark.parametrize("D", [3, 8])
def test_verify_many_items_per_cta(D):
    """800 (sequence, head) items, more than the GPU has SMs, so the pipelined
    kernel's CTAs cycle both buffers several times; padding and out-of-range
    slots are mixed in.  Every output and record checked."""
    kda = _kda()
    B, H, dk, dv, NS = 200, 4, 128, 128, 256
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype="bf16", num_slots=NS, seed=40 + D)
    slots = x.slot_ids.clone()
    slots[7] = -1
    slots[100] = NS + 5
    slots[199] = -1
    pool = x.pool.cuda()
    pool_before = pool.clone()
    flag = err_flag()
    out, rec = kda.verify_record(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(),
                                 x.b.cuda(), slots.cuda(), pool, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == kda.KDA_DEVERR_SLOT
    assert torch.equal(pool, pool_before)
    o_ref, r_ref, e = oracle.verify(x.q, x.k, x.v, x.g, x.b, slots, x.pool)
    assert e == H
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), atol, rtol, "verify outputs")
    for n in (7, 100, 199):
        assert torch.all(out[n] == 0)
    assert_close(to_np64(rec["k_hat"]), r_ref["k_hat"], 1e-6, 1e-5, "k_hat records")
    assert torch.equal(rec["v"].cpu(), x.v)
    assert torch.equal(rec["g"].cpu(), x.g)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("g_mean,D", [(-14.0, 8), (-8.0, 16), (-8.0, 8), (-6.0, 8), (-3.0, 7),
                                      (6.0, 16), (6.0, 5), (3.0, 9)])
def test_verify_decay_range(dtype, g_mean, D):
    """Near-total decay (alpha ~ 1e-6 and 3e-4 per token: the window's decay
    products fall below 1e-30 and underflow), strong, negligible and typical
    decay, over windows that take each verify path (bf16 windows of up to 8
    tokens at dk = dv = 128 use the window + tensor-core state kernels, whose
    factored window products give way to running products when a decay
    product drops below 1e-30: at g_mean -14 and -8 every window does, at -6
    the factored form runs with decay products down to ~4e-25)."""
    kda = _kda()
    B, H, dk, dv, NS = 4, 2, 128, 128, 6
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype=dtype, num_slots=NS, seed=31 + D,
                             g_mean=g_mean)
    out, _ = kda.verify_record(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(),
                               x.b.cuda(), x.slot_ids.cuda(), x.pool.cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    o_ref, _, e = oracle.verify(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool)
    assert e == 0
    dt = inputs.torch_dtype(dtype)
    atol, rtol = tol_for(dt)
    assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, "verify outputs")


def test_replay_rejects_bad_accepted_length_and_slot():
    kda = _kda()
    B, D, H, dk, dv, NS = 3, 4, 2, 64, 64, 6
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype="bf16", num_slots=NS, seed=2)
    slots = x.slot_ids.clone()
    _, rec = kda.verify_record(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(),
                               x.b.cuda(), slots.cuda(), x.pool.cuda())
    pool = x.pool.cuda()
    flag = err_flag()
    kda.replay_commit(rec, torch.tensor([D + 1, 0, 2], dtype=torch.int32).cuda(),
                      slots.cuda(), pool, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == kda.KDA_DEVERR_ACCEPTED
    assert torch.equal(pool[int(slots[0])].cpu(), x.pool[int(slots[0])])
    assert not torch.equal(pool[int(slots[2])].cpu(), x.pool[int(slots[2])])
    flag.zero_()
    slots2 = slots.clone()
    slots2[2] = NS
    kda.replay_commit(rec, torch.tensor([1, 1, 2], dtype=torch.int32).cuda(),
                      slots2.cuda(), x.pool.cuda(), err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == kda.KDA_DEVERR_SLOT
    with pytest.raises(kda.KdaError):
        kda.verify_record(*[torch.zeros((1, 17, H, d), device="cuda", dtype=torch.bfloat16)
                            for d in (dk, dk, dv)],
                          torch.zeros((1, 17, H, dk), device="cuda"),
                          torch.zeros((1, 17, H), device="cuda", dtype=torch.bfloat16),
                          torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.zeros((1, H, dv, dk), device="cuda"))


def test_verify_commit_full_size_sampled():
    """128 sequences x 7 draft tokens x 32 heads, dk = dv = 128, bf16, 4096-slot
    pool, accepted length uniform on 0..7: the configuration the benchmark
    times.  Sampled sequences are checked against the oracle."""
    kda = _kda()
    w = inputs.WORKLOADS["verify_commit_b128_d7_h32_d128_bf16"]
    B, D, H, dk, dv, NS = w["B"], w["D"], w["H"], w["dk"], w["dv"], w["num_slots"]
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype="bf16", num_slots=NS, seed=0,
                             device="cuda")
    rng = np.random.default_rng(1)
    sn = torch.as_tensor(np.sort(rng.choice(B, 8, replace=False)))
    ss = x.slot_ids.cpu()[sn].long()
    before = x.pool[ss.cuda()].cpu()
    pool_before = x.pool.clone()
    flag = err_flag()
    out, rec = kda.verify_record(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool, err_flag=flag)
    torch.cuda.synchronize()
    assert torch.equal(x.pool, pool_before)
    kda.replay_commit(rec, x.num_accepted, x.slot_ids, x.pool, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    cpu = lambda t: t.cpu()[sn]  # noqa: E731
    local = torch.arange(len(sn), dtype=torch.int32)
    o_ref, r_ref, _ = oracle.verify(cpu(x.q), cpu(x.k), cpu(x.v), cpu(x.g), cpu(x.b),
                                    local, before)
    p_ref, _ = oracle.replay(r_ref, cpu(x.num_accepted), local, before)
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out.cpu()[sn]), round_to(o_ref, torch.bfloat16), atol, rtol,
                 "verify outputs")
    assert_close(to_np64(x.pool[ss.cuda()].cpu()), p_ref, atol, rtol, "committed states")
    touched = torch.zeros(NS, dtype=torch.bool, device="cuda")
    touched[x.slot_ids.long()[x.num_accepted > 0]] = True
    assert torch.equal(x.pool[~touched], pool_before[~touched])


def _verify_with(kda, x, workspace, stream=None):
    args = [t.cuda() for t in (x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool)]
    out, rec = kda.verify_record(*args, workspace=workspace, stream=stream)
    return out, rec


@pytest.mark.parametrize("D", [1, 5, 8])
def test_verify_workspace_contents_do_not_matter(D):
    """The window + state kernels (bf16, dk = dv = 128, D <= 8) pass a scratch
    record through the caller's workspace.  Whatever the workspace held before
    (here NaN bit patterns), every byte the state kernel uses is written first:
    outputs and records are the same bits as with a zeroed workspace."""
    kda = _kda()
    B, H, NS = 6, 4, 10
    x = inputs.verify_inputs(B, D, H, 128, 128, dtype="bf16", num_slots=NS, seed=70 + D)
    need = kda.verify_workspace_bytes(H, 128, 128, kda.KDA_DT_BF16, B, D)
    assert need == B * H * 12928
    ws0 = torch.zeros(need, dtype=torch.uint8, device="cuda")
    wsn = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # all-ones: NaN floats
    out0, rec0 = _verify_with(kda, x, ws0)
    outn, recn = _verify_with(kda, x, wsn)
    torch.cuda.synchronize()
    assert torch.isfinite(outn.float()).all()
    assert torch.equal(out0, outn)
    for key in ("k_hat", "v", "g", "beta"):
        assert torch.equal(rec0[key], recn[key]), key


def test_verify_workspace_reused_across_batches():
    """One workspace serving two different batches in turn (and a side
    stream): the second batch gets the same bits as with fresh scratch, and
    both match the oracle."""
    kda = _kda()
    H, D, NS = 4, 7, 16
    xa = inputs.verify_inputs(8, D, H, 128, 128, dtype="bf16", num_slots=NS, seed=81)
    xb = inputs.verify_inputs(5, D, H, 128, 128, dtype="bf16", num_slots=NS, seed=82, g_mean=-5.0)
    need = kda.verify_workspace_bytes(H, 128, 128, kda.KDA_DT_BF16, 8, D)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        out_a, _ = _verify_with(kda, xa, ws, stream=side)
        out_b, rec_b = _verify_with(kda, xb, ws, stream=side)
    side.synchronize()
    out_b2, rec_b2 = _verify_with(kda, xb, None)
    torch.cuda.synchronize()
    assert torch.equal(out_b, out_b2)
    for key in ("k_hat", "v", "g", "beta"):
        assert torch.equal(rec_b[key], rec_b2[key]), key
    atol, rtol = tol_for(torch.bfloat16)
    for x, out in ((xa, out_a), (xb, out_b)):
        o_ref, _, e = oracle.verify(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool)
        assert e == 0
        assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), atol, rtol, "verify outputs")


def test_verify_rejects_missing_or_small_workspace():
    kda = _kda()
    B, D, H = 2, 7, 2
    x = inputs.verify_inputs(B, D, H, 128, 128, dtype="bf16", num_slots=4, seed=5)
    need = kda.verify_workspace_bytes(H, 128, 128, kda.KDA_DT_BF16, B, D)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError) as ei:
        _verify_with(kda, x, small)
    assert ei.value.status == -4  # KDA_ERR_WORKSPACE
