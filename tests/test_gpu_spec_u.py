"""GPU checks of the ReplaySSM u-record variant ("2.8x faster Kimi K3
inference on CANN", section 04 "ReplaySSM"): verify writes u = beta (v - S'k^)
per value row, the commit applies S <- S diag(exp g) + u k^^T, and
kda_commit_verify_u does the previous window's commit and this window's
verify in one call (one launch on the CUDA-core shapes, the commit and the
verify launches on the tensor-core one).  Outputs and committed states are
compared with the fp64 oracle; the call is compared bit for bit with the
separate commit + verify calls."""
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for

pytestmark = pytest.mark.gpu

# (dtype, dk = dv, draft length): the first is the tensor-core verify shape
CASES = [("bf16", 128, 7), ("f32", 64, 5), ("bf16", 32, 12), ("bf16", 128, 3)]


def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


def _dev(x):
    return {k: v.cuda() if torch.is_tensor(v) else v for k, v in vars(x).items()}


@pytest.mark.parametrize("dtype,d,D", CASES)
def test_u_verify_equals_value_verify_and_commit_matches_oracle(dtype, d, D):
    kda = _kda()
    B, H = 6, 3
    x = inputs.verify_inputs(B, D, H, d, d, dtype=dtype, num_slots=9, seed=31 + d + D)
    x.slot_ids = torch.tensor([4, -1, 0, 7, 2, 5], dtype=torch.int32)
    x.num_accepted = torch.tensor([D, 3, 0, 1, min(2, D), D - 1], dtype=torch.int32)
    g = _dev(x)
    pool_v = g["pool"].clone()
    out_v, rec_v = kda.verify_record(g["q"], g["k"], g["v"], g["g"], g["b"], g["slot_ids"], pool_v)
    out_u, rec_u = kda.verify_record_u(g["q"], g["k"], g["v"], g["g"], g["b"], g["slot_ids"], g["pool"])
    torch.cuda.synchronize()
    # the same kernels: the same outputs, keys and gates, bit for bit
    assert torch.equal(out_u, out_v)
    assert torch.equal(rec_u["k_hat"], rec_v["k_hat"])
    assert torch.equal(rec_u["g"], rec_v["g"])
    assert torch.all(rec_u["u"][1] == 0)  # padding entry
    flag = err_flag()
    pool_u = g["pool"].clone()
    kda.replay_commit_u(rec_u, g["num_accepted"], g["slot_ids"], pool_u, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    atol, rtol = tol_for(inputs.torch_dtype(dtype))
    o_ref, r_ref, _ = oracle.verify(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool)
    p_ref, _ = oracle.replay(r_ref, x.num_accepted, x.slot_ids, x.pool)
    assert_close(to_np64(out_u), round_to(o_ref, inputs.torch_dtype(dtype)), atol, rtol, "outputs")
    assert_close(to_np64(pool_u), p_ref, atol, rtol, "u-record commit")
    # slots with nothing accepted and slots nobody names keep their bits
    for sl in (0, 1, 3, 6, 8):
        assert torch.equal(pool_u[sl].cpu(), x.pool[sl]), sl


@pytest.mark.parametrize("dtype,d,D", CASES)
def test_commit_verify_fused_equals_separate(dtype, d, D):
    """Window 1 verified into u records; window 2 either (a) after a separate
    u-record commit or (b) by the fused launch: the same committed state,
    outputs and records, bit for bit, and both match the oracle."""
    kda = _kda()
    B, H = 6, 3
    w1 = inputs.verify_inputs(B, D, H, d, d, dtype=dtype, num_slots=8, seed=41 + d)
    w2 = inputs.verify_inputs(B, D, H, d, d, dtype=dtype, num_slots=8, seed=42 + d)
    slots = torch.tensor([3, 0, -1, 6, 1, 5], dtype=torch.int32)
    acc1 = torch.tensor([D, 0, 2, 1, D - 1, 2], dtype=torch.int32)
    g1, g2 = _dev(w1), _dev(w2)
    dslots, dacc = slots.cuda(), acc1.cuda()
    pool0 = g1["pool"]
    _, rec1 = kda.verify_record_u(g1["q"], g1["k"], g1["v"], g1["g"], g1["b"], dslots, pool0)
    # (a) separate
    pool_a = pool0.clone()
    kda.replay_commit_u(rec1, dacc, dslots, pool_a)
    out_a, rec_a = kda.verify_record_u(g2["q"], g2["k"], g2["v"], g2["g"], g2["b"], dslots, pool_a)
    # (b) fused
    pool_b = pool0.clone()
    flag = err_flag()
    out_b, rec_b = kda.commit_verify_u(rec1, dacc, g2["q"], g2["k"], g2["v"], g2["g"], g2["b"], dslots,
                                       pool_b, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    assert torch.equal(pool_b, pool_a)
    assert torch.equal(out_b, out_a)
    for key in ("k_hat", "g", "u"):
        assert torch.equal(rec_b[key], rec_a[key]), key
    # the oracle: window 1's accepted prefix, then window 2 from that state
    atol, rtol = tol_for(inputs.torch_dtype(dtype))
    _, r1, _ = oracle.verify(w1.q, w1.k, w1.v, w1.g, w1.b, slots, w1.pool)
    p1, _ = oracle.replay(r1, acc1, slots, w1.pool)
    o2, _, _ = oracle.verify(w2.q, w2.k, w2.v, w2.g, w2.b, slots, torch.from_numpy(p1))
    assert_close(to_np64(pool_b), p1, atol, rtol, "committed state")
    assert_close(to_np64(out_b), round_to(o2, inputs.torch_dtype(dtype)), atol, rtol, "window 2 outputs")


def test_commit_verify_bad_accepted_length():
    kda = _kda()
    B, H, d, D = 3, 2, 128, 7
    w1 = inputs.verify_inputs(B, D, H, d, d, dtype="bf16", num_slots=4, seed=51)
    w2 = inputs.verify_inputs(B, D, H, d, d, dtype="bf16", num_slots=4, seed=52)
    g1, g2 = _dev(w1), _dev(w2)
    slots = g1["slot_ids"]
    _, rec1 = kda.verify_record_u(g1["q"], g1["k"], g1["v"], g1["g"], g1["b"], slots, g1["pool"])
    acc = torch.tensor([2, 9, -1], dtype=torch.int32, device="cuda")  # one valid, two out of range
    pool = g1["pool"].clone()
    flag = err_flag()
    kda.commit_verify_u(rec1, acc, g2["q"], g2["k"], g2["v"], g2["g"], g2["b"], slots, pool,
                        err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == kda.KDA_DEVERR_ACCEPTED
    for n in (1, 2):  # not committed
        sl = int(w1.slot_ids[n])
        assert torch.equal(pool[sl].cpu(), w1.pool[sl])


def test_u_records_full_size_b128_d7_h32():
    """The benchmark's verify shape: the commit + verify call against the
    separate calls, bit for bit, on a 4096-slot pool."""
    kda = _kda()
    B, D, H, d = 128, 7, 32, 128
    w1 = inputs.verify_inputs(B, D, H, d, d, dtype="bf16", num_slots=4096, seed=61, device="cuda")
    w2 = inputs.verify_inputs(B, D, H, d, d, dtype="bf16", num_slots=1, seed=62, device="cuda")
    slots, acc = w1.slot_ids, w1.num_accepted
    _, rec1 = kda.verify_record_u(w1.q, w1.k, w1.v, w1.g, w1.b, slots, w1.pool)
    pool_a = w1.pool.clone()
    kda.replay_commit_u(rec1, acc, slots, pool_a)
    out_a, rec_a = kda.verify_record_u(w2.q, w2.k, w2.v, w2.g, w2.b, slots, pool_a)
    out_b, rec_b = kda.commit_verify_u(rec1, acc, w2.q, w2.k, w2.v, w2.g, w2.b, slots, w1.pool)
    torch.cuda.synchronize()
    assert torch.equal(w1.pool, pool_a)
    assert torch.equal(out_b, out_a)
    assert torch.equal(rec_b["u"], rec_a["u"])
