"""GPU parity of kda_decode_fused (ShortConv + decode step + RMS norm and
sigmoid gate) against the fp64 oracle in oracle/megakda.py, through the C ABI."""
import numpy as np
import pytest
import torch

from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for
from oracle import megakda

pytestmark = pytest.mark.gpu


def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


def _split_w(conv_w, dk):
    w = to_np64(conv_w)
    return w[:, :dk], w[:, dk:2 * dk], w[:, 2 * dk:]


def _oracle_step(x, ex, slots, pool, cpool, dk, eps_o):
    wq, wk, wv = _split_w(ex.conv_w, dk)
    return megakda.decode_fused(x.q, x.k, x.v, x.g, x.b, ex.z, wq, wk, wv, to_np64(ex.norm_w),
                                slots, pool, cpool, eps_o=eps_o)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 128), (64, 128), (128, 32)])
def test_fused_decode_parity_shapes(dtype, dk, dv):
    kda = _kda()
    B, H, NS = 7, 3, 11
    x = inputs.decode_inputs(B, H, dk, dv, dtype=dtype, num_slots=NS, seed=dk + 3 * dv)
    ex = inputs.fused_extras(B, H, dk, dv, dtype=dtype, num_slots=NS, seed=dk + 3 * dv)
    slots = x.slot_ids.clone()
    slots[2] = -1           # padding
    slots[5] = NS + 3       # out of range -> error flag
    pool, cst = x.pool.cuda(), ex.conv_state.cuda()
    flag = err_flag()
    out = kda.decode_fused(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(), ex.z.cuda(),
                           slots.cuda(), pool, cst, ex.conv_w.cuda(), ex.norm_w.cuda(),
                           eps_o=1e-5, err_flag=flag)
    o_ref, p_ref, c_ref, e = _oracle_step(x, ex, slots, x.pool, ex.conv_state, dk, 1e-5)
    torch.cuda.synchronize()
    assert e == H
    assert flag.item() == kda.KDA_DEVERR_SLOT
    dt = inputs.torch_dtype(dtype)
    atol, rtol = tol_for(dt)
    assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, "outputs")
    assert torch.all(out[2] == 0) and torch.all(out[5] == 0)
    assert_close(to_np64(pool), p_ref, atol, rtol, "pool")
    # the conv state holds raw inputs: the shift is exact
    assert np.array_equal(to_np64(cst), c_ref)
    touched = {int(s) for s in slots.tolist() if 0 <= s < NS}
    untouched = [s for s in range(NS) if s not in touched]
    assert torch.equal(pool.cpu()[untouched], x.pool[untouched])
    assert torch.equal(cst.cpu()[untouched], ex.conv_state[untouched])


def test_fused_decode_sequence_from_empty_conv_state():
    """A new sequence: conv state and KDA state start at zero, then 6 fused
    decode steps in a row against 6 oracle steps."""
    kda = _kda()
    B, H, dk, dv, NS, steps = 3, 2, 128, 128, 4, 6
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=31, tokens=steps,
                             zero_state=True)
    ex = inputs.fused_extras(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=31)
    cst0 = torch.zeros_like(ex.conv_state)
    pool, cst = x.pool.cuda(), cst0.cuda()
    p_ref, c_ref = to_np64(x.pool), to_np64(cst0)
    wq, wk, wv = _split_w(ex.conv_w, dk)
    z = ex.z.cuda()
    atol, rtol = tol_for(torch.bfloat16)
    flag = err_flag()
    for t in range(steps):
        out = kda.decode_fused(x.q[t].cuda(), x.k[t].cuda(), x.v[t].cuda(), x.g[t].cuda(),
                               x.b[t].cuda(), z, x.slot_ids.cuda(), pool, cst, ex.conv_w.cuda(),
                               ex.norm_w.cuda(), err_flag=flag)
        o_ref, p_ref, c_ref, e = megakda.decode_fused(x.q[t], x.k[t], x.v[t], x.g[t], x.b[t], ex.z,
                                                      wq, wk, wv, to_np64(ex.norm_w), x.slot_ids,
                                                      p_ref, c_ref)
        assert e == 0
        assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), atol, rtol, f"step {t} output")
    torch.cuda.synchronize()
    assert flag.item() == 0
    assert_close(to_np64(pool), p_ref, atol, rtol, "states")
    assert np.array_equal(to_np64(cst), c_ref)


def test_fused_decode_deterministic_and_batch_order_invariant():
    kda = _kda()
    B, H, dk, dv, NS = 33, 4, 128, 128, 64
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=5)
    ex = inputs.fused_extras(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=5)
    args = [t.cuda() for t in (x.q, x.k, x.v, x.g, x.b, ex.z)]
    slots = x.slot_ids.cuda()
    w, nw = ex.conv_w.cuda(), ex.norm_w.cuda()
    runs = []
    for perm in (None, None, torch.randperm(B, generator=torch.Generator().manual_seed(1)).cuda()):
        p, c = x.pool.cuda(), ex.conv_state.cuda()
        a = args if perm is None else [t[perm].contiguous() for t in args]
        s = slots if perm is None else slots[perm].contiguous()
        o = kda.decode_fused(*a, s, p, c, w, nw)
        runs.append((o if perm is None else o[torch.argsort(perm)], p, c))
    torch.cuda.synchronize()
    for o, p, c in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(p, runs[0][1]) and torch.equal(c, runs[0][2])


def test_fused_decode_bad_arguments_launch_nothing():
    kda = _kda()
    B, H, dk, dv, NS = 2, 2, 64, 64, 4
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=2, device="cuda")
    ex = inputs.fused_extras(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=2, device="cuda")
    pool0, c0 = x.pool.clone(), ex.conv_state.clone()
    with pytest.raises(kda.KdaError) as ei:
        kda.decode_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.slot_ids, x.pool, ex.conv_state,
                         ex.conv_w, ex.norm_w, eps_o=-1.0)
    assert ei.value.status == kda.KDA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(x.pool, pool0) and torch.equal(ex.conv_state, c0)
    # empty batch: nothing launched, nothing changed
    e = lambda *s, dt=torch.bfloat16: torch.empty(s, device="cuda", dtype=dt)  # noqa: E731
    out = kda.decode_fused(e(0, H, dk), e(0, H, dk), e(0, H, dv), e(0, H, dk, dt=torch.float32),
                           e(0, H), e(0, H, dv), torch.empty(0, dtype=torch.int32, device="cuda"),
                           x.pool, ex.conv_state, ex.conv_w, ex.norm_w)
    assert out.shape == (0, H, dv)
    assert torch.equal(x.pool, pool0) and torch.equal(ex.conv_state, c0)


def test_fused_decode_full_size_sampled():
    """256 sequences x 32 heads, dk = dv = 128, bf16, 4096-slot pool: sampled
    (sequence) outputs, states and conv states against the oracle; untouched
    slots of both pools bit-exact."""
    kda = _kda()
    B, H, dk, dv, NS = 256, 32, 128, 128, 4096
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=0, device="cuda")
    ex = inputs.fused_extras(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=0, device="cuda")
    sn = torch.as_tensor(np.sort(np.random.default_rng(0).choice(B, 10, replace=False)))
    ss = x.slot_ids.cpu()[sn].long()
    before, cbefore = x.pool[ss.cuda()].cpu(), ex.conv_state[ss.cuda()].cpu()
    pool0, c0 = x.pool.clone(), ex.conv_state.clone()
    flag = err_flag()
    out = kda.decode_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.slot_ids, x.pool, ex.conv_state,
                           ex.conv_w, ex.norm_w, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    wq, wk, wv = _split_w(ex.conv_w, dk)
    o_ref, p_ref, c_ref, e = megakda.decode_fused(
        x.q.cpu()[sn], x.k.cpu()[sn], x.v.cpu()[sn], x.g.cpu()[sn], x.b.cpu()[sn], ex.z.cpu()[sn],
        wq, wk, wv, to_np64(ex.norm_w), torch.arange(len(sn), dtype=torch.int32), before, cbefore)
    assert e == 0
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out.cpu()[sn]), round_to(o_ref, torch.bfloat16), atol, rtol, "outputs")
    assert_close(to_np64(x.pool[ss.cuda()].cpu()), p_ref, atol, rtol, "states")
    assert np.array_equal(to_np64(ex.conv_state[ss.cuda()].cpu()), c_ref)
    touched = torch.zeros(NS, dtype=torch.bool, device="cuda")
    touched[x.slot_ids.long()] = True
    assert torch.equal(x.pool[~touched], pool0[~touched])
    assert torch.equal(ex.conv_state[~touched], c0[~touched])


def _preactivations(x, ex, dk):
    """The conv pre-activations w . (x_{t-3}, x_{t-2}, x_{t-1}, x_t) of every
    (sequence, head, channel) of the step, from the slots' conv states."""
    slots = x.slot_ids.long()
    hist = to_np64(ex.conv_state[slots])                          # [B, H, 3, nc]
    cur = np.concatenate([to_np64(x.q), to_np64(x.k), to_np64(x.v)], axis=-1)  # [B, H, nc]
    w = to_np64(ex.conv_w)                                        # [H, nc, 4]
    return (w[None, :, :, 0] * hist[:, :, 0] + w[None, :, :, 1] * hist[:, :, 1] +
            w[None, :, :, 2] * hist[:, :, 2] + w[None, :, :, 3] * cur)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_fused_decode_saturated_conv(dtype):
    """Conv taps 40 times the usual ones: a few percent of the SiLU arguments
    lie beyond +-88, where e^{-x} leaves the fp32 range, so the fast
    exponential and division must give silu(x) = -0 for x << 0 and x for
    x >> 0 (no NaN), and the step still matches the oracle."""
    kda = _kda()
    B, H, NS, d = 7, 3, 9, 128
    x = inputs.decode_inputs(B, H, d, d, dtype=dtype, num_slots=NS, seed=77)
    ex = inputs.fused_extras(B, H, d, d, dtype=dtype, num_slots=NS, seed=77)
    ex.conv_w = ex.conv_w * 40.0
    pre = _preactivations(x, ex, d)
    assert (pre < -88).sum() > 20 and (pre > 88).sum() > 20
    pool, cst = x.pool.cuda(), ex.conv_state.cuda()
    flag = err_flag()
    out = kda.decode_fused(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(), ex.z.cuda(),
                           x.slot_ids.cuda(), pool, cst, ex.conv_w.cuda(), ex.norm_w.cuda(),
                           eps_o=1e-5, err_flag=flag)
    o_ref, p_ref, c_ref, e = _oracle_step(x, ex, x.slot_ids, x.pool, ex.conv_state, d, 1e-5)
    torch.cuda.synchronize()
    assert e == 0 and flag.item() == 0
    assert torch.isfinite(out).all() and torch.isfinite(pool).all()
    dt = inputs.torch_dtype(dtype)
    atol, rtol = tol_for(dt)
    assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, "outputs")
    assert_close(to_np64(pool), p_ref, atol, rtol, "pool")
    assert np.array_equal(to_np64(cst), c_ref)
