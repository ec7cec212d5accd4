"""GPU parity of kda_prefill_fused (ShortConv along each sequence + the
tensor-core chunked prefill + gated RMS norm) against the fp64 oracle in
oracle/megakda.py, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for
from oracle import megakda

pytestmark = pytest.mark.gpu
D = 128

# The fused prefill's outputs are divided by their token's RMS, which the
# plain prefill's outputs (bf16 bound: 2e-3 absolute + 1e-2 relative) are
# not: with outputs of typical magnitude ~0.4 the plain path's absolute bound
# becomes about 5e-3 on the normalised scale.  States and conv states keep
# the plain bound (bit-exactness for the conv states).
ATOL_OUT, RTOL_OUT = 5e-3, 1e-2


def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


def _split_w(conv_w):
    w = to_np64(conv_w)
    return w[:, :D], w[:, D:2 * D], w[:, 2 * D:]


def _run(lens, slots, H, num_slots, seed, init_from_pool, eps_o=1e-5, conv_scale=1.0):
    kda = _kda()
    oracle.set_threads(16)
    x = inputs.prefill_inputs(lens, H, D, D, dtype="bf16", num_slots=num_slots, seed=seed,
                              zero_state=False, pool_std=0.05)
    x.slot_ids = torch.tensor(slots, dtype=torch.int32)
    T = int(x.cu_seqlens[-1])
    ex = inputs.fused_prefill_extras(T, len(lens), H, D, D, dtype="bf16", num_slots=num_slots, seed=seed)
    ex.conv_w = ex.conv_w * conv_scale
    pool, cst = x.pool.cuda(), ex.conv_state.cuda()
    flag = err_flag()
    out = kda.prefill_fused(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(), ex.z.cuda(),
                            x.cu_seqlens.cuda(), x.slot_ids.cuda(), pool, cst, ex.conv_w.cuda(),
                            ex.norm_w.cuda(), init_from_pool=init_from_pool, eps_o=eps_o, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    wq, wk, wv = _split_w(ex.conv_w)
    o_ref, p_ref, c_ref, e = megakda.prefill_fused(x.q, x.k, x.v, x.g, x.b, ex.z, wq, wk, wv,
                                                   to_np64(ex.norm_w), x.cu_seqlens, x.slot_ids, x.pool,
                                                   ex.conv_state, init_from_pool=init_from_pool, eps_o=eps_o)
    assert e == 0
    return x, ex, pool, cst, out, o_ref, p_ref, c_ref


@pytest.mark.parametrize("init_from_pool", [True, False])
def test_fused_prefill_mixed_batch(init_from_pool):
    """Sequences of 300, 130, 2, 0 and 64 tokens x 3 heads, the fourth
    padding: outputs, states and conv states (bit-exact: raw inputs)."""
    lens = [300, 130, 2, 0, 64]
    slots = [4, 0, 2, -1, 5]
    x, ex, pool, cst, out, o_ref, p_ref, c_ref = _run(lens, slots, 3, 7, 51, init_from_pool)
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), ATOL_OUT, RTOL_OUT, "outputs")
    live = [4, 0, 2, 5]
    assert_close(to_np64(pool[live]), p_ref[live], atol, rtol, "states")
    assert np.array_equal(to_np64(cst), c_ref)
    cu = x.cu_seqlens.tolist()
    assert torch.all(out[cu[3]:cu[4]] == 0)
    for sl in (1, 3, 6):  # slots nobody names keep their bits
        assert torch.equal(pool[sl].cpu(), x.pool[sl])
        assert torch.equal(cst[sl].cpu(), ex.conv_state[sl])


def test_fused_prefill_then_fused_decode():
    """A fused prefill of 200 and 3 tokens, then 3 fused decode steps per
    sequence from the state and conv state it left: against the oracle's
    prefill followed by its decodes."""
    kda = _kda()
    lens = [200, 3]
    slots = [1, 0]
    H = 2
    x, ex, pool, cst, out, o_ref, p_ref, c_ref = _run(lens, slots, H, 2, 52, True)
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), ATOL_OUT, RTOL_OUT, "prefill outputs")
    wq, wk, wv = _split_w(ex.conv_w)
    y = inputs.decode_inputs(2, H, D, D, dtype="bf16", num_slots=2, seed=53, tokens=3)
    dz = inputs.fused_extras(2, H, D, D, dtype="bf16", num_slots=2, seed=53).z
    sl = torch.tensor(slots, dtype=torch.int32)
    for t in range(3):
        o = kda.decode_fused(y.q[t].cuda(), y.k[t].cuda(), y.v[t].cuda(), y.g[t].cuda(), y.b[t].cuda(),
                             dz.cuda(), sl.cuda(), pool, cst, ex.conv_w.cuda(), ex.norm_w.cuda(), eps_o=1e-5)
        o2, p_ref, c_ref, e = megakda.decode_fused(y.q[t], y.k[t], y.v[t], y.g[t], y.b[t], dz, wq, wk, wv,
                                                   to_np64(ex.norm_w), sl, p_ref, c_ref, eps_o=1e-5)
        assert e == 0
        assert_close(to_np64(o), round_to(o2, torch.bfloat16), atol, rtol, f"decode step {t}")
    torch.cuda.synchronize()
    assert_close(to_np64(pool), p_ref, atol, rtol, "states")
    assert np.array_equal(to_np64(cst), c_ref)


def test_fused_prefill_pipelined_segments():
    """One sequence of 3 x 8192 + 337 tokens x 16 heads, which the library
    pipelines in seven growing segments: the conv history crosses chunk and
    segment boundaries and the conv state is written by the last segment's
    chain."""
    lens = [3 * 8192 + 337]
    x, ex, pool, cst, out, o_ref, p_ref, c_ref = _run(lens, [0], 16, 2, 54, True)
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), ATOL_OUT, RTOL_OUT, "outputs")
    assert_close(to_np64(pool[:1]), p_ref[:1], atol, rtol, "state")
    assert np.array_equal(to_np64(cst), c_ref)


def test_fused_prefill_saturated_conv():
    """Conv taps 40 times the usual ones (pre-activations of about N(0, 40^2)):
    a few percent of the SiLU arguments lie beyond +-88, where e^{-x} leaves
    the fp32 range, in the k/q conv of step 0 and in v's conv inside beta
    V^T; the approximate exponential and reciprocal must give -0 and x there
    (no NaN), and the prefill still matches the oracle."""
    lens = [200, 70]
    x, ex, pool, cst, out, o_ref, p_ref, c_ref = _run(lens, [0, 1], 2, 2, 58, True, conv_scale=40.0)
    w = to_np64(ex.conv_w)
    raw = np.concatenate([to_np64(x.q), to_np64(x.k), to_np64(x.v)], axis=-1)  # [T, H, nc]
    pre = sum(w[None, :, :, j] * raw[j:raw.shape[0] - 3 + j] for j in range(4))  # windows inside the batch
    assert (pre < -88).sum() > 100 and (pre > 88).sum() > 100
    assert torch.isfinite(out).all() and torch.isfinite(pool).all()
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), ATOL_OUT, RTOL_OUT, "outputs")
    # the chain's fp16 operands round relative to the magnitudes of the state
    # and the WY factors, here up to about 45 instead of about 1 (v ~ 40x):
    # the absolute part of the bound scales with the largest |state|
    s_atol = atol * max(1.0, float(np.abs(p_ref[:2]).max()))
    assert_close(to_np64(pool[:2]), p_ref[:2], s_atol, rtol, "states")
    assert np.array_equal(to_np64(cst), c_ref)


def test_fused_prefill_unsupported_shape_launches_nothing():
    kda = _kda()
    H, d = 2, 64
    x = inputs.prefill_inputs([70], H, d, d, dtype="bf16", num_slots=1, seed=55, device="cuda")
    ex = inputs.fused_prefill_extras(70, 1, H, d, d, dtype="bf16", num_slots=1, seed=55, device="cuda")
    p0, c0 = x.pool.clone(), ex.conv_state.clone()
    with pytest.raises(kda.KdaError) as ei:
        kda.prefill_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.cu_seqlens, x.slot_ids, x.pool, ex.conv_state,
                          ex.conv_w, ex.norm_w)
    assert ei.value.status == kda.KDA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.equal(x.pool, p0) and torch.equal(ex.conv_state, c0)
