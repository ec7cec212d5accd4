"""GPU parity of kda_decode against the fp64 oracle (through the C ABI)."""
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


def test_tiny_eight_sequential_decode_tokens_fp32():
    """2 sequences x 2 heads, dk = dv = 32, 8 decode calls, fp32, zero state."""
    kda = _kda()
    w = inputs.WORKLOADS["tiny_decode_2x2_d32_8tok_f32"]
    x = inputs.decode_inputs(w["B"], w["H"], w["dk"], w["dv"], dtype="f32",
                             num_slots=w["num_slots"], seed=0, g_mean=2.0,
                             zero_state=True, tokens=w["tokens"])
    pool_ref = to_np64(x.pool)
    pool = x.pool.cuda()
    slots = x.slot_ids.cuda()
    atol, rtol = tol_for(torch.float32)
    flag = err_flag()
    for t in range(w["tokens"]):
        out = kda.decode(x.q[t].cuda(), x.k[t].cuda(), x.v[t].cuda(), x.g[t].cuda(),
                         x.b[t].cuda(), slots, pool, err_flag=flag)
        o_ref, pool_ref, e = oracle.decode(x.q[t], x.k[t], x.v[t], x.g[t], x.b[t],
                                           x.slot_ids, pool_ref)
        assert e == 0
        assert_close(to_np64(out), o_ref, atol, rtol, f"token {t} output")
    torch.cuda.synchronize()
    assert flag.item() == 0
    got = to_np64(pool)
    assert_close(got, pool_ref, atol, rtol, "final states")
    untouched = [s for s in range(w["num_slots"]) if s not in set(x.slot_ids.tolist())]
    assert torch.equal(pool.cpu()[untouched], x.pool[untouched])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 128), (64, 128), (128, 32)])
def test_decode_parity_shapes(dtype, dk, dv):
    kda = _kda()
    B, H, NS = 7, 3, 11
    x = inputs.decode_inputs(B, H, dk, dv, dtype=dtype, num_slots=NS, seed=dk + dv,
                             g_mean=3.0, pool_std=0.02)
    slots = x.slot_ids.clone()
    slots[2] = -1           # padding
    slots[5] = NS + 3       # out of range -> error flag
    pool = x.pool.cuda()
    flag = err_flag()
    out = kda.decode(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(),
                     slots.cuda(), pool, err_flag=flag)
    o_ref, p_ref, e = oracle.decode(x.q, x.k, x.v, x.g, x.b, slots, x.pool)
    torch.cuda.synchronize()
    assert e == H
    assert flag.item() == kda.KDA_DEVERR_SLOT
    dt = inputs.torch_dtype(dtype)
    atol, rtol = tol_for(dt)
    assert_close(to_np64(out), round_to(o_ref, dt), atol, rtol, "outputs")
    assert torch.all(out[2] == 0) and torch.all(out[5] == 0)
    assert_close(to_np64(pool), p_ref, atol, rtol, "pool")
    touched = {int(s) for s in slots.tolist() if 0 <= s < NS}
    untouched = [s for s in range(NS) if s not in touched]
    assert torch.equal(pool.cpu()[untouched], x.pool[untouched])


def test_decode_deterministic_and_batch_order_invariant():
    kda = _kda()
    B, H, dk, dv, NS = 33, 4, 128, 128, 64
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=5)
    args = [t.cuda() for t in (x.q, x.k, x.v, x.g, x.b)]
    slots = x.slot_ids.cuda()
    p1 = x.pool.cuda()
    p2 = x.pool.cuda()
    o1 = kda.decode(*args, slots, p1)
    o2 = kda.decode(*args, slots, p2)
    assert torch.equal(o1, o2) and torch.equal(p1, p2)
    perm = torch.randperm(B, generator=torch.Generator().manual_seed(1)).cuda()
    p3 = x.pool.cuda()
    o3 = kda.decode(*[a[perm].contiguous() for a in args], slots[perm].contiguous(), p3)
    assert torch.equal(o3, o1[perm])
    assert torch.equal(p3, p1)


def test_decode_empty_batch_and_bad_arguments():
    kda = _kda()
    H, dk, dv = 2, 64, 64
    pool = torch.zeros((4, H, dv, dk), device="cuda")
    e = lambda *s: torch.empty(s, device="cuda")  # noqa: E731
    out = kda.decode(e(0, H, dk), e(0, H, dk), e(0, H, dv), e(0, H, dk), e(0, H),
                     torch.empty(0, dtype=torch.int32, device="cuda"), pool)
    assert out.shape == (0, H, dv)
    # unsupported head size is refused before any launch
    with pytest.raises(kda.KdaError) as ei:
        kda.decode(e(1, H, 48), e(1, H, 48), e(1, H, dv), e(1, H, 48), e(1, H),
                   torch.zeros(1, dtype=torch.int32, device="cuda"),
                   torch.zeros((4, H, dv, 48), device="cuda"))
    assert ei.value.status == kda.KDA_ERR_UNSUPPORTED


def test_decode_full_size_sampled():
    """256 sequences x 32 heads, dk = dv = 128, bf16, 4096-slot pool (8 GiB):
    the launch configuration the benchmark times; outputs and states checked
    on a sample of (sequence, head) pairs, untouched slots bit-exact."""
    kda = _kda()
    w = inputs.WORKLOADS["decode_b256_h32_d128_pool4096_bf16"]
    B, H, dk, dv, NS = w["B"], w["H"], w["dk"], w["dv"], w["num_slots"]
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=0,
                             g_mean=3.0, pool_std=0.02, device="cuda")
    rng = np.random.default_rng(0)
    sample_n = np.sort(rng.choice(B, 12, replace=False))
    sample_slots = x.slot_ids[torch.as_tensor(sample_n, device="cuda")].long()
    before = x.pool[sample_slots].cpu()          # [12, H, dv, dk]
    pool_before = x.pool.clone()
    flag = err_flag()
    out = kda.decode(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    sn = torch.as_tensor(sample_n)
    o_ref, p_ref, e = oracle.decode(x.q.cpu()[sn], x.k.cpu()[sn], x.v.cpu()[sn],
                                    x.g.cpu()[sn], x.b.cpu()[sn],
                                    torch.arange(len(sample_n), dtype=torch.int32), before)
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out.cpu()[sn]), round_to(o_ref, torch.bfloat16), atol, rtol, "outputs")
    assert_close(to_np64(x.pool[sample_slots].cpu()), p_ref, atol, rtol, "states")
    touched = torch.zeros(NS, dtype=torch.bool, device="cuda")
    touched[x.slot_ids.long()] = True
    assert torch.equal(x.pool[~touched], pool_before[~touched])


def test_decode_rows_per_cta_do_not_change_bits():
    """The launcher picks 64, 32 or 16 state rows per CTA from the grid size;
    the same tokens decoded as one large batch (64 rows per CTA) and as small
    slices (fewer rows per CTA) give the same bits."""
    kda = _kda()
    B, H, dk, dv, NS = 192, 8, 128, 128, 256
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=23)
    args = [t.cuda() for t in (x.q, x.k, x.v, x.g, x.b)]
    slots = x.slot_ids.cuda()
    p_big = x.pool.cuda()
    o_big = kda.decode(*args, slots, p_big)
    p_small = x.pool.cuda()
    outs = []
    for s0 in range(0, B, 3):
        sl = slice(s0, min(s0 + 3, B))
        outs.append(kda.decode(*[a[sl].contiguous() for a in args], slots[sl].contiguous(), p_small))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs), o_big)
    assert torch.equal(p_small, p_big)


def test_decode_full_size_1024x64_pool16384_sampled():
    """The long-context mix's decode batch: 1024 sequences x 64 heads over a
    16384-slot pool (64 GiB of state, so slot offsets run far past 2^32
    bytes).  Sampled sequences, including the highest slots, against the
    oracle; untouched slots bit-exact on a sample."""
    kda = _kda()
    B, H, dk, dv, NS = 1024, 64, 128, 128, 16384
    x = inputs.decode_inputs(B, H, dk, dv, dtype="bf16", num_slots=NS, seed=11, g_mean=3.0,
                             pool_std=0.02, device="cuda")
    order = torch.argsort(x.slot_ids.cpu())
    sample_n = torch.cat([order[-3:], order[:2], torch.tensor([5, 500, 1000])]).unique()
    sample_slots = x.slot_ids.cpu()[sample_n].long()
    before = x.pool[sample_slots.cuda()].cpu()
    touched = torch.zeros(NS, dtype=torch.bool)
    touched[x.slot_ids.cpu().long()] = True
    probe = torch.nonzero(~touched).flatten()[-4:]  # untouched slots near the top of the pool
    probe_before = x.pool[probe.cuda()].cpu()
    flag = err_flag()
    out = kda.decode(x.q, x.k, x.v, x.g, x.b, x.slot_ids, x.pool, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    sn = sample_n
    o_ref, p_ref, e = oracle.decode(x.q.cpu()[sn], x.k.cpu()[sn], x.v.cpu()[sn], x.g.cpu()[sn],
                                    x.b.cpu()[sn], torch.arange(len(sn), dtype=torch.int32), before)
    atol, rtol = tol_for(torch.bfloat16)
    assert_close(to_np64(out.cpu()[sn]), round_to(o_ref, torch.bfloat16), atol, rtol, "outputs")
    assert_close(to_np64(x.pool[sample_slots.cuda()].cpu()), p_ref, atol, rtol, "states")
    assert torch.equal(x.pool[probe.cuda()].cpu(), probe_before)


def test_decode_in_cuda_graph_equals_eager():
    """Decode steps captured in a CUDA graph (as the long-context mix runs
    them) give the same bits as the same calls issued eagerly."""
    kda = _kda()
    H, steps = 32, 16
    x = inputs.decode_inputs(1, H, 128, 128, dtype="bf16", num_slots=1, seed=7, device="cuda",
                             tokens=steps, zero_state=False)
    slots = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool_e = x.pool.clone()
    out_e = torch.empty((steps, 1, H, 128), dtype=torch.bfloat16, device="cuda")
    for t in range(steps):
        kda.decode(x.q[t], x.k[t], x.v[t], x.g[t], x.b[t], slots, pool_e, out_e[t])
    pool_g = x.pool.clone()
    out_g = torch.empty_like(out_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for t in range(steps):
            kda.decode(x.q[t], x.k[t], x.v[t], x.g[t], x.b[t], slots, pool_g, out_g[t], stream=s)
    pool_g.copy_(x.pool)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e)
    assert torch.equal(pool_g, pool_e)
