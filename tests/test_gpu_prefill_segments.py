"""GPU parity of the pipelined tensor-core prefill: when a few (sequence,
head) chains each walk many chunks, the chunks are cut into segments and
segment k's prep runs beside segment k - 1's chain.  The library sizes the
segments as a geometric series (ratio 0.16 x free SMs / chains, at least
16 chunks, chunks / 50 and 256 prep CTAs each) when (sequences x heads) is
below the SM count; the last segment takes the rest.  These batches take
that path with shrinking (32 chains) and growing (8 and 16 chains)
segments; outputs, final states and snapshots on both sides of segment
boundaries are compared with the fp64 oracle."""
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, segment_starts, to_np64, tol_for

pytestmark = pytest.mark.gpu




def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


def _run(lens, slots, H, reqs, num_slots, seed):
    kda = _kda()
    oracle.set_threads(16)
    x = inputs.prefill_inputs(lens, H, 128, 128, dtype="bf16", num_slots=num_slots, seed=seed,
                              zero_state=False, pool_std=0.05)
    x.slot_ids = torch.tensor(slots, dtype=torch.int32)
    pool = x.pool.cuda()
    flag = err_flag()
    snaps = tuple(torch.tensor(c, dtype=torch.int32, device="cuda") for c in zip(*reqs)) if reqs else None
    out = kda.prefill_chunked(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda(), x.b.cuda(),
                              x.cu_seqlens.cuda(), x.slot_ids.cuda(), pool, init_from_pool=True,
                              snapshots=snaps, err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0
    atol, rtol = tol_for(torch.bfloat16)
    o_ref, p_ref, e = oracle.prefill(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                                     init_from_pool=True)
    assert e == 0
    assert_close(to_np64(out), round_to(o_ref, torch.bfloat16), atol, rtol, "outputs")
    live = sorted(s for s in slots if s >= 0)
    assert_close(to_np64(pool[live]), p_ref[live], atol, rtol, "final states")
    cu = x.cu_seqlens.tolist()
    for s, t, sl in reqs:
        for h in range(H):
            sel = lambda a: a[cu[s]:cu[s] + t, h]  # noqa: E731
            _, S_ref = oracle.recurrence(sel(x.q), sel(x.k), sel(x.v), sel(x.g), sel(x.b),
                                         S0=x.pool[slots[s], h])
            assert_close(to_np64(pool[sl, h]), S_ref, atol, rtol, f"snapshot seq {s} at {t} head {h}")
    return x, pool, out


def _starts(lens, H):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_seq = (sum(lens) + 63) // 64 // len(lens)
    return segment_starts(len(lens) * H, sms, per_seq)


def test_segments_mixed_batch():
    """Five sequences (60000, 26000, 100, 0 and 300 tokens; the third is
    padding) x 8 heads: 1350 chunks, 270 per sequence on average, in growing
    segments; the short sequences lie in the first only.  Snapshots at the
    second segment's start, one chunk past it and deep in the last
    segment."""
    lens = [60000, 26000, 100, 0, 300]
    lo = _starts(lens, 8)
    assert len(lo) >= 3, lo
    b = lo[1] * 64
    slots = [0, 1, -1, 2, 3]
    reqs = [(0, b, 4), (0, b + 64, 5), (1, 25600, 6), (4, 256, 7)]
    x, pool, out = _run(lens, slots, 8, reqs, num_slots=9, seed=41)
    cu = x.cu_seqlens.tolist()
    assert torch.all(out[cu[2]:cu[3]] == 0)          # padding sequence: zero outputs
    assert torch.equal(pool[8].cpu(), x.pool[8])     # a slot nobody names keeps its bits


def test_growing_segments_one_sequence():
    """One sequence of 3 x 8192 + 337 tokens x 16 heads (390 chunks, the last
    partial): growing segments; snapshots at two segment boundaries and at
    the last whole chunk."""
    T = 3 * 8192 + 337
    lo = _starts([T], 16)
    assert len(lo) >= 4, lo
    reqs = [(0, lo[1] * 64, 1), (0, lo[-1] * 64, 2), (0, 3 * 8192 + 320, 3)]
    _run([T], [0], 16, reqs, num_slots=4, seed=42)


def test_shrinking_segments_one_sequence():
    """One sequence of 8172 tokens x 32 heads (128 chunks, the last partial):
    shrinking segments.  Snapshots at the first boundary, one chunk past it,
    at the last boundary and at the last whole chunk."""
    lo = _starts([8172], 32)
    assert len(lo) >= 3, lo
    reqs = [(0, lo[1] * 64, 1), (0, lo[1] * 64 + 64, 2), (0, lo[-1] * 64, 3), (0, 127 * 64, 4)]
    _run([8172], [0], 32, reqs, num_slots=5, seed=43)
