"""GPU parity of the pipelined tensor-core prefill: when a few (sequence,
head) chains each walk many chunks, the chunks are cut into segments and
segment k's prep runs beside segment k - 1's chain.  The library takes about
sqrt(mean chunks per sequence / 10) segments (rounded up after the length
is fixed), each of at least 64 chunks and at least 2048 prep CTAs, when
(sequences x heads) is at most the SM count; the last segment takes the
rest.  These batches take that path (5 and 4 segments); outputs, final
states and snapshots on both sides of segment boundaries are compared with
the fp64 oracle."""
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for

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


def test_five_segments_mixed_batch():
    """Five sequences (60000, 26000, 100, 0 and 300 tokens; the third is
    padding) x 8 heads: 1350 chunks, 270 per sequence on average, so five
    segments of 64 chunks (the last takes the rest); the short sequences lie
    in the first only.  Snapshots at a segment boundary (4096 tokens), one
    chunk past it and deep in the last segment."""
    seg = 64 * 64
    lens = [60000, 26000, 100, 0, 300]
    slots = [0, 1, -1, 2, 3]
    reqs = [(0, seg, 4), (0, seg + 64, 5), (1, 25600, 6), (4, 256, 7)]
    x, pool, out = _run(lens, slots, 8, reqs, num_slots=9, seed=41)
    cu = x.cu_seqlens.tolist()
    assert torch.all(out[cu[2]:cu[3]] == 0)          # padding sequence: zero outputs
    assert torch.equal(pool[8].cpu(), x.pool[8])     # a slot nobody names keeps its bits


def test_four_segments_one_sequence():
    """One sequence of 3 x 8192 + 337 tokens x 16 heads (390 chunks): three
    segments of 128 chunks and a last one of 6 ending in a partial chunk;
    snapshots at two segment boundaries and at the last whole chunk."""
    seg = 128 * 64
    T = 3 * seg + 337
    reqs = [(0, seg, 1), (0, 2 * seg, 2), (0, 3 * seg + 320, 3)]
    _run([T], [0], 16, reqs, num_slots=4, seed=42)


def test_two_uneven_segments_one_sequence():
    """One sequence of 8172 tokens x 32 heads (128 chunks, the last partial):
    two segments, the first holding 72 % of the chunks (92).  Snapshots at
    the boundary, one chunk past it and at the last whole chunk."""
    reqs = [(0, 92 * 64, 1), (0, 93 * 64, 2), (0, 127 * 64, 3)]
    _run([8172], [0], 32, reqs, num_slots=4, seed=43)
