"""The long-context mix end to end: a 102 400-token chunked prefill of one
sequence (32 heads, dk = dv = 128, bf16), then 256 decode steps on the
prefill's final state, captured in one CUDA graph as the benchmark runs them.
Every prefill and decode output of the checked heads, and their state after
the last decode step, are compared element by element with the fp64 oracle's
token recurrence over all 102 656 tokens ("2.8x faster Kimi K3 inference on
CANN", section 01: 100K input and 256 output tokens at batch 1)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_decode_gb300 import inputs
from kda_testutil import assert_close, err_flag, round_to, to_np64, tol_for

pytestmark = pytest.mark.gpu


def test_longmix_prefill_then_256_graph_decodes_match_oracle():
    from gated_delta_rule_decode_gb300 import kda
    T, H, d, steps = 102400, 32, 128, 256
    x = inputs.prefill_inputs([T], H, d, d, dtype="bf16", seed=0, device="cuda")
    y = inputs.decode_inputs(1, H, d, d, dtype="bf16", num_slots=1, seed=7, device="cuda",
                             tokens=steps)
    flag = err_flag()
    out_p = kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, x.pool,
                                err_flag=flag)
    # the decode steps run on the slot the prefill wrote
    slots = x.slot_ids.clone()
    out_d = torch.empty((steps, 1, H, d), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    pool_after_prefill = x.pool.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for t in range(steps):
            kda.decode(y.q[t], y.k[t], y.v[t], y.g[t], y.b[t], slots, x.pool, out_d[t], stream=s)
    x.pool.copy_(pool_after_prefill)  # capture launches nothing; start from the prefill's state
    graph.replay()
    torch.cuda.synchronize()
    assert flag.item() == 0
    atol, rtol = tol_for(torch.bfloat16)
    slot = int(x.slot_ids[0])
    for h in (7, 25):
        cat = lambda a, b: torch.cat([a[:, h].cpu(), b[:, 0, h].cpu()])  # noqa: E731
        o_ref, S_ref = oracle.recurrence(cat(x.q, y.q), cat(x.k, y.k), cat(x.v, y.v),
                                         cat(x.g, y.g), cat(x.b, y.b))
        assert o_ref.shape == (T + steps, d)
        assert_close(to_np64(out_p[:, h]), round_to(o_ref[:T], torch.bfloat16), atol, rtol,
                     f"head {h}: prefill outputs")
        assert_close(to_np64(out_d[:, 0, h]), round_to(o_ref[T:], torch.bfloat16), atol, rtol,
                     f"head {h}: the 256 decode outputs")
        assert_close(to_np64(x.pool[slot, h]), S_ref, atol, rtol,
                     f"head {h}: state after the 256 decode steps")
    assert np.isfinite(to_np64(x.pool)).all()
