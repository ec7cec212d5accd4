"""Canary pages around every buffer the library writes (compute-sanitizer
is not available here, so out-of-bounds writes are looked for this way).

Each output, record, conv-state, pool and workspace buffer is the middle of
a larger allocation whose first and last 4 KiB hold a byte pattern; after
the call those bytes must be unchanged.  Buffers the call only reads (the
verify's pool) must be unchanged entirely.  The shapes cover the
tensor-core paths (bf16, dk = dv = 128) and the CUDA-core ones (fp32, other
head sizes), ragged and empty sequences, padding slots, and snapshots."""
import pytest
import torch

from gated_delta_rule_decode_gb300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


def _kda():
    from gated_delta_rule_decode_gb300 import kda
    return kda


class Guarded:
    """Tensors carved out of allocations with canary pages on both sides."""

    def __init__(self):
        self.bufs = []

    def like(self, t: torch.Tensor) -> torch.Tensor:
        g = self.empty(t.shape, t.dtype)
        g.copy_(t)
        return g

    def empty(self, shape, dtype) -> torch.Tensor:
        n = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.bufs.append((buf, n))
        return buf[GUARD:GUARD + n].view(dtype).view(shape)

    def workspace(self, nbytes: int) -> torch.Tensor:
        return self.empty((nbytes,), torch.uint8)

    def check(self):
        torch.cuda.synchronize()
        for i, (buf, n) in enumerate(self.bufs):
            head, tail = buf[:GUARD], buf[GUARD + n:]
            assert torch.all(head == PATTERN), f"buffer {i}: bytes before it were written"
            assert torch.all(tail == PATTERN), f"buffer {i}: bytes after it were written"


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 32), ("bf16", 32, 64)])
def test_decode_canaries(dtype, dk, dv):
    kda = _kda()
    x = inputs.decode_inputs(5, 3, dk, dv, dtype=dtype, num_slots=7, seed=1, device="cuda")
    x.slot_ids[1] = -1  # a padding entry
    gd = Guarded()
    pool = gd.like(x.pool)
    out = gd.empty((5, 3, dv), x.q.dtype)
    kda.decode(x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool, out)
    gd.check()


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_fused_decode_canaries(dtype, d):
    kda = _kda()
    x = inputs.decode_inputs(3, 2, d, d, dtype=dtype, num_slots=4, seed=2, device="cuda")
    ex = inputs.fused_extras(3, 2, d, d, dtype=dtype, num_slots=4, seed=2, device="cuda")
    gd = Guarded()
    pool, cst = gd.like(x.pool), gd.like(ex.conv_state)
    out = gd.empty((3, 2, d), x.q.dtype)
    kda.decode_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.slot_ids, pool, cst, ex.conv_w, ex.norm_w, out)
    gd.check()


def _guarded_records(gd, B, D, H, dk, dv, dt):
    return dict(k_hat=gd.empty((B, D, H, dk), torch.float32), v=gd.empty((B, D, H, dv), dt),
                g=gd.empty((B, D, H, dk), torch.float32), beta=gd.empty((B, D, H), torch.float32))


def _guarded_records_u(gd, B, D, H, dk, dv):
    return dict(k_hat=gd.empty((B, D, H, dk), torch.float32), g=gd.empty((B, D, H, dk), torch.float32),
                u=gd.empty((B, D, H, dv), torch.float32))


@pytest.mark.parametrize("dtype,dk,dv,D", [("bf16", 128, 128, 7), ("f32", 64, 64, 5), ("bf16", 128, 128, 12)])
def test_verify_and_commit_canaries(dtype, dk, dv, D):
    kda = _kda()
    B, H = 3, 2
    x = inputs.verify_inputs(B, D, H, dk, dv, dtype=dtype, num_slots=5, seed=3, device="cuda")
    gd = Guarded()
    pool = gd.like(x.pool)
    pool0 = pool.clone()
    code = kda.KDA_DT_BF16 if dtype == "bf16" else kda.KDA_DT_F32
    need = kda.verify_workspace_bytes(H, dk, dv, code, B, D)
    ws = gd.workspace(need) if need > 0 else None
    out = gd.empty((B, D, H, dv), x.q.dtype)
    rec = _guarded_records(gd, B, D, H, dk, dv, x.q.dtype)
    kda.verify_record(x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool, out, rec, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(pool, pool0)  # verify only reads the pool
    kda.replay_commit(rec, x.num_accepted, x.slot_ids, pool)
    gd.check()
    # the u-record variant and the commit-then-verify call
    out_u = gd.empty((B, D, H, dv), x.q.dtype)
    rec_u = _guarded_records_u(gd, B, D, H, dk, dv)
    kda.verify_record_u(x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool, out_u, rec_u, workspace=ws)
    kda.replay_commit_u(rec_u, x.num_accepted, x.slot_ids, pool)
    out2 = gd.empty((B, D, H, dv), x.q.dtype)
    rec2 = _guarded_records_u(gd, B, D, H, dk, dv)
    kda.commit_verify_u(rec_u, x.num_accepted, x.q, x.k, x.v, x.g, x.b, x.slot_ids, pool, out2, rec2,
                        workspace=ws)
    gd.check()


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 64), ("bf16", 32, 128)])
def test_prefill_canaries(dtype, dk, dv):
    kda = _kda()
    lens = [70, 0, 130, 64, 1]
    H = 2
    x = inputs.prefill_inputs(lens, H, dk, dv, dtype=dtype, num_slots=9, seed=4, device="cuda",
                              zero_state=False)
    x.slot_ids = torch.tensor([0, 1, -1, 3, 4], dtype=torch.int32, device="cuda")
    gd = Guarded()
    pool = gd.like(x.pool)
    T = sum(lens)
    out = gd.empty((T, H, dv), x.q.dtype)
    code = kda.KDA_DT_BF16 if dtype == "bf16" else kda.KDA_DT_F32
    ws = gd.workspace(kda.prefill_workspace_bytes(H, dk, dv, code, len(lens), T))
    snaps = (torch.tensor([0, 3], dtype=torch.int32, device="cuda"),
             torch.tensor([64, 64], dtype=torch.int32, device="cuda"),
             torch.tensor([5, 6], dtype=torch.int32, device="cuda"))
    kda.prefill_chunked(x.q, x.k, x.v, x.g, x.b, x.cu_seqlens, x.slot_ids, pool, out, init_from_pool=True,
                        workspace=ws, snapshots=snaps)
    gd.check()


def test_prefill_fused_canaries():
    kda = _kda()
    lens = [100, 3, 200]
    H, d = 2, 128
    x = inputs.prefill_inputs(lens, H, d, d, dtype="bf16", num_slots=4, seed=5, device="cuda",
                              zero_state=False)
    ex = inputs.fused_prefill_extras(sum(lens), len(lens), H, d, d, dtype="bf16", num_slots=4, seed=5,
                                     device="cuda")
    gd = Guarded()
    pool, cst = gd.like(x.pool), gd.like(ex.conv_state)
    T = sum(lens)
    out = gd.empty((T, H, d), x.q.dtype)
    ws = gd.workspace(kda.prefill_workspace_bytes(H, d, d, kda.KDA_DT_BF16, len(lens), T))
    kda.prefill_fused(x.q, x.k, x.v, x.g, x.b, ex.z, x.cu_seqlens, x.slot_ids, pool, cst, ex.conv_w, ex.norm_w,
                      out, init_from_pool=True, workspace=ws)
    gd.check()
