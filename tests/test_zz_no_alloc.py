"""pkv_paged_attn_static: attention for callers that cannot allocate device memory.

Such callers (a process whose device memory another framework's caching
allocator owns, code inside an allocator or stream callback, or a loop that
must not take cudaMalloc's device-wide synchronisation) cannot hand
pkv_paged_attn a workspace, so this entry point keeps its work lists and
split-KV partials in a fixed static device array.  These tests call it through
the C ABI and check it against the CPU oracle and, bit for bit, against
pkv_paged_attn on the same batch (both run the same plan), on two calls in a
row; check that calls on different pools and streams, issued back to back
without a host synchronisation, do not disturb one another in the shared
array; and check that a batch too large for the array is refused.  This file
is collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_25_gb300 import pkv
from paged_kv_attention_25_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_25_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


class Case:
    """A batch appended into its own pool, with its pkv_paged_attn result and the oracle's."""

    def __init__(self, batch):
        self.b = b = batch
        self.pool = pkv.Pool(b.num_blocks, b.num_kv_heads, b.head_dim)
        wl.fill_pool(b, self.pool.k, self.pool.v)
        self.d = d = wl.upload(b)
        self.meta = pkv.HostMeta(b.cu_q_lens, b.ctx_lens, b.q_positions)
        pkv.pkv_append(self.pool, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])
        self.ref_o, self.ref_lse = pkv.pkv_paged_attn(self.pool, d["q"], d["q_positions"], d["block_tables"],
                                                      d["ctx_lens"], d["cu_q_lens"], self.meta, b.scale)
        torch.cuda.synchronize()
        kp, vp = b.pool_arrays()
        oracle.append(kp, vp, b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
        self.O, self.L = oracle.paged_attn(b.q, kp, vp, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions,
                                           b.scale)

    def static_call(self, out=None, lse=None, stream=None):
        d = self.d
        return pkv.pkv_paged_attn_static(self.pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                         d["cu_q_lens"], self.meta, self.b.scale, out=out, lse=lse, stream=stream)

    def check(self, o, lse, what):
        assert torch.equal(o, self.ref_o) and torch.equal(lse, self.ref_lse), f"{what}: differs from pkv_paged_attn"
        o64 = o.float().cpu().numpy().astype(np.float64)
        err = np.abs(o64 - self.O)
        assert (err <= ATOL + RTOL * np.abs(self.O)).all(), f"{what}: max err {err.max():.3e} against the oracle"
        assert np.abs(lse.cpu().numpy() - self.L).max() <= LSE_TOL, f"{what}: LSE against the oracle"


def test_static_scratch_matches_workspace_entry_point_and_oracle_twice():
    reqs = [wl._decode(30000), wl._new_turn(3000, 100), wl._decode(500), wl._recompute(2000, 64, 16)]
    c = Case(wl.build_batch("no_alloc", reqs, num_q_heads=8, num_kv_heads=2, head_dim=128, seed=77))
    stats = pkv.pkv_last_plan_stats(c.pool)
    assert stats["num_partial_rows"] > 0, "the batch must put split partials into the scratch"
    assert stats["workspace_bytes"] <= pkv.PKV_STATIC_SCRATCH_BYTES
    built_before = stats["plans_built"]
    for call in range(2):
        o, lse = c.static_call()
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_errors(c.pool) == 0
        c.check(o, lse, f"call {call}")
    # The same metadata reuses the pool's cached plan: no call above planned again.
    assert pkv.pkv_last_plan_stats(c.pool)["plans_built"] == built_before


def test_static_calls_on_two_pools_back_to_back():
    """Calls on different pools share the array: each call's upload must wait for the previous
    call's kernels, on one stream and across two streams, with no host synchronisation between."""
    a = Case(wl.build_batch("no_alloc_a", [wl._decode(20000), wl._new_turn(1000, 300), wl._decode(70)],
                            num_q_heads=8, num_kv_heads=2, head_dim=128, seed=78))
    b = Case(wl.build_batch("no_alloc_b", [wl._decode(9000), wl._decode(12000), wl._recompute(3000, 500, 40)],
                            num_q_heads=4, num_kv_heads=4, head_dim=128, seed=79))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for rnd in range(3):
        streams = (None, None) if rnd == 0 else (s1, s2) if rnd == 1 else (s2, s1)
        for case, st in zip((a, b, a, b), streams + streams):
            o = torch.empty_like(case.ref_o)
            lse = torch.empty_like(case.ref_lse)
            case.static_call(out=o, lse=lse, stream=st)
            outs.append((case, o, lse, rnd))
    torch.cuda.synchronize()
    for case in (a, b):
        assert pkv.pkv_check_device_errors(case.pool) == 0
    for i, (case, o, lse, rnd) in enumerate(outs):
        case.check(o, lse, f"round {rnd} call {i}")


def test_static_scratch_refuses_batch_above_its_limit():
    # 600,000 one-token requests make 600,000 work items (48 bytes each): more
    # than the static array holds, whatever the split policy.
    R = 600_000
    pool = pkv.Pool(1, 1, 64)
    q = torch.zeros((R, 1, 64), dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(R, dtype=torch.int32, device="cuda")
    bt = torch.zeros((R, 1), dtype=torch.int32, device="cuda")
    ctx = torch.ones(R, dtype=torch.int32, device="cuda")
    cu = torch.arange(R + 1, dtype=torch.int32, device="cuda")
    meta = pkv.HostMeta(np.arange(R + 1, dtype=np.int32), np.ones(R, np.int32), np.zeros(R, np.int32))
    assert pkv.pkv_paged_attn_workspace_size(pool, 1, meta) > pkv.PKV_STATIC_SCRATCH_BYTES
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_attn_static(pool, q, pos, bt, ctx, cu, meta, 0.125)
    assert e.value.code == pkv.PKV_EINVAL
    assert "static limit" in str(e.value)
