"""pkv_paged_attn_static: attention for callers that cannot allocate device memory.

Such callers (a process whose device memory another framework's caching
allocator owns, code inside an allocator or stream callback, or a loop that
must not take cudaMalloc's device-wide synchronisation) cannot hand
pkv_paged_attn a workspace, so this entry point keeps its work lists and
split-KV partials in a fixed static device array.  These tests call it through
the C ABI and compare it with pkv_paged_attn, twice in a row, and check that a
batch too large for the array is refused.  This file is collected last.
"""
import numpy as np
import pytest
import torch

from paged_kv_attention_25_gb300 import pkv
from paged_kv_attention_25_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_25_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def test_static_scratch_matches_workspace_entry_point_twice():
    reqs = [wl._decode(30000), wl._new_turn(3000, 100), wl._decode(500), wl._recompute(2000, 64, 16)]
    b = wl.build_batch("no_alloc", reqs, num_q_heads=8, num_kv_heads=2, head_dim=128, seed=77)
    pool = pkv.Pool(b.num_blocks, b.num_kv_heads, b.head_dim)
    wl.fill_pool(b, pool.k, pool.v)
    d = wl.upload(b)
    meta = pkv.HostMeta(b.cu_q_lens, b.ctx_lens, b.q_positions)
    pkv.pkv_append(pool, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])
    ref_o, ref_lse = pkv.pkv_paged_attn(pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                        d["cu_q_lens"], meta, b.scale)
    torch.cuda.synchronize()
    stats = pkv.pkv_last_plan_stats(pool)
    assert stats["num_partial_rows"] > 0, "the batch must put split partials into the scratch"
    assert stats["workspace_bytes"] <= pkv.PKV_STATIC_SCRATCH_BYTES
    ref_o = ref_o.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    for call in range(2):
        o, lse = pkv.pkv_paged_attn_static(pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                           d["cu_q_lens"], meta, b.scale)
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_errors(pool) == 0
        o = o.float().cpu().numpy()
        err = np.abs(o - ref_o)
        assert (err <= ATOL + RTOL * np.abs(ref_o)).all(), f"call {call}: max err {err.max():.3e}"
        assert np.abs(lse.cpu().numpy() - ref_lse).max() <= LSE_TOL, f"call {call}"


def test_static_scratch_refuses_batch_above_its_limit():
    # 600,000 one-token requests make 600,000 work items (32 bytes each): more
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
