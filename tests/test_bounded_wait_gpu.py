"""Failure detection without a GPU fault: a bounded wait inside a kernel that
runs out is reported, and the pool stays usable.

A pool's test setting withholds one K copy in the first CTA of the split-KV
(or tensor-core) kernel, so that the wait for it can never be satisfied, and
shortens the wait limit to a few milliseconds.  The kernel must then record
PKV_DEVERR_TIMEOUT, drain its copies in flight, free what it holds and return;
pkv_check_device_errors reports PKV_ETIMEOUT; and the next normal call on the
same pool matches the oracle.
"""
import ctypes

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


FP8_SCALE = 2.0 ** -6


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("kernel", [1, 2])
def test_wait_that_runs_out_is_reported_and_pool_recovers(kernel, dtype):
    # Decodes for the split-KV kernel and new turns for the tensor-core kernel.  FP8 pools take
    # other waits: the tensor-core producers poll their barriers and give up on their own limit.
    fp8 = dtype == "fp8_e4m3"
    reqs = [wl._decode(5000), wl._decode(700), wl._new_turn(2000, 300), wl._new_turn(0, 130)]
    b = wl.build_batch(f"timeout_{kernel}_{dtype}", reqs, num_q_heads=4, num_kv_heads=4, head_dim=128,
                       seed=90 + kernel)
    if fp8:
        pool = pkv.Pool(b.num_blocks, b.num_kv_heads, b.head_dim, dtype=dtype, k_scale=FP8_SCALE, v_scale=FP8_SCALE)
        wl.fill_pool_fp8(b, pool.k, pool.v)
    else:
        pool = pkv.Pool(b.num_blocks, b.num_kv_heads, b.head_dim)
        wl.fill_pool(b, pool.k, pool.v)
    d = wl.upload(b)
    meta = pkv.HostMeta(b.cu_q_lens, b.ctx_lens, b.q_positions)
    pkv.pkv_append(pool, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])
    st = pkv.pkv_plan_inspect(b.num_q_heads, b.num_kv_heads, b.head_dim, pkv.pkv_device_sm_count(), meta)[1]
    assert st["num_decode_items"] > 0 and st["num_tc_items"] > 0

    def attn():
        return pkv.pkv_paged_attn(pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                  d["cu_q_lens"], meta, b.scale)

    pkv.pkv_debug_set(pool, pkv.PKV_DEBUG_WAIT_LIMIT_NS, 2_000_000)    # 2 ms
    pkv.pkv_debug_set(pool, pkv.PKV_DEBUG_WITHHOLD_COPY, kernel)
    attn()
    flags = ctypes.c_uint()
    rc = pkv.load_library().pkv_check_device_errors(pool.handle, pkv._stream(None), ctypes.byref(flags))
    assert rc == pkv.PKV_ETIMEOUT, pkv.pkv_last_error()
    assert flags.value & pkv.PKV_DEVERR_TIMEOUT
    assert "bounded wait" in pkv.pkv_last_error()

    # Back to normal on the same pool: the error word was cleared by the check.
    pkv.pkv_debug_set(pool, pkv.PKV_DEBUG_WITHHOLD_COPY, 0)
    pkv.pkv_debug_set(pool, pkv.PKV_DEBUG_WAIT_LIMIT_NS, 1_000_000_000)
    o, lse = attn()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(pool) == 0
    if fp8:
        kp, vp = wl.fp8_pool_arrays(b)
        oracle.append_fp8(kp, vp, np.float32(FP8_SCALE), np.float32(FP8_SCALE), b.block_tables, b.cu_q_lens,
                          b.q_positions, b.k_new, b.v_new)
        O, L = oracle.paged_attn_fp8(b.q, kp, vp, FP8_SCALE, FP8_SCALE, b.block_tables, b.ctx_lens, b.cu_q_lens,
                                     b.q_positions, b.scale)
    else:
        kp, vp = b.pool_arrays()
        oracle.append(kp, vp, b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
        O, L = oracle.paged_attn(b.q, kp, vp, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions, b.scale)
    err = np.abs(o.float().cpu().numpy() - O)
    assert (err <= ATOL + RTOL * np.abs(O)).all(), f"max err {err.max():.3e}"
    assert np.abs(lse.cpu().numpy() - L).max() <= LSE_TOL


def test_debug_settings_are_validated():
    pool = pkv.Pool(4, 1, 64)
    for what, value in ((pkv.PKV_DEBUG_WAIT_LIMIT_NS, 0), (pkv.PKV_DEBUG_WITHHOLD_COPY, 3), (99, 0)):
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_debug_set(pool, what, value)
        assert e.value.code == pkv.PKV_EINVAL
