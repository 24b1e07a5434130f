"""FP8 (E4M3) KV cache through the C ABI, against the CPU oracle.

Bars: the quantising append leaves the pools bit-identical to the oracle's
(every code of every block, saturating and subnormal quotients included); swaps
move the code bytes exactly; split-KV attention over FP8 pools is within
|gpu - ref| <= 2e-2 + 1e-2 |ref| (O) and 1e-3 (LSE) of the fp64 oracle on the
dequantised values, and so is tensor-core attention over FP8 pools (codes
widened to f16 in shared memory) on prefill, recompute and grouped-query
batches.
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


def fp8_pool(batch, ks, vs):
    pool = pkv.Pool(batch.num_blocks, batch.num_kv_heads, batch.head_dim, dtype="fp8_e4m3", k_scale=ks, v_scale=vs)
    wl.fill_pool_fp8(batch, pool.k, pool.v)
    torch.cuda.synchronize()
    return pool


def append(pool, d):
    pkv.pkv_append(pool, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])


@pytest.mark.parametrize("hkv,d,ks,vs", [(2, 64, 0.0123, 0.5), (4, 128, 2.0 ** -6, 0.03),
                                          (2, 128, 2.0 ** -12, 2.0 ** 10)])   # saturating K, subnormal V
def test_fp8_append_bit_exact_whole_pool(hkv, d, ks, vs):
    b = wl.random_small(51, num_q_heads=hkv * 2, num_kv_heads=hkv, head_dim=d)
    pool = fp8_pool(b, ks, vs)
    append(pool, wl.upload(b))
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(pool) == 0
    k8, v8 = wl.fp8_pool_arrays(b)
    oracle.append_fp8(k8, v8, np.float32(ks), np.float32(vs), b.block_tables, b.cu_q_lens, b.q_positions,
                      b.k_new, b.v_new)
    assert np.array_equal(pool.k.cpu().numpy(), k8)
    assert np.array_equal(pool.v.cpu().numpy(), v8)
    pool.close()


def check_attention(b, ks, vs, rows=None, want_tc=False):
    pool = fp8_pool(b, ks, vs)
    dv = wl.upload(b)
    append(pool, dv)
    meta = pkv.HostMeta(b.cu_q_lens, b.ctx_lens, b.q_positions)
    o, lse = pkv.pkv_paged_attn(pool, dv["q"], dv["q_positions"], dv["block_tables"], dv["ctx_lens"],
                                dv["cu_q_lens"], meta, b.scale)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(pool) == 0
    st = pkv.pkv_last_plan_stats(pool)
    assert (st["num_tc_items"] > 0) == want_tc
    k8, v8 = wl.fp8_pool_arrays(b)
    oracle.append_fp8(k8, v8, np.float32(ks), np.float32(vs), b.block_tables, b.cu_q_lens, b.q_positions,
                      b.k_new, b.v_new)
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    if rows is None:
        O, L = oracle.paged_attn_fp8(b.q, k8, v8, ks, vs, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions,
                                     b.scale)
    else:
        rt, rh = rows
        O, L = oracle.paged_attn_rows_fp8(b.q, k8, v8, ks, vs, b.block_tables, b.ctx_lens, b.cu_q_lens,
                                          b.q_positions, b.scale, rt, rh)
        o, lse = o[rt, rh], lse[rt, rh]
    err = np.abs(o - O)
    bad = err > ATOL + RTOL * np.abs(O)
    assert not bad.any(), f"{bad.sum()} O elements out of tolerance; max err {err.max():.3e}"
    assert np.abs(lse - L).max() <= LSE_TOL
    pool.close()
    return st


@pytest.mark.parametrize("hq,hkv,d,tokens", [(4, 4, 128, 1), (8, 8, 64, 2), (8, 4, 128, 2), (16, 4, 128, 1),
                                             (8, 2, 64, 1)])
def test_fp8_split_kv_attention_matches_oracle(hq, hkv, d, tokens):
    b = wl.decode_small(60 + hq + d + tokens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, tokens=tokens)
    st = check_attention(b, 2.0 ** -6, 0.0217)
    assert st["num_decode_items"] > b.num_reqs * hkv   # the long request is split over several items


def test_fp8_full_size_decode_workload_every_row():
    check_attention(wl.decode_lognormal(), 2.0 ** -6, 2.0 ** -6)


def test_fp8_swap_bit_exact():
    b = wl.decode_small(70, num_q_heads=8, num_kv_heads=8, head_dim=128)
    pool = fp8_pool(b, 1.0, 1.0)
    ids = b.used_blocks[:7].astype(np.int32)
    host = torch.empty((7, 2, 8, 16, 128), dtype=torch.uint8).pin_memory()
    pkv.pkv_swap_out(pool, ids, host)
    torch.cuda.synchronize()
    k8, v8 = wl.fp8_pool_arrays(b)
    assert np.array_equal(host[:, 0].numpy(), k8[ids]) and np.array_equal(host[:, 1].numpy(), v8[ids])
    free = np.setdiff1d(np.arange(b.num_blocks), b.used_blocks)[:7].astype(np.int32)
    pkv.pkv_swap_in(pool, free, host)
    copy = torch.cuda.Stream()
    pkv.pkv_swap_in_ahead(pool, free[::-1].copy(), host, copy)
    pkv.pkv_swap_in_finish(pool)
    torch.cuda.synchronize()
    k8[free[::-1]] = k8[ids]
    v8[free[::-1]] = v8[ids]
    assert np.array_equal(pool.k.cpu().numpy(), k8) and np.array_equal(pool.v.cpu().numpy(), v8)
    pool.close()


@pytest.mark.parametrize("maker,ks,vs", [
    (lambda: wl.random_small(71, num_q_heads=4, num_kv_heads=2, head_dim=64), 2.0 ** -6, 0.0217),
    (lambda: wl.random_small(72, num_q_heads=4, num_kv_heads=4, head_dim=128, max_ctx=2000, max_q=300), 0.0123, 0.5),
    (lambda: wl.random_small(73, num_q_heads=16, num_kv_heads=2, head_dim=128, max_ctx=1500, max_q=100),
     2.0 ** -6, 2.0 ** -6),
    # Saturating K codes and subnormal V codes: every key is a new token, so every code comes from
    # quantising N(0,1) values (history codes times a scale of 2^10 would give values near 1e5,
    # where the rounding of P alone exceeds an absolute tolerance of 2e-2).
    (lambda: wl.build_batch("fp8_extreme", [wl._new_turn(0, n) for n in (37, 130, 250, 61)], num_q_heads=10,
                            num_kv_heads=2, head_dim=128, seed=74), 2.0 ** -12, 2.0 ** 10),
    (lambda: wl.random_small(75, num_q_heads=10, num_kv_heads=2, head_dim=128, max_ctx=900, max_q=60),
     2.0 ** -6, 2.0 ** -6),
    # The other way round: subnormal K codes (the widened tiles then hold f16 subnormals) and
    # saturating V codes.
    (lambda: wl.build_batch("fp8_extreme_k", [wl._new_turn(0, n) for n in (45, 129, 260, 3)], num_q_heads=8,
                            num_kv_heads=2, head_dim=128, seed=76), 2.0 ** 10, 2.0 ** -12),
])
def test_fp8_tensor_core_attention_matches_oracle(maker, ks, vs):
    check_attention(maker(), ks, vs, want_tc=True)


@pytest.mark.parametrize("G,D", [(1, 128), (8, 128), (2, 64)])
def test_fp8_tensor_core_edge_shapes(G, D):
    tq = 128 // G
    reqs = [wl._decode(63), wl._new_turn(0, tq - 1), wl._new_turn(7, tq), wl._new_turn(64, tq + 1),
            wl._new_turn(1, 2 * tq + 3), wl._recompute(200, 17, 5), wl._recompute(129, 128, 1)]
    b = wl.build_batch(f"fp8_edges_G{G}_D{D}", reqs, num_q_heads=2 * G, num_kv_heads=2, head_dim=D, seed=80 + G + D)
    check_attention(b, 2.0 ** -6, 2.0 ** -6, want_tc=True)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama13b_mixed", "llama70b_gqa", "long_skewed_evict"])
def test_fp8_full_size_mixed_workloads_every_row(name):
    check_attention(wl.WORKLOADS[name](), 2.0 ** -6, 2.0 ** -6, want_tc=True)


def test_fp8_pool_rejects_bad_scales():
    with pytest.raises(pkv.PkvError):
        pkv.Pool(16, 2, 64, dtype="fp8_e4m3", k_scale=0.0, v_scale=1.0)
