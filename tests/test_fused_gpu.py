"""Fused paged KV append + attention (pkv_append_paged_attn) through the C ABI.

Bars: after the call the whole pool equals the oracle's append, bit for bit
(untouched slots included); O and LSE are within |gpu - ref| <= 2e-2 + 1e-2
|ref| and 1e-3 of the fp64 oracle, and bit-identical to pkv_append followed by
pkv_paged_attn on the same batch (the same plan and the same values: the fused
kernels only take the step's own keys and values from the new rows instead of
the pool).  A NaN canary in every slot the append is about to write shows the
attention never reads those slots from the pool.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_25_gb300 import pkv
from paged_kv_attention_25_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3
FP8_SCALE = 2.0 ** -6


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_25_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_pool(b, fp8):
    if fp8:
        pool = pkv.Pool(b.num_blocks, b.num_kv_heads, b.head_dim, dtype="fp8_e4m3", k_scale=FP8_SCALE,
                        v_scale=FP8_SCALE)
        wl.fill_pool_fp8(b, pool.k, pool.v)
    else:
        pool = pkv.Pool(b.num_blocks, b.num_kv_heads, b.head_dim)
        wl.fill_pool(b, pool.k, pool.v)
    return pool


def poison_new_slots(b, pool):
    """NaN (bf16) or the E4M3 NaN code in every slot this step's append writes."""
    nan = 0x7F if pool.k.dtype == torch.uint8 else float("nan")
    for r in range(b.num_reqs):
        for p in b.q_positions[b.cu_q_lens[r]:b.cu_q_lens[r + 1]]:
            blk = int(b.block_tables[r, p // 16])
            pool.k[blk, :, p % 16] = nan
            pool.v[blk, :, p % 16] = nan


def oracle_after(b, fp8):
    if fp8:
        kp, vp = wl.fp8_pool_arrays(b)
        oracle.append_fp8(kp, vp, np.float32(FP8_SCALE), np.float32(FP8_SCALE), b.block_tables, b.cu_q_lens,
                          b.q_positions, b.k_new, b.v_new)
        O, L = oracle.paged_attn_rows_fp8(b.q, kp, vp, FP8_SCALE, FP8_SCALE, b.block_tables, b.ctx_lens,
                                          b.cu_q_lens, b.q_positions, b.scale,
                                          np.repeat(np.arange(b.num_tokens, dtype=np.int32), b.num_q_heads),
                                          np.tile(np.arange(b.num_q_heads, dtype=np.int32), b.num_tokens))
        O = O.reshape(b.num_tokens, b.num_q_heads, b.head_dim)
        L = L.reshape(b.num_tokens, b.num_q_heads)
    else:
        kp, vp = b.pool_arrays()
        oracle.append(kp, vp, b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
        O, L = oracle.paged_attn(b.q, kp, vp, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions, b.scale)
    return kp, vp, O, L


def run_both(b, fp8=False, poison=True, form=1):
    """(fused O, LSE, pool K, pool V) and (unfused O, LSE) on fresh pools holding the same history.
    form: PKV_DEBUG_FUSED_FORM of the fused call's pool (1, in-kernel append wherever the pool allows
    it, unless a test asks for the per-batch choice (0) or append-first (2))."""
    d = wl.upload(b)
    meta = pkv.HostMeta(b.cu_q_lens, b.ctx_lens, b.q_positions)
    ref_pool = make_pool(b, fp8)
    pkv.pkv_append(ref_pool, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])
    o_ref, l_ref = pkv.pkv_paged_attn(ref_pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                      d["cu_q_lens"], meta, b.scale)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(ref_pool) == 0
    pool = make_pool(b, fp8)
    pkv.pkv_debug_set(pool, pkv.PKV_DEBUG_FUSED_FORM, form)
    if poison:
        poison_new_slots(b, pool)
    torch.cuda.synchronize()
    o, lse = pkv.pkv_append_paged_attn(pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                       d["cu_q_lens"], meta, d["k_new"], d["v_new"], b.scale)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(pool) == 0
    st = pkv.pkv_last_plan_stats(pool)
    return (o, lse, pool), (o_ref, l_ref), st


def check(b, fp8=False, poison=True, need_tc=None, form=1):
    (o, lse, pool), (o_ref, l_ref), st = run_both(b, fp8, poison, form)
    if need_tc is not None:
        assert (st["num_tc_items"] > 0) == need_tc
    kp, vp, O, L = oracle_after(b, fp8)
    assert np.array_equal(bits(pool.k), kp), f"{b.name}: K pool differs from the oracle's append"
    assert np.array_equal(bits(pool.v), vp), f"{b.name}: V pool differs from the oracle's append"
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), f"{b.name}: a NaN reached the output"
    err = np.abs(o.float().cpu().numpy() - O)
    bad = err > ATOL + RTOL * np.abs(O)
    assert not bad.any(), f"{b.name}: {bad.sum()} O elements out of tolerance, max err {err.max():.3e}"
    assert np.abs(lse.cpu().numpy() - L).max() <= LSE_TOL, f"{b.name}: LSE"
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), f"{b.name}: fused and unfused outputs differ"
    return st


@pytest.mark.parametrize("maker", [
    lambda: wl.tiny_mixed(1),
    lambda: wl.random_small(1),
    lambda: wl.random_small(2, num_q_heads=4, num_kv_heads=4, head_dim=128),
    lambda: wl.random_small(3, num_q_heads=8, num_kv_heads=1, head_dim=64),
    lambda: wl.random_small(4, num_q_heads=16, num_kv_heads=2, head_dim=128, max_ctx=2000, max_q=300),
    lambda: wl.random_small(5, num_q_heads=2, num_kv_heads=2, head_dim=128, num_reqs=12, max_ctx=5000, max_q=200),
    lambda: wl.random_small(6, num_q_heads=10, num_kv_heads=2, head_dim=64, max_ctx=700, max_q=90),
])
def test_fused_matches_oracle_and_unfused(maker):
    check(maker())


@pytest.mark.parametrize("G,D", [(1, 64), (1, 128), (2, 128), (8, 128), (5, 128)])
def test_fused_edge_shapes(G, D):
    """New runs starting and ending inside blocks and 8-key groups (patched blocks), runs on block
    edges (blocks taken whole from the new rows), recompute prefixes, and a request with no tokens."""
    tq = 128 // G
    reqs = [wl._decode(0), wl._decode(15), wl._decode(16), wl._decode(63), wl._new_turn(0, tq - 1),
            wl._new_turn(7, tq), wl._new_turn(64, tq + 1), wl._new_turn(1, 2 * tq + 3), wl._new_turn(13, 37),
            wl._new_turn(16, 48), wl._recompute(200, 17, 5), wl._recompute(129, 128, 1), wl._recompute(300, 40, 3),
            wl.RequestSpec(ctx=50, q_positions=np.zeros(0, np.int32))]
    check(wl.build_batch(f"fused_edges_G{G}_D{D}", reqs, num_q_heads=2 * G, num_kv_heads=2, head_dim=D,
                         seed=140 + G + D))


def test_fused_positions_out_of_token_order():
    """A request whose tokens are not in position order (runs sorted by the planner), with one
    tensor-core tile spanning both runs."""
    reqs = [wl.RequestSpec(ctx=400, q_positions=np.concatenate([np.arange(350, 400), np.arange(100, 180)]).astype(
                np.int32)),
            wl.RequestSpec(ctx=90, q_positions=np.array([89, 3, 40, 41, 42, 7], np.int32)), wl._decode(500)]
    check(wl.build_batch("fused_order", reqs, num_q_heads=4, num_kv_heads=2, head_dim=128, seed=150), need_tc=True)


def test_fused_split_key_ranges():
    """Long contexts cut into several key splits on both kernels; the new tokens fall in the last split."""
    reqs = [wl._decode(9000), wl._new_turn(6000, 400), wl._new_turn(3000, 1), wl._recompute(7000, 900, 100)]
    st = check(wl.build_batch("fused_splits", reqs, num_q_heads=8, num_kv_heads=2, head_dim=128, seed=151))
    assert st["num_merge_items"] > 0


@pytest.mark.parametrize("maker", [lambda: wl.decode_small(61, num_q_heads=4, num_kv_heads=4, head_dim=128),
                                   lambda: wl.decode_small(62, num_q_heads=4, num_kv_heads=2, head_dim=64,
                                                           tokens=2)])
def test_fused_fp8_decode_regime(maker):
    check(maker(), fp8=True, need_tc=False)


@pytest.mark.parametrize("maker", [lambda: wl.random_small(63, num_q_heads=4, num_kv_heads=2, head_dim=128,
                                                           max_ctx=1500, max_q=200),
                                   lambda: wl.random_small(64, num_q_heads=16, num_kv_heads=2, head_dim=64,
                                                           max_ctx=700, max_q=50)])
def test_fused_fp8_tensor_core(maker):
    check(maker(), fp8=True, need_tc=True)


@pytest.mark.parametrize("form", [0, 2])
@pytest.mark.parametrize("maker", [
    lambda: wl.random_small(4, num_q_heads=16, num_kv_heads=2, head_dim=128, max_ctx=2000, max_q=300),
    lambda: wl.random_small(5, num_q_heads=2, num_kv_heads=2, head_dim=128, num_reqs=12, max_ctx=5000, max_q=200),
    lambda: wl.decode_small(61, num_q_heads=4, num_kv_heads=4, head_dim=128),
])
def test_fused_other_forms_same_bits(maker, form):
    """The per-batch choice (0) and append-first (2) give the oracle's pool and the unfused outputs,
    bit for bit, as the in-kernel append does."""
    check(maker(), form=form)


def test_fused_form_setting_range():
    b = wl.tiny_mixed(1)
    pool = make_pool(b, False)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_debug_set(pool, pkv.PKV_DEBUG_FUSED_FORM, 3)
    assert e.value.code == pkv.PKV_EINVAL
    pool.close()


def test_fused_needs_host_positions():
    b = wl.tiny_mixed(1)
    pool = make_pool(b, False)
    d = wl.upload(b)
    meta = pkv.HostMeta(b.cu_q_lens, b.ctx_lens, None)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_append_paged_attn(pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"], d["cu_q_lens"],
                                  meta, d["k_new"], d["v_new"], b.scale)
    assert e.value.code == pkv.PKV_EINVAL


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama13b_mixed", "llama70b_gqa", "long_skewed_evict"])
def test_fused_full_size(name):
    """Full-size workloads: the pool's used blocks against the oracle's append, every output row
    bit-identical to the unfused path, and a sample of rows against the oracle."""
    b = wl.WORKLOADS[name]()
    (o, lse, pool), (o_ref, l_ref), _ = run_both(b, poison=False)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    kp, vp = b.pool_arrays()
    oracle.append(kp, vp, b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
    idx = torch.from_numpy(b.used_blocks.astype(np.int64)).cuda()
    assert np.array_equal(bits(pool.k[idx]), kp[b.used_blocks])
    assert np.array_equal(bits(pool.v[idx]), vp[b.used_blocks])
    rng = np.random.default_rng(3)
    t = rng.integers(0, b.num_tokens, 400).astype(np.int32)
    h = rng.integers(0, b.num_q_heads, 400).astype(np.int32)
    O, L = oracle.paged_attn_rows(b.q, kp, vp, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions, b.scale, t, h)
    err = np.abs(o.float().cpu().numpy()[t, h] - O)
    assert (err <= ATOL + RTOL * np.abs(O)).all()
    assert np.abs(lse.cpu().numpy()[t, h] - L).max() <= LSE_TOL
