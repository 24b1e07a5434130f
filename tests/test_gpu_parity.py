"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: the append and every swap are bit-exact; attention output O (bf16) is
within |gpu - ref| <= 2e-2 + 1e-2 * |ref| element-wise and LSE within 1e-3
absolute of the fp64 oracle; a physical-block permutation leaves the GPU
output bit-identical.
"""
import math

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


def to_np_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class GpuRun:
    """Pool + device inputs for a batch; append then attention through the C ABI."""

    def __init__(self, batch, with_positions_meta=True):
        self.b = batch
        self.pool = pkv.Pool(batch.num_blocks, batch.num_kv_heads, batch.head_dim)
        wl.fill_pool(batch, self.pool.k, self.pool.v)
        self.d = wl.upload(batch)
        self.meta = pkv.HostMeta(batch.cu_q_lens, batch.ctx_lens, batch.q_positions if with_positions_meta else None)

    def append(self):
        d = self.d
        pkv.pkv_append(self.pool, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])

    def attn(self):
        d = self.d
        return pkv.pkv_paged_attn(self.pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                  d["cu_q_lens"], self.meta, self.b.scale)

    def step(self):
        self.append()
        o, lse = self.attn()
        torch.cuda.synchronize()
        assert pkv.pkv_check_device_errors(self.pool) == 0
        return o, lse


def oracle_pools(batch):
    kp, vp = batch.pool_arrays()
    oracle.append(kp, vp, batch.block_tables, batch.cu_q_lens, batch.q_positions, batch.k_new, batch.v_new)
    return kp, vp


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    err = np.abs(o_gpu - o_ref)
    bound = ATOL + RTOL * np.abs(o_ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} O elements out of tolerance; max err {err.max():.3e}"
    lerr = np.abs(lse_gpu - lse_ref)
    assert lerr.max() <= LSE_TOL, f"{what}: LSE max err {lerr.max():.3e}"


def full_parity(batch, **kw):
    run = GpuRun(batch, **kw)
    o, lse = run.step()
    kp, vp = oracle_pools(batch)
    O, L = oracle.paged_attn(batch.q, kp, vp, batch.block_tables, batch.ctx_lens, batch.cu_q_lens,
                             batch.q_positions, batch.scale)
    assert_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), O, L, batch.name)
    return run, o, lse


# ----------------------------------------------------------------------------- append

@pytest.mark.parametrize("maker", [lambda: wl.tiny_mixed(1), lambda: wl.random_small(3),
                                   lambda: wl.random_small(8, num_q_heads=8, num_kv_heads=2, head_dim=128)])
def test_append_bit_exact_whole_pool(maker):
    batch = maker()
    run = GpuRun(batch)
    run.append()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(run.pool) == 0
    kp, vp = oracle_pools(batch)
    assert np.array_equal(to_np_bits(run.pool.k), kp)   # includes every untouched slot
    assert np.array_equal(to_np_bits(run.pool.v), vp)


def test_append_more_requests_than_staged_offsets():
    """2,100 requests: the append's request search then reads cu_q_lens from global memory rather
    than from its shared-memory copy (which holds up to 2,048 entries); empty requests among them
    share offsets with their neighbours.  The pool must still match the oracle bit for bit."""
    rng = np.random.default_rng(61)
    reqs = []
    for i in range(2100):
        if i % 97 == 5:
            reqs.append(wl.RequestSpec(ctx=int(rng.integers(1, 40)), q_positions=np.zeros(0, np.int32)))
        elif i % 5 == 0:
            reqs.append(wl._new_turn(int(rng.integers(0, 30)), int(rng.integers(1, 20))))
        else:
            reqs.append(wl._decode(int(rng.integers(0, 60))))
    batch = wl.build_batch("many_requests", reqs, num_q_heads=4, num_kv_heads=2, head_dim=64, seed=61)
    assert batch.num_reqs + 1 > 2048
    run = GpuRun(batch)
    run.append()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(run.pool) == 0
    kp, vp = oracle_pools(batch)
    assert np.array_equal(to_np_bits(run.pool.k), kp)
    assert np.array_equal(to_np_bits(run.pool.v), vp)
    o, lse = run.attn()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(run.pool) == 0
    O, L = oracle.paged_attn(batch.q, kp, vp, batch.block_tables, batch.ctx_lens, batch.cu_q_lens,
                             batch.q_positions, batch.scale)
    assert_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), O, L, batch.name)


def test_append_full_size_gqa_workload():
    batch = wl.llama70b_gqa()
    run = GpuRun(batch)
    run.append()
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(run.pool) == 0
    kp, vp = oracle_pools(batch)
    idx = torch.from_numpy(batch.used_blocks.astype(np.int64)).cuda()
    assert np.array_equal(to_np_bits(run.pool.k[idx]), kp[batch.used_blocks])
    assert np.array_equal(to_np_bits(run.pool.v[idx]), vp[batch.used_blocks])
    unused = torch.ones(batch.num_blocks, dtype=torch.bool, device="cuda")
    unused[idx] = False
    assert int(run.pool.k[unused].view(torch.int16).abs().sum()) == 0


def test_append_flags_bad_slot_without_writing():
    batch = wl.tiny_mixed(1)
    run = GpuRun(batch)
    before = run.pool.k.clone()
    bad = run.d["q_positions"].clone()
    bad[0] = batch.max_blocks * 16 + 5          # beyond the block table: the kernel's bounds check skips it
    pkv.pkv_append(run.pool, run.d["block_tables"], run.d["cu_q_lens"], bad[:1].contiguous(),
                   run.d["k_new"][:1].contiguous(), run.d["v_new"][:1].contiguous())
    flags = pkv.pkv_check_device_errors(run.pool)
    assert flags & pkv.PKV_DEVERR_POSITION
    assert torch.equal(run.pool.k, before)


# ----------------------------------------------------------------------------- attention, small

@pytest.mark.parametrize("maker", [
    lambda: wl.tiny_mixed(1),
    lambda: wl.random_small(1),
    lambda: wl.random_small(2, num_q_heads=4, num_kv_heads=4, head_dim=128),
    lambda: wl.random_small(3, num_q_heads=8, num_kv_heads=1, head_dim=64),
    lambda: wl.random_small(4, num_q_heads=16, num_kv_heads=2, head_dim=128, max_ctx=2000, max_q=300),
    lambda: wl.random_small(5, num_q_heads=2, num_kv_heads=2, head_dim=128, num_reqs=12, max_ctx=5000, max_q=200),
    lambda: wl.random_small(6, num_q_heads=10, num_kv_heads=2, head_dim=64, max_ctx=700, max_q=90),
])
def test_attention_matches_oracle_small(maker):
    full_parity(maker())


def test_attention_without_host_positions():
    full_parity(wl.random_small(7, num_q_heads=4, num_kv_heads=2, head_dim=128, max_ctx=900), with_positions_meta=False)


def _edge_batch(G, D, seed):
    """q_len at 1, tile-1, tile, tile+1 and two tiles; contexts on and off block / tile edges."""
    tq = 128 // G
    reqs = [wl._decode(0), wl._decode(15), wl._decode(16), wl._decode(63), wl._decode(64), wl._decode(65),
            wl._new_turn(0, tq - 1), wl._new_turn(7, tq), wl._new_turn(64, tq + 1), wl._new_turn(1, 2 * tq + 3),
            wl._new_turn(0, 1), wl._recompute(200, 17, 5), wl._recompute(129, 128, 1),
            wl.RequestSpec(ctx=50, q_positions=np.zeros(0, np.int32))]   # a request with no query tokens
    return wl.build_batch(f"edges_G{G}_D{D}", reqs, num_q_heads=2 * G, num_kv_heads=2, head_dim=D, seed=seed)


@pytest.mark.parametrize("G,D", [(1, 64), (1, 128), (2, 128), (8, 128), (8, 64), (5, 128)])
def test_attention_edge_shapes(G, D):
    full_parity(_edge_batch(G, D, seed=40 + G + D))


@pytest.mark.parametrize("G", [1, 2, 4])
def test_split_kv_groups_merged_by_their_last_split(G):
    """Long decodes with 1, 2 or 4 query rows per KV head, cut into many splits: every
    group is combined inside the split-KV kernel by whichever split finishes last."""
    reqs = [wl._decode(9000), wl._decode(4100), wl._decode(777), wl._new_turn(3000, 1)]
    batch = wl.build_batch(f"splits_G{G}", reqs, num_q_heads=2 * G, num_kv_heads=2, head_dim=128, seed=70 + G)
    meta = pkv.HostMeta(batch.cu_q_lens, batch.ctx_lens, batch.q_positions)
    _, st = pkv.pkv_plan_inspect(batch.num_q_heads, batch.num_kv_heads, batch.head_dim,
                                 torch.cuda.get_device_properties(0).multi_processor_count, meta)
    assert st["num_tc_items"] == 0 and st["num_merge_items"] >= 4
    full_parity(batch)


def test_block_permutation_gives_bit_identical_gpu_output():
    batch = wl.random_small(11, num_q_heads=8, num_kv_heads=2, head_dim=128, max_ctx=1500, max_q=150)
    _, o1, l1 = full_parity(batch)
    perm = np.random.default_rng(5).permutation(batch.num_blocks).astype(np.int32)
    b2 = wl.Batch(**{**batch.__dict__})
    b2.block_tables = np.where(batch.block_tables >= 0, perm[np.maximum(batch.block_tables, 0)], -1).astype(np.int32)
    order = np.argsort(perm[batch.used_blocks])
    b2.used_blocks = perm[batch.used_blocks][order].astype(np.int32)
    b2.k_used = batch.k_used[order]
    b2.v_used = batch.v_used[order]
    run = GpuRun(b2)
    o2, l2 = run.step()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_peaky_scores_select_one_value():
    """q = 8 * k_j for one visible key j: softmax concentrates on j, so O ~ v_j (far from zero)."""
    batch = wl.random_small(12, num_q_heads=4, num_kv_heads=4, head_dim=128, max_ctx=600)
    kp, vp = oracle_pools(batch)
    q = batch.q.copy()
    rng = np.random.default_rng(0)
    for t in range(batch.num_tokens):
        r = int(np.searchsorted(batch.cu_q_lens, t, side="right") - 1)
        j = int(rng.integers(0, batch.q_positions[t] + 1))
        blk = batch.block_tables[r, j // 16]
        for h in range(4):
            kvec = oracle.bf16_bits_to_f64(kp[blk, h, j % 16]) * 8.0      # exact in bf16 (power of two)
            q[t, h] = wl.f32_to_bf16_bits(kvec.astype(np.float32))
    batch.q = q
    _, o, _ = full_parity(batch)
    assert float(o.float().abs().mean()) > 0.3


@pytest.mark.parametrize("G", [1, 8])
def test_nan_in_slots_past_the_context_does_not_leak(G):
    """Pool slots no request may see (unused blocks, and the slots past each context in its last
    block) hold NaN: masked keys must contribute exactly nothing (a 0 * NaN product in the split-KV
    FMAs or the tensor-core PV would spread NaN to every row of the tile)."""
    batch = wl.random_small(21 + G, num_q_heads=2 * G, num_kv_heads=2, head_dim=128, num_reqs=8, max_ctx=700,
                            max_q=150)
    run = GpuRun(batch)
    nan = float("nan")
    unused = torch.from_numpy(np.setdiff1d(np.arange(batch.num_blocks), batch.used_blocks)).long().cuda()
    for pool in (run.pool.k, run.pool.v):
        pool[unused] = nan
        for r in range(batch.num_reqs):
            c = int(batch.ctx_lens[r])
            if c % 16:
                pool[int(batch.block_tables[r, c // 16]), :, c % 16:, :] = nan
    o, lse = run.step()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    kp, vp = oracle_pools(batch)
    O, L = oracle.paged_attn(batch.q, kp, vp, batch.block_tables, batch.ctx_lens, batch.cu_q_lens,
                             batch.q_positions, batch.scale)
    assert_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), O, L, batch.name)


def test_output_16_byte_aligned_matches_32_byte_aligned():
    """The tensor-core epilogue stores 32 bytes a row at a time when the output is 32-byte aligned,
    else 16; an output 16 bytes past a 32-byte boundary must get the same bits."""
    batch = wl.random_small(31, num_q_heads=8, num_kv_heads=2, head_dim=128, max_ctx=900, max_q=300)
    run, o1, l1 = full_parity(batch)
    assert pkv.pkv_plan_inspect(batch.num_q_heads, batch.num_kv_heads, batch.head_dim, 148, run.meta)[1][
        "num_tc_items"] > 0
    T, Hq, D = o1.shape
    flat = torch.full((T * Hq * D + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = flat[8:].view(T, Hq, D)
    assert out.data_ptr() % 32 == 16
    d = run.d
    o2, l2 = pkv.pkv_paged_attn(run.pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                d["cu_q_lens"], run.meta, batch.scale, out=out)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(run.pool) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.isnan(flat[:8].float()).all()   # nothing written before the output


def test_zero_tokens_is_a_no_op():
    batch = wl.tiny_mixed(1)
    run = GpuRun(batch)
    empty_q = torch.empty((0, 4, 64), dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(4, dtype=torch.int32, device="cuda")
    meta = pkv.HostMeta(np.zeros(4, np.int32), batch.ctx_lens, np.zeros(0, np.int32))
    out, _ = pkv.pkv_paged_attn(run.pool, empty_q, torch.empty(0, dtype=torch.int32, device="cuda"),
                                run.d["block_tables"], run.d["ctx_lens"], cu, meta, batch.scale)
    assert out.numel() == 0


def test_host_validation_rejects_bad_positions():
    batch = wl.tiny_mixed(1)
    run = GpuRun(batch)
    bad = batch.q_positions.copy()
    bad[-1] = batch.ctx_lens[-1]
    meta = pkv.HostMeta(batch.cu_q_lens, batch.ctx_lens, bad)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_attn(run.pool, run.d["q"], run.d["q_positions"], run.d["block_tables"], run.d["ctx_lens"],
                           run.d["cu_q_lens"], meta, batch.scale)
    assert e.value.code == pkv.PKV_EINVAL


def test_invalid_block_id_is_flagged_not_faulted():
    batch = wl.tiny_mixed(1)
    run = GpuRun(batch)
    run.step()
    bt = run.d["block_tables"].clone()
    bt[0, 0] = batch.num_blocks + 100          # outside the pool: kernels skip the copy and flag it
    pkv.pkv_paged_attn(run.pool, run.d["q"], run.d["q_positions"], bt, run.d["ctx_lens"], run.d["cu_q_lens"],
                       run.meta, batch.scale)
    flags = pkv.pkv_check_device_errors(run.pool)
    assert flags & pkv.PKV_DEVERR_BLOCK_ID


# ----------------------------------------------------------------------------- swap

def test_swap_out_in_bit_exact():
    batch = wl.random_small(13, num_q_heads=4, num_kv_heads=2, head_dim=128)
    run = GpuRun(batch)
    run.step()
    kp, vp = oracle_pools(batch)
    ids = np.concatenate([batch.used_blocks[:6], batch.used_blocks[-3:][::-1]]).astype(np.int32)
    n = ids.shape[0]
    host = torch.empty((n, 2, 2, 16, 128), dtype=torch.bfloat16).pin_memory()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        pkv.pkv_swap_out(run.pool, ids, host)
    side.synchronize()
    ref = oracle.swap_out(kp, vp, ids)
    assert np.array_equal(host.view(torch.int16).numpy().view(np.uint16), ref)
    free = np.setdiff1d(np.arange(batch.num_blocks), batch.used_blocks)[:n].astype(np.int32)
    pkv.pkv_swap_in(run.pool, free, host)
    torch.cuda.synchronize()
    oracle.swap_in(kp, vp, free, ref)
    assert np.array_equal(to_np_bits(run.pool.k), kp) and np.array_equal(to_np_bits(run.pool.v), vp)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_swap_out(run.pool, np.array([batch.num_blocks], np.int32), host)


# ----------------------------------------------------------------------------- full-size workloads

@pytest.mark.slow
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("nbytes,offset", [(1 << 20, 0), (12345, 0), (4099, 3), (16, 0), (0, 0)])
def test_host_copies_bit_exact(pinned, nbytes, offset):
    """pkv_copy_to_device / pkv_copy_to_host: every byte, aligned or not, pinned or pageable host memory."""
    rng = np.random.default_rng(nbytes + offset)
    src = torch.from_numpy(rng.integers(0, 256, nbytes + offset + 8, dtype=np.uint8))
    if pinned:
        src = src.pin_memory()
    dev = torch.full((nbytes + offset + 8,), 7, dtype=torch.uint8, device="cuda")
    pkv.pkv_copy_to_device(dev[offset:offset + nbytes], src[offset:offset + nbytes])
    back = torch.zeros(nbytes + offset + 8, dtype=torch.uint8)
    if pinned:
        back = back.pin_memory()
    pkv.pkv_copy_to_host(back[offset:offset + nbytes], dev[offset:offset + nbytes])
    torch.cuda.synchronize()
    d = dev.cpu().numpy()
    assert np.array_equal(d[offset:offset + nbytes], src.numpy()[offset:offset + nbytes])
    assert (d[:offset] == 7).all() and (d[offset + nbytes:] == 7).all()   # nothing outside the range
    assert np.array_equal(back.numpy()[offset:offset + nbytes], src.numpy()[offset:offset + nbytes])
    assert (back.numpy()[offset + nbytes:] == 0).all()


@pytest.mark.parametrize("name", ["llama13b_mixed", "decode_lognormal", "llama70b_gqa", "long_skewed_evict"])
def test_full_size_workloads_every_row(name):
    """Every (token, head) row of the full-size workload against the fp64 oracle, in the bench's launch shape."""
    batch = wl.WORKLOADS[name]()
    run = GpuRun(batch)
    o, lse = run.step()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    kp, vp = oracle_pools(batch)
    O, L = oracle.paged_attn(batch.q, kp, vp, batch.block_tables, batch.ctx_lens, batch.cu_q_lens,
                             batch.q_positions, batch.scale)
    assert_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), O, L, name)


def test_plan_cache_tells_apart_batches_of_one_shape():
    """Two batches with the same request and token counts on one pool: the second differs only in
    one decode's context length and position, so it must be planned again (the cached plan's key
    ranges would read one key too many) and still match the oracle."""
    a = wl.random_small(31, num_q_heads=4, num_kv_heads=2, head_dim=128, num_reqs=8, max_ctx=3000, max_q=60)
    dec = [r for r in range(a.num_reqs) if a.cu_q_lens[r + 1] - a.cu_q_lens[r] == 1 and a.ctx_lens[r] > 2]
    assert dec, "the batch needs a decode request"
    run = GpuRun(a)
    run.step()
    built = pkv.pkv_last_plan_stats(run.pool)["plans_built"]
    kp, vp = oracle_pools(a)
    b = wl.Batch(**{**a.__dict__})
    b.ctx_lens = a.ctx_lens.copy()
    b.q_positions = a.q_positions.copy()
    r = dec[0]
    b.ctx_lens[r] -= 1
    b.q_positions[a.cu_q_lens[r]] -= 1
    d = wl.upload(b)
    meta = pkv.HostMeta(b.cu_q_lens, b.ctx_lens, b.q_positions)
    pkv.pkv_append(run.pool, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])
    o, lse = pkv.pkv_paged_attn(run.pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                d["cu_q_lens"], meta, b.scale)
    torch.cuda.synchronize()
    assert pkv.pkv_check_device_errors(run.pool) == 0
    assert pkv.pkv_last_plan_stats(run.pool)["plans_built"] == built + 1
    oracle.append(kp, vp, b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
    O, L = oracle.paged_attn(b.q, kp, vp, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions, b.scale)
    assert_close(bf16_to_f64(o), lse.cpu().numpy().astype(np.float64), O, L, "second batch")


@pytest.mark.parametrize("name,mode", [("llama13b_mixed", 1), ("llama13b_mixed", 2), ("long_skewed_evict", 1)])
def test_repeated_calls_bit_identical_without_device_errors(name, mode):
    """Forty calls on one full-size batch (the persistent tensor-core kernel reuses every barrier across the
    items of a CTA, including single-tile items): no bounded wait gives up, and every output equals the first."""
    batch = wl.WORKLOADS[name]()
    run = GpuRun(batch)
    o0, l0 = run.step()
    pkv.pkv_profile_enable(run.pool, mode)
    for _ in range(40):
        o, lse = run.attn()
    torch.cuda.synchronize()
    pkv.pkv_profile_enable(run.pool, 0)
    assert pkv.pkv_check_device_errors(run.pool) == 0
    assert torch.equal(o, o0) and torch.equal(lse, l0)
