"""Ahead-of-time swap-in (pkv_swap_in_ahead / pkv_swap_in_finish) through the C ABI.

Bars: the pool after the blocks land equals the oracle's swap-in bit for bit
(untouched blocks included); calls take effect in call order (a swap-out after
an ahead-of-time swap-in reads the new blocks; a transfer reads a host buffer
that a swap-out queued before it filled); and layer-pipelined attention over
pools whose evicted history came back ahead of time is bit-identical to the
same attention over pools that never lost it, and within the parity tolerance
of the fp64 oracle.
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


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def rand_host(n, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((n, 2, hkv, 16, d), generator=g).to(torch.bfloat16).pin_memory()


def filled_pool(batch):
    pool = pkv.Pool(batch.num_blocks, batch.num_kv_heads, batch.head_dim)
    wl.fill_pool(batch, pool.k, pool.v)
    torch.cuda.synchronize()
    return pool


@pytest.mark.parametrize("hkv,d,n", [(2, 64, 5), (2, 128, 9), (8, 128, 40)])
def test_swap_in_ahead_lands_bit_exact(hkv, d, n):
    batch = wl.random_small(21, num_q_heads=hkv * 2, num_kv_heads=hkv, head_dim=d)
    pool = filled_pool(batch)
    kp, vp = bits(pool.k), bits(pool.v)
    rng = np.random.default_rng(n)
    ids = rng.choice(batch.num_blocks, size=min(n, batch.num_blocks), replace=False).astype(np.int32)
    host = rand_host(ids.shape[0], hkv, d, seed=n)
    copy = torch.cuda.Stream()
    pkv.pkv_swap_in_ahead(pool, ids, host, copy)
    copy.synchronize()
    # the transfer is done, but the blocks land only at the pool's next call
    assert np.array_equal(bits(pool.k), kp) and np.array_equal(bits(pool.v), vp)
    pkv.pkv_swap_in_finish(pool)
    pkv.pkv_swap_in_finish(pool)   # nothing pending: a no-op
    torch.cuda.synchronize()
    oracle.swap_in(kp, vp, ids, host.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(bits(pool.k), kp) and np.array_equal(bits(pool.v), vp)
    assert pkv.pkv_check_device_errors(pool) == 0
    pool.close()


def test_calls_take_effect_in_call_order():
    hkv, d = 2, 128
    batch = wl.random_small(22, num_q_heads=4, num_kv_heads=hkv, head_dim=d)
    pool = filled_pool(batch)
    kp, vp = bits(pool.k), bits(pool.v)
    copy = torch.cuda.Stream()
    a = np.array([3, 7, 1, 12], np.int32)
    b = np.array([7, 2, 12, 5, 9, 0, 4], np.int32)   # overlaps a, and more blocks (the staging grows)
    ha, hb = rand_host(a.shape[0], hkv, d, 1), rand_host(b.shape[0], hkv, d, 2)
    # a swap-out after an ahead-of-time swap-in reads the swapped-in blocks
    pkv.pkv_swap_in_ahead(pool, a, ha, copy)
    back = torch.empty_like(ha).pin_memory()
    pkv.pkv_swap_out(pool, a, back)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), ha.view(torch.int16))
    # two ahead-of-time swap-ins in a row: the first lands before the second
    pkv.pkv_swap_in_ahead(pool, a, ha, copy)
    pkv.pkv_swap_in_ahead(pool, b, hb, copy)
    pkv.pkv_swap_in_finish(pool)
    torch.cuda.synchronize()
    oracle.swap_in(kp, vp, a, ha.view(torch.int16).numpy().view(np.uint16))
    oracle.swap_in(kp, vp, b, hb.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(bits(pool.k), kp) and np.array_equal(bits(pool.v), vp)
    # a bad id starts nothing and leaves nothing pending
    with pytest.raises(pkv.PkvError):
        pkv.pkv_swap_in_ahead(pool, np.array([0, batch.num_blocks], np.int32), ha[:2], copy)
    pkv.pkv_swap_in_finish(pool)
    torch.cuda.synchronize()
    assert np.array_equal(bits(pool.k), kp) and np.array_equal(bits(pool.v), vp)
    pool.close()


def test_transfer_follows_swap_out_queued_before_it():
    # The CPU tier's round trip in one go: blocks x go out to a host buffer on
    # the compute stream, and the same buffer comes back ahead of time into
    # blocks y; the transfer must wait for the swap-out that fills the buffer.
    hkv, d = 8, 128
    batch = wl.random_small(23, num_q_heads=16, num_kv_heads=hkv, head_dim=d)
    pool = filled_pool(batch)
    kp, vp = bits(pool.k), bits(pool.v)
    free = np.setdiff1d(np.arange(batch.num_blocks), batch.used_blocks)
    k = min(16, free.shape[0], batch.used_blocks.shape[0])
    assert k >= 8
    x = batch.used_blocks[:k].astype(np.int32)
    y = free[:k].astype(np.int32)
    host = torch.zeros((x.shape[0], 2, hkv, 16, d), dtype=torch.bfloat16).pin_memory()
    copy = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    for _ in range(3):
        pkv.pkv_swap_out(pool, x, host, stream=main)
        pkv.pkv_swap_in_ahead(pool, y, host, copy, stream=main)
        pkv.pkv_swap_in_finish(pool, stream=main)
    torch.cuda.synchronize()
    oracle.swap_in(kp, vp, y, oracle.swap_out(kp, vp, x))
    assert np.array_equal(bits(pool.k), kp) and np.array_equal(bits(pool.v), vp)
    pool.close()


def history_blocks(batch):
    """Whole blocks of each request below its first query position: cached history that the append leaves alone."""
    ids = []
    for r in range(batch.num_reqs):
        q = batch.q_positions[batch.cu_q_lens[r]:batch.cu_q_lens[r + 1]]
        first = int(q.min()) if q.size else int(batch.ctx_lens[r])
        ids.extend(int(x) for x in batch.block_tables[r, :first // 16])
    return np.array(sorted(set(ids)), np.int32)


class Layer:
    def __init__(self, batch):
        self.b = batch
        self.pool = filled_pool(batch)
        self.d = wl.upload(batch)
        self.meta = pkv.HostMeta(batch.cu_q_lens, batch.ctx_lens, batch.q_positions)

    def attend(self):
        d = self.d
        pkv.pkv_append(self.pool, d["block_tables"], d["cu_q_lens"], d["q_positions"], d["k_new"], d["v_new"])
        return pkv.pkv_paged_attn(self.pool, d["q"], d["q_positions"], d["block_tables"], d["ctx_lens"],
                                  d["cu_q_lens"], self.meta, self.b.scale)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 2, 128), (4, 4, 64)])
def test_layer_pipelined_attention_matches_unevicted(hq, hkv, d):
    layers_n = 3
    batches = [wl.random_small(40 + l, num_q_heads=hq, num_kv_heads=hkv, head_dim=d) for l in range(layers_n)]
    # reference: the same layers, history never evicted
    ref = []
    for b in batches:
        lay = Layer(b)
        o, lse = lay.attend()
        torch.cuda.synchronize()
        ref.append((o.clone(), lse.clone()))
        lay.pool.close()
    # evict each layer's history to a pinned host buffer, poison the pool blocks
    layers, hosts, ids = [], [], []
    for b in batches:
        lay = Layer(b)
        h_ids = history_blocks(b)
        assert h_ids.size > 0
        host = torch.empty((h_ids.shape[0], 2, hkv, 16, d), dtype=torch.bfloat16).pin_memory()
        pkv.pkv_swap_out(lay.pool, h_ids, host)
        torch.cuda.synchronize()
        idx = torch.from_numpy(h_ids.astype(np.int64)).cuda()
        lay.pool.k[idx] = float("nan")
        lay.pool.v[idx] = float("nan")
        layers.append(lay)
        hosts.append(host)
        ids.append(h_ids)
    torch.cuda.synchronize()
    # every layer's swap-in ahead of time on one copy stream, then the layers in order
    copy, main = torch.cuda.Stream(), torch.cuda.current_stream()
    for lay, h_ids, host in zip(layers, ids, hosts):
        pkv.pkv_swap_in_ahead(lay.pool, h_ids, host, copy, stream=main)
    outs = [lay.attend() for lay in layers]
    torch.cuda.synchronize()
    for l, ((o, lse), (o_ref, lse_ref), lay) in enumerate(zip(outs, ref, layers)):
        assert pkv.pkv_check_device_errors(lay.pool) == 0
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), f"layer {l}: O differs"
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), f"layer {l}: LSE differs"
    # and against the oracle, for the first layer
    b = batches[0]
    kp, vp = b.pool_arrays()
    oracle.append(kp, vp, b.block_tables, b.cu_q_lens, b.q_positions, b.k_new, b.v_new)
    O, L = oracle.paged_attn(b.q, kp, vp, b.block_tables, b.ctx_lens, b.cu_q_lens, b.q_positions, b.scale)
    o = outs[0][0].float().cpu().numpy().astype(np.float64)
    assert (np.abs(o - O) <= ATOL + RTOL * np.abs(O)).all()
    assert np.abs(outs[0][1].cpu().numpy().astype(np.float64) - L).max() <= LSE_TOL
    for lay in layers:
        lay.pool.close()
